// Grouped GEMMs of the MoE layer on the 5th-generation tensor cores (tcgen05 + TMEM + TMA).
//
// Expert FFN (sebask.de MoK article, intro: up, gate and down projection; stamatios.com,
// "Outras caracteristicas": SwiGLU, router-weight gradient fused into the SwiGLU
// backward). One persistent, warp-specialised kernel serves every GEMM of the layer:
//
//   warp 0      TMA producer: one elected lane streams A/B tiles into a 4-stage ring of
//               shared-memory buffers (128-byte swizzle), mbarrier-tracked;
//   warp 1      MMA issuer: allocates 512 TMEM columns (two 128x256 fp32 accumulators)
//               and issues tcgen05.mma (M=128, N=256, K=16) from one lane;
//   warps 2..5  epilogue: tcgen05.ld the accumulator (one TMEM lane per output row),
//               apply the mode's fused math, store bf16 rows; the accumulator is handed
//               back so the next tile's MMAs overlap this tile's epilogue.
//
// Tiles of the routed row space are 128 rows of one expert (segments are padded to 128
// rows by the schedule), so a tile never mixes experts. Each output element is one fp32
// sum in a fixed K order, so results are bitwise reproducible. Every mbarrier wait is
// bounded by a deadline; on expiry the kernel records MOK_ERR_TIMEOUT in the status
// word, drains its outstanding copies and returns.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdio>
#include <cstring>
#include <mutex>

#include "mok_internal.h"
#include "mok_ptx.cuh"

namespace mok {

namespace {

constexpr int BM = 128;
constexpr int BK = 64;                      // bf16 elements per 128-byte swizzle row
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;        // 16 KB
constexpr int B_BYTES = 256 * BK * 2;       // 32 KB (N up to 256)
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int TMEM_COLS = 512;
constexpr int ACC_COLS = 256;
constexpr int NUM_THREADS = 192;
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 /*align*/ + 256 /*barriers*/;
constexpr uint64_t kTimeoutNs = 2000000000ull;

struct Params {
  int mode;
  int dense;        // 1: one group over M_rows rows (shared expert)
  int M_rows;       // dense rows (T)
  int H, I;         // hidden, intermediate of this FFN
  int k;            // top-k (gate lookup)
  int BN;           // MMA N (256 or 128)
  int n_tiles;      // tiles along N
  int m_tiles_dw;   // dW modes: tiles along M of one expert's dW
  int groups;
  int kiters;       // row-space modes: K / 64
  // schedule
  const int32_t* poff;
  const int32_t* counts;
  const int32_t* offsets;
  const int32_t* tile_expert;
  const int32_t* num_mtiles;
  const int32_t* table;
  const float* gates;
  // epilogue
  __nv_bfloat16* out0;
  __nv_bfloat16* out1;
  __nv_bfloat16* out2;
  const __nv_bfloat16* aux0;
  const __nv_bfloat16* aux1;
  float* dgp;
  uint32_t* status;
};

struct TileInfo {
  int e;        // expert (0 when dense)
  int row0;     // first row of the row space (row-space modes) / first dW row (dW modes)
  int n0;       // first output column
  int kiters;   // K iterations of 64
  int krow0;    // dW modes: first row of the contraction range
};

__device__ __forceinline__ bool is_dw(int mode) { return mode == kBwdDWDown || mode == kBwdDWUpGate; }

__device__ __forceinline__ int num_tiles_of(const Params& p) {
  if (is_dw(p.mode)) return p.groups * p.m_tiles_dw * p.n_tiles;
  int mt = (p.M_rows + BM - 1) / BM;            // dense rows, or the padded-row bound
  if (!p.dense) mt = min(max(*p.num_mtiles, 0), mt);
  return mt * p.n_tiles;
}

__device__ __forceinline__ TileInfo tile_info(const Params& p, int tile) {
  TileInfo ti;
  if (is_dw(p.mode)) {
    const int per_e = p.m_tiles_dw * p.n_tiles;
    ti.e = tile / per_e;
    const int rem = tile - ti.e * per_e;
    const int mt = rem / p.n_tiles;
    ti.row0 = mt * BM;
    ti.n0 = (rem - mt * p.n_tiles) * (p.mode == kBwdDWUpGate ? 128 : p.BN);
    if (p.dense) {
      ti.krow0 = 0;
      ti.kiters = (p.M_rows + BK - 1) / BK;
    } else {
      ti.krow0 = p.poff[ti.e];
      ti.kiters = (p.poff[ti.e + 1] - ti.krow0) / BK;
    }
  } else {
    const int mt = tile / p.n_tiles;
    ti.e = p.dense ? 0 : min(max(p.tile_expert[mt], 0), p.groups - 1);
    ti.row0 = mt * BM;
    ti.n0 = (tile - mt * p.n_tiles) * (p.mode == kFwdUpGate ? 128 : p.BN);
    ti.kiters = p.kiters;
    ti.krow0 = 0;
  }
  return ti;
}

__device__ __forceinline__ void set_error(uint32_t* status, uint32_t bit) {
  atomicOr(status, bit);
}

__device__ __forceinline__ void store_bf16x32(__nv_bfloat16* dst, const float* v) {
  uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint4 w;
    __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&w);
#pragma unroll
    for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(v[8 * q + 2 * i], v[8 * q + 2 * i + 1]);
    d[q] = w;
  }
}
__device__ __forceinline__ void load_bf16x32(const __nv_bfloat16* src, float* v) {
  const uint4* s = reinterpret_cast<const uint4*>(src);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint4 w = __ldg(s + q);
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&w);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float2 f = __bfloat1622float2(h[i]);
      v[8 * q + 2 * i] = f.x;
      v[8 * q + 2 * i + 1] = f.y;
    }
  }
}
__device__ __forceinline__ float sigmoidf_(float v) { return 1.f / (1.f + __expf(-v)); }

// ------------------------------------------------------------------ producer
__device__ void produce(const Params& p, const CUtensorMap* tA0, const CUtensorMap* tA1,
                        const CUtensorMap* tB0, const CUtensorMap* tB1, uint8_t* smem,
                        uint64_t* full, uint64_t* empty, volatile int* abort_flag) {
  const int ntiles = num_tiles_of(p);
  uint32_t it = 0;
  const uint32_t b_bytes = (p.mode == kFwdUpGate || p.mode == kBwdDWUpGate) ? 256 * BK * 2
                                                                              : p.BN * BK * 2;
  bool ok = true;
  for (int tile = blockIdx.x; tile < ntiles && ok; tile += gridDim.x) {
    const TileInfo ti = tile_info(p, tile);
    for (int kb = 0; kb < ti.kiters; ++kb, ++it) {
      const int stage = it % STAGES;
      const uint32_t round = it / STAGES;
      if (round > 0 && !mbar_wait(&empty[stage], (round - 1) & 1, globaltimer_ns() + kTimeoutNs)) {
        set_error(p.status, kErrTimeout);
        *abort_flag = 1;
        ok = false;
        break;
      }
      uint8_t* sa = smem + stage * STAGE_BYTES;
      uint8_t* sb = sa + A_BYTES;
      mbar_arrive_expect_tx(&full[stage], A_BYTES + b_bytes);
      const int k0 = kb * BK;
      switch (p.mode) {
        case kFwdUpGate: {   // A: Xg rows (K-major); B: W_up|W_gate cols n0..n0+127 (MN-major)
          tma_load_2d(sa, tA0, &full[stage], k0, ti.row0);
          const int brow = ti.e * p.H + k0;
          tma_load_2d(sb + 0 * 8192, tB0, &full[stage], ti.n0, brow);
          tma_load_2d(sb + 1 * 8192, tB0, &full[stage], ti.n0 + 64, brow);
          tma_load_2d(sb + 2 * 8192, tB1, &full[stage], ti.n0, brow);
          tma_load_2d(sb + 3 * 8192, tB1, &full[stage], ti.n0 + 64, brow);
          break;
        }
        case kFwdDown: {     // A: h rows (K-major); B: W_down cols (MN-major)
          tma_load_2d(sa, tA0, &full[stage], k0, ti.row0);
          const int brow = ti.e * p.I + k0;
          for (int c = 0; c < p.BN / 64; ++c)
            tma_load_2d(sb + c * 8192, tB0, &full[stage], ti.n0 + 64 * c, brow);
          break;
        }
        case kBwdDH: {       // A: dYg rows (K-major); B: W_down rows i (K-major over H)
          tma_load_2d(sa, tA0, &full[stage], k0, ti.row0);
          tma_load_2d(sb, tB0, &full[stage], k0, ti.e * p.I + ti.n0);
          break;
        }
        case kBwdDX: {       // K = [I of du | I of dv]; B: W_up / W_gate rows h (K-major over I)
          const int half = p.I / BK;
          const bool second = kb >= half;
          const int kk = (second ? kb - half : kb) * BK;
          tma_load_2d(sa, second ? tA1 : tA0, &full[stage], kk, ti.row0);
          tma_load_2d(sb, second ? tB1 : tB0, &full[stage], kk, ti.e * p.H + ti.n0);
          break;
        }
        case kBwdDWDown: {   // A: (g h)^T (MN-major, M = I); B: dYg (MN-major, N = H)
          const int kr = ti.krow0 + k0;
          tma_load_2d(sa, tA0, &full[stage], ti.row0, kr);
          tma_load_2d(sa + 8192, tA0, &full[stage], ti.row0 + 64, kr);
          for (int c = 0; c < p.BN / 64; ++c)
            tma_load_2d(sb + c * 8192, tB0, &full[stage], ti.n0 + 64 * c, kr);
          break;
        }
        default: {           // kBwdDWUpGate: A: Xg^T (M = H); B: du | dv cols n0..n0+127
          const int kr = ti.krow0 + k0;
          tma_load_2d(sa, tA0, &full[stage], ti.row0, kr);
          tma_load_2d(sa + 8192, tA0, &full[stage], ti.row0 + 64, kr);
          tma_load_2d(sb + 0 * 8192, tB0, &full[stage], ti.n0, kr);
          tma_load_2d(sb + 1 * 8192, tB0, &full[stage], ti.n0 + 64, kr);
          tma_load_2d(sb + 2 * 8192, tB1, &full[stage], ti.n0, kr);
          tma_load_2d(sb + 3 * 8192, tB1, &full[stage], ti.n0 + 64, kr);
          break;
        }
      }
    }
  }
  // Drain: make sure every issued copy has landed and every MMA commit has arrived
  // before the CTA's shared memory goes away.
  const uint32_t n_armed = it;
  for (uint32_t s = 0; s < STAGES && s < n_armed; ++s) {
    const uint32_t last = ((n_armed - 1 - s) / STAGES) * STAGES + s;  // last use of stage s
    const uint32_t round = last / STAGES;
    if (!mbar_wait(&empty[s], round & 1, globaltimer_ns() + kTimeoutNs)) {
      set_error(p.status, kErrTimeout);
      mbar_wait(&full[s], round & 1, globaltimer_ns() + kTimeoutNs);
    }
  }
}

// ------------------------------------------------------------------ MMA issuer
__device__ void mma_issue(const Params& p, uint8_t* smem, uint64_t* full, uint64_t* empty,
                          uint64_t* acc_full, uint64_t* acc_empty, uint32_t tmem_base,
                          volatile int* abort_flag) {
  const int ntiles = num_tiles_of(p);
  uint32_t it = 0;
  int local = 0;
  // operand majorness and descriptor strides per mode
  bool a_mn = false, b_mn = false;
  int n_mma = p.BN;
  switch (p.mode) {
    case kFwdUpGate: b_mn = true; n_mma = 256; break;
    case kFwdDown: b_mn = true; break;
    case kBwdDH: break;
    case kBwdDX: break;
    case kBwdDWDown: a_mn = true; b_mn = true; break;
    default: a_mn = true; b_mn = true; n_mma = 256; break;
  }
  const uint32_t idesc = idesc_bf16(BM, n_mma, a_mn, b_mn);
  for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x, ++local) {
    const TileInfo ti = tile_info(p, tile);
    const int acc = local & 1;
    const uint32_t use = local >> 1;
    if (use > 0 && !mbar_wait(&acc_empty[acc], (use - 1) & 1, globaltimer_ns() + kTimeoutNs)) {
      set_error(p.status, kErrTimeout);
      *abort_flag = 1;
      return;
    }
    tc_fence_after();
    const uint32_t d_tmem = tmem_base + acc * ACC_COLS;
    for (int kb = 0; kb < ti.kiters; ++kb, ++it) {
      const int stage = it % STAGES;
      const uint32_t round = it / STAGES;
      if (!mbar_wait(&full[stage], round & 1, globaltimer_ns() + kTimeoutNs)) {
        set_error(p.status, kErrTimeout);
        *abort_flag = 1;
        return;
      }
      tc_fence_after();
      const uint32_t sa = smem_u32(smem + stage * STAGE_BYTES);
      const uint32_t sb = sa + A_BYTES;
#pragma unroll
      for (int kk = 0; kk < BK / 16; ++kk) {
        // K-major: the k-th 16-element slice starts 32 bytes further along the row.
        // MN-major: it starts 16 rows (2048 bytes) further; 64-element MN chunks are
        // 8 KB apart (leading byte offset), 8-row groups 1 KB apart (stride offset).
        const uint64_t ad = a_mn ? umma_desc_sw128(sa + kk * 2048, 8192, 1024)
                                 : umma_desc_sw128(sa + kk * 32, 16, 1024);
        const uint64_t bd = b_mn ? umma_desc_sw128(sb + kk * 2048, 8192, 1024)
                                 : umma_desc_sw128(sb + kk * 32, 16, 1024);
        umma_bf16(d_tmem, ad, bd, idesc, (kb > 0 || kk > 0) ? 1u : 0u);
      }
      umma_commit(&empty[stage]);   // frees the stage once these MMAs have read it
    }
    if (ti.kiters > 0) umma_commit(&acc_full[acc]);
    else mbar_arrive(&acc_full[acc]);  // nothing to accumulate: epilogue writes zeros
  }
}

// ------------------------------------------------------------------ epilogue
__device__ void epilogue(const Params& p, uint64_t* acc_full, uint64_t* acc_empty,
                         uint32_t tmem_base, volatile int* abort_flag) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int quarter = warp & 3;             // TMEM lanes 32*quarter .. +31
  const int r = quarter * 32 + lane;        // row inside the tile
  const int ntiles = num_tiles_of(p);
  int local = 0;
  for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x, ++local) {
    const TileInfo ti = tile_info(p, tile);
    const int acc = local & 1;
    const uint32_t use = local >> 1;
    if (!mbar_wait(&acc_full[acc], use & 1, globaltimer_ns() + kTimeoutNs)) {
      set_error(p.status, kErrTimeout);
      *abort_flag = 1;
      return;
    }
    tc_fence_after();
    const uint32_t t_row = tmem_base + acc * ACC_COLS + ((uint32_t)(quarter * 32) << 16);
    const bool have = ti.kiters > 0;
    float a[32], b[32];
    // tcgen05.ld is warp-collective: every lane loads, rows outside the problem only
    // skip their global loads and stores.
    const int row = ti.row0 + r;
    const bool valid = !(p.dense && !is_dw(p.mode) && row >= p.M_rows);
    switch (p.mode) {
      case kFwdUpGate: {
        const size_t o = (size_t)row * p.I + ti.n0;
        for (int c = 0; c < 4; ++c) {
          tmem_ld32(t_row + c * 32, a);          // U
          tmem_ld32(t_row + 128 + c * 32, b);    // V
          if (!valid) continue;
          float h[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) h[i] = b[i] * sigmoidf_(b[i]) * a[i];
          store_bf16x32(p.out0 + o + c * 32, h);
          store_bf16x32(p.out1 + o + c * 32, a);
          store_bf16x32(p.out2 + o + c * 32, b);
        }
        break;
      }
      case kFwdDown:
      case kBwdDX: {
        const size_t o = (size_t)row * p.H + ti.n0;
        for (int c = 0; c < p.BN / 32; ++c) {
          tmem_ld32(t_row + c * 32, a);
          if (valid) store_bf16x32(p.out0 + o + c * 32, a);
        }
        break;
      }
      case kBwdDH: {
        float g = 1.f;
        if (!p.dense) {
          const int rl = row - p.poff[ti.e];
          g = 0.f;
          if (rl < p.counts[ti.e]) {
            const int tr = p.offsets[ti.e] + rl;
            g = p.gates[(size_t)p.table[2 * tr] * p.k + p.table[2 * tr + 1]];
          }
        }
        const size_t o = (size_t)row * p.I + ti.n0;
        float dg = 0.f;
        for (int c = 0; c < p.BN / 32; ++c) {
          tmem_ld32(t_row + c * 32, a);          // D = dY W_down^T
          if (!valid) continue;
          float u[32], v[32];
          load_bf16x32(p.aux0 + o + c * 32, u);  // saved U
          load_bf16x32(p.aux1 + o + c * 32, v);  // saved V
          float du[32], dv[32], hg[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const float sg = sigmoidf_(v[i]);
            const float sl = v[i] * sg;
            const float hv = sl * u[i];
            dg = fmaf(a[i], hv, dg);
            const float dh = g * a[i];
            du[i] = dh * sl;
            dv[i] = dh * u[i] * (sg * (1.f + v[i] * (1.f - sg)));
            hg[i] = g * hv;
          }
          store_bf16x32(p.out0 + o + c * 32, du);
          store_bf16x32(p.out1 + o + c * 32, dv);
          store_bf16x32(p.out2 + o + c * 32, hg);
        }
        if (valid && p.dgp) p.dgp[(size_t)row * p.n_tiles + ti.n0 / p.BN] = dg;
        break;
      }
      case kBwdDWDown: {                         // row = i index of dW_down[e]
        __nv_bfloat16* dst = p.out0 + ((size_t)ti.e * p.I + row) * p.H + ti.n0;
        for (int c = 0; c < p.BN / 32; ++c) {
          if (have) tmem_ld32(t_row + c * 32, a);
          else {
#pragma unroll
            for (int i = 0; i < 32; ++i) a[i] = 0.f;
          }
          store_bf16x32(dst + c * 32, a);
        }
        break;
      }
      default: {                                 // kBwdDWUpGate; row = h index
        const size_t o = ((size_t)ti.e * p.H + row) * p.I + ti.n0;
        for (int c = 0; c < 4; ++c) {
          if (have) {
            tmem_ld32(t_row + c * 32, a);
            tmem_ld32(t_row + 128 + c * 32, b);
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) a[i] = b[i] = 0.f;
          }
          store_bf16x32(p.out0 + o + c * 32, a);
          store_bf16x32(p.out1 + o + c * 32, b);
        }
        break;
      }
    }
    tc_fence_before();
    mbar_arrive(&acc_empty[acc]);
  }
}

__global__ void __launch_bounds__(NUM_THREADS, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tA0, const __grid_constant__ CUtensorMap tA1,
                        const __grid_constant__ CUtensorMap tB0, const __grid_constant__ CUtensorMap tB1,
                        const Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE_BYTES);
  uint64_t* empty = full + STAGES;
  uint64_t* acc_full = empty + STAGES;
  uint64_t* acc_empty = acc_full + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_empty + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&acc_full[a], 1);
      mbar_init(&acc_empty[a], 128);
    }
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tA0);
    tma_prefetch_desc(&tB0);
  }
  if (warp == 1) tmem_alloc(tmem_slot, TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    if (threadIdx.x == 0) produce(p, &tA0, &tA1, &tB0, &tB1, smem, full, empty, abort_flag);
  } else if (warp == 1) {
    if ((threadIdx.x & 31) == 0)
      mma_issue(p, smem, full, empty, acc_full, acc_empty, tmem_base, abort_flag);
  } else {
    epilogue(p, acc_full, acc_empty, tmem_base, abort_flag);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

// ------------------------------------------------------------------ host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// 2-D bf16 tensor map over a row-major [rows][cols] matrix, box (64 cols, box_rows rows),
// 128-byte swizzle; reads outside the matrix return zeros.
bool make_map(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows, int box_rows) {
  EncodeTiledFn enc = get_encode_fn();
  if (!enc || base == nullptr) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace

int gemm_dh_parts(int I) { return (I % 256 == 0) ? I / 256 : I / 128; }

cudaError_t launch_gemm(const GemmCall& c, int num_sms, cudaStream_t s) {
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(grouped_gemm_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  Params p;
  memset(&p, 0, sizeof(p));
  p.mode = c.mode;
  p.dense = c.dense ? 1 : 0;
  p.M_rows = c.M_rows;
  p.H = c.H;
  p.I = c.I;
  p.k = c.k;
  p.groups = c.dense ? 1 : c.groups;
  p.poff = c.poff;
  p.counts = c.counts;
  p.offsets = c.offsets;
  p.tile_expert = c.tile_expert;
  p.num_mtiles = c.num_mtiles;
  p.table = c.table;
  p.gates = c.gates;
  p.out0 = static_cast<__nv_bfloat16*>(c.out0);
  p.out1 = static_cast<__nv_bfloat16*>(c.out1);
  p.out2 = static_cast<__nv_bfloat16*>(c.out2);
  p.aux0 = static_cast<const __nv_bfloat16*>(c.aux0);
  p.aux1 = static_cast<const __nv_bfloat16*>(c.aux1);
  p.dgp = c.dgp;
  p.status = c.status;

  const uint64_t rows = (uint64_t)c.M_rows;  // rows of the row-space buffers
  const uint64_t G = (uint64_t)p.groups;
  CUtensorMap tA0, tA1, tB0, tB1;
  memset(&tA1, 0, sizeof(tA1));
  memset(&tB1, 0, sizeof(tB1));
  bool ok = true;
  int max_tiles = 0;
  const int mt_rows = (int)((rows + BM - 1) / BM);
  switch (c.mode) {
    case kFwdUpGate:
      p.BN = 256;
      p.n_tiles = c.I / 128;
      p.kiters = c.H / BK;
      ok = make_map(&tA0, c.a0, c.H, rows, BM) && make_map(&tB0, c.b0, c.I, G * c.H, BK) &&
           make_map(&tB1, c.b1, c.I, G * c.H, BK);
      max_tiles = mt_rows * p.n_tiles;
      break;
    case kFwdDown:
      p.BN = (c.H % 256 == 0) ? 256 : 128;
      p.n_tiles = c.H / p.BN;
      p.kiters = c.I / BK;
      ok = make_map(&tA0, c.a0, c.I, rows, BM) && make_map(&tB0, c.b0, c.H, G * c.I, BK);
      max_tiles = mt_rows * p.n_tiles;
      break;
    case kBwdDH:
      p.BN = (c.I % 256 == 0) ? 256 : 128;
      p.n_tiles = c.I / p.BN;
      p.kiters = c.H / BK;
      ok = make_map(&tA0, c.a0, c.H, rows, BM) && make_map(&tB0, c.b0, c.H, G * c.I, p.BN);
      max_tiles = mt_rows * p.n_tiles;
      break;
    case kBwdDX:
      p.BN = (c.H % 256 == 0) ? 256 : 128;
      p.n_tiles = c.H / p.BN;
      p.kiters = 2 * (c.I / BK);
      ok = make_map(&tA0, c.a0, c.I, rows, BM) && make_map(&tA1, c.a1, c.I, rows, BM) &&
           make_map(&tB0, c.b0, c.I, G * c.H, p.BN) && make_map(&tB1, c.b1, c.I, G * c.H, p.BN);
      max_tiles = mt_rows * p.n_tiles;
      break;
    case kBwdDWDown:
      p.BN = (c.H % 256 == 0) ? 256 : 128;
      p.n_tiles = c.H / p.BN;
      p.m_tiles_dw = c.I / BM;
      ok = make_map(&tA0, c.a0, c.I, rows, BK) && make_map(&tB0, c.b0, c.H, rows, BK);
      max_tiles = p.groups * p.m_tiles_dw * p.n_tiles;
      break;
    case kBwdDWUpGate:
      p.BN = 256;
      p.n_tiles = c.I / 128;
      p.m_tiles_dw = c.H / BM;
      ok = make_map(&tA0, c.a0, c.H, rows, BK) && make_map(&tB0, c.b0, c.I, rows, BK) &&
           make_map(&tB1, c.b1, c.I, rows, BK);
      max_tiles = p.groups * p.m_tiles_dw * p.n_tiles;
      break;
  }
  if (!ok) return cudaErrorInvalidValue;
  if (c.mode != kBwdDX) tA1 = tA0;  // second maps only used by the modes that set them
  if (c.mode == kFwdDown || c.mode == kBwdDH || c.mode == kBwdDWDown) tB1 = tB0;
  int grid = max_tiles < num_sms ? max_tiles : num_sms;
  if (grid < 1) grid = 1;
  grouped_gemm_kernel<<<grid, NUM_THREADS, SMEM_BYTES, s>>>(tA0, tA1, tB0, tB1, p);
  return cudaGetLastError();
}

}  // namespace mok
