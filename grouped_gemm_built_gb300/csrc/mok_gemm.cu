// Grouped GEMMs of the MoE layer on the 5th-generation tensor cores (tcgen05 + TMEM + TMA).
//
// Expert FFN (sebask.de MoK article, intro: up, gate and down projection; stamatios.com,
// "Outras caracteristicas": SwiGLU, router-weight gradient fused into the SwiGLU
// backward, MXFP8 with a BF16 shared expert). One persistent, warp-specialised kernel
// template serves every GEMM of the layer, instantiated per mode (and, for the dW modes,
// per hi/lo split) so that each launch carries only its own code:
//
//   warp 0      TMA producer: one lane streams A/B tiles (and, in MXFP8, their scale
//               atoms) into a ring of shared-memory stages (128-byte swizzle);
//   warp 1      MMA issuer: allocates 512 TMEM columns and issues tcgen05.mma
//               (M=128, N=256) from one lane; BF16: kind::f16, K=16 per instruction, two
//               256-column accumulators; MXFP8: kind::mxf8f6f4.block_scale, K=32 per
//               instruction, one 256-column accumulator (dH: two of 128 columns) plus
//               per-stage scale columns filled by tcgen05.cp;
//   warps 2..5  epilogue: tcgen05.ld the accumulator (one TMEM lane per output row), run
//               the mode's fused math, stage 32-row boxes in shared memory and store them
//               with TMA; with two accumulators the next tile's MMAs overlap this epilogue.
//
// Tiles of the routed row space are 128 rows of one expert (segments are padded to 128
// rows by the schedule), so a tile never mixes experts. Each output element is one fp32
// sum in a fixed K order, so results are bitwise reproducible.
//
// Precision of the BF16 backward: the computed operands du, dv and g*h are also kept as a
// pair of bf16 values (hi = bf16(v), lo = bf16(v - hi)); the dW GEMMs run both halves of
// each K chunk back to back into the same fp32 accumulator, so there these operands carry
// a 16-bit significand while the tensor cores still take bf16. (The dX GEMM sums over I
// and takes the bf16 hi parts only.) One pipeline stage then holds a K chunk of the other
// operand once and both halves of the split one (SPLIT_STAGE_BYTES), so the shared
// operand crosses shared memory once per chunk.
//
// Every mbarrier wait is bounded by a deadline; on expiry the kernel records
// MOK_ERR_TIMEOUT in the status word, drains its outstanding copies and returns.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include <cstdio>
#include <cstring>
#include <mutex>

#include "mok_internal.h"
#include "mok_mx.cuh"
#include "mok_ptx.cuh"

namespace mok {

namespace {

constexpr int BM = 128;
constexpr int A_BYTES = 16384;              // 128 rows x 128 bytes
constexpr int B_BYTES = 32768;              // 256 rows x 128 bytes
constexpr int TMEM_COLS = 512;
constexpr int NUM_THREADS = 192;
constexpr uint64_t kTimeoutNs = 2000000000ull;
constexpr int STAGE_OUT_BYTES = 4096;               // one 32-row epilogue staging box
constexpr int TQ = 4;                               // slots of the dynamic tile queue
constexpr int OUT_STAGING = 4 * 2 * STAGE_OUT_BYTES;  // 4 epilogue warps x 2 buffers
// split (hi/lo) dW stage: [A 16 KB][B 32 KB][second half: B lo 32 KB, or A lo 16 KB]
constexpr int SPLIT_STAGE_BYTES = A_BYTES + 2 * B_BYTES;
constexpr int SPLIT_EXTRA_OFF = A_BYTES + B_BYTES;
// row-tile pair stage (BF16): [A0 16 KB][B 32 KB][A1 16 KB]
constexpr int PAIR_STAGE_BYTES = 2 * A_BYTES + B_BYTES;
constexpr int PAIR_A1_OFF = A_BYTES + B_BYTES;
// SM-pair dW stage (BF16, clusters of two CTAs): [A: this CTA's 128 rows][B: its half of the
// tile's columns, at most 128], 16 KB each; six stages and two staging boxes per warp
constexpr int SMP_STAGE_BYTES = 2 * A_BYTES;
constexpr int SMP_STAGES = 6;

template <bool MX>
struct Cfg {
  // barrier slots: the most stages a launch uses (MXFP8: 3 or 4 full stages, or 6 of the
  // dH launch's 128-column tiles, which need a third less)
  static constexpr int STAGES = MX ? 6 : 4;
  static constexpr int BK = MX ? 128 : 64;           // K elements per stage (128 bytes/row)
  static constexpr int MMA_K = MX ? 32 : 16;         // K elements per instruction
  static constexpr int MN_CHUNK = MX ? 128 : 64;     // elements per 128-byte MN-major chunk
  static constexpr int MN_LBO = BK * 128;            // bytes between MN chunks in smem
  static constexpr int MN_KSTEP = MMA_K * 128;       // bytes per instruction along K, MN-major
  static constexpr int SF_OFF = A_BYTES + B_BYTES;   // scale atoms: A 512 B, B 1024 B
  static constexpr int STAGE_BYTES = MX ? 51200 : 49152;
  static constexpr int MX_STAGES = 3;                // MXFP8 stages of STAGE_BYTES (up|gate: 4)
  static constexpr int MX_DH_STAGE_BYTES = 67584;    // 2 x (A 16 KB, B 16 KB, atoms 1 KB)
  static constexpr int MX_DH_STAGES = 3;
  static constexpr int NACC = MX ? 1 : 2;             // accumulators of ACC_COLS columns
  static constexpr int ACC_COLS = 256;
  static constexpr int SF_TMEM = 256;                // MX: scale columns start here
  // data area, then barriers. BF16: the larger of (STAGES stages + 2 staging boxes per
  // warp) and (STAGES - 1 stages + 4 staging boxes per warp). MXFP8 (one accumulator per
  // tile), per mode: the up|gate launch takes 4 stages and 1 staging box per warp (its
  // tiles' K is long, the operands in flight bound it); the launches that store 256
  // columns of results per tile take 3 stages and 4 boxes per warp, which hold a whole
  // 128 x 256 tile of bf16 results, so the tile leaves its accumulator at once and the
  // stores drain during the next tile's MMAs; dH (plain stores) takes 6 of its smaller
  // stages. The largest of the three.
  static constexpr int DATA_BYTES =
      MX ? (4 * STAGE_BYTES + OUT_STAGING / 2)
         : ((STAGES * STAGE_BYTES + OUT_STAGING > (STAGES - 1) * STAGE_BYTES + 2 * OUT_STAGING)
                ? STAGES * STAGE_BYTES + OUT_STAGING
                : (STAGES - 1) * STAGE_BYTES + 2 * OUT_STAGING);
  // + 1024 alignment slack, + barriers and flags (256), + the cluster-launch-control
  // barrier and answer (at BAR_BYTES / 2 of the barrier area)
  static constexpr int BAR_BYTES = 512;
  static constexpr int SMEM_BYTES = DATA_BYTES + 1024 + BAR_BYTES;
};

// Tensor maps of one launch: operands a[], b[] (loads) and outputs o[] (stores).
struct Maps {
  CUtensorMap a[4];
  CUtensorMap b[4];
  CUtensorMap o[6];
};

struct Params {
  int mode;
  int dense;        // 1: one group over M_rows rows (shared expert)
  int M_rows;       // rows of the row space (dense: T)
  int H, I;         // hidden, intermediate of this FFN
  int k;            // top-k (gate lookup)
  int BN;           // MMA N (256 or 128)
  int n_tiles;      // tiles along N
  int m_tiles_dw;   // dW modes: tiles along M of one expert's dW
  int groups;
  int kiters;       // row-space modes: K iterations per tile
  int split;        // 1: the dW GEMMs run hi and lo halves of their computed operand
  int stage_bytes;  // bytes of one pipeline stage (Cfg::STAGE_BYTES or SPLIT_STAGE_BYTES)
  int sf_off;       // MXFP8: offset of the stage's scale atoms
  int kdouble;      // MXFP8 dH: a stage holds two 128-element K chunks of each operand (A0,
                    // A1, B0, B1 of 16 KB, then the atoms A0, A1, B0, B1): half the barrier,
                    // scale-copy and commit work per MMA of these short 128-column tiles
  int lo_out;       // kBwdDH (bf16): also write the lo halves of du, dv, g*h
  int out_bf16;     // kFwdDown, kBwdDX, dW modes: round the outputs to bf16 (64-column boxes)
  int* tile_counter;// dynamic tile order: the next tile is atomicAdd(tile_counter, 1) (zero at
                    // launch); null: the static order (tile blockIdx.x, + gridDim.x, ...)
  int clc;          // cluster launch control: one CTA per tile; a CTA runs tile blockIdx.x,
                    // then the tiles of the not yet launched CTAs it cancels
  int pair;         // BF16 routed up|gate, down and dX: a tile is a pair of row tiles of one
                    // expert (ptile), two M=128 accumulators side by side against one
                    // weight tile; stages [A0 | B | A1]
  const int32_t* ptile;
  const int32_t* num_ptiles;
  int max_ptiles;
  // MXFP8 forward launches that also run the BF16 shared expert ([C] "Outras
  // caracteristicas": MXFP8 training with the shared expert in BF16): shared_tiles BF16
  // tiles follow the routed ones (kernel variant 3), with their own maps a[2], b[2..3],
  // o[3..5]: s_rows = T rows, s_n_tiles column tiles of s_BN, s_kiters K blocks of 64
  int shared_tiles;
  int s_rows, s_n_tiles, s_kiters, s_BN, s_I;
  uint64_t timeout_ns;  // bound of every wait (MOK_ERR_TIMEOUT when it passes)
  int n_out;        // kRouter: output columns (E)
  const float* bias;// kRouter: logit bias or null
  float* logits;    // kRouter: [M_rows][n_out]
  int stages;       // shared-memory stages of the operand ring
  int nbuf;         // epilogue staging boxes per warp (2 or 4)
  int nacc;         // TMEM accumulators (Cfg::NACC; MXFP8 dH: 2 of 128 columns)
  int acc_cols;     // columns of one accumulator
  // schedule
  const int32_t* poff;
  const int32_t* counts;
  const int32_t* offsets;
  const int32_t* tile_expert;
  const int32_t* num_mtiles;
  const int32_t* table;
  const float* gates;
  // epilogue inputs
  const void* u;    // kBwdDH: saved U, V [rows][I] bf16
  const void* v;
  const int32_t* uv_row;   // kBwdDH: row of U, V per row of the row space (null: the same)
  float* dgp;
  uint32_t* status;
  // MXFP8 scale atoms (512 B each): A side [row tile][kcs_a], B side [e][kcs_b][ncs_b]
  const uint8_t* sfa;
  const uint8_t* sfa1;
  const uint8_t* sfb0;
  const uint8_t* sfb1;
  int kcs_a, kcs_b, ncs_b;
  // MX outputs. kFwdUpGate: q[0] = h along I. kBwdDH: q[0], q[1] = du, dv along I;
  // q[2], q[3], q[4] = du, dv, g*h in 32-row blocks. E4M3 [rows][I], atoms [row tile][I/128].
  uint8_t* out_q[5];
  uint8_t* out_sf[5];
  int smpair;       // BF16 dW modes on SM pairs: the two CTAs of a cluster share M = 256
                    // MMAs (rank 0 issues them); a tile is 256 rows of dW, 128 per CTA, and
                    // each CTA loads its A rows and half of the B columns
  int crank;        // SM pairs: this CTA's rank in its cluster (set at kernel entry)
  int t0, tstep;    // SM pairs, static order: the cluster's index and the cluster count
};

struct TileInfo {
  int e;        // expert (0 when dense)
  int row0;     // first row of the row space (row-space modes) / first dW row (dW modes)
  int arow0;    // row-space modes: first row of the A operand (row0 unless A lives elsewhere)
  int n0;       // first output column
  int kiters;   // K iterations
  int krow0;    // dW modes: first row of the contraction range
  int klast;    // dW modes: MMA K steps of the last K iteration that hold rows
  int skip;     // 1: no tile here (the unmatched half of the last row-tile pair)
  int nrt;      // row tiles in this tile: 1, or 2 (a row-tile pair: rows row0 .. row0+255)
  int bf;       // 1: a BF16 shared-expert tile of an MXFP8 forward launch (rows of x / hs)
  int norows;   // SM pairs, row-space modes: this CTA's half of the pair tile has no rows
                // (the pair's odd last row tile): it loads and takes part, writes nothing
};

__host__ __device__ __forceinline__ bool is_dw(int mode) { return mode == kBwdDWDown || mode == kBwdDWUpGate; }

__device__ __forceinline__ int routed_mtiles(const Params& p) {
  return min(max(*p.num_mtiles, 0), (p.M_rows + BM - 1) / BM);
}

// Routed row-space modes number their tiles in pairs of row tiles: tile 2g + r is row tile
// 2 (g / n_tiles) + r of column block g mod n_tiles. The two row tiles of a pair usually
// belong to one expert and read the same weight slice; with this order two neighbouring
// CTAs take them in the same round, so the second read of the slice is an L2 hit.
__device__ __forceinline__ int num_tiles_of(const Params& p) {
  if (is_dw(p.mode)) return p.groups * (p.smpair ? p.m_tiles_dw / 2 : p.m_tiles_dw) * p.n_tiles;
  if (p.smpair) {   // row-space modes on SM pairs: pairs of row tiles
    if (p.dense) return (((p.M_rows + BM - 1) / BM + 1) / 2) * p.n_tiles;
    return min(max(*p.num_ptiles, 0), p.max_ptiles) * p.n_tiles;
  }
  if (p.pair) return min(max(*p.num_ptiles, 0), p.max_ptiles) * p.n_tiles;
  if (p.dense) return ((p.M_rows + BM - 1) / BM) * p.n_tiles;
  return ((routed_mtiles(p) + 1) / 2) * 2 * p.n_tiles + p.shared_tiles;
}

template <bool MX>
__device__ __forceinline__ TileInfo tile_info(const Params& p, int tile) {
  constexpr int BK = Cfg<MX>::BK;
  constexpr int MMA_K = Cfg<MX>::MMA_K;
  TileInfo ti;
  ti.skip = 0;
  ti.nrt = 1;
  ti.bf = 0;
  ti.norows = 0;
  ti.klast = BK / MMA_K;
  if (p.smpair && !is_dw(p.mode)) {
    // SM pair over a pair of row tiles of one expert (routed: the plan's list; dense:
    // consecutive): rank 0 takes the first, rank 1 the second, or no rows when there is none
    const int q = tile / p.n_tiles;
    const int nt = tile - q * p.n_tiles;
    int mt, two;
    if (p.dense) {
      mt = 2 * q;
      two = mt + 1 < (p.M_rows + BM - 1) / BM;
      ti.e = 0;
    } else {
      const int pt = p.ptile[q];
      mt = pt >> 1;
      ti.skip = mt >= routed_mtiles(p);   // both CTAs see the same list entry
      two = (pt & 1) && mt + 1 < routed_mtiles(p);
      ti.e = ti.skip ? 0 : min(max(p.tile_expert[mt], 0), p.groups - 1);
      if (ti.skip) mt = 0;
    }
    ti.norows = p.crank == 1 && !two;
    ti.row0 = (mt + p.crank) * BM;
    ti.arow0 = ti.row0;
    ti.n0 = nt * p.BN;
    ti.kiters = p.kiters;
    ti.krow0 = 0;
    return ti;
  }
  if (p.pair) {   // tile = pair q of column block nt; the pair's tiles share the expert
    const int q = tile / p.n_tiles;
    const int nt = tile - q * p.n_tiles;
    const int pt = p.ptile[q];
    const int mt = pt >> 1;
    ti.skip = mt >= routed_mtiles(p);
    ti.nrt = (pt & 1) && mt + 1 < routed_mtiles(p) ? 2 : 1;
    ti.e = ti.skip ? 0 : min(max(p.tile_expert[mt], 0), p.groups - 1);
    ti.row0 = ti.skip ? 0 : mt * BM;
    ti.n0 = nt * (p.mode == kFwdUpGate ? 128 : p.BN);
    ti.kiters = p.kiters;
    ti.krow0 = 0;
    ti.arow0 = ti.row0;
    return ti;
  }
  if (is_dw(p.mode)) {
    const int per_e = (p.smpair ? p.m_tiles_dw / 2 : p.m_tiles_dw) * p.n_tiles;
    ti.e = tile / per_e;
    const int rem = tile - ti.e * per_e;
    const int mt = rem / p.n_tiles;
    ti.row0 = (p.smpair ? 2 * mt + p.crank : mt) * BM;   // SM pair: this CTA's 128 rows
    ti.n0 = (rem - mt * p.n_tiles) * (p.mode == kBwdDWUpGate ? 128 : p.BN);
    int krows;
    if (p.dense) {
      ti.krow0 = 0;
      krows = p.M_rows;
      ti.kiters = (p.M_rows + BK - 1) / BK;
    } else {
      // the expert's rows rounded up to the K step; the segment's padding rows are zero
      ti.krow0 = p.poff[ti.e];
      krows = max(p.counts[ti.e], 0);
      ti.kiters = min((krows + BK - 1) / BK, (p.poff[ti.e + 1] - ti.krow0) / BK);
    }
    // the last K iteration's MMAs stop after the last row (the rest would add zeros)
    if (ti.kiters > 0) {
      const int rem = krows - (ti.kiters - 1) * BK;
      if (rem > 0 && rem < BK) ti.klast = (rem + MMA_K - 1) / MMA_K;
    }
  } else {
    int mt, nt;
    const int nr = p.shared_tiles ? ((routed_mtiles(p) + 1) / 2) * 2 * p.n_tiles : 0;
    if (p.shared_tiles && tile >= nr) {   // a BF16 shared-expert tile after the routed ones
      const int l = tile - nr;
      mt = l / p.s_n_tiles;
      ti.bf = 1;
      ti.e = 0;
      ti.row0 = mt * BM;
      ti.arow0 = ti.row0;
      ti.n0 = (l - mt * p.s_n_tiles) * (p.mode == kFwdUpGate ? 128 : p.s_BN);
      ti.kiters = p.s_kiters;
      ti.krow0 = 0;
      return ti;
    }
    if (p.dense) {
      mt = tile / p.n_tiles;
      nt = tile - mt * p.n_tiles;
    } else {
      const int g = tile >> 1;
      mt = (g / p.n_tiles) * 2 + (tile & 1);
      nt = g % p.n_tiles;
      ti.skip = mt >= routed_mtiles(p);
      if (ti.skip) mt = 0;
    }
    ti.e = p.dense ? 0 : min(max(p.tile_expert[mt], 0), p.groups - 1);
    ti.row0 = mt * BM;
    ti.n0 = nt * (p.mode == kFwdUpGate ? 128 : p.BN);
    ti.kiters = p.kiters;
    ti.krow0 = 0;
  }
  ti.arow0 = ti.row0;
  return ti;
}

__device__ __forceinline__ void set_error(uint32_t* status, uint32_t bit) {
  atomicOr(status, bit);
}

// Fast division: the SwiGLU epilogues run one warp per SM sub-partition and are
// latency-bound; IEEE division made the MXFP8 forward up|gate launch 19% slower.
__device__ __forceinline__ void load_bf16x32(const __nv_bfloat16* src, float* v) {
  const uint4* s = reinterpret_cast<const uint4*>(src);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const uint4 w = __ldg(s + q);
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&w);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = __bfloat1622float2(h[i]);
      v[8 * q + 2 * i] = f.x;
      v[8 * q + 2 * i + 1] = f.y;
    }
  }
}
__device__ __forceinline__ float sigmoidf_(float v) { return __fdividef(1.f, 1.f + __expf(-v)); }

// bf16 pair of an fp32 value: hi = bf16(v), lo = bf16(v - hi) (v - hi is exact in fp32).
__device__ __forceinline__ void split_bf16(const float* v, float* hi, float* lo) {
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    hi[i] = __bfloat162float(__float2bfloat16_rn(v[i]));
    lo[i] = v[i] - hi[i];
  }
}

// MXFP8 block of 32 (one thread's chunk): returns the scale byte, writes 32 E4M3 codes.
__device__ __forceinline__ uint32_t quant32_e4m3(const float* v, uint4* q2) {
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(v[i]));
  uint32_t sb = 127u;
  if (amax != 0.f) {
    const int b = (int)((__float_as_uint(amax) >> 23) & 0xFF) - 8;
    sb = (uint32_t)(b < 0 ? 0 : b);
  }
  const float inv = __uint_as_float((254u - sb) << 23);
  uint32_t w[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(v[4 * i] * inv, v[4 * i + 1] * inv),
                                                 __NV_SATFINITE, __NV_E4M3);
    const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(v[4 * i + 2] * inv, v[4 * i + 3] * inv),
                                                 __NV_SATFINITE, __NV_E4M3);
    w[i] = (lo & 0xFFFFu) | (hi << 16);
  }
  q2[0] = make_uint4(w[0], w[1], w[2], w[3]);
  q2[1] = make_uint4(w[4], w[5], w[6], w[7]);
  return sb;
}

// MXFP8 blocks of 32 rows (the warp's rows, one per lane) for this lane's 32 columns of
// one row: per column a warp-wide maximum gives the block's scale; lane i keeps the scale
// of column i. Writes the row's 32 codes (when valid) and this lane's scale byte.
__device__ __forceinline__ void quant_rowblock(const float (&x)[32], int lane, bool valid,
                                               uint8_t* codes, uint8_t* scale) {
  uint32_t w[8];
  uint32_t my_sb = 127u;
#pragma unroll
  for (int i = 0; i < 32; i += 2) {
    // two columns per step: each its own warp-wide maximum and scale, one conversion
    float inv[2];
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      const uint32_t am = __reduce_max_sync(0xffffffffu, __float_as_uint(fabsf(x[i + c])));
      uint32_t sb = 127u;
      if (am != 0u) {
        const int bb = (int)((am >> 23) & 0xFF) - 8;
        sb = (uint32_t)(bb < 0 ? 0 : bb);
      }
      if (i + c == lane) my_sb = sb;
      inv[c] = __uint_as_float((254u - sb) << 23);
    }
    const uint32_t code2 = __nv_cvt_float2_to_fp8x2(make_float2(x[i] * inv[0], x[i + 1] * inv[1]),
                                                    __NV_SATFINITE, __NV_E4M3) & 0xFFFFu;
    if ((i & 3) == 0) w[i >> 2] = 0;
    w[i >> 2] |= code2 << (8 * (i & 3));
  }
  if (valid) {
    uint4* dq = reinterpret_cast<uint4*>(codes);
    dq[0] = make_uint4(w[0], w[1], w[2], w[3]);
    dq[1] = make_uint4(w[4], w[5], w[6], w[7]);
  }
  *scale = (uint8_t)my_sb;
}

// Epilogue output path: a warp stages its 32 rows x 128 bytes in shared memory (swizzled
// like the TMA box, so the 16-byte stores of 32 lanes spread over all banks) and one lane
// stores the box with TMA. Two buffers per warp: a buffer is refilled only after the TMA
// store issued two boxes earlier has finished reading it. Every lane calls these.
struct Stager {
  uint8_t* buf;   // this warp's nbuf x 4 KB, 1024-byte aligned
  uint32_t n;
  int lane;
  int nbuf;       // 2 or 4
  __device__ __forceinline__ uint8_t* next() {
    uint8_t* b = buf + (n & (nbuf - 1)) * STAGE_OUT_BYTES;
    if (n >= (uint32_t)nbuf && lane == 0) {
      if (nbuf == 4) bulk_wait_read<3>();
      else if (nbuf == 2) bulk_wait_read<1>();
      else bulk_wait_read<0>();
    }
    __syncwarp();
    return b;
  }
  __device__ __forceinline__ void issue(const CUtensorMap* m, const uint8_t* b, int col, int row) {
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      tma_store_2d(m, b, col, row);
      bulk_commit();
    }
    ++n;
  }
  // 32 fp32 of this lane's row -> box (32 cols, 32 rows), 128-byte swizzle
  __device__ __forceinline__ void f32(const CUtensorMap* m, const float* v, int col, int row) {
    uint8_t* b = next();
    uint8_t* r = b + lane * 128;
#pragma unroll
    for (int j = 0; j < 8; ++j)
      *reinterpret_cast<float4*>(r + ((j ^ (lane & 7)) << 4)) =
          make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
    issue(m, b, col, row);
  }
  // 32 bf16 of this lane's row -> box (32 cols, 32 rows), 64-byte swizzle
  __device__ __forceinline__ void bf16(const CUtensorMap* m, const float* v, int col, int row) {
    uint8_t* b = next();
    uint8_t* r = b + lane * 64;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      uint4 w;
      __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&w);
#pragma unroll
      for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(v[8 * j + 2 * i], v[8 * j + 2 * i + 1]);
      *reinterpret_cast<uint4*>(r + ((j ^ ((lane >> 1) & 3)) << 4)) = w;
    }
    issue(m, b, col, row);
  }
  // 64 values of this lane's row (v0: columns 0..31, v1: 32..63), rounded to bf16 ->
  // box (64 cols, 32 rows), 128-byte rows with the 128-byte swizzle of the fp32 boxes: half
  // the bytes of two fp32 boxes in one store
  __device__ __forceinline__ void bf16x64(const CUtensorMap* m, const float* v0, const float* v1,
                                          int col, int row) {
    uint8_t* b = next();
    uint8_t* r = b + lane * 128;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float* v = j < 4 ? v0 + 8 * j : v1 + 8 * (j - 4);
      uint4 w;
      __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&w);
#pragma unroll
      for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
      *reinterpret_cast<uint4*>(r + ((j ^ (lane & 7)) << 4)) = w;
    }
    issue(m, b, col, row);
  }
  __device__ __forceinline__ void drain() {
    if (lane == 0) bulk_wait_all();
    __syncwarp();
  }
};

// ------------------------------------------------------------------ tile order
// Static order: CTA b takes tiles b, b + G, b + 2G, ... (SM pairs: cluster b of G, both of
// its CTAs the same tiles, each its half of the rows). Dynamic order (a tile counter in
// global memory): the producer lane of each CTA takes the next tile with an atomic add when
// it is ready for one, and passes it to the CTA's MMA lane and epilogue warps through a
// queue of TQ slots in shared memory (slot q: tile id, "full" barrier of 1 arrival, "empty"
// barrier of 5: the MMA lane and one lane per epilogue warp). A CTA whose tiles run long
// then simply takes fewer of them. The queue ends with tile -1. Cluster launch control
// ([I], the paragraph on CLC) feeds the same queue: the grid has a CTA per tile, a CTA
// starts with tile blockIdx.x, and the producer lane asks the hardware to cancel a CTA that
// has not been launched yet and takes over its tile; it asks for the next one as soon as it
// starts a tile, so the answer is there when the tile's loads are issued. Which CTA runs a
// tile changes nothing in it: each output tile is one CTA's fixed-order sum in every order.
struct TileQueue {
  volatile int* tile;
  uint64_t* full;
  uint64_t* empty;
};

// Producer: publish entry n (tile id or -1). False after a timed-out wait.
__device__ __forceinline__ bool tq_publish(const Params& p, const TileQueue& tq, uint32_t n,
                                           int tile) {
  const int q = n % TQ;
  const uint32_t round = n / TQ;
  if (round > 0 && !mbar_wait(&tq.empty[q], (round - 1) & 1, globaltimer_ns() + p.timeout_ns))
    return false;
  tq.tile[q] = tile;
  mbar_arrive(&tq.full[q]);   // release: the id is visible to the waiters' acquire
  return true;
}

// Consumer (one lane): read entry n and free its slot. False after a timed-out wait.
__device__ __forceinline__ bool tq_take(const Params& p, const TileQueue& tq, uint32_t n,
                                        int& tile) {
  const int q = n % TQ;
  if (!mbar_wait(&tq.full[q], (n / TQ) & 1, globaltimer_ns() + p.timeout_ns)) return false;
  tile = tq.tile[q];
  mbar_arrive(&tq.empty[q]);
  return true;
}

// ------------------------------------------------------------------ producer
// One tile's K loop: fills stages it, it+1, ... (it counts stage uses over the CTA's
// whole task sequence). Returns false after a timed-out wait.
// SMP: the SM-pair kernel (its tcgen05 and TMA instructions of the CTA pair may not share a
// kernel with single-CTA ones, so the pair paths exist only in that instantiation).
template <bool MX, bool SMP = false>
__device__ bool produce_tile(const Params& p, const Maps& mp, uint8_t* smem, uint64_t* full,
                             uint64_t* empty, volatile int* abort_flag, const TileInfo& ti,
                             uint32_t& it) {
  using C = Cfg<MX>;
  constexpr int BK = C::BK;
  const int STAGES = p.stages;
  constexpr int CH = C::MN_LBO;        // bytes of one MN-major chunk
  const int sp = p.split;
  uint32_t b_bytes = (p.mode == kFwdUpGate || p.mode == kBwdDWUpGate) ? 256 * 128 : p.BN * 128;
  if (MX) b_bytes += 512 + ((p.mode == kFwdUpGate || p.mode == kBwdDWUpGate) ? 1024 : p.BN * 4);
  if (MX && ti.bf) {
    // BF16 shared-expert tile in an MXFP8 launch: the BF16 stage layout (K blocks of 64
    // elements, 64-element MN chunks Cfg<false>::MN_LBO apart), no scale atoms
    using CB = Cfg<false>;
    const uint32_t bb = p.mode == kFwdUpGate ? 256 * 128 : p.s_BN * 128;
    for (int kb = 0; kb < ti.kiters; ++kb, ++it) {
      const int stage = it % STAGES;
      const uint32_t round = it / STAGES;
      if (round > 0 && !mbar_wait(&empty[stage], (round - 1) & 1, globaltimer_ns() + p.timeout_ns)) {
        set_error(p.status, kErrTimeout);
        *abort_flag = 1;
        return false;
      }
      uint8_t* sa = smem + stage * p.stage_bytes;
      uint8_t* sb = sa + A_BYTES;
      uint64_t* bar = &full[stage];
      mbar_arrive_expect_tx(bar, A_BYTES + bb);
      const int k0 = kb * CB::BK;
      tma_load_2d(sa, &mp.a[2], bar, k0, ti.arow0);
      if (p.mode == kFwdUpGate) {
        for (int c = 0; c < 128 / CB::MN_CHUNK; ++c) {
          tma_load_2d(sb + c * CB::MN_LBO, &mp.b[2], bar, ti.n0 + c * CB::MN_CHUNK, k0);
          tma_load_2d(sb + (128 / CB::MN_CHUNK + c) * CB::MN_LBO, &mp.b[3], bar,
                      ti.n0 + c * CB::MN_CHUNK, k0);
        }
      } else {
        for (int c = 0; c < p.s_BN / CB::MN_CHUNK; ++c)
          tma_load_2d(sb + c * CB::MN_LBO, &mp.b[2], bar, ti.n0 + c * CB::MN_CHUNK, k0);
      }
    }
    return true;
  }
  {
    for (int kb = 0; kb < ti.kiters; ++kb, ++it) {
      const int stage = it % STAGES;
      const uint32_t round = it / STAGES;
      if (round > 0 && !mbar_wait(&empty[stage], (round - 1) & 1, globaltimer_ns() + p.timeout_ns)) {
        set_error(p.status, kErrTimeout);
        *abort_flag = 1;
        return false;
      }
      uint8_t* sa = smem + stage * p.stage_bytes;
      uint8_t* sb = sa + A_BYTES;
      uint8_t* sf = sa + p.sf_off;
      uint64_t* bar = &full[stage];
      if constexpr (!MX && SMP) {
        // SM pair: this CTA's 128 rows of A and its half of B's columns (dW up|gate: rank
        // 0 du, rank 1 dv, columns n0..n0+127; dW down: columns n0 + rank * BN/2 ..; dH:
        // rows n0 + rank * BN/2 .. of W_down), the copies of both CTAs counted on rank 0's
        // barrier, which rank 0 arms for both
        const uint32_t lbar = mapa_rank(bar, 0);
        const int nb = p.BN / 2;
        if (p.crank == 0) mbar_arrive_expect_tx(bar, 2 * (A_BYTES + nb * 128));
        if (p.mode == kBwdDH) {   // A: dYg rows (K-major); B: nb rows of W_down (K-major)
          tma_load_2d_pair(sa, &mp.a[0], lbar, kb * BK, ti.arow0);
          tma_load_2d_pair(sb, &mp.b[0], lbar, kb * BK, ti.e * p.I + ti.n0 + p.crank * nb);
          continue;
        }
        const int kr = ti.krow0 + kb * BK;
        for (int c = 0; c < BM / C::MN_CHUNK; ++c)
          tma_load_2d_pair(sa + c * CH, &mp.a[0], lbar, ti.row0 + c * C::MN_CHUNK, kr);
        const bool ug = p.mode == kBwdDWUpGate;
        const CUtensorMap* bmap = ug ? &mp.b[p.crank] : &mp.b[0];
        const int bc = ug ? ti.n0 : ti.n0 + p.crank * nb;
        for (int c = 0; c < nb / C::MN_CHUNK; ++c)
          tma_load_2d_pair(sb + c * CH, bmap, lbar, bc + c * C::MN_CHUNK, kr);
        continue;
      }
      uint32_t extra = 0;   // split dW stages also carry the lo half of the split operand
      if (sp) extra = p.mode == kBwdDWUpGate ? 2 * 128 * 128 : BM * 128;
      if (MX && p.kdouble) extra = A_BYTES + b_bytes;   // the second K chunk
      const bool a1 = !MX && ti.nrt == 2;              // the pair's second row tile
      if (a1) extra += A_BYTES;
      mbar_arrive_expect_tx(bar, A_BYTES + b_bytes + extra);
      const int k0 = kb * BK;
      switch (p.mode) {
        case kFwdUpGate: {   // A: Xg rows (K-major); B: W_up|W_gate cols n0..n0+127 (MN-major)
          tma_load_2d(sa, &mp.a[0], bar, k0, ti.arow0);
          if (a1) tma_load_2d(sa + PAIR_A1_OFF, &mp.a[0], bar, k0, ti.arow0 + BM);
          const int brow = ti.e * p.H + k0;
          for (int c = 0; c < 128 / C::MN_CHUNK; ++c) {
            tma_load_2d(sb + c * CH, &mp.b[0], bar, ti.n0 + c * C::MN_CHUNK, brow);
            tma_load_2d(sb + (128 / C::MN_CHUNK + c) * CH, &mp.b[1], bar, ti.n0 + c * C::MN_CHUNK,
                        brow);
          }
          if (MX) {
            bulk_load(sf, p.sfa + ((size_t)(ti.arow0 / BM) * p.kcs_a + kb) * 512, 512, bar);
            const size_t bi = (((size_t)ti.e * p.kcs_b + kb) * p.ncs_b + ti.n0 / 128) * 512;
            bulk_load(sf + 512, p.sfb0 + bi, 512, bar);
            bulk_load(sf + 1024, p.sfb1 + bi, 512, bar);
          }
          break;
        }
        case kFwdDown: {     // A: h rows (K-major); B: W_down cols (MN-major)
          tma_load_2d(sa, &mp.a[0], bar, k0, ti.arow0);
          if (a1) tma_load_2d(sa + PAIR_A1_OFF, &mp.a[0], bar, k0, ti.arow0 + BM);
          const int brow = ti.e * p.I + k0;
          for (int c = 0; c < p.BN / C::MN_CHUNK; ++c)
            tma_load_2d(sb + c * CH, &mp.b[0], bar, ti.n0 + c * C::MN_CHUNK, brow);
          if (MX) {
            bulk_load(sf, p.sfa + ((size_t)(ti.arow0 / BM) * p.kcs_a + kb) * 512, 512, bar);
            const size_t bi = (((size_t)ti.e * p.kcs_b + kb) * p.ncs_b + ti.n0 / 128) * 512;
            bulk_load(sf + 512, p.sfb0 + bi, p.BN * 4, bar);
          }
          break;
        }
        case kRouter: {      // A: x rows (K-major, K chunk wraps per part); B: Wr parts (MN-major)
          tma_load_2d(sa, &mp.a[0], bar, (kb % (p.H / BK)) * BK, ti.arow0);
          for (int c = 0; c < p.BN / C::MN_CHUNK; ++c)
            tma_load_2d(sb + c * CH, &mp.b[0], bar, ti.n0 + c * C::MN_CHUNK, k0);
          break;
        }
        case kBwdDH: {       // A: dYg rows (K-major); B: W_down rows i (K-major over H)
          if (MX && p.kdouble) {   // two K chunks: A0 A1 B0 B1, then atoms A0 A1 B0 B1
            for (int h = 0; h < 2; ++h) {
              const int kc = 2 * kb + h;
              tma_load_2d(sa + h * A_BYTES, &mp.a[0], bar, kc * BK, ti.arow0);
              tma_load_2d(sa + (2 + h) * A_BYTES, &mp.b[0], bar, kc * BK, ti.e * p.I + ti.n0);
              bulk_load(sf + h * 512, p.sfa + ((size_t)(ti.arow0 / BM) * p.kcs_a + kc) * 512, 512,
                        bar);
              const size_t bi = (((size_t)ti.e * p.kcs_b + kc) * p.ncs_b + ti.n0 / 128) * 512;
              bulk_load(sf + 1024 + h * 512, p.sfb0 + bi, 512, bar);
            }
            break;
          }
          tma_load_2d(sa, &mp.a[0], bar, k0, ti.arow0);
          if (a1) tma_load_2d(sa + PAIR_A1_OFF, &mp.a[0], bar, k0, ti.arow0 + BM);
          tma_load_2d(sb, &mp.b[0], bar, k0, ti.e * p.I + ti.n0);
          if (MX) {
            bulk_load(sf, p.sfa + ((size_t)(ti.arow0 / BM) * p.kcs_a + kb) * 512, 512, bar);
            const size_t bi = (((size_t)ti.e * p.kcs_b + kb) * p.ncs_b + ti.n0 / 128) * 512;
            bulk_load(sf + 512, p.sfb0 + bi, p.BN * 4, bar);
          }
          break;
        }
        case kBwdDX: {       // K = [I of du | I of dv]; B: W_up / W_gate rows h (K-major over I)
          const int per_half = p.I / BK;
          const int second = kb >= per_half ? 1 : 0;
          const int kq = kb - second * per_half;   // K chunk inside the half
          tma_load_2d(sa, &mp.a[second], bar, kq * BK, ti.arow0);
          if (a1) tma_load_2d(sa + PAIR_A1_OFF, &mp.a[second], bar, kq * BK, ti.arow0 + BM);
          tma_load_2d(sb, &mp.b[second], bar, kq * BK, ti.e * p.H + ti.n0);
          if (MX) {
            bulk_load(sf, (second ? p.sfa1 : p.sfa) + ((size_t)(ti.arow0 / BM) * p.kcs_a + kq) * 512,
                      512, bar);
            const size_t bi = (((size_t)ti.e * p.kcs_b + kq) * p.ncs_b + ti.n0 / 128) * 512;
            bulk_load(sf + 512, (second ? p.sfb1 : p.sfb0) + bi, p.BN * 4, bar);
          }
          break;
        }
        case kBwdDWDown: {   // A: (g h)^T (MN-major, M = I), hi (+ lo); B: dYg (MN-major, N = H)
          const int kr = ti.krow0 + kb * BK;
          for (int c = 0; c < BM / C::MN_CHUNK; ++c) {
            tma_load_2d(sa + c * CH, &mp.a[0], bar, ti.row0 + c * C::MN_CHUNK, kr);
            if (sp)
              tma_load_2d(sa + SPLIT_EXTRA_OFF + c * CH, &mp.a[1], bar, ti.row0 + c * C::MN_CHUNK, kr);
          }
          for (int c = 0; c < p.BN / C::MN_CHUNK; ++c)
            tma_load_2d(sb + c * CH, &mp.b[0], bar, ti.n0 + c * C::MN_CHUNK, kr);
          if (MX) {   // row-block atoms [row tile][M/128] and [row tile][N/128]
            bulk_load(sf, p.sfa + ((size_t)(kr / BM) * (p.I / 128) + ti.row0 / 128) * 512, 512, bar);
            bulk_load(sf + 512, p.sfb0 + ((size_t)(kr / BM) * (p.H / 128) + ti.n0 / 128) * 512,
                      p.BN * 4, bar);
          }
          break;
        }
        default: {           // kBwdDWUpGate: A: Xg^T (M = H); B: du | dv cols n0..n0+127 (+ lo)
          const int kr = ti.krow0 + kb * BK;
          for (int c = 0; c < BM / C::MN_CHUNK; ++c)
            tma_load_2d(sa + c * CH, &mp.a[0], bar, ti.row0 + c * C::MN_CHUNK, kr);
          for (int part = 0; part <= sp; ++part) {
            uint8_t* dst = part ? sa + SPLIT_EXTRA_OFF : sb;
            for (int c = 0; c < 128 / C::MN_CHUNK; ++c) {
              tma_load_2d(dst + c * CH, &mp.b[2 * part], bar, ti.n0 + c * C::MN_CHUNK, kr);
              tma_load_2d(dst + (128 / C::MN_CHUNK + c) * CH, &mp.b[2 * part + 1], bar,
                          ti.n0 + c * C::MN_CHUNK, kr);
            }
          }
          if (MX) {
            bulk_load(sf, p.sfa + ((size_t)(kr / BM) * (p.H / 128) + ti.row0 / 128) * 512, 512, bar);
            const size_t bi = ((size_t)(kr / BM) * (p.I / 128) + ti.n0 / 128) * 512;
            bulk_load(sf + 512, p.sfb0 + bi, 512, bar);
            bulk_load(sf + 1024, p.sfb1 + bi, 512, bar);
          }
          break;
        }
      }
    }
  }
  return true;
}

// Drain: every issued copy has landed and every MMA commit has arrived before the CTA's
// shared memory goes away (n_armed = stage uses issued).
template <bool MX>
__device__ void produce_drain(const Params& p, uint64_t* full, uint64_t* empty,
                              uint32_t n_armed) {
  const int STAGES = p.stages;
  for (uint32_t s = 0; s < (uint32_t)STAGES && s < n_armed; ++s) {
    const uint32_t last = ((n_armed - 1 - s) / STAGES) * STAGES + s;  // last use of stage s
    const uint32_t round = last / STAGES;
    if (!mbar_wait(&empty[s], round & 1, globaltimer_ns() + p.timeout_ns)) {
      set_error(p.status, kErrTimeout);
      mbar_wait(&full[s], round & 1, globaltimer_ns() + p.timeout_ns);
    }
  }
}

// Cluster-launch-control requests of one producer lane: at most one in flight.
struct ClcState {
  uint64_t* bar;
  uint8_t* answer;     // 16 bytes, 16-byte aligned
  uint32_t made = 0;   // answered requests (the phase of bar)
  bool in_flight = false;
  bool ended = false;  // an answer said no CTA was left: no further request may be made
};
__device__ __forceinline__ void clc_ask(ClcState& c) {
  if (c.ended || c.in_flight) return;
  if (c.made) fence_proxy_async_smem();   // the last answer's reads before the next write
  mbar_arrive_expect_tx(c.bar, 16);
  clc_try_cancel(c.answer, c.bar);
  c.in_flight = true;
}
// The answer of the request in flight: the cancelled CTA's index, or -1 (none left). False
// after a timed-out wait.
__device__ __forceinline__ bool clc_answer(const Params& p, ClcState& c, int& x) {
  if (!mbar_wait(c.bar, c.made & 1, globaltimer_ns() + p.timeout_ns)) return false;
  ++c.made;
  c.in_flight = false;
  x = clc_cancelled_x(c.answer);
  if (x < 0) c.ended = true;
  return true;
}

template <bool MX, bool SMP = false>
__device__ void produce(const Params& p, const Maps& mp, uint8_t* smem, uint64_t* full,
                        uint64_t* empty, volatile int* abort_flag, const TileQueue& tq,
                        ClcState& clc) {
  const int ntiles = num_tiles_of(p);
  uint32_t it = 0;
  if (!p.tile_counter && !p.clc) {
    const int t0 = SMP ? p.t0 : (int)blockIdx.x, step = SMP ? p.tstep : (int)gridDim.x;
    for (int tile = t0; tile < ntiles; tile += step) {
      const TileInfo ti = tile_info<MX>(p, tile);
      if (ti.skip) continue;
      if (!produce_tile<MX, SMP>(p, mp, smem, full, empty, abort_flag, ti, it)) break;
    }
  } else {
    int own = p.clc ? (int)blockIdx.x : -1;   // CLC: the CTA's own tile comes first
    for (uint32_t n = 0;; ++n) {
      int tile;
      TileInfo ti;
      bool ok = true;
      for (;;) {   // the next tile that is not the unmatched half of a row-tile pair
        if (!p.clc) {
          tile = atomicAdd(p.tile_counter, 1);
        } else if (own >= 0) {
          tile = own;
          own = -1;
        } else {
          clc_ask(clc);                 // (already in flight after the previous tile)
          if (clc.ended) {
            tile = -1;
            break;
          }
          if (!clc_answer(p, clc, tile)) {
            ok = false;
            break;
          }
          if (tile < 0) break;
        }
        if (tile >= ntiles) {
          tile = -1;
          break;
        }
        ti = tile_info<MX>(p, tile);
        if (!ti.skip) break;
      }
      if (!ok) {   // no answer in time: end the queue so the consumers stop too
        set_error(p.status, kErrTimeout);
        *abort_flag = 1;
        tile = -1;
      } else if (p.clc && tile >= 0) {
        clc_ask(clc);   // the answer arrives while this tile's loads run
      }
      if (!tq_publish(p, tq, n, tile)) {
        set_error(p.status, kErrTimeout);
        *abort_flag = 1;
        break;
      }
      if (tile < 0) break;
      if (!produce_tile<MX>(p, mp, smem, full, empty, abort_flag, ti, it)) break;
    }
  }
  produce_drain<MX>(p, full, empty, it);
}

// ------------------------------------------------------------------ MMA issuer
// SM pair, rank 0: one tile's M = 256 MMAs over both CTAs' stages (both operands MN-major);
// each commit arrives on the barrier at the same offset in both CTAs. Returns false after a
// timed-out wait.
template <bool MX>
__device__ bool mma_tile_pair(const Params& p, uint8_t* smem, uint64_t* full, uint64_t* empty,
                              uint64_t* acc_full, uint64_t* acc_empty, uint32_t tmem_base,
                              volatile int* abort_flag, const TileInfo& ti, uint32_t& it,
                              int local) {
  using C = Cfg<MX>;
  const int STAGES = p.stages;
  // the weight gradients' operands are MN-major, dH's K-major
  const bool mn = is_dw(p.mode);
  const uint32_t idp = idesc_bf16(2 * BM, p.BN, mn, mn);
  const int acc = local % p.nacc;
  const uint32_t use = local / p.nacc;
  if (use > 0 &&
      !mbar_wait(&acc_empty[acc], (use - 1) & 1, globaltimer_ns() + p.timeout_ns)) {
    set_error(p.status, kErrTimeout);
    *abort_flag = 1;
    return false;
  }
  tc_fence_after();
  const uint32_t d_tmem = tmem_base + acc * p.acc_cols;
  for (int kb = 0; kb < ti.kiters; ++kb, ++it) {
    const int stage = it % STAGES;
    if (!mbar_wait(&full[stage], (it / STAGES) & 1, globaltimer_ns() + p.timeout_ns)) {
      set_error(p.status, kErrTimeout);
      *abort_flag = 1;
      return false;
    }
    tc_fence_after();
    const uint32_t sa = smem_u32(smem + stage * p.stage_bytes);
    const uint32_t sb = sa + A_BYTES;
    const int nk = kb == ti.kiters - 1 ? ti.klast : 4;
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      if (kk >= nk) break;
      const uint64_t ad = mn ? umma_desc_sw128(sa + kk * C::MN_KSTEP, C::MN_LBO, 1024)
                             : umma_desc_sw128(sa + kk * 32, 16, 1024);
      const uint64_t bd = mn ? umma_desc_sw128(sb + kk * C::MN_KSTEP, C::MN_LBO, 1024)
                             : umma_desc_sw128(sb + kk * 32, 16, 1024);
      umma_bf16_pair(d_tmem, ad, bd, idp, (kb > 0 || kk > 0) ? 1u : 0u);
    }
    umma_commit_pair(&empty[stage]);
  }
  if (ti.kiters > 0) {
    umma_commit_pair(&acc_full[acc]);
  } else {   // nothing to accumulate: both epilogues write zeros
    mbar_arrive(&acc_full[acc]);
    mbar_arrive_cluster(mapa_rank(&acc_full[acc], 1));
  }
  return true;
}

// One tile: waits for a free accumulator (local = the CTA's tile count so far), issues the
// K loop's MMAs and commits the accumulator. Returns false after a timed-out wait.
template <bool MX>
__device__ bool mma_tile(const Params& p, uint8_t* smem, uint64_t* full, uint64_t* empty,
                         uint64_t* acc_full, uint64_t* acc_empty, uint32_t tmem_base,
                         volatile int* abort_flag, const TileInfo& ti, uint32_t& it, int local) {
  using C = Cfg<MX>;
  const int STAGES = p.stages;
  bool a_mn = false, b_mn = false;
  int n_mma = p.BN;
  switch (p.mode) {
    case kFwdUpGate: b_mn = true; n_mma = 256; break;
    case kFwdDown: b_mn = true; break;
    case kRouter: b_mn = true; break;
    case kBwdDH: break;
    case kBwdDX: break;
    case kBwdDWDown: a_mn = true; b_mn = true; break;
    default: a_mn = true; b_mn = true; n_mma = 256; break;
  }
  const uint32_t idesc = idesc_bf16(BM, n_mma, a_mn, b_mn);
  if (MX && ti.bf) {   // BF16 shared-expert tile: kind::f16 MMAs on the BF16 stage layout
    using CB = Cfg<false>;
    const uint32_t idb = idesc_bf16(BM, p.mode == kFwdUpGate ? 256 : p.s_BN, false, true);
    const int acc = local % p.nacc;
    const uint32_t use = local / p.nacc;
    if (use > 0 && !mbar_wait(&acc_empty[acc], (use - 1) & 1, globaltimer_ns() + p.timeout_ns)) {
      set_error(p.status, kErrTimeout);
      *abort_flag = 1;
      return false;
    }
    tc_fence_after();
    const uint32_t d_tmem = tmem_base + acc * p.acc_cols;
    for (int kb = 0; kb < ti.kiters; ++kb, ++it) {
      const int stage = it % STAGES;
      if (!mbar_wait(&full[stage], (it / STAGES) & 1, globaltimer_ns() + p.timeout_ns)) {
        set_error(p.status, kErrTimeout);
        *abort_flag = 1;
        return false;
      }
      tc_fence_after();
      const uint32_t sa = smem_u32(smem + stage * p.stage_bytes);
      const uint32_t sb = sa + A_BYTES;
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
        umma_bf16(d_tmem, umma_desc_sw128(sa + kk * 32, 16, 1024),
                  umma_desc_sw128(sb + kk * CB::MN_KSTEP, CB::MN_LBO, 1024), idb,
                  (kb > 0 || kk > 0) ? 1u : 0u);
      umma_commit(&empty[stage]);
    }
    if (ti.kiters > 0) umma_commit(&acc_full[acc]);
    else mbar_arrive(&acc_full[acc]);
    return true;
  }
  {
    const int acc = local % p.nacc;
    const uint32_t use = local / p.nacc;
    if (use > 0 && !mbar_wait(&acc_empty[acc], (use - 1) & 1, globaltimer_ns() + p.timeout_ns)) {
      set_error(p.status, kErrTimeout);
      *abort_flag = 1;
      return false;
    }
    tc_fence_after();
    const uint32_t d_tmem = tmem_base + acc * p.acc_cols;
    for (int kb = 0; kb < ti.kiters; ++kb, ++it) {
      const int stage = it % STAGES;
      const uint32_t round = it / STAGES;
      if (!mbar_wait(&full[stage], round & 1, globaltimer_ns() + p.timeout_ns)) {
        set_error(p.status, kErrTimeout);
        *abort_flag = 1;
        return false;
      }
      tc_fence_after();
      const uint32_t sa = smem_u32(smem + stage * p.stage_bytes);
      const uint32_t sb = sa + A_BYTES;
      // MMA K steps of this stage: all four, except in a dW tile's last K iteration
      const int nk = (is_dw(p.mode) && kb == ti.kiters - 1) ? ti.klast : 4;
      uint32_t t_sfa = 0, t_sfb = 0;
      if (MX && p.kdouble) {
        // two K chunks of 128: atoms A0, A1 -> columns 0-3, 4-7; B0, B1 -> 8-11, 12-15
        const uint32_t t_sf = tmem_base + C::SF_TMEM + stage * 16;
        for (int j = 0; j < 4; ++j)
          tmem_cp_32x128b_x4(t_sf + 4 * j, smem_desc_rows16(sa + p.sf_off + 512 * j));
#pragma unroll
        for (int h = 0; h < 2; ++h) {
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t ad = umma_desc_sw128(sa + h * A_BYTES + kk * 32, 16, 1024);
            const uint64_t bd = umma_desc_sw128(sa + (2 + h) * A_BYTES + kk * 32, 16, 1024);
            const uint32_t accum = (kb > 0 || h > 0 || kk > 0) ? 1u : 0u;
            umma_mxf8(d_tmem, ad, bd, idesc_mxf8(BM, n_mma, false, false, kk), t_sf + 4 * h,
                      t_sf + 8 + 4 * h, accum);
          }
        }
        umma_commit(&empty[stage]);
        continue;
      }
      if (MX) {
        // scale atoms -> TMEM: A in 4 columns, B in 4 columns per 128 rows of N
        const uint32_t col = C::SF_TMEM + stage * 16;
        t_sfa = tmem_base + col;
        t_sfb = tmem_base + col + 4;
        tmem_cp_32x128b_x4(t_sfa, smem_desc_rows16(sa + p.sf_off));
        for (int j = 0; j < n_mma / 128; ++j)
          tmem_cp_32x128b_x4(t_sfb + 4 * j, smem_desc_rows16(sa + p.sf_off + 512 + 512 * j));
      }
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        if (kk >= nk) break;
        // K-major: the kk-th K slice starts 32 bytes further along each 128-byte row.
        // MN-major: it starts MMA_K rows further; 128-byte MN chunks are MN_LBO apart
        // (leading byte offset), 8-row groups 1 KB apart (stride byte offset).
        const uint64_t ad = a_mn ? umma_desc_sw128(sa + kk * C::MN_KSTEP, C::MN_LBO, 1024)
                                 : umma_desc_sw128(sa + kk * 32, 16, 1024);
        const uint64_t bd = b_mn ? umma_desc_sw128(sb + kk * C::MN_KSTEP, C::MN_LBO, 1024)
                                 : umma_desc_sw128(sb + kk * 32, 16, 1024);
        const uint32_t accum = (kb > 0 || kk > 0) ? 1u : 0u;
        if (MX) {
          umma_mxf8(d_tmem, ad, bd, idesc_mxf8(BM, n_mma, a_mn, b_mn, kk), t_sfa, t_sfb, accum);
        } else {
          umma_bf16(d_tmem, ad, bd, idesc, accum);
          if (ti.nrt == 2)   // the pair's second row tile (K-major A), same B, columns +256
            umma_bf16(d_tmem + 256, umma_desc_sw128(sa + PAIR_A1_OFF + kk * 32, 16, 1024), bd,
                      idesc, accum);
        }
      }
      if (!MX && p.split) {
        // the lo half of the K chunk, after the hi half, into the same accumulator:
        // dW_up|gate pairs A with B lo, dW_down pairs A lo with B
        const uint32_t sx = sa + SPLIT_EXTRA_OFF;
        const uint32_t a2 = p.mode == kBwdDWDown ? sx : sa;
        const uint32_t b2 = p.mode == kBwdDWDown ? sb : sx;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          if (kk >= nk) break;
          umma_bf16(d_tmem, umma_desc_sw128(a2 + kk * C::MN_KSTEP, C::MN_LBO, 1024),
                    umma_desc_sw128(b2 + kk * C::MN_KSTEP, C::MN_LBO, 1024), idesc, 1u);
        }
      }
      umma_commit(&empty[stage]);   // frees the stage once these MMAs have read it
    }
    if (ti.kiters > 0) umma_commit(&acc_full[acc]);
    else mbar_arrive(&acc_full[acc]);  // nothing to accumulate: epilogue writes zeros
  }
  return true;
}

template <bool MX>
__device__ void mma_issue(const Params& p, uint8_t* smem, uint64_t* full, uint64_t* empty,
                          uint64_t* acc_full, uint64_t* acc_empty, uint32_t tmem_base,
                          volatile int* abort_flag, const TileQueue& tq) {
  const int ntiles = num_tiles_of(p);
  uint32_t it = 0;
  int local = 0;
  if (!p.tile_counter && !p.clc) {
    for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
      const TileInfo ti = tile_info<MX>(p, tile);
      if (ti.skip) continue;
      if (!mma_tile<MX>(p, smem, full, empty, acc_full, acc_empty, tmem_base, abort_flag, ti,
                        it, local++))
        return;
    }
    return;
  }
  for (uint32_t n = 0;; ++n) {
    int tile;
    if (!tq_take(p, tq, n, tile)) {
      set_error(p.status, kErrTimeout);
      *abort_flag = 1;
      return;
    }
    if (tile < 0) return;
    const TileInfo ti = tile_info<MX>(p, tile);
    if (!mma_tile<MX>(p, smem, full, empty, acc_full, acc_empty, tmem_base, abort_flag, ti, it,
                      local++))
      return;
  }
}

// SM pair, rank 0: the cluster's tiles in the static order. Returns the number of tiles
// whose MMAs were issued.
template <bool MX>
__device__ int mma_issue_pair(const Params& p, uint8_t* smem, uint64_t* full, uint64_t* empty,
                              uint64_t* acc_full, uint64_t* acc_empty, uint32_t tmem_base,
                              volatile int* abort_flag) {
  const int ntiles = num_tiles_of(p);
  uint32_t it = 0;
  int local = 0;
  for (int tile = p.t0; tile < ntiles; tile += p.tstep) {
    const TileInfo ti = tile_info<MX>(p, tile);
    if (ti.skip) continue;   // as the producer and the epilogue
    if (!mma_tile_pair<MX>(p, smem, full, empty, acc_full, acc_empty, tmem_base, abort_flag, ti,
                           it, local))
      return local;
    ++local;
  }
  return local;
}

// SM pair, rank 0 after its last tile: every epilogue release of both CTAs has arrived
// (the other CTA's arrivals target this CTA's shared memory), n = tiles issued.
__device__ void mma_drain_pair(const Params& p, uint64_t* acc_empty, int n) {
  for (int a = 0; a < p.nacc && a < n; ++a) {
    const uint32_t uses = (uint32_t)((n - 1 - a) / p.nacc + 1);
    if (!mbar_wait(&acc_empty[a], (uses - 1) & 1, globaltimer_ns() + p.timeout_ns))
      set_error(p.status, kErrTimeout);
  }
}

// ------------------------------------------------------------------ epilogue
// One tile (local = the CTA's tile count so far): waits for its accumulator, runs the
// mode's epilogue and frees the accumulator. Warp-collective over the 4 epilogue warps.
// Returns false after a timed-out wait.
template <bool MX, bool SMP = false>
__device__ bool epilogue_tile(const Params& p, const Maps& mp, Stager& st, uint64_t* acc_full,
                              uint64_t* acc_empty, uint32_t tmem_base, volatile int* abort_flag,
                              const TileInfo& tile_in, int local) {
  using C = Cfg<MX>;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int quarter = warp & 3;             // TMEM lanes 32*quarter .. +31
  const int r = quarter * 32 + lane;        // row inside the tile
  {
    const int acc = local % p.nacc;
    const uint32_t use = local / p.nacc;
    if (!mbar_wait(&acc_full[acc], use & 1, globaltimer_ns() + p.timeout_ns)) {
      set_error(p.status, kErrTimeout);
      *abort_flag = 1;
      return false;
    }
    tc_fence_after();
    const bool have = tile_in.kiters > 0;
    float a[32], b[32];
    // The accumulator is handed back to the MMA lane right after this thread's last TMEM
    // load (before that chunk's math and stores), so the next tile's MMAs can start while
    // the stores drain; with one accumulator (MXFP8) this is the overlap there is. A
    // row-tile pair hands both back after its second row tile's last load.
    bool released = false;
    int half = 0;
    auto release = [&]() {
      if (!released && half >= tile_in.nrt - 1) {
        tc_fence_before();
        if constexpr (SMP) {   // one arrival per warp on rank 0's barrier (8 in all)
          __syncwarp();
          if (lane == 0) mbar_arrive_cluster(mapa_rank(&acc_empty[acc], 0));
        } else {
          mbar_arrive(&acc_empty[acc]);
        }
        released = true;
      }
    };
    for (; half < tile_in.nrt; ++half) {
    TileInfo ti = tile_in;   // row tile `half` of a pair: rows +128, accumulator columns +256
    ti.row0 += half * BM;
    ti.arow0 += half * BM;
    const uint32_t t_row =
        tmem_base + acc * p.acc_cols + half * 256 + ((uint32_t)(quarter * 32) << 16);
    // tcgen05.ld and the staged stores are warp-collective: every lane takes part, rows
    // outside the problem only skip their global loads (TMA drops their stores).
    const int row = ti.row0 + r;
    const int wrow = ti.row0 + quarter * 32;  // first row of this warp's 32-row box
    const bool valid = !(p.dense && !is_dw(p.mode) && row >= p.M_rows);
    switch (p.mode) {
      case kFwdUpGate: {
        const size_t o = (size_t)row * p.I + ti.n0;
        // BF16: h as the down GEMM's bf16 operand; U, V kept as bf16 for the backward, two
        // 32-column chunks at a time in 64-column boxes (maps o[m0..m0+2])
        auto bf16_upgate = [&](int m0) {
          for (int c = 0; c < 4; c += 2) {
            float a1[32], b1[32];
            tmem_ld32(t_row + c * 32, a);                // U
            tmem_ld32(t_row + 128 + c * 32, b);          // V
            tmem_ld32(t_row + (c + 1) * 32, a1);
            tmem_ld32(t_row + 128 + (c + 1) * 32, b1);
            if (c == 2) release();
            const int col = ti.n0 + c * 32;
            float h[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) h[i] = b[i] * sigmoidf_(b[i]) * a[i];
            st.bf16(&mp.o[m0], h, col, wrow);
#pragma unroll
            for (int i = 0; i < 32; ++i) h[i] = b1[i] * sigmoidf_(b1[i]) * a1[i];
            st.bf16(&mp.o[m0], h, col + 32, wrow);
            st.bf16x64(&mp.o[m0 + 1], a, a1, col, wrow);
            st.bf16x64(&mp.o[m0 + 2], b, b1, col, wrow);
          }
        };
        if constexpr (MX) {
          if (ti.bf) {   // the shared expert's tile of a mixed launch
            bf16_upgate(3);
            break;
          }
          uint32_t sbytes = 0;
          // two 32-column chunks at a time: U, V leave as bf16 in 64-column boxes, h as
          // MXFP8 blocks of 32 along I (plain stores of the codes, the scale word below)
          for (int c = 0; c < 4; c += 2) {
            float a1[32], b1[32];
            tmem_ld32(t_row + c * 32, a);               // U
            tmem_ld32(t_row + 128 + c * 32, b);         // V
            tmem_ld32(t_row + (c + 1) * 32, a1);
            tmem_ld32(t_row + 128 + (c + 1) * 32, b1);
            if (c == 2) release();
            for (int half = 0; half < 2; ++half) {
              const float* uu = half ? a1 : a;
              const float* vv = half ? b1 : b;
              float h[32];
#pragma unroll
              for (int i = 0; i < 32; ++i) h[i] = vv[i] * sigmoidf_(vv[i]) * uu[i];
              uint4 q[2];
              sbytes |= quant32_e4m3(h, q) << (8 * (c + half));
              if (valid) {
                uint4* dq = reinterpret_cast<uint4*>(p.out_q[0] + o + (c + half) * 32);
                dq[0] = q[0];
                dq[1] = q[1];
              }
            }
            st.bf16x64(&mp.o[1], a, a1, ti.n0 + c * 32, wrow);
            st.bf16x64(&mp.o[2], b, b1, ti.n0 + c * 32, wrow);
          }
          if (valid) {
            const size_t atom = (size_t)(row / BM) * (p.I / 128) + ti.n0 / 128;
            *reinterpret_cast<uint32_t*>(p.out_sf[0] + atom * 512 + 16 * (r & 31) + 4 * (r >> 5)) =
                sbytes;
          }
        } else {
          bf16_upgate(0);
        }
        break;
      }
      case kRouter: {  // logits fp32 (+ bias), ordinary stores of the row's valid columns
        for (int c = 0; c < p.BN / 32; ++c) {
          tmem_ld32(t_row + c * 32, a);
          if (c == p.BN / 32 - 1) release();
          const int col0 = ti.n0 + c * 32;
          if (valid) {
            float* dst = p.logits + (size_t)row * p.n_out;
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (col0 + i < p.n_out) dst[col0 + i] = a[i] + (p.bias ? p.bias[col0 + i] : 0.f);
          }
        }
        break;
      }
      case kFwdDown:
      case kBwdDX: {   // expert outputs / routed dX rows (shared expert output: o[3]), fp32 or bf16
        const int bn = ti.bf ? p.s_BN : p.BN;
        const CUtensorMap* om = &mp.o[ti.bf ? 3 : 0];
        if (p.out_bf16) {
          for (int c = 0; c < bn / 32; c += 2) {
            tmem_ld32(t_row + c * 32, a);
            tmem_ld32(t_row + (c + 1) * 32, b);
            if (c + 2 >= bn / 32) release();
            st.bf16x64(om, a, b, ti.n0 + c * 32, wrow);
          }
        } else {
          for (int c = 0; c < bn / 32; ++c) {
            tmem_ld32(t_row + c * 32, a);
            if (c == bn / 32 - 1) release();
            st.f32(om, a, ti.n0 + c * 32, wrow);
          }
        }
        break;
      }
      case kBwdDH: {
        if (ti.norows) {   // SM pair without a second row tile: nothing to read or write
          release();
          break;
        }
        float g = 1.f;
        bool real = true;   // a row of the expert, not segment padding
        if (!p.dense) {
          const int rl = row - p.poff[ti.e];
          g = 0.f;
          real = rl < p.counts[ti.e];
          if (real) {
            const int tr = p.offsets[ti.e] + rl;
            g = p.gates[(size_t)p.table[2 * tr] * p.k + p.table[2 * tr + 1]];
          }
        }
        const size_t o = (size_t)row * p.I + ti.n0;
        // U, V of this row: the same row, or its row in the layout the forward kept them in.
        // A padding row reads neither and gives exact zeros (its D, U, V may be anything)
        const int urow = p.uv_row ? p.uv_row[row] : row;
        const bool have_uv = valid && real && urow >= 0;
        const size_t ouv = (size_t)(urow < 0 ? 0 : urow) * p.I + ti.n0;
        float dg = 0.f;
        for (int c = 0; c < p.BN / 32; ++c) {
          const int col = ti.n0 + c * 32;
          tmem_ld32(t_row + c * 32, a);          // D = dY W_down^T
          if (c == p.BN / 32 - 1) release();
          float u[32], v[32];
          if (have_uv) {                         // U, V as the forward kept them (bf16)
            load_bf16x32(reinterpret_cast<const __nv_bfloat16*>(p.u) + ouv + c * 32, u);
            load_bf16x32(reinterpret_cast<const __nv_bfloat16*>(p.v) + ouv + c * 32, v);
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) u[i] = v[i] = a[i] = 0.f;
          }
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
          if (!MX) {   // bf16 hi/lo pairs of du, dv, g*h
            float hi[32], lo[32];
            split_bf16(du, hi, lo);
            st.bf16(&mp.o[0], hi, col, wrow);
            if (p.lo_out) st.bf16(&mp.o[1], lo, col, wrow);
            split_bf16(dv, hi, lo);
            st.bf16(&mp.o[2], hi, col, wrow);
            if (p.lo_out) st.bf16(&mp.o[3], lo, col, wrow);
            split_bf16(hg, hi, lo);
            st.bf16(&mp.o[4], hi, col, wrow);
            if (p.lo_out) st.bf16(&mp.o[5], lo, col, wrow);
          } else {
            // du, dv feed the dX GEMM (K = I): per-thread blocks of 32 along I
            const size_t atom_i = ((size_t)(row / BM) * (p.I / 128) + col / 128) * 512 +
                                  16 * (r & 31) + 4 * (r >> 5) + ((col & 127) >> 5);
            uint4 q[2];
            const uint8_t sb_du = (uint8_t)quant32_e4m3(du, q);
            if (valid) {
              p.out_sf[0][atom_i] = sb_du;
              reinterpret_cast<uint4*>(p.out_q[0] + o + c * 32)[0] = q[0];
              reinterpret_cast<uint4*>(p.out_q[0] + o + c * 32)[1] = q[1];
            }
            const uint8_t sb_dv = (uint8_t)quant32_e4m3(dv, q);
            if (valid) {
              p.out_sf[1][atom_i] = sb_dv;
              reinterpret_cast<uint4*>(p.out_q[1] + o + c * 32)[0] = q[0];
              reinterpret_cast<uint4*>(p.out_q[1] + o + c * 32)[1] = q[1];
            }
            // du, dv, g*h also feed the dW GEMMs (K = rows): blocks of the warp's 32 rows,
            // one warp-wide maximum per column. Every lane takes part (rows outside the
            // problem are zero), so the reductions stay converged.
            const size_t atom_r = ((size_t)(row / BM) * (p.I / 128) + col / 128) * 512 +
                                  16 * (lane & 31) + 4 * (((col & 127) + lane) >> 5) + quarter;
            quant_rowblock(du, lane, valid, p.out_q[2] + o + c * 32, p.out_sf[2] + atom_r);
            quant_rowblock(dv, lane, valid, p.out_q[3] + o + c * 32, p.out_sf[3] + atom_r);
            quant_rowblock(hg, lane, valid, p.out_q[4] + o + c * 32, p.out_sf[4] + atom_r);
          }
        }
        if (valid && p.dgp) p.dgp[(size_t)row * p.n_tiles + ti.n0 / p.BN] = dg;
        break;
      }
      case kBwdDWDown: {                         // rows = i of dW_down[e], fp32 or bf16
        const int orow = ti.e * p.I + wrow;
        if (p.out_bf16) {
          for (int c = 0; c < p.BN / 32; c += 2) {
            if (have) {
              tmem_ld32(t_row + c * 32, a);
              tmem_ld32(t_row + (c + 1) * 32, b);
            } else {
#pragma unroll
              for (int i = 0; i < 32; ++i) a[i] = b[i] = 0.f;
            }
            if (c + 2 >= p.BN / 32) release();
            st.bf16x64(&mp.o[0], a, b, ti.n0 + c * 32, orow);
          }
          break;
        }
        for (int c = 0; c < p.BN / 32; ++c) {
          if (have) tmem_ld32(t_row + c * 32, a);
          else {
#pragma unroll
            for (int i = 0; i < 32; ++i) a[i] = 0.f;
          }
          if (c == p.BN / 32 - 1) release();
          st.f32(&mp.o[0], a, ti.n0 + c * 32, orow);
        }
        break;
      }
      default: {                                 // kBwdDWUpGate; rows = h, fp32 or bf16
        const int orow = ti.e * p.H + wrow;
        if (p.out_bf16) {
          // columns c*32 .. c*32+63 of dW_up (accumulator columns 0..127) and of dW_gate
          // (columns 128..255), one 64-column box each
          for (int c = 0; c < 4; c += 2) {
            float a1[32];
            if (have) {
              tmem_ld32(t_row + c * 32, a);
              tmem_ld32(t_row + (c + 1) * 32, a1);
            } else {
#pragma unroll
              for (int i = 0; i < 32; ++i) a[i] = a1[i] = 0.f;
            }
            st.bf16x64(&mp.o[0], a, a1, ti.n0 + c * 32, orow);
            if (have) {
              tmem_ld32(t_row + 128 + c * 32, b);
              tmem_ld32(t_row + 128 + (c + 1) * 32, a1);
            } else {
#pragma unroll
              for (int i = 0; i < 32; ++i) b[i] = a1[i] = 0.f;
            }
            if (c == 2) release();
            st.bf16x64(&mp.o[1], b, a1, ti.n0 + c * 32, orow);
          }
          break;
        }
        for (int c = 0; c < 4; ++c) {
          if (have) {
            tmem_ld32(t_row + c * 32, a);
            tmem_ld32(t_row + 128 + c * 32, b);
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) a[i] = b[i] = 0.f;
          }
          if (c == 3) release();
          st.f32(&mp.o[0], a, ti.n0 + c * 32, orow);
          st.f32(&mp.o[1], b, ti.n0 + c * 32, orow);
        }
        break;
      }
    }
    }
    half = tile_in.nrt - 1;
    release();
  }
  return true;
}

template <bool MX, bool SMP = false>
__device__ void epilogue(const Params& p, const Maps& mp, uint8_t* staging, uint64_t* acc_full,
                         uint64_t* acc_empty, uint32_t tmem_base, volatile int* abort_flag,
                         const TileQueue& tq) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ntiles = num_tiles_of(p);
  Stager st{staging + (warp - 2) * p.nbuf * STAGE_OUT_BYTES, 0u, lane, p.nbuf};
  int local = 0;
  if (!p.tile_counter && !p.clc) {
    const int t0 = SMP ? p.t0 : (int)blockIdx.x, step = SMP ? p.tstep : (int)gridDim.x;
    for (int tile = t0; tile < ntiles; tile += step) {
      const TileInfo ti = tile_info<MX>(p, tile);
      if (ti.skip) continue;
      if (!epilogue_tile<MX, SMP>(p, mp, st, acc_full, acc_empty, tmem_base, abort_flag, ti,
                                  local++))
        break;
    }
  } else {
    for (uint32_t n = 0;; ++n) {
      // lane 0 takes the warp's queue entry, the warp learns it by a shuffle
      int tile = -1;
      int ok = 1;
      if (lane == 0) ok = tq_take(p, tq, n, tile) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      tile = __shfl_sync(0xffffffffu, tile, 0);
      if (!ok) {
        if (lane == 0) {
          set_error(p.status, kErrTimeout);
          *abort_flag = 1;
        }
        break;
      }
      if (tile < 0) break;
      const TileInfo ti = tile_info<MX>(p, tile);
      if (!epilogue_tile<MX>(p, mp, st, acc_full, acc_empty, tmem_base, abort_flag, ti,
                             local++))
        break;
    }
  }
  st.drain();
}

// One instantiation per mode (and, for the dW modes, per hi/lo split): with both
// compile-time constants the compiler keeps only that launch's producer, MMA and epilogue
// code (a smaller instruction footprint, a straight-line MMA issue).
// VAR: 0 plain, 1 split (hi/lo dW operands), 2 row-tile pairs, 3 MXFP8 forward with the
// BF16 shared expert's tiles, 4 BF16 dW on SM pairs (clusters of two CTAs, M = 256 MMAs).
// Fixing the variant at compile time keeps those paths out of the other kernels' code.
template <bool MX, int MODE, int VAR>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    grouped_gemm_kernel(const __grid_constant__ Maps mp, const Params p_in) {
  using C = Cfg<MX>;
  Params p = p_in;
  p.mode = MODE;
  p.split = VAR == 1;
  p.pair = VAR == 2;
  if (VAR != 3) p.shared_tiles = 0;   // variant 3: MXFP8 forward with BF16 shared tiles
  p.smpair = VAR == 4;
  p.crank = VAR == 4 ? (int)cluster_ctarank() : 0;
  p.t0 = VAR == 4 ? (int)cluster_id_x() : 0;
  p.tstep = VAR == 4 ? (int)cluster_count_x() : 1;
  // CLC: the grid is sized to the largest tile count; a CTA past the actual count (which
  // the plan wrote to device memory) has no tile and leaves before taking any resource
  if (p.clc && (int)blockIdx.x >= num_tiles_of(p)) return;
  // barrier slots; the launch uses p.stages of them
  constexpr int STAGES = VAR == 4 ? SMP_STAGES : C::STAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* staging = smem + p.stages * p.stage_bytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::DATA_BYTES);
  uint64_t* empty = full + STAGES;
  uint64_t* acc_full = empty + STAGES;
  uint64_t* acc_empty = acc_full + 2;
  TileQueue tq;
  tq.full = acc_empty + 2;
  tq.empty = tq.full + TQ;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tq.empty + TQ);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  tq.tile = abort_flag + 1;
  ClcState clc;
  clc.bar = reinterpret_cast<uint64_t*>(smem + C::DATA_BYTES + C::BAR_BYTES / 2);
  clc.answer = smem + C::DATA_BYTES + C::BAR_BYTES / 2 + 16;
  static_assert(C::DATA_BYTES % 16 == 0 && 2 * TQ * 8 + 2 * STAGES * 8 + 32 + 8 + 4 * TQ <=
                    C::BAR_BYTES / 2, "barrier area overlaps the CLC answer");

  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&acc_full[a], 1);
      // SM pair: one arrival per epilogue warp of both CTAs, on rank 0's barrier
      mbar_init(&acc_empty[a], VAR == 4 ? 8 : 128);
    }
    for (int q = 0; q < TQ; ++q) {
      mbar_init(&tq.full[q], 1);
      mbar_init(&tq.empty[q], 5);   // the MMA lane and lane 0 of each epilogue warp
    }
    mbar_init(clc.bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&mp.a[0]);
    tma_prefetch_desc(&mp.b[0]);
  }
  if (warp == 1) {
    if constexpr (VAR == 4) tmem_alloc_pair(tmem_slot, TMEM_COLS);
    else tmem_alloc(tmem_slot, TMEM_COLS);
  }
  tc_fence_before();
  if (VAR == 4) cluster_sync_all();   // both CTAs' barriers initialised, TMEM allocated
  else __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    if (threadIdx.x == 0) {
      produce<MX, VAR == 4>(p, mp, smem, full, empty, abort_flag, tq, clc);
      // leave no request in flight: its answer is written to this CTA's shared memory
      int unused;
      if (clc.in_flight && !clc_answer(p, clc, unused)) set_error(p.status, kErrTimeout);
    }
  } else if (warp == 1) {
    if constexpr (VAR == 4) {
      if ((threadIdx.x & 31) == 0 && p.crank == 0) {
        const int n = mma_issue_pair<MX>(p, smem, full, empty, acc_full, acc_empty, tmem_base,
                                         abort_flag);
        mma_drain_pair(p, acc_empty, n);
      }
    } else if ((threadIdx.x & 31) == 0) {
      mma_issue<MX>(p, smem, full, empty, acc_full, acc_empty, tmem_base, abort_flag, tq);
    }
  } else {
    epilogue<MX, VAR == 4>(p, mp, staging, acc_full, acc_empty, tmem_base, abort_flag, tq);
  }
  tc_fence_before();
  if constexpr (VAR == 4) {
    __syncwarp();
    cluster_sync_all();   // no traffic of either CTA into the other is left
  } else {
    __syncthreads();
  }
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    if constexpr (VAR == 4) tmem_dealloc_pair(tmem_base, TMEM_COLS);
    else tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

// ------------------------------------------------------------------ forward megakernel
// One persistent launch for dispatch, the grouped up|gate and down GEMMs and the combine
// of the routed experts ([C] "O que e o MoK", "Granularidade do overlap", "Ring token
// buffers (macrobatch)"; [S] "Das Scheduling"). Its CTAs (one per SM, co-resident by a
// cooperative launch) are split in software:
//
//   CTAs 0 .. n_comm-1   gather/combine SMs: move the dispatched rows of macrobatch m into
//                        ring slot m % S with TMA bulk copies (MXFP8: quantised along H on
//                        the way), 128-row tile by tile, and combine finished macrobatches;
//   the other CTAs       GEMM SMs: the warp-specialised tcgen05 pipeline above, over a fixed
//                        task order: for each macrobatch, its up|gate tiles, then its down
//                        tiles; task i goes to GEMM CTA i mod G.
//
// The sides signal through device counters (release adds, acquire loads):
//   gathered[m][r]  row tile r of m is in its slot           (up|gate tiles of r wait)
//   hcnt[m][r]      up|gate tiles of row tile r done         (down tiles of r wait for all)
//   upg_done[m]     up|gate tiles of m done: slot m % S is free again (gather m + S waits)
//   down_done[m]    down tiles of m done                     (combine of m waits)
// Every dependency points to an earlier task, and each CTA takes its tasks in order, so the
// earliest unfinished task can always run. Every wait is bounded; on expiry the waiter
// records MOK_ERR_TIMEOUT, raises the shared abort flag and returns.
struct MegaParams {
  Params up, down;
  int M, S, P_slot, Tm, T, H, I, E, k, mt_m_max, n_comm, has_shared;
  const int32_t* mstart;
  const int32_t* mcount;
  const int32_t* mpoff;
  const int32_t* mtile_expert;
  const int32_t* mtiles;
  const int32_t* mrow0;
  const int32_t* table;
  const int32_t* topk_idx;
  const int32_t* inv;
  const float* gates;
  const uint8_t* x;     // [T][H] bf16
  uint8_t* ring;        // [S][P_slot][H] bf16 (MXFP8: e4m3)
  uint8_t* ring_sf;     // MXFP8: atoms [S][P_slot/128][H/128]
  const void* O;        // expert outputs [P_cat][H]: fp32, or bf16 with out_bf16
  const void* Os;       // shared expert output [T][H] or null (O's type)
  void* y;              // [T][H] (O's type)
  int out_bf16;
  int* cnt;             // counters (MegaCnt layout), zero at launch
  uint32_t* status;
  unsigned long long* trace;   // optional: kTraceStamps %globaltimer stamps per CTA
  int withhold;                // test hook: never publish row tile 0 of macrobatch 0
};
struct MegaMaps {
  Maps up, down;
};

constexpr int kCommWarps = NUM_THREADS / 32;
constexpr int kCopyChunk = 8192;                 // bytes per bulk copy
// chunk buffers per warp: loads in flight = buffers - 1 (MXFP8 has less shared memory)
template <bool MX>
__host__ __device__ constexpr int copy_bufs() { return MX ? 3 : 4; }
template <bool MX>
__host__ __device__ constexpr int comm_zero_off() { return kCommWarps * copy_bufs<MX>() * kCopyChunk; }
template <bool MX>
__host__ __device__ constexpr int comm_src_off() { return comm_zero_off<MX>() + kCopyChunk; }   // 128 ints

// Bounded wait until *c >= need (acquire). False if the deadline passed or another CTA
// raised the abort flag.
__device__ bool wait_count(const int* c, int need, int* abort_g, uint32_t* status,
                           uint64_t timeout_ns) {
  const uint64_t deadline = globaltimer_ns() + timeout_ns;
  uint32_t spins = 0;
  while (ld_acquire(c) < need) {
    if ((++spins & 63u) == 0) {
      if (ld_relaxed(abort_g)) return false;
      if (globaltimer_ns() > deadline) {
        set_error(status, kErrTimeout);
        atomicExch(abort_g, 1);
        return false;
      }
    }
    __nanosleep(64);
  }
  return true;
}

__device__ __forceinline__ int mega_mtiles(const MegaParams& q, int m) {
  return min(max(q.mtiles[m], 0), q.mt_m_max);
}

// Task t of a phase: the pair-interleaved order of the standalone routed GEMMs (row tile
// 2 (g / n_tiles) + (t & 1), column block g mod n_tiles with g = t / 2).
__device__ __forceinline__ int mega_row_tile(const Params& p, int t) {
  return ((t >> 1) / p.n_tiles) * 2 + (t & 1);
}

__device__ __forceinline__ TileInfo mega_tile(const MegaParams& q, int m, int ph, int t) {
  const Params& p = ph ? q.down : q.up;
  const int r = mega_row_tile(p, t), n = (t >> 1) % p.n_tiles;
  TileInfo ti;
  const int e = r < q.mt_m_max ? q.mtile_expert[(size_t)m * q.mt_m_max + r] : 0;
  ti.e = (e < 0 || e >= q.E) ? 0 : e;
  ti.row0 = q.mrow0[m] + r * BM;                                   // h, U, V, O rows
  ti.arow0 = ph ? ti.row0 : (m % q.S) * q.P_slot + r * BM;        // ring slot rows
  ti.n0 = n * (ph ? p.BN : 128);
  ti.kiters = p.kiters;
  ti.krow0 = 0;
  ti.klast = 4;
  ti.skip = r >= mega_mtiles(q, m);
  ti.nrt = 1;
  ti.bf = 0;
  ti.norows = 0;
  return ti;
}

// Calls f(m, phase, t) for GEMM CTA g's tasks in order; stops when f returns false.
template <class F>
__device__ void mega_for_each(const MegaParams& q, int g, int G, F&& f) {
  int base = 0;   // tasks before the current phase, mod G
  for (int m = 0; m < q.M; ++m) {
    const int mt = mega_mtiles(q, m);
    for (int ph = 0; ph < 2; ++ph) {
      const int n = ((mt + 1) / 2) * 2 * (ph ? q.down.n_tiles : q.up.n_tiles);
      int t = (g - base) % G;
      if (t < 0) t += G;
      for (; t < n; t += G)
        if (!f(m, ph, t)) return;
      base = (base + n) % G;
    }
  }
}

// Gather row tile r of macrobatch m into its ring slot. The tile's 128 source tokens are
// looked up once (all threads) into shared memory. Each warp then moves rows warp, warp+6,
// ...: lane 0 keeps NB - 1 bulk loads (global -> shared) in flight over NB chunk buffers;
// the lanes copy each landed chunk to the ring (MXFP8: convert it, blocks of 32 along H,
// to E4M3 codes and scale bytes). Padding rows are
// zeros. Called by all threads of the CTA.
//
// The lanes write the ring with ordinary stores from the shared-memory chunk: bulk stores
// would queue behind the bulk loads in flight on the SM's copy engine, leaving one load in
// flight per warp.
template <bool MX>
__device__ bool mega_gather_tile(const MegaParams& q, int m, int r, uint8_t* bufs, const uint8_t* zero,
                                 int* s_src, uint64_t* bars, uint32_t& phase, int* abort_g) {
  constexpr int NB = copy_bufs<MX>();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int e_raw = q.mtile_expert[(size_t)m * q.mt_m_max + r];
  const int e = (e_raw < 0 || e_raw >= q.E) ? 0 : e_raw;
  const int slot_row0 = (m % q.S) * q.P_slot + r * BM;   // ring row of the tile's row 0
  const uint32_t rowbytes = (uint32_t)q.H * 2;          // bf16 source row
  __syncthreads();   // s_src of the previous tile is no longer read
  if (threadIdx.x < BM) {
    const int po = q.mpoff[(size_t)m * (q.E + 1) + e];
    const int cnt = q.mcount[(size_t)m * q.E + e];
    const int st = q.mstart[(size_t)m * q.E + e];
    const int local = r * BM + (int)threadIdx.x - po;   // row of e inside macrobatch m
    s_src[threadIdx.x] = (local >= 0 && local < cnt) ? q.table[2 * (size_t)(st + local)] : -1;
  }
  __syncthreads();
  const int nch = (int)((rowbytes + kCopyChunk - 1) / kCopyChunk);
  const int nrows = (BM - warp + kCommWarps - 1) / kCommWarps;
  const int V = nrows * nch;
  uint8_t* mybuf = bufs + (size_t)warp * NB * kCopyChunk;
  uint64_t* mybar = bars + warp * NB;
  // chunk v: row i = warp + (v / nch) * 6 of the tile, bytes [c * chunk, ...) of the row
  auto src_of = [&](int v, uint32_t& off, uint32_t& bytes, int& i) -> const uint8_t* {
    i = warp + (v / nch) * kCommWarps;
    const int c = v - (v / nch) * nch;
    off = (uint32_t)c * kCopyChunk;
    bytes = min((uint32_t)kCopyChunk, rowbytes - off);
    const int t = s_src[i];
    return t < 0 ? nullptr : q.x + (size_t)t * rowbytes + off;
  };
  uint32_t pending = 0;   // buffers with a load in flight (every lane tracks the same)
  auto issue_load = [&](int v) {   // lane 0 issues; every lane records it
    uint32_t off, bytes;
    int i;
    const uint8_t* src = src_of(v, off, bytes, i);
    if (src) {
      if (lane == 0) {
        uint64_t* bar = mybar + v % NB;
        mbar_arrive_expect_tx(bar, bytes);
        bulk_load(mybuf + (v % NB) * kCopyChunk, src, bytes, bar);
      }
      pending |= 1u << (v % NB);
    }
  };
  bool ok = true;
  for (int v = 0; v < min(NB - 1, V); ++v) issue_load(v);
  for (int v = 0; v < V; ++v) {
    uint32_t off, bytes;
    int i;
    const uint8_t* src = src_of(v, off, bytes, i);
    const int b = v % NB;
    uint8_t* buf = mybuf + b * kCopyChunk;
    const size_t ring_row = (size_t)slot_row0 + i;
    if (src) {   // every lane waits for the load (the MXFP8 path reads it)
      const bool got = mbar_wait(mybar + b, (phase >> b) & 1u, globaltimer_ns() + q.up.timeout_ns);
      if (!__all_sync(0xffffffffu, got)) {
        if (lane == 0) {
          set_error(q.status, kErrTimeout);
          atomicExch(abort_g, 1);
        }
        ok = false;
        break;
      }
      phase ^= 1u << b;
      pending &= ~(1u << b);
    }
    if (!MX) {
      // the lanes store the chunk with 16-byte stores, so stores never queue behind the
      // bulk loads in flight
      uint4* dst = reinterpret_cast<uint4*>(q.ring + ring_row * rowbytes + off);
      const uint4* from = reinterpret_cast<const uint4*>(src ? buf : zero);
      for (int u = lane; u < (int)(bytes / 16); u += 32) dst[u] = from[u];
    } else {
      // groups of 8 bf16 (16 bytes): 4 neighbouring lanes hold one block of 32 along H
      // (conflict-free 16-byte reads; the block maximum over two shuffles). Every lane runs
      // the same number of passes so the shuffles stay converged.
      const int ngrp = (int)(bytes / 16);
      const size_t hrow = ring_row * (size_t)q.H;          // e4m3 row start
      for (int g0 = 0; g0 < ngrp; g0 += 32) {
        const int gi = g0 + lane;
        const bool act = gi < ngrp;
        float f[8];
        float amax = 0.f;
        if (src && act) {
          const uint4 w = *reinterpret_cast<const uint4*>(buf + gi * 16);
          const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&w);
#pragma unroll
          for (int z = 0; z < 4; ++z) {
            const float2 t2 = __bfloat1622float2(h2[z]);
            f[2 * z] = t2.x;
            f[2 * z + 1] = t2.y;
            amax = fmaxf(amax, fmaxf(fabsf(t2.x), fabsf(t2.y)));
          }
        } else {
#pragma unroll
          for (int z = 0; z < 8; ++z) f[z] = 0.f;
        }
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
        if (!act) continue;
        const uint32_t sb = mx_scale_byte(amax);
        const float inv = mx_inv_scale(sb);
        uint2 qv;
        qv.x = (uint32_t)f32x2_to_e4m3x2(f[0] * inv, f[1] * inv) |
               ((uint32_t)f32x2_to_e4m3x2(f[2] * inv, f[3] * inv) << 16);
        qv.y = (uint32_t)f32x2_to_e4m3x2(f[4] * inv, f[5] * inv) |
               ((uint32_t)f32x2_to_e4m3x2(f[6] * inv, f[7] * inv) << 16);
        const int hk = (int)(off / 2) + gi * 8;              // H index of the group
        *reinterpret_cast<uint2*>(q.ring + hrow + hk) = qv;
        if ((lane & 3) == 0) {
          const size_t atom = (ring_row >> 7) * (size_t)(q.H / 128) + (size_t)(hk >> 7);
          q.ring_sf[atom * 512 + atom_byte((int)(ring_row & 127), hk)] = (uint8_t)sb;
        }
      }
    }
    // every lane has consumed chunk v - 1's buffer (its values fed stores already issued),
    // so the next bulk load may refill it
    __syncwarp();
    if (v + NB - 1 < V) issue_load(v + NB - 1);
  }
  if (!ok) {   // let the loads still in flight land before the CTA can leave
    for (int b = 0; b < NB; ++b)
      if (pending & (1u << b))
        mbar_wait(mybar + b, (phase >> b) & 1u, globaltimer_ns() + q.up.timeout_ns);
  }
  if (lane == 0) {
    bulk_wait_all();
    fence_proxy_async_global();
  }
  __threadfence();
  return ok;
}

// y[t] = sum_j g_tj O[row(t, j)] (+ Os[t]) for the tokens of macrobatch m, one warp per
// token, warps wi, wi + nw, ... (same arithmetic and order as the standalone combine:
// fp32 sums in slot order, then the shared expert; bf16 mode rounds y once at the end).
__device__ __forceinline__ void bf16x8_to_f32(const uint4& w, float* f) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&w);
#pragma unroll
  for (int z = 0; z < 4; ++z) {
    const float2 t2 = __bfloat1622float2(h[z]);
    f[2 * z] = t2.x;
    f[2 * z + 1] = t2.y;
  }
}
__device__ __forceinline__ uint4 f32_to_bf16x8(const float* f) {
  uint4 w;
  __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&w);
#pragma unroll
  for (int z = 0; z < 4; ++z) h[z] = __floats2bfloat162_rn(f[2 * z], f[2 * z + 1]);
  return w;
}

__device__ void mega_combine(const MegaParams& q, int m, int wi, int nw) {
  const int lane = threadIdx.x & 31;
  const int t0 = m * q.Tm, t1 = min(q.T, t0 + q.Tm);
  for (int t = t0 + wi; t < t1; t += nw) {
    int my_row = 0;
    float my_g = 0.f;
    if (lane < q.k) {
      const int sl = t * q.k + lane;
      int e = q.topk_idx[sl];
      e = (e < 0 || e >= q.E) ? 0 : e;
      my_row = q.mrow0[m] + q.mpoff[(size_t)m * (q.E + 1) + e] +
               (q.inv[sl] - q.mstart[(size_t)m * q.E + e]);
      my_g = q.gates[sl];
    }
    int rows[kMaxK];
    float g[kMaxK];
#pragma unroll
    for (int j = 0; j < kMaxK; ++j) {
      rows[j] = __shfl_sync(0xffffffffu, my_row, j);
      g[j] = __shfl_sync(0xffffffffu, my_g, j);
    }
    if (q.out_bf16) {
      // 8 bf16 (16 bytes) per vector; 2 vectors per lane per pass
      const int nvec = q.H / 8;
      const uint4* O = reinterpret_cast<const uint4*>(q.O);
      const uint4* Os = reinterpret_cast<const uint4*>(q.Os);
      uint4* y = reinterpret_cast<uint4*>(q.y);
      // every load of a pass first (k rows x U vectors, and the shared rows), then the
      // sums in slot order: with 6 warps per SM the loads in flight come from each lane
      constexpr int U = 2;
      for (int i0 = lane; i0 < nvec; i0 += 32 * U) {
        uint4 w[kMaxK][U], ws[U];
#pragma unroll
        for (int j = 0; j < kMaxK; ++j) {
          if (j < q.k) {
#pragma unroll
            for (int u = 0; u < U; ++u) {
              const int i = i0 + 32 * u;
              w[j][u] = i < nvec ? __ldcg(O + (size_t)rows[j] * nvec + i) : make_uint4(0, 0, 0, 0);
            }
          }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int i = i0 + 32 * u;
          ws[u] = (Os && i < nvec) ? __ldcg(Os + (size_t)t * nvec + i) : make_uint4(0, 0, 0, 0);
        }
        float acc[U][8];
#pragma unroll
        for (int u = 0; u < U; ++u)
#pragma unroll
          for (int z = 0; z < 8; ++z) acc[u][z] = 0.f;
#pragma unroll
        for (int j = 0; j < kMaxK; ++j) {
          if (j < q.k) {
#pragma unroll
            for (int u = 0; u < U; ++u) {
              float f[8];
              bf16x8_to_f32(w[j][u], f);
#pragma unroll
              for (int z = 0; z < 8; ++z) acc[u][z] = fmaf(g[j], f[z], acc[u][z]);
            }
          }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int i = i0 + 32 * u;
          if (i >= nvec) continue;
          if (Os) {
            float f[8];
            bf16x8_to_f32(ws[u], f);
#pragma unroll
            for (int z = 0; z < 8; ++z) acc[u][z] += f[z];
          }
          y[(size_t)t * nvec + i] = f32_to_bf16x8(acc[u]);
        }
      }
      continue;
    }
    const int nvec = q.H / 4;
    const float4* O = reinterpret_cast<const float4*>(q.O);
    const float4* Os = reinterpret_cast<const float4*>(q.Os);
    float4* y = reinterpret_cast<float4*>(q.y);
    // 4 vectors per lane per pass: with 6 warps per SM, loads in flight come from width
    constexpr int U = 4;
    for (int i0 = lane; i0 < nvec; i0 += 32 * U) {
      float4 f[kMaxK][U];   // every load of the pass first, then the sums in slot order
#pragma unroll
      for (int j = 0; j < kMaxK; ++j) {
        if (j < q.k) {
#pragma unroll
          for (int u = 0; u < U; ++u) {
            const int i = i0 + 32 * u;
            f[j][u] = i < nvec ? __ldcg(O + (size_t)rows[j] * nvec + i)
                               : make_float4(0.f, 0.f, 0.f, 0.f);
          }
        }
      }
      float4 acc[U];
#pragma unroll
      for (int u = 0; u < U; ++u) acc[u] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int j = 0; j < kMaxK; ++j) {
        if (j < q.k) {
#pragma unroll
          for (int u = 0; u < U; ++u) {
            acc[u].x = fmaf(g[j], f[j][u].x, acc[u].x);
            acc[u].y = fmaf(g[j], f[j][u].y, acc[u].y);
            acc[u].z = fmaf(g[j], f[j][u].z, acc[u].z);
            acc[u].w = fmaf(g[j], f[j][u].w, acc[u].w);
          }
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int i = i0 + 32 * u;
        if (i >= nvec) continue;
        if (Os) {
          const float4 f = __ldcg(Os + (size_t)t * nvec + i);
          acc[u].x += f.x;
          acc[u].y += f.y;
          acc[u].z += f.z;
          acc[u].w += f.w;
        }
        y[(size_t)t * nvec + i] = acc[u];
      }
    }
  }
}

// All threads: thread 0 waits for *c >= need, the CTA learns the outcome.
__device__ bool cta_wait_count(const int* c, int need, int* abort_g, uint32_t* status,
                               uint64_t timeout_ns, volatile int* s_ok) {
  if (threadIdx.x == 0) *s_ok = wait_count(c, need, abort_g, status, timeout_ns) ? 1 : 0;
  __syncthreads();
  const bool ok = *s_ok != 0;
  __syncthreads();
  return ok;
}

template <bool MX>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    fwd_mega_kernel(const __grid_constant__ MegaMaps mm, const MegaParams q) {
  using C = Cfg<MX>;
  constexpr int STAGES = C::STAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::DATA_BYTES);
  uint64_t* empty = full + STAGES;
  uint64_t* acc_full = empty + STAGES;
  uint64_t* acc_empty = acc_full + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_empty + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* s_ok = abort_flag + 1;
  volatile int* s_pub = abort_flag + 2;   // epilogue: the tile's outcome, read by all 4 warps
  // gather SMs: 6 x NB copy barriers in the data area, after the token indices
  uint64_t* copy_bars = reinterpret_cast<uint64_t*>(smem + comm_src_off<MX>() + BM * 4);
  const MegaCnt CN = {0, q.M * q.mt_m_max, 2 * q.M * q.mt_m_max, 2 * q.M * q.mt_m_max + q.M,
                      2 * q.M * q.mt_m_max + 2 * q.M, 0};
  int* cnt = q.cnt;
  int* abort_g = cnt + CN.abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool comm = (int)blockIdx.x < q.n_comm;
  const int G = (int)gridDim.x - q.n_comm;
  unsigned long long* stamps = q.trace ? q.trace + (size_t)blockIdx.x * kTraceStamps : nullptr;
  if (stamps && threadIdx.x == 0) stamps[kStampStart] = globaltimer_ns();

  if (comm) {
    // ---------------- gather / combine SM
    uint8_t* bufs = smem;                                 // 6 warps x NB x 8 KB
    uint8_t* zero = smem + comm_zero_off<MX>();           // 8 KB of zeros
    int* s_src = reinterpret_cast<int*>(smem + comm_src_off<MX>());
    for (int i = threadIdx.x; i < kCopyChunk / 16; i += blockDim.x)
      reinterpret_cast<uint4*>(zero)[i] = make_uint4(0, 0, 0, 0);
    if (threadIdx.x == 0) {
      for (int i = 0; i < kCommWarps * copy_bufs<MX>(); ++i) mbar_init(&copy_bars[i], 1);
      fence_mbar_init();
    }
    fence_proxy_async_smem();   // the zero chunk is read by bulk stores
    __syncthreads();
    uint32_t phase = 0;
    const int c = blockIdx.x;
    bool ok = true;
    for (int m = 0; m < q.M && ok; ++m) {
      if (m >= q.S)   // slot m % S drains when every up|gate tile of m - S has read it
        ok = cta_wait_count(cnt + CN.upg_done + (m - q.S), mega_mtiles(q, m - q.S) * q.up.n_tiles,
                            abort_g, q.status, q.up.timeout_ns, s_ok);
      const int mt = mega_mtiles(q, m);
      for (int r = c; r < mt && ok; r += q.n_comm) {
        ok = mega_gather_tile<MX>(q, m, r, bufs, zero, s_src, copy_bars, phase, abort_g);
        ok = __syncthreads_and(ok ? 1 : 0) != 0;
        if (ok && threadIdx.x == 0 && !(q.withhold && m == 0 && r == 0))
          red_release_add(cnt + CN.gathered + m * q.mt_m_max + r, 1);
      }
      if (ok && m >= 1) {   // combine the previous macrobatch while the GEMMs run this one
        ok = cta_wait_count(cnt + CN.down_done + (m - 1),
                            mega_mtiles(q, m - 1) * q.down.n_tiles, abort_g, q.status, q.up.timeout_ns, s_ok);
        if (ok) mega_combine(q, m - 1, c * kCommWarps + warp, q.n_comm * kCommWarps);
      }
    }
    if (stamps && threadIdx.x == 0) stamps[kStampCommDone] = globaltimer_ns();
    if (!ok) return;
  } else {
    // ---------------- GEMM SM
    const int g = (int)blockIdx.x - q.n_comm;
    uint8_t* staging = smem + q.up.stages * q.up.stage_bytes;
    if (threadIdx.x == 0) {
      for (int s2 = 0; s2 < STAGES; ++s2) {
        mbar_init(&full[s2], 1);
        mbar_init(&empty[s2], 1);
      }
      for (int a = 0; a < 2; ++a) {
        mbar_init(&acc_full[a], 1);
        mbar_init(&acc_empty[a], 128);
      }
      *abort_flag = 0;
      fence_mbar_init();
    }
    if (warp == 1) tmem_alloc(tmem_slot, TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    if (warp == 0) {
      if (lane == 0) {
        uint32_t it = 0;
        mega_for_each(q, g, G, [&](int m, int ph, int t) {
          const Params& p = ph ? q.down : q.up;
          const TileInfo ti = mega_tile(q, m, ph, t);
          if (ti.skip) return true;
          const int r = mega_row_tile(p, t);
          const int* dep = cnt + (ph ? CN.hcnt : CN.gathered) + m * q.mt_m_max + r;
          if (!wait_count(dep, ph ? q.up.n_tiles : 1, abort_g, q.status, q.up.timeout_ns)) {
            *abort_flag = 1;
            return false;
          }
          fence_proxy_async_global();   // the TMA reads below follow the acquire
          return produce_tile<MX>(p, ph ? mm.down : mm.up, smem, full, empty, abort_flag, ti, it);
        });
        produce_drain<MX>(q.up, full, empty, it);
        if (stamps) stamps[kStampProducerDone] = globaltimer_ns();
      }
    } else if (warp == 1) {
      if (lane == 0) {
        uint32_t it = 0;
        int local = 0;
        mega_for_each(q, g, G, [&](int m, int ph, int t) {
          const TileInfo ti = mega_tile(q, m, ph, t);
          if (ti.skip) return true;
          return mma_tile<MX>(ph ? q.down : q.up, smem, full, empty, acc_full, acc_empty,
                              tmem_base, abort_flag, ti, it, local++);
        });
      }
    } else {
      Stager st{staging + (warp - 2) * q.up.nbuf * STAGE_OUT_BYTES, 0u, lane, q.up.nbuf};
      int local = 0;
      mega_for_each(q, g, G, [&](int m, int ph, int t) {
        const Params& p = ph ? q.down : q.up;
        const TileInfo ti = mega_tile(q, m, ph, t);
        if (ti.skip) return true;   // every epilogue warp skips the same tasks
        // a warp that timed out has raised the CTA's abort flag; every warp still meets
        // the others at the barrier below, and after it all of them see the flag
        epilogue_tile<MX>(p, ph ? mm.down : mm.up, st, acc_full, acc_empty, tmem_base,
                          abort_flag, ti, local++);
        // publish the tile: its TMA stores have landed (and, MXFP8, the plain stores of h)
        if (lane == 0) {
          bulk_wait_all();
          fence_proxy_async_global();
        }
        __threadfence();
        named_bar_sync(1, 128);
        if (threadIdx.x == 64) {   // one reader, so the four warps decide alike
          const int ok64 = *abort_flag == 0;
          *s_pub = ok64;
          if (ok64) {
            const int r = mega_row_tile(p, t);
            if (ph == 0) {
              red_release_add(cnt + CN.hcnt + m * q.mt_m_max + r, 1);
              red_release_add(cnt + CN.upg_done + m, 1);
            } else {
              red_release_add(cnt + CN.down_done + m, 1);
            }
          }
        }
        named_bar_sync(1, 128);
        const bool ok = *s_pub != 0;
        named_bar_sync(1, 128);   // s_pub is rewritten only after every warp has read it
        return ok;
      });
      st.drain();
      if (stamps && threadIdx.x == 64) stamps[kStampGemmDone] = globaltimer_ns();
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
      __syncwarp();
      tc_fence_after();
      tmem_dealloc(tmem_base, TMEM_COLS);
    }
  }
  // ---------------- last macrobatch: every CTA combines
  const int mlast = q.M - 1;
  if (!cta_wait_count(cnt + CN.down_done + mlast, mega_mtiles(q, mlast) * q.down.n_tiles,
                      abort_g, q.status, q.up.timeout_ns, s_ok))
    return;
  if (stamps && threadIdx.x == 0) stamps[kStampCombine] = globaltimer_ns();
  mega_combine(q, mlast, (int)blockIdx.x * kCommWarps + warp, (int)gridDim.x * kCommWarps);
  if (stamps) {
    __syncthreads();
    if (threadIdx.x == 0) stamps[kStampEnd] = globaltimer_ns();
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

// 2-D tensor map over a row-major [rows][cols] matrix of 1- or 2-byte elements, box
// (128 bytes of columns, box_rows rows), 128-byte swizzle; reads outside return zeros.
bool make_map(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows, int box_rows,
              int elem_bytes) {
  EncodeTiledFn enc = get_encode_fn();
  if (!enc || base == nullptr) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * elem_bytes};
  cuuint32_t box[2] = {(cuuint32_t)(128 / elem_bytes), (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(m, elem_bytes == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8,
                   2, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Output map for the epilogue's boxes of 32 rows: fp32 32 columns (128-byte rows,
// 128-byte swizzle), bf16 32 columns (64-byte rows, 64-byte swizzle) or, with wide, bf16 64
// columns (128-byte rows, 128-byte swizzle); stores outside the matrix are dropped.
bool make_out_map(CUtensorMap* m, void* base, uint64_t cols, uint64_t rows, int elem_bytes,
                  bool wide = false) {
  EncodeTiledFn enc = get_encode_fn();
  if (!enc || base == nullptr) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * elem_bytes};
  const bool sw128 = elem_bytes == 4 || wide;
  cuuint32_t box[2] = {(cuuint32_t)(elem_bytes == 2 && wide ? 64 : 32), 32};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(m, elem_bytes == 4 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                   2, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   sw128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                   CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}
// the map of an fp32 or (out_bf16) bf16 64-column-box output
bool make_res_map(CUtensorMap* m, void* base, uint64_t cols, uint64_t rows, bool out_bf16) {
  return out_bf16 ? make_out_map(m, base, cols, rows, 2, true) : make_out_map(m, base, cols, rows, 4);
}

// Kernel parameters and tensor maps of one grouped-GEMM call; max_tiles = tiles of the
// largest possible problem (the launch's grid bound).
template <bool MX>
cudaError_t build_call(const GemmCall& c, Params& p, Maps& mp, int& max_tiles) {
  using C = Cfg<MX>;
  if (MX && c.dense) return cudaErrorNotSupported;  // the shared expert stays BF16
  memset(&p, 0, sizeof(p));
  p.mode = c.mode;
  p.dense = c.dense ? 1 : 0;
  p.M_rows = c.M_rows;
  p.H = c.H;
  p.I = c.I;
  p.k = c.k;
  p.groups = c.dense ? 1 : c.groups;
  p.split = (!MX && c.split && (c.mode == kBwdDWDown || c.mode == kBwdDWUpGate)) ? 1 : 0;
  static_assert(2 * SPLIT_STAGE_BYTES + 2 * OUT_STAGING <= Cfg<false>::DATA_BYTES,
                "split stages and staging exceed the data area");
  p.lo_out = (!MX && c.mode == kBwdDH && c.out[1] && c.out[3] && c.out[5]) ? 1 : 0;
  p.out_bf16 = (c.out_bf16 && (c.mode == kFwdDown || c.mode == kBwdDX || c.mode == kBwdDWDown ||
                               c.mode == kBwdDWUpGate)) ? 1 : 0;
  const bool ob = p.out_bf16 != 0;
  p.timeout_ns = c.timeout_ns > 0 ? c.timeout_ns : kTimeoutNs;
  // Modes without split keep the full operand ring (trading a stage for deeper output
  // staging made the dW modes slower).
  p.stages = MX ? C::MX_STAGES : C::STAGES;
  p.nbuf = 2;
  p.stage_bytes = C::STAGE_BYTES;
  p.sf_off = C::SF_OFF;
  p.nacc = C::NACC;
  p.acc_cols = C::ACC_COLS;
  if (p.split) {   // two chunk-sized hi/lo stages leave room for 4 staging boxes per warp
    p.stages = 2;
    p.nbuf = 4;
    p.stage_bytes = SPLIT_STAGE_BYTES;
  }
  // MXFP8 stages and staging per mode (see Cfg::DATA_BYTES)
  if (MX) {
    p.nbuf = 4;
    if (c.mode == kFwdUpGate) {
      p.stages = 4;
      p.nbuf = 1;
    } else if (c.mode == kBwdDH && c.H % 256 == 0) {
      p.stages = C::MX_DH_STAGES;
      p.stage_bytes = C::MX_DH_STAGE_BYTES;
      p.sf_off = 4 * A_BYTES;
      p.kdouble = 1;
    }
  }
  static_assert(4 * Cfg<true>::STAGE_BYTES + OUT_STAGING / 2 <= Cfg<true>::DATA_BYTES &&
                    3 * Cfg<true>::STAGE_BYTES + 2 * OUT_STAGING <= Cfg<true>::DATA_BYTES &&
                    Cfg<true>::MX_DH_STAGES * Cfg<true>::MX_DH_STAGE_BYTES <= Cfg<true>::DATA_BYTES,
                "MXFP8 stages and staging exceed the data area");
  static_assert(Cfg<true>::MX_DH_STAGE_BYTES % 1024 == 0 && Cfg<true>::STAGE_BYTES % 1024 == 0,
                "stages must keep the 1024-byte alignment of the swizzled tiles");
  p.poff = c.poff;
  p.counts = c.counts;
  p.offsets = c.offsets;
  p.tile_expert = c.tile_expert;
  p.num_mtiles = c.num_mtiles;
  p.table = c.table;
  p.gates = c.gates;
  p.u = c.u;
  p.v = c.v;
  p.uv_row = c.uv_row;
  p.tile_counter = c.tile_counter;
  p.clc = c.clc ? 1 : 0;
  p.pair = (!MX && c.pair && !c.dense && !p.split && c.ptile && c.num_ptiles &&
            (c.mode == kFwdUpGate || c.mode == kFwdDown || c.mode == kBwdDX))
               ? 1 : 0;
  p.ptile = c.ptile;
  p.num_ptiles = c.num_ptiles;
  p.max_ptiles = c.max_ptiles;
  p.smpair = (!MX && c.smpair && !p.split && !c.tile_counter && !c.clc &&
              (c.mode == kBwdDWDown || c.mode == kBwdDWUpGate ||
               (c.mode == kBwdDH && (c.dense || (c.ptile && c.num_ptiles))))) ? 1 : 0;
  const bool mixed = MX && c.s_a && (c.mode == kFwdUpGate || c.mode == kFwdDown);
  p.dgp = c.dgp;
  p.status = c.status;
  p.sfa = static_cast<const uint8_t*>(c.sfa);
  p.sfa1 = static_cast<const uint8_t*>(c.sfa1);
  p.sfb0 = static_cast<const uint8_t*>(c.sfb0);
  p.sfb1 = static_cast<const uint8_t*>(c.sfb1);
  for (int i = 0; i < 5; ++i) {
    p.out_q[i] = static_cast<uint8_t*>(c.out_q[i]);
    p.out_sf[i] = static_cast<uint8_t*>(c.out_sf[i]);
  }

  const int eb = MX ? 1 : 2;                  // element bytes of the GEMM operands
  const uint64_t rows = (uint64_t)c.M_rows;   // rows of the row-space buffers
  const uint64_t arows = c.a_rows > 0 ? (uint64_t)c.a_rows : rows;  // rows of A's buffer
  const uint64_t G = (uint64_t)p.groups;
  memset(&mp, 0, sizeof(mp));
  bool ok = true;
  max_tiles = 0;
  const int mt_rows = (int)((rows + BM - 1) / BM);
  const int BK = C::BK;
  switch (c.mode) {
    case kFwdUpGate:
      p.BN = 256;
      p.n_tiles = c.I / 128;
      p.kiters = c.H / BK;
      p.kcs_a = c.H / 128;
      p.kcs_b = c.H / 128;
      p.ncs_b = c.I / 128;
      ok = make_map(&mp.a[0], c.a[0], c.H, arows, BM, eb) &&
           make_map(&mp.b[0], c.b[0], c.I, G * c.H, BK, eb) &&
           make_map(&mp.b[1], c.b[1], c.I, G * c.H, BK, eb) &&
           (MX || make_out_map(&mp.o[0], c.out[0], c.I, rows, 2)) &&
           make_out_map(&mp.o[1], c.out[1], c.I, rows, 2, true) &&
           make_out_map(&mp.o[2], c.out[2], c.I, rows, 2, true);
      max_tiles = mt_rows * p.n_tiles;
      break;
    case kFwdDown:
      p.BN = (c.H % 256 == 0) ? 256 : 128;
      p.n_tiles = c.H / p.BN;
      p.kiters = c.I / BK;
      p.kcs_a = c.I / 128;
      p.kcs_b = c.I / 128;
      p.ncs_b = c.H / 128;
      ok = make_map(&mp.a[0], c.a[0], c.I, rows, BM, eb) &&
           make_map(&mp.b[0], c.b[0], c.H, G * c.I, BK, eb) &&
           make_res_map(&mp.o[0], c.out[0], c.H, rows, ob);
      max_tiles = mt_rows * p.n_tiles;
      break;
    case kRouter:
      if (MX || !c.dense) return cudaErrorNotSupported;
      // the fewest column tiles of at most 256 columns (one launch round of long-K tiles,
      // K = 3H, and the fewest x re-reads), each as narrow as they allow in steps of 64
      // (E = 384: two of 192, not 256 + 128 of which half past E); columns past E load as
      // zeros
      p.n_tiles = (c.n_out + 255) / 256;
      p.BN = ((c.n_out + p.n_tiles - 1) / p.n_tiles + 63) / 64 * 64;
      p.n_out = c.n_out;
      p.bias = c.bias;
      p.logits = static_cast<float*>(c.out[0]);
      p.kiters = 3 * (c.H / BK);
      ok = c.ld_b % 64 == 0 && c.ld_b >= c.n_out &&
           make_map(&mp.a[0], c.a[0], c.H, rows, BM, eb) &&
           make_map(&mp.b[0], c.b[0], c.ld_b, 3 * (uint64_t)c.H, BK, eb);
      max_tiles = mt_rows * p.n_tiles;
      break;
    case kBwdDH:
      // MXFP8: 128-column tiles, so that two accumulators fit next to the scale columns
      // and the long epilogue overlaps the next tile's MMAs
      p.BN = (!MX && c.I % 256 == 0) ? 256 : 128;
      if (MX) {
        p.nacc = 2;
        p.acc_cols = 128;
      }
      p.n_tiles = c.I / p.BN;
      p.kiters = c.H / BK / (p.kdouble ? 2 : 1);
      p.kcs_a = c.H / 128;
      p.kcs_b = c.H / 128;
      p.ncs_b = c.I / 128;
      // SM pairs: each CTA copies half of the weight tile's rows
      ok = make_map(&mp.a[0], c.a[0], c.H, rows, BM, eb) &&
           make_map(&mp.b[0], c.b[0], c.H, G * c.I, p.smpair ? p.BN / 2 : p.BN, eb);
      for (int i = 0; i < 6 && ok && !MX; ++i)
        if (i % 2 == 0 || p.lo_out) ok = make_out_map(&mp.o[i], c.out[i], c.I, rows, 2);
      max_tiles = mt_rows * p.n_tiles;
      break;
    case kBwdDX:
      p.BN = (c.H % 256 == 0) ? 256 : 128;
      p.n_tiles = c.H / p.BN;
      p.kiters = 2 * (c.I / BK);
      p.kcs_a = c.I / 128;
      p.kcs_b = c.I / 128;
      p.ncs_b = c.H / 128;
      for (int i = 0; i < 2 && ok; ++i) ok = make_map(&mp.a[i], c.a[i], c.I, rows, BM, eb);
      ok = ok && make_map(&mp.b[0], c.b[0], c.I, G * c.H, p.BN, eb) &&
           make_map(&mp.b[1], c.b[1], c.I, G * c.H, p.BN, eb) &&
           make_res_map(&mp.o[0], c.out[0], c.H, rows, ob);
      max_tiles = mt_rows * p.n_tiles;
      break;
    case kBwdDWDown:
      p.BN = (c.H % 256 == 0) ? 256 : 128;
      p.n_tiles = c.H / p.BN;
      p.m_tiles_dw = c.I / BM;
      for (int i = 0; i < (p.split ? 2 : 1) && ok; ++i) ok = make_map(&mp.a[i], c.a[i], c.I, rows, BK, eb);
      ok = ok && make_map(&mp.b[0], c.b[0], c.H, rows, BK, eb) &&
           make_res_map(&mp.o[0], c.out[0], c.H, G * c.I, ob);
      max_tiles = p.groups * p.m_tiles_dw * p.n_tiles;
      break;
    case kBwdDWUpGate:
      p.BN = 256;
      p.n_tiles = c.I / 128;
      p.m_tiles_dw = c.H / BM;
      ok = make_map(&mp.a[0], c.a[0], c.H, rows, BK, eb);
      for (int i = 0; i < (p.split ? 4 : 2) && ok; ++i) ok = make_map(&mp.b[i], c.b[i], c.I, rows, BK, eb);
      ok = ok && make_res_map(&mp.o[0], c.out[0], c.I, G * c.H, ob) &&
           make_res_map(&mp.o[1], c.out[1], c.I, G * c.H, ob);
      max_tiles = p.groups * p.m_tiles_dw * p.n_tiles;
      break;
  }
  // routed row-space launches number their tiles in row-tile pairs (num_tiles_of)
  if (!p.dense && !is_dw(c.mode)) max_tiles = (mt_rows + 1) / 2 * 2 * p.n_tiles;
  if (mixed && ok) {   // the BF16 shared expert's tiles after the routed ones
    const uint64_t T = (uint64_t)c.s_rows;
    if (c.s_rows <= 0 || c.s_I <= 0 || c.s_I % 128) return cudaErrorInvalidValue;
    p.s_rows = c.s_rows;
    p.s_I = c.s_I;
    if (c.mode == kFwdUpGate) {
      p.s_n_tiles = c.s_I / 128;
      p.s_kiters = c.H / Cfg<false>::BK;
      p.s_BN = 256;
      ok = make_map(&mp.a[2], c.s_a, c.H, T, BM, 2) &&
           make_map(&mp.b[2], c.s_b[0], c.s_I, c.H, Cfg<false>::BK, 2) &&
           make_map(&mp.b[3], c.s_b[1], c.s_I, c.H, Cfg<false>::BK, 2) &&
           make_out_map(&mp.o[3], c.s_out[0], c.s_I, T, 2) &&
           make_out_map(&mp.o[4], c.s_out[1], c.s_I, T, 2, true) &&
           make_out_map(&mp.o[5], c.s_out[2], c.s_I, T, 2, true);
    } else {
      p.s_BN = (c.H % 256 == 0) ? 256 : 128;
      p.s_n_tiles = c.H / p.s_BN;
      p.s_kiters = c.s_I / Cfg<false>::BK;
      ok = make_map(&mp.a[2], c.s_a, c.s_I, T, BM, 2) &&
           make_map(&mp.b[2], c.s_b[0], c.H, c.s_I, Cfg<false>::BK, 2) &&
           make_res_map(&mp.o[3], c.s_out[0], c.H, T, ob);
    }
    p.shared_tiles = (int)((T + BM - 1) / BM) * p.s_n_tiles;
    max_tiles += p.shared_tiles;
  }
  if (p.smpair && is_dw(c.mode) && p.m_tiles_dw % 2) p.smpair = 0;   // 256-row tiles only
  if (p.smpair) {   // six [A | half of B] stages; max_tiles counts pair tiles
    static_assert(SMP_STAGES * SMP_STAGE_BYTES + OUT_STAGING <= Cfg<false>::DATA_BYTES &&
                      SMP_STAGE_BYTES % 1024 == 0,
                  "SM-pair stages exceed the data area");
    p.stages = SMP_STAGES;
    p.stage_bytes = SMP_STAGE_BYTES;
    p.nbuf = 2;
    if (is_dw(c.mode))
      max_tiles = p.groups * (p.m_tiles_dw / 2) * p.n_tiles;
    else
      max_tiles = (p.dense ? (mt_rows + 1) / 2 : (p.max_ptiles > 0 ? p.max_ptiles : 0)) * p.n_tiles;
  }
  if (p.pair) {   // three [A0 | B | A1] stages, both accumulators for one tile
    static_assert(3 * PAIR_STAGE_BYTES + OUT_STAGING <= Cfg<false>::DATA_BYTES &&
                      PAIR_STAGE_BYTES % 1024 == 0 && PAIR_A1_OFF % 1024 == 0,
                  "row-tile pair stages exceed the data area");
    p.stages = 3;
    p.stage_bytes = PAIR_STAGE_BYTES;
    p.nbuf = 2;
    p.nacc = 1;
    p.acc_cols = 512;
    max_tiles = (p.max_ptiles > 0 ? p.max_ptiles : 0) * p.n_tiles;
  }
  if (!ok) return cudaErrorInvalidValue;
  return cudaSuccess;
}

using GemmKernel = void (*)(const Maps, const Params);

template <bool MX>
GemmKernel gemm_kernel_for(int mode, int split, int pair, int mixed, int smpair) {
  switch (mode) {
    case kFwdUpGate:
      if (MX && mixed) return grouped_gemm_kernel<MX, kFwdUpGate, MX ? 3 : 0>;
      return pair ? grouped_gemm_kernel<MX, kFwdUpGate, MX ? 0 : 2>
                  : grouped_gemm_kernel<MX, kFwdUpGate, 0>;
    case kFwdDown:
      if (MX && mixed) return grouped_gemm_kernel<MX, kFwdDown, MX ? 3 : 0>;
      return pair ? grouped_gemm_kernel<MX, kFwdDown, MX ? 0 : 2>
                  : grouped_gemm_kernel<MX, kFwdDown, 0>;
    case kBwdDH:
      if (!MX && smpair) return grouped_gemm_kernel<MX, kBwdDH, MX ? 0 : 4>;
      return grouped_gemm_kernel<MX, kBwdDH, 0>;
    case kBwdDX:
      return pair ? grouped_gemm_kernel<MX, kBwdDX, MX ? 0 : 2>
                  : grouped_gemm_kernel<MX, kBwdDX, 0>;
    case kBwdDWDown:
      if (!MX && smpair) return grouped_gemm_kernel<MX, kBwdDWDown, MX ? 0 : 4>;
      return split ? grouped_gemm_kernel<MX, kBwdDWDown, !MX> : grouped_gemm_kernel<MX, kBwdDWDown, 0>;
    case kBwdDWUpGate:
      if (!MX && smpair) return grouped_gemm_kernel<MX, kBwdDWUpGate, MX ? 0 : 4>;
      return split ? grouped_gemm_kernel<MX, kBwdDWUpGate, !MX>
                   : grouped_gemm_kernel<MX, kBwdDWUpGate, 0>;
    case kRouter: return grouped_gemm_kernel<MX, kRouter, 0>;
    default: return nullptr;
  }
}

template <bool MX>
cudaError_t launch_impl(const GemmCall& c, int num_sms, cudaStream_t s) {
  using C = Cfg<MX>;
  static bool attr_set[8][5] = {};
  static int pair_clusters[8] = {};   // SM pairs: clusters of two that fit at once (0: not asked)
  if (c.mode < 0 || c.mode >= 8) return cudaErrorInvalidValue;
  Params p;
  Maps mp;
  int max_tiles = 0;
  cudaError_t e = build_call<MX>(c, p, mp, max_tiles);
  if (e != cudaSuccess) return e;
  const GemmKernel kern =
      gemm_kernel_for<MX>(c.mode, p.split, p.pair, p.shared_tiles > 0, p.smpair);
  if (!kern) return cudaErrorInvalidValue;
  const int var = p.split ? 1 : p.pair ? 2 : p.shared_tiles > 0 ? 3 : p.smpair ? 4 : 0;
  if (!attr_set[c.mode][var]) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    attr_set[c.mode][var] = true;
  }
  if (p.smpair) {
    // persistent clusters of two: as many as fit on the device at once (a GPC with an odd
    // number of free SMs leaves one out), at most one per two SMs of the limit
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = 2;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cudaLaunchConfig_t cfg;
    memset(&cfg, 0, sizeof(cfg));
    cfg.blockDim = dim3(NUM_THREADS, 1, 1);
    cfg.dynamicSmemBytes = C::SMEM_BYTES;
    cfg.stream = s;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    if (pair_clusters[c.mode] == 0) {
      cfg.gridDim = dim3(2, 1, 1);
      int n = 0;
      e = cudaOccupancyMaxActiveClusters(&n, reinterpret_cast<const void*>(kern), &cfg);
      if (e != cudaSuccess) return e;
      pair_clusters[c.mode] = n > 0 ? n : -1;
    }
    if (pair_clusters[c.mode] < 0 || num_sms < 2) {   // no cluster of two: one CTA per tile
      GemmCall c1 = c;
      c1.smpair = false;
      return launch_impl<MX>(c1, num_sms, s);
    }
    int clusters = pair_clusters[c.mode] < num_sms / 2 ? pair_clusters[c.mode] : num_sms / 2;
    if (clusters > max_tiles) clusters = max_tiles;
    if (clusters < 1) clusters = 1;
    cfg.gridDim = dim3(2 * clusters, 1, 1);
    e = cudaLaunchKernelEx(&cfg, kern, mp, p);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
  }
  // persistent: one CTA per SM; CLC: one CTA per tile (the hardware keeps one per SM
  // running and the running CTAs cancel the rest)
  int grid = p.clc ? max_tiles : (max_tiles < num_sms ? max_tiles : num_sms);
  if (grid < 1) grid = 1;
  kern<<<grid, NUM_THREADS, C::SMEM_BYTES, s>>>(mp, p);
  return cudaGetLastError();
}

}  // namespace

template <bool MX>
cudaError_t launch_mega_impl(const MegaCall& c, int num_sms, cudaStream_t s) {
  using C = Cfg<MX>;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(fwd_mega_kernel<MX>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  static_assert(comm_src_off<MX>() + BM * 4 + kCommWarps * copy_bufs<MX>() * 8 <= C::DATA_BYTES,
                "gather buffers exceed the data area");
  MegaParams q;
  MegaMaps mm;
  memset(&q, 0, sizeof(q));
  int mt = 0;
  cudaError_t e = build_call<MX>(c.up, q.up, mm.up, mt);
  if (e != cudaSuccess) return e;
  if ((e = build_call<MX>(c.down, q.down, mm.down, mt)) != cudaSuccess) return e;
  // both phases share the CTA's stage ring, staging boxes and accumulator sequence: MXFP8
  // takes the down GEMM's setting for both
  if (MX) {
    q.up.stages = q.down.stages;
    q.up.nbuf = q.down.nbuf;
  }
  if (q.up.stages != q.down.stages || q.up.stage_bytes != q.down.stage_bytes ||
      q.up.nbuf != q.down.nbuf || q.up.nacc != q.down.nacc || q.up.acc_cols != q.down.acc_cols)
    return cudaErrorInvalidValue;
  q.M = c.M;
  q.S = c.S;
  q.P_slot = c.P_slot;
  q.Tm = c.Tm;
  q.T = c.T;
  q.H = c.up.H;
  q.I = c.up.I;
  q.E = c.up.groups;
  q.k = c.up.k;
  q.mt_m_max = c.mt_m_max;
  q.has_shared = c.Os != nullptr;
  q.mstart = c.mstart;
  q.mcount = c.mcount;
  q.mpoff = c.mpoff;
  q.mtile_expert = c.mtile_expert;
  q.mtiles = c.mtiles;
  q.mrow0 = c.mrow0;
  q.table = c.up.table;
  q.topk_idx = c.topk_idx;
  q.inv = c.inv;
  q.gates = c.up.gates;
  q.x = static_cast<const uint8_t*>(c.x);
  q.ring = static_cast<uint8_t*>(c.ring);
  q.ring_sf = static_cast<uint8_t*>(c.ring_sf);
  q.O = c.O;
  q.Os = c.Os;
  q.y = c.y;
  q.out_bf16 = c.down.out_bf16 ? 1 : 0;
  q.cnt = c.cnt;
  q.status = c.up.status;
  q.trace = c.trace;
  q.withhold = c.withhold;
  int per_sm = 0;
  if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fwd_mega_kernel<MX>, NUM_THREADS,
                                                         C::SMEM_BYTES)) != cudaSuccess)
    return e;
  if (per_sm < 1) return cudaErrorInvalidConfiguration;
  const int grid = num_sms;   // one CTA per SM, all resident (cooperative launch)
  // gather SMs: they move every dispatched row and, with several macrobatches, combine
  // (their copies are bound by memory latency: with several macrobatches, whose gathers
  // must keep ahead of the GEMMs, one SM in five gathers and combines)
  q.n_comm = c.n_comm > 0 ? c.n_comm : (grid < 32 ? 1 : (c.M == 1 ? 8 : grid / 5));
  if (grid - q.n_comm < 1) return cudaErrorInvalidConfiguration;
  void* args[] = {&mm, &q};
  return cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(fwd_mega_kernel<MX>), grid,
                                     NUM_THREADS, args, C::SMEM_BYTES, s);
}

int gemm_dh_parts(int I, bool mx) { return (!mx && I % 256 == 0) ? I / 256 : I / 128; }

cudaError_t launch_fwd_mega(const MegaCall& c, int num_sms, cudaStream_t s) {
  return c.up.mx ? launch_mega_impl<true>(c, num_sms, s) : launch_mega_impl<false>(c, num_sms, s);
}

cudaError_t launch_gemm(const GemmCall& c, int num_sms, cudaStream_t s) {
  return c.mx ? launch_impl<true>(c, num_sms, s) : launch_impl<false>(c, num_sms, s);
}

}  // namespace mok
