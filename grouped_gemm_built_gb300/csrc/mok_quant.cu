// MXFP8 quantisation (E4M3 elements, one UE8M0 scale per 32 elements along a GEMM's
// contraction axis), fused into the producers that need it.
//
// "Determinismus und MXFP8-Unterstuetzung" (sebask.de MoK article): MXFP8 support lives
// in the kernel, with no separate conversion kernel for activations. The block rule is
// the OCP Microscaling one: scale 2^(floor(log2 amax) - 8) stored as the biased byte,
// elements v / scale rounded to nearest-even E4M3 with saturation, all-zero block ->
// scale byte 127.
//
// Scale "atoms". The block-scaled tcgen05.mma reads its scales from TMEM; a 512-byte atom
// in shared memory covers 128 rows (M or N index m) x 4 blocks of 32 along K (128 K
// elements), with byte (m, b) at 16*(m%32) + 4*(m/32) + b. tcgen05.cp (32x128b, warpx4)
// moves one atom into 4 TMEM columns. Producers write scales straight into this layout so
// that a GEMM stage fetches its scales with one bulk copy.
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include "mok_internal.h"
#include "mok_mx.cuh"

namespace mok {


// ---------------------------------------------------------------- blocks along columns
// src [rows][cols] bf16 (batch z at src + z*batch_elems), K = the column axis.
// Each warp quantises one row, 8 elements per lane per step (4 lanes = one block).
// Atom (kc = col/128, mc = row/128) lives at atoms + z*atom_batch + (kc*s_kc + mc*s_mc)*512.
__global__ void __launch_bounds__(256) mx_quant_cols_kernel(
    const __nv_bfloat16* __restrict__ src, int rows, int cols, size_t batch_elems,
    uint8_t* __restrict__ dst, uint8_t* __restrict__ atoms, size_t atom_batch, int s_kc,
    int s_mc) {
  const int lane = threadIdx.x & 31;
  const int z = blockIdx.y;
  const int row = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (row >= rows) return;
  const uint4* s = reinterpret_cast<const uint4*>(src + z * batch_elems + (size_t)row * cols);
  uint2* d = reinterpret_cast<uint2*>(dst + z * batch_elems + (size_t)row * cols);
  uint8_t* at = atoms + z * atom_batch;
  for (int v = lane; v < cols / 8; v += 32) {
    uint4 w = __ldg(s + v);
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&w);
    float f[8];
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float2 t = __bfloat1622float2(h[i]);
      f[2 * i] = t.x;
      f[2 * i + 1] = t.y;
      amax = fmaxf(amax, fmaxf(fabsf(t.x), fabsf(t.y)));
    }
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    const uint32_t sb = mx_scale_byte(amax);
    const float inv = mx_inv_scale(sb);
    uint2 q;
    q.x = (uint32_t)f32x2_to_e4m3x2(f[0] * inv, f[1] * inv) |
          ((uint32_t)f32x2_to_e4m3x2(f[2] * inv, f[3] * inv) << 16);
    q.y = (uint32_t)f32x2_to_e4m3x2(f[4] * inv, f[5] * inv) |
          ((uint32_t)f32x2_to_e4m3x2(f[6] * inv, f[7] * inv) << 16);
    d[v] = q;
    if ((lane & 3) == 0) {
      const int k = v * 8;
      at[(size_t)((k >> 7) * s_kc + (row >> 7) * s_mc) * 512 + atom_byte(row, k)] = (uint8_t)sb;
    }
  }
}

// ---------------------------------------------------------------- blocks along rows
// src [rows][cols] bf16, K = the row axis (rows multiple of 32). Thread per column, 32
// rows per block; atom (kc = row/128, mc = col/128).
__global__ void __launch_bounds__(256) mx_quant_rows_kernel(
    const __nv_bfloat16* __restrict__ src, int rows, int cols, size_t batch_elems,
    uint8_t* __restrict__ dst, uint8_t* __restrict__ atoms, size_t atom_batch, int s_kc,
    int s_mc) {
  const int z = blockIdx.z;
  const int col = blockIdx.x * blockDim.x + threadIdx.x;
  const int r0 = blockIdx.y * 32;
  if (col >= cols || r0 >= rows) return;
  const __nv_bfloat16* s = src + z * batch_elems + (size_t)r0 * cols + col;
  uint8_t* d = dst + z * batch_elems + (size_t)r0 * cols + col;
  float f[32];
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    f[i] = __bfloat162float(s[(size_t)i * cols]);
    amax = fmaxf(amax, fabsf(f[i]));
  }
  const uint32_t sb = mx_scale_byte(amax);
  const float inv = mx_inv_scale(sb);
#pragma unroll
  for (int i = 0; i < 32; i += 2) {
    uint16_t q = f32x2_to_e4m3x2(f[i] * inv, f[i + 1] * inv);
    d[(size_t)i * cols] = (uint8_t)(q & 0xFF);
    d[(size_t)(i + 1) * cols] = (uint8_t)(q >> 8);
  }
  atoms[z * atom_batch + (size_t)((r0 >> 7) * s_kc + (col >> 7) * s_mc) * 512 +
        atom_byte(col, r0)] = (uint8_t)sb;
}

cudaError_t launch_mx_quant(const void* src, int rows, int cols, int batch, bool k_along_cols,
                            void* dst, void* atoms, int s_kc, int s_mc, cudaStream_t s) {
  const size_t be = (size_t)rows * cols;
  const size_t ab = (size_t)(rows / 128) * (cols / 128) * 512;
  if (k_along_cols) {
    dim3 grid((rows * 32 + 255) / 256, batch);
    mx_quant_cols_kernel<<<grid, 256, 0, s>>>(static_cast<const __nv_bfloat16*>(src), rows, cols,
                                             be, static_cast<uint8_t*>(dst),
                                             static_cast<uint8_t*>(atoms), ab, s_kc, s_mc);
  } else {
    dim3 grid((cols + 255) / 256, rows / 32, batch);
    mx_quant_rows_kernel<<<grid, 256, 0, s>>>(static_cast<const __nv_bfloat16*>(src), rows, cols,
                                             be, static_cast<uint8_t*>(dst),
                                             static_cast<uint8_t*>(atoms), ab, s_kc, s_mc);
  }
  return cudaGetLastError();
}

// ---------------------------------------------------------------- dispatch + quantise
// The forward dispatch in MXFP8 mode: pull x rows through the table and quantise them
// along H on the way (zero padding rows get scale byte 127). Atoms [P/128][H/128].
__global__ void __launch_bounds__(256) gather_quant_kernel(
    int H, int E, const uint4* __restrict__ src, const int32_t* __restrict__ table,
    const int32_t* __restrict__ counts, const int32_t* __restrict__ offsets,
    const int32_t* __restrict__ poff, const int32_t* __restrict__ tile_expert,
    const int32_t* __restrict__ num_mtiles, int P_max, uint2* __restrict__ dst,
    uint8_t* __restrict__ atoms) {
  const int lane = threadIdx.x & 31;
  const int nvec = H / 8;
  const int P = min(*num_mtiles, P_max / kRowPad) * kRowPad;
  const int nwarps = (gridDim.x * blockDim.x) >> 5;
  const int kcs = H / 128;
  for (int p = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; p < P; p += nwarps) {
    int e = tile_expert[p / kRowPad];
    e = (e < 0 || e >= E) ? 0 : e;
    const int r = p - poff[e];
    const uint4* s = nullptr;
    if (r < counts[e]) s = src + (size_t)table[2 * (size_t)(offsets[e] + r)] * nvec;
    uint2* d = dst + (size_t)p * nvec;
    uint8_t* at = atoms + (size_t)(p >> 7) * kcs * 512;
    for (int v = lane; v < nvec; v += 32) {
      float f[8];
      float amax = 0.f;
      if (s) {
        uint4 w = __ldg(s + v);
        const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&w);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          float2 t = __bfloat1622float2(h[i]);
          f[2 * i] = t.x;
          f[2 * i + 1] = t.y;
          amax = fmaxf(amax, fmaxf(fabsf(t.x), fabsf(t.y)));
        }
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) f[i] = 0.f;
      }
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
      const uint32_t sb = mx_scale_byte(amax);
      const float inv = mx_inv_scale(sb);
      uint2 q;
      q.x = (uint32_t)f32x2_to_e4m3x2(f[0] * inv, f[1] * inv) |
            ((uint32_t)f32x2_to_e4m3x2(f[2] * inv, f[3] * inv) << 16);
      q.y = (uint32_t)f32x2_to_e4m3x2(f[4] * inv, f[5] * inv) |
            ((uint32_t)f32x2_to_e4m3x2(f[6] * inv, f[7] * inv) << 16);
      d[v] = q;
      if ((lane & 3) == 0) {
        const int k = v * 8;
        at[(size_t)(k >> 7) * 512 + atom_byte(p, k)] = (uint8_t)sb;
      }
    }
  }
}

cudaError_t launch_gather_quant(const Dims& d, const void* src, const mok_sched& sc,
                                const AuxPtrs& a, void* dst, void* atoms, int num_sms,
                                cudaStream_t s) {
  gather_quant_kernel<<<num_sms * 8, 256, 0, s>>>(
      d.H, d.E, static_cast<const uint4*>(src), sc.table, sc.counts, sc.offsets, a.poff,
      a.tile_expert, a.num_mtiles, d.P_max, static_cast<uint2*>(dst),
      static_cast<uint8_t*>(atoms));
  return cudaGetLastError();
}

}  // namespace mok

namespace mok {

// ---------------------------------------------------------------- dispatch + row blocks
__device__ __forceinline__ float2 bf16x2_to_float2(uint32_t w) {
  return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w));
}

// Pull rows by the table and quantise them in blocks of 32 consecutive padded rows (the
// contraction axis of the dW GEMMs). Blocks start at each expert segment's first row,
// since segments start on 128-row boundaries. A CTA takes 512 columns (two per thread) of
// every gridDim.y-th 32-row block; atoms [P/128][H/128], m = column, b = block inside the
// 128-row tile.
__global__ void __launch_bounds__(256, 2) gather_quant_rows_kernel(
    int H, int E, const __nv_bfloat16* __restrict__ src, const int32_t* __restrict__ table,
    const int32_t* __restrict__ counts, const int32_t* __restrict__ offsets,
    const int32_t* __restrict__ poff, const int32_t* __restrict__ tile_expert,
    const int32_t* __restrict__ num_mtiles, int P_max, uint8_t* __restrict__ dst,
    uint8_t* __restrict__ atoms) {
  // source tokens of the CTA's next 8 blocks (blockIdx.y + q gridDim.y), one lookup per
  // thread, so the table's dependent loads are paid once per 8 blocks
  __shared__ int s_tok[8][32];
  const int P = min(*num_mtiles, P_max / kRowPad) * kRowPad;
  const int nblocks = P / 32;
  const int kcs = H / 128;
  // two neighbouring columns per thread (a warp loads a whole 128-byte line of each row);
  // the 32 rows stay in registers as the loaded bf16 pairs and are widened twice
  const int col = (blockIdx.x * 256 + threadIdx.x) * 2;
  for (int base = blockIdx.y; base < nblocks; base += 8 * gridDim.y) {
    __syncthreads();
    {
      const int b = base + (threadIdx.x >> 5) * gridDim.y;
      int tok = -1;
      if (b < nblocks) {
        const int p = b * 32 + (threadIdx.x & 31);
        int e = tile_expert[p / kRowPad];
        e = (e < 0 || e >= E) ? 0 : e;
        const int r = p - poff[e];
        if (r < counts[e]) tok = table[2 * (size_t)(offsets[e] + r)];
      }
      s_tok[threadIdx.x >> 5][threadIdx.x & 31] = tok;
    }
    __syncthreads();
    if (col >= H) continue;
    for (int q = 0; q < 8; ++q) {
      const int blk = base + q * gridDim.y;
      if (blk >= nblocks) break;
      const int p0 = blk * 32;
      uint32_t raw[32];
      float amax0 = 0.f, amax1 = 0.f;
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const int t = s_tok[q][i];
        raw[i] = 0u;
        if (t >= 0) raw[i] = __ldg(reinterpret_cast<const uint32_t*>(src + (size_t)t * H + col));
      }
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const float2 f = bf16x2_to_float2(raw[i]);
        amax0 = fmaxf(amax0, fabsf(f.x));
        amax1 = fmaxf(amax1, fabsf(f.y));
      }
      const uint32_t sb0 = mx_scale_byte(amax0), sb1 = mx_scale_byte(amax1);
      const float inv0 = mx_inv_scale(sb0), inv1 = mx_inv_scale(sb1);
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const float2 f = bf16x2_to_float2(raw[i]);
        *reinterpret_cast<uint16_t*>(dst + (size_t)(p0 + i) * H + col) =
            (uint16_t)f32x2_to_e4m3x2(f.x * inv0, f.y * inv1);
      }
      atoms[((size_t)(p0 >> 7) * kcs + (col >> 7)) * 512 + atom_byte(col, p0)] = (uint8_t)sb0;
      atoms[((size_t)(p0 >> 7) * kcs + ((col + 1) >> 7)) * 512 + atom_byte(col + 1, p0)] =
          (uint8_t)sb1;
    }
  }
}

cudaError_t launch_gather_quant_rows(const Dims& d, const void* src, const mok_sched& sc,
                                     const AuxPtrs& a, void* dst, void* atoms, int num_sms,
                                     cudaStream_t s) {
  dim3 grid((d.H / 2 + 255) / 256, num_sms * 4);
  gather_quant_rows_kernel<<<grid, 256, 0, s>>>(
      d.H, d.E, static_cast<const __nv_bfloat16*>(src), sc.table, sc.counts, sc.offsets, a.poff,
      a.tile_expert, a.num_mtiles, d.P_max, static_cast<uint8_t*>(dst),
      static_cast<uint8_t*>(atoms));
  return cudaGetLastError();
}

}  // namespace mok
