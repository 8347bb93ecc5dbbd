// Row movement driven by the schedule table: dispatch (pull gather into expert order),
// combine, reverse-dispatch, reverse-combine; plus the router backward.
//
// "Push oder Pull?" (sebask.de MoK article): dispatch pulls rows by the table; combine
// keeps token order; the one plan serves all four exchange steps. On one GPU the four
// steps are HBM-to-HBM moves: a warp moves one 2*H-byte row with 16-byte accesses.
// Reductions over a token's k slots run in slot order j = 0..k-1 in fp32, so y and dX
// are bitwise reproducible.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "mok_internal.h"

namespace mok {

namespace {

__device__ __forceinline__ int clamp_expert(int e, int E) { return (e < 0 || e >= E) ? 0 : e; }

// padded row of slot (t, j): its table row moved from the unpadded to the padded layout
__device__ __forceinline__ int padded_row(int sl, int E, const int32_t* topk_idx,
                                          const int32_t* inv, const int32_t* offsets,
                                          const int32_t* poff) {
  int e = clamp_expert(topk_idx[sl], E);
  return inv[sl] - offsets[e] + poff[e];
}

}  // namespace

// ---------------------------------------------------------------- dispatch (pull gather)
__global__ void __launch_bounds__(256) gather_rows_kernel(
    int H, int E, const uint4* __restrict__ src, const int32_t* __restrict__ table,
    const int32_t* __restrict__ counts, const int32_t* __restrict__ offsets,
    const int32_t* __restrict__ poff, const int32_t* __restrict__ tile_expert,
    const int32_t* __restrict__ num_mtiles, int P_max, uint4* __restrict__ dst) {
  const int lane = threadIdx.x & 31;
  const int nvec = H / 8;
  const int P = min(*num_mtiles, P_max / kRowPad) * kRowPad;
  const int nwarps = (gridDim.x * blockDim.x) >> 5;
  for (int p = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; p < P; p += nwarps) {
    const int e = clamp_expert(tile_expert[p / kRowPad], E);
    const int r = p - poff[e];
    uint4* d = dst + (size_t)p * nvec;
    if (r < counts[e]) {
      const int t = table[2 * (size_t)(offsets[e] + r)];
      const uint4* s = src + (size_t)t * nvec;
#pragma unroll 4
      for (int i = lane; i < nvec; i += 32) d[i] = __ldg(s + i);
    } else {
      const uint4 z = make_uint4(0, 0, 0, 0);
      for (int i = lane; i < nvec; i += 32) d[i] = z;
    }
  }
}

cudaError_t launch_gather_rows(const Dims& d, const void* src, const mok_sched& sc,
                               const AuxPtrs& a, void* dst, int num_sms, cudaStream_t s) {
  int blocks = num_sms * 8;
  gather_rows_kernel<<<blocks, 256, 0, s>>>(d.H, d.E, static_cast<const uint4*>(src), sc.table,
                                            sc.counts, sc.offsets, a.poff, a.tile_expert,
                                            a.num_mtiles, d.P_max, static_cast<uint4*>(dst));
  return cudaGetLastError();
}

// ---------------------------------------------------------------- combine
// One warp per token, fp32 rows. weighted: y = sum_j g_tj O[row(t,j)] (+ add[t]);
// otherwise the plain sum (the reverse combine of the backward), plus the router path
// sum_j dl_tj Wr[:, e_j] when dl is given.
constexpr int kCombineWarps = 4;   // warps per token: more loads in flight per SM

__global__ void __launch_bounds__(256) combine_kernel(
    int T, int H, int E, int k, const float4* __restrict__ O, const int32_t* __restrict__ topk_idx,
    const float* __restrict__ gates, const int32_t* __restrict__ inv,
    const int32_t* __restrict__ offsets, const int32_t* __restrict__ poff,
    const float4* __restrict__ add, const float* __restrict__ dl, const float* __restrict__ WrT,
    int weighted, float4* __restrict__ y) {
  const int lane = threadIdx.x & 31;
  // kCombineWarps warps per token, each taking every kCombineWarps-th block of 32 vectors
  const int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int t = gw / kCombineWarps, part = gw % kCombineWarps;
  if (t >= T) return;
  const int nvec = H / 4;
  int my_row = 0, my_e = 0;
  float my_g = 0.f, my_dl = 0.f;
  if (lane < k) {
    const int sl = t * k + lane;
    my_e = clamp_expert(topk_idx[sl], E);
    my_row = padded_row(sl, E, topk_idx, inv, offsets, poff);
    my_g = weighted ? gates[sl] : 1.f;
    my_dl = dl ? dl[sl] : 0.f;
  }
  int rows[kMaxK], ex[kMaxK];
  float g[kMaxK], dls[kMaxK];
#pragma unroll
  for (int j = 0; j < kMaxK; ++j) {
    rows[j] = __shfl_sync(0xffffffffu, my_row, j);
    ex[j] = __shfl_sync(0xffffffffu, my_e, j);
    g[j] = __shfl_sync(0xffffffffu, my_g, j);
    dls[j] = __shfl_sync(0xffffffffu, my_dl, j);
  }
  for (int i = part * 32 + lane; i < nvec; i += 32 * kCombineWarps) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int j = 0; j < kMaxK; ++j) {
      if (j < k) {
        const float4 f = __ldg(O + (size_t)rows[j] * nvec + i);
        if (weighted) {
          acc.x = fmaf(g[j], f.x, acc.x);
          acc.y = fmaf(g[j], f.y, acc.y);
          acc.z = fmaf(g[j], f.z, acc.z);
          acc.w = fmaf(g[j], f.w, acc.w);
        } else {
          acc.x += f.x;
          acc.y += f.y;
          acc.z += f.z;
          acc.w += f.w;
        }
      }
    }
    if (add) {
      const float4 f = __ldg(add + (size_t)t * nvec + i);
      acc.x += f.x;
      acc.y += f.y;
      acc.z += f.z;
      acc.w += f.w;
    }
    if (dl) {
#pragma unroll
      for (int j = 0; j < kMaxK; ++j) {
        if (j < k) {
          const float4 w = __ldg(reinterpret_cast<const float4*>(WrT + (size_t)ex[j] * H) + i);
          acc.x = fmaf(dls[j], w.x, acc.x);
          acc.y = fmaf(dls[j], w.y, acc.y);
          acc.z = fmaf(dls[j], w.z, acc.z);
          acc.w = fmaf(dls[j], w.w, acc.w);
        }
      }
    }
    y[(size_t)t * nvec + i] = acc;
  }
}

cudaError_t launch_combine(const Dims& d, const void* O, const mok_sched& sc, const AuxPtrs& a,
                           const void* add, bool weighted, void* y, cudaStream_t s) {
  int blocks = (d.T * kCombineWarps * 32 + 255) / 256;
  combine_kernel<<<blocks, 256, 0, s>>>(d.T, d.H, d.E, d.k, static_cast<const float4*>(O),
                                        sc.topk_idx, sc.gates, sc.inv, sc.offsets, a.poff,
                                        static_cast<const float4*>(add), nullptr, nullptr,
                                        weighted ? 1 : 0, static_cast<float4*>(y));
  return cudaGetLastError();
}

// ---------------------------------------------------------------- reverse combine
__global__ void transpose_f32_kernel(int rows, int cols, const float* __restrict__ in,
                                     float* __restrict__ out) {
  __shared__ float tile[32][33];
  int c = blockIdx.x * 32 + threadIdx.x, r = blockIdx.y * 32 + threadIdx.y;
  for (int i = 0; i < 32; i += 8)
    if (r + i < rows && c < cols) tile[threadIdx.y + i][threadIdx.x] = in[(size_t)(r + i) * cols + c];
  __syncthreads();
  c = blockIdx.y * 32 + threadIdx.x;
  r = blockIdx.x * 32 + threadIdx.y;
  for (int i = 0; i < 32; i += 8)
    if (r + i < cols && c < rows) out[(size_t)(r + i) * rows + c] = tile[threadIdx.x][threadIdx.y + i];
}

cudaError_t launch_transpose_wr(const Dims& d, const float* Wr, float* WrT, cudaStream_t s) {
  dim3 grid((d.E + 31) / 32, (d.H + 31) / 32), block(32, 8);
  transpose_f32_kernel<<<grid, block, 0, s>>>(d.H, d.E, Wr, WrT);
  return cudaGetLastError();
}

cudaError_t launch_reverse_combine(const Dims& d, const void* dXg, const mok_sched& sc,
                                   const AuxPtrs& a, const void* dXs, const float* dl,
                                   const float* WrT, void* dX, cudaStream_t s) {
  int blocks = (d.T * kCombineWarps * 32 + 255) / 256;
  combine_kernel<<<blocks, 256, 0, s>>>(d.T, d.H, d.E, d.k, static_cast<const float4*>(dXg),
                                        sc.topk_idx, sc.gates, sc.inv, sc.offsets, a.poff,
                                        static_cast<const float4*>(dXs), dl, dl ? WrT : nullptr,
                                        0, static_cast<float4*>(dX));
  return cudaGetLastError();
}

// ---------------------------------------------------------------- router backward
// dg_tj = sum over the kBwdDH partial sums (fixed order); with the set S fixed,
// dl_j = g_j (dg_j - sum_i g_i dg_i) for the k chosen experts.
__global__ void router_grad_kernel(int T, int E, int k, const float* __restrict__ dgp, int n_parts,
                                   const int32_t* __restrict__ topk_idx,
                                   const float* __restrict__ gates, const int32_t* __restrict__ inv,
                                   const int32_t* __restrict__ offsets,
                                   const int32_t* __restrict__ poff, float* __restrict__ dgates,
                                   float* __restrict__ dl) {
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= T) return;
  float dg[kMaxK], g[kMaxK];
  float s = 0.f;
  for (int j = 0; j < k; ++j) {
    const int sl = t * k + j;
    const int p = padded_row(sl, E, topk_idx, inv, offsets, poff);
    float v = 0.f;
    for (int q = 0; q < n_parts; ++q) v += dgp[(size_t)p * n_parts + q];
    dg[j] = v;
    g[j] = gates[sl];
    dgates[sl] = v;
    s = fmaf(g[j], v, s);
  }
  if (dl)
    for (int j = 0; j < k; ++j) dl[(size_t)t * k + j] = g[j] * (dg[j] - s);
}

cudaError_t launch_router_grad(const Dims& d, const float* dgp, int n_parts, const mok_sched& sc,
                               const AuxPtrs& a, float* dgates, float* dl, cudaStream_t s) {
  router_grad_kernel<<<(d.T + 127) / 128, 128, 0, s>>>(d.T, d.E, d.k, dgp, n_parts, sc.topk_idx,
                                                       sc.gates, sc.inv, sc.offsets, a.poff,
                                                       dgates, dl);
  return cudaGetLastError();
}

// dWr[h][e] = sum over expert e's table rows r (ascending) of x[t_r][h] * dl[t_r][j_r].
// Grid (E, H/256); each thread owns one h, so the row loop is one fixed-order fp32 sum.
__global__ void __launch_bounds__(256) router_dwr_kernel(int H, int E, int k,
                                                         const __nv_bfloat16* __restrict__ x,
                                                         const int32_t* __restrict__ table,
                                                         const int32_t* __restrict__ counts,
                                                         const int32_t* __restrict__ offsets,
                                                         const float* __restrict__ dl,
                                                         float* __restrict__ dWr) {
  const int e = blockIdx.x;
  const int h = blockIdx.y * 256 + threadIdx.x;
  __shared__ int s_tok[256];
  __shared__ float s_w[256];
  const int n = counts[e], r0 = offsets[e];
  float acc = 0.f;
  for (int c = 0; c < n; c += 256) {
    __syncthreads();
    if (c + (int)threadIdx.x < n) {
      const int r = r0 + c + threadIdx.x;
      const int t = table[2 * (size_t)r], j = table[2 * (size_t)r + 1];
      s_tok[threadIdx.x] = t;
      s_w[threadIdx.x] = dl[(size_t)t * k + j];
    }
    __syncthreads();
    const int m = min(256, n - c);
    if (h < H) {
#pragma unroll 8
      for (int i = 0; i < m; ++i)
        acc = fmaf(__bfloat162float(x[(size_t)s_tok[i] * H + h]), s_w[i], acc);
    }
  }
  if (h < H) dWr[(size_t)h * E + e] = acc;
}

cudaError_t launch_router_dwr(const Dims& d, const void* x, const mok_sched& sc, const AuxPtrs& a,
                              const float* dl, float* dWr, cudaStream_t s) {
  (void)a;
  dim3 grid(d.E, (d.H + 255) / 256);
  router_dwr_kernel<<<grid, 256, 0, s>>>(d.H, d.E, d.k, static_cast<const __nv_bfloat16*>(x),
                                         sc.table, sc.counts, sc.offsets, dl, dWr);
  return cudaGetLastError();
}

}  // namespace mok
