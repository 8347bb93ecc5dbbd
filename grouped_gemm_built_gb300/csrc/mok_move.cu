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
// Rows of the padded row space: an expert's rows from the table; after them, zeros up to the
// next multiple of 16 rows (the weight-gradient GEMMs' last MMA K step reads that far and
// multiplies these rows by zero operands, which must not meet a NaN); the rest of the
// segment is left as it is (no GEMM result that is read depends on it).
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
    } else if (r < (counts[e] + 15) / 16 * 16) {
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
// kCombineWarps warps per token. weighted: y = sum_j g_tj O[row(t,j)] (+ add[t]); otherwise
// the plain sum (the reverse combine of the backward), plus the router path
// sum_j dl_tj Wr[:, e_j] when dl is given. Sums in fp32, slot order, then add, then the
// router path. Rows are fp32 (4 per 16-byte vector) or, with BF16, bf16 (8 per vector) with
// the result rounded to bf16 once.
constexpr int kCombineWarps = 4;   // warps per token: more loads in flight per SM

template <bool BF16>
struct RowVec {
  static constexpr int N = BF16 ? 8 : 4;   // values per 16-byte vector
  __device__ static void load(const uint4* p, float* f) { unpack(__ldg(p), f); }
  __device__ static void unpack(const uint4 w, float* f) {
    if (BF16) {
      const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&w);
#pragma unroll
      for (int z = 0; z < 4; ++z) {
        const float2 t2 = __bfloat1622float2(h[z]);
        f[2 * z] = t2.x;
        f[2 * z + 1] = t2.y;
      }
    } else {
      f[0] = __uint_as_float(w.x);
      f[1] = __uint_as_float(w.y);
      f[2] = __uint_as_float(w.z);
      f[3] = __uint_as_float(w.w);
    }
  }
  __device__ static void store(uint4* p, const float* f) {
    uint4 w;
    if (BF16) {
      __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&w);
#pragma unroll
      for (int z = 0; z < 4; ++z) h[z] = __floats2bfloat162_rn(f[2 * z], f[2 * z + 1]);
    } else {
      w = make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]),
                     __float_as_uint(f[3]));
    }
    *p = w;
  }
};

template <bool BF16>
__global__ void __launch_bounds__(256) combine_kernel(
    int T, int H, int E, int k, const uint4* __restrict__ O, const int32_t* __restrict__ topk_idx,
    const float* __restrict__ gates, const int32_t* __restrict__ inv,
    const int32_t* __restrict__ offsets, const int32_t* __restrict__ poff,
    const uint4* __restrict__ add, const float* __restrict__ dl, const float* __restrict__ WrT,
    int weighted, uint4* __restrict__ y) {
  using V = RowVec<BF16>;
  constexpr int N = V::N;
  const int lane = threadIdx.x & 31;
  // kCombineWarps warps per token, each taking every kCombineWarps-th block of 32 vectors
  const int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int t = gw / kCombineWarps, part = gw % kCombineWarps;
  if (t >= T) return;
  const int nvec = H / N;
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
    // every load of this vector first (the k rows and the added row are independent),
    // then the sums in slot order
    uint4 w[kMaxK], wa = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
    for (int j = 0; j < kMaxK; ++j)
      if (j < k) w[j] = __ldg(O + (size_t)rows[j] * nvec + i);
    if (add) wa = __ldg(add + (size_t)t * nvec + i);
    float acc[N];
#pragma unroll
    for (int z = 0; z < N; ++z) acc[z] = 0.f;
#pragma unroll
    for (int j = 0; j < kMaxK; ++j) {
      if (j < k) {
        float f[N];
        V::unpack(w[j], f);
        if (weighted) {
#pragma unroll
          for (int z = 0; z < N; ++z) acc[z] = fmaf(g[j], f[z], acc[z]);
        } else {
#pragma unroll
          for (int z = 0; z < N; ++z) acc[z] += f[z];
        }
      }
    }
    if (add) {
      float f[N];
      V::unpack(wa, f);
#pragma unroll
      for (int z = 0; z < N; ++z) acc[z] += f[z];
    }
    if (dl) {   // the router weights' columns, four slots' loads at a time, in slot order
#pragma unroll
      for (int j0 = 0; j0 < kMaxK; j0 += 4) {
        float4 wv[4][N / 4];
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
          if (j0 + jj < k) {
            const float4* w =
                reinterpret_cast<const float4*>(WrT + (size_t)ex[j0 + jj] * H + (size_t)i * N);
#pragma unroll
            for (int q = 0; q < N / 4; ++q) wv[jj][q] = __ldg(w + q);
          }
        }
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
          const int j = j0 + jj;
          if (j < k) {
#pragma unroll
            for (int q = 0; q < N / 4; ++q) {
              acc[4 * q] = fmaf(dls[j], wv[jj][q].x, acc[4 * q]);
              acc[4 * q + 1] = fmaf(dls[j], wv[jj][q].y, acc[4 * q + 1]);
              acc[4 * q + 2] = fmaf(dls[j], wv[jj][q].z, acc[4 * q + 2]);
              acc[4 * q + 3] = fmaf(dls[j], wv[jj][q].w, acc[4 * q + 3]);
            }
          }
        }
      }
    }
    V::store(y + (size_t)t * nvec + i, acc);
  }
}

namespace {
cudaError_t launch_combine_impl(const Dims& d, const void* rows, const mok_sched& sc,
                                const AuxPtrs& a, const void* add, const float* dl,
                                const float* WrT, bool weighted, bool bf16, void* out,
                                cudaStream_t s) {
  int blocks = (d.T * kCombineWarps * 32 + 255) / 256;
  auto kern = bf16 ? combine_kernel<true> : combine_kernel<false>;
  kern<<<blocks, 256, 0, s>>>(d.T, d.H, d.E, d.k, static_cast<const uint4*>(rows), sc.topk_idx,
                              sc.gates, sc.inv, sc.offsets, a.poff,
                              static_cast<const uint4*>(add), dl, dl ? WrT : nullptr,
                              weighted ? 1 : 0, static_cast<uint4*>(out));
  return cudaGetLastError();
}
}  // namespace

cudaError_t launch_combine(const Dims& d, const void* O, const mok_sched& sc, const AuxPtrs& a,
                           const void* add, bool weighted, bool bf16, void* y, cudaStream_t s) {
  return launch_combine_impl(d, O, sc, a, add, nullptr, nullptr, weighted, bf16, y, s);
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
                                   const float* WrT, bool bf16, void* dX, cudaStream_t s) {
  return launch_combine_impl(d, dXg, sc, a, dXs, dl, WrT, false, bf16, dX, s);
}

// ---------------------------------------------------------------- U, V row map
__global__ void uv_rowmap_kernel(int E, int Tm, int P_max, const int32_t* __restrict__ table,
                                 const int32_t* __restrict__ counts,
                                 const int32_t* __restrict__ offsets,
                                 const int32_t* __restrict__ poff,
                                 const int32_t* __restrict__ tile_expert,
                                 const int32_t* __restrict__ num_mtiles,
                                 const int32_t* __restrict__ mstart,
                                 const int32_t* __restrict__ mpoff,
                                 const int32_t* __restrict__ mrow0, int32_t* __restrict__ map) {
  const int P = min(*num_mtiles, P_max / kRowPad) * kRowPad;
  for (int p = blockIdx.x * blockDim.x + threadIdx.x; p < P_max; p += gridDim.x * blockDim.x) {
    int out = -1;
    if (p < P) {
      const int e = clamp_expert(tile_expert[p / kRowPad], E);
      const int rl = p - poff[e];
      if (rl >= 0 && rl < counts[e]) {
        const int tr = offsets[e] + rl;
        const int m = table[2 * (size_t)tr] / Tm;
        out = mrow0[m] + mpoff[(size_t)m * (E + 1) + e] + (tr - mstart[(size_t)m * E + e]);
      }
    }
    map[p] = out;
  }
}

cudaError_t launch_uv_rowmap(const Dims& d, const mok_sched& sc, const AuxPtrs& a, int32_t* map,
                             cudaStream_t s) {
  const int blocks = (d.P_max + 255) / 256;
  uv_rowmap_kernel<<<blocks, 256, 0, s>>>(d.E, d.Tm, d.P_max, sc.table, sc.counts, sc.offsets,
                                          a.poff, a.tile_expert, a.num_mtiles, a.mstart, a.mpoff,
                                          a.mrow0, map);
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

// dWr[h][e] = sum over expert e's table rows r of x[t_r][h] * dl[t_r][j_r], in two fixed-order
// passes. Pass 1, grid (chunk items, H/256): a CTA takes one chunk of kDwrChunk rows of one
// expert and 256 columns h; warp w sums the chunk's rows w, w+8, w+16, ... (ascending), each
// lane 8 consecutive h from one 16-byte load per row; the eight warp sums are added in warp
// order into part[q][h]. Pass 2, grid (E, H/256): dWr[h][e] = the expert's chunk sums in
// chunk order. A busy expert (the biased experts take most tokens) spreads over many CTAs.
constexpr int kDwrWarps = 8;
__global__ void __launch_bounds__(kDwrWarps * 32) router_dwr_part_kernel(
    int H, int k, const uint4* __restrict__ x, const int32_t* __restrict__ table,
    const int32_t* __restrict__ counts, const int32_t* __restrict__ offsets,
    const int32_t* __restrict__ dwr_q0, const int32_t* __restrict__ dwr_item_e, int E,
    const float* __restrict__ dl, float* __restrict__ part) {
  __shared__ int s_tok[kDwrChunk];
  __shared__ float s_w[kDwrChunk];
  __shared__ float s_red[kDwrWarps][256];
  const int q = blockIdx.x;
  if (q >= dwr_q0[E]) return;
  const int e = dwr_item_e[q];
  const int c0 = (q - dwr_q0[e]) * kDwrChunk;
  const int m = min(kDwrChunk, counts[e] - c0);
  const int r0 = offsets[e] + c0;
  for (int i = threadIdx.x; i < m; i += blockDim.x) {
    const int t = table[2 * (size_t)(r0 + i)], j = table[2 * (size_t)(r0 + i) + 1];
    s_tok[i] = t;
    s_w[i] = dl[(size_t)t * k + j];
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h0 = blockIdx.y * 256 + lane * 8;   // this lane's 8 columns
  const bool on = h0 < H;
  const int hv = H / 8;                         // 16-byte vectors per row of x
  float acc[8];
#pragma unroll
  for (int z = 0; z < 8; ++z) acc[z] = 0.f;
  if (on) {
#pragma unroll 4
    for (int i = warp; i < m; i += kDwrWarps) {
      const uint4 w = __ldg(x + (size_t)s_tok[i] * hv + h0 / 8);
      const float wt = s_w[i];
      const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&w);
#pragma unroll
      for (int z = 0; z < 4; ++z) {
        const float2 f = __bfloat1622float2(b[z]);
        acc[2 * z] = fmaf(f.x, wt, acc[2 * z]);
        acc[2 * z + 1] = fmaf(f.y, wt, acc[2 * z + 1]);
      }
    }
  }
#pragma unroll
  for (int z = 0; z < 8; ++z) s_red[warp][lane * 8 + z] = acc[z];
  __syncthreads();
  const int h = blockIdx.y * 256 + threadIdx.x;
  if (h < H) {
    float v = 0.f;
#pragma unroll
    for (int w2 = 0; w2 < kDwrWarps; ++w2) v += s_red[w2][threadIdx.x];
    part[(size_t)q * H + h] = v;
  }
}

__global__ void __launch_bounds__(256) router_dwr_sum_kernel(int H, int E,
                                                             const int32_t* __restrict__ dwr_q0,
                                                             const float* __restrict__ part,
                                                             float* __restrict__ dWr) {
  const int e = blockIdx.x;
  const int h = blockIdx.y * 256 + threadIdx.x;
  if (h >= H) return;
  const int q0 = dwr_q0[e], q1 = dwr_q0[e + 1];
  float v = 0.f;
  for (int q = q0; q < q1; ++q) v += part[(size_t)q * H + h];
  dWr[(size_t)h * E + e] = v;
}

cudaError_t launch_router_dwr(const Dims& d, const void* x, const mok_sched& sc, const AuxPtrs& a,
                              float* part, const float* dl, float* dWr, cudaStream_t s) {
  if (d.H % 8 != 0) return cudaErrorInvalidValue;
  dim3 g1(dwr_items_max(d), (d.H + 255) / 256);
  router_dwr_part_kernel<<<g1, kDwrWarps * 32, 0, s>>>(
      d.H, d.k, static_cast<const uint4*>(x), sc.table, sc.counts, sc.offsets, a.dwr_q0,
      a.dwr_item_e, d.E, dl, part);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  dim3 g2(d.E, (d.H + 255) / 256);
  router_dwr_sum_kernel<<<g2, 256, 0, s>>>(d.H, d.E, a.dwr_q0, part, dWr);
  return cudaGetLastError();
}

}  // namespace mok
