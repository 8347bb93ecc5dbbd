// Routing and the no-sort schedule table.
//
// "Das Scheduling" (sebask.de MoK article): a pull schedule is a list of source indices
// whose order follows from the routing itself, built entirely on the GPU without a sort;
// "Escolha da direcao de comunicacao" (stamatios.com): the table is built once and reused
// by forward dispatch/combine and backward reverse-dispatch/reverse-combine.
//
// Construction (deterministic, no sort, no atomics):
//   1. router logits, softmax top-k and renormalised gates per token;
//   2. per block of 32 tokens, one warp walks the block's slots in ascending (t, j) and
//      gives each slot its rank among the block's slots of the same expert
//      (__match_any_sync + popc), producing a per-block expert histogram;
//   3. one CTA scans the histograms over blocks (per expert) and over experts (warp-scan)
//      into counts, offsets and 128-row padded offsets, and maps each 128-row tile of the
//      padded row space to its expert;
//   4. every slot lands at offsets[e] + (rows of e in earlier blocks) + its block rank.
#include <algorithm>

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "mok_internal.h"

namespace mok {

// ---------------------------------------------------------------- 1a. logits on tensor cores
// The logits x Wr are fp32 sums of bf16 x fp32 products. Wr splits exactly into three
// bf16 matrices (hi = bf16(w), mid = bf16(w - hi), lo = bf16(w - hi - mid): 8 + 8 + 8
// significant bits hold fp32's 24), so x Wr = x hi + x mid + x lo with every product exact
// in fp32; the grouped-GEMM kernel's router mode sums them on the tensor cores with fp32
// accumulation and adds the bias in its epilogue.
__global__ void __launch_bounds__(256) split_wr_kernel(int H, int E, int ld,
                                                       const float* __restrict__ Wr,
                                                       __nv_bfloat16* __restrict__ out) {
  const size_t n = (size_t)H * ld;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n;
       i += (size_t)gridDim.x * blockDim.x) {
    const int h = (int)(i / ld), e = (int)(i % ld);
    const float w = e < E ? Wr[(size_t)h * E + e] : 0.f;
    const __nv_bfloat16 hi = __float2bfloat16_rn(w);
    const float r1 = w - __bfloat162float(hi);
    const __nv_bfloat16 mid = __float2bfloat16_rn(r1);
    const float r2 = r1 - __bfloat162float(mid);
    out[i] = hi;
    out[n + i] = mid;
    out[2 * n + i] = __float2bfloat16_rn(r2);
  }
}

cudaError_t launch_split_wr(const Dims& d, const float* Wr, int ld, void* out, cudaStream_t s) {
  const size_t n = (size_t)d.H * ld;
  const int blocks = (int)std::min<size_t>((n + 255) / 256, 4096);
  split_wr_kernel<<<blocks, 256, 0, s>>>(d.H, d.E, ld, Wr, static_cast<__nv_bfloat16*>(out));
  return cudaGetLastError();
}

// ---------------------------------------------------------------- 1b+2. top-k and ranks
// One CTA per block of 32 tokens (8 warps, 4 tokens each). logits == nullptr: topk_idx is
// an input (expert ids are range-checked; a bad id is flagged and replaced by 0 so that
// every later index stays in bounds).
__global__ void __launch_bounds__(256) topk_rank_kernel(int T, int E, int k,
                                                        const float* __restrict__ logits,
                                                        int32_t* __restrict__ topk_idx,
                                                        float* __restrict__ gates,
                                                        int32_t* __restrict__ hist,
                                                        int32_t* __restrict__ lrank,
                                                        uint32_t* __restrict__ status) {
  __shared__ int32_t s_idx[kTokBlock * kMaxK];
  __shared__ int32_t s_hist[kMaxE];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int blk = blockIdx.x;
  const int t0 = blk * kTokBlock;
  const int ntok = min(kTokBlock, T - t0);
  for (int e = tid; e < E; e += 256) s_hist[e] = 0;

  if (logits != nullptr) {
    for (int tt = warp; tt < ntok; tt += 8) {
      const int t = t0 + tt;
      float v[kMaxE / 32];
      const float* lg = logits + (size_t)t * E;
#pragma unroll
      for (int i = 0; i < kMaxE / 32; ++i) {
        int e = lane + 32 * i;
        v[i] = (e < E) ? lg[e] : -INFINITY;
      }
      uint32_t taken = 0;
      float top_l[kMaxK];
      int top_e[kMaxK];
      for (int j = 0; j < k; ++j) {
        // lane-local best: larger value, ties to the lower expert id
        float bv = -INFINITY;
        int be = 0x7fffffff;  // sentinel: no candidate yet
#pragma unroll
        for (int i = 0; i < kMaxE / 32; ++i) {
          int e = lane + 32 * i;
          bool ok = (e < E) && !((taken >> i) & 1u);
          if (ok && (be == 0x7fffffff || v[i] > bv || (v[i] == bv && e < be))) {
            bv = v[i];
            be = e;
          }
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
          float ov = __shfl_xor_sync(0xffffffffu, bv, off);
          int oe = __shfl_xor_sync(0xffffffffu, be, off);
          if (ov > bv || (ov == bv && oe < be)) {
            bv = ov;
            be = oe;
          }
        }
        if (be == 0x7fffffff) {  // only NaN logits left: flag, keep indices in range
          if (lane == 0) atomicOr(status, kErrBadExpert);
          be = 0;
        }
        if ((be & 31) == lane) taken |= 1u << (be >> 5);
        top_l[j] = bv;
        top_e[j] = be;
      }
      if (lane == 0) {
        // gates = softmax over the chosen logits (= renormalised softmax probabilities)
        float z = 0.f, p[kMaxK];
        for (int j = 0; j < k; ++j) {
          p[j] = expf(top_l[j] - top_l[0]);
          z += p[j];
        }
        for (int j = 0; j < k; ++j) {
          topk_idx[(size_t)t * k + j] = top_e[j];
          gates[(size_t)t * k + j] = p[j] / z;
          s_idx[tt * k + j] = top_e[j];
        }
      }
    }
  } else {
    for (int i = tid; i < ntok * k; i += 256) {
      int e = topk_idx[(size_t)t0 * k + i];
      if (e < 0 || e >= E) {
        atomicOr(status, kErrBadExpert);
        e = 0;
      }
      s_idx[i] = e;
    }
  }
  __syncthreads();

  // ranks inside the block, walking slots in ascending (t, j)
  if (warp == 0) {
    const int nslots = ntok * k;
    const unsigned lt_mask = (1u << lane) - 1u;
    for (int c = 0; c < nslots; c += 32) {
      int sl = c + lane;
      int e = (sl < nslots) ? s_idx[sl] : -1 - lane;  // idle lanes match nobody
      unsigned peers = __match_any_sync(0xffffffffu, e);
      int r = 0;
      if (sl < nslots) r = s_hist[e] + __popc(peers & lt_mask);
      __syncwarp();
      if (sl < nslots) {
        lrank[(size_t)t0 * k + sl] = r;
        if ((__ffs(peers) - 1) == lane) s_hist[e] += __popc(peers);
      }
      __syncwarp();
    }
  }
  __syncthreads();
  for (int e = tid; e < E; e += 256) hist[(size_t)blk * E + e] = s_hist[e];
}

cudaError_t launch_topk_rank(const Dims& d, const float* logits, int32_t* topk_idx, float* gates,
                             int32_t* hist, int32_t* lrank, uint32_t* status, cudaStream_t s) {
  topk_rank_kernel<<<d.nblk, 256, 0, s>>>(d.T, d.E, d.k, logits, topk_idx, gates, hist, lrank,
                                          status);
  return cudaGetLastError();
}

// ---------------------------------------------------------------- 3. scans (one CTA)
__device__ __forceinline__ int warp_inclusive_scan(int v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    int u = __shfl_up_sync(0xffffffffu, v, off);
    if (lane >= off) v += u;
  }
  return v;
}

// Exclusive scan of one value per thread over the CTA (blockDim.x multiple of 32).
__device__ int block_exclusive_scan(int v, int* s_warp, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  int inc = warp_inclusive_scan(v);
  if (lane == 31) s_warp[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    int w = (lane < nw) ? s_warp[lane] : 0;
    int wi = warp_inclusive_scan(w);
    if (lane < nw) s_warp[lane] = wi - w;
    if (lane == 31) *total = wi;
  }
  __syncthreads();
  int r = s_warp[warp] + inc - v;
  __syncthreads();
  return r;
}

__global__ void __launch_bounds__(kMaxE) plan_scan_kernel(int E, int nblk, int32_t* hist,
                                                          int32_t* counts, int32_t* offsets,
                                                          int32_t* poff, int32_t* tile_expert,
                                                          int32_t* num_mtiles, int32_t* ptile,
                                                          int32_t* num_ptiles, int32_t* dwr_q0,
                                                          int32_t* dwr_item_e) {
  __shared__ int s_warp[32];
  __shared__ int s_total;
  const int e = threadIdx.x;
  int run = 0;
  if (e < E) {
    // rows of e in earlier blocks (exclusive, in place); loads batched for latency
    for (int b0 = 0; b0 < nblk; b0 += 32) {
      int v[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) v[i] = (b0 + i < nblk) ? hist[(size_t)(b0 + i) * E + e] : 0;
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        if (b0 + i < nblk) hist[(size_t)(b0 + i) * E + e] = run;
        run += v[i];
      }
    }
  }
  const int cnt = (e < E) ? run : 0;
  const int pcnt = (cnt + kRowPad - 1) / kRowPad * kRowPad;
  int off = block_exclusive_scan(cnt, s_warp, &s_total);
  const int R = s_total;
  int poff_e = block_exclusive_scan(pcnt, s_warp, &s_total);
  const int P = s_total;
  // row-tile pairs of the expert's segment: tiles 0-1, 2-3, ...; an odd last one alone
  const int mt_e = pcnt / kRowPad;
  const int np_e = (mt_e + 1) / 2;
  const int pq0 = block_exclusive_scan(np_e, s_warp, &s_total);
  const int NP = s_total;
  // chunks of the router weight gradient's row sums
  const int nq_e = (cnt + kDwrChunk - 1) / kDwrChunk;
  const int q0 = block_exclusive_scan(nq_e, s_warp, &s_total);
  const int NQ = s_total;
  if (e < E) {
    counts[e] = cnt;
    offsets[e] = off;
    poff[e] = poff_e;
    for (int m = poff_e / kRowPad; m < (poff_e + pcnt) / kRowPad; ++m) tile_expert[m] = e;
    for (int q = 0; q < np_e; ++q)
      ptile[pq0 + q] = ((poff_e / kRowPad + 2 * q) << 1) | (2 * q + 1 < mt_e ? 1 : 0);
    dwr_q0[e] = q0;
    for (int q = 0; q < nq_e; ++q) dwr_item_e[q0 + q] = e;
  }
  if (e == 0) {
    offsets[E] = R;
    poff[E] = P;
    *num_mtiles = P / kRowPad;
    *num_ptiles = NP;
    dwr_q0[E] = NQ;
  }
}

// 3b. macrobatches ([C] "Ring token buffers (macrobatch)"): macrobatch m holds tokens
// [m*Tm, (m+1)*Tm). Inside an expert the table is in ascending token order, so m's rows of
// expert e are one contiguous run of e's table rows; its start and length follow from the
// scanned block histograms. Each macrobatch gets its own 128-row padded expert segments
// and tile map; mrow0 places the macrobatches one after another.
__global__ void __launch_bounds__(kMaxE) plan_macro_kernel(int E, int nblk, int M, int blk_m,
                                                           int mt_m_max,
                                                           const int32_t* __restrict__ hist,
                                                           const int32_t* __restrict__ counts,
                                                           const int32_t* __restrict__ offsets,
                                                           int32_t* mstart, int32_t* mcount,
                                                           int32_t* mpoff, int32_t* mtile_expert,
                                                           int32_t* mtiles, int32_t* mrow0) {
  __shared__ int s_warp[32];
  __shared__ int s_total;
  const int e = threadIdx.x;
  int row0 = 0;
  for (int m = 0; m < M; ++m) {
    int st = 0, cnt = 0;
    if (e < E) {
      const int b0 = m * blk_m, b1 = (m + 1) * blk_m;
      const int before = b0 < nblk ? hist[(size_t)b0 * E + e] : counts[e];
      const int upto = b1 < nblk ? hist[(size_t)b1 * E + e] : counts[e];
      st = offsets[e] + before;
      cnt = upto - before;
    }
    const int pcnt = (cnt + kRowPad - 1) / kRowPad * kRowPad;
    const int po = block_exclusive_scan(pcnt, s_warp, &s_total);
    const int P = s_total;
    if (e < E) {
      mstart[(size_t)m * E + e] = st;
      mcount[(size_t)m * E + e] = cnt;
      mpoff[(size_t)m * (E + 1) + e] = po;
      for (int t = po / kRowPad; t < (po + pcnt) / kRowPad && t < mt_m_max; ++t)
        mtile_expert[(size_t)m * mt_m_max + t] = e;
    }
    if (e == 0) {
      mpoff[(size_t)m * (E + 1) + E] = P;
      mtiles[m] = P / kRowPad;
      mrow0[m] = row0;
    }
    row0 += P;
  }
  if (e == 0) mrow0[M] = row0;
}

cudaError_t launch_plan_scan(const Dims& d, int32_t* hist, int32_t* counts, int32_t* offsets,
                             const AuxPtrs& a, cudaStream_t s) {
  int threads = (d.E + 31) / 32 * 32;
  plan_scan_kernel<<<1, threads, 0, s>>>(d.E, d.nblk, hist, counts, offsets, a.poff,
                                         a.tile_expert, a.num_mtiles, a.ptile, a.num_ptiles,
                                         a.dwr_q0, a.dwr_item_e);
  return cudaGetLastError();
}

cudaError_t launch_plan_macro(const Dims& d, const int32_t* hist, const int32_t* counts,
                              const int32_t* offsets, const AuxPtrs& a, cudaStream_t s) {
  int threads = (d.E + 31) / 32 * 32;
  plan_macro_kernel<<<1, threads, 0, s>>>(d.E, d.nblk, d.M, d.Tm / kTokBlock, d.mt_m_max, hist,
                                          counts, offsets, a.mstart, a.mcount, a.mpoff,
                                          a.mtile_expert, a.mtiles, a.mrow0);
  return cudaGetLastError();
}

// ---------------------------------------------------------------- 4. scatter into the table
__global__ void plan_scatter_kernel(int R, int k, int E, const int32_t* __restrict__ topk_idx,
                                    const int32_t* __restrict__ hist,
                                    const int32_t* __restrict__ lrank,
                                    const int32_t* __restrict__ offsets,
                                    int32_t* __restrict__ table, int32_t* __restrict__ inv) {
  int sl = blockIdx.x * blockDim.x + threadIdx.x;
  if (sl >= R) return;
  int t = sl / k, j = sl - t * k;
  int e = topk_idx[sl];
  if (e < 0 || e >= E) e = 0;  // already flagged by the rank kernel
  int row = offsets[e] + hist[(size_t)(t / kTokBlock) * E + e] + lrank[sl];
  table[2 * (size_t)row] = t;
  table[2 * (size_t)row + 1] = j;
  inv[sl] = row;
}

cudaError_t launch_plan_scatter(const Dims& d, const int32_t* topk_idx, const int32_t* hist,
                                const int32_t* lrank, const int32_t* offsets, int32_t* table,
                                int32_t* inv, cudaStream_t s) {
  int threads = 256;
  int blocks = (d.R + threads - 1) / threads;
  plan_scatter_kernel<<<blocks, threads, 0, s>>>(d.R, d.k, d.E, topk_idx, hist, lrank, offsets,
                                                 table, inv);
  return cudaGetLastError();
}

}  // namespace mok
