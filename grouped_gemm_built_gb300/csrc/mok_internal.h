// Library-internal declarations: buffer layouts and kernel launchers.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/mok.h"

namespace mok {

constexpr int kRowPad = 128;          // expert segments are padded to whole 128-row tiles
constexpr int kTokBlock = 32;         // tokens per block of the schedule histogram
constexpr int kMaxE = 512;
constexpr int kMaxK = 8;
constexpr uint32_t kErrTimeout = 1u;  // device status bits
constexpr uint32_t kErrBadExpert = 2u;

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

struct Dims {
  int T, H, I, E, k, Is;
  int router;
  int R;        // T*k routed rows
  int P_max;    // upper bound of padded rows: R + E*127, rounded up to 128
  int mt_max;   // P_max / 128
  int nblk;     // ceil(T / 32) histogram blocks
};

// aux buffer (persists from mok_plan to mok_moe_fwd / mok_moe_bwd)
struct AuxLayout {
  size_t status, poff, tile_expert, num_mtiles, total;
};
// scratch for mok_plan
struct PlanWs {
  size_t logits, hist, lrank, total;
};
// scratch for the forward
struct FwdWs {
  size_t xg, h, o, hs, os, total;
};
// scratch for the backward
struct BwdWs {
  size_t dyg, xg, du, dv, hg, dxg, dgp, dl, dus, dvs, hsg, dxs, total;
};
// saved activations (forward -> backward)
struct SavedLayout {
  size_t u, v, us, vs, total;
};

Dims make_dims(const mok_dims& d);
AuxLayout aux_layout(const Dims& d);
PlanWs plan_ws(const Dims& d);
FwdWs fwd_ws(const Dims& d);
BwdWs bwd_ws(const Dims& d);
SavedLayout saved_layout(const Dims& d);

// Pointers into the aux buffer.
struct AuxPtrs {
  uint32_t* status;
  int32_t* poff;        // [E+1] padded offsets (multiples of 128)
  int32_t* tile_expert; // [mt_max] expert of each 128-row tile of the padded row space
  int32_t* num_mtiles;  // [1]
};
inline AuxPtrs aux_ptrs(const Dims& d, void* aux) {
  AuxLayout L = aux_layout(d);
  char* b = static_cast<char*>(aux);
  return AuxPtrs{reinterpret_cast<uint32_t*>(b + L.status), reinterpret_cast<int32_t*>(b + L.poff),
                 reinterpret_cast<int32_t*>(b + L.tile_expert),
                 reinterpret_cast<int32_t*>(b + L.num_mtiles)};
}

// ---------------------------------------------------------------- launchers (mok_route.cu)
cudaError_t launch_router_logits(const Dims& d, const void* x, const float* Wr, const float* bias,
                                 float* logits, cudaStream_t s);
cudaError_t launch_topk_rank(const Dims& d, const float* logits, int32_t* topk_idx, float* gates,
                             int32_t* hist, int32_t* lrank, uint32_t* status, cudaStream_t s);
cudaError_t launch_plan_scan(const Dims& d, int32_t* hist, int32_t* counts, int32_t* offsets,
                             const AuxPtrs& a, cudaStream_t s);
cudaError_t launch_plan_scatter(const Dims& d, const int32_t* topk_idx, const int32_t* hist,
                                const int32_t* lrank, const int32_t* offsets, int32_t* table,
                                int32_t* inv, cudaStream_t s);

// ---------------------------------------------------------------- launchers (mok_move.cu)
// Xg[p] = src[table token of padded row p] (zero rows for padding); optional per-row gate.
cudaError_t launch_gather_rows(const Dims& d, const void* src, const mok_sched& sc,
                               const AuxPtrs& a, void* dst, int num_sms, cudaStream_t s);
// y[t] = sum_j gates[t][j] * O[row(t,j)] (+ add[t]) in fp32, slot order, -> bf16.
cudaError_t launch_combine(const Dims& d, const void* O, const mok_sched& sc, const AuxPtrs& a,
                           const void* add, bool weighted, void* y, cudaStream_t s);
// WrT [E][H] = Wr [H][E]^T (router rows made contiguous for the reverse combine)
cudaError_t launch_transpose_wr(const Dims& d, const float* Wr, float* WrT, cudaStream_t s);
// dX[t] = sum_j dXg[row(t,j)] + dXs[t] + sum_j dl[t][j] * WrT[e_j][:]  (dl may be null)
cudaError_t launch_reverse_combine(const Dims& d, const void* dXg, const mok_sched& sc,
                                   const AuxPtrs& a, const void* dXs, const float* dl,
                                   const float* WrT, void* dX, cudaStream_t s);
// dg[t][j] = sum of the per-tile partial dot products; dl = softmax-renorm backward.
cudaError_t launch_router_grad(const Dims& d, const float* dgp, int n_parts, const mok_sched& sc,
                               const AuxPtrs& a, float* dgates, float* dl, cudaStream_t s);
// dWr[:, e] = sum over expert e's table rows of x[t] * dl[t][j]   (fixed row order)
cudaError_t launch_router_dwr(const Dims& d, const void* x, const mok_sched& sc, const AuxPtrs& a,
                              const float* dl, float* dWr, cudaStream_t s);

// ---------------------------------------------------------------- grouped GEMMs (mok_gemm.cu)
enum GemmMode : int {
  kFwdUpGate = 0,   // [U V] = Xg [W_up W_gate]; h = silu(V) * U
  kFwdDown = 1,     // O = h W_down
  kBwdDH = 2,       // D = dYg W_down^T; SwiGLU' fused with the router-weight gradient
  kBwdDX = 3,       // dXg = du W_up^T + dv W_gate^T
  kBwdDWDown = 4,   // dW_down = (g h)^T dYg
  kBwdDWUpGate = 5, // dW_up = Xg^T du, dW_gate = Xg^T dv
};

struct GemmCall {
  GemmMode mode;
  // problem
  int M_rows;           // rows of the row space (padded rows, or T for the dense case)
  bool dense;           // one group over M_rows rows (shared expert); else routed groups
  int H, I;             // hidden size and this FFN's intermediate size
  int groups;           // experts (dense: 1)
  // operands (device pointers)
  const void* a0; const void* a1;      // row-space operands (Xg / h / dYg / du, dv ...)
  const void* b0; const void* b1;      // weights
  void* out0; void* out1; void* out2;  // outputs
  const void* aux0; const void* aux1;  // extra epilogue inputs (saved U, V)
  float* dgp;                          // kBwdDH: per-tile partial router-weight gradients
  // schedule (routed case)
  const int32_t* poff; const int32_t* counts; const int32_t* offsets;
  const int32_t* tile_expert; const int32_t* num_mtiles;
  const int32_t* table; const float* gates; int k;
  uint32_t* status;
};
cudaError_t launch_gemm(const GemmCall& c, int num_sms, cudaStream_t s);
int gemm_dh_parts(int I);  // number of partial dg columns kBwdDH writes per row

}  // namespace mok
