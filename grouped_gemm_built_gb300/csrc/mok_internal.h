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
constexpr int kTileCounters = 16;     // GEMM launches of one call with a dynamic tile order

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

struct Dims {
  int T, H, I, E, k, Is;
  int router;
  int R;        // T*k routed rows
  int P_max;    // upper bound of padded rows: R + E*127, rounded up to 128
  int mt_max;   // P_max / 128
  int nblk;     // ceil(T / 32) histogram blocks
  // macrobatches: consecutive token ranges of Tm tokens (a multiple of 128), each with its
  // own 128-row padded expert segments; their padded row spaces are concatenated (P_cat
  // rows) for h, U, V and O. Dispatched rows pass through a ring of S slots of P_slot rows.
  int M;        // macrobatches
  int Tm;       // tokens per macrobatch (the last one may hold fewer)
  int mt_m_max; // most 128-row tiles of one macrobatch
  int P_slot;   // rows of one ring slot (mt_m_max * 128)
  int S;        // ring slots (1 <= S <= M)
  int P_cat;    // concatenated padded rows of all macrobatches, bound
};

// aux buffer (persists from mok_plan to mok_moe_fwd / mok_moe_bwd). Per macrobatch m and
// expert e: mstart[m][e] (table row of e's first row in m), mcount[m][e], mpoff[m][e]
// (padded offset inside m, E+1 entries), mtile_expert[m][tile], mtiles[m], mrow0[m] (first
// row of m in the concatenated padded space, M+1 entries).
// ptile[q] = (first row tile << 1) | (1 if the pair has a second row tile): the row-tile
// pairs of each expert's segment (tiles 0-1, 2-3, ...; an odd last tile alone), expert
// by expert; num_ptiles[0] = their count (at most max_ptiles(d)).
struct AuxLayout {
  size_t status, poff, tile_expert, num_mtiles;
  size_t mstart, mcount, mpoff, mtile_expert, mtiles, mrow0, ptile, num_ptiles;
  size_t dwr_q0, dwr_item_e, total;
};
inline int max_ptiles(const Dims& d) { return (d.mt_max + d.E + 1) / 2; }
// The router weight gradient sums each expert's table rows in chunks of kDwrChunk rows
// (a busy expert spreads over many CTAs): dwr_q0[e] = the expert's first chunk (E+1
// entries, exclusive scan of ceil(count / kDwrChunk)), dwr_item_e[q] = the expert of chunk q.
constexpr int kDwrChunk = 1024;
inline int dwr_items_max(const Dims& d) { return (d.R + kDwrChunk - 1) / kDwrChunk + d.E; }
// scratch for mok_plan
struct PlanWs {
  size_t logits, hist, lrank, wr3, total;
};
inline int router_ld(const Dims& d) { return (d.E + 63) / 64 * 64; }
// scratch for the forward (xq/xsf, hq/hsf: MXFP8 operands and their scale atoms; ring:
// S slots of dispatched rows (bf16, or E4M3 + atoms at ring_sf); cnt: megakernel counters)
struct FwdWs {
  size_t h, o, hs, os, xq, xsf, hq, hsf, ring, ring_sf, cnt, tcnt, total;
};
// device counters of the forward megakernel (ints, zeroed before each launch)
struct MegaCnt {
  int gathered, hcnt, upg_done, down_done, abort_flag, total;
};
inline MegaCnt mega_cnt(const Dims& d) {
  MegaCnt c;
  c.gathered = 0;
  c.hcnt = c.gathered + d.M * d.mt_m_max;
  c.upg_done = c.hcnt + d.M * d.mt_m_max;
  c.down_done = c.upg_done + d.M;
  c.abort_flag = c.down_done + d.M;
  c.total = c.abort_flag + 1;
  return c;
}
// MXFP8 copies of the routed weights (mok_quantize_weights_mxfp8): data in the weights'
// own layouts, atoms [e][K/128][N/128]. *_h: blocks along H; *_i: blocks along I.
struct MxWeights {
  size_t up_h, up_h_sf, gate_h, gate_h_sf, down_i, down_i_sf;  // forward GEMMs
  size_t down_h, down_h_sf, up_i, up_i_sf, gate_i, gate_i_sf;  // backward dH / dX GEMMs
  size_t total;
};
// scratch for the backward. MXFP8 operands (E4M3 + atoms): dY along H (dH GEMM), dY and
// x in 32-row blocks (dW GEMMs), du/dv along I (dX GEMM), du/dv/g*h in 32-row blocks.
struct BwdWs {
  size_t dyg, du, dv, hg, du_lo, dv_lo, hg_lo, dxg, dgp, dl, dus, dvs, hsg, dus_lo,
      dvs_lo, hsg_lo, dxs;
  size_t uvmap, xr;   // after a multi-macrobatch megakernel forward: U, V row map; x rows
  size_t tcnt;        // tile counters (dynamic tile order)
  size_t dwr_part;    // router weight gradient: per-chunk partial sums [dwr_items_max][H]
  size_t q_dy_h, sf_dy_h, q_dy_r, sf_dy_r, q_x_r, sf_x_r;
  size_t q_du_i, sf_du_i, q_dv_i, sf_dv_i, q_du_r, sf_du_r, q_dv_r, sf_dv_r, q_hg_r, sf_hg_r;
  size_t total;
};
// saved activations (forward -> backward): U, V bf16; xg: the gathered rows of x in the
// padded row space (BF16 forward), which the backward's weight gradients read again
struct SavedLayout {
  size_t u, v, us, vs, xg, total;
};

// num_sms: the device's SM count (0 without a device), for the two-wave minibatch rule
Dims make_dims(const mok_dims& d, int num_sms);
AuxLayout aux_layout(const Dims& d);
PlanWs plan_ws(const Dims& d);
FwdWs fwd_ws(const Dims& d);
BwdWs bwd_ws(const Dims& d);
SavedLayout saved_layout(const Dims& d);
MxWeights mx_weights_layout(const Dims& d);

// Pointers into the aux buffer.
struct AuxPtrs {
  uint32_t* status;
  int32_t* poff;        // [E+1] padded offsets (multiples of 128)
  int32_t* tile_expert; // [mt_max] expert of each 128-row tile of the padded row space
  int32_t* num_mtiles;  // [1]
  int32_t* mstart;      // [M][E]
  int32_t* mcount;      // [M][E]
  int32_t* mpoff;       // [M][E+1]
  int32_t* mtile_expert;// [M][mt_m_max]
  int32_t* mtiles;      // [M]
  int32_t* mrow0;       // [M+1]
  int32_t* ptile;       // [max_ptiles] row-tile pairs of the padded row space
  int32_t* num_ptiles;  // [1]
  int32_t* dwr_q0;      // [E+1]
  int32_t* dwr_item_e;  // [dwr_items_max]
};
inline AuxPtrs aux_ptrs(const Dims& d, void* aux) {
  AuxLayout L = aux_layout(d);
  char* b = static_cast<char*>(aux);
  auto I32 = [&](size_t off) { return reinterpret_cast<int32_t*>(b + off); };
  return AuxPtrs{reinterpret_cast<uint32_t*>(b + L.status), I32(L.poff), I32(L.tile_expert),
                 I32(L.num_mtiles), I32(L.mstart), I32(L.mcount), I32(L.mpoff),
                 I32(L.mtile_expert), I32(L.mtiles), I32(L.mrow0), I32(L.ptile),
                 I32(L.num_ptiles), I32(L.dwr_q0), I32(L.dwr_item_e)};
}

// Read-only views of a context (defined in mok_api.cu).
const Dims* ctx_dims(mok_ctx_t ctx);
int ctx_num_sms(mok_ctx_t ctx);

// ---------------------------------------------------------------- launchers (mok_route.cu)
cudaError_t launch_topk_rank(const Dims& d, const float* logits, int32_t* topk_idx, float* gates,
                             int32_t* hist, int32_t* lrank, uint32_t* status, cudaStream_t s);
cudaError_t launch_plan_scan(const Dims& d, int32_t* hist, int32_t* counts, int32_t* offsets,
                             const AuxPtrs& a, cudaStream_t s);
// per-macrobatch arrays from the scanned histograms (after launch_plan_scan)
cudaError_t launch_plan_macro(const Dims& d, const int32_t* hist, const int32_t* counts,
                              const int32_t* offsets, const AuxPtrs& a, cudaStream_t s);
cudaError_t launch_plan_scatter(const Dims& d, const int32_t* topk_idx, const int32_t* hist,
                                const int32_t* lrank, const int32_t* offsets, int32_t* table,
                                int32_t* inv, cudaStream_t s);

// Wr [H][E] fp32 -> three bf16 matrices stacked [3][H][ld] (columns >= E zero) with
// Wr = hi + mid + lo exactly: hi = bf16(w), mid = bf16(w - hi), lo = bf16(w - hi - mid).
cudaError_t launch_split_wr(const Dims& d, const float* Wr, int ld, void* out, cudaStream_t s);

// ---------------------------------------------------------------- launchers (mok_move.cu)
// Xg[p] = src[table token of padded row p] (zero rows for padding); optional per-row gate.
cudaError_t launch_gather_rows(const Dims& d, const void* src, const mok_sched& sc,
                               const AuxPtrs& a, void* dst, int num_sms, cudaStream_t s);
// y[t] = sum_j gates[t][j] * O[row(t,j)] (+ add[t]) in slot order, summed in fp32. O, add
// and y are fp32, or (bf16) all three bf16 with y rounded once from the fp32 sum.
cudaError_t launch_combine(const Dims& d, const void* O, const mok_sched& sc, const AuxPtrs& a,
                           const void* add, bool weighted, bool bf16, void* y, cudaStream_t s);
// WrT [E][H] = Wr [H][E]^T (router rows made contiguous for the reverse combine)
cudaError_t launch_transpose_wr(const Dims& d, const float* Wr, float* WrT, cudaStream_t s);
// dX[t] = sum_j dXg[row(t,j)] + dXs[t] + sum_j dl[t][j] * WrT[e_j][:], summed in fp32
// (dl may be null); dXg, dXs and dX fp32, or (bf16) all three bf16
cudaError_t launch_reverse_combine(const Dims& d, const void* dXg, const mok_sched& sc,
                                   const AuxPtrs& a, const void* dXs, const float* dl,
                                   const float* WrT, bool bf16, void* dX, cudaStream_t s);
// dg[t][j] = sum of the per-tile partial dot products; dl = softmax-renorm backward.
cudaError_t launch_router_grad(const Dims& d, const float* dgp, int n_parts, const mok_sched& sc,
                               const AuxPtrs& a, float* dgates, float* dl, cudaStream_t s);
// After a forward that kept U, V in the per-macrobatch padded layout: for every row p of the
// whole-batch padded row space, the row of the same (token, slot) in that layout (mrow0[m] +
// mpoff[m][e] + its place in m's run of e's rows), -1 for padding rows.
cudaError_t launch_uv_rowmap(const Dims& d, const mok_sched& sc, const AuxPtrs& a, int32_t* map,
                             cudaStream_t s);
// dWr[:, e] = sum over expert e's table rows of x[t] * dl[t][j]   (fixed row order)
cudaError_t launch_router_dwr(const Dims& d, const void* x, const mok_sched& sc, const AuxPtrs& a,
                              float* part,
                              const float* dl, float* dWr, cudaStream_t s);

// ---------------------------------------------------------------- grouped GEMMs (mok_gemm.cu)
enum GemmMode : int {
  kFwdUpGate = 0,   // [U V] = Xg [W_up W_gate]; h = silu(V) * U
  kFwdDown = 1,     // O = h W_down
  kBwdDH = 2,       // D = dYg W_down^T; SwiGLU' fused with the router-weight gradient
  kBwdDX = 3,       // dXg = du W_up^T + dv W_gate^T
  kBwdDWDown = 4,   // dW_down = (g h)^T dYg
  kBwdDWUpGate = 5, // dW_up = Xg^T du, dW_gate = Xg^T dv
  kRouter = 6,      // logits = x [Wr_hi; Wr_mid; Wr_lo] (+ bias): fp32 router on tensor cores
};

// Operands per mode (BF16; MXFP8 in brackets):
//   kFwdUpGate   a0 = Xg [x_q]; b0, b1 = W_up, W_gate; out0 = h bf16 [out_q0 + atoms],
//                out1, out2 = U, V bf16 (saved)
//   kFwdDown     a0 = h [h_q]; b0 = W_down; out0 = O fp32 (out_bf16: bf16)
//   kBwdDH       a0 = dYg [dY_q]; b0 = W_down; u, v = saved U, V; out0..5 = du, dv, g*h as
//                bf16 hi/lo pairs [out_q0..4 + atoms]; dgp
//   kBwdDX       a0, a1 = du_hi, dv_hi [du_q, dv_q]; b0, b1 = W_up, W_gate; out0 = dXg fp32
//                (out_bf16: bf16)
//   kBwdDWDown   a0, a1 = g*h hi, lo [a0 = g*h_q]; b0 = dYg [dY_q]; out0 = dW_down fp32
//                (out_bf16: bf16)
//   kBwdDWUpGate a0 = Xg [x_q]; b0, b1 = du_hi, dv_hi; b2, b3 = du_lo, dv_lo
//                [b0, b1 = du_q, dv_q]; out0, out1 = dW_up, dW_gate fp32 (out_bf16: bf16)
//   kRouter      a0 = x; b0 = [Wr_hi; Wr_mid; Wr_lo] [3H][ld_b] bf16; out0 = logits [T][E]
//                fp32 (dense, BF16 only)
struct GemmCall {
  GemmMode mode;
  // problem
  int M_rows;           // rows of the row space (padded rows, or T for the dense case)
  int a_rows;           // rows of a[0]'s buffer when it differs from M_rows (0: M_rows)
  bool dense;           // one group over M_rows rows (shared expert); else routed groups
  int H, I;             // hidden size and this FFN's intermediate size
  int groups;           // experts (dense: 1)
  int n_out;            // kRouter: E (output columns); the B operand has ld_b columns
  int ld_b;             // kRouter: columns of the stacked bf16 router weights (E rounded to 64)
  const float* bias;    // kRouter: logit bias [E] or null
  const void* a[4];     // row-space operands
  const void* b[4];     // weights / second row-space operand
  void* out[6];         // outputs (kBwdDH: du, du lo, dv, dv lo, g*h, g*h lo; lo optional)
  bool split;           // dW modes (bf16): operands a[1] / b[2..3] hold the lo halves
  bool out_bf16;        // kFwdDown, kBwdDX, dW modes: outputs rounded to bf16 (else fp32)
  const void* u;        // kBwdDH: saved U, V (bf16)
  const void* v;
  const int32_t* uv_row;// kBwdDH: row of U, V for each row of the row space (null: the same
                        // row; -1: a padding row, read as zeros)
  float* dgp;           // kBwdDH: per-tile partial router-weight gradients
  // schedule (routed case)
  const int32_t* poff; const int32_t* counts; const int32_t* offsets;
  const int32_t* tile_expert; const int32_t* num_mtiles;
  const int32_t* table; const float* gates; int k;
  // row-tile pairs (BF16 routed row-space modes): one CTA runs both row tiles of a pair
  // against one weight tile, two accumulators side by side (AuxLayout::ptile)
  bool pair;
  const int32_t* ptile; const int32_t* num_ptiles; int max_ptiles;
  // BF16 dW modes without hi/lo split and dH, static tile order: run on SM pairs
  // (clusters of two CTAs sharing M = 256 MMAs; dW when the dW rows per expert are a whole
  // number of 256-row tiles, dH over the plan's pairs of row tiles); otherwise the launch
  // runs one CTA per tile as usual
  bool smpair;
  // MXFP8 kFwdUpGate / kFwdDown: the BF16 shared expert's tiles in the same launch
  // (s_a: x, or the shared h; s_b: Ws_up, Ws_gate, or Ws_down; s_out: hs, Us, Vs, or the
  // shared output rows; s_rows = T; s_I the shared expert's intermediate size); null: none
  const void* s_a; const void* s_b[2]; void* s_out[3]; int s_rows, s_I;
  uint32_t* status;
  uint64_t timeout_ns;  // bound of every device wait (0: 2 s)
  int* tile_counter;    // dynamic tile order: a zeroed int of device memory (null: static)
  bool clc;             // tiles handed out by cluster launch control (one CTA per tile)
  // MXFP8 (E4M3 operands with 512-byte scale atoms; see mok_quant.cu)
  bool mx;
  const void* sfa; const void* sfa1;                   // A scale atoms (second: kBwdDX dv)
  const void* sfb0; const void* sfb1;                  // B scale atoms
  void* out_q[5]; void* out_sf[5];                     // quantised epilogue outputs + atoms
};
cudaError_t launch_gemm(const GemmCall& c, int num_sms, cudaStream_t s);

// Forward megakernel (mok_gemm.cu): dispatch into the ring, routed up|gate and down GEMMs
// and the combine in one cooperative launch over all SMs. up / down describe the two
// routed GEMMs (up.a[0] = ring, up.a_rows = S * P_slot; rows of h, U, V, O = P_cat).
struct MegaCall {
  GemmCall up, down;
  int M, S, P_slot, Tm, T, mt_m_max, n_comm;   // n_comm 0: default
  const int32_t* mstart; const int32_t* mcount; const int32_t* mpoff;
  const int32_t* mtile_expert; const int32_t* mtiles; const int32_t* mrow0;
  const int32_t* topk_idx; const int32_t* inv;
  const void* x; void* ring; void* ring_sf;
  const void* O; const void* Os; void* y;   // fp32, or bf16 when down.out_bf16
  int* cnt;
  unsigned long long* trace;   // profiling: kTraceStamps stamps per CTA, or null
  int withhold;                // test hook: row tile 0 of macrobatch 0 is never published
};
// megakernel phase stamps (%globaltimer ns), per CTA
constexpr int kTraceStamps = 8;
constexpr int kStampStart = 0, kStampCommDone = 1, kStampGemmDone = 2, kStampProducerDone = 3,
              kStampCombine = 4, kStampEnd = 5;
constexpr int kTraceSlots = 64;   // megakernel launches kept between two reports
cudaError_t launch_fwd_mega(const MegaCall& c, int num_sms, cudaStream_t s);

// ---------------------------------------------------------------- MXFP8 quantisers (mok_quant.cu)
// src [batch][rows][cols] bf16 -> dst e4m3 (same layout) + 512-byte scale atoms; blocks of
// 32 along the columns (k_along_cols) or along the rows. Atom (kc, mc) of batch z is at
// atoms + z*(rows/128)*(cols/128)*512 + (kc*s_kc + mc*s_mc)*512, kc indexing K / 128 and
// mc the other axis / 128.
cudaError_t launch_mx_quant(const void* src, int rows, int cols, int batch, bool k_along_cols,
                            void* dst, void* atoms, int s_kc, int s_mc, cudaStream_t s);
// forward dispatch in MXFP8: pull x rows by the table and quantise along H
// (atoms [P/128][H/128]).
cudaError_t launch_gather_quant(const Dims& d, const void* src, const mok_sched& sc,
                                const AuxPtrs& a, void* dst, void* atoms, int num_sms,
                                cudaStream_t s);
// the same pull, quantised in blocks of 32 padded rows (contraction axis of the dW GEMMs):
// atoms [P/128][H/128] with m = column, b = 32-row block inside the 128-row tile.
cudaError_t launch_gather_quant_rows(const Dims& d, const void* src, const mok_sched& sc,
                                     const AuxPtrs& a, void* dst, void* atoms, int num_sms,
                                     cudaStream_t s);
int gemm_dh_parts(int I, bool mx);  // partial dg columns kBwdDH writes per row

}  // namespace mok
