/*
 * mok.h - C ABI of the GB300 (sm_103a) MoE SwiGLU layer library.
 *
 * The library runs the data-parallel hot path of a Mixture-of-Experts layer as the
 * Mixture-of-Kittens articles describe it, on one GPU:
 *   top-k routing -> schedule table built on the GPU with no sort -> gather of token rows
 *   into expert order -> grouped up/gate GEMM with SwiGLU -> grouped down GEMM ->
 *   weighted combine; and the backward pass (SwiGLU derivative fused with the
 *   router-weight gradient, then dX, dW_up, dW_gate, dW_down in a fixed order).
 *
 * Sources for what is computed (page title, then section):
 *   [S] "Mixture-of-Kittens: Cursors Open-Source-Ansatz fuer effizientes MoE-Training auf
 *       NVL72" (sebask.de): intro (router, experts with up/gate/down projection);
 *       "Push oder Pull?" (pull dispatch, push combine, one plan for the four exchange
 *       steps); "Das Scheduling" (table of source indices, order follows from routing,
 *       no sort, built on the GPU); "Determinismus und MXFP8-Unterstuetzung".
 *   [C] "Cursor abre codigo de megakernel MoE para GPUs NVL72" (stamatios.com):
 *       "Escolha da direcao de comunicacao" (table built once, reused by the four ops);
 *       "Granularidade do overlap" (minibatch of at least two full SM waves);
 *       "Ring token buffers (macrobatch)"; "Outras caracteristicas" (determinism,
 *       MXFP8 with BF16 shared expert, router-weight gradient fused into SwiGLU bwd).
 *
 * Conventions (every entry point):
 *   - All tensors are row-major and dense. "bf16" buffers hold IEEE bfloat16 bits.
 *   - Every data pointer is a DEVICE pointer owned by the caller. The library never
 *     allocates device memory inside these calls; scratch space is the caller's
 *     `workspace`, whose size mok_get_sizes reports.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream). Calls only enqueue work
 *     on it; none synchronises with the host except mok_get_status.
 *   - Argument errors are detected on the host and returned before anything is launched.
 *     Errors found on the device (bounded waits that time out, out-of-range expert ids)
 *     set bits in a device status word kept in the schedule's aux buffer; mok_get_status
 *     reads and clears it.
 *   - Results are bitwise reproducible from run to run: every reduction has a fixed
 *     order that depends only on the schedule table.
 */
#ifndef MOK_H_
#define MOK_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MOK_OK = 0,
  MOK_ERR_INVALID_ARG = -1, /* bad pointer, size or combination of arguments        */
  MOK_ERR_UNSUPPORTED = -2, /* valid request the library does not support           */
  MOK_ERR_WORKSPACE = -3,   /* workspace/aux/saved buffer missing or misaligned     */
  MOK_ERR_CUDA = -4,        /* a CUDA runtime/driver call failed                    */
  MOK_ERR_TIMEOUT = -5,     /* a device-side bounded wait expired                   */
  MOK_ERR_DEVICE = -6       /* the device flagged bad data (e.g. expert id >= E)    */
} mok_status;

/* MOK_BF16: bf16 tensor-core operands with fp32 accumulation (results in the type that
 *   mok_set_output_dtype selects). Inputs,
 *   weights, h and the dX GEMM's du, dv are bf16; the weight-gradient GEMMs take du, dv
 *   and g*h as bf16 hi + lo pairs (two MMAs per K step), close to fp32 operands.
 * MOK_MXFP8: E4M3 elements with one UE8M0 scale per 32 along each GEMM's contraction axis;
 *   the shared expert stays BF16 (as in MOK_BF16); in the forward its BF16 tiles run in
 *   the same launches as the routed MXFP8 tiles (up|gate, then down), after them.
 * In every precision the forward keeps U = x W_up and V = x W_gate for the backward as bf16
 *   values (h itself is formed from the fp32 accumulators).
 * MOK_BF16_WGRAD_PLAIN: as MOK_BF16 with single bf16 du, dv, g*h in the weight-gradient
 *   GEMMs: half their MMAs, at the cost of one bf16 rounding of each operand. The pages
 *   name BF16 and MXFP8 only; how BF16 feeds the weight gradients is this library's
 *   choice. */
typedef enum { MOK_BF16 = 0, MOK_MXFP8 = 1, MOK_BF16_WGRAD_PLAIN = 2 } mok_precision;

/* Type of the layer's results, in every precision:
 * MOK_OUT_BF16 (default): y, dX and the weight gradients dW_up, dW_gate, dW_down, dWs_* are
 *   bf16, each rounded once (to nearest even) from its fp32 accumulator; the expert output
 *   rows and routed dX rows that the combines add up are bf16 too, and the combines sum in
 *   fp32 before their one rounding.
 * MOK_OUT_F32: all of these in fp32, and the expert output rows and routed dX rows too.
 * dgates and dWr are fp32 in both. The pages fix no output type; BF16 training reads as
 * bf16 results accumulated in fp32, with fp32 results as the option. */
typedef enum { MOK_OUT_BF16 = 0, MOK_OUT_F32 = 1 } mok_out_dtype;

/* How mok_moe_fwd runs the routed experts:
 * MOK_FWD_MEGAKERNEL: one persistent cooperative launch over all SMs, split in software
 *   into gather/combine SMs and GEMM SMs that move macrobatches through the ring token
 *   buffer and signal each other with device counters ([C] "O que e o MoK", "Ring token
 *   buffers (macrobatch)"; [S] "Das Scheduling").
 * MOK_FWD_LAUNCHES: one launch per step (gather, up|gate GEMM, down GEMM, combine) over
 *   the whole batch; macrobatches are ignored. Same arithmetic, same bits.
 * MOK_FWD_AUTO (default): one launch per step, the faster path on one GPU. There the
 *   megakernel's gather SMs copy rows between two places of the same HBM while the GEMM
 *   SMs already keep it busy: their copies wait on memory latency with at most a
 *   shared-memory's worth of bytes in flight, and the SMs they take are missing from the
 *   GEMMs. Its overlap pays where the gather side moves rows between GPUs instead. */
typedef enum { MOK_FWD_MEGAKERNEL = 0, MOK_FWD_LAUNCHES = 1, MOK_FWD_AUTO = 2 } mok_fwd_path;

/* Order in which the persistent grouped-GEMM launches take their tiles ([C] "Outras
 * caracteristicas" and the ihal.it article: tiles scheduled on the GPU at run time rather
 * than fixed ahead):
 * MOK_TILES_STATIC (default): CTA b takes tiles b, b + G, b + 2G, ... (G CTAs);
 * MOK_TILES_DYNAMIC: each CTA takes the next tile from a device counter when it is ready
 *   for one, so CTAs whose tiles run long (the weight gradients of busy experts) take
 *   fewer;
 * MOK_TILES_CLC: cluster launch control, the hardware scheduler of the ihal.it article's
 *   paragraph on CLC: the launch has one CTA per tile; a running CTA, when it is ready
 *   for another tile, cancels a CTA that has not been launched yet and runs that CTA's
 *   tile, so about one CTA per SM runs while the hardware hands out the rest. A launch
 *   whose tile count lives on the device (routed experts) is sized to the largest count
 *   the context's dimensions allow; CTAs beyond the actual count return at once. The
 *   hardware places these CTAs on every SM: mok_set_sm_limit does not apply to them.
 * Every output tile is one CTA's fixed-order sum in each order: same bits. */
typedef enum { MOK_TILES_STATIC = 0, MOK_TILES_DYNAMIC = 1, MOK_TILES_CLC = 2 } mok_tile_order;

/* Row-tile pairs in the BF16 routed GEMMs of the forward and of dX: one CTA runs two
 * 128-row tiles of one expert against one weight tile (two accumulators side by side,
 * pipeline stages [rows 0-127 | weight tile | rows 128-255]), so each SM keeps more weight
 * bytes in flight. MOK_PAIRS_AUTO (default): on when the experts average more than 128 and
 * at most 256 rows (weight-streaming launches); MOK_PAIRS_ON / MOK_PAIRS_OFF force it.
 * Same bits either way. MXFP8 launches, the shared expert and the forward megakernel run
 * single row tiles. */
typedef enum { MOK_PAIRS_AUTO = 0, MOK_PAIRS_ON = 1, MOK_PAIRS_OFF = 2 } mok_row_pairs;

/* SM pairs in the BF16 weight-gradient GEMMs (dW_up|dW_gate, dW_down, without the hi/lo
 * split) and the BF16 dH GEMM: the two CTAs of a cluster of two share each tensor-core MMA
 * of 256 rows (tcgen05 cta_group::2). Each CTA loads its 128 rows of A (a row tile of dY for
 * dH; 128 rows of the transposed operand for dW) and half of the other operand's 256
 * columns, so a tile moves a third less through its SM's shared memory; dH's two row tiles
 * of an expert share one weight tile. Needs the static tile order; the dW launches need dW
 * rows per expert (H, I) in whole 256-row tiles. Otherwise, and when no cluster of two
 * fits, the launch runs one CTA per tile. MOK_SMPAIRS_AUTO (default): the routed experts'
 * weight-gradient launches, and their dH launch when the experts average more than 128
 * and at most 256 rows (an expert's odd last row tile leaves half a cluster idle);
 * MOK_SMPAIRS_ON: every eligible launch, the shared expert's as well; MOK_SMPAIRS_OFF: none.
 * Every output element is the same fixed-order sum either way. */
typedef enum { MOK_SMPAIRS_AUTO = 0, MOK_SMPAIRS_ON = 1, MOK_SMPAIRS_OFF = 2 } mok_sm_pairs;

typedef struct mok_ctx_s* mok_ctx_t;

/* Layer dimensions. T tokens, H hidden, I expert intermediate size, E routed experts,
 * k experts per token. H and I must be multiples of 128; 1 <= k <= 8 <= ... E <= 512;
 * shared_I (0 = no shared expert) a multiple of 128. router = 1: mok_plan routes from
 * x and Wr; router = 0: the caller supplies topk_idx and gates (an expert slice fed by
 * an external dispatcher). macrobatches splits the token range into consecutive chunks of
 * ceil(T / macrobatches) tokens rounded up to 128 (0 or 1: one chunk), which the forward
 * megakernel passes through the ring token buffer one after another; ring_bytes bounds
 * that buffer: it holds ring_bytes / (one macrobatch's padded rows of bf16) slots, at
 * most one per macrobatch (0: one per macrobatch); fewer than one slot is
 * MOK_ERR_INVALID_ARG ([C] "Ring token buffers"). minibatch_tokens sizes the macrobatches
 * by tokens instead: 0 = not used (macrobatches decides); > 0 = that many tokens per
 * macrobatch (rounded up to 128); -1 = the two-wave rule of [C] "Granularidade do
 * overlap": mok_minibatch_tokens(H, I, k, SMs of the current device) tokens, rounded up
 * to 128, so that every macrobatch's grouped GEMMs have at least two full waves of row
 * tiles (one macrobatch when there is no device); setting both it and macrobatches is
 * MOK_ERR_INVALID_ARG. mok_get_sizes reports the resolved counts. */
typedef struct {
  int T, H, I, E, k;
  int shared_I;
  int router;
  int macrobatches;
  size_t ring_bytes;
  int minibatch_tokens;
} mok_dims;

/* Schedule produced by mok_plan and passed unchanged to mok_moe_fwd and mok_moe_bwd
 * ([S] "Push oder Pull?": the dispatch plan is reused by the other exchange steps).
 * All device pointers, caller-owned:
 *   topk_idx [T][k] int32  expert of slot (t, j); slot order = descending gate
 *   gates    [T][k] fp32   renormalised routing weights
 *   counts   [E]    int32  rows routed to each expert
 *   offsets  [E+1]  int32  exclusive prefix sum of counts
 *   table    [T*k][2] int32 for expert row r: (source token t, slot j), rows of expert e
 *                          at offsets[e] .. offsets[e+1]-1 in ascending (t, j)
 *   inv      [T][k] int32  row of (t, j) in the table
 *   aux      mok_sizes.aux_bytes, 256-byte aligned: library-private schedule data
 *            (padded offsets, tile maps, per-block histograms, device status word). */
typedef struct {
  int32_t* topk_idx;
  float* gates;
  int32_t* counts;
  int32_t* offsets;
  int32_t* table;
  int32_t* inv;
  void* aux;
} mok_sched;

/* Weights (device, bf16 unless noted):
 *   W_up, W_gate [E][H][I]; W_down [E][I][H]
 *   Ws_up, Ws_gate [H][shared_I]; Ws_down [shared_I][H]  (NULL when shared_I == 0)
 *   mx: MXFP8 copies of W_up, W_gate, W_down written by mok_quantize_weights_mxfp8
 *       (mok_sizes.mx_weight_bytes, library-private layout); required in MXFP8 mode. */
typedef struct {
  const void* W_up;
  const void* W_gate;
  const void* W_down;
  const void* Ws_up;
  const void* Ws_gate;
  const void* Ws_down;
  const void* mx;
} mok_weights;

/* Gradients written by mok_moe_bwd (device): dW_* with the weights' shapes (fp32 sums of
 * bf16/MXFP8 products, stored as bf16 or fp32 per mok_set_output_dtype); dgates [T][k] fp32
 * (dL/dgate, the router-weight gradient); dWr [H][E] fp32 (NULL when there is no router);
 * dWs_* (output type; NULL when there is no shared expert). */
typedef struct {
  void* dW_up;
  void* dW_gate;
  void* dW_down;
  float* dgates;
  float* dWr;
  void* dWs_up;
  void* dWs_gate;
  void* dWs_down;
} mok_grads;

typedef struct {
  size_t aux_bytes;        /* mok_sched.aux                                   */
  size_t workspace_bytes;  /* scratch for mok_plan / mok_moe_fwd / mok_moe_bwd  */
  size_t saved_bytes;      /* forward activations kept for the backward        */
  size_t mx_weight_bytes;  /* mok_weights.mx                                    */
  int padded_rows_max;     /* upper bound of expert rows after 128-row padding  */
  int macrobatches;        /* resolved macrobatch count                         */
  int ring_slots;          /* macrobatch slots of the ring token buffer         */
  int macrobatch_tokens;   /* resolved tokens per macrobatch (the last may hold fewer) */
} mok_sizes;

/* ---- helpers (host only; nothing is launched) ---------------------------------- */

/* Validate dims and create a context for the current CUDA device. *out owns no device
 * memory. Returns MOK_ERR_INVALID_ARG for unsupported shapes. */
mok_status mok_create(const mok_dims* dims, mok_ctx_t* out);
void mok_destroy(mok_ctx_t ctx);
/* Buffer sizes for the context's dims and precision. */
mok_status mok_get_sizes(mok_ctx_t ctx, mok_sizes* out);
/* Smallest token count whose routed rows fill at least two full waves of `num_sms` SMs
 * when every SM takes 64 rows of a grouped-GEMM tile per wave ([C] "Granularidade do
 * overlap": two waves; the page gives T >= 2368 for H=7168, I=2048, k=8, 148 SMs).
 * Returns -1 on bad arguments. */
int mok_minibatch_tokens(int H, int I, int k, int num_sms);
const char* mok_status_string(mok_status s);

/* ---- the layer ----------------------------------------------------------------- */

/* Select the arithmetic of later mok_moe_fwd / mok_moe_bwd calls (mok_precision above;
 * BF16 and MXFP8 from [S] "Determinismus und MXFP8-Unterstuetzung"; [C] "Outras
 * caracteristicas"). Host-only state change; MOK_ERR_INVALID_ARG for other values. */
mok_status mok_set_precision(mok_ctx_t ctx, mok_precision p);

/* Select the tile order of later mok_moe_fwd / mok_moe_bwd grouped GEMMs (mok_tile_order
 * above). Host-only state change; MOK_ERR_INVALID_ARG for other values. */
mok_status mok_set_tile_order(mok_ctx_t ctx, mok_tile_order order);

/* Select the row-tile pairing of later mok_moe_fwd / mok_moe_bwd BF16 routed GEMMs
 * (mok_row_pairs above). Host-only state change; MOK_ERR_INVALID_ARG for other values. */
mok_status mok_set_row_pairs(mok_ctx_t ctx, mok_row_pairs mode);

/* Select SM pairs for later mok_moe_bwd BF16 dH and weight-gradient GEMMs (mok_sm_pairs above).
 * Host-only state change; MOK_ERR_INVALID_ARG for other values. */
mok_status mok_set_sm_pairs(mok_ctx_t ctx, mok_sm_pairs mode);

/* Select the type of later mok_moe_fwd / mok_moe_bwd results (mok_out_dtype above).
 * Host-only state change; MOK_ERR_INVALID_ARG for other values. */
mok_status mok_set_output_dtype(mok_ctx_t ctx, mok_out_dtype t);

/* Select how later mok_moe_fwd calls run (mok_fwd_path above). Host-only state change;
 * MOK_ERR_INVALID_ARG for other values. */
mok_status mok_set_fwd_path(mok_ctx_t ctx, mok_fwd_path path);

/* Most SMs the context's kernels use (0 = all): persistent grids are sized to it. Results
 * do not depend on it (every sum has a fixed order), which the tests check; it also lets a
 * caller leave SMs to other work. Host-only state change. */
mok_status mok_set_sm_limit(mok_ctx_t ctx, int n);

/* Number of the forward megakernel's SMs that gather and combine (the rest run the GEMMs):
 * 0 = automatic, else 1 .. SMs - 1 (MOK_ERR_INVALID_ARG otherwise, checked at launch
 * against the device's SM count). Host-only state change. */
mok_status mok_set_comm_sms(mok_ctx_t ctx, int n);

/* Bound, in nanoseconds, of every device-side wait of later calls (pipeline barriers and
 * the megakernel's counters); 0 = 2 s, at most 60 s. A wait that passes it records
 * MOK_ERR_TIMEOUT in the status word (mok_get_status), the kernel lets its copies in
 * flight land, frees its TMEM and returns; nothing traps. Host-only state change. */
mok_status mok_set_wait_timeout(mok_ctx_t ctx, uint64_t ns);

/* Test hook (no counterpart in the articles): while on, the forward megakernel never
 * publishes the first gathered row tile, so the GEMM SMs' bounded wait for it passes its
 * limit and the call's status reads MOK_ERR_TIMEOUT. Failure detection is tested this
 * way, with no fault. Host-only state change. */
mok_status mok_test_withhold_signal(mok_ctx_t ctx, int on);

/* Routing and schedule on the device ([S] "Das Scheduling"; [C] "Escolha da direcao").
 *   x [T][H] bf16; Wr [H][E] fp32; logit_bias [E] fp32 or NULL.
 * With dims.router = 1, writes topk_idx and gates (softmax of x Wr + bias, top-k, gates
 * renormalised over the k chosen experts; ties go to the lower expert id). With
 * dims.router = 0, x/Wr/logit_bias must be NULL and sched->topk_idx, sched->gates are
 * inputs. Then, with no sort, writes counts, offsets, table, inv and the aux data.
 * Deterministic: depends only on topk_idx. */
mok_status mok_plan(mok_ctx_t ctx, const void* x, const float* Wr, const float* logit_bias,
                    mok_sched* sched, void* workspace, void* stream);

/* Forward: y [T][H] (bf16, or fp32 per mok_set_output_dtype) = sum_j gates[t][j] *
 * FFN_{topk_idx[t][j]}(x[t]) (+ shared expert), FFN_e(v) = (silu(v W_gate[e]) *
 * (v W_up[e])) W_down[e]; the GEMMs take bf16 (or MXFP8) operands with fp32 accumulation,
 * h is rounded to the operand format, each expert output row to the output type, and the
 * k terms are added in slot order in fp32. `saved` (mok_sizes.saved_bytes) receives what
 * mok_moe_bwd needs; it must stay untouched until then. */
mok_status mok_moe_fwd(mok_ctx_t ctx, const mok_sched* sched, const void* x,
                       const mok_weights* w, void* y, void* saved, void* workspace,
                       void* stream);

/* Backward for upstream gradient dY [T][H] bf16. Writes dX [T][H] (output type: routed
 * experts, shared expert and, when routing ran on the device, the router path, summed in
 * fp32 in slot order and rounded once) and `grads`.
 * Wr must be the router weight given to mok_plan (NULL when dims.router = 0). */
mok_status mok_moe_bwd(mok_ctx_t ctx, const mok_sched* sched, const void* x, const float* Wr,
                       const mok_weights* w, const void* saved, const void* dY, void* dX,
                       mok_grads* grads, void* workspace, void* stream);

/* MXFP8 copies of the routed expert weights in every layout the forward and backward
 * GEMMs read (blocks of 32 along H and along I), into w->mx. */
mok_status mok_quantize_weights_mxfp8(mok_ctx_t ctx, const mok_weights* w, void* mx_out,
                                      void* stream);

/* Synchronise `stream`, read and clear the device status word of `sched`. */
mok_status mok_get_status(mok_ctx_t ctx, const mok_sched* sched, void* stream);

/* Schedule construction that allocates nothing and takes no workspace. The articles have
 * no counterpart: this serves callers that cannot allocate device memory, e.g. code
 * embedded in a host runtime that owns every device allocation, or code that runs where
 * the allocator must not be called. They still pass inputs and outputs (sched, with
 * topk_idx and gates filled in by the caller, and aux), but not a workspace.
 *
 * Computes exactly what mok_plan computes for a context created with router = 0 (counts,
 * offsets, table, inv and the aux data, bitwise the same). Its scratch (per-block expert
 * histograms and slot ranks, (ceil(T/32)*E + T*k) * 4 bytes, the first part rounded up
 * to 256) lives in a fixed 4 MiB device array inside the library, which every GPU that
 * loads the library holds until the process exits. Larger problems return
 * MOK_ERR_UNSUPPORTED; contexts with router = 1 return MOK_ERR_INVALID_ARG.
 *
 * The first call on a device looks up that array's device address (with the device
 * current) and caches it with the CUDA context it belongs to; make that first call before
 * any stream capture. After a device reset the next call finds another context and looks
 * the address up again (make that call before any capture too). Every call
 * shares the one array: calls whose work overlaps on the GPU (other streams, other host
 * threads) race and must be serialised by the caller. No state carries over from one
 * call to the next: the scratch is fully rewritten before it is read. Does not call
 * cudaMalloc, cudaFree or any allocating routine. */
mok_status mok_plan_noalloc(mok_ctx_t ctx, mok_sched* sched, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* MOK_H_ */
