// Host side of the C ABI declared in include/mok.h: argument checks, buffer layouts and
// the launch sequences of mok_plan, mok_moe_fwd and mok_moe_bwd.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <new>
#include <string>
#include <vector>

#include "../../include/mok_profile.h"

#include "mok_internal.h"

#define MOK_CHECK_CUDA(expr)                    \
  do {                                          \
    cudaError_t _e = (expr);                    \
    if (_e != cudaSuccess) return MOK_ERR_CUDA; \
  } while (0)

struct mok_ctx_s {
  mok_dims dims;
  mok::Dims d;
  mok_precision precision;
  mok_out_dtype out_dtype = MOK_OUT_BF16;
  mok_fwd_path fwd_path = MOK_FWD_AUTO;
  int comm_sms = 0;
  int sm_limit = 0;               // 0: every SM
  uint64_t wait_timeout_ns = 0;   // 0: the kernels' default (2 s)
  int withhold = 0;               // test hook of mok_test_withhold_signal
  mok_tile_order tile_order = MOK_TILES_STATIC;
  mok_row_pairs row_pairs = MOK_PAIRS_AUTO;
  mok_sm_pairs sm_pairs = MOK_SMPAIRS_AUTO;
  int* tcnt = nullptr;            // tile counters of the current call (dynamic order)
  int tcnt_used = 0;
  // the latest forward kept U, V (and the gathered rows) in the per-macrobatch padded
  // layout: the megakernel with more than one macrobatch
  bool fwd_cat = false;
  int device;
  int num_sms;
  // optional per-launch timing (mok_profile.h)
  bool profile = false;
  struct Rec {
    const char* name;
    cudaEvent_t a, b;
  };
  std::vector<Rec> recs;
  std::vector<cudaEvent_t> pool;
  size_t pool_used = 0;
  // megakernel phase stamps: kTraceSlots launches x num_sms CTAs x kTraceStamps
  unsigned long long* trace = nullptr;
  int trace_launches = 0;
  cudaEvent_t ev() {
    if (pool_used == pool.size()) {
      cudaEvent_t e;
      if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
      pool.push_back(e);
    }
    return pool[pool_used++];
  }
  ~mok_ctx_s() {
    for (auto e : pool) cudaEventDestroy(e);
  }
};
// SMs the context's kernels may use (persistent grids are sized to it)
static int launch_sms(mok_ctx_t ctx) {
  return ctx->sm_limit > 0 && ctx->sm_limit < ctx->num_sms ? ctx->sm_limit : ctx->num_sms;
}

// Row-tile pairs for the BF16 routed forward and dX GEMMs. Automatic: when the experts average
// more than one and at most two 128-row tiles of rows. There the launches stream weights
// (a weight tile meets 129..256 rows, below the tensor cores' ridge) and are bound by the
// bytes each SM keeps in flight; a pair tile streams its weight tile once into three stages
// of [A0 | B | A1] instead of two CTAs each keeping four [A | B] stages, half of whose
// weight bytes the other CTA also requests. With more rows per expert the GEMMs are
// compute-bound and keep their two accumulators for overlapping the epilogue. The dH launch
// keeps single row tiles: a pair holds both accumulators through its long SwiGLU'
// epilogue, which measured 10% slower at the Kimi shape.
// experts that average more than one and at most two 128-row tiles of rows
static bool two_row_tiles(const mok::Dims& d) {
  const long long R = (long long)d.R, E = d.E;
  return R > 128 * E && R <= 256 * E;
}
static bool use_pairs(mok_ctx_t ctx) {
  if (ctx->row_pairs == MOK_PAIRS_ON) return true;
  if (ctx->row_pairs == MOK_PAIRS_OFF) return false;
  return two_row_tiles(ctx->d);
}

// SM pairs for the routed dH launch: a cluster takes a pair of an expert's row tiles, and
// an expert's odd last row tile leaves one of its two CTAs without rows. Automatic, like
// the row-tile pairs, where that is rare: at 384 rows per expert (three row tiles) the
// idle halves made dH 16% slower than single CTAs (0.199 to 0.231 ms), at about 171 rows
// it is 6% faster.
static bool use_dh_sm_pairs(mok_ctx_t ctx) {
  if (ctx->sm_pairs == MOK_SMPAIRS_ON) return true;
  if (ctx->sm_pairs == MOK_SMPAIRS_OFF) return false;
  return two_row_tiles(ctx->d);
}

// the context's bound on device waits and its tile order, applied to one GEMM call
// (ordered = false: the static order, for the router GEMM of mok_plan)
static mok::GemmCall timed(mok::GemmCall c, mok_ctx_t ctx, bool ordered = true) {
  c.timeout_ns = ctx->wait_timeout_ns;
  c.tile_counter = nullptr;
  if (ordered && ctx->tcnt && ctx->tcnt_used < mok::kTileCounters)
    c.tile_counter = ctx->tcnt + ctx->tcnt_used++;
  c.clc = ordered && ctx->tile_order == MOK_TILES_CLC;
  return c;
}
// start of a call's launches: its tile counters (zeroed here, one per GEMM launch)
static cudaError_t begin_counters(mok_ctx_t ctx, void* base, cudaStream_t s) {
  ctx->tcnt_used = 0;
  ctx->tcnt = nullptr;
  if (ctx->tile_order != MOK_TILES_DYNAMIC) return cudaSuccess;
  ctx->tcnt = static_cast<int*>(base);
  return cudaMemsetAsync(base, 0, sizeof(int) * mok::kTileCounters, s);
}

namespace {
// Run a launcher; when profiling, bracket it with two events on the launch stream.
template <class F>
cudaError_t prof_launch(mok_ctx_s* c, const char* name, cudaStream_t s, F&& f) {
  if (!c->profile) return f();
  cudaEvent_t a = c->ev(), b = c->ev();
  if (a) cudaEventRecord(a, s);
  cudaError_t e = f();
  if (b) cudaEventRecord(b, s);
  if (a && b) c->recs.push_back({name, a, b});
  return e;
}
}  // namespace
#define MOK_LAUNCH(name, expr) MOK_CHECK_CUDA(prof_launch(ctx, name, s, [&]() { return (expr); }))

namespace mok {

Dims make_dims(const mok_dims& x, int num_sms) {
  Dims d;
  d.T = x.T;
  d.H = x.H;
  d.I = x.I;
  d.E = x.E;
  d.k = x.k;
  d.Is = x.shared_I;
  d.router = x.router;
  d.R = x.T * x.k;
  d.P_max = (int)align_up((size_t)d.R + (size_t)d.E * (kRowPad - 1), kRowPad);
  d.mt_max = d.P_max / kRowPad;
  d.nblk = (x.T + kTokBlock - 1) / kTokBlock;
  // macrobatches: Tm tokens each, a multiple of 128 (so a macrobatch is whole histogram
  // blocks and whole 128-token tiles); 0 means one. By tokens: minibatch_tokens, or the
  // two-wave rule at the device's SM count.
  if (x.minibatch_tokens != 0) {
    int tok = x.minibatch_tokens;
    if (tok < 0) tok = num_sms > 0 ? mok_minibatch_tokens(x.H, x.I, x.k, num_sms) : x.T;
    d.Tm = (int)align_up((size_t)std::max(tok, 1), kRowPad);
  } else {
    const int want = x.macrobatches > 0 ? x.macrobatches : 1;
    d.Tm = (int)align_up((size_t)((x.T + want - 1) / want), kRowPad);
  }
  d.M = (x.T + d.Tm - 1) / d.Tm;
  const long long rows_m = (long long)std::min(d.Tm, x.T) * x.k;
  d.mt_m_max = (int)((rows_m + (long long)std::min<long long>(x.E, rows_m) * (kRowPad - 1) +
                      kRowPad - 1) / kRowPad);
  d.P_slot = d.mt_m_max * kRowPad;
  d.P_cat = (int)align_up((size_t)d.R + (size_t)d.E * (kRowPad - 1) * d.M, kRowPad);
  if (d.M == 1) d.P_cat = std::max(d.P_cat, d.P_max);
  // ring slots: as many as ring_bytes holds at bf16 (the larger row format), at most M
  const size_t slot_bytes = (size_t)d.P_slot * d.H * 2;
  d.S = d.M;
  if (x.ring_bytes > 0) d.S = (int)std::min<size_t>((size_t)d.M, x.ring_bytes / slot_bytes);
  return d;
}

namespace {
struct Bump {
  size_t off = 0;
  size_t take(size_t bytes) {
    size_t o = off;
    off = align_up(off + bytes, 256);
    return o;
  }
};
}  // namespace

AuxLayout aux_layout(const Dims& d) {
  Bump b;
  AuxLayout L;
  L.status = b.take(sizeof(uint32_t));
  L.poff = b.take(sizeof(int32_t) * (d.E + 1));
  L.tile_expert = b.take(sizeof(int32_t) * d.mt_max);
  L.num_mtiles = b.take(sizeof(int32_t));
  L.mstart = b.take(sizeof(int32_t) * (size_t)d.M * d.E);
  L.mcount = b.take(sizeof(int32_t) * (size_t)d.M * d.E);
  L.mpoff = b.take(sizeof(int32_t) * (size_t)d.M * (d.E + 1));
  L.mtile_expert = b.take(sizeof(int32_t) * (size_t)d.M * d.mt_m_max);
  L.mtiles = b.take(sizeof(int32_t) * (size_t)d.M);
  L.mrow0 = b.take(sizeof(int32_t) * (size_t)(d.M + 1));
  L.ptile = b.take(sizeof(int32_t) * (size_t)max_ptiles(d));
  L.num_ptiles = b.take(sizeof(int32_t));
  L.dwr_q0 = b.take(sizeof(int32_t) * (size_t)(d.E + 1));
  L.dwr_item_e = b.take(sizeof(int32_t) * (size_t)dwr_items_max(d));
  L.total = b.off;
  return L;
}

PlanWs plan_ws(const Dims& d) {
  Bump b;
  PlanWs L;
  L.logits = b.take(sizeof(float) * (size_t)d.T * d.E);
  L.hist = b.take(sizeof(int32_t) * (size_t)d.nblk * d.E);
  L.lrank = b.take(sizeof(int32_t) * (size_t)d.R);
  L.wr3 = d.router ? b.take(2 * 3 * (size_t)d.H * router_ld(d)) : b.off;
  L.total = b.off;
  return L;
}

FwdWs fwd_ws(const Dims& d) {
  Bump b;
  FwdWs L;
  const size_t P = d.P_cat;
  L.h = b.take(2 * P * d.I);
  L.o = b.take(4 * P * d.H);
  L.hs = b.take(2 * (size_t)d.T * d.Is);
  L.os = b.take(4 * (size_t)d.T * d.H);
  L.xq = b.take(P * d.H);
  L.xsf = b.take(P * d.H / 32);
  L.hq = b.take(P * d.I);
  L.hsf = b.take(P * d.I / 32);
  L.ring = b.take((size_t)d.S * d.P_slot * d.H * 2);
  L.ring_sf = b.take((size_t)d.S * d.P_slot * d.H / 32);
  L.cnt = b.take(sizeof(int) * (size_t)mega_cnt(d).total);
  L.tcnt = b.take(sizeof(int) * kTileCounters);
  L.total = b.off;
  return L;
}

MxWeights mx_weights_layout(const Dims& d) {
  Bump b;
  MxWeights L;
  const size_t n = (size_t)d.E * d.H * d.I;
  L.up_h = b.take(n);
  L.up_h_sf = b.take(n / 32);
  L.gate_h = b.take(n);
  L.gate_h_sf = b.take(n / 32);
  L.down_i = b.take(n);
  L.down_i_sf = b.take(n / 32);
  L.down_h = b.take(n);
  L.down_h_sf = b.take(n / 32);
  L.up_i = b.take(n);
  L.up_i_sf = b.take(n / 32);
  L.gate_i = b.take(n);
  L.gate_i_sf = b.take(n / 32);
  L.total = b.off;
  return L;
}

BwdWs bwd_ws(const Dims& d) {
  Bump b;
  BwdWs L;
  const size_t P = d.P_max;
  L.dyg = b.take(2 * P * d.H);
  L.du = b.take(2 * P * d.I);   // du, dv, g*h: bf16 hi parts ...
  L.dv = b.take(2 * P * d.I);
  L.hg = b.take(2 * P * d.I);
  L.du_lo = b.take(2 * P * d.I);  // ... and lo parts
  L.dv_lo = b.take(2 * P * d.I);
  L.hg_lo = b.take(2 * P * d.I);
  L.dxg = b.take(4 * P * d.H);
  L.dgp = b.take(sizeof(float) * P * gemm_dh_parts(d.I, true));   // the larger count
  L.dl = b.take(sizeof(float) * (size_t)d.R);
  L.dus = b.take(2 * (size_t)d.T * d.Is);
  L.dvs = b.take(2 * (size_t)d.T * d.Is);
  L.hsg = b.take(2 * (size_t)d.T * d.Is);
  L.dus_lo = b.take(2 * (size_t)d.T * d.Is);
  L.dvs_lo = b.take(2 * (size_t)d.T * d.Is);
  L.hsg_lo = b.take(2 * (size_t)d.T * d.Is);
  L.dxs = b.take(4 * (size_t)d.T * d.H + sizeof(float) * (size_t)d.E * d.H);  // + Wr^T
  L.q_dy_h = b.take(P * d.H);
  L.sf_dy_h = b.take(P * d.H / 32);
  L.q_dy_r = b.take(P * d.H);
  L.sf_dy_r = b.take(P * d.H / 32);
  L.q_x_r = b.take(P * d.H);
  L.sf_x_r = b.take(P * d.H / 32);
  L.q_du_i = b.take(P * d.I);
  L.sf_du_i = b.take(P * d.I / 32);
  L.q_dv_i = b.take(P * d.I);
  L.sf_dv_i = b.take(P * d.I / 32);
  L.q_du_r = b.take(P * d.I);
  L.sf_du_r = b.take(P * d.I / 32);
  L.q_dv_r = b.take(P * d.I);
  L.sf_dv_r = b.take(P * d.I / 32);
  L.q_hg_r = b.take(P * d.I);
  L.sf_hg_r = b.take(P * d.I / 32);
  // only after a multi-macrobatch megakernel forward
  L.uvmap = d.M > 1 ? b.take(sizeof(int32_t) * P) : b.off;
  L.xr = d.M > 1 ? b.take(2 * P * d.H) : b.off;
  L.tcnt = b.take(sizeof(int) * kTileCounters);
  L.dwr_part = d.router ? b.take(sizeof(float) * (size_t)dwr_items_max(d) * d.H) : b.off;
  L.total = b.off;
  return L;
}

SavedLayout saved_layout(const Dims& d) {
  Bump b;
  SavedLayout L;
  const size_t P = d.P_cat;
  L.u = b.take(2 * P * d.I);   // U, V kept for the backward as bf16
  L.v = b.take(2 * P * d.I);
  L.us = b.take(2 * (size_t)d.T * d.Is);
  L.vs = b.take(2 * (size_t)d.T * d.Is);
  L.xg = b.take(2 * P * d.H);
  L.total = b.off;
  return L;
}

}  // namespace mok

namespace mok {
const Dims* ctx_dims(mok_ctx_t ctx) { return ctx ? &ctx->d : nullptr; }
int ctx_num_sms(mok_ctx_t ctx) { return ctx ? ctx->num_sms : 0; }
}  // namespace mok

using namespace mok;

namespace {

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

mok_status check_sched(const Dims& d, const mok_sched* s) {
  if (!s || !s->topk_idx || !s->gates || !s->counts || !s->offsets || !s->table || !s->inv)
    return MOK_ERR_INVALID_ARG;
  if (!s->aux || !aligned(s->aux, 256)) return MOK_ERR_WORKSPACE;
  (void)d;
  return MOK_OK;
}

char* at(void* base, size_t off) { return static_cast<char*>(base) + off; }

const char* gemm_name(const GemmCall& c) {
  static const char* routed[] = {"gemm_fwd_upgate_swiglu", "gemm_fwd_down", "gemm_bwd_dh_swiglu",
                                 "gemm_bwd_dx", "gemm_bwd_dw_down", "gemm_bwd_dw_upgate"};
  static const char* dense[] = {"shared_fwd_upgate_swiglu", "shared_fwd_down",
                                "shared_bwd_dh_swiglu", "shared_bwd_dx", "shared_bwd_dw_down",
                                "shared_bwd_dw_upgate"};
  return c.dense ? dense[c.mode] : routed[c.mode];
}

}  // namespace

extern "C" {

const char* mok_status_string(mok_status s) {
  switch (s) {
    case MOK_OK: return "ok";
    case MOK_ERR_INVALID_ARG: return "invalid argument";
    case MOK_ERR_UNSUPPORTED: return "unsupported";
    case MOK_ERR_WORKSPACE: return "workspace missing or misaligned";
    case MOK_ERR_CUDA: return "CUDA error";
    case MOK_ERR_TIMEOUT: return "device wait timed out";
    case MOK_ERR_DEVICE: return "device flagged bad data";
  }
  return "unknown status";
}

int mok_minibatch_tokens(int H, int I, int k, int num_sms) {
  // Two full waves: every SM takes one 64-row slice of a grouped-GEMM tile per wave, so a
  // minibatch must route at least 2 * num_sms * 64 rows, i.e. ceil(that / k) tokens.
  if (H <= 0 || I <= 0 || k <= 0 || num_sms <= 0) return -1;
  const long rows = 2L * num_sms * 64;
  return (int)((rows + k - 1) / k);
}

mok_status mok_create(const mok_dims* dims, mok_ctx_t* out) {
  if (!dims || !out) return MOK_ERR_INVALID_ARG;
  *out = nullptr;
  const mok_dims& x = *dims;
  if (x.T < 1 || x.H < 128 || x.I < 128 || x.E < 1 || x.k < 1) return MOK_ERR_INVALID_ARG;
  if (x.H % 128 || x.I % 128) return MOK_ERR_INVALID_ARG;
  if (x.E > kMaxE || x.k > kMaxK) return MOK_ERR_INVALID_ARG;
  if (x.router && x.k > x.E) return MOK_ERR_INVALID_ARG;
  if (x.shared_I < 0 || (x.shared_I % 128) != 0) return MOK_ERR_INVALID_ARG;
  if (x.router != 0 && x.router != 1) return MOK_ERR_INVALID_ARG;
  if (x.macrobatches < 0) return MOK_ERR_INVALID_ARG;
  if (x.minibatch_tokens < -1 || (x.minibatch_tokens != 0 && x.macrobatches > 0))
    return MOK_ERR_INVALID_ARG;
  if ((long long)x.T * x.k + (long long)x.E * 127 > (1LL << 30)) return MOK_ERR_INVALID_ARG;
  if ((long long)x.E * x.H > (1LL << 31) || (long long)x.E * x.I > (1LL << 31))
    return MOK_ERR_INVALID_ARG;
  mok_ctx_s* c = new (std::nothrow) mok_ctx_s;
  if (!c) return MOK_ERR_INVALID_ARG;
  c->dims = x;
  c->precision = MOK_BF16;
  // Without a usable device the context still answers the host-only queries
  // (mok_get_sizes); every call that launches work then returns MOK_ERR_CUDA.
  c->device = -1;
  c->num_sms = 0;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) == cudaSuccess &&
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess) {
    c->device = dev;
    c->num_sms = sms;
  } else {
    cudaGetLastError();
  }
  c->d = make_dims(x, c->num_sms);
  if (c->d.S < 1) {   // ring_bytes below one slot
    delete c;
    return MOK_ERR_INVALID_ARG;
  }
  *out = c;
  return MOK_OK;
}

void mok_destroy(mok_ctx_t ctx) {
  if (ctx && ctx->trace) cudaFree(ctx->trace);
  delete ctx;
}

mok_status mok_set_precision(mok_ctx_t ctx, mok_precision p) {
  if (!ctx) return MOK_ERR_INVALID_ARG;
  if (p != MOK_BF16 && p != MOK_MXFP8 && p != MOK_BF16_WGRAD_PLAIN) return MOK_ERR_INVALID_ARG;
  ctx->precision = p;
  return MOK_OK;
}

mok_status mok_set_tile_order(mok_ctx_t ctx, mok_tile_order order) {
  if (!ctx) return MOK_ERR_INVALID_ARG;
  if (order != MOK_TILES_STATIC && order != MOK_TILES_DYNAMIC && order != MOK_TILES_CLC)
    return MOK_ERR_INVALID_ARG;
  ctx->tile_order = order;
  return MOK_OK;
}

mok_status mok_set_sm_pairs(mok_ctx_t ctx, mok_sm_pairs mode) {
  if (!ctx) return MOK_ERR_INVALID_ARG;
  if (mode != MOK_SMPAIRS_AUTO && mode != MOK_SMPAIRS_ON && mode != MOK_SMPAIRS_OFF)
    return MOK_ERR_INVALID_ARG;
  ctx->sm_pairs = mode;
  return MOK_OK;
}

mok_status mok_set_row_pairs(mok_ctx_t ctx, mok_row_pairs mode) {
  if (!ctx) return MOK_ERR_INVALID_ARG;
  if (mode != MOK_PAIRS_AUTO && mode != MOK_PAIRS_ON && mode != MOK_PAIRS_OFF)
    return MOK_ERR_INVALID_ARG;
  ctx->row_pairs = mode;
  return MOK_OK;
}

mok_status mok_set_output_dtype(mok_ctx_t ctx, mok_out_dtype t) {
  if (!ctx) return MOK_ERR_INVALID_ARG;
  if (t != MOK_OUT_BF16 && t != MOK_OUT_F32) return MOK_ERR_INVALID_ARG;
  ctx->out_dtype = t;
  return MOK_OK;
}

mok_status mok_set_fwd_path(mok_ctx_t ctx, mok_fwd_path path) {
  if (!ctx) return MOK_ERR_INVALID_ARG;
  if (path != MOK_FWD_MEGAKERNEL && path != MOK_FWD_LAUNCHES && path != MOK_FWD_AUTO)
    return MOK_ERR_INVALID_ARG;
  ctx->fwd_path = path;
  return MOK_OK;
}

mok_status mok_set_wait_timeout(mok_ctx_t ctx, uint64_t ns) {
  if (!ctx || ns > 60000000000ull) return MOK_ERR_INVALID_ARG;
  ctx->wait_timeout_ns = ns;
  return MOK_OK;
}

mok_status mok_test_withhold_signal(mok_ctx_t ctx, int on) {
  if (!ctx) return MOK_ERR_INVALID_ARG;
  ctx->withhold = on ? 1 : 0;
  return MOK_OK;
}

mok_status mok_set_sm_limit(mok_ctx_t ctx, int n) {
  if (!ctx || n < 0) return MOK_ERR_INVALID_ARG;
  ctx->sm_limit = n;
  return MOK_OK;
}

mok_status mok_set_comm_sms(mok_ctx_t ctx, int n) {
  if (!ctx || n < 0) return MOK_ERR_INVALID_ARG;
  ctx->comm_sms = n;
  return MOK_OK;
}

mok_status mok_get_sizes(mok_ctx_t ctx, mok_sizes* out) {
  if (!ctx || !out) return MOK_ERR_INVALID_ARG;
  const Dims& d = ctx->d;
  out->aux_bytes = aux_layout(d).total;
  size_t ws = plan_ws(d).total;
  size_t f = fwd_ws(d).total, b = bwd_ws(d).total;
  if (f > ws) ws = f;
  if (b > ws) ws = b;
  out->workspace_bytes = ws;
  out->saved_bytes = saved_layout(d).total;
  out->mx_weight_bytes = mx_weights_layout(d).total;
  out->padded_rows_max = d.P_max;
  out->macrobatches = d.M;
  out->ring_slots = d.S;
  out->macrobatch_tokens = d.Tm;
  return MOK_OK;
}

mok_status mok_plan(mok_ctx_t ctx, const void* x, const float* Wr, const float* logit_bias,
                    mok_sched* sched, void* workspace, void* stream) {
  if (!ctx) return MOK_ERR_INVALID_ARG;
  const Dims& d = ctx->d;
  mok_status st = check_sched(d, sched);
  if (st != MOK_OK) return st;
  if (!workspace || !aligned(workspace, 256)) return MOK_ERR_WORKSPACE;
  if (d.router) {
    if (!x || !Wr || !aligned(x, 16)) return MOK_ERR_INVALID_ARG;
  } else if (x || Wr || logit_bias) {
    return MOK_ERR_INVALID_ARG;
  }
  if (ctx->num_sms <= 0) return MOK_ERR_CUDA;  // no usable device
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  ctx->tcnt = nullptr;   // the router GEMM takes the static tile order
  ctx->tcnt_used = 0;
  AuxPtrs a = aux_ptrs(d, sched->aux);
  PlanWs L = plan_ws(d);
  float* logits = reinterpret_cast<float*>(at(workspace, L.logits));
  int32_t* hist = reinterpret_cast<int32_t*>(at(workspace, L.hist));
  int32_t* lrank = reinterpret_cast<int32_t*>(at(workspace, L.lrank));
  MOK_CHECK_CUDA(cudaMemsetAsync(a.status, 0, sizeof(uint32_t), s));
  if (d.router) {
    // logits = x Wr (+ bias) on the tensor cores, Wr split exactly into three bf16 parts
    void* wr3 = at(workspace, L.wr3);
    MOK_LAUNCH("router_split", launch_split_wr(d, Wr, router_ld(d), wr3, s));
    GemmCall c;
    memset(&c, 0, sizeof(c));
    c.mode = kRouter;
    c.dense = true;
    c.M_rows = d.T;
    c.H = d.H;
    c.I = d.H;
    c.groups = 1;
    c.n_out = d.E;
    c.ld_b = router_ld(d);
    c.bias = logit_bias;
    c.a[0] = x;
    c.b[0] = wr3;
    c.out[0] = logits;
    c.status = a.status;
    MOK_LAUNCH("router_logits", launch_gemm(timed(c, ctx, false), launch_sms(ctx), s));
  }
  MOK_LAUNCH("topk_rank", launch_topk_rank(d, d.router ? logits : nullptr, sched->topk_idx,
                                            sched->gates, hist, lrank, a.status, s));
  MOK_LAUNCH("plan_scan", launch_plan_scan(d, hist, sched->counts, sched->offsets, a, s));
  MOK_LAUNCH("plan_macro", launch_plan_macro(d, hist, sched->counts, sched->offsets, a, s));
  MOK_LAUNCH("plan_scatter", launch_plan_scatter(d, sched->topk_idx, hist, lrank,
                                                  sched->offsets, sched->table, sched->inv, s));
  return MOK_OK;
}

static mok_status check_weights(const Dims& d, const mok_weights* w) {
  if (!w || !w->W_up || !w->W_gate || !w->W_down) return MOK_ERR_INVALID_ARG;
  if (!aligned(w->W_up, 16) || !aligned(w->W_gate, 16) || !aligned(w->W_down, 16))
    return MOK_ERR_INVALID_ARG;
  if (d.Is) {
    if (!w->Ws_up || !w->Ws_gate || !w->Ws_down) return MOK_ERR_INVALID_ARG;
    if (!aligned(w->Ws_up, 16) || !aligned(w->Ws_gate, 16) || !aligned(w->Ws_down, 16))
      return MOK_ERR_INVALID_ARG;
  }
  return MOK_OK;
}

// pair: the launch may run row-tile pairs (BF16 row-space modes; see use_pairs)
static GemmCall routed_call(const Dims& d, const mok_sched* sc, const AuxPtrs& a, GemmMode m,
                            bool pair = false) {
  GemmCall c;
  memset(&c, 0, sizeof(c));
  c.pair = pair;
  c.ptile = a.ptile;
  c.num_ptiles = a.num_ptiles;
  c.max_ptiles = max_ptiles(d);
  c.mode = m;
  c.M_rows = d.P_max;
  c.dense = false;
  c.H = d.H;
  c.I = d.I;
  c.groups = d.E;
  c.poff = a.poff;
  c.counts = sc->counts;
  c.offsets = sc->offsets;
  c.tile_expert = a.tile_expert;
  c.num_mtiles = a.num_mtiles;
  c.table = sc->table;
  c.gates = sc->gates;
  c.k = d.k;
  c.status = a.status;
  return c;
}

static GemmCall dense_call(const Dims& d, const AuxPtrs& a, GemmMode m) {
  GemmCall c;
  memset(&c, 0, sizeof(c));
  c.mode = m;
  c.M_rows = d.T;
  c.dense = true;
  c.H = d.H;
  c.I = d.Is;
  c.groups = 1;
  c.k = d.k;
  c.status = a.status;
  return c;
}

mok_status mok_moe_fwd(mok_ctx_t ctx, const mok_sched* sched, const void* x,
                       const mok_weights* w, void* y, void* saved, void* workspace,
                       void* stream) {
  if (!ctx) return MOK_ERR_INVALID_ARG;
  const Dims& d = ctx->d;
  mok_status st = check_sched(d, sched);
  if (st != MOK_OK) return st;
  if ((st = check_weights(d, w)) != MOK_OK) return st;
  if (ctx->precision == MOK_MXFP8 && (!w->mx || !aligned(w->mx, 256))) return MOK_ERR_INVALID_ARG;
  if (!x || !y || !aligned(x, 16) || !aligned(y, 16)) return MOK_ERR_INVALID_ARG;
  if (!workspace || !aligned(workspace, 256) || !saved || !aligned(saved, 256))
    return MOK_ERR_WORKSPACE;
  if (ctx->num_sms <= 0) return MOK_ERR_CUDA;  // no usable device
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  AuxPtrs a = aux_ptrs(d, sched->aux);
  FwdWs L = fwd_ws(d);
  SavedLayout S = saved_layout(d);
  auto W = [&](size_t off) -> void* { return at(workspace, off); };
  void* o = W(L.o);
  const bool mx = ctx->precision == MOK_MXFP8;
  const bool ob = ctx->out_dtype == MOK_OUT_BF16;   // O, Os, y in bf16
  MOK_CHECK_CUDA(begin_counters(ctx, W(L.tcnt), s));

  const bool mega = ctx->fwd_path == MOK_FWD_MEGAKERNEL;
  if (mega) {
    // shared expert first (BF16, dense launches); the megakernel's combine adds its output
    const void* os = nullptr;
    if (d.Is) {
      GemmCall cs = dense_call(d, a, kFwdUpGate);
      cs.a[0] = x;
      cs.b[0] = w->Ws_up;
      cs.b[1] = w->Ws_gate;
      cs.out[0] = W(L.hs);
      cs.out[1] = at(saved, S.us);
      cs.out[2] = at(saved, S.vs);
      MOK_LAUNCH(gemm_name(cs), launch_gemm(timed(cs, ctx), launch_sms(ctx), s));
      cs = dense_call(d, a, kFwdDown);
      cs.a[0] = W(L.hs);
      cs.b[0] = w->Ws_down;
      cs.out[0] = W(L.os);
      cs.out_bf16 = ob;
      MOK_LAUNCH(gemm_name(cs), launch_gemm(timed(cs, ctx), launch_sms(ctx), s));
      os = W(L.os);
    }
    MegaCall mc;
    memset(&mc, 0, sizeof(mc));
    mc.up = routed_call(d, sched, a, kFwdUpGate);
    mc.down = routed_call(d, sched, a, kFwdDown);
    mc.up.M_rows = mc.down.M_rows = d.P_cat;
    mc.down.out_bf16 = ob;
    mc.up.a_rows = d.S * d.P_slot;
    mc.up.mx = mc.down.mx = mx;
    // one macrobatch, BF16: the ring's only slot is the saved gathered rows, which the
    // backward reads again
    void* ring = (d.M == 1 && !mx) ? at(saved, S.xg) : W(L.ring);
    mc.up.a[0] = ring;
    mc.up.out[1] = at(saved, S.u);
    mc.up.out[2] = at(saved, S.v);
    mc.down.out[0] = o;
    if (!mx) {
      mc.up.b[0] = w->W_up;
      mc.up.b[1] = w->W_gate;
      mc.up.out[0] = W(L.h);
      mc.down.a[0] = W(L.h);
      mc.down.b[0] = w->W_down;
    } else {
      MxWeights M = mx_weights_layout(d);
      char* mxw = static_cast<char*>(const_cast<void*>(w->mx));
      mc.up.sfa = W(L.ring_sf);
      mc.up.b[0] = mxw + M.up_h;
      mc.up.b[1] = mxw + M.gate_h;
      mc.up.sfb0 = mxw + M.up_h_sf;
      mc.up.sfb1 = mxw + M.gate_h_sf;
      mc.up.out_q[0] = W(L.hq);
      mc.up.out_sf[0] = W(L.hsf);
      mc.down.a[0] = W(L.hq);
      mc.down.sfa = W(L.hsf);
      mc.down.b[0] = mxw + M.down_i;
      mc.down.sfb0 = mxw + M.down_i_sf;
    }
    if (ctx->comm_sms >= launch_sms(ctx)) return MOK_ERR_INVALID_ARG;
    mc.n_comm = ctx->comm_sms;
    mc.up.timeout_ns = mc.down.timeout_ns = ctx->wait_timeout_ns;
    mc.withhold = ctx->withhold;
    mc.M = d.M;
    mc.S = d.S;
    mc.P_slot = d.P_slot;
    mc.Tm = d.Tm;
    mc.T = d.T;
    mc.mt_m_max = d.mt_m_max;
    mc.mstart = a.mstart;
    mc.mcount = a.mcount;
    mc.mpoff = a.mpoff;
    mc.mtile_expert = a.mtile_expert;
    mc.mtiles = a.mtiles;
    mc.mrow0 = a.mrow0;
    mc.topk_idx = sched->topk_idx;
    mc.inv = sched->inv;
    mc.x = x;
    mc.ring = ring;
    mc.ring_sf = W(L.ring_sf);
    mc.O = o;
    mc.Os = os;
    mc.y = y;
    mc.cnt = reinterpret_cast<int*>(W(L.cnt));
    MOK_CHECK_CUDA(cudaMemsetAsync(mc.cnt, 0, sizeof(int) * (size_t)mega_cnt(d).total, s));
    if (ctx->profile && ctx->trace) {
      const size_t per = (size_t)ctx->num_sms * kTraceStamps;
      mc.trace = ctx->trace + (size_t)(ctx->trace_launches % kTraceSlots) * per;
      MOK_CHECK_CUDA(cudaMemsetAsync(mc.trace, 0, per * sizeof(unsigned long long), s));
      ++ctx->trace_launches;
    }
    MOK_LAUNCH(mx ? "fwd_megakernel_mxfp8" : "fwd_megakernel", launch_fwd_mega(mc, launch_sms(ctx), s));
    ctx->fwd_cat = d.M > 1;
    return MOK_OK;
  }

  if (!mx) {
    // dispatch: pull token rows into expert order through the table
    MOK_LAUNCH("dispatch_gather",
               launch_gather_rows(d, x, *sched, a, at(saved, S.xg), launch_sms(ctx), s));
    // grouped up|gate GEMM + SwiGLU (h bf16; U, V saved as bf16)
    GemmCall c = routed_call(d, sched, a, kFwdUpGate, use_pairs(ctx));
    c.a[0] = at(saved, S.xg);
    c.b[0] = w->W_up;
    c.b[1] = w->W_gate;
    c.out[0] = W(L.h);
    c.out[1] = at(saved, S.u);
    c.out[2] = at(saved, S.v);
    MOK_LAUNCH(gemm_name(c), launch_gemm(timed(c, ctx), launch_sms(ctx), s));
    // grouped down GEMM
    c = routed_call(d, sched, a, kFwdDown, use_pairs(ctx));
    c.a[0] = W(L.h);
    c.b[0] = w->W_down;
    c.out[0] = o;
    c.out_bf16 = ob;
    MOK_LAUNCH(gemm_name(c), launch_gemm(timed(c, ctx), launch_sms(ctx), s));
  } else {
    MxWeights M = mx_weights_layout(d);
    char* mxw = static_cast<char*>(const_cast<void*>(w->mx));
    // dispatch with MXFP8 quantisation along H fused in
    MOK_LAUNCH("dispatch_gather_mxfp8",
               launch_gather_quant(d, x, *sched, a, W(L.xq), W(L.xsf), launch_sms(ctx), s));
    GemmCall c = routed_call(d, sched, a, kFwdUpGate);
    c.mx = true;
    c.a[0] = W(L.xq);
    c.sfa = W(L.xsf);
    c.b[0] = mxw + M.up_h;
    c.b[1] = mxw + M.gate_h;
    c.sfb0 = mxw + M.up_h_sf;
    c.sfb1 = mxw + M.gate_h_sf;
    c.out_q[0] = W(L.hq);
    c.out_sf[0] = W(L.hsf);
    c.out[1] = at(saved, S.u);
    c.out[2] = at(saved, S.v);
    // the BF16 shared expert's tiles run in the same launches ([C] "Outras
    // caracteristicas": MXFP8 training with the shared expert in BF16)
    if (d.Is) {
      c.s_a = x;
      c.s_b[0] = w->Ws_up;
      c.s_b[1] = w->Ws_gate;
      c.s_out[0] = W(L.hs);
      c.s_out[1] = at(saved, S.us);
      c.s_out[2] = at(saved, S.vs);
      c.s_rows = d.T;
      c.s_I = d.Is;
    }
    MOK_LAUNCH(d.Is ? "gemm_fwd_upgate_swiglu_mxfp8_shared" : "gemm_fwd_upgate_swiglu_mxfp8",
               launch_gemm(timed(c, ctx), launch_sms(ctx), s));
    c = routed_call(d, sched, a, kFwdDown);
    c.mx = true;
    c.a[0] = W(L.hq);
    c.sfa = W(L.hsf);
    c.b[0] = mxw + M.down_i;
    c.sfb0 = mxw + M.down_i_sf;
    c.out[0] = o;
    c.out_bf16 = ob;
    if (d.Is) {
      c.s_a = W(L.hs);
      c.s_b[0] = w->Ws_down;
      c.s_out[0] = W(L.os);
      c.s_rows = d.T;
      c.s_I = d.Is;
    }
    MOK_LAUNCH(d.Is ? "gemm_fwd_down_mxfp8_shared" : "gemm_fwd_down_mxfp8",
               launch_gemm(timed(c, ctx), launch_sms(ctx), s));
  }
  const void* shared_out = nullptr;
  if (d.Is && mx) {
    shared_out = W(L.os);   // written by the MXFP8 launches above
  } else if (d.Is) {
    GemmCall cs = dense_call(d, a, kFwdUpGate);
    cs.a[0] = x;
    cs.b[0] = w->Ws_up;
    cs.b[1] = w->Ws_gate;
    cs.out[0] = W(L.hs);
    cs.out[1] = at(saved, S.us);
    cs.out[2] = at(saved, S.vs);
    MOK_LAUNCH(gemm_name(cs), launch_gemm(timed(cs, ctx), launch_sms(ctx), s));
    cs = dense_call(d, a, kFwdDown);
    cs.a[0] = W(L.hs);
    cs.b[0] = w->Ws_down;
    cs.out[0] = W(L.os);
    cs.out_bf16 = ob;
    MOK_LAUNCH(gemm_name(cs), launch_gemm(timed(cs, ctx), launch_sms(ctx), s));
    shared_out = W(L.os);
  }
  // weighted combine in slot order
  MOK_LAUNCH("combine", launch_combine(d, o, *sched, a, shared_out, true, ob, y, s));
  ctx->fwd_cat = false;
  return MOK_OK;
}

mok_status mok_moe_bwd(mok_ctx_t ctx, const mok_sched* sched, const void* x, const float* Wr,
                       const mok_weights* w, const void* saved, const void* dY, void* dX,
                       mok_grads* g, void* workspace, void* stream) {
  if (!ctx) return MOK_ERR_INVALID_ARG;
  const Dims& d = ctx->d;
  mok_status st = check_sched(d, sched);
  if (st != MOK_OK) return st;
  if ((st = check_weights(d, w)) != MOK_OK) return st;
  if (!x || !dY || !dX || !aligned(x, 16) || !aligned(dY, 16) || !aligned(dX, 16))
    return MOK_ERR_INVALID_ARG;
  if (!g || !g->dW_up || !g->dW_gate || !g->dW_down || !g->dgates) return MOK_ERR_INVALID_ARG;
  if (!aligned(g->dW_up, 16) || !aligned(g->dW_gate, 16) || !aligned(g->dW_down, 16))
    return MOK_ERR_INVALID_ARG;
  if (ctx->precision == MOK_MXFP8 && (!w->mx || !aligned(w->mx, 256))) return MOK_ERR_INVALID_ARG;
  if (d.router && (!Wr || !g->dWr)) return MOK_ERR_INVALID_ARG;
  if (!d.router && (Wr || g->dWr)) return MOK_ERR_INVALID_ARG;
  if (d.Is && (!g->dWs_up || !g->dWs_gate || !g->dWs_down)) return MOK_ERR_INVALID_ARG;
  if (!workspace || !aligned(workspace, 256) || !saved || !aligned(saved, 256))
    return MOK_ERR_WORKSPACE;
  if (ctx->num_sms <= 0) return MOK_ERR_CUDA;  // no usable device
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  AuxPtrs a = aux_ptrs(d, sched->aux);
  BwdWs L = bwd_ws(d);
  SavedLayout S = saved_layout(d);
  auto W = [&](size_t off) -> void* { return at(workspace, off); };
  MOK_CHECK_CUDA(begin_counters(ctx, W(L.tcnt), s));
  const void* su = at(const_cast<void*>(saved), S.u);   // U, V kept as bf16
  const void* sv = at(const_cast<void*>(saved), S.v);
  void* dxg = W(L.dxg);
  float* dgp = reinterpret_cast<float*>(W(L.dgp));
  float* dl = reinterpret_cast<float*>(W(L.dl));
  const bool mx = ctx->precision == MOK_MXFP8;
  const bool ob = ctx->out_dtype == MOK_OUT_BF16;   // dXg, dXs, dX and every dW in bf16
  const bool hilo = ctx->precision == MOK_BF16;  // dW operands as bf16 hi + lo pairs
  // After a megakernel forward over several macrobatches, U, V sit in the per-macrobatch
  // padded rows where the megakernel wrote them: the dH GEMM reads them there through a
  // row map (no copy). The gathered x rows of the weight gradients passed through the
  // ring, whose slots later macrobatches reuse: they are gathered again from x (the same
  // HBM bytes that reading resident ring slots would cost on one GPU).
  const int32_t* uvmap = nullptr;
  void* xrows = at(const_cast<void*>(saved), S.xg);
  if (ctx->fwd_cat) {
    int32_t* map = reinterpret_cast<int32_t*>(W(L.uvmap));
    MOK_LAUNCH("uv_rowmap", launch_uv_rowmap(d, *sched, a, map, s));
    uvmap = map;
    if (!mx) {
      xrows = W(L.xr);
      MOK_LAUNCH("replay_gather", launch_gather_rows(d, x, *sched, a, xrows, launch_sms(ctx), s));
    }
  }
  // the shared expert is BF16 in the MXFP8 mode too, with that mode's dW operands
  const bool hilo_s = ctx->precision != MOK_BF16_WGRAD_PLAIN;
  MxWeights M = mx_weights_layout(d);
  char* mxw = static_cast<char*>(const_cast<void*>(w->mx));

  if (!mx) {
    // reverse dispatch of dY through the table
    MOK_LAUNCH("reverse_dispatch_gather",
               launch_gather_rows(d, dY, *sched, a, W(L.dyg), launch_sms(ctx), s));
    // x's gathered rows come from the forward (saved), no replay
    // D = dYg W_down^T with SwiGLU' and the router-weight gradient fused in
    // (single row tiles: its long epilogue needs the second accumulator to overlap)
    GemmCall c = routed_call(d, sched, a, kBwdDH);
    c.a[0] = W(L.dyg);
    c.b[0] = w->W_down;
    c.u = su;
    c.v = sv;
    c.uv_row = uvmap;
    c.out[0] = W(L.du);
    c.out[2] = W(L.dv);
    c.out[4] = W(L.hg);
    if (hilo) {
      c.out[1] = W(L.du_lo);
      c.out[3] = W(L.dv_lo);
      c.out[5] = W(L.hg_lo);
    }
    c.dgp = dgp;
    c.smpair = use_dh_sm_pairs(ctx);
    MOK_LAUNCH(gemm_name(c), launch_gemm(timed(c, ctx), launch_sms(ctx), s));
    // dXg = du W_up^T + dv W_gate^T (bf16 du, dv)
    c = routed_call(d, sched, a, kBwdDX, use_pairs(ctx));
    c.a[0] = W(L.du);
    c.a[1] = W(L.dv);
    c.b[0] = w->W_up;
    c.b[1] = w->W_gate;
    c.out[0] = dxg;
    c.out_bf16 = ob;
    MOK_LAUNCH(gemm_name(c), launch_gemm(timed(c, ctx), launch_sms(ctx), s));
  } else {
    // reverse dispatch of dY (blocks along H for the dH GEMM, 32-row blocks for dW_down)
    // and replay of x (32-row blocks for dW_up / dW_gate), all through the table
    MOK_LAUNCH("reverse_dispatch_gather_mxfp8",
               launch_gather_quant(d, dY, *sched, a, W(L.q_dy_h), W(L.sf_dy_h), launch_sms(ctx), s));
    MOK_LAUNCH("reverse_dispatch_gather_rows_mxfp8",
               launch_gather_quant_rows(d, dY, *sched, a, W(L.q_dy_r), W(L.sf_dy_r),
                                        launch_sms(ctx), s));
    MOK_LAUNCH("replay_gather_rows_mxfp8",
               launch_gather_quant_rows(d, x, *sched, a, W(L.q_x_r), W(L.sf_x_r), launch_sms(ctx),
                                        s));
    GemmCall c = routed_call(d, sched, a, kBwdDH);
    c.mx = true;
    c.a[0] = W(L.q_dy_h);
    c.sfa = W(L.sf_dy_h);
    c.b[0] = mxw + M.down_h;
    c.sfb0 = mxw + M.down_h_sf;
    c.u = su;
    c.v = sv;
    c.uv_row = uvmap;
    c.out_q[0] = W(L.q_du_i);
    c.out_sf[0] = W(L.sf_du_i);
    c.out_q[1] = W(L.q_dv_i);
    c.out_sf[1] = W(L.sf_dv_i);
    c.out_q[2] = W(L.q_du_r);
    c.out_sf[2] = W(L.sf_du_r);
    c.out_q[3] = W(L.q_dv_r);
    c.out_sf[3] = W(L.sf_dv_r);
    c.out_q[4] = W(L.q_hg_r);
    c.out_sf[4] = W(L.sf_hg_r);
    c.dgp = dgp;
    MOK_LAUNCH("gemm_bwd_dh_swiglu_mxfp8", launch_gemm(timed(c, ctx), launch_sms(ctx), s));
    c = routed_call(d, sched, a, kBwdDX);
    c.mx = true;
    c.a[0] = W(L.q_du_i);
    c.sfa = W(L.sf_du_i);
    c.a[1] = W(L.q_dv_i);
    c.sfa1 = W(L.sf_dv_i);
    c.b[0] = mxw + M.up_i;
    c.sfb0 = mxw + M.up_i_sf;
    c.b[1] = mxw + M.gate_i;
    c.sfb1 = mxw + M.gate_i_sf;
    c.out[0] = dxg;
    c.out_bf16 = ob;
    MOK_LAUNCH("gemm_bwd_dx_mxfp8", launch_gemm(timed(c, ctx), launch_sms(ctx), s));
  }
  // router-weight gradient and the renormalised-softmax backward
  MOK_LAUNCH("router_grad", launch_router_grad(d, dgp, gemm_dh_parts(d.I, mx), *sched, a,
                                              g->dgates, d.router ? dl : nullptr, s));
  const void* dxs = nullptr;
  if (d.Is) {
    GemmCall cs = dense_call(d, a, kBwdDH);
    cs.a[0] = dY;
    cs.b[0] = w->Ws_down;
    cs.u = at(const_cast<void*>(saved), S.us);
    cs.v = at(const_cast<void*>(saved), S.vs);
    cs.out[0] = W(L.dus);
    cs.out[2] = W(L.dvs);
    cs.out[4] = W(L.hsg);
    if (hilo_s) {
      cs.out[1] = W(L.dus_lo);
      cs.out[3] = W(L.dvs_lo);
      cs.out[5] = W(L.hsg_lo);
    }
    cs.smpair = ctx->sm_pairs == MOK_SMPAIRS_ON;   // shared expert: on request only
    MOK_LAUNCH(gemm_name(cs), launch_gemm(timed(cs, ctx), launch_sms(ctx), s));
    cs = dense_call(d, a, kBwdDX);
    cs.a[0] = W(L.dus);
    cs.a[1] = W(L.dvs);
    cs.b[0] = w->Ws_up;
    cs.b[1] = w->Ws_gate;
    cs.out[0] = W(L.dxs);
    cs.out_bf16 = ob;
    MOK_LAUNCH(gemm_name(cs), launch_gemm(timed(cs, ctx), launch_sms(ctx), s));
    dxs = W(L.dxs);
  }
  // dX: reverse combine in slot order (+ shared expert, + router path)
  float* wrt = reinterpret_cast<float*>(at(workspace, L.dxs + 4 * (size_t)d.T * d.H));
  if (d.router) MOK_LAUNCH("transpose_wr", launch_transpose_wr(d, Wr, wrt, s));
  MOK_LAUNCH("reverse_combine", launch_reverse_combine(d, dxg, *sched, a, dxs,
                                                       d.router ? dl : nullptr, wrt, ob, dX, s));
  // weight gradients, each a fixed-order sum over the expert's rows
  GemmCall c = routed_call(d, sched, a, kBwdDWUpGate);
  c.mx = mx;
  if (mx) {
    c.a[0] = W(L.q_x_r);
    c.b[0] = W(L.q_du_r);
    c.b[1] = W(L.q_dv_r);
    c.sfa = W(L.sf_x_r);
    c.sfb0 = W(L.sf_du_r);
    c.sfb1 = W(L.sf_dv_r);
  } else {
    c.a[0] = xrows;
    c.b[0] = W(L.du);
    c.b[1] = W(L.dv);
    if (hilo) {
      c.split = true;
      c.b[2] = W(L.du_lo);
      c.b[3] = W(L.dv_lo);
    }
  }
  c.out[0] = g->dW_up;
  c.out[1] = g->dW_gate;
  c.out_bf16 = ob;
  c.smpair = ctx->sm_pairs != MOK_SMPAIRS_OFF;
  MOK_LAUNCH(mx ? "gemm_bwd_dw_upgate_mxfp8" : gemm_name(c), launch_gemm(timed(c, ctx), launch_sms(ctx), s));
  c = routed_call(d, sched, a, kBwdDWDown);
  c.mx = mx;
  if (mx) {
    c.a[0] = W(L.q_hg_r);
    c.b[0] = W(L.q_dy_r);
    c.sfa = W(L.sf_hg_r);
    c.sfb0 = W(L.sf_dy_r);
  } else {
    c.a[0] = W(L.hg);
    c.b[0] = W(L.dyg);
    if (hilo) {
      c.split = true;
      c.a[1] = W(L.hg_lo);
    }
  }
  c.out[0] = g->dW_down;
  c.out_bf16 = ob;
  c.smpair = ctx->sm_pairs != MOK_SMPAIRS_OFF;
  MOK_LAUNCH(mx ? "gemm_bwd_dw_down_mxfp8" : gemm_name(c), launch_gemm(timed(c, ctx), launch_sms(ctx), s));
  if (d.Is) {
    GemmCall cs = dense_call(d, a, kBwdDWUpGate);
    cs.a[0] = x;
    cs.b[0] = W(L.dus);
    cs.b[1] = W(L.dvs);
    if (hilo_s) {
      cs.split = true;
      cs.b[2] = W(L.dus_lo);
      cs.b[3] = W(L.dvs_lo);
    }
    cs.out[0] = g->dWs_up;
    cs.out[1] = g->dWs_gate;
    cs.out_bf16 = ob;
    cs.smpair = ctx->sm_pairs == MOK_SMPAIRS_ON;   // shared expert: on request only
    MOK_LAUNCH(gemm_name(cs), launch_gemm(timed(cs, ctx), launch_sms(ctx), s));
    cs = dense_call(d, a, kBwdDWDown);
    cs.a[0] = W(L.hsg);
    cs.b[0] = dY;
    if (hilo_s) {
      cs.split = true;
      cs.a[1] = W(L.hsg_lo);
    }
    cs.out[0] = g->dWs_down;
    cs.out_bf16 = ob;
    cs.smpair = ctx->sm_pairs == MOK_SMPAIRS_ON;   // shared expert: on request only
    MOK_LAUNCH(gemm_name(cs), launch_gemm(timed(cs, ctx), launch_sms(ctx), s));
  }
  if (d.router)
    MOK_LAUNCH("router_dwr", launch_router_dwr(d, x, *sched, a, reinterpret_cast<float*>(W(L.dwr_part)),
                                               dl, g->dWr, s));
  return MOK_OK;
}

mok_status mok_quantize_weights_mxfp8(mok_ctx_t ctx, const mok_weights* w, void* mx_out,
                                      void* stream) {
  if (!ctx) return MOK_ERR_INVALID_ARG;
  const Dims& d = ctx->d;
  if (!w || !w->W_up || !w->W_gate || !w->W_down) return MOK_ERR_INVALID_ARG;
  if (!aligned(w->W_up, 16) || !aligned(w->W_gate, 16) || !aligned(w->W_down, 16))
    return MOK_ERR_INVALID_ARG;
  if (!mx_out || !aligned(mx_out, 256)) return MOK_ERR_INVALID_ARG;
  if (ctx->num_sms <= 0) return MOK_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  MxWeights M = mx_weights_layout(d);
  char* o = static_cast<char*>(mx_out);
  // W_up / W_gate [E][H][I]: blocks along H (the rows), atoms [e][H/128][I/128]
  MOK_LAUNCH("quant_w_up", launch_mx_quant(w->W_up, d.H, d.I, d.E, false, o + M.up_h,
                                           o + M.up_h_sf, d.I / 128, 1, s));
  MOK_LAUNCH("quant_w_gate", launch_mx_quant(w->W_gate, d.H, d.I, d.E, false, o + M.gate_h,
                                             o + M.gate_h_sf, d.I / 128, 1, s));
  // W_down [E][I][H]: blocks along I (the rows), atoms [e][I/128][H/128]
  MOK_LAUNCH("quant_w_down", launch_mx_quant(w->W_down, d.I, d.H, d.E, false, o + M.down_i,
                                             o + M.down_i_sf, d.H / 128, 1, s));
  // backward copies: W_down along H (dH GEMM, N = I), W_up / W_gate along I (dX GEMM,
  // N = H); atoms [e][K/128][N/128]
  MOK_LAUNCH("quant_w_down_h", launch_mx_quant(w->W_down, d.I, d.H, d.E, true, o + M.down_h,
                                               o + M.down_h_sf, d.I / 128, 1, s));
  MOK_LAUNCH("quant_w_up_i", launch_mx_quant(w->W_up, d.H, d.I, d.E, true, o + M.up_i,
                                             o + M.up_i_sf, d.H / 128, 1, s));
  MOK_LAUNCH("quant_w_gate_i", launch_mx_quant(w->W_gate, d.H, d.I, d.E, true, o + M.gate_i,
                                               o + M.gate_i_sf, d.H / 128, 1, s));
  return MOK_OK;
}

mok_status mok_get_status(mok_ctx_t ctx, const mok_sched* sched, void* stream) {
  if (!ctx || !sched || !sched->aux) return MOK_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  AuxPtrs a = aux_ptrs(ctx->d, sched->aux);
  uint32_t v = 0;
  MOK_CHECK_CUDA(cudaMemcpyAsync(&v, a.status, sizeof(v), cudaMemcpyDeviceToHost, s));
  MOK_CHECK_CUDA(cudaMemsetAsync(a.status, 0, sizeof(uint32_t), s));
  MOK_CHECK_CUDA(cudaStreamSynchronize(s));
  if (v & kErrTimeout) return MOK_ERR_TIMEOUT;
  if (v & kErrBadExpert) return MOK_ERR_DEVICE;
  return MOK_OK;
}

mok_status mok_profile_enable(mok_ctx_t ctx, int enable) {
  if (!ctx) return MOK_ERR_INVALID_ARG;
  ctx->profile = enable != 0;
  ctx->recs.clear();
  ctx->pool_used = 0;
  ctx->trace_launches = 0;
  if (ctx->profile && !ctx->trace && ctx->num_sms > 0) {
    const size_t bytes = sizeof(unsigned long long) * kTraceSlots * ctx->num_sms * kTraceStamps;
    if (cudaMalloc(&ctx->trace, bytes) != cudaSuccess) {
      ctx->trace = nullptr;
      return MOK_ERR_CUDA;
    }
  }
  return MOK_OK;
}

namespace {
// Phase times of the recorded megakernel launches (ms, summed over launches), from the
// per-CTA stamps: gather = last gather SM done - first start; gemm = last GEMM SM done -
// first start; gemm_spread = last - first GEMM SM done (load imbalance); combine = last
// end - first final-combine start; total = last end - first start.
void megakernel_phases(mok_ctx_t ctx, std::string& out) {
  const int n = std::min(ctx->trace_launches, kTraceSlots);
  if (n <= 0 || !ctx->trace) return;
  const size_t per = (size_t)ctx->num_sms * kTraceStamps;
  std::vector<unsigned long long> h(per * n);
  if (cudaMemcpy(h.data(), ctx->trace, h.size() * sizeof(unsigned long long),
                 cudaMemcpyDeviceToHost) != cudaSuccess)
    return;
  const char* names[5] = {"gather", "gemm", "gemm_spread", "combine", "total"};
  double sum[5] = {0, 0, 0, 0, 0};
  for (int l = 0; l < n; ++l) {
    const unsigned long long* s = h.data() + per * l;
    unsigned long long t0 = ~0ull, comm_end = 0, gemm_end = 0, gemm_first = ~0ull,
                       comb0 = ~0ull, end = 0;
    for (int c = 0; c < ctx->num_sms; ++c) {
      const unsigned long long* x = s + (size_t)c * kTraceStamps;
      if (x[kStampStart]) t0 = std::min(t0, x[kStampStart]);
      comm_end = std::max(comm_end, x[kStampCommDone]);
      if (x[kStampGemmDone]) {
        gemm_end = std::max(gemm_end, x[kStampGemmDone]);
        gemm_first = std::min(gemm_first, x[kStampGemmDone]);
      }
      if (x[kStampCombine]) comb0 = std::min(comb0, x[kStampCombine]);
      end = std::max(end, x[kStampEnd]);
    }
    if (t0 == ~0ull || end == 0) continue;
    sum[0] += comm_end > t0 ? (comm_end - t0) * 1e-6 : 0.0;
    sum[1] += gemm_end > t0 ? (gemm_end - t0) * 1e-6 : 0.0;
    sum[2] += (gemm_first != ~0ull && gemm_end > gemm_first) ? (gemm_end - gemm_first) * 1e-6 : 0.0;
    sum[3] += (comb0 != ~0ull && end > comb0) ? (end - comb0) * 1e-6 : 0.0;
    sum[4] += (end - t0) * 1e-6;
  }
  for (int i = 0; i < 5; ++i) {
    char line[128];
    snprintf(line, sizeof(line), "fwd_megakernel:%s %d %.6f\n", names[i], n, sum[i]);
    out += line;
  }
}
}  // namespace

mok_status mok_profile_report(mok_ctx_t ctx, char* buf, size_t len, int* total_launches) {
  if (!ctx || !buf || len == 0) return MOK_ERR_INVALID_ARG;
  std::vector<std::string> names;
  std::vector<int> cnt;
  std::vector<double> ms;
  for (auto& r : ctx->recs) {
    if (cudaEventSynchronize(r.b) != cudaSuccess) return MOK_ERR_CUDA;
    float t = 0.f;
    if (cudaEventElapsedTime(&t, r.a, r.b) != cudaSuccess) return MOK_ERR_CUDA;
    size_t i = 0;
    while (i < names.size() && names[i] != r.name) ++i;
    if (i == names.size()) {
      names.push_back(r.name);
      cnt.push_back(0);
      ms.push_back(0.0);
    }
    cnt[i] += 1;
    ms[i] += t;
  }
  std::string out;
  for (size_t i = 0; i < names.size(); ++i) {
    char line[256];
    snprintf(line, sizeof(line), "%s %d %.6f\n", names[i].c_str(), cnt[i], ms[i]);
    out += line;
  }
  megakernel_phases(ctx, out);
  ctx->trace_launches = 0;
  size_t n = out.size() < len - 1 ? out.size() : len - 1;
  memcpy(buf, out.data(), n);
  buf[n] = 0;
  if (total_launches) *total_launches = (int)ctx->recs.size();
  ctx->recs.clear();
  ctx->pool_used = 0;
  return MOK_OK;
}

}  // extern "C"
