"""GPU parity of the whole layer through the C ABI against the fp64 oracle."""
import numpy as np
import pytest
import torch

import moe_inputs as mi
from grouped_gemm_built_gb300 import mok
from tests import gpu_util as gu
from tests import out_slack as osl

pytestmark = pytest.mark.gpu

CASES = {
    "tiny": mi.CONFIGS["tiny"],
    # ragged token count, shared expert, several 128-row tiles per expert
    "ragged_shared": mi.MoEConfig("ragged_shared", T=300, H=256, I=256, E=12, k=3,
                                  shared_I=128),
    # most experts empty (zero-row segments, zero dW)
    "sparse": mi.MoEConfig("sparse", T=64, H=128, I=128, E=64, k=1),
    "single_token": mi.MoEConfig("single_token", T=1, H=128, I=128, E=4, k=2),
    # routing supplied by the caller, a token may pick one expert twice
    "external_routing": mi.MoEConfig("external_routing", T=100, H=256, I=128, E=6, k=8,
                                     router=False, zipf_s=1.2, macrobatches=0),
    "mid": mi.CONFIGS["mid"],
    # weight-gradient GEMMs on single bf16 operands (compared with the flip allowance)
    "ragged_shared_plain": mi.MoEConfig("ragged_shared_plain", T=300, H=256, I=256, E=12, k=3,
                                        shared_I=128, precision="bf16_plain"),
    "mid_plain": mi.scaled(mi.CONFIGS["mid"], name="mid_plain", precision="bf16_plain"),
    "sparse_plain": mi.MoEConfig("sparse_plain", T=64, H=128, I=128, E=64, k=1,
                                 precision="bf16_plain"),
    # the largest expert count and top-k the library takes, Zipf(1.2) loads: a few busy
    # experts, hundreds with one row or none
    "max_experts": mi.MoEConfig("max_experts", T=200, H=128, I=128, E=512, k=8, router=False,
                                zipf_s=1.2, macrobatches=0),
    # degenerate: one expert, top-1 (a dense SwiGLU FFN with gate 1)
    "single_expert": mi.MoEConfig("single_expert", T=130, H=128, I=128, E=1, k=1),
    # degenerate: every token routed to every expert (k = E)
    "all_experts": mi.MoEConfig("all_experts", T=96, H=128, I=256, E=4, k=4, shared_I=128),
}


def _check_route_and_plan(cfg, inp, res, orc_idx, orc_gates, logits):
    if cfg.router:
        amb = set(gu.ambiguous_tokens(cfg, inp, logits).tolist())
        diff = np.where((res["topk_idx"] != orc_idx).any(axis=1))[0]
        bad = [t for t in diff if t not in amb]
        assert not bad, f"top-k differs outside near-ties: tokens {bad[:10]}"
        assert len(diff) == 0, f"near-tie tokens routed differently: {diff[:10]}"
        assert np.abs(res["gates"] - orc_gates).max() < 1e-4   # tensor-core sum order
        assert np.allclose(res["gates"].sum(1), 1.0, atol=1e-5)
    pl = gu.moe.plan(orc_idx, cfg.E)
    assert np.array_equal(res["counts"], pl.counts)
    assert np.array_equal(res["offsets"], pl.offsets)
    assert np.array_equal(res["table"], pl.table)
    assert np.array_equal(res["inv"], pl.inv)


RESULTS = ["y", "dX", "dW_up", "dW_gate", "dW_down", "dWs_up", "dWs_gate", "dWs_down"]


@pytest.mark.parametrize("out", ["bf16", "fp32"])
@pytest.mark.parametrize("name", list(CASES))
def test_layer_matches_oracle(name, out):
    """Every result against the oracle at the tolerance. With bf16 results the oracle
    rounds them too, and an element may land a bf16 step either side where a rounding
    midpoint lies within the propagated bound of the two values before rounding
    (tests/out_slack.py); the tolerance applies to what remains."""
    cfg = mi.scaled(CASES[name], out=out)
    inp = gu.gpu_inputs(cfg, seed=0)
    idx, gates, logits = gu.oracle_route(cfg, inp)
    res, _ = gu.run_gpu(cfg, inp, backward=True)
    assert res["status"] == 0
    _check_route_and_plan(cfg, inp, res, idx, gates, logits)
    ref = gu.run_oracle(cfg, inp, idx, gates, backward=True)
    tol = gu.TOL[cfg.precision]
    fields = ["y", "dX", "dW_up", "dW_gate", "dW_down", "dgates"]
    if cfg.router:
        fields.append("dWr")
    if cfg.shared_I:
        fields += ["dWs_up", "dWs_gate", "dWs_down"]
    errs = {f: gu.rel_err(res[f], ref[f]) for f in fields}
    print(name, out, errs)
    if out == "bf16":
        slack = osl.layer_slack(cfg, inp, idx, gates, logits)
        for f in list(errs):
            if f in slack:
                errs[f] = gu.rel_err_slack(res[f], ref[f], slack[f])
        print(name, out, "with the rounding allowance:", errs)
    elif cfg.precision in ("bf16", "bf16_plain"):
        # U, V are kept as bf16 for the backward (and in bf16_plain du, dv, g*h are rounded
        # to bf16 before the weight-gradient GEMMs): values whose exact value sits within
        # the fp32 error bound of a rounding midpoint may round either way, and with few
        # rows per expert one such flip is visible in dW
        slack, frac = gu.bf16_flip_slack(cfg, inp, idx, gates)
        for f in list(errs):
            if f in slack:
                errs[f] = gu.rel_err_slack(res[f], ref[f], slack[f])
        print(name, f"with flip slack ({frac:.4f} of dW operands near a midpoint):", errs)
    # reported, not gated: the error against the unquantised fp64 layer (no rounding of h,
    # du, dv or the results), the quantisation's own effect included
    ref64 = gu.run_oracle(cfg, inp, idx, gates, backward=True, precision="fp64", out="fp32")
    print(name, out, "against unrounded fp64 (not gated):",
          {f: round(gu.rel_err(res[f], ref64[f]), 5) for f in fields})
    for f, e in errs.items():
        assert e <= tol, (f, e)


def test_plan_bit_exact_with_oracle_routing():
    """The schedule built on the GPU from the oracle's expert ids equals the oracle's."""
    cfg = mi.MoEConfig("plan_ext", T=999, H=128, I=128, E=37, k=5, router=False)
    inp = gu.gpu_inputs(cfg, seed=3)
    rng = np.random.default_rng(5)
    idx = np.stack([rng.choice(37, 5, replace=False) for _ in range(999)])
    idx[::7, 1] = idx[::7, 0]          # some tokens hit one expert twice
    g = rng.uniform(0.1, 1, idx.shape)
    g = g / g.sum(1, keepdims=True)
    res, _ = gu.run_gpu(cfg, inp, backward=False, routing=(idx, g))
    pl = gu.moe.plan(idx, cfg.E)
    for f in ("counts", "offsets", "table", "inv"):
        assert np.array_equal(res[f], getattr(pl, f)), f


@pytest.mark.parametrize("name,path", [("ragged_shared", "launches"),
                                       ("ragged_shared", "megakernel"),
                                       ("ragged_shared_mx", "megakernel")])
def test_bitwise_deterministic_over_10_runs(name, path):
    cfg = CASES.get(name) or MX_CASES[name]
    inp = gu.gpu_inputs(cfg, seed=1)
    L0 = gu.make_layer(cfg)
    L0.set_fwd_path(path)
    first, L = gu.run_gpu(cfg, inp, layer=L0)
    for _ in range(9):
        again, _ = gu.run_gpu(cfg, inp, layer=L)
        for f in ("y", "dX", "dW_up", "dW_gate", "dW_down", "dgates", "dWr", "dWs_up"):
            assert torch.equal(torch.as_tensor(first[f]), torch.as_tensor(again[f])), f


def test_bad_expert_id_is_flagged():
    cfg = mi.MoEConfig("bad_id", T=40, H=128, I=128, E=4, k=2, router=False)
    inp = gu.gpu_inputs(cfg)
    idx = np.zeros((40, 2), np.int64)
    idx[3, 1] = 9                       # out of range
    res, _ = gu.run_gpu(cfg, inp, backward=False, routing=(idx, np.full((40, 2), 0.5)))
    from grouped_gemm_built_gb300 import mok
    assert res["status"] == mok.MOK_ERR_DEVICE


# ----------------------------------------------------------------------------- MXFP8
MX_CASES = {
    "tiny_mx": mi.MoEConfig("tiny_mx", T=256, H=256, I=256, E=8, k=2, precision="mxfp8"),
    "biased_mx": mi.MoEConfig("biased_mx", T=512, H=512, I=256, E=16, k=4,
                              bias_experts=(0, 1, 2, 3), bias_value=3.0, precision="mxfp8"),
    "ep64_slice_small": mi.MoEConfig("ep64_slice_small", T=256, H=512, I=256, E=6, k=8,
                                     router=False, zipf_s=1.2, precision="mxfp8",
                                     backward=False),
    "ragged_shared_mx": mi.MoEConfig("ragged_shared_mx", T=300, H=256, I=256, E=12, k=3,
                                     shared_I=128, precision="mxfp8"),
    "max_experts_mx": mi.MoEConfig("max_experts_mx", T=128, H=256, I=256, E=512, k=8,
                                   router=False, zipf_s=1.2, macrobatches=0, precision="mxfp8"),
}


def test_mxfp8_weight_quantizer_is_bit_exact():
    from oracle import numerics as nu
    cfg = MX_CASES["tiny_mx"]
    inp = gu.gpu_inputs(cfg)
    L = gu.make_layer(cfg)
    d = gu.to_dev(inp)
    mx = L.quantize_weights(d["W_up"], d["W_gate"], d["W_down"]).cpu().numpy()
    E, H, I = cfg.E, cfg.H, cfg.I
    off = gu.mx_weight_offsets(E, H, I)
    for name, wname, K, N in (("up_h", "W_up", H, I), ("gate_h", "W_gate", H, I),
                              ("down_i", "W_down", I, H)):
        o, n = off[name]
        codes = mx[o:o + n].reshape(E, K, N)
        so, sn = off[name + "_sf"]
        scales = gu.unpack_atoms(mx[so:so + sn], E, K, N)
        rc, rs = nu.mx_quantize(gu.np64(inp[wname]), axis=1)
        assert np.array_equal(codes, rc), name
        assert np.array_equal(scales, rs), name + " scales"


@pytest.mark.parametrize("out", ["bf16", "fp32"])
@pytest.mark.parametrize("name", list(MX_CASES))
def test_mxfp8_layer_matches_oracle(name, out):
    """MXFP8 layer against the oracle. With an in-layer router, the GPU's gates come from
    fp32 logits and the oracle's from exact ones; in MXFP8 a gate scales du and g*h before
    they are quantised, and E4M3 codes are 2^-3 apart, so a 1e-5 gate difference flips
    codes near a rounding boundary that the two sides then decide differently. The router
    run therefore checks routing, y, dX and the router gradients; the weight gradients are
    compared in a second run that takes the oracle's routing (expert ids and fp32 gates)
    as its input, so both sides quantise the same values. With bf16 results each result
    element may also land one bf16 step either side of the oracle's (the value before its
    rounding is known only to the E4M3 operands' flips)."""
    cfg = mi.scaled(MX_CASES[name], out=out)
    inp = gu.gpu_inputs(cfg, seed=0)
    idx, gates, logits = gu.oracle_route(cfg, inp)
    res, _ = gu.run_gpu(cfg, inp, backward=cfg.backward)
    assert res["status"] == 0
    _check_route_and_plan(cfg, inp, res, idx, gates, logits)
    ref = gu.run_oracle(cfg, inp, idx, gates, backward=cfg.backward)
    fields = ["y"]
    dw = ["dW_up", "dW_gate", "dW_down"] + (["dWs_up", "dWs_gate", "dWs_down"] if cfg.shared_I
                                            else [])
    if cfg.backward:
        fields += ["dX", "dgates"] + (["dWr"] if cfg.router else dw)
    def cmp(gpu, r, f):
        if out == "bf16" and f in RESULTS:
            return gu.rel_err_slack(gpu[f], r[f], osl.bf16_spacing(r["unrounded"][f]))
        return gu.rel_err(gpu[f], r[f])
    errs = {f: cmp(res, ref, f) for f in fields}
    if cfg.backward and cfg.router:
        # weight gradients with the oracle's routing as the input
        ext = mi.scaled(cfg, router=False)
        g32 = gates.astype(np.float32)
        res2, _ = gu.run_gpu(ext, inp, backward=True, routing=(idx, g32))
        assert res2["status"] == 0
        ref2 = gu.run_oracle(ext, inp, idx, g32.astype(np.float64), backward=True)
        for f in ["y", "dX"] + dw:
            errs[f + " (oracle routing)"] = cmp(res2, ref2, f)
    print(name, out, errs)
    ref64 = gu.run_oracle(cfg, inp, idx, gates, backward=cfg.backward, precision="fp64",
                          out="fp32")
    print(name, out, "against unrounded fp64 (not gated):",
          {f: round(gu.rel_err(res[f], ref64[f]), 5) for f in fields})
    for f, e in errs.items():
        assert e <= gu.TOL["mxfp8"], (f, e)


@pytest.mark.parametrize("name,bias", [("mid", False), ("biased_mx", True)])
def test_router_logits_within_fp32_bound(name, bias):
    """The tensor-core router's logits (fp32 accumulation of exact bf16 x bf16-part
    products) stay inside the worst-case fp32 error bound of the exact logits."""
    cfg = CASES.get(name) or MX_CASES[name]
    inp = gu.gpu_inputs(cfg, seed=2)
    L = gu.make_layer(cfg)
    d = gu.to_dev(inp)
    L.plan(x=d["x"], Wr=d["Wr"], bias=d["bias"])
    torch.cuda.synchronize()
    assert L.status() == 0
    got = L.workspace[: cfg.T * cfg.E * 4].view(torch.float32).reshape(cfg.T, cfg.E)
    got = got.cpu().double().numpy()
    x, Wr = gu.np64(inp["x"]), gu.np64(inp["Wr"])
    exact = x @ Wr + (gu.np64(inp["bias"])[None, :] if inp["bias"] is not None else 0.0)
    bound = gu.logit_margins(cfg, inp, exact)
    ratio = np.abs(got - exact) / bound
    print(name, "max |err| / bound", float(ratio.max()))
    assert float(ratio.max()) <= 1.0


@pytest.mark.parametrize("E,k,bias", [(512, 8, True), (4, 4, False), (1, 1, False)])
def test_topk_of_gpu_logits_is_exact(E, k, bias):
    """The integer decision in the GPU's own precision: the oracle's top-k (same rule:
    larger logit first, equal logits in ascending expert order) of the router's fp32
    logits equals the GPU's expert ids on every token, at the largest expert count and
    top-k and at k = E and E = 1; gates agree to fp32 rounding; the schedule of those ids
    is the oracle's, bit for bit."""
    cfg = mi.MoEConfig(f"topk_{E}_{k}", T=300, H=256, I=128, E=E, k=k,
                       bias_experts=(0, 1, 2, 3) if bias else (), bias_value=1.0)
    inp = gu.gpu_inputs(cfg, seed=4)
    L = gu.make_layer(cfg)
    d = gu.to_dev(inp)
    L.plan(x=d["x"], Wr=d["Wr"], bias=d["bias"])
    torch.cuda.synchronize()
    assert L.status() == 0
    lg = L.workspace[: cfg.T * cfg.E * 4].view(torch.float32).reshape(cfg.T, cfg.E)
    lg = lg.cpu().double().numpy()
    x, Wr = gu.np64(inp["x"]), gu.np64(inp["Wr"])
    exact = x @ Wr + (gu.np64(inp["bias"])[None, :] if inp["bias"] is not None else 0.0)
    assert float((np.abs(lg - exact) / gu.logit_margins(cfg, inp, exact)).max()) <= 1.0
    idx, gates = gu.moe.select(lg, cfg.k)
    gi = L.topk_idx.cpu().numpy()
    assert np.array_equal(gi, idx)
    assert np.abs(L.gates.cpu().numpy() - gates).max() < 2e-6
    pl = gu.moe.plan(idx, cfg.E)
    for f in ("counts", "offsets", "table", "inv"):
        assert np.array_equal(getattr(L, f).cpu().numpy(), getattr(pl, f)), f


@pytest.mark.parametrize("name", ["ragged_shared", "tiny_mx"])
def test_split_invariance(name):
    """Every sum has a fixed order, so the results do not depend on how many SMs the
    persistent kernels spread their tiles over: 152 (all), 37 and 5 SMs give the same bits,
    and so does the forward megakernel with 1 or 3 gather SMs on 9 SMs, and so do tiles
    taken in a dynamic order (from a device counter) on all SMs and on 7, and tiles handed
    out by cluster launch control (which always spreads over every SM)."""
    cfg = CASES.get(name) or MX_CASES[name]
    inp = gu.gpu_inputs(cfg, seed=5)
    fields = ("y", "dX", "dW_up", "dW_gate", "dW_down", "dgates")
    ref = None
    for limit, path, comm, order in ((0, "launches", 0, 0), (37, "launches", 0, 0),
                                     (5, "launches", 0, 0), (9, "megakernel", 1, 0),
                                     (9, "megakernel", 3, 0), (0, "launches", 0, 1),
                                     (7, "launches", 0, 1), (0, "launches", 0, 2)):
        L = gu.make_layer(cfg)
        mok.mok_set_sm_limit(L.ctx, limit)
        L.set_fwd_path(path)
        mok.mok_set_comm_sms(L.ctx, comm)
        mok.mok_set_tile_order(L.ctx, order)
        res, _ = gu.run_gpu(cfg, inp, backward=True, layer=L)
        assert res["status"] == 0
        if ref is None:
            ref = res
            continue
        for f in fields:
            assert torch.equal(res[f], ref[f]), (limit, path, comm, order, f)


@pytest.mark.parametrize("name", ["mid", "mid_plain", "external_routing", "max_experts"])
def test_row_tile_pairs_keep_the_bits(name):
    """Row-tile pairs (one CTA runs two 128-row tiles of an expert against one weight tile,
    or the odd last tile alone) give the single-tile launches' bits in every tile order:
    each output row is the same fixed-order K sum. The cases have experts of one, two,
    three and more row tiles."""
    cfg = CASES[name]
    inp = gu.gpu_inputs(cfg, seed=8)
    fields = ("y", "dX", "dW_up", "dW_gate", "dW_down", "dgates")
    ref = None
    for pairs, order in ((mok.MOK_PAIRS_OFF, 0), (mok.MOK_PAIRS_ON, 0), (mok.MOK_PAIRS_ON, 1),
                         (mok.MOK_PAIRS_ON, 2)):
        L = gu.make_layer(cfg)
        mok.mok_set_row_pairs(L.ctx, pairs)
        mok.mok_set_tile_order(L.ctx, order)
        res, _ = gu.run_gpu(cfg, inp, backward=True, layer=L)
        assert res["status"] == 0
        if ref is None:
            ref = res
            continue
        for f in fields:
            assert torch.equal(res[f], ref[f]), (pairs, order, f)


SM_PAIR_CASES = {
    # dW rows in whole 256-row tiles in every weight-gradient launch (routed and shared)
    "even": mi.MoEConfig("smp_even", T=512, H=512, I=256, E=8, k=2, shared_I=256,
                         precision="bf16_plain"),
    # I = 384: the routed and shared dW_down launches (rows = I) fall back to single CTAs,
    # dW up/gate (rows = H) runs on pairs; ragged experts, some with no rows
    "odd_I": mi.MoEConfig("smp_odd", T=300, H=512, I=384, E=16, k=2, shared_I=384,
                          precision="bf16_plain"),
    # fp32 results, no shared expert
    "fp32": mi.MoEConfig("smp_f32", T=700, H=256, I=256, E=8, k=4, precision="bf16_plain",
                         out="fp32"),
}


@pytest.mark.parametrize("name", sorted(SM_PAIR_CASES))
def test_sm_pairs_keep_the_bits(name):
    """SM pairs (clusters of two CTAs sharing the M = 256 MMAs of the dH and weight-gradient
    GEMMs) give the single-CTA launches' results bit for bit: each output element is the
    same fixed-order K sum. Every eligible launch on pairs (ON), the routed ones only
    (AUTO), with an SM limit that leaves room for one pair, and with one SM (no pair fits:
    single CTAs). The layer against the oracle is covered by the cases of
    test_layer_matches_oracle, whose BF16 cases run on pairs by default."""
    cfg = SM_PAIR_CASES[name]
    inp = gu.gpu_inputs(cfg, seed=14)
    fields = ("dW_up", "dW_gate", "dW_down", "dX", "dgates", "dWr") + (
        ("dWs_up", "dWs_gate", "dWs_down") if cfg.shared_I else ())
    ref = None
    for pairs, limit in ((mok.MOK_SMPAIRS_OFF, 0), (mok.MOK_SMPAIRS_ON, 0),
                         (mok.MOK_SMPAIRS_AUTO, 0), (mok.MOK_SMPAIRS_ON, 2),
                         (mok.MOK_SMPAIRS_ON, 1)):
        L = gu.make_layer(cfg)
        mok.mok_set_sm_pairs(L.ctx, pairs)
        mok.mok_set_sm_limit(L.ctx, limit)
        res, _ = gu.run_gpu(cfg, inp, backward=True, layer=L)
        assert res["status"] == 0, (pairs, limit)
        if ref is None:
            ref = res
            continue
        for f in fields:
            assert torch.equal(res[f], ref[f]), (pairs, limit, f)


@pytest.mark.parametrize("shared_I", [128, 384])
def test_mxfp8_launches_carry_the_bf16_shared_expert(shared_I):
    """In MXFP8 the routed forward launches also run the BF16 shared expert's tiles
    (after the routed ones, with their own operands and stage layout). The shared expert's
    weight gradients, which read the U, V those tiles kept, equal bit for bit the BF16
    layer's, whose shared expert runs in launches of its own (both take hi/lo shared
    operands); the layer against the oracle is covered by ragged_shared_mx."""
    base = mi.scaled(MX_CASES["ragged_shared_mx"], shared_I=shared_I)
    inp = gu.gpu_inputs(base, seed=3)
    rm, _ = gu.run_gpu(base, inp)
    rb, _ = gu.run_gpu(mi.scaled(base, precision="bf16"), inp)
    assert rm["status"] == 0 and rb["status"] == 0
    for f in ("dWs_up", "dWs_gate", "dWs_down"):
        assert torch.equal(rm[f], rb[f]), f
    for order in (1, 2):   # the shared tiles in the dynamic and CLC tile orders
        L = gu.make_layer(base)
        mok.mok_set_tile_order(L.ctx, order)
        ro, _ = gu.run_gpu(base, inp, layer=L)
        assert ro["status"] == 0
        for f in ("y", "dX", "dWs_up", "dWs_gate", "dWs_down"):
            assert torch.equal(ro[f], rm[f]), (order, f)


@pytest.mark.parametrize("name", ["ragged_shared", "ragged_shared_plain", "ragged_shared_mx"])
def test_bf16_results_are_the_fp32_sums_rounded(name):
    """The weight gradients come out of the same fp32 accumulators in both result types:
    the bf16 ones are those fp32 values rounded to nearest even (torch's conversion), bit
    for bit; dgates and dWr do not depend on the result type."""
    base = CASES.get(name) or MX_CASES[name]
    inp = gu.gpu_inputs(base, seed=6)
    r32, _ = gu.run_gpu(mi.scaled(base, out="fp32"), inp)
    r16, _ = gu.run_gpu(mi.scaled(base, out="bf16"), inp)
    assert r32["status"] == 0 and r16["status"] == 0
    assert r16["y"].dtype == torch.bfloat16 and r32["y"].dtype == torch.float32
    for f in ("dW_up", "dW_gate", "dW_down", "dWs_up", "dWs_gate", "dWs_down"):
        assert torch.equal(r16[f], r32[f].to(torch.bfloat16)), f
    for f in ("dgates", "dWr"):
        assert torch.equal(r16[f], r32[f]), f
