"""The allowance for bf16 results (tests/out_slack.py): it admits a GPU-like result and
still rejects planted mistakes. Everything here runs on the CPU. The "GPU-like" side is an
fp32 emulation of the library's arithmetic with the library's rounding points (fp32 GEMM
sums, bf16 h, U and V kept as bf16 for the backward, bf16 du, dv for the dX GEMM, hi + lo
weight-gradient operands, bf16 expert output rows, routed dX rows and results, fp32
combines in slot order); the oracle side is
the fp64 oracle with bf16 results modelled (``out="bf16"``)."""
import numpy as np
import pytest

import moe_inputs as mi
from oracle import moe
from oracle.numerics import bf16_round
from tests import gpu_util as gu
from tests import out_slack as osl

F = np.float32


def _bf(a):
    return bf16_round(np.asarray(a, np.float64)).astype(F)


def _silu32(v):
    s = (1 / (1 + np.exp(-v.astype(F)))).astype(F)
    return s, (v * s).astype(F)


def emulate(cfg, inp, idx, mistake=None):
    """fp32 emulation of plan + forward + backward with bf16 results. ``idx``: the expert
    ids (the GPU's router picks the same sets on these inputs). Returns a dict of float64
    results like the GPU tests read them."""
    x = gu.np64(inp["x"]).astype(F)
    dY = gu.np64(inp["dY"]).astype(F)
    Wu, Wg, Wd = (gu.np64(inp[n]).astype(F) for n in ("W_up", "W_gate", "W_down"))
    T, H, k = cfg.T, cfg.H, cfg.k
    plain = cfg.precision == "bf16_plain"
    if cfg.router:
        Wr = gu.np64(inp["Wr"]).astype(F)
        lg = x @ Wr
        lS = np.take_along_axis(lg, idx, axis=1)
        p = np.exp(lS - lS.max(axis=1, keepdims=True)).astype(F)
        gates = (p / p.sum(axis=1, keepdims=True)).astype(F)
    else:
        gates = gu.np64(inp["gates"]).astype(F)
    if mistake == "dropped_gate":
        gates = np.ones_like(gates)
    pl = moe.plan(idx, cfg.E)
    R = T * k
    O = np.zeros((R, H), F)
    dXg = np.zeros((R, H), F)
    dg = np.zeros((T, k), F)
    res = {"dW_up": np.zeros(Wu.shape), "dW_gate": np.zeros(Wg.shape),
           "dW_down": np.zeros(Wd.shape)}
    dwu_raw = []
    emulate_dw_unrounded = np.zeros(Wu.shape)

    def ffn(X, dYr, g, A, B, C):
        U, V = X @ A, X @ B
        s, s0 = _silu32(V)
        h = _bf(s0 * U)
        Orow = _bf(h @ C)
        U, V = _bf(U), _bf(V)             # kept as bf16 for the backward
        s, s0 = _silu32(V)
        D = dYr @ C.T
        s1 = (s * (1 + V * (1 - s))).astype(F)
        hv = (s0 * U).astype(F)
        du = (g * D * s0).astype(F)
        dv = (g * D * U * s1).astype(F)
        if mistake == "dv_sign":
            dv = -dv
        hg = (g * hv).astype(F)
        dxr = _bf(_bf(du) @ A.T + _bf(dv) @ B.T)

        def op(v):
            if plain:
                return _bf(v)
            hi = _bf(v)
            return (hi + _bf(v - hi)).astype(F)
        dwu_raw.append(X.T @ op(du))
        dwu = _bf(dwu_raw[-1])
        dwg = _bf(X.T @ op(dv))
        dwd = _bf(op(hg).T @ dYr)
        return Orow, dxr, (D * hv).sum(axis=1, dtype=F), dwu, dwg, dwd

    for e in range(cfg.E):
        r0, r1 = pl.offsets[e], pl.offsets[e + 1]
        if r0 == r1:
            continue
        t, j = pl.table[r0:r1, 0], pl.table[r0:r1, 1]
        g = gates[t, j][:, None]
        O[r0:r1], dXg[r0:r1], dg[t, j], a, b, c = ffn(x[t], dY[t], g, Wu[e], Wg[e], Wd[e])
        res["dW_up"][e], res["dW_gate"][e], res["dW_down"][e] = a, b, c
        emulate_dw_unrounded[e] = dwu_raw[-1]
    y = np.zeros((T, H), F)
    dX = np.zeros((T, H), F)
    for jj in range(k):
        rows = pl.inv[:, jj]
        y = (gates[:, jj:jj + 1] * O[rows] + y).astype(F)
        dX = (dX + dXg[rows]).astype(F)
    if cfg.shared_I:
        Su, Sg, Sd = (gu.np64(inp[n]).astype(F) for n in ("Ws_up", "Ws_gate", "Ws_down"))
        Os, dXs, _, a, b, c = ffn(x, dY, np.ones((T, 1), F), Su, Sg, Sd)
        y = (y + Os).astype(F)
        dX = (dX + dXs).astype(F)
        res["dWs_up"], res["dWs_gate"], res["dWs_down"] = a, b, c
    if cfg.router:
        S = (gates * dg).sum(axis=1, keepdims=True, dtype=F)
        dl = (gates * (dg - S)).astype(F)
        for jj in range(k):
            dX = (dl[:, jj:jj + 1] * Wr[:, idx[:, jj]].T + dX).astype(F)
    res["y"] = _bf(y)
    res["dX"] = _bf(dX)
    if mistake == "scaled_row":
        e = int(np.argmax(pl.counts))
        res["dW_down"][e, 3] *= 1.05
    if mistake == "truncated_dw":     # rounding toward zero instead of to nearest
        raw = emulate_dw_unrounded
        m, ex = np.frexp(raw)
        res["dW_up"] = np.ldexp(np.trunc(np.ldexp(m, 8)), ex - 8)
    return {n: v.astype(np.float64) for n, v in res.items()}


CASES = {
    "ragged_shared": mi.MoEConfig("ragged_shared", T=300, H=256, I=256, E=12, k=3,
                                  shared_I=128),
    "sparse": mi.MoEConfig("sparse", T=64, H=128, I=128, E=64, k=1),
    "external": mi.MoEConfig("external", T=100, H=256, I=128, E=6, k=8, router=False,
                             zipf_s=1.2),
    "ragged_plain": mi.MoEConfig("ragged_plain", T=300, H=256, I=256, E=12, k=3,
                                 shared_I=128, precision="bf16_plain"),
}
FIELDS = ["y", "dX", "dW_up", "dW_gate", "dW_down"]


def _ref(cfg, inp):
    idx, gates, logits = gu.oracle_route(cfg, inp)
    ref = gu.run_oracle(cfg, inp, idx, gates, backward=True, out="bf16")
    return idx, gates, logits, ref


@pytest.mark.parametrize("name", list(CASES))
def test_allowance_admits_the_fp32_emulation(name):
    cfg = CASES[name]
    inp = gu.gpu_inputs(cfg, seed=0)
    idx, gates, logits, ref = _ref(cfg, inp)
    slack = osl.layer_slack(cfg, inp, idx, gates, logits)
    got = emulate(cfg, inp, idx)
    fields = FIELDS + (["dWs_up", "dWs_gate", "dWs_down"] if cfg.shared_I else [])
    for f in fields:
        rms = np.sqrt((ref[f] ** 2).mean())
        ex = gu.rel_err_slack(got[f], ref[f], slack[f])
        raw = gu.rel_err(got[f], ref[f])
        frac = float((slack[f] > 0).mean())
        print(name, f, f"raw {raw:.3g} with allowance {ex:.3g}, {frac:.4f} may flip")
        # the emulation's only departures are rounding flips the allowance admits, plus
        # small fp32 differences far below the tolerance
        assert ex <= 2e-3, f
        # (the bounds are conservative: most y and dX elements may flip)
        # the allowance is small: a bf16 spacing or so at the elements that may flip
        assert float(np.median(slack[f][slack[f] > 0]) / rms if frac else 0) < 0.1, f


@pytest.mark.parametrize("mistake,field", [("dv_sign", "dW_gate"), ("dropped_gate", "y"),
                                           ("scaled_row", "dW_down")])
def test_allowance_still_rejects_planted_mistakes(mistake, field):
    cfg = CASES["ragged_shared"]
    inp = gu.gpu_inputs(cfg, seed=0)
    idx, gates, logits, ref = _ref(cfg, inp)
    slack = osl.layer_slack(cfg, inp, idx, gates, logits)
    bad = emulate(cfg, inp, idx, mistake=mistake)
    assert gu.rel_err_slack(bad[field], ref[field], slack[field]) > gu.TOL["bf16"]


def test_allowance_catches_a_wrong_rounding_mode():
    """Rounding the weight gradients toward zero instead of to nearest moves about half of
    them by up to a bf16 spacing; where no midpoint lies within the bound, that is beyond
    the allowance, and the excess shows at many elements (the tolerance alone would not
    show it: a spacing is far below 2e-2 of the RMS at most elements). Routing is an
    input here, so the gates carry no router error."""
    cfg = CASES["external"]
    inp = gu.gpu_inputs(cfg, seed=0)
    idx, gates, logits, ref = _ref(cfg, inp)
    slack = osl.layer_slack(cfg, inp, idx, gates, logits)
    sp = osl.bf16_spacing(ref["dW_up"])
    good = emulate(cfg, inp, idx)
    bad = emulate(cfg, inp, idx, mistake="truncated_dw")
    ex_good = np.maximum(np.abs(good["dW_up"] - ref["dW_up"]) - slack["dW_up"], 0)
    ex_bad = np.maximum(np.abs(bad["dW_up"] - ref["dW_up"]) - slack["dW_up"], 0)
    assert float((ex_good > 0.25 * sp).mean()) < 1e-3
    assert float((ex_bad > 0.25 * sp).mean()) > 0.1


def test_flip_dev_and_spacing():
    assert osl.bf16_spacing(np.array([1.0]))[0] == 2.0 ** -7
    assert osl.bf16_spacing(np.array([-3.0]))[0] == 2.0 ** -6
    v = np.array([1.0, 1.0 + 2.0 ** -7])
    assert np.all(osl.flip_dev(v, np.full(2, 1e-6)) == 0)
    mid = np.array([1.0 + 2.0 ** -8])
    assert osl.flip_dev(mid, np.array([1e-9]))[0] == 2.0 ** -7


def test_oracle_bf16_results_are_rounded_unrounded_kept():
    cfg = CASES["ragged_shared"]
    inp = gu.gpu_inputs(cfg, seed=0)
    idx, gates, _, ref = _ref(cfg, inp)
    for f in ("y", "dX", "dW_up", "dWs_down"):
        assert np.array_equal(ref[f], bf16_round(ref[f])), f
        assert np.array_equal(ref[f], bf16_round(ref["unrounded"][f])), f
