"""Pins of the layer oracle: brute force on tiny inputs, finite differences, invariants
and special cases (no GPU)."""
import math

import numpy as np
import pytest

import moe_inputs as mi
from oracle import moe
from oracle.numerics import silu


def small_problem(rng, T=12, H=16, I=8, E=5, k=2, shared=False, bias=False):
    x = rng.normal(0, 1, (T, H))
    Wr = rng.normal(0, 0.3, (H, E))
    b = rng.normal(0, 0.5, E) if bias else None
    Wu = rng.normal(0, 0.3, (E, H, I))
    Wg = rng.normal(0, 0.3, (E, H, I))
    Wd = rng.normal(0, 0.3, (E, I, H))
    sh = None
    if shared:
        sh = (rng.normal(0, 0.3, (H, 6)), rng.normal(0, 0.3, (H, 6)), rng.normal(0, 0.3, (6, H)))
    dY = rng.normal(0, 1, (T, H))
    return x, Wr, b, Wu, Wg, Wd, sh, dY


# ----------------------------------------------------------------------------- routing
def test_route_matches_python_brute_force(rng):
    x, Wr, b, *_ = small_problem(rng, T=20, E=7, k=3, bias=True)
    r = moe.route(x, Wr, 3, b)
    for t in range(20):
        logits = [math.fsum(x[t, h] * Wr[h, e] for h in range(x.shape[1])) + b[e]
                  for e in range(7)]
        m = max(logits)
        p = [math.exp(l - m) for l in logits]
        z = math.fsum(p)
        p = [v / z for v in p]
        chosen = sorted(range(7), key=lambda e: (-logits[e], e))[:3]
        assert list(r.idx[t]) == chosen
        zS = math.fsum(p[e] for e in chosen)
        assert np.allclose(r.gates[t], [p[e] / zS for e in chosen], rtol=1e-13, atol=0)


def test_route_ties_go_to_lower_expert():
    x = np.ones((1, 2))
    Wr = np.array([[1.0, 2.0, 2.0, 0.5, 2.0], [0.0, 0.0, 0.0, 0.0, 0.0]])
    r = moe.route(x, Wr, 3)
    assert list(r.idx[0]) == [1, 2, 4]
    assert np.allclose(r.gates[0], 1 / 3)


def test_route_invariants(rng):
    cfg = mi.CONFIGS["tiny"]
    inp = mi.make_inputs(cfg)
    r = moe.route(mi.to_f64(inp["x"]), mi.to_f64(inp["Wr"]), cfg.k)
    assert np.allclose(r.gates.sum(1), 1.0, atol=1e-14)
    assert np.all(np.diff(r.gates, axis=1) <= 0)          # slot order: descending gate
    assert np.all(r.gates > 0)
    assert np.all([len(set(row)) == cfg.k for row in r.idx])


# ----------------------------------------------------------------------------- schedule
@pytest.mark.parametrize("T,E,k", [(1, 1, 1), (7, 3, 2), (64, 8, 2), (33, 40, 6)])
def test_plan_matches_loops_and_invariants(rng, T, E, k):
    idx = np.stack([rng.choice(E, k, replace=k > E) for _ in range(T)])
    p = moe.plan(idx, E)
    q = moe.plan_loops(idx, E)
    for f in ("counts", "offsets", "table", "inv"):
        assert np.array_equal(getattr(p, f), getattr(q, f)), f
    R = T * k
    assert p.counts.sum() == R and p.offsets[-1] == R
    assert np.all(np.diff(p.offsets) >= 0)
    # every (t, j) appears exactly once; each token exactly k times
    pairs = {tuple(v) for v in p.table}
    assert len(pairs) == R
    assert np.all(np.bincount(p.table[:, 0], minlength=T) == k)
    # inverse of the table
    assert np.array_equal(p.inv[p.table[:, 0], p.table[:, 1]], np.arange(R))
    # rows of one expert hold that expert, in ascending (t, j)
    for e in range(E):
        seg = p.table[p.offsets[e]:p.offsets[e + 1]]
        assert np.all(idx[seg[:, 0], seg[:, 1]] == e)
        key = seg[:, 0] * k + seg[:, 1]
        assert np.all(np.diff(key) > 0)


def test_plan_duplicate_expert_in_one_token():
    idx = np.array([[2, 2, 0], [0, 2, 2]])
    p = moe.plan(idx, 3)
    assert list(p.counts) == [2, 0, 4]
    assert p.table.tolist() == [[0, 2], [1, 0], [0, 0], [0, 1], [1, 1], [1, 2]]


def test_zipf_counts_of_the_ep64_slice():
    c = mi.zipf_counts(16384, 6, 1.2)
    assert sum(c) == 16384
    w = np.arange(1, 7) ** -1.2
    assert np.all(np.abs(np.array(c) - 16384 * w / w.sum()) < 1.0)


# ----------------------------------------------------------------------------- forward
def test_forward_matches_per_token_brute_force(rng):
    x, Wr, b, Wu, Wg, Wd, _, _ = small_problem(rng, T=16, E=6, k=3)
    r = moe.route(x, Wr, 3)
    y, _ = moe.forward(x, r.idx, r.gates, Wu, Wg, Wd)
    for t in range(16):
        yt = moe.token_forward_bruteforce(x[t], r.idx[t], r.gates[t], Wu, Wg, Wd)
        assert np.allclose(y[t], yt, rtol=1e-12, atol=1e-12)


def test_forward_identity_experts_return_input(rng):
    """combine(dispatch(x)) = sum_j g_tj x_t = x_t when every expert is the identity."""
    x, Wr, _, Wu, Wg, Wd, _, _ = small_problem(rng, T=30, E=5, k=3)
    r = moe.route(x, Wr, 3)
    y, _ = moe.forward(x, r.idx, r.gates, Wu, Wg, Wd, expert_fn=lambda e, X: X)
    assert np.allclose(y, x, rtol=0, atol=1e-14)


def test_forward_single_expert_is_dense_swiglu(rng):
    x, _, _, Wu, Wg, Wd, _, _ = small_problem(rng, T=9, E=1, k=1)
    idx = np.zeros((9, 1), np.int64)
    g = np.ones((9, 1))
    y, _ = moe.forward(x, idx, g, Wu, Wg, Wd)
    u = np.einsum("th,hi->ti", x, Wu[0])
    v = np.einsum("th,hi->ti", x, Wg[0])
    dense = np.einsum("ti,ih->th", v / (1 + np.exp(-v)) * u, Wd[0])
    assert np.allclose(y, dense, rtol=1e-12, atol=1e-13)


def test_forward_is_linear_in_gates(rng):
    x, Wr, _, Wu, Wg, Wd, _, _ = small_problem(rng, T=10, E=4, k=2)
    r = moe.route(x, Wr, 2)
    y1, _ = moe.forward(x, r.idx, r.gates, Wu, Wg, Wd)
    y2, _ = moe.forward(x, r.idx, 2 * r.gates, Wu, Wg, Wd)
    assert np.allclose(y2, 2 * y1, rtol=1e-13, atol=1e-14)


def test_shared_expert_adds_dense_ffn(rng):
    x, Wr, _, Wu, Wg, Wd, sh, _ = small_problem(rng, T=8, E=3, k=1, shared=True)
    r = moe.route(x, Wr, 1)
    y0, _ = moe.forward(x, r.idx, r.gates, Wu, Wg, Wd)
    y1, _ = moe.forward(x, r.idx, r.gates, Wu, Wg, Wd, shared=sh)
    for t in range(8):
        u, v = x[t] @ sh[0], x[t] @ sh[1]
        assert np.allclose(y1[t] - y0[t], (silu(v) * u) @ sh[2], rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("mode,tol", [("bf16", 1e-2), ("bf16_plain", 1e-2), ("mxfp8", 1.5e-1)])
def test_rounded_modes_stay_near_fp64(mode, tol):
    """The rounding model only perturbs: rms(rounded - fp64) / rms(fp64) stays near the
    formats' unit roundoff (2^-9 for bf16, about 2^-4 per MXFP8 element)."""
    cfg = mi.CONFIGS["tiny"]
    inp = mi.make_inputs(cfg)
    x, Wr = mi.to_f64(inp["x"]), mi.to_f64(inp["Wr"])
    W = [mi.to_f64(inp[n]) for n in ("W_up", "W_gate", "W_down")]
    r = moe.route(x, Wr, cfg.k)
    y0, s0 = moe.forward(x, r.idx, r.gates, *W)
    y1, s1 = moe.forward(x, r.idx, r.gates, *W, precision=mode)
    def rel(a, b):
        return np.sqrt(((a - b) ** 2).mean()) / np.sqrt((a ** 2).mean())

    assert rel(y0, y1) < tol
    dY = mi.to_f64(inp["dY"])
    g0 = moe.backward(x, r.idx, r.gates, *W, s0, dY, Wr=Wr)
    g1 = moe.backward(x, r.idx, r.gates, *W, s1, dY, precision=mode, Wr=Wr)
    for f in ("dX", "dW_up", "dW_gate", "dW_down", "dgates", "dWr"):
        assert rel(getattr(g0, f), getattr(g1, f)) < tol, f


# ----------------------------------------------------------------------------- backward
def _fd_check(f, arr, grad, rng, n=12, eps=1e-6, rtol=1e-6):
    flat = arr.reshape(-1)
    gflat = grad.reshape(-1)
    picks = rng.choice(flat.size, size=min(n, flat.size), replace=False)
    scale = max(np.abs(gflat).max(), 1e-30)
    for i in picks:
        old = flat[i]
        flat[i] = old + eps
        lp = f()
        flat[i] = old - eps
        lm = f()
        flat[i] = old
        fd = (lp - lm) / (2 * eps)
        assert abs(fd - gflat[i]) <= rtol * scale + 1e-9 * abs(fd), (i, fd, gflat[i])


@pytest.mark.parametrize("shared,bias", [(False, False), (True, True)])
def test_backward_matches_finite_differences(rng, shared, bias):
    x, Wr, b, Wu, Wg, Wd, sh, dY = small_problem(rng, T=10, H=12, I=6, E=4, k=2,
                                                 shared=shared, bias=bias)
    r = moe.route(x, Wr, 2, b)
    S = r.idx.copy()
    y, saved = moe.forward(x, S, r.gates, Wu, Wg, Wd, shared=sh)
    g = moe.backward(x, S, r.gates, Wu, Wg, Wd, saved, dY, shared=sh, Wr=Wr)

    def L():
        return moe.layer_loss(x, Wr, b, S, Wu, Wg, Wd, dY, shared=sh)

    _fd_check(L, x, g.dX, rng)
    _fd_check(L, Wu, g.dW_up, rng)
    _fd_check(L, Wg, g.dW_gate, rng)
    _fd_check(L, Wd, g.dW_down, rng)
    _fd_check(L, Wr, g.dWr, rng)
    if shared:
        for arr, gr in zip(sh, (g.dWs_up, g.dWs_gate, g.dWs_down)):
            _fd_check(L, arr, gr, rng)


def test_dgates_match_finite_differences(rng):
    x, Wr, _, Wu, Wg, Wd, _, dY = small_problem(rng, T=8, E=4, k=3)
    r = moe.route(x, Wr, 3)
    gates = r.gates.copy()
    y, saved = moe.forward(x, r.idx, gates, Wu, Wg, Wd)
    g = moe.backward(x, r.idx, gates, Wu, Wg, Wd, saved, dY)

    def L():
        yy, _ = moe.forward(x, r.idx, gates, Wu, Wg, Wd)
        return float((yy * dY).sum())

    _fd_check(L, gates, g.dgates, rng, n=24)


def test_router_backward_invariants(rng):
    x, Wr, _, Wu, Wg, Wd, _, dY = small_problem(rng, T=15, E=6, k=3)
    r = moe.route(x, Wr, 3)
    dg = rng.normal(0, 1, r.gates.shape)
    dl, dWr, dx = moe.router_backward(x, Wr, r.idx, r.gates, dg)
    # softmax over S is shift invariant: the logit gradient sums to zero per token
    assert np.allclose(dl.sum(1), 0, atol=1e-14)
    # zero outside the selected set
    mask = np.zeros_like(dl, bool)
    np.put_along_axis(mask, r.idx, True, axis=1)
    assert np.all(dl[~mask] == 0)
    # dg equal on every slot of a token is a pure shift: no logit gradient
    dl2, _, _ = moe.router_backward(x, Wr, r.idx, r.gates, np.ones_like(dg) * 3.0)
    assert np.allclose(dl2, 0, atol=1e-14)


def test_backward_linear_in_dY(rng):
    x, Wr, _, Wu, Wg, Wd, _, dY = small_problem(rng, T=10, E=4, k=2)
    r = moe.route(x, Wr, 2)
    _, saved = moe.forward(x, r.idx, r.gates, Wu, Wg, Wd)
    g1 = moe.backward(x, r.idx, r.gates, Wu, Wg, Wd, saved, dY, Wr=Wr)
    g2 = moe.backward(x, r.idx, r.gates, Wu, Wg, Wd, saved, 2 * dY, Wr=Wr)
    for f in ("dX", "dW_up", "dW_gate", "dW_down", "dgates", "dWr"):
        assert np.allclose(getattr(g2, f), 2 * getattr(g1, f), rtol=1e-12, atol=1e-14)


def test_empty_experts_get_zero_gradients(rng):
    x, _, _, Wu, Wg, Wd, _, dY = small_problem(rng, T=6, E=5, k=1)
    idx = np.zeros((6, 1), np.int64)           # only expert 0 is used
    gates = np.ones((6, 1))
    _, saved = moe.forward(x, idx, gates, Wu, Wg, Wd)
    g = moe.backward(x, idx, gates, Wu, Wg, Wd, saved, dY)
    assert np.all(g.dW_up[1:] == 0) and np.all(g.dW_down[1:] == 0)
    assert np.abs(g.dW_up[0]).max() > 0


@pytest.mark.parametrize("out", ["fp32", "bf16"])
def test_sampled_evaluators_match_the_dense_oracle(rng, out):
    """Per-token and per-element evaluators (no table, no streaming) against the dense
    per-expert oracle, bf16 rounding model, shared expert and router path included; both
    result types (with bf16 results the values before the last rounding too)."""
    from oracle import sampled
    x, Wr, b, Wu, Wg, Wd, sh, dY = small_problem(rng, T=14, H=16, I=8, E=5, k=2, shared=True)
    r = moe.route(x, Wr, 2)
    y, saved = moe.forward(x, r.idx, r.gates, Wu, Wg, Wd, shared=sh, precision="bf16", out=out)
    g = moe.backward(x, r.idx, r.gates, Wu, Wg, Wd, saved, dY, shared=sh, precision="bf16",
                     Wr=Wr, out=out)
    W = lambda e: (Wu[e], Wg[e], Wd[e])
    for t in range(14):
        o = sampled.token_outputs(t, x, r.idx, r.gates, W, dY=dY, shared=sh, Wr=Wr, out=out)
        assert np.allclose(o["y"], y[t], rtol=1e-12, atol=1e-12)
        assert np.allclose(o["dX"], g.dX[t], rtol=1e-12, atol=1e-12)
        assert np.allclose(o["y_unrounded"], saved["y_unrounded"][t], rtol=1e-12, atol=1e-12)
        assert np.allclose(o["dX_unrounded"], g.unrounded["dX"][t], rtol=1e-12, atol=1e-12)
        assert np.allclose(o["dgates"], g.dgates[t], rtol=1e-12, atol=1e-12)
    pl = saved["plan"]
    for e in range(5):
        pairs = sampled.expert_rows(pl, e)
        picks = [("dW_up", 3, 5), ("dW_gate", 15, 0), ("dW_down", 7, 11), ("dW_down", 0, 0)]
        got = sampled.dw_elements(e, pairs, x, dY, r.gates, Wu[e], Wg[e], Wd[e], picks)
        G = g.unrounded
        ref = [G["dW_up"][e, 3, 5], G["dW_gate"][e, 15, 0], G["dW_down"][e, 7, 11],
               G["dW_down"][e, 0, 0]]
        assert np.allclose(got, ref, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("mode,out", [("bf16", "fp32"), ("bf16_plain", "fp32"),
                                      ("bf16", "bf16")])
def test_dw_lines_and_mx_token_forward_match_the_dense_oracle(rng, mode, out):
    """The full-size evaluators (whole dW lines; MXFP8 per-token forward) against the
    dense per-expert oracle, in both result types."""
    from oracle import sampled
    from oracle.numerics import bf16_round
    x, Wr, b, Wu, Wg, Wd, sh, dY = small_problem(rng, T=20, H=64, I=32, E=4, k=2, shared=True)
    x = bf16_round(x)
    r = moe.route(x, Wr, 2)
    y, saved = moe.forward(x, r.idx, r.gates, Wu, Wg, Wd, shared=sh, precision=mode, out=out)
    g = moe.backward(x, r.idx, r.gates, Wu, Wg, Wd, saved, dY, shared=sh, precision=mode,
                     out=out)
    pl = saved["plan"]
    for e in range(4):
        for i in (0, 17, 31):
            L = sampled.dw_lines(sampled.expert_rows(pl, e), x, dY, r.gates, Wu[e], Wg[e], Wd[e], i,
                                 plain=mode != "bf16", out=out)
            assert np.allclose(L["dW_down"], g.dW_down[e, i, :], rtol=1e-12, atol=1e-12)
            assert np.allclose(L["dW_up"], g.dW_up[e, :, i], rtol=1e-12, atol=1e-12)
            assert np.allclose(L["dW_gate"], g.dW_gate[e, :, i], rtol=1e-12, atol=1e-12)
    ym, _ = moe.forward(x, r.idx, r.gates, Wu, Wg, Wd, shared=sh, precision="mxfp8", out=out)
    cache = {}

    def wq(e):
        if e not in cache:
            cache[e] = sampled.mx_expert_weights(Wu[e], Wg[e], Wd[e])
        return cache[e]

    for t in range(20):
        yt = sampled.token_forward_mx(t, x, r.idx, r.gates, wq, shared=sh, out=out)
        assert np.allclose(yt, ym[t], rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("out", ["fp32", "bf16"])
def test_mx_backward_evaluators_match_the_dense_oracle(rng, out):
    """The MXFP8 full-size backward evaluators (one token's dgates and dX at sampled
    hidden indices with the router path; whole dW lines of one expert) against the dense
    per-expert oracle in mxfp8 mode, in both result types."""
    from oracle import sampled
    from oracle.numerics import bf16_round
    x, Wr, b, Wu, Wg, Wd, sh, dY = small_problem(rng, T=64, H=64, I=64, E=3, k=2)
    x = bf16_round(x)
    r = moe.route(x, Wr, 2)
    _, saved = moe.forward(x, r.idx, r.gates, Wu, Wg, Wd, precision="mxfp8", out=out)
    g = moe.backward(x, r.idx, r.gates, Wu, Wg, Wd, saved, dY, precision="mxfp8", Wr=Wr,
                     out=out)
    hs = np.array([0, 5, 31, 63])
    wq = lambda e: sampled.mx_expert_weights_bwd(Wu[e], Wg[e], Wd[e], hs)
    for t in range(40):
        o = sampled.token_backward_mx(t, x, r.idx, r.gates, wq, dY, Wr=Wr[hs], out=out)
        assert np.allclose(o["dgates"], g.dgates[t], rtol=1e-12, atol=1e-12)
        assert np.allclose(o["dX"], g.dX[t, hs], rtol=1e-12, atol=1e-12)
    pl = saved["plan"]
    assert pl.counts.max() > 32          # an expert with more than one 32-row block
    for e in range(3):
        L = sampled.dw_lines_mx(sampled.expert_rows(pl, e), x, dY, r.gates, Wu[e], Wg[e],
                                Wd[e], [0, 17, 63], out=out)
        for i, li in L.items():
            assert np.allclose(li["dW_down"], g.dW_down[e, i, :], rtol=1e-12, atol=1e-12)
            assert np.allclose(li["dW_up"], g.dW_up[e, :, i], rtol=1e-12, atol=1e-12)
            assert np.allclose(li["dW_gate"], g.dW_gate[e, :, i], rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("mode,out", [("bf16", "fp32"), ("bf16_plain", "fp32"),
                                      ("mxfp8", "fp32"), ("bf16", "bf16")])
def test_shared_dw_lines_match_the_dense_oracle(rng, mode, out):
    from oracle import sampled
    x, Wr, b, Wu, Wg, Wd, sh, dY = small_problem(rng, T=12, H=32, I=32, E=3, k=1, shared=True)
    r = moe.route(x, Wr, 1)
    _, saved = moe.forward(x, r.idx, r.gates, Wu, Wg, Wd, shared=sh, precision=mode, out=out)
    g = moe.backward(x, r.idx, r.gates, Wu, Wg, Wd, saved, dY, shared=sh, precision=mode,
                     out=out)
    for i in range(6):
        L = sampled.shared_dw_lines(x, dY, *sh, i, plain=mode == "bf16_plain", out=out)
        assert np.allclose(L["dWs_down"], g.dWs_down[i], rtol=1e-12, atol=1e-12)
        assert np.allclose(L["dWs_up"], g.dWs_up[:, i], rtol=1e-12, atol=1e-12)
        assert np.allclose(L["dWs_gate"], g.dWs_gate[:, i], rtol=1e-12, atol=1e-12)


def test_saved_uv_rounding_point(rng):
    """The forward keeps U, V for the backward as bf16 values in mxfp8 and in bf16 mode
    (the shared expert's too), while h (and so y) is formed from the unrounded U, V; fp64
    mode keeps them exact."""
    from oracle.numerics import bf16_round, mx_qdq, silu
    x, Wr, b, Wu, Wg, Wd, sh, dY = small_problem(rng, T=24, H=64, I=64, E=3, k=2, shared=True)
    r = moe.route(x, Wr, 2)
    y, saved = moe.forward(x, r.idx, r.gates, Wu, Wg, Wd, precision="mxfp8")
    U, V = saved["U"], saved["V"]
    assert np.array_equal(U, bf16_round(U)) and np.array_equal(V, bf16_round(V))
    pl = saved["plan"]
    e = int(np.argmax(pl.counts))
    r0, r1 = pl.offsets[e], pl.offsets[e + 1]
    A = mx_qdq(x[pl.table[r0:r1, 0]], 1)
    Ue, Ve = A @ mx_qdq(Wu[e], 0), A @ mx_qdq(Wg[e], 0)
    assert np.array_equal(U[r0:r1], bf16_round(Ue))          # rounded where they are saved
    assert not np.array_equal(Ue, bf16_round(Ue))             # (so rounding changes them)
    Xe = x[pl.table[r0:r1, 0]]
    _, saved16 = moe.forward(x, r.idx, r.gates, Wu, Wg, Wd, precision="bf16")
    assert np.array_equal(saved16["U"][r0:r1], bf16_round(Xe @ Wu[e]))
    assert np.array_equal(saved16["V"][r0:r1], bf16_round(Xe @ Wg[e]))
    _, saved64 = moe.forward(x, r.idx, r.gates, Wu, Wg, Wd, precision="fp64")
    assert np.allclose(saved64["U"][r0:r1], Xe @ Wu[e], rtol=0, atol=1e-12)
    assert not np.array_equal(saved64["U"], bf16_round(saved64["U"]))
    _, ssh = moe.shared_forward(x, *sh, "bf16")
    assert np.array_equal(ssh["Us"], bf16_round(x @ sh[0]))
    assert np.array_equal(ssh["Vs"], bf16_round(x @ sh[1]))
    _, ssh64 = moe.shared_forward(x, *sh, "fp64")
    assert np.allclose(ssh64["Us"], x @ sh[0], rtol=0, atol=1e-12)
    # h, the down GEMM's operand, comes from the unrounded U, V: y matches that, not the
    # rounded values
    h_exact = mx_qdq(silu(Ve) * Ue, 1)
    h_saved = mx_qdq(silu(V[r0:r1]) * U[r0:r1], 1)
    assert not np.array_equal(h_exact, h_saved)
    ytok = np.zeros(x.shape[1])
    t, j = pl.table[r0]
    others = [jj for jj in range(2) if jj != j]
    for jj in others:
        ee = int(r.idx[t, jj])
        rr = pl.inv[t, jj] - pl.offsets[ee]
        s0 = pl.offsets[ee]
        Ax = mx_qdq(x[pl.table[s0:pl.offsets[ee + 1], 0]], 1)
        hh = mx_qdq(silu(Ax @ mx_qdq(Wg[ee], 0)) * (Ax @ mx_qdq(Wu[ee], 0)), 1)
        ytok += r.gates[t, jj] * (hh[rr] @ mx_qdq(Wd[ee], 0))
    ytok += r.gates[t, j] * (h_exact[0] @ mx_qdq(Wd[e], 0))
    assert np.allclose(ytok, y[t], rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("mode", ["bf16", "bf16_plain"])
def test_weight_gradient_operand_rounding_point(rng, mode):
    """One token routed to one expert, x made of powers of two: dW_up[e][h][i] =
    x[h] * du[i] exactly, so dW_up / x is du itself. In the bf16_plain mode every such du
    is a bf16 value; with hi/lo operands (bf16) it is the unrounded du (a bf16 value only
    by chance)."""
    from oracle.numerics import bf16_round
    H, I = 32, 64
    x = np.ldexp(1.0, rng.integers(-3, 3, (1, H))) * rng.choice([-1.0, 1.0], (1, H))
    Wu = bf16_round(rng.normal(0, 0.2, (1, H, I)))
    Wg = bf16_round(rng.normal(0, 0.2, (1, H, I)))
    Wd = bf16_round(rng.normal(0, 0.2, (1, I, H)))
    dY = bf16_round(rng.normal(0, 1, (1, H)))
    idx = np.zeros((1, 1), np.int64)
    gates = np.ones((1, 1))
    _, saved = moe.forward(x, idx, gates, Wu, Wg, Wd, precision=mode)
    g = moe.backward(x, idx, gates, Wu, Wg, Wd, saved, dY, precision=mode)
    du = g.dW_up[0] / x[0][:, None]
    assert np.allclose(du, du[0][None, :], rtol=0, atol=0)     # one du row, scaled by x[h]
    n_bf16 = int((bf16_round(du[0]) == du[0]).sum())
    if mode == "bf16_plain":
        assert n_bf16 == I
    else:
        assert n_bf16 < I // 4


def _one_token_one_expert(rng, H, c=0.5):
    """x, dY bf16 values; W_up and W_down the identity, W_gate c times it (H = I): then
    U = x, V = c x and D = dY exactly in every precision mode (MXFP8 blocks of an identity
    row or column hold a single power of two)."""
    from oracle.numerics import bf16_round
    x = bf16_round(rng.normal(0, 1, (1, H)))
    dY = bf16_round(rng.normal(0, 1, (1, H)))
    eye = np.eye(H)[None]
    return x, dY, eye, c * eye, eye


@pytest.mark.parametrize("mode", ["fp64", "bf16", "mxfp8"])
def test_down_gemm_operand_rounding_point(rng, mode):
    """With W_down the identity, gate 1 and one slot, y is h itself, so it shows where h
    is rounded: to bf16 in the bf16 mode (h is stored as bf16 for the down GEMM), to MXFP8
    blocks of 32 along I in the mxfp8 mode, not at all in fp64."""
    from oracle.numerics import bf16_round, mx_qdq, silu
    H = 64
    x, _, _, _, Wd = _one_token_one_expert(rng, H)
    Wu = bf16_round(rng.normal(0, 0.2, (1, H, H)))
    Wg = bf16_round(rng.normal(0, 0.2, (1, H, H)))
    y, _ = moe.forward(x, np.zeros((1, 1), np.int64), np.ones((1, 1)), Wu, Wg, Wd,
                       precision=mode)
    if mode == "mxfp8":
        A = mx_qdq(x, 1)
        h = silu(A @ mx_qdq(Wg[0], 0)) * (A @ mx_qdq(Wu[0], 0))
        want = mx_qdq(h, 1)
    else:
        h = silu(x @ Wg[0]) * (x @ Wu[0])
        want = bf16_round(h) if mode == "bf16" else h
    assert np.array_equal(y, want)
    if mode != "fp64":
        assert not np.array_equal(want, h)


@pytest.mark.parametrize("mode", ["fp64", "bf16", "mxfp8"])
def test_dx_gemm_operand_rounding_point(rng, mode):
    """With W_up, W_down the identity and W_gate = identity / 2, gate 1 and one slot,
    dX = du' + dv' / 2, where du', dv' are du = D silu(V) and dv = D U silu'(V) as the dX
    GEMM reads them: bf16 in the bf16 mode, MXFP8 blocks of 32 along I in the mxfp8 mode,
    unrounded in fp64."""
    from oracle.numerics import bf16_round, dsilu, mx_qdq, silu
    H, c = 64, 0.5
    x, dY, Wu, Wg, Wd = _one_token_one_expert(rng, H, c)
    idx, gates = np.zeros((1, 1), np.int64), np.ones((1, 1))
    _, saved = moe.forward(x, idx, gates, Wu, Wg, Wd, precision=mode)
    g = moe.backward(x, idx, gates, Wu, Wg, Wd, saved, dY, precision=mode)
    mx = mode == "mxfp8"
    A, D = (mx_qdq(x, 1), mx_qdq(dY, 1)) if mx else (x, dY)
    U, V = A, c * A
    du, dv = D * silu(V), D * U * dsilu(V)
    rd = {"fp64": lambda a: a, "bf16": bf16_round, "mxfp8": lambda a: mx_qdq(a, 1)}[mode]
    assert np.array_equal(g.dX, rd(du) + c * rd(dv))
    if mode != "fp64":
        assert not np.array_equal(rd(du), du) and not np.array_equal(rd(dv), dv)


# ----------------------------------------------------------------------------- result type
def test_result_rounding_points_forward(rng):
    """bf16 results: with W_down = c * identity (c = 1 + 2^-10, so c h is not a bf16 value
    while bf16(c h) is h's neighbourhood), two slots to two experts with gates 1/3, 2/3 and
    a shared expert of the same form, the value before y's rounding is
    g1 bf16(c h1) + g2 bf16(c h2) + bf16(c hs) exactly: each expert output row and the
    shared output rounded on its own, then summed; y is that sum rounded once. With fp32
    results nothing is rounded: g1 c h1 + g2 c h2 + c hs."""
    from oracle.numerics import bf16_round, silu
    H, c = 64, 1.0 + 2.0 ** -10
    x = bf16_round(rng.normal(0, 1, (1, H)))
    Wu = bf16_round(rng.normal(0, 0.2, (2, H, H)))
    Wg = bf16_round(rng.normal(0, 0.2, (2, H, H)))
    Wd = c * np.stack([np.eye(H), np.eye(H)])
    sh = (bf16_round(rng.normal(0, 0.2, (H, H))), bf16_round(rng.normal(0, 0.2, (H, H))),
          c * np.eye(H))
    idx, gates = np.array([[1, 0]]), np.array([[1 / 3, 2 / 3]])
    h = [bf16_round(silu(x @ Wg[e]) * (x @ Wu[e])) for e in (0, 1)]
    hs = bf16_round(silu(x @ sh[1]) * (x @ sh[0]))
    y, saved = moe.forward(x, idx, gates, Wu, Wg, Wd, shared=sh, precision="bf16", out="bf16")
    pre = gates[0, 0] * bf16_round(c * h[1]) + gates[0, 1] * bf16_round(c * h[0]) \
        + bf16_round(c * hs)
    assert np.array_equal(saved["y_unrounded"], pre)
    assert np.array_equal(y, bf16_round(pre))
    assert not np.array_equal(bf16_round(pre), pre)
    y32, s32 = moe.forward(x, idx, gates, Wu, Wg, Wd, shared=sh, precision="bf16", out="fp32")
    want = gates[0, 0] * (c * h[1]) + gates[0, 1] * (c * h[0]) + c * hs
    assert np.array_equal(y32, want) and np.array_equal(s32["y_unrounded"], want)
    assert not np.array_equal(pre, want)


def test_result_rounding_points_backward(rng):
    """bf16 results: one token, both slots to one expert (gates 1/4, 3/4), a shared expert,
    W_down the identity, W_up = c I and W_gate = (c/2) I (c = 1 + 2^-10). Each routed dX
    row is bf16(c du' + (c/2) dv') with du', dv' the dX GEMM's bf16 operands (formed from
    U = bf16(c x), V = bf16(c x / 2), as the forward keeps them), the shared expert's dX
    row likewise with gate 1; dX is their sum rounded once; every weight gradient is its
    exact sum over the rows rounded once (dW_up = x^T du per slot)."""
    from oracle.numerics import bf16_round, dsilu, silu
    H, c = 64, 1.0 + 2.0 ** -10
    x = bf16_round(rng.normal(0, 1, (1, H)))
    dY = bf16_round(rng.normal(0, 1, (1, H)))
    eye = np.eye(H)
    Wu, Wg, Wd = (c * eye)[None], (c / 2 * eye)[None], eye[None]
    sh = (c * eye, c / 2 * eye, eye)
    idx, gates = np.array([[0, 0]]), np.array([[0.25, 0.75]])
    _, saved = moe.forward(x, idx, gates, Wu, Wg, Wd, shared=sh, precision="bf16", out="bf16")
    g = moe.backward(x, idx, gates, Wu, Wg, Wd, saved, dY, shared=sh, precision="bf16",
                     out="bf16")
    U, V = bf16_round(c * x), bf16_round(c / 2 * x)
    assert not np.array_equal(U, c * x)   # (the kept values differ from the exact ones)

    def rows(gt):
        du, dv = gt * dY * silu(V), gt * dY * U * dsilu(V)
        return bf16_round(c * bf16_round(du) + c / 2 * bf16_round(dv)), du
    r1, du1 = rows(0.25)
    r2, du2 = rows(0.75)
    rs, _ = rows(1.0)
    pre = r1 + r2 + rs
    assert np.array_equal(g.unrounded["dX"], pre)
    assert np.array_equal(g.dX, bf16_round(pre))
    assert not np.array_equal(bf16_round(pre), pre)
    dwu = x.T @ du1 + x.T @ du2
    assert np.allclose(g.unrounded["dW_up"][0], dwu, rtol=1e-14, atol=0)
    assert np.array_equal(g.dW_up, bf16_round(g.unrounded["dW_up"]))
    assert not np.array_equal(g.dW_up, g.unrounded["dW_up"])
    for n in ("dW_gate", "dW_down", "dWs_up", "dWs_gate", "dWs_down"):
        assert np.array_equal(getattr(g, n), bf16_round(g.unrounded[n])), n
    g32 = moe.backward(x, idx, gates, Wu, Wg, Wd, saved, dY, shared=sh, precision="bf16",
                       out="fp32")
    pre32 = (c * bf16_round(rows(0.25)[1]) + c / 2 * bf16_round(0.25 * dY * U * dsilu(V))) \
        + (c * bf16_round(rows(0.75)[1]) + c / 2 * bf16_round(0.75 * dY * U * dsilu(V)))
    assert np.allclose(g32.dX - (c * bf16_round(dY * silu(V))
                                 + c / 2 * bf16_round(dY * U * dsilu(V))), pre32,
                       rtol=1e-14, atol=1e-15)
    assert np.allclose(g32.dW_up[0], dwu, rtol=1e-14, atol=0)
