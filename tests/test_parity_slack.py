"""The bf16 rounding-flip allowance used by the weight-gradient parity checks with fp32
results: it admits a GPU-like result (fp32 GEMM errors within the bound, then bf16
rounding of U, V and, in bf16_plain, of du, dv, g*h) and still rejects planted mistakes,
in both BF16 modes. Everything here runs on the CPU; the "GPU-like" side is the oracle's
own arithmetic with perturbed intermediates."""
import numpy as np
import pytest

import moe_inputs as mi
from oracle import moe
from oracle.numerics import bf16_round, dsilu, silu
from tests import gpu_util as gu


def _case(seed=0, precision="bf16_plain"):
    cfg = mi.MoEConfig("slack", T=64, H=128, I=128, E=32, k=2, precision=precision)
    inp = mi.make_inputs(cfg, seed=seed, with_dy=True)
    idx, gates, _ = gu.oracle_route(cfg, inp)
    return cfg, inp, idx, gates


def _dw_with(cfg, inp, idx, gates, perturb, rng, sign_dv=1.0):
    """dW_up, dW_gate, dW_down with U, V, D perturbed by up to ``perturb`` times their
    fp32-sum bound, U, V then kept as bf16 (as the forward keeps them), du, dv, g*h rounded
    to bf16 in bf16_plain (the GPU's operand points; bf16 takes them as hi + lo pairs,
    close to exact)."""
    x, dY = gu.np64(inp["x"]), gu.np64(inp["dY"])
    Wu, Wg, Wd = (gu.np64(inp[n]) for n in ("W_up", "W_gate", "W_down"))
    gam = 6.0 * np.sqrt(cfg.H) * 2.0 ** -24      # the bound the allowance assumes
    pl = moe.plan(idx, cfg.E)
    rnd = bf16_round if cfg.precision == "bf16_plain" else (lambda v: v)
    out = [np.zeros(Wu.shape), np.zeros(Wg.shape), np.zeros(Wd.shape)]
    for e in range(cfg.E):
        r0, r1 = pl.offsets[e], pl.offsets[e + 1]
        if r0 == r1:
            continue
        t, j = pl.table[r0:r1, 0], pl.table[r0:r1, 1]
        X, dYe, g = x[t], dY[t], gates[t, j][:, None]
        U, V, D = X @ Wu[e], X @ Wg[e], dYe @ Wd[e].T
        bU = gam * (np.abs(X) @ np.abs(Wu[e]))
        bV = gam * (np.abs(X) @ np.abs(Wg[e]))
        bD = gam * (np.abs(dYe) @ np.abs(Wd[e]).T)
        U = U + perturb * bU * rng.uniform(-1, 1, U.shape)
        V = V + perturb * bV * rng.uniform(-1, 1, V.shape)
        D = D + perturb * bD * rng.uniform(-1, 1, D.shape)
        U, V = bf16_round(U), bf16_round(V)
        du = rnd(g * D * silu(V))
        dv = rnd(sign_dv * g * D * U * dsilu(V))
        hg = rnd(g * silu(V) * U)
        out[0][e], out[1][e], out[2][e] = X.T @ du, X.T @ dv, hg.T @ dYe
    return dict(zip(("dW_up", "dW_gate", "dW_down"), out))


@pytest.mark.parametrize("precision", ["bf16_plain", "bf16"])
def test_slack_admits_perturbations_within_the_bound(precision):
    cfg, inp, idx, gates = _case(precision=precision)
    rng = np.random.default_rng(1)
    ref = _dw_with(cfg, inp, idx, gates, 0.0, rng)
    slack, frac = gu.bf16_flip_slack(cfg, inp, idx, gates)
    assert 0 < frac < 0.5
    for f in ref:    # the allowance is a few bf16 spacings, far below the tolerance
        rms = np.sqrt((ref[f] ** 2).mean())
        assert np.median(slack[f]) / rms < 1e-3, f
    for trial in range(3):
        got = _dw_with(cfg, inp, idx, gates, 1.0, rng)
        for f in ref:
            assert gu.rel_err_slack(got[f], ref[f], slack[f]) <= 1e-12, f


def test_slack_is_zero_away_from_midpoints():
    v = np.array([1.0, 1.0 + 2.0 ** -7, 3.0, -0.75])      # bf16 values: far from midpoints
    dev, frac = gu._flip_dev(v, np.full(4, 1e-6))
    assert np.all(dev == 0) and frac == 0
    mid = np.array([1.0 + 2.0 ** -7 + 2.0 ** -8])          # a midpoint between two bf16
    dev, frac = gu._flip_dev(mid, np.array([1e-9]))
    assert dev[0] == 2.0 ** -7 and frac == 1.0
    # a bound of 2.5 spacings around 1 + 2^-7: upwards 1 + 3.5 * 2^-7 is a tie that goes to
    # the even neighbour 1 + 4 * 2^-7 (3 spacings); downwards 1 - 3 * 2^-8 (2.5 spacings)
    wide = np.array([1.0 + 2.0 ** -7])
    dev, _ = gu._flip_dev(wide, np.array([2.5 * 2.0 ** -7]))
    assert dev[0] == 3 * 2.0 ** -7


@pytest.mark.parametrize("precision", ["bf16_plain", "bf16"])
@pytest.mark.parametrize("mistake", ["dv_sign", "dropped_gate", "scaled_row"])
def test_slack_still_rejects_planted_mistakes(mistake, precision):
    cfg, inp, idx, gates = _case(precision=precision)
    rng = np.random.default_rng(2)
    ref = _dw_with(cfg, inp, idx, gates, 0.0, rng)
    slack, _ = gu.bf16_flip_slack(cfg, inp, idx, gates)
    if mistake == "dv_sign":
        bad = _dw_with(cfg, inp, idx, gates, 0.0, rng, sign_dv=-1.0)["dW_gate"]
        f = "dW_gate"
    elif mistake == "dropped_gate":
        bad = _dw_with(cfg, inp, idx, np.ones_like(gates), 0.0, rng)["dW_up"]
        f = "dW_up"
    else:
        f = "dW_down"
        bad = ref[f].copy()
        e = int(np.argmax(np.abs(bad).sum(axis=(1, 2))))   # an expert with rows
        bad[e, 7] *= 1.05
    assert gu.rel_err_slack(bad, ref[f], slack[f]) > gu.TOL["bf16_plain"]
