"""Allowance for comparing bf16 results of the GPU with the oracle's (test helper).

With bf16 results the GPU rounds its fp32 sums once, and the oracle rounds its fp64 values
once, both to nearest-even bf16. Where the two values before rounding lie on the same side
of every bf16 rounding midpoint, the results are equal; where a midpoint lies between them,
they differ by one bf16 spacing (more if the gap spans several). So each result element
gets an allowance: the largest distance between bf16(a') and bf16(a) over every a' within
delta of the oracle's value a, where delta bounds |GPU value - oracle value| before the
rounding. The allowance is 0 wherever no midpoint lies within delta.

delta is a first-order bound propagated through the GPU's arithmetic, step by step:
* an fp32 sum of n products errs by at most lam * sqrt(n) * u * sum|terms| (u = 2^-24,
  lam = 6): the probabilistic bound of Higham and Mary ("A New Approach to Probabilistic
  Rounding Error Analysis", 2019), which fails for a given sum with probability below
  2 exp(-lam^2 / 2);
* errors of the operands of a sum (each within its own bound c_i, of either sign, from
  roundings of different elements) add up, under the same model of independent errors of
  mean zero, to at most lam * sqrt(sum c_i^2) (Hoeffding's inequality, failing with the
  same probability); a worst-case sum of the c_i would flag most results of a long
  contraction as near a midpoint and say little;
* elementwise fp32 arithmetic (SwiGLU, its derivative, the gate products) errs by a few
  units, taken as 8 u relative;
* an intermediate rounded on both sides (h, U and V as kept for the backward, and du, dv
  for the dX GEMM, in bf16; the expert output rows and routed dX rows with bf16 results;
  du, dv, g*h with single bf16 weight-gradient operands) moves by its own rounding flip,
  found the same way;
* the weight-gradient GEMMs' bf16 hi + lo operand pairs carry a 16-bit significand:
  2^-17 relative;
* the router's gates: the GPU's fp32 logits lie within the worst-case bound of
  ``gpu_util.logit_margins``; a renormalised gate then moves by at most
  g (m_j + sum_i g_i m_i) <= 2 g max m (plus fp32 rounding), m the logit bounds.

In MXFP8 the operands themselves are E4M3 values whose quantisation can flip by an E4M3
step (2^-4 relative), and the comparison's tolerance covers those; the value before the
result's rounding is then not known to better than a bf16 spacing, and the allowance is one
bf16 spacing of each element.
"""
from __future__ import annotations

import numpy as np

from oracle import moe
from oracle.numerics import bf16_round, dsilu, sigmoid

U32 = 2.0 ** -24
LAM = 6.0
HILO_REL = 2.0 ** -17
ELT_REL = 8 * U32


def gam(n):
    return LAM * np.sqrt(max(int(n), 1)) * U32


def prop(A, Bm):
    """Bound on the sum's error from operand errors: lam * sqrt((A^2) @ (Bm^2)), A holding
    the operand error bounds and Bm the other operand (or the reverse)."""
    return LAM * np.sqrt(np.square(A) @ np.square(Bm))


def flip_dev(a, delta):
    """Largest |bf16(a') - bf16(a)| over |a' - a| <= delta (bf16 rounding is monotone,
    so the ends of the interval give it)."""
    r = bf16_round(a)
    return np.maximum(np.abs(bf16_round(a + delta) - r), np.abs(bf16_round(a - delta) - r))


def bf16_spacing(a):
    """The distance between neighbouring bf16 values at |a| (8 significant bits)."""
    a = np.abs(np.asarray(a, np.float64))
    _, e = np.frexp(np.where(a > 0, a, 1.0))
    return np.where(a > 0, np.ldexp(1.0, np.maximum(e - 8, -133)), np.ldexp(1.0, -133))


def gate_bounds(cfg, inp, idx, gates, logits=None):
    """Bound on |GPU gate - oracle gate| per slot: 0 when the routing is an input (the
    oracle takes the same fp32 gates), else from the logit bound."""
    if not cfg.router:
        return np.zeros_like(gates)
    from tests import gpu_util as gu
    if logits is None:
        logits = gu.np64(inp["x"]) @ gu.np64(inp["Wr"])
        if inp.get("bias") is not None:
            logits = logits + gu.np64(inp["bias"])[None, :]
    m = np.take_along_axis(gu.logit_margins(cfg, inp, logits), idx, axis=1)
    return 2.0 * gates * m.max(axis=1, keepdims=True) * (1 + 1e-6) + 4 * U32 * gates


# ----------------------------------------------------------------------------- per rows
def fwd_rows(X, Wu, Wg, Wd, out_bf16=True):
    """Forward of some routed rows X (any subset of one expert's rows; bf16 precision):
    the oracle's values and the bounds of the GPU's. Returns a dict with U, V, their
    bounds bU, bV, h (bf16), Opre (h W_down) and O (the result row), d_O (bound before the
    rounding) and f_O (bound on |GPU O - oracle O|)."""
    H, I = Wu.shape
    aX = np.abs(X)
    U, V = X @ Wu, X @ Wg
    bU, bV = gam(H) * (aX @ np.abs(Wu)), gam(H) * (aX @ np.abs(Wg))
    s = sigmoid(V)
    s0 = V * s
    s1 = s * (1 + V * (1 - s))
    hpre = s0 * U
    d_h = np.abs(s1 * U) * bV + np.abs(s0) * bU + ELT_REL * np.abs(hpre)
    f_h = flip_dev(hpre, d_h)
    h = bf16_round(hpre)
    Opre = h @ Wd
    d_O = prop(f_h, Wd) + gam(I) * (np.abs(h) @ np.abs(Wd))
    if out_bf16:
        O, f_O = bf16_round(Opre), flip_dev(Opre, d_O)
    else:
        O, f_O = Opre, d_O
    return {"U": U, "V": V, "bU": bU, "bV": bV, "s": s, "s0": s0, "s1": s1,
            "Opre": Opre, "O": O, "d_O": d_O, "f_O": f_O}


def bwd_rows(f, dYr, g, dgb, Wu, Wg, Wd, plain=False, out_bf16=True):
    """Backward of the same rows (``f`` from ``fwd_rows``) with upstream rows dYr and gates
    g, gate bounds dgb ([n, 1] each). Returns the oracle's operands (du, dv, g*h as the
    weight-gradient GEMMs take them), their bounds E_* (|GPU operand - oracle operand|),
    the routed dX rows (dXg, with bound f_dXg), the router-weight gradient dg and its
    bound d_dg."""
    H, I = Wu.shape
    # the backward reads U, V as the forward kept them, bf16 on both sides: they differ
    # by the rounding flip of the GPU's fp32 sums
    U, V = bf16_round(f["U"]), bf16_round(f["V"])
    bU, bV = flip_dev(f["U"], f["bU"]), flip_dev(f["V"], f["bV"])
    s = sigmoid(V)
    s0 = V * s
    s1 = s * (1 + V * (1 - s))
    s2 = s * (1 - s) * (2 + V * (1 - 2 * s))
    D = dYr @ Wd.T
    bD = gam(H) * (np.abs(dYr) @ np.abs(Wd).T)
    ag = np.abs(g)
    hv = s0 * U
    du, dv, hg = g * D * s0, g * D * U * s1, g * hv
    d_du = ag * (bD * np.abs(s0) + np.abs(D * s1) * bV) + dgb * np.abs(D * s0) \
        + ELT_REL * np.abs(du)
    d_dv = ag * (bD * np.abs(U * s1) + np.abs(D * s1) * bU + np.abs(D * U * s2) * bV) \
        + dgb * np.abs(D * U * s1) + ELT_REL * np.abs(dv)
    d_hv = np.abs(s1 * U) * bV + np.abs(s0) * bU + ELT_REL * np.abs(hv)
    d_hg = ag * d_hv + dgb * np.abs(hv) + ELT_REL * np.abs(hg)
    # the dX GEMM takes du, dv rounded to bf16 on both sides
    du_b, dv_b = bf16_round(du), bf16_round(dv)
    f_du, f_dv = flip_dev(du, d_du), flip_dev(dv, d_dv)
    dXpre = du_b @ Wu.T + dv_b @ Wg.T
    d_dXg = LAM * np.sqrt(np.square(f_du) @ np.square(Wu).T + np.square(f_dv) @ np.square(Wg).T) \
        + gam(2 * I) * (np.abs(du_b) @ np.abs(Wu).T + np.abs(dv_b) @ np.abs(Wg).T)
    if out_bf16:
        dXg, f_dXg = bf16_round(dXpre), flip_dev(dXpre, d_dXg)
    else:
        dXg, f_dXg = dXpre, d_dXg
    # the weight-gradient GEMMs' operands: hi + lo pairs, or single bf16 values
    if plain:
        ops = {n: (bf16_round(v), flip_dev(v, dv_)) for n, v, dv_ in
               (("du", du, d_du), ("dv", dv, d_dv), ("hg", hg, d_hg))}
    else:
        ops = {n: (v, dv_ + HILO_REL * np.abs(v)) for n, v, dv_ in
               (("du", du, d_du), ("dv", dv, d_dv), ("hg", hg, d_hg))}
    dg = (D * hv).sum(axis=1)
    d_dg = LAM * np.sqrt((np.square(bD * hv) + np.square(D * d_hv)).sum(axis=1)) \
        + gam(I) * (np.abs(D * hv)).sum(axis=1)
    return {"ops": ops, "dXg": dXg, "f_dXg": f_dXg, "dg": dg, "d_dg": d_dg}


def dw_slack(X, dYr, ops, plain=False):
    """Allowance of one expert's bf16 weight gradients from its rows: X and dYr the rows'
    x and dY, ``ops`` from ``bwd_rows``. Returns (dW_up, dW_gate, dW_down) allowances and
    the unrounded oracle values."""
    n = X.shape[0]
    kf = n if plain else 2 * n          # hi + lo: two MMAs per K step
    aX, adY = np.abs(X), np.abs(dYr)
    res, pre = [], []
    for name, A, aA in (("du", X, aX), ("dv", X, aX)):
        op, E = ops[name]
        v = A.T @ op
        d = prop(A.T, E) + gam(kf) * (aA.T @ np.abs(op))
        res.append(flip_dev(v, d))
        pre.append(v)
    op, E = ops["hg"]
    v = op.T @ dYr
    d = prop(E.T, dYr) + gam(kf) * (np.abs(op).T @ adY)
    res.append(flip_dev(v, d))
    pre.append(v)
    return res, pre


# ----------------------------------------------------------------------------- whole layer
def layer_slack(cfg, inp, idx, gates, logits=None):
    """Allowances for every bf16 result of a small layer (dense in memory): a dict with
    y, dX, dW_up, dW_gate, dW_down and, with a shared expert, dWs_*. ``idx``, ``gates``:
    the oracle's routing (the GPU's is the same expert sets, tested separately)."""
    from tests import gpu_util as gu
    if cfg.precision == "mxfp8":
        raise ValueError("MXFP8 results take one bf16 spacing (spacing_slack)")
    plain = cfg.precision == "bf16_plain"
    x, dY = gu.np64(inp["x"]), gu.np64(inp["dY"])
    Wu, Wg, Wd = (gu.np64(inp[n]) for n in ("W_up", "W_gate", "W_down"))
    T, H, k = cfg.T, cfg.H, cfg.k
    dgb_all = gate_bounds(cfg, inp, idx, gates, logits)
    pl = moe.plan(idx, cfg.E)
    R = T * k
    O, f_O = np.zeros((R, H)), np.zeros((R, H))
    dXg, f_dXg = np.zeros((R, H)), np.zeros((R, H))
    dg, d_dg = np.zeros((T, k)), np.zeros((T, k))
    out = {n: np.zeros(w.shape) for n, w in (("dW_up", Wu), ("dW_gate", Wg), ("dW_down", Wd))}
    for e in range(cfg.E):
        r0, r1 = pl.offsets[e], pl.offsets[e + 1]
        if r0 == r1:
            continue
        t, j = pl.table[r0:r1, 0], pl.table[r0:r1, 1]
        g = gates[t, j][:, None]
        f = fwd_rows(x[t], Wu[e], Wg[e], Wd[e])
        b = bwd_rows(f, dY[t], g, dgb_all[t, j][:, None], Wu[e], Wg[e], Wd[e], plain)
        O[r0:r1], f_O[r0:r1] = f["O"], f["f_O"]
        dXg[r0:r1], f_dXg[r0:r1] = b["dXg"], b["f_dXg"]
        dg[t, j], d_dg[t, j] = b["dg"], b["d_dg"]
        (su, sg, sd), _ = dw_slack(x[t], dY[t], b["ops"], plain)
        out["dW_up"][e], out["dW_gate"][e], out["dW_down"][e] = su, sg, sd
    # combine: y = sum_j g O (slot order, fp32) + Os
    y_pre = np.zeros((T, H))
    d_y = np.zeros((T, H))
    mag_y = np.zeros((T, H))
    dX_pre = np.zeros((T, H))
    d_dX = np.zeros((T, H))
    mag_dx = np.zeros((T, H))
    for jj in range(k):
        rows = pl.inv[:, jj]
        gj = gates[:, jj:jj + 1]
        y_pre += gj * O[rows]
        d_y += np.abs(gj) * f_O[rows] + dgb_all[:, jj:jj + 1] * np.abs(O[rows])
        mag_y += np.abs(gj * O[rows])
        dX_pre += dXg[rows]
        d_dX += f_dXg[rows]
        mag_dx += np.abs(dXg[rows])
    if cfg.shared_I:
        Su, Sg, Sd = (gu.np64(inp[n]) for n in ("Ws_up", "Ws_gate", "Ws_down"))
        fs = fwd_rows(x, Su, Sg, Sd)
        ones = np.ones((T, 1))
        bs = bwd_rows(fs, dY, ones, np.zeros((T, 1)), Su, Sg, Sd,
                      plain=plain)
        y_pre += fs["O"]
        d_y += fs["f_O"]
        mag_y += np.abs(fs["O"])
        dX_pre += bs["dXg"]
        d_dX += bs["f_dXg"]
        mag_dx += np.abs(bs["dXg"])
        (su, sg, sd), _ = dw_slack(x, dY, bs["ops"], plain)
        out["dWs_up"], out["dWs_gate"], out["dWs_down"] = su, sg, sd
    if cfg.router:
        Wr = gu.np64(inp["Wr"])
        S = (gates * dg).sum(axis=1, keepdims=True)
        dl = gates * (dg - S)
        dS = (dgb_all * np.abs(dg) + np.abs(gates) * d_dg).sum(axis=1, keepdims=True)
        d_dl = dgb_all * np.abs(dg - S) + np.abs(gates) * (d_dg + dS) \
            + 4 * U32 * np.abs(gates) * (np.abs(dg) + np.abs(S))
        for jj in range(k):
            w = Wr[:, idx[:, jj]].T                    # [T, H]
            dX_pre += dl[:, jj:jj + 1] * w
            d_dX += d_dl[:, jj:jj + 1] * np.abs(w)
            mag_dx += np.abs(dl[:, jj:jj + 1] * w)
    d_y += (k + 2) * U32 * mag_y
    d_dX += (2 * k + 2) * U32 * mag_dx
    out["y"] = flip_dev(y_pre, d_y)
    out["dX"] = flip_dev(dX_pre, d_dX)
    return out


def spacing_slack(ref_unrounded: dict):
    """One bf16 spacing per element (the MXFP8 allowance)."""
    return {n: bf16_spacing(v) for n, v in ref_unrounded.items()}


def rel_err_slack(gpu, ref, slack) -> float:
    """max(|gpu - oracle| - allowance, 0) / rms(oracle)."""
    from tests import gpu_util as gu
    return gu.rel_err_slack(gpu, ref, slack)


# ----------------------------------------------------------------------------- full size
def token_slack(t, x, idx, gates, dgb, weights, dY=None, shared=None, Wr=None, plain=False):
    """Allowances of one token's bf16 y and dX rows (full-size workloads, bf16
    precision). weights(e) -> (W_up[e], W_gate[e], W_down[e]) float64; dgb: gate bounds
    [T, k]. Returns (y allowance, dX allowance or None)."""
    k = idx.shape[1]
    x_t = np.asarray(x[t], np.float64)[None, :]
    H = x_t.shape[1]
    y_pre, d_y, mag_y = np.zeros(H), np.zeros(H), np.zeros(H)
    dX_pre, d_dX, mag_dx = np.zeros(H), np.zeros(H), np.zeros(H)
    dg, d_dg = np.zeros(k), np.zeros(k)
    dY_t = None if dY is None else np.asarray(dY[t], np.float64)[None, :]
    for j in range(k):
        e, g = int(idx[t, j]), float(gates[t, j])
        Wu, Wg, Wd = weights(e)
        f = fwd_rows(x_t, Wu, Wg, Wd)
        y_pre += g * f["O"][0]
        d_y += abs(g) * f["f_O"][0] + dgb[t, j] * np.abs(f["O"][0])
        mag_y += np.abs(g * f["O"][0])
        if dY_t is not None:
            b = bwd_rows(f, dY_t, np.array([[g]]), np.array([[dgb[t, j]]]), Wu, Wg, Wd, plain)
            dX_pre += b["dXg"][0]
            d_dX += b["f_dXg"][0]
            mag_dx += np.abs(b["dXg"][0])
            dg[j], d_dg[j] = b["dg"][0], b["d_dg"][0]
    if shared is not None:
        Su, Sg, Sd = shared
        fs = fwd_rows(x_t, Su, Sg, Sd)
        y_pre += fs["O"][0]
        d_y += fs["f_O"][0]
        mag_y += np.abs(fs["O"][0])
        if dY_t is not None:
            bs = bwd_rows(fs, dY_t, np.ones((1, 1)), np.zeros((1, 1)), Su, Sg, Sd, plain)
            dX_pre += bs["dXg"][0]
            d_dX += bs["f_dXg"][0]
            mag_dx += np.abs(bs["dXg"][0])
    d_y += (k + 2) * U32 * mag_y
    y_sl = flip_dev(y_pre, d_y)
    if dY_t is None:
        return y_sl, None
    if Wr is not None:
        g = np.asarray(gates[t], np.float64)
        S = float((g * dg).sum())
        dl = g * (dg - S)
        dS = float((dgb[t] * np.abs(dg) + np.abs(g) * d_dg).sum())
        d_dl = dgb[t] * np.abs(dg - S) + np.abs(g) * (d_dg + dS) \
            + 4 * U32 * np.abs(g) * (np.abs(dg) + abs(S))
        for j in range(k):
            w = np.asarray(Wr[:, int(idx[t, j])], np.float64)
            dX_pre += dl[j] * w
            d_dX += d_dl[j] * np.abs(w)
            mag_dx += np.abs(dl[j] * w)
    d_dX += (2 * k + 2) * U32 * mag_dx
    return y_sl, flip_dev(dX_pre, d_dX)


def dw_line_slack(pairs, x, dY, gates, dgb, Wu, Wg, Wd, i, plain=False):
    """Allowances of one expert's bf16 weight-gradient lines for intermediate index i:
    dW_down[e][i, :], dW_up[e][:, i], dW_gate[e][:, i] (full-size workloads). ``gates``
    and ``dgb`` [T, k]; pairs: the expert's (t, j) table rows."""
    t, j = pairs[:, 0], pairs[:, 1]
    X = np.asarray(x[t], np.float64)
    dYr = np.asarray(dY[t], np.float64)
    g = np.asarray(gates[t, j], np.float64)[:, None]
    f = fwd_rows(X, Wu[:, i:i + 1], Wg[:, i:i + 1], Wd[i:i + 1, :])
    b = bwd_rows(f, dYr, g, np.asarray(dgb[t, j], np.float64)[:, None], Wu[:, i:i + 1],
                 Wg[:, i:i + 1], Wd[i:i + 1, :], plain)
    (su, sg, sd), _ = dw_slack(X, dYr, b["ops"], plain)
    return {"dW_up": su[:, 0], "dW_gate": sg[:, 0], "dW_down": sd[0]}
