"""Single-output evaluators of the layer for full-size workloads (fp64, NumPy).

TEST INFRASTRUCTURE ONLY (see oracle/__init__.py). The dense oracle in ``moe`` holds every
routed row of every expert; at the Kimi/DeepSeek sizes that is too much, so these
functions compute one token's y or dX row, or one element or line of a weight gradient,
straight from the definition (with the same rounding model as ``moe``, precision "bf16":
h, the down GEMM's operand, and du, dv as operands of the dX GEMM are rounded to bf16,
and the backward reads U, V as bf16 values, as the forward keeps them; the
weight-gradient functions take ``plain`` to choose "bf16_plain" over "bf16"):

* y_t = sum_j g_tj O_(t,j) + shared(x_t), O = bf16(silu(x W_gate) * (x W_up)) W_down;
* dX_t = sum_j (bf16(du) W_up^T + bf16(dv) W_gate^T) + dXs_t + sum_j dl_tj Wr[:, e_j],
  with D = dY_t W_down^T, du = g D silu(V), dv = g D U silu'(V) (U, V the kept bf16 values);
* dW_down[e][i][h] = sum over e's rows of (g silu(V) U)[i] dY[t][h];
* dW_up[e][h][i] = sum over e's rows of x[t][h] du[i] (dW_gate with dv).

The ``*_mx`` functions follow ``moe``'s precision "mxfp8" instead: every GEMM operand in
MXFP8 blocks of 32 along that GEMM's contraction axis (x, h and dY along H or I per row;
du, dv, g*h, x and dY along the expert rows for the weight gradients), and the backward
reads U, V as bf16 values.

``out`` ("fp32" or "bf16", as in ``moe``) models the result type: with "bf16" the expert
output rows, the shared expert's output, the routed dX rows and the shared expert's dX are
rounded to bf16, and so is each returned y, dX and weight-gradient line (once, after the
exact sum); dgates stay unrounded. The values before that last rounding come back too
(keys ending in ``_unrounded``).

``W`` arguments are callables returning one expert's float64 matrices on demand, so the
caller can stream them from wherever they live.
"""
from __future__ import annotations

import numpy as np

from .moe import out_round
from .numerics import bf16_round, dsilu, mx_qdq, mx_qdq_rows_padded, silu


def _row_terms(x_t, dY_t, g, Wu, Wg, Wd, out="fp32"):
    rnd = out_round(out)
    U = x_t @ Wu
    V = x_t @ Wg
    h = bf16_round(silu(V) * U)
    O = rnd(h @ Wd)
    res = {"O": O}
    if dY_t is not None:
        U, V = bf16_round(U), bf16_round(V)   # as kept for the backward
        D = Wd @ dY_t                      # = dY_t W_down^T
        hv = silu(V) * U
        res["dg"] = float(D @ hv)
        du = g * D * silu(V)
        dv = g * D * U * dsilu(V)
        res["dXg"] = rnd(Wu @ bf16_round(du) + Wg @ bf16_round(dv))
    return res


def token_outputs(t, x, idx, gates, weights, dY=None, shared=None, Wr=None, out="fp32"):
    """y_t, and with dY: dX_t and dg_t (the k router-weight gradients) for token t.
    weights(e) -> (W_up[e], W_gate[e], W_down[e]) float64; shared = (Ws_up, Ws_gate,
    Ws_down) float64 or None; Wr [H][E] float64 or None (router path of dX)."""
    rnd = out_round(out)
    x_t = np.asarray(x[t], np.float64)
    dY_t = None if dY is None else np.asarray(dY[t], np.float64)
    k = idx.shape[1]
    y = np.zeros(x_t.shape[0])
    dX = np.zeros(x_t.shape[0])
    dg = np.zeros(k)
    for j in range(k):
        e = int(idx[t, j])
        g = float(gates[t, j])
        r = _row_terms(x_t, dY_t, g, *weights(e), out=out)
        y += g * r["O"]
        if dY_t is not None:
            dg[j] = r["dg"]
            dX += r["dXg"]
    if shared is not None:
        Ws_up, Ws_gate, Ws_down = shared
        u = x_t @ Ws_up
        v = x_t @ Ws_gate
        y += rnd(bf16_round(silu(v) * u) @ Ws_down)
        if dY_t is not None:
            u, v = bf16_round(u), bf16_round(v)   # as kept for the backward
            D = Ws_down @ dY_t
            du = D * silu(v)
            dv = D * u * dsilu(v)
            dX += rnd(Ws_up @ bf16_round(du) + Ws_gate @ bf16_round(dv))
    res = {"y": rnd(y), "y_unrounded": y}
    if dY_t is not None:
        if Wr is not None:
            s = float((gates[t] * dg).sum())
            dl = gates[t] * (dg - s)
            for j in range(k):
                dX += dl[j] * Wr[:, int(idx[t, j])]
        res["dX"] = rnd(dX)
        res["dX_unrounded"] = dX
        res["dgates"] = dg
    return res


def expert_rows(plan, e):
    """(token, slot) pairs of expert e in table order."""
    return plan.table[plan.offsets[e]:plan.offsets[e + 1]]


def dw_elements(e, pairs, x, dY, gates, Wu, Wg, Wd, picks, plain=False):
    """Elements of expert e's weight gradients. pairs: [n, 2] (t, j) rows of e;
    picks: list of (name, a, b) with name in dW_up (a=h, b=i), dW_gate (a=h, b=i),
    dW_down (a=i, b=h). Wu, Wg [H][I], Wd [I][H] float64."""
    rnd = bf16_round if plain else (lambda v: v)
    t = pairs[:, 0]
    g = np.asarray(gates[t, pairs[:, 1]], np.float64)
    X = np.asarray(x[t], np.float64)
    dYe = np.asarray(dY[t], np.float64)
    out = []
    for name, a, b in picks:
        if len(t) == 0:
            out.append(0.0)
            continue
        if name == "dW_down":
            i, h = a, b
            U = bf16_round(X @ Wu[:, i])   # U, V as kept for the backward
            V = bf16_round(X @ Wg[:, i])
            hg = rnd(g * silu(V) * U)
            out.append(float(hg @ dYe[:, h]))
        else:
            h, i = a, b
            U = bf16_round(X @ Wu[:, i])
            V = bf16_round(X @ Wg[:, i])
            D = dYe @ Wd[i, :]
            if name == "dW_up":
                d = rnd(g * D * silu(V))
            else:
                d = rnd(g * D * U * dsilu(V))
            out.append(float(X[:, h] @ d))
    return np.array(out)


# ----------------------------------------------------------------------------- whole dW lines
def dw_lines(pairs, x, dY, gates, Wu, Wg, Wd, i, plain=False, out="fp32"):
    """For one expert (its table rows ``pairs``) and one intermediate index i: the row
    dW_down[e][i, :] (length H) and the columns dW_up[e][:, i], dW_gate[e][:, i]
    (length H); du, dv, g*h unrounded (rounded to bf16 with ``plain``); each line rounded
    to the result type."""
    rnd = bf16_round if plain else (lambda v: v)
    t = pairs[:, 0]
    g = np.asarray(gates[t, pairs[:, 1]], np.float64)
    X = np.asarray(x[t], np.float64)
    dYe = np.asarray(dY[t], np.float64)
    U = bf16_round(X @ Wu[:, i])   # U, V as kept for the backward
    V = bf16_round(X @ Wg[:, i])
    D = dYe @ Wd[i, :]
    hg = rnd(g * silu(V) * U)
    du = rnd(g * D * silu(V))
    dv = rnd(g * D * U * dsilu(V))
    ro = out_round(out)
    return {"dW_down": ro(hg @ dYe), "dW_up": ro(X.T @ du), "dW_gate": ro(X.T @ dv)}


# ----------------------------------------------------------------------------- MXFP8 forward
def mx_expert_weights(Wu, Wg, Wd):
    """The MXFP8 values the forward GEMMs see for one expert: W_up, W_gate quantised in
    blocks of 32 along H, W_down in blocks of 32 along I."""
    return mx_qdq(Wu, 0), mx_qdq(Wg, 0), mx_qdq(Wd, 0)


def token_forward_mx(t, x, idx, gates, weights_q, shared=None, out="fp32"):
    """y_t in MXFP8 mode: x_t in blocks of 32 along H, h in blocks of 32 along I; the
    shared expert BF16 (h rounded to bf16). weights_q(e) -> mx_expert_weights(...)."""
    rnd = out_round(out)
    x_t = np.asarray(x[t], np.float64)
    xq = mx_qdq(x_t[None, :], 1)[0]
    y = np.zeros(x_t.shape[0])
    for j in range(idx.shape[1]):
        Wu, Wg, Wd = weights_q(int(idx[t, j]))
        U = xq @ Wu
        V = xq @ Wg
        hq = mx_qdq((silu(V) * U)[None, :], 1)[0]
        y += float(gates[t, j]) * rnd(hq @ Wd)
    if shared is not None:
        Ws_up, Ws_gate, Ws_down = shared
        u = x_t @ Ws_up
        v = x_t @ Ws_gate
        y += rnd(bf16_round(silu(v) * u) @ Ws_down)
    return rnd(y)


# ----------------------------------------------------------------------------- MXFP8 backward
def mx_expert_weights_bwd(Wu, Wg, Wd, hs):
    """What the MXFP8 GEMMs of one token's backward see of one expert: W_up, W_gate in
    blocks of 32 along H (the forward's U, V), W_down in blocks along H (dH GEMM), and rows
    ``hs`` of W_up, W_gate in blocks along I (dX GEMM; a row's blocks lie in that row)."""
    hs = np.asarray(hs)
    return mx_qdq(Wu, 0), mx_qdq(Wg, 0), mx_qdq(Wd, 1), mx_qdq(Wu[hs], 1), mx_qdq(Wg[hs], 1)


def token_backward_mx(t, x, idx, gates, weights_q, dY, Wr=None, out="fp32"):
    """MXFP8 mode, token t: the k router-weight gradients dg_t and dX_t at the hidden
    indices the weights were cut to (``weights_q(e)`` -> mx_expert_weights_bwd(..., hs)).
    D = dY_t W_down^T with dY_t and W_down in blocks along H; dg = D . (silu(V) U);
    du = g D silu(V), dv = g D U silu'(V), each in blocks along I before the dX GEMM;
    with Wr ([H][E], rows hs only) the router path dl Wr^T is added. With bf16 results
    the routed dX rows and the sum are rounded (the rows are rounded over the hidden
    indices given, which is what the full rows' rounding gives there)."""
    rnd = out_round(out)
    x_t = np.asarray(x[t], np.float64)
    xq = mx_qdq(x_t[None, :], 1)[0]
    dYq = mx_qdq(np.asarray(dY[t], np.float64)[None, :], 1)[0]
    k = idx.shape[1]
    dg = np.zeros(k)
    dX = None
    for j in range(k):
        e = int(idx[t, j])
        g = float(gates[t, j])
        Wu, Wg, Wd, Wu_rows, Wg_rows = weights_q(e)
        U = bf16_round(xq @ Wu)          # U, V as saved for the backward
        V = bf16_round(xq @ Wg)
        D = Wd @ dYq
        dg[j] = float(D @ (silu(V) * U))
        du = mx_qdq((g * D * silu(V))[None, :], 1)[0]
        dv = mx_qdq((g * D * U * dsilu(V))[None, :], 1)[0]
        part = rnd(Wu_rows @ du + Wg_rows @ dv)
        dX = part if dX is None else dX + part
    if Wr is not None:
        s = float((gates[t] * dg).sum())
        dl = gates[t] * (dg - s)
        for j in range(k):
            dX = dX + dl[j] * np.asarray(Wr, np.float64)[:, int(idx[t, j])]
    return {"dX": rnd(dX), "dX_unrounded": dX, "dgates": dg}


def dw_lines_mx(pairs, x, dY, gates, Wu, Wg, Wd, i_list, out="fp32"):
    """MXFP8 mode, one expert (its table rows ``pairs``), for each i in ``i_list``: the
    row dW_down[e][i, :] and the columns dW_up[e][:, i], dW_gate[e][:, i]. U, V from x in
    blocks along H and W_up, W_gate columns in blocks along H; D from dY in blocks along
    H and the W_down row in blocks along H; then g*h, du, dv, x and dY in blocks of 32
    expert rows (the last block completed with zero rows); each line rounded to the
    result type."""
    ro = out_round(out)
    t = pairs[:, 0]
    g = np.asarray(gates[t, pairs[:, 1]], np.float64)
    X = np.asarray(x[t], np.float64)
    dYe = np.asarray(dY[t], np.float64)
    Xq = mx_qdq(X, 1)
    dYq = mx_qdq(dYe, 1)
    XR = mx_qdq_rows_padded(X)
    dYR = mx_qdq_rows_padded(dYe)
    res = {}
    for i in i_list:
        U = bf16_round(Xq @ mx_qdq(Wu[:, i:i + 1], 0)[:, 0])   # as saved for the backward
        V = bf16_round(Xq @ mx_qdq(Wg[:, i:i + 1], 0)[:, 0])
        D = dYq @ mx_qdq(Wd[i:i + 1, :], 1)[0]
        col = lambda v: mx_qdq_rows_padded(v[:, None])[:, 0]
        hg = col(g * silu(V) * U)
        du = col(g * D * silu(V))
        dv = col(g * D * U * dsilu(V))
        res[i] = {"dW_down": ro(hg @ dYR), "dW_up": ro(XR.T @ du), "dW_gate": ro(XR.T @ dv)}
    return res


def shared_dw_lines(x, dY, Ws_up, Ws_gate, Ws_down, i, plain=False, out="fp32"):
    """Shared expert (gate 1, every token): dWs_down[i, :], dWs_up[:, i], dWs_gate[:, i],
    each rounded to the result type."""
    rnd = bf16_round if plain else (lambda v: v)
    ro = out_round(out)
    x = np.asarray(x, np.float64)
    dY = np.asarray(dY, np.float64)
    U = bf16_round(x @ Ws_up[:, i])   # U, V as kept for the backward
    V = bf16_round(x @ Ws_gate[:, i])
    D = dY @ Ws_down[i, :]
    return {"dWs_down": ro(rnd(silu(V) * U) @ dY), "dWs_up": ro(x.T @ rnd(D * silu(V))),
            "dWs_gate": ro(x.T @ rnd(D * U * dsilu(V)))}
