"""fp64 CPU oracle of the MoE SwiGLU layer: routing, schedule, experts, combine, backward.

TEST INFRASTRUCTURE ONLY (see oracle/__init__.py): the plain definition of what the layer
computes, in NumPy float64, streamed one expert at a time. No blocking, fusion or
reordering beyond the definition.

What the articles fix, and where:
* tokens go from a router to a selection of experts; each expert is a small feed-forward
  net with an up, a gate and a down projection ("Mixture-of-Kittens: Cursors
  Open-Source-Ansatz ...", sebask.de, intro);
* the expert non-linearity is SwiGLU and the router-weight gradient is computed inside the
  SwiGLU backward ("Cursor abre código de megakernel MoE para GPUs NVL72",
  stamatios.com, section "Outras características"; ihal.it article, paragraph on BF16,
  MXFP8, router weights and SwiGLU);
* dispatch follows a pull-style schedule: for every expert row, the source token index
  (and, here, its top-k slot), in an order that follows from the routing with no sort,
  and the one table serves all four exchange steps (sebask.de, sections "Push oder Pull?"
  and "Das Scheduling"; stamatios.com, section "Escolha da direção de comunicação");
* an always-on shared expert runs in BF16 next to the routed experts (stamatios.com,
  "Outras características").

Readings taken where the pages are silent (each is also listed in the design notes):
* router: logits l = x Wr (+ bias); p = softmax(l); S = the k largest (larger value first,
  ties to the lower expert index); gates g_j = p_j / sum_{i in S} p_i. Selection is made on
  l, which orders exactly like p;
* slot order j = 0..k-1 is the top-k order (descending gate, ties to the lower expert);
* SwiGLU: h = silu(x W_gate) * (x W_up); the gate multiplies the expert output at the
  combine: y_t = sum_j g_tj O_(t,j) (+ shared expert output, weight 1);
* schedule order inside an expert: ascending token, then ascending slot;
* gradients at the top-k boundary are taken with the selected set S held fixed.

Precision model (``precision``): "fp64" applies no rounding at all. "bf16" (the articles'
BF16 mode: bf16 tensor-core operands, fp32 accumulation) rounds h, the down GEMM's
operand, and du, dv as operands of the dX GEMM to bf16; the GPU feeds du, dv and g*h to
the weight-gradient GEMMs as bf16 hi + lo pairs (a 16-bit significand), so there they
stay unrounded here; expert outputs, routed dX rows and all results stay unrounded too
(the GPU keeps them in fp32 until the result's own rounding). "bf16_plain" is "bf16" with
du, dv and g*h rounded to bf16 for the weight-gradient GEMMs as well. "mxfp8" quantises
every GEMM operand to MXFP8 blocks of 32 along that GEMM's contraction axis (inputs,
weights, h, du, dv, g*h, dY). Every mode but "fp64" keeps U, V for the backward as bf16
values, the routed experts' and the shared expert's (h is formed from the unrounded
ones in the forward; the backward's SwiGLU', du, dv and g*h read the kept values).
Everything else is float64. The shared expert is always BF16: single bf16
weight-gradient operands in "bf16_plain", hi/lo ones in "bf16" and "mxfp8".

Result type (``out``): "fp32" keeps every result unrounded (the GPU writes fp32, whose
rounding the comparison's tolerance covers). "bf16" models bf16 results: each expert output
row O and the shared expert's output, each routed dX row and the shared expert's dX, and
then y, dX and every weight gradient are rounded to bf16 once (nearest, ties to even); the
combines add the rounded rows up exactly and round their sum. dgates and dWr stay
unrounded. The values just before the last rounding are kept (``y_unrounded`` in the
forward's saved dict, ``Grads.unrounded``), since a result that lies close to a bf16
rounding midpoint may round either way on a GPU that sums in fp32.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np

from .numerics import bf16_round, dsilu, mx_qdq, mx_qdq_rows_padded, silu


# ----------------------------------------------------------------------------- routing
@dataclasses.dataclass
class Route:
    logits: np.ndarray   # [T, E] float64 (bias included)
    idx: np.ndarray      # [T, k] int64, slot order
    gates: np.ndarray    # [T, k] float64


def select(logits, k: int):
    """Top-k of softmax(logits) per row with renormalised gates: the k largest logits in
    descending order, equal logits in ascending expert order; gates = the chosen
    probabilities over their sum. Returns (idx [T, k] int64, gates [T, k] float64)."""
    logits = np.asarray(logits, np.float64)
    m = logits.max(axis=1, keepdims=True)
    p = np.exp(logits - m)
    p = p / p.sum(axis=1, keepdims=True)
    # stable sort of -l: equal logits keep ascending expert order
    order = np.argsort(-logits, axis=1, kind="stable")
    idx = order[:, :k]
    pS = np.take_along_axis(p, idx, axis=1)
    gates = pS / pS.sum(axis=1, keepdims=True)
    return idx.astype(np.int64), gates


def route(x, Wr, k: int, bias=None) -> Route:
    """Softmax top-k router with renormalised gates (reading stated in the module doc)."""
    x = np.asarray(x, np.float64)
    logits = x @ np.asarray(Wr, np.float64)
    if bias is not None:
        logits = logits + np.asarray(bias, np.float64)[None, :]
    idx, gates = select(logits, k)
    return Route(logits=logits, idx=idx, gates=gates)


# ----------------------------------------------------------------------------- schedule
@dataclasses.dataclass
class Plan:
    counts: np.ndarray   # [E] rows per expert
    offsets: np.ndarray  # [E+1] exclusive prefix sum of counts
    table: np.ndarray    # [R, 2] (token t, slot j) for every expert row
    inv: np.ndarray      # [T, k] expert row of (t, j)


def plan(idx, E: int) -> Plan:
    """Pull-style schedule: expert e's rows are offsets[e] .. offsets[e+1]-1, holding the
    (token, slot) pairs routed to e in ascending (token, slot) order."""
    idx = np.asarray(idx, np.int64)
    T, k = idx.shape
    flat = idx.reshape(-1)                  # slot id s = t*k + j, ascending in (t, j)
    counts = np.bincount(flat, minlength=E)
    offsets = np.zeros(E + 1, np.int64)
    offsets[1:] = np.cumsum(counts)
    order = np.argsort(flat, kind="stable")  # grouped by expert, slot ids ascending inside
    table = np.stack([order // k, order % k], axis=1)
    inv = np.empty(T * k, np.int64)
    inv[order] = np.arange(T * k)
    return Plan(counts=counts, offsets=offsets, table=table, inv=inv.reshape(T, k))


def plan_loops(idx, E: int) -> Plan:
    """The same schedule built with plain Python loops (brute force, small cases)."""
    idx = [[int(v) for v in row] for row in np.asarray(idx)]
    T, k = len(idx), len(idx[0])
    counts = [0] * E
    rows = [[] for _ in range(E)]
    for t in range(T):
        for j in range(k):
            counts[idx[t][j]] += 1
            rows[idx[t][j]].append((t, j))
    offsets = [0]
    for e in range(E):
        offsets.append(offsets[-1] + counts[e])
    table = [tj for e in range(E) for tj in rows[e]]
    inv = [[0] * k for _ in range(T)]
    for r, (t, j) in enumerate(table):
        inv[t][j] = r
    return Plan(counts=np.array(counts), offsets=np.array(offsets),
                table=np.array(table, dtype=np.int64).reshape(-1, 2),
                inv=np.array(inv, dtype=np.int64))


# ----------------------------------------------------------------------------- precision
class Precision:
    """Where the GPU path rounds. See the module docstring."""

    def __init__(self, mode: str):
        if mode not in ("fp64", "bf16", "bf16_plain", "mxfp8"):
            raise ValueError(mode)
        self.mode = mode

    @property
    def mx(self):
        return self.mode == "mxfp8"

    def op(self, a, axis):
        """A GEMM operand that is already bf16-exact (inputs, weights): MXFP8 blocks of 32
        along the contraction axis ``axis`` in mxfp8 mode, unchanged otherwise."""
        return mx_qdq(a, axis) if self.mx else a

    def op_rows(self, a):
        """A GEMM operand whose contraction axis is the (ragged) expert-row axis 0."""
        return mx_qdq_rows_padded(a) if self.mx else a

    def fwd_act(self, a, axis):
        """h, the forward down GEMM's operand: bf16, or MXFP8 blocks along ``axis``."""
        if self.mode == "fp64":
            return a
        return mx_qdq(a, axis) if self.mx else bf16_round(a)

    def dx_act(self, a, axis):
        """du, dv feeding the dX GEMM along ``axis`` (I): bf16, or MXFP8 blocks."""
        return self.fwd_act(a, axis)

    def saved_uv(self, a):
        """U, V as kept for the backward: bf16 values (unrounded in fp64 mode)."""
        return a if self.mode == "fp64" else bf16_round(a)

    def bwd_act_rows(self, a):
        """du, dv, g*h feeding a weight-gradient GEMM (K = expert rows): MXFP8 blocks of 32
        rows in mxfp8 mode, bf16 in bf16_plain mode; bf16 mode carries them as a bf16
        hi + lo pair, which this model takes as exact (the pair's error, 2^-16 relative,
        is far below the comparison's tolerance)."""
        if self.mx:
            return mx_qdq_rows_padded(a)
        if self.mode == "bf16_plain":
            return bf16_round(a)
        return a


# ----------------------------------------------------------------------------- results
def out_round(out: str):
    """The rounding of a result of type ``out``: bf16 for "bf16", none for "fp32"."""
    if out not in ("fp32", "bf16"):
        raise ValueError(out)
    return bf16_round if out == "bf16" else (lambda v: v)


# ----------------------------------------------------------------------------- forward
def shared_forward(x, Ws_up, Ws_gate, Ws_down, mode: str, out: str = "fp32"):
    """Always-on shared expert (BF16 in the bf16 and mxfp8 modes), gate 1; its output
    is a result row, rounded to the result type."""
    P = Precision("fp64" if mode == "fp64" else "bf16")
    U = x @ Ws_up
    V = x @ Ws_gate
    h = P.fwd_act(silu(V) * U, 1)
    O = out_round(out)(h @ Ws_down)
    return O, {"Us": P.saved_uv(U), "Vs": P.saved_uv(V)}


def forward(x, idx, gates, W_up, W_gate, W_down, shared=None, precision="fp64",
            expert_fn=None, out="fp32"):
    """Layer forward. ``shared`` = (Ws_up, Ws_gate, Ws_down) or None.
    ``expert_fn(e, Xe)`` (test hook) replaces expert e's FFN with any row-wise map.
    ``out``: the result type (module docstring). Returns (y [T,H] float64, saved dict)."""
    P = Precision(precision)
    rnd = out_round(out)
    x = np.asarray(x, np.float64)
    T, H = x.shape
    E = W_up.shape[0]
    k = idx.shape[1]
    pl = plan(idx, E)
    R = T * k
    I = W_up.shape[2]
    O_rows = np.zeros((R, H))
    U_s = np.zeros((R, I))
    V_s = np.zeros((R, I))
    for e in range(E):
        r0, r1 = pl.offsets[e], pl.offsets[e + 1]
        if r0 == r1:
            continue
        Xe = x[pl.table[r0:r1, 0]]                      # dispatch: pull rows by table
        if expert_fn is not None:
            O_rows[r0:r1] = expert_fn(e, Xe)
            continue
        A = P.op(Xe, 1)
        U = A @ P.op(W_up[e], 0)
        V = A @ P.op(W_gate[e], 0)
        h = P.fwd_act(silu(V) * U, 1)
        O_rows[r0:r1] = rnd(h @ P.op(W_down[e], 0))
        U_s[r0:r1] = P.saved_uv(U)
        V_s[r0:r1] = P.saved_uv(V)
    y = np.zeros((T, H))
    for j in range(k):                                  # combine in slot order
        y += gates[:, j:j + 1] * O_rows[pl.inv[:, j]]
    saved = {"plan": pl, "U": U_s, "V": V_s}
    if shared is not None:
        Os, ss = shared_forward(x, *shared, precision, out)
        y = y + Os
        saved.update(ss)
    saved["y_unrounded"] = y
    return rnd(y), saved


# ----------------------------------------------------------------------------- backward
@dataclasses.dataclass
class Grads:
    dX: np.ndarray
    dW_up: np.ndarray
    dW_gate: np.ndarray
    dW_down: np.ndarray
    dgates: np.ndarray
    dlogits: Optional[np.ndarray] = None
    dWr: Optional[np.ndarray] = None
    dWs_up: Optional[np.ndarray] = None
    dWs_gate: Optional[np.ndarray] = None
    dWs_down: Optional[np.ndarray] = None
    # the results before their last rounding (the same values when out is "fp32")
    unrounded: Optional[dict] = None


def shared_backward(x, Ws_up, Ws_gate, Ws_down, saved, dY, mode: str, out: str = "fp32"):
    """Shared expert backward: BF16 (single bf16 weight-gradient operands in bf16_plain,
    hi/lo ones in the bf16 and mxfp8 modes). dXs is a result row, rounded to the result
    type; the weight gradients are returned unrounded."""
    P = Precision(mode if mode in ("fp64", "bf16_plain") else "bf16")
    Us, Vs = saved["Us"], saved["Vs"]
    D = dY @ Ws_down.T
    hv = silu(Vs) * Us
    du = D * silu(Vs)
    dv = D * Us * dsilu(Vs)
    dXs = out_round(out)(P.dx_act(du, 1) @ Ws_up.T + P.dx_act(dv, 1) @ Ws_gate.T)
    dWs_down = P.bwd_act_rows(hv).T @ dY
    dWs_up = x.T @ P.bwd_act_rows(du)
    dWs_gate = x.T @ P.bwd_act_rows(dv)
    return dXs, dWs_up, dWs_gate, dWs_down


def router_backward(x, Wr, idx, gates, dgates):
    """Gradient of the renormalised top-k softmax with S fixed:
    dl_i = g_i (dg_i - sum_j g_j dg_j) for i in S, 0 elsewhere; dWr = x^T dl;
    dx = dl Wr^T."""
    T, k = idx.shape
    E = Wr.shape[1]
    s = (gates * dgates).sum(axis=1, keepdims=True)
    dlS = gates * (dgates - s)
    dl = np.zeros((T, E))
    for j in range(k):
        np.add.at(dl, (np.arange(T), idx[:, j]), dlS[:, j])
    return dl, x.T @ dl, dl @ np.asarray(Wr, np.float64).T


def backward(x, idx, gates, W_up, W_gate, W_down, saved, dY, shared=None,
             precision="fp64", Wr=None, out="fp32"):
    """Layer backward for upstream gradient dY; ``out``: the result type (module
    docstring). Returns Grads (float64)."""
    P = Precision(precision)
    rnd = out_round(out)
    x = np.asarray(x, np.float64)
    dY = np.asarray(dY, np.float64)
    T, H = x.shape
    E = W_up.shape[0]
    k = idx.shape[1]
    pl = saved["plan"]
    R = T * k
    dXg = np.zeros((R, H))
    dgates = np.zeros((T, k))
    dW_up = np.zeros(W_up.shape)
    dW_gate = np.zeros(W_gate.shape)
    dW_down = np.zeros(W_down.shape)
    for e in range(E):
        r0, r1 = pl.offsets[e], pl.offsets[e + 1]
        if r0 == r1:
            continue
        t = pl.table[r0:r1, 0]
        j = pl.table[r0:r1, 1]
        g = gates[t, j][:, None]
        Xe = x[t]
        dYe = dY[t]                                      # reverse dispatch
        Us, Vs = saved["U"][r0:r1], saved["V"][r0:r1]
        D = P.op(dYe, 1) @ P.op(W_down[e], 1).T          # rows x I
        hv = silu(Vs) * Us
        dgates[t, j] = (D * hv).sum(axis=1)              # router-weight gradient
        dh = g * D
        du = dh * silu(Vs)
        dv = dh * Us * dsilu(Vs)
        dXg[r0:r1] = rnd(P.dx_act(du, 1) @ P.op(W_up[e], 1).T
                          + P.dx_act(dv, 1) @ P.op(W_gate[e], 1).T)
        dW_down[e] = P.bwd_act_rows(g * hv).T @ P.op_rows(dYe)
        XR = P.op_rows(Xe)
        dW_up[e] = XR.T @ P.bwd_act_rows(du)
        dW_gate[e] = XR.T @ P.bwd_act_rows(dv)
    dX = np.zeros((T, H))
    for j in range(k):                                   # reverse combine in slot order
        dX += dXg[pl.inv[:, j]]
    res = Grads(dX=dX, dW_up=dW_up, dW_gate=dW_gate, dW_down=dW_down, dgates=dgates)
    if shared is not None:
        dXs, res.dWs_up, res.dWs_gate, res.dWs_down = shared_backward(
            x, *shared, saved, dY, precision, out)
        res.dX = res.dX + dXs
    if Wr is not None:
        res.dlogits, res.dWr, dxr = router_backward(x, Wr, idx, gates, dgates)
        res.dX = res.dX + dxr
    names = ["dX", "dW_up", "dW_gate", "dW_down"] + \
        (["dWs_up", "dWs_gate", "dWs_down"] if shared is not None else [])
    res.unrounded = {n: getattr(res, n) for n in names}
    for n in names:
        setattr(res, n, rnd(getattr(res, n)))
    return res


# ----------------------------------------------------------------------------- per token
def token_forward_bruteforce(x_t, experts, gates_t, W_up, W_gate, W_down):
    """One token's routed output, straight from the definition: sum over its slots of
    gate * down(silu(gate_proj) * up_proj), with no table, in float64."""
    y = np.zeros(W_down.shape[2])
    for e, g in zip(experts, gates_t):
        u = x_t @ W_up[e]
        v = x_t @ W_gate[e]
        y += g * ((silu(v) * u) @ W_down[e])
    return y


def layer_loss(x, Wr, bias, S, W_up, W_gate, W_down, dY, shared=None):
    """Scalar L = <y, dY> of the fp64 layer with the expert set S [T,k] held fixed and
    gates recomputed from the logits (for finite-difference checks)."""
    x = np.asarray(x, np.float64)
    logits = x @ Wr + (0 if bias is None else bias)
    lS = np.take_along_axis(logits, S, axis=1)
    pS = np.exp(lS - lS.max(axis=1, keepdims=True))
    gates = pS / pS.sum(axis=1, keepdims=True)
    y, _ = forward(x, S, gates, W_up, W_gate, W_down, shared=shared, precision="fp64")
    return float((y * dY).sum())
