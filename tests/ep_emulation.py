"""Expert parallelism emulated on one GPU (test harness around the C ABI).

Under expert parallelism each of P ranks owns E/P experts; a token's rows travel to the
ranks that own its experts (dispatch) and their outputs travel back (combine). The MoK
articles build that exchange from one table built on the GPU: for every expert row, its
source (rank, token), in an order that follows from the routing, reused by the dispatch,
the combine and their reverses ("Push oder Pull?" and "Das Scheduling" on the sebask.de
page; "Escolha da direção de comunicação" on the stamatios.com page).

On one GPU the P ranks are P expert slices, each a router-less layer of its own (E/P
experts, one slot per row, the row's gate). The schedule that connects them is built on
the host from the one global table ``mok_plan`` writes: because the table lists the rows
expert by expert, slice s's rows are the contiguous run of table rows of its experts, in
the table's (token, slot) order; the slice pulls those rows of x (and of dY) by token,
and pushes each output row back to its (token, slot). Nothing else is shared: every slice
runs the library's own plan, forward and backward.

Results match the single-layer run: a slice's expert GEMMs see the same rows in the same
order, so its expert outputs, dX rows, weight gradients and router-weight gradients are
the single layer's, bit for bit; y and dX are sums over the k slots, which the harness
adds up in slot order (the single layer fuses the gate into that sum, so y may differ in
the last bits).
"""
from __future__ import annotations

import dataclasses

import numpy as np
import torch


@dataclasses.dataclass
class Slice:
    experts: tuple          # [e0, e1): the experts this slice owns
    rows: np.ndarray        # global table rows, in table order
    tokens: np.ndarray      # source token of each row
    slots: np.ndarray       # slot j of each row
    local_expert: np.ndarray


def cross_slice_schedule(counts, offsets, table, E: int, P: int):
    """Per slice, the global table rows of its experts (a contiguous run, since the table
    lists rows expert by expert), their tokens, slots and local expert ids."""
    counts, offsets, table = (np.asarray(a) for a in (counts, offsets, table))
    if E % P:
        raise ValueError("E must be a multiple of the number of slices")
    per = E // P
    out = []
    for s in range(P):
        e0, e1 = s * per, (s + 1) * per
        r0, r1 = int(offsets[e0]), int(offsets[e1])
        rows = np.arange(r0, r1)
        local = np.repeat(np.arange(per), counts[e0:e1])
        out.append(Slice((e0, e1), rows, table[r0:r1, 0].copy(), table[r0:r1, 1].copy(), local))
    return out


def run_ep(cfg, d, P: int, backward=True):
    """Plan on the whole batch, then P router-less slices, pull dispatch and push
    combine by the cross-slice schedule. ``d``: device inputs (moe_inputs names), fp32
    results. Returns (results dict, slices)."""
    from grouped_gemm_built_gb300.layer import MoELayer
    T, H, I, E, k = cfg.T, cfg.H, cfg.I, cfg.E, cfg.k
    g_layer = MoELayer(T, H, I, E, k, router=True, out="fp32")
    g_layer.plan(x=d["x"], Wr=d["Wr"], bias=d["bias"])
    torch.cuda.synchronize()
    sched = cross_slice_schedule(g_layer.counts.cpu().numpy(), g_layer.offsets.cpu().numpy(),
                                 g_layer.table.cpu().numpy(), E, P)
    gates = g_layer.gates
    y_rows = torch.zeros((T, k, H), dtype=torch.float32, device="cuda")
    dx_rows = torch.zeros((T, k, H), dtype=torch.float32, device="cuda")
    dgates = torch.zeros((T, k), dtype=torch.float32, device="cuda")
    dW = {n: torch.zeros(d[n].shape, dtype=torch.float32, device="cuda")
          for n in ("W_up", "W_gate", "W_down")}
    for sl in sched:
        n = len(sl.rows)
        if n == 0:
            continue
        e0, e1 = sl.experts
        tok = torch.as_tensor(sl.tokens, dtype=torch.long, device="cuda")
        slot = torch.as_tensor(sl.slots, dtype=torch.long, device="cuda")
        L = MoELayer(n, H, I, e1 - e0, 1, router=False, out="fp32")
        L.plan(topk_idx=torch.as_tensor(sl.local_expert, dtype=torch.int32, device="cuda")
               .reshape(n, 1),
               gates=gates[tok, slot].reshape(n, 1).contiguous())
        xs = d["x"].index_select(0, tok).contiguous()          # pull dispatch
        w = L.weights(d["W_up"][e0:e1].contiguous(), d["W_gate"][e0:e1].contiguous(),
                      d["W_down"][e0:e1].contiguous())
        ys = L.forward(xs, w)
        y_rows[tok, slot] = ys                                  # push combine, by (t, j)
        if backward:
            dys = d["dY"].index_select(0, tok).contiguous()     # reverse dispatch
            g = L.backward(xs, None, w, dys)
            dx_rows[tok, slot] = g["dX"]                        # reverse combine
            dgates[tok, slot] = g["dgates"].reshape(-1)
            dW["W_up"][e0:e1] = g["dW_up"]
            dW["W_gate"][e0:e1] = g["dW_gate"]
            dW["W_down"][e0:e1] = g["dW_down"]
        torch.cuda.synchronize()
        assert L.status() == 0
    # slot-ordered sums of the pushed rows
    y = y_rows[:, 0].clone()
    for j in range(1, k):
        y += y_rows[:, j]
    res = {"y": y, "topk_idx": g_layer.topk_idx, "gates": gates}
    if backward:
        dX = dx_rows[:, 0].clone()
        for j in range(1, k):
            dX += dx_rows[:, j]
        # router path: renormalised-softmax backward with the chosen set fixed
        s = (gates * dgates).sum(dim=1, keepdim=True)
        dl = gates * (dgates - s)
        dlog = torch.zeros((T, E), dtype=torch.float32, device="cuda")
        dlog.scatter_add_(1, g_layer.topk_idx.long(), dl)
        dX += dlog @ d["Wr"].t()
        res.update({"dX": dX, "dgates": dgates, "dW_up": dW["W_up"], "dW_gate": dW["W_gate"],
                    "dW_down": dW["W_down"], "dWr": d["x"].float().t() @ dlog})
    return res, sched
