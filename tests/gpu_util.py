"""Helpers for the GPU parity tests: run the CUDA path through the C ABI and the fp64
oracle on the same seeded inputs, and compare.

Error metric (from the layer's acceptance bar): err = max|gpu - oracle| / rms(oracle),
gated at 2e-2 for BF16 and 6e-2 for MXFP8.
"""
from __future__ import annotations

import numpy as np
import torch

import moe_inputs as mi
from oracle import moe

TOL = {"bf16": 2e-2, "bf16_plain": 2e-2, "mxfp8": 6e-2}


def rel_err(gpu, ref) -> float:
    gpu = mi.to_f64(gpu) if isinstance(gpu, torch.Tensor) else np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    rms = np.sqrt((ref ** 2).mean())
    if rms == 0:
        return float(np.abs(gpu).max())
    return float(np.abs(gpu - ref).max() / rms)


def np64(t):
    return mi.to_f64(t)


def make_layer(cfg, device="cuda"):
    from grouped_gemm_built_gb300.layer import MoELayer
    return MoELayer(cfg.T, cfg.H, cfg.I, cfg.E, cfg.k, shared_I=cfg.shared_I,
                    router=cfg.router, macrobatches=cfg.macrobatches,
                    ring_bytes=cfg.ring_bytes, precision=cfg.precision, device=device,
                    out=cfg.out, minibatch_tokens=cfg.minibatch_tokens)


def gpu_inputs(cfg, seed=0):
    return mi.make_inputs(cfg, seed=seed, device="cpu", with_dy=True)


def to_dev(inp):
    return {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}


def run_gpu(cfg, inp_cpu, backward=True, layer=None, routing=None):
    """Plan + forward (+ backward) on the GPU. ``routing`` = (idx, gates) numpy arrays
    to feed as inputs (router-less mode). Returns numpy results and the layer."""
    d = to_dev(inp_cpu)
    L = layer or make_layer(cfg)
    if cfg.router and routing is None:
        L.plan(x=d["x"], Wr=d["Wr"], bias=d["bias"])
    elif routing is None:
        L.plan(topk_idx=d["topk_idx"], gates=d["gates"])
    else:
        idx, g = routing
        L.plan(topk_idx=torch.as_tensor(np.asarray(idx), dtype=torch.int32).cuda(),
               gates=torch.as_tensor(np.asarray(g), dtype=torch.float32).cuda())
    mx = None
    if cfg.precision == "mxfp8":
        mx = L.quantize_weights(d["W_up"], d["W_gate"], d["W_down"])
    w = L.weights(d["W_up"], d["W_gate"], d["W_down"], d["Ws_up"], d["Ws_gate"], d["Ws_down"],
                  mx=mx)
    y = L.forward(d["x"], w)
    out = {"y": y}
    if backward:
        g = L.backward(d["x"], d["Wr"] if cfg.router else None, w, d["dY"])
        out.update(g)
    torch.cuda.synchronize()
    res = {k: (v.detach().cpu() if isinstance(v, torch.Tensor) else v) for k, v in out.items()}
    res["topk_idx"] = L.topk_idx.cpu().numpy()
    res["gates"] = L.gates.cpu().numpy()
    res["counts"] = L.counts.cpu().numpy()
    res["offsets"] = L.offsets.cpu().numpy()
    res["table"] = L.table.cpu().numpy()
    res["inv"] = L.inv.cpu().numpy()
    res["status"] = L.status()
    return res, L


def oracle_route(cfg, inp):
    if cfg.router:
        r = moe.route(np64(inp["x"]), np64(inp["Wr"]), cfg.k, np64(inp["bias"]))
        return r.idx, r.gates, r.logits
    return inp["topk_idx"].numpy().astype(np.int64), np64(inp["gates"]), None


def run_oracle(cfg, inp, idx, gates, backward=True, precision=None, out=None):
    """The oracle on the same inputs; ``out`` (default: the config's) models the result
    type. ``unrounded`` holds the results before their last rounding."""
    precision = precision or cfg.precision
    out = out or cfg.out
    x = np64(inp["x"])
    W = [np64(inp[n]) for n in ("W_up", "W_gate", "W_down")]
    shared = None
    if cfg.shared_I:
        shared = tuple(np64(inp[n]) for n in ("Ws_up", "Ws_gate", "Ws_down"))
    y, saved = moe.forward(x, idx, gates, *W, shared=shared, precision=precision, out=out)
    res = {"y": y, "plan": saved["plan"], "unrounded": {"y": saved["y_unrounded"]}}
    if backward:
        g = moe.backward(x, idx, gates, *W, saved, np64(inp["dY"]), shared=shared,
                         precision=precision, Wr=np64(inp["Wr"]) if cfg.router else None,
                         out=out)
        res.update({"dX": g.dX, "dW_up": g.dW_up, "dW_gate": g.dW_gate, "dW_down": g.dW_down,
                    "dgates": g.dgates, "dWr": g.dWr, "dWs_up": g.dWs_up,
                    "dWs_gate": g.dWs_gate, "dWs_down": g.dWs_down})
        res["unrounded"].update(g.unrounded)
    return res


def logit_margins(cfg, inp, logits):
    """Per-logit bound on |GPU logit - exact logit|. The GPU sums the 3H exact products
    x_h * (hi, mid, lo parts of w_h) in fp32 on the tensor cores in an order of its own:
    any order of n rounded additions errs by at most (n-1) u sum|terms|, and an accumulator
    that truncates instead of rounding to nearest at most twice that; so
    6 H u sum|x_h w_h|, plus the bias add."""
    x = np.abs(np64(inp["x"]))
    w = np.abs(np64(inp["Wr"]))
    u = 2.0 ** -24
    gam = 6 * cfg.H * u
    return gam * (x @ w) + u * np.abs(logits) + 1e-30


def ambiguous_tokens(cfg, inp, logits):
    """Tokens whose top-(k+1) logits (oracle, fp64) are closer than the fp32 error bound:
    the GPU may legitimately order or pick them differently."""
    bound = logit_margins(cfg, inp, logits)
    order = np.argsort(-logits, axis=1, kind="stable")[:, :cfg.k + 1]
    lv = np.take_along_axis(logits, order, axis=1)
    bv = np.take_along_axis(bound, order, axis=1)
    gaps = lv[:, :-1] - lv[:, 1:]
    if cfg.k == cfg.E:
        gaps = gaps[:, :cfg.k - 1]
        bsum = (bv[:, :-1] + bv[:, 1:])[:, :cfg.k - 1]
    else:
        bsum = bv[:, :-1] + bv[:, 1:]
    return np.where((gaps <= bsum).any(axis=1))[0]


def mx_weight_offsets(E, H, I):
    """Byte offsets of the MXFP8 weight copies written by mok_quantize_weights_mxfp8
    (the library's bump layout: 256-byte aligned, in this order)."""
    def al(v):
        return (v + 255) // 256 * 256
    n = E * H * I
    names = ["up_h", "up_h_sf", "gate_h", "gate_h_sf", "down_i", "down_i_sf"]
    sizes = [n, n // 32, n, n // 32, n, n // 32]
    off, out = 0, {}
    for nm, sz in zip(names, sizes):
        out[nm] = (off, sz)
        off = al(off + sz)
    return out


def unpack_atoms(buf, E, K, N):
    """Scale bytes [E][K/32][N] from 512-byte atoms laid out [e][K/128][N/128], byte
    (m, b) of an atom at 16*(m%32) + 4*((m%128)//32) + b (m the N index, b the 32-block
    inside the atom's 128 K elements)."""
    a = np.asarray(buf).reshape(E, K // 128, N // 128, 512)
    m = np.arange(128)
    out = np.empty((E, K // 32, N), np.uint8)
    for b in range(4):
        pos = 16 * (m % 32) + 4 * (m // 32) + b
        blk = a[:, :, :, pos]                      # [E, K/128, N/128, 128]
        out[:, b::4, :] = blk.reshape(E, K // 128, N)
    return out


# ----------------------------------------------------------------------------- rounding flips
def _flip_dev(a, delta):
    """Per element: how far bf16(a') can land from bf16(a) for any a' within delta of the
    exact value a (bf16 rounding is monotone, so the ends a - delta and a + delta give the
    extremes); 0 unless a rounding midpoint lies within delta of a. Returns (deviation,
    fraction of elements with a nonzero deviation)."""
    from oracle.numerics import bf16_round
    r = bf16_round(a)
    dev = np.maximum(np.abs(bf16_round(a + delta) - r), np.abs(bf16_round(a - delta) - r))
    return dev, float((dev > 0).mean()) if dev.size else 0.0


def bf16_flip_slack(cfg, inp, idx, gates):
    """Elementwise allowance for the weight gradients in the BF16 modes with fp32 results.
    The backward reads U, V as the forward kept them, bf16 on both sides: the GPU rounds
    its fp32 sums, the oracle exact values. In bf16_plain, du, dv and g*h are rounded to
    bf16 again before the weight-gradient GEMMs; in bf16 they go in as hi + lo pairs
    (a 16-bit significand). The fp32 sums U, V, D are taken to be within
    6 sqrt(H) u sum|a b| of the exact ones (u = 2^-24): the probabilistic bound of Higham
    and Mary ("A New Approach to Probabilistic Rounding Error Analysis", 2019) with
    lambda = 6, which fails for a given sum with probability below 2 exp(-18); the
    worst-case bound H u sum|a b| flags about half of all operands at these sizes and
    would say little. A U or V within that bound of a rounding midpoint may keep another
    bf16 value; propagated to first order through SwiGLU', that moves du, dv, g*h, and in
    bf16_plain one of those within its moved bound of a midpoint may round to another bf16
    value. The slack of a dW element is the sum, over its contraction, of |other operand|
    * (largest such move) for its operands.
    Returns (dict of slack arrays shaped like the gradients, fraction of operands whose
    value may differ by a rounding flip: du, dv, g*h in bf16_plain, U, V in bf16)."""
    from oracle import moe
    from oracle.numerics import bf16_round, sigmoid
    x = np64(inp["x"])
    dY = np64(inp["dY"])
    Wu, Wg, Wd = (np64(inp[n]) for n in ("W_up", "W_gate", "W_down"))
    H = cfg.H
    u = 2.0 ** -24
    gam = 6.0 * np.sqrt(H) * u   # see the docstring
    plain = cfg.precision == "bf16_plain"

    def operand_flips(X, dYr, g, A, B, C):
        U, V, D = X @ A, X @ B, dYr @ C.T
        aX, adY = np.abs(X), np.abs(dYr)
        bU, bV, bD = gam * (aX @ np.abs(A)), gam * (aX @ np.abs(B)), gam * (adY @ np.abs(C).T)
        # the backward reads U, V kept as bf16 on both sides: they differ by the rounding
        # flip of the GPU's fp32 sums
        (bU, nU), (bV, nV) = _flip_dev(U, bU), _flip_dev(V, bV)
        U, V = bf16_round(U), bf16_round(V)
        sg = sigmoid(V)
        s0 = V * sg
        s1 = sg * (1 + V * (1 - sg))
        s2 = sg * (1 - sg) * (2 + V * (1 - 2 * sg))
        ag = np.abs(g)
        du, dv, hg = g * D * s0, g * D * U * s1, g * s0 * U
        d_du = ag * (bD * np.abs(s0) + np.abs(D * s1) * bV) + 8 * u * np.abs(du)
        d_dv = ag * (bD * np.abs(U * s1) + np.abs(D * s1) * bU + np.abs(D * U * s2) * bV) \
            + 8 * u * np.abs(dv)
        d_hg = ag * (np.abs(s1 * U) * bV + np.abs(s0) * bU) + 8 * u * np.abs(hg)
        if plain:
            f_du, n1 = _flip_dev(du, d_du)
            f_dv, n2 = _flip_dev(dv, d_dv)
            f_hg, n3 = _flip_dev(hg, d_hg)
            n = (n1 + n2 + n3) / 3
        else:   # hi + lo operands: their bound, plus the pair's 2^-17
            hl = 2.0 ** -17
            f_du, f_dv, f_hg = (d + hl * np.abs(v) for d, v in
                                ((d_du, du), (d_dv, dv), (d_hg, hg)))
            n = (nU + nV) / 2
        return (aX.T @ f_du, aX.T @ f_dv, f_hg.T @ adY), n

    pl = moe.plan(idx, cfg.E)
    out = {"dW_up": np.zeros(Wu.shape), "dW_gate": np.zeros(Wg.shape),
           "dW_down": np.zeros(Wd.shape)}
    fr, n = [], []
    for e in range(cfg.E):
        r0, r1 = pl.offsets[e], pl.offsets[e + 1]
        if r0 == r1:
            continue
        t, j = pl.table[r0:r1, 0], pl.table[r0:r1, 1]
        g = gates[t, j][:, None]
        (su, sgt, sd), f = operand_flips(x[t], dY[t], g, Wu[e], Wg[e], Wd[e])
        out["dW_up"][e], out["dW_gate"][e], out["dW_down"][e] = su, sgt, sd
        fr.append(f * (r1 - r0))
        n.append(r1 - r0)
    if cfg.shared_I:
        Su, Sg, Sd = (np64(inp[n_]) for n_ in ("Ws_up", "Ws_gate", "Ws_down"))
        (su, sgt, sd), _ = operand_flips(x, dY, np.ones((cfg.T, 1)), Su, Sg, Sd)
        out["dWs_up"], out["dWs_gate"], out["dWs_down"] = su, sgt, sd
    return out, float(sum(fr) / max(sum(n), 1))


def rel_err_slack(gpu, ref, slack) -> float:
    """max(|gpu - oracle| - slack, 0) / rms(oracle)."""
    gpu = mi.to_f64(gpu) if isinstance(gpu, torch.Tensor) else np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    rms = np.sqrt((ref ** 2).mean())
    ex = np.maximum(np.abs(gpu - ref) - slack, 0.0)
    return float(ex.max() / rms) if rms else float(ex.max())
