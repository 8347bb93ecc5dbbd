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

TOL = {"bf16": 2e-2, "mxfp8": 6e-2}


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
                    ring_bytes=cfg.ring_bytes, precision=cfg.precision, device=device)


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


def run_oracle(cfg, inp, idx, gates, backward=True, precision=None):
    precision = precision or cfg.precision
    x = np64(inp["x"])
    W = [np64(inp[n]) for n in ("W_up", "W_gate", "W_down")]
    shared = None
    if cfg.shared_I:
        shared = tuple(np64(inp[n]) for n in ("Ws_up", "Ws_gate", "Ws_down"))
    y, saved = moe.forward(x, idx, gates, *W, shared=shared, precision=precision)
    out = {"y": y, "plan": saved["plan"]}
    if backward:
        g = moe.backward(x, idx, gates, *W, saved, np64(inp["dY"]), shared=shared,
                         precision=precision, Wr=np64(inp["Wr"]) if cfg.router else None)
        out.update({"dX": g.dX, "dW_up": g.dW_up, "dW_gate": g.dW_gate, "dW_down": g.dW_down,
                    "dgates": g.dgates, "dWr": g.dWr, "dWs_up": g.dWs_up,
                    "dWs_gate": g.dWs_gate, "dWs_down": g.dWs_down})
    return out


def logit_margins(cfg, inp, logits):
    """Per-token bound on |fp32 logit - exact logit| for the GPU's sequential fp32 FMA
    sum over H terms (gamma_H * sum|x_h w_h|, plus the bias add)."""
    x = np.abs(np64(inp["x"]))
    w = np.abs(np64(inp["Wr"]))
    u = 2.0 ** -24
    gam = cfg.H * u / (1 - cfg.H * u)
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
