"""Parity at full size, in the launch sequence bench.py times (MoELayer plan + forward +
backward), on outputs the oracle can compute one at a time: routing and the whole
schedule exactly; sampled tokens' y, dX and router-weight gradients; whole rows and
columns of the weight gradients. The error of a sampled set is max|gpu - oracle| over
the RMS of the oracle's values in that set."""
import numpy as np
import pytest
import torch

import moe_inputs as mi
from oracle import moe, sampled
from tests import gpu_util as gu

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


def f64(t):
    return t.detach().float().cpu().double().numpy()


def err(gpu, ref):
    ref = np.asarray(ref, np.float64)
    return float(np.abs(np.asarray(gpu, np.float64) - ref).max() / np.sqrt((ref ** 2).mean()))


def _run(cfg, seed, backward):
    inp = mi.make_inputs(cfg, seed=seed, device="cuda", with_dy=backward)
    L = gu.make_layer(cfg)
    if cfg.router:
        L.plan(x=inp["x"], Wr=inp["Wr"], bias=inp["bias"])
    else:
        L.plan(topk_idx=inp["topk_idx"], gates=inp["gates"])
    mx = L.quantize_weights(inp["W_up"], inp["W_gate"], inp["W_down"]) \
        if cfg.precision == "mxfp8" else None
    w = L.weights(inp["W_up"], inp["W_gate"], inp["W_down"], inp["Ws_up"], inp["Ws_gate"],
                  inp["Ws_down"], mx=mx)
    y = L.forward(inp["x"], w)
    g = L.backward(inp["x"], inp["Wr"], w, inp["dY"]) if backward else None
    torch.cuda.synchronize()
    assert L.status() == 0
    return inp, L, y, g


def _check_schedule(cfg, inp, L):
    """Routing: equal to the oracle's on every token whose top-(k+1) logits are farther
    apart than the fp32 error bound; on the others the GPU's choice must be one the bound
    allows. The schedule of the GPU's expert ids is compared bit for bit. Returns the
    expert ids and the oracle's gates for those ids (fp64), for the sampled checks."""
    x = f64(inp["x"])
    gi = L.topk_idx.cpu().numpy().astype(np.int64)
    if cfg.router:
        r = moe.route(x, f64(inp["Wr"]), cfg.k, None if inp["bias"] is None else f64(inp["bias"]))
        amb = set(gu.ambiguous_tokens(cfg, inp, r.logits).tolist())
        diff = np.where((gi != r.idx).any(axis=1))[0]
        assert all(t in amb for t in diff), f"top-k differs outside near-ties: {diff[:10]}"
        if len(diff):
            bound = gu.logit_margins(cfg, inp, r.logits)[diff]
            kth = np.sort(r.logits[diff], axis=1)[:, -cfg.k]
            chosen = np.take_along_axis(r.logits[diff], gi[diff], axis=1)
            cb = np.take_along_axis(bound, gi[diff], axis=1)
            assert np.all(chosen + 2 * cb.max(1, keepdims=True) >= kth[:, None])
        m = r.logits.max(axis=1, keepdims=True)
        p = np.exp(r.logits - m)
        pS = np.take_along_axis(p, gi, axis=1)
        gates = pS / pS.sum(axis=1, keepdims=True)
        # the tensor-core router sums 3H products in its own order: observed 2e-5 at the
        # Kimi size; the layer outputs carry their own tolerance
        assert np.abs(L.gates.cpu().numpy() - gates).max() < 1e-4
        print(f"{cfg.name}: {len(amb)} near-tie tokens, {len(diff)} routed differently")
    else:
        assert np.array_equal(gi, inp["topk_idx"].cpu().numpy())
        gates = f64(inp["gates"])
    pl = moe.plan(gi, cfg.E)
    assert np.array_equal(L.counts.cpu().numpy(), pl.counts)
    assert np.array_equal(L.offsets.cpu().numpy(), pl.offsets)
    assert np.array_equal(L.table.cpu().numpy(), pl.table)
    assert np.array_equal(L.inv.cpu().numpy(), pl.inv)
    return x, gi, gates, pl


def test_kimi_8192_bf16_full_size_sampled():
    cfg = mi.CONFIGS["kimi_8192"]
    inp, L, y, g = _run(cfg, seed=7, backward=True)
    x, idx, gates, pl = _check_schedule(cfg, inp, L)
    dY = f64(inp["dY"])
    Wr = f64(inp["Wr"])
    shared = tuple(f64(inp[n]) for n in ("Ws_up", "Ws_gate", "Ws_down"))
    cache = {}

    def W(e):
        if e not in cache:
            cache.clear()
            cache[e] = tuple(f64(inp[n][e]) for n in ("W_up", "W_gate", "W_down"))
        return cache[e]

    tokens = [0, 2049, 5000, cfg.T - 1]
    gy, gdx, gdg, ry, rdx, rdg = [], [], [], [], [], []
    for t in tokens:
        o = sampled.token_outputs(t, x, idx, gates, W, dY=dY, shared=shared, Wr=Wr)
        ry.append(o["y"]); rdx.append(o["dX"]); rdg.append(o["dgates"])
        gy.append(f64(y[t])); gdx.append(f64(g["dX"][t])); gdg.append(g["dgates"][t].cpu().numpy())
    errs = {"y": err(gy, ry), "dX": err(gdx, rdx), "dgates": err(gdg, rdg)}
    # whole weight-gradient lines of the busiest expert and of a typical one
    busiest = int(np.argmax(pl.counts))
    for e in (busiest, int(idx[0, 0])):
        pairs = sampled.expert_rows(pl, e)
        Wu, Wg, Wd = W(e)
        for i in (5, cfg.I - 3):
            ref = sampled.dw_lines(pairs, x, dY, gates, Wu, Wg, Wd, i)
            for name, gv in (("dW_down", g["dW_down"][e, i, :]), ("dW_up", g["dW_up"][e, :, i]),
                             ("dW_gate", g["dW_gate"][e, :, i])):
                errs[f"{name}[{e}][{i}]"] = err(f64(gv), ref[name])
    for i in (7, cfg.shared_I - 1):
        ref = sampled.shared_dw_lines(x, dY, *shared, i)
        errs[f"dWs_down[{i}]"] = err(f64(g["dWs_down"][i, :]), ref["dWs_down"])
        errs[f"dWs_up[{i}]"] = err(f64(g["dWs_up"][:, i]), ref["dWs_up"])
        errs[f"dWs_gate[{i}]"] = err(f64(g["dWs_gate"][:, i]), ref["dWs_gate"])
    print("kimi_8192", errs)
    for k, v in errs.items():
        assert v <= gu.TOL["bf16"], (k, v)


def _mx_forward_sampled(cfg, inp, L, y, tokens):
    x, idx, gates, pl = _check_schedule(cfg, inp, L)
    cache = {}

    def Wq(e):
        if e not in cache:
            cache.clear()
            cache[e] = sampled.mx_expert_weights(*(f64(inp[n][e]) for n in
                                                   ("W_up", "W_gate", "W_down")))
        return cache[e]

    ref = [sampled.token_forward_mx(t, x, idx, gates, Wq) for t in tokens]
    got = [f64(y[t]) for t in tokens]
    e = err(got, ref)
    print(cfg.name, "y", e)
    assert e <= gu.TOL["mxfp8"]
    return pl


def test_ep64_slice_mxfp8_full_size_sampled():
    """Per-GPU slice of EP=64 (2048 tokens, 6 local experts, Zipf(1.2) loads), MXFP8,
    forward only, ring of 256 MB in 4 macrobatches."""
    cfg = mi.CONFIGS["ep64_slice"]
    inp, L, y, _ = _run(cfg, seed=3, backward=False)
    pl = _mx_forward_sampled(cfg, inp, L, y, [0, 777, cfg.T - 1])
    assert list(pl.counts) == mi.zipf_counts(cfg.T * cfg.k, cfg.E, cfg.zipf_s)


def test_dsv3_imbalanced_mxfp8_forward_sampled():
    """256 experts, 16384 tokens, router bias +3 on experts 0-3 (hot experts), MXFP8."""
    cfg = mi.CONFIGS["dsv3_imbalanced"]
    inp, L, y, _ = _run(cfg, seed=11, backward=False)
    pl = _mx_forward_sampled(cfg, inp, L, y, [1, cfg.T // 2, cfg.T - 2])
    assert pl.counts[:4].min() > 4 * np.median(pl.counts)


def test_ep64_slice_megakernel_matches_launches_full_size():
    """The full EP=64 slice through the forward megakernel (4 macrobatches, a 256 MB ring
    of 3 slots, so slots are reused) gives the same bits as one launch per step."""
    cfg = mi.CONFIGS["ep64_slice"]
    inp = mi.make_inputs(cfg, seed=3, device="cuda", with_dy=False)
    ys = {}
    for path in ("megakernel", "launches"):
        L = gu.make_layer(cfg)
        assert (L.sizes.macrobatches, L.sizes.ring_slots) == (4, 3)
        L.set_fwd_path(path)
        L.plan(topk_idx=inp["topk_idx"], gates=inp["gates"])
        mx = L.quantize_weights(inp["W_up"], inp["W_gate"], inp["W_down"])
        w = L.weights(inp["W_up"], inp["W_gate"], inp["W_down"], mx=mx)
        ys[path] = L.forward(inp["x"], w)
        torch.cuda.synchronize()
        assert L.status() == 0
        del L
    assert torch.equal(ys["megakernel"], ys["launches"])
