"""Parity at full size, in the launch sequence bench.py times (MoELayer plan + forward +
backward, bf16 results), on outputs the oracle can compute one at a time: routing and
the whole schedule exactly; sampled tokens' y, dX and router-weight gradients; whole rows
and columns of the weight gradients. The error of a sampled set is max|gpu - oracle| over
the RMS of the oracle's values in that set, less each element's rounding allowance
(tests/out_slack.py: a bf16 step where a rounding midpoint lies within the propagated
bound; one bf16 step in MXFP8)."""
import numpy as np
import pytest
import torch

import moe_inputs as mi
from oracle import moe, sampled
from tests import gpu_util as gu
from tests import out_slack as osl

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


def f64(t):
    return t.detach().float().cpu().double().numpy()


def err(gpu, ref, slack=0.0):
    ref = np.asarray(ref, np.float64)
    ex = np.maximum(np.abs(np.asarray(gpu, np.float64) - ref) - slack, 0.0)
    return float(ex.max() / np.sqrt((ref ** 2).mean()))


def _run(cfg, seed, backward):
    inp = mi.make_inputs(cfg, seed=seed, device="cuda", with_dy=backward)
    L = gu.make_layer(cfg)
    if cfg.router:
        L.plan(x=inp["x"], Wr=inp["Wr"], bias=inp["bias"])
        torch.cuda.synchronize()
        # the router's fp32 logits (bias included) open the workspace until the forward
        L.gpu_logits = f64(L.workspace[: cfg.T * cfg.E * 4].view(torch.float32)
                           .reshape(cfg.T, cfg.E))
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
    """Routing, in three parts. (1) The GPU's fp32 logits lie inside the worst-case fp32
    error bound of the exact ones. (2) The integer decision, taken in the GPU's precision:
    the oracle's top-k of the GPU's own logits equals the GPU's expert ids on every token,
    and its gates agree to fp32 rounding. (3) Against the exact logits: a token may be
    routed differently only where the exact logits of its choice are within twice the
    largest measured logit error of the exact k-th logit. The schedule of the GPU's
    expert ids is compared bit for bit. Returns the expert ids and the oracle's gates
    (exact logits) for those ids, for the sampled checks."""
    x = f64(inp["x"])
    gi = L.topk_idx.cpu().numpy().astype(np.int64)
    if cfg.router:
        r = moe.route(x, f64(inp["Wr"]), cfg.k, None if inp["bias"] is None else f64(inp["bias"]))
        lg = L.gpu_logits
        lerr = np.abs(lg - r.logits)
        assert float((lerr / gu.logit_margins(cfg, inp, r.logits)).max()) <= 1.0
        sel_idx, sel_g = moe.select(lg, cfg.k)
        assert np.array_equal(gi, sel_idx), "top-k of the GPU's own logits differs"
        assert np.abs(L.gates.cpu().numpy() - sel_g).max() < 2e-6
        emax = float(lerr.max())
        diff = np.where((np.sort(gi, axis=1) != np.sort(r.idx, axis=1)).any(axis=1))[0]
        if len(diff):
            kth = np.sort(r.logits[diff], axis=1)[:, -cfg.k]
            chosen = np.take_along_axis(r.logits[diff], gi[diff], axis=1)
            assert np.all(chosen + 2 * emax >= kth[:, None])
        m = r.logits.max(axis=1, keepdims=True)
        p = np.exp(r.logits - m)
        pS = np.take_along_axis(p, gi, axis=1)
        gates = pS / pS.sum(axis=1, keepdims=True)
        # the tensor-core router sums 3H products in its own order: observed 2e-5 at the
        # Kimi size; the layer outputs carry their own tolerance
        assert np.abs(L.gates.cpu().numpy() - gates).max() < 1e-4
        print(f"{cfg.name}: max logit error {emax:.3g}, {len(diff)} tokens routed to another "
              f"expert set than the exact logits give")
    else:
        assert np.array_equal(gi, inp["topk_idx"].cpu().numpy())
        gates = f64(inp["gates"])
    pl = moe.plan(gi, cfg.E)
    assert np.array_equal(L.counts.cpu().numpy(), pl.counts)
    assert np.array_equal(L.offsets.cpu().numpy(), pl.offsets)
    assert np.array_equal(L.table.cpu().numpy(), pl.table)
    assert np.array_equal(L.inv.cpu().numpy(), pl.inv)
    return x, gi, gates, pl


@pytest.mark.parametrize("name,seed", [("kimi_8192", 7), ("kimi_2368", 5),
                                       ("kimi_8192_plain", 7)])
def test_kimi_bf16_full_size_sampled(name, seed):
    """Kimi-2.5 expert shape with all 384 experts on one GPU: T=8192 (about 171 rows per
    expert) and T=2368 (about 49, most experts a single partly filled row tile); and T=8192
    with single bf16 weight-gradient operands."""
    cfg = mi.CONFIGS[name]
    plain = cfg.precision == "bf16_plain"
    inp, L, y, g = _run(cfg, seed=seed, backward=True)
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

    out = cfg.out
    bf = out == "bf16"
    dgb = osl.gate_bounds(cfg, inp, idx, gates, None) if bf else None
    tokens = [0, cfg.T // 4 + 1, (5 * cfg.T) // 8, cfg.T - 1]
    gy, gdx, gdg, ry, rdx, rdg, sy, sdx = [], [], [], [], [], [], [], []
    for t in tokens:
        o = sampled.token_outputs(t, x, idx, gates, W, dY=dY, shared=shared, Wr=Wr, out=out)
        ry.append(o["y"]); rdx.append(o["dX"]); rdg.append(o["dgates"])
        gy.append(f64(y[t])); gdx.append(f64(g["dX"][t])); gdg.append(g["dgates"][t].cpu().numpy())
        if bf:
            a, b = osl.token_slack(t, x, idx, gates, dgb, W, dY=dY, shared=shared, Wr=Wr,
                                   plain=plain)
            sy.append(a); sdx.append(b)
    errs = {"y": err(gy, ry, np.array(sy) if bf else 0.0),
            "dX": err(gdx, rdx, np.array(sdx) if bf else 0.0), "dgates": err(gdg, rdg)}
    # whole weight-gradient lines of the busiest expert and of a typical one
    busiest = int(np.argmax(pl.counts))
    for e in (busiest, int(idx[0, 0])):
        pairs = sampled.expert_rows(pl, e)
        Wu, Wg, Wd = W(e)
        for i in (5, cfg.I - 3):
            ref = sampled.dw_lines(pairs, x, dY, gates, Wu, Wg, Wd, i, plain=plain, out=out)
            sl = osl.dw_line_slack(pairs, x, dY, gates, dgb, Wu, Wg, Wd, i, plain=plain) \
                if bf else {}
            for name, gv in (("dW_down", g["dW_down"][e, i, :]), ("dW_up", g["dW_up"][e, :, i]),
                             ("dW_gate", g["dW_gate"][e, :, i])):
                errs[f"{name}[{e}][{i}]"] = err(f64(gv), ref[name], sl.get(name, 0.0))
    sh_pairs = np.stack([np.arange(cfg.T), np.zeros(cfg.T, np.int64)], axis=1)
    for i in (7, cfg.shared_I - 1):
        ref = sampled.shared_dw_lines(x, dY, *shared, i, plain=plain, out=out)
        sl = osl.dw_line_slack(sh_pairs, x, dY, np.ones((cfg.T, 1)), np.zeros((cfg.T, 1)),
                               *shared, i, plain=plain) if bf else {}
        errs[f"dWs_down[{i}]"] = err(f64(g["dWs_down"][i, :]), ref["dWs_down"],
                                     sl.get("dW_down", 0.0))
        errs[f"dWs_up[{i}]"] = err(f64(g["dWs_up"][:, i]), ref["dWs_up"], sl.get("dW_up", 0.0))
        errs[f"dWs_gate[{i}]"] = err(f64(g["dWs_gate"][:, i]), ref["dWs_gate"],
                                     sl.get("dW_gate", 0.0))
    print(name, errs)
    for k, v in errs.items():
        assert v <= gu.TOL[cfg.precision], (k, v)


def _mx_forward_sampled(cfg, inp, L, y, tokens):
    x, idx, gates, pl = _check_schedule(cfg, inp, L)
    cache = {}

    def Wq(e):
        if e not in cache:
            cache.clear()
            cache[e] = sampled.mx_expert_weights(*(f64(inp[n][e]) for n in
                                                   ("W_up", "W_gate", "W_down")))
        return cache[e]

    ref = [sampled.token_forward_mx(t, x, idx, gates, Wq, out=cfg.out) for t in tokens]
    got = [f64(y[t]) for t in tokens]
    e = err(got, ref, osl.bf16_spacing(np.array(ref)) if cfg.out == "bf16" else 0.0)
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


def test_dsv3_imbalanced_mxfp8_backward_sampled():
    """MXFP8 backward at the DeepSeek-V3 shape (T=16384, 256 experts, four hot experts).
    In the bench's configuration (router in the layer): the schedule, one token's
    router-weight gradients and its dX at 64 hidden indices (router path included).
    Weight gradients: whole lines of the busiest expert in a second run that takes the
    oracle's routing (expert ids and fp32 gates) as its input, so that both sides quantise
    the same g*du values (see test_mxfp8_layer_matches_oracle)."""
    cfg = mi.CONFIGS["dsv3_imbalanced"]
    inp, L, y, g = _run(cfg, seed=11, backward=True)
    x, idx, gates, pl = _check_schedule(cfg, inp, L)
    dY = f64(inp["dY"])
    hs = np.arange(0, cfg.H, cfg.H // 64) + 3
    Wr_hs = f64(inp["Wr"])[hs]

    def wq(e):
        return sampled.mx_expert_weights_bwd(*(f64(inp[n][e]) for n in
                                               ("W_up", "W_gate", "W_down")), hs)

    t = cfg.T // 3
    bf = cfg.out == "bf16"
    o = sampled.token_backward_mx(t, x, idx, gates, wq, dY, Wr=Wr_hs, out=cfg.out)
    errs = {"dX": err(f64(g["dX"][t])[hs], o["dX"],
                      osl.bf16_spacing(o["dX_unrounded"]) if bf else 0.0),
            "dgates": err(g["dgates"][t].cpu().numpy(), o["dgates"])}
    del L, y, g
    torch.cuda.empty_cache()

    r = moe.route(x, f64(inp["Wr"]), cfg.k, f64(inp["bias"]))
    g32 = r.gates.astype(np.float32)
    ext = mi.scaled(cfg, router=False)
    L2 = gu.make_layer(ext)
    L2.plan(topk_idx=torch.as_tensor(r.idx, dtype=torch.int32).cuda(),
            gates=torch.as_tensor(g32).cuda())
    mx = L2.quantize_weights(inp["W_up"], inp["W_gate"], inp["W_down"])
    w = L2.weights(inp["W_up"], inp["W_gate"], inp["W_down"], mx=mx)
    L2.forward(inp["x"], w)
    g2 = L2.backward(inp["x"], None, w, inp["dY"])
    torch.cuda.synchronize()
    assert L2.status() == 0
    pl2 = moe.plan(r.idx, cfg.E)
    e = int(np.argmax(pl2.counts))
    assert pl2.counts[e] > 4 * np.median(pl2.counts)
    lines = sampled.dw_lines_mx(sampled.expert_rows(pl2, e), x, dY, g32.astype(np.float64),
                                *(f64(inp[n][e]) for n in ("W_up", "W_gate", "W_down")),
                                [5, cfg.I - 3], out=cfg.out)
    sp = (lambda v: osl.bf16_spacing(v)) if bf else (lambda v: 0.0)
    for i, li in lines.items():
        errs[f"dW_down[{e}][{i}]"] = err(f64(g2["dW_down"][e, i, :]), li["dW_down"],
                                         sp(li["dW_down"]))
        errs[f"dW_up[{e}][{i}]"] = err(f64(g2["dW_up"][e, :, i]), li["dW_up"], sp(li["dW_up"]))
        errs[f"dW_gate[{e}][{i}]"] = err(f64(g2["dW_gate"][e, :, i]), li["dW_gate"],
                                         sp(li["dW_gate"]))
    print("dsv3_imbalanced backward", int(pl2.counts[e]), "rows", errs)
    for k, v in errs.items():
        assert v <= gu.TOL["mxfp8"], (k, v)


def _bit_checksums(t):
    """Two 64-bit checksums of a tensor's 32-bit words, in chunks on the device: the plain
    sum and a sum weighted by position (mod 65521), so that a changed or moved word
    changes them."""
    w = t.detach().contiguous().view(torch.int32).reshape(-1)
    n = w.numel()
    chunk = 1 << 27
    pos = (torch.arange(chunk, device=w.device, dtype=torch.int64) % 65521) + 1
    s1 = torch.zeros((), dtype=torch.int64, device=w.device)
    s2 = torch.zeros((), dtype=torch.int64, device=w.device)
    for i in range(0, n, chunk):
        c = w[i:i + chunk].to(torch.int64)
        s1 += c.sum()
        s2 += (c * pos[:c.numel()]).sum()
    return int(s1), int(s2)


@pytest.mark.parametrize("name", ["dsv3_imbalanced", "kimi_8192", "kimi_8192_plain"])
def test_full_size_bitwise_deterministic_over_10_runs(name):
    """Ten plan + forward + backward steps at full size, in the bench's launch sequence,
    give the same bits for the routing, y, dX and every gradient (checksums of the 32-bit
    words, compared run by run)."""
    cfg = mi.CONFIGS[name]
    inp = mi.make_inputs(cfg, seed=13, device="cuda", with_dy=True)
    L = gu.make_layer(cfg)
    mx = L.quantize_weights(inp["W_up"], inp["W_gate"], inp["W_down"]) \
        if cfg.precision == "mxfp8" else None
    w = L.weights(inp["W_up"], inp["W_gate"], inp["W_down"], inp["Ws_up"], inp["Ws_gate"],
                  inp["Ws_down"], mx=mx)
    grads = L.alloc_grads()
    y = torch.empty((cfg.T, cfg.H), dtype=L.out_dtype, device="cuda")
    first = None
    for run in range(10):
        L.plan(x=inp["x"], Wr=inp["Wr"], bias=inp["bias"])
        L.forward(inp["x"], w, y)
        L.backward(inp["x"], inp["Wr"], w, inp["dY"], grads)
        torch.cuda.synchronize()
        assert L.status() == 0
        sums = {"topk_idx": _bit_checksums(L.topk_idx), "gates": _bit_checksums(L.gates),
                "y": _bit_checksums(y)}
        for f, v in grads.items():
            if v is not None:
                sums[f] = _bit_checksums(v)
        if first is None:
            first = sums
        else:
            assert sums == first, (run, [f for f in sums if sums[f] != first[f]])


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
