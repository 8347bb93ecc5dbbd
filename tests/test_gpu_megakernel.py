"""The forward megakernel (one cooperative launch: gather/combine SMs and GEMM SMs that
pass macrobatches through the ring token buffer) against the one-launch-per-step forward
and against the oracle. Both paths do the same arithmetic in the same order, so their
outputs must agree bit for bit."""
import numpy as np
import pytest
import torch

import moe_inputs as mi
from grouped_gemm_built_gb300 import mok
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu

ONE_MACROBATCH = {
    "tiny": mi.CONFIGS["tiny"],
    "ragged_shared": mi.MoEConfig("ragged_shared", T=300, H=256, I=256, E=12, k=3,
                                  shared_I=128),
    "sparse": mi.MoEConfig("sparse", T=64, H=128, I=128, E=64, k=1),
    "tiny_mx": mi.MoEConfig("tiny_mx", T=256, H=256, I=256, E=8, k=2, precision="mxfp8"),
    "ragged_shared_mx": mi.MoEConfig("ragged_shared_mx", T=300, H=256, I=256, E=12, k=3,
                                     shared_I=128, precision="mxfp8"),
}


def _run(cfg, inp, path, backward):
    L = gu.make_layer(cfg)
    L.set_fwd_path(path)
    res, _ = gu.run_gpu(cfg, inp, backward=backward, layer=L)
    saved = L.saved.cpu().numpy().copy()
    return res, saved


@pytest.mark.parametrize("name", list(ONE_MACROBATCH))
def test_megakernel_matches_launches_bitwise(name):
    cfg = ONE_MACROBATCH[name]
    inp = gu.gpu_inputs(cfg, seed=4)
    a, sa = _run(cfg, inp, "megakernel", backward=True)
    b, sb = _run(cfg, inp, "launches", backward=True)
    assert a["status"] == 0 and b["status"] == 0
    assert torch.equal(a["y"], b["y"]), "y differs between the two forward paths"
    assert np.array_equal(sa, sb), "saved U, V differ between the two forward paths"
    for f in ("dX", "dW_up", "dW_gate", "dW_down", "dgates"):
        assert torch.equal(a[f], b[f]), f


def _ring_case(precision):
    return mi.MoEConfig(f"ring_{precision}", T=1000, H=256, I=128, E=6, k=8, router=False,
                        zipf_s=1.2, precision=precision, backward=False, macrobatches=4)


@pytest.mark.parametrize("precision", ["bf16", "mxfp8"])
def test_ring_wraps_and_reuses_slots_bitwise(precision):
    """Four macrobatches through a ring of two slots, of four slots, and the whole batch
    at once: the same bits; and the oracle's forward within the tolerance."""
    base = _ring_case(precision)
    inp = gu.gpu_inputs(base, seed=6)
    two = mi.scaled(base, ring_bytes=2 * _slot_bytes(base) + _slot_bytes(base) // 2)
    outs = {}
    for label, cfg, path, slots in (("4 slots", base, "megakernel", 4),
                                     ("2 slots", two, "megakernel", 2),
                                     ("launches", base, "launches", 4)):
        L = gu.make_layer(cfg)
        assert L.sizes.macrobatches == 4 and L.sizes.ring_slots == slots, label
        L.set_fwd_path(path)
        res, _ = gu.run_gpu(cfg, inp, backward=False, layer=L)
        assert res["status"] == 0, label
        outs[label] = res["y"]
    assert torch.equal(outs["4 slots"], outs["2 slots"])
    assert torch.equal(outs["4 slots"], outs["launches"])
    idx, gates, _ = gu.oracle_route(base, inp)
    ref = gu.run_oracle(base, inp, idx, gates, backward=False)
    assert gu.rel_err(outs["2 slots"], ref["y"]) <= gu.TOL[precision]


def _slot_bytes(cfg):
    """Bytes of one ring slot: a macrobatch's padded rows (whole 128-row tiles), bf16."""
    M = max(cfg.macrobatches, 1)
    Tm = -(-(-(-cfg.T // M)) // 128) * 128          # ceil(T / M) rounded up to 128
    rows = min(Tm, cfg.T) * cfg.k
    mt = (rows + min(cfg.E, rows) * 127 + 127) // 128
    return mt * 128 * cfg.H * 2


@pytest.mark.parametrize("precision,slots", [("bf16", 4), ("bf16", 2), ("bf16", 1),
                                             ("mxfp8", 2)])
def test_backward_after_macrobatches_matches_one_launch_per_step(precision, slots):
    """Forward through the megakernel over four macrobatches (ring of 4, 2 or 1 slots) and
    the backward after it: U, V are read where the megakernel left them (per-macrobatch
    padded rows) and the x rows are gathered again. y and every gradient equal, bit for
    bit, those of the one-launch-per-step path; and they match the oracle."""
    base = mi.scaled(_ring_case(precision), backward=True, router=True, zipf_s=0.0,
                     shared_I=128, E=12, k=4)
    sb = _slot_bytes(base)
    cfg = mi.scaled(base, ring_bytes=0 if slots == 4 else slots * sb + sb // 2)
    inp = gu.gpu_inputs(cfg, seed=9)
    res = {}
    for path in ("megakernel", "launches"):
        L = gu.make_layer(cfg)
        assert (L.sizes.macrobatches, L.sizes.ring_slots) == (4, slots)
        L.set_fwd_path(path)
        res[path], _ = gu.run_gpu(cfg, inp, backward=True, layer=L)
        assert res[path]["status"] == 0, path
    for f in ("y", "dX", "dW_up", "dW_gate", "dW_down", "dgates", "dWr", "dWs_up",
              "dWs_gate", "dWs_down"):
        assert torch.equal(res["megakernel"][f], res["launches"][f]), f
    if slots == 2:
        idx, gates, logits = gu.oracle_route(cfg, inp)
        ref = gu.run_oracle(cfg, inp, idx, gates, backward=True)
        from tests import out_slack as osl
        r = res["megakernel"]
        for f in ("y", "dX", "dgates"):
            sl = (osl.bf16_spacing(ref["unrounded"][f]) if f != "dgates" and precision == "mxfp8"
                  else osl.layer_slack(cfg, inp, idx, gates, logits)[f] if f != "dgates"
                  else 0.0)
            assert gu.rel_err_slack(r[f], ref[f], sl) <= gu.TOL[precision], f


def test_two_wave_macrobatches_resolve_and_keep_the_bits():
    """minibatch_tokens = -1 sizes macrobatches by the two-wave rule at the device's SM
    count (ceil(2 * SMs * 64 / k) tokens, rounded up to 128). Through the megakernel, with
    the backward, the results equal the one-launch-per-step path's bit for bit."""
    props = torch.cuda.get_device_properties(0)
    cfg = mi.MoEConfig("two_wave", T=5000, H=256, I=128, E=16, k=8, shared_I=0,
                       minibatch_tokens=-1, macrobatches=0)
    want = -(-mok.mok_minibatch_tokens(256, 128, 8, props.multi_processor_count) // 128) * 128
    inp = gu.gpu_inputs(cfg, seed=10)
    res = {}
    for path in ("megakernel", "launches"):
        L = gu.make_layer(cfg)
        assert L.sizes.macrobatch_tokens == want
        assert L.sizes.macrobatches == -(-5000 // want) and L.sizes.macrobatches > 1
        L.set_fwd_path(path)
        res[path], _ = gu.run_gpu(cfg, inp, backward=True, layer=L)
        assert res[path]["status"] == 0
    for f in ("y", "dX", "dW_up", "dW_gate", "dW_down", "dgates", "dWr"):
        assert torch.equal(res["megakernel"][f], res["launches"][f]), f


def test_withheld_signal_times_out_and_the_context_recovers():
    """Failure detection without a fault: with the test hook on, the megakernel never
    publishes one gathered row tile, so the GEMM SM waiting for it passes its bound
    (20 ms here); the call must end with MOK_ERR_TIMEOUT in the status word, quickly and
    with no trap, and the same context must then run correctly."""
    import time
    cfg = ONE_MACROBATCH["ragged_shared"]
    inp = gu.gpu_inputs(cfg, seed=8)
    d = gu.to_dev(inp)
    L = gu.make_layer(cfg)
    L.set_fwd_path("megakernel")
    mok.mok_set_wait_timeout(L.ctx, 20_000_000)
    L.plan(x=d["x"], Wr=d["Wr"], bias=d["bias"])
    w = L.weights(d["W_up"], d["W_gate"], d["W_down"], d["Ws_up"], d["Ws_gate"], d["Ws_down"])
    assert L.status() == 0
    mok.mok_test_withhold_signal(L.ctx, True)
    t0 = time.time()
    L.forward(d["x"], w)
    torch.cuda.synchronize()
    elapsed = time.time() - t0
    assert L.status() == mok.MOK_ERR_TIMEOUT
    assert elapsed < 5.0, elapsed
    mok.mok_test_withhold_signal(L.ctx, False)
    y = L.forward(d["x"], w).clone()
    torch.cuda.synchronize()
    assert L.status() == 0
    L2 = gu.make_layer(cfg)
    L2.set_fwd_path("launches")
    L2.plan(x=d["x"], Wr=d["Wr"], bias=d["bias"])
    y2 = L2.forward(d["x"], w)
    torch.cuda.synchronize()
    assert torch.equal(y, y2)
