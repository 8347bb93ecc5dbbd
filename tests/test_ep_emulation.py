"""Expert parallelism emulated on one GPU (tests/ep_emulation.py): the cross-slice
schedule on the CPU, and the sliced layer against the single layer on the GPU."""
import numpy as np
import pytest
import torch

import moe_inputs as mi
from oracle import moe
from tests import ep_emulation as ep
from tests import gpu_util as gu


@pytest.mark.parametrize("P", [1, 2, 4, 8])
def test_cross_slice_schedule_partitions_the_table(P):
    """Every (token, slot) lands in exactly one slice, the slice that owns its expert, in
    the table's order; the local expert ids are the global ones less the slice's first."""
    rng = np.random.default_rng(P)
    T, E, k = 300, 16, 4
    idx = np.stack([rng.choice(E, k, replace=False) for _ in range(T)])
    pl = moe.plan(idx, E)
    sl = ep.cross_slice_schedule(pl.counts, pl.offsets, pl.table, E, P)
    assert len(sl) == P
    seen = np.concatenate([s.rows for s in sl])
    assert np.array_equal(seen, np.arange(T * k))          # a partition, in table order
    for s in sl:
        e0, e1 = s.experts
        assert e1 - e0 == E // P
        ex = idx[s.tokens, s.slots]
        assert np.all((ex >= e0) & (ex < e1))
        assert np.array_equal(s.local_expert, ex - e0)
        # inside an expert, ascending (token, slot)
        key = s.local_expert * (T * k) + s.tokens * k + s.slots
        assert np.all(np.diff(key) > 0)
    with pytest.raises(ValueError):
        ep.cross_slice_schedule(pl.counts, pl.offsets, pl.table, E, 3)


@pytest.mark.gpu
@pytest.mark.parametrize("P", [2, 4, 8])
def test_ep_slices_match_the_single_layer(P):
    """P expert slices, each a router-less layer fed by the cross-slice schedule, give the
    single layer's weight gradients and router-weight gradients bit for bit, and its y,
    dX and dWr to fp32 rounding (the slot sums are added outside the fused combine)."""
    cfg = mi.MoEConfig("ep_emul", T=512, H=256, I=128, E=16, k=4, out="fp32")
    inp = gu.gpu_inputs(cfg, seed=12)
    d = gu.to_dev(inp)
    res, sched = ep.run_ep(cfg, d, P)
    assert sum(len(s.rows) for s in sched) == cfg.T * cfg.k
    full, _ = gu.run_gpu(cfg, inp, backward=True)
    assert full["status"] == 0
    assert np.array_equal(res["topk_idx"].cpu().numpy(), full["topk_idx"])
    for f in ("dW_up", "dW_gate", "dW_down", "dgates"):
        assert torch.equal(res[f].cpu(), full[f]), f
    for f in ("y", "dX", "dWr"):
        err = gu.rel_err(res[f].cpu(), gu.np64(full[f]))
        assert err < 1e-5, (f, err)
    # and the oracle, at the layer's tolerance (weight gradients with the allowance for
    # U, V rounding flips)
    idx, gates, _ = gu.oracle_route(cfg, inp)
    ref = gu.run_oracle(cfg, inp, idx, gates, backward=True)
    slack, _ = gu.bf16_flip_slack(cfg, inp, idx, gates)
    for f in ("y", "dX", "dW_up", "dW_down", "dWr"):
        err = gu.rel_err_slack(res[f].cpu(), ref[f], slack.get(f, 0.0))
        assert err <= gu.TOL["bf16"], (f, err)
