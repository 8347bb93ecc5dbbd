"""The allocation-free schedule entry point (mok_plan_noalloc) against mok_plan.

Callers that cannot allocate device memory pass no workspace; the schedule builder's
scratch then lives in a fixed array inside the library. Through the C ABI, two calls in a
row (different routing each time, so the second call also shows that nothing left in the
shared array by the first leaks into the result) must give exactly the schedule that
mok_plan writes with a workspace. This file is collected last on purpose.
"""
import numpy as np
import pytest
import torch

from grouped_gemm_built_gb300 import mok

pytestmark = pytest.mark.gpu


def _sched(T, k, E, aux_bytes):
    d = "cuda"
    t = {
        "topk_idx": torch.zeros((T, k), dtype=torch.int32, device=d),
        "gates": torch.zeros((T, k), dtype=torch.float32, device=d),
        "counts": torch.full((E,), -1, dtype=torch.int32, device=d),
        "offsets": torch.full((E + 1,), -1, dtype=torch.int32, device=d),
        "table": torch.full((T * k, 2), -1, dtype=torch.int32, device=d),
        "inv": torch.full((T, k), -1, dtype=torch.int32, device=d),
        "aux": torch.zeros(aux_bytes, dtype=torch.uint8, device=d),
    }
    s = mok.MokSched(**{n: v.data_ptr() for n, v in t.items()})
    return t, s


def test_noalloc_schedule_equals_mok_plan_twice():
    T, H, I, E, k = 1000, 256, 128, 37, 5
    dims = mok.MokDims(T=T, H=H, I=I, E=E, k=k, shared_I=0, router=0, macrobatches=0,
                       ring_bytes=0)
    ctx = mok.mok_create(dims)
    sizes = mok.mok_get_sizes(ctx)
    ws = torch.empty(sizes.workspace_bytes, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    rng = np.random.default_rng(11)
    try:
        for call in range(2):
            idx = np.stack([rng.choice(E, k, replace=False) for _ in range(T)])
            if call == 1:
                idx[::3, 2] = idx[::3, 0]        # repeated experts inside a token
            g = rng.uniform(0.1, 1.0, idx.shape)
            g = g / g.sum(1, keepdims=True)
            ref_t, ref_s = _sched(T, k, E, sizes.aux_bytes)
            new_t, new_s = _sched(T, k, E, sizes.aux_bytes)
            for t in (ref_t, new_t):
                t["topk_idx"].copy_(torch.as_tensor(idx, dtype=torch.int32))
                t["gates"].copy_(torch.as_tensor(g, dtype=torch.float32))
            mok.mok_plan(ctx, None, None, None, ref_s, ws.data_ptr(), stream)
            mok.mok_plan_noalloc(ctx, new_s, stream)
            torch.cuda.synchronize()
            assert mok.mok_get_status(ctx, new_s, stream) == 0
            for name in ("counts", "offsets", "table", "inv", "aux"):
                assert torch.equal(ref_t[name], new_t[name]), (call, name)
    finally:
        mok.mok_destroy(ctx)
