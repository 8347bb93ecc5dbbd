"""The allocation-free schedule entry point (mok_plan_noalloc) against mok_plan and the
oracle.

Callers that cannot allocate device memory pass no workspace; the schedule builder's
scratch then lives in a fixed array inside the library. Through the C ABI, two calls in a
row (different routing each time, so the second call also shows that nothing left in the
shared array by the first leaks into the result) must give exactly the schedule that
mok_plan writes with a workspace, and the oracle's schedule.

The file name makes pytest collect it last: the entry point is an addition outside the
layer's own path, and a run that stops at the first failure has then already run every
other test. It passes on its own in a fresh process as well as after the others (the shared
array is rewritten by every call before it is read). Its host-side checks, which launch
nothing, run without a GPU.
"""
import numpy as np
import pytest
import torch

from grouped_gemm_built_gb300 import mok
from oracle import moe


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


@pytest.mark.gpu
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
            assert mok.mok_get_status(ctx, ref_s, stream) == 0
            assert mok.mok_get_status(ctx, new_s, stream) == 0
            for name in ("counts", "offsets", "table", "inv", "aux"):
                assert torch.equal(ref_t[name], new_t[name]), (call, name)
            pl = moe.plan(idx, E)
            for name in ("counts", "offsets", "table", "inv"):
                got = new_t[name].cpu().numpy()
                assert np.array_equal(got, getattr(pl, name).reshape(got.shape)), (call, name)
    finally:
        mok.mok_destroy(ctx)


def _dims(T, E, k, router=0):
    return mok.MokDims(T=T, H=128, I=128, E=E, k=k, shared_I=0, router=router,
                       macrobatches=0, ring_bytes=0)


def _dummy_sched():
    # stand-in addresses: these calls return before anything is launched or read
    return mok.MokSched(topk_idx=256, gates=512, counts=768, offsets=1024, table=1280,
                        inv=1536, aux=4096)


def test_noalloc_rejects_problems_beyond_its_scratch():
    """(ceil(T/32) * E int32 histograms, rounded up to 256 bytes, + T*k int32 ranks) must fit
    in the 4 MiB array: 65536 tokens, 512 experts, top-8 need 6 MiB, which is
    MOK_ERR_UNSUPPORTED before any launch; at 512 experts and top-8 the largest token count
    that fits passes the size check, 32 tokens more do not."""
    L = mok.lib()
    big = mok.mok_create(_dims(65536, 512, 8))
    try:
        assert L.mok_plan_noalloc(big, mok.ctypes.byref(_dummy_sched()), None) == \
            mok.MOK_ERR_UNSUPPORTED
    finally:
        mok.mok_destroy(big)
    # the bound is exact: the largest T with E = 512, k = 8 that fits
    E, k = 512, 8

    def need(T):
        hist = ((T + 31) // 32) * E * 4
        return (hist + 255) // 256 * 256 + T * k * 4
    T_ok = max(T for T in range(1, 100000) if need(T) <= (4 << 20))
    for T, want_unsupported in ((T_ok, False), (T_ok + 32, True)):
        c = mok.mok_create(_dims(T, E, k))
        try:
            st = L.mok_plan_noalloc(c, mok.ctypes.byref(_dummy_sched()), None)
            if want_unsupported:
                assert st == mok.MOK_ERR_UNSUPPORTED, T
            else:   # past the size check: on a machine without a GPU the launch fails
                assert st != mok.MOK_ERR_UNSUPPORTED, T
        finally:
            mok.mok_destroy(c)


def test_noalloc_refuses_a_context_that_routes():
    """The entry point takes routing from the caller: a context made with router = 1 gets
    MOK_ERR_INVALID_ARG, before any launch."""
    L = mok.lib()
    c = mok.mok_create(_dims(64, 8, 2, router=1))
    try:
        assert L.mok_plan_noalloc(c, mok.ctypes.byref(_dummy_sched()), None) == \
            mok.MOK_ERR_INVALID_ARG
        assert L.mok_plan_noalloc(None, mok.ctypes.byref(_dummy_sched()), None) == \
            mok.MOK_ERR_INVALID_ARG
    finally:
        mok.mok_destroy(c)
