"""The C ABI without a GPU: the library loads, exports what include/*.h declares, and its
host-only logic (argument checks, sizes, the minibatch planner) behaves."""
import ctypes
import os

import pytest

from grouped_gemm_built_gb300 import build, mok

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module", autouse=True)
def built():
    build.build()
    mok.lib()


def test_exports_every_declared_symbol():
    declared = mok.declared_symbols()
    assert {"mok_plan", "mok_moe_fwd", "mok_moe_bwd", "mok_set_precision"} <= set(declared)
    L = ctypes.CDLL(build.lib_path())
    for name in declared:
        assert hasattr(L, name), name


def test_two_wave_minibatch_matches_the_page():
    line = [l for l in open(os.path.join(GOLDEN, "two_wave_minibatch.txt"))
            if not l.startswith("#") and l.strip()][0]
    kv = dict(p.split("=") for p in line.split())
    got = mok.mok_minibatch_tokens(int(kv["H"]), int(kv["I"]), int(kv["k"]), int(kv["sms"]))
    assert got == int(kv["tokens"])
    assert mok.mok_minibatch_tokens(7168, 2048, 8, 0) == -1


def dims(**over):
    base = dict(T=256, H=256, I=128, E=8, k=2, shared_I=0, router=1, macrobatches=0,
                ring_bytes=0)
    base.update(over)
    return mok.MokDims(**base)


@pytest.mark.parametrize("bad", [dict(H=200), dict(I=96), dict(E=0), dict(E=513), dict(k=9),
                                 dict(k=9, E=4, router=0), dict(k=5, E=4), dict(T=0),
                                 dict(shared_I=100), dict(router=2)])
def test_create_rejects_bad_dims(bad):
    with pytest.raises(mok.MokError) as ei:
        mok.mok_create(dims(**bad))
    assert ei.value.status == mok.MOK_ERR_INVALID_ARG


def test_sizes_cover_the_padded_row_space():
    ctx = mok.mok_create(dims(T=300, E=12, k=3, I=256, shared_I=128))
    s = mok.mok_get_sizes(ctx)
    R = 300 * 3
    assert s.padded_rows_max >= R + 12 * 127 and s.padded_rows_max % 128 == 0
    assert s.saved_bytes >= 2 * 2 * s.padded_rows_max * 256 + 2 * 2 * 300 * 128
    assert s.workspace_bytes >= 2 * s.padded_rows_max * 256 * 4
    assert s.aux_bytes >= 4 * (12 + 1)
    mok.mok_destroy(ctx)


def test_calls_check_arguments_before_touching_the_device():
    ctx = mok.mok_create(dims())
    sched = mok.MokSched()          # all null
    with pytest.raises(mok.MokError) as ei:
        mok.mok_plan(ctx, 16, 16, None, sched, 256, None)
    assert ei.value.status == mok.MOK_ERR_INVALID_ARG
    full = mok.MokSched(*([256] * 6), 1000)  # aux not 256-byte aligned
    with pytest.raises(mok.MokError) as ei:
        mok.mok_plan(ctx, 16, 16, None, full, 256, None)
    assert ei.value.status == mok.MOK_ERR_WORKSPACE
    with pytest.raises(mok.MokError) as ei:
        mok.mok_set_precision(ctx, 7)
    assert ei.value.status == mok.MOK_ERR_INVALID_ARG
    mok.mok_destroy(ctx)


def test_status_strings():
    for st in (0, -1, -2, -3, -4, -5, -6):
        assert mok.mok_status_string(st)


def test_macrobatches_and_ring_slots():
    """Macrobatches are ceil(T / M) tokens rounded up to 128; the ring holds as many
    macrobatch slots (bf16 rows, whole 128-row tiles) as ring_bytes allows, at most M;
    a ring smaller than one slot is rejected."""
    def slot_bytes(T, H, E, k, M):
        Tm = -(-(-(-T // M)) // 128) * 128
        rows = min(Tm, T) * k
        return ((rows + min(E, rows) * 127 + 127) // 128) * 128 * H * 2

    d = dict(T=1000, H=256, I=128, E=6, k=8, router=0)
    ctx = mok.mok_create(dims(**d, macrobatches=4))
    s = mok.mok_get_sizes(ctx)
    assert (s.macrobatches, s.ring_slots) == (4, 4)
    mok.mok_destroy(ctx)
    sb = slot_bytes(1000, 256, 6, 8, 4)
    for ring, slots in ((sb, 1), (2 * sb + sb // 2, 2), (100 * sb, 4)):
        ctx = mok.mok_create(dims(**d, macrobatches=4, ring_bytes=ring))
        assert mok.mok_get_sizes(ctx).ring_slots == slots
        mok.mok_destroy(ctx)
    with pytest.raises(mok.MokError) as ei:
        mok.mok_create(dims(**d, macrobatches=4, ring_bytes=sb - 1))
    assert ei.value.status == mok.MOK_ERR_INVALID_ARG
    # 128-token granularity: 7 macrobatches of 1000 tokens become ceil(1000/7)=143 -> 256
    # tokens each, so 4 of them
    ctx = mok.mok_create(dims(**d, macrobatches=7))
    assert mok.mok_get_sizes(ctx).macrobatches == 4
    mok.mok_destroy(ctx)
    ctx = mok.mok_create(dims(**d))
    assert mok.mok_get_sizes(ctx).macrobatches == 1
    mok.mok_destroy(ctx)


def test_fwd_path_option():
    ctx = mok.mok_create(dims())
    mok.mok_set_fwd_path(ctx, mok.MOK_FWD_LAUNCHES)
    mok.mok_set_fwd_path(ctx, mok.MOK_FWD_MEGAKERNEL)
    with pytest.raises(mok.MokError) as ei:
        mok.mok_set_fwd_path(ctx, 7)
    assert ei.value.status == mok.MOK_ERR_INVALID_ARG
    mok.mok_destroy(ctx)


def test_tile_order_row_pairs_sm_pairs_and_output_type_options():
    ctx = mok.mok_create(dims())
    for order in (mok.MOK_TILES_DYNAMIC, mok.MOK_TILES_CLC, mok.MOK_TILES_STATIC):
        mok.mok_set_tile_order(ctx, order)
    for out in (mok.MOK_OUT_F32, mok.MOK_OUT_BF16):
        mok.mok_set_output_dtype(ctx, out)
    for mode in (mok.MOK_PAIRS_ON, mok.MOK_PAIRS_OFF, mok.MOK_PAIRS_AUTO):
        mok.mok_set_row_pairs(ctx, mode)
    for mode in (mok.MOK_SMPAIRS_ON, mok.MOK_SMPAIRS_OFF, mok.MOK_SMPAIRS_AUTO):
        mok.mok_set_sm_pairs(ctx, mode)
    for setter, bad in ((mok.mok_set_tile_order, 3), (mok.mok_set_output_dtype, 2),
                        (mok.mok_set_row_pairs, 3), (mok.mok_set_sm_pairs, 3),
                        (mok.mok_set_sm_pairs, -1)):
        with pytest.raises(mok.MokError) as ei:
            setter(ctx, bad)
        assert ei.value.status == mok.MOK_ERR_INVALID_ARG
    mok.mok_destroy(ctx)
    assert mok.lib().mok_set_tile_order(None, 0) == mok.MOK_ERR_INVALID_ARG
    assert mok.lib().mok_set_output_dtype(None, 0) == mok.MOK_ERR_INVALID_ARG
    assert mok.lib().mok_set_row_pairs(None, 0) == mok.MOK_ERR_INVALID_ARG
    assert mok.lib().mok_set_sm_pairs(None, 0) == mok.MOK_ERR_INVALID_ARG


def test_wait_timeout_and_test_hook_are_host_settings():
    ctx = mok.mok_create(dims())
    mok.mok_set_wait_timeout(ctx, 5_000_000)
    mok.mok_set_wait_timeout(ctx, 0)
    with pytest.raises(mok.MokError) as ei:
        mok.mok_set_wait_timeout(ctx, 61_000_000_000)
    assert ei.value.status == mok.MOK_ERR_INVALID_ARG
    mok.mok_test_withhold_signal(ctx, True)
    mok.mok_test_withhold_signal(ctx, False)
    mok.mok_destroy(ctx)


# ----------------------------------------------------------------- argument checks of the calls
# Every case below is rejected before the call touches a device: the checks run first and
# return a status, so fake (never dereferenced) addresses are enough.
A = 1 << 20                                   # a fake, 256-byte aligned address


def _sched():
    return mok.MokSched(*([A] * 7))


def _weights(shared=False, mx=False):
    return mok.MokWeights(A, A, A, *((A, A, A) if shared else (None, None, None)),
                          A if mx else None)


def _grads(router=True, shared=False):
    return mok.MokGrads(A, A, A, A, A if router else None,
                        *((A, A, A) if shared else (None, None, None)))


def _status(fn, *args):
    with pytest.raises(mok.MokError) as ei:
        fn(*args)
    return ei.value.status


def test_fwd_rejects_bad_arguments():
    ctx = mok.mok_create(dims())
    S, W = _sched(), _weights()
    fwd = mok.mok_moe_fwd
    assert _status(fwd, ctx, S, A, mok.MokWeights(None, A, A), A, A, A, None) == \
        mok.MOK_ERR_INVALID_ARG                                        # missing W_up
    assert _status(fwd, ctx, S, A + 8, W, A, A, A, None) == mok.MOK_ERR_INVALID_ARG  # x
    assert _status(fwd, ctx, S, A, W, None, A, A, None) == mok.MOK_ERR_INVALID_ARG   # y
    assert _status(fwd, ctx, S, A, W, A, A, None, None) == mok.MOK_ERR_WORKSPACE
    assert _status(fwd, ctx, S, A, W, A, A + 16, A, None) == mok.MOK_ERR_WORKSPACE  # saved
    assert _status(fwd, ctx, mok.MokSched(*([A] * 6), None), A, W, A, A, A, None) == \
        mok.MOK_ERR_WORKSPACE                                          # no aux
    mok.mok_set_precision(ctx, mok.MOK_MXFP8)
    assert _status(fwd, ctx, S, A, W, A, A, A, None) == mok.MOK_ERR_INVALID_ARG  # no mx
    mok.mok_destroy(ctx)
    ctx = mok.mok_create(dims(shared_I=128))
    assert _status(fwd, ctx, S, A, W, A, A, A, None) == mok.MOK_ERR_INVALID_ARG  # no Ws_*
    mok.mok_destroy(ctx)


def test_bwd_rejects_bad_arguments():
    ctx = mok.mok_create(dims())
    S, W, G = _sched(), _weights(), _grads()
    bwd = mok.mok_moe_bwd
    assert _status(bwd, ctx, S, A, None, W, A, A, A, G, A, None) == \
        mok.MOK_ERR_INVALID_ARG                                        # router needs Wr
    assert _status(bwd, ctx, S, A, A, W, A, A, A, _grads(router=False), A, None) == \
        mok.MOK_ERR_INVALID_ARG                                        # and dWr
    assert _status(bwd, ctx, S, A, A, W, A, None, A, G, A, None) == mok.MOK_ERR_INVALID_ARG
    assert _status(bwd, ctx, S, A, A, W, A, A, A,
                   mok.MokGrads(A, A, A, None, A, None, None, None), A, None) == \
        mok.MOK_ERR_INVALID_ARG                                        # dgates
    assert _status(bwd, ctx, S, A, A, W, None, A, A, G, A, None) == mok.MOK_ERR_WORKSPACE
    mok.mok_destroy(ctx)
    ctx = mok.mok_create(dims(router=0))
    assert _status(bwd, ctx, S, A, A, W, A, A, A, _grads(router=False), A, None) == \
        mok.MOK_ERR_INVALID_ARG                                        # Wr without a router
    assert _status(bwd, ctx, S, A, None, W, A, A, A, G, A, None) == \
        mok.MOK_ERR_INVALID_ARG                                        # dWr without a router
    mok.mok_destroy(ctx)
    ctx = mok.mok_create(dims(shared_I=128))
    assert _status(bwd, ctx, S, A, A, _weights(shared=True), A, A, A, G, A, None) == \
        mok.MOK_ERR_INVALID_ARG                                        # shared grads
    mok.mok_destroy(ctx)
    ctx = mok.mok_create(dims(router=0, macrobatches=2))
    assert mok.mok_get_sizes(ctx).macrobatches == 2
    # several macrobatches are accepted: past the argument checks, a machine without a
    # GPU then fails at the launch
    assert _status(bwd, ctx, S, A, None, W, A, A, A, _grads(router=False), A, None) == \
        mok.MOK_ERR_CUDA
    mok.mok_destroy(ctx)


def test_minibatch_tokens_resolve_macrobatches():
    """minibatch_tokens > 0 sizes macrobatches by tokens (rounded up to 128); -1 takes the
    two-wave rule at the device's SM count, which without a device is one macrobatch;
    setting it together with macrobatches, or below -1, is rejected."""
    d = dict(T=1000, H=256, I=128, E=6, k=8, router=0)
    ctx = mok.mok_create(dims(**d, minibatch_tokens=300))
    s = mok.mok_get_sizes(ctx)
    assert (s.macrobatch_tokens, s.macrobatches) == (384, 3)
    mok.mok_destroy(ctx)
    ctx = mok.mok_create(dims(**d, minibatch_tokens=-1))
    s = mok.mok_get_sizes(ctx)
    import torch
    if not torch.cuda.is_available():
        assert s.macrobatches == 1 and s.macrobatch_tokens >= 1000
    mok.mok_destroy(ctx)
    for bad in (dict(minibatch_tokens=256, macrobatches=2), dict(minibatch_tokens=-2)):
        with pytest.raises(mok.MokError) as ei:
            mok.mok_create(dims(**d, **bad))
        assert ei.value.status == mok.MOK_ERR_INVALID_ARG


def test_plan_and_quantize_reject_bad_arguments():
    ctx = mok.mok_create(dims())
    S = _sched()
    assert _status(mok.mok_plan, ctx, A, None, None, S, A, None) == mok.MOK_ERR_INVALID_ARG
    assert _status(mok.mok_plan, ctx, A + 4, A, None, S, A, None) == mok.MOK_ERR_INVALID_ARG
    assert _status(mok.mok_plan, ctx, A, A, None, S, A + 64, None) == mok.MOK_ERR_WORKSPACE
    assert _status(mok.mok_quantize_weights_mxfp8, ctx, _weights(), A + 128, None) == \
        mok.MOK_ERR_INVALID_ARG
    assert _status(mok.mok_quantize_weights_mxfp8, ctx, mok.MokWeights(A, None, A), A,
                   None) == mok.MOK_ERR_INVALID_ARG
    mok.mok_destroy(ctx)
    ctx = mok.mok_create(dims(router=0))
    for x, Wr, b in ((A, None, None), (None, A, None), (None, None, A)):
        assert _status(mok.mok_plan, ctx, x, Wr, b, S, A, None) == mok.MOK_ERR_INVALID_ARG
    mok.mok_destroy(ctx)


def _no_device():
    import torch
    return not torch.cuda.is_available() and not os.path.exists("/dev/nvidia0")


@pytest.mark.skipif(not _no_device(), reason="only where no GPU exists: the call would launch")
def test_valid_calls_without_a_device_return_cuda_error():
    """With every argument valid, the calls get as far as the device and report that there
    is none, without launching anything."""
    ctx = mok.mok_create(dims())
    S, W = _sched(), _weights()
    assert _status(mok.mok_plan, ctx, A, A, None, S, A, None) == mok.MOK_ERR_CUDA
    assert _status(mok.mok_moe_fwd, ctx, S, A, W, A, A, A, None) == mok.MOK_ERR_CUDA
    assert _status(mok.mok_moe_bwd, ctx, S, A, A, W, A, A, A, _grads(), A, None) == \
        mok.MOK_ERR_CUDA
    assert _status(mok.mok_quantize_weights_mxfp8, ctx, W, A, None) == mok.MOK_ERR_CUDA
    mok.mok_destroy(ctx)


def test_a_plain_c_program_uses_the_abi(tmp_path):
    """tests/abi_consumer.c includes the headers as C99 (-pedantic, warnings as errors),
    links libmok.so and runs the host-side calls; its view of the sizes equals the
    binding's."""
    import shutil
    import subprocess
    gcc = shutil.which("gcc") or shutil.which("cc")
    if gcc is None:
        pytest.skip("no C compiler")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    libdir = os.path.dirname(build.lib_path())
    exe = str(tmp_path / "abi_consumer")
    cmd = [gcc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic",
           "-I", os.path.join(root, "include"), os.path.join(root, "tests", "abi_consumer.c"),
           "-L", libdir, "-lmok", f"-Wl,-rpath,{libdir}", "-o", exe]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    out = dict(line.split(" ", 1) for line in r.stdout.splitlines())
    assert out["failures"] == "0"
    assert int(out["minibatch_148"]) == 2368
    ctx = mok.mok_create(dims(T=300, H=256, I=256, E=12, k=3, shared_I=128))
    s = mok.mok_get_sizes(ctx)
    mok.mok_destroy(ctx)
    want = [s.aux_bytes, s.workspace_bytes, s.saved_bytes, s.mx_weight_bytes,
            s.padded_rows_max, s.macrobatches, s.ring_slots]
    assert [int(v) for v in out["sizes"].split()] == want


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    """No fallback: without the built library every call raises at once."""
    monkeypatch.setattr(mok, "_LIB", None)
    monkeypatch.setattr(mok, "lib_path", lambda: str(tmp_path / "libmok.so"))
    with pytest.raises(RuntimeError, match="not built"):
        mok.mok_status_string(0)
    with pytest.raises(RuntimeError, match="not built"):
        mok.mok_create(dims())


def test_product_path_never_imports_the_oracle():
    """The library package and its binding import nothing from oracle/ (the oracle is
    test infrastructure); checked on the source text of every module in the package."""
    import ast
    pkg = os.path.dirname(os.path.abspath(mok.__file__))
    for name in sorted(os.listdir(pkg)):
        if not name.endswith(".py"):
            continue
        tree = ast.parse(open(os.path.join(pkg, name)).read())
        for node in ast.walk(tree):
            if isinstance(node, ast.Import):
                mods = [a.name for a in node.names]
            elif isinstance(node, ast.ImportFrom):
                mods = [node.module or ""]
            else:
                continue
            assert not any(m == "oracle" or m.startswith("oracle.") for m in mods), name
