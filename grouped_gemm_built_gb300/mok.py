"""ctypes binding of libmok (the C ABI in include/mok.h), with the same names.

Argument marshalling only: every step of the layer runs in the library's CUDA kernels.
Pointers are passed as Python ints (e.g. ``tensor.data_ptr()``), streams as the raw
``cudaStream_t`` value (``torch.cuda.current_stream().cuda_stream``). A missing library
raises immediately; there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os
import re

from .build import lib_path

c_int, c_size_t, c_void_p, c_char_p = ctypes.c_int, ctypes.c_size_t, ctypes.c_void_p, ctypes.c_char_p

MOK_OK = 0
MOK_ERR_INVALID_ARG = -1
MOK_ERR_UNSUPPORTED = -2
MOK_ERR_WORKSPACE = -3
MOK_ERR_CUDA = -4
MOK_ERR_TIMEOUT = -5
MOK_ERR_DEVICE = -6
MOK_BF16 = 0
MOK_MXFP8 = 1
MOK_BF16_WGRAD_PLAIN = 2
MOK_OUT_BF16 = 0
MOK_OUT_F32 = 1
MOK_TILES_STATIC = 0
MOK_TILES_DYNAMIC = 1
MOK_TILES_CLC = 2
MOK_PAIRS_AUTO = 0
MOK_PAIRS_ON = 1
MOK_PAIRS_OFF = 2
MOK_SMPAIRS_AUTO = 0
MOK_SMPAIRS_ON = 1
MOK_SMPAIRS_OFF = 2
MOK_FWD_MEGAKERNEL = 0
MOK_FWD_LAUNCHES = 1
MOK_FWD_AUTO = 2


class MokDims(ctypes.Structure):
    _fields_ = [("T", c_int), ("H", c_int), ("I", c_int), ("E", c_int), ("k", c_int),
                ("shared_I", c_int), ("router", c_int), ("macrobatches", c_int),
                ("ring_bytes", c_size_t), ("minibatch_tokens", c_int)]


class MokSched(ctypes.Structure):
    _fields_ = [(n, c_void_p) for n in ("topk_idx", "gates", "counts", "offsets", "table",
                                        "inv", "aux")]


class MokWeights(ctypes.Structure):
    _fields_ = [(n, c_void_p) for n in ("W_up", "W_gate", "W_down", "Ws_up", "Ws_gate",
                                        "Ws_down", "mx")]


class MokGrads(ctypes.Structure):
    _fields_ = [(n, c_void_p) for n in ("dW_up", "dW_gate", "dW_down", "dgates", "dWr",
                                        "dWs_up", "dWs_gate", "dWs_down")]


class MokSizes(ctypes.Structure):
    _fields_ = [("aux_bytes", c_size_t), ("workspace_bytes", c_size_t),
                ("saved_bytes", c_size_t), ("mx_weight_bytes", c_size_t),
                ("padded_rows_max", c_int), ("macrobatches", c_int), ("ring_slots", c_int),
                ("macrobatch_tokens", c_int)]


class MokError(RuntimeError):
    def __init__(self, what, status):
        super().__init__(f"{what}: {mok_status_string(status)} ({status})")
        self.status = status


_LIB = None
_P = ctypes.POINTER


def _declare(L):
    sig = {
        "mok_create": (c_int, [_P(MokDims), _P(c_void_p)]),
        "mok_destroy": (None, [c_void_p]),
        "mok_get_sizes": (c_int, [c_void_p, _P(MokSizes)]),
        "mok_minibatch_tokens": (c_int, [c_int, c_int, c_int, c_int]),
        "mok_status_string": (c_char_p, [c_int]),
        "mok_set_precision": (c_int, [c_void_p, c_int]),
        "mok_set_output_dtype": (c_int, [c_void_p, c_int]),
        "mok_set_tile_order": (c_int, [c_void_p, c_int]),
        "mok_set_row_pairs": (c_int, [c_void_p, c_int]),
        "mok_set_sm_pairs": (c_int, [c_void_p, c_int]),
        "mok_set_fwd_path": (c_int, [c_void_p, c_int]),
        "mok_set_comm_sms": (c_int, [c_void_p, c_int]),
        "mok_set_sm_limit": (c_int, [c_void_p, c_int]),
        "mok_set_wait_timeout": (c_int, [c_void_p, ctypes.c_uint64]),
        "mok_test_withhold_signal": (c_int, [c_void_p, c_int]),
        "mok_plan": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, _P(MokSched), c_void_p,
                             c_void_p]),
        "mok_moe_fwd": (c_int, [c_void_p, _P(MokSched), c_void_p, _P(MokWeights), c_void_p,
                                c_void_p, c_void_p, c_void_p]),
        "mok_moe_bwd": (c_int, [c_void_p, _P(MokSched), c_void_p, c_void_p, _P(MokWeights),
                                c_void_p, c_void_p, c_void_p, _P(MokGrads), c_void_p,
                                c_void_p]),
        "mok_quantize_weights_mxfp8": (c_int, [c_void_p, _P(MokWeights), c_void_p, c_void_p]),
        "mok_get_status": (c_int, [c_void_p, _P(MokSched), c_void_p]),
        "mok_plan_noalloc": (c_int, [c_void_p, _P(MokSched), c_void_p]),
        "mok_profile_enable": (c_int, [c_void_p, c_int]),
        "mok_profile_report": (c_int, [c_void_p, c_char_p, c_size_t, _P(c_int)]),
    }
    for name, (res, args) in sig.items():
        f = getattr(L, name)
        f.restype = res
        f.argtypes = args


def lib():
    """The loaded libmok (raises if it has not been built)."""
    global _LIB
    if _LIB is None:
        p = lib_path()
        if not os.path.exists(p):
            raise RuntimeError(f"libmok is not built ({p}); run __graft_entry__.build()")
        L = ctypes.CDLL(p)
        _declare(L)
        _LIB = L
    return _LIB


def declared_symbols():
    """Names of the functions declared in include/*.h."""
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    inc = os.path.join(root, "include")
    names = set()
    for f in sorted(os.listdir(inc)):
        if f.endswith(".h"):
            text = re.sub(r"/\*.*?\*/", "", open(os.path.join(inc, f)).read(), flags=re.S)
            names.update(re.findall(r"\b(mok_[a-z0-9_]+)\s*\(", text))
    return sorted(names)


def _check(st, what):
    if st != MOK_OK:
        raise MokError(what, st)


def _v(p):
    return None if p is None or p == 0 else ctypes.c_void_p(int(p))


# ----------------------------------------------------------------- same names as the ABI
def mok_status_string(status: int) -> str:
    return lib().mok_status_string(int(status)).decode()


def mok_minibatch_tokens(H: int, I: int, k: int, num_sms: int) -> int:
    return lib().mok_minibatch_tokens(H, I, k, num_sms)


def mok_create(dims: MokDims):
    h = c_void_p()
    _check(lib().mok_create(ctypes.byref(dims), ctypes.byref(h)), "mok_create")
    return h


def mok_destroy(ctx) -> None:
    lib().mok_destroy(ctx)


def mok_get_sizes(ctx) -> MokSizes:
    s = MokSizes()
    _check(lib().mok_get_sizes(ctx, ctypes.byref(s)), "mok_get_sizes")
    return s


def mok_set_precision(ctx, precision: int) -> None:
    _check(lib().mok_set_precision(ctx, int(precision)), "mok_set_precision")


def mok_set_tile_order(ctx, order: int) -> None:
    _check(lib().mok_set_tile_order(ctx, int(order)), "mok_set_tile_order")


def mok_set_row_pairs(ctx, mode: int) -> None:
    _check(lib().mok_set_row_pairs(ctx, int(mode)), "mok_set_row_pairs")


def mok_set_sm_pairs(ctx, mode: int) -> None:
    _check(lib().mok_set_sm_pairs(ctx, int(mode)), "mok_set_sm_pairs")


def mok_set_output_dtype(ctx, out_dtype: int) -> None:
    _check(lib().mok_set_output_dtype(ctx, int(out_dtype)), "mok_set_output_dtype")


def mok_set_fwd_path(ctx, path: int) -> None:
    _check(lib().mok_set_fwd_path(ctx, int(path)), "mok_set_fwd_path")


def mok_set_sm_limit(ctx, n: int) -> None:
    _check(lib().mok_set_sm_limit(ctx, int(n)), "mok_set_sm_limit")


def mok_set_comm_sms(ctx, n: int) -> None:
    _check(lib().mok_set_comm_sms(ctx, int(n)), "mok_set_comm_sms")


def mok_set_wait_timeout(ctx, ns: int) -> None:
    _check(lib().mok_set_wait_timeout(ctx, int(ns)), "mok_set_wait_timeout")


def mok_test_withhold_signal(ctx, on: bool) -> None:
    _check(lib().mok_test_withhold_signal(ctx, 1 if on else 0), "mok_test_withhold_signal")


def mok_plan(ctx, x, Wr, bias, sched: MokSched, workspace, stream) -> None:
    _check(lib().mok_plan(ctx, _v(x), _v(Wr), _v(bias), ctypes.byref(sched), _v(workspace),
                          _v(stream)), "mok_plan")


def mok_moe_fwd(ctx, sched: MokSched, x, weights: MokWeights, y, saved, workspace,
                stream) -> None:
    _check(lib().mok_moe_fwd(ctx, ctypes.byref(sched), _v(x), ctypes.byref(weights), _v(y),
                             _v(saved), _v(workspace), _v(stream)), "mok_moe_fwd")


def mok_moe_bwd(ctx, sched: MokSched, x, Wr, weights: MokWeights, saved, dY, dX,
                grads: MokGrads, workspace, stream) -> None:
    _check(lib().mok_moe_bwd(ctx, ctypes.byref(sched), _v(x), _v(Wr), ctypes.byref(weights),
                             _v(saved), _v(dY), _v(dX), ctypes.byref(grads), _v(workspace),
                             _v(stream)), "mok_moe_bwd")


def mok_quantize_weights_mxfp8(ctx, weights: MokWeights, mx_out, stream) -> None:
    _check(lib().mok_quantize_weights_mxfp8(ctx, ctypes.byref(weights), _v(mx_out),
                                            _v(stream)), "mok_quantize_weights_mxfp8")


def mok_get_status(ctx, sched: MokSched, stream) -> int:
    """Synchronises the stream; returns the device status (0 = ok) and clears it."""
    return lib().mok_get_status(ctx, ctypes.byref(sched), _v(stream))


def mok_plan_noalloc(ctx, sched: MokSched, stream) -> None:
    """Schedule from caller-supplied routing, with no workspace (see include/mok.h)."""
    _check(lib().mok_plan_noalloc(ctx, ctypes.byref(sched), _v(stream)), "mok_plan_noalloc")


def mok_profile_enable(ctx, enable: bool) -> None:
    _check(lib().mok_profile_enable(ctx, 1 if enable else 0), "mok_profile_enable")


def mok_profile_report(ctx):
    """Returns ({kernel name: (launches, total_ms)}, total launches); clears the records."""
    buf = ctypes.create_string_buffer(1 << 16)
    n = c_int(0)
    _check(lib().mok_profile_report(ctx, buf, len(buf), ctypes.byref(n)), "mok_profile_report")
    out = {}
    for line in buf.value.decode().splitlines():
        name, cnt, ms = line.split()
        out[name] = (int(cnt), float(ms))
    return out, n.value
