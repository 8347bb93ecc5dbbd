"""Number formats for the oracle: bf16 rounding, OCP E4M3 and MXFP8 (E4M3 + UE8M0 per 32).

TEST INFRASTRUCTURE ONLY (see oracle/__init__.py). Plain NumPy, float64 throughout.

The articles name the format only: "MXFP8" ("Determinismus und MXFP8-Unterstützung" on
the sebask.de page; "Outras características" on the stamatios.com page). The block rule
written out here is the plain reading of that name, the OCP Microscaling format:

* a block is 32 consecutive elements along the contraction (K) axis of the GEMM that
  consumes the operand;
* its shared scale is a power of two X = 2^(floor(log2(amax)) - 8), 8 being the exponent
  of E4M3's largest normal (448 = 1.75 * 2^8); the exponent is clamped to [-127, 127]
  and stored as UE8M0, i.e. the biased byte e + 127;
* an all-zero block gets exponent 0 (byte 127);
* each element is v / X rounded to nearest-even E4M3, saturating at +-448.
"""
from __future__ import annotations

import numpy as np

MX_BLOCK = 32
E4M3_MAX = 448.0
E4M3_EMAX = 8


# ----------------------------------------------------------------------------- bf16
def bf16_round(a) -> np.ndarray:
    """Round float64 values to the nearest bf16 value, ties to even (8-bit significand,
    8-bit exponent). Returns float64 holding bf16-representable values. Values beyond
    the bf16 range become +-inf (not reached by the layer's data)."""
    a = np.asarray(a, dtype=np.float64)
    out = np.zeros_like(a)
    nz = (a != 0) & np.isfinite(a)
    m, e = np.frexp(a[nz])              # a = m * 2^e, 0.5 <= |m| < 1
    # bf16 normal: 8 significant bits -> quantum 2^(e-8); subnormal quantum 2^-133.
    q_exp = np.maximum(e - 8, -133)
    scaled = np.ldexp(a[nz], -q_exp)    # exact: a / 2^q_exp
    r = np.round(scaled)                # numpy rounds half to even
    out[nz] = np.ldexp(r, q_exp)
    out[~np.isfinite(a)] = a[~np.isfinite(a)]
    big = np.abs(out) > 3.3895313892515355e38
    out[big] = np.sign(out[big]) * np.inf
    return out


# ----------------------------------------------------------------------------- E4M3
def e4m3_decode_table() -> np.ndarray:
    """Value of each of the 256 E4M3 codes (sign, 4 exponent bits with bias 7, 3 mantissa
    bits; exponent field 0 is subnormal 2^-6 * m/8; S.1111.111 is NaN; no infinities)."""
    vals = np.empty(256, dtype=np.float64)
    for c in range(256):
        s = -1.0 if c & 0x80 else 1.0
        ef = (c >> 3) & 0xF
        mf = c & 0x7
        if ef == 0xF and mf == 0x7:
            vals[c] = np.nan
        elif ef == 0:
            vals[c] = s * (mf / 8.0) * 2.0 ** -6
        else:
            vals[c] = s * (1.0 + mf / 8.0) * 2.0 ** (ef - 7)
    return vals


_E4M3 = e4m3_decode_table()
_POS_CODES = np.arange(0, 0x7F)          # 0x00 .. 0x7E: the finite non-negative codes
_POS_VALS = _E4M3[_POS_CODES]            # ascending


def e4m3_encode(v) -> np.ndarray:
    """Round float64 values to E4M3 codes: nearest, ties to the even code, saturating
    at +-448 (values beyond the largest finite value map to it); the sign bit is the
    input's sign bit, so small negative values give -0 (0x80). NaN -> 0x7F."""
    v = np.asarray(v, dtype=np.float64)
    a = np.minimum(np.abs(v), E4M3_MAX)
    hi = np.searchsorted(_POS_VALS, a, side="left")          # first value >= a
    hi = np.clip(hi, 0, len(_POS_VALS) - 1)
    lo = np.clip(hi - 1, 0, len(_POS_VALS) - 1)
    d_hi = _POS_VALS[hi] - a
    d_lo = a - _POS_VALS[lo]
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (_POS_CODES[hi] % 2 == 0))
    code = np.where(pick_hi, _POS_CODES[hi], _POS_CODES[lo]).astype(np.uint8)
    # the sign is kept, also when the magnitude rounds to zero (IEEE-style -0 = 0x80)
    code = np.where(np.signbit(v), code | 0x80, code).astype(np.uint8)
    code = np.where(np.isnan(v), np.uint8(0x7F), code).astype(np.uint8)
    return code


def e4m3_decode(codes) -> np.ndarray:
    return _E4M3[np.asarray(codes, dtype=np.uint8)]


# ----------------------------------------------------------------------------- MXFP8
def _floor_log2(a: np.ndarray) -> np.ndarray:
    """Exact floor(log2(a)) for positive finite float64 values."""
    _, e = np.frexp(a)   # a = m 2^e with 0.5 <= m < 1  ->  floor(log2 a) = e - 1
    return e - 1


def mx_quantize(a, axis: int = -1):
    """MXFP8 quantisation of ``a`` in blocks of 32 along ``axis`` (whose length must be a
    multiple of 32). Returns (codes uint8 with a's shape, scale bytes uint8 with the
    axis length divided by 32)."""
    a = np.asarray(a, dtype=np.float64)
    a_m = np.moveaxis(a, axis, -1)
    K = a_m.shape[-1]
    if K % MX_BLOCK:
        raise ValueError("MX block axis length must be a multiple of 32")
    blk = a_m.reshape(a_m.shape[:-1] + (K // MX_BLOCK, MX_BLOCK))
    amax = np.max(np.abs(blk), axis=-1)
    e = np.zeros(amax.shape, dtype=np.int64)
    pos = amax > 0
    e[pos] = _floor_log2(amax[pos]) - E4M3_EMAX
    e = np.clip(e, -127, 127)
    scale = np.ldexp(1.0, e)
    codes = e4m3_encode(blk / scale[..., None]).reshape(a_m.shape)
    return np.moveaxis(codes, -1, axis), np.moveaxis((e + 127).astype(np.uint8), -1, axis)


def mx_dequantize(codes, scales, axis: int = -1) -> np.ndarray:
    c = np.moveaxis(np.asarray(codes), axis, -1)
    s = np.moveaxis(np.asarray(scales), axis, -1)
    vals = e4m3_decode(c)
    K = vals.shape[-1]
    vals = vals.reshape(vals.shape[:-1] + (K // MX_BLOCK, MX_BLOCK))
    vals = vals * np.ldexp(1.0, s.astype(np.int64) - 127)[..., None]
    return np.moveaxis(vals.reshape(c.shape), -1, axis)


def mx_qdq(a, axis: int = -1) -> np.ndarray:
    """Quantise then dequantise: the values an MXFP8 GEMM sees for operand ``a``."""
    c, s = mx_quantize(a, axis)
    return mx_dequantize(c, s, axis)


def mx_qdq_rows_padded(a) -> np.ndarray:
    """MXFP8 along axis 0 for a (rows x N) operand whose row count need not be a multiple
    of 32: blocks start at row 0; the last block is completed with zero rows, which do
    not change its amax."""
    a = np.asarray(a, dtype=np.float64)
    n = a.shape[0]
    pad = (-n) % MX_BLOCK
    if pad:
        a = np.concatenate([a, np.zeros((pad,) + a.shape[1:])], axis=0)
    return mx_qdq(a, axis=0)[:n]


# ----------------------------------------------------------------------------- SwiGLU
def sigmoid(v):
    v = np.asarray(v, dtype=np.float64)
    return 1.0 / (1.0 + np.exp(-v))


def silu(v):
    return np.asarray(v, dtype=np.float64) * sigmoid(v)


def dsilu(v):
    """d/dv [v * sigmoid(v)] = sigmoid(v) * (1 + v * (1 - sigmoid(v)))."""
    s = sigmoid(v)
    return s * (1.0 + v * (1.0 - s))
