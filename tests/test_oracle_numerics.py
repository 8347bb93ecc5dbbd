"""Pins of the oracle's number formats against library routines, closed forms and
exhaustive enumeration (no GPU)."""
import math

import numpy as np
import pytest
import torch

from oracle import numerics as nu


def test_bf16_round_matches_torch(rng):
    v = np.concatenate([
        rng.normal(0, 1, 20000), rng.normal(0, 1e-3, 2000), rng.normal(0, 1e4, 2000),
        [0.0, -0.0, 1.0, -2.5, 3.0e38, 1e-40],
    ])
    # exact halfway cases between neighbouring bf16 values: ties go to even
    base = torch.tensor(rng.normal(0, 1, 500), dtype=torch.float32).to(torch.bfloat16).float()
    bits = base.view(torch.int32)
    nxt = (bits + (1 << 16)).view(torch.float32)
    mid = ((base.double() + nxt.double()) / 2).numpy()
    v = np.concatenate([v, mid])
    ref = torch.tensor(v, dtype=torch.float64).to(torch.bfloat16).double().numpy()
    got = nu.bf16_round(v)
    assert np.array_equal(got, ref)


def test_e4m3_table_known_values():
    t = nu.e4m3_decode_table()
    assert t[0x7E] == 448.0                    # largest finite
    assert t[0x01] == 2.0 ** -9                # smallest subnormal
    assert t[0x08] == 2.0 ** -6                # smallest normal
    assert t[0x38] == 1.0
    assert t[0x78] == 256.0
    assert math.isnan(t[0x7F]) and math.isnan(t[0xFF])
    assert t[0x80] == 0.0 and math.copysign(1, t[0x80]) == -1.0
    finite = t[~np.isnan(t)]
    assert len(finite) == 254


def test_e4m3_roundtrip_all_codes():
    t = nu.e4m3_decode_table()
    codes = np.array([c for c in range(256) if not np.isnan(t[c])], dtype=np.uint8)
    assert np.array_equal(nu.e4m3_encode(t[codes]), codes)


def test_e4m3_encode_matches_torch_in_range(rng):
    v = np.concatenate([rng.uniform(-448, 448, 20000), rng.normal(0, 0.01, 5000),
                        rng.normal(0, 1, 5000)])
    t = nu.e4m3_decode_table()
    pos = t[:0x7F]
    mids = (pos[1:] + pos[:-1]) / 2                 # every tie between neighbours
    v = np.concatenate([v, mids, -mids])
    ref = torch.tensor(v, dtype=torch.float32).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(nu.e4m3_encode(v), ref)


def test_e4m3_saturates():
    codes = nu.e4m3_encode(np.array([448.0, 460.0, 464.0, 500.0, 1e30, -1e30, -449.0]))
    assert list(codes) == [0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0xFE]


@pytest.mark.parametrize("s", [-20, -3, 0, 5, 40])
def test_mx_scale_for_amax_448_times_power_of_two(s, rng):
    blk = rng.uniform(-1, 1, (4, 32)) * 448.0 * 2.0 ** s
    blk[:, 7] = 448.0 * 2.0 ** s                     # amax = 448 * 2^s exactly
    codes, scales = nu.mx_quantize(blk, axis=1)
    assert np.all(scales == 127 + s)
    ref = torch.tensor(blk / 2.0 ** s, dtype=torch.float32).to(torch.float8_e4m3fn)
    assert np.array_equal(codes, ref.view(torch.uint8).numpy())


def test_mx_powers_of_two_closed_form():
    for p in (-30, -1, 0, 1, 7, 60):
        blk = np.full((1, 32), 2.0 ** p)
        codes, scales = nu.mx_quantize(blk, axis=1)
        assert scales[0, 0] == 127 + p - 8           # X = 2^(p-8)
        assert np.all(codes == 0x78)                 # element 2^8 = 256


def test_mx_zero_block_and_saturation():
    codes, scales = nu.mx_quantize(np.zeros((2, 64)), axis=1)
    assert np.all(scales == 127) and np.all(codes == 0)
    blk = np.zeros((1, 32))
    blk[0, 0] = 500.0                                # floor(log2 500) = 8 -> X = 1
    codes, scales = nu.mx_quantize(blk, axis=1)
    assert scales[0, 0] == 127 and codes[0, 0] == 0x7E


def test_mx_axis_and_error_bound(rng):
    a = rng.normal(0, 1, (64, 96)) * np.exp(rng.normal(0, 2, (64, 1)))
    for axis in (0, 1):
        q = nu.mx_qdq(a, axis)
        c, s = nu.mx_quantize(a, axis)
        assert s.shape[axis] == a.shape[axis] // 32
        X = np.repeat(np.ldexp(1.0, s.astype(int) - 127), 32, axis=axis)
        # normal E4M3 range: relative error <= 2^-4; subnormal range: <= 2^-10 * X;
        # |a|/X in (448, 512) saturates to 448 X
        bound = np.maximum.reduce([2.0 ** -4 * np.abs(a), 2.0 ** -10 * X, np.abs(a) - 448 * X])
        assert np.all(np.abs(q - a) <= bound * (1 + 1e-12))
    # blocks along axis 0 of the transposed matrix equal blocks along axis 1
    assert np.array_equal(nu.mx_qdq(a.T, 0), nu.mx_qdq(a, 1).T)


def test_mx_rows_padded_equals_explicit_zero_rows(rng):
    a = rng.normal(0, 1, (45, 64))
    q = nu.mx_qdq_rows_padded(a)
    full = np.concatenate([a, np.zeros((19, 64))])
    assert np.array_equal(q, nu.mx_qdq(full, 0)[:45])


def test_silu_and_derivative():
    v = np.linspace(-8, 8, 161)
    assert np.allclose(nu.silu(v), v / (1 + np.exp(-v)), rtol=1e-15, atol=0)
    eps = 1e-6
    fd = (nu.silu(v + eps) - nu.silu(v - eps)) / (2 * eps)
    assert np.allclose(nu.dsilu(v), fd, rtol=1e-8, atol=1e-10)
