"""Pins for the oracle's E4M3 codec (CPU only): values fixed by the format's
definition, round trips, torch's float8_e4m3fn conversion inside the finite
range (a library routine), saturation, and ties to even."""

import numpy as np
import pytest
import torch

from oracle import fp8


def test_decode_known_codes():
    # (code, value) fixed by the format: bias 7, 3 mantissa bits, subnormals below 2^-6
    table = {0x00: 0.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6, 0x38: 1.0, 0x3C: 1.5,
             0x40: 2.0, 0x7E: 448.0, 0x80: -0.0, 0xB8: -1.0, 0xFE: -448.0}
    for code, value in table.items():
        assert fp8.e4m3_decode(np.uint8(code)) == value
    assert np.isnan(fp8.e4m3_decode(np.uint8(0x7F))) and np.isnan(fp8.e4m3_decode(np.uint8(0xFF)))


def test_every_finite_code_round_trips():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    assert np.array_equal(fp8.e4m3_encode(fp8.e4m3_decode(codes)), codes)


def test_matches_torch_float8_inside_the_finite_range():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(20000) * s for s in (0.01, 1.0, 30.0, 150.0)])
    x = np.clip(x, -448, 448).astype(np.float32)
    want = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = fp8.e4m3_encode(x.astype(np.float64))
    assert np.array_equal(got, want)


def test_saturation_and_nan():
    assert fp8.e4m3_encode(500.0) == 0x7E
    assert fp8.e4m3_encode(-1e9) == 0xFE
    assert fp8.e4m3_encode(464.0) == 0x7E  # beyond the largest value, not rounded up to NaN
    assert fp8.e4m3_encode(np.nan) == 0x7F


@pytest.mark.parametrize("x,code", [(232.0, 0x76), (248.0, 0x78), (1.0625, 0x38), (1.1875, 0x3A),
                                    (2.0 ** -10, 0x00), (3 * 2.0 ** -10, 0x02)])
def test_ties_go_to_even(x, code):
    # each x lies exactly halfway between two neighbours; the even code wins
    assert fp8.e4m3_encode(x) == code


def test_quantize_divides_in_float32():
    x = np.float32(3.0)
    assert fp8.quantize(x, 0.1) == fp8.e4m3_encode(np.float64(np.float32(3.0) / np.float32(0.1)))
    assert fp8.dequantize(fp8.quantize(np.float32(1.0), 0.5), 0.5) == 1.0


def test_quantize_rounds_the_float32_quotient():
    # The store divides in float32 (the kernel's input precision).  For these
    # inputs the float32 quotient x / scale lands exactly on the midpoint
    # between two E4M3 values while the exact quotient lies just above it, so
    # the stored code must be the midpoint's even neighbour.  Expected codes
    # come from numpy's IEEE float32 division and torch's float8 conversion.
    found = 0
    for mid in (1.0625, 2.125, 17.0):  # midpoints of (1, 1.125), (2, 2.25), (16, 18)
        for k in range(200):
            s = np.float32(0.1 + 0.00037 * k)
            x = np.float32(mid * float(s))
            q32 = x / s
            if q32 != np.float32(mid) or not float(x) / float(s) > mid:
                continue
            want = torch.tensor(float(q32), dtype=torch.float32).to(torch.float8_e4m3fn).view(torch.uint8).item()
            assert fp8.quantize(x, float(s)) == want
            found += 1
    assert found >= 10


def test_kv_store_fp8_closed_form():
    # each token's K and V rows land, quantized with their own scale, at (block, offset) found by
    # walking the pool block by block; slot -1 and every other byte are left as they were
    rng = np.random.default_rng(7)
    num_blocks, bs, hkv, d = 6, 4, 2, 8
    k_cache = rng.integers(0, 256, (num_blocks, bs, hkv, d), dtype=np.uint8)
    v_cache = rng.integers(0, 256, (num_blocks, bs, hkv, d), dtype=np.uint8)
    slots = [9, -1, 0, 23, 14]
    k = (rng.standard_normal((len(slots), hkv, d)) * 3).astype(np.float32)
    v = (rng.standard_normal((len(slots), hkv, d)) * 3).astype(np.float32)
    k_scale, v_scale = 0.05, 0.02
    k_out, v_out = fp8.kv_store_fp8(k_cache, v_cache, k, v, slots, k_scale, v_scale)
    want_k, want_v = k_cache.copy(), v_cache.copy()
    def code(x, scale):  # float32 quotient, saturated at the largest finite value, then torch's conversion
        quot = min(max(float(np.float32(x) / np.float32(scale)), -448.0), 448.0)
        return torch.tensor(quot).to(torch.float8_e4m3fn).view(torch.uint8).item()

    flat = 0
    for blk in range(num_blocks):
        for off in range(bs):
            if flat in slots:
                i = slots.index(flat)
                want_k[blk, off] = [[code(x, k_scale) for x in row] for row in k[i]]
                want_v[blk, off] = [[code(x, v_scale) for x in row] for row in v[i]]
            flat += 1
    assert np.array_equal(k_out, want_k)
    assert np.array_equal(v_out, want_v)
    with pytest.raises(IndexError):
        fp8.kv_store_fp8(k_cache, v_cache, k[:1], v[:1], [num_blocks * bs], k_scale, v_scale)
