"""Oracle for the FP8 (E4M3) KV-cache codec.

TEST INFRASTRUCTURE ONLY (see the package docstring).

The pages name a reduced-precision KV cache (vLLM's --kv-cache-dtype, in
"10 Serving Engines", section 10.2.2; "3.6 ModelRunner, CUDA Graph, and
benchmarks", section 4 notes nano-vllm has none) without fixing a format.
The reading taken here is the common one: OCP FP8 E4M3 with a per-tensor
float scale.  An element x is stored as e4m3(x / scale) and read back as
decode(code) * scale.

E4M3 by its definition: 1 sign bit, 4 exponent bits with bias 7, 3 mantissa
bits; exponent field 0 encodes subnormals mantissa/8 * 2^-6; codes 0x7F and
0xFF are NaN; there are no infinities, so the largest finite magnitude is
(1 + 6/8) * 2^8 = 448.  Encoding rounds to the nearest representable value,
ties to the even code, and saturates finite values beyond +-448 to +-448.
"""

from __future__ import annotations

import numpy as np


def e4m3_decode(codes) -> np.ndarray:
    """float64 values of E4M3 codes (uint8); NaN for 0x7F / 0xFF."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    exp = (c >> 3) & 0xF
    mant = c & 0x7
    sub = mant / 8.0 * 2.0 ** -6
    normal = (1.0 + mant / 8.0) * np.power(2.0, exp - 7)
    mag = np.where(exp == 0, sub, normal)
    mag = np.where((exp == 15) & (mant == 7), np.nan, mag)
    return sign * mag


# all non-negative finite codes 0x00..0x7E in increasing value order
_POS_CODES = np.arange(0x7F, dtype=np.uint8)
_POS_VALUES = e4m3_decode(_POS_CODES)


def e4m3_encode(x) -> np.ndarray:
    """Nearest E4M3 code (uint8) of each value, ties to even, finite values saturating at +-448.

    NaN maps to 0x7F; the sign of zero is kept.
    """
    x = np.asarray(x, dtype=np.float64)
    neg = np.signbit(x)
    mag = np.minimum(np.abs(x), 448.0)
    hi = np.searchsorted(_POS_VALUES, mag, side="left")  # first value >= mag
    hi = np.minimum(hi, len(_POS_VALUES) - 1)
    lo = np.maximum(hi - 1, 0)
    d_lo = mag - _POS_VALUES[lo]
    d_hi = _POS_VALUES[hi] - mag
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (_POS_CODES[hi] % 2 == 0) & (hi != lo))
    exact = _POS_VALUES[hi] == mag
    code = np.where(exact | pick_hi, _POS_CODES[hi], _POS_CODES[lo]).astype(np.uint8)
    code = np.where(neg, code | 0x80, code).astype(np.uint8)
    return np.where(np.isnan(x), np.uint8(0x7F), code).astype(np.uint8)


def quantize(x, scale: float) -> np.ndarray:
    """Stored codes of x / scale, the division done in float32 like the kernel's input."""
    q = np.asarray(x, dtype=np.float32) / np.float32(scale)
    return e4m3_encode(q.astype(np.float64))


def dequantize(codes, scale: float) -> np.ndarray:
    """float64 values read back from the cache: decode(code) * scale."""
    return e4m3_decode(codes) * float(np.float32(scale))


def kv_store_fp8(k_cache, v_cache, k, v, slot_mapping, k_scale: float, v_scale: float):
    """Quantizing slot scatter: cache[slot] = e4m3(row / scale) for slot >= 0; returns copies.

    Same slot rule as the bf16 store ("3.6 ModelRunner ...", sections 2 and 5):
    slot = block * block_size + offset, -1 writes nothing.
    """
    k_out = np.array(k_cache, dtype=np.uint8, copy=True)
    v_out = np.array(v_cache, dtype=np.uint8, copy=True)
    bs = k_out.shape[1]
    for i, slot in enumerate(np.asarray(slot_mapping).tolist()):
        if slot == -1:
            continue
        if not 0 <= slot < k_out.shape[0] * bs:
            raise IndexError(f"slot {slot} outside the cache")
        blk, off = divmod(slot, bs)
        k_out[blk, off] = quantize(k[i], k_scale)
        v_out[blk, off] = quantize(v[i], v_scale)
    return k_out, v_out
