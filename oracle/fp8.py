"""Oracle FP8 (E4M3) KV cache: the 8-bit storage format, quantised writes, dequantisation.

Test infrastructure (see the package docstring). Plain Python / NumPy, code by code.

Source: vLLM docs page (docs.acceleratez.fun, "vLLM"), 量化支持 (quantisation support),
its format table: FP8, 8-bit, 2x compression against 16-bit storage, for newer GPUs.

The pages name the format only. Readings (the plainest ones):
- FP8 is E4M3 as NVIDIA GPUs implement it (the OCP 8-bit "E4M3" encoding): 1 sign bit,
  4 exponent bits with bias 7, 3 mantissa bits; exponent field 0 is subnormal
  (value m/8 * 2^-6); there are no infinities; S.1111.111 is NaN, so the largest
  finite magnitude is 1.75 * 2^8 = 448.
- One scale per cache tensor (one for K, one for V), given by the caller: the stored
  code of a value x is E4M3(x / scale) and it stands for E4M3-value * scale.
- x / scale is one IEEE binary32 division (x first widened to binary32), rounded to
  nearest even; the binary32 result is rounded to E4M3 to nearest, ties to even, and a
  magnitude beyond 448 saturates to 448 (the inputs are finite).
- Attention reads the dequantised values; everything after that is the bf16 path's
  arithmetic (float64 here).
"""
from __future__ import annotations

import numpy as np

MAX_E4M3 = 448.0


def e4m3_decode(code: int) -> float:
    """The value of one E4M3 code (NaN for the two NaN codes)."""
    code = int(code) & 0xFF
    s = -1.0 if code & 0x80 else 1.0
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0xF and m == 0x7:
        return float("nan")
    if e == 0:
        return s * (m / 8.0) * 2.0 ** -6
    return s * (1.0 + m / 8.0) * 2.0 ** (e - 7)


DECODE_TABLE = np.array([e4m3_decode(c) for c in range(256)], np.float64)


def e4m3_encode(x: float) -> int:
    """Round a finite value to the nearest E4M3 code, ties to the even code, saturating at
    +-448. Written over the list of finite non-negative codes (0x00 .. 0x7E, increasing)."""
    x = float(x)
    sign = 0x80 if (x < 0 or (x == 0 and np.signbit(x))) else 0
    a = abs(x)
    if a >= MAX_E4M3:
        return sign | 0x7E
    lo = 0
    while lo + 1 <= 0x7E and DECODE_TABLE[lo + 1] <= a:
        lo += 1
    if DECODE_TABLE[lo] == a or lo == 0x7E:
        return sign | lo
    hi = lo + 1
    d_lo, d_hi = a - DECODE_TABLE[lo], DECODE_TABLE[hi] - a
    if d_lo < d_hi:
        return sign | lo
    if d_hi < d_lo:
        return sign | hi
    return sign | (lo if lo % 2 == 0 else hi)  # a tie: the even code (mantissa LSB 0)


_POS = DECODE_TABLE[:0x7F]  # finite non-negative codes 0x00 .. 0x7E, increasing values


def e4m3_encode_array(a: np.ndarray) -> np.ndarray:
    """``e4m3_encode`` over an array (the same rule, vectorised): the largest code whose
    value is <= |x|, or the next one if that is nearer or equally near and even."""
    a = np.asarray(a, np.float64)
    mag = np.abs(a)
    lo = np.searchsorted(_POS, mag, side="right") - 1
    lo = np.clip(lo, 0, 0x7E)
    hi = np.minimum(lo + 1, 0x7E)
    d_lo, d_hi = mag - _POS[lo], _POS[hi] - mag
    up = (d_hi < d_lo) | ((d_hi == d_lo) & (lo % 2 == 1))
    code = np.where(up & (hi != lo), hi, lo)
    code = np.where(mag >= MAX_E4M3, 0x7E, code)
    sign = np.where(np.signbit(a), 0x80, 0)
    return (code | sign).astype(np.uint8)


def quantize(x: np.ndarray, scale: float) -> np.ndarray:
    """float32 values -> E4M3 codes (uint8, same shape): E4M3(float32(x) / float32(scale))."""
    x32 = np.asarray(x, np.float32)
    q32 = (x32 / np.float32(scale)).astype(np.float32)
    return e4m3_encode_array(q32)


def dequantize(codes: np.ndarray, scale: float) -> np.ndarray:
    """E4M3 codes -> float64 values times the scale."""
    return DECODE_TABLE[np.asarray(codes, np.uint8)] * float(scale)


def kv_write_fp8_ref(k_cache, v_cache, k32, v32, slot_mapping, block_size, k_scale, v_scale):
    """For every t with s = slot_mapping[t] >= 0: cache[s // B, s % B] = E4M3(x[t] / scale).

    k32, v32: [T, Hkv, D] float32 (inputs widened exactly); caches: uint8 arrays
    [NB, B, Hkv, D] (or BlockStores of uint8 blocks)."""
    kq, vq = quantize(k32, k_scale), quantize(v32, v_scale)
    for t, s in enumerate(np.asarray(slot_mapping).tolist()):
        if s < 0:
            continue
        b, o = s // block_size, s % block_size
        kb = k_cache.block_for_write(b) if hasattr(k_cache, "block_for_write") else k_cache[b]
        vb = v_cache.block_for_write(b) if hasattr(v_cache, "block_for_write") else v_cache[b]
        kb[o] = kq[t]
        vb[o] = vq[t]
