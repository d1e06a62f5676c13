"""Counter-based Philox4x32-10 generator and the integer Irwin-Hall normal built on it.

Philox4x32-10 is the counter-based generator of Salmon, Moraes, Dror and Shaw,
"Parallel random numbers: as easy as 1, 2, 3" (SC'11): ten rounds of two 32x32->64
multiplies, with a Weyl-sequence key schedule.  It is written here from that
definition, vectorised over numpy uint32 arrays.  The CUDA twin in
``synth/csrc/synth.cu`` implements the same definition and must produce the same
bytes; ``tests/test_synth.py`` checks that.

Normal variates: the sum of twelve independent uniform 16-bit integers minus its
mean, divided by 2**16 (Irwin-Hall with n = 12).  Every step is exact in float32
(the sum is below 2**24 and the divisor is a power of two), so host and device
agree bit for bit.  The tails are cut at +-6 sigma, which is irrelevant for the
synthetic calibration data it feeds.

This module holds no arithmetic of the compression method itself.
"""
from __future__ import annotations

import numpy as np

PHILOX_M0 = np.uint64(0xD2511F53)
PHILOX_M1 = np.uint64(0xCD9E8D57)
PHILOX_W0 = np.uint32(0x9E3779B9)
PHILOX_W1 = np.uint32(0xBB67AE85)
_MASK32 = np.uint64(0xFFFFFFFF)
_SHIFT32 = np.uint64(32)

# Irwin-Hall with twelve 16-bit uniforms: mean 12 * 65535 / 2.
IH_TERMS = 12
IH_MEAN = 393210
IH_SCALE = np.float32(1.0 / 65536.0)


def philox4x32_10(c0, c1, c2, c3, k0, k1):
    """Ten Philox4x32 rounds on uint32 counter words (arrays broadcast) and a 2-word key."""
    c0 = np.asarray(c0, dtype=np.uint32)
    c1 = np.asarray(c1, dtype=np.uint32)
    c2 = np.asarray(c2, dtype=np.uint32)
    c3 = np.asarray(c3, dtype=np.uint32)
    k0 = np.uint32(k0)
    k1 = np.uint32(k1)
    with np.errstate(over="ignore"):
        for _ in range(10):
            p0 = PHILOX_M0 * c0.astype(np.uint64)
            p1 = PHILOX_M1 * c2.astype(np.uint64)
            hi0 = (p0 >> _SHIFT32).astype(np.uint32)
            lo0 = (p0 & _MASK32).astype(np.uint32)
            hi1 = (p1 >> _SHIFT32).astype(np.uint32)
            lo1 = (p1 & _MASK32).astype(np.uint32)
            c0, c1, c2, c3 = hi1 ^ c1 ^ k0, lo1, hi0 ^ c3 ^ k1, lo0
            k0 = np.uint32(k0 + PHILOX_W0)
            k1 = np.uint32(k1 + PHILOX_W1)
    return c0, c1, c2, c3


def key_words(seed: int):
    seed &= (1 << 64) - 1
    return np.uint32(seed & 0xFFFFFFFF), np.uint32(seed >> 32)


def _halves(w):
    return (w & np.uint32(0xFFFF)).astype(np.int64) + (w >> np.uint32(16)).astype(np.int64)


def standard_normal(elem_index, seed: int) -> np.ndarray:
    """Irwin-Hall normal for each 64-bit element index (uint64 array) under one seed.

    Element e uses the counters (e_lo, e_hi, 0, 0) and (e_lo, e_hi, 0, 1); the six
    words r0..r3 of the first call and r0, r1 of the second give the twelve 16-bit
    uniforms.  Returns float32.
    """
    e = np.asarray(elem_index, dtype=np.uint64)
    lo = (e & _MASK32).astype(np.uint32)
    hi = (e >> _SHIFT32).astype(np.uint32)
    k0, k1 = key_words(seed)
    zero = np.zeros_like(lo)
    a0, a1, a2, a3 = philox4x32_10(lo, hi, zero, zero, k0, k1)
    b0, b1, _, _ = philox4x32_10(lo, hi, zero, zero + np.uint32(1), k0, k1)
    s = _halves(a0) + _halves(a1) + _halves(a2) + _halves(a3) + _halves(b0) + _halves(b1)
    return (s - IH_MEAN).astype(np.float32) * IH_SCALE


def uniform_u32(index, seed: int, lane: int = 2) -> np.ndarray:
    """One raw 32-bit Philox word per index (counter (i_lo, i_hi, lane, 0), word 0)."""
    e = np.asarray(index, dtype=np.uint64)
    lo = (e & _MASK32).astype(np.uint32)
    hi = (e >> _SHIFT32).astype(np.uint32)
    k0, k1 = key_words(seed)
    r0, _, _, _ = philox4x32_10(lo, hi, np.zeros_like(lo) + np.uint32(lane), np.zeros_like(lo), k0, k1)
    return r0


# ---------------------------------------------------------------- bf16 helpers
def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """IEEE round-to-nearest-even float32 -> bfloat16, returned as uint16 bit patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    with np.errstate(over="ignore"):
        r = u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    out = (r >> np.uint32(16)).astype(np.uint16)
    nan = np.isnan(np.asarray(x, dtype=np.float32))
    if nan.any():
        out[nan] = np.uint16(0x7FC0)
    return out


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)
