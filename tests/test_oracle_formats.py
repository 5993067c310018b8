"""Pins for the oracle's block formats (hand-built blocks, bounds, bijection)."""
import struct

import numpy as np
import pytest

from oracle import formats as F


def _fp16_bytes(v):
    return struct.pack("<e", v)


# ---------------------------------------------------------------- Q8_0
def test_q8_0_hand_built_block_roundtrip():
    # w = 2^-7 * q with max |q| = 127: d = 127 * 2^-7 / 127 = 2^-7 exactly.
    q = np.arange(-127, 128, 8)  # 32 codes, -127 .. 121
    q[5] = 127
    w = (q.astype(np.float64) * 2.0 ** -7).astype(np.float32)[None, :]
    blob = F.q8_0_quantize(w)
    expect = _fp16_bytes(2.0 ** -7) + bytes((int(v) & 0xFF) for v in q)
    assert blob.tobytes() == expect
    assert np.array_equal(F.q8_0_dequantize(blob, 1, 32), w)


def test_q8_0_zero_block():
    blob = F.q8_0_quantize(np.zeros((2, 64), np.float32))
    assert not blob.any()
    assert not F.q8_0_dequantize(blob, 2, 64).any()


def test_q8_0_decode_hand_bytes():
    # d = 0.5, q = -16..15 -> w = 0.5 q exactly
    q = np.arange(-16, 16)
    raw = _fp16_bytes(0.5) + bytes((int(v) & 0xFF) for v in q)
    w = F.q8_0_dequantize(np.frombuffer(raw, np.uint8)[None, :], 1, 32)
    assert np.array_equal(w[0], 0.5 * q.astype(np.float32))


def test_q8_0_sign_symmetry_and_half_away():
    rng = np.random.default_rng(3)
    w = rng.normal(0, 0.02, (8, 256)).astype(np.float32)
    a, b = F.q8_0_quantize(w), F.q8_0_quantize(-w)
    a3, b3 = a.reshape(8, 8, 34), b.reshape(8, 8, 34)
    assert np.array_equal(a3[..., :2], b3[..., :2])
    qa = a3[..., 2:].view(np.int8).astype(int)
    qb = b3[..., 2:].view(np.int8).astype(int)
    assert np.array_equal(qa, -qb)
    # an exact half rounds away from zero: max 127 (d = 1), w = 2.5 -> 3, -2.5 -> -3
    w = np.zeros((1, 32), np.float32)
    w[0, 0], w[0, 1], w[0, 2] = 127.0, 2.5, -2.5
    q = F.q8_0_quantize(w)[0, 2:].view(np.int8)
    assert (q[0], q[1], q[2]) == (127, 3, -3)


def test_q8_0_error_bound():
    rng = np.random.default_rng(4)
    w = rng.normal(0, 0.02, (64, 512)).astype(np.float32)
    r = F.q8_0_dequantize(F.q8_0_quantize(w), 64, 512)
    b = w.reshape(64, 16, 32).astype(np.float64)
    d32 = (np.abs(b).max(axis=2) / 127.0)
    d16 = d32.astype(np.float32).astype(np.float16).astype(np.float64)
    # |w - d16 q| <= d32/2 + 127 |d32 - d16| (rounding of q, then of d)
    bound = d32 / 2 + 127 * np.abs(d32 - d16) + 1e-12
    err = np.abs(r.reshape(64, 16, 32) - b).max(axis=2)
    assert (err <= bound * (1 + 1e-6)).all()


# ---------------------------------------------------------------- Q4KS
def _pack_bits_reference(fields):
    v = 0
    for i, f in enumerate(fields):
        assert 0 <= f < 64
        v |= int(f) << (6 * i)
    return v.to_bytes(12, "little")


def test_fields6_bijection_exhaustive_per_field():
    rng = np.random.default_rng(5)
    base = rng.integers(0, 64, 16)
    for pos in range(16):
        for val in range(64):
            f = base.copy()
            f[pos] = val
            packed = F.pack_fields6(f[None, :])[0]
            assert packed.tobytes() == _pack_bits_reference(f)
            assert np.array_equal(F.unpack_fields6(packed[None, :])[0], f)


def _hand_superblock(d, dmin, sc, m, q):
    raw = _fp16_bytes(d) + _fp16_bytes(dmin) + _pack_bits_reference(list(sc) + list(m))
    qb = bytes(int(q[2 * i]) | (int(q[2 * i + 1]) << 4) for i in range(128))
    return np.frombuffer(raw + qb, np.uint8)


def test_q4ks_decode_hand_built():
    rng = np.random.default_rng(6)
    d, dmin = 2.0 ** -9, 3 * 2.0 ** -10
    sc = rng.integers(0, 64, 8)
    m = rng.integers(0, 64, 8)
    q = rng.integers(0, 16, 256)
    blob = _hand_superblock(d, dmin, sc, m, q)
    w = F.q4ks_dequantize(blob[None, :], 1, 256)[0]
    exact = np.array([d * sc[i // 32] * q[i] - dmin * m[i // 32] for i in range(256)])
    assert np.array_equal(w, exact.astype(np.float32))


def test_q4ks_quantize_recovers_hand_built():
    # Sub-blocks whose codes reach 0 and 15 and whose largest sc / m are 63
    # are reproduced exactly by the closed-form quantiser.
    rng = np.random.default_rng(7)
    d, dmin = 2.0 ** -10, 2.0 ** -11
    sc = np.array([63, 40, 17, 5, 63, 1, 30, 22])
    m = np.array([12, 63, 0, 9, 33, 63, 2, 50])
    q = rng.integers(0, 16, 256)
    for s in range(8):
        q[32 * s] = 0
        q[32 * s + 1] = 15
    w = np.array([d * sc[i // 32] * q[i] - dmin * m[i // 32] for i in range(256)])
    w = w.astype(np.float32)[None, :]
    blob = F.q4ks_quantize(w)
    assert blob.tobytes() == _hand_superblock(d, dmin, sc, m, q).tobytes()


def test_q4ks_error_bound():
    rng = np.random.default_rng(8)
    w = rng.normal(0, 0.02, (16, 1024)).astype(np.float32)
    r = F.q4ks_dequantize(F.q4ks_quantize(w), 16, 1024)
    sub = w.reshape(16, 4, 8, 32).astype(np.float64)
    lo = np.minimum(0, sub.min(axis=3))
    A = (sub.max(axis=3) - lo) / 15
    err = np.abs(r.reshape(16, 4, 8, 32) - sub).max(axis=3)
    # half a code step plus what the 6-bit scale / min rounding moves:
    # |a - A| <= d/2 per step over 15 steps, |b - B| <= dmin/2
    blob = F.q4ks_quantize(w).reshape(16, 4, 144)
    d = np.ascontiguousarray(blob[..., 0:2]).view("<f2").astype(np.float64)
    dm = np.ascontiguousarray(blob[..., 2:4]).view("<f2").astype(np.float64)
    bound = A / 2 + d * (0.5 + 7.5) + dm / 2 + 1e-9
    assert (err <= bound).all()
    assert np.median(err / A) < 0.6


def test_q4ks_zero_and_constant():
    assert not F.q4ks_dequantize(F.q4ks_quantize(np.zeros((1, 256), np.float32)), 1, 256).any()
    w = np.full((1, 256), -0.25, np.float32)
    r = F.q4ks_dequantize(F.q4ks_quantize(w), 1, 256)
    assert np.abs(r - w).max() <= 0.25 / 63 / 2 * 1.01 + 0.25 * 2 ** -11
