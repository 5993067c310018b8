"""Block formats Q8_0 and Q4KS (this library's Q4_K-style type), numpy.

TEST INFRASTRUCTURE ONLY (see the package docstring).

The pages list Q8_0 for shared experts, attention and the output matrix and
Q4_K for routed experts ("Step-5 Preview GGUF", "Precision distribution"
table; "Step 3.7 Flash Mixed-Quant GGUF", "Tensor recipe" table) without
defining either layout.  The definitions used here:

Q8_0 -- 32 weights along a row, serialised as 34 bytes:
    bytes 0-1  d  (IEEE fp16, little endian), d = max|w| / 127 computed in fp32
               and rounded to fp16 (round to nearest even);
    bytes 2-33 q  (int8), q = clamp(round_half_away(w / d_fp32), -127, 127).
  An all-zero block has d = 0 and q = 0.  Decoding: w = float(d) * q, exact in
  fp32.

Q4KS -- 256 weights along a row (8 sub-blocks of 32), serialised as 144 bytes:
    bytes 0-1   d     (fp16), bytes 2-3 dmin (fp16);
    bytes 4-15  sixteen 6-bit fields as one little-endian bit stream, field f
                at bits [6f, 6f+6): fields 0-7 are sc[s], fields 8-15 are m[s];
    bytes 16-143 4-bit codes, weight i in byte 16 + i//2, low nibble for even i.
  Decoding: a = d*sc, b = dmin*m (both exact in fp32), w = fp32(a*q - b) with
  a*q exact, so one round-to-nearest on the subtraction.
  Quantiser (closed form, no search), per sub-block s:
    lo = min(0, min w), hi = max w, A_s = (hi - lo)/15, B_s = 0 - lo  (fp32)
    d = fp16(max_s A_s / 63), dmin = fp16(max_s B_s / 63)
    sc = clamp(round_half_away(A_s / d), 0, 63), m likewise from B_s / dmin
        (d and dmin are the decoded fp16 values; a zero divisor gives 0)
    q = clamp(round_half_away((w + dmin*m) / (d*sc)), 0, 15)   (0 if d*sc == 0)
"""

import numpy as np

F32 = np.float32

Q8_0_BLOCK = 32
Q8_0_BYTES = 34
Q4KS_BLOCK = 256
Q4KS_BYTES = 144


def round_half_away(v):
    """Round to the nearest integer, halves away from zero (C ``roundf``).

    ``v - trunc(v)`` is exact in binary floating point, so the comparison with
    0.5 decides the halfway cases exactly.
    """
    v = np.asarray(v)
    t = np.trunc(v)
    frac = v - t
    return t + np.where(np.abs(frac) >= 0.5, np.sign(v), 0).astype(v.dtype)


# --------------------------------------------------------------------------
# Q8_0
# --------------------------------------------------------------------------
def q8_0_quantize(w):
    """fp32 [rows, K] -> serialised Q8_0 bytes uint8 [rows, K/32*34]."""
    w = np.ascontiguousarray(w, dtype=F32)
    rows, K = w.shape
    if K % Q8_0_BLOCK:
        raise ValueError("Q8_0 needs K divisible by 32")
    nb = K // Q8_0_BLOCK
    b = w.reshape(rows, nb, Q8_0_BLOCK)
    amax = np.max(np.abs(b), axis=2)
    d = (amax / F32(127)).astype(F32)
    nz = d > 0
    safe = np.where(nz, d, F32(1))
    v = (b / safe[..., None]).astype(F32)
    q = np.clip(round_half_away(v), -127, 127)
    q = np.where(nz[..., None], q, 0).astype(np.int8)
    out = np.empty((rows, nb, Q8_0_BYTES), np.uint8)
    out[..., 0:2] = d.astype("<f2").view(np.uint8).reshape(rows, nb, 2)
    out[..., 2:] = q.view(np.uint8)
    return out.reshape(rows, nb * Q8_0_BYTES)


def q8_0_dequantize(blob, rows, K):
    """Serialised Q8_0 bytes -> fp32 [rows, K]."""
    nb = K // Q8_0_BLOCK
    a = np.asarray(blob, np.uint8).reshape(rows, nb, Q8_0_BYTES)
    d = np.ascontiguousarray(a[..., 0:2]).view("<f2").astype(F32)  # [rows, nb, 1]
    q = np.ascontiguousarray(a[..., 2:]).view(np.int8).astype(F32)
    return (d * q).astype(F32).reshape(rows, K)


# --------------------------------------------------------------------------
# Q4KS
# --------------------------------------------------------------------------
def pack_fields6(fields):
    """uint [..., 16] 6-bit fields -> uint8 [..., 12], little-endian bit stream."""
    f = np.asarray(fields).astype(np.uint64)
    words = np.zeros(f.shape[:-1] + (3,), np.uint64)
    for i in range(16):
        p = 6 * i
        wi, sh = divmod(p, 32)
        words[..., wi] |= (f[..., i] << np.uint64(sh)) & np.uint64(0xFFFFFFFF)
        if sh + 6 > 32:
            words[..., wi + 1] |= f[..., i] >> np.uint64(32 - sh)
    return words.astype("<u4").view(np.uint8).reshape(f.shape[:-1] + (12,))


def unpack_fields6(b12):
    """uint8 [..., 12] -> int64 [..., 16] 6-bit fields."""
    b = np.ascontiguousarray(np.asarray(b12, np.uint8))
    words = b.view("<u4").astype(np.uint64)  # [..., 3]
    out = np.empty(b.shape[:-1] + (16,), np.int64)
    for i in range(16):
        p = 6 * i
        wi, sh = divmod(p, 32)
        v = words[..., wi] >> np.uint64(sh)
        if sh + 6 > 32:
            v = v | (words[..., wi + 1] << np.uint64(32 - sh))
        out[..., i] = (v & np.uint64(63)).astype(np.int64)
    return out


def q4ks_quantize(w):
    """fp32 [rows, K] -> serialised Q4KS bytes uint8 [rows, K/256*144]."""
    w = np.ascontiguousarray(w, dtype=F32)
    rows, K = w.shape
    if K % Q4KS_BLOCK:
        raise ValueError("Q4KS needs K divisible by 256")
    ns = K // Q4KS_BLOCK
    sub = w.reshape(rows, ns, 8, 32)
    lo = np.minimum(F32(0), sub.min(axis=3))
    hi = sub.max(axis=3)
    A = ((hi - lo) / F32(15)).astype(F32)
    B = (F32(0) - lo).astype(F32)
    d16 = (A.max(axis=2) / F32(63)).astype(F32).astype("<f2")
    m16 = (B.max(axis=2) / F32(63)).astype(F32).astype("<f2")
    dF = d16.astype(F32)[..., None]
    mF = m16.astype(F32)[..., None]
    sc = np.where(dF > 0, round_half_away((A / np.where(dF > 0, dF, F32(1))).astype(F32)), 0)
    mm = np.where(mF > 0, round_half_away((B / np.where(mF > 0, mF, F32(1))).astype(F32)), 0)
    sc = np.clip(sc, 0, 63).astype(np.int64)
    mm = np.clip(mm, 0, 63).astype(np.int64)
    a = (dF * sc.astype(F32)).astype(F32)[..., None]
    bq = (mF * mm.astype(F32)).astype(F32)[..., None]
    num = (sub + bq).astype(F32)
    q = round_half_away((num / np.where(a > 0, a, F32(1))).astype(F32))
    q = np.where(a > 0, np.clip(q, 0, 15), 0).astype(np.uint8).reshape(rows, ns, 256)
    out = np.empty((rows, ns, Q4KS_BYTES), np.uint8)
    out[..., 0:2] = d16.view(np.uint8).reshape(rows, ns, 2)
    out[..., 2:4] = m16.view(np.uint8).reshape(rows, ns, 2)
    out[..., 4:16] = pack_fields6(np.concatenate([sc, mm], axis=2))
    out[..., 16:] = q[..., 0::2] | (q[..., 1::2] << 4)
    return out.reshape(rows, ns * Q4KS_BYTES)


def q4ks_dequantize(blob, rows, K):
    """Serialised Q4KS bytes -> fp32 [rows, K]."""
    ns = K // Q4KS_BLOCK
    a8 = np.asarray(blob, np.uint8).reshape(rows, ns, Q4KS_BYTES)
    d = np.ascontiguousarray(a8[..., 0:2]).view("<f2").astype(F32)      # [rows, ns, 1]
    dm = np.ascontiguousarray(a8[..., 2:4]).view("<f2").astype(F32)
    fld = unpack_fields6(a8[..., 4:16])                                  # [rows, ns, 16]
    sc = fld[..., 0:8].astype(F32)
    mm = fld[..., 8:16].astype(F32)
    qb = a8[..., 16:]
    q = np.empty((rows, ns, 256), F32)
    q[..., 0::2] = (qb & 0x0F).astype(F32)
    q[..., 1::2] = (qb >> 4).astype(F32)
    q = q.reshape(rows, ns, 8, 32)
    a = (d * sc)[..., None].astype(F32)
    b = (dm * mm)[..., None].astype(F32)
    return ((a * q).astype(F32) - b).astype(F32).reshape(rows, K)


# --------------------------------------------------------------------------
# format table
# --------------------------------------------------------------------------
FMT_F32, FMT_BF16, FMT_Q8_0, FMT_Q4KS = 0, 1, 2, 3


def quantize(fmt, w):
    if fmt == FMT_Q8_0:
        return q8_0_quantize(w)
    if fmt == FMT_Q4KS:
        return q4ks_quantize(w)
    if fmt == FMT_F32:
        return np.ascontiguousarray(w, F32).view(np.uint8).reshape(w.shape[0], -1)
    raise ValueError(f"unsupported format {fmt}")


def dequantize(fmt, blob, rows, K):
    if fmt == FMT_Q8_0:
        return q8_0_dequantize(blob, rows, K)
    if fmt == FMT_Q4KS:
        return q4ks_dequantize(blob, rows, K)
    if fmt == FMT_F32:
        return np.ascontiguousarray(blob).view(F32).reshape(rows, K)
    raise ValueError(f"unsupported format {fmt}")


def row_bytes(fmt, K):
    if fmt == FMT_Q8_0:
        return K // Q8_0_BLOCK * Q8_0_BYTES
    if fmt == FMT_Q4KS:
        return K // Q4KS_BLOCK * Q4KS_BYTES
    if fmt == FMT_F32:
        return 4 * K
    raise ValueError(f"unsupported format {fmt}")
