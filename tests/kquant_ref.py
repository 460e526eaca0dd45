"""Test-side k-quant encoder and a second, independently written decoder.

The encoder builds super-blocks from their fields (d, dmin, s_j, m_j, q_i) with
Python integers, so that a hand-constructed block has a value that follows from
its fields alone. The decoder reads the packed bytes with 64-bit shifts and
index arithmetic, a different route from the oracle's bit-stream unpacking; the
brute-force checks use it so that they share no dequantisation code with the
oracle.
"""

from __future__ import annotations

import numpy as np


def encode_header(d: float, dmin: float, s, m) -> bytes:
    acc = 0
    for j in range(8):
        assert 0 <= s[j] < 64 and 0 <= m[j] < 64
        acc |= int(s[j]) << (6 * j)
        acc |= int(m[j]) << (48 + 6 * j)
    return (np.float16(d).tobytes() + np.float16(dmin).tobytes()
            + acc.to_bytes(12, "little"))


def encode_q4k(d, dmin, s, m, q) -> np.ndarray:
    assert len(q) == 256 and all(0 <= v < 16 for v in q)
    qs = bytes(int(q[2 * b]) | (int(q[2 * b + 1]) << 4) for b in range(128))
    return np.frombuffer(encode_header(d, dmin, s, m) + qs, dtype=np.uint8).copy()


def encode_q5k(d, dmin, s, m, q) -> np.ndarray:
    assert len(q) == 256 and all(0 <= v < 32 for v in q)
    hi = 0
    for i in range(256):
        hi |= (int(q[i]) >> 4) << i
    low = [int(v) & 15 for v in q]
    qs = bytes(low[2 * b] | (low[2 * b + 1] << 4) for b in range(128))
    return np.frombuffer(encode_header(d, dmin, s, m) + hi.to_bytes(32, "little") + qs,
                         dtype=np.uint8).copy()


def expected_weights(d, dmin, s, m, q) -> np.ndarray:
    """w_i = d * s_j * q_i - dmin * m_j, j = i // 32, from the fields."""
    d64 = float(np.float16(d))
    m64 = float(np.float16(dmin))
    return np.array([d64 * s[i // 32] * q[i] - m64 * m[i // 32] for i in range(256)])


def _le_u64(b: np.ndarray) -> np.ndarray:
    out = np.zeros(b.shape[:-1], dtype=np.uint64)
    for n in range(b.shape[-1]):
        out |= b[..., n].astype(np.uint64) << np.uint64(8 * n)
    return out


def decode(blocks: np.ndarray) -> np.ndarray:
    """[..., 144 or 176] uint8 -> [..., 256] float64 (second implementation)."""
    nb = blocks.shape[-1]
    d = blocks[..., 0:2].copy().view(np.float16)[..., 0].astype(np.float64)
    dmin = blocks[..., 2:4].copy().view(np.float16)[..., 0].astype(np.float64)
    lo = _le_u64(blocks[..., 4:12])          # field bits 0..63
    hi = _le_u64(blocks[..., 12:16])         # field bits 64..95
    fields = []
    for f in range(16):
        p = 6 * f
        if p + 6 <= 64:
            v = (lo >> np.uint64(p)) & np.uint64(63)
        elif p >= 64:
            v = (hi >> np.uint64(p - 64)) & np.uint64(63)
        else:
            v = ((lo >> np.uint64(p)) | (hi << np.uint64(64 - p))) & np.uint64(63)
        fields.append(v.astype(np.float64))
    i = np.arange(256)
    if nb == 144:
        qs = blocks[..., 16:144]
        qh = None
    else:
        qs = blocks[..., 48:176]
        qh = blocks[..., 16:48]
    q = (qs[..., i // 2].astype(np.int64) >> (4 * (i % 2))) & 15
    if qh is not None:
        q = q + 16 * ((qh[..., i // 8].astype(np.int64) >> (i % 8)) & 1)
    s = np.stack(fields[0:8], axis=-1)[..., i // 32]
    m = np.stack(fields[8:16], axis=-1)[..., i // 32]
    return d[..., None] * s * q - dmin[..., None] * m


def encode_q6k(d, s, q) -> np.ndarray:
    """Q6_K super-block (210 B) from d, sixteen signed scales and 256 quants
    in 0..63, packed with Python integers."""
    assert len(s) == 16 and all(-128 <= v < 128 for v in s)
    assert len(q) == 256 and all(0 <= v < 64 for v in q)
    scales = bytes(int(v) & 0xFF for v in s)
    high = 0
    for i in range(256):
        high |= (int(q[i]) >> 4) << (2 * i)
    low = bytes((int(q[2 * b]) & 15) | ((int(q[2 * b + 1]) & 15) << 4) for b in range(128))
    raw = np.float16(d).tobytes() + scales + high.to_bytes(64, "little") + low
    return np.frombuffer(raw, dtype=np.uint8).copy()


def expected_weights_q6k(d, s, q) -> np.ndarray:
    """w_i = d * s_{i // 16} * (q_i - 32), from the fields."""
    d64 = float(np.float16(d))
    return np.array([d64 * s[i // 16] * (q[i] - 32) for i in range(256)])


def decode_q6k(blocks: np.ndarray) -> np.ndarray:
    """[..., 210] uint8 -> [..., 256] float64 (second implementation: the
    high parts read as eight little-endian 64-bit words)."""
    d = blocks[..., 0:2].copy().view(np.float16)[..., 0].astype(np.float64)
    sc = blocks[..., 2:18].astype(np.int64)
    sc = np.where(sc >= 128, sc - 256, sc)
    words = [_le_u64(blocks[..., 18 + 8 * w:26 + 8 * w]) for w in range(8)]
    i = np.arange(256)
    high = np.stack([(words[n // 32] >> np.uint64(2 * (n % 32))) & np.uint64(3) for n in range(256)],
                    axis=-1).astype(np.int64)
    low = (blocks[..., 82 + i // 2].astype(np.int64) >> (4 * (i % 2))) & 15
    q = low + 16 * high
    return d[..., None] * sc[..., i // 16] * (q - 32)


def encode_mxfp4(e, codes) -> np.ndarray:
    """MXFP4 super-block (136 B) from eight E8M0 exponents and 256 4-bit codes."""
    assert len(e) == 8 and all(0 <= v < 256 for v in e)
    assert len(codes) == 256 and all(0 <= c < 16 for c in codes)
    nib = bytes(int(codes[2 * b]) | (int(codes[2 * b + 1]) << 4) for b in range(128))
    return np.frombuffer(bytes(int(v) for v in e) + nib, dtype=np.uint8).copy()


def e2m1_value(code: int) -> float:
    """FP4 E2M1 from its definition: sign, exponent (2 bits, bias 1), mantissa
    (1 bit); exponent 0 is subnormal (0.m * 2^0)."""
    sign = -1.0 if code & 8 else 1.0
    ex, man = (code >> 1) & 3, code & 1
    mag = man * 0.5 if ex == 0 else (1.0 + 0.5 * man) * 2.0 ** (ex - 1)
    return sign * mag


def decode_mxfp4(blocks: np.ndarray) -> np.ndarray:
    """[..., 136] uint8 -> [..., 256] float64 (second implementation, from the
    bit-level definition of E2M1 and E8M0)."""
    out = np.empty(blocks.shape[:-1] + (256,))
    flat_b = blocks.reshape(-1, 136)
    flat_o = out.reshape(-1, 256)
    for r in range(flat_b.shape[0]):
        for i in range(256):
            e = int(flat_b[r, i // 32])
            code = (int(flat_b[r, 8 + i // 2]) >> (4 * (i % 2))) & 15
            flat_o[r, i] = float("nan") if e == 255 else e2m1_value(code) * 2.0 ** (e - 127)
    return out


def dense(W: np.ndarray) -> np.ndarray:
    """[..., rows, nblk, bytes] -> [..., rows, nblk*256] via this module's
    decoders (``decode`` for Q4_K/Q5_K, ``decode_q6k``, ``decode_mxfp4``)."""
    nb = W.shape[-1]
    v = decode_q6k(W) if nb == 210 else (decode_mxfp4(W) if nb == 136 else decode(W))
    return v.reshape(*W.shape[:-2], W.shape[-2] * 256)
