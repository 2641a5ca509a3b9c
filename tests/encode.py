"""Independent encoders for q6_K / q4_K super-blocks (test helper).

They build a raw block from chosen fields so that oracle pins can start from known
values instead of from the oracle's own decoder.  The field placement follows
the byte layouts the pages give (q6_K: ql@0, qh@128, scales@192, d@208; q4_K:
d@0, dmin@2, scales[12]@4, qs@16); the bit mapping inside ql/qh/qs and the
scales[12] packing are the same readings the oracle documents, written here as
the inverse operation (Python big-int packing rather than byte shifts).
"""
from __future__ import annotations

import numpy as np

QK_K = 256


def f16_bits(v: float) -> int:
    return int(np.array([v], np.float16).view(np.uint16)[0])


def encode_q6k(d_bits: int, sc, q) -> np.ndarray:
    """sc: 16 ints in [-128,127]; q: 256 ints in [-32,31]."""
    sc = [int(s) for s in sc]
    q = [int(v) for v in q]
    assert len(sc) == 16 and len(q) == QK_K
    out = np.zeros(210, np.uint8)
    for e, v in enumerate(q):
        u = v + 32
        assert 0 <= u < 64
        lo, hi = u % 16, u // 16
        out[e // 2] |= lo << (4 * (e % 2))
        out[128 + e // 4] |= hi << (2 * (e % 4))
    for i, s in enumerate(sc):
        out[192 + i] = s & 0xFF
    out[208] = d_bits & 0xFF
    out[209] = d_bits >> 8
    return out


def encode_q4k(d_bits: int, dmin_bits: int, sc, m, q) -> np.ndarray:
    """sc, m: 8 ints in [0,63]; q: 256 ints in [0,15]."""
    fields = [int(s) for s in sc] + [int(v) for v in m]
    assert len(fields) == 16 and all(0 <= f < 64 for f in fields)
    packed = 0
    for i, f in enumerate(fields):
        packed += f << (6 * i)
    out = np.zeros(144, np.uint8)
    out[0], out[1] = d_bits & 0xFF, d_bits >> 8
    out[2], out[3] = dmin_bits & 0xFF, dmin_bits >> 8
    out[4:16] = np.frombuffer(packed.to_bytes(12, "little"), np.uint8)
    for e, v in enumerate(q):
        v = int(v)
        assert 0 <= v < 16
        out[16 + e // 2] |= v << (4 * (e % 2))
    return out


def random_q6k_fields(rng: np.random.Generator, sc_range=(-32, 31)):
    d = float(np.float16(abs(rng.standard_normal()) * 1e-3))
    sc = rng.integers(sc_range[0], sc_range[1] + 1, 16)
    q = rng.integers(-32, 32, QK_K)
    return d, sc, q


def random_q4k_fields(rng: np.random.Generator):
    d = float(np.float16(abs(rng.standard_normal()) * 1e-3))
    dmin = float(np.float16(abs(rng.standard_normal()) * 1e-3))
    sc = rng.integers(0, 64, 8)
    m = rng.integers(0, 64, 8)
    q = rng.integers(0, 16, QK_K)
    return d, dmin, sc, m, q


def q6k_matrix(rng, od, id_, sc_range=(-32, 31)):
    """Random q6_K rows built from known fields: returns (raw [od,nsb,210], W f64 [od,id])."""
    nsb = id_ // QK_K
    raw = np.zeros((od, nsb, 210), np.uint8)
    W = np.zeros((od, id_), np.float64)
    for j in range(od):
        for b in range(nsb):
            d, sc, q = random_q6k_fields(rng, sc_range)
            raw[j, b] = encode_q6k(f16_bits(d), sc, q)
            for e in range(QK_K):
                W[j, b * QK_K + e] = d * float(sc[e // 16]) * float(q[e])
    return raw, W


def q4k_matrix(rng, od, id_):
    nsb = id_ // QK_K
    raw = np.zeros((od, nsb, 144), np.uint8)
    W = np.zeros((od, id_), np.float64)
    for j in range(od):
        for b in range(nsb):
            d, dmin, sc, m, q = random_q4k_fields(rng)
            raw[j, b] = encode_q4k(f16_bits(d), f16_bits(dmin), sc, m, q)
            for e in range(QK_K):
                c = e // 32
                W[j, b * QK_K + e] = d * float(sc[c]) * float(q[e]) - dmin * float(m[c])
    return raw, W


# --------------------------------------------------------------------------- ggml layout
# Encoders for the public ggml (llama.cpp) block layouts, written from the format's
# description of where each value lives (the inverse of the oracle's conversion, so the
# two are independent statements of the same mapping):
#   q4_K: the 256 values in four groups of 64; in group j, value l < 32 is the low
#         nibble of qs[32j + l] and value 32 + l its high nibble; scale/min of sub-block
#         s (32 values): s < 4 in the low 6 bits of S[s] / S[s + 4]; s >= 4 split into a
#         low nibble (S[s + 4], sc in bits 0-3, m in bits 4-7) and the top two bits of
#         S[s - 4] (sc) / S[s] (m).
#   q6_K: two halves of 128; in half n, quarter p (32 values), value l: low 4 bits in
#         nibble p // 2 of ql[64n + 32(p % 2) + l], high 2 bits at bit 2p of qh[32n + l];
#         scales[16] and d as in the reading.
def encode_q4k_ggml(d_bits: int, dmin_bits: int, sc, m, q) -> np.ndarray:
    sc = [int(v) for v in sc]
    m = [int(v) for v in m]
    out = np.zeros(144, np.uint8)
    out[0], out[1] = d_bits & 0xFF, d_bits >> 8
    out[2], out[3] = dmin_bits & 0xFF, dmin_bits >> 8
    S = [0] * 12
    for s in range(4):
        S[s] = sc[s] | ((sc[s + 4] >> 4) << 6)
        S[s + 4] = m[s] | ((m[s + 4] >> 4) << 6)
        S[s + 8] = (sc[s + 4] & 15) | ((m[s + 4] & 15) << 4)
    out[4:16] = S
    for group in range(4):
        for l in range(32):
            lo = int(q[64 * group + l])
            hi = int(q[64 * group + 32 + l])
            out[16 + 32 * group + l] = lo | (hi << 4)
    return out


def encode_q6k_ggml(d_bits: int, sc, q) -> np.ndarray:
    out = np.zeros(210, np.uint8)
    for n in range(2):
        for p in range(4):
            for l in range(32):
                u = int(q[128 * n + 32 * p + l]) + 32
                assert 0 <= u < 64
                out[64 * n + 32 * (p % 2) + l] |= (u & 15) << (4 * (p // 2))
                out[128 + 32 * n + l] |= (u >> 4) << (2 * p)
    for i, s in enumerate(sc):
        out[192 + i] = int(s) & 0xFF
    out[208] = d_bits & 0xFF
    out[209] = d_bits >> 8
    return out
