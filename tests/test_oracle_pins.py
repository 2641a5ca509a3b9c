"""Pins of the CPU oracle against things other than itself (no GPU).

Each test fixes the oracle to a source outside its own code: hand-worked golden
blocks, a library routine (numpy's binary16 conversion, numpy's f64 matmul),
exact rational arithmetic, closed forms and invariants.  The choice covers the
plausible mistakes: a wrong bit or field position, a wrong scale index (16 vs
32), a dropped or sign-flipped min term, a transposed operand, a wrong rounding
rule, an f16 subnormal slip.
"""
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
from tests.encode import (encode_q4k, encode_q4k_ggml, encode_q6k, encode_q6k_ggml, f16_bits, q4k_matrix, q6k_matrix,
                          random_q4k_fields, random_q6k_fields)

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _lines(name):
    with open(os.path.join(GOLDEN, name)) as f:
        for ln in f:
            ln = ln.strip()
            if ln and not ln.startswith("#"):
                yield ln.split()


# --------------------------------------------------------------------------- f16
def test_f16_to_f32_matches_numpy_on_all_patterns(oracle_lib):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = oracle.f16_to_f32(bits)
    ref = bits.view(np.float16).astype(np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan].view(np.uint32), ref[~nan].view(np.uint32))


# --------------------------------------------------------------------------- quantize
def _golden_chunks():
    chunks, cur = [], None
    for tok in _lines("quantize_chunks.txt"):
        key, vals = tok[0], tok[1:]
        if key == "chunk":
            cur = {"x": [float(v) for v in vals]}
            chunks.append(cur)
        elif key == "d":
            cur["d"] = None if vals[0] == "any" else float(vals[0])
        elif key == "q":
            cur["q"] = [int(v) for v in vals]
        elif key == "ssum":
            cur["ssum"] = int(vals[0])
    return chunks


def test_quantize_golden_chunks(oracle_lib):
    chunks = _golden_chunks()
    assert len(chunks) == 4
    x = np.zeros((1, 32 * len(chunks)), np.float32)
    for c, ch in enumerate(chunks):
        x[0, 32 * c: 32 * c + len(ch["x"])] = ch["x"]
    q, d, s = oracle.quantize_act(x)
    for c, ch in enumerate(chunks):
        want = np.zeros(32, np.int64)
        want[: len(ch["q"])] = ch["q"]
        assert np.array_equal(q[0, 32 * c: 32 * c + 32], want), c
        assert s[0, c] == ch["ssum"], c
        if ch["d"] is not None:
            assert d[0, c] == ch["d"], c
    # chunk D: d is the f32 nearest 0.75/127 -> within half an ulp of the real quotient
    dD = Fraction(float(d[0, 3]))
    exact = Fraction(3, 4) / 127
    ulp = Fraction(np.spacing(np.float32(d[0, 3])).item())
    assert abs(dD - exact) <= ulp / 2


@pytest.mark.parametrize("scale", [1.0, 1e-3, 3e4, 1e-30, 2.0 ** -120])
def test_quantize_invariants(oracle_lib, scale):
    rng = np.random.default_rng(11)
    x = (rng.standard_normal((37, 256)) * scale).astype(np.float32)
    x[3, 32:64] = 0.0                                   # all-zero chunk
    x[4, 64:96] = 0.0
    x[4, 70] = np.float32(-5.0 * scale)                 # single non-zero chunk
    q, d, s = oracle.quantize_act(x)
    xc = x.reshape(37, 8, 32).astype(np.float64)
    qc = q.reshape(37, 8, 32).astype(np.int64)
    dc = d.astype(np.float64)[..., None]
    assert np.abs(qc).max() <= 127
    assert np.array_equal(s, qc.sum(-1))
    assert np.all(qc[3, 1] == 0) and d[3, 1] == 0 and s[3, 1] == 0
    assert qc[4, 2, 6] == -127 and np.count_nonzero(qc[4, 2]) == 1
    nz = d > 0
    # the element at |x| = amax maps to +-127 (d normal)
    amax_idx = np.abs(xc).argmax(-1)
    qa = np.take_along_axis(qc, amax_idx[..., None], -1)[..., 0]
    normal = d >= np.finfo(np.float32).tiny * 128
    assert np.all(np.abs(qa[normal]) == 127)
    # reconstruction error at most half a step (plus f32 rounding of the quotient)
    err = np.abs(xc - dc * qc)
    bound = dc * (0.5 + 2.0 ** -17) + np.abs(xc) * 2.0 ** -22
    assert np.all(err[nz & normal] <= bound[nz & normal])
    # sign preserved (or zero)
    assert np.all((np.sign(qc) == np.sign(xc)) | (qc == 0))


def test_quantize_power_of_two_scaling(oracle_lib):
    # multiplying x by 2^k scales d by 2^k exactly and leaves the codes unchanged
    x = np.random.default_rng(5).standard_normal((9, 128)).astype(np.float32)
    q0, d0, s0 = oracle.quantize_act(x)
    for k in (-20, -3, 5, 40):
        q1, d1, s1 = oracle.quantize_act(np.ldexp(x, k).astype(np.float32))
        assert np.array_equal(q0, q1) and np.array_equal(s0, s1)
        assert np.array_equal(np.ldexp(d0, k).astype(np.float32), d1)


def test_quantize_ties_away_from_zero(oracle_lib):
    # amax = 127 -> d = 1; every k + 0.5 must round away from zero
    halves = np.array([0.5, 1.5, 2.5, 3.5, 125.5, 126.5], np.float32)
    x = np.zeros((1, 32), np.float32)
    x[0, 0] = 127
    x[0, 1:7] = halves
    x[0, 7:13] = -halves
    q, _, _ = oracle.quantize_act(x)
    assert list(q[0, 1:7]) == [1, 2, 3, 4, 126, 127]
    assert list(q[0, 7:13]) == [-1, -2, -3, -4, -126, -127]


# --------------------------------------------------------------------------- decode
def test_q6k_golden_block(oracle_lib):
    spec = {}
    codes, dscs = [], []
    for tok in _lines("q6k_block.txt"):
        if tok[0] == "code":
            codes.append((int(tok[1]), int(tok[2]), float(tok[3])))
        elif tok[0] == "dsc":
            dscs.append((int(tok[1]), int(tok[2]), float(tok[3])))
        else:
            spec[tok[0]] = tok[1:]
    blk = np.zeros(210, np.uint8)
    blk[0:128] = int(spec["fill_ql"][0], 16)
    blk[128:192] = int(spec["fill_qh"][0], 16)
    blk[192:208] = np.array([int(v) for v in spec["scales"]], np.int8).view(np.uint8)
    dbits = int(spec["d_bits"][0], 16)
    blk[208], blk[209] = dbits & 0xFF, dbits >> 8
    d, sc, q = oracle.decode_q6k(blk)
    assert d == 1.0
    W = oracle.dequant_q6k(blk.reshape(1, 1, 210))
    for e, code, w in codes:
        assert q[e] == code, e
        assert W[0, e] == w, e
    dsc = oracle.scale_planes_q6k(blk.reshape(1, 1, 210))
    for c, h, v in dscs:
        assert dsc[0, c, h] == v


def test_q4k_golden_block(oracle_lib):
    spec = {}
    codes, dscs = [], []
    for tok in _lines("q4k_block.txt"):
        if tok[0] == "code":
            codes.append((int(tok[1]), int(tok[2]), float(tok[3])))
        elif tok[0] == "dsc":
            dscs.append((int(tok[1]), float(tok[2]), float(tok[3])))
        else:
            spec[tok[0]] = tok[1:]
    blk = np.zeros(144, np.uint8)
    db, mb = int(spec["d_bits"][0], 16), int(spec["dmin_bits"][0], 16)
    blk[0], blk[1], blk[2], blk[3] = db & 0xFF, db >> 8, mb & 0xFF, mb >> 8
    blk[4:16] = [int(v, 16) for v in spec["scales_bytes"]]
    blk[16:144] = int(spec["fill_qs"][0], 16)
    d, dmin, sc, m, q = oracle.decode_q4k(blk)
    assert (d, dmin) == (1.0, 0.5)
    assert list(sc) == [int(v) for v in spec["sc"]]
    assert list(m) == [int(v) for v in spec["m"]]
    W = oracle.dequant_q4k(blk.reshape(1, 1, 144))
    for e, code, w in codes:
        assert q[e] == code, e
        assert W[0, e] == w, e
    dsc, dmn = oracle.scale_planes_q4k(blk.reshape(1, 1, 144))
    for c, a, b in dscs:
        assert dsc[0, c] == a and dmn[0, c] == b


def test_decode_roundtrip_against_independent_encoder(oracle_lib):
    rng = np.random.default_rng(3)
    for _ in range(40):
        d, sc, q = random_q6k_fields(rng, (-128, 127))
        blk = encode_q6k(f16_bits(d), sc, q)
        d2, sc2, q2 = oracle.decode_q6k(blk)
        assert d2 == np.float32(np.float16(d)) and np.array_equal(sc2, sc) and np.array_equal(q2, q)
        d, dmin, sc, m, q = random_q4k_fields(rng)
        blk = encode_q4k(f16_bits(d), f16_bits(dmin), sc, m, q)
        d2, dm2, sc2, m2, q2 = oracle.decode_q4k(blk)
        assert (d2, dm2) == (np.float32(np.float16(d)), np.float32(np.float16(dmin)))
        assert np.array_equal(sc2, sc) and np.array_equal(m2, m) and np.array_equal(q2, q)


def test_f16_subnormal_scales_decode(oracle_lib):
    # d in the binary16 subnormal range must decode exactly (man * 2^-24)
    for bits in (0x0001, 0x03FF, 0x8001, 0x0200):
        blk = encode_q6k(bits, [1] * 16, [1] * 256)
        d, _, _ = oracle.decode_q6k(blk)
        man = bits & 0x3FF
        want = (-1.0 if bits & 0x8000 else 1.0) * man * 2.0 ** -24
        assert d == want


# --------------------------------------------------------------------------- planes
@pytest.mark.parametrize("kind", ["q6_K", "q4_K"])
def test_scale_planes_are_exact_products(oracle_lib, kind):
    """Closed form: d (11 significant bits) * a scale of <= 8 bits has <= 19 bits,
    so the f32 product is the exact real product (no rounding)."""
    rng = np.random.default_rng(8)
    if kind == "q6_K":
        raw, _ = q6k_matrix(rng, 6, 512, (-128, 127))
        dsc = oracle.scale_planes_q6k(raw)
        for j in range(6):
            for b in range(2):
                d, sc, _ = oracle.decode_q6k(raw[j, b])
                for cc in range(8):
                    for h in range(2):
                        exact = Fraction(d) * sc[2 * cc + h]
                        assert Fraction(float(dsc[j, 8 * b + cc, h])) == exact
    else:
        raw, _ = q4k_matrix(rng, 6, 512)
        dsc, dmn = oracle.scale_planes_q4k(raw)
        for j in range(6):
            for b in range(2):
                d, dmin, sc, m, _ = oracle.decode_q4k(raw[j, b])
                for cc in range(8):
                    assert Fraction(float(dsc[j, 8 * b + cc])) == Fraction(d) * int(sc[cc])
                    assert Fraction(float(dmn[j, 8 * b + cc])) == Fraction(dmin) * int(m[cc])


# --------------------------------------------------------------------------- dots
def test_dots_brute_force_from_known_fields(oracle_lib):
    """Plain loops over the fields the encoder was given (not the oracle's decode)."""
    rng = np.random.default_rng(21)
    od, id_, M = 3, 512, 2
    qa = rng.integers(-127, 128, (M, id_)).astype(np.int8)
    raw6 = np.zeros((od, 2, 210), np.uint8)
    raw4 = np.zeros((od, 2, 144), np.uint8)
    codes6 = np.zeros((od, id_), np.int64)
    codes4 = np.zeros((od, id_), np.int64)
    for j in range(od):
        for b in range(2):
            d, sc, q = random_q6k_fields(rng)
            raw6[j, b] = encode_q6k(f16_bits(d), sc, q)
            codes6[j, 256 * b: 256 * b + 256] = q
            d, dmin, sc, m, q = random_q4k_fields(rng)
            raw4[j, b] = encode_q4k(f16_bits(d), f16_bits(dmin), sc, m, q)
            codes4[j, 256 * b: 256 * b + 256] = q
    D6 = oracle.dots_q6k(raw6, qa)
    D4 = oracle.dots_q4k(raw4, qa)
    for t in range(M):
        for j in range(od):
            for s in range(id_ // 16):
                acc = 0
                for e in range(16 * s, 16 * s + 16):
                    acc += int(codes6[j, e]) * int(qa[t, e])
                assert D6[t, j, s] == acc
            for c in range(id_ // 32):
                acc = 0
                for e in range(32 * c, 32 * c + 32):
                    acc += int(codes4[j, e]) * int(qa[t, e])
                assert D4[t, j, c] == acc


# --------------------------------------------------------------------------- Y
def _act(rng, M, K):
    x = rng.standard_normal((M, K)).astype(np.float32)
    return oracle.quantize_act(x)


@pytest.mark.parametrize("kind", ["q6_K", "q4_K"])
def test_gemm_equals_dense_f64_matmul(oracle_lib, kind):
    """Y == (d_a*q_a) @ W^T with W built from the encoder's fields (numpy f64 matmul)."""
    rng = np.random.default_rng(31 if kind == "q6_K" else 32)
    od, id_, M = 24, 768, 9
    raw, W = (q6k_matrix(rng, od, id_, (-128, 127)) if kind == "q6_K" else q4k_matrix(rng, od, id_))
    q, d, s = _act(rng, M, id_)
    A = (np.repeat(d.astype(np.float64), 32, axis=1) * q.astype(np.float64))
    ref = A @ W.T
    fn = oracle.gemm_q6k if kind == "q6_K" else oracle.gemm_q4k
    Y, S = fn(raw, q, d, s, with_abs=True)
    assert np.all(S >= np.abs(Y))
    assert np.max(np.abs(Y - ref)) <= 1e-12 * np.max(np.abs(ref))
    # the oracle's own dequantized weights agree exactly with the encoder's
    Wo = oracle.dequant_q6k(raw) if kind == "q6_K" else oracle.dequant_q4k(raw)
    assert np.array_equal(Wo, W)


@pytest.mark.parametrize("kind", ["q6_K", "q4_K"])
def test_gemm_exact_rational_tiny(oracle_lib, kind):
    rng = np.random.default_rng(41 if kind == "q6_K" else 42)
    for od, id_, M in ((1, 256, 1), (3, 512, 2), (4, 256, 3)):
        raw, _ = (q6k_matrix(rng, od, id_, (-128, 127)) if kind == "q6_K" else q4k_matrix(rng, od, id_))
        q, d, s = _act(rng, M, id_)
        fn = oracle.gemm_q6k if kind == "q6_K" else oracle.gemm_q4k
        Y, S = fn(raw, q, d, s, with_abs=True)
        for j in range(od):
            # exact weights from the encoded blocks, as rationals
            Wj = []
            for b in range(id_ // 256):
                if kind == "q6_K":
                    dd, sc, qq = oracle.decode_q6k(raw[j, b])
                    Wj += [Fraction(dd) * int(sc[e // 16]) * int(qq[e]) for e in range(256)]
                else:
                    dd, dm, sc, m, qq = oracle.decode_q4k(raw[j, b])
                    Wj += [Fraction(dd) * int(sc[e // 32]) * int(qq[e]) - Fraction(dm) * int(m[e // 32])
                           for e in range(256)]
            for t in range(M):
                exact = sum(Fraction(float(d[t, e // 32])) * int(q[t, e]) * Wj[e] for e in range(id_))
                assert abs(Fraction(Y[t, j]) - exact) <= Fraction(1e-14) * Fraction(S[t, j]) + Fraction(1e-300)


@pytest.mark.parametrize("kind", ["q6_K", "q4_K"])
def test_gemm_one_hot_activation(oracle_lib, kind):
    """A single non-zero activation x_e = v gives d_a = |v|/127, q = +-127 and
    Y[j] = d_a * (+-127) * w[j, e] (up to one f64 rounding)."""
    rng = np.random.default_rng(51)
    od, id_ = 5, 512
    raw, W = (q6k_matrix(rng, od, id_) if kind == "q6_K" else q4k_matrix(rng, od, id_))
    x = np.zeros((1, id_), np.float32)
    e = 299
    x[0, e] = -2.75
    q, d, s = oracle.quantize_act(x)
    assert q[0, e] == -127 and s[0, e // 32] == -127
    fn = oracle.gemm_q6k if kind == "q6_K" else oracle.gemm_q4k
    Y = fn(raw, q, d, s)
    want = float(d[0, e // 32]) * -127.0 * W[:, e]
    np.testing.assert_allclose(Y[0], want, rtol=1e-15, atol=0)


def test_gemm_zero_scales_and_zero_dmin(oracle_lib):
    rng = np.random.default_rng(61)
    q, d, s = _act(rng, 4, 256)
    # q6_K with every scale 0 -> Y = 0
    blk = encode_q6k(f16_bits(0.5), [0] * 16, rng.integers(-32, 32, 256))
    assert np.all(oracle.gemm_q6k(blk.reshape(1, 1, 210), q, d, s) == 0)
    # q4_K with dmin = 0 reduces to sum_c d_a * d*sc_c * I_c (integer dots from the brute force)
    sc = rng.integers(0, 64, 8)
    codes = rng.integers(0, 16, 256)
    blk4 = encode_q4k(f16_bits(0.25), f16_bits(0.0), sc, rng.integers(0, 64, 8), codes)
    Y = oracle.gemm_q4k(blk4.reshape(1, 1, 144), q, d, s)
    for t in range(4):
        want = 0.0
        for c in range(8):
            I = int(np.dot(codes[32 * c: 32 * c + 32].astype(np.int64), q[t, 32 * c: 32 * c + 32].astype(np.int64)))
            want += float(d[t, c]) * 0.25 * int(sc[c]) * I
        assert abs(Y[t, 0] - want) <= 1e-13 * max(1.0, abs(want))
    # q4_K with every sc = 0: only the min term remains, -sum_c d_a*dmin*m_c*ssum_c
    m = rng.integers(0, 64, 8)
    blk0 = encode_q4k(f16_bits(0.25), f16_bits(0.125), [0] * 8, m, codes)
    Y0 = oracle.gemm_q4k(blk0.reshape(1, 1, 144), q, d, s)
    for t in range(4):
        want = -sum(float(d[t, c]) * 0.125 * int(m[c]) * int(s[t, c]) for c in range(8))
        assert abs(Y0[t, 0] - want) <= 1e-13 * max(1.0, abs(want))


@pytest.mark.parametrize("kind", ["q6_K", "q4_K"])
def test_gemm_token_permutation_and_threads(oracle_lib, kind):
    rng = np.random.default_rng(71)
    od, id_, M = 17, 512, 7
    raw, _ = (q6k_matrix(rng, od, id_) if kind == "q6_K" else q4k_matrix(rng, od, id_))
    q, d, s = _act(rng, M, id_)
    fn = oracle.gemm_q6k if kind == "q6_K" else oracle.gemm_q4k
    Y = fn(raw, q, d, s)
    perm = rng.permutation(M)
    Yp = fn(raw, q[perm], d[perm], s[perm])
    assert np.array_equal(Yp, Y[perm])
    Yt = fn(raw, q, d, s, nthreads=4)
    assert np.array_equal(Yt, Y)


def test_whole_matrix_codes_match_encoder(oracle_lib):
    rng = np.random.default_rng(81)
    od, id_ = 5, 512
    raw6 = np.zeros((od, 2, 210), np.uint8)
    raw4 = np.zeros((od, 2, 144), np.uint8)
    want6 = np.zeros((od, id_), np.int64)
    want4 = np.zeros((od, id_), np.int64)
    for j in range(od):
        for b in range(2):
            d, sc, q = random_q6k_fields(rng)
            raw6[j, b] = encode_q6k(f16_bits(d), sc, q)
            want6[j, 256 * b: 256 * b + 256] = q
            d, dmin, sc, m, q = random_q4k_fields(rng)
            raw4[j, b] = encode_q4k(f16_bits(d), f16_bits(dmin), sc, m, q)
            want4[j, 256 * b: 256 * b + 256] = q
    assert np.array_equal(oracle.codes_q6k(raw6), want6)
    assert np.array_equal(oracle.codes_q4k(raw4), want4)


def test_block_fields_match_encoder(oracle_lib):
    rng = np.random.default_rng(91)
    raw6 = np.zeros((3, 2, 210), np.uint8)
    raw4 = np.zeros((3, 2, 144), np.uint8)
    want6, want4 = [], []
    for j in range(3):
        for b in range(2):
            d, sc, q = random_q6k_fields(rng, (-128, 127))
            raw6[j, b] = encode_q6k(f16_bits(d), sc, q)
            want6.append((np.float32(np.float16(d)), sc))
            d, dmin, sc, m, q = random_q4k_fields(rng)
            raw4[j, b] = encode_q4k(f16_bits(d), f16_bits(dmin), sc, m, q)
            want4.append((np.float32(np.float16(d)), np.float32(np.float16(dmin)), sc, m))
    d6, sc6 = oracle.fields_q6k(raw6)
    d4, dm4, sc4, m4 = oracle.fields_q4k(raw4)
    for i, (d, sc) in enumerate(want6):
        assert d6.reshape(-1)[i] == d and np.array_equal(sc6.reshape(-1, 16)[i], sc)
    for i, (d, dmin, sc, m) in enumerate(want4):
        assert d4.reshape(-1)[i] == d and dm4.reshape(-1)[i] == dmin
        assert np.array_equal(sc4.reshape(-1, 8)[i], sc) and np.array_equal(m4.reshape(-1, 8)[i], m)


# --------------------------------------------------------------------------- ggml interop
def test_ggml_q4k_hand_worked_block(oracle_lib):
    """Bytes placed by hand in the ggml q4_K layout; the decoded values are worked out
    from the layout's description (value 64j + l < 32: low nibble of qs[32j + l];
    64j + 32 + l: its high nibble; sub-block 4: sc from S[8] low nibble and S[0] top
    bits, m from S[8] high nibble and S[4] top bits)."""
    g = np.zeros(144, np.uint8)
    g[0:4] = [0x00, 0x3C, 0x00, 0x38]             # d = 1.0, dmin = 0.5
    g[4 + 0] = 0xC5                               # sc_0 = 5, top bits 3 -> sc_4 += 48
    g[4 + 4] = 0x87                               # m_0 = 7, top bits 2 -> m_4 += 32
    g[4 + 8] = 0x9A                               # sc_4 low 10, m_4 low 9
    g[16 + 0], g[16 + 31], g[16 + 32] = 0x21, 0x43, 0x65
    r = oracle.ggml_to_reading("q4_K", g)
    d, dmin, sc, m, q = oracle.decode_q4k(r)
    assert (d, dmin) == (1.0, 0.5)
    assert (sc[0], m[0], sc[4], m[4]) == (5, 7, 58, 41)
    assert sc[1] == sc[2] == sc[3] == sc[5] == 0 and m[1] == m[5] == 0
    assert (q[0], q[32], q[31], q[63], q[64], q[96]) == (1, 2, 3, 4, 5, 6)
    assert q[1] == q[33] == q[65] == q[255] == 0


def test_ggml_q6k_hand_worked_block(oracle_lib):
    """Value 128n + 32p + l: low 4 bits = nibble p // 2 of ql[64n + 32(p % 2) + l],
    high 2 bits = bits 2p of qh[32n + l], code = that 6-bit value - 32."""
    g = np.zeros(210, np.uint8)
    g[0], g[32], g[64] = 0x21, 0x43, 0x0F
    g[128 + 0], g[128 + 32] = 0xE4, 0x01
    g[192:208] = np.arange(16, dtype=np.int8).view(np.uint8) - 8
    g[208], g[209] = 0x00, 0x3C
    r = oracle.ggml_to_reading("q6_K", g)
    d, sc, q = oracle.decode_q6k(r)
    assert d == 1.0 and list(sc) == list(range(-8, 8))
    assert (q[0], q[32], q[64], q[96], q[128]) == (-31, -13, 2, 20, -1)
    assert q[1] == q[33] == q[129] == q[255] == -32


def test_ggml_roundtrip_against_independent_encoder(oracle_lib):
    """Fields -> ggml bytes (tests/encode.py) -> oracle conversion -> the reading's
    decoder gives the same fields, and equals the reading's own encoder byte for byte."""
    rng = np.random.default_rng(11)
    for _ in range(30):
        d, dmin, sc, m, q = random_q4k_fields(rng)
        g = encode_q4k_ggml(f16_bits(d), f16_bits(dmin), sc, m, q)
        r = oracle.ggml_to_reading("q4_K", g)
        assert np.array_equal(r, encode_q4k(f16_bits(d), f16_bits(dmin), sc, m, q))
        d, sc, q = random_q6k_fields(rng, (-128, 127))
        g = encode_q6k_ggml(f16_bits(d), sc, q)
        r = oracle.ggml_to_reading("q6_K", g)
        assert np.array_equal(r, encode_q6k(f16_bits(d), sc, q))
    # in place (the same buffer as source and destination)
    blocks = np.stack([encode_q6k_ggml(f16_bits(1.0), np.zeros(16), rng.integers(-32, 32, 256)) for _ in range(3)])
    want = oracle.ggml_to_reading("q6_K", blocks)
    lib = oracle._load()
    lib.oracle_ggml_to_reading(14, blocks.ctypes.data, 3, blocks.ctypes.data)
    assert np.array_equal(blocks, want)
