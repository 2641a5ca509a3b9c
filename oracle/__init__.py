"""CPU oracle for the q6_K / q4_K x q8 prefill MMQ (numpy wrappers over mmq_oracle.c).

TEST INFRASTRUCTURE ONLY: tests/, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` are the only callers.  Nothing in ``quant_int8_mmq_gb300``
imports this package, and this package imports nothing from it.

Every function is a thin ctypes call into ``mmq_oracle.c``; the C file cites the
page and section each step follows.  Pins (what the oracle is checked against,
other than itself) live in ``tests/test_oracle_pins.py``.  Parity unpinned: none
of the functions below; the bit mapping inside ql/qh/qs and the scales[12]
packing are readings of silent pages (pinned only against the reading, by an
independent encoder and hand-worked golden blocks).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mmq_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

QK_K = 256
CHUNK = 32
Q6K_BYTES = 210
Q4K_BYTES = 144


def build(force: bool = False) -> str:
    """Compile mmq_oracle.c into liboracle.so (gcc, IEEE arithmetic, no contraction)."""
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-std=c11", "-fPIC", "-shared",
           "-pthread", "-Wall", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        I = ctypes.c_int
        lib.oracle_f16_to_f32_array.argtypes = [P, P, ctypes.c_size_t]
        lib.oracle_quantize_act.argtypes = [P, I, I, I, P, P, P]
        lib.oracle_ggml_to_reading.argtypes = [I, P, ctypes.c_longlong, P]
        lib.oracle_decode_q6k.argtypes = [P, P, P, P]
        lib.oracle_decode_q4k.argtypes = [P, P, P, P, P, P]
        lib.oracle_scale_planes_q6k.argtypes = [P, I, I, P]
        lib.oracle_scale_planes_q4k.argtypes = [P, I, I, P, P]
        lib.oracle_dots_q6k.argtypes = [P, I, I, P, I, P]
        lib.oracle_dots_q4k.argtypes = [P, I, I, P, I, P]
        lib.oracle_gemm_q6k.argtypes = [P, I, I, P, P, P, I, P, P, I]
        lib.oracle_gemm_q4k.argtypes = [P, I, I, P, P, P, I, P, P, I]
        lib.oracle_dequant_q6k.argtypes = [P, I, I, P]
        lib.oracle_dequant_q4k.argtypes = [P, I, I, P]
        lib.oracle_codes_q6k.argtypes = [P, I, I, P]
        lib.oracle_codes_q4k.argtypes = [P, I, I, P]
        lib.oracle_fields_q6k.argtypes = [P, I, I, P, P]
        lib.oracle_fields_q4k.argtypes = [P, I, I, P, P, P, P]
        for name in ("oracle_f16_to_f32_array", "oracle_quantize_act", "oracle_decode_q6k",
                     "oracle_decode_q4k", "oracle_scale_planes_q6k", "oracle_scale_planes_q4k",
                     "oracle_dots_q6k", "oracle_dots_q4k", "oracle_gemm_q6k", "oracle_gemm_q4k",
                     "oracle_dequant_q6k", "oracle_dequant_q4k", "oracle_codes_q6k", "oracle_codes_q4k", "oracle_fields_q6k",
                     "oracle_fields_q4k"):
            getattr(lib, name).restype = None
        _lib = lib
        return lib


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return ctypes.c_void_p(a.ctypes.data)


def _raw(raw: np.ndarray, block_bytes: int, od: int | None = None):
    raw = np.ascontiguousarray(raw, dtype=np.uint8)
    if raw.ndim == 3:
        od = raw.shape[0]
        assert raw.shape[2] == block_bytes
        nsb = raw.shape[1]
    else:
        assert od is not None
        nsb = raw.size // (od * block_bytes)
    return raw, od, nsb * QK_K


def f16_to_f32(h: np.ndarray) -> np.ndarray:
    h = np.ascontiguousarray(h, dtype=np.uint16)
    out = np.empty(h.shape, np.float32)
    _load().oracle_f16_to_f32_array(_p(h), _p(out), h.size)
    return out


def quantize_act(x: np.ndarray):
    """q8 per 32-chunk: returns (q int8 [M,K], d f32 [M,K/32], ssum int32 [M,K/32])."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    M, K = x.shape
    assert K % CHUNK == 0
    q = np.empty((M, K), np.int8)
    d = np.empty((M, K // CHUNK), np.float32)
    s = np.empty((M, K // CHUNK), np.int32)
    _load().oracle_quantize_act(_p(x), M, K, K, _p(q), _p(d), _p(s))
    return q, d, s


def decode_q6k(block: np.ndarray):
    b = np.ascontiguousarray(block, dtype=np.uint8).reshape(Q6K_BYTES)
    d = np.zeros(1, np.float32)
    sc = np.zeros(16, np.int8)
    q = np.zeros(QK_K, np.int8)
    _load().oracle_decode_q6k(_p(b), _p(d), _p(sc), _p(q))
    return float(d[0]), sc, q


def decode_q4k(block: np.ndarray):
    b = np.ascontiguousarray(block, dtype=np.uint8).reshape(Q4K_BYTES)
    d = np.zeros(1, np.float32)
    dmin = np.zeros(1, np.float32)
    sc = np.zeros(8, np.uint8)
    m = np.zeros(8, np.uint8)
    q = np.zeros(QK_K, np.uint8)
    _load().oracle_decode_q4k(_p(b), _p(d), _p(dmin), _p(sc), _p(m), _p(q))
    return float(d[0]), float(dmin[0]), sc, m, q


def scale_planes_q6k(raw: np.ndarray) -> np.ndarray:
    """dsc [od, id/32, 2] f32 = d * scales[2*(c%8)+h]."""
    raw, od, id_ = _raw(raw, Q6K_BYTES)
    dsc = np.empty((od, id_ // CHUNK, 2), np.float32)
    _load().oracle_scale_planes_q6k(_p(raw), od, id_, _p(dsc))
    return dsc


def scale_planes_q4k(raw: np.ndarray):
    """(dsc, dmn), each [od, id/32] f32: d*sc_c and dmin*m_c."""
    raw, od, id_ = _raw(raw, Q4K_BYTES)
    dsc = np.empty((od, id_ // CHUNK), np.float32)
    dmn = np.empty((od, id_ // CHUNK), np.float32)
    _load().oracle_scale_planes_q4k(_p(raw), od, id_, _p(dsc), _p(dmn))
    return dsc, dmn


def dots_q6k(raw: np.ndarray, qa: np.ndarray) -> np.ndarray:
    """Per-16 sub-block int32 dots [M, od, id/16]."""
    raw, od, id_ = _raw(raw, Q6K_BYTES)
    qa = np.ascontiguousarray(qa, dtype=np.int8)
    M = qa.shape[0]
    out = np.empty((M, od, id_ // 16), np.int32)
    _load().oracle_dots_q6k(_p(raw), od, id_, _p(qa), M, _p(out))
    return out


def dots_q4k(raw: np.ndarray, qa: np.ndarray) -> np.ndarray:
    """Per-32 chunk int32 dots [M, od, id/32]."""
    raw, od, id_ = _raw(raw, Q4K_BYTES)
    qa = np.ascontiguousarray(qa, dtype=np.int8)
    M = qa.shape[0]
    out = np.empty((M, od, id_ // CHUNK), np.int32)
    _load().oracle_dots_q4k(_p(raw), od, id_, _p(qa), M, _p(out))
    return out


def _gemm(fn, block_bytes, raw, qa, da, ssum, nthreads, with_abs):
    raw, od, id_ = _raw(raw, block_bytes)
    qa = np.ascontiguousarray(qa, dtype=np.int8)
    da = np.ascontiguousarray(da, dtype=np.float32)
    ssum = np.ascontiguousarray(ssum, dtype=np.int32)
    M = qa.shape[0]
    assert qa.shape == (M, id_) and da.shape == (M, id_ // CHUNK) and ssum.shape == da.shape
    Y = np.empty((M, od), np.float64)
    S = np.empty((M, od), np.float64) if with_abs else None
    fn(_p(raw), od, id_, _p(qa), _p(da), _p(ssum), M, _p(Y), _p(S) if S is not None else None,
       int(nthreads or 1))
    return (Y, S) if with_abs else Y


def gemm_q6k(raw, qa, da, ssum, nthreads: int = 1, with_abs: bool = False):
    """f64 Y [M, od] (and the sum of |terms| when with_abs)."""
    return _gemm(_load().oracle_gemm_q6k, Q6K_BYTES, raw, qa, da, ssum, nthreads, with_abs)


def gemm_q4k(raw, qa, da, ssum, nthreads: int = 1, with_abs: bool = False):
    return _gemm(_load().oracle_gemm_q4k, Q4K_BYTES, raw, qa, da, ssum, nthreads, with_abs)


def dequant_q6k(raw: np.ndarray) -> np.ndarray:
    raw, od, id_ = _raw(raw, Q6K_BYTES)
    W = np.empty((od, id_), np.float64)
    _load().oracle_dequant_q6k(_p(raw), od, id_, _p(W))
    return W


def dequant_q4k(raw: np.ndarray) -> np.ndarray:
    raw, od, id_ = _raw(raw, Q4K_BYTES)
    W = np.empty((od, id_), np.float64)
    _load().oracle_dequant_q4k(_p(raw), od, id_, _p(W))
    return W


def codes_q6k(raw: np.ndarray) -> np.ndarray:
    """Decoded codes [od, id] int8 in [-32, 31]."""
    raw, od, id_ = _raw(raw, Q6K_BYTES)
    out = np.empty((od, id_), np.int8)
    _load().oracle_codes_q6k(_p(raw), od, id_, _p(out))
    return out


def codes_q4k(raw: np.ndarray) -> np.ndarray:
    """Decoded codes [od, id] uint8 in [0, 15]."""
    raw, od, id_ = _raw(raw, Q4K_BYTES)
    out = np.empty((od, id_), np.uint8)
    _load().oracle_codes_q4k(_p(raw), od, id_, _p(out))
    return out


def fields_q6k(raw: np.ndarray):
    """(d [od, nsb] f32, scales [od, nsb, 16] int8) of every super-block."""
    raw, od, id_ = _raw(raw, Q6K_BYTES)
    nsb = id_ // QK_K
    d = np.empty((od, nsb), np.float32)
    sc = np.empty((od, nsb, 16), np.int8)
    _load().oracle_fields_q6k(_p(raw), od, id_, _p(d), _p(sc))
    return d, sc


def fields_q4k(raw: np.ndarray):
    """(d, dmin [od, nsb] f32, sc, m [od, nsb, 8] uint8) of every super-block."""
    raw, od, id_ = _raw(raw, Q4K_BYTES)
    nsb = id_ // QK_K
    d = np.empty((od, nsb), np.float32)
    dmin = np.empty((od, nsb), np.float32)
    sc = np.empty((od, nsb, 8), np.uint8)
    m = np.empty((od, nsb, 8), np.uint8)
    _load().oracle_fields_q4k(_p(raw), od, id_, _p(d), _p(dmin), _p(sc), _p(m))
    return d, dmin, sc, m


def cpu_threads() -> int:
    return len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)


def ggml_to_reading(typ: str, blocks: np.ndarray) -> np.ndarray:
    """Blocks in the public ggml q4_K / q6_K layout (uint8, any leading shape, last
    axis the block bytes) -> the same blocks in the reading the oracle decodes
    (see mmq_oracle.c, "GGUF interop").  Parity unpinned against real GGUF files."""
    nb = Q4K_BYTES if typ == "q4_K" else Q6K_BYTES
    src = np.ascontiguousarray(blocks, dtype=np.uint8)
    assert src.shape[-1] == nb
    out = np.empty_like(src)
    _load().oracle_ggml_to_reading(12 if typ == "q4_K" else 14, src.ctypes.data, src.size // nb, out.ctypes.data)
    return out
