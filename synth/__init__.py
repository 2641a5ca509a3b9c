"""Seeded synthetic inputs for the q6_K / q4_K x q8 MMQ workloads.

Shared by the oracle tests, the GPU tests and bench.py.  It holds none of the
method's arithmetic: it only draws random numbers and places them at the byte
offsets the pages give for each super-block (q6_K: ql[128] at 0, qh[64] at 128,
int8 scales[16] at 192, f16 d at 208; q4_K: f16 d at 0, f16 dmin at 2, scales[12]
at 4, qs[128] at 16).

Distributions (the workload configurations):
  q6_K: ql/qh uniform bytes; scales int8 uniform in [-32, 31]; d = f16(|N(0,1)| * 1e-3)
  q4_K: d, dmin = f16(|N(0,1)| * 1e-3); scales[12] uniform bytes (so every six-bit
        scale and min is uniform in [0, 63]); qs uniform bytes (uniform nibbles)
  x:    N(0,1) float32
Generator: numpy PCG64 seeded per tensor.
"""
from __future__ import annotations

import numpy as np

QK_K = 256
Q6K_BYTES = 210
Q4K_BYTES = 144


def _rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def _ubytes(rng: np.random.Generator, shape) -> np.ndarray:
    n = int(np.prod(shape))
    return np.frombuffer(rng.bytes(n), dtype=np.uint8).reshape(shape)


def _absnormal_f16(rng: np.random.Generator, n: int, scale: float) -> np.ndarray:
    return (np.abs(rng.standard_normal(n)) * scale).astype(np.float16)


def q6k_blocks(od: int, id_: int, seed: int, sc_lo: int = -32, sc_hi: int = 31,
               d_scale: float = 1e-3) -> np.ndarray:
    """Raw q6_K weight rows, shape [od, id/256, 210] uint8."""
    assert id_ % QK_K == 0
    nsb = id_ // QK_K
    rng = _rng(seed)
    blk = np.empty((od, nsb, Q6K_BYTES), np.uint8)
    blk[:, :, 0:192] = _ubytes(rng, (od, nsb, 192))
    blk[:, :, 192:208] = rng.integers(sc_lo, sc_hi + 1, (od, nsb, 16)).astype(np.int8).view(np.uint8)
    blk[:, :, 208:210] = _absnormal_f16(rng, od * nsb, d_scale).view(np.uint8).reshape(od, nsb, 2)
    return blk


def q4k_blocks(od: int, id_: int, seed: int, d_scale: float = 1e-3) -> np.ndarray:
    """Raw q4_K weight rows, shape [od, id/256, 144] uint8."""
    assert id_ % QK_K == 0
    nsb = id_ // QK_K
    rng = _rng(seed)
    blk = np.empty((od, nsb, Q4K_BYTES), np.uint8)
    blk[:, :, 0:2] = _absnormal_f16(rng, od * nsb, d_scale).view(np.uint8).reshape(od, nsb, 2)
    blk[:, :, 2:4] = _absnormal_f16(rng, od * nsb, d_scale).view(np.uint8).reshape(od, nsb, 2)
    blk[:, :, 4:144] = _ubytes(rng, (od, nsb, 140))
    return blk


def activations(M: int, K: int, seed: int, scale: float = 1.0) -> np.ndarray:
    """x ~ N(0,1) float32, shape [M, K]."""
    rng = _rng(seed)
    x = rng.standard_normal((M, K), dtype=np.float32)
    if scale != 1.0:
        x *= np.float32(scale)
    return x


# ---------------------------------------------------------------------------
# The workload configurations (sizes and seeds).
# ---------------------------------------------------------------------------
CONFIGS = {
    "q6k_64x512_m16": dict(type="q6_K", od=64, id=512, M=16, seed=0),
    "q4k_attn_4096x4096_m512": dict(type="q4_K", od=4096, id=4096, M=512, seed=1),
    "q4k_ffn_gate_11008x4096_m2048": dict(type="q4_K", od=11008, id=4096, M=2048, seed=2, tail_M=2047),
    "q6k_ffn_down_4096x11008_m2048": dict(type="q6_K", od=4096, id=11008, M=2048, seed=3,
                                      tail=dict(od=4097, M=(1, 31))),
}

# 7B-shaped prefill GEMM stack: per layer (name, type, od, id, slot)
STACK_LAYER = [
    ("q", "q4_K", 4096, 4096, 0),
    ("k", "q4_K", 4096, 4096, 1),
    ("v", "q6_K", 4096, 4096, 2),
    ("o", "q4_K", 4096, 4096, 3),
    ("gate", "q4_K", 11008, 4096, 4),
    ("up", "q4_K", 11008, 4096, 5),
    ("down", "q6_K", 4096, 11008, 6),
]
STACK_LAYERS = 32
STACK_LM_HEAD = ("lm_head", "q6_K", 32000, 4096)
STACK_M = 3314
STACK_SEED = 4


def stack_seed(layer: int, slot: int) -> int:
    """Independent seed per stack tensor: seed*1000 + layer*10 + slot (lm_head: layer 32, slot 0)."""
    return STACK_SEED * 1000 + layer * 10 + slot


def stack_gemms():
    """Yield (name, type, od, id, seed) for every GEMM of the 7B-shaped stack, in order."""
    for layer in range(STACK_LAYERS):
        for name, typ, od, id_, slot in STACK_LAYER:
            yield (f"l{layer}.{name}", typ, od, id_, stack_seed(layer, slot))
    name, typ, od, id_ = STACK_LM_HEAD
    yield (name, typ, od, id_, stack_seed(STACK_LAYERS, 0))


def blocks(typ: str, od: int, id_: int, seed: int) -> np.ndarray:
    if typ == "q6_K":
        return q6k_blocks(od, id_, seed)
    if typ == "q4_K":
        return q4k_blocks(od, id_, seed)
    raise ValueError(typ)
