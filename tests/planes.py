"""Read the library's tile-major planes back into row-major numpy arrays.

Implements the layouts documented in include/mmq.h (test helper; no method
arithmetic): 16384-byte operand tiles of 128 rows x 64 values of binary16 with
the 128-byte swizzle, and tile-major 8-byte scale entries.
"""
import numpy as np

TILE_ROWS = 128
TILE_K = 64


def _tile_index():
    r = np.arange(TILE_ROWS)[:, None]
    k = np.arange(TILE_K)[None, :]
    byte = r * 128 + (((k >> 3) ^ (r & 7)) << 4) + ((k & 7) << 1)
    return byte // 2  # index in binary16 units


_IDX = _tile_index()


def untile_codes(buf: np.ndarray, rows_padded: int, K: int) -> np.ndarray:
    """Code plane (uint8 bytes) -> int64 codes [rows_padded, K]."""
    nt, nkb = rows_padded // TILE_ROWS, K // TILE_K
    u16 = np.ascontiguousarray(buf[: rows_padded * K * 2]).view(np.uint16).reshape(nt, nkb, TILE_ROWS * TILE_K)
    assert not np.any(u16 == 0x8000), "code 0 must be stored as +0"   # pins the bits, not only the values
    tiles = u16[:, :, _IDX]                         # [nt, nkb, 128, 64]
    vals = tiles.view(np.float16).astype(np.float64)
    out = vals.transpose(0, 2, 1, 3).reshape(rows_padded, K)
    assert np.all(out == np.round(out)), "codes must be exact integers"
    return out.astype(np.int64)


def untile_pairs(buf: np.ndarray, rows_padded: int, nchunk: int, dtype0, dtype1):
    """Scale plane (uint8 bytes) -> two arrays [rows_padded, nchunk]."""
    nt = rows_padded // TILE_ROWS
    raw = np.ascontiguousarray(buf[: rows_padded * nchunk * 8]).view(np.uint32).reshape(nt, nchunk, TILE_ROWS, 2)
    raw = raw.transpose(0, 2, 1, 3).reshape(rows_padded, nchunk, 2)
    return raw[..., 0].copy().view(dtype0), raw[..., 1].copy().view(dtype1)


def padded(n: int) -> int:
    return (n + TILE_ROWS - 1) // TILE_ROWS * TILE_ROWS


def _tf32_index():
    r = np.arange(TILE_ROWS)[:, None]
    k = np.arange(8)[None, :]
    return ((r >> 3) * 256 + (k >> 2) * 128 + (r & 7) * 16 + (k & 3) * 4) // 4


_TF32_IDX = _tf32_index()


def untile_tf32_pair(buf: np.ndarray, rows_padded: int, nsb: int):
    """hi/lo tf32 tile plane (8192-byte blocks per (row tile, super-block)) -> two
    float32 arrays [rows_padded, nsb*8]."""
    nt = rows_padded // TILE_ROWS
    f = np.ascontiguousarray(buf[: nt * nsb * 8192]).view(np.float32).reshape(nt, nsb, 2, 1024)
    tiles = f[:, :, :, _TF32_IDX]                       # [nt, nsb, 2, 128, 8]
    hi = tiles[:, :, 0].transpose(0, 2, 1, 3).reshape(rows_padded, nsb * 8)
    lo = tiles[:, :, 1].transpose(0, 2, 1, 3).reshape(rows_padded, nsb * 8)
    return hi, lo


def untile_rows(buf: np.ndarray, rows_padded: int, n: int, dtype=np.float32):
    """[row tile][n][128] plane -> [rows_padded, n]."""
    nt = rows_padded // TILE_ROWS
    a = np.ascontiguousarray(buf[: nt * n * TILE_ROWS * 4]).view(dtype).reshape(nt, n, TILE_ROWS)
    return a.transpose(0, 2, 1).reshape(rows_padded, n)


def is_tf32(a: np.ndarray) -> bool:
    return bool(np.all((a.view(np.uint32) & 0x1FFF) == 0))


def compact_plane(typ: str, codes: np.ndarray, rows_padded: int) -> np.ndarray:
    """The compact code plane documented in include/mmq.h (CW), built from decoded codes
    [od, id] (q4_K 0..15; q6_K -32..31): uint8 bytes of [row tile][k-block][word][128][16 B]."""
    od, K = codes.shape
    v = np.zeros((rows_padded, K), np.uint32)
    v[:od] = codes.astype(np.int64) + (32 if typ == "q6_K" else 0)
    nt, nkb = rows_padded // TILE_ROWS, K // TILE_K
    if typ == "q6_K":
        # word w = sub-block w of the k-block (16 values), value 4u + o in 32-bit word u at
        # byte 2 (o & 1) + (o >> 1), holding 4 (q + 32)
        vv = (4 * v).reshape(nt, TILE_ROWS, nkb, 4, 4, 4)          # [nt, r, kb, w, u, o]
        byte_of_o = np.array([0, 2, 1, 3])
        b = np.zeros((nt, TILE_ROWS, nkb, 4, 4, 4), np.uint8)
        b[..., byte_of_o] = vv.astype(np.uint8)
        return np.ascontiguousarray(b.transpose(0, 2, 3, 1, 4, 5)).reshape(-1)
    W = 2
    # v[nt, r, kb, hc, i] for the 32 values i of chunk hc of k-block kb
    vv = v.reshape(nt, TILE_ROWS, nkb, 2, 32)
    i = np.arange(32)
    u, p, h = i // 8, (i % 8) // 2, i % 2
    out = np.zeros((nt, nkb, W, TILE_ROWS, 4), np.uint32)
    for hc in range(2):
        for uu in range(4):
            sel = u == uu
            sh = (4 * p + 16 * h)[sel]
            out[:, :, hc, :, uu] = np.bitwise_or.reduce(vv[:, :, :, hc][..., sel] << sh, axis=-1).transpose(0, 2, 1)
    return out.reshape(-1).view(np.uint8)


def scale_plane(rows: np.ndarray, rows_padded: int) -> np.ndarray:
    """The sub-block scale plane (SC) from per-row bytes [od, nsb, 16]: uint8 bytes of
    [row tile][super-block][128][16 B], padded rows zero."""
    od, nsb, _ = rows.shape
    full = np.zeros((rows_padded, nsb, 16), np.uint8)
    full[:od] = rows
    return full.reshape(rows_padded // TILE_ROWS, TILE_ROWS, nsb, 16).transpose(0, 2, 1, 3).reshape(-1)


def untile_token_operand(buf: np.ndarray, n: int, K: int):
    """Few-token operand plane (tq) -> (hi, lo) float16 arrays [n, K]."""
    nkb = K // TILE_K
    u16 = np.ascontiguousarray(buf[: nkb * 2 * n * 128]).view(np.uint16).reshape(nkb, 2, n * 64)
    idx = _IDX[:n]                                           # rows 0..n-1 of the swizzled tile
    t = u16[:, :, idx]                                       # [nkb, 2, n, 64]
    hi = t[:, 0].transpose(1, 0, 2).reshape(n, K).view(np.float16)
    lo = t[:, 1].transpose(1, 0, 2).reshape(n, K).view(np.float16)
    return hi, lo
