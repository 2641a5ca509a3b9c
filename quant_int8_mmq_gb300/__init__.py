"""GB300 (sm_103a) prefill MMQ: q6_K / q4_K weight super-blocks x per-32 q8 activations.

Thin ctypes binding over the C ABI in ``include/mmq.h`` (``libmmq_gb300.so``, built
in-tree by ``quant_int8_mmq_gb300.build``).  The functions named like the C entry
points take raw device pointers and a stream handle and only marshal arguments;
every step of the computation runs in the library's CUDA kernels.  The tensor
helpers below them use PyTorch for device memory and streams only.

There is no fallback: if the library is missing or fails to load, every call
raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

from .build import LIB_PATH

__all__ = [
    "MMQError", "MMQ_Q4_K", "MMQ_Q6_K", "load", "lib_path",
    "mmq_act_plane_bytes", "mmq_act_scale_layout", "mmq_act_ft_layout", "mmq_quantize_act",
    "mmq_packed_weight_bytes",
    "mmq_packed_weight_layout",
    "mmq_pack_weights", "mmq_pack_weights_fused", "mmq_convert_ggml_blocks", "mmq_gemm_q6k", "mmq_gemm_q4k", "mmq_debug_gemm_dots", "mmq_debug_select_large_m_kernel",
    "mmq_debug_inject_wait_timeout", "mmq_debug_route", "ROUTES",
    "mmq_get_device_error", "mmq_status_string", "mmq_last_path", "mmq_version", "mmq_launch_count",
    "quantize_act", "pack_weights", "pack_weights_fused", "gemm", "gemm_dots", "TYPES",
]

MMQ_Q4_K = 12
MMQ_Q6_K = 14
TYPES = {"q4_K": MMQ_Q4_K, "q6_K": MMQ_Q6_K}
BLOCK_BYTES = {MMQ_Q4_K: 144, MMQ_Q6_K: 210}

STATUS = {0: "MMQ_OK", 1: "MMQ_ERR_ARG", 2: "MMQ_ERR_SHAPE", 3: "MMQ_ERR_ALIGN", 4: "MMQ_ERR_CUDA",
          5: "MMQ_ERR_TIMEOUT", 6: "MMQ_ERR_UNSUPPORTED"}

_lib = None
_lock = threading.Lock()


class MMQError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {STATUS.get(status, status)}")


def lib_path() -> str:
    return LIB_PATH


def load():
    """Load libmmq_gb300.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is not built; run quant_int8_mmq_gb300.build.build() "
                               "(or __graft_entry__.build())")
        lib = ctypes.CDLL(LIB_PATH)
        P, I, S = ctypes.c_void_p, ctypes.c_int, ctypes.POINTER(ctypes.c_size_t)
        sig = {
            "mmq_act_plane_bytes": [I, I, S, S],
            "mmq_quantize_act": [P, I, I, I, P, P, P],
            "mmq_packed_weight_bytes": [I, I, I, S],
            "mmq_packed_weight_layout": [I, I, I, S, S],
            "mmq_act_scale_layout": [I, I, S, S, S, S],
            "mmq_act_ft_layout": [I, I, S, S, S, S, S, S],
            "mmq_pack_weights": [I, P, I, I, P, P],
            "mmq_pack_weights_fused": [I, P, I, P, I, I, P, P],
            "mmq_convert_ggml_blocks": [I, P, ctypes.c_size_t, P, P],
            "mmq_gemm_q6k": [P, I, I, P, P, I, P, I, P],
            "mmq_gemm_q4k": [P, I, I, P, P, I, P, I, P],
            "mmq_debug_gemm_dots": [I, P, I, I, P, P, I, P, P],
            "mmq_debug_select_large_m_kernel": [I],
            "mmq_debug_route": [I, I, I, I, I, I, ctypes.POINTER(ctypes.c_int)],
            "mmq_debug_inject_wait_timeout": [I, ctypes.c_ulonglong],
            "mmq_get_device_error": [P],
        }
        for name, args in sig.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = ctypes.c_int
        for name in ("mmq_status_string",):
            getattr(lib, name).argtypes = [ctypes.c_int]
            getattr(lib, name).restype = ctypes.c_char_p
        for name in ("mmq_last_path", "mmq_version"):
            getattr(lib, name).argtypes = []
            getattr(lib, name).restype = ctypes.c_char_p
        _lib = lib
        return lib


def _check(st: int, what: str):
    if st != 0:
        raise MMQError(st, what)


# ----------------------------------------------------------------------------
# Same names as the C entry points (pointers and streams as Python ints).
# ----------------------------------------------------------------------------
def mmq_act_plane_bytes(M: int, K: int):
    qa, sc = ctypes.c_size_t(), ctypes.c_size_t()
    _check(load().mmq_act_plane_bytes(M, K, ctypes.byref(qa), ctypes.byref(sc)), "mmq_act_plane_bytes")
    return qa.value, sc.value


def mmq_quantize_act(x, M, K, ldx, qa, scales, stream=0):
    _check(load().mmq_quantize_act(x, M, K, ldx, qa, scales, stream or None), "mmq_quantize_act")


def mmq_packed_weight_bytes(t, od, id_):
    b = ctypes.c_size_t()
    _check(load().mmq_packed_weight_bytes(t, od, id_, ctypes.byref(b)), "mmq_packed_weight_bytes")
    return b.value


PLANES = ("codes", "pairs", "sbd", "aux", "flag", "raw", "cw", "sc", "dm", "codes2")
SMALL_M = 8          # token counts up to this take the weight-streaming path
FT_MAX_M = 64        # token counts up to this take the few-token GEMM (and get its planes)


def mmq_packed_weight_layout(t, od, id_):
    """{plane name: (offset, size)} of a packed weight buffer."""
    off = (ctypes.c_size_t * len(PLANES))()
    size = (ctypes.c_size_t * len(PLANES))()
    _check(load().mmq_packed_weight_layout(t, od, id_, off, size), "mmq_packed_weight_layout")
    return {name: (off[i], size[i]) for i, name in enumerate(PLANES)}


def mmq_act_scale_layout(M, K):
    """{"pairs": (offset, size), "am": (offset, size)} of the activation scale buffer."""
    v = [ctypes.c_size_t() for _ in range(4)]
    _check(load().mmq_act_scale_layout(M, K, *[ctypes.byref(x) for x in v]), "mmq_act_scale_layout")
    return {"pairs": (v[0].value, v[1].value), "am": (v[2].value, v[3].value)}


def mmq_act_ft_layout(M, K):
    """{"tq", "ip", "fm": (offset, size)} of the few-token planes (sizes 0 when M > 64)."""
    v = [ctypes.c_size_t() for _ in range(6)]
    _check(load().mmq_act_ft_layout(M, K, *[ctypes.byref(x) for x in v]), "mmq_act_ft_layout")
    return {"tq": (v[0].value, v[1].value), "ip": (v[2].value, v[3].value), "fm": (v[4].value, v[5].value)}


def mmq_pack_weights(t, raw, od, id_, packed, stream=0):
    _check(load().mmq_pack_weights(t, raw, od, id_, packed, stream or None), "mmq_pack_weights")


def mmq_pack_weights_fused(t, raw_a, od_a, raw_b, od_b, id_, packed, stream=0):
    _check(load().mmq_pack_weights_fused(t, raw_a, od_a, raw_b, od_b, id_, packed, stream or None),
           "mmq_pack_weights_fused")


def mmq_convert_ggml_blocks(t, src, nblocks, dst, stream=0):
    _check(load().mmq_convert_ggml_blocks(t, src, nblocks, dst, stream or None), "mmq_convert_ggml_blocks")


def mmq_gemm_q6k(packed, od, id_, qa, scales, M, Y, ldy, stream=0):
    _check(load().mmq_gemm_q6k(packed, od, id_, qa, scales, M, Y, ldy, stream or None), "mmq_gemm_q6k")


def mmq_gemm_q4k(packed, od, id_, qa, scales, M, Y, ldy, stream=0):
    _check(load().mmq_gemm_q4k(packed, od, id_, qa, scales, M, Y, ldy, stream or None), "mmq_gemm_q4k")


def mmq_debug_gemm_dots(t, packed, od, id_, qa, scales, M, dots, stream=0):
    _check(load().mmq_debug_gemm_dots(t, packed, od, id_, qa, scales, M, dots, stream or None),
           "mmq_debug_gemm_dots")


def mmq_debug_select_large_m_kernel(which: int):
    _check(load().mmq_debug_select_large_m_kernel(which), "mmq_debug_select_large_m_kernel")


ROUTES = {0: "weight-streaming", 1: "chunk", 2: "super-block", 3: "few-token"}


def mmq_debug_route(t, od: int, id_: int, M: int, fold: int = 1, nsm: int = 152) -> str:
    """The kernel the default selection gives (t, od, id, M) on a device with nsm SMs,
    for q6_K codes folded (fold 1), in two tiles (0) or of unknown state (-1); host
    logic only, no CUDA call."""
    out = ctypes.c_int(-1)
    _check(load().mmq_debug_route(TYPES.get(t, t), od, id_, M, fold, nsm, ctypes.byref(out)), "mmq_debug_route")
    return ROUTES[out.value]


def mmq_debug_inject_wait_timeout(fill: int, limit_ns: int = 0):
    """Arm (fill >= 0) or disarm (fill < 0) the one-shot wait-timeout injection of the
    next tile-GEMM launch (see include/mmq.h)."""
    _check(load().mmq_debug_inject_wait_timeout(fill, limit_ns), "mmq_debug_inject_wait_timeout")


def mmq_get_device_error(stream=0) -> int:
    """Returns the raw status (0 ok, 5 timeout, 4 CUDA error)."""
    return load().mmq_get_device_error(stream or None)


def mmq_status_string(st: int) -> str:
    return load().mmq_status_string(st).decode()


def mmq_launch_count():
    """Kernel launches the library has made in this process."""
    lib = load()
    lib.mmq_launch_count.restype = ctypes.c_ulonglong
    return int(lib.mmq_launch_count())


def mmq_last_path() -> str:
    return load().mmq_last_path().decode()


def mmq_version() -> str:
    return load().mmq_version().decode()


# ----------------------------------------------------------------------------
# Tensor helpers: PyTorch provides device memory and the current stream only.
# ----------------------------------------------------------------------------
def _torch():
    import torch
    return torch


def _stream(stream):
    torch = _torch()
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _type_id(t) -> int:
    return TYPES[t] if isinstance(t, str) else int(t)


def _nbytes(t) -> int:
    return t.numel() * t.element_size()


def _require(cond, msg):
    # ValueError rather than assert: a buffer too small for the kernel must never reach it
    if not cond:
        raise ValueError(msg)


def _check_gemm_buffers(tid, packed, od, id_, qa, scales, M):
    """Sizes first (testable without a GPU), then placement: every buffer a GEMM kernel reads
    must hold what the size queries of the C ABI say it reads."""
    _require(packed.is_contiguous() and _nbytes(packed) >= mmq_packed_weight_bytes(tid, od, id_),
             f"packed holds {_nbytes(packed)} bytes, the ({od} x {id_}) weights need "
             f"{mmq_packed_weight_bytes(tid, od, id_)}")
    qb, sb = mmq_act_plane_bytes(M, id_)
    _require(qa.is_contiguous() and _nbytes(qa) >= qb, f"qa holds {_nbytes(qa)} bytes, M={M} K={id_} needs {qb}")
    _require(scales.is_contiguous() and _nbytes(scales) >= sb,
             f"scales holds {_nbytes(scales)} bytes, M={M} K={id_} needs {sb}")
    _require(packed.is_cuda and qa.is_cuda and scales.is_cuda, "packed, qa and scales must be CUDA tensors")
    _require(packed.device == qa.device == scales.device, "packed, qa and scales must be on one device")


def quantize_act(x, qa=None, scales=None, stream=None):
    """x: float32 CUDA tensor [M, K] (row stride >= K).  Returns (qa, scales) uint8 buffers."""
    torch = _torch()
    _require(x.dtype == torch.float32 and x.dim() == 2 and x.stride(1) == 1,
             "x must be a float32 [M, K] tensor with unit column stride")
    M, K = x.shape
    qb, sb = mmq_act_plane_bytes(M, K)
    _require(x.is_cuda, "x must be a CUDA tensor")
    if qa is None:
        qa = torch.empty(qb, dtype=torch.uint8, device=x.device)
    if scales is None:
        scales = torch.empty(sb, dtype=torch.uint8, device=x.device)
    _require(qa.is_contiguous() and _nbytes(qa) >= qb, f"qa holds {_nbytes(qa)} bytes, M={M} K={K} needs {qb}")
    _require(scales.is_contiguous() and _nbytes(scales) >= sb,
             f"scales holds {_nbytes(scales)} bytes, M={M} K={K} needs {sb}")
    _require(qa.is_cuda and scales.is_cuda and qa.device == x.device == scales.device,
             "qa and scales must be CUDA tensors on x's device")
    mmq_quantize_act(x.data_ptr(), M, K, x.stride(0), qa.data_ptr(), scales.data_ptr(), _stream(stream))
    return qa, scales


def pack_weights(t, raw, od, id_, packed=None, stream=None):
    """raw: uint8 CUDA tensor holding od * id/256 super-blocks.  Returns the packed buffer."""
    torch = _torch()
    tid = _type_id(t)
    _require(raw.dtype == torch.uint8 and raw.is_contiguous(), "raw must be a contiguous uint8 tensor")
    _require(raw.numel() == od * (id_ // 256) * BLOCK_BYTES[tid],
             f"raw holds {raw.numel()} bytes, {od} x {id_} {t} weights are {od * (id_ // 256) * BLOCK_BYTES[tid]}")
    _require(raw.is_cuda, "raw must be a CUDA tensor")
    nb = mmq_packed_weight_bytes(tid, od, id_)
    if packed is None:
        packed = torch.empty(nb, dtype=torch.uint8, device=raw.device)
    _require(packed.is_cuda and packed.is_contiguous() and _nbytes(packed) >= nb,
             f"packed must be a contiguous CUDA buffer of at least {nb} bytes")
    mmq_pack_weights(tid, raw.data_ptr(), od, id_, packed.data_ptr(), _stream(stream))
    return packed


def pack_weights_fused(t, raw_a, od_a, raw_b, od_b, id_, packed=None, stream=None):
    """Two raw weights of one type and width (uint8 CUDA tensors) packed as one weight of
    od_a + od_b rows (a's rows first); one GEMM on it computes both outputs."""
    torch = _torch()
    tid = _type_id(t)
    for raw, od in ((raw_a, od_a), (raw_b, od_b)):
        _require(raw.dtype == torch.uint8 and raw.is_contiguous() and raw.is_cuda,
                 "raw weights must be contiguous uint8 CUDA tensors")
        _require(raw.numel() == od * (id_ // 256) * BLOCK_BYTES[tid],
                 f"raw holds {raw.numel()} bytes, {od} x {id_} {t} weights are {od * (id_ // 256) * BLOCK_BYTES[tid]}")
    _require(raw_a.device == raw_b.device, "both raw weights must be on one device")
    nb = mmq_packed_weight_bytes(tid, od_a + od_b, id_)
    if packed is None:
        packed = torch.empty(nb, dtype=torch.uint8, device=raw_a.device)
    _require(packed.is_cuda and packed.is_contiguous() and _nbytes(packed) >= nb,
             f"packed must be a contiguous CUDA buffer of at least {nb} bytes")
    mmq_pack_weights_fused(tid, raw_a.data_ptr(), od_a, raw_b.data_ptr(), od_b, id_, packed.data_ptr(),
                           _stream(stream))
    return packed


def gemm(t, packed, od, id_, qa, scales, M, Y=None, stream=None):
    """Y [M, od] float32 (allocated if not given; a given Y may have row stride >= od)."""
    torch = _torch()
    tid = _type_id(t)
    _check_gemm_buffers(tid, packed, od, id_, qa, scales, M)
    if Y is None:
        Y = torch.empty((M, od), dtype=torch.float32, device=packed.device)
    _require(Y.dtype == torch.float32 and Y.dim() == 2 and Y.stride(1) == 1 and Y.shape[0] >= M
             and Y.shape[1] >= od and Y.is_cuda and Y.device == packed.device,
             f"Y must be a float32 CUDA tensor [>= {M}, >= {od}] with unit column stride on the weights' device")
    fn = mmq_gemm_q6k if tid == MMQ_Q6_K else mmq_gemm_q4k
    fn(packed.data_ptr(), od, id_, qa.data_ptr(), scales.data_ptr(), M, Y.data_ptr(), Y.stride(0), _stream(stream))
    return Y


def gemm_dots(t, packed, od, id_, qa, scales, M, stream=None):
    """Raw integer dots from the GEMM kernel as a flat f32 buffer of M*od*(id/32)
    values, one per (token, row, chunk); see include/mmq.h."""
    torch = _torch()
    tid = _type_id(t)
    _check_gemm_buffers(tid, packed, od, id_, qa, scales, M)
    nsub = id_ // 32
    dots = torch.full((M * od * nsub,), float("nan"), dtype=torch.float32, device=packed.device)
    mmq_debug_gemm_dots(tid, packed.data_ptr(), od, id_, qa.data_ptr(), scales.data_ptr(), M, dots.data_ptr(),
                        _stream(stream))
    return dots
