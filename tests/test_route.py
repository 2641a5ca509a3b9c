"""Default kernel choice of the GEMM calls, through the host-only query mmq_debug_route
(no GPU needed).  The expected choices are the kernels that were faster on GB300
(152 SMs) in paired CUDA-graph timings of the chunk and super-block kernels (µs in the
comments: chunk / super-block); the GPU suite checks that real calls take the kernel
this query names."""
import pytest

import quant_int8_mmq_gb300 as mmq

GB300_SMS = 152


@pytest.mark.parametrize("typ,od,id_,M,want,note", [
    ("q4_K", 4096, 4096, 1024, "super-block", "69.5 / 53.9; 128 tiles of 128x256, fewer than the SMs"),
    ("q4_K", 4096, 4096, 512, "chunk", "36.5 / 39.3; 64 tiles, every one split in K"),
    ("q4_K", 4096, 4096, 129, "chunk", "24.0 / 37.0"),
    ("q4_K", 11008, 4096, 256, "super-block", "58.9 / 55.0"),
    ("q4_K", 11008, 4096, 3314, "super-block", "the prompt-length FFN gate GEMM"),
    ("q4_K", 4096, 14336, 450, "super-block", "110.1 / 98.0"),
    ("q4_K", 2560, 768, 1024, "super-block", "22.8 / 16.3"),
    ("q6_K", 4097, 11008, 896, "super-block", "169.6 / 125.7"),
    ("q6_K", 4097, 11008, 1152, "chunk", "170.8 / 196.0; 153 tiles: one left for a second round"),
    ("q6_K", 4096, 11008, 384, "super-block", "78.2 / 72.6"),
    ("q6_K", 4096, 4096, 450, "chunk", "33.8 / 37.2"),
    ("q6_K", 5100, 768, 1300, "chunk", "26.5 / 33.3"),
    ("q6_K", 32000, 4096, 129, "super-block", "113.6 / 95.5"),
])
def test_route_follows_the_measured_winner(mmq_lib, typ, od, id_, M, want, note):
    assert mmq.mmq_debug_route(typ, od, id_, M, 1, GB300_SMS) == want, note


@pytest.mark.parametrize("od,id_,M", [(4096, 11008, 129), (4096, 4096, 1024), (4096, 11008, 3314),
                                      (32000, 4096, 3314), (4097, 11008, 2048)])
def test_two_tile_q6k_takes_the_chunk_kernel(mmq_lib, od, id_, M):
    """q6_K whose scales do not fold (some |sc| > 64) runs two tiles per k-block; the
    chunk kernel was faster at every M measured (e.g. 4096x11008 at M = 3314: 472.5
    against 697.9 µs), so only the fold state decides.  An unknown fold state routes as
    folded."""
    assert mmq.mmq_debug_route("q6_K", od, id_, M, 0, GB300_SMS) == "chunk"
    assert mmq.mmq_debug_route("q6_K", od, id_, M, -1, GB300_SMS) == mmq.mmq_debug_route(
        "q6_K", od, id_, M, 1, GB300_SMS)


def test_q4k_ignores_the_fold_state(mmq_lib):
    for M in (129, 700, 3314):
        got = {mmq.mmq_debug_route("q4_K", 4096, 4096, M, f, GB300_SMS) for f in (-1, 0, 1)}
        assert len(got) == 1


@pytest.mark.parametrize("typ,od,id_,M,want", [
    ("q4_K", 11008, 4096, 1, "weight-streaming"),
    ("q4_K", 11008, 4096, 8, "few-token"),          # large weight: few-token from 7 tokens
    ("q4_K", 1024, 1024, 8, "weight-streaming"),
    ("q6_K", 4097, 11008, 31, "few-token"),
    ("q6_K", 4097, 11008, 64, "few-token"),
    ("q6_K", 4097, 11008, 65, "chunk"),             # 33 tiles: every one split in K
])
def test_route_below_the_tile_kernels(mmq_lib, typ, od, id_, M, want):
    assert mmq.mmq_debug_route(typ, od, id_, M, 1, GB300_SMS) == want


def test_route_is_one_of_the_tile_kernels_above_64_tokens(mmq_lib):
    for typ in ("q4_K", "q6_K"):
        for od in (256, 4096, 11008, 32000):
            for id_ in (256, 4096, 14336):
                for M in (65, 128, 1000, 3314, 20000):
                    assert mmq.mmq_debug_route(typ, od, id_, M, 1, GB300_SMS) in ("chunk", "super-block")


def test_route_argument_errors(mmq_lib):
    lib = mmq.load()
    import ctypes
    out = ctypes.c_int(-1)
    assert lib.mmq_debug_route(12, 4096, 4096, 512, 1, 152, None) == 1
    assert lib.mmq_debug_route(12, 4096, 4096, 512, 1, 0, ctypes.byref(out)) == 1
    assert lib.mmq_debug_route(12, 4096, 4096, 512, 2, 152, ctypes.byref(out)) == 1
    assert lib.mmq_debug_route(12, 4096, 4096, 0, 1, 152, ctypes.byref(out)) == 2
    assert lib.mmq_debug_route(12, 4096, 300, 512, 1, 152, ctypes.byref(out)) == 2
    assert lib.mmq_debug_route(7, 4096, 4096, 512, 1, 152, ctypes.byref(out)) == 1
    assert out.value == -1
