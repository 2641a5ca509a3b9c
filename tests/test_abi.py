"""The C-ABI library builds, loads, exports every symbol include/mmq.h declares,
and validates arguments on the host before touching CUDA (no GPU needed)."""
import ctypes
import os
import re

import pytest

import quant_int8_mmq_gb300 as mmq

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mmq.h")


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mmq_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = _declared_functions()
    for must in ("mmq_quantize_act", "mmq_pack_weights", "mmq_gemm_q6k", "mmq_gemm_q4k",
                 "mmq_act_plane_bytes", "mmq_packed_weight_bytes", "mmq_get_device_error",
                 "mmq_status_string", "mmq_last_path", "mmq_debug_gemm_dots"):
        assert must in names


def test_library_exports_every_declared_symbol(mmq_lib):
    lib = ctypes.CDLL(mmq.lib_path())
    for name in _declared_functions():
        assert hasattr(lib, name), name


def test_python_binding_has_same_names(mmq_lib):
    for name in _declared_functions():
        assert callable(getattr(mmq, name)), name


def test_size_queries_follow_the_documented_layout(mmq_lib):
    qa, sc = mmq.mmq_act_plane_bytes(130, 512)
    lay = mmq.mmq_act_scale_layout(130, 512)
    assert qa == 256 * 512 * 2
    assert lay["pairs"] == (0, 256 * 16 * 8)
    assert lay["am"] == (256 * 16 * 8, 2 * 2 * 8192)            # 2 token tiles x 2 super-blocks
    assert sc == lay["am"][0] + lay["am"][1]
    # token counts up to 8 add the int8 code plane after the tiles, up to 64 the few-token
    # operand (8 k-blocks x hi, lo x 16 * ceil(M/16) rows of 128 B) and 1/p (2 x 64 floats)
    assert mmq.mmq_act_plane_bytes(5, 512) == (128 * 512 * 2 + 5 * 512 + 8 * 2 * 16 * 128,
                                               128 * 16 * 8 + 2 * 8192 + 2 * 64 * 4 + 2 * 64 * 8 * 4)
    assert mmq.mmq_act_plane_bytes(8, 512)[0] == 128 * 512 * 2 + 8 * 512 + 8 * 2 * 16 * 128
    assert mmq.mmq_act_plane_bytes(9, 512)[0] == 128 * 512 * 2 + 8 * 2 * 16 * 128
    assert mmq.mmq_act_plane_bytes(64, 512)[0] == 128 * 512 * 2 + 8 * 2 * 64 * 128
    assert mmq.mmq_act_plane_bytes(65, 512)[0] == 128 * 512 * 2
    assert mmq.mmq_act_ft_layout(33, 512) == {"tq": (128 * 512 * 2, 8 * 2 * 48 * 128),
                                              "ip": (128 * 16 * 8 + 2 * 8192, 2 * 64 * 4),
                                              "fm": (128 * 16 * 8 + 2 * 8192 + 2 * 64 * 4, 2 * 64 * 8 * 4)}
    assert mmq.mmq_act_ft_layout(65, 512) == {"tq": (0, 0), "ip": (0, 0), "fm": (0, 0)}
    for t in (mmq.MMQ_Q4_K, mmq.MMQ_Q6_K):
        L = mmq.mmq_packed_weight_layout(t, 4097, 1024)
        Np, nsb = 4224, 4
        assert L["codes"] == (0, Np * 1024 * 2)
        assert L["pairs"] == (Np * 1024 * 2, Np * 32 * 8)
        assert L["sbd"] == (sum(L["pairs"]), Np * nsb * 4)
        assert L["aux"] == (sum(L["sbd"]), Np * nsb * 64)
        assert L["flag"][0] == sum(L["aux"])
        assert L["raw"] == (sum(L["flag"]), 4097 * 4 * (144 if t == mmq.MMQ_Q4_K else 224))
        words = 2 if t == mmq.MMQ_Q4_K else 4          # q4_K: 4-bit codes; q6_K: one byte per value
        assert L["cw"] == (-(-sum(L["raw"]) // 256) * 256, (Np // 128) * 16 * words * 128 * 16)
        assert L["sc"] == (sum(L["cw"]), Np * nsb * 16)
        assert L["dm"] == (sum(L["sc"]), Np * nsb * 4 if t == mmq.MMQ_Q4_K else 0)
        assert L["codes2"] == (sum(L["dm"]), Np * 1024 * 2 if t == mmq.MMQ_Q6_K else 0)
        assert all(off % 16 == 0 for off, _ in L.values())
        assert mmq.mmq_packed_weight_bytes(t, 4097, 1024) == sum(L["codes2"])


@pytest.mark.parametrize("M,K,err", [(0, 256, 2), (1, 255, 2), (1, 0, 2), (5, 300, 2), (1 << 23, 256, 2)])
def test_shape_errors(mmq_lib, M, K, err):
    with pytest.raises(mmq.MMQError) as e:
        mmq.mmq_act_plane_bytes(M, K)
    assert e.value.status == err


def test_argument_errors_are_synchronous_and_cuda_free(mmq_lib):
    lib = mmq.load()
    p16 = 0x10000          # aligned fake pointers: never dereferenced on the error paths
    # null pointers
    assert lib.mmq_quantize_act(None, 4, 256, 256, p16, p16, None) == 1
    assert lib.mmq_gemm_q4k(None, 8, 256, p16, p16, 4, p16, 8, None) == 1
    # ldx < K, ldy < od
    assert lib.mmq_quantize_act(p16, 4, 256, 200, p16, p16, None) == 1
    assert lib.mmq_gemm_q6k(p16, 8, 256, p16, p16, 4, p16, 7, None) == 1
    # shapes
    assert lib.mmq_gemm_q4k(p16, 0, 256, p16, p16, 4, p16, 8, None) == 2
    assert lib.mmq_gemm_q4k(p16, 8, 320, p16, p16, 4, p16, 8, None) == 2
    assert lib.mmq_gemm_q4k(p16, 8, 256, p16, p16, 0, p16, 8, None) == 2
    # alignment
    assert lib.mmq_gemm_q4k(p16 + 8, 8, 256, p16, p16, 4, p16, 8, None) == 3
    assert lib.mmq_gemm_q4k(p16, 8, 256, p16 + 4, p16, 4, p16, 8, None) == 3
    assert lib.mmq_gemm_q4k(p16, 8, 256, p16, p16, 4, p16 + 2, 8, None) == 3
    assert lib.mmq_quantize_act(p16 + 2, 4, 256, 256, p16, p16, None) == 3
    assert lib.mmq_pack_weights(14, p16, 8, 256, p16 + 8, None) == 3
    # bad type id
    assert lib.mmq_pack_weights(7, p16, 8, 256, p16, None) == 1
    assert lib.mmq_debug_gemm_dots(7, p16, 8, 256, p16, p16, 4, p16, None) == 1
    # fused pack: bad type, empty part, null pointer, misaligned output
    assert lib.mmq_pack_weights_fused(7, p16, 8, p16, 8, 256, p16, None) == 1
    assert lib.mmq_pack_weights_fused(12, p16, 0, p16, 8, 256, p16, None) == 2
    assert lib.mmq_pack_weights_fused(12, p16, 8, p16, 8, 300, p16, None) == 2
    assert lib.mmq_pack_weights_fused(12, p16, 8, None, 8, 256, p16, None) == 1
    assert lib.mmq_pack_weights_fused(12, p16, 8, p16, 8, 256, p16 + 8, None) == 3
    # ggml conversion: bad type, null pointers
    assert lib.mmq_convert_ggml_blocks(7, p16, 4, p16, None) == 1
    assert lib.mmq_convert_ggml_blocks(12, None, 4, p16, None) == 1
    assert lib.mmq_convert_ggml_blocks(14, p16, 4, None, None) == 1
    # kernel selector: 0 to 4 only (host state, no CUDA call)
    assert lib.mmq_debug_select_large_m_kernel(5) == 1
    assert lib.mmq_debug_select_large_m_kernel(-1) == 1
    assert lib.mmq_debug_select_large_m_kernel(4) == 0
    assert lib.mmq_debug_select_large_m_kernel(0) == 0
    # wait-timeout injection: limit 1 us .. 2 s when arming; disarming takes any limit
    assert lib.mmq_debug_inject_wait_timeout(0, 999) == 1
    assert lib.mmq_debug_inject_wait_timeout(0, 2000000001) == 1
    assert lib.mmq_debug_inject_wait_timeout(-1, 0) == 0


def test_valid_calls_without_a_gpu_report_unsupported(mmq_lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    lib = mmq.load()
    p16 = 0x10000
    assert lib.mmq_quantize_act(p16, 4, 256, 256, p16, p16, None) == 6
    assert lib.mmq_gemm_q4k(p16, 8, 256, p16, p16, 4, p16, 8, None) == 6


def test_launch_counter_counts_only_launches(mmq_lib):
    before = mmq.mmq_launch_count()
    lib = mmq.load()
    p16 = 0x10000
    assert lib.mmq_gemm_q4k(None, 8, 256, p16, p16, 4, p16, 8, None) == 1      # argument error
    assert mmq.mmq_launch_count() == before


def test_status_strings_and_labels(mmq_lib):
    for st in range(7):
        assert mmq.mmq_status_string(st).startswith(mmq.STATUS[st])
    assert "sm_103a" in mmq.mmq_version()
    assert isinstance(mmq.mmq_last_path(), str)


def test_python_helpers_refuse_short_or_host_buffers(mmq_lib):
    """The tensor helpers check every buffer a GEMM kernel reads against the size queries
    before calling the library, so a wrong buffer raises instead of reaching the GPU."""
    torch = pytest.importorskip("torch")
    od, id_, M = 300, 768, 20
    nb = mmq.mmq_packed_weight_bytes(mmq.MMQ_Q4_K, od, id_)
    qb, sb = mmq.mmq_act_plane_bytes(M, id_)
    p = torch.empty(nb, dtype=torch.uint8)
    q = torch.empty(qb, dtype=torch.uint8)
    s = torch.empty(sb, dtype=torch.uint8)
    for args, what in (((p[:-1], q, s), "packed"), ((p, q[:-16], s), "qa"), ((p, q, s[:-8]), "scales")):
        with pytest.raises(ValueError, match=what):
            mmq.gemm("q4_K", args[0], od, id_, args[1], args[2], M)
        with pytest.raises(ValueError, match=what):
            mmq.gemm_dots("q4_K", args[0], od, id_, args[1], args[2], M)
    with pytest.raises(ValueError, match="qa"):          # planes sized for fewer tokens
        mmq.gemm("q4_K", p, od, id_, q, s, 200)
    with pytest.raises(ValueError, match="packed"):      # weights of another shape
        mmq.gemm("q6_K", p, od + 128, id_, q, s, M)
    with pytest.raises(ValueError, match="CUDA"):        # right sizes, host memory
        mmq.gemm("q4_K", p, od, id_, q, s, M)


def test_quantize_and_pack_helpers_refuse_bad_inputs(mmq_lib):
    torch = pytest.importorskip("torch")
    x = torch.zeros(4, 512)
    with pytest.raises(ValueError, match="float32"):
        mmq.quantize_act(x.double())
    with pytest.raises(ValueError, match="CUDA"):
        mmq.quantize_act(x)
    raw = torch.zeros(3 * 2 * 144, dtype=torch.uint8)
    with pytest.raises(ValueError, match="raw holds"):
        mmq.pack_weights("q4_K", raw[:-1], 3, 512)
    with pytest.raises(ValueError, match="CUDA"):
        mmq.pack_weights("q4_K", raw, 3, 512)
