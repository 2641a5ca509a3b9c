"""The timeout path of the boundary, on the GPU.

A bounded in-kernel wait that runs out must be reported by mmq_get_device_error as
MMQ_ERR_TIMEOUT whichever kernel waited (one error word for the whole library), the
report must clear the word, and the next call must compute the right result.

The wait is made to run out on the host's say-so, with no GPU fault:
mmq_debug_inject_wait_timeout arms a one-shot injection under which the first CTA's
producer leaves one operand fill out (its barrier is never armed and no copy is
issued) and every wait of that launch gives up after 1 ms.  The kernel then leaves
its loops, drains its own copies and MMAs, frees TMEM and exits.  Launches that
split a tile over a CTA cluster are not injected (a cluster barrier has no time
limit); injected few-token launches run without the cluster split.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
import quant_int8_mmq_gb300 as mmq

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
TIMEOUT = 5


@pytest.fixture(scope="module", autouse=True)
def _lib(mmq_lib):
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    yield


def _raw(typ, od, id_, seed):
    if typ == "q4_K":
        return synth.q4k_blocks(od, id_, seed)
    full = typ == "q6_K_full"
    return synth.q6k_blocks(od, id_, seed, sc_lo=-128 if full else -32, sc_hi=127 if full else 31)


@pytest.mark.parametrize("selector,typ,M,od,id_,label", [
    (2, "q4_K", 200, 300, 768, "super-block tcgen05 GEMM"),
    (2, "q6_K", 200, 300, 768, "super-block tcgen05 GEMM"),
    (1, "q4_K", 200, 300, 768, "chunk GEMM"),
    (1, "q6_K_full", 200, 300, 768, "chunk GEMM"),
    (0, "q4_K", 31, 259, 768, "few-token GEMM"),
    (0, "q6_K_full", 31, 259, 768, "few-token GEMM"),
])
def test_expired_wait_is_reported_then_cleared(selector, typ, M, od, id_, label):
    t = "q6_K" if typ.startswith("q6_K") else typ
    raw = _raw(typ, od, id_, seed=od + M + selector)
    x = synth.activations(M, id_, seed=M + 3)
    xt = torch.from_numpy(x).to(DEV)
    packed = mmq.pack_weights(t, torch.from_numpy(raw.reshape(-1)).to(DEV), od, id_)
    qa, sc = mmq.quantize_act(xt)
    torch.cuda.synchronize()
    assert mmq.mmq_get_device_error() == 0
    mmq.mmq_debug_select_large_m_kernel(selector)
    try:
        mmq.mmq_debug_inject_wait_timeout(1, 1_000_000)          # fill 1 of CTA 0, 1 ms waits
        mmq.gemm(t, packed, od, id_, qa, sc, M)
        assert label in mmq.mmq_last_path()
        assert mmq.mmq_get_device_error() == TIMEOUT
        assert mmq.mmq_get_device_error() == 0                    # the report cleared the word
        Y = mmq.gemm(t, packed, od, id_, qa, sc, M)               # the next call runs clean
        assert mmq.mmq_get_device_error() == 0
    finally:
        mmq.mmq_debug_inject_wait_timeout(-1)
        mmq.mmq_debug_select_large_m_kernel(0)
    q, d, s = oracle.quantize_act(x)
    fn = oracle.gemm_q6k if t == "q6_K" else oracle.gemm_q4k
    Yo, S = fn(raw, q, d, s, nthreads=oracle.cpu_threads(), with_abs=True)
    err = np.abs(Y.cpu().numpy().astype(np.float64) - Yo)
    assert err.max() <= 1e-5 * np.abs(Yo).max()
    assert np.all(err <= 1e-5 * S + 1e-30)


def test_injection_is_one_shot_and_skips_the_streaming_path():
    """An armed injection waits for the next tile-GEMM launch: a weight-streaming call
    (M <= 8, no waits) leaves it armed, the next tile GEMM consumes it, and the one after
    runs clean."""
    od, id_ = 130, 512
    raw = _raw("q4_K", od, id_, seed=5)
    packed = mmq.pack_weights("q4_K", torch.from_numpy(raw.reshape(-1)).to(DEV), od, id_)
    qa1, sc1 = mmq.quantize_act(torch.from_numpy(synth.activations(4, id_, 6)).to(DEV))
    qa2, sc2 = mmq.quantize_act(torch.from_numpy(synth.activations(40, id_, 7)).to(DEV))
    torch.cuda.synchronize()
    assert mmq.mmq_get_device_error() == 0
    try:
        mmq.mmq_debug_inject_wait_timeout(0, 1_000_000)
        mmq.gemm("q4_K", packed, od, id_, qa1, sc1, 4)
        assert "weight-streaming" in mmq.mmq_last_path()
        assert mmq.mmq_get_device_error() == 0
        mmq.gemm("q4_K", packed, od, id_, qa2, sc2, 40)
        assert mmq.mmq_get_device_error() == TIMEOUT
        mmq.gemm("q4_K", packed, od, id_, qa2, sc2, 40)
        assert mmq.mmq_get_device_error() == 0
    finally:
        mmq.mmq_debug_inject_wait_timeout(-1)
