"""Host logic of bench.py that needs no GPU: the stack of GEMM shapes it times, the
fused-pair bookkeeping of --fuse-shared-inputs, and the rule that committed ncu counters
count only for the exact kernel sources they were captured from."""
import hashlib
import json
import os
import shutil
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402

SHAPES = {("q4_K", 4096, 4096), ("q6_K", 4096, 4096), ("q4_K", 11008, 4096), ("q6_K", 4096, 11008),
          ("q6_K", 32000, 4096)}


def test_stack_is_32_layers_of_seven_gemms_plus_lm_head():
    g = bench.stack_list(32)
    assert len(g) == 32 * 7 + 1
    assert {(t, od, i) for _, t, od, i, _ in g} == SHAPES
    assert g[-1][:4] == ("lm_head", "q6_K", 32000, 4096)
    assert len({seed for *_, seed in g}) == len(g)            # every tensor has its own seed
    per_layer = sum(od * i for name, _, od, i, _ in g if name.startswith("l0."))
    assert per_layer == 4 * 4096 * 4096 + 2 * 11008 * 4096 + 4096 * 11008
    assert [x[0] for x in bench.stack_list(2, "l1.gate,lm_head")] == ["l1.gate", "lm_head"]


def test_fused_pairs_keep_every_row_and_seed():
    g = bench.stack_list(32)
    f = bench.fuse_shared_inputs(g)
    assert len(f) == 32 * 5 + 1                                # q+k and gate+up merge per layer
    assert sum(od * i for _, _, od, i, _ in f) == sum(od * i for _, _, od, i, _ in g)
    parts = [p for *_, ps in f for p in ps]
    assert sorted(s for _, s in parts) == sorted(s for *_, s in g)
    for name, typ, od, i, ps in f:
        assert od == sum(o for o, _ in ps)
        if "+" in name:
            a, b = name.split(".")[1].split("+")
            assert (a, b) in bench.FUSED_PAIRS and len(ps) == 2
            src = {n: (t, o, ii) for n, t, o, ii, _ in g}
            layer = name.split(".")[0]
            assert src[f"{layer}.{a}"][0] == src[f"{layer}.{b}"][0] == typ   # same type and id
            assert src[f"{layer}.{a}"][2] == src[f"{layer}.{b}"][2] == i


def _sha(paths):
    h = hashlib.sha256()
    for p in paths:
        h.update(open(p, "rb").read())
    return h.hexdigest()


def test_counters_count_only_for_the_captured_sources(tmp_path, monkeypatch):
    d = json.load(open(os.path.join(ROOT, "profiles", "gemm_counters.json")))
    key, want = next(iter(d["kernels"].items()))
    srcs = [os.path.join(ROOT, "quant_int8_mmq_gb300", "csrc", n) for n in d["sources"]]
    fresh = _sha(srcs) == d["sources_sha256"]
    assert bench.kernel_traffic(key) == (want["dram_bytes"] if fresh else None)
    # a copy of the tree whose kernel sources differ by one byte reports nothing
    fake = tmp_path / "root"
    (fake / "profiles").mkdir(parents=True)
    (fake / "quant_int8_mmq_gb300" / "csrc").mkdir(parents=True)
    shutil.copy(os.path.join(ROOT, "profiles", "gemm_counters.json"), fake / "profiles")
    for n, src in zip(d["sources"], srcs):
        shutil.copy(src, fake / "quant_int8_mmq_gb300" / "csrc" / n)
    monkeypatch.setattr(bench, "ROOT", str(fake))
    assert bench.kernel_traffic(key) == (want["dram_bytes"] if fresh else None)
    last = fake / "quant_int8_mmq_gb300" / "csrc" / d["sources"][-1]
    last.write_bytes(last.read_bytes() + b"\n")
    assert bench.kernel_traffic(key) is None
    assert bench.kernel_counters(key) is None
    assert bench.kernel_traffic("no_such_kernel") is None


def test_measured_peaks_read_the_probe_and_the_driver_file():
    p = bench.measured_peaks()
    assert p["bf16_tflops_sustained"] > 0 and p["hbm_gbs"] > 0
    assert p["probe"]["int8_mma_sync_tops"] > 0
