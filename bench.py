#!/usr/bin/env python3
"""Benchmark: the 7B-shaped q4_K_M prefill GEMM stack on GB300.

One step = one pass of the whole hot path over one prompt of M = 3314 tokens:
for every GEMM of the stack (32 layers x {q, k, o, gate, up: q4_K; v, down:
q6_K} + lm_head q6_K, 225 GEMMs) the activation quantize prepass and the MMQ
GEMM, through the C ABI.  Weights are random (seeded, the pages' block
distributions), repacked once at registration (outside the timed region).

Prints one JSON line (rank 0).  `--impl reference` times the CPU oracle on a
bounded token sample of the same workload instead.

Multi-GPU: one process per GPU (torchrun); every rank runs its own replica of
the prefill (independent prompts, no collective on the data path): weak scaling.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import synth  # noqa: E402

METRIC = "q4_K/q6_K MMQ GEMM int8 TOPS and prefill-GEMM tok/s; % of GB300 int8 peak"
WORKLOAD = ("7B-shaped q4_K_M prefill GEMM stack: 32 layers x (q,k,o 4096x4096 q4_K; v 4096x4096 q6_K; "
            "gate,up 11008x4096 q4_K; down 4096x11008 q6_K) + lm_head 32000x4096 q6_K; "
            "quantize prepass per GEMM")
FALLBACK_TFLOPS_SUSTAINED = 1700.0
FALLBACK_TFLOPS_BURST = 1900.0
FALLBACK_HBM_GBS = 6800.0


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=10)
    p.add_argument("--warmup", type=int, default=3)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--layers", type=int, default=synth.STACK_LAYERS, help="fewer layers: a quick look only")
    p.add_argument("--tokens", type=int, default=synth.STACK_M)
    p.add_argument("--cpu-seconds", type=float, default=12.0, help="oracle sample budget (CPU baseline)")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--peaks", action="store_true", help="run the throughput probes and print their JSON")
    p.add_argument("--small-m-only", action="store_true",
                   help="run only the few-token cases and print their JSON (for profiling)")
    p.add_argument("--small-m-shape", default="", help="with --small-m-only: one shape, e.g. q6_K:4097x11008")
    p.add_argument("--small-m-tokens", default="", help="with --small-m-only: token counts, e.g. 1,31")
    p.add_argument("--no-configs", action="store_true", help="skip the per-configuration GEMM figures")
    p.add_argument("--q6k-scales", choices=["narrow", "full"], default="narrow",
                   help="q6_K sub-block scales of the stack: narrow = U[-32,31] (the workload's distribution), "
                        "full = U[-128,127] (the whole int8 range, as a quantizer that spreads scales produces)")
    p.add_argument("--kernel", choices=["default", "exact"], default="default",
                   help="exact: every stack GEMM on the chunk GEMM (per-sub-block f32 scale order, exact "
                        "integer dots) instead of the super-block kernel")
    p.add_argument("--no-parity", action="store_true", help="skip the sampled-token oracle check of the stack")
    p.add_argument("--only", default="", help="comma-separated GEMM names of the stack (e.g. l0.gate): "
                   "a small case for profiling, not a bench line")
    p.add_argument("--fuse-shared-inputs", action="store_true",
                   help="run q+k and gate+up of every layer as one GEMM each over one fused packed weight "
                        "(same outputs, one prepass per GEMM), reported as its own line")
    return p.parse_args()


def stack_list(layers, only=""):
    keep = {x for x in only.split(",") if x}
    out = []
    for name, typ, od, id_, seed in synth.stack_gemms():
        if name[0] == "l" and name[1].isdigit() and int(name[1:].split(".")[0]) >= layers:
            continue
        if keep and name not in keep:
            continue
        out.append((name, typ, od, id_, seed))
    return out


# Pairs of stack GEMMs that read the same activations and share type and id: with
# --fuse-shared-inputs each pair runs as one GEMM over one fused packed weight.
FUSED_PAIRS = (("q", "k"), ("gate", "up"))


def fuse_shared_inputs(gemms):
    """[(name, typ, od, id, seed)] -> [(name, typ, od, id, [(od_part, seed), ...])]."""
    by_name = {g[0]: g for g in gemms}
    out, done = [], set()
    for name, typ, od, id_, seed in gemms:
        if name in done:
            continue
        layer, _, short = name.partition(".")
        pair = next((p for p in FUSED_PAIRS if short == p[0]), None)
        if pair and f"{layer}.{pair[1]}" in by_name:
            other = by_name[f"{layer}.{pair[1]}"]
            out.append((f"{layer}.{pair[0]}+{pair[1]}", typ, od + other[2], id_, [(od, seed), (other[2], other[4])]))
            done.add(other[0])
        else:
            out.append((name, typ, od, id_, [(od, seed)]))
    return out


def config(args, extra=None):
    gemms = stack_list(args.layers, getattr(args, "only", ""))
    if getattr(args, "fuse_shared_inputs", False):
        gemms = fuse_shared_inputs(gemms)
    c = {"workload": WORKLOAD, "tokens": args.tokens, "layers": args.layers,
         "gemms_per_step": len(gemms),
         "prepass_per_gemm": True,
         "l2": "inputs larger than L2: every step streams ~14.9 GB of repacked weights (129 MB L2)"}
    if getattr(args, "only", ""):
        c["only"] = args.only
    if getattr(args, "q6k_scales", "narrow") == "full":
        c["q6k_scales"] = "U[-128,127] (whole int8 range)"
    if getattr(args, "kernel", "default") == "exact":
        c["kernel"] = "chunk GEMM for every GEMM (exact integer dots, per-sub-block f32 scale order)"
    if getattr(args, "fuse_shared_inputs", False):
        c["fused"] = ("q+k and gate+up of every layer as one GEMM each over one fused packed weight "
                      "(same outputs and MACs, one prepass per GEMM)")
    if extra:
        c.update(extra)
    return c


# ----------------------------------------------------------------------------- peaks
def _find_key(obj, names):
    if isinstance(obj, dict):
        for k, v in obj.items():
            if k in names and isinstance(v, (int, float)):
                return float(v)
        for v in obj.values():
            r = _find_key(v, names)
            if r is not None:
                return r
    return None


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    out = {"source": "fallback", "bf16_tflops_sustained": FALLBACK_TFLOPS_SUSTAINED,
           "bf16_tflops": FALLBACK_TFLOPS_BURST, "hbm_gbs": FALLBACK_HBM_GBS}
    if os.path.exists(path):
        try:
            d = json.load(open(path))
            sus = _find_key(d, {"bf16_tflops_sustained"})
            burst = _find_key(d, {"bf16_tflops"})
            hbm = _find_key(d, {"hbm_gbs"})
            if sus or burst:
                out["source"] = "measured"
                out["bf16_tflops_sustained"] = sus or burst
                out["bf16_tflops"] = burst or sus
            if hbm:
                out["hbm_gbs"] = hbm
        except Exception:
            pass
    probe = os.path.join(ROOT, "profiles", "peaks_gb300.json")
    if os.path.exists(probe):
        try:
            out["probe"] = json.load(open(probe))
        except Exception:
            pass
    return out


COUNTERS_FILE = os.path.join("profiles", "gemm_counters.json")


def _sources_sha(names):
    h = hashlib.sha256()
    for name in names:
        h.update(open(os.path.join(ROOT, "quant_int8_mmq_gb300", "csrc", name), "rb").read())
    return h.hexdigest()


def kernel_counters(kernel_key):
    """ncu counters of one launch of a kernel class from the committed summary (DRAM bytes,
    tensor-pipe and FMA-pipe shares), valid only for the unchanged kernel sources."""
    path = os.path.join(ROOT, COUNTERS_FILE)
    if not os.path.exists(path):
        return None
    try:
        d = json.load(open(path))
        if d.get("sources_sha256") != _sources_sha(d["sources"]):
            return None
        return d.get("kernels", {}).get(kernel_key)
    except Exception:
        return None


def kernel_traffic(kernel_key):
    """DRAM bytes per launch from the committed ncu summary, or None."""
    c = kernel_counters(kernel_key)
    return None if c is None else c.get("dram_bytes")


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.QUERY}", "--format=csv,noheader",
                                          "-lms", "200", "-i", self.gpu_id],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1].split()[0]))
                mx.append(float(f[2].split()[0]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------------------- nvtx
def nvtx_push(name):
    try:
        import torch
        torch.cuda.nvtx.range_push(name)
    except Exception:
        pass


def nvtx_pop():
    try:
        import torch
        torch.cuda.nvtx.range_pop()
    except Exception:
        pass


# ----------------------------------------------------------------------------- dist
def dist_init():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(world, value: float, device=None) -> float:
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------------- oracle stack
def oracle_stack_tokens(raws, xh, xf, n_tokens, threads):
    """Run the CPU oracle over the first n_tokens of the prompt through every GEMM."""
    import oracle
    for (name, typ, od, id_, seed), raw in raws:
        x = xh if id_ == 4096 else xf
        q, d, s = oracle.quantize_act(x[:n_tokens])
        fn = oracle.gemm_q6k if typ == "q6_K" else oracle.gemm_q4k
        fn(raw, q, d, s, nthreads=threads)


Q6K_SC = (-32, 31)      # q6_K sub-block scale range of the stack's weights (--q6k-scales)


def stack_blocks(typ, od, id_, seed):
    if typ == "q6_K":
        return synth.q6k_blocks(od, id_, seed, sc_lo=Q6K_SC[0], sc_hi=Q6K_SC[1])
    return synth.blocks(typ, od, id_, seed)


def host_weights(gemms):
    return [((name, typ, od, id_, seed), stack_blocks(typ, od, id_, seed)) for name, typ, od, id_, seed in gemms]


def host_acts(tokens):
    return (synth.activations(tokens, 4096, synth.STACK_SEED * 1000 + 900),
            synth.activations(tokens, 11008, synth.STACK_SEED * 1000 + 901))


def cpu_sample_run(raws, xh, xf, seconds, threads):
    """Time the oracle on the first n tokens, growing n until one pass takes about `seconds`."""
    n = 4
    while True:
        t0 = time.perf_counter()
        oracle_stack_tokens(raws, xh, xf, n, threads)
        dt = time.perf_counter() - t0
        if dt >= 0.5 * seconds or n >= xh.shape[0]:
            return n / dt, n, dt
        n = min(xh.shape[0], max(n + 1, int(n * seconds / max(dt, 1e-3))))


# ----------------------------------------------------------------------------- few tokens
SMALL_M_SHAPES = (("q6_K", 4097, 11008, "FFN down, odd od"), ("q4_K", 11008, 4096, "FFN gate"))
SMALL_M_TOKENS = (1, 4, 8, 31)
RAW_BLOCK = {"q4_K": 144, "q6_K": 210}


def graph_time(fn_calls, stream, reps):
    """Per-launch device time of the calls (cycled), from one CUDA graph of `reps`
    launches replayed three times (median), CUDA events on the replaying stream."""
    import torch
    dev = torch.cuda.current_device()
    cap = torch.cuda.Stream(dev)
    cap.wait_stream(stream)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(cap):
        with torch.cuda.graph(graph, stream=cap):
            for i in range(reps):
                fn_calls[i % len(fn_calls)](cap.cuda_stream)
    torch.cuda.synchronize()
    graph.replay()
    torch.cuda.synchronize()
    ts = []
    for _ in range(3):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        graph.replay()
        b.record(stream)
        torch.cuda.synchronize()
        ts.append(a.elapsed_time(b) * 1e-3 / reps)
    return statistics.median(ts)


def small_m_cases(lib, dev, stream, peaks, shapes=SMALL_M_SHAPES, tokens=SMALL_M_TOKENS, copies=8, reps=48):
    """Decode and prompt-tail token counts on the FFN shapes: the weights are read once per
    launch, so the figure is HBM bandwidth on the raw k-quant bytes (210 / 144 B per 256
    values).  `copies` packed weight buffers are rotated so that neither the raw plane
    nor the compact plane stays in L2."""
    import torch
    import quant_int8_mmq_gb300 as mmq
    out = []
    for typ, od, id_, what in shapes:
        raw = torch.from_numpy(synth.blocks(typ, od, id_, 77).reshape(-1)).to(dev)
        pks = [mmq.pack_weights(typ, raw, od, id_) for _ in range(copies)]
        fn = lib.mmq_gemm_q6k if typ == "q6_K" else lib.mmq_gemm_q4k
        alg = od * (id_ // 256) * RAW_BLOCK[typ]
        for M in tokens:
            x = torch.from_numpy(synth.activations(M, id_, 78)).to(dev)
            qa, sc = mmq.quantize_act(x)
            Y = torch.empty((M, od), dtype=torch.float32, device=dev)
            calls = [(lambda s, p=pk: fn(p.data_ptr(), od, id_, qa.data_ptr(), sc.data_ptr(), M, Y.data_ptr(), od, s))
                     for pk in pks]
            for c in calls:
                c(stream.cuda_stream)
            torch.cuda.synchronize()
            label = mmq.mmq_last_path()
            t = graph_time(calls, stream, reps)
            if mmq.mmq_get_device_error() != 0:
                raise RuntimeError("device error in a few-token case")
            out.append({"workload": f"{typ} {od}x{id_} ({what}), M={M}", "us": t * 1e6,
                        "achieved_gbs": alg / t / 1e9, "frac_hbm": alg / t / 1e9 / peaks["hbm_gbs"],
                        "path": label.split(":")[1].split("(")[0].strip() if ":" in label else label})
        del pks
    planes = mmq.mmq_packed_weight_layout(mmq.TYPES[SMALL_M_SHAPES[0][0]], SMALL_M_SHAPES[0][1], SMALL_M_SHAPES[0][2])
    return {"cases": out, "peak_gbs": peaks["hbm_gbs"],
            "bytes_def": "raw block bytes od*id/256*(210 q6_K | 144 q4_K) per launch",
            "l2": f"{copies} rotated weight copies per shape (q6_K FFN down: raw plane "
                  f"{planes['raw'][1] / 1e6:.1f} MB, compact plane {planes['cw'][1] / 1e6:.1f} MB each)",
            "timing": f"CUDA graph of {reps} launches, median of 3 replays, CUDA events"}


def run_small_m_only(args=None):
    import torch
    import quant_int8_mmq_gb300 as mmq
    lib = mmq.load()
    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    shapes, tokens = SMALL_M_SHAPES, SMALL_M_TOKENS
    if args is not None and args.small_m_shape:
        typ, dims = args.small_m_shape.split(":")
        od, id_ = (int(v) for v in dims.split("x"))
        shapes = ((typ, od, id_, "selected"),)
    if args is not None and args.small_m_tokens:
        tokens = tuple(int(v) for v in args.small_m_tokens.split(","))
    print(json.dumps(small_m_cases(lib, dev, stream, measured_peaks(), shapes, tokens)), flush=True)
    return 0


# ----------------------------------------------------------------------------- the configurations
def config_cases(lib, dev, stream, peaks, threads):
    """The workload's single-GEMM configurations (and their tail variants), each timed on
    the GPU and checked against the CPU oracle run in full on the same inputs, which is
    timed beside it."""
    import torch
    import oracle
    import quant_int8_mmq_gb300 as mmq
    cases = []
    for key, c in synth.CONFIGS.items():
        cases.append((key, c["type"], c["od"], c["id"], c["M"], c["seed"]))
        if "tail_M" in c:
            cases.append((key + "_tail", c["type"], c["od"], c["id"], c["tail_M"], c["seed"]))
        if "tail" in c:
            for M in c["tail"]["M"]:
                cases.append((key + f"_od{c['tail']['od']}_m{M}", c["type"], c["tail"]["od"], c["id"], M, c["seed"]))
    out = []
    probe = (peaks.get("probe") or {}).get("tcgen05_f16_tflops_n128")
    for name, typ, od, id_, M, seed in cases:
        raw = synth.blocks(typ, od, id_, seed)
        x = synth.activations(M, id_, seed + 100)
        rt = torch.from_numpy(raw.reshape(-1)).to(dev)
        nbytes = mmq.mmq_packed_weight_bytes(mmq.TYPES[typ], od, id_)
        copies = max(1, min(8, -(-256_000_000 // nbytes)))      # rotate copies past L2
        pks = [mmq.pack_weights(typ, rt, od, id_) for _ in range(copies)]
        qa, sc = mmq.quantize_act(torch.from_numpy(x).to(dev))
        Y = torch.empty((M, od), dtype=torch.float32, device=dev)
        fn = lib.mmq_gemm_q6k if typ == "q6_K" else lib.mmq_gemm_q4k
        calls = [(lambda s, p=pk: fn(p.data_ptr(), od, id_, qa.data_ptr(), sc.data_ptr(), M, Y.data_ptr(), od, s))
                 for pk in pks]
        for cl in calls:
            cl(stream.cuda_stream)
        torch.cuda.synchronize()
        label = mmq.mmq_last_path()
        t = graph_time(calls, stream, 20)
        calls[0](stream.cuda_stream)
        torch.cuda.synchronize()
        if mmq.mmq_get_device_error() != 0:
            raise RuntimeError(f"device error in configuration {name}")
        Yg = Y.cpu().numpy().astype(np.float64)
        t0 = time.perf_counter()
        q, d, s = oracle.quantize_act(x)
        ofn = oracle.gemm_q6k if typ == "q6_K" else oracle.gemm_q4k
        Yo, S = ofn(raw, q, d, s, nthreads=threads, with_abs=True)
        t_cpu = time.perf_counter() - t0
        err = np.abs(Yg - Yo)
        rel = float(err.max() / max(np.abs(Yo).max(), 1e-300))
        ok = bool(rel <= 1e-5 and np.all(err <= 1e-5 * S + 1e-30))
        ops = 2.0 * M * od * id_
        e = {"config": name, "type": typ, "od": od, "id": id_, "M": M, "us": t * 1e6, "tops_int8_equiv": ops / t / 1e12,
             "frac_of_bf16_sustained": ops / t / 1e12 / peaks["bf16_tflops_sustained"],
             "path": label.split(":")[1].split("(")[0].strip() if ":" in label else label,
             "oracle_s": t_cpu, "oracle_cores": threads, "gpu_vs_oracle": t_cpu / t,
             "parity": {"normwise_rel_err": rel, "ok": ok}}
        if probe:
            e["frac_of_tcgen05_probe"] = ops / t / 1e12 / probe
        if M <= 64:
            e["frac_hbm_raw_bytes"] = od * (id_ // 256) * RAW_BLOCK[typ] / t / 1e9 / peaks["hbm_gbs"]
        out.append(e)
        del pks, rt
    return out


# ----------------------------------------------------------------------------- stack side figures
PARITY_TOKENS = 6


def stack_parity(packed, ys, xh, xf, M):
    """The last step's output buffers (one per output width: the last GEMM of that width
    in the step wrote it) against the CPU oracle on a few sampled tokens, first and last
    included.  The prepass quantises each token on its own, so a token subset quantises
    as in the full prompt.  Bound: |Y - Y_oracle| <= 1e-5 * sum|terms| per output."""
    import oracle
    oracle.build()
    last = {}
    for name, typ, od, id_, parts, pk in packed:
        last[od] = (name, typ, od, id_, parts)
    rng = np.random.default_rng(M)
    toks = sorted({0, M - 1, *rng.choice(M, size=PARITY_TOKENS - 2, replace=False).tolist()})
    out, worst = [], 0.0
    for od, (name, typ, _, id_, parts) in sorted(last.items()):
        raw = np.concatenate([stack_blocks(typ, od_p, id_, seed) for od_p, seed in parts], axis=0)
        x = (xh if id_ == 4096 else xf)[toks]
        q, d, s = oracle.quantize_act(x)
        fn = oracle.gemm_q6k if typ == "q6_K" else oracle.gemm_q4k
        Yo, S = fn(raw, q, d, s, nthreads=oracle.cpu_threads(), with_abs=True)
        Yg = ys[od][toks].cpu().numpy().astype(np.float64)
        err = np.abs(Yg - Yo)
        ratio = float((err / (S + 1e-30)).max())
        worst = max(worst, ratio)
        out.append({"gemm": name, "od": od, "id": id_, "max_abs_err": float(err.max()),
                    "max_err_over_abs_sum": ratio})
    return {"ok": bool(worst <= 1e-5), "tokens": toks, "bound": "|Y - Y_oracle| <= 1e-5 * sum|terms|",
            "checked": out}


def exact_path_case(lib, packed, qa, sc, xh, stream, M, peaks):
    """The dominant shape (q4_K 11008x4096 at the prompt length) on the chunk GEMM, whose
    per-sub-block accumulators reproduce the pages' per-block f32 order, beside the default
    super-block kernel, both over the stack's own weights (32 copies rotated)."""
    import quant_int8_mmq_gb300 as mmq
    pks = [pk for _, typ, od, id_, _, pk in packed if (typ, od, id_) == ("q4_K", 11008, 4096)]
    if not pks:
        return None
    import torch
    Y = torch.empty((M, 11008), dtype=torch.float32, device=xh.device)
    lib.mmq_quantize_act(xh.data_ptr(), M, 4096, 4096, qa.data_ptr(), sc.data_ptr(), stream.cuda_stream)
    calls = [(lambda s, p=pk: lib.mmq_gemm_q4k(p.data_ptr(), 11008, 4096, qa.data_ptr(), sc.data_ptr(), M,
                                               Y.data_ptr(), 11008, s)) for pk in pks]
    out = {"workload": f"q4_K 11008x4096, M={M}"}
    for key, sel in (("default", 0), ("exact_chunk", 1)):
        mmq.mmq_debug_select_large_m_kernel(sel)
        try:
            calls[0](stream.cuda_stream)
            torch.cuda.synchronize()
            label = mmq.mmq_last_path()
            t = graph_time(calls, stream, len(calls))
        finally:
            mmq.mmq_debug_select_large_m_kernel(0)
        tf = 2.0 * M * 11008 * 4096 / t / 1e12
        out[key] = {"us": t * 1e6, "tflops_int8_equiv": tf, "frac": tf / peaks["bf16_tflops_sustained"],
                    "path": label.split(":")[1].split("(")[0].split(",")[0].strip() if ":" in label else label}
    if mmq.mmq_get_device_error() != 0:
        raise RuntimeError("device error in the exact-path case")
    return out


def q6k_full_range_cases(lib, dev, stream, M, xh, xf, qa, sc, peaks, min_bytes=300e6):
    """The stack's q6_K shapes with sub-block scales over the whole int8 range, as a
    quantizer that maps each super-block's largest scale to +-127 makes them (no tensor
    folds into one f16 tile): per shape the default choice, steered by the fold state the
    pack recorded (the chunk kernel), beside the super-block kernel forced, at the prompt
    length over rotated weight copies (at least 300 MB, more than L2)."""
    import torch
    import quant_int8_mmq_gb300 as mmq
    out = []
    for od, id_, x in ((4096, 11008, xf), (4096, 4096, xh), (32000, 4096, xh)):
        lib.mmq_quantize_act(x.data_ptr(), M, id_, id_, qa.data_ptr(), sc.data_ptr(), stream.cuda_stream)
        nb = mmq.mmq_packed_weight_bytes(mmq.MMQ_Q6_K, od, id_)
        pks = []
        for c in range(max(2, int(-(-min_bytes // nb)))):
            raw = torch.from_numpy(synth.q6k_blocks(od, id_, 7100 + c, sc_lo=-128, sc_hi=127).reshape(-1)).to(dev)
            pks.append(mmq.pack_weights("q6_K", raw, od, id_))
            del raw
        Y = torch.empty((M, od), dtype=torch.float32, device=dev)
        calls = [(lambda s, p=p: lib.mmq_gemm_q6k(p.data_ptr(), od, id_, qa.data_ptr(), sc.data_ptr(), M,
                                                  Y.data_ptr(), od, s)) for p in pks]
        case = {"shape": f"q6_K {od}x{id_}", "M": M, "weight_copies": len(pks)}
        for key, sel in (("default", 0), ("super_block_forced", 2)):
            mmq.mmq_debug_select_large_m_kernel(sel)
            try:
                calls[0](stream.cuda_stream)
                torch.cuda.synchronize()
                label = mmq.mmq_last_path()
                t = graph_time(calls, stream, 4 * len(calls))
            finally:
                mmq.mmq_debug_select_large_m_kernel(0)
            tf = 2.0 * M * od * id_ / t / 1e12
            case[key] = {"us": t * 1e6, "tflops_int8_equiv": tf, "frac": tf / peaks["bf16_tflops_sustained"],
                         "path": label.split(":")[1].split("(")[0].split(",")[0].strip() if ":" in label else label}
        out.append(case)
        del pks, calls, Y
    if mmq.mmq_get_device_error() != 0:
        raise RuntimeError("device error in the full-range q6_K cases")
    return {"scales": "q6_K sub-block scales U[-128,127]: two exact tiles per k-block", "cases": out}


def fused_pair_cases(lib, dev, stream, M, xh, qa, sc, copies=2):
    """q+k and gate+up of one layer as one GEMM over a fused packed weight (one weight
    pass, one launch) against the two GEMMs on the same quantised activations."""
    import torch
    import quant_int8_mmq_gb300 as mmq
    lib.mmq_quantize_act(xh.data_ptr(), M, 4096, 4096, qa.data_ptr(), sc.data_ptr(), stream.cuda_stream)
    out = []
    for a, b in FUSED_PAIRS:
        (typ, od_a, id_, slot_a), = [(t, o, i, sl) for n, t, o, i, sl in synth.STACK_LAYER if n == a]
        (_, od_b, _, slot_b), = [(t, o, i, sl) for n, t, o, i, sl in synth.STACK_LAYER if n == b]
        seps, fus = [], []
        for c in range(copies):
            ra = torch.from_numpy(synth.blocks(typ, od_a, id_, synth.stack_seed(c, slot_a)).reshape(-1)).to(dev)
            rb = torch.from_numpy(synth.blocks(typ, od_b, id_, synth.stack_seed(c, slot_b)).reshape(-1)).to(dev)
            seps.append((mmq.pack_weights(typ, ra, od_a, id_), mmq.pack_weights(typ, rb, od_b, id_)))
            fus.append(mmq.pack_weights_fused(typ, ra, od_a, rb, od_b, id_))
            del ra, rb
        fn = lib.mmq_gemm_q6k if typ == "q6_K" else lib.mmq_gemm_q4k
        Ya = torch.empty((M, od_a), dtype=torch.float32, device=dev)
        Yb = torch.empty((M, od_b), dtype=torch.float32, device=dev)
        Yf = torch.empty((M, od_a + od_b), dtype=torch.float32, device=dev)
        q, s_ = qa.data_ptr(), sc.data_ptr()
        sep_calls = [(lambda st, pa=pa, pb=pb: (fn(pa.data_ptr(), od_a, id_, q, s_, M, Ya.data_ptr(), od_a, st),
                                                fn(pb.data_ptr(), od_b, id_, q, s_, M, Yb.data_ptr(), od_b, st)))
                     for pa, pb in seps]
        fus_calls = [(lambda st, pf=pf: fn(pf.data_ptr(), od_a + od_b, id_, q, s_, M, Yf.data_ptr(), od_a + od_b, st))
                     for pf in fus]
        for cl in sep_calls + fus_calls:
            cl(stream.cuda_stream)
        torch.cuda.synchronize()
        # the two arms may split K differently in their last round, so the f32 sums can
        # differ in rounding; both are checked against the oracle by the parity tests
        ref = torch.cat([Ya, Yb], dim=1)
        diff = float((Yf - ref).abs().max() / ref.abs().max().clamp_min(1e-30))
        t_sep = graph_time(sep_calls, stream, 8)
        t_fus = graph_time(fus_calls, stream, 8)
        out.append({"pair": f"{a}+{b}", "type": typ, "od": [od_a, od_b], "id": id_, "M": M,
                    "separate_us": t_sep * 1e6, "fused_us": t_fus * 1e6, "saving": 1.0 - t_fus / t_sep,
                    "max_rel_diff_fused_vs_separate": diff})
        del seps, fus
    if mmq.mmq_get_device_error() != 0:
        raise RuntimeError("device error in the fused-pair case")
    return {"cases": out, "note": "both weights of a pair packed into one buffer (mmq_pack_weights_fused); "
                                  f"{copies} layers' weights rotated; one prepass shared by both arms"}


# ----------------------------------------------------------------------------- reference arm
def run_reference(args, world, rank):
    if rank != 0:
        return 0
    import oracle
    oracle.build()
    threads = oracle.cpu_threads()
    gemms = stack_list(args.layers)
    raws = host_weights(gemms)
    xh, xf = host_acts(args.tokens)
    # size one step's token sample so the whole run stays within a few minutes
    t0 = time.perf_counter()
    oracle_stack_tokens(raws, xh, xf, 4, threads)
    t_tok = (time.perf_counter() - t0) / 4
    # whole run (warm-up + timed steps) sized to about two minutes of CPU work
    per_step = max(1, int(120.0 / max(t_tok, 1e-6) / max(1, args.steps + args.warmup)))
    per_step = min(per_step, args.tokens)
    for _ in range(args.warmup):
        oracle_stack_tokens(raws, xh, xf, per_step, threads)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_stack_tokens(raws, xh, xf, per_step, threads)
    dt = time.perf_counter() - t0
    value = per_step * args.steps / dt
    sample = (f"{per_step} token(s) of the {args.tokens}-token prompt per step through all {len(gemms)} GEMMs "
              f"(prepass + f64 oracle GEMM, all output columns)")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tok/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64 (CPU oracle)",
            "data": "synthetic", "config": config(args),
            "cpu_baseline": {"value": value, "unit": "tok/s", "cores": threads, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------------------- our arm
def run_ours(args, world, rank, local):
    import torch

    import quant_int8_mmq_gb300 as mmq
    from quant_int8_mmq_gb300 import build as mmq_build

    if rank == 0 or world == 1:
        mmq_build.build()
    barrier(world)
    lib = mmq.load()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    sptr = stream.cuda_stream
    M = args.tokens
    gemms = stack_list(args.layers, args.only)
    if not gemms:
        raise SystemExit(f"--only {args.only!r} matches no GEMM of the stack")
    mmq.mmq_debug_select_large_m_kernel(1 if args.kernel == "exact" else 0)

    # ---- registration (untimed): generate raw blocks, upload, repack, keep the packed planes
    want_cpu = (rank == 0 and world == 1 and not args.no_cpu_baseline)
    host_raws = []
    packed = []
    for g in gemms:
        if want_cpu:
            host_raws.append((g, stack_blocks(*g[1:])))
    units = fuse_shared_inputs(gemms) if args.fuse_shared_inputs else [g[:4] + ([(g[2], g[4])],) for g in gemms]
    for name, typ, od, id_, parts in units:
        rts = [torch.from_numpy(stack_blocks(typ, od_p, id_, seed).reshape(-1)).to(dev) for od_p, seed in parts]
        if len(rts) == 1:
            pk = mmq.pack_weights(typ, rts[0], od, id_)
        else:                        # two weights that read the same activations: one GEMM
            pk = mmq.pack_weights_fused(typ, rts[0], parts[0][0], rts[1], parts[1][0], id_)
        packed.append((name, typ, od, id_, parts, pk))
        del rts
    xh_np, xf_np = host_acts(M)
    xh = torch.from_numpy(xh_np).to(dev)
    xf = torch.from_numpy(xf_np).to(dev)
    qa_b, sc_b = mmq.mmq_act_plane_bytes(M, 11008)
    qa = torch.empty(qa_b, dtype=torch.uint8, device=dev)
    sc = torch.empty(sc_b, dtype=torch.uint8, device=dev)
    ys = {od: torch.empty((M, od), dtype=torch.float32, device=dev) for od in sorted({p[2] for p in packed})}
    torch.cuda.synchronize()
    assert mmq.mmq_get_device_error() == 0

    calls = []
    for name, typ, od, id_, parts, pk in packed:
        x = xh if id_ == 4096 else xf
        gemm_fn = lib.mmq_gemm_q6k if typ == "q6_K" else lib.mmq_gemm_q4k
        calls.append((typ, od, id_, x.data_ptr(), pk.data_ptr(), ys[od].data_ptr(), gemm_fn))
    qa_p, sc_p = qa.data_ptr(), sc.data_ptr()
    quant = lib.mmq_quantize_act

    paths = {}

    def step(events=None, record_paths=False, call_list=None, before_last=None):
        cl = calls if call_list is None else call_list
        for i, (typ, od, id_, xp, pkp, yp, gemm_fn) in enumerate(cl):
            if before_last is not None and i == len(cl) - 1:
                before_last()
            st = quant(xp, M, id_, id_, qa_p, sc_p, sptr)
            if events is not None:
                events[i][0].record(stream)
            st |= gemm_fn(pkp, od, id_, qa_p, sc_p, M, yp, od, sptr)
            if events is not None:
                events[i][1].record(stream)
            if st:
                raise RuntimeError(f"launch failed with status {st}")
            if record_paths:
                paths[f"gemm_{typ}_{od}x{id_}"] = mmq.mmq_last_path()

    for w in range(args.warmup):
        step(record_paths=(w == 0))
    torch.cuda.synchronize()
    if mmq.mmq_get_device_error() != 0:
        raise RuntimeError("device error during warm-up")

    ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in calls]
          for _ in range(args.steps)]
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    try:
        uuid = str(torch.cuda.get_device_properties(dev).uuid)
        gpu_id = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
    except Exception:
        gpu_id = str(local)
    barrier(world)
    torch.cuda.synchronize()
    launches0 = mmq.mmq_launch_count()
    with ClockSampler(gpu_id) as clocks:
        nvtx_push("timed")            # lets a profiler capture exactly the timed launches
        e0.record(stream)
        for k in range(args.steps):
            step(ev[k])
        e1.record(stream)
        nvtx_pop()
        torch.cuda.synchronize()
    launches = mmq.mmq_launch_count() - launches0
    barrier(world)
    t = e0.elapsed_time(e1) * 1e-3
    if mmq.mmq_get_device_error() != 0:
        raise RuntimeError("device error in the timed region")
    t_max = max_over_ranks(world, t, dev if world > 1 else None)
    value = world * M * args.steps / t_max

    # per-kernel time by GEMM shape (events on the launching stream, inside the timed region)
    cls_time, cls_flops, cls_n = {}, {}, {}
    for k in range(args.steps):
        for (typ, od, id_, *_), (a, b) in zip(calls, ev[k]):
            key = f"gemm_{typ}_{od}x{id_}"
            cls_time[key] = cls_time.get(key, 0.0) + a.elapsed_time(b) * 1e-3
            cls_flops[key] = cls_flops.get(key, 0.0) + 2.0 * M * od * id_
            cls_n[key] = cls_n.get(key, 0) + 1
    dom = max(cls_time, key=cls_time.get)
    gemm_time = sum(cls_time.values())
    total_flops = sum(cls_flops.values())
    peaks = measured_peaks()
    achieved = cls_flops[dom] / cls_time[dom] / 1e12
    peak = peaks["bf16_tflops_sustained"]
    roof = {"bound": "tensor", "kernel": dom, "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
            "frac": achieved / peak, "traffic": kernel_traffic(dom),
            "launches": cls_n[dom], "time_share": cls_time[dom] / t,
            "achieved_def": "2*M*od*id per launch (int8-equivalent MACs x2) / mean launch time, CUDA events",
            "peak_source": f"{peaks['source']} dense bf16 sustained (f16 operands run at the bf16 rate)"}
    roof["path"] = paths.get(dom, "")
    probe = peaks.get("probe") or {}
    if probe.get("tcgen05_f16_tflops_n128"):
        # the same figure against the tcgen05 kind::f16 rate this GPU reached in a bare MMA loop
        roof["frac_of_tcgen05_probe"] = achieved / probe["tcgen05_f16_tflops_n128"]
    if "super-block tcgen05 GEMM" in roof["path"]:
        # the super-block kernel runs every contraction twice on the tensor pipe (the hi and
        # lo halves of the activation operand); the q4_K min term is not counted here
        roof["tensor_pipe_work"] = {"achieved": 2.0 * achieved, "frac": 2.0 * achieved / peak, "unit": "TFLOP/s",
                                    "def": "2 x achieved: hi and lo passes of the split activation operand"}
    counters = kernel_counters(dom)
    if counters:
        roof["ncu"] = {k: v for k, v in counters.items() if k != "dram_bytes"}

    classes = {k: {"launches": cls_n[k], "us_per_launch": cls_time[k] / cls_n[k] * 1e6,
                   "tflops_int8_equiv": cls_flops[k] / cls_time[k] / 1e12,
                   "frac_of_bf16_sustained": cls_flops[k] / cls_time[k] / 1e12 / peak,
                   "share_of_step": cls_time[k] / t} for k in sorted(cls_time, key=cls_time.get, reverse=True)}
    line = {"metric": METRIC, "value": value, "unit": "tok/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": t_max / args.steps * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f16 operands: exact int weight codes x activations p*d_a*q_a as f16 hi+lo -> f32",
            "data": "synthetic (seeded random k-quant blocks, N(0,1) activations)",
            "config": config(args, {"parallelism": f"replicas x{world}"}),
            "tops_int8_equiv": world * total_flops / args.steps / (t_max / args.steps) / 1e12,
            "gemm_only_tops": total_flops / gemm_time / 1e12,
            "gemm_share_of_step": gemm_time / t,
            "gemm_only_tok_s": world * M * args.steps / gemm_time,
            "roofline": roof,
            "gemm_classes": classes,
            "gpu_launches": launches,
            "path": mmq.mmq_last_path()}
    if probe.get("int8_mma_sync_tops"):
        line["int8_peak_tops"] = probe["int8_mma_sync_tops"]
        line["frac_of_int8_peak"] = line["gemm_only_tops"] / probe["int8_mma_sync_tops"]
    line["clocks"] = clocks.summary()

    # ---- outputs of the last step against the oracle, on sampled tokens
    if rank == 0 and not args.no_parity:
        line["parity"] = stack_parity(packed, ys, xh_np, xf_np, M)

    # ---- side measurements on rank 0 (not part of the step; default kernel choice only)
    side = not (args.only or args.fuse_shared_inputs or args.kernel != "default" or args.q6k_scales != "narrow")
    if rank == 0 and side:
        line["exact_path"] = exact_path_case(lib, packed, qa, sc, xh, stream, M, peaks)
        line["fused_shared_inputs"] = fused_pair_cases(lib, dev, stream, M, xh, qa, sc)
        line["q6k_full_range"] = q6k_full_range_cases(lib, dev, stream, M, xh, xf, qa, sc, peaks)
        line["small_m"] = small_m_cases(lib, dev, stream, peaks)
        if not args.no_configs:
            import oracle
            oracle.build()
            line["configs"] = config_cases(lib, dev, stream, peaks, oracle.cpu_threads())

    # ---- end to end through the public API: pinned host inputs in, logits out, every step.
    # The copies run on a second stream, pipelined with the GEMMs: step k + 1's inputs go
    # into the other of two device input buffers while step k computes, and step k's
    # logits come back while step k + 1 computes (its lm_head waits for that copy).
    if not args.no_e2e:
        xh_host = torch.from_numpy(xh_np).pin_memory()
        xf_host = torch.from_numpy(xf_np).pin_memory()
        y_last = ys[calls[-1][1]]
        y_host = torch.empty(y_last.shape, dtype=torch.float32).pin_memory()
        h2d = xh_host.numel() * 4 + xf_host.numel() * 4
        d2h = y_host.numel() * 4
        xin = [(xh, xf), (torch.empty_like(xh), torch.empty_like(xf))]
        call_sets = [[(c[0], c[1], c[2], (xin[b][0] if c[2] == 4096 else xin[b][1]).data_ptr()) + c[4:] for c in calls]
                     for b in range(2)]
        cstream = torch.cuda.Stream(dev)
        ev = lambda: torch.cuda.Event()
        in_ready, in_free, out_ready, out_done = [ev(), ev()], [ev(), ev()], ev(), ev()

        def fetch(b, after=None):
            with torch.cuda.stream(cstream):
                if after is not None:
                    cstream.wait_event(after)
                xin[b][0].copy_(xh_host, non_blocking=True)
                xin[b][1].copy_(xf_host, non_blocking=True)
                in_ready[b].record(cstream)

        barrier(world)
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        l0 = mmq.mmq_launch_count()
        a.record(stream)
        fetch(0, after=a)
        for k in range(args.steps):
            cur = k % 2
            if k + 1 < args.steps:
                fetch(1 - cur, after=in_free[1 - cur] if k >= 1 else None)
            stream.wait_event(in_ready[cur])
            step(call_list=call_sets[cur], before_last=(lambda: stream.wait_event(out_done)) if k >= 1 else None)
            in_free[cur].record(stream)
            out_ready.record(stream)
            with torch.cuda.stream(cstream):
                cstream.wait_event(out_ready)
                y_host.copy_(y_last, non_blocking=True)
                out_done.record(cstream)
        stream.wait_event(out_done)
        b.record(stream)
        torch.cuda.synchronize()
        barrier(world)
        te = max_over_ranks(world, a.elapsed_time(b) * 1e-3, dev if world > 1 else None)
        line["e2e"] = {"value": world * M * args.steps / te, "unit": "tok/s", "h2d_bytes_per_step": h2d,
                       "d2h_bytes_per_step": d2h}
        line["gpu_launches_e2e"] = mmq.mmq_launch_count() - l0

    if want_cpu:
        import oracle
        oracle.build()
        threads = oracle.cpu_threads()
        v, n, dt = cpu_sample_run(host_raws, xh_np, xf_np, args.cpu_seconds, threads)
        line["cpu_baseline"] = {"value": v, "unit": "tok/s", "cores": threads, "kind": "oracle",
                                "sample": f"first {n} token(s) of the prompt through all {len(gemms)} GEMMs "
                                          f"(oracle quantize + f64 GEMM, all columns), {dt:.1f} s"}
    mmq.mmq_debug_select_large_m_kernel(0)
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


def run_peaks():
    from quant_int8_mmq_gb300 import build as mmq_build
    exe = mmq_build.build_peaks()
    r = subprocess.run([exe], capture_output=True, text=True, timeout=600)
    sys.stderr.write(r.stderr)
    print(r.stdout.strip(), flush=True)
    return r.returncode


def main():
    args = parse_args()
    if args.peaks:
        return run_peaks()
    if args.small_m_only:
        return run_small_m_only(args)
    global Q6K_SC
    if args.q6k_scales == "full":
        Q6K_SC = (-128, 127)
    world, rank, local = dist_init()
    try:
        if args.impl == "reference":
            return run_reference(args, world, rank)
        return run_ours(args, world, rank, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    sys.exit(main())
