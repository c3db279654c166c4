#!/usr/bin/env python3
"""Batch-1 decode benchmark of the megakernel on the Llama-1B shape.

One step = one greedy decode token (one megakernel launch) of the Llama-1B
shaped model (16 layers, d 2048, 32/8 heads x 64, SwiGLU 8192, vocab 128256,
tied embedding) with random bf16 weights, after a 128-token seeded prompt:
the timed steps are positions 128..128+K-1 with the token fed back on the
device. Weights (2.47 GB) exceed L2, so every step streams them from HBM.

Prints ONE JSON line (rank 0). `--impl reference` times the fp64 CPU oracle
on the host cores instead (a bounded sample of the same workload).
With torchrun (--gpus N > 1) every rank runs an independent replica.
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
sys.path.insert(0, ROOT)

WORKLOAD = "llama1b"
FALLBACK_HBM_GBS = 6800.0


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=128)
    ap.add_argument("--warmup", type=int, default=8)
    ap.add_argument("--impl", default="mk", choices=["mk", "reference"])
    ap.add_argument("--workload", default=WORKLOAD)
    ap.add_argument("--no-comparators", action="store_true",
                    help="skip the unfused-chain timings")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the prefill, tensor-core GEMM and W2A8 GEMV timings")
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="budget of each timed oracle CPU-baseline sample (all cores, one thread); 0 skips it")
    ap.add_argument("--profile", action="store_true",
                    help="only W warm-up and K decode steps (for ncu captures); prints one line")
    ap.add_argument("--profile-prefill", action="store_true",
                    help="only W + K prefills of the workload's prompt (for ncu captures); prints one line")
    ap.add_argument("--profile-twell", action="store_true",
                    help="only mk_twell_down over 8 W_down^T copies of the workload's FFN shape at 0, 50 "
                         "and 90%% zero activations (for ncu captures); prints one line")
    ap.add_argument("--profile-gemm", action="store_true",
                    help="only W + K runs of the prefill's gate contraction (tensor cores) for the "
                         "workload's prompt (for ncu captures); prints one line")
    ap.add_argument("--profile-w2a8", action="store_true",
                    help="only W + K launches of the W2A8 GEMV over the bench's 134 MB packed matrix "
                         "(for ncu captures); prints one line")
    ap.add_argument("--trace", default=None,
                    help="also record one traced step and write its summary (JSON) here")
    return ap.parse_args()


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(x: float, ws: int, device) -> float:
    """The largest x over the ranks (the slowest replica sets the job's time)."""
    if ws == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_us_per_token(t_max_s: float, k: int, ws: int) -> float:
    """Whole-job time per token: ws replicas each decode k tokens in t_max_s."""
    return 1e6 * t_max_s / (k * ws)


def algorithmic_bytes(shape, pos: int) -> int:
    """Weights read by one step + keys/values attended over (positions 0..pos)."""
    return shape.step_weight_bytes() + shape.kv_read_bytes(pos + 1)


def shape_desc(shape) -> str:
    return (f"{shape.name} shape ({shape.n_layers} layers, d {shape.d_model}, {shape.n_heads} q / "
            f"{shape.n_kv_heads} kv heads x {shape.head_dim}, SwiGLU {shape.ffn_dim}, vocab {shape.vocab} tied)")


def l2_note(shape) -> str:
    gb = shape.step_weight_bytes() / 1e9
    if shape.step_weight_bytes() > 129e6:
        return f"inputs larger than L2: {gb:.2f} GB of weights streamed every step"
    return f"weights ({shape.step_weight_bytes() / 1e6:.1f} MB) fit in the 129 MB L2: a latency test, not a bandwidth one"


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            d = json.load(open(path))
            for k in ("hbm_gbs", "hbm_GBs", "hbm_copy_gbs"):
                if k in d and d[k]:
                    return float(d[k]), "of measured"
        except Exception:
            pass
    return FALLBACK_HBM_GBS, "of fallback"


def kernel_sha() -> str:
    h = hashlib.sha256()
    for f in ("mk_kernel.cuh", "mk_kernel_hd64.cu", "mk_kernel_hd128.cu", "mk_kernel.cu", "mk_plan.h",
              "mk_host.cpp"):
        h.update(open(os.path.join(ROOT, "decode_megakernel_llama_gb300", "csrc", f), "rb").read())
    return h.hexdigest()[:16]


def committed_traffic():
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel source (else None)."""
    path = os.path.join(ROOT, "profiles", "megakernel_llama1b_traffic.json")
    if not os.path.exists(path):
        return None
    try:
        d = json.load(open(path))
        if d.get("kernel_sha") == kernel_sha():
            return int(d["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu: int):
        self.gpu = gpu
        self.p = None

    def __enter__(self):
        try:
            self.p = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.p = None
        return self

    def __exit__(self, *a):
        self.lines = []
        if self.p is not None:
            self.p.terminate()
            try:
                out, _ = self.p.communicate(timeout=5)
            except Exception:
                self.p.kill()
                out = ""
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in getattr(self, "lines", []):
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else platform)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    import platform
    return platform.processor() or platform.machine()


def host_cores() -> int:
    """Cores this process may run on (affinity), else the machine's count."""
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def oracle_model(shape, host_w, max_seq: int):
    import oracle
    cfg = oracle.OracleConfig(shape.n_layers, shape.d_model, shape.n_heads, shape.n_kv_heads,
                              shape.head_dim, shape.ffn_dim, shape.vocab, shape.rms_eps,
                              shape.rope_theta)
    return oracle.OracleModel(cfg, host_w, max_seq)


def oracle_baseline(shape, host_w, prompt, P0: int, K: int, budget_all: float, budget_one: float):
    """The oracle as it stands on the host cores, on the bench's own positions:
    the prompt (positions 0..P0-1) untimed with all cores, then up to K decode
    steps at positions P0.. timed with all cores (at most budget_all seconds),
    then again from P0 with one thread (at most budget_one seconds)."""
    import oracle
    oracle.build()
    cores = host_cores()
    oracle.set_threads(cores)
    m = oracle_model(shape, host_w, P0 + K)
    tok = 0
    for i in range(P0):
        _, tok = m.decode_step(int(prompt[i]), i)

    def timed(budget):
        t, n, cur = 0.0, 0, tok
        while n < K:
            t0 = time.perf_counter()
            _, cur = m.decode_step(cur, P0 + n)
            t += time.perf_counter() - t0
            n += 1
            if t >= budget:
                break
        return 1e6 * t / n, n

    us_all, n_all = timed(budget_all)
    threads_all = oracle.get_threads()
    oracle.set_threads(1)
    us_one, n_one = timed(budget_one)
    oracle.set_threads(cores)
    return {"value": us_all, "unit": "us/token", "cores": threads_all, "kind": "oracle",
            "sample": f"{n_all} fp64 oracle decode steps at positions {P0}..{P0 + n_all - 1} of the same "
                      f"model after its {P0}-token prompt, {threads_all} OpenMP threads",
            "single_thread": {"value": us_one, "unit": "us/token", "cores": 1,
                              "sample": f"{n_one} steps at positions {P0}..{P0 + n_one - 1}, 1 thread"},
            "cpu_model": cpu_model(), "affinity_cores": cores}


def run_reference(args, ws, rank):
    """The oracle as it stands, on the host cores, on the GPU arm's workload:
    the prompt untimed, W warm-up steps, then K timed decode steps at the
    same positions the GPU arm times (P0..P0+K-1)."""
    if rank != 0:
        return
    import oracle
    from decode_megakernel_llama_gb300 import synth
    from decode_megakernel_llama_gb300.configs import WORKLOADS
    oracle.build()
    wl = WORKLOADS[args.workload]
    shape = wl.shape
    K, W = args.steps, args.warmup
    if wl.batch > 1 or wl.prefill:
        raise SystemExit("--impl reference times the batch-1 workloads without pre-filled caches")
    P0 = wl.prompt_len
    host_w = synth.host_weights(synth.make_weights(shape, "cpu", 0))
    cores = host_cores()
    oracle.set_threads(cores)
    m = oracle_model(shape, host_w, P0 + max(K, W))
    prompt = synth.prompt_tokens(shape.vocab, P0)
    tok = 0
    for i in range(P0):
        _, tok = m.decode_step(int(prompt[i]), i)
    tok = int(prompt[-1])
    for s in range(W):
        _, tok = m.decode_step(tok, P0 + s)
    t0 = time.perf_counter()
    for s in range(K):
        _, tok = m.decode_step(tok, P0 + s)
    us = 1e6 * (time.perf_counter() - t0) / K
    thr = oracle.get_threads()
    line = {
        "impl": "reference", "metric": "batch-1 decode us/token (Llama-1B shape) and achieved HBM GB/s vs peak",
        "value": us, "unit": "us/token", "n_gpus": ws, "steps": K,
        "warmup": W, "ms_per_step": us / 1e3, "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{wl.name}: {shape_desc(shape)}, batch 1, {P0}-token prompt, "
                               f"timed decode positions {P0}..{P0 + K - 1} (fp64 CPU oracle)"},
        "cpu_baseline": {"value": us, "unit": "us/token", "cores": thr, "kind": "oracle",
                         "sample": f"the {P0}-token prompt untimed, {W} warm-up steps, then {K} timed "
                                   f"decode steps at positions {P0}..{P0 + K - 1}",
                         "cpu_model": cpu_model(), "affinity_cores": cores},
        "e2e": {"value": us, "unit": "us/token", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def projection_params(shape) -> int:
    """Weights of one layer's seven projections."""
    d, F, qd, kvd = shape.d_model, shape.ffn_dim, shape.q_dim, shape.kv_dim
    return qd * d + 2 * kvd * d + d * qd + 3 * F * d


def bf16_tensor_peak():
    """Measured dense bf16 tensor peak (TFLOP/s) and its kind."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            d = json.load(open(path))
            if d.get("bf16_tflops"):
                return float(d["bf16_tflops"]), "of measured (burst)"
        except Exception:
            pass
    return 1900.0, "of fallback"


def measure_extras(mk, shape, prompt, P, W, dev, stream, decode_us):
    """Prefill of the P-token prompt (mk_prefill), its gate contraction alone
    (mk_tc_gemm), the W2A8 GEMV (mk_w2a8_gemv) and the activation-sparse down
    projection (mk_twell_down), timed with CUDA events on the launching stream
    after W warm-up runs."""
    import torch
    from decode_megakernel_llama_gb300 import _lib
    out = {}

    def timed(fn, reps):
        for _ in range(W):
            fn()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        a.record(stream)
        for _ in range(reps):
            fn()
        b.record(stream)
        torch.cuda.synchronize()
        return 1e3 * a.elapsed_time(b) / reps  # us

    peak_tf, peak_kind = bf16_tensor_peak()
    # prefill: the prompt at positions 0 .. P-1 (rewrites the same cache rows)
    toks = prompt.to(dev)
    tok = torch.zeros(1, dtype=torch.int32, device=dev)
    us = timed(lambda: mk.prefill(toks, 0, tok, None, stream), 10)
    if mk.status() != 0:
        raise SystemExit("prefill status error")
    flops = 2 * 2 * P * shape.n_layers * projection_params(shape)  # hi and lo terms
    out["prefill"] = {"prompt_tokens": P, "us_per_prompt": us, "us_per_token": us / P,
                      "vs_token_by_token_us": decode_us * P,
                      "projection_tflops": flops / (us * 1e-6) / 1e12,
                      "note": "tcgen05 bf16 contractions (activations as hi + lo bf16 terms), "
                              "causal attention, KV append; TFLOP/s counts the projections only, over the whole prefill"}
    # the gate contraction of that prompt on its own
    g = torch.Generator(device="cpu").manual_seed(7)
    F, d = shape.ffn_dim, shape.d_model
    w = (torch.randn(F, d, generator=g) * 0.02).to(torch.bfloat16).to(dev)
    x = torch.randn(P, d, generator=g)
    hi = x.to(torch.bfloat16)
    lo = (x - hi.float()).to(torch.bfloat16)
    hi, lo = hi.to(dev), lo.to(dev)
    y = torch.empty(P, F, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    gus = timed(lambda: _lib.tc_gemm(w, hi, lo, y, status=st, stream=stream), 20)
    if int(st.item()) != 0:
        raise SystemExit("tensor-core contraction status error")
    gflop = 2 * 2 * P * F * d
    achieved = gflop / (gus * 1e-6) / 1e12
    out["prefill"]["gate_gemm"] = {"M": F, "K": d, "N": P, "us": gus,
                                   "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak_tf,
                                                "unit": "TFLOP/s", "frac": achieved / peak_tf,
                                                "peak_source": peak_kind}}
    del w, hi, lo, y
    # W2A8 GEMV over a 134 MB packed matrix (larger than L2)
    rows, cols = 65536, 8192
    packed = torch.randint(0, 2 ** 31 - 1, (rows, cols // 16), generator=g, dtype=torch.int32)
    packed = (packed & 0x55555555).to(dev)  # codes 0 or 1 (weights -1 / 0): valid words
    xv = torch.randn(cols, generator=g).to(dev)
    yv = torch.empty(rows, device=dev)
    wus = timed(lambda: _lib.w2a8_gemv(packed, 0.02, rows, cols, xv, yv, stream=stream), 20)
    nbytes = rows * cols // 4 + 4 * cols + 4 * rows
    gbs = nbytes / (wus * 1e-6) / 1e9
    hbm, hbm_kind = measured_peak()
    out["w2a8_gemv"] = {"rows": rows, "cols": cols, "us": wus, "weights_per_s": rows * cols / (wus * 1e-6),
                        "roofline": {"bound": "hbm", "achieved": gbs, "peak": hbm, "unit": "GB/s",
                                     "frac": gbs / hbm, "peak_source": hbm_kind, "bytes_per_launch": nbytes}}
    del packed
    out["twell_down"] = measure_twell(shape, dev, stream, timed, hbm, hbm_kind)
    return out


def measure_twell(shape, dev, stream, timed, hbm, hbm_kind):
    """mk_twell_down at the model's FFN shape over seeded activations with
    0, 50 and 90 % zeros; copies of W_down^T (about 256 MB in all, larger than
    L2) are cycled so that every call reads its rows from HBM. The calls over
    all copies are captured once in a CUDA graph and the graph is replayed, so
    the time is the device's (two short kernels per call), not the host's
    launch rate. Bytes per call: the rows of the non-zero units, h, the row
    blocks' partial sums written and read back, and y."""
    import math
    import torch
    from decode_megakernel_llama_gb300 import _lib, synth
    F, d = shape.ffn_dim, shape.d_model
    ncopy = max(2, math.ceil(256e6 / (F * d * 2)))
    gen = torch.Generator(device=dev).manual_seed(21)
    wts = [(torch.randn(F, d, generator=gen, device=dev) * 0.02).to(torch.bfloat16) for _ in range(ncopy)]
    y = torch.empty(d, device=dev)
    n_sm = torch.cuda.get_device_properties(dev).multi_processor_count
    R = min(2048, max(1, -(-F // (2 * n_sm))))  # rows per block, as the unit plans them
    nb = -(-F // R)
    res = {}
    for s in (0.0, 0.5, 0.9):
        h = synth.sparse_activations(F, s, seed=22).to(dev)
        for w in wts:  # first calls outside the capture (workspace, kernel attributes)
            _lib.twell_down(w, h, y, stream=stream)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):  # captured on torch's side stream
            cap = torch.cuda.current_stream(dev)
            for w in wts:
                _lib.twell_down(w, h, y, stream=cap)
        torch.cuda.synchronize()

        def replay():
            with torch.cuda.stream(stream):
                graph.replay()
        us = timed(replay, 8) / ncopy
        nnz = int((h != 0).sum().item())
        nbytes = nnz * d * 2 + F * 4 + 2 * nb * d * 4 + d * 4
        gbs = nbytes / (us * 1e-6) / 1e9
        res[f"{s:.2f}"] = {"us": us, "nonzero_units": nnz, "bytes_per_call": nbytes, "achieved_gbs": gbs,
                           "frac": gbs / hbm}
    dense_us = res["0.00"]["us"]
    for v in res.values():
        v["speedup_vs_dense"] = dense_us / v["us"]
    half = res["0.50"]
    return {"F": F, "d": d, "by_sparsity": res,
            "roofline": {"bound": "hbm", "achieved": half["achieved_gbs"], "peak": hbm, "unit": "GB/s",
                         "frac": half["frac"], "peak_source": hbm_kind, "bytes_per_launch": half["bytes_per_call"],
                         "at_sparsity": 0.5},
            "note": "activations are seeded N(0,1) with exact zeros at random units (a stand-in for a "
                    "ReLU-gated FFN of a trained model); W_down^T copies cycled, every call reads HBM"}


def run_profile_gemm(args):
    """W + K launches of the tensor-core contraction of the prompt's gate
    projection (M = ffn, K = d_model, N = prompt tokens), nothing else."""
    import torch
    from decode_megakernel_llama_gb300 import _lib
    from decode_megakernel_llama_gb300.build import build
    from decode_megakernel_llama_gb300.configs import WORKLOADS
    build()
    dev = torch.device("cuda", 0)
    wl = WORKLOADS[args.workload]
    shape, P = wl.shape, wl.prompt_len
    g = torch.Generator(device="cpu").manual_seed(7)
    w = (torch.randn(shape.ffn_dim, shape.d_model, generator=g) * 0.02).to(torch.bfloat16).to(dev)
    x = torch.randn(P, shape.d_model, generator=g)
    hi = x.to(torch.bfloat16)
    lo = (x - hi.float()).to(torch.bfloat16)
    hi, lo = hi.to(dev), lo.to(dev)
    y = torch.empty(P, shape.ffn_dim, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    for _ in range(args.warmup + args.steps):
        _lib.tc_gemm(w, hi, lo, y, status=st)
    torch.cuda.synchronize()
    print(json.dumps({"profile_gemm": True, "status": int(st.item()), "launches": args.warmup + args.steps}),
          flush=True)


def run_profile_w2a8(args):
    """W + K launches of the W2A8 GEMV over the same 65,536 x 8,192 packed
    matrix the bench line times, nothing else."""
    import torch
    from decode_megakernel_llama_gb300 import _lib
    from decode_megakernel_llama_gb300.build import build
    build()
    dev = torch.device("cuda", 0)
    g = torch.Generator(device="cpu").manual_seed(7)
    rows, cols = 65536, 8192
    packed = torch.randint(0, 2 ** 31 - 1, (rows, cols // 16), generator=g, dtype=torch.int32)
    packed = (packed & 0x55555555).to(dev)  # codes 0 or 1 (weights -1 / 0): valid words
    xv = torch.randn(cols, generator=g).to(dev)
    yv = torch.empty(rows, device=dev)
    for _ in range(args.warmup + args.steps):
        _lib.w2a8_gemv(packed, 0.02, rows, cols, xv, yv)
    torch.cuda.synchronize()
    print(json.dumps({"profile_w2a8": True, "launches": args.warmup + args.steps}), flush=True)


def run_profile_prefill(args):
    """W + K prefills (mk_prefill) of the workload's prompt, nothing else."""
    import torch
    from decode_megakernel_llama_gb300 import _lib, synth
    from decode_megakernel_llama_gb300.build import build
    from decode_megakernel_llama_gb300.configs import WORKLOADS
    build()
    dev = torch.device("cuda", 0)
    wl = WORKLOADS[args.workload]
    shape, P = wl.shape, wl.prompt_len
    w = synth.make_weights(shape, dev, 0)
    kc, vc = synth.kv_cache(shape, P + 1, 1, dev)
    mk = _lib.Megakernel(shape, w, kc, vc)
    toks = synth.prompt_tokens(shape.vocab, P).to(dev)
    tok = torch.zeros(1, dtype=torch.int32, device=dev)
    for _ in range(args.warmup + args.steps):
        mk.prefill(toks, 0, tok)
    torch.cuda.synchronize()
    print(json.dumps({"profile_prefill": True, "status": mk.status(), "prefills": args.warmup + args.steps}),
          flush=True)
    mk.close()


def run_profile_twell(args):
    """24 calls of the activation-sparse down projection (mk_twell_down): 8
    W_down^T copies of the workload's FFN shape, each at 0, 50 and 90 % zero
    activations; 48 launches (twell_part, twell_reduce), nothing else timed."""
    import torch
    from decode_megakernel_llama_gb300 import _lib, synth
    from decode_megakernel_llama_gb300.build import build
    from decode_megakernel_llama_gb300.configs import WORKLOADS
    build()
    dev = torch.device("cuda", 0)
    shape = WORKLOADS[args.workload].shape
    F, d = shape.ffn_dim, shape.d_model
    gen = torch.Generator(device=dev).manual_seed(21)
    wts = [(torch.randn(F, d, generator=gen, device=dev) * 0.02).to(torch.bfloat16) for _ in range(8)]
    y = torch.empty(d, device=dev)
    for s in (0.0, 0.5, 0.9):
        h = synth.sparse_activations(F, s, seed=22).to(dev)
        for w in wts:
            _lib.twell_down(w, h, y)
    torch.cuda.synchronize()
    print(json.dumps({"profile_twell": True, "calls": 24, "F": F, "d": d}), flush=True)


def run_batch(args, ws, rank, local):
    """The batched workload (llama1b_b8): B sequences per step in one launch
    through the last layer, then the LM head as one tensor-core contraction
    and the tokens' draw (mk_decode_step_batch), their caches pre-filled with seeded keys/values up
    to the prompt length (a stand-in for B prompts run in lockstep), then K
    timed steps with tokens and positions chained on the device."""
    import torch
    from decode_megakernel_llama_gb300 import _lib, synth
    from decode_megakernel_llama_gb300.build import build
    from decode_megakernel_llama_gb300.configs import WORKLOADS
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    build()
    wl = WORKLOADS[args.workload]
    shape, B, P = wl.shape, wl.batch, wl.prompt_len
    K, W = args.steps, args.warmup
    max_seq = P + W + K + 1
    w = synth.make_weights(shape, dev, 0)
    kc, vc = synth.kv_cache(shape, max_seq, B, dev)
    synth.prefill_cache(kc, vc, P)
    mk = _lib.Megakernel(shape, w, kc, vc)
    stream = torch.cuda.current_stream(dev)
    toks = torch.stack([synth.prompt_tokens(shape.vocab, 1, seq=b) for b in range(B)]).view(B).to(dev)
    pos = torch.full((B,), P, dtype=torch.int32, device=dev)
    out = torch.zeros(B, dtype=torch.int32, device=dev)
    one = torch.ones(B, dtype=torch.int32, device=dev)

    def step():
        mk.step_batch(toks, pos, out, None, stream)
        toks.copy_(out)
        pos.add_(one)

    for _ in range(W):
        step()
    torch.cuda.synchronize()
    if mk.status() != 0:
        raise SystemExit("megakernel status error in the batched warm-up")
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        a.record(stream)
        for _ in range(K):
            step()
        b.record(stream)
        torch.cuda.synchronize()
    if mk.status() != 0:
        raise SystemExit("megakernel status error in the batched steps")
    ms = a.elapsed_time(b) / K
    kv = shape.kv_read_bytes(P + W + K // 2 + 1, B)
    bytes_step = shape.step_weight_bytes() + kv
    achieved = bytes_step / (ms * 1e-3) / 1e9
    peak, peak_kind = measured_peak()
    line = {
        "metric": f"batch-{B} decode us/token ({shape.name} shape), one megakernel launch per step for all {B} "
                  "sequences",
        "value": 1e3 * ms / B, "unit": "us/token", "n_gpus": 1, "steps": K, "warmup": W,
        "ms_per_step": ms, "higher_is_better": False, "scaling": "weak", "vs_baseline": None,
        "dtype": "f16", "data": "synthetic",
        "config": {"workload": f"{wl.name}: {B} sequences, caches pre-filled to {P} positions, "
                               f"timed positions {P + W}..{P + W + K - 1}",
                   "arithmetic": "layer GEMVs on fp16 tensor-core inputs (exact fp16 copy of the bf16 weights, "
                                 "inputs rounded to fp16), fp32 accumulation; LM head on tcgen05 over the bf16 "
                                 "embedding with hi/lo bf16 inputs; attention and norms in fp32",
                   "l2": "weights (2.5 GB) far exceed the 129 MB L2"},
        "tokens_per_s": B * 1e3 / ms,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_source": peak_kind, "bytes_per_launch": bytes_step,
                     "traffic": None, "kernel": "whole step: mk_megakernel (batched) + final norm + "
                                                "tc_gemm LM head + draw"},
        # per step: the megakernel, the final norm, the LM-head contraction
        # and the draw's two kernels
        "gpu_launches": 5 * K,
        "clocks": clk.summary(),
    }
    if args.trace:
        from decode_megakernel_llama_gb300 import trace as mktrace
        mk.set_trace(True)
        step()
        torch.cuda.synchronize()
        rec = mk.read_trace()
        mk.set_trace(False)
        with open(args.trace, "w") as f:
            json.dump(mktrace.summarize(rec), f, indent=1)
        mktrace.to_chrome(rec, os.path.splitext(args.trace)[0] + ".chrome.json")
    print(json.dumps(line), flush=True)
    mk.close()


def run_mk(args, ws, rank, local):
    import torch
    import torch.distributed as dist

    from decode_megakernel_llama_gb300 import _lib, synth
    from decode_megakernel_llama_gb300.build import build
    from decode_megakernel_llama_gb300.configs import WORKLOADS

    if ws > 1 and not dist.is_initialized():
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if rank == 0 or ws == 1:
        build()
    if ws > 1:
        dist.barrier()
    wl = WORKLOADS[args.workload]
    shape = wl.shape
    K, W = args.steps, args.warmup
    P = wl.prompt_len
    P0 = wl.prefill + P  # first decode position after the (pre-filled) context and the prompt
    if W < 3:
        raise SystemExit("--warmup must be >= 3")
    max_seq = P0 + max(K, wl.decode_steps)
    w = synth.make_weights(shape, dev, 0)
    kc, vc = synth.kv_cache(shape, max_seq, 1, dev)
    if wl.prefill:
        synth.prefill_cache(kc, vc, wl.prefill)
    mk = _lib.Megakernel(shape, w, kc, vc)
    prompt = synth.prompt_tokens(shape.vocab, P)
    stream = torch.cuda.current_stream(dev)
    tok = torch.zeros(1, dtype=torch.int32, device=dev)
    logits = torch.empty(shape.vocab, dtype=torch.float32, device=dev)

    def run_prompt(step_fn):
        for i in range(P):
            step_fn(int(prompt[i]), wl.prefill + i)

    if args.profile:
        for s in range(W + K):
            mk.step(int(prompt[s % P]), s, tok, None, stream)
        torch.cuda.synchronize()
        print(json.dumps({"profile": True, "status": mk.status(), "launches": W + K}), flush=True)
        mk.close()
        return

    # prompt through the decode step (its last W steps are the warm-up)
    run_prompt(lambda t, i: mk.step(t, i, tok, None, stream))
    torch.cuda.synchronize()
    if mk.status() != 0:
        raise SystemExit("megakernel status error during the prompt")
    tok.fill_(int(prompt[-1]))

    # keep the clocks sampled under load around the timed region
    def timed_decode():
        start = torch.cuda.Event(enable_timing=True)
        end = torch.cuda.Event(enable_timing=True)
        if ws > 1:
            dist.barrier()
        torch.cuda.synchronize()
        start.record(stream)
        for s in range(K):
            mk.step_dev(tok, P0 + s, tok, None, stream)
        end.record(stream)
        torch.cuda.synchronize()
        return start.elapsed_time(end)  # ms

    with ClockSampler(local) as clk:
        t_end = time.time() + 1.0
        while time.time() < t_end:      # load the GPU before the timed region
            for s in range(W):
                mk.step_dev(tok, P0 + s, tok, None, stream)
            torch.cuda.synchronize()
        # W warm-up steps on the exact positions, then the timed K
        for s in range(W):
            mk.step_dev(tok, P0 + s, tok, None, stream)
        ms = timed_decode()
    if mk.status() != 0:
        raise SystemExit("megakernel status error during timing")
    t_max = max_over_ranks(ms, ws, dev)
    us_per_tok_launch = 1e3 * ms / K                  # this rank's per-launch average
    value = aggregate_us_per_token(t_max * 1e-3, K, ws)  # aggregate us per token

    # ---- end to end: the public call with host buffers (token H2D, token D2H)
    h_in = torch.zeros(1, dtype=torch.int32).pin_memory()
    h_out = torch.zeros(1, dtype=torch.int32).pin_memory()
    # the host side reads and writes the pinned words through numpy views (a
    # torch scalar index costs microseconds per access)
    v_in, v_out = h_in.numpy(), h_out.numpy()
    v_in[0] = int(prompt[-1])
    for s in range(W):
        mk.step_host(h_in, P0 + s, h_out, None, stream)
        v_in[0] = v_out[0]
    if ws > 1:
        dist.barrier()
    t0 = time.perf_counter()
    for s in range(K):
        mk.step_host(h_in, P0 + s, h_out, None, stream)
        v_in[0] = v_out[0]
    e2e_s = time.perf_counter() - t0
    e2e_val = aggregate_us_per_token(max_over_ranks(e2e_s, ws, dev), K, ws)

    # ---- the same decode loop with the sampling epilogue on (temperature 0.8)
    mk.set_sampling(0.8, 1234)
    for s in range(W):
        mk.step_dev(tok, P0 + s, tok, None, stream)
    sampled_us = 1e3 * timed_decode() / K
    # ... and with the top-k / top-p filter on the draw
    mk.set_sampling_filter(50, 0.9)
    for s in range(W):
        mk.step_dev(tok, P0 + s, tok, None, stream)
    filtered_us = 1e3 * timed_decode() / K
    mk.set_sampling_filter(0, 1.0)
    mk.set_sampling(0.0)
    if mk.status() != 0:
        raise SystemExit("megakernel status error with sampling")
    sampling_line = {"us_per_token": sampled_us, "temperature": 0.8,
                     "filtered_us_per_token": filtered_us, "top_k": 50, "top_p": 0.9,
                     "note": "Gumbel-max draw from softmax(logits/T), Philox4x32-10 noise per vocabulary entry; "
                             "filtered: the draw among the top_k best logits, cut to the shortest prefix whose "
                             "softmax mass reaches top_p"}

    # ---- comparators: the same kernels as an unfused chain (and as a graph)
    comp = None
    if not args.no_comparators:
        torch.cuda.synchronize()
        for s in range(W):
            mk.step_unfused(int(prompt[-1]), P0 + s, tok, None, stream)
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for s in range(K):
            mk.step_unfused(int(prompt[-1]), P0 + s, tok, None, stream)
        b.record(stream)
        torch.cuda.synchronize()
        unfused_us = 1e3 * a.elapsed_time(b) / K
        graph_us = None
        try:
            g = torch.cuda.CUDAGraph()
            cs = torch.cuda.Stream(dev)
            cs.wait_stream(stream)
            with torch.cuda.stream(cs):
                mk.step_unfused(int(prompt[-1]), P0, tok, None, cs)  # warm the capture stream
            torch.cuda.synchronize()
            with torch.cuda.graph(g, stream=cs):
                mk.step_unfused(int(prompt[-1]), P0, tok, None, cs)
            for _ in range(W):
                g.replay()
            torch.cuda.synchronize()
            a.record(stream)
            for _ in range(K):
                g.replay()
            b.record(stream)
            torch.cuda.synchronize()
            graph_us = 1e3 * a.elapsed_time(b) / K
        except Exception as e:  # capture support is a comparator, not the product
            graph_us = f"unavailable: {type(e).__name__}"
        if mk.status() != 0:
            raise SystemExit("status error in comparators")
        comp = {"unfused_chain_us_per_token": unfused_us,
                "unfused_chain_graph_us_per_token": graph_us,
                "unfused_launches_per_token": 5 * shape.n_layers + 1,
                "megakernel_speedup_vs_unfused": unfused_us / us_per_tok_launch}

    # ---- optional per-instruction trace of one step
    if args.trace:
        from decode_megakernel_llama_gb300 import trace as mktrace
        mk.set_trace(True)
        mk.step_dev(tok, P0 + K // 2, tok, None, stream)  # a position in the middle of the timed range
        torch.cuda.synchronize()
        rec = mk.read_trace()
        mk.set_trace(False)
        summ = mktrace.summarize(rec)
        with open(args.trace, "w") as f:
            json.dump(summ, f, indent=1)
        mktrace.to_chrome(rec, os.path.splitext(args.trace)[0] + ".chrome.json")

    # ---- multi-token prefill of the workload's prompt (tensor cores), the
    # contraction alone, and the W2A8 GEMV
    extras = None if args.no_extras or ws > 1 else measure_extras(mk, shape, prompt, P, W, dev, stream, us_per_tok_launch)

    # ---- roofline of the megakernel (the only kernel)
    mean_bytes = sum(algorithmic_bytes(shape, P0 + s) for s in range(K)) / K
    achieved = mean_bytes / (us_per_tok_launch * 1e-6) / 1e9
    peak, peak_kind = measured_peak()
    roof = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
            "frac": achieved / peak, "peak_source": peak_kind,
            "traffic": committed_traffic(), "bytes_per_launch": mean_bytes,
            "kernel": "mk_megakernel"}

    # ---- oracle on the host cores (rank 0 at N=1 only)
    cpu = None
    if rank == 0 and ws == 1 and args.cpu_seconds > 0 and not wl.prefill:
        cpu = oracle_baseline(shape, synth.host_weights(w), prompt, P0, K, args.cpu_seconds,
                              args.cpu_seconds)

    if rank == 0:
        line = {
            "metric": "batch-1 decode us/token (Llama-1B shape) and achieved HBM GB/s vs peak",
            "value": value, "unit": "us/token", "n_gpus": ws, "steps": K, "warmup": W,
            "ms_per_step": t_max / K, "higher_is_better": False, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": f"{wl.name}: {shape_desc(shape)}, batch 1, "
                                   + (f"KV cache pre-filled to {wl.prefill} positions, " if wl.prefill else "")
                                   + f"{wl.prompt_len}-token prompt, timed decode positions {P0}..{P0 + K - 1}",
                       "l2": l2_note(shape),
                       "parallelism": f"replicas x{ws}"},
            "tokens_per_s": 1e6 / value,
            "achieved_hbm_gbs": achieved,
            "roofline": roof,
            "e2e": {"value": e2e_val, "unit": "us/token", "h2d_bytes_per_step": 4,
                    "d2h_bytes_per_step": 4},
            "gpu_launches": K,
            "clocks": clk.summary(),
            "comparators": comp,
            "sampling": sampling_line,
            "prefill": extras.get("prefill") if extras else None,
            "w2a8_gemv": extras.get("w2a8_gemv") if extras else None,
            "twell_down": extras.get("twell_down") if extras else None,
            "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)
    mk.close()
    if ws > 1:
        dist.barrier()
        dist.destroy_process_group()


def main():
    args = parse()
    ws, rank, local = dist_env()
    from decode_megakernel_llama_gb300.configs import WORKLOADS
    if args.impl == "reference":
        run_reference(args, ws, rank)
    elif args.profile_gemm:
        run_profile_gemm(args)
    elif args.profile_prefill:
        run_profile_prefill(args)
    elif args.profile_twell:
        run_profile_twell(args)
    elif args.profile_w2a8:
        run_profile_w2a8(args)
    elif WORKLOADS[args.workload].batch > 1:
        run_batch(args, ws, rank, local)
    else:
        run_mk(args, ws, rank, local)


if __name__ == "__main__":
    main()
