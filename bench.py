#!/usr/bin/env python3
"""Benchmark of the MoE layer hot path on one B300.

Default workload: one full-size MoE layer (hidden 2816, 128 experts, top-8, expert
inter 704, shared inter 2112, 4-bit g64 experts, 8-bit g64 router), one decode
token per step, uniform router logits.  A step is one moe_layer_decode call
(router + top-8 + softmax gates, 8 routed experts and the shared expert with
GeGLU, gate-weighted combine).  Weights rotate over enough distinct copies of the
layer that no step finds its weights in L2.

The JSON line reports decode tokens/s (value), the HBM roofline fraction of the
layer kernel, the end-to-end rate through the public API with host buffers, the
oracle timed on the host cores, and side measurements (decode batch sweep with
Zipf(1.1) popularity, the 128-token prefill chunk).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

H, E, TOPK, I, IS = 2816, 128, 8, 704, 2112
EXPERT_BYTES = 3 * I * H * 36 // 64          # 3,345,408 B at 4.5 bit/weight
SHARED_BYTES = 3 * IS * H * 36 // 64         # 10,036,224 B
ROUTER_BYTES = E * H * 68 // 64              # 382,976 B at 8.5 bit/weight
DECODE_BYTES = TOPK * EXPERT_BYTES + SHARED_BYTES + ROUTER_BYTES  # 37,182,464 B per token

# DRAM traffic (read + write) of one decode launch at T = 1 from an ncu capture of
# `bench.py --quick` (dram__bytes_read.sum + dram__bytes_write.sum); reported only
# while the decode kernel's sources are the ones it was taken on (their SHA-1
# without comments)
DECODE_NCU_TRAFFIC = {"sha1": "7592a6f2f37b04b4e4046e9ce355b0291db78325", "bytes": 37_332_224}
DECODE_SOURCES = ["bit_affine_quantised_affine4_b300/csrc/" + f for f in
                  ("decode.cuh", "common.cuh", "mma_core.cuh", "route.cuh", "sync.cuh", "tile.cuh",
                   "moe_api.cu")] + ["include/moe.h"]


DECODE_API_END = "int run_layer_chunk("


def decode_sources_sha1():
    """SHA-1 of the decode kernel's sources with comments and blank space removed
    (a change of documentation does not change the kernel)."""
    import hashlib
    import re
    h = hashlib.sha1()
    for f in DECODE_SOURCES:
        with open(os.path.join(ROOT, f), encoding="utf-8") as fh:
            text = fh.read()
        # of the ABI implementation only the decode path: what precedes the prefill
        # and cache entry points (workspace binding, decode plan and launch)
        if f.endswith("moe_api.cu") and DECODE_API_END in text:
            text = text[:text.index(DECODE_API_END)]
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        h.update(" ".join(text.split()).encode())
    return h.hexdigest()


def decode_traffic():
    return DECODE_NCU_TRAFFIC["bytes"] if decode_sources_sha1() == DECODE_NCU_TRAFFIC["sha1"] else None


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "source": "measured"}
    return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "source": "fallback"}


# ---------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index=0):
        self.dev = device_index
        self.proc = None
        self.path = None

    def __enter__(self):
        try:
            import tempfile
            self.path = os.path.join(os.environ.get("MOE_BENCH_CLOCKS_DIR", tempfile.gettempdir()),
                                     "moe_bench_clocks_%d.csv" % os.getpid())
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"], stdout=self.fh,
                stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.fh.close()

    def summary(self):
        if not self.path or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            f = [v.strip() for v in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------- oracle (CPU) leg
def cpu_model():
    try:
        for line in open("/proc/cpuinfo"):
            if line.startswith("model name"):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


def _omp():
    """The OpenMP runtime the oracle library runs on (to set its thread count)."""
    import ctypes
    try:
        return ctypes.CDLL("libgomp.so.1")
    except OSError:
        return None


def oracle_decode_rate(seconds=15.0, max_tokens=64, single_tokens=3):
    """The oracle as it stands: full-size layer, one token per call, timed on the
    host cores over a bounded sample of tokens (each call timed on its own; the
    rate is 1 / median).  A single-thread figure comes from a few more calls with
    the OpenMP runtime set to one thread."""
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    from layers import OracleLayer  # test-side builder around the oracle
    s = synth.FULL
    ol = OracleLayer(s, seed=0)
    n_all = max_tokens + single_tokens
    x = synth.tokens(s, n_all, seed=0, stream=9000)
    # route everything first so expert quantisation (data preparation) is untimed
    for t in range(n_all):
        _, idx, _ = ol.route(x[t:t + 1])
        for e in np.unique(idx):
            ol.expert(int(e))
    omp = _omp()
    cores = omp.omp_get_max_threads() if omp else int(os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1))
    times = []
    t0 = time.perf_counter()
    while len(times) < max_tokens and (len(times) < 3 or time.perf_counter() - t0 < seconds):
        t1 = time.perf_counter()
        ol.layer(x[len(times):len(times) + 1])
        times.append(time.perf_counter() - t1)
    single = None
    if omp:
        omp.omp_set_num_threads(1)
        st = []
        for t in range(single_tokens):
            t1 = time.perf_counter()
            ol.layer(x[max_tokens + t:max_tokens + t + 1])
            st.append(time.perf_counter() - t1)
        omp.omp_set_num_threads(cores)
        single = 1.0 / statistics.median(st)
    med = statistics.median(times)
    return {"value": 1.0 / med, "unit": "tok/s", "cores": cores, "kind": "oracle",
            "cpu_model": cpu_model(), "single_thread_tok_s": single,
            "sample": "%d decode tokens of the full-size layer (uniform routing), each timed alone, "
                      "rate = 1 / median (%.1f ms); single thread: median of %d more tokens"
                      % (len(times), med * 1e3, single_tokens)}


# ---------------------------------------------------------------- GPU leg
def build_layer(moe, copies, bias=None):
    s = synth.FULL
    return moe.make_layer(s.H, s.E, s.topk, s.I, s.Is, synth.router_weights(s, 0),
                          lambda e: synth.expert_weights(s, e, 0), synth.shared_weights(s, 0),
                          bias=bias, copies=copies)


def ranks_barrier(torch):
    """Barrier over the ranks of the process group (no-op without one)."""
    import torch.distributed as td
    if td.is_available() and td.is_initialized():
        td.barrier()


def max_over_ranks(torch, value, device="cpu"):
    """The largest of every rank's value (the value itself without a process group)."""
    import torch.distributed as td
    if not (td.is_available() and td.is_initialized()):
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    td.all_reduce(t, op=td.ReduceOp.MAX)
    return float(t.item())


def job_rate(world, steps, seconds):
    """Whole-job throughput: every rank processes `steps` units in at most `seconds`."""
    return world * steps / seconds


def time_graph(torch, fn_steps, K, W):
    """Capture K steps (and W warm-up steps) as CUDA graphs; time the K-step replay
    with CUDA events on the capturing stream, between barriers over the ranks."""
    st = torch.cuda.Stream()
    torch.cuda.synchronize()
    gW, gK = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
    with torch.cuda.stream(st):
        fn_steps(W, 0)  # eager warm-up (also loads the module on the device)
    torch.cuda.synchronize()
    with torch.cuda.graph(gW, stream=st):
        fn_steps(W, 0)
    with torch.cuda.graph(gK, stream=st):
        fn_steps(K, W)
    with torch.cuda.stream(st):
        gW.replay()
        gK.replay()  # untimed replay: uploads the timed graph
    torch.cuda.synchronize()
    ranks_barrier(torch)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(st):
        ev0.record(st)
        gK.replay()
        ev1.record(st)
    ev1.synchronize()
    torch.cuda.synchronize()
    ranks_barrier(torch)
    return ev0.elapsed_time(ev1) / 1e3


def run_ours(args):
    import torch
    import bit_affine_quantised_affine4_b300 as moe

    dist = args.gpus > 1
    rank, world = 0, 1
    if dist:
        import torch.distributed as td
        td.init_process_group("nccl")
        rank, world = td.get_rank(), td.get_world_size()
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", rank)))
    dev = torch.device("cuda")
    peaks = load_peaks()
    props = torch.cuda.get_device_properties(dev)
    l2 = getattr(props, "L2_cache_size", 126 * 2**20)

    # enough distinct layer copies that a step never finds its weights in L2
    copies = args.copies or max(4, int(np.ceil(4 * l2 / DECODE_BYTES)))
    layer = build_layer(moe, copies)
    views = [layer.view(c) for c in range(copies)]
    NX = 64
    X = torch.from_numpy(synth.tokens(synth.FULL, NX, seed=0, stream=rank)).to(dev)
    Y = torch.empty((NX, H), device=dev)
    ws = moe.new_workspace(views[0], moe.MOE_MAX_PREFILL_TOKENS)
    torch.cuda.synchronize()

    def decode_steps(n, first):
        for i in range(first, first + n):
            moe.moe_layer_decode(views[i % copies], X[i % NX:i % NX + 1], ws, y=Y[i % NX:i % NX + 1])

    # ---- headline: decode T=1, CUDA-graph replay, clocks sampled during it
    with ClockSampler(torch.cuda.current_device()) as clk:
        dt = time_graph(torch, decode_steps, args.steps, args.warmup)
    clocks = clk.summary()
    dt = max_over_ranks(torch, dt, dev)
    per_step = dt / args.steps
    value = job_rate(world, args.steps, dt)  # tokens/s over all ranks (one token per step per rank)
    achieved_gbs = DECODE_BYTES / per_step / 1e9

    # ---- end to end through the public API with host buffers: one call per step
    # copies the token in (pinned host memory), runs the decode, copies y back and
    # returns once it is there -- through the prepared host call (moe_host_call,
    # a recorded graph per layer) and, for comparison, moe_layer_decode_host
    xh = torch.from_numpy(synth.tokens(synth.FULL, NX, seed=0, stream=rank)).pin_memory()
    yh = torch.empty((NX, H)).pin_memory()
    st = torch.cuda.Stream()
    xrows = [xh[i:i + 1] for i in range(NX)]  # a caller's per-token host buffers
    yrows = [yh[i:i + 1] for i in range(NX)]

    prepared = [moe.HostCall(v, ws, T=1, stream=st) for v in views]  # one per layer copy
    unprepared = [moe.DecodeHostCall(v, ws, stream=st) for v in views]  # arguments marshalled once per layer

    def e2e_time(calls):
        def e2e_steps(n, first):
            for i in range(first, first + n):
                calls[i % copies](xrows[i % NX], yrows[i % NX])

        e2e_steps(args.warmup, 0)
        torch.cuda.synchronize()
        passes = []
        for _ in range(3):  # the host-bound call varies with the host: the median of three passes of K steps
            ranks_barrier(torch)
            t0 = time.perf_counter()
            e2e_steps(args.steps, args.warmup)
            torch.cuda.synchronize()
            passes.append(time.perf_counter() - t0)
        ranks_barrier(torch)
        return max_over_ranks(torch, statistics.median(passes), dev)

    e2e_dt = e2e_time(prepared)
    e2e_host_dt = e2e_time(unprepared)
    for c in prepared:
        c.close()

    extra = {}
    if not args.quick and rank == 0:
        extra = side_measurements(torch, moe, layer, copies, ws, args)
    if not args.quick and rank == 0:
        extra["attention_block"] = attention_measurement(torch, moe, args, peaks)
        extra["qgemv_affine4"] = qgemv_measurement(torch, moe, args, peaks)
        extra["sampling_and_rmsnorm"] = sample_norm_measurement(torch, moe, args, peaks)
    if args.stack and rank == 0:
        del layer, views
        torch.cuda.empty_cache()
        stack_layers = build_stack_layers(torch, moe)
        extra["stack_decode_attention"] = stack_attn_measurement(torch, moe, args, stack_layers)
        extra["stack_decode_lfu"] = stack_measurement(torch, moe, args, layers=stack_layers)
        del stack_layers

    line = {
        "metric": "MoE decode tokens/s (one full-size layer, T=1) and % of B300 HBM roofline; prefill-chunk tok/s",
        "value": value, "unit": "tok/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": per_step * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": "u4 weights (affine g64, fp16 scale/bias), u8 router; fp16 activations (x, h) "
                 "as tensor-core operands, f32 accumulate",
        "data": "synthetic: weights N(0,0.02) quantised 4-bit g64 (router 8-bit g64), tokens N(0,1), seed 0",
        "config": {"workload": "moe_layer_decode, hidden 2816, 128 experts top-8, inter 704, shared 2112, "
                               "GeGLU, T=1, uniform router logits",
                   "algorithmic_bytes_per_step": DECODE_BYTES,
                   "l2": "weights rotate over %d distinct layer copies (%.1f GB) > L2 (%d MB)"
                         % (copies, copies * (E * EXPERT_BYTES + SHARED_BYTES + ROUTER_BYTES) / 1e9, l2 >> 20),
                   "timing": "CUDA graph of K steps, CUDA events on the capturing stream; "
                             "warm-up = W steps + one untimed replay of the timed graph",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "roofline": {"bound": "hbm", "achieved": achieved_gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": achieved_gbs / peaks["hbm_gbs"], "traffic": decode_traffic(),
                     "peak_source": peaks["source"], "kernel": "moe_layer_decode (whole call)"},
        "e2e": {"value": job_rate(world, args.steps, e2e_dt), "unit": "tok/s",
                "h2d_bytes_per_step": H * 4, "d2h_bytes_per_step": H * 4,
                "note": "moe_host_call_run through the Python binding (HostCall, one prepared handle per "
                        "layer copy), one call per step on pinned host rows: x copied into the handle's "
                        "mapped staging row and read by the device, the step's recorded graph launched, "
                        "y written by the decode kernel into the mapped row and copied out once the "
                        "completion word arrives; median of three passes of K steps",
                "moe_layer_decode_host": {"value": job_rate(world, args.steps, e2e_host_dt), "unit": "tok/s",
                                          "note": "the unprepared host-buffer call (DecodeHostCall): mapped "
                                                  "rows, two launches and a stream poll per step"}},
        "gpu_launches": args.steps,  # one persistent k_decode launch per step
        "clocks": clocks,
    }
    line.update(extra)
    if rank == 0 and not args.no_cpu:
        line["cpu_baseline"] = oracle_decode_rate(seconds=args.cpu_seconds)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()


def unique_experts(idx, written):
    """Mean number of distinct experts per step over the routing rows the steps
    wrote (row i % NX for steps i = 0 .. written - 1; the others were never run)."""
    rows = idx[:min(idx.shape[0], written)].cpu().numpy()
    assert (rows >= 0).all(), "a routing row the steps should have written is unset"
    return float(np.mean([len(np.unique(r)) for r in rows]))


def side_measurements(torch, moe, layer, copies, ws, args):
    """Decode batch sweep and the 128-token prefill chunk, both with Zipf(1.1)
    popularity (router logit bias), timed the same way as the headline."""
    s = synth.FULL
    layer.set_bias(synth.popularity_bias(s, seed=0))
    views = [layer.view(c) for c in range(copies)]
    dev = layer.device
    out = {}
    sweep = []
    for T in (1, 2, 4, 8, 16):
        NX = 32
        X = torch.from_numpy(synth.tokens(s, NX * T, seed=0, stream=1000 + T)).to(dev).view(NX, T, H)
        Y = torch.empty_like(X)
        idx = torch.full((NX, T, TOPK), -1, dtype=torch.int32, device=dev)

        def steps(n, first):
            for i in range(first, first + n):
                moe.moe_layer_decode(views[i % copies], X[i % NX], ws, y=Y[i % NX], idx=idx[i % NX])

        K = max(20, args.steps // 4)
        dt = time_graph(torch, steps, K, args.warmup)
        U = unique_experts(idx, args.warmup + K)
        bytes_step = U * EXPERT_BYTES + SHARED_BYTES + ROUTER_BYTES
        sweep.append({"T": T, "tok_s": K * T / dt, "us_per_step": dt / K * 1e6, "unique_experts": U,
                      "GB_s": bytes_step / (dt / K) / 1e9})
    out["decode_batch_zipf"] = sweep
    # prefill chunk of 128 tokens
    T = 128
    NX = 4
    X = torch.from_numpy(synth.tokens(s, NX * T, seed=0, stream=2000)).to(dev).view(NX, T, H)
    Y = torch.empty_like(X)
    idx = torch.full((NX, T, TOPK), -1, dtype=torch.int32, device=dev)

    def psteps(n, first):
        for i in range(first, first + n):
            moe.moe_layer_prefill_chunk(views[i % copies], X[i % NX], ws, y=Y[i % NX], idx=idx[i % NX])

    K = 10
    dt = time_graph(torch, psteps, K, args.warmup)
    U = unique_experts(idx, args.warmup + K)
    bytes_step = U * EXPERT_BYTES + SHARED_BYTES + ROUTER_BYTES
    flops = 2 * T * (TOPK * 3 * I * H + 3 * IS * H + E * H)
    out["prefill_chunk_zipf"] = {"T": T, "tok_s": K * T / dt, "us_per_chunk": dt / K * 1e6,
                                 "unique_experts": U, "GB_s": bytes_step / (dt / K) / 1e9,
                                 "TFLOP_s": flops / (dt / K) / 1e12}
    layer.set_bias(None)
    return out


ATTN_SLIDING, ATTN_GLOBAL = synth.ATTN_FULL_SLIDING, synth.ATTN_FULL_GLOBAL


def attn_weight_bytes(a):
    """4-bit weights (4.5 bits with scale and bias) of one attention block."""
    return (a.n_qkv * a.H + a.H * a.nq * a.d) * 9 // 16


def attn_call_bytes(a, attended):
    """Algorithmic bytes of one T = 1 attention call that attends to `attended`
    positions: the weights, the binary16 keys and values read, the new key and value
    written, x read and y written."""
    return attn_weight_bytes(a) + 2 * a.nkv * attended * a.d * 2 + 2 * a.nkv * a.d * 2 + 2 * a.H * 4


def new_attn_layer(torch, moe, a, gen, dev):
    L = moe.AttnLayer(a.H, a.nq, a.nkv, a.d, a.window, a.kv_len, a.theta, device=dev)
    L.set_weights(torch.randn(a.n_qkv, a.H, generator=gen, device=dev) * 0.02,
                  torch.randn(a.H, a.nq * a.d, generator=gen, device=dev) * 0.02)
    L.set_cache(torch.randn(a.nkv, a.kv_len, a.d, generator=gen, device=dev).half().view(torch.int16),
                torch.randn(a.nkv, a.kv_len, a.d, generator=gen, device=dev).half().view(torch.int16))
    L.set_norm(1.0 + 0.1 * torch.randn(a.H, generator=gen, device=dev), 1e-6)
    return L


def attention_measurement(torch, moe, args, peaks):
    """One attention block (pre-norm, residual), T = 1, for a sliding-window layer
    (window 1024, ring of 1151) and a full layer (store of 4096, at its last
    position), rotating over enough layer copies that weights and caches do not
    fit in L2; CUDA-graph replay timed with events."""
    dev = torch.device("cuda")
    gen = torch.Generator(device=dev)
    gen.manual_seed(1)
    out = {}
    for a, pos, attended in ((ATTN_SLIDING, 5000, ATTN_SLIDING.window), (ATTN_GLOBAL, ATTN_GLOBAL.kv_len - 1,
                                                                         ATTN_GLOBAL.kv_len)):
        per = attn_weight_bytes(a) + 2 * a.nkv * a.kv_len * a.d * 2
        copies = max(4, int(np.ceil(3 * (128 << 20) / per)))
        layers = [new_attn_layer(torch, moe, a, gen, dev) for _ in range(copies)]
        views = [l.view() for l in layers]
        ws = moe.new_attn_workspace(views[0], 1)
        x = torch.randn(1, a.H, generator=gen, device=dev)
        y = torch.empty_like(x)

        def steps(n, first):
            for i in range(first, first + n):
                moe.moe_attn_step(views[i % copies], x, ws, pos, y=y, flags=moe.MOE_RESIDUAL | moe.MOE_PRENORM)

        K = max(40, args.steps // 2)
        dt = time_graph(torch, steps, K, args.warmup)
        status = moe.moe_attn_workspace_status(ws)
        b = attn_call_bytes(a, attended)
        gbs = b / (dt / K) / 1e9
        out[a.name] = {"us_per_call": dt / K * 1e6, "attended_positions": attended, "algorithmic_bytes": b,
                       "GB_s": gbs, "frac_of_hbm": gbs / peaks["hbm_gbs"], "layer_copies": copies,
                       "status": moe.status_string(status)}
        del layers, views, ws
        torch.cuda.empty_cache()
    out["shape"] = ("hidden 2816, 16 query heads and 8 key/value heads of 256, 4-bit Wqkv [8192 x 2816] and "
                    "Wo [2816 x 4096], binary16 cache; three kernels per call (QKV + RoPE + cache store, "
                    "attention, output projection + residual) with programmatic dependent launch")
    return out


def qgemv_measurement(torch, moe, args, peaks):
    """qgemv_affine4 alone, one token: the attention block's two matrix shapes
    ([8192 x 2816] and [2816 x 4096]), rotating over copies whose total exceeds L2;
    CUDA-graph replay timed with events.  Bytes: the 4-bit weights at 4.5 bits plus
    x and y."""
    dev = torch.device("cuda")
    gen = torch.Generator(device=dev)
    gen.manual_seed(3)
    out = {}
    for N, K in ((8192, 2816), (2816, 4096)):
        wbytes = N * K * 9 // 16
        copies = max(4, int(np.ceil(3 * (128 << 20) / wbytes)))
        mats = [moe.affine_quantise(torch.randn(N, K, generator=gen, device=dev) * 0.02, 4) for _ in range(copies)]
        x = torch.randn(K, generator=gen, device=dev)
        y = torch.empty(N, device=dev)

        def steps(n, first):
            for i in range(first, first + n):
                q, sc, b = mats[i % copies]
                moe.qgemv_affine4(q, sc, b, K, x, y=y)

        K_steps = max(40, args.steps // 2)
        dt = time_graph(torch, steps, K_steps, args.warmup)
        b = wbytes + K * 4 + N * 4
        gbs = b / (dt / K_steps) / 1e9
        out["%dx%d" % (N, K)] = {"us_per_call": dt / K_steps * 1e6, "algorithmic_bytes": b, "GB_s": gbs,
                                 "frac_of_hbm": gbs / peaks["hbm_gbs"], "copies": copies}
        del mats
        torch.cuda.empty_cache()
    return out


def sample_norm_measurement(torch, moe, args, peaks):
    """Token sampling (the engine's defaults: temperature 0.2, top-K 64, top-P 0.95)
    over a 262,144-entry vocabulary for 1 and 16 rows, and RMSNorm of 1 and 16
    rows of 2816, rotating over inputs larger than L2; CUDA-graph replay timed with
    events.  Bytes: logits read (sampling), x read + y written + the gain (RMSNorm)."""
    dev = torch.device("cuda")
    gen = torch.Generator(device=dev)
    gen.manual_seed(4)
    out = {}
    V = 262144
    for T in (1, 16):
        n = max(4, int(np.ceil(3 * (128 << 20) / (T * V * 4))))
        logits = [torch.randn(T, V, generator=gen, device=dev) * 3.0 for _ in range(n)]
        u = torch.rand(T, generator=gen, device=dev)
        tok = torch.empty(T, dtype=torch.int32, device=dev)

        def steps(k, first):
            for i in range(first, first + k):
                moe.moe_sample(logits[i % n], 0.2, 64, 0.95, u, tokens=tok)

        K = max(40, args.steps // 2)
        dt = time_graph(torch, steps, K, args.warmup)
        gbs = T * V * 4 / (dt / K) / 1e9
        out["sample_V262144_T%d" % T] = {"us_per_call": dt / K * 1e6, "GB_s": gbs,
                                         "frac_of_hbm": gbs / peaks["hbm_gbs"]}
        del logits
    w = 1.0 + 0.1 * torch.randn(H, generator=gen, device=dev)
    for T in (1, 16):
        n = max(4, int(np.ceil(3 * (128 << 20) / (T * H * 8))))
        xs = [torch.randn(T, H, generator=gen, device=dev) for _ in range(n)]
        ys = [torch.empty(T, H, device=dev) for _ in range(n)]

        def nsteps(k, first):
            for i in range(first, first + k):
                moe.moe_rmsnorm(xs[i % n], w, 1e-6, y=ys[i % n])

        K = max(40, args.steps // 2)
        dt = time_graph(torch, nsteps, K, args.warmup)
        b = 2 * T * H * 4 + H * 4
        out["rmsnorm_H2816_T%d" % T] = {"us_per_call": dt / K * 1e6, "GB_s": b / (dt / K) / 1e9}
        del xs, ys
    torch.cuda.empty_cache()
    return out


def build_stack_layers(torch, moe, n_layers=30):
    """The 30 MoE layers of the decode stacks, experts resident on the device: router,
    experts and shared expert from the GPU's seeded normal generator (N(0, 0.02)),
    quantised and tiled by the library; Zipf(1.1) logit bias per layer; RMSNorm
    weights 1 + N(0, 0.1^2)."""
    s = synth.FULL
    dev = torch.device("cuda")
    gen = torch.Generator(device=dev)
    gen.manual_seed(0)
    layers = []
    for l in range(n_layers):
        L = moe.Layer(H, E, TOPK, I, IS, device=dev, copies=1)
        L.set_router(torch.randn(E, H, generator=gen, device=dev) * 0.02)
        for e in range(E):
            L.set_expert(e, torch.randn(2 * I, H, generator=gen, device=dev) * 0.02,
                         torch.randn(H, I, generator=gen, device=dev) * 0.02)
        L.set_shared(torch.randn(2 * IS, H, generator=gen, device=dev) * 0.02,
                     torch.randn(H, IS, generator=gen, device=dev) * 0.02)
        L.set_bias(synth.popularity_bias(s, seed=0, layer=l))
        L.set_norm(1.0 + 0.1 * torch.randn(H, generator=gen, device=dev), 1e-6)
        layers.append(L)
    torch.cuda.synchronize()
    return layers


def stack_attn_measurement(torch, moe, args, layers, steps=64):
    """The 30-layer decode step with attention: per layer the pre-norm attention
    block h <- h + Attn(RMSNorm(h)) over a binary16 key/value cache, then the
    pre-norm MoE block h <- h + MoE(RMSNorm(h)) with every expert resident.  Layers
    6, 12, ..., 30 attend to the whole context (a linear store of 4096), the other 25
    to a window of 1024 (a ring of 1151).  The context holds 4096 - 64 synthetic
    tokens when the 64 timed steps start.  Each step is 30 x (3 attention kernels +
    1 MoE decode kernel), replayed from a CUDA graph; the same steps are also
    timed with the attention blocks alone and the MoE blocks alone."""
    dev = torch.device("cuda")
    gen = torch.Generator(device=dev)
    gen.manual_seed(2)
    n_layers = len(layers)
    attn = [new_attn_layer(torch, moe, ATTN_GLOBAL if l % 6 == 5 else ATTN_SLIDING, gen, dev) for l in range(n_layers)]
    aviews = [a.view() for a in attn]
    mviews = [L.view() for L in layers]
    # one workspace for both layer kinds: the larger of their sizes
    big = max((aviews[0], aviews[n_layers // 6 * 6 - 1]), key=lambda v: moe.moe_attn_workspace_bytes(v, 1))
    aws = moe.new_attn_workspace(big, 1)
    mws = moe.new_workspace(mviews[0], 1)
    X = torch.from_numpy(synth.token_sequence(synth.FULL, steps, seed=0)).to(dev)
    ha = torch.empty((1, H), device=dev)
    hb = [torch.empty((1, H), device=dev), torch.empty((1, H), device=dev)]  # the decode's y must not alias x
    pos0 = ATTN_GLOBAL.kv_len - steps
    flags = moe.MOE_RESIDUAL | moe.MOE_PRENORM

    def run(which):
        def fn(n, first):
            for st in range(first, first + n):
                cur = X[st % steps:st % steps + 1]
                for l in range(n_layers):
                    if which != "moe":
                        moe.moe_attn_step(aviews[l], cur, aws, pos0 + st % steps, y=ha, flags=flags)
                        cur = ha
                    if which != "attn":
                        moe.moe_layer_decode(mviews[l], cur, mws, y=hb[l & 1], flags=flags)
                        cur = hb[l & 1]
        return fn

    res = {}
    for which in ("both", "attn", "moe"):
        dt = time_graph(torch, run(which), steps, 2)
        res[which] = dt / steps
    status = moe.moe_attn_workspace_status(aws)
    attended = sum((ATTN_GLOBAL.kv_len - steps // 2) if l % 6 == 5 else ATTN_SLIDING.window for l in range(n_layers))
    attn_bytes = sum(attn_weight_bytes(ATTN_GLOBAL if l % 6 == 5 else ATTN_SLIDING) for l in range(n_layers)) + \
        2 * ATTN_SLIDING.nkv * attended * ATTN_SLIDING.d * 2
    moe_bytes = n_layers * DECODE_BYTES
    out = {"layers": n_layers, "full_attention_layers": n_layers // 6, "context": ATTN_GLOBAL.kv_len,
           "steps_timed": steps, "tok_s": 1.0 / res["both"], "ms_per_token": res["both"] * 1e3,
           "attention_only_ms": res["attn"] * 1e3, "moe_only_ms": res["moe"] * 1e3,
           "bytes_per_token": attn_bytes + moe_bytes,
           "GB_s": (attn_bytes + moe_bytes) / res["both"] / 1e9, "attn_status": moe.status_string(status),
           "note": "experts resident; the routing follows Zipf(1.1) with an AR(1) token sequence; "
                   "bytes: 4-bit weights at 4.5 bits + binary16 keys/values attended (mean context of the "
                   "timed steps for the full layers)"}
    del attn, aviews, aws
    torch.cuda.empty_cache()
    return out


def stack_measurement(torch, moe, args, layers=None, n_layers=30, steps=256, slots=16):
    """30-layer MoE stack decode (MoE part only: attention is the identity), one
    token per step, experts in page-locked host memory behind a 16-slot LFU cache
    per layer.  Each layer is the pre-norm block h <- h + MoE(RMSNorm(h)) (without
    the norm the residual stream grows layer over layer).  Routing follows Zipf(1.1)
    popularity (a per-layer logit bias) and the step inputs are an AR(1) sequence
    (rho 0.9), so consecutive steps route alike.  `layers`: the resident layers of
    build_stack_layers, whose experts move to host memory here."""
    s = synth.FULL
    dev = torch.device("cuda")
    blob = moe.moe_tile_blob_bytes(H, I)
    if layers is None:
        layers = build_stack_layers(torch, moe, n_layers)
    n_layers = len(layers)
    hosts, caches, views = [], [], []
    n_host = 0
    for l, L in enumerate(layers):
        try:
            host = torch.empty((E, blob), dtype=torch.uint8).pin_memory()
            host.copy_(L.experts[0])
            n_host += 1
        except RuntimeError:
            host = hosts[l % max(n_host, 1)]  # host memory ran short: reuse a layer's experts
        L.experts = None
        hosts.append(host)
        views.append(L.view(experts=False))
        caches.append(moe.Cache(H, E, I, host, slots=slots))
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    X = torch.from_numpy(synth.token_sequence(s, steps, seed=0)).to(dev)
    h = [torch.empty((1, H), device=dev), torch.empty((1, H), device=dev)]
    ws = moe.new_workspace(views[0], 1)
    warm = 8

    def run(first, n):
        for st in range(first, first + n):
            cur = X[st:st + 1]
            for l in range(n_layers):
                moe.moe_layer_decode(views[l], cur, ws, y=h[l & 1], flags=moe.MOE_RESIDUAL | moe.MOE_PRENORM,
                                     cache=caches[l])
                cur = h[l & 1]

    def timed(first, n, fn=None):
        torch.cuda.synchronize()
        st0 = [c.stats() for c in caches]
        t0 = time.perf_counter()
        (fn or run)(first, n)
        torch.cuda.synchronize()
        dt = time.perf_counter() - t0
        st1 = [c.stats() for c in caches]
        hits = sum(b[0] - a[0] for a, b in zip(st0, st1))
        misses = sum(b[1] - a[1] for a, b in zip(st0, st1))
        h2d = sum(b[2] - a[2] for a, b in zip(st0, st1))
        return {"steps_timed": n, "tok_s": n / dt, "ms_per_token": dt / n * 1e3,
                "hit_rate": hits / max(hits + misses, 1), "misses_per_token": misses / n,
                "h2d_GB_s": h2d / dt / 1e9}

    # a third of the sequence with the host policy, a third with the policy on the
    # device, the last third with the device policy replayed from a CUDA graph (a
    # layer call then needs no host involvement at all); all on warm caches
    third = (steps - warm) // 3
    run(0, warm)
    host = timed(warm, third)
    for c in caches:
        c.set_device_policy(True)
    device = timed(warm + third, third)
    first = warm + 2 * third
    st = torch.cuda.Stream()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=st):
        run(first, third)

    def replay(first_, n_):
        with torch.cuda.stream(st):
            g.replay()

    graph = timed(first, third, replay)
    out = {"layers": n_layers, "slots_per_layer": slots, "host_layers_distinct": n_host,
           "device_bytes_per_token": n_layers * DECODE_BYTES}
    out.update(graph)
    out["policy"] = "device, CUDA graph of the steps"
    out["device_policy_eager"] = device
    out["host_policy"] = host
    out["note"] = ("pre-norm blocks h + MoE(RMSNorm(h)).  Device policy: per layer the router's ranking CTA "
                   "runs the LFU step on device state, a kernel copies the misses from the mapped host "
                   "blobs, the decode reads the slot map on the device: no host round trip.  Host policy: "
                   "the router writes the routing into mapped host memory, the host polls a flag, runs "
                   "the policy and copies the misses on a side stream while the shared expert runs")
    out["h2d_link_probe_GB_s"] = h2d_link_probe(torch, caches[0].host_experts)
    out["h2d_link_use"] = out["h2d_GB_s"] / max(out["h2d_link_probe_GB_s"]["expert_copies"], 1e-9)
    for c in caches:
        c.close()
    return out


def h2d_link_probe(torch, host):
    """Host -> device copy rate of this box's link, measured here: back-to-back
    cudaMemcpyAsync copies from page-locked memory, (a) of one expert blob at a time
    (what a cache miss copies), (b) of 64 MB at a time."""
    blob = host.shape[1]
    st = torch.cuda.Stream()
    res = {}
    for name, nbytes, reps in (("expert_copies", blob, 32), ("copies_64MB", 64 << 20, 8)):
        src = host.view(-1)[:min(nbytes, host.numel())] if nbytes <= host.numel() else None
        if src is None:
            big = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
            src = big
        dst = torch.empty(src.numel(), dtype=torch.uint8, device="cuda")
        with torch.cuda.stream(st):
            for _ in range(2):
                dst.copy_(src, non_blocking=True)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(st)
            for _ in range(reps):
                dst.copy_(src, non_blocking=True)
            e1.record(st)
        e1.synchronize()
        res[name] = src.numel() * reps / (e0.elapsed_time(e1) * 1e-3) / 1e9
    return res


def run_prefill_only(args):
    """The 128-token prefill chunk of one full-size layer with Zipf(1.1) routing,
    run K times after W warm-ups (a short, single-layer case for profilers)."""
    import torch
    import bit_affine_quantised_affine4_b300 as moe
    s = synth.FULL
    layer = build_layer(moe, 1, bias=synth.popularity_bias(s, seed=0))
    view = layer.view()
    x = torch.from_numpy(synth.tokens(s, 128, seed=0, stream=2000)).cuda()
    ws = moe.new_workspace(view, 128)
    for _ in range(args.warmup):
        moe.moe_layer_prefill_chunk(view, x, ws)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        moe.moe_layer_prefill_chunk(view, x, ws)
    e1.record()
    e1.synchronize()
    us = e0.elapsed_time(e1) * 1000 / args.steps
    print(json.dumps({"workload": "prefill chunk, 128 tokens, full-size layer, Zipf(1.1)",
                      "us_per_chunk": us, "tok_s": 128e6 / us, "note": "single layer, weights may sit in L2"}))


def run_decode_only(args):
    """Decode steps of T tokens on the full-size layer with Zipf(1.1) routing,
    rotating over 2 layer copies, K times after W warm-ups (a short case for
    profilers: the batch sweep's configuration at one T)."""
    import torch
    import bit_affine_quantised_affine4_b300 as moe
    s, T = synth.FULL, args.decode_only
    layer = build_layer(moe, 2, bias=synth.popularity_bias(s, seed=0))
    views = [layer.view(c) for c in range(2)]
    x = torch.from_numpy(synth.tokens(s, T, seed=0, stream=3000 + T)).cuda()
    ws = moe.new_workspace(views[0], T)
    for i in range(args.warmup):
        moe.moe_layer_decode(views[i % 2], x, ws)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for i in range(args.steps):
        moe.moe_layer_decode(views[i % 2], x, ws)
    e1.record()
    e1.synchronize()
    us = e0.elapsed_time(e1) * 1000 / args.steps
    print(json.dumps({"workload": "decode, %d tokens, full-size layer, Zipf(1.1)" % T, "us_per_step": us,
                      "note": "eager launches, 2 layer copies (weights may sit in L2)"}))


def run_attention_only(args):
    """Attention blocks alone (T = 1, pre-norm, residual) on the sliding-window shape
    (window 1024, ring 1151) or the full shape (store of 4096, last position),
    rotating over 2 layers, K times after W warm-ups (a short case for profilers)."""
    import torch
    import bit_affine_quantised_affine4_b300 as moe
    a = ATTN_GLOBAL if args.attention_only == "global" else ATTN_SLIDING
    pos = a.kv_len - 1 if a.window == 0 else 5000
    dev = torch.device("cuda")
    gen = torch.Generator(device=dev)
    gen.manual_seed(1)
    layers = [new_attn_layer(torch, moe, a, gen, dev) for _ in range(2)]
    views = [l.view() for l in layers]
    ws = moe.new_attn_workspace(views[0], 1)
    x = torch.randn(1, a.H, generator=gen, device=dev)
    y = torch.empty_like(x)
    flags = moe.MOE_RESIDUAL | moe.MOE_PRENORM
    for i in range(args.warmup):
        moe.moe_attn_step(views[i % 2], x, ws, pos, y=y, flags=flags)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for i in range(args.steps):
        moe.moe_attn_step(views[i % 2], x, ws, pos, y=y, flags=flags)
    e1.record()
    e1.synchronize()
    status = moe.moe_attn_workspace_status(ws)
    print(json.dumps({"workload": "attention block, T=1, %s" % a.name, "us_per_call": e0.elapsed_time(e1) * 1000 /
                      args.steps, "status": moe.status_string(status),
                      "note": "eager launches, 2 layers (weights and caches may sit in L2)"}))


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    cb = oracle_decode_rate(seconds=args.cpu_seconds)
    line = {
        "impl": "reference",
        "metric": "MoE decode tokens/s (one full-size layer, T=1) and % of B300 HBM roofline; prefill-chunk tok/s",
        "value": cb["value"], "unit": "tok/s", "n_gpus": args.gpus, "steps": args.steps,
        "warmup": args.warmup, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic, seed 0",
        "config": {"workload": "moe_layer_decode, hidden 2816, 128 experts top-8, inter 704, shared 2112, "
                               "GeGLU, T=1, uniform router logits"},
        "cpu_baseline": cb,
        "e2e": {"value": cb["value"], "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "note": "the plain CPU oracle (no reference implementation exists for this hardware)",
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--quick", action="store_true", help="headline only, no side measurements")
    ap.add_argument("--no-cpu", action="store_true", help="skip the oracle timing")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--attention-only", choices=["sliding", "global"], default=None,
                    help="attention blocks alone (a short case for profilers)")
    ap.add_argument("--prefill-only", action="store_true",
                    help="only the 128-token prefill chunk of one layer (for profilers)")
    ap.add_argument("--decode-only", type=int, default=0, metavar="T",
                    help="only decode steps of T tokens with Zipf routing on one layer (for profilers)")
    ap.add_argument("--stack", action=argparse.BooleanOptionalAction, default=True,
                    help="also run the 30-layer stack decode with per-layer LFU caches")
    ap.add_argument("--copies", type=int, default=0,
                    help="distinct layer copies to rotate over (default: enough to exceed 4x L2)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.decode_only and not 1 <= args.decode_only <= 16:
        ap.error("--decode-only takes 1..16 tokens")
    if args.attention_only:
        run_attention_only(args)
    elif args.prefill_only:
        run_prefill_only(args)
    elif args.decode_only:
        run_decode_only(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
