"""Benchmark of the grouped-expert MoE FFN layer on one GB300 (one JSON line on stdout).

Default workload: the 40-layer stacked prefill at T=2600 (35B-A3B-shaped layers, H=2048,
E=128, top_k=8, I=512, shared expert I=512, distinct seeded weights per layer; per layer the
input is RMS-normalised (parameter-free pre-norm), router logits = x_in @ W_r, and the
residual x <- bf16(x + y)). One step = the whole stack over one batch.
`value` = MoE-layer tokens per second (T x 40 per step). The same run also measures batched
decode at C=8 rows through the same 40 layers' weights (microseconds per layer and the HBM
roofline over the unique experts' bytes).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun each rank runs an independent replica on its own GPU (the layer has no
exchange step); rank 0 prints the line with the whole-job throughput.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import synth  # noqa: E402

METRIC = "MoE layer tokens/s (prefill) & µs/layer decode C=8; % int8/HBM roofline"
# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) of one gate/up GEMM launch on the
# stacked-prefill layer (T=2600), from one ncu capture of the kernel as it is now. Set to None
# whenever the kernel changes, until it is captured again.
GU_TRAFFIC_BYTES = 399.5e6
# Kernels one stacked-prefill layer launches: RMS pre-norm, router projection, and the
# forward's routing + histogram + scan, scatter, gate/up GEMM, requantisation, down GEMM.
LAUNCHES_PER_LAYER = 7
# moe_forward's default dispatch threshold (T <= this runs the weight-streaming kernels).
DEFAULT_DECODE_ROWS = 24
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def load_peaks():
    try:
        with open(PEAKS_FILE) as f:
            p = json.load(f)
        return p, "measured"
    except Exception:
        return dict(FALLBACK), "fallback"


# ---------------------------------------------------------------- distributed plumbing

def dist_init(n_gpus):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
            torch.distributed.init_process_group("nccl")
        else:
            # host-only runs (the tests of this plumbing): the same path over gloo
            torch.distributed.init_process_group("gloo")
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return world, rank


def barrier(world):
    if world > 1:
        torch.distributed.barrier()


def max_over_ranks(v, world):
    if world == 1:
        return v
    dev = "cuda" if torch.distributed.get_backend() == "nccl" else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return t.item()


def replica_throughput(units_per_step, world, ms_step):
    """Whole-job rate of `world` independent replicas (weak scaling): every rank processes
    units_per_step per step, and the step takes the slowest rank's time ms_step."""
    return units_per_step * world / (ms_step / 1e3)


# ---------------------------------------------------------------- clocks

class Clocks:
    """nvidia-smi sampling during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self):
        try:
            self.idx = "GPU-" + str(torch.cuda.get_device_properties(torch.cuda.current_device()).uuid)
        except Exception:
            self.idx = "0"
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in open(self.path):
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "samples": len(sm), "reasons": sorted(reasons)}


# ---------------------------------------------------------------- our arm

def build_stack(moe, wl, n_layers, dev):
    sh = wl.shape
    plan = moe.moe_plan(sh.E, sh.k, sh.H, sh.I, sh.Is, sh.T)
    layers = []
    for l in range(n_layers):
        seed = synth.layer_seed(wl, l)
        W = synth.make_weights(sh, seed, device=dev)
        wr = synth.make_router_weight(sh.H, sh.E, seed, device=dev)
        packed = moe.moe_pack_weights(plan, W)
        layers.append((W, moe.moe_router_pack(wr), packed))
    torch.cuda.synchronize()
    return plan, layers


def oracle_sample_rate(W_dev, wl, n_tokens, nthreads):
    """Oracle (as it stands) on n_tokens tokens of one stacked-prefill layer; returns
    (layer-tokens per second, seconds, threads)."""
    import oracle
    sh = wl.shape
    L = oracle.Layer({k: v.cpu() for k, v in W_dev.items()}, sh.E, sh.k, sh.H, sh.I, sh.Is)
    x = synth.make_activations(sh.T, sh.H, wl.seed)[:n_tokens].contiguous()
    wr = synth.make_router_weight(sh.H, sh.E, wl.seed)
    t0 = time.perf_counter()
    _, x = oracle.rmsnorm_residual(x)
    lg = oracle.router_logits(x, wr, nthreads=nthreads).astype(np.float32)
    idx, w = oracle.route(lg, sh.k)
    oracle.forward(L, x, idx, w, nthreads=nthreads)
    dt = time.perf_counter() - t0
    return n_tokens / dt, dt


def measure_decode(moe, plan, packed_list, peaks, H, E, k, bytes_per_expert, steps, stream,
                   what="int8 weights of the stack's 40 layers"):
    """Batched decode, C=8 rows, through one packed weight set per layer (CUDA graph of one
    moe_route_forward per layer: routing from the logits inside the forward); microseconds
    per layer and the HBM roofline of the unique experts' bytes."""
    dev = torch.device("cuda")
    dwl = synth.WORKLOADS["decode"]
    xd = synth.make_activations(dwl.shape.T, H, dwl.seed, dwl.outliers, dev)
    lgd = synth.make_logits(dwl.shape.T, E, dwl.seed, dwl.zipf_s, dev)
    idd = torch.empty((dwl.shape.T, k), dtype=torch.int32, device=dev)
    wd = torch.empty((dwl.shape.T, k), dtype=torch.float32, device=dev)
    yd = torch.empty((dwl.shape.T, H), dtype=torch.float32, device=dev)

    def decode_stack():
        for packed in packed_list:
            moe.moe_route_forward(plan, packed, xd, lgd, idd, wd, yd)

    n_layers = len(packed_list)
    decode_stack()
    torch.cuda.synchronize()
    counts = moe.moe_debug_tap(plan, moe.TAP_COUNTS)
    U = int((counts > 0).sum())
    g = torch.cuda.CUDAGraph()
    s2 = torch.cuda.Stream()
    s2.wait_stream(stream)
    with torch.cuda.stream(s2):
        with torch.cuda.graph(g, stream=s2):
            decode_stack()
    torch.cuda.synchronize()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    d0, d1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    reps = max(steps, 20)
    torch.cuda.nvtx.range_push("timed_decode")
    d0.record(stream)
    for _ in range(reps):
        g.replay()
    d1.record(stream)
    torch.cuda.nvtx.range_pop()
    torch.cuda.synchronize()
    us_layer = d0.elapsed_time(d1) * 1e3 / reps / n_layers
    # per-stage decode timing (eager, profiled)
    moe.moe_profile_enable(plan, True)
    for _ in range(3):
        decode_stack()
    torch.cuda.synchronize()
    st, calls = moe.moe_profile_read(plan, 1)
    moe.moe_profile_enable(plan, False)
    dstage_us = [v * 1e3 / max(calls, 1) for v in st][:3]
    uniq_bytes = (U + 1) * bytes_per_expert
    hbm = peaks.get("hbm_gbs", FALLBACK["hbm_gbs"])
    dec_gbs = uniq_bytes / (us_layer * 1e-6) / 1e9
    kern_us = dstage_us[1] + dstage_us[2]

    return {"workload": f"C=8 rows, T=8, Zipf(1.1) routing, outliers, through the {what}",
            "us_per_layer": us_layer, "unique_experts": U,
            "unique_bytes_per_layer": uniq_bytes, "achieved_gbs": dec_gbs,
            "hbm_peak_gbs": hbm, "frac": dec_gbs / hbm,
            "stage_us": {"route_dedup_quant": dstage_us[0], "gate_up_stream_requant": dstage_us[1],
                         "down_stream_into_y": dstage_us[2]},
            "kernel_gbs": uniq_bytes / (kern_us * 1e-6) / 1e9 if kern_us > 0 else None}


def measure_decode_nvfp4(moe, plan, wl, n_layers, peaks, steps, stream):
    """The C=8 decode measurement with NVFP4 expert weights (one NVFP4 weight set per layer,
    the same shapes): microseconds per layer and the HBM roofline of the unique experts'
    NVFP4 bytes (codes + block scales)."""
    sh = wl.shape
    dev = torch.device("cuda")
    Ws, packed = [], []
    for l in range(n_layers):
        W4 = synth.make_weights_nvfp4(sh, synth.layer_seed(wl, l), device=dev)
        Ws.append(W4)
        packed.append(moe.moe_pack_weights_nvfp4(plan, W4))
    torch.cuda.synchronize()
    assert moe.moe_get_error(plan) == 0
    try:
        return measure_decode(moe, plan, packed, peaks, sh.H, sh.E, sh.k,
                              synth.weight_bytes_per_expert_nvfp4(sh.H, sh.I), steps, stream,
                              what=f"NVFP4 weights of {n_layers} layers")
    finally:
        for pk in packed:
            moe.moe_packed_destroy(pk)
        del Ws
        torch.cuda.empty_cache()


def measure_crossover(moe, plan, layers, H, E, k, steps, stream,
                      Ts=(1, 2, 4, 8, 12, 16, 24, 32, 48, 64)):
    """Both paths of moe_forward at small T (the decode/grouped-GEMM crossover): each T runs
    through the stack's 40 layers' weights (CUDA graph of moe_route_forward per layer) once on
    the weight-streaming decode kernels and once on the grouped GEMMs; microseconds per
    layer. Zipf(1.1) routing as in the decode workload."""
    dev = torch.device("cuda")
    dwl = synth.WORKLOADS["decode"]
    out = {"T": [], "stream_us": [], "grouped_us": []}
    for T in Ts:
        xd = synth.make_activations(T, H, 500 + T, dwl.outliers, dev)
        lgd = synth.make_logits(T, E, 500 + T, dwl.zipf_s, dev)
        idd = torch.empty((T, k), dtype=torch.int32, device=dev)
        wd = torch.empty((T, k), dtype=torch.float32, device=dev)
        yd = torch.empty((T, H), dtype=torch.float32, device=dev)

        def run():
            for (W, wr, packed) in layers:
                moe.moe_route_forward(plan, packed, xd, lgd, idd, wd, yd)

        out["T"].append(T)
        for rows, key in ((64, "stream_us"), (0, "grouped_us")):
            moe.moe_plan_set_decode_rows(plan, rows)
            run()
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            s2 = torch.cuda.Stream()
            s2.wait_stream(stream)
            with torch.cuda.stream(s2):
                with torch.cuda.graph(g, stream=s2):
                    run()
            torch.cuda.synchronize()
            for _ in range(3):
                g.replay()
            d0, d1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            reps = max(steps, 10)
            d0.record(stream)
            for _ in range(reps):
                g.replay()
            d1.record(stream)
            torch.cuda.synchronize()
            out[key].append(round(d0.elapsed_time(d1) * 1e3 / reps / len(layers), 2))
            del g
    moe.moe_plan_set_decode_rows(plan, DEFAULT_DECODE_ROWS)
    assert moe.moe_get_error(plan) == 0
    faster = [T for T, a, b in zip(out["T"], out["stream_us"], out["grouped_us"]) if b < a]
    out["grouped_faster_from_T"] = min(faster) if faster else None
    out["plan_default_decode_rows"] = DEFAULT_DECODE_ROWS
    return out


def layer_work(sh, counts=None):
    """(int-ops of the layer, weight bytes the layer touches) for routing counts `counts`
    (experts with no row touch no bytes); 2*M*N*K over routed rows plus the shared expert."""
    R = sh.T * sh.k
    ops = 2.0 * R * 3 * sh.I * sh.H + 2.0 * sh.T * 3 * sh.Is * sh.H
    used = sh.E if counts is None else int((counts > 0).sum())
    wbytes = used * (3 * sh.H * sh.I + 4 * (2 * sh.I + sh.H))
    if sh.Is:
        wbytes += 3 * sh.H * sh.Is + 4 * (2 * sh.Is + sh.H)
    return ops, wbytes


def measure_layer(moe, name, peaks, steps, fmt="int8"):
    """One layer of a single-layer workload (the 256-token prefill chunk, the 8192-token
    stress layer) with int8 or NVFP4 expert weights: routing once, then `steps` timed
    forwards (CUDA events on the stream); tokens/s, microseconds per layer, and the layer's
    tensor and HBM roofline fractions."""
    dev = torch.device("cuda")
    wl = synth.WORKLOADS[name]
    sh = wl.shape
    W = (synth.make_weights if fmt == "int8" else synth.make_weights_nvfp4)(sh, wl.seed, device=dev)
    x = synth.make_activations(sh.T, sh.H, wl.seed, wl.outliers, dev)
    lg = synth.make_logits(sh.T, sh.E, wl.seed, wl.zipf_s, dev)
    lay = moe.MoELayer(sh.E, sh.k, sh.H, sh.I, sh.Is, sh.T, W)
    try:
        idx, w = lay.route(lg)
        y = torch.empty((sh.T, sh.H), dtype=torch.float32, device=dev)
        for _ in range(3):
            lay.forward(x, idx, w, y)
        torch.cuda.synchronize()
        counts = moe.moe_debug_tap(lay.plan, moe.TAP_COUNTS)
        stream = torch.cuda.current_stream()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        reps = max(steps, 10)
        e0.record(stream)
        for _ in range(reps):
            lay.forward(x, idx, w, y)
        e1.record(stream)
        torch.cuda.synchronize()
        us = e0.elapsed_time(e1) * 1e3 / reps
        moe.moe_profile_enable(lay.plan, True)
        for _ in range(3):
            lay.forward(x, idx, w, y)
        torch.cuda.synchronize()
        st, calls = moe.moe_profile_read(lay.plan, 0)
        moe.moe_profile_enable(lay.plan, False)
        if moe.moe_get_error(lay.plan):
            raise moe.MoeError(moe.moe_get_error(lay.plan), name)
    finally:
        lay.close()
    ops, wbytes = layer_work(sh, counts)
    if fmt == "nvfp4":  # the same experts at NVFP4 width
        used = int((counts > 0).sum())
        wbytes = used * synth.weight_bytes_per_expert_nvfp4(sh.H, sh.I) + \
            (synth.weight_bytes_per_expert_nvfp4(sh.H, sh.Is) if sh.Is else 0)
    act_bytes = sh.T * sh.H * 2 + sh.T * sh.H * 4  # x in (bf16), y out (fp32)
    tf = ops / (us * 1e-6) / 1e12
    gbs = (wbytes + act_bytes) / (us * 1e-6) / 1e9
    return {"workload": wl.note + ("" if fmt == "int8" else ", NVFP4 expert weights"),
            "tokens_per_s": sh.T / (us * 1e-6), "us_per_layer": us,
            "int_ops": ops, "achieved_tops": tf,
            "tensor_frac": tf / peaks.get("bf16_tflops", FALLBACK["bf16_tflops"]),
            "hbm_bytes": wbytes + act_bytes, "achieved_gbs": gbs,
            "hbm_frac": gbs / peaks.get("hbm_gbs", FALLBACK["hbm_gbs"]),
            "experts_used": int((counts > 0).sum()),
            "stage_us": [v * 1e3 / max(calls, 1) for v in st]}


def measure_prefill_formats(moe, peaks, steps, n_layers=8):
    """The stacked-prefill layer shape (T=2600, H=2048, E=128, top_k=8, I=512, shared 512) with
    int8 and with NVFP4 expert weights, in the same harness: n_layers layers of each (weights
    above L2 in total), N(0,1) router logits per layer, moe_forward per layer timed with CUDA
    events; microseconds per layer, the two GEMM stages and the gate/up GEMM's tensor
    fraction."""
    dev = torch.device("cuda")
    wl = synth.WORKLOADS["stack"]
    sh = wl.shape
    T, H, E, k = sh.T, sh.H, sh.E, sh.k
    x = synth.make_activations(T, H, wl.seed, wl.outliers, dev)
    y = torch.empty((T, H), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()
    R = T * k + T
    gu_flops = 2.0 * R * 2 * sh.I * H
    peak_tf = peaks.get("bf16_tflops", FALLBACK["bf16_tflops"])
    out = {"workload": f"{n_layers} layers x T={T}, H={H}, E={E}, top_k={k}, I={sh.I}, shared I={sh.Is}, "
                       "N(0,1) router logits"}
    for fmt in ("int8", "nvfp4"):
        plan = moe.moe_plan(E, k, H, sh.I, sh.Is, T)
        Ws, packed, routes = [], [], []
        try:
            for l in range(n_layers):
                seed = synth.layer_seed(wl, l)
                if fmt == "int8":
                    W = synth.make_weights(sh, seed, device=dev)
                    packed.append(moe.moe_pack_weights(plan, W))
                else:
                    W = synth.make_weights_nvfp4(sh, seed, device=dev)
                    packed.append(moe.moe_pack_weights_nvfp4(plan, W))
                Ws.append(W)
                lg = synth.make_logits(T, E, seed, 0.0, dev)
                idx = torch.empty((T, k), dtype=torch.int32, device=dev)
                w = torch.empty((T, k), dtype=torch.float32, device=dev)
                moe.moe_route(plan, lg, idx, w)
                routes.append((idx, w))

            def run():
                for pk, (idx, w) in zip(packed, routes):
                    moe.moe_forward(plan, pk, x, idx, w, y)

            for _ in range(3):
                run()
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            reps = max(steps, 5)
            e0.record(stream)
            for _ in range(reps):
                run()
            e1.record(stream)
            torch.cuda.synchronize()
            us = e0.elapsed_time(e1) * 1e3 / reps / n_layers
            moe.moe_profile_enable(plan, True)
            for _ in range(2):
                run()
            torch.cuda.synchronize()
            st, calls = moe.moe_profile_read(plan, 0)
            moe.moe_profile_enable(plan, False)
            if moe.moe_get_error(plan):
                raise moe.MoeError(moe.moe_get_error(plan), f"prefill {fmt}")
        finally:
            for pk in packed:
                moe.moe_packed_destroy(pk)
            moe.moe_plan_destroy(plan)
            del Ws
            torch.cuda.empty_cache()
        stage = [v * 1e3 / max(calls, 1) for v in st]
        gu_tf = gu_flops / (stage[1] * 1e-6) / 1e12
        out[fmt] = {"us_per_layer": us, "tokens_per_s": T / (us * 1e-6),
                    "stage_us": {"permute_quant": stage[0], "gate_up_gemm": stage[1],
                                 "requant": stage[2], "down_gemm_into_y": stage[3]},
                    "gate_up_tflops": gu_tf, "gate_up_frac": gu_tf / peak_tf}
    return out


def oracle_one_core(names, max_tokens):
    """The oracle (as it stands) on one host core: MoE-layer tokens/s per workload, on the
    first min(T, max_tokens[name]) tokens of the workload's layer."""
    import oracle
    out = {}
    for name in names:
        wl = synth.WORKLOADS[name]
        sh = wl.shape
        d = synth.make_layer(wl, device="cpu")
        n = min(sh.T, max_tokens.get(name, sh.T))
        L = oracle.Layer(d["weights"], sh.E, sh.k, sh.H, sh.I, sh.Is)
        x = d["x"][:n].contiguous()
        lg = d["logits"][:n].contiguous()
        t0 = time.perf_counter()
        idx, w = oracle.route(lg, sh.k)
        oracle.forward(L, x, idx, w, nthreads=1)
        dt = time.perf_counter() - t0
        out[name] = {"value": n / dt, "unit": "MoE-layer tokens/s", "cores": 1, "kind": "oracle",
                     "sample": f"{n} of {sh.T} tokens of the {name} layer (route + layer), {dt:.2f} s"}
    return out


def run_ours(args, world, rank):
    import grouped_expert_ffn_gb300 as moe
    peaks, peak_src = load_peaks()
    dev = torch.device("cuda")
    wl = synth.WORKLOADS["stack"]
    sh = wl.shape
    n_layers = args.layers
    plan, layers = build_stack(moe, wl, n_layers, dev)
    T, H, E, k = sh.T, sh.H, sh.E, sh.k
    x0 = synth.make_activations(T, H, wl.seed, wl.outliers, dev)
    x = torch.empty_like(x0)
    x_in = torch.empty_like(x0)
    logits = torch.empty((T, E), dtype=torch.float32, device=dev)
    idx = torch.empty((T, k), dtype=torch.int32, device=dev)
    w = torch.empty((T, k), dtype=torch.float32, device=dev)
    y = torch.empty((T, H), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()

    prof_layer = n_layers // 2

    def stack(profile=False):
        # layer l: x_in = rmsnorm(x) -> logits = x_in @ W_r -> routing and y = moe(x_in), the
        # routing inside the forward's first kernel -> x += y
        # With profile, one layer per step records the plan's per-stage CUDA events (events
        # between every layer's kernels would add their own cost to the step).
        for l, (W, wr, packed) in enumerate(layers):
            moe.moe_rmsnorm_residual(x, y if l else None, x_in)
            moe.moe_router_logits_packed(x_in, wr, logits)
            if profile and l == prof_layer:
                moe.moe_profile_enable(plan, True)
            moe.moe_route_forward(plan, packed, x_in, logits, idx, w, y)
            if profile and l == prof_layer:
                moe.moe_profile_enable(plan, False)
        moe.moe_residual_add(x, y)

    def step(profile=False):
        x.copy_(x0)
        stack(profile)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    err = moe.moe_get_error(plan)
    if err:
        raise moe.MoeError(err, "stacked prefill warm-up")
    clocks = Clocks()
    barrier(world)
    torch.cuda.synchronize()
    clocks.start()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.nvtx.range_push("timed_prefill")
    ev0.record(stream)
    for _ in range(args.steps):
        step(profile=True)
    ev1.record(stream)
    torch.cuda.nvtx.range_pop()
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop()
    ms_total = max_over_ranks(ev0.elapsed_time(ev1), world)
    st, calls = moe.moe_profile_read(plan, 0)
    stage_ms = [v / max(calls, 1) for v in st]
    assert moe.moe_get_error(plan) == 0
    ms_step = ms_total / args.steps
    layer_tokens = T * n_layers
    value = replica_throughput(layer_tokens, world, ms_step)

    # roofline of the dominant kernel (gate/up GEMM): 2*R*2I*H flops per launch
    R = T * k + T
    gu_flops = 2.0 * R * 2 * sh.I * H
    gu_ms = stage_ms[1]
    peak_tf = peaks.get("bf16_tflops", FALLBACK["bf16_tflops"])
    peak_sus = peaks.get("bf16_tflops_sustained", FALLBACK["bf16_tflops_sustained"])
    achieved_tf = gu_flops / (gu_ms / 1e3) / 1e12
    down_flops = 2.0 * R * H * sh.I
    layer_flops = gu_flops + down_flops
    moe_ms = sum(stage_ms)
    layer_tf = layer_flops / (moe_ms / 1e3) / 1e12

    # ---- e2e: host (pinned) x in, host result out, inside the timed region
    e2e = None
    if not args.no_e2e:
        x_host = x0.cpu().pin_memory()
        out_host = torch.empty_like(x_host).pin_memory()

        def step_e2e():
            x.copy_(x_host, non_blocking=True)
            stack()
            out_host.copy_(x, non_blocking=True)

        step_e2e()
        torch.cuda.synchronize()
        barrier(world)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            step_e2e()
        e1.record(stream)
        torch.cuda.synchronize()
        ms_e2e = max_over_ranks(e0.elapsed_time(e1), world) / args.steps
        e2e_value = replica_throughput(layer_tokens, world, ms_e2e)

        e2e = {"value": e2e_value, "unit": "MoE-layer tokens/s",
               "h2d_bytes_per_step": x_host.numel() * 2, "d2h_bytes_per_step": out_host.numel() * 2}

    decode = None if args.no_decode else measure_decode(
        moe, plan, [pk for (_, _, pk) in layers], peaks, H, E, k,
        synth.weight_bytes_per_expert(H, sh.I), args.steps, stream)

    # ---- oracle CPU baseline (bounded sample, rank 0 only, N=1 only)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        nthreads = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
        n_tok = args.cpu_tokens
        rate, secs = oracle_sample_rate(layers[0][0], wl, n_tok, nthreads)
        cpu = {"value": rate, "unit": "MoE-layer tokens/s", "cores": nthreads, "kind": "oracle",
               "sample": f"{n_tok} tokens of layer 0 of the stack (router projection + route + "
                         f"layer), {secs:.1f} s"}

    extra = {}
    if rank == 0 and not args.no_extra:
        extra["prefill_chunk_T256"] = measure_layer(moe, "prefill", peaks, args.steps)
        extra["stress_T8192"] = measure_layer(moe, "stress", peaks, args.steps)
        extra["stress_T8192_nvfp4"] = measure_layer(moe, "stress", peaks, args.steps, fmt="nvfp4")
        extra["decode_crossover"] = measure_crossover(moe, plan, layers, H, E, k, args.steps, stream)
        if not args.no_decode:
            extra["decode_nvfp4"] = measure_decode_nvfp4(moe, plan, wl, n_layers, peaks, args.steps,
                                                         stream)
        extra["prefill_int8_vs_nvfp4"] = measure_prefill_formats(moe, peaks, args.steps)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        extra["cpu_baseline_1core"] = oracle_one_core(["tiny", "decode", "prefill"],
                                                      {"prefill": args.cpu_tokens_1core})

    n_launch = (n_layers * LAUNCHES_PER_LAYER + 1) * args.steps
    line = {
        "metric": METRIC,
        "value": value,
        "unit": "MoE-layer tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "int8 (W8A8) on the fp16 tensor pipe, fp32 epilogue",
        "data": "synthetic (seeded, random-init weights)",
        "config": {"workload": f"stacked prefill {n_layers} layers x T={T}, H={H}, E={E}, top_k={k}, "
                               f"I={sh.I}, shared I={sh.Is}",
                   "global_batch": T * world, "seq_len": T, "layers": n_layers,
                   "parallelism": f"replicas x{world}",
                   "l2": "inputs larger than L2 (each layer's weights > 129 MB)"},
        "per_layer_us": ms_step * 1e3 / n_layers,
        "moe_layer_us": moe_ms * 1e3,
        "stack_prompt_tokens_per_s": replica_throughput(T, world, ms_step),
        "stage_us": {"permute_quant": stage_ms[0] * 1e3, "gate_up_gemm": stage_ms[1] * 1e3,
                     "requant": stage_ms[2] * 1e3, "down_gemm_into_y": stage_ms[3] * 1e3},
        "roofline": {"bound": "tensor", "kernel": "grouped gate/up GEMM (tcgen05 kind::f16)",
                     "achieved": achieved_tf, "peak": peak_tf, "unit": "TFLOP/s",
                     "frac": achieved_tf / peak_tf, "traffic": GU_TRAFFIC_BYTES,
                     "traffic_unit": "bytes per launch (ncu)",
                     "peak_source": f"{peak_src} bf16_tflops (burst; fp16 = bf16 rate)",
                     "frac_of_sustained": achieved_tf / peak_sus,
                     "flops_per_launch": gu_flops},
        "layer_roofline": {"bound": "tensor", "achieved": layer_tf, "unit": "TFLOP/s",
                           "flops_per_layer": layer_flops, "layer_us": moe_ms * 1e3,
                           "frac": layer_tf / peak_tf, "frac_of_sustained": layer_tf / peak_sus,
                           "gate_up_frac": achieved_tf / peak_tf,
                           "down_frac": down_flops / (stage_ms[3] / 1e3) / 1e12 / peak_tf,
                           "peak_source": f"{peak_src} bf16_tflops (burst)"},
        "layer_tflops": layer_tf,
        "decode": decode,
        "e2e": e2e,
        "gpu_launches": n_launch,
        "clocks": clk,
        "cpu_baseline": cpu,
        **extra,
    }
    if rank == 0:
        print(json.dumps(line))


# ---------------------------------------------------------------- reference arm (the oracle)

def run_reference(args, world, rank):
    if rank != 0:
        return
    import oracle
    wl = synth.WORKLOADS["stack"]
    sh = wl.shape
    nthreads = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    W = synth.make_weights(sh, synth.layer_seed(wl, 0), device="cpu")
    L = oracle.Layer(W, sh.E, sh.k, sh.H, sh.I, sh.Is)
    wr = synth.make_router_weight(sh.H, sh.E, wl.seed)
    x_all = synth.make_activations(sh.T, sh.H, wl.seed)
    n_tok = args.ref_tokens

    def step(i):
        off = (i * n_tok) % (sh.T - n_tok)
        x = x_all[off:off + n_tok].contiguous()
        _, x = oracle.rmsnorm_residual(x)
        lg = oracle.router_logits(x, wr, nthreads=nthreads).astype(np.float32)
        idx, w = oracle.route(lg, sh.k)
        oracle.forward(L, x, idx, w, nthreads=nthreads)

    for i in range(args.warmup):
        step(i)
    t0 = time.perf_counter()
    for i in range(args.steps):
        step(args.warmup + i)
    dt = time.perf_counter() - t0
    value = n_tok * args.steps / dt
    line = {"metric": METRIC, "value": value, "unit": "MoE-layer tokens/s", "impl": "reference",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": dt * 1e3 / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "int8 W8A8, fp32 epilogue (scalar C++)",
            "data": "synthetic (seeded, random-init weights)",
            "config": {"workload": f"stacked prefill layer, T={sh.T} sampled {n_tok} tokens per step, "
                                   f"H={sh.H}, E={sh.E}, top_k={sh.k}, I={sh.I}, shared I={sh.Is}",
                       "global_batch": n_tok, "seq_len": sh.T, "parallelism": "host cores"},
            "cpu_baseline": {"value": value, "unit": "MoE-layer tokens/s", "cores": nthreads,
                             "kind": "oracle", "sample": f"{n_tok} tokens of one layer per step"},
            "e2e": {"value": value, "unit": "MoE-layer tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


def nvfp4_probe():
    """A short fixed launch sequence for a profiler capture of the NVFP4 kernels (no timing,
    no JSON line): one plan and one NVFP4 weight set of the stacked layer's shape, two
    moe_route_forward calls at T=2600 (grouped GEMMs, N(0,1) router logits), then two at T=8
    (streaming decode kernels, the decode workload's Zipf(1.1) logits)."""
    import grouped_expert_ffn_gb300 as moe
    dev = torch.device("cuda")
    wl = synth.WORKLOADS["stack"]
    sh = wl.shape
    plan = moe.moe_plan(sh.E, sh.k, sh.H, sh.I, sh.Is, sh.T)
    W = synth.make_weights_nvfp4(sh, synth.layer_seed(wl, 0), device=dev)
    pk = moe.moe_pack_weights_nvfp4(plan, W)
    dwl = synth.WORKLOADS["decode"]
    for T, x, lg in ((sh.T, synth.make_activations(sh.T, sh.H, wl.seed, wl.outliers, dev),
                      synth.make_logits(sh.T, sh.E, wl.seed, 0.0, dev)),
                     (8, synth.make_activations(8, sh.H, dwl.seed, dwl.outliers, dev),
                      synth.make_logits(8, sh.E, dwl.seed, dwl.zipf_s, dev))):
        idx = torch.empty((T, sh.k), dtype=torch.int32, device=dev)
        w = torch.empty((T, sh.k), dtype=torch.float32, device=dev)
        y = torch.empty((T, sh.H), dtype=torch.float32, device=dev)
        for _ in range(2):
            moe.moe_route_forward(plan, pk, x, lg, idx, w, y)
    torch.cuda.synchronize()
    if moe.moe_get_error(plan):
        raise moe.MoeError(moe.moe_get_error(plan), "nvfp4 probe")
    moe.moe_packed_destroy(pk)
    moe.moe_plan_destroy(plan)
    print("nvfp4 probe ok")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--layers", type=int, default=40)
    ap.add_argument("--cpu-tokens", type=int, default=2600,
                    help="tokens of layer 0 the oracle baseline runs (our arm)")
    ap.add_argument("--ref-tokens", type=int, default=512,
                    help="tokens per step of the reference (oracle) arm")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-decode", action="store_true", help="skip the decode measurement")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end pass")
    ap.add_argument("--no-extra", action="store_true",
                    help="skip the T=256 prefill-chunk and T=8192 stress layer lines")
    ap.add_argument("--cpu-tokens-1core", type=int, default=48,
                    help="tokens of the T=256 prefill layer the one-core oracle runs")
    ap.add_argument("--nvfp4-probe", action="store_true",
                    help="only run the short NVFP4 launch sequence a profiler capture uses")
    args = ap.parse_args()
    if args.nvfp4_probe:
        nvfp4_probe()
        return
    if args.impl == "reference":
        rank = int(os.environ.get("RANK", "0"))
        world = int(os.environ.get("WORLD_SIZE", "1"))
        run_reference(args, world, rank)
        return
    world, rank = dist_init(args.gpus)
    run_ours(args, world, rank)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
