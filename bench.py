#!/usr/bin/env python
"""GPT-2 pretraining-step benchmark on B300: train tokens/s and MFU.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--config 124m|350m|1558m|attn|classifier] [--no-cpu-baseline]

Step configs (124m default, 350m, 1558m = the d48 model): one step = forward
(embedding, L pre-LN blocks, tied lm_head over the padded vocabulary, mean
cross-entropy) + full backward + global-norm clip + AdamW, on one batch of
synthetic Zipf(1.1) token streams (B=16, T=1024 for 124M).  The step runs
through the C ABI of libgpt2.so, captured once in a CUDA graph and replayed;
`value` is device-timed with CUDA events over K replays with the inputs
resident in HBM.  `e2e` times gpt2_train_step_host with pinned host token
buffers (host->device copies and the loss / norm readback inside the timed
region).  Under torchrun every rank runs an independent replica of the step
(weak scaling; the replicas exchange nothing but the timing barrier).

Microbench configs: `attn` times attn_fwd and attn_bwd on bf16 [16, 12, T, 64]
tensors for T in {256, 512, 1024, 2048, 4096}; `classifier` times
classifier_fwd_bwd at M=16384, C=768, V=50257 -> 50304.  Both flush L2 between
timed calls.

--impl reference times the CPU oracle (plain numpy, float64) on the host
cores, on rank 0 only, each step a bounded sample of the same workload (the
same sample the `cpu_baseline` object of the GPU line reports).
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

CONFIGS = {
    "124m": dict(L=12, H=12, C=768, V=50257, Vpad=50304, T=1024, B=16),
    "350m": dict(L=24, H=16, C=1024, V=50257, Vpad=50304, T=1024, B=8),
    "1558m": dict(L=48, H=25, C=1600, V=50257, Vpad=50304, T=1024, B=16),
}
MICRO = ("attn", "classifier")
ATTN_T = (256, 512, 1024, 2048, 4096)
LR, B1, B2, EPS, WD, CLIP = 6e-4, 0.9, 0.95, 1e-8, 0.1, 1.0
NOMINAL_BF16_TFLOPS = 2250.0
METRIC = "GPT-2 124M train tokens/sec on 1 B300 (bf16, T=1024); MFU vs dense BF16 peak"
LLMC_124M_TOK_S = 223000.0  # llm.c GPT-2 124M throughput quoted on the pages (hardware not stated)


def flops_per_token(c):
    """6N + 6 L C T with N the padded parameter count incl. wpe (the convention that
    reproduces the llm.c run log's 47.3% bf16 MFU)."""
    L, C, Vpad, T = c["L"], c["C"], c["Vpad"], c["T"]
    N = Vpad * C + T * C + L * (12 * C * C + 13 * C) + 2 * C
    return 6.0 * N + 6.0 * L * C * T, N


def measured_peaks():
    try:
        return json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except Exception:
        return {}


PROF_STEPS = 5  # instrumented eager steps behind the per-kernel and per-GEMM-shape breakdown
TRAFFIC = os.path.join(ROOT, "profiles", "traffic.json")


def sources_sha256(files):
    import hashlib
    h = hashlib.sha256()
    for f in files:
        h.update(open(os.path.join(ROOT, "pretraining_step_train_b300", "csrc", f), "rb").read())
    return h.hexdigest()


def traffic_per_launch(kernel):
    """ncu DRAM bytes (read + write) per launch of `kernel` from profiles/traffic.json,
    or None when the kernel's sources changed since those counters were taken (hash
    mismatch) or there is no entry."""
    try:
        e = json.load(open(TRAFFIC))[kernel]
        if sources_sha256(e["sources"]) != e["source_sha256"]:
            return None
        return int(e["bytes_per_launch"])
    except Exception:
        return None


def device_init_params(c, seed=43, std=0.02):
    """The init recipe (every weight matrix, wte and wpe ~ N(0, std), the two residual
    projections scaled by 1/sqrt(2L), biases 0, LayerNorm gamma 1 / beta 0, padded wte
    rows 0) drawn on the device with torch's seeded generator: the same distribution as
    synth.init_params without generating billions of values on the host.  Returns the
    flat fp32 CUDA tensor in the canonical order."""
    import torch
    from pretraining_step_train_b300 import synth
    L, C, V, Vpad, T = c["L"], c["C"], c["V"], c["Vpad"], c["T"]
    g = torch.Generator(device="cuda").manual_seed(seed)
    parts = []
    for name, shape in synth.param_shapes(L, C, Vpad, T):
        n = 1
        for d in shape:
            n *= d
        if name.startswith("ln") and name.endswith("w"):
            t = torch.ones(n, device="cuda")
        elif name in ("wte", "wpe", "qkvw", "attprojw", "fcw", "fcprojw"):
            sd = std / (2.0 * L) ** 0.5 if name in ("attprojw", "fcprojw") else std
            t = torch.randn(n, generator=g, device="cuda") * sd
            if name == "wte":
                t.view(Vpad, C)[V:] = 0.0
        else:
            t = torch.zeros(n, device="cuda")
        parts.append(t)
    return torch.cat(parts)


def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


class Clocks:
    """nvidia-smi sampler over the timed region (SM clock, throttle reasons)."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        self.p = None

    def start(self):
        try:
            self.p = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                                       "--format=csv,noheader,nounits", "-lms", "100"],
                                      stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.p = None

    def stop(self):
        if self.p is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.p.terminate()
        try:
            self.p.wait(timeout=5)
        except Exception:
            self.p.kill()
        self.f.flush()
        rows = []
        for line in open(self.f.name):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 9:
                rows.append(parts)
        os.unlink(self.f.name)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


def count_graph_kernels(graph):
    """Number of kernel nodes in a captured cudaGraph_t (cuda-python bindings)."""
    try:
        import cuda.bindings.runtime as rt
        g = rt.cudaGraph_t(graph.raw_cuda_graph())
        err, _, n = rt.cudaGraphGetNodes(g, numNodes=0)
        err, nodes, n = rt.cudaGraphGetNodes(g, numNodes=n)
        k = 0
        for nd in nodes:
            e, t = rt.cudaGraphNodeGetType(nd)
            if t == rt.cudaGraphNodeType.cudaGraphNodeTypeKernel:
                k += 1
        return k
    except Exception:
        return None


def host_cores():
    try:
        import threadpoolctl
        return max(i.get("num_threads", 1) for i in threadpoolctl.threadpool_info())
    except Exception:
        return os.cpu_count()


class OracleStep:
    """The oracle's training step on a bounded sample of a step workload.

    The sample is the first Ts positions of one sequence of the batch (attention
    is causal, so a prefix is a self-contained sub-problem) with Ts = T when a
    full sequence fits the time budget, else the longest multiple of 64 that
    does.  Its cost is fitted as fixed + per-position from two calibration
    steps (64 and 128 positions), so the GPU line's `cpu_baseline` and the
    reference arm pick the same Ts for the same --steps / --warmup."""

    def __init__(self, c):
        import numpy as np  # noqa: F401
        from oracle import gpt2_oracle as O
        from pretraining_step_train_b300 import synth
        self.O, self.c = O, c
        self.cfg = O.Config(c["L"], c["H"], c["C"], c["V"], c["Vpad"], c["T"])
        self.P = synth.init_params(43, c["L"], c["C"], c["V"], c["Vpad"], c["T"], bf16_representable=True)
        self.tok, self.tgt = synth.token_batch(42, 1, c["T"], c["V"])
        t64 = self.time(64)
        t128 = self.time(128)
        self.per_pos = max(1e-6, (t128 - t64) / 64.0)
        self.fixed = max(0.0, t64 - 64 * self.per_pos)

    def time(self, Ts):
        t0 = time.perf_counter()
        self.last = self.O.train_step(self.P, self.tok[:, :Ts], self.tgt[:, :Ts], self.cfg, lr=LR, t=1)
        return time.perf_counter() - t0

    def sample_len(self, steps, warmup, budget_s=170.0):
        per_step = budget_s / max(1, steps + warmup)
        ts = int((per_step - self.fixed) / self.per_pos) // 64 * 64
        return max(64, min(self.c["T"], ts))

    def describe(self, Ts):
        return (f"first {Ts} positions of 1 of the {self.c['B']} sequences (T={self.c['T']}) per step: "
                f"forward + mean CE + backward + clip + AdamW over all {self.O.num_params(self.c['L'], self.c['C'], self.c['Vpad'], self.c['T'])} "
                f"parameters, numpy float64")


def cpu_baseline(c, steps, warmup, budget_s=25.0):
    """The oracle on the host cores, timed on the sample the reference arm uses for
    the same --steps / --warmup: tokens/s of the sampled positions."""
    o = OracleStep(c)
    Ts = o.sample_len(steps, warmup)
    n = max(1, int(budget_s / (o.fixed + o.per_pos * Ts)))
    dt = sum(o.time(Ts) for _ in range(n)) / n
    return {"value": round(Ts / dt, 3), "unit": "tokens/s", "cores": host_cores(), "kind": "oracle",
            "sample": o.describe(Ts) + f"; mean of {n} step(s) of {dt:.2f} s", "loss": o.last["loss"]}


def run_reference(args, c):
    """The oracle on the host cores, K timed steps after W warm-up steps, each on
    the bounded sample described by OracleStep (rank 0 only)."""
    rank, world, _ = dist_env()
    if rank != 0:
        return
    if args.config in MICRO:
        return run_reference_micro(args, world)
    if args.config == "1558m":
        print(json.dumps({"impl": "reference", "unavailable": "the float64 oracle's parameter, gradient and "
                          "AdamW arrays for 1.56B parameters need about 90 GB of host memory"}), flush=True)
        return
    o = OracleStep(c)
    Ts = o.sample_len(args.steps, args.warmup)
    for _ in range(args.warmup):
        o.time(Ts)
    dt = sum(o.time(Ts) for _ in range(args.steps)) / args.steps
    val = Ts / dt
    out = {"impl": "reference", "metric": METRIC if args.config == "124m" else step_metric(args.config),
           "value": round(val, 3), "unit": "tokens/s", "n_gpus": world,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 2),
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
           "data": "synthetic",
           "config": {"workload": f"GPT-2 {args.config} train step (fwd+CE+bwd+clip+AdamW)", **c,
                      "parallelism": "host cores"},
           "cpu_baseline": {"value": round(val, 3), "unit": "tokens/s", "cores": host_cores(), "kind": "oracle",
                            "sample": o.describe(Ts)},
           "e2e": {"value": round(val, 3), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


def step_metric(config):
    return f"GPT-2 {config} train tokens/sec on 1 B300 (bf16, T=1024); MFU vs dense BF16 peak"


# ------------------------------------------------------------------ microbenches
def attn_flops(B, H, T, d=64):
    """Causal-useful forward FLOPs: QK^T and PV over the pairs j <= i (2 d each)."""
    return 4.0 * B * H * d * T * (T + 1) / 2.0


def oracle_attention_rate(T, pairs=2):
    """The oracle's materialised attention forward + backward on `pairs` (b, h) heads of
    [T, 64]: causal-useful TFLOP/s on the host cores."""
    import numpy as np
    from oracle import gpt2_oracle as O
    from pretraining_step_train_b300 import synth
    q, k, v, do = (x.astype(np.float64) for x in synth.attention_inputs(T, 1, pairs, T, 64))
    t0 = time.perf_counter()
    _, p, _ = O.attention_forward(q, k, v, 0.125)
    O.attention_backward(do, q, k, v, p, 0.125)
    dt = time.perf_counter() - t0
    return 3.5 * attn_flops(1, pairs, T) / dt / 1e12, dt


def l2_flush_buffer():
    import torch
    return torch.empty(256 << 20, dtype=torch.uint8, device="cuda")  # twice the 126 MB L2


def time_calls(fn, n, flush, stream):
    """Mean CUDA-event time (ms) of fn() over n calls on `stream`, L2 flushed before each."""
    import torch
    tot = 0.0
    with torch.cuda.stream(stream):
        for _ in range(n):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            e1.synchronize()
            tot += e0.elapsed_time(e1)
    return tot / n


def bench_attn(args, peaks, clocks):
    import torch
    from pretraining_step_train_b300 import binding
    L = binding.lib()
    B, H, d = 16, 12, 64
    stream = torch.cuda.Stream()
    flush = l2_flush_buffer()
    gen = torch.Generator(device="cuda").manual_seed(42)
    peak = peaks.get("bf16_tflops") or 1800.0
    rows = {}
    launches = 0
    clocks.start()
    for T in ATTN_T:
        q, k, v, do = (torch.randn((B, H, T, d), generator=gen, device="cuda").to(torch.bfloat16) for _ in range(4))
        o, dq, dk, dv = (torch.empty_like(q) for _ in range(4))
        lse = torch.empty((B, H, T), dtype=torch.float32, device="cuda")
        ws = torch.empty(L.attn_workspace_bytes(B, H, T), dtype=torch.uint8, device="cuda")
        st = (H * T * d, T * d, d)
        sp = int(stream.cuda_stream)
        fwd = lambda: binding.check(L.attn_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                                               B, H, T, d, *st, *st, 0.125, sp))
        bwd = lambda: binding.check(L.attn_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                                               do.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H, T, d,
                                               *st, *st, 0.125, ws.data_ptr(), ws.numel(), sp))
        with torch.cuda.stream(stream):
            for _ in range(args.warmup):
                fwd(); bwd()
        stream.synchronize()
        tf = time_calls(fwd, args.steps, flush, stream)
        tb = time_calls(bwd, args.steps, flush, stream)
        launches += 3 * args.steps
        ff = attn_flops(B, H, T)
        rows[T] = {"fwd_ms": round(tf, 4), "bwd_ms": round(tb, 4),
                   "fwd_tflops": round(ff / tf / 1e9, 1), "bwd_tflops": round(2.5 * ff / tb / 1e9, 1),
                   "fwd_bwd_tflops": round(3.5 * ff / (tf + tb) / 1e9, 1),
                   "frac_of_burst_peak": round(3.5 * ff / (tf + tb) / 1e9 / peak, 4)}
        del q, k, v, do, o, dq, dk, dv, lse, ws
    clk = clocks.stop()
    # end to end at T = 1024: q, k, v, dO from pinned host memory, dq, dk, dv back
    T = 1024
    host = [torch.randn((B, H, T, d), generator=torch.Generator().manual_seed(i)).to(torch.bfloat16).pin_memory()
            for i in range(4)]
    outs = [torch.empty_like(host[0]).pin_memory() for _ in range(3)]
    dev = [torch.empty_like(host[0], device="cuda") for _ in range(4)]
    o, dq, dk, dv = (torch.empty_like(dev[0]) for _ in range(4))
    lse = torch.empty((B, H, T), dtype=torch.float32, device="cuda")
    ws = torch.empty(L.attn_workspace_bytes(B, H, T), dtype=torch.uint8, device="cuda")
    st = (H * T * d, T * d, d)
    sp = int(stream.cuda_stream)

    def e2e_call():
        with torch.cuda.stream(stream):
            for hsrc, ddst in zip(host, dev):
                ddst.copy_(hsrc, non_blocking=True)
            binding.check(L.attn_fwd(dev[0].data_ptr(), dev[1].data_ptr(), dev[2].data_ptr(), o.data_ptr(),
                                     lse.data_ptr(), B, H, T, d, *st, *st, 0.125, sp))
            binding.check(L.attn_bwd(dev[0].data_ptr(), dev[1].data_ptr(), dev[2].data_ptr(), o.data_ptr(),
                                     lse.data_ptr(), dev[3].data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
                                     B, H, T, d, *st, *st, 0.125, ws.data_ptr(), ws.numel(), sp))
            for dsrc, hdst in zip((dq, dk, dv), outs):
                hdst.copy_(dsrc, non_blocking=True)
        stream.synchronize()

    for _ in range(2):
        e2e_call()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        e2e_call()
    e2e_s = (time.perf_counter() - t0) / args.steps
    ff = attn_flops(B, H, T)
    head = rows[1024]
    out = {
        "metric": "causal attention fwd+bwd TFLOP/s (causal-useful), bf16 [16,12,T,64], T=1024",
        "value": head["fwd_bwd_tflops"], "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(head["fwd_ms"] + head["bwd_ms"], 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "attention microbench: attn_fwd + attn_bwd, Q,K,V,dO ~ N(0,1) bf16 "
                               "[B=16,H=12,T,64], scale 1/8, T swept", "T_sweep": list(ATTN_T),
                   "l2": "flushed (256 MB write) before every timed call",
                   "flops": "forward 4*B*H*d*T(T+1)/2, backward 2.5x forward"},
        "per_T": rows,
        "roofline": {"bound": "tensor", "achieved": head["fwd_bwd_tflops"], "peak": peak, "unit": "TFLOP/s",
                     "frac": head["frac_of_burst_peak"],
                     "peak_source": "MEASURED_PEAKS.json bf16_tflops (burst: the kernels are timed alone)",
                     "traffic": None},
        "e2e": {"value": round(3.5 * ff / e2e_s / 1e12, 1), "unit": "TFLOP/s",
                "h2d_bytes_per_step": 4 * B * H * T * d * 2, "d2h_bytes_per_step": 3 * B * H * T * d * 2,
                "path": "attn_fwd + attn_bwd through the C ABI, q/k/v/dO copied from pinned host memory and "
                        "dq/dk/dv copied back inside the timed region"},
        "gpu_launches": launches,
        "clocks": clk,
    }
    if not args.no_cpu_baseline:
        rate, dt = oracle_attention_rate(1024)
        out["cpu_baseline"] = {"value": round(rate, 6), "unit": "TFLOP/s", "cores": host_cores(), "kind": "oracle",
                               "sample": f"2 of the 192 (b, h) heads at T=1024, materialised T x T softmax, "
                                         f"forward + backward, numpy float64, {dt:.2f} s"}
    print(json.dumps(out), flush=True)


def bench_classifier(args, peaks, clocks):
    import torch
    from pretraining_step_train_b300 import binding, synth
    L = binding.lib()
    M, C, V, Vpad = 16384, 768, 50257, 50304
    x, w, tgt = synth.classifier_inputs(42, M, C, V, Vpad)
    xd = torch.from_numpy(x).cuda().to(torch.bfloat16)
    wd = torch.from_numpy(w).cuda().to(torch.bfloat16)
    td = torch.from_numpy(tgt.astype("int32")).cuda()
    loss = torch.zeros(1, dtype=torch.float32, device="cuda")
    dx = torch.empty((M, C), dtype=torch.bfloat16, device="cuda")
    dw = torch.empty((Vpad, C), dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(L.classifier_workspace_bytes(M, C, Vpad), dtype=torch.uint8, device="cuda")
    stream = torch.cuda.Stream()
    sp = int(stream.cuda_stream)
    flush = l2_flush_buffer()
    call = lambda: binding.check(L.classifier_fwd_bwd(xd.data_ptr(), wd.data_ptr(), td.data_ptr(), M, C, V, Vpad,
                                                      loss.data_ptr(), dx.data_ptr(), dw.data_ptr(), ws.data_ptr(),
                                                      ws.numel(), sp))
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            call()
    stream.synchronize()
    clocks.start()
    ms = time_calls(call, args.steps, flush, stream)
    clk = clocks.stop()
    flops = 6.0 * M * V * C
    peak = peaks.get("bf16_tflops") or 1800.0
    tflops = flops / ms / 1e9
    zb = M * Vpad * 2
    # end to end: x and targets from pinned host memory, loss, dx, dw back
    xh, th = xd.cpu().pin_memory(), td.cpu().pin_memory()
    lh, dxh, dwh = (torch.empty_like(t, device="cpu").pin_memory() for t in (loss, dx, dw))

    def e2e_call():
        with torch.cuda.stream(stream):
            xd.copy_(xh, non_blocking=True)
            td.copy_(th, non_blocking=True)
            call()
            for dsrc, hdst in ((loss, lh), (dx, dxh), (dw, dwh)):
                hdst.copy_(dsrc, non_blocking=True)
        stream.synchronize()

    e2e_call()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        e2e_call()
    e2e_s = (time.perf_counter() - t0) / args.steps
    out = {
        "metric": "fused classifier (tied lm_head + mean CE + dlogits -> dX, dW) TFLOP/s, M=16384, C=768, V=50257",
        "value": round(tflops, 1), "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms, 4), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "classifier microbench: X ~ N(0,1) bf16 [16384,768], W ~ N(0,0.02) bf16 [50304,768] "
                               "(pad rows zero), Zipf(1.1) targets", "flops": "6*M*V*C (V = 50257)",
                   "l2": "flushed (256 MB write) before every timed call"},
        "logits_round_trip_bytes": {"logits_write": zb, "dlogits_read_write_in_place": 2 * zb,
                                    "dlogits_read_by_dx_and_dw_gemms": 2 * zb, "total": 5 * zb,
                                    "note": "bf16 [M, Vpad]; the CE statistics come out of the logits GEMM epilogue, "
                                            "so no separate pass reads the logits for the softmax"},
        "roofline": {"bound": "tensor", "achieved": round(tflops, 1), "peak": peak, "unit": "TFLOP/s",
                     "frac": round(tflops / peak, 4),
                     "peak_source": "MEASURED_PEAKS.json bf16_tflops (burst: the call is timed alone)",
                     "traffic": None},
        "e2e": {"value": round(flops / e2e_s / 1e12, 1), "unit": "TFLOP/s",
                "h2d_bytes_per_step": M * C * 2 + M * 4, "d2h_bytes_per_step": 4 + M * C * 2 + Vpad * C * 2,
                "path": "classifier_fwd_bwd through the C ABI, x and targets copied from pinned host memory, "
                        "loss, dx, dw copied back inside the timed region"},
        "gpu_launches": 6 * args.steps,
        "clocks": clk,
    }
    if not args.no_cpu_baseline:
        import numpy as np
        from oracle import gpt2_oracle as O
        rows = 512
        t0 = time.perf_counter()
        O.classifier_forward_backward(x[:rows].astype(np.float64), w.astype(np.float64), tgt[:rows], V)
        dt = time.perf_counter() - t0
        out["cpu_baseline"] = {"value": round(6.0 * rows * V * C / dt / 1e12, 6), "unit": "TFLOP/s",
                               "cores": host_cores(), "kind": "oracle",
                               "sample": f"{rows} of the {M} rows, full [rows, 50304] logits, numpy float64, {dt:.2f} s"}
    print(json.dumps(out), flush=True)


def run_reference_micro(args, world):
    if args.config == "attn":
        rates = []
        for _ in range(args.warmup):
            oracle_attention_rate(1024)
        for _ in range(args.steps):
            rates.append(oracle_attention_rate(1024))
        val = len(rates) / sum(1.0 / r for r, _ in rates)
        dt = sum(t for _, t in rates) / len(rates)
        metric = "causal attention fwd+bwd TFLOP/s (causal-useful), bf16 [16,12,T,64], T=1024"
        sample = "2 of the 192 (b, h) heads at T=1024 per step, materialised T x T softmax, numpy float64"
    else:
        import numpy as np
        from oracle import gpt2_oracle as O
        from pretraining_step_train_b300 import synth
        M, C, V, Vpad, rows = 16384, 768, 50257, 50304, 512
        x, w, tgt = synth.classifier_inputs(42, M, C, V, Vpad)
        x64, w64 = x[:rows].astype(np.float64), w.astype(np.float64)
        for _ in range(args.warmup):
            O.classifier_forward_backward(x64, w64, tgt[:rows], V)
        t0 = time.perf_counter()
        for _ in range(args.steps):
            O.classifier_forward_backward(x64, w64, tgt[:rows], V)
        dt = (time.perf_counter() - t0) / args.steps
        val = 6.0 * rows * V * C / dt / 1e12
        metric = "fused classifier (tied lm_head + mean CE + dlogits -> dX, dW) TFLOP/s, M=16384, C=768, V=50257"
        sample = f"{rows} of the {M} rows per step, full logits, numpy float64"
    out = {"impl": "reference", "metric": metric, "value": round(val, 6), "unit": "TFLOP/s", "n_gpus": world,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 2), "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
           "config": {"workload": f"{args.config} microbench", "parallelism": "host cores"},
           "cpu_baseline": {"value": round(val, 6), "unit": "TFLOP/s", "cores": host_cores(), "kind": "oracle",
                            "sample": sample},
           "e2e": {"value": round(val, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default="124m", choices=sorted(CONFIGS) + list(MICRO))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-graph", action="store_true", help="eager launches instead of a CUDA graph")
    ap.add_argument("--one-step", action="store_true",
                    help="set up, run one eager step and exit (for profiler launch lists)")
    ap.add_argument("--batch", type=int, default=0,
                    help="override the sequences per step (smaller profiler captures)")
    args = ap.parse_args()
    c = dict(CONFIGS.get(args.config, {}))
    if args.batch > 0 and c:
        c["B"] = args.batch
    if args.impl == "reference":
        run_reference(args, c)
        return
    rank, world, local = dist_env()
    import numpy as np
    import torch
    from pretraining_step_train_b300 import binding, build, synth

    torch.cuda.set_device(local)
    if args.config in MICRO:  # single-GPU microbenches: rank 0 runs them, other ranks have no work
        if rank == 0:
            build.build()
            (bench_attn if args.config == "attn" else bench_classifier)(args, measured_peaks(), Clocks(local))
        return
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        pg = dist
    if rank == 0:
        build.build()
    if pg:
        pg.barrier()
    L, H, C, V, Vpad, T, B = (c[k] for k in ("L", "H", "C", "V", "Vpad", "T", "B"))
    M = B * T
    if args.config == "124m":
        P = synth.init_params(43, L, C, V, Vpad, T, bf16_representable=True)
        flat = synth.flatten_params(P, L, C, Vpad, T)
        del P
    else:
        flat = device_init_params(c)
    NB = 4
    host_batches = [synth.token_batch(42 + 1000 * rank + i, B, T, V) for i in range(NB)]
    dev_tok = torch.stack([torch.from_numpy(b[0]) for b in host_batches]).cuda()
    dev_tgt = torch.stack([torch.from_numpy(b[1]) for b in host_batches]).cuda()
    src_tok = torch.empty((B, T), dtype=torch.int32, device="cuda")
    src_tgt = torch.empty((B, T), dtype=torch.int32, device="cuda")
    stream = torch.cuda.Stream()
    step = binding.Step(L, H, C, V, Vpad, T, B, precision=binding.GPT2_BF16, stream=stream)
    step.set_params(flat)

    def one_step():
        step.forward(src_tok, src_tgt, want_loss=False)
        step.backward()
        step.clip_adamw(LR, B1, B2, EPS, WD, CLIP, 0, want_norm=False)

    with torch.cuda.stream(stream):
        src_tok.copy_(dev_tok[0]); src_tgt.copy_(dev_tgt[0])
        one_step()  # eager warm-up (one-time host set-up inside the library)
    stream.synchronize()
    if args.one_step:
        st = step.sync_status()
        print(json.dumps({"one_step": True, "status": st}), flush=True)
        sys.exit(0 if st == 0 else 1)
    graph = None
    n_kernels = None
    if not args.no_graph:
        graph = torch.cuda.CUDAGraph(keep_graph=True)
        with torch.cuda.graph(graph, stream=stream):
            one_step()
        n_kernels = count_graph_kernels(graph)
        graph.instantiate()

    def run(i):
        with torch.cuda.stream(stream):
            src_tok.copy_(dev_tok[i % NB], non_blocking=True)
            src_tgt.copy_(dev_tgt[i % NB], non_blocking=True)
            if graph is not None:
                graph.replay()
            else:
                one_step()

    for i in range(args.warmup):
        run(i)
    stream.synchronize()
    clocks = Clocks(local)
    clocks.start()
    time.sleep(0.3)
    if pg:
        pg.barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(args.steps):
        run(i)
    e1.record(stream)
    e1.synchronize()
    torch.cuda.synchronize()
    if pg:
        pg.barrier()
    clk = clocks.stop()
    ms = e0.elapsed_time(e1) / args.steps
    t_max = torch.tensor([ms], dtype=torch.float64, device="cuda")
    if pg:
        pg.all_reduce(t_max, op=pg.ReduceOp.MAX)
    ms_max = float(t_max.item())
    status = step.sync_status()

    # per-kernel-class timing of instrumented (uncaptured) steps on the same stream, per-step means
    step.profile(True)
    with torch.cuda.stream(stream):
        for _ in range(PROF_STEPS):
            one_step()
    prof = {k: (v[0] // PROF_STEPS, v[1] / PROF_STEPS, v[2] / PROF_STEPS, v[3] / PROF_STEPS)
            for k, v in step.profile_read().items()}
    regions = [(c, d, ms / PROF_STEPS, fl / PROF_STEPS, by / PROF_STEPS) for c, d, ms, fl, by in step.profile_regions()]
    step.profile(False)
    shapes = {}
    epi_names = ["store", "bias", "bias+resid", "bias+gelu", "gelu'", "ce", "f32"]
    for cls, dims, rms, rfl, rby in regions:
        if cls != "gemm":
            continue
        Mx, Nx, Kx, amn, bmn, epi = dims
        key = f"{Mx}x{Nx}x{Kx} {'MN' if amn else 'K'}{'MN' if bmn else 'K'} {epi_names[epi]}"
        e = shapes.setdefault(key, [0, 0.0, 0.0])
        e[0] += 1; e[1] += rms; e[2] += rfl
    gemm_shapes = {k: {"calls": v[0] // PROF_STEPS, "ms": round(v[1], 4), "tflops": round(v[2] / (v[1] / 1e3) / 1e12, 1)}
                   for k, v in sorted(shapes.items(), key=lambda kv: -kv[1][1])}

    # end to end through the C ABI from pinned host buffers
    pin_tok = [torch.from_numpy(b[0]).pin_memory() for b in host_batches]
    pin_tgt = [torch.from_numpy(b[1]).pin_memory() for b in host_batches]
    e2e_steps = max(3, min(args.steps, 20))
    for i in range(2):
        step.train_step_host(pin_tok[i % NB], pin_tgt[i % NB], LR, B1, B2, EPS, WD, CLIP, 0)
    if pg:
        pg.barrier()
    t0 = time.perf_counter()
    last = None
    for i in range(e2e_steps):
        last = step.train_step_host(pin_tok[i % NB], pin_tgt[i % NB], LR, B1, B2, EPS, WD, CLIP, 0)
    e2e_s = (time.perf_counter() - t0) / e2e_steps
    t_e2e = torch.tensor([e2e_s], dtype=torch.float64, device="cuda")
    if pg:
        pg.all_reduce(t_e2e, op=pg.ReduceOp.MAX)
    e2e_s = float(t_e2e.item())

    if rank != 0:
        if pg:
            pg.destroy_process_group()
        return
    fpt, N = flops_per_token(c)
    tok_s = world * M / (ms_max / 1e3)
    peaks = measured_peaks()
    peak_burst = peaks.get("bf16_tflops")
    peak_sust = peaks.get("bf16_tflops_sustained")
    achieved_tflops = tok_s / world * fpt / 1e12
    g_regions, g_ms, g_flops, g_bytes = prof["gemm"]
    gemm_tflops = g_flops / (g_ms / 1e3) / 1e12 if g_ms > 0 else None
    # the sustained figure was measured at a power-capped clock this step does not run at
    # (the clocks object records the step's own), so the burst figure is the comparator
    gemm_peak = peak_burst or 1800.0
    kernels = {k: {"regions": v[0], "ms": round(v[1], 4), "share": round(v[1] / max(1e-9, sum(x[1] for x in prof.values())), 4),
                   "tflops": round(v[2] / (v[1] / 1e3) / 1e12, 1) if v[1] > 0 and v[2] > 0 else None,
                   "gbs": round(v[3] / (v[1] / 1e3) / 1e9, 1) if v[1] > 0 and v[3] > 0 else None}
               for k, v in prof.items()}
    out = {
        "metric": METRIC if args.config == "124m" else step_metric(args.config),
        "value": round(tok_s, 1),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_max, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": round(tok_s / LLMC_124M_TOK_S, 3) if args.config == "124m" else None,
        "vs_baseline_ref": ("llm.c GPT-2 124M 223k tok/s quoted on the pages (hardware not stated; context)"
                            if args.config == "124m" else None),
        "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": f"GPT-2 {args.config} train step (fwd+CE+bwd+clip+AdamW)", "B": B, "T": T, "L": L,
                   "H": H, "C": C, "V": V, "Vpad": Vpad, "global_batch_tokens": world * M,
                   "parallelism": f"{world} independent replica(s)", "graph": graph is not None,
                   "l2": "working set (params, optimizer state, activations: 9 GB and up) far exceeds L2; no flush",
                   "tokens": "Zipf(1.1) streams over the vocab, targets shifted by one"},
        "mfu": {"flops_per_token": fpt, "convention": "6N+6LCT, N padded incl. wpe",
                "vs_nominal_2250": round(achieved_tflops / NOMINAL_BF16_TFLOPS, 4),
                "vs_measured_burst": round(achieved_tflops / peak_burst, 4) if peak_burst else None,
                "achieved_tflops": round(achieved_tflops, 1)},
        "roofline": {"bound": "tensor", "kernel": "k_gemm_tc (all Linears + classifier logits)",
                     "achieved": round(gemm_tflops, 1) if gemm_tflops else None,
                     "peak": gemm_peak, "unit": "TFLOP/s",
                     "frac": round(gemm_tflops / gemm_peak, 4) if gemm_tflops else None,
                     "peak_source": "MEASURED_PEAKS.json bf16_tflops (burst); the sustained figure was taken "
                                    "at a median 1.19 GHz, below the clocks this step runs at",
                     "frac_vs_sustained": round(gemm_tflops / peak_sust, 4) if (gemm_tflops and peak_sust) else None,
                     "achieved_source": "sum of 2MNK over the step's GEMM launches / their CUDA-event time, "
                                        "instrumented eager steps on the bench stream (mean of 5)",
                     "traffic": traffic_per_launch("k_gemm_tc") if args.config == "124m" else None,
                     "traffic_source": "ncu dram__bytes_read+write per k_gemm_tc launch of the 124M step, "
                                       "profiles/traffic.json (null if the kernel changed since)"},
        "kernels": kernels,
        "gemm_shapes": gemm_shapes,
        "e2e": {"value": round(world * M / e2e_s, 1), "unit": "tokens/s", "h2d_bytes_per_step": 2 * M * 4 + 32,
                "d2h_bytes_per_step": 12,
                "path": "gpt2_train_step_host from pinned host tokens: the library copies them into its pinned "
                        "staging and replays its CUDA graph of the step (tokens, targets, hyperparameters in; "
                        "loss, norm, status out)"},
        "gpu_launches": (n_kernels * args.steps) if n_kernels else None,
        "kernels_per_step": n_kernels,
        "gemm_cta_pairs": binding.lib().gemm_bf16_pairs(),
        "clocks": clk,
        "loss_last_e2e": last[0] if last else None,
        "status": status,
    }
    if world == 1 and not args.no_cpu_baseline:
        del flat
        if args.config == "1558m":
            out["cpu_baseline"] = {"value": None, "unit": "tokens/s", "cores": host_cores(), "kind": "oracle",
                                   "sample": "not run: the float64 oracle's parameter, gradient and AdamW arrays "
                                             "for 1.56B parameters need about 90 GB of host memory"}
        else:
            out["cpu_baseline"] = cpu_baseline(c, args.steps, args.warmup)
    print(json.dumps(out), flush=True)
    if pg:
        pg.destroy_process_group()


if __name__ == "__main__":
    main()
