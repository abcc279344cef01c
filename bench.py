#!/usr/bin/env python
"""GPT-2 pretraining-step benchmark on B300: train tokens/s and MFU.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--config 124m|350m] [--no-cpu-baseline]

One step = forward (embedding, 12 pre-LN blocks, tied lm_head over the padded
vocabulary, mean cross-entropy) + full backward + global-norm clip + AdamW,
on one batch of synthetic Zipf(1.1) token streams (B=16, T=1024 for 124M).
The step runs through the C ABI of libgpt2.so, captured once in a CUDA graph
and replayed; `value` is device-timed with CUDA events over K replays with
the inputs resident in HBM.  `e2e` times gpt2_train_step_host with pinned
host token buffers (host->device copies and the loss / norm readback inside
the timed region).  Under torchrun every rank runs an independent replica of
the step (weak scaling; the replicas exchange nothing but the timing barrier).

--impl reference times the CPU oracle (plain numpy, float64) on the host
cores, one sequence of the same workload per step, on rank 0 only.
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
}
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


GEMM_SOURCES = ["gemm_tc.cu", "tc_ptx.cuh", "common.cuh", "internal.h"]
TRAFFIC_SUMMARY = os.path.join(ROOT, "profiles", "gemm_tc_dram_step_124m_b16.md")
PROF_STEPS = 5  # instrumented eager steps behind the per-kernel and per-GEMM-shape breakdown


def gemm_traffic_per_launch():
    """DRAM bytes per k_gemm_tc launch from the committed ncu summary, or None when the
    GEMM sources changed since those counters were taken (hash mismatch) or the
    summary is missing."""
    import hashlib
    try:
        text = open(TRAFFIC_SUMMARY).read()
        fields = dict(line.split(": ", 1) for line in text.splitlines()
                      if line.startswith(("traffic_bytes_per_launch:", "source_sha256:")))
        h = hashlib.sha256()
        for f in GEMM_SOURCES:
            h.update(open(os.path.join(ROOT, "pretraining_step_train_b300", "csrc", f), "rb").read())
        if h.hexdigest() != fields["source_sha256"].strip():
            return None
        return int(fields["traffic_bytes_per_launch"])
    except Exception:
        return None


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


def cpu_baseline(c, budget_s=20.0):
    """The oracle (numpy float64) on a bounded sample of the workload: tokens/s on host cores.

    The sample is a prefix of Ts positions of one sequence (causal, so a prefix
    is a self-contained sub-problem) with Ts sized from a 64-position
    calibration run so that the timed oracle step takes about budget_s."""
    import numpy as np
    from oracle import gpt2_oracle as O
    from pretraining_step_train_b300 import synth
    try:
        import threadpoolctl
        cores = max(i.get("num_threads", 1) for i in threadpoolctl.threadpool_info())
    except Exception:
        cores = os.cpu_count()
    cfg = O.Config(c["L"], c["H"], c["C"], c["V"], c["Vpad"], c["T"])
    P = synth.init_params(43, c["L"], c["C"], c["V"], c["Vpad"], c["T"], bf16_representable=True)
    tok, tgt = synth.token_batch(42, 1, c["T"], c["V"])
    t0 = time.perf_counter()
    O.train_step(P, tok[:, :64], tgt[:, :64], cfg, lr=LR, t=1)  # calibration, untimed
    per64 = time.perf_counter() - t0
    Ts = int(max(64, min(c["T"], 64 * int(budget_s / per64))))
    t0 = time.perf_counter()
    r = O.train_step(P, tok[:, :Ts], tgt[:, :Ts], cfg, lr=LR, t=1)
    dt = time.perf_counter() - t0
    return {"value": round(Ts / dt, 3), "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"prefix of {Ts} positions of 1 of {c['B']} sequences (T={c['T']}): "
                      f"forward+backward+clip+AdamW, numpy float64, {dt:.1f} s", "loss": r["loss"]}


def run_reference(args, c):
    """The oracle on the host cores, K timed steps after W warm-up steps.

    Each step is a bounded sample of the workload: forward + backward + clip +
    AdamW over a prefix of Ts positions of one sequence (causal, so a prefix is
    a self-contained sub-problem), Ts sized so that the whole run stays within
    about three minutes."""
    rank, world, _ = dist_env()
    if rank != 0:
        return
    from oracle import gpt2_oracle as O
    from pretraining_step_train_b300 import synth
    try:
        import threadpoolctl
        cores = max(i.get("num_threads", 1) for i in threadpoolctl.threadpool_info())
    except Exception:
        cores = os.cpu_count()
    cfg = O.Config(c["L"], c["H"], c["C"], c["V"], c["Vpad"], c["T"])
    P = synth.init_params(43, c["L"], c["C"], c["V"], c["Vpad"], c["T"], bf16_representable=True)
    tok, tgt = synth.token_batch(42, 1, c["T"], c["V"])
    t0 = time.perf_counter()
    O.train_step(P, tok[:, :64], tgt[:, :64], cfg, lr=LR, t=1)  # calibration, untimed
    per64 = time.perf_counter() - t0
    budget = 180.0 / max(1, args.steps + args.warmup)
    Ts = int(max(64, min(c["T"], 64 * int(budget / per64))))
    for i in range(args.warmup):
        O.train_step(P, tok[:, :Ts], tgt[:, :Ts], cfg, lr=LR, t=1)
    t0 = time.perf_counter()
    for i in range(args.steps):
        O.train_step(P, tok[:, :Ts], tgt[:, :Ts], cfg, lr=LR, t=1)
    dt = (time.perf_counter() - t0) / args.steps
    val = Ts / dt
    sample = f"prefix of {Ts} positions of 1 sequence per step (workload B={c['B']}, T={c['T']})"
    out = {"impl": "reference", "metric": METRIC, "value": round(val, 2), "unit": "tokens/s", "n_gpus": world,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 2),
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
           "data": "synthetic",
           "config": {"workload": f"GPT-2 {args.config} train step (fwd+CE+bwd+clip+AdamW)", **c,
                      "parallelism": "host cores"},
           "cpu_baseline": {"value": round(val, 2), "unit": "tokens/s", "cores": cores, "kind": "oracle",
                            "sample": sample},
           "e2e": {"value": round(val, 2), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default="124m", choices=sorted(CONFIGS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-graph", action="store_true", help="eager launches instead of a CUDA graph")
    ap.add_argument("--one-step", action="store_true",
                    help="set up, run one eager step and exit (for profiler launch lists)")
    ap.add_argument("--batch", type=int, default=0,
                    help="override the sequences per step (smaller profiler captures)")
    args = ap.parse_args()
    c = dict(CONFIGS[args.config])
    if args.batch > 0:
        c["B"] = args.batch
    if args.impl == "reference":
        run_reference(args, c)
        return
    rank, world, local = dist_env()
    import numpy as np
    import torch
    from pretraining_step_train_b300 import binding, build, synth

    torch.cuda.set_device(local)
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
    P = synth.init_params(43, L, C, V, Vpad, T, bf16_representable=True)
    flat = synth.flatten_params(P, L, C, Vpad, T)
    del P
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
    gemm_peak = peak_sust or 1400.0
    kernels = {k: {"regions": v[0], "ms": round(v[1], 4), "share": round(v[1] / max(1e-9, sum(x[1] for x in prof.values())), 4),
                   "tflops": round(v[2] / (v[1] / 1e3) / 1e12, 1) if v[1] > 0 and v[2] > 0 else None,
                   "gbs": round(v[3] / (v[1] / 1e3) / 1e9, 1) if v[1] > 0 and v[3] > 0 else None}
               for k, v in prof.items()}
    out = {
        "metric": METRIC,
        "value": round(tok_s, 1),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_max, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": round(tok_s / LLMC_124M_TOK_S, 3),
        "vs_baseline_ref": "llm.c GPT-2 124M 223k tok/s quoted on the pages (hardware not stated; context)",
        "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": f"GPT-2 {args.config} train step (fwd+CE+bwd+clip+AdamW)", "B": B, "T": T, "L": L,
                   "H": H, "C": C, "V": V, "Vpad": Vpad, "global_batch_tokens": world * M,
                   "parallelism": f"{world} independent replica(s)", "graph": graph is not None,
                   "l2": "working set (params, optimizer state, activations: ~9 GB) exceeds L2; no flush",
                   "tokens": "Zipf(1.1) streams over the vocab, targets shifted by one"},
        "mfu": {"flops_per_token": fpt, "convention": "6N+6LCT, N padded incl. wpe",
                "vs_nominal_2250": round(achieved_tflops / NOMINAL_BF16_TFLOPS, 4),
                "vs_measured_burst": round(achieved_tflops / peak_burst, 4) if peak_burst else None,
                "achieved_tflops": round(achieved_tflops, 1)},
        "roofline": {"bound": "tensor", "kernel": "k_gemm_tc (all Linears + classifier logits)",
                     "achieved": round(gemm_tflops, 1) if gemm_tflops else None,
                     "peak": gemm_peak, "unit": "TFLOP/s",
                     "frac": round(gemm_tflops / gemm_peak, 4) if gemm_tflops else None,
                     "peak_source": "MEASURED_PEAKS.json bf16_tflops_sustained (kernel timed inside a long step)",
                     "achieved_source": "sum of 2MNK over the step's GEMM launches / their CUDA-event time, "
                                        "instrumented eager steps on the bench stream (mean of 5)",
                     "traffic": gemm_traffic_per_launch(),
                     "traffic_source": "ncu dram__bytes_read+write per k_gemm_tc launch, "
                                       "profiles/gemm_tc_dram_step_124m_b16.md (null if the kernel changed)"},
        "kernels": kernels,
        "gemm_shapes": gemm_shapes,
        "e2e": {"value": round(world * M / e2e_s, 1), "unit": "tokens/s", "h2d_bytes_per_step": 2 * M * 4 + 32,
                "d2h_bytes_per_step": 12,
                "path": "gpt2_train_step_host from pinned host tokens: the library copies them into its pinned "
                        "staging and replays its CUDA graph of the step (tokens, targets, hyperparameters in; "
                        "loss, norm, status out)"},
        "gpu_launches": (n_kernels * args.steps) if n_kernels else None,
        "kernels_per_step": n_kernels,
        "clocks": clk,
        "loss_last_e2e": last[0] if last else None,
        "status": status,
    }
    if world == 1 and not args.no_cpu_baseline:
        del flat
        out["cpu_baseline"] = cpu_baseline(c)
    print(json.dumps(out), flush=True)
    if pg:
        pg.destroy_process_group()


if __name__ == "__main__":
    main()
