#!/usr/bin/env python
"""Throughput of one GPT-2 training step (forward + zero_grad + backward +
AdamW) on B300 GPUs, through libgpt2b300's C ABI.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
    python bench.py --impl reference ...     # the CPU oracle, timed alone

Default workload: GPT-2 124M (L=12, C=768, NH=12, V=50257 padded to 50304),
fp32, B=4, T=64 -- the configuration of the llm.c console log (page
«千行C代码训完GPT-2», section «快速入门»: 124,439,808 parameters, B*T = 256,
about 1.3 s per step on an M3 Max CPU).  Inputs are synthetic: seeded
Zipf(1.1) token streams and a seeded N(0, 0.02) init.

Prints one JSON line (rank 0).  ``value`` is whole-job tokens/s with the
token batches resident in HBM; ``e2e`` is the same metric through
``gpt2_train_step`` with pinned host token arrays copied every step and the
loss read back every step.  Multi-GPU runs are independent replicas (the path
is not sharded across GPUs), so ``scaling`` is weak.
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "GPT-2 124M train tokens/sec (fwd+bwd+AdamW) on 1 B300; MFU; per-kernel HBM GB/s"
DEFAULT_WORKLOAD = "gpt2_124m_B4_T64_fp32"
L2_BYTES = 126 * 1024 * 1024


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        p = json.load(open(path))
        return {"hbm_gbs": p["hbm_gbs"], "bf16_tflops": p["bf16_tflops"],
                "bf16_tflops_sustained": p.get("bf16_tflops_sustained"), "sm_max_mhz": p.get("sm_max_mhz", 2032.0),
                "source": "measured"}
    return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0, "sm_max_mhz": 2032.0,
            "source": "fallback"}


def flops_per_token(w) -> float:
    """Algorithmic training FLOPs per token: 3 x forward, causal attention
    counts only keys t2 <= t, the LM head over the real vocabulary."""
    L, C, T, V = w.num_layers, w.channels, w.T, w.vocab_size
    return 3.0 * (L * (24.0 * C * C + 4.0 * C * (T + 1) / 2.0) + 2.0 * C * V)


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0, "note": "nvidia-smi unavailable"}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), parts[5:9]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i, v in enumerate(r[2]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows)}


# ---------------------------------------------------------------------------
# CPU oracle timing (rank 0)
# ---------------------------------------------------------------------------
def oracle_sample_run(w, seconds_target: float = 12.0, max_steps: int = 50, B_sample: int | None = None):
    """Times full oracle training steps (forward, zero_grad, backward, AdamW)
    on B_sample sequences of the workload's batch until seconds_target has
    passed.  Returns (tokens/s, steps, tokens per step, seconds)."""
    from oracle import ref

    B = B_sample or w.B
    m = ref.RefModel(ref.config_from(w), B, w.T, np.float32)
    m.set_params(synth.init_params(w))
    inp, tgt = synth.batch(w, step=0)
    inp, tgt = inp[:B].copy(), tgt[:B].copy()
    steps = 0
    t0 = time.perf_counter()
    while True:
        m.step(inp, tgt, steps + 1, lr=w.lr)
        steps += 1
        el = time.perf_counter() - t0
        if el >= seconds_target or steps >= max_steps:
            break
    m.close()
    return B * w.T * steps / el, steps, B * w.T, el


def oracle_one_thread(w, seconds: float = 4.0):
    """The oracle on one host thread, beside the all-cores figure: the same
    kind of sample (training steps on one sequence of the batch) in a child
    process started with OMP_NUM_THREADS=1, which OpenMP reads at start-up.
    Returns the child's JSON record, or None when it did not complete."""
    cmd = [sys.executable, os.path.abspath(__file__), "--workload", w.name, "--oracle-one-thread", str(seconds)]
    try:
        out = subprocess.run(cmd, env=dict(os.environ, OMP_NUM_THREADS="1"), capture_output=True, text=True,
                             timeout=60.0 + 10.0 * seconds)
        return json.loads(out.stdout.strip().splitlines()[-1]) if out.returncode == 0 else None
    except (subprocess.TimeoutExpired, ValueError, IndexError):
        return None


def cpu_cores() -> int:
    n = int(os.environ.get("OMP_NUM_THREADS", "0") or 0)
    return n if n > 0 else len(os.sched_getaffinity(0))


# ---------------------------------------------------------------------------
def run_reference(args, w):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    # each step: one full oracle training step on one sequence of the batch
    B_sample = 1 if w.BT >= 256 else w.B
    from oracle import ref

    m = ref.RefModel(ref.config_from(w), B_sample, w.T, np.float32)
    m.set_params(synth.init_params(w))
    # exactly the K timed and W warm-up steps asked for; each is one full
    # oracle training step on a bounded sample of the batch
    steps = args.steps
    warm = args.warmup
    batches = [synth.batch(w, step=s) for s in range(warm + steps)]
    for s in range(warm):
        m.step(batches[s][0][:B_sample], batches[s][1][:B_sample], s + 1, lr=w.lr)
    t0 = time.perf_counter()
    for s in range(steps):
        i, t = batches[warm + s]
        m.step(i[:B_sample], t[:B_sample], warm + s + 1, lr=w.lr)
    el = time.perf_counter() - t0
    m.close()
    tok = B_sample * w.T * steps
    value = tok / el
    sample = (f"{steps} oracle training steps (forward, zero_grad, backward, AdamW) on {B_sample} of the "
              f"{w.B} sequences of each batch (T={w.T}); tokens/s counts the tokens processed")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": steps, "warmup": warm, "ms_per_step": 1000.0 * el / steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": workload_config(w, args.gpus),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cpu_cores(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def workload_config(w, n_gpus):
    return {"workload": w.name, "B": w.B, "T": w.T, "tokens_per_step_per_gpu": w.BT,
            "global_batch_tokens": w.BT * n_gpus, "precision": w.precision, "tokens": f"{w.tokens} (seeded)",
            "parallelism": "replicas" if n_gpus > 1 else "single",
            "l2": "no flush: each step streams params+grads+AdamW moments (> 126 MB L2)"}


def measure_tf32_peak():
    """Dense TF32 tensor-core rate of this GPU, measured the way the bf16 peak
    is: torch.matmul (cuBLAS) of two 8192 x 8192 fp32 matrices with TF32
    allowed, 2 * 8192^3 FLOPs, best of 10 (CUDA events).  TFLOP/s."""
    import torch

    n = 8192
    prev = torch.backends.cuda.matmul.allow_tf32
    torch.backends.cuda.matmul.allow_tf32 = True
    try:
        a = torch.randn(n, n, device="cuda")
        b = torch.randn(n, n, device="cuda")
        c = torch.empty(n, n, device="cuda")
        for _ in range(3):
            torch.matmul(a, b, out=c)
        best = float("inf")
        for _ in range(10):
            s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s.record()
            torch.matmul(a, b, out=c)
            e.record()
            e.synchronize()
            best = min(best, s.elapsed_time(e))
        del a, b, c
        torch.cuda.empty_cache()
    finally:
        torch.backends.cuda.matmul.allow_tf32 = prev
    return 2.0 * n ** 3 / (best * 1e-3) / 1e12


KERNEL_CLASSES = ("gemm", "adamw", "xent", "layernorm", "attn_fwd", "attn_bwd", "encoder")


def measure(w, K, W, peaks, g, rank=0, world=1, barrier=lambda: None, reduce_max=lambda x: x, with_e2e=True):
    """Times K graph-replayed training steps of workload w (after W warm-up
    steps) with CUDA events on the handle's stream, samples the SM clocks
    during them, times every kernel class with events around each launch,
    and (with_e2e) times K steps through gpt2_train_step from pinned host
    tokens with the loss read back every step."""
    import torch

    model = g.GPT2(w, seed=synth.INIT_SEED)
    stream = model.stream
    # token batches for every step, resident in HBM before timing (distinct per rank)
    nb = W + K
    host_in = np.empty((nb, w.B, w.T), np.int32)
    host_tg = np.empty((nb, w.B, w.T), np.int32)
    for s in range(nb):
        host_in[s], host_tg[s] = synth.batch(w, step=rank * 1_000_003 + s)
    d_in = torch.from_numpy(host_in).cuda()
    d_tg = torch.from_numpy(host_tg).cuda()
    torch.cuda.synchronize()

    t = 0
    for s in range(W):
        t += 1
        model.train_step_device(d_in[s], d_tg[s], t, lr=w.lr)
    torch.cuda.synchronize()
    barrier()

    local = torch.cuda.current_device()
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.25)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    barrier()
    start.record(stream)
    for s in range(K):
        t += 1
        model.train_step_device(d_in[W + s], d_tg[W + s], t, lr=w.lr)
    end.record(stream)
    torch.cuda.synchronize()
    barrier()
    clk = clocks.stop()
    ms = reduce_max(start.elapsed_time(end))
    launches_per_step = model.last_launch_count()
    last_loss = model.sync()
    ms_per_step = ms / K
    value = world * w.BT * K / (ms / 1000.0)

    # per-kernel-class timing (events around each launch, direct launches)
    kinds = {}
    ksteps = min(K, 5)
    for kind in KERNEL_CLASSES:
        g.gpt2_kernel_timer(model.h, kind)
        for s in range(ksteps):
            t += 1
            model.train_step_device(d_in[s % nb], d_tg[s % nb], t, lr=w.lr)
        kms, kn, kwork = g.gpt2_kernel_timer_read(model.h)
        kinds[kind] = {"ms_per_step": kms / ksteps, "launches_per_step": kn / ksteps,
                       "work_per_launch": kwork / max(kn, 1), "avg_launch_ms": kms / max(kn, 1)}
    g.gpt2_kernel_timer(model.h, "off")
    dom = max(kinds, key=lambda k: kinds[k]["ms_per_step"])
    roof = roofline_for(dom, kinds[dom], peaks, w)
    # every timed class against its own bound (the dominant one is `roofline`)
    rooflines = {kd: roofline_for(kd, kinds[kd], peaks, w) for kd in kinds if kinds[kd]["launches_per_step"] > 0}

    e2e = None
    if with_e2e:
        # end to end: pinned host tokens, H2D every step, loss read back every step
        pin_in = torch.from_numpy(host_in).pin_memory().numpy()
        pin_tg = torch.from_numpy(host_tg).pin_memory().numpy()
        for s in range(min(W, 3)):
            t += 1
            model.train_step(pin_in[s], pin_tg[s], t, lr=w.lr)
        barrier()
        t0 = time.perf_counter()
        for s in range(K):
            t += 1
            model.train_step(pin_in[W + s], pin_tg[W + s], t, lr=w.lr)
        e2e_s = reduce_max(time.perf_counter() - t0)
        barrier()
        e2e = {"value": world * w.BT * K / e2e_s, "unit": "tokens/s", "h2d_bytes_per_step": 2 * w.BT * 4,
               "d2h_bytes_per_step": 4, "api": "gpt2_train_step (host tokens, loss returned every step)"}
    model.close()
    del d_in, d_tg
    torch.cuda.empty_cache()
    f_tok = flops_per_token(w)
    return {
        "value": value, "ms_per_step": ms_per_step, "launches_per_step": launches_per_step, "clocks": clk,
        "roofline": roof, "rooflines": rooflines, "kernels": kinds, "e2e": e2e, "last_loss": last_loss,
        "mfu": {"vs_bf16_dense_measured": value * f_tok / (peaks["bf16_tflops"] * 1e12 * world),
                "vs_bf16_dense_sustained_measured": (value * f_tok / (peaks["bf16_tflops_sustained"] * 1e12 * world)
                                                     if peaks.get("bf16_tflops_sustained") else None),
                "vs_tf32_dense_measured": value * f_tok / (peaks["tf32_tflops"] * 1e12 * world),
                "flops_per_token": f_tok},
    }


# the T = 1024 bf16 workloads, timed after the headline in a default single-GPU run
EXTRA_WORKLOADS = ("gpt2_124m_B16_T1024_bf16", "gpt2_350m_B8_T1024_bf16", "gpt2_774m_B4_T1024_bf16")


def run_ours(args, w):
    import torch

    import gpt_train_step_02_b300 as g

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    def barrier():
        if dist is not None:
            dist.barrier()

    def reduce_max(v):
        if dist is None:
            return v
        x = torch.tensor([v], device="cuda", dtype=torch.float64)
        dist.all_reduce(x, op=dist.ReduceOp.MAX)
        return float(x.item())

    peaks = load_peaks()
    peaks["tf32_tflops"] = measure_tf32_peak()
    peaks["tf32_source"] = "measured in this run: torch.matmul fp32 8192^3 with TF32 allowed, best of 10"
    res = measure(w, args.steps, args.warmup, peaks, g, rank, world, barrier, reduce_max)
    extra = {}
    if world == 1 and not args.no_extra:
        for name in EXTRA_WORKLOADS:
            if name == w.name:
                continue
            xw = synth.WORKLOADS[name]
            r = measure(xw, args.extra_steps, 3, peaks, g, with_e2e=False)
            extra[name] = {
                "config": workload_config(xw, 1), "tokens_per_s": r["value"], "ms_per_step": r["ms_per_step"],
                "steps": args.extra_steps, "warmup": 3, "mfu": r["mfu"], "roofline": r["roofline"],
                "rooflines": r["rooflines"], "kernels": r["kernels"], "clocks": r["clocks"],
                "gpu_launches_per_step": r["launches_per_step"],
                "last_loss": r["last_loss"],
            }

    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return 0
    cpu = None
    if not args.no_cpu_baseline and world == 1:
        v, steps, tok, el = oracle_sample_run(w, seconds_target=args.cpu_seconds)
        cpu = {"value": v, "unit": "tokens/s", "cores": cpu_cores(), "kind": "oracle",
               "sample": f"{steps} full oracle training step(s) of the same workload ({tok} tokens each), "
                         f"{el:.1f} s of CPU time",
               "one_thread": oracle_one_thread(w)}
    line = {
        "metric": METRIC, "value": res["value"], "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": res["ms_per_step"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32" if w.precision == "fp32" else "bf16", "data": "synthetic",
        "config": workload_config(w, world),
        "mfu": res["mfu"],
        "roofline": res["roofline"],
        "rooflines": res["rooflines"],
        "cpu_baseline": cpu,
        "e2e": res["e2e"],
        "gpu_launches": int(res["launches_per_step"] * args.steps),
        "clocks": res["clocks"],
        "kernels": res["kernels"],
        "last_loss": res["last_loss"],
        "peaks": {k: peaks[k] for k in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained", "tf32_tflops", "source",
                                        "tf32_source")},
        "workloads_t1024": extra,
    }
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


# Sources of each kernel class: DRAM traffic recorded by ncu stays valid only
# while these files are unchanged.
# Sources of each kernel class: DRAM traffic recorded by ncu stays valid only
# while these are unchanged -- whole files for the matmuls, the named
# functions (their full definitions) for the others, so that an edit to an
# unrelated kernel in the same file does not invalidate a record.
KERNEL_SOURCES = {
    "gemm": ["gemm_common.cuh", "k_gemm_tc.cuh", "k_gemm_bf16.cuh"],
    "adamw": [("k_misc.cuh", "adamw_f4"), ("k_misc.cuh", "adamw_kernel"), ("k_misc.cuh", "adamw_rows_kernel"),
              ("k_misc.cuh", "adamw_sorted_rows_kernel")],
    "xent": [("k_xent.cuh", "online_merge"), ("k_xent.cuh", "xent_fused_kernel"), ("k_xent.cuh", "xent_bf16_kernel")],
    "layernorm": [("k_layernorm.cuh", "layernorm_fwd_kernel"), ("k_layernorm.cuh", "layernorm_bwd_kernel"),
                  ("k_layernorm.cuh", "layernorm_bwd_stride_kernel"), ("k_misc.cuh", "col_finish_kernel")],
    "encoder": [("k_misc.cuh", "encoder_fwd_kernel")],
    "attn_fwd": ["k_attention_tc.cuh", "k_attention_tf32.cuh"],
    "attn_bwd": ["k_attention_tc.cuh", "k_attention_tf32.cuh"],
}


def function_source(text, name):
    """The definition of function `name` in a CUDA source: from the line that
    declares it to the brace closing its body."""
    import re

    m = re.search(r"^[^\n]*\b" + re.escape(name) + r"\(", text, re.M)
    if not m:
        raise KeyError(name)
    i = text.index("{", m.end())
    depth = 0
    for j in range(i, len(text)):
        depth += {"{": 1, "}": -1}.get(text[j], 0)
        if depth == 0:
            return text[m.start():j + 1]
    raise ValueError(name)


def kernel_source_sha(kind):
    import hashlib

    h = hashlib.sha256()
    for src in KERNEL_SOURCES.get(kind, []):
        f, fn = (src, None) if isinstance(src, str) else src
        with open(os.path.join(ROOT, "gpt_train_step_02_b300", "csrc", f), encoding="utf-8") as fh:
            text = fh.read()
        h.update((text if fn is None else function_source(text, fn)).encode())
    return h.hexdigest()[:16]


def recorded_traffic(kind, w):
    """DRAM bytes per launch of this kernel class from the committed ncu
    capture (profiles/roofline_traffic.json), or None when there is none or
    the kernel sources changed since it was taken."""
    path = os.path.join(ROOT, "profiles", "roofline_traffic.json")
    if not os.path.exists(path):
        return None
    rec = json.load(open(path)).get(w.name, {}).get(kind)
    if not rec or rec.get("source_sha") != kernel_source_sha(kind):
        return None
    return rec["dram_bytes_per_launch"]


def tf32_peak(peaks):
    """Dense TF32 rate for the 3xTF32 kernels: the rate measured in this run
    (cuBLAS, TF32 allowed), else the bf16 burst figure x the nominal ratio."""
    if peaks.get("tf32_tflops"):
        return peaks["tf32_tflops"], peaks["tf32_source"]
    return (peaks["bf16_tflops"] * 1.1 / 2.25,
            f"{peaks['source']} bf16 dense burst x nominal tf32/bf16 ratio 1.1/2.25")


def bf16_peak(peaks):
    """Dense bf16 rate for kernels timed inside a long graph-replayed step at
    the power cap: the sustained figure when it was measured, else the burst."""
    if peaks.get("bf16_tflops_sustained"):
        return peaks["bf16_tflops_sustained"], f"{peaks['source']} bf16 dense sustained"
    return peaks["bf16_tflops"], f"{peaks['source']} bf16 dense burst"


def tensor_line(kernel, achieved, peaks, w, three_mmas, traffic=None):
    """A tensor-bound roofline entry: 3xTF32 kernels against the TF32 rate
    (three MMAs per product, so a third of it is their ceiling), bf16 kernels
    against the sustained bf16 rate (the burst fraction alongside)."""
    if three_mmas:
        peak, src = tf32_peak(peaks)
        return {"kernel": kernel, "bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak, "frac_of_3xtf32_ceiling": 3.0 * achieved / peak, "traffic": traffic,
                "peak_source": src + "; 3 MMAs per product"}
    peak, src = bf16_peak(peaks)
    return {"kernel": kernel, "bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
            "frac": achieved / peak, "frac_of_burst": achieved / peaks["bf16_tflops"], "traffic": traffic,
            "peak_source": src}


# B300 HBM3e nominal bandwidth (the datasheet figure; the measured copy rate
# is the roofline peak, this one is reported beside it)
HBM_NOMINAL_GBS = 7700.0


def roofline_for(kind, k, peaks, w):
    if kind == "gemm":
        # fp32 matmuls run as 3xTF32 on tcgen05 kind::tf32, bf16 ones on kind::f16
        achieved = k["work_per_launch"] / (k["avg_launch_ms"] * 1e-3) / 1e12
        return tensor_line("matmul (all tcgen05 launches of the step)", achieved, peaks, w, w.precision == "fp32",
                           recorded_traffic(kind, w))
    if kind in ("attn_fwd", "attn_bwd"):
        # the timer's work figure is FLOPs: 4 (forward) or 8 (backward) x B NH hs T(T+1)/2
        achieved = k["work_per_launch"] / (k["avg_launch_ms"] * 1e-3) / 1e12
        hs = w.channels // w.num_heads
        if w.precision == "bf16" and hs == 64 and w.T % 128 == 0:  # tcgen05 kind::f16 products
            return tensor_line(kind, achieved, peaks, w, False, recorded_traffic(kind, w))
        if w.precision == "fp32" and hs == 64 and w.T <= 64:  # tcgen05 kind::tf32, 3xTF32 products
            return tensor_line(kind, achieved, peaks, w, True, recorded_traffic(kind, w))
        # CUDA-core fp32: 148 SMs x 128 FMA lanes x 2 FLOPs x the maximum SM clock
        peak = 148 * 128 * 2 * peaks["sm_max_mhz"] * 1e6 / 1e12
        return {"kernel": kind, "bound": "alu", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak, "traffic": None,
                "peak_source": "fp32 FMA issue rate: 148 SMs x 128 lanes x 2 FLOPs x max SM clock"}
    achieved = k["work_per_launch"] / (k["avg_launch_ms"] * 1e-3) / 1e9
    return {"kernel": kind, "bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
            "frac": achieved / peaks["hbm_gbs"], "frac_of_nominal": achieved / HBM_NOMINAL_GBS,
            "traffic": recorded_traffic(kind, w), "peak_source": peaks["source"]}


# kernel-name fragments of each class in an ncu capture
TRAFFIC_KERNELS = {"gemm": ("gemm_tf32x3", "gemm_bf16"),
                   "adamw": ("adamw_kernel", "adamw_rows_kernel", "adamw_sorted_rows_kernel"),
                   "xent": ("xent_fused_kernel", "xent_bf16_kernel"),
                   "layernorm": ("layernorm_fwd_kernel", "layernorm_bwd_kernel", "layernorm_bwd_stride_kernel"),
                   "encoder": ("encoder_fwd_kernel",),
                   "attn_fwd": ("attn_fwd_tc_kernel", "attn_fwd_tf32_kernel"),
                   "attn_bwd": ("attn_bwd_ld_bf16_kernel", "attn_bwd_dkv_tc_kernel", "attn_bwd_dq_tc_kernel",
                                "attn_bwd_tf32_kernel")}
# Classes whose timed launch is one layer's attention op: one launch of each of
# the class's kernels that the path takes (the bf16 backward: the (-lse log2 e,
# -D) pass, dK/dV and dQ).  Their record is the sum, over the kernels seen in
# the capture, of each kernel's mean DRAM bytes per launch.
TRAFFIC_PER_OP = ("attn_fwd", "attn_bwd")
BYTE_UNITS = {"byte": 1.0, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9, "KB": 1e3, "MB": 1e6, "GB": 1e9}


def record_traffic(csv_path, w, kind="gemm"):
    """Average DRAM bytes (read + write) per launch of one kernel class, from
    an ncu capture of the launches of whole steps of workload w
    (``--metrics dram__bytes_read.sum,dram__bytes_write.sum --csv``), stored
    in profiles/roofline_traffic.json with the hash of the kernel sources it
    was taken on.  Every step launches the same sequence, so any run of one
    step's launch count covers each launch of a step once.  For the attention
    classes (TRAFFIC_PER_OP) one timed launch is one layer's op, several
    kernels: the record sums the kernels' means."""
    import csv as _csv

    rows = list(_csv.DictReader(l for l in open(csv_path) if not l.startswith("==")))
    launches = {}
    for r in rows:
        name = r["Kernel Name"]
        hit = [k for k in TRAFFIC_KERNELS[kind] if k in name]
        if not hit:
            continue
        m = r["Metric Name"]
        if m not in ("dram__bytes_read.sum", "dram__bytes_write.sum"):
            continue
        v = float(r["Metric Value"].replace(",", "")) * BYTE_UNITS[r["Metric Unit"]]
        launches.setdefault(int(r["ID"]), {"kernel": hit[0]})[m] = v
    full = [d for d in launches.values() if len(d) == 3]
    if not full:
        print(f"no {kind} launches with both DRAM metrics in {csv_path}", file=sys.stderr)
        return 1
    if kind in TRAFFIC_PER_OP:
        by_kernel = {}
        for d in full:
            by_kernel.setdefault(d["kernel"], []).append(d["dram__bytes_read.sum"] + d["dram__bytes_write.sum"])
        per_launch = sum(sum(v) / len(v) for v in by_kernel.values())
    else:
        per_launch = sum(d["dram__bytes_read.sum"] + d["dram__bytes_write.sum"] for d in full) / len(full)
    path = os.path.join(ROOT, "profiles", "roofline_traffic.json")
    data = json.load(open(path)) if os.path.exists(path) else {}
    data.setdefault(w.name, {})[kind] = {
        "dram_bytes_per_launch": per_launch,
        "launches_captured": len(full),
        "source_sha": kernel_source_sha(kind),
        "capture": os.path.basename(csv_path),
    }
    with open(path, "w") as fh:
        json.dump(data, fh, indent=1, sort_keys=True)
        fh.write("\n")
    print(json.dumps({"workload": w.name, "kind": kind, "dram_bytes_per_launch": per_launch, "launches": len(full)}))
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(synth.WORKLOADS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-extra", action="store_true", help="skip the T = 1024 bf16 workloads after the headline")
    ap.add_argument("--extra-steps", type=int, default=10)
    ap.add_argument("--record-traffic", metavar="NCU_CSV",
                    help="store the DRAM bytes per launch of one kernel class (--traffic-kind) from an ncu capture "
                         "of --workload and exit")
    ap.add_argument("--traffic-kind", default="gemm", choices=sorted(TRAFFIC_KERNELS))
    ap.add_argument("--oracle-one-thread", type=float, metavar="SECONDS",
                    help="time the oracle alone for about SECONDS on one sequence of --workload's batch, print "
                         "one JSON record and exit (the cpu_baseline's one-thread figure runs this with "
                         "OMP_NUM_THREADS=1)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)  # at least three untimed warm-up steps
    w = synth.WORKLOADS[args.workload]
    if args.oracle_one_thread is not None:
        v, steps, tok, el = oracle_sample_run(w, seconds_target=args.oracle_one_thread, B_sample=1)
        print(json.dumps({"value": v, "unit": "tokens/s", "cores": cpu_cores(),
                          "sample": f"{steps} oracle training step(s) on one sequence ({tok} tokens each), "
                                    f"{el:.1f} s"}))
        return 0
    if args.record_traffic:
        return record_traffic(args.record_traffic, w, args.traffic_kind)
    if args.impl == "reference":
        return run_reference(args, w)
    return run_ours(args, w)


if __name__ == "__main__":
    sys.exit(main())
