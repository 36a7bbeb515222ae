"""Benchmark of the attention backward on GB300.

One step = one full backward (preprocess, KV-tile-parallel main kernel, dQ
convert) over the headline workload: B=4, Hq=32, Hkv=8, Nq=Nkv=8192, d=128,
bf16, causal (the Llama-3-8B shaped sweep of "[Kernel] Flash attention 2",
Liger-Kernel #275, "Benchmarking", at its 8192 point).  Inputs are seeded
synthetic N(0,1) tensors resident in HBM; O and L come from this library's
forward, outside the timed region.  Every input is larger than L2.

Metric: backward TFLOP/s counting 10*B*Hq*Nq*Nkv*d FLOPs, halved for causal.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference] [--deterministic]
    python bench.py --feature {varlen,bias,bshd} [--steps K] [--warmup W]

--feature times one of the widened paths on its own workload (one JSON line,
same metric; not part of the headline):
  varlen  packed batch of 16 Llama-3 shaped sequences, seeded lengths 512..8192, causal
  bias    the headline shape at N=4096 with a per-head bias [1, 32, N, N] and dBias
  bshd    the headline workload with every tensor stored [B, N, H, d] (strided)

Under torchrun (N > 1) every rank runs the same workload on its own GPU (the
problem shards by (batch, kv-head) groups with no exchange): weak scaling,
replicas only, with a barrier and the max over ranks of the timed region.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "attention backward TFLOP/s (bf16/fp16) and % of GB300 dense tensor peak"
PEAKS_FALLBACK = {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0}
# fa_bwd_host pipeline of the e2e leg: (batch, kv-head) groups per chunk, staging slots
HOST_CHUNK_GROUPS = 4
HOST_SLOTS = 4


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--deterministic", action="store_true")
    ap.add_argument("--n", type=int, default=8192, help="sequence length of the Llama-3 shaped workload")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--feature", choices=["varlen", "bias", "bshd"], default=None)
    return ap.parse_args()


def workload(n):
    from attn_bwd_gb300 import inputs
    return inputs.llama_gqa(n)


def flops(sh) -> float:
    f = 10.0 * sh.B * sh.Hq * sh.Nq * sh.Nkv * sh.d
    return f / 2 if sh.causal else f


def max_over_ranks(x: float, world: int, device=None) -> float:
    """The slowest rank's figure: the whole job is done only when every replica is."""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(flops_per_step: float, steps: int, world: int, ms_max: float) -> float:
    """Every replica runs the same workload (weak scaling): total FLOPs of all ranks / slowest time."""
    return world * flops_per_step * steps / (ms_max * 1e-3) / 1e12


def config_dict(sh, det, n_gpus):
    in_bytes = 2 * (2 * sh.B * sh.Hq * sh.Nq * sh.d + 3 * sh.B * sh.Hkv * sh.Nkv * sh.d) + 4 * sh.B * sh.Hq * sh.Nq
    return {"workload": f"llama3-8b-shaped GQA causal attention backward B={sh.B} Hq={sh.Hq} Hkv={sh.Hkv} "
                        f"Nq=Nkv={sh.Nq} d={sh.d} {sh.dtype}",
            "B": sh.B, "Hq": sh.Hq, "Hkv": sh.Hkv, "Nq": sh.Nq, "Nkv": sh.Nkv, "d": sh.d,
            "causal": sh.causal, "dtype": sh.dtype, "deterministic": det,
            "inputs": "seeded synthetic N(0,1), O and L from fa_fwd",
            "l2": f"inputs larger than L2 ({in_bytes / 2**20:.0f} MiB read per step, L2 = 129 MB)",
            "parallelism": "replicas" if n_gpus > 1 else "single GPU"}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return PEAKS_FALLBACK, "fallback"


def main_kernel_sha() -> str:
    h = hashlib.sha256()
    for f in ("bwd_main_persist.cu", "bwd_main.cu", "ptx.cuh", "kernels.h"):
        with open(os.path.join(ROOT, "attn_bwd_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def traffic_per_launch(sh, det):
    """DRAM bytes per main-kernel launch from the committed ncu record, if it still matches the source."""
    p = os.path.join(ROOT, "profiles", "bwd_main_traffic.txt")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        rec = json.load(f)
    if rec.get("source_sha") != main_kernel_sha() or bool(rec.get("deterministic")) != det:
        return None
    # scale a smaller capture by the tiles processed (traffic grows with the work)
    return rec["bytes_per_launch"] * flops(sh) / rec["flops_per_launch"]


class ClockSampler:
    """Samples nvidia-smi clocks and throttle reasons during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        self.out = ""
        if self.proc is not None:
            time.sleep(0.3)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self):
        rows = [r.split(",") for r in self.out.strip().splitlines() if r.count(",") >= 8]
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].strip().replace(".", "").isdigit()]
        mx = max(float(r[2]) for r in rows if r[2].strip().replace(".", "").isdigit())
        pw = [float(r[3]) for r in rows if r[3].strip().replace(".", "").isdigit()]
        loaded = [s for s, p in zip(sm, pw) if p > 300] or sm
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].strip() == "Active"})
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": mx, "reasons": reasons,
                "samples": len(rows), "power_w_max": max(pw) if pw else None}


def group_parity(grads, ref) -> dict:
    """max|gpu - oracle| / (1e-2 max|oracle| + 1e-3) per tensor (<= 1 passes), for the GPU's
    (dq, dk, dv) of one group against the oracle's dict of fp64 arrays."""
    import numpy as np
    out = {}
    for name, got in zip(("dq", "dk", "dv"), grads):
        g = got.detach().cpu().double().numpy()
        r = ref[name]
        out[name] = float(np.abs(g - r).max()) / (1e-2 * float(np.abs(r).max()) + 1e-3)
    return out


def run_cpu_baseline(sh, group=None):
    """The fp64 oracle, as it stands, on one (batch, kv-head) group of the workload (all of its
    query heads).  `group` = (q, k, v, do, dq, dk, dv) of that group as the GPU saw and produced
    them (batch 0, kv head 0): the oracle then runs on those inputs, and the GPU's gradients are
    compared with its result.  Returns (baseline, parity or None)."""
    from attn_bwd_gb300 import inputs
    from oracle import attn_ref
    G = sh.Hq // sh.Hkv
    if group is None:
        sub = inputs.Shape(1, G, 1, sh.Nq, sh.Nkv, sh.d, sh.causal, sh.dtype)
        q, k, v, do = inputs.draw(sub, 12345)
    else:
        q, k, v, do = group[:4]
    t0 = time.perf_counter()
    ref = attn_ref.backward(q, k, v, do, sh.softmax_scale, sh.causal)
    dt = time.perf_counter() - t0
    f = 10.0 * G * sh.Nq * sh.Nkv * sh.d / (2 if sh.causal else 1)
    cores = len(os.sched_getaffinity(0))
    base = {"value": f / dt / 1e12, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
            "sample": f"{G} query heads of one (batch, kv-head) group at Nq=Nkv={sh.Nq}, "
                      f"fp64 numpy/OpenBLAS, {dt:.1f} s wall"}
    return base, (group_parity(group[4:], ref) if group is not None else None)


def reference_arm(args):
    """--impl reference: the fp64 oracle timed on the host cores, one query head per step."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    from attn_bwd_gb300 import inputs
    from oracle import attn_ref
    sh = workload(args.n)
    sub = inputs.Shape(1, 1, 1, sh.Nq, sh.Nkv, sh.d, sh.causal, sh.dtype)
    q, k, v, do = inputs.draw(sub, 777)
    f = 10.0 * sh.Nq * sh.Nkv * sh.d / (2 if sh.causal else 1)
    for _ in range(args.warmup):
        attn_ref.backward(q, k, v, do, sh.softmax_scale, sh.causal)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        attn_ref.backward(q, k, v, do, sh.softmax_scale, sh.causal)
    dt = time.perf_counter() - t0
    val = f * args.steps / dt / 1e12
    cores = len(os.sched_getaffinity(0))
    line = {"metric": METRIC, "value": val, "unit": "TFLOP/s", "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1e3 * dt / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "impl": "reference", "config": config_dict(sh, args.deterministic, args.gpus),
            "cpu_baseline": {"value": val, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                             "sample": f"one query head per step (B=1, H=1, Nq=Nkv={sh.Nq}, d={sh.d}, causal)"},
            "e2e": {"value": val, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_feature(args):
    """Times one widened path (packed batch, bias with dBias, strided storage) on its workload."""
    import random

    import torch
    from attn_bwd_gb300 import _lib, inputs, torch_api

    torch.cuda.set_device(0)
    _lib.load()
    det = args.deterministic
    if args.feature == "varlen":
        rnd = random.Random(7)
        lens = [rnd.randrange(512, 8193, 64) for _ in range(16)]
        pk = inputs.Packed(tuple(lens), tuple(lens), 32, 8, 128, 1, "bf16")
        q, k, v, do = inputs.draw_packed(pk, 7, device="cuda")
        o, lse = torch_api.forward_varlen(q, k, v, pk.cu_q, pk.cu_k, pk.softmax_scale, 1)
        fl = sum(10.0 * 32 * n * n * 128 / 2 for n in lens)
        call = lambda: torch_api.backward_varlen(q, k, v, o, do, lse, pk.cu_q, pk.cu_k, pk.softmax_scale, 1, det)  # noqa: E731
        desc = {"workload": f"packed batch of 16 causal sequences, lengths {min(lens)}..{max(lens)} "
                            f"(total {sum(lens)} tokens), Hq=32 Hkv=8 d=128 bf16", "lengths": lens}
    elif args.feature == "bias":
        n = 4096
        sh = inputs.Shape(4, 32, 8, n, n, 128, True, "bf16")
        q, k, v, do = inputs.draw(sh, 8, device="cuda")
        g = torch.Generator(device="cuda").manual_seed(9)
        bias = torch.randn(1, 32, n, n, generator=g, device="cuda").to(torch.bfloat16)
        o, lse = torch_api.forward_bias(q, k, v, bias, sh.softmax_scale, True)
        fl = flops(sh)
        call = lambda: torch_api.backward_bias(q, k, v, o, do, lse, bias, sh.softmax_scale, True, det)  # noqa: E731
        desc = {"workload": f"B=4 Hq=32 Hkv=8 N={n} d=128 bf16 causal, bias [1, 32, N, N], dBias [4, 32, N, N]"}
    else:
        sh = workload(args.n)
        q, k, v, do = (t.transpose(1, 2).contiguous().transpose(1, 2) for t in inputs.draw(sh, 10, device="cuda"))
        o, lse = torch_api.forward_strided(q, k, v, sh.softmax_scale, True)
        fl = flops(sh)
        call = lambda: torch_api.backward_strided(q, k, v, o, do, lse, sh.softmax_scale, True, det)  # noqa: E731
        desc = {"workload": "headline workload stored [B, N, H, d] (strided views)"}
    for _ in range(max(3, args.warmup)):
        call()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        call()
    e1.record()
    torch.cuda.synchronize()
    if _lib.fa_last_device_error() != 0:
        raise RuntimeError("device status reported a failure")
    ms = e0.elapsed_time(e1) / args.steps
    peaks, _ = load_peaks()
    tf = fl / (ms * 1e-3) / 1e12
    print(json.dumps({"metric": METRIC, "feature": args.feature, "value": tf, "unit": "TFLOP/s", "n_gpus": 1,
                      "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
                      "dtype": "bf16", "data": "synthetic", "deterministic": det,
                      "frac_of_measured_bf16_peak": tf / float(peaks["bf16_tflops"]),
                      "note": "whole backward through the torch front end (workspace and outputs allocated per call)",
                      "config": desc}), flush=True)


def main():
    args = parse()
    if args.impl == "reference":
        reference_arm(args)
        return
    if args.feature:
        run_feature(args)
        return
    import torch
    import torch.distributed as dist
    from attn_bwd_gb300 import _lib, inputs, torch_api

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    _lib.load()
    sh = workload(args.n)
    det = args.deterministic
    B, Hq, Hkv, N, d = sh.B, sh.Hq, sh.Hkv, sh.Nq, sh.d
    dt_code = _lib.FA_BF16 if sh.dtype == "bf16" else _lib.FA_F16
    q, k, v, do = inputs.draw(sh, 1000 + rank, device=dev)
    o, lse = torch_api.forward(q, k, v, sh.softmax_scale, sh.causal)
    ws = torch_api.workspace(q, k, det)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    stream = torch.cuda.current_stream(dev)
    scale, causal = sh.softmax_scale, int(sh.causal)

    def step(ev=None):
        st = _lib.fa_bwd_preprocess(o, do, lse, B, Hq, Hkv, N, N, d, dt_code, det, ws, ws.numel(), stream)
        if ev is not None:
            ev[0].record(stream)
        st |= _lib.fa_bwd_main(q, k, v, do, dk, dv, B, Hq, Hkv, N, N, d, scale, causal, dt_code, det, ws,
                               ws.numel(), stream)
        if ev is not None:
            ev[1].record(stream)
        st |= _lib.fa_bwd_dq(q, k, v, do, dq, B, Hq, Hkv, N, N, d, scale, causal, dt_code, det, ws, ws.numel(),
                             stream)
        if st:
            raise RuntimeError(f"fa_bwd stage failed: {st}")

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    if _lib.fa_last_device_error(stream) != 0:
        raise RuntimeError("device status reported a failure during warm-up")

    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        t_start.record(stream)
        for i in range(args.steps):
            step(evs[i])
        t_end.record(stream)
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
    ms_total = t_start.elapsed_time(t_end)
    main_ms = [a.elapsed_time(b) for a, b in evs]
    ms_total = max_over_ranks(ms_total, world, dev)
    if _lib.fa_last_device_error(stream) != 0:
        raise RuntimeError("device status reported a failure in the timed region")

    fl = flops(sh)
    value = whole_job_tflops(fl, args.steps, world, ms_total)
    peaks, peaks_src = load_peaks()
    main_avg = sum(main_ms) / len(main_ms)
    # the main kernel runs all five contractions in atomic mode, four in deterministic mode
    # (dQ = dS K moves to the separate pass)
    main_flops = fl * (0.8 if det else 1.0)
    achieved = main_flops / (main_avg * 1e-3) / 1e12
    peak = float(peaks["bf16_tflops"])
    traffic = traffic_per_launch(sh, det)

    # ---- the forward that makes O and L (not part of the step): timed separately, same roofline
    fwd_iters = 10
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    f0.record(stream)
    for _ in range(fwd_iters):
        st = _lib.fa_fwd(q, k, v, o, lse, B, Hq, Hkv, N, N, d, scale, causal, dt_code, stream)
        if st:
            raise RuntimeError(f"fa_fwd failed: {st}")
    f1.record(stream)
    torch.cuda.synchronize()
    fwd_ms = f0.elapsed_time(f1) / fwd_iters
    fwd_flops = 4.0 * B * Hq * N * N * d / (2 if causal else 1)

    # ---- end to end through the C ABI with host buffers (pinned), copies inside the timed region:
    # fa_bwd_host takes the host tensors and overlaps their transfers with the computation,
    # in chunks of (batch, kv-head) groups through a ring of device staging slots
    host_in = [t.cpu().pin_memory() for t in (q, k, v, o, do, lse)]
    host_out = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in (dq, dk, dv)]
    h2d = sum(t.numel() * t.element_size() for t in host_in)
    d2h = sum(t.numel() * t.element_size() for t in host_out)
    e2e_steps = max(3, args.steps // 4)
    chunk_groups, slots = HOST_CHUNK_GROUPS, HOST_SLOTS
    st_bytes = _lib.fa_bwd_host_staging_size(B, Hq, Hkv, N, N, d, det, chunk_groups, slots)
    staging = torch.empty(st_bytes, dtype=torch.uint8, device=dev)

    def e2e_step():
        st = _lib.fa_bwd_host(*host_in, *host_out, B, Hq, Hkv, N, N, d, scale, causal, dt_code, det, chunk_groups,
                              slots, staging, st_bytes, stream)
        if st:
            raise RuntimeError(f"fa_bwd_host failed: {st}")

    e2e_step()
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1)
    e2e_ms = max_over_ranks(e2e_ms, world, dev)
    e2e_val = whole_job_tflops(fl, e2e_steps, world, e2e_ms)

    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": max(3, args.warmup), "ms_per_step": ms_total / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": sh.dtype, "data": "synthetic",
        "config": config_dict(sh, det, world),
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak, "traffic": traffic},
        "peak_source": f"{peaks_src} bf16 burst (MEASURED_PEAKS.json); main-kernel fraction of the sustained "
                       f"{peaks.get('bf16_tflops_sustained')} TFLOP/s: {achieved / float(peaks.get('bf16_tflops_sustained', peak)):.3f}",
        "percent_of_peak": 100.0 * value / peak,
        "kernel_ms": {"bwd_main_avg": main_avg, "bwd_main_min": min(main_ms),
                      "other_avg": ms_total / args.steps - main_avg},
        "e2e": {"value": e2e_val, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "api": f"fa_bwd_host (pinned host tensors, transfers overlapped in chunks of {chunk_groups} "
                       f"(batch, kv-head) groups through {slots} staging slots)"},
        "gpu_launches": 3 * args.steps,
        "forward": {"kernel": "fwd_persist_kernel (makes O and L; outside the timed step)", "ms": fwd_ms,
                    "tflops": fwd_flops / (fwd_ms * 1e-3) / 1e12,
                    "frac": fwd_flops / (fwd_ms * 1e-3) / 1e12 / peak,
                    "flops": "4*B*Hq*Nq*Nkv*d, halved for causal"},
        "clocks": clk.summary(),
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        # the oracle on batch 0 / kv head 0 of this run's own inputs; the same run's gradients of
        # that group are checked against it (the last timed step wrote dq, dk, dv)
        G = Hq // Hkv
        try:
            grp = tuple(t[0:1, 0:n].cpu() for t, n in ((q, G), (k, 1), (v, 1), (do, G), (dq, G), (dk, 1), (dv, 1)))
            base, par = run_cpu_baseline(sh, grp)
            line["cpu_baseline"] = base
            line["parity"] = dict(par, group="batch 0, kv head 0 with its query heads, full length",
                                  bound="max|gpu - oracle| / (1e-2 max|oracle| + 1e-3), <= 1 passes")
        except Exception as e:   # the measurement line is printed whatever happens here
            line["parity"] = {"error": f"{type(e).__name__}: {e}"}
            try:
                line["cpu_baseline"], _ = run_cpu_baseline(sh)
            except Exception as e2:
                line["cpu_baseline"] = None
                line["cpu_baseline_error"] = f"{type(e2).__name__}: {e2}"
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
