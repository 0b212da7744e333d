"""Benchmark: MM-DiT joint attention (QK-RMSNorm + softmax attention) fwd+bwd on GB300.

One step = jattn_fwd_train + jattn_bwd_train over one batch of the 512 px
workload (B=16, H=12, N = 1024 image + 77 text tokens, d=64), inputs resident
in HBM: a training step's attention, whose forward keeps the normalised q / k
and the rows' 1/rms for its backward.
The metric is TFLOP/s of the fwd+bwd pair at 14*B*H*N^2*d FLOP per step
(forward 4 B H N^2 d; backward 10 B H N^2 d, the five N x N x d products
including the recomputed scores), with the true N, so tile padding counts
against the kernels.

Prints ONE JSON line (rank 0).  Multi-GPU (torchrun): every rank runs its own
replica of the workload (the path has no exchange step: (b, h) pairs are
independent), a barrier + synchronize brackets the timed region, the time is
the max over ranks and the value is the work of all ranks over that time.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
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
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "joint-attn fwd+bwd TFLOP/s and % of GB300 dense-BF16 peak at B16 H12 N1101 d64"
UNIT = "TFLOP/s"
WORKLOAD = "512px"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# Rotating input sets: 3 x (q, k, v, dout, out, lse, dq, dk, dv) at 512 px is
# about 3 x 245 MB, well beyond the 129 MB L2, so no step starts warm.
N_SETS = 3
FWD_RESULTS = ("out", "lse")  # written by the forward, downloaded while the backward runs


def flops_fwd(B, H, N, d):
    return 4.0 * B * H * N * N * d


def flops_bwd(B, H, N, d):
    return 10.0 * B * H * N * N * d


# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) per launch, stored from one ncu capture
# of the 512 px workload and keyed to the kernel source they were taken on: a changed source
# reports null until it is captured again.  The line labels the figure as stored, with its capture.
_CAPTURE = ("ncu --set full --clock-control none -k regex:attn_ -s 2 -c 2, "
            "python bench.py --steps 2 --warmup 3 --no-cpu-baseline --no-e2e --no-per-config")
NCU_TRAFFIC = {
    "attn_bwd": {"bytes": 197.58464e6 + 64.802304e6, "source": "attn_bwd.cu", "sha1": "f7d6bf58b915",
                 "capture": _CAPTURE},
    "attn_fwd": {"bytes": 81.322496e6 + 57.446144e6, "source": "attn_fwd.cu", "sha1": "1e3f9884fd9f",
                 "capture": _CAPTURE},
}


def ncu_traffic(kernel):
    import hashlib

    rec = NCU_TRAFFIC.get(kernel)
    if rec is None:
        return None
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "joint_attention_gb300", "csrc", rec["source"])
    try:
        cur = hashlib.sha1(open(path, "rb").read()).hexdigest()[:12]
    except OSError:
        return None
    return rec["bytes"] if cur == rec["sha1"] else None


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            data = json.load(open(path))
            flat = {}

            def walk(o):
                if isinstance(o, dict):
                    for key, val in o.items():
                        if isinstance(val, (int, float)) and key in FALLBACK_PEAKS:
                            flat[key] = float(val)
                        walk(val)
            walk(data)
            if "bf16_tflops" in flat and "hbm_gbs" in flat:
                flat.setdefault("bf16_tflops_sustained", flat["bf16_tflops"])
                cl = data.get("clocks_under_load") if isinstance(data, dict) else None
                if isinstance(cl, dict) and isinstance(cl.get("sm_mhz_median"), (int, float)):
                    flat["sustained_sm_mhz"] = float(cl["sm_mhz_median"])
                return flat, "measured"
        except (OSError, ValueError):
            pass
    return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.file = None
        self.window = None  # (t0, t1) wall-clock seconds of the timed loop

    def mark(self, t0: float, t1: float):
        self.window = (t0, t1)

    def __enter__(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"], stdout=self.file,
                                         stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, ValueError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.proc is None or self.file is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.file.flush()
        rows = []
        with open(self.file.name) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 10:
                    rows.append(parts)
        os.unlink(self.file.name)
        scope = "all samples"
        if self.window is not None:
            import datetime

            def stamp(r):
                try:
                    return datetime.datetime.strptime(r[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                except ValueError:
                    return None
            inside = [r for r in rows if stamp(r) is not None and self.window[0] <= stamp(r) <= self.window[1]]
            if inside:
                rows, scope = inside, "timed loop"
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[2]) for r in rows if num(r[2]) is not None]
        mx = [num(r[3]) for r in rows if num(r[3]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[6 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows), "scope": scope,
                "power_w_median": statistics.median([num(r[4]) for r in rows if num(r[4]) is not None] or [0])}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def aggregate_over_ranks(ms_total, steps, fl_step, world, dist=None, device="cpu"):
    """The job's timed-loop duration (the slowest rank's) and whole-job throughput in TFLOP/s:
    every rank ran `steps` steps of `fl_step` FLOP on its own replica."""
    if world > 1:
        import torch

        t = torch.tensor([ms_total], device=device, dtype=torch.float64)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms_total = float(t.item())
    return ms_total, fl_step * steps * world / (ms_total * 1e-3) / 1e12


def cpu_oracle_sample(B, H, N, d, seed, budget_s: float, max_heads: int):
    """Times the float64 oracle on whole heads of the workload until budget_s."""
    import numpy as np

    import oracle
    from joint_attention_gb300.inputs import make_inputs

    inp = make_inputs(1, 1, N, d, seed=seed)
    heads = 0
    t0 = time.perf_counter()
    while heads < max_heads:
        oracle.joint_attention_bwd(inp.q, inp.k, inp.v, inp.gq, inp.gk, inp.dout)
        heads += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    el = time.perf_counter() - t0
    fl = (flops_fwd(1, 1, N, d) + flops_bwd(1, 1, N, d)) * heads
    del np
    return {"value": fl / el / 1e12, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"{heads} head(s) of the {WORKLOAD} workload (N={N}, d={d}) fwd+bwd in float64 NumPy, "
                      f"materialised N x N scores, {el:.2f} s; BLAS threads = all host cores"}


def cpu_oracle_per_config(budget_s: float):
    """The float64 oracle timed on each workload of the parity suite, on the host cores.

    A sample of whole (b, h) heads of each workload runs through the oracle (fwd+bwd for the
    training workloads; the forward for the CFG sampling workload) until budget_s has passed or
    every head is done; the time of the full workload is the per-head time times its heads (times
    its denoising steps for CFG sampling), stated as extrapolated unless every head ran."""
    import oracle
    from joint_attention_gb300.inputs import CONFIGS, make_inputs

    res = {}
    for name, c in CONFIGS.items():
        fwd_only = c.mode == "cfg_fwd"
        inp = make_inputs(1, 1, c.N, c.d, seed=c.seed, value_scale=c.value_scale, with_dout=not fwd_only)
        heads_total = c.B * c.H
        heads = 0
        t0 = time.perf_counter()
        while heads < heads_total:
            if fwd_only:
                oracle.joint_attention_fwd(inp.q, inp.k, inp.v, inp.gq, inp.gk)
            else:
                oracle.joint_attention_bwd(inp.q, inp.k, inp.v, inp.gq, inp.gk, inp.dout)
            heads += 1
            if time.perf_counter() - t0 >= budget_s:
                break
        el = time.perf_counter() - t0
        fl_head = flops_fwd(1, 1, c.N, c.d) + (0.0 if fwd_only else flops_bwd(1, 1, c.N, c.d))
        steps = c.steps if fwd_only else 1
        full_s = el / heads * heads_total * steps
        res[name] = {"value": fl_head * heads / el / 1e12, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
                     "full_workload_s": full_s, "extrapolated": heads < heads_total or steps > 1,
                     "sample": f"{heads} of {heads_total} heads ({'forward' if fwd_only else 'fwd+bwd'}, N={c.N}, "
                               f"d={c.d}) in {el:.2f} s" + (f"; x{steps} denoising steps" if steps > 1 else "")}
    return res


def run_reference(args):
    """The CPU oracle as the reference arm (rank 0 only).

    A step is one head of the workload run through the oracle's own steps (RMSNorm of q and k,
    bf16 rounding of q_hat and k_hat, softmax attention with materialised scores, its exact
    backward, the RMSNorm backward), restricted to R of the head's N query rows against all N
    keys.  R is the full N when K steps of whole heads fit the time budget, otherwise the largest
    row count that does; the FLOP per step is 14·R·N·d, the same count per query row as the GPU
    arm's 14·B·H·N²·d."""
    world, rank, _ = dist_setup()
    if rank != 0:
        return 0
    import numpy as np

    import oracle
    from joint_attention_gb300.inputs import CONFIGS, make_inputs

    c = CONFIGS[WORKLOAD]
    N, d = c.N, c.d
    inp = make_inputs(1, 1, N, d, seed=c.seed)
    q, k, v, dout = (np.asarray(x[0, 0], dtype=np.float64) for x in (inp.q, inp.k, inp.v, inp.dout))
    gq, gk = np.asarray(inp.gq, dtype=np.float64), np.asarray(inp.gk, dtype=np.float64)
    scale = 1.0 / np.sqrt(d)

    def step(R):
        qh, rq = oracle.rmsnorm_fwd(q[:R], gq)
        kh, rk = oracle.rmsnorm_fwd(k, gk)
        qh, kh = oracle.round_to_bf16(qh), oracle.round_to_bf16(kh)
        O, _, P = oracle.attention_fwd_head(qh, kh, v, scale)
        dqh, dkh, _ = oracle.attention_bwd_head(qh, kh, v, P, O, dout[:R], scale)
        oracle.rmsnorm_bwd(q[:R], gq, rq, dqh)
        oracle.rmsnorm_bwd(k, gk, rk, dkh)

    t0 = time.perf_counter()
    step(N)
    t_head = time.perf_counter() - t0
    budget_s = 120.0
    R = N
    if (args.steps + args.warmup) * t_head > budget_s:
        R = max(16, int(N * budget_s / ((args.steps + args.warmup) * t_head)))
    for _ in range(args.warmup):
        step(R)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step(R)
    el = time.perf_counter() - t0
    fl = 14.0 * R * N * d * args.steps
    val = fl / el / 1e12
    sample = (f"each step = {R} of the N={N} query rows of one (b, h) head of the {WORKLOAD} workload "
              f"(d={d}) against all N keys, fwd+bwd with the RMSNorm steps, float64 NumPy with "
              f"materialised scores")
    line = {"metric": METRIC, "value": val, "unit": UNIT, "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "impl": "reference",
            "config": {"workload": f"{WORKLOAD} B16 H12 N_img1024 N_txt77 d64 (a bounded sample per step)",
                       "sample": sample},
            "cpu_baseline": {"value": val, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": val, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def per_config_throughput(ja, torch, dev, stream, peaks, reps=50, warmup=10, only=None):
    """TFLOP/s and images-equivalent/s of every workload of the parity suite (one GPU, eager
    calls, inputs resident on the device; the fwd+bwd rows are 14·B·H·N²·d per step, the CFG
    sampling row is its forward, 4·B·H·N²·d per denoising step).  Inputs are seeded device
    normals of each workload's shape (values do not change the work), in N_SETS rotating sets
    whose combined size exceeds L2 for every workload but the tiny one.  Each row is the median
    of `reps` steps, each timed alone with CUDA events on the launching stream, after `warmup`
    untimed steps."""
    from joint_attention_gb300.inputs import CONFIGS

    def median_ms(one):
        for i in range(warmup):
            one(i)
        torch.cuda.synchronize(dev)
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
        for i, (a, b) in enumerate(evs):
            a.record(stream)
            one(i)
            b.record(stream)
        torch.cuda.synchronize(dev)
        return statistics.median(a.elapsed_time(b) for a, b in evs)

    res = {}
    gen = torch.Generator(device=dev)
    for name, c in CONFIGS.items():
        if only and name not in only:
            continue
        B, H, N, d = c.B, c.H, c.N, c.d
        gen.manual_seed(1000 + c.seed)
        shape = (B, H, N, d)
        sets = [{key: (torch.randn(shape, generator=gen, device=dev) * c.value_scale).to(torch.bfloat16)
                 for key in ("q", "k", "v", "dout")} for _ in range(N_SETS)]
        gq = torch.rand(d, generator=gen, device=dev) + 0.5
        gk = torch.rand(d, generator=gen, device=dev) + 0.5
        out, lse = torch.empty_like(sets[0]["q"]), torch.empty((B, H, N), device=dev, dtype=torch.float32)
        dq, dk, dv = torch.empty_like(out), torch.empty_like(out), torch.empty_like(out)
        dgq, dgk = torch.empty_like(gq), torch.empty_like(gk)
        fwd_only = c.mode == "cfg_fwd"
        saved = torch.empty(ja.jattn_saved_bytes(B, H, c.N_img, c.N_txt, d), dtype=torch.uint8, device=dev)

        def one(i):
            t = sets[i % N_SETS]
            if fwd_only:
                ja.jattn_fwd(t["q"], t["k"], t["v"], gq, gk, B, H, c.N_img, c.N_txt, d, out, lse, stream)
            else:
                ja.jattn_fwd_train(t["q"], t["k"], t["v"], gq, gk, B, H, c.N_img, c.N_txt, d, out, lse, saved,
                                   stream)
                ja.jattn_bwd_train(t["q"], t["k"], t["v"], gq, gk, out, lse, t["dout"], saved, dq, dk, dv, dgq,
                                   dgk, B, H, c.N_img, c.N_txt, d, stream)

        ms = median_ms(one)
        fl = flops_fwd(B, H, N, d) + (0.0 if fwd_only else flops_bwd(B, H, N, d))
        row = {"mode": "fwd (CFG sampling step)" if fwd_only else "fwd+bwd", "B": B, "H": H, "N": N, "d": d,
               "ms": ms, "tflops": fl / (ms * 1e-3) / 1e12}
        if fwd_only:
            row["images_per_s"] = c.n_uncond / (c.steps * 12 * ms * 1e-3)
        else:
            row["images_equiv_per_s"] = B / (12 * ms * 1e-3)
        res[name] = row
        if name == WORKLOAD:
            # The same workload with dQ added in a fixed order (jattn_set_deterministic): the
            # cost of bit-for-bit repeatable gradients.
            ja.jattn_set_deterministic(True)
            try:
                ms_det = median_ms(one)
            finally:
                ja.jattn_set_deterministic(False)
            res[name + "_deterministic"] = dict(row, mode="fwd+bwd, deterministic dQ order", ms=ms_det,
                                                tflops=fl / (ms_det * 1e-3) / 1e12,
                                                images_equiv_per_s=B / (12 * ms_det * 1e-3))
        del sets, out, lse, dq, dk, dv, saved
    if only and "varlen_mix" not in only:
        return _per_config_tail(ja, torch, dev, stream, median_ms, peaks, res, only)
    # Packed variable-length call (the training pair's varlen form): the 512 px and 256 px joint
    # lengths mixed in one call, 8 x 1101 + 16 x 333 rows per head, H = 12, d = 64.
    lens = [1101] * 8 + [333] * 16
    H, d = 12, 64
    cu = [0]
    for n in lens:
        cu.append(cu[-1] + n)
    T = cu[-1]
    gen.manual_seed(2000)
    sets = [{key: torch.randn((H, T, d), generator=gen, device=dev).to(torch.bfloat16)
             for key in ("q", "k", "v", "dout")} for _ in range(N_SETS)]
    gq = torch.rand(d, generator=gen, device=dev) + 0.5
    gk = torch.rand(d, generator=gen, device=dev) + 0.5
    out, lse = torch.empty_like(sets[0]["q"]), torch.empty((H, T), device=dev, dtype=torch.float32)
    dq, dk, dv = torch.empty_like(out), torch.empty_like(out), torch.empty_like(out)
    dgq, dgk = torch.empty_like(gq), torch.empty_like(gk)
    saved = torch.empty(ja.jattn_saved_bytes_varlen(cu, H, d), dtype=torch.uint8, device=dev)

    def one_varlen(i):
        t = sets[i % N_SETS]
        ja.jattn_fwd_train_varlen(t["q"], t["k"], t["v"], gq, gk, cu, H, d, out, lse, saved, stream)
        ja.jattn_bwd_train_varlen(t["q"], t["k"], t["v"], gq, gk, out, lse, t["dout"], saved, dq, dk, dv, dgq,
                                  dgk, cu, H, d, stream)

    ms = median_ms(one_varlen)
    fl = sum(flops_fwd(1, H, n, d) + flops_bwd(1, H, n, d) for n in lens)
    res["varlen_mix"] = {"mode": "fwd+bwd, packed sequences", "sequences": "8 x 1101 + 16 x 333", "H": H, "T": T,
                         "d": d, "ms": ms, "tflops": fl / (ms * 1e-3) / 1e12,
                         "images_equiv_per_s": len(lens) / (12 * ms * 1e-3)}
    del sets, out, lse, dq, dk, dv, saved
    return _per_config_tail(ja, torch, dev, stream, median_ms, peaks, res, only)


def _per_config_tail(ja, torch, dev, stream, median_ms, peaks, res, only):
    if not only or WORKLOAD + "_projected" in only:
        res[WORKLOAD + "_projected"] = projected_step_throughput(ja, torch, dev, stream, median_ms, peaks)
    if ja.jattn_last_device_error(stream) != 0:
        raise RuntimeError("device-side wait timed out in the per-config pass")
    return res


def projected_step_throughput(ja, torch, dev, stream, median_ms, peaks):
    """The 512 px training step from the tokens: both streams' QKV projections (width C = 768,
    W [3 H d, C] per stream) with QK-RMSNorm in the projection's epilogue (jattn_qkv_norm), then
    the attention forward from the saved q_hat / k_hat (jattn_fwd_saved) and the training
    backward.  Beside it the same step with the projection as two cuBLAS GEMMs (torch F.linear,
    bf16), the heads copied into the joint layout, and the training pair normalising q / k
    itself.  Reports both step times, the fused kernel's own time (CUDA events around each
    launch) and its TFLOP/s against the measured bf16 peak."""
    from joint_attention_gb300.inputs import CONFIGS

    c = CONFIGS[WORKLOAD]
    B, H, N_img, N_txt, d, N = c.B, c.H, c.N_img, c.N_txt, c.d, c.N
    C = H * d
    gen = torch.Generator(device=dev)
    gen.manual_seed(3000)
    sets = [{"x_img": torch.randn((B, N_img, C), generator=gen, device=dev).to(torch.bfloat16),
             "x_txt": torch.randn((B, N_txt, C), generator=gen, device=dev).to(torch.bfloat16),
             "dout": torch.randn((B, H, N, d), generator=gen, device=dev).to(torch.bfloat16)}
            for _ in range(N_SETS)]
    w = {s: (torch.randn((3 * H * d, C), generator=gen, device=dev) * C ** -0.5).to(torch.bfloat16)
         for s in ("img", "txt")}
    b = {s: torch.randn(3 * H * d, generator=gen, device=dev) * 0.1 for s in ("img", "txt")}
    b16 = {s: b[s].to(torch.bfloat16) for s in b}
    gq = torch.rand(d, generator=gen, device=dev) + 0.5
    gk = torch.rand(d, generator=gen, device=dev) + 0.5
    q = torch.empty((B, H, N, d), dtype=torch.bfloat16, device=dev)
    k, v, out = torch.empty_like(q), torch.empty_like(q), torch.empty_like(q)
    lse = torch.empty((B, H, N), device=dev, dtype=torch.float32)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(q), torch.empty_like(q)
    dgq, dgk = torch.empty_like(gq), torch.empty_like(gk)
    saved = torch.empty(ja.jattn_saved_bytes(B, H, N_img, N_txt, d), dtype=torch.uint8, device=dev)

    def fused(i):
        t = sets[i % N_SETS]
        ja.jattn_qkv_norm(t["x_img"], w["img"], b["img"], t["x_txt"], w["txt"], b["txt"], gq, gk, B, H, N_img,
                          N_txt, d, C, q, k, v, saved, stream)
        ja.jattn_fwd_saved(v, B, H, N_img, N_txt, d, out, lse, saved, stream)
        ja.jattn_bwd_train(q, k, v, gq, gk, out, lse, t["dout"], saved, dq, dk, dv, dgq, dgk, B, H, N_img, N_txt,
                           d, stream)

    def unfused(i):
        t = sets[i % N_SETS]
        # torch's current stream is `stream` (the bench launches everything on it)
        for s, x, rows in (("txt", t["x_txt"], slice(0, N_txt)), ("img", t["x_img"], slice(N_txt, N))):
            y = torch.nn.functional.linear(x, w[s], b16[s]).view(B, -1, 3, H, d).permute(2, 0, 3, 1, 4)
            q[:, :, rows], k[:, :, rows], v[:, :, rows] = y[0], y[1], y[2]
        ja.jattn_fwd_train(q, k, v, gq, gk, B, H, N_img, N_txt, d, out, lse, saved, stream)
        ja.jattn_bwd_train(q, k, v, gq, gk, out, lse, t["dout"], saved, dq, dk, dv, dgq, dgk, B, H, N_img, N_txt,
                           d, stream)

    ms_fused = median_ms(fused)
    ms_unfused = median_ms(unfused)
    ja.jattn_profile_reset()
    ja.jattn_profile_enable(True)
    for i in range(20):
        fused(i)
    torch.cuda.synchronize(dev)
    ja.jattn_profile_enable(False)
    kinds = {ja.jattn_kernel_name(kk): ja.jattn_profile_read(kk) for kk in range(ja.KERNEL_KINDS)}
    n, tot = kinds["qkv_norm"]
    qkv_us = tot / max(n, 1) * 1e3
    proj_fl = 2.0 * B * N * (3 * H * d) * C
    qkv_tf = proj_fl / (qkv_us * 1e-6) / 1e12
    fl = proj_fl + flops_fwd(B, H, N, d) + flops_bwd(B, H, N, d)
    row = {"mode": "QKV projection + QK-RMSNorm epilogue, attention fwd from saved, training bwd",
           "B": B, "H": H, "N": N, "d": d, "C": C, "ms": ms_fused, "tflops": fl / (ms_fused * 1e-3) / 1e12,
           "ms_projection_by_cublas_and_norm_pass": ms_unfused,
           "qkv_norm_us": qkv_us, "qkv_norm_tflops": qkv_tf,
           "qkv_norm_frac_of_measured_bf16": qkv_tf / peaks["bf16_tflops"],
           "kernel_us": {name: tot_ms / max(cnt, 1) * 1e3 for name, (cnt, tot_ms) in kinds.items() if cnt},
           "images_equiv_per_s": B / (12 * ms_fused * 1e-3)}
    del sets, q, k, v, out, lse, dq, dk, dv, saved
    return row


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    # The default timed loop runs about a second, so that the 200 ms clock samples fall inside it.
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--cpu-budget-s", type=float, default=10.0)
    ap.add_argument("--cpu-config-budget-s", type=float, default=3.0,
                    help="host seconds of oracle time per workload in the per-config pass")
    ap.add_argument("--no-per-config", action="store_true", help="skip the per-workload throughput pass")
    ap.add_argument("--per-config", default="",
                    help="comma-separated rows of the per-workload pass to run (default: all)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        return run_reference(args)

    import torch
    import torch.distributed as dist

    world, rank, local = dist_setup()
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)

    from joint_attention_gb300.build import build

    if rank == 0:
        build()
    if world > 1:
        dist.barrier()
    import joint_attention_gb300 as ja
    from joint_attention_gb300.inputs import CONFIGS, make_config_inputs

    ja.load_library()
    c = CONFIGS[WORKLOAD]
    B, H, N, d = c.B, c.H, c.N, c.d
    inp = make_config_inputs(c)

    def bf(a):
        return torch.from_numpy(a).to(dev).to(torch.bfloat16).contiguous()

    gq = torch.from_numpy(inp.gq).to(dev).float().contiguous()
    gk = torch.from_numpy(inp.gk).to(dev).float().contiguous()
    sets = []
    for s in range(N_SETS):
        # set 0 is the seeded workload; the others are permutations of it
        # (same values and statistics, different addresses).
        roll = s * 7
        q = bf(inp.q).roll(roll, dims=2).contiguous()
        k = bf(inp.k).roll(roll, dims=2).contiguous()
        v = bf(inp.v).roll(roll, dims=2).contiguous()
        do = bf(inp.dout).roll(roll, dims=2).contiguous()
        sets.append(dict(q=q, k=k, v=v, dout=do, out=torch.empty_like(q),
                         lse=torch.empty((B, H, N), device=dev, dtype=torch.float32),
                         dq=torch.empty_like(q), dk=torch.empty_like(q), dv=torch.empty_like(q),
                         dgq=torch.empty_like(gq), dgk=torch.empty_like(gk),
                         saved=torch.empty(ja.jattn_saved_bytes(B, H, c.N_img, c.N_txt, d), dtype=torch.uint8,
                                           device=dev)))
    stream = torch.cuda.current_stream(dev)
    n_img, n_txt = c.N_img, c.N_txt

    def step(i):
        t = sets[i % N_SETS]
        ja.jattn_fwd_train(t["q"], t["k"], t["v"], gq, gk, B, H, n_img, n_txt, d, t["out"], t["lse"], t["saved"],
                           stream)
        ja.jattn_bwd_train(t["q"], t["k"], t["v"], gq, gk, t["out"], t["lse"], t["dout"], t["saved"], t["dq"],
                           t["dk"], t["dv"], t["dgq"], t["dgk"], B, H, n_img, n_txt, d, stream)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize(dev)
    if ja.jattn_last_device_error(stream) != 0:
        raise RuntimeError("device-side wait timed out during warm-up")

    # ---- timed region (device time, CUDA events on the launching stream) ----
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(dev.index) as clocks:
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize(dev)
        wall0 = time.time()
        ev0.record(stream)
        for i in range(args.steps):
            step(i)
        ev1.record(stream)
        torch.cuda.synchronize(dev)
        clocks.mark(wall0, time.time())
        if world > 1:
            dist.barrier()
    ms_total = ev0.elapsed_time(ev1)
    # ---- per-kernel breakdown: the same steps again, each launch bracketed by CUDA events
    # on the launching stream (the library's profiling mode).  A separate pass, because the
    # per-launch events sit between kernels and would hold back the overlap of one kernel's
    # launch with the previous one's tail (programmatic dependent launch) in the timed region.
    torch.cuda.synchronize(dev)
    ja.jattn_profile_reset()
    ja.jattn_profile_enable(True)
    for i in range(args.steps):
        step(i)
    torch.cuda.synchronize(dev)
    ja.jattn_profile_enable(False)
    prof = ja.profile_snapshot()
    if ja.jattn_last_device_error(stream) != 0:
        raise RuntimeError("device-side wait timed out in the timed region")
    fl_step = flops_fwd(B, H, N, d) + flops_bwd(B, H, N, d)
    ms_total, value = aggregate_over_ranks(ms_total, args.steps, fl_step, world, dist, dev)
    ms_step = ms_total / args.steps

    # ---- end to end: pinned host buffers, copies inside the timed region ----
    # Each step copies its inputs host -> device, runs fwd + bwd through the C ABI and copies
    # every result device -> host.  As in a training loop that prefetches, the copies of one
    # step overlap the kernels of its neighbours: three device buffer sets, the uploads on one
    # stream, the kernels on the launching stream, the downloads on a third; events order
    # each buffer set's upload -> kernels -> download -> next upload.  out and lse leave as
    # soon as the forward has written them, while the backward runs.  The copy engines move
    # about 200 GB/s each way and 320 GB/s both ways at once on this machine, so the copies,
    # not the kernels, set the end-to-end step time.
    e2e = None
    if not args.no_e2e:
        nbuf = N_SETS
        h_in = {n: sets[0][n].cpu().pin_memory() for n in ("q", "k", "v", "dout")}
        h_g = {"gq": gq.cpu().pin_memory(), "gk": gk.cpu().pin_memory()}
        h_out = {n: torch.empty_like(sets[0][n], device="cpu").pin_memory()
                 for n in ("out", "lse", "dq", "dk", "dv", "dgq", "dgk")}
        d_g = [{"gq": torch.empty_like(gq), "gk": torch.empty_like(gk)} for _ in range(nbuf)]
        h2d = sum(x.numel() * x.element_size() for x in list(h_in.values()) + list(h_g.values()))
        d2h = sum(x.numel() * x.element_size() for x in h_out.values())
        s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        ev_in = [torch.cuda.Event() for _ in range(nbuf)]
        ev_fwd = [torch.cuda.Event() for _ in range(nbuf)]
        ev_comp = [torch.cuda.Event() for _ in range(nbuf)]
        ev_out = [torch.cuda.Event() for _ in range(nbuf)]
        used = [False] * nbuf

        def e2e_step(i):
            kb = i % nbuf
            t, g = sets[kb], d_g[kb]
            with torch.cuda.stream(s_in):
                if used[kb]:
                    s_in.wait_event(ev_out[kb])
                for n, x in h_in.items():
                    t[n].copy_(x, non_blocking=True)
                for n, x in h_g.items():
                    g[n].copy_(x, non_blocking=True)
                ev_in[kb].record(s_in)
            stream.wait_event(ev_in[kb])
            ja.jattn_fwd_train(t["q"], t["k"], t["v"], g["gq"], g["gk"], B, H, n_img, n_txt, d, t["out"], t["lse"],
                               t["saved"], stream)
            ev_fwd[kb].record(stream)
            ja.jattn_bwd_train(t["q"], t["k"], t["v"], g["gq"], g["gk"], t["out"], t["lse"], t["dout"], t["saved"],
                               t["dq"], t["dk"], t["dv"], t["dgq"], t["dgk"], B, H, n_img, n_txt, d, stream)
            ev_comp[kb].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_fwd[kb])
                for n in FWD_RESULTS:
                    h_out[n].copy_(t[n], non_blocking=True)
                s_out.wait_event(ev_comp[kb])
                for n, x in h_out.items():
                    if n not in FWD_RESULTS:
                        x.copy_(t[n], non_blocking=True)
                ev_out[kb].record(s_out)
            used[kb] = True

        for i in range(4):
            e2e_step(i)
        torch.cuda.synchronize(dev)
        if world > 1:
            dist.barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        n_e2e = max(3, min(args.steps, 300))
        e0.record(s_in)
        for i in range(n_e2e):
            e2e_step(i)
        e1.record(s_out)
        torch.cuda.synchronize(dev)
        ms_e2e = e0.elapsed_time(e1)
        if world > 1:
            tt = torch.tensor([ms_e2e], device=dev, dtype=torch.float64)
            dist.all_reduce(tt, op=dist.ReduceOp.MAX)
            ms_e2e = float(tt.item())
        e2e = {"value": fl_step * n_e2e * world / (ms_e2e * 1e-3) / 1e12, "unit": UNIT,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "ms_per_step": ms_e2e / n_e2e,
               "overlap": "three buffer sets: later steps' uploads and earlier steps' downloads run during "
                          "step i's kernels; out and lse download while the backward runs"}

    if rank != 0:
        dist.destroy_process_group()
        return 0

    # ---- roofline of the dominant kernel ----
    peaks, peak_src = load_peaks()
    kern = {name: {"launches": n, "total_ms": ms, "avg_us": (ms / n * 1e3) if n else None}
            for name, (n, ms) in prof.items()}
    tot = sum(v["total_ms"] for v in kern.values()) or 1.0
    for v in kern.values():
        v["share"] = v["total_ms"] / tot
    dom = max(kern, key=lambda k: kern[k]["total_ms"])
    algo = {  # algorithmic work per launch (FLOP for contractions, bytes for HBM-bound kernels)
        "attn_fwd": ("tensor", flops_fwd(B, H, N, d)),
        "attn_bwd": ("tensor", flops_bwd(B, H, N, d)),
        # read q, k; write q_hat, k_hat and the rows' 1/rms (kept for the backward)
        "qk_norm_fwd": ("hbm", 4.0 * B * H * N * d * 2 + 2 * B * H * N * 4),
        # read out, dout, lse; write the zeroed dq accumulator and the statistics chunks
        # (16 bf16 per row of the 128-row-padded layout)
        "bwd_prep": ("hbm", B * H * N * d * 2 * 2 + B * H * N * 4 + B * H * N * d * 4
                     + B * H * (-(-N // 128) * 128) * 32),
        # read the dq accumulator, q and rq; write dq
        "q_norm_bwd": ("hbm", B * H * N * d * (4 + 2 + 2) + B * H * N * 4),
    }
    bound, work = algo[dom]
    avg_s = kern[dom]["avg_us"] * 1e-6
    clk = clocks.summary()
    extra = {}
    if bound == "tensor":
        achieved = work / avg_s / 1e12
        unit = "TFLOP/s"
        # The burst bf16 peak is a GEMM timed alone at full clock; the sustained one is a
        # seconds-long GEMM loop at the clock the power cap settles it to.  The peak taken is the
        # one whose clock the timed loop ran at: burst when its median SM clock is within 10 % of
        # the maximum.
        sm, mx = clk.get("sm_mhz"), clk.get("sm_max_mhz")
        full_clock = sm is None or mx is None or sm >= 0.9 * mx
        peak = peaks["bf16_tflops"] if full_clock else peaks["bf16_tflops_sustained"]
        which = "burst bf16" if full_clock else "sustained bf16"
        extra = {"frac_vs_sustained": achieved / peaks["bf16_tflops_sustained"],
                 "sustained_peak": peaks["bf16_tflops_sustained"],
                 "sustained_peak_clock_mhz": peaks.get("sustained_sm_mhz")}
    else:
        achieved = work / avg_s / 1e9
        peak = peaks["hbm_gbs"]
        unit = "GB/s"
        which = "HBM copy"
    traffic = ncu_traffic(dom)
    roofline = {"kernel": dom, "bound": bound, "achieved": achieved, "peak": peak, "unit": unit,
                "frac": achieved / peak, "traffic": traffic,
                "traffic_source": (f"stored: dram__bytes_read.sum + dram__bytes_write.sum of one ncu capture "
                                   f"of {dom} on this workload, keyed to its source file "
                                   f"({NCU_TRAFFIC[dom]['capture']})") if traffic is not None else None,
                "peak_source": f"{peak_src} ({which})", **extra}
    per_cfg = None
    if not args.no_per_config and world == 1:
        only = {x for x in args.per_config.split(",") if x}
        per_cfg = per_config_throughput(ja, torch, dev, stream, peaks, only=only)
    cpu = None
    if not args.no_cpu_baseline and world == 1:
        cpu = cpu_oracle_sample(B, H, N, d, c.seed, args.cpu_budget_s, max_heads=64)
        if per_cfg is not None:
            for name, row in cpu_oracle_per_config(args.cpu_config_budget_s).items():
                if name in per_cfg:
                    per_cfg[name]["cpu_baseline"] = row
    launches = sum(v["launches"] for v in kern.values())
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"{WORKLOAD} MM-DiT joint attention fwd+bwd: B={B} H={H} N_img={c.N_img} "
                               f"N_txt={c.N_txt} (N={N}) d={d}, QK-RMSNorm eps=1e-6",
                   "flop_per_step": fl_step, "l2": f"{N_SETS} rotating input sets, each larger than L2 "
                                                   f"together (~{N_SETS * 245} MB vs 129 MB)",
                   "parallelism": f"replicas x{world}"},
        "pct_of_peak_bf16": value / world / peaks["bf16_tflops"] * 100.0,
        "peak_bf16_tflops": peaks["bf16_tflops"], "peak_source": peak_src,
        "images_equiv_per_s": B * world / (12 * ms_step * 1e-3),
        "model_tflops": 12.0 * B * H * N * N * d * args.steps * world / (ms_total * 1e-3) / 1e12,
        "roofline": roofline, "kernels": kern, "gpu_launches": launches,
        "cpu_baseline": cpu, "e2e": e2e, "clocks": clk, "per_config": per_cfg,
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
