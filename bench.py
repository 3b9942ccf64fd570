"""Benchmark: causal multi-head attention forward + backward on one GB300.

One step = attn_fwd + attn_bwd (every kernel of the hot path) over one batch
of the GPT-2 small attention layer, bf16: B=16, T=1024, C=768, NH=12 (hs=64),
causal. Metric: causal-adjusted TFLOP/s, FLOPs counted the FlashAttention way:
fwd = 4*B*NH*T^2*hs/2 (x2 without the mask), bwd = 2.5*fwd, step = 3.5*fwd.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
                    [--workload NAME]

--workload times another of the attention-layer shapes (inputs.WORKLOADS,
e.g. gpt2s_f32 for fp32 inputs on the tf32 tensor-core path); the default is
the GPT-2 small bf16 layer the metric is quoted on.

Prints ONE JSON line (rank 0). For N>1 launch with torch.distributed.run; each
rank runs its own independent batch (weak scaling, no collective on the data
path; one barrier and a max-reduction of the timing only).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import pathlib
import statistics
import subprocess
import sys
import time

ROOT = pathlib.Path(__file__).resolve().parent
sys.path.insert(0, str(ROOT))

WORKLOAD = "gpt2s_bf16"
METRIC = "attention fwd+bwd causal TFLOP/s at 1 GB300 and % of dense tensor peak"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
TF32_PER_BF16 = 1.1 / 2.25    # nominal dense tf32 / bf16 tensor rate of the GB300
FLUSH_BYTES = 512 << 20   # > 129 MB L2


# ----------------------------------------------------------------------------- helpers
def flops(B, T, C, NH, causal):
    hs = C // NH
    fwd = 4.0 * B * NH * T * T * hs * (0.5 if causal else 1.0)
    return {"fwd": fwd, "bwd": 2.5 * fwd, "step": 3.5 * fwd}


def algo_bytes(B, T, C, NH, e):
    """Algorithmic HBM bytes: fwd reads qkv, writes out + lse; bwd reads qkv, out,
    dout, lse, writes dqkv and D."""
    btc = B * T * C
    return {"fwd": 4 * btc * e + 4 * B * NH * T, "bwd": 8 * btc * e + 8 * B * NH * T}


def load_peaks():
    p = ROOT / "MEASURED_PEAKS.json"
    if p.exists():
        d = json.loads(p.read_text())
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def reduce_max(x: float, world: int, device=None) -> float:
    """Max of a scalar over all ranks (identity for world == 1)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate(units_per_rank: float, t_ms_rank: float, world: int, device=None):
    """Whole-job throughput: units over all ranks / the slowest rank's time."""
    t = reduce_max(t_ms_rank, world, device)
    return units_per_rank * world / (t * 1e-3), t


class ClockSampler:
    """nvidia-smi clock/throttle sampling while the timed region runs."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        self.out = ""
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self):
        rows = []
        for line in (self.out or "").splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                rows.append((float(f[1]), float(f[2]), f[5], f[6], f[7], f[8]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[2 + i] == "Active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows)}


# ----------------------------------------------------------------------------- CPU oracle
_CPU_CHILD = r"""
import json, sys, time
sys.path.insert(0, sys.argv[1])
import numpy as np
import oracle
from causal_head_attention_fwd_gb300 import inputs
w = inputs.WORKLOADS[sys.argv[2]]
budget = float(sys.argv[3]); max_heads = int(sys.argv[4])
x, _ = inputs.draw((w.B, w.T, 3 * w.C), w.sigma_qkv, w.seed_qkv, w.dtype)
d, _ = inputs.draw((w.B, w.T, w.C), w.sigma_dout, w.seed_dout, w.dtype)
heads, t0 = 0, time.perf_counter()
fwd_times, bwd_times = [], []
while heads < max_heads and (time.perf_counter() - t0) < budget:
    # the batch's (b, h) heads in order, wrapping around after the last
    b, h = (heads // w.NH) % w.B, heads % w.NH
    xb = x[b:b + 1].astype(np.float64); db = d[b:b + 1].astype(np.float64)
    s = time.perf_counter()
    oracle.forward(xb, 1, w.T, w.C, w.NH, bool(w.causal), heads=[(0, h)])
    m = time.perf_counter()
    oracle.backward(db, xb, 1, w.T, w.C, w.NH, bool(w.causal), heads=[(0, h)])
    e = time.perf_counter()
    fwd_times.append(m - s); bwd_times.append(e - m)
    heads += 1
print(json.dumps({"heads": heads, "seconds": time.perf_counter() - t0, "fwd_times": fwd_times,
                  "bwd_times": bwd_times}))
"""


def run_oracle_child(workload: str, budget_s: float, max_heads: int):
    cores = os.cpu_count() or 1
    env = dict(os.environ)
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        env[k] = str(cores)
    r = subprocess.run([sys.executable, "-c", _CPU_CHILD, str(ROOT), workload, str(budget_s), str(max_heads)],
                       capture_output=True, text=True, env=env, timeout=min(budget_s * 4 + 600, 7200))
    if r.returncode != 0:
        raise RuntimeError("oracle child failed: " + r.stderr[-2000:])
    return json.loads(r.stdout.strip().splitlines()[-1]), cores


def _oracle_rates(w, fwd_times, bwd_times):
    """TFLOP/s of the oracle's forward, backward and forward + backward per head."""
    f_head = {k: v / (w.B * w.NH) for k, v in flops(w.B, w.T, w.C, w.NH, w.causal).items()}
    tf, tb = sum(fwd_times), sum(bwd_times)
    n = len(fwd_times)
    return {"fwd": n * f_head["fwd"] / tf / 1e12, "bwd": n * f_head["bwd"] / tb / 1e12,
            "step": n * f_head["step"] / (tf + tb) / 1e12, "fwd_s_per_head": tf / n, "bwd_s_per_head": tb / n}


def _sample_text(w, n_heads, seconds, what):
    return (f"{what}: {n_heads} (b,h) heads of {w.name} taken in order from (0,0) "
            f"({w.B * w.NH} heads in the batch{', wrapping around' if n_heads > w.B * w.NH else ''}), "
            f"forward and backward timed apart (the oracle's backward recomputes att itself), "
            f"float64 numpy oracle, {seconds:.1f} s")


def cpu_baseline(workload: str, budget_s: float = 15.0):
    from causal_head_attention_fwd_gb300 import inputs
    w = inputs.WORKLOADS[workload]
    res, cores = run_oracle_child(workload, budget_s, 10_000)
    r = _oracle_rates(w, res["fwd_times"], res["bwd_times"])
    return {"value": r["step"], "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
            "fwd_tflops": r["fwd"], "bwd_tflops": r["bwd"],
            "fwd_s_per_head": r["fwd_s_per_head"], "bwd_s_per_head": r["bwd_s_per_head"],
            "sample": _sample_text(w, res["heads"], res["seconds"], "fwd+bwd")}


def run_reference(args):
    """The oracle as the reference arm: each step = fwd+bwd of one (b, h) head."""
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    from causal_head_attention_fwd_gb300 import inputs
    w = inputs.WORKLOADS[args.workload]
    res, cores = run_oracle_child(args.workload, 1e9, args.warmup + args.steps)
    ft, bt = res["fwd_times"][args.warmup:], res["bwd_times"][args.warmup:]
    r = _oracle_rates(w, ft, bt)
    value = r["step"]
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": (sum(ft) + sum(bt)) / len(ft) * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_dict(w), "fwd_tflops": r["fwd"], "bwd_tflops": r["bwd"],
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "fwd_tflops": r["fwd"], "bwd_tflops": r["bwd"],
                         "sample": f"one (b,h) head of {w.name} per step (1/{w.B * w.NH} of the batch), "
                                   f"heads in order from (0,0); " + _sample_text(w, len(ft), sum(ft) + sum(bt),
                                                                                   "timed steps")},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def launch_plan(gpus: int, env) -> tuple:
    """How to honour --gpus N: ("run", None) in this process (N == 1, or N
    ranks already started by torch.distributed.run with WORLD_SIZE == N),
    ("spawn", argv) to start N ranks with torch.distributed.run, or
    ("refuse", reason) when the environment's world size contradicts N."""
    if gpus < 1:
        return "refuse", f"--gpus must be >= 1, got {gpus}"
    ws = env.get("WORLD_SIZE")
    if ws is not None:
        if int(ws) != gpus:
            return "refuse", f"--gpus {gpus} but WORLD_SIZE={ws}: launch {gpus} ranks or pass --gpus {ws}"
        return "run", None
    if gpus == 1:
        return "run", None
    port = env.get("MASTER_PORT") or str(_free_port())
    return "spawn", [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={gpus}",
                     "--master-addr", "127.0.0.1", "--master-port", port]


def _free_port() -> int:
    import socket
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        return sk.getsockname()[1]


def config_dict(w):
    mask = "causal" if w.causal else "non-causal"
    return {"workload": f"{w.name}: attention layer, B={w.B} T={w.T} C={w.C} NH={w.NH} "
                        f"hs={w.hs}, {mask}, {w.dtype} qkv~N(0,{w.sigma_qkv}^2) dout~N(0,{w.sigma_dout}^2)",
            "B": w.B, "T": w.T, "C": w.C, "NH": w.NH, "causal": w.causal,
            "l2": "flushed between timed steps (512 MiB write)"}


# ----------------------------------------------------------------------------- llm.c drop-in mode
def run_att(args):
    """Times attn_fwd_att (preatt and att materialised, fp32 B x NH x T x T) on
    one GPU. Bound by the HBM writes of the two matrices."""
    import torch
    from causal_head_attention_fwd_gb300 import build, inputs
    build.build()
    from causal_head_attention_fwd_gb300 import api, ops
    dev = torch.device("cuda", 0)
    w = inputs.WORKLOADS[args.workload]
    B, T, C, NH, causal = w.B, w.T, w.C, w.NH, w.causal
    host = inputs.make_inputs(B, T, C, NH, w.dtype, w.sigma_qkv, w.sigma_dout, w.seed_qkv, w.seed_dout)
    qkv = ops.upload(host.qkv_dev, w.dtype, dev)
    out, lse = ops.attention_forward(qkv, NH, bool(causal))
    pre = torch.empty((B, NH, T, T), dtype=torch.float32, device=dev)
    att = torch.empty_like(pre)
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    for _ in range(args.warmup):
        ops.attention_matrices(qkv, lse, NH, bool(causal), preatt=pre, att=att, stream=stream)
    torch.cuda.synchronize(dev)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    with ClockSampler(0) as cs:
        for a, b in ev:
            flush.fill_(1.0)
            a.record(stream)
            ops.attention_matrices(qkv, lse, NH, bool(causal), preatt=pre, att=att, stream=stream)
            b.record(stream)
        torch.cuda.synchronize(dev)
    if api.attn_last_device_error(stream) != api.ATTN_OK:
        raise RuntimeError("device error in the timed region")
    t_ms = sum(a.elapsed_time(b) for a, b in ev) / len(ev)
    esz = 2 if w.dtype == "bf16" else 4
    nbytes = 2 * B * NH * T * T * 4 + B * T * 2 * C * esz + B * NH * T * 4   # writes + q,k + lse reads
    peaks, src = load_peaks()
    gbs = nbytes / (t_ms * 1e-3) / 1e9
    line = {"metric": "llm.c drop-in attention matrices (preatt + att) GB/s at 1 GB300", "value": gbs,
            "unit": "GB/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": t_ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": w.dtype,
            "data": "synthetic", "config": config_dict(w),
            "roofline": {"kernel": "attn_att_kernel", "bound": "hbm", "achieved": gbs,
                         "peak": float(peaks["hbm_gbs"]), "unit": "GB/s", "frac": gbs / float(peaks["hbm_gbs"]),
                         "traffic": None, "peak_source": f"{src} HBM copy (MEASURED_PEAKS.json hbm_gbs)"},
            "bytes_per_step": nbytes, "gpu_launches": args.steps, "clocks": cs.summary()}
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------------------- FP8 forward
FP8_PER_BF16 = 4.5 / 2.25     # nominal dense e4m3 / bf16 tensor rate of the GB300


def run_fp8(args):
    """Times attn_fwd_fp8 (e4m3 qkv with per-tile descales, bf16 out) on one
    GPU; FLOPs of the forward against the e4m3 tensor peak."""
    import torch
    from causal_head_attention_fwd_gb300 import build, inputs
    build.build()
    from causal_head_attention_fwd_gb300 import api, ops
    dev = torch.device("cuda", 0)
    w = inputs.FP8_WORKLOADS[args.fp8]
    B, T, C, NH, causal = w["B"], w["T"], w["C"], w["NH"], w["causal"]
    f = inputs.make_fp8_inputs(B, T, C, sigma=w["sigma"], seed=w["seed"], NH=NH)
    codes = torch.from_numpy(f.codes).to(dev)
    descale = torch.from_numpy(f.descale).to(dev)
    out = torch.empty((B, T, C), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((B, NH, T), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    def step():
        api.attn_fwd_fp8(codes, descale, out, lse, B, T, C, NH, int(causal), stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    with ClockSampler(0) as cs:
        for a, b in ev:
            flush.fill_(1.0)
            a.record(stream)
            step()
            b.record(stream)
        torch.cuda.synchronize(dev)
    if api.attn_last_device_error(stream) != api.ATTN_OK:
        raise RuntimeError("device error in the timed region")
    t_ms = sum(a.elapsed_time(b) for a, b in ev) / len(ev)
    fl = flops(B, T, C, NH, causal)["fwd"]
    tf = fl / (t_ms * 1e-3) / 1e12
    peaks, src = load_peaks()
    peak = float(peaks["bf16_tflops"]) * FP8_PER_BF16
    line = {"metric": "FP8 (e4m3) attention forward TFLOP/s at 1 GB300", "value": tf, "unit": "TFLOP/s",
            "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": t_ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "e4m3",
            "data": "synthetic",
            "config": {"workload": f"{args.fp8}: B={B} T={T} C={C} NH={NH} causal={int(causal)}, e4m3 qkv, bf16 out",
                       "B": B, "T": T, "C": C, "NH": NH, "l2": "flushed between timed steps (512 MiB write)"},
            "roofline": {"kernel": "attn_fwd_fp8_kernel", "bound": "tensor", "achieved": tf, "peak": peak,
                         "unit": "TFLOP/s", "frac": tf / peak, "traffic": None,
                         "peak_source": f"e4m3 = {src} bf16 burst (MEASURED_PEAKS.json bf16_tflops) x nominal 4.5/2.25"},
            "gpu_launches": args.steps, "clocks": cs.summary()}
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------------------- attention block
def run_block(args):
    """Times the GPT-2 attention block forward: c_attn GEMM (+bias) -> attention
    forward -> c_proj GEMM (+bias), three launches on one stream."""
    import torch
    from causal_head_attention_fwd_gb300 import build, inputs
    build.build()
    from causal_head_attention_fwd_gb300 import api, ops
    dev = torch.device("cuda", 0)
    w = inputs.BLOCK_WORKLOADS[args.block]
    B, T, C, NH, causal = w["B"], w["T"], w["C"], w["NH"], w["causal"]
    bi = inputs.make_block_inputs(B, T, C, seed=w["seed"])
    d = {k: ops.upload(v, "bf16", dev) for k, v in bi.bits.items()}
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    qkv = torch.empty((B, T, 3 * C), dtype=torch.bfloat16, device=dev)
    out = torch.empty((B, T, C), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((B, NH, T), dtype=torch.float32, device=dev)
    y = torch.empty((B, T, C), dtype=torch.bfloat16, device=dev)
    M = B * T

    def step():
        api.attn_linear_fwd(d["x"], d["w_attn"], d["b_attn"], qkv, M, 3 * C, C, stream)
        api.attn_fwd(qkv, out, lse, B, T, C, NH, int(causal), api.ATTN_BF16, stream)
        api.attn_linear_fwd(out, d["w_proj"], d["b_proj"], y, M, C, C, stream)

    def timed(n):
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
        for a, b in ev:
            flush.fill_(1.0)
            a.record(stream)
            step()
            b.record(stream)
        torch.cuda.synchronize(dev)
        return [a.elapsed_time(b) for a, b in ev]

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    with ClockSampler(0) as cs:
        times = timed(args.steps)
    if api.attn_last_device_error(stream) != api.ATTN_OK:
        raise RuntimeError("device error in the timed region")
    t_ms = sum(times) / len(times)
    f_lin = 2.0 * M * 3 * C * C + 2.0 * M * C * C
    f_att = flops(B, T, C, NH, causal)["fwd"]
    tf = (f_lin + f_att) / (t_ms * 1e-3) / 1e12
    api.attn_profile_reset()
    api.attn_profile_enable(True)
    timed(20)
    api.attn_profile_enable(False)
    lin_ms, lin_n = api.attn_profile_read(api.K_LINEAR)
    att_ms, att_n = api.attn_profile_read(api.K_FWD)
    peaks, src = load_peaks()
    peak = float(peaks["bf16_tflops"])
    lin_tf = f_lin / (lin_ms / max(lin_n, 1) * 2 * 1e-3) / 1e12
    line = {"metric": "GPT-2 attention block forward (c_attn + attention + c_proj) TFLOP/s at 1 GB300",
            "value": tf, "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": t_ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": f"{args.block}: B={B} T={T} C={C} NH={NH} causal={int(causal)}, bf16",
                       "B": B, "T": T, "C": C, "NH": NH, "l2": "flushed between timed steps (512 MiB write)"},
            "kernels": {"attn_linear_kernel": {"launches": lin_n, "avg_ms": lin_ms / max(lin_n, 1)},
                        "attn_fwd_kernel": {"launches": att_n, "avg_ms": att_ms / max(att_n, 1)}},
            "roofline": {"kernel": "attn_linear_kernel (c_attn + c_proj)", "bound": "tensor", "achieved": lin_tf,
                         "peak": peak, "unit": "TFLOP/s", "frac": lin_tf / peak, "traffic": None,
                         "peak_source": f"{src} bf16 burst (MEASURED_PEAKS.json bf16_tflops)"},
            "gpu_launches": 3 * args.steps, "clocks": cs.summary()}
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------------------- decode forward
def run_decode(args):
    """Times attn_decode (the last Tq tokens of each sequence against its whole
    key/value cache). Bound by reading the cache from HBM."""
    import torch
    from causal_head_attention_fwd_gb300 import build, inputs
    build.build()
    from causal_head_attention_fwd_gb300 import api, ops
    dev = torch.device("cuda", 0)
    w = inputs.DECODE_WORKLOADS[args.decode]
    B, L, C, NH, Tq = w.B, w.L, w.C, w.NH, w.Tq
    _, qkv_dev = inputs.draw((B, L, 3 * C), w.sigma_qkv, w.seed_qkv, w.dtype)
    qkv = ops.upload(qkv_dev, w.dtype, dev)
    tdt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    out = torch.empty((B, Tq, C), dtype=tdt, device=dev)
    lse = torch.empty((B, NH, Tq), dtype=torch.float32, device=dev)
    adt = api.ATTN_BF16 if w.dtype == "bf16" else api.ATTN_F32
    nws = api.attn_decode_workspace_size(B, L, C, NH, Tq, adt)
    ws = torch.empty(nws, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    def step():
        api.attn_decode(qkv, out, lse, B, L, C, NH, Tq, adt, ws, nws, stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    with ClockSampler(0) as cs:
        for a, b in ev:
            flush.fill_(1.0)
            a.record(stream)
            step()
            b.record(stream)
        torch.cuda.synchronize(dev)
    if api.attn_last_device_error(stream) != api.ATTN_OK:
        raise RuntimeError("device error in the timed region")
    t_ms = sum(a.elapsed_time(b) for a, b in ev) / len(ev)
    esz = 2 if w.dtype == "bf16" else 4
    cache = 2 * B * L * C * esz                                   # K and V of every position
    nbytes = cache + B * Tq * C * esz * 2 + 2 * nws + B * NH * Tq * 4
    peaks, src = load_peaks()
    gbs = nbytes / (t_ms * 1e-3) / 1e9
    line = {"metric": "decode forward (KV-cache stream) GB/s at 1 GB300", "value": gbs, "unit": "GB/s",
            "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": t_ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": w.dtype,
            "data": "synthetic",
            "config": {"workload": f"{w.name}: B={B} cached L={L} new Tq={Tq} C={C} NH={NH} hs={w.hs}, {w.dtype}",
                       "B": B, "L": L, "Tq": Tq, "C": C, "NH": NH,
                       "l2": "flushed between timed steps (512 MiB write)"},
            "roofline": {"kernel": "attn_decode_split", "bound": "hbm", "achieved": gbs,
                         "peak": float(peaks["hbm_gbs"]), "unit": "GB/s", "frac": gbs / float(peaks["hbm_gbs"]),
                         "traffic": stored_traffic("attn_decode_split", w.name),
                         "peak_source": f"{src} HBM copy (MEASURED_PEAKS.json hbm_gbs)"},
            "bytes_per_step": nbytes, "cache_bytes": cache, "tokens_per_s": B * Tq / (t_ms * 1e-3),
            "gpu_launches": 2 * args.steps, "clocks": cs.summary()}
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------------------- GPU arm
def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--workload", default=WORKLOAD)
    ap.add_argument("--decode", default=None, metavar="NAME",
                    help="time the decode forward (attn_decode) on a decode workload, e.g. gpt2s_decode")
    ap.add_argument("--fp8", default=None, metavar="NAME",
                    help="time the FP8 forward (attn_fwd_fp8) on an FP8 workload, e.g. gpt2s_fp8")
    ap.add_argument("--block", default=None, metavar="NAME",
                    help="time the GPT-2 attention block forward (c_attn -> attention -> c_proj), e.g. gpt2s_block")
    ap.add_argument("--att", action="store_true",
                    help="time the llm.c drop-in mode (attn_fwd_att: preatt and att, B x NH x T x T fp32) "
                         "instead of the fwd+bwd step")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    how, detail = launch_plan(args.gpus, os.environ)
    if how == "refuse":
        ap.error(detail)
    if how == "spawn":
        # one rank per GPU on this node, each running this same command line
        return subprocess.call(detail + [str(pathlib.Path(__file__).resolve())] +
                               list(sys.argv[1:] if argv is None else argv))
    if args.impl == "reference":
        return run_reference(args)
    if args.att:
        return run_att(args)
    if args.decode:
        return run_decode(args)
    if args.fp8:
        return run_fp8(args)
    if args.block:
        return run_block(args)

    import numpy as np
    import torch
    rank, world, local_rank = dist_env()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    from causal_head_attention_fwd_gb300 import build, inputs
    build.build()
    from causal_head_attention_fwd_gb300 import api, ops

    w = inputs.WORKLOADS[args.workload]
    B, T, C, NH, causal = w.B, w.T, w.C, w.NH, w.causal
    is_bf16 = w.dtype == "bf16"
    adt = api.ATTN_BF16 if is_bf16 else api.ATTN_F32
    tdt = torch.bfloat16 if is_bf16 else torch.float32
    esz = 2 if is_bf16 else 4
    host = inputs.make_inputs(B, T, C, NH, w.dtype, w.sigma_qkv, w.sigma_dout,
                              w.seed_qkv + 7919 * rank, w.seed_dout + 7919 * rank)
    qkv = ops.upload(host.qkv_dev, w.dtype, dev)
    dout = ops.upload(host.dout_dev, w.dtype, dev)
    out = torch.empty((B, T, C), dtype=tdt, device=dev)
    lse = torch.empty((B, NH, T), dtype=torch.float32, device=dev)
    dqkv = torch.empty_like(qkv)
    ws_bytes = api.attn_bwd_workspace_size(B, T, C, NH, causal, adt)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        api.attn_fwd(qkv, out, lse, B, T, C, NH, causal, adt, stream)
        api.attn_bwd(dout, qkv, out, lse, dqkv, B, T, C, NH, causal, adt, ws, ws_bytes, stream)

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize(dev)

    def timed(n, body):
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
        barrier()
        for a, b in ev:
            flush.fill_(1.0)            # evict L2 between steps (not timed)
            a.record(stream)
            body()
            b.record(stream)
        barrier()
        return [a.elapsed_time(b) for a, b in ev]

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    if api.attn_last_device_error(stream) != api.ATTN_OK:
        raise RuntimeError("device error during warm-up")

    # ---- main timed region (uninstrumented)
    with ClockSampler(local_rank) as cs:
        times = timed(args.steps, step)
    clocks = cs.summary()
    if api.attn_last_device_error(stream) != api.ATTN_OK:
        raise RuntimeError("device error in the timed region")
    t_ms = sum(times) / len(times)
    f = flops(B, T, C, NH, causal)
    value_flops, t_max = aggregate(f["step"], t_ms, world, dev)
    value = value_flops / 1e12

    # ---- per-kernel device times (library event profiling), same workload
    api.attn_profile_reset()
    api.attn_profile_enable(True)
    timed(max(20, min(args.steps, 200)), step)
    api.attn_profile_enable(False)
    kern = {}
    for kid, name in (api.KERNEL_NAMES if is_bf16 else api.KERNEL_NAMES_F32).items():
        ms, n = api.attn_profile_read(kid)
        kern[name] = {"launches": n, "avg_ms": ms / max(n, 1)}
    tot = sum(k["avg_ms"] for k in kern.values())
    for k in kern.values():
        k["share"] = k["avg_ms"] / tot if tot > 0 else None
    peaks, peak_src = load_peaks()
    dom = max(kern, key=lambda k: kern[k]["avg_ms"])
    # algorithmic FLOPs per launch; the fp32 backward splits the five matmuls
    # into dK/dV (S, dP, dV, dK) and dQ (dQ; its S and dP recompute is not counted)
    dom_flops = {"attn_fwd_kernel": f["fwd"], "attn_bwd_kernel": f["bwd"], "attn_fwd_f32_kernel": f["fwd"],
                 "attn_bwd_dkdv_f32": 2.0 * f["fwd"], "attn_bwd_dq_f32": 0.5 * f["fwd"]}.get(dom)
    peak_tf = float(peaks["bf16_tflops"]) * (1.0 if is_bf16 else TF32_PER_BF16)
    if dom_flops is not None:
        ach = dom_flops / (kern[dom]["avg_ms"] * 1e-3) / 1e12
        src = (f"{peak_src} bf16 burst (MEASURED_PEAKS.json bf16_tflops)" if peak_src == "measured"
               else "fallback 1.9 PFLOP/s bf16")
        if not is_bf16:
            src = f"tf32 = {src} x nominal 1.1/2.25"
        roofline = {"kernel": dom, "bound": "tensor", "achieved": ach, "peak": peak_tf, "unit": "TFLOP/s",
                    "frac": ach / peak_tf, "traffic": None, "peak_source": src}
    else:
        roofline = {"kernel": dom, "bound": "hbm", "achieved": None, "peak": float(peaks["hbm_gbs"]),
                    "unit": "GB/s", "frac": None, "traffic": None}
    roofline["traffic"] = stored_traffic(dom, w.name)
    names = list(kern)
    fwd_ms = kern[names[0]]["avg_ms"]
    bwd_ms = sum(kern[k]["avg_ms"] for k in names[1:])
    ab = algo_bytes(B, T, C, NH, esz)

    # ---- end to end through the public API with host buffers
    # Every step copies its inputs from pinned host memory and its results
    # (out, dqkv) back; the copies of neighbouring steps overlap the compute on
    # three streams (h2d, compute, d2h) with two device buffer sets, as a
    # data-loading training loop would run it. Time = the whole sequence / K.
    # (A second copy stream per direction measured no faster: the host link is
    # the limit at ~160 GB/s each way.)
    h_qkv = ops.upload(host.qkv_dev, w.dtype, pin=True)
    h_dout = ops.upload(host.dout_dev, w.dtype, pin=True)
    bufs = []
    for _ in range(2):
        bufs.append({"qkv": torch.empty_like(qkv), "dout": torch.empty_like(dout),
                     "out": torch.empty_like(out), "lse": torch.empty_like(lse), "dqkv": torch.empty_like(dqkv),
                     "h_out": torch.empty((B, T, C), dtype=tdt).pin_memory(),
                     "h_dqkv": torch.empty((B, T, 3 * C), dtype=tdt).pin_memory(),
                     "ev_in": torch.cuda.Event(), "ev_comp": torch.cuda.Event(), "ev_out": torch.cuda.Event()})
    s_h2d, s_d2h = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    e2e_ws = ops.Workspace()

    def e2e_run(n):
        for k in range(n):
            bf = bufs[k % 2]
            with torch.cuda.stream(s_h2d):
                if k >= 2:
                    s_h2d.wait_event(bf["ev_comp"])        # step k-2 no longer reads these inputs
                bf["qkv"].copy_(h_qkv, non_blocking=True)
                bf["dout"].copy_(h_dout, non_blocking=True)
                bf["ev_in"].record(s_h2d)
            stream.wait_event(bf["ev_in"])
            if k >= 2:
                stream.wait_event(bf["ev_out"])            # step k-2's results have been read out
            ops.attention_forward(bf["qkv"], NH, bool(causal), out=bf["out"], lse=bf["lse"], stream=stream)
            ops.attention_backward(bf["dout"], bf["qkv"], bf["out"], bf["lse"], NH, bool(causal), dqkv=bf["dqkv"],
                                   workspace=e2e_ws, stream=stream)
            bf["ev_comp"].record(stream)
            with torch.cuda.stream(s_d2h):
                s_d2h.wait_event(bf["ev_comp"])
                bf["h_out"].copy_(bf["out"], non_blocking=True)
                bf["h_dqkv"].copy_(bf["dqkv"], non_blocking=True)
                bf["ev_out"].record(s_d2h)

    e2e_run(4)
    barrier()
    n_e2e = max(20, min(args.steps, 200))
    ev_a, ev_b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev_a.record(s_h2d)
    stream.wait_event(ev_a)
    s_d2h.wait_event(ev_a)
    e2e_run(n_e2e)
    s_h2d.wait_stream(s_d2h)
    s_h2d.wait_stream(stream)
    ev_b.record(s_h2d)
    barrier()
    e2e_ms = ev_a.elapsed_time(ev_b) / n_e2e
    e2e_val, _ = aggregate(f["step"], e2e_ms, world, dev)

    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": t_max, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": w.dtype, "data": "synthetic", "config": config_dict(w),
        "pct_of_peak": value / peak_tf,
        "fwd_tflops": f["fwd"] / (fwd_ms * 1e-3) / 1e12, "bwd_tflops": f["bwd"] / (bwd_ms * 1e-3) / 1e12,
        "fwd_hbm_gbs": ab["fwd"] / (fwd_ms * 1e-3) / 1e9, "bwd_hbm_gbs": ab["bwd"] / (bwd_ms * 1e-3) / 1e9,
        "roofline": roofline, "kernels": kern,
        "e2e": {"value": e2e_val / 1e12, "unit": "TFLOP/s",
                "h2d_bytes_per_step": int((qkv.numel() + dout.numel()) * esz),
                "d2h_bytes_per_step": int((out.numel() + dqkv.numel()) * esz),
                "ms_per_step": e2e_ms,
                "pipeline": "h2d, compute and d2h on three streams, two device buffer sets; "
                            "time of the whole sequence / steps"},
        "gpu_launches": 4 * args.steps,
        "clocks": clocks,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args.workload)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


# CUDA sources each kernel is compiled from (its translation unit and headers)
_KERNEL_SOURCES = {
    "attn_fwd_kernel": ["attn_fwd.cu", "fwd_deal.cuh", "common.cuh", "ptx.cuh"],
    "attn_bwd_kernel": ["attn_bwd.cu", "fwd_deal.cuh", "common.cuh", "ptx.cuh"],
    "attn_decode_split": ["attn_decode.cu", "common.cuh", "ptx.cuh"],
    "f32": ["attn_f32.cu", "tf32.cuh", "common.cuh", "ptx.cuh"],
}


def stored_traffic(kernel: str, workload: str):
    """DRAM bytes per launch of `kernel` on `workload` from one ncu capture
    (profiles/traffic.json, key "<kernel>@<workload>"), or None when there is
    no capture of this workload or the kernel's code has changed since."""
    f = ROOT / "profiles" / "traffic.json"
    if not f.exists():
        return None
    tr = json.loads(f.read_text()).get(f"{kernel}@{workload}")
    if tr and tr.get("source_hash") == kernel_source_hash(kernel):
        return tr["bytes_per_launch"]
    return None


def _code_only(text: str) -> str:
    """C++ source with its comments and blank lines taken out, so that a change
    to a comment keeps a kernel's hash."""
    import re
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return "\n".join(ln.rstrip() for ln in text.splitlines() if ln.strip())


def kernel_source_hash(kernel: str = "attn_bwd_kernel") -> str:
    """Hash of the code (comments excluded) of the CUDA sources a kernel is
    built from; ties a stored ncu traffic figure to the kernel version it
    measured."""
    import hashlib
    h = hashlib.sha256()
    csrc = ROOT / "causal_head_attention_fwd_gb300" / "csrc"
    names = _KERNEL_SOURCES.get("f32" if "f32" in kernel else kernel)
    if names is None:
        return ""
    for name in names:
        h.update(name.encode())
        h.update(_code_only((csrc / name).read_text()).encode())
    return h.hexdigest()[:16]


if __name__ == "__main__":
    sys.exit(main())
