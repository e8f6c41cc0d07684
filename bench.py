#!/usr/bin/env python
"""Benchmark of causal RoPE self-attention forward + backward on GB300.

One step = the training pair ne_attn_fwd_train + ne_attn_bwd_train (all
kernels of the path: the q, k rotation pass, the forward, the backward's
preprocess, main kernel and postprocess) over one batch of the GPT-2-small
training shape, B=8, H=12, T=1024, D=64, bf16 inputs drawn N(0,1) from a fixed
seed, inputs resident in HBM.  The plain pair ne_attn_fwd + ne_attn_bwd (same
results, RoPE applied in both directions) is timed beside it.  The L2 is flushed (a 512 MiB
write) between timed steps, outside the timed region.  Throughput counts the
causal FLOPs: 2*B*H*T^2*D forward plus 2.5x that backward.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

N > 1 runs N independent replicas (the operation needs no exchange between
GPUs), one process per GPU under torch.distributed; value = all ranks' FLOPs /
the slowest rank's time.  ``--impl reference`` times the CPU oracle (the
plain double-precision C implementation) on a bounded sample of the same
workload on this host's cores.  Prints one JSON line.
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

METRIC = "RoPE causal attention fwd+bwd TFLOP/s at B8 H12 T1024 D64; % of BF16 peak"
UNIT = "TFLOP/s"
WORKLOAD = "gpt2s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--e2e-steps", type=int, default=100)
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="target CPU time of the oracle baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--path", choices=("train", "decode"), default="train",
                    help="train: the fwd+bwd step (the headline); decode: one generation "
                         "step against a KV cache (decode16k)")
    ap.add_argument("--extra-steps", type=int, default=50,
                    help="timed steps of each longer workload reported beside the headline")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the longer workloads and the decode step")
    ap.add_argument("--cpu-sample", type=float, default=None, help=argparse.SUPPRESS)
    return ap.parse_args()


def flops_fwd_bwd(B, H, T, D):
    fwd = 2.0 * B * H * T * T * D
    return fwd, 2.5 * fwd


def workload_flops(inp):
    """Causal fwd and bwd FLOPs of a workload: 2*H*D*sum(L^2) forward (2*B*H*T^2*D
    for a fixed-length batch), 2.5x that backward."""
    H, D = inp["H"], inp["D"]
    lengths = inp["lengths"] if "lengths" in inp else [inp["T"]] * inp["B"]
    fwd = 2.0 * H * D * sum(float(L) * L for L in lengths)
    return fwd, 2.5 * fwd


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f), "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def rank_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0")),
            int(os.environ.get("WORLD_SIZE", "1")))


def slowest_rank_ms(ms, world, device=None):
    """The largest of the ranks' times (every rank gets it).  Replicas share
    nothing, so the job is as fast as its slowest rank."""
    if world <= 1:
        return ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tflops(flops_per_step_per_rank, steps, ms, world):
    """Whole-job throughput: the FLOPs of all ranks' steps over the slowest
    rank's time for them (ms)."""
    return world * flops_per_step_per_rank * steps / (ms * 1e-3) / 1e12


# --------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi clock/throttle samples of one GPU while it runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.proc = None
        self.out = None
        try:
            self.out = open(f"/tmp/ne_clocks_{os.getpid()}.csv", "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", str(device_index), "-lms", "50"], stdout=self.out,
                stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.out.close()
        rows = []
        with open(self.out.name) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.out.name)
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i] == "Active"})
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": reasons, "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(sm)}


# ------------------------------------------------------------------ CPU oracle
def oracle_sample(seconds_target, inp, fixed_T=None):
    """Time the oracle (as it stands) on whole heads of the workload until about
    `seconds_target` seconds have been spent; returns (flops, seconds, heads, T)."""
    import oracle
    B, T, H, D = inp["B"], inp["T"], inp["H"], inp["D"]
    T = fixed_T or T
    fwd, bwd = flops_fwd_bwd(1, 1, T, D)
    heads = 0
    t0 = time.perf_counter()
    while True:
        b, h = divmod(heads % (B * H), H)
        q, k, v, do = (inp[n][b, :T, h:h + 1] for n in ("q", "k", "v", "dout"))
        oracle.attention(q, k, v, do, [0, T], base=inp["rope_base"], scale=inp["scale"])
        heads += 1
        el = time.perf_counter() - t0
        if el >= seconds_target or heads >= 4 * B * H:
            break
    return heads * (fwd + bwd), el, heads, T


def run_cpu_sample(args):
    """Print the oracle's throughput on a bounded sample of the headline workload
    (used by the benchmark to time the oracle on one core in a child process)."""
    import oracle
    from causal_self_attention_gb300.inputs import make_inputs
    oracle.build()
    fl, sec, heads, Ts = oracle_sample(args.cpu_sample, make_inputs(WORKLOAD))
    print(json.dumps({"flops": fl, "seconds": sec, "heads": heads, "T": Ts,
                      "cores": oracle.num_threads()}))
    return 0


def oracle_one_core(seconds):
    """The oracle's TFLOP/s on one host core, measured in a child process with
    OMP_NUM_THREADS=1 (spawned with exec, so it shares nothing with this
    process's CUDA context)."""
    env = dict(os.environ, OMP_NUM_THREADS="1")
    for k in ("RANK", "LOCAL_RANK", "WORLD_SIZE"):
        env.pop(k, None)
    r = subprocess.run([sys.executable, os.path.abspath(__file__), "--cpu-sample", str(seconds)],
                       env=env, capture_output=True, text=True, timeout=600)
    if r.returncode != 0:
        return None
    rec = json.loads(r.stdout.strip().splitlines()[-1])
    return {"value": rec["flops"] / rec["seconds"] / 1e12, "unit": UNIT, "cores": rec["cores"],
            "sample": f"{rec['heads']} whole heads (b, h) of the {WORKLOAD} workload, "
                      f"T={rec['T']}, fwd+bwd in fp64, {rec['seconds']:.1f} s"}


def run_reference(args):
    rank, _, world = rank_env()
    if world > 1 and rank != 0:
        return 0
    import oracle
    from causal_self_attention_gb300.inputs import make_inputs
    inp = make_inputs(WORKLOAD)
    B, T, H, D = inp["B"], inp["T"], inp["H"], inp["D"]
    # Calibrate one head, then size each step so the whole run stays within minutes.
    oracle.build()
    t0 = time.perf_counter()
    oracle_sample(0.0, inp)
    t_head = time.perf_counter() - t0
    budget = 150.0
    Ts = T
    while (args.steps + args.warmup) * t_head * (Ts / T) ** 2 > budget and Ts > 64:
        Ts //= 2
    for _ in range(args.warmup):
        oracle_sample(0.0, inp, fixed_T=Ts)
    total_flops, total_s = 0.0, 0.0
    for _ in range(args.steps):
        f, s, _, _ = oracle_sample(0.0, inp, fixed_T=Ts)
        total_flops += f
        total_s += s
    value = total_flops / total_s / 1e12
    sample = (f"one head (b, h) of the {WORKLOAD} workload per step, positions 0..{Ts - 1}, "
              f"fwd+bwd in fp64, all of the oracle's OpenMP threads")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * total_s / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{WORKLOAD}: B={B} H={H} T={T} D={D}, causal, RoPE base 10000, "
                               "fwd+bwd", "sample_T": Ts},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.num_threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


# --------------------------------------------------------------------- ours
def source_sha(paths):
    h = hashlib.sha256()
    for p in paths:
        with open(os.path.join(ROOT, p), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel):
    """Per-launch DRAM bytes of `kernel` from the committed ncu summary, or None
    when the kernel source has changed since the counters were taken."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f).get(kernel)
    if not rec:
        return None
    if rec.get("source_sha") != source_sha(rec["sources"]):
        return None
    return rec.get("dram_bytes_per_launch")


def bench_workloads(args, dev, stream, flush, peak_tf):
    """Fwd+bwd throughput of the longer workloads (byte-level contexts and the
    packed varlen batch), each with the L2 flushed before every timed step.
    The headline stays the GPT-2-small line; these are reported beside it."""
    import torch

    from causal_self_attention_gb300 import ne_attn as na
    from causal_self_attention_gb300.inputs import make_inputs
    res = {}
    for name in ("byte4k", "long16k", "varlen"):
        inp = make_inputs(name)
        q, k, v, do = (inp[n].to(dev) for n in ("q", "k", "v", "dout"))
        base, scale = inp["rope_base"], inp["scale"]
        H, D = inp["H"], inp["D"]
        N = q.shape[0] * (q.shape[1] if q.dim() == 4 else 1)
        ws = torch.empty(na.ne_attn_bwd_workspace_bytes(N, H, D), dtype=torch.uint8, device=dev)
        out = torch.empty_like(q)
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        qr, kr = torch.empty_like(q), torch.empty_like(k)
        if "cu_seqlens" in inp:
            cu, mx = inp["cu_seqlens"].to(dev), inp["max_seqlen"]
            lse = torch.empty((H, N), dtype=torch.float32, device=dev)

            def fwd():
                na.ne_attn_varlen_fwd_train(q, k, v, cu, mx, base, scale, out=out, lse=lse,
                                            qr=qr, kr=kr, stream=stream)

            def bwd():
                na.ne_attn_varlen_bwd_train(qr, kr, v, out, do, lse, cu, mx, base, scale,
                                            dq=dq, dk=dk, dv=dv, workspace=ws, stream=stream)
        else:
            B, T = inp["B"], inp["T"]
            lse = torch.empty((B, H, T), dtype=torch.float32, device=dev)

            def fwd():
                na.ne_attn_fwd_train(q, k, v, base, scale, out=out, lse=lse, qr=qr, kr=kr,
                                     stream=stream)

            def bwd():
                na.ne_attn_bwd_train(qr, kr, v, out, do, lse, base, scale, dq=dq, dk=dk, dv=dv,
                                     workspace=ws, stream=stream)
        for _ in range(3):
            flush.zero_()
            fwd()
            bwd()
        n = max(args.extra_steps, 3)
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(n)]
        for e in ev:
            flush.zero_()
            e[0].record(stream)
            fwd()
            e[1].record(stream)
            bwd()
            e[2].record(stream)
        torch.cuda.synchronize()
        assert na.ne_attn_get_device_status() == 0
        f_fwd, f_bwd = workload_flops(inp)
        t_all = [e[0].elapsed_time(e[2]) for e in ev]
        t_f = [e[0].elapsed_time(e[1]) for e in ev]
        t_b = [e[1].elapsed_time(e[2]) for e in ev]
        mean, medi = statistics.mean(t_all), statistics.median(t_all)
        shape = (f"B={inp['B']} H={H} T={inp['T']} D={D}" if "B" in inp else
                 f"{len(inp['lengths'])} sequences, L~U[64,2048] (sum {N}), H={H} D={D}")
        res[name] = {
            "shape": shape, "steps": n, "gflop_per_step": (f_fwd + f_bwd) / 1e9,
            "ms_per_step": mean, "ms_per_step_median": medi,
            "tflops": (f_fwd + f_bwd) / (mean * 1e-3) / 1e12,
            "tflops_at_median": (f_fwd + f_bwd) / (medi * 1e-3) / 1e12,
            "pct_bf16_peak": 100.0 * (f_fwd + f_bwd) / (mean * 1e-3) / 1e12 / peak_tf,
            "fwd_ms_median": statistics.median(t_f), "bwd_ms_median": statistics.median(t_b),
            "fwd_tflops_at_median": f_fwd / (statistics.median(t_f) * 1e-3) / 1e12,
            "bwd_tflops_at_median": f_bwd / (statistics.median(t_b) * 1e-3) / 1e12,
        }
        del q, k, v, do, ws, out, dq, dk, dv, lse, qr, kr
    return res


def proj_summary(args, dev, stream, flush, peak_tf):
    """The projections around the attention at the GPT-2-small shape (B=8,
    T=1024, C=768): RMSNorm + QKV projection with RoPE in the epilogue, and
    the output projection + residual; each timed with CUDA events, the L2
    flushed before every step, beside the same products by torch.matmul
    (cuBLAS) for context."""
    import torch

    from causal_self_attention_gb300 import ne_attn as na
    B, T, H = 8, 1024, 12
    C, M = H * 64, B * T
    g = torch.Generator().manual_seed(77)
    x = torch.randn((M, C), generator=g).to(torch.bfloat16).to(dev)
    gw = (torch.randn((C,), generator=g) * 0.1 + 1.0).to(torch.bfloat16).to(dev)
    wq = (torch.randn((3 * C, C), generator=g) / C ** 0.5).to(torch.bfloat16).to(dev)
    wo = (torch.randn((C, C), generator=g) / C ** 0.5).to(torch.bfloat16).to(dev)
    res = torch.randn((M, C), generator=g).to(torch.bfloat16).to(dev)
    xn = torch.empty_like(x)
    rstd = torch.empty(M, dtype=torch.float32, device=dev)
    q, k, v = (torch.empty((B, T, H, 64), dtype=torch.bfloat16, device=dev) for _ in range(3))
    y = torch.empty_like(x)

    def qkv():
        na.ne_rmsnorm_qkv_rope(x, gw, wq, T, x_norm=xn, rstd=rstd, q=q, k=k, v=v, stream=stream)

    def outp():
        na.ne_out_proj_residual(x, wo, res, y=y, stream=stream)

    def cublas_qkv():
        torch.matmul(xn, wq.t())

    def cublas_out():
        torch.addmm(res, x, wo.t())

    n = max(args.extra_steps, 3)
    res_ms = {}
    for name, fn in (("qkv", qkv), ("out", outp), ("cublas_qkv", cublas_qkv),
                     ("cublas_out", cublas_out)):
        for _ in range(3):
            fn()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(n)]
        for a, b in ev:
            flush.zero_()
            a.record(stream)
            fn()
            b.record(stream)
        torch.cuda.synchronize()
        res_ms[name] = statistics.median(a.elapsed_time(b) for a, b in ev)
    assert na.ne_attn_get_device_status() == 0
    fq, fo = 2.0 * M * 3 * C * C, 2.0 * M * C * C
    return {
        "shape": f"M={M} (B={B} T={T}), C={C}: QKV [M,{C}]x[{3 * C},{C}]^T, out [M,{C}]x[{C},{C}]^T",
        "steps": n,
        "rmsnorm_qkv_rope": {"ms_median": res_ms["qkv"],
                             "tflops": fq / (res_ms["qkv"] * 1e-3) / 1e12,
                             "frac_bf16_peak": fq / (res_ms["qkv"] * 1e-3) / 1e12 / peak_tf,
                             "cublas_gemm_only_ms_median": res_ms["cublas_qkv"]},
        "out_proj_residual": {"ms_median": res_ms["out"],
                              "tflops": fo / (res_ms["out"] * 1e-3) / 1e12,
                              "frac_bf16_peak": fo / (res_ms["out"] * 1e-3) / 1e12 / peak_tf,
                              "cublas_addmm_ms_median": res_ms["cublas_out"]},
    }


def mtp_summary(args, dev, stream, flush, peak_tf):
    """The multi-token prediction head at the GPT-2-small shape (8192 tokens of
    width 768, heads for the next token and the one after it, a 256-way byte
    vocabulary): logits with the cross-entropy in the GEMM epilogue, dh and dW;
    timed with CUDA events, the L2 flushed before every step, beside torch's
    three bare products (cuBLAS) for context."""
    import torch

    from causal_self_attention_gb300 import ne_attn as na
    M, C, K, V = 8192, 768, 2, 256
    g = torch.Generator().manual_seed(91)
    h = torch.randn((M, C), generator=g).to(torch.bfloat16).to(dev)
    w = (torch.randn((K * V, C), generator=g) * (2.0 / C ** 0.5)).to(torch.bfloat16).to(dev)
    tg = torch.randint(0, V, (M, K), generator=g, dtype=torch.int32)
    tg[-1, 1] = -1  # the last token has no token two ahead
    tg = tg.to(dev)
    loss = torch.empty(1, dtype=torch.float32, device=dev)
    row = torch.empty((M, K), dtype=torch.float32, device=dev)
    dh = torch.empty_like(h)
    dw = torch.empty((K * V, C), dtype=torch.float32, device=dev)
    ws = torch.empty(na.ne_mtp_head_workspace_bytes(M, K, V), dtype=torch.uint8, device=dev)
    dl = torch.empty((M, K * V), dtype=torch.bfloat16, device=dev)

    def ours():
        na.ne_mtp_head(h, w, tg, K, loss=loss, row_loss=row, dh=dh, dw=dw, workspace=ws,
                       stream=stream)

    def cublas():
        torch.matmul(h, w.t())
        torch.matmul(dl, w)
        torch.matmul(dl.t(), h)

    n = max(args.extra_steps, 3)
    res_ms = {}
    for name, fn in (("ours", ours), ("cublas", cublas)):
        for _ in range(3):
            fn()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(n)]
        for a, b in ev:
            flush.zero_()
            a.record(stream)
            fn()
            b.record(stream)
        torch.cuda.synchronize()
        res_ms[name] = statistics.median(a.elapsed_time(b) for a, b in ev)
    assert na.ne_attn_get_device_status() == 0
    fl = 3 * 2.0 * M * C * K * V  # logits, dh, dW
    return {
        "shape": f"M={M} tokens, C={C}, K={K} heads (next token and the one after), V={V}",
        "steps": n, "gflop": fl / 1e9,
        "ms_median": res_ms["ours"], "tflops": fl / (res_ms["ours"] * 1e-3) / 1e12,
        "frac_bf16_peak": fl / (res_ms["ours"] * 1e-3) / 1e12 / peak_tf,
        "cublas_three_products_ms_median": res_ms["cublas"],
        "loss": float(loss.cpu()[0]),
    }


def _time_calls(fn, n, stream):
    """Per-call device times (ms) of n calls of fn on stream, CUDA events."""
    import torch
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(n)]
    for a, b in ev:
        a.record(stream)
        fn()
        b.record(stream)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in ev]


def decode_summary(args, dev, stream, peaks):
    """One decode step over a KV cache (decode16k), timed with CUDA events:
    GB/s of K and V read, against the measured HBM bandwidth.  Also the same
    step on a cache of rotated keys (ne_attn_decode_rotated: q' and k' given,
    nothing rotated, no table read)."""
    import torch

    from causal_self_attention_gb300 import ne_attn as na
    from causal_self_attention_gb300.inputs import make_decode
    inp = make_decode(DECODE_WORKLOAD)
    B, H, Tmax = inp["B"], inp["H"], inp["Tmax"]
    q, kc, vc, pos = (inp[n].to(dev) for n in ("q", "k_cache", "v_cache", "pos"))
    out = torch.empty_like(q)
    lse = torch.empty((B, H), dtype=torch.float32, device=dev)
    ws = torch.empty(na.ne_attn_decode_workspace_bytes(B, H, Tmax), dtype=torch.uint8, device=dev)

    def rotating():
        na.ne_attn_decode(q, kc, vc, pos, inp["rope_base"], inp["scale"], out=out, lse=lse,
                          workspace=ws, stream=stream)

    def rotated():  # timing only: the cache's contents do not change the work
        na.ne_attn_decode_rotated(q, kc, vc, pos, inp["scale"], out=out, lse=lse, workspace=ws,
                                  stream=stream)

    n = max(4 * args.extra_steps, 3)
    kv = decode_kv_bytes(inp)
    res = {}
    for name, fn in (("rotating", rotating), ("rotated", rotated)):
        for _ in range(5):
            fn()
        # the cache (2 x 403 MB) is larger than L2: no flush needed
        res[name] = _time_calls(fn, n, stream)
    assert na.ne_attn_get_device_status() == 0
    t = res["rotating"]
    medi = statistics.median(t)
    medr = statistics.median(res["rotated"])
    return {"workload": f"{DECODE_WORKLOAD}: B={B} H={H} Tmax={Tmax} D=64, one new token per "
                        "sequence at the last cache row", "steps": n,
            "ms_per_step": statistics.mean(t), "ms_per_step_median": medi,
            "gbs_at_median": kv / (medi * 1e-3) / 1e9, "kv_bytes_per_step": kv,
            "frac_hbm": kv / (medi * 1e-3) / 1e9 / peaks["hbm_gbs"],
            "rotated_cache": {"how": "ne_attn_decode_rotated: cache of k' = R(n) k, q' given",
                              "ms_per_step_median": medr,
                              "gbs_at_median": kv / (medr * 1e-3) / 1e9,
                              "frac_hbm": kv / (medr * 1e-3) / 1e9 / peaks["hbm_gbs"]}}


def run_ours(args):
    import torch
    import torch.distributed as dist

    from causal_self_attention_gb300 import build as nb
    rank, local_rank, world = rank_env()
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    if rank == 0 or world == 1:
        nb.build()
    if world > 1:
        dist.barrier()
    from causal_self_attention_gb300 import ne_attn as na
    from causal_self_attention_gb300.inputs import make_inputs

    inp = make_inputs(WORKLOAD)
    B, T, H, D = inp["B"], inp["T"], inp["H"], inp["D"]
    base, scale = inp["rope_base"], inp["scale"]
    f_fwd, f_bwd = flops_fwd_bwd(B, H, T, D)
    f_step = f_fwd + f_bwd
    q, k, v, do = (inp[n].to(dev) for n in ("q", "k", "v", "dout"))
    out = torch.empty_like(q)
    lse = torch.empty((B, H, T), dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    qr, kr = torch.empty_like(q), torch.empty_like(k)  # rotated operands kept for the backward
    ws = torch.empty(na.ne_attn_bwd_workspace_bytes(B * T, H, D), dtype=torch.uint8, device=dev)
    flush = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()

    def fwd():
        na.ne_attn_fwd_train(q, k, v, base, scale, out=out, lse=lse, qr=qr, kr=kr, stream=stream)

    def bwd():
        na.ne_attn_bwd_train(qr, kr, v, out, do, lse, base, scale, dq=dq, dk=dk, dv=dv,
                             workspace=ws, stream=stream)

    def plain_step():
        na.ne_attn_fwd(q, k, v, base, scale, out=out, lse=lse, stream=stream)
        na.ne_attn_bwd(q, k, v, out, do, lse, base, scale, dq=dq, dk=dk, dv=dv, workspace=ws,
                       stream=stream)

    for _ in range(max(args.warmup, 3)):
        flush.zero_()
        fwd()
        bwd()
        flush.zero_()
        plain_step()
    torch.cuda.synchronize()
    assert na.ne_attn_get_device_status() == 0

    K = args.steps
    # Timed region: K whole steps, one event pair per step and nothing between
    # the kernels of a step (they run back to back, each launched so that it
    # may start while the previous one drains).
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
    for e in ev:  # torch creates the CUDA event on first record: create them all now
        for x in e:
            x.record(stream)
    torch.cuda.synchronize()
    clocks = ClockSampler(local_rank)
    time.sleep(0.3)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    w0 = time.perf_counter()
    for i in range(K):
        e = ev[i]
        flush.zero_()
        e[0].record(stream)
        fwd()
        bwd()
        e[1].record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    wall = time.perf_counter() - w0
    clk = clocks.stop()
    status = na.ne_attn_get_device_status()
    t_step = [e[0].elapsed_time(e[1]) for e in ev]
    total_ms = slowest_rank_ms(sum(t_step), world, dev)
    value = job_tflops(f_step, K, total_ms, world)
    median_ms = slowest_rank_ms(statistics.median(t_step), world, dev)

    # Per-kernel breakdown (outside the timed region): the same steps with an
    # event between every two kernels, which times each kernel on its own.
    KB = min(K, 300)
    evb = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(KB)]
    for e in evb:  # the library records three of them: torch must have created them first
        for x in e:
            x.record(stream)
    for i in range(KB):
        e = evb[i]
        flush.zero_()
        na.ne_attn_set_fwd_phase_event(e[1])
        na.ne_attn_set_bwd_phase_events(e[3], e[4])
        e[0].record(stream)
        fwd()
        e[2].record(stream)
        bwd()
        e[5].record(stream)
    torch.cuda.synchronize()
    na.ne_attn_set_fwd_phase_event(None)
    na.ne_attn_set_bwd_phase_events(None, None)
    status = status or na.ne_attn_get_device_status()
    t_rot = [e[0].elapsed_time(e[1]) for e in evb]
    t_fwd = [e[1].elapsed_time(e[2]) for e in evb]
    t_pre = [e[2].elapsed_time(e[3]) for e in evb]
    t_main = [e[3].elapsed_time(e[4]) for e in evb]
    t_post = [e[4].elapsed_time(e[5]) for e in evb]
    t_sep = [e[0].elapsed_time(e[5]) for e in evb]

    # The plain pair (RoPE inside both directions), for comparison.
    KP = min(K, 300)
    evp = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(KP)]
    for e in evp:
        flush.zero_()
        e[0].record(stream)
        plain_step()
        e[1].record(stream)
    torch.cuda.synchronize()
    status = status or na.ne_attn_get_device_status()
    t_plain = [e[0].elapsed_time(e[1]) for e in evp]

    # ---- end to end through the public API with host buffers ------------------
    # Every step uploads its q, k, v, dO from pinned host memory and downloads
    # all of its results (O, LSE, dQ, dK, dV).  As a training pipeline would,
    # the copies run on their own streams with three device buffer sets: step
    # i+1's inputs upload while step i computes and step i-1's results
    # download.  Each direction moves one contiguous block (q, k, v, dO as
    # [4, B, T, H, 64]; O, dQ, dK, dV likewise; the tensors the calls take are
    # views of it) plus LSE: measured 8% faster than one copy per tensor, the
    # host link being the bound (~200 GB/s each way, ~330 GB/s both at once).
    # The timed region spans the first upload to the last download.
    h_in = torch.stack([inp[n] for n in ("q", "k", "v", "dout")]).pin_memory()
    h_res = torch.empty((4,) + tuple(q.shape), dtype=torch.bfloat16).pin_memory()
    h_lse = torch.empty(lse.shape, dtype=torch.float32).pin_memory()
    h2d = h_in.numel() * h_in.element_size()
    d2h = h_res.numel() * h_res.element_size() + h_lse.numel() * h_lse.element_size()
    KE = max(args.e2e_steps, 2)
    NSETS = 3
    s_in = torch.cuda.Stream(dev)
    s_out = torch.cuda.Stream(dev)
    s_comp = stream
    sets = []
    for _ in range(NSETS):
        d_in = torch.empty_like(h_in, device=dev)
        d_res = torch.empty_like(h_res, device=dev)
        sets.append({"in": d_in, "res": d_res, "q": d_in[0], "k": d_in[1], "v": d_in[2],
                     "dout": d_in[3], "out": d_res[0], "dq": d_res[1], "dk": d_res[2],
                     "dv": d_res[3], "lse": torch.empty_like(lse), "qr": torch.empty_like(q),
                     "kr": torch.empty_like(q)})

    def e2e_run(n_steps):
        ev_in = [torch.cuda.Event() for _ in range(n_steps)]
        ev_comp = [torch.cuda.Event() for _ in range(n_steps)]
        ev_out = [torch.cuda.Event() for _ in range(n_steps)]
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(s_in)
        for i in range(n_steps):
            d = sets[i % NSETS]
            if i >= NSETS:
                s_in.wait_event(ev_comp[i - NSETS])  # step i-3 no longer reads these inputs
            with torch.cuda.stream(s_in):
                d["in"].copy_(h_in, non_blocking=True)
            ev_in[i].record(s_in)
            s_comp.wait_event(ev_in[i])
            if i >= NSETS:
                s_comp.wait_event(ev_out[i - NSETS])  # step i-3's results have been read out
            na.ne_attn_fwd_train(d["q"], d["k"], d["v"], base, scale, out=d["out"],
                                 lse=d["lse"], qr=d["qr"], kr=d["kr"], stream=s_comp)
            na.ne_attn_bwd_train(d["qr"], d["kr"], d["v"], d["out"], d["dout"], d["lse"], base,
                                 scale, dq=d["dq"], dk=d["dk"], dv=d["dv"], workspace=ws,
                                 stream=s_comp)
            ev_comp[i].record(s_comp)
            s_out.wait_event(ev_comp[i])
            with torch.cuda.stream(s_out):
                h_res.copy_(d["res"], non_blocking=True)
                h_lse.copy_(d["lse"], non_blocking=True)
            ev_out[i].record(s_out)
        t1.record(s_out)
        torch.cuda.synchronize()
        return t0.elapsed_time(t1) / n_steps

    e2e_run(3)  # warm-up
    e2e_ms = slowest_rank_ms(e2e_run(KE), world, dev)
    e2e_value = job_tflops(f_step, 1, e2e_ms, world)

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return 0

    peaks, peak_kind = load_peaks()
    peak_tf = peaks["bf16_tflops"]
    per_kernel = {
        "ne_attn_rope_rows_kernel": statistics.mean(t_rot),
        "ne_attn_fwd_kernel": statistics.mean(t_fwd),
        "ne_attn_bwd_prep_stream_kernel": statistics.mean(t_pre),
        "ne_attn_bwd_kernel": statistics.mean(t_main),
        "ne_attn_dq_postprocess_kernel": statistics.mean(t_post),
    }
    dom = max(per_kernel, key=per_kernel.get)
    kernel_flops = {"ne_attn_fwd_kernel": f_fwd, "ne_attn_bwd_kernel": f_bwd}
    achieved = kernel_flops.get(dom, 0.0) / (per_kernel[dom] * 1e-3) / 1e12
    roofline = {"bound": "tensor", "kernel": dom, "achieved": achieved, "peak": peak_tf,
                "unit": "TFLOP/s", "frac": achieved / peak_tf,
                "peak_source": f"{peak_kind} bf16 burst (MEASURED_PEAKS.json)"
                if peak_kind == "measured" else "fallback bf16 burst",
                "traffic": recorded_traffic(dom)}
    # HBM-bound helpers: algorithmic bytes / time.
    n_el = B * T * H * D
    rot_bytes = 4 * n_el * 2                                  # read q, k; write q', k'
    pre_bytes = 2 * n_el * 2 + B * H * T * 4 + n_el * 4       # read O, dO; write D; zero dQ'
    post_bytes = n_el * 4 + n_el * 2 + 2 * n_el * 2       # read dQ', write dQ; dK in place
    med = {"ne_attn_rope_rows_kernel": statistics.median(t_rot),
           "ne_attn_fwd_kernel": statistics.median(t_fwd),
           "ne_attn_bwd_prep_stream_kernel": statistics.median(t_pre),
           "ne_attn_bwd_kernel": statistics.median(t_main),
           "ne_attn_dq_postprocess_kernel": statistics.median(t_post)}
    kernels = {
        "ne_attn_rope_rows_kernel": {
            "ms": per_kernel["ne_attn_rope_rows_kernel"],
            "gbs": rot_bytes / (per_kernel["ne_attn_rope_rows_kernel"] * 1e-3) / 1e9},
        "ne_attn_fwd_kernel": {"ms": per_kernel["ne_attn_fwd_kernel"],
                               "tflops": f_fwd / (per_kernel["ne_attn_fwd_kernel"] * 1e-3) / 1e12},
        "ne_attn_bwd_kernel": {"ms": per_kernel["ne_attn_bwd_kernel"],
                               "tflops": f_bwd / (per_kernel["ne_attn_bwd_kernel"] * 1e-3) / 1e12},
        "ne_attn_bwd_prep_stream_kernel": {
            "ms": per_kernel["ne_attn_bwd_prep_stream_kernel"],
            "gbs": pre_bytes / (per_kernel["ne_attn_bwd_prep_stream_kernel"] * 1e-3) / 1e9},
        "ne_attn_dq_postprocess_kernel": {
            "ms": per_kernel["ne_attn_dq_postprocess_kernel"],
            "gbs": post_bytes / (per_kernel["ne_attn_dq_postprocess_kernel"] * 1e-3) / 1e9},
    }
    for name in kernels:
        kernels[name]["ms_median"] = med[name]
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": max(args.warmup, 3), "ms_per_step": total_ms / K,
        "ms_per_step_median": median_ms,
        "value_at_median": job_tflops(f_step, 1, median_ms, world), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"{WORKLOAD}: B={B} H={H} T={T} D={D}, causal, RoPE base 10000, "
                               "fwd+bwd (training pair)", "B": B, "H": H, "T": T, "D": D,
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": "flushed (512 MiB write) between timed steps"},
        "pct_bf16_peak": 100.0 * value / (world * peak_tf),
        "pct_bf16_peak_sustained": 100.0 * value / (world * peaks.get("bf16_tflops_sustained",
                                                                      peak_tf)),
        "roofline": roofline,
        "kernels": kernels,
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                "how": "pinned host buffers; each step one upload of q, k, v, dO (one "
                       "contiguous block, the calls take views of it) and one download of O, "
                       "dQ, dK, dV plus LSE, on their own streams; three device buffer sets "
                       "(step i+1 uploads while step i computes and step i-1 downloads); "
                       f"{KE} steps timed from the first upload to the last download"},
        "breakdown": {"steps": KB, "ms_per_step_kernels_apart": statistics.mean(t_sep),
                      "how": "events between the kernels (outside the timed region): each "
                             "kernel timed on its own, without the overlap of one kernel's "
                             "start with the previous one's drain"},
        "plain_pair": {"steps": KP, "ms_per_step_median": statistics.median(t_plain),
                       "tflops_at_median": f_step / (statistics.median(t_plain) * 1e-3) / 1e12,
                       "how": "ne_attn_fwd + ne_attn_bwd (RoPE applied inside the forward and "
                              "again in the backward's preprocess), L2 flushed, outside the "
                              "timed region"},
        "gpu_launches": 5 * K,
        "clocks": clk,
        "wall_s": wall,
        "device_status": status,
    }
    if not args.no_extras:
        line["workloads"] = bench_workloads(args, dev, stream, flush, peak_tf)
        line["decode"] = decode_summary(args, dev, stream, peaks)
        line["projections"] = proj_summary(args, dev, stream, flush, peak_tf)
        line["mtp_head"] = mtp_summary(args, dev, stream, flush, peak_tf)
    if not args.no_cpu_baseline and (world == 1 or rank == 0):
        import oracle
        oracle.build()
        fl, s, heads, Ts = oracle_sample(args.cpu_seconds, inp)
        line["cpu_baseline"] = {
            "value": fl / s / 1e12, "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"{heads} whole heads (b, h) of the {WORKLOAD} workload, T={Ts}, fwd+bwd "
                      f"in fp64, {s:.1f} s"}
        one = oracle_one_core(args.cpu_seconds)
        if one is not None:
            line["cpu_baseline"]["one_core"] = one
    print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()
    return 0


# ------------------------------------------------------------------- decode
DECODE_WORKLOAD = "decode16k"
DECODE_METRIC = "decode attention KV-cache read GB/s at B8 H12 Tmax16384 D64"


def decode_kv_bytes(inp):
    """Algorithmic bytes of one decode step: every attended K and V row once."""
    return sum(int(p) + 1 for p in inp["pos"]) * inp["H"] * inp["D"] * 2 * 2


def run_decode(args):
    import torch

    from causal_self_attention_gb300 import build as nb
    rank, local_rank, world = rank_env()
    if world > 1 and rank != 0:
        return 0  # one GPU is enough: the decode line is measured on rank 0 only
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    nb.build()
    from causal_self_attention_gb300 import ne_attn as na
    from causal_self_attention_gb300.inputs import make_decode

    inp = make_decode(DECODE_WORKLOAD)
    B, H, Tmax, D = inp["B"], inp["H"], inp["Tmax"], inp["D"]
    base, scale = inp["rope_base"], inp["scale"]
    q, kc, vc, pos = (inp[n].to(dev) for n in ("q", "k_cache", "v_cache", "pos"))
    out = torch.empty_like(q)
    lse = torch.empty((B, H), dtype=torch.float32, device=dev)
    ws = torch.empty(na.ne_attn_decode_workspace_bytes(B, H, Tmax), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    kv_bytes = decode_kv_bytes(inp)

    def step(s=stream):
        na.ne_attn_decode(q, kc, vc, pos, base, scale, out=out, lse=lse, workspace=ws, stream=s)

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    assert na.ne_attn_get_device_status() == 0
    K = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(K)]
    clocks = ClockSampler(local_rank)
    time.sleep(0.3)
    torch.cuda.synchronize()
    for i in range(K):  # the cache (2 x 403 MB) is larger than L2: no flush needed
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    status = na.ne_attn_get_device_status()
    ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
    gbs = kv_bytes / (ms * 1e-3) / 1e9

    # End to end: the new token's q, k, v rows uploaded (one copy of one
    # contiguous block) and written into the cache, O and LSE read back (one
    # copy: both are views of one device block), every step, one step after
    # the other as a generation loop runs (the cache itself stays resident,
    # as a KV cache does).
    h_in = torch.stack([inp["q"], inp["k_cache"][:, -1], inp["v_cache"][:, -1]]).pin_memory()
    d_in = torch.empty_like(h_in, device=dev)
    o_bytes = out.numel() * out.element_size()
    d_res = torch.empty(o_bytes + lse.numel() * 4, dtype=torch.uint8, device=dev)
    h_res = torch.empty(d_res.shape, dtype=torch.uint8).pin_memory()
    e_out = d_res[:o_bytes].view(torch.bfloat16).view(out.shape)
    e_lse = d_res[o_bytes:].view(torch.float32).view(lse.shape)
    h2d = h_in.numel() * h_in.element_size()
    d2h = h_res.numel()
    KE = max(args.e2e_steps, 2)
    last = int(inp["pos"][0])

    def e2e_step():
        d_in.copy_(h_in, non_blocking=True)
        kc[:, last].copy_(d_in[1])
        vc[:, last].copy_(d_in[2])
        na.ne_attn_decode(d_in[0], kc, vc, pos, base, scale, out=e_out, lse=e_lse, workspace=ws,
                          stream=stream)
        h_res.copy_(d_res, non_blocking=True)

    for _ in range(3):  # warm-up: the first pass pays one-time set-up (~0.6 s measured)
        e2e_step()
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(KE):
        e2e_step()
    t1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = t0.elapsed_time(t1) / KE

    # The same step on a cache of rotated keys (outside the timed region).
    def step_rot(s=stream):
        na.ne_attn_decode_rotated(q, kc, vc, pos, scale, out=out, lse=lse, workspace=ws, stream=s)

    for _ in range(3):
        step_rot()
    t_rot = statistics.median(_time_calls(step_rot, max(K, 3), stream))
    assert na.ne_attn_get_device_status() == 0

    peaks, peak_kind = load_peaks()
    line = {
        "metric": DECODE_METRIC, "value": gbs, "unit": "GB/s", "n_gpus": 1, "steps": K,
        "warmup": max(args.warmup, 3), "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"{DECODE_WORKLOAD}: B={B} H={H} Tmax={Tmax} D={D}, one new "
                               "token per sequence at the last cache row, RoPE base 10000",
                   "B": B, "H": H, "Tmax": Tmax, "D": D,
                   "l2": "cache larger than L2 (2 x 403 MB)"},
        "roofline": {"bound": "hbm", "kernel": "ne_attn_decode_split_kernel", "achieved": gbs,
                     "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": gbs / peaks["hbm_gbs"],
                     "peak_source": f"{peak_kind} HBM copy (MEASURED_PEAKS.json)",
                     "traffic": recorded_traffic("ne_attn_decode_split_kernel")},
        "e2e": {"value": kv_bytes / (e2e_ms * 1e-3) / 1e9, "unit": "GB/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms},
        "gpu_launches": 2 * K,
        "clocks": clk,
        "device_status": status,
        "rotated_cache": {"how": "ne_attn_decode_rotated on a cache of k' = R(n) k with q' "
                                 "given (nothing rotated, no table read); outside the timed "
                                 "region", "ms_per_step_median": t_rot,
                          "gbs_at_median": kv_bytes / (t_rot * 1e-3) / 1e9,
                          "frac_hbm": kv_bytes / (t_rot * 1e-3) / 1e9 / peaks["hbm_gbs"]},
    }
    if not args.no_cpu_baseline:
        import oracle
        oracle.build()
        t_start = time.perf_counter()
        done = 0
        Lc = int(inp["pos"][0]) + 1
        for b in range(B):
            qs = torch.zeros((Lc, H, D), dtype=torch.bfloat16)
            qs[Lc - 1] = inp["q"][b]
            oracle.attention_sampled(qs, inp["k_cache"][b, :Lc], inp["v_cache"][b, :Lc], None,
                                     [0, Lc], [(0, h, [Lc - 1], []) for h in range(H)],
                                     base=base, scale=scale, mode=1)
            done += Lc * H * D * 2 * 2
            if time.perf_counter() - t_start > args.cpu_seconds:
                break
        sec = time.perf_counter() - t_start
        line["cpu_baseline"] = {"value": done / sec / 1e9, "unit": "GB/s",
                                "cores": oracle.num_threads(), "kind": "oracle",
                                "sample": f"{done // (Lc * H * D * 4)} of {B} sequences' decode "
                                          f"rows (all heads), {sec:.1f} s"}
    print(json.dumps(line))
    return 0


def main():
    args = parse()
    if args.cpu_sample is not None:
        return run_cpu_sample(args)
    if args.path == "decode":
        return run_decode(args)
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
