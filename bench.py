"""Benchmark of the block-sparse attention hot path on GB300.

One step = one pass of the whole path over one batch of the video-DiT
workload: tile map -> mean pool -> route (E + TopK) -> block-sparse
attention.  B=1, h=24, D=128, token grid (T,H,W)=(30,48,80) (N=115200),
(4,4,8) blocks of 128 tokens (J=960, the last temporal block row holds 2
frames), k=96 kept blocks per query block, bf16 inputs, fp32 accumulation.

Metric: effective sparse-attention TFLOP/s = 4*Hq*N*d*k*B_k / step time
(the FLOP count of the "MSA ... KV-outer" page, eq. 13/15).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line on rank 0.  With --impl reference the CPU oracle is
timed on the host cores on a bounded sample of the same workload.
"""

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOAD = dict(name="video_dit_bsa", B=1, heads=24, D=128, grid=(30, 48, 80), block=(4, 4, 8), M=128,
                k=96, seed=202)


def metric_flops(w):
    T, H, W = w["grid"]
    N = T * H * W
    return 4.0 * w["B"] * w["heads"] * N * w["D"] * w["k"] * w["M"]


def read_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    except (OSError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


# ---------------------------------------------------------------- clocks

class ClockSampler:
    """Samples nvidia-smi clocks and throttle reasons while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------- CPU oracle sample

ORACLE_SAMPLE = r"""
import json, os, sys, time
sys.path.insert(0, {root!r})
import numpy as np, torch
import oracle
from block_sparse_attention_tile_gb300 import synthetic
w = json.loads({w!r})
budget_s = {budget}
T, H, W = w["grid"]; bT, bH, bW = w["block"]; D = w["D"]; k = w["k"]
t0 = time.perf_counter()
q, kk, v = synthetic.video_qkv(1, 1, T, H, W, D, w["seed"], torch.bfloat16, field=True)
Q, K, V = (x[0].float().numpy().astype(np.float64) for x in (q, kk, v))
gen_s = time.perf_counter() - t0
t0 = time.perf_counter()
blocks = oracle.tile_3d(T, H, W, bT, bH, bW)
qbar, kbar = oracle.pool_blocks(Q, blocks), oracle.pool_blocks(K, blocks)
E = oracle.routing_scores(qbar, kbar, D)
idx, num = oracle.route(E, k, k)
route_s = time.perf_counter() - t0
rng = np.random.default_rng(0)
order = rng.permutation(len(blocks))
t0 = time.perf_counter(); done = 0
while done < len(order) and (done < 2 or time.perf_counter() - t0 < budget_s):
    oracle.block_sparse_attention(Q, K, V, blocks, idx, num, D ** -0.5, query_blocks=[int(order[done])])
    done += 1
attn_s = time.perf_counter() - t0
J = len(blocks)
step_s = w["B"] * w["heads"] * (route_s + J * attn_s / done)
print(json.dumps(dict(step_s=step_s, blocks=done, J=J, route_s=route_s, attn_s=attn_s, gen_s=gen_s)))
"""


def run_oracle_sample(budget_s=15.0):
    """Times the CPU oracle in a fresh interpreter (spawned, never forked)."""
    cores = os.cpu_count() or 1
    env = dict(os.environ)
    for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        env[var] = str(cores)
    env["CUDA_VISIBLE_DEVICES"] = ""
    code = ORACLE_SAMPLE.format(root=ROOT, w=json.dumps(WORKLOAD), budget=budget_s)
    out = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env, timeout=900)
    if out.returncode != 0:
        raise RuntimeError("oracle sample failed:\n" + out.stderr[-2000:])
    r = json.loads(out.stdout.strip().splitlines()[-1])
    value = metric_flops(WORKLOAD) / r["step_s"] / 1e12
    sample = ("1 of %d heads: tile map, pool and route of all %d blocks (%.1f s) plus %d of %d query blocks "
              "attended (%.1f s); step time scaled by heads and blocks"
              % (WORKLOAD["heads"], r["J"], r["route_s"], r["blocks"], r["J"], r["attn_s"]))
    return {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "sample": sample,
            "step_s_extrapolated": r["step_s"]}


# ---------------------------------------------------------------- GPU arm

def kernel_source_hash(files):
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "block_sparse_attention_tile_gb300", "csrc")
    for name in files:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def read_traffic(kernel):
    """Per-launch DRAM bytes of `kernel` from the committed ncu summary, only if
    it was taken on the kernel's current source files."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            t = json.load(f)
        e = t[kernel]
        if e.get("source_hash") != kernel_source_hash(e["source_files"]):
            return None
        return e.get("bytes_per_launch")
    except (OSError, ValueError, KeyError):
        return None


def gpu_arm(args):
    import torch
    import torch.distributed as dist

    from block_sparse_attention_tile_gb300 import bsa, pipeline, synthetic

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    w = dict(WORKLOAD)
    if args.heads:
        w["heads"] = args.heads
        w["name"] = WORKLOAD["name"] + "_%dheads" % args.heads
    T, H, W = w["grid"]
    N = T * H * W
    BH, D, M, k = w["B"] * w["heads"], w["D"], w["M"], w["k"]

    # inputs resident in HBM (seeded generator on the device; per-rank seed)
    with torch.no_grad():
        q, kk, v = synthetic.video_qkv(w["B"], w["heads"], T, H, W, D, w["seed"] + 1000 * rank,
                                       torch.bfloat16, device=dev, field=True)
    geom = pipeline.Geometry(T, H, W, *w["block"], M=M)
    geo = geom.geometry
    J = geom.num_blocks
    scale = D ** -0.5
    im = torch.empty((J, M), dtype=torch.int32, device=dev)
    bs = torch.empty((J,), dtype=torch.int32, device=dev)
    qbar = torch.empty((BH, J, D), dtype=torch.float32, device=dev)
    kbar = torch.empty_like(qbar)
    q2k = torch.empty((BH, J, k), dtype=torch.int32, device=dev)
    q2n = torch.empty((BH, J), dtype=torch.int32, device=dev)
    out = torch.empty_like(q)
    lse = torch.empty((BH, N), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()

    def step(ev=None):
        if ev: ev[0].record(stream)
        bsa.bsa_tile_map(T, H, W, *w["block"], 0, None, M, im, bs)
        if ev: ev[1].record(stream)
        bsa.bsa_pool_blocks(q, kk, None, BH, N, D, im, bs, J, M, qbar, kbar)
        if ev: ev[2].record(stream)
        bsa.bsa_route_topk(qbar, kbar, BH, J, D, J * D, k, scale, k, q2k, q2n)
        if ev: ev[3].record(stream)
        bsa.bsa_fwd_qouter(q, kk, v, BH, N, D, im, bs, J, M, 0, geo, q2k, q2n, k, scale, out, lse)
        if ev: ev[4].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if bsa.bsa_device_status() != bsa.BSA_OK:
        raise RuntimeError("device status after warm-up: " + bsa.bsa_last_error())

    # algorithmic work of one attention launch: 4*D per valid (query, key) pair
    sizes = bs.long()
    sel_sizes = sizes[q2k.long()].sum(-1)                        # [BH, J] keys visited
    pairs = (sizes[None, :] * sel_sizes).sum().item()
    attn_flops = 4.0 * D * pairs
    pool_bytes = 2 * BH * N * D * 2 + 2 * BH * J * D * 4 + J * M * 4 + J * 4

    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(args.steps)]
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for i in range(args.steps):
        step(ev[i])
    t_end.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clk = clocks.stop()
    ms_total = t_start.elapsed_time(t_end)
    stage_ms = {name: statistics.mean(e[j].elapsed_time(e[j + 1]) for e in ev)
                for j, name in enumerate(["tile_map", "pool", "route", "attention"])}
    if bsa.bsa_device_status() != bsa.BSA_OK:
        raise RuntimeError("device status after timing: " + bsa.bsa_last_error())

    # end to end through the public API with host buffers
    hq, hk, hv = (x.cpu().pin_memory() for x in (q, kk, v))
    hout = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    dq, dk, dv = torch.empty_like(q), torch.empty_like(kk), torch.empty_like(v)

    def e2e_step():
        dq.copy_(hq, non_blocking=True)
        dk.copy_(hk, non_blocking=True)
        dv.copy_(hv, non_blocking=True)
        bsa.bsa_tile_map(T, H, W, *w["block"], 0, None, M, im, bs)
        bsa.bsa_pool_blocks(dq, dk, None, BH, N, D, im, bs, J, M, qbar, kbar)
        bsa.bsa_route_topk(qbar, kbar, BH, J, D, J * D, k, scale, k, q2k, q2n)
        bsa.bsa_fwd_qouter(dq, dk, dv, BH, N, D, im, bs, J, M, 0, geo, q2k, q2n, k, scale, out, lse)
        hout.copy_(out, non_blocking=True)

    for _ in range(max(1, args.warmup)):
        e2e_step()
    e2e_steps = max(1, min(args.steps, 5))
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / e2e_steps

    # max over ranks
    t = torch.tensor([ms_total, e2e_ms], device=dev)
    if world > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    ms_total, e2e_ms = t.tolist()
    ms_step = ms_total / args.steps

    if rank == 0:
        peaks, peak_kind = read_peaks()
        flops = metric_flops(w)
        tensor_peak = peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"])
        attn_tflops = attn_flops / (stage_ms["attention"] * 1e-3) / 1e12
        pool_gbs = pool_bytes / (stage_ms["pool"] * 1e-3) / 1e9
        props = torch.cuda.get_device_properties(dev)
        fp32_peak = props.multi_processor_count * 128 * 2 * peaks.get("sm_max_mhz", 2070.0) * 1e6 / 1e12
        route_tflops = 2.0 * BH * J * J * D / (stage_ms["route"] * 1e-3) / 1e12
        line = {
            "metric": "sparse-attn effective TFLOP/s (4*Hq*N*d*k*Bk/s)",
            "value": world * flops / (ms_step * 1e-3) / 1e12,
            "unit": "TFLOP/s",
            "n_gpus": world,
            "steps": args.steps,
            "warmup": args.warmup,
            "ms_per_step": ms_step,
            "higher_is_better": True,
            "scaling": "weak" if world > 1 else "none",
            "vs_baseline": None,
            "dtype": "bf16",
            "data": "synthetic (seeded N(0,1) + smooth space-time field on Q/K; no dataset or weights)",
            "config": {"workload": w["name"], "B": w["B"], "heads": w["heads"], "D": w["D"], "seq_len": N,
                       "grid": list(w["grid"]), "block": list(w["block"]), "J": J, "k": k,
                       "global_batch": w["B"] * world, "parallelism": "replicas%d" % world if world > 1 else "single",
                       "l2": "inputs larger than L2: Q,K,V = %.2f GB per step" % (3 * q.numel() * 2 / 1e9)},
            "stages_us": {kname: round(v * 1e3, 1) for kname, v in stage_ms.items()},
            "roofline": {"bound": "tensor", "achieved": attn_tflops, "peak": tensor_peak, "unit": "TFLOP/s",
                         "frac": attn_tflops / tensor_peak, "traffic": read_traffic("attention"),
                         "kernel": "bsa_fwd_qouter attention", "peak_kind": peak_kind + " bf16 sustained",
                         "algorithmic_flops_per_launch": attn_flops},
            "rooflines_secondary": {
                "pool": {"bound": "hbm", "achieved": pool_gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": pool_gbs / peaks["hbm_gbs"], "bytes_per_launch": pool_bytes},
                "route": {"bound": "alu", "achieved": route_tflops, "peak": fp32_peak, "unit": "TFLOP/s",
                          "frac": route_tflops / fp32_peak, "flops_per_launch": 2.0 * BH * J * J * D,
                          "peak_note": "SMs x 128 FP32 lanes x 2 x max SM clock"}},
            "e2e": {"value": world * flops / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
                    "h2d_bytes_per_step": 3 * q.numel() * 2, "d2h_bytes_per_step": out.numel() * 2,
                    "ms_per_step": e2e_ms},
            "gpu_launches": 4 * args.steps,
            "clocks": clk,
        }
        if not args.no_cpu_baseline and world == 1:
            try:
                line["cpu_baseline"] = run_oracle_sample(args.cpu_budget)
            except Exception as exc:  # noqa: BLE001
                line["cpu_baseline"] = {"value": None, "error": str(exc)[:300]}
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def reference_arm(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    steps = []
    cb = None
    for i in range(args.warmup + args.steps):
        cb = run_oracle_sample(max(2.0, args.cpu_budget / 3))
        if i >= args.warmup:
            steps.append(cb["step_s_extrapolated"])
    step_s = statistics.mean(steps)
    value = metric_flops(WORKLOAD) / step_s / 1e12
    line = {"impl": "reference", "metric": "sparse-attn effective TFLOP/s (4*Hq*N*d*k*Bk/s)",
            "value": value, "unit": "TFLOP/s", "n_gpus": int(os.environ.get("WORLD_SIZE", "1")),
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_s * 1e3,
            "higher_is_better": True, "scaling": "none", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": WORKLOAD["name"], "seq_len": 115200,
                                            "heads": 24, "D": 128, "k": 96},
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cb["cores"], "kind": "oracle",
                             "sample": cb["sample"]},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--heads", type=int, default=0,
                    help="fewer heads than the workload's 24 (a small case for profiler captures)")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        print("warning: fewer than 3 warm-up steps", file=sys.stderr)
    if args.impl == "reference":
        reference_arm(args)
    else:
        gpu_arm(args)


if __name__ == "__main__":
    main()
