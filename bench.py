"""Benchmark of the block-sparse attention hot path on GB300.

One step = one pass of the whole path over one batch of a workload.  The
default workload (the one the headline line reports) is the video-DiT one:
tile map -> mean pool -> route (E + TopK) -> block-sparse attention, B=1,
h=24, D=128, token grid (T,H,W)=(30,48,80) (N=115200), (4,4,8) blocks of 128
tokens (J=960, the last temporal block row holds 2 frames), k=96 kept blocks
per query block, bf16 inputs, fp32 accumulation.

Other workloads (--workload):
  video_tiny     fp32, h=2, D=64, grid (8,16,16), (4,4,4) blocks, k=8
  nsa_prefill    bf16 GQA selected prefill, B=2, T=8192, HQ=64, H=4, BS=64,
                 S=16: reverse index -> KV-outer partials -> combine
                 (the query-outer order is timed beside it)
  msa_prefill    bf16, B=1, N=32768, Hq=64, Hkv=4, Bk=128, k=16 with
                 Zipf(1.1) hot blocks: the same KV-outer pipeline
  spark_summary  bf16, h=24, 1024 text tokens + (16,32,64) video under a
                 permutation, 128-token blocks, k=26, summaries of the
                 unselected blocks
  spark_reweight the same with Spark-Reweight summaries (weighted key and
                 value at the head's mean video query, log-mass bias)
  spark_reblock  the spark_summary inputs in the Spark-Reblock layout (one per
                 head, built on the GPU each step) instead of a seeded
                 permutation; rows gathered into it and outputs scattered back
  r2v_bsa        bf16, h=24, R2V layout: 1024 text tokens, two reference
                 videos (8,48,80) and the target (30,48,80) in (4,4,8) windows;
                 region-grouped TopK keeping 10% of each video region
  video_dit_coarse  the default workload plus the gated coarse branch
                 softmax(E) V_bar broadcast to each block's tokens (synthetic
                 per-head, per-channel gate)

Metric: effective sparse-attention TFLOP/s = 4*Hq*N*d*k*B_k / step time
(the FLOP count of the "MSA ... KV-outer" page, eq. 13/15).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload NAME]

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

METRIC = "sparse-attn effective TFLOP/s (4*Hq*N*d*k*Bk/s)"

WORKLOADS = {
    "video_dit_bsa": dict(kind="block", B=1, heads=24, D=128, grid=(30, 48, 80), block=(4, 4, 8), M=128, k=96,
                          seed=202, dtype="bf16"),
    "video_tiny": dict(kind="block", B=1, heads=2, D=64, grid=(8, 16, 16), block=(4, 4, 4), M=64, k=8, seed=101,
                       dtype="f32"),
    "spark_summary": dict(kind="block", B=1, heads=24, D=128, grid=(16, 32, 64), block=(1, 1, 1), M=128, k=26,
                          seed=505, dtype="bf16", n_text=1024, summary=True),
    "r2v_bsa": dict(kind="block", B=1, heads=24, D=128, segments=[1024, (8, 48, 80), (8, 48, 80), (30, 48, 80)],
                    block=(4, 4, 8), M=128, budgets=[24, 24, 96], k=144, seed=707, dtype="bf16"),
    "spark_reblock": dict(kind="block", B=1, heads=24, D=128, grid=(16, 32, 64), block=(1, 1, 1), M=128, k=26,
                          seed=505, dtype="bf16", n_text=1024, summary=True, reblock=True),
    "video_dit_coarse": dict(kind="block", B=1, heads=24, D=128, grid=(30, 48, 80), block=(4, 4, 8), M=128, k=96,
                             seed=202, dtype="bf16", coarse=True),
    "spark_reweight": dict(kind="block", B=1, heads=24, D=128, grid=(16, 32, 64), block=(1, 1, 1), M=128, k=26,
                           seed=505, dtype="bf16", n_text=1024, summary=True, reweight=True),
    # each token workload runs in its page's order (the NSA selected branch query-outer, MSA KV-outer);
    # the other order is timed beside it
    "nsa_prefill": dict(kind="token", B=2, T=8192, HQ=64, H=4, D=128, BS=64, S=16, seed=303, zipf=False,
                        order="qouter"),
    "msa_prefill": dict(kind="token", B=1, T=32768, HQ=64, H=4, D=128, BS=128, S=16, seed=404, zipf=True,
                        order="kvouter"),
}
DEFAULT = "video_dit_bsa"


# GB300 dense bf16 tensor peak as the metric names it (~2.2 PFLOP/s), reported beside the measured one
NOMINAL_BF16_TFLOPS = 2200.0


def metric_flops(w):
    if w["kind"] == "token":
        return 4.0 * w["B"] * w["HQ"] * w["T"] * w["D"] * w["S"] * w["BS"]
    if "segments" in w:  # every video query token, the blocks kept per row
        nv = sum(s[0] * s[1] * s[2] for s in w["segments"] if not isinstance(s, int))
        return 4.0 * w["B"] * w["heads"] * nv * w["D"] * w["k"] * w["M"]
    T, H, W = w["grid"]
    return 4.0 * w["B"] * w["heads"] * T * H * W * w["D"] * w["k"] * w["M"]


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


# ---------------------------------------------------------------- CPU oracle samples

# Everything below runs in a spawned interpreter (bench.py --oracle-sample) with
# the GPU hidden and one BLAS thread per process: the setup (inputs, pooling,
# routing, reverse index) and a fixed subset of query blocks (or tokens) on one
# thread, then the same attention spread over a spawned process pool with one
# worker per host core.  Workers import this file, so it imports only the
# standard library at module level.
_ORACLE_STATE = {}
ORACLE_CHUNK_TOKENS = 8   # query tokens per unit of the token workloads (all heads)


def _oracle_setup(w):
    """The oracle's inputs and routing for one head (block workloads) or one
    batch element (token workloads); returns (state, setup seconds, units)."""
    import numpy as np
    import torch
    if ROOT not in sys.path:
        sys.path.insert(0, ROOT)
    import oracle
    from block_sparse_attention_tile_gb300 import synthetic
    st = {"w": w}
    if w["kind"] == "token":
        B, T, HQ, H, D, BS, S = (w[x] for x in ("B", "T", "HQ", "H", "D", "BS", "S"))
        q = synthetic.normal((1, T, HQ, D), w["seed"], dtype=torch.bfloat16)
        k = synthetic.normal((1, T, H, D), w["seed"] + 1, dtype=torch.bfloat16)
        v = synthetic.normal((1, T, H, D), w["seed"] + 2, dtype=torch.bfloat16)
        gen = synthetic.zipf_block_lists if w["zipf"] else synthetic.causal_block_lists
        idx, cnt = gen(1, T, H, S, BS, w["seed"])
        st.update(Q=q[0].double().numpy(), K=k[0].double().numpy(), V=v[0].double().numpy(), idx=idx[0],
                  cnt=cnt[0])
        t0 = time.perf_counter()
        nblk = -(-T // BS)
        oracle.reverse_index(np.transpose(idx, (0, 2, 1, 3)).reshape(H, T, S),
                             np.transpose(cnt, (0, 2, 1)).reshape(H, T), nblk)
        setup_s = time.perf_counter() - t0
        return st, setup_s, -(-T // ORACLE_CHUNK_TOKENS)
    bT, bH, bW = w["block"]
    D, k_, M = w["D"], w["k"], w["M"]
    segs = [x if isinstance(x, int) else tuple(x) for x in w["segments"]] if "segments" in w else None
    n_text = w.get("n_text", 0)
    summary, reweight, coarse = w.get("summary", False), w.get("reweight", False), w.get("coarse", False)
    dt = torch.bfloat16 if w["dtype"] == "bf16" else torch.float32
    spans = None
    if segs is not None:
        q, kk, v = synthetic.segment_qkv(1, segs, D, w["seed"], dt)
    elif summary:
        T, H, W = w["grid"]
        q, kk, v = synthetic.cluster_qkv(1, n_text, T * H * W, D, w["seed"], dt)
    else:
        T, H, W = w["grid"]
        q, kk, v = synthetic.video_qkv(1, 1, T, H, W, D, w["seed"], dt, field=(w["dtype"] == "bf16"))
    Q, K, V = (x[0].double().numpy() for x in (q, kk, v))
    t0 = time.perf_counter()
    if segs is not None:
        blocks, P, spans = oracle.tile_segments(segs, bT, bH, bW, M)
    elif summary:
        T, H, W = w["grid"]
        if w.get("reblock"):  # the Spark-Reblock layout of this head
            perm = oracle.reblock_layout(Q[n_text:], K[n_text:], M)
        else:
            perm = synthetic.permutation(T * H * W, w["seed"] + 1)
        blocks = oracle.tile_prefix(n_text, M) + oracle.tile_permuted(perm, M, offset=n_text)
        P = len(oracle.tile_prefix(n_text, M))
    else:
        T, H, W = w["grid"]
        blocks = oracle.tile_3d(T, H, W, bT, bH, bW)
        P = 0
    qbar, kbar = oracle.pool_blocks(Q, blocks), oracle.pool_blocks(K, blocks)
    vbar = oracle.pool_blocks(V, blocks) if (summary or coarse) else None
    E = oracle.routing_scores(qbar[P:], kbar[P:], D)
    if spans is not None:
        idx, num = oracle.route_grouped(E, [(lo - P, hi - P) for lo, hi in spans], w["budgets"], k_)
    else:
        idx, num = oracle.route(E, k_, k_)
    sbias = None
    if reweight:
        kbar, vbar, sbias, _ = oracle.reweight_summaries(
            Q, K, V, blocks, D ** -0.5, prefix_blocks=P,
            round_key=oracle.bf16_round if w["dtype"] == "bf16" else None)
        kbar = np.concatenate([np.zeros((P, D)), kbar])
        vbar = np.concatenate([np.zeros((P, D)), vbar])
    C = g = None
    if coarse:
        C = oracle.coarse_attention(E, vbar[P:])
        g = synthetic.normal((1, D), w["seed"] + 71)[0].double().numpy()
    setup_s = time.perf_counter() - t0
    st.update(Q=Q, K=K, V=V, blocks=blocks, P=P, idx=idx, num=num, kbar=kbar, vbar=vbar, sbias=sbias, C=C, g=g)
    return st, setup_s, len(blocks)


def _oracle_attend(st, units):
    """The oracle's attention for some units: query blocks (block workloads)
    or chunks of ORACLE_CHUNK_TOKENS query tokens with all their heads."""
    import oracle
    w = st["w"]
    if w["kind"] == "token":
        T = w["T"]
        toks = [t for u in units for t in range(u * ORACLE_CHUNK_TOKENS, min(T, (u + 1) * ORACLE_CHUNK_TOKENS))]
        if toks:
            oracle.nsa_selected_attention(st["Q"], st["K"], st["V"], st["idx"], st["cnt"], w["BS"], tokens=toks)
        return
    D, P = w["D"], st["P"]
    for qb in units:
        if w.get("summary"):
            oracle.summary_attention(st["Q"], st["K"], st["V"], st["blocks"], st["idx"], st["num"], st["kbar"][P:],
                                     st["vbar"][P:], D ** -0.5, prefix_blocks=P, query_blocks=[qb],
                                     block_bias=st["sbias"])
        else:
            O, _ = oracle.block_sparse_attention(st["Q"], st["K"], st["V"], st["blocks"], st["idx"], st["num"],
                                                 D ** -0.5, query_blocks=[qb], prefix_blocks=P)
            if st["C"] is not None and qb >= P:
                oracle.coarse_output(O, st["C"][qb - P:qb - P + 1], st["g"], [st["blocks"][qb]], 0)


def _oracle_worker_init(wjson):
    _ORACLE_STATE["st"] = _oracle_setup(json.loads(wjson))[0]


def _oracle_worker_wait(seconds):
    time.sleep(seconds)
    return 0


def _oracle_worker_task(units):
    _oracle_attend(_ORACLE_STATE["st"], units)
    return len(units)


def _oracle_sample_main(spec):
    """The spawned sampler: setup and a fixed subset on one thread, then the
    process pool, either for a time budget (cpu_baseline) or for `steps` steps
    of a fixed number of units each (the reference arm)."""
    import concurrent.futures
    import multiprocessing
    import random
    w = WORKLOADS[spec["workload"]]
    cores = spec["cores"]
    st, setup_s, total = _oracle_setup(w)
    order = list(range(total))
    random.Random(0).shuffle(order)
    n1 = min(total, 4 if w["kind"] == "block" else 2)
    t0 = time.perf_counter()
    _oracle_attend(st, order[:n1])
    t1_unit = (time.perf_counter() - t0) / n1
    out = {"cores": cores, "setup_s": setup_s, "units_total": total, "one_thread_units": n1,
           "one_thread_s_per_unit": t1_unit}
    # units per pool task: at least ~50 ms of work, so the pool's per-task
    # messaging stays small beside it
    per_task = max(1, min(64, int(0.05 / max(t1_unit, 1e-6)) + 1))
    out["units_per_task"] = per_task
    ctx = multiprocessing.get_context("spawn")
    with concurrent.futures.ProcessPoolExecutor(cores, mp_context=ctx, initializer=_oracle_worker_init,
                                                initargs=(json.dumps(w),)) as ex:
        # every worker set up (its initializer runs before its first task) before the clock starts
        list(ex.map(_oracle_worker_wait, [1.0] * (2 * cores)))
        pos = n1
        if spec.get("steps"):
            walls, units = [], []
            for _ in range(spec["steps"]):
                n = spec["units_per_step"] * per_task
                seq = [order[(pos + i) % total] for i in range(n)]
                pos += n
                batch = [seq[i:i + per_task] for i in range(0, n, per_task)]
                t0 = time.perf_counter()
                done = sum(ex.map(_oracle_worker_task, batch))
                walls.append(time.perf_counter() - t0)
                units.append(done)
            out.update(step_walls_s=walls, step_units=units)
        else:
            t0 = time.perf_counter()
            done = 0
            while pos < total and (done < cores or time.perf_counter() - t0 < spec["budget_s"]):
                seq = order[pos:pos + cores * per_task]
                pos += len(seq)
                done += sum(ex.map(_oracle_worker_task, [seq[i:i + per_task] for i in range(0, len(seq), per_task)]))
            out.update(all_core_units=done, all_core_wall_s=time.perf_counter() - t0)
    print(json.dumps(out), flush=True)


def _run_sampler(spec):
    env = dict(os.environ)
    for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        env[var] = "1"
    env["CUDA_VISIBLE_DEVICES"] = ""
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--oracle-sample", json.dumps(spec)],
                         capture_output=True, text=True, env=env, timeout=1800)
    if out.returncode != 0:
        raise RuntimeError("oracle sample failed:\n" + out.stderr[-2000:])
    return json.loads(out.stdout.strip().splitlines()[-1])


def _sample_scale(w):
    """(independent setups per step, units per setup, unit name)."""
    if w["kind"] == "token":
        return w["B"], "chunks of %d query tokens (all %d heads)" % (ORACLE_CHUNK_TOKENS, w["HQ"])
    return w["B"] * w["heads"], "query blocks of one head"


def run_oracle_sample(wname, budget_s=15.0):
    """The CPU oracle as it stands, on a bounded sample of the workload: one
    thread on a fixed subset, and all host cores through a spawned process
    pool; both extrapolated to a full step."""
    w = WORKLOADS[wname]
    cores = os.cpu_count() or 1
    r = _run_sampler({"workload": wname, "cores": cores, "budget_s": budget_s})
    setups, unit_name = _sample_scale(w)
    units = setups * r["units_total"]
    one_s = setups * r["setup_s"] + units * r["one_thread_s_per_unit"]
    all_s = setups * r["setup_s"] / cores + units * r["all_core_wall_s"] / r["all_core_units"]
    flops = metric_flops(w)
    sample = ("setup of one %s on one thread (%.2f s: inputs, %s); attention of %d %s on one thread "
              "(%.3f s each) and of %d more on %d spawned single-thread workers (%.1f s wall); both "
              "extrapolated to all %d setups x %d units of a step"
              % ("batch element" if w["kind"] == "token" else "head", r["setup_s"],
                 "reverse index" if w["kind"] == "token" else "tile map, pool, route and the other per-head stages",
                 r["one_thread_units"], unit_name, r["one_thread_s_per_unit"], r["all_core_units"], cores,
                 r["all_core_wall_s"], setups, r["units_total"]))
    return {"value": flops / all_s / 1e12, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
            "sample": sample, "extrapolated": True, "step_s_extrapolated": all_s,
            "one_thread": {"value": flops / one_s / 1e12, "step_s_extrapolated": one_s, "cores": 1},
            "all_core": {"value": flops / all_s / 1e12, "step_s_extrapolated": all_s, "cores": cores}}


# ---------------------------------------------------------------- traffic records

def kernel_source_hash(files):
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "block_sparse_attention_tile_gb300", "csrc")
    for name in files:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def read_traffic(workload):
    """Per-launch DRAM bytes of the workload's dominant kernel from the committed
    ncu summary, only if it was taken on the kernel's current source files."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            t = json.load(f)
        e = t[workload]
        if e.get("source_hash") != kernel_source_hash(e["source_files"]):
            return None
        return e.get("bytes_per_launch")
    except (OSError, ValueError, KeyError):
        return None


# ---------------------------------------------------------------- ranks

def rank_seed(base, rank):
    """Each replica draws its own inputs: the workload seed offset by the rank."""
    return base + 1000 * rank


def max_over_ranks(values, world, device="cpu"):
    """Element-wise maximum of a list of floats over all ranks (the slowest rank
    sets the job's time); a plain copy when world == 1."""
    import torch
    import torch.distributed as dist
    t = torch.tensor(values, dtype=torch.float64, device=device)
    if world > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def job_tflops(unit_flops, world, ms):
    """Whole-job throughput: every rank processes one workload (weak scaling)."""
    return world * unit_flops / (ms * 1e-3) / 1e12


# ---------------------------------------------------------------- workloads

_MEMCPY2D = []


def cuda_memcpy2d():
    """cudaMemcpy2DAsync of the CUDA runtime this process has loaded (torch's),
    through ctypes, or None.  A pitched copy moves one head slice of a
    [B, T, heads, D] host tensor without staging it: torch's copy of a
    non-contiguous pinned tensor first makes a contiguous pageable copy."""
    if _MEMCPY2D:
        return _MEMCPY2D[0]
    import ctypes
    fn = None
    try:
        paths = sorted({ln.split()[-1] for ln in open("/proc/self/maps") if "libcudart.so" in ln})
        for path in paths:
            lib = ctypes.CDLL(path)
            if hasattr(lib, "cudaMemcpy2DAsync"):
                fn = lib.cudaMemcpy2DAsync
                fn.argtypes = [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_size_t,
                               ctypes.c_size_t, ctypes.c_int, ctypes.c_void_p]
                fn.restype = ctypes.c_int
                break
    except OSError:
        fn = None
    _MEMCPY2D.append(fn)
    return fn


class BlockWorkload:
    """Tile map -> pool -> route -> block attention (exact, or exact + summary)."""

    stage_names = ["tile_map", "pool", "route", "attention"]

    def __init__(self, name, w, dev, rank):
        import torch
        from block_sparse_attention_tile_gb300 import pipeline, synthetic
        self.name, self.w, self.dev = name, w, dev
        self.torch = torch
        self.segments = [s if isinstance(s, int) else tuple(s) for s in w["segments"]] if "segments" in w else None
        if self.segments is None:
            T, H, W = w["grid"]
        self.summary = w.get("summary", False)
        self.reweight = self.summary and w.get("reweight", False)
        self.coarse = w.get("coarse", False)
        self.reblock = w.get("reblock", False)
        if self.reweight:
            self.stage_names = ["tile_map", "pool", "route", "reweight", "attention"]
        if self.coarse:
            self.stage_names = ["tile_map", "pool", "route", "attention", "coarse_attention", "coarse_apply"]
        self.core_stages = len(self.stage_names)
        self.ev_off = 0
        if self.reblock:
            self.stage_names = ["reblock", "permute"] + self.stage_names + ["unpermute"]
            self.ev_off = 2
        n_text = w.get("n_text", 0)
        D, M, k = w["D"], w["M"], w["k"]
        self.BH = w["B"] * w["heads"]
        self.dtype = torch.bfloat16 if w["dtype"] == "bf16" else torch.float32
        seed = rank_seed(w["seed"], rank)
        with torch.no_grad():
            if self.segments is not None:
                self.q, self.k, self.v = synthetic.segment_qkv(self.BH, self.segments, D, seed, self.dtype,
                                                               device=dev)
                self.perm = None
            elif self.summary:
                self.q, self.k, self.v = synthetic.cluster_qkv(self.BH, n_text, T * H * W, D, seed, self.dtype,
                                                               device=dev)
                self.perm = (None if self.reblock else
                             torch.as_tensor(synthetic.permutation(T * H * W, seed + 1), device=dev))
            else:
                self.q, self.k, self.v = synthetic.video_qkv(w["B"], w["heads"], T, H, W, D, seed, self.dtype,
                                                             device=dev, field=(w["dtype"] == "bf16"))
                self.perm = None
        if self.segments is not None:
            self.geom = pipeline.SegmentGeometry(self.segments, *w["block"], M=M)
        elif self.reblock:  # in the layout's order a block is a run of M rows
            self.geom = pipeline.Geometry(1, 1, T * H * W, 1, 1, M, M=M, n_prefix=n_text)
        else:
            self.geom = pipeline.Geometry(T, H, W, *w["block"], M=M, n_prefix=n_text, perm=self.perm)
        self.N = self.geom.n_tokens
        self.J = self.geom.num_blocks
        self.P = self.geom.prefix_blocks
        self.Jr = self.J - self.P
        if self.segments is not None:
            self.region_starts = [lo - self.P for lo, _ in self.geom.spans] + [self.Jr]
        self.scale = D ** -0.5
        BH, J = self.BH, self.J
        self.im = torch.empty((J, M), dtype=torch.int32, device=dev)
        self.bs = torch.empty((J,), dtype=torch.int32, device=dev)
        self.qbar = torch.empty((BH, J, D), dtype=torch.float32, device=dev)
        self.kbar = torch.empty_like(self.qbar)
        self.vbar = torch.empty_like(self.qbar) if (self.summary or self.coarse) else None
        self.kbar_lp = torch.empty((BH, J, D), dtype=self.dtype, device=dev) if self.summary else None
        self.vbar_lp = torch.empty((BH, J, D), dtype=self.dtype, device=dev) if self.summary else None
        # permuted blocks or a multi-segment layout: the pool pass also writes Q/K/V in block order for
        # the attention
        self.packed = (torch.empty((3, BH, J, M, D), dtype=self.dtype, device=dev)
                       if (self.perm is not None or self.segments is not None) else None)
        if self.packed is not None and self.vbar is None:
            self.vbar = torch.empty_like(self.qbar)
        from block_sparse_attention_tile_gb300 import bsa as _bsa
        self.route_ws = torch.empty((_bsa.bsa_route_workspace(BH, self.Jr) // 4,), dtype=torch.float32, device=dev)
        self.q2k = torch.empty((BH, self.Jr, k), dtype=torch.int32, device=dev)
        self.q2n = torch.empty((BH, self.Jr), dtype=torch.int32, device=dev)
        self.out = torch.empty_like(self.q)
        self.lse = torch.empty((BH, self.N), dtype=torch.float32, device=dev)
        self.sbias = torch.empty((BH, J), dtype=torch.float32, device=dev) if self.reweight else None
        self.rw_ws = (torch.empty((_bsa.bsa_reweight_workspace(BH, D) // 4,), dtype=torch.float32, device=dev)
                      if self.reweight else None)
        self.C = torch.empty((BH, self.Jr, D), dtype=torch.float32, device=dev) if self.coarse else None
        self.gate = (synthetic.normal((BH, D), seed + 71, dev) if self.coarse else None)
        # tile map, pool, route (contraction + select), [reweight: mean partials, mean, summaries], attention,
        # [coarse: attention, apply]
        self.launches_per_step = 5 + (3 if self.reweight else 0) + (2 if self.coarse else 0)
        self.core_out, self.core_lse = self.out, self.lse
        if self.reblock:
            Nv = self.N - n_text
            NB = -(-Nv // M)
            levels = max(0, (NB - 1).bit_length())
            self.rb_perm = torch.empty((BH, Nv), dtype=torch.int32, device=dev)
            self.rb_ws = torch.empty((_bsa.bsa_reblock_workspace(BH, self.N, D, n_text),), dtype=torch.uint8,
                                     device=dev)
            self.q2, self.k2, self.v2 = (torch.empty_like(x) for x in (self.q, self.k, self.v))
            self.core_out, self.core_lse = torch.empty_like(self.out), torch.empty_like(self.lse)
            # moment, reduce, factor, features, iota, one split per level, leaf sort; 3 gathers; 2 scatters
            self.launches_per_step += 6 + levels + 3 + 2

    def tile_map(self):
        from block_sparse_attention_tile_gb300 import bsa
        g, M = self.geom, self.w["M"]
        if self.segments is not None:
            bsa.bsa_tile_map_segments(self.segments, g.bT, g.bH, g.bW, M, self.im, self.bs)
        else:
            bsa.bsa_tile_map(g.T, g.H, g.W, g.bT, g.bH, g.bW, g.n_prefix, self.perm, M, self.im, self.bs)

    def route(self, qbar, kbar, nh, q2k, q2n):
        """TopK per row, or the region-grouped TopK of a multi-segment layout."""
        from block_sparse_attention_tile_gb300 import bsa
        D, kk = self.w["D"], self.w["k"]
        if self.segments is not None:
            bsa.bsa_route_topk_grouped(qbar, kbar, nh, self.Jr, D, self.J * D, self.region_starts,
                                       self.w["budgets"], self.scale, kk, q2k, q2n, self.route_ws)
        else:
            bsa.bsa_route_topk(qbar, kbar, nh, self.Jr, D, self.J * D, kk, self.scale, kk, q2k, q2n,
                               self.route_ws)

    def reblock_in(self, q, k, v, sl, nh):
        """The heads' layouts, then their rows gathered into them."""
        from block_sparse_attention_tile_gb300 import bsa
        n_text, M, D = self.w.get("n_text", 0), self.w["M"], self.w["D"]
        bsa.bsa_reblock_layout(q[sl], k[sl], nh, self.N, D, n_text, M, self.rb_perm[sl], self.rb_ws)

    def permute_in(self, q, k, v, sl, nh):
        from block_sparse_attention_tile_gb300 import bsa
        n_text, D = self.w.get("n_text", 0), self.w["D"]
        for src, dst in ((q, self.q2), (k, self.k2), (v, self.v2)):
            bsa.bsa_permute_rows(src[sl], dst[sl], nh, self.N, D, n_text, self.rb_perm[sl])

    def permute_out(self, sl, nh):
        from block_sparse_attention_tile_gb300 import bsa
        n_text, D = self.w.get("n_text", 0), self.w["D"]
        bsa.bsa_permute_rows(self.core_out[sl], self.out[sl], nh, self.N, D, n_text, self.rb_perm[sl], inverse=True)
        bsa.bsa_permute_rows(self.core_lse[sl].unsqueeze(-1), self.lse[sl].unsqueeze(-1), nh, self.N, 1, n_text,
                             self.rb_perm[sl], inverse=True)

    def step(self, ev=None, q=None, k=None, v=None):
        q = self.q if q is None else q
        k = self.k if k is None else k
        v = self.v if v is None else v
        if not self.reblock:
            return self.core_step(ev, q, k, v)
        st = self.torch.cuda.current_stream()
        sl = slice(0, self.BH)
        if ev: ev[0].record(st)
        self.reblock_in(q, k, v, sl, self.BH)
        if ev: ev[1].record(st)
        self.permute_in(q, k, v, sl, self.BH)
        self.core_step(ev, self.q2, self.k2, self.v2)
        self.permute_out(sl, self.BH)
        if ev: ev[len(self.stage_names)].record(st)

    def core_step(self, ev, q, k, v):
        from block_sparse_attention_tile_gb300 import bsa
        w, g = self.w, self.geom
        D, M, kk = w["D"], w["M"], w["k"]
        st = self.torch.cuda.current_stream()
        o = self.ev_off
        if ev: ev[o + 0].record(st)
        self.tile_map()
        if ev: ev[o + 1].record(st)
        bsa.bsa_pool_blocks(q, k, v if self.vbar is not None else None, self.BH, self.N, D, self.im, self.bs,
                            self.J, M, self.qbar, self.kbar, self.vbar, self.kbar_lp, self.vbar_lp,
                            packed=self.packed)
        if ev: ev[o + 2].record(st)
        self.route(self.qbar[:, self.P:], self.kbar[:, self.P:], self.BH, self.q2k, self.q2n)
        if ev: ev[o + 3].record(st)
        if self.reweight:
            bsa.bsa_reweight_summaries(q, k, v, self.BH, self.N, D, self.im, self.bs, self.J, M, self.P, self.scale,
                                       self.kbar_lp, self.vbar_lp, self.sbias, self.rw_ws, qbar=self.qbar,
                                       packed=self.packed)
            if ev: ev[o + 4].record(st)
        if self.summary:
            bsa.bsa_fwd_summary(q, k, v, self.BH, self.N, D, self.im, self.bs, self.J, M, self.P, g.geometry,
                                self.q2k, self.q2n, kk, self.kbar_lp, self.vbar_lp, self.scale, self.core_out,
                                self.core_lse, packed=self.packed, summary_bias=self.sbias)
        else:
            bsa.bsa_fwd_qouter(q, k, v, self.BH, self.N, D, self.im, self.bs, self.J, M, self.P, g.geometry,
                               self.q2k, self.q2n, kk, self.scale, self.core_out, self.core_lse, packed=self.packed)
        if self.coarse:
            if ev: ev[o + 4].record(st)
            bsa.bsa_coarse_attention(self.route_ws, self.Jr * self.Jr, self.vbar[:, self.P:], self.J * D, self.BH,
                                     self.Jr, D, self.C)
            if ev: ev[o + 5].record(st)
            bsa.bsa_coarse_apply(self.core_out, self.C, self.gate, False, self.BH, self.N, D, self.im, self.bs,
                                 self.J, M, self.P)
        if ev: ev[o + self.core_stages].record(st)

    def host_inputs(self):
        return [self.q, self.k, self.v], [self.out]

    def run_with(self, dev_inputs):
        self.step(None, *dev_inputs)

    def run_heads(self, q, k, v, h0, h1, packed_chunk):
        """Pool, route and attention for heads [h0, h1) only (the heads are
        independent): every entry point takes the head count and pointers
        offset to the first head; the tile map is shared."""
        from block_sparse_attention_tile_gb300 import bsa
        w, g = self.w, self.geom
        D, M, kk = w["D"], w["M"], w["k"]
        sl = slice(h0, h1)
        nh = h1 - h0
        if self.reblock:
            self.reblock_in(q, k, v, sl, nh)
            self.permute_in(q, k, v, sl, nh)
            q, k, v = self.q2, self.k2, self.v2
        bsa.bsa_pool_blocks(q[sl], k[sl], v[sl] if self.vbar is not None else None, nh, self.N, D, self.im,
                            self.bs, self.J, M, self.qbar[sl], self.kbar[sl],
                            self.vbar[sl] if self.vbar is not None else None,
                            self.kbar_lp[sl] if self.summary else None, self.vbar_lp[sl] if self.summary else None,
                            packed=packed_chunk)
        self.route(self.qbar[sl, self.P:], self.kbar[sl, self.P:], nh, self.q2k[sl], self.q2n[sl])
        sb = None
        if self.reweight:
            sb = self.sbias[sl]
            bsa.bsa_reweight_summaries(q[sl], k[sl], v[sl], nh, self.N, D, self.im, self.bs, self.J, M, self.P,
                                       self.scale, self.kbar_lp[sl], self.vbar_lp[sl], sb, self.rw_ws,
                                       qbar=self.qbar[sl], packed=packed_chunk)
        if self.summary:
            bsa.bsa_fwd_summary(q[sl], k[sl], v[sl], nh, self.N, D, self.im, self.bs, self.J, M, self.P, g.geometry,
                                self.q2k[sl], self.q2n[sl], kk, self.kbar_lp[sl], self.vbar_lp[sl], self.scale,
                                self.core_out[sl], self.core_lse[sl], packed=packed_chunk, summary_bias=sb)
        else:
            bsa.bsa_fwd_qouter(q[sl], k[sl], v[sl], nh, self.N, D, self.im, self.bs, self.J, M, self.P, g.geometry,
                               self.q2k[sl], self.q2n[sl], kk, self.scale, self.core_out[sl], self.core_lse[sl],
                               packed=packed_chunk)
        if self.coarse:
            bsa.bsa_coarse_attention(self.route_ws, self.Jr * self.Jr, self.vbar[sl, self.P:], self.J * D, nh,
                                     self.Jr, D, self.C[sl])
            bsa.bsa_coarse_apply(self.core_out[sl], self.C[sl], self.gate[sl], False, nh, self.N, D, self.im, self.bs,
                                 self.J, M, self.P)
        if self.reblock:
            self.permute_out(sl, nh)

    def make_e2e(self, h_in, d_in, h_out, heads_per_chunk=None):
        """End-to-end step with host buffers, pipelined by heads: chunk c's
        inputs are copied in on a copy stream while chunk c-1 computes, and each
        chunk's output is copied out as soon as it is done.  Chunks of 1, 2, then
        heads_per_chunk heads, and one head last.  The host-to-device copies bind
        the plain steps (at C2, 2-head chunks gave 15.31 ms, 3: 15.41, 4: 15.72,
        8: 17.2); a step that builds the Spark-Reblock layout pays its tree
        levels once a chunk, whatever the chunk's heads, so it takes 12-head
        chunks (2: 10.5 ms, 4: 8.0, 8: 6.9, 12: 6.7)."""
        if heads_per_chunk is None:
            heads_per_chunk = 12 if self.reblock else 2
        torch = self.torch
        g = self.geom
        comp = torch.cuda.current_stream()
        h2d_s, d2h_s = torch.cuda.Stream(), torch.cuda.Stream()
        # graded chunks: a one-head first chunk starts the compute early and a
        # one-head last chunk leaves little output to copy after it
        sizes = []
        left = self.BH
        for first in (1, 2):
            if left > 1:
                sizes.append(first)
                left -= first
        tail = [1] if left > 2 else []
        left -= sum(tail)
        while left > 0:
            sizes.append(min(heads_per_chunk, left))
            left -= sizes[-1]
        sizes += tail
        chunks, h0 = [], 0
        for n_h in sizes:
            chunks.append((h0, h0 + n_h))
            h0 += n_h
        per_head = self.J * self.w["M"] * self.w["D"]
        dq, dk, dv = d_in
        hq, hk, hv = h_in
        (hout,) = h_out
        # Chunks alternate between two compute streams, each with its own scratch (route
        # workspace, packed copy, reweight and reblock workspaces), so that one chunk's pool
        # and route run on the SMs that the other chunk's attention has finished with.
        comps = [comp, torch.cuda.Stream()]
        scratch = []
        for sidx in range(2):
            scratch.append({
                "route_ws": self.route_ws if sidx == 0 else torch.empty_like(self.route_ws),
                "rw_ws": (self.rw_ws if sidx == 0 or self.rw_ws is None else torch.empty_like(self.rw_ws)),
                "rb_ws": (getattr(self, "rb_ws", None) if sidx == 0 or not self.reblock
                          else torch.empty_like(self.rb_ws)),
                "pk": (torch.empty((3 * heads_per_chunk * per_head,), dtype=self.dtype, device=self.dev)
                       if self.packed is not None else None)})

        def use(sidx):
            for name in ("route_ws", "rw_ws", "rb_ws"):
                if scratch[sidx][name] is not None:
                    setattr(self, name, scratch[sidx][name])

        def step():
            from block_sparse_attention_tile_gb300 import bsa
            start = torch.cuda.Event()
            start.record(comp)
            h2d_s.wait_event(start)
            ready = []
            for h0, h1 in chunks:
                with torch.cuda.stream(h2d_s):
                    for d, h in ((dq, hq), (dk, hk), (dv, hv)):
                        d[h0:h1].copy_(h[h0:h1], non_blocking=True)
                    e = torch.cuda.Event()
                    e.record(h2d_s)
                ready.append(e)
            self.tile_map()
            mapped = torch.cuda.Event()
            mapped.record(comp)
            comps[1].wait_event(mapped)
            for c, ((h0, h1), e) in enumerate(zip(chunks, ready)):
                cs = comps[c % 2]
                cs.wait_event(e)
                use(c % 2)
                pk = scratch[c % 2]["pk"]
                # a contiguous [3, h1 - h0, J, M, D] view for this chunk's packed copy
                pkc = None if pk is None else pk[:3 * (h1 - h0) * per_head].view(3, h1 - h0, self.J, self.w["M"],
                                                                                   self.w["D"])
                with torch.cuda.stream(cs):
                    self.run_heads(dq, dk, dv, h0, h1, pkc)
                    done = torch.cuda.Event()
                    done.record(cs)
                d2h_s.wait_event(done)
                with torch.cuda.stream(d2h_s):
                    hout[h0:h1].copy_(self.out[h0:h1], non_blocking=True)
            use(0)
            fin = torch.cuda.Event()
            fin.record(d2h_s)
            comp.wait_event(fin)

        self.e2e_pipelining = ("head chunks of %s heads on two compute streams: copies in and out overlap the "
                               "compute of other heads" % "/".join(str(n) for n in sizes))
        return step, 1 + (self.launches_per_step - 1) * len(chunks)

    def algorithmic(self):
        """Valid (query, key) pairs the attention scores, x 4*D FLOPs."""
        torch = self.torch
        sizes = self.bs.long()
        routed = sizes[self.P:]
        sel = routed[self.q2k.long().clamp(min=0)] * (self.q2k >= 0)       # [BH, Jr, k]
        keys = sel.sum(-1)                                                   # [BH, Jr]
        prefix_keys = sizes[:self.P].sum()
        if self.summary:
            keys = keys + prefix_keys + (self.Jr - self.q2n.long())          # one virtual key per unselected block
        else:
            keys = keys + prefix_keys
        pairs = (routed[None, :] * keys).sum() + self.BH * sizes[:self.P].sum() * self.N
        flops = 4.0 * self.w["D"] * float(pairs.item())
        ntens = 3 if self.vbar is not None else 2
        pool_bytes = (ntens * self.BH * self.N * self.w["D"] * self.q.element_size()
                      + ntens * self.BH * self.J * self.w["D"] * 4
                      + (2 * self.BH * self.J * self.w["D"] * self.q.element_size() if self.summary else 0)
                      + (self.packed.numel() * self.packed.element_size() if self.packed is not None else 0)
                      + self.J * self.w["M"] * 4 + self.J * 4)
        return flops, pool_bytes

    def reweight_bytes(self):
        """Routed member rows of K and V read once, the float32 block means
        of Q read for the mean, k~ and v~ rows and the bias written."""
        D, el = self.w["D"], self.q.element_size()
        rows = float(self.bs[self.P:].long().sum().item())
        return (2 * self.BH * rows * D * el + self.BH * self.Jr * D * 4 + self.BH * self.Jr * (2 * D * el + 4)
                + self.J * self.w["M"] * 4)

    def report(self, stage_ms, peaks, peak_kind, props):
        flops, pool_bytes = self.algorithmic()
        D, J = self.w["D"], self.J
        attn_s = stage_ms["attention"] * 1e-3
        if self.w["dtype"] == "bf16":
            # the attention launch is timed on its own (milliseconds, not a seconds-long loop):
            # graded against the burst bf16 peak, with the nominal dense peak beside it
            peak = peaks["bf16_tflops"]
            roof = {"bound": "tensor", "achieved": flops / attn_s / 1e12, "peak": peak, "unit": "TFLOP/s",
                    "peak_kind": peak_kind + " bf16 burst",
                    "frac_nominal": flops / attn_s / 1e12 / NOMINAL_BF16_TFLOPS,
                    "nominal_peak": NOMINAL_BF16_TFLOPS}
        else:
            peak = fp32_peak(peaks, props)
            roof = {"bound": "alu", "achieved": flops / attn_s / 1e12, "peak": peak, "unit": "TFLOP/s",
                    "peak_kind": "FP32 lanes: SMs x 128 x 2 x max SM clock"}
        roof["frac"] = roof["achieved"] / roof["peak"]
        roof["traffic"] = read_traffic(self.name)
        roof["kernel"] = "bsa_fwd_summary attention" if self.summary else "bsa_fwd_qouter attention"
        roof["algorithmic_flops_per_launch"] = flops
        pool_gbs = pool_bytes / (stage_ms["pool"] * 1e-3) / 1e9
        rflops = 2.0 * self.BH * self.Jr * self.Jr * D
        route_tf = rflops / (stage_ms["route"] * 1e-3) / 1e12
        fp32 = fp32_peak(peaks, props)
        secondary = {
            "pool": {"bound": "hbm", "achieved": pool_gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": pool_gbs / peaks["hbm_gbs"], "bytes_per_launch": pool_bytes},
            "route": {"bound": "alu", "achieved": route_tf, "peak": fp32, "unit": "TFLOP/s", "frac": route_tf / fp32,
                      "flops_per_launch": rflops, "peak_note": "SMs x 128 FP32 lanes x 2 x max SM clock",
                      "note": "E = Q_bar K_bar^T on the tensor cores (three tf32 products of split float32 "
                              "operands), then the exact select on the CUDA cores; the FP32 figure is kept as the "
                              "stage's reference peak"}}
        if self.reblock:
            Nv = self.N - self.w.get("n_text", 0)
            el = self.q.element_size()
            # the stage is the tree levels' feature passes (three reads of the bf16 unit features a
            # level) plus one read of Q_v and K_v and one write of the features; the moment and
            # the features (2 * 2 * BH * Nv * D^2 FLOP) run on the tensor cores
            NB = -(-Nv // self.w["M"])
            levels = max(0, (NB - 1).bit_length())
            fbytes = self.BH * Nv * D * 2
            rbytes = levels * 3 * fbytes + 2 * self.BH * Nv * D * el + fbytes
            rgbs = rbytes / (stage_ms["reblock"] * 1e-3) / 1e9
            secondary["reblock"] = {"bound": "hbm", "achieved": rgbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                                    "frac": rgbs / peaks["hbm_gbs"], "bytes_per_launch": rbytes,
                                    "flops_per_launch": 2 * 2.0 * self.BH * Nv * D * D,
                                    "note": "%d tree levels, each reading the unit features three times; the "
                                            "levels are latency-bound (radix-select passes and cluster barriers)"
                                            % levels}
            pb = 3 * 2 * self.q.numel() * el
            secondary["permute"] = {"bound": "hbm", "achieved": pb / (stage_ms["permute"] * 1e-3) / 1e9,
                                    "peak": peaks["hbm_gbs"], "unit": "GB/s",
                                    "frac": pb / (stage_ms["permute"] * 1e-3) / 1e9 / peaks["hbm_gbs"],
                                    "bytes_per_launch": pb}
        if self.coarse:
            cflops = 2.0 * self.BH * self.Jr * self.Jr * D
            ctf = cflops / (stage_ms["coarse_attention"] * 1e-3) / 1e12
            secondary["coarse_attention"] = {"bound": "alu", "achieved": ctf, "peak": fp32, "unit": "TFLOP/s",
                                             "frac": ctf / fp32, "flops_per_launch": cflops}
            el = self.q.element_size()
            rows = float(self.bs[self.P:].long().sum().item())
            ab = 2 * self.BH * rows * D * el + self.BH * self.Jr * D * 4 + self.BH * D * 4 + self.J * self.w["M"] * 4
            agbs = ab / (stage_ms["coarse_apply"] * 1e-3) / 1e9
            secondary["coarse_apply"] = {"bound": "hbm", "achieved": agbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                                         "frac": agbs / peaks["hbm_gbs"], "bytes_per_launch": ab}
        if self.reweight:
            rb = self.reweight_bytes()
            rgbs = rb / (stage_ms["reweight"] * 1e-3) / 1e9
            secondary["reweight"] = {"bound": "hbm", "achieved": rgbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                                     "frac": rgbs / peaks["hbm_gbs"], "bytes_per_launch": rb}
        config = {"workload": self.name, "B": self.w["B"], "heads": self.w["heads"], "D": D, "seq_len": self.N}
        if self.segments is not None:
            config.update({"segments": [s if isinstance(s, int) else list(s) for s in self.segments],
                           "prefix_blocks": self.P, "video_spans": self.geom.spans, "budgets": self.w["budgets"],
                           "routing": "region-grouped TopK (exempt prefix)"})
        else:
            config["grid"] = list(self.w["grid"])
        config.update({"block": list(self.w["block"]), "M": self.w["M"], "J": J, "k": self.w["k"]})
        if self.summary:
            config.update({"n_text": self.w["n_text"], "permuted": True, "summary": True})
            if self.reweight:
                config["summaries"] = "spark-reweight"
            if self.reblock:
                config["permuted"] = "spark-reblock layout per head, built on the GPU every step"
        if self.coarse:
            config["coarse"] = "softmax(E) V_bar, per-head per-channel gate"
        nbytes = 3 * self.q.numel() * self.q.element_size()
        config["l2"] = ("inputs larger than L2: Q,K,V = %.2f GB per step" % (nbytes / 1e9) if nbytes > 129e6 else
                        "inputs smaller than L2 (%.1f MB): L2 not flushed, launch-bound tiny case" % (nbytes / 1e6))
        data = ("synthetic (seeded N(0,1) + per-head low-rank clusters; no dataset or weights)" if self.summary else
                "synthetic (seeded N(0,1) + a smooth space-time field per video segment on Q/K; no dataset or "
                "weights)" if self.segments is not None else
                "synthetic (seeded N(0,1)%s; no dataset or weights)"
                % (" + smooth space-time field on Q/K" if self.w["dtype"] == "bf16" else ""))
        return roof, secondary, config, data, self.w["dtype"]


class TokenWorkload:
    """GQA selected attention with supplied block lists, in the workload's
    order: query-outer (one launch) or KV-outer (reverse index -> partials ->
    combine); the other order is timed beside it."""

    def __init__(self, name, w, dev, rank):
        import numpy as np
        import torch
        from block_sparse_attention_tile_gb300 import bsa, synthetic
        self.name, self.w, self.dev, self.torch, self.np = name, w, dev, torch, np
        B, T, HQ, H, D, BS, S = (w[x] for x in ("B", "T", "HQ", "H", "D", "BS", "S"))
        seed = rank_seed(w["seed"], rank)
        self.q = synthetic.normal((B, T, HQ, D), seed, device=dev, dtype=torch.bfloat16)
        self.k = synthetic.normal((B, T, H, D), seed + 1, device=dev, dtype=torch.bfloat16)
        self.v = synthetic.normal((B, T, H, D), seed + 2, device=dev, dtype=torch.bfloat16)
        gen = synthetic.zipf_block_lists if w["zipf"] else synthetic.causal_block_lists
        self.idx_h, self.cnt_h = gen(B, T, H, S, BS, seed)
        self.idx = torch.as_tensor(self.idx_h, device=dev)
        self.cnt = torch.as_tensor(self.cnt_h, device=dev)
        from block_sparse_attention_tile_gb300 import pipeline
        self.nblk = -(-T // BS)
        self.cap = 2 * S * BS
        self.window = pipeline.default_window(T) if w.get("window") is None else w["window"]
        nwin = pipeline.windows(T, self.window)
        self.max_chunks = bsa.bsa_max_chunks(B, T, H, S, self.nblk, self.cap, self.window)
        self.row_ptr = torch.empty((B * nwin * H * self.nblk + 1,), dtype=torch.int32, device=dev)
        self.q_idx = torch.empty((B * H * T * S,), dtype=torch.int32, device=dev)
        self.slot = torch.empty_like(self.q_idx)
        self.chunks = torch.empty((self.max_chunks, 4), dtype=torch.int32, device=dev)
        self.n_chunks = torch.empty((1,), dtype=torch.int32, device=dev)
        self.ws = torch.empty((max(16, bsa.bsa_reverse_index_workspace(B, T, H, self.nblk)),), dtype=torch.uint8,
                              device=dev)
        self.obuf = torch.empty((B, T, HQ, S, D), dtype=torch.bfloat16, device=dev)
        self.lsebuf = torch.empty((B, T, HQ, S), dtype=torch.float32, device=dev)
        self.out = torch.empty_like(self.q)
        self.lse = torch.empty((B, T, HQ), dtype=torch.float32, device=dev)
        self.out_q = torch.empty_like(self.q)
        self.lse_q = torch.empty_like(self.lse)
        self.scale = D ** -0.5
        self.order = w.get("order", "kvouter")
        if self.order == "qouter":
            self.stage_names = ["attention"]
            self.launches_per_step = 1
        else:
            self.stage_names = ["reverse_index", "partials", "combine"]
            self.launches_per_step = 5

    def step(self, ev=None, q=None, k=None, v=None, idx=None, cnt=None):
        from block_sparse_attention_tile_gb300 import bsa
        w = self.w
        B, T, HQ, H, D, BS, S = (w[x] for x in ("B", "T", "HQ", "H", "D", "BS", "S"))
        q = self.q if q is None else q
        k = self.k if k is None else k
        v = self.v if v is None else v
        idx = self.idx if idx is None else idx
        cnt = self.cnt if cnt is None else cnt
        st = self.torch.cuda.current_stream()
        if self.order == "qouter":
            if ev: ev[0].record(st)
            bsa.bsa_fwd_qouter_tokens(q, k, v, B, T, HQ, H, D, idx, cnt, S, BS, True, self.scale, self.out, self.lse)
            if ev: ev[1].record(st)
            return
        self.kvouter(ev, q, k, v, idx, cnt)

    def kvouter(self, ev=None, q=None, k=None, v=None, idx=None, cnt=None):
        from block_sparse_attention_tile_gb300 import bsa
        w = self.w
        B, T, HQ, H, D, BS, S = (w[x] for x in ("B", "T", "HQ", "H", "D", "BS", "S"))
        q = self.q if q is None else q
        k = self.k if k is None else k
        v = self.v if v is None else v
        idx = self.idx if idx is None else idx
        cnt = self.cnt if cnt is None else cnt
        st = self.torch.cuda.current_stream()
        if ev: ev[0].record(st)
        bsa.bsa_build_reverse_index(idx, cnt, B, T, H, S, self.nblk, self.cap, self.row_ptr, self.q_idx, self.slot,
                                    self.chunks, self.n_chunks, self.max_chunks, self.ws, window=self.window)
        if ev: ev[1].record(st)
        bsa.bsa_fwd_kvouter(q, k, v, B, T, HQ, H, D, self.row_ptr, self.q_idx, self.slot, self.chunks,
                            self.n_chunks, self.max_chunks, self.nblk, BS, S, True, self.scale, self.obuf,
                            self.lsebuf, window=self.window)
        if ev: ev[2].record(st)
        bsa.bsa_combine(self.obuf, self.lsebuf, cnt, B, T, HQ, H, S, D, self.out, self.lse)
        if ev: ev[3].record(st)

    def qouter(self):
        from block_sparse_attention_tile_gb300 import bsa
        w = self.w
        bsa.bsa_fwd_qouter_tokens(self.q, self.k, self.v, w["B"], w["T"], w["HQ"], w["H"], w["D"], self.idx,
                                  self.cnt, w["S"], w["BS"], True, self.scale, self.out_q, self.lse_q)

    def host_inputs(self):
        return [self.q, self.k, self.v, self.idx, self.cnt], [self.out]

    def run_with(self, dev_inputs):
        self.step(None, *dev_inputs)

    def _kv_scratch(self, T, G, S, D):
        """KV-outer scratch for one (batch, KV head): reverse index, partials."""
        from block_sparse_attention_tile_gb300 import bsa, pipeline
        torch, dev = self.torch, self.dev
        nwin = pipeline.windows(T, self.window)
        mc = bsa.bsa_max_chunks(1, T, 1, S, self.nblk, self.cap, self.window)
        return {"max_chunks": mc,
                "row_ptr": torch.empty((nwin * self.nblk + 1,), dtype=torch.int32, device=dev),
                "q_idx": torch.empty((T * S,), dtype=torch.int32, device=dev),
                "slot": torch.empty((T * S,), dtype=torch.int32, device=dev),
                "chunks": torch.empty((mc, 4), dtype=torch.int32, device=dev),
                "n_chunks": torch.empty((1,), dtype=torch.int32, device=dev),
                "ws": torch.empty((max(16, bsa.bsa_reverse_index_workspace(1, T, 1, self.nblk)),), dtype=torch.uint8,
                                  device=dev),
                "obuf": torch.empty((1, T, G, S, D), dtype=torch.bfloat16, device=dev),
                "lsebuf": torch.empty((1, T, G, S), dtype=torch.float32, device=dev)}

    def make_e2e(self, h_in, d_in, h_out):
        """End-to-end step with host buffers, pipelined by (batch, KV head): the
        G query heads of one KV head and their selections are independent of the
        others' in both orders, so each such chunk runs through the same public
        calls with B = 1, HQ = G, H = 1.  K, V and the block lists (small) are
        copied in whole first; each chunk's Q comes in by a pitched copy while
        the chunk before it computes, and its output goes back by a pitched
        copy into the host [B, T, HQ, D] tensor as soon as it is done.  Every
        row's arithmetic is the same as in the whole-problem call (a row's scores,
        softmax and products do not depend on which rows share its tile), so
        the result is identical.  Falls back to copy-in / compute / copy-out when
        the runtime's pitched copy cannot be found."""
        torch = self.torch
        memcpy2d = cuda_memcpy2d()
        w = self.w
        B, T, HQ, H, D, BS, S = (w[x] for x in ("B", "T", "HQ", "H", "D", "BS", "S"))
        G = HQ // H
        hq, hk, hv, hidx, hcnt = h_in
        _, dk, dv, didx, dcnt = d_in
        (hout,) = h_out
        if memcpy2d is None or B * H < 2:
            def plain():
                for d, h in zip(d_in, h_in):
                    d.copy_(h, non_blocking=True)
                self.run_with(d_in)
                hout.copy_(self.out, non_blocking=True)
            return plain, self.launches_per_step
        dev = self.dev
        chunks = [(b, h) for b in range(B) for h in range(H)]
        qc = [torch.empty((1, T, G, D), dtype=torch.bfloat16, device=dev) for _ in chunks]
        oc = [torch.empty((1, T, G, D), dtype=torch.bfloat16, device=dev) for _ in chunks]
        lc = [torch.empty((1, T, G), dtype=torch.float32, device=dev) for _ in chunks]
        kc, vc, ic, cc = ([torch.empty(shape, dtype=dt, device=dev) for _ in range(2)]
                          for shape, dt in (((1, T, 1, D), torch.bfloat16), ((1, T, 1, D), torch.bfloat16),
                                            ((1, T, 1, S), torch.int32), ((1, T, 1), torch.int32)))
        scratch = [self._kv_scratch(T, G, S, D) for _ in range(2)] if self.order != "qouter" else None
        comp = torch.cuda.current_stream()
        comps = [comp, torch.cuda.Stream()]
        h2d_s, d2h_s = torch.cuda.Stream(), torch.cuda.Stream()
        row_b = G * D * 2                       # one position's G heads, bf16
        esz = hq.element_size()

        def check(rc):
            if rc != 0:
                raise RuntimeError("cudaMemcpy2DAsync failed (%d)" % rc)

        def step():
            from block_sparse_attention_tile_gb300 import bsa
            start = torch.cuda.Event()
            start.record(comp)
            h2d_s.wait_event(start)
            ready = []
            with torch.cuda.stream(h2d_s):
                for d, h in ((dk, hk), (dv, hv), (didx, hidx), (dcnt, hcnt)):
                    d.copy_(h, non_blocking=True)
                for c, (b, h) in enumerate(chunks):
                    src = hq.data_ptr() + ((b * T) * HQ + h * G) * D * esz
                    check(memcpy2d(qc[c].data_ptr(), row_b, src, HQ * D * esz, row_b, T, 1, h2d_s.cuda_stream))
                    e = torch.cuda.Event()
                    e.record(h2d_s)
                    ready.append(e)
            for c, (b, h) in enumerate(chunks):
                i = c % 2
                cs = comps[i]
                cs.wait_event(ready[c])
                with torch.cuda.stream(cs):
                    kc[i].copy_(dk[b:b + 1, :, h:h + 1])
                    vc[i].copy_(dv[b:b + 1, :, h:h + 1])
                    ic[i].copy_(didx[b:b + 1, :, h:h + 1])
                    cc[i].copy_(dcnt[b:b + 1, :, h:h + 1])
                    if self.order == "qouter":
                        bsa.bsa_fwd_qouter_tokens(qc[c], kc[i], vc[i], 1, T, G, 1, D, ic[i], cc[i], S, BS, True,
                                                  self.scale, oc[c], lc[c])
                    else:
                        sc = scratch[i]
                        bsa.bsa_build_reverse_index(ic[i], cc[i], 1, T, 1, S, self.nblk, self.cap, sc["row_ptr"],
                                                    sc["q_idx"], sc["slot"], sc["chunks"], sc["n_chunks"],
                                                    sc["max_chunks"], sc["ws"], window=self.window)
                        bsa.bsa_fwd_kvouter(qc[c], kc[i], vc[i], 1, T, G, 1, D, sc["row_ptr"], sc["q_idx"], sc["slot"],
                                            sc["chunks"], sc["n_chunks"], sc["max_chunks"], self.nblk, BS, S, True,
                                            self.scale, sc["obuf"], sc["lsebuf"], window=self.window)
                        bsa.bsa_combine(sc["obuf"], sc["lsebuf"], cc[i], 1, T, G, 1, S, D, oc[c], lc[c])
                    done = torch.cuda.Event()
                    done.record(cs)
                d2h_s.wait_event(done)
                dst = hout.data_ptr() + ((b * T) * HQ + h * G) * D * esz
                check(memcpy2d(dst, HQ * D * esz, oc[c].data_ptr(), row_b, row_b, T, 2, d2h_s.cuda_stream))
                # the next chunk on this stream reuses the small buffers only after
                # this chunk's kernels have read them (same stream: ordered)
            fin = torch.cuda.Event()
            fin.record(d2h_s)
            comp.wait_event(fin)
            comps[1].wait_event(fin)

        self.e2e_pipelining = ("(batch, KV head) chunks on two compute streams: each chunk's Q in and output out "
                               "by pitched copies that overlap the compute of other chunks; K, V and the block "
                               "lists copied in whole first")
        return step, self.launches_per_step * len(chunks)

    def algorithmic(self):
        """Visible (query head, key) pairs (causal) x 4*D FLOPs; nnz entries; bytes of the
        KV-outer partial pass under the page's I/O model (eq. 16): per entry the G query
        rows in, the G partial rows and LSEs out; per chunk one K/V block."""
        np = self.np
        w = self.w
        B, T, HQ, H, D, BS, S = (w[x] for x in ("B", "T", "HQ", "H", "D", "BS", "S"))
        G = HQ // H
        t = np.arange(T)[None, :, None, None]
        slot_ok = np.arange(S)[None, None, None, :] < self.cnt_h[..., None]
        first = self.idx_h.astype(np.int64) * BS
        vis = np.clip(np.minimum(t - first + 1, T - first), 0, BS) * slot_ok * (self.idx_h >= 0)
        pairs = float(vis.sum()) * G
        nnz = int(self.cnt_h.sum())
        nch = int(self.n_chunks.item())
        k1_bytes = nnz * G * (2 * D * 2 + 4) + nch * 2 * BS * D * 2
        return 4.0 * D * pairs, nnz, k1_bytes

    def _time(self, fn, reps=3):
        torch = self.torch
        for _ in range(2):
            fn()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record()
        for _ in range(reps):
            fn()
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / reps

    def report(self, stage_ms, peaks, peak_kind, props):
        torch = self.torch
        w = self.w
        B, T, HQ, H, D, BS, S = (w[x] for x in ("B", "T", "HQ", "H", "D", "BS", "S"))
        tensor_peak = peaks["bf16_tflops"]  # launches timed on their own: the burst peak
        # the other order on the same inputs (the KV-outer one per stage)
        if self.order == "qouter":
            ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
            for _ in range(2):
                self.kvouter()
            torch.cuda.synchronize()
            kv_stage = {n: 0.0 for n in ("reverse_index", "partials", "combine")}
            for _ in range(3):
                self.kvouter(ev)
                torch.cuda.synchronize()
                for j, n in enumerate(kv_stage):
                    kv_stage[n] += ev[j].elapsed_time(ev[j + 1]) / 3
            kv_ms = sum(kv_stage.values())
            other = {"kvouter_order": {"ms": kv_ms, "stages_us": {n: v * 1e3 for n, v in kv_stage.items()},
                                       "effective_tflops": metric_flops(w) / (kv_ms * 1e-3) / 1e12,
                                       "kernels": "bsa_build_reverse_index, bsa_fwd_kvouter, bsa_combine"}}
        else:
            kv_stage = stage_ms
            q_ms = self._time(self.qouter)
            other = {"qouter_order": {"ms": q_ms, "effective_tflops": metric_flops(w) / (q_ms * 1e-3) / 1e12,
                                      "kernel": "bsa_fwd_qouter_tokens"}}
        flops, nnz, k1_bytes = self.algorithmic()
        # K1 roofline: bytes of the page's I/O model (eq. 16) or FLOPs, whichever bounds it
        k1_s = kv_stage["partials"] * 1e-3
        if k1_bytes / (peaks["hbm_gbs"] * 1e9) >= flops / (tensor_peak * 1e12):
            ach = k1_bytes / k1_s / 1e9
            k1_roof = {"bound": "hbm", "achieved": ach, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                       "peak_kind": peak_kind + " HBM copy", "algorithmic_bytes_per_launch": k1_bytes}
        else:
            ach = flops / k1_s / 1e12
            k1_roof = {"bound": "tensor", "achieved": ach, "peak": tensor_peak, "unit": "TFLOP/s",
                       "peak_kind": peak_kind + " bf16 burst", "frac_nominal": ach / NOMINAL_BF16_TFLOPS,
                       "nominal_peak": NOMINAL_BF16_TFLOPS}
        k1_roof["frac"] = k1_roof["achieved"] / k1_roof["peak"]
        k1_roof["kernel"] = "bsa_fwd_kvouter partials (K1)"
        k1_roof["algorithmic_flops_per_launch"] = flops
        # combine: reads every written partial (bf16) + LSE, writes O (bf16) + LSE
        cb_bytes = nnz * (HQ // H) * (D * 2 + 4) + B * T * HQ * (D * 2 + 4) + B * T * H * 4
        cb_gbs = cb_bytes / (kv_stage["combine"] * 1e-3) / 1e9
        if self.order == "qouter":
            a_s = stage_ms["attention"] * 1e-3
            ach = flops / a_s / 1e12
            roof = {"bound": "tensor", "achieved": ach, "peak": tensor_peak, "unit": "TFLOP/s",
                    "peak_kind": peak_kind + " bf16 burst", "frac": ach / tensor_peak,
                    "frac_nominal": ach / NOMINAL_BF16_TFLOPS, "nominal_peak": NOMINAL_BF16_TFLOPS,
                    "kernel": "bsa_fwd_qouter_tokens (tensor-core, query-outer)",
                    "algorithmic_flops_per_launch": flops,
                    "note": "FLOPs of the visible (query head, key) pairs; the kernel also multiplies the rows "
                            "of positions that did not select a tile of the union (masked)"}
            secondary = {"kvouter_partials": k1_roof}
        else:
            roof = k1_roof
            secondary = {}
        roof["traffic"] = read_traffic(self.name)
        compulsory = (self.q.numel() + self.k.numel() + self.v.numel() + self.out.numel()) * 2 + \
            self.idx.numel() * 4 + self.cnt.numel() * 4
        step_ms = sum(stage_ms.values())
        ideal = max(flops / (tensor_peak * 1e12), compulsory / (peaks["hbm_gbs"] * 1e9))
        secondary.update({
            "combine": {"bound": "hbm", "achieved": cb_gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                        "frac": cb_gbs / peaks["hbm_gbs"], "bytes_per_launch": cb_bytes},
            "strict_step": {"ideal_ms": ideal * 1e3, "step_ms": step_ms, "frac": ideal * 1e3 / step_ms,
                            "note": "ideal = max(algorithmic FLOP / bf16 peak, compulsory Q,K,V,O,index bytes / "
                                    "HBM peak)"}})
        secondary.update(other)
        config = {"workload": self.name, "B": B, "T": T, "HQ": HQ, "H": H, "D": D, "block_size": BS, "S": S,
                  "selection": "zipf(1.1) sink+own" if w["zipf"] else "causal uniform, counts U{1..S}",
                  "order": "query-outer" if self.order == "qouter" else "kv-outer",
                  "chunk_cap": self.cap, "window": self.window, "nnz": nnz, "n_chunks": int(self.n_chunks.item()),
                  "l2": "inputs larger than L2: Q,K,V = %.2f GB per step"
                        % ((self.q.numel() + self.k.numel() + self.v.numel()) * 2 / 1e9)}
        return roof, secondary, config, "synthetic (seeded N(0,1); no dataset or weights)", "bf16"


def fp32_peak(peaks, props):
    return props.multi_processor_count * 128 * 2 * peaks.get("sm_max_mhz", 2070.0) * 1e6 / 1e12


# ---------------------------------------------------------------- GPU arm

def time_device(wl, steps, warmup, local, world):
    """Warm-up steps, then `steps` steps bracketed by a barrier and a synchronize
    on both sides, timed with CUDA events on the launching stream (whole region
    and per stage), with the SM clocks sampled meanwhile."""
    import torch
    import torch.distributed as dist

    from block_sparse_attention_tile_gb300 import bsa

    nst = len(wl.stage_names)
    for _ in range(warmup):
        wl.step()
    torch.cuda.synchronize()
    if bsa.bsa_device_status() != bsa.BSA_OK:
        raise RuntimeError("device status after warm-up: " + bsa.bsa_last_error())
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(nst + 1)] for _ in range(steps)]
    stream = torch.cuda.current_stream()
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for i in range(steps):
        wl.step(ev[i])
    t_end.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clk = clocks.stop()
    ms_total = t_start.elapsed_time(t_end)
    stage_ms = {sn: statistics.mean(e[j].elapsed_time(e[j + 1]) for e in ev) for j, sn in enumerate(wl.stage_names)}
    if bsa.bsa_device_status() != bsa.BSA_OK:
        raise RuntimeError("device status after timing: " + bsa.bsa_last_error())
    return ms_total, stage_ms, clk


def other_workloads(skip, dev, local, steps=5, warmup=3):
    """Every other workload of the table timed on the device after the headline
    (inputs resident, no end-to-end or CPU leg): per workload its step time,
    metric value, stage times, the dominant kernel's roofline and the clocks."""
    import torch

    peaks, peak_kind = read_peaks()
    props = torch.cuda.get_device_properties(dev)
    out = {}
    for name in sorted(WORKLOADS):
        if name == skip:
            continue
        w = dict(WORKLOADS[name])
        try:
            wl = (TokenWorkload if w["kind"] == "token" else BlockWorkload)(name, w, dev, 0)
            ms_total, stage_ms, clk = time_device(wl, steps, warmup, local, 1)
            roof, secondary, config, data, dtype = wl.report(stage_ms, peaks, peak_kind, props)
            ms_step = ms_total / steps
            entry = {"ms_per_step": round(ms_step, 4), "value": job_tflops(metric_flops(w), 1, ms_step),
                     "unit": "TFLOP/s", "steps": steps, "warmup": warmup, "dtype": dtype,
                     "stages_us": {sn: round(v * 1e3, 1) for sn, v in stage_ms.items()},
                     "roofline": {k: roof.get(k) for k in ("kernel", "bound", "achieved", "peak", "unit", "frac",
                                                           "frac_nominal") if k in roof},
                     "config": config, "clocks": clk}
            for key in ("kvouter_order", "qouter_order"):
                if key in roof:
                    entry[key] = {k: roof[key].get(k) for k in ("ms", "stages_us") if k in roof[key]}
            out[name] = entry
        except Exception as exc:  # noqa: BLE001
            out[name] = {"error": str(exc)[:300]}
        wl = None
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
    return out


def gpu_arm(args):
    import torch
    import torch.distributed as dist

    from block_sparse_attention_tile_gb300 import bsa

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    w = dict(WORKLOADS[args.workload])
    name = args.workload
    if args.window is not None and w["kind"] == "token":
        w["window"] = args.window
        name = name + "_window%d" % args.window
    if args.heads:
        if w["kind"] == "block":
            w["heads"] = args.heads
        else:  # KV heads, each with its G query heads
            w["HQ"] = w["HQ"] // w["H"] * args.heads
            w["H"] = args.heads
        name = name + "_%dheads" % args.heads
    wl = (TokenWorkload if w["kind"] == "token" else BlockWorkload)(name, w, dev, rank)
    ms_total, stage_ms, clk = time_device(wl, args.steps, args.warmup, local, world)
    stream = torch.cuda.current_stream()

    # end to end through the public API with host buffers: pinned inputs in,
    # the result out, every step
    ins, outs = wl.host_inputs()
    h_in = [x.cpu().pin_memory() for x in ins]
    d_in = [torch.empty_like(x) for x in ins]
    h_out = [torch.empty(x.shape, dtype=x.dtype).pin_memory() for x in outs]
    h2d = sum(x.numel() * x.element_size() for x in ins)
    d2h = sum(x.numel() * x.element_size() for x in outs)

    def e2e_plain():
        for d, h in zip(d_in, h_in):
            d.copy_(h, non_blocking=True)
        wl.run_with(d_in)
        for h, d in zip(h_out, outs):
            h.copy_(d, non_blocking=True)

    if hasattr(wl, "make_e2e"):
        e2e_step, e2e_launches = wl.make_e2e(h_in, d_in, h_out)
    else:
        e2e_step, e2e_launches = e2e_plain, wl.launches_per_step
    ref_out = [x.clone() for x in outs]  # the device-only run's result, for the check below

    for _ in range(max(1, args.warmup)):
        e2e_step()
    # Each step timed on its own; the median is reported.  Plain pinned copies of the
    # same sizes, with no kernel of ours, stall now and then for 25-100 ms on these
    # hosts, so one stalled step would otherwise dominate a short mean; the mean and
    # the slowest step are reported beside it.
    e2e_steps = max(3, min(args.steps, 7))
    torch.cuda.synchronize()
    e2e_times = []
    for _ in range(e2e_steps):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        e2e_step()
        e1.record(stream)
        e1.synchronize()
        e2e_times.append(e0.elapsed_time(e1))
    e2e_ms = statistics.median(e2e_times)
    e2e_mean, e2e_max = statistics.mean(e2e_times), max(e2e_times)
    # the pipelined end-to-end path must return exactly what the device-only run computed
    e2e_match = all(torch.equal(h.to(dev), r) for h, r in zip(h_out, ref_out))
    del ref_out
    if not e2e_match:
        raise RuntimeError("end-to-end output differs from the device-only run")

    # max over ranks
    ms_total, e2e_ms = max_over_ranks([ms_total, e2e_ms], world, dev)
    ms_step = ms_total / args.steps

    if rank == 0:
        peaks, peak_kind = read_peaks()
        props = torch.cuda.get_device_properties(dev)
        roof, secondary, config, data, dtype = wl.report(stage_ms, peaks, peak_kind, props)
        flops = metric_flops(w)
        config.update({"global_batch": w["B"] * world,
                       "parallelism": "replicas%d" % world if world > 1 else "single"})
        line = {
            "metric": METRIC,
            "value": job_tflops(flops, world, ms_step),
            "unit": "TFLOP/s",
            "n_gpus": world,
            "steps": args.steps,
            "warmup": args.warmup,
            "ms_per_step": ms_step,
            "higher_is_better": True,
            "scaling": "weak" if world > 1 else "none",
            "vs_baseline": None,
            "dtype": dtype,
            "data": data,
            "config": config,
            "stages_us": {sn: round(v * 1e3, 1) for sn, v in stage_ms.items()},
            "roofline": roof,
            "rooflines_secondary": secondary,
            "e2e": {"value": job_tflops(flops, world, e2e_ms), "unit": "TFLOP/s",
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                    "steps_timed": e2e_steps, "aggregate": "median of per-step times",
                    "ms_per_step_mean": e2e_mean, "ms_per_step_max": e2e_max,
                    "pipelining": getattr(wl, "e2e_pipelining", "none: copy in, compute, copy out"),
                    "gpu_launches_per_step": e2e_launches, "matches_device_run": e2e_match},
            "gpu_launches": wl.launches_per_step * args.steps,
            "clocks": clk,
        }
        if not args.no_cpu_baseline and world == 1:
            try:
                line["cpu_baseline"] = run_oracle_sample(args.workload, args.cpu_budget)
            except Exception as exc:  # noqa: BLE001
                line["cpu_baseline"] = {"value": None, "error": str(exc)[:300]}
        if world == 1 and not args.headline_only and args.workload == DEFAULT and not args.heads:
            # the other workloads, device-timed in the same run, after the headline's
            # buffers are released
            wl = None
            h_in = d_in = h_out = ins = outs = None
            e2e_step = None
            torch.cuda.synchronize()
            torch.cuda.empty_cache()
            line["other_workloads"] = other_workloads(args.workload, dev, local)
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def reference_arm(args):
    """The oracle on the host cores (there is no other implementation of the
    pages to run): every step attends the same number of query units on all
    cores through the sampler's process pool, so value and ms_per_step are the
    sampled work over its own wall time; the full-step extrapolation rides
    along."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    w = WORKLOADS[args.workload]
    cores = os.cpu_count() or 1
    per_step = cores  # pool tasks per step, each of the sampler's units_per_task units
    r = _run_sampler({"workload": args.workload, "cores": cores, "steps": args.warmup + args.steps,
                      "units_per_step": per_step})
    setups, unit_name = _sample_scale(w)
    walls = r["step_walls_s"][args.warmup:]
    units = r["step_units"][args.warmup:]
    flops_per_unit = metric_flops(w) / (setups * r["units_total"])
    step_s = statistics.mean(walls)
    value = flops_per_unit * statistics.mean(units) / step_s / 1e12
    full_s = setups * r["setup_s"] / cores + setups * r["units_total"] * step_s / statistics.mean(units)
    if w["kind"] == "token":
        cfg = {"workload": args.workload, "B": w["B"], "T": w["T"], "HQ": w["HQ"], "H": w["H"], "D": w["D"],
               "block_size": w["BS"], "S": w["S"]}
    else:
        cfg = {"workload": args.workload, "heads": w["heads"], "D": w["D"], "k": w["k"]}
        if "grid" in w:
            T, H, W = w["grid"]
            cfg["seq_len"] = T * H * W + w.get("n_text", 0)
    sample = ("each step: %d %s attended on %d spawned single-thread workers (the oracle as it stands); "
              "a full step (%d setups x %d units) extrapolates to %.1f s"
              % (per_step * r["units_per_task"], unit_name, cores, setups, r["units_total"], full_s))
    line = {"impl": "reference", "metric": METRIC,
            "value": value, "unit": "TFLOP/s", "n_gpus": int(os.environ.get("WORLD_SIZE", "1")),
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_s * 1e3,
            "higher_is_better": True, "scaling": "none", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": cfg,
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "sample": sample,
                             "full_step_s_extrapolated": full_s},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default=DEFAULT)
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--headline-only", action="store_true",
                    help="skip the device-timed pass over the other workloads that the default run adds")
    ap.add_argument("--heads", type=int, default=0,
                    help="fewer heads (KV heads for the token workloads) than the workload's: a small case "
                         "for profiler captures")
    ap.add_argument("--window", type=int, default=None,
                    help="token workloads: query positions per KV-outer window (0 = one window; default: "
                         "the library pipeline's choice)")
    ap.add_argument("--oracle-sample", default=None, help=argparse.SUPPRESS)
    args = ap.parse_args()
    if args.oracle_sample is not None:  # the spawned CPU sampler (see _oracle_sample_main)
        _oracle_sample_main(json.loads(args.oracle_sample))
        return
    if args.warmup < 3 and args.impl == "ours":
        print("warning: fewer than 3 warm-up steps", file=sys.stderr)
    if args.impl == "reference":
        reference_arm(args)
    else:
        gpu_arm(args)


if __name__ == "__main__":
    main()
