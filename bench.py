#!/usr/bin/env python
"""Paged decode-attention benchmark on one GB300 (replicas for N > 1).

Workload: the continuous-batching rollout with Qwen3-4B head shapes — 64
slots, 32 q / 8 kv heads, head_dim 128, page 64, max_seq 1024, prompts
U[100, 400], 512 decode steps, each sequence stopping at a seeded length and
its slot and pages reused at once (fragmented placement). A step is one
layer's decode step: q/k RMSNorm + RoPE, the K/V append, split-KV attention
and combine — by default the fused paged_decode_step kernel plus the combine
(--chain: three separate kernels). --workload picks one of the static decode
layers instead (qwen3 B=8, llama B=16, gemma sliding D=256 / full D=512).

The rollout schedule always has its 512 steps. --steps K times K steps drawn
evenly across it (step floor((i + 1/2) * 512 / K) for i < K: every step once
at K = 512), so a short run samples the whole schedule, not its opening. The
whole schedule is also timed once per run (config.schedule), with the
attention split by quarter (admission-heavy opening vs long-row end).

value      algorithmic KV-read bytes of the attention (K+V of every key,
           q in, out, table entries) / device time of the whole step, GB/s;
           inputs resident in HBM, 4+ layer caches cycled so every step's
           keys come from DRAM (working set > 4x L2).
roofline   the same bytes / the attention kernels' own time, vs the measured
           HBM copy bandwidth; config.hot_l2 repeats it on one layer cache.
e2e        the same metric through the public Python API with pinned host
           inputs copied in and the output read back every step.
cpu_baseline / --impl reference: the float64 CPU oracle on a bounded sample
           (a process pool over (row, kv head) on the host cores, and one
           thread); config.pt_us times the host allocator calls.
"""
from __future__ import annotations

import os

for _v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")

import argparse  # noqa: E402
import hashlib  # noqa: E402
import json  # noqa: E402
import math  # noqa: E402
import statistics  # noqa: E402
import subprocess  # noqa: E402
import sys  # noqa: E402
import time  # noqa: E402

import numpy as np  # noqa: E402
import torch  # noqa: E402

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as wl  # noqa: E402

METRIC = "paged decode-attn KV-read GB/s (% of GB300 HBM peak); µs per decode step"
UNIT = "GB/s"
WORKLOAD_DESC = ("512-step rollout, continuous batching: B=64 slots, Qwen3-4B heads 32/8, D=128, "
                 "page 64, max_seq 1024, prompts U[100,400]")


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=512)
    ap.add_argument("--warmup", type=int, default=16)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--e2e-steps", type=int, default=400)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--num-splits", type=int, default=0)
    ap.add_argument("--no-clocks", action="store_true")
    ap.add_argument("--chain", action="store_true",
                    help="layer step as three kernels (qk_norm_rope, kv_append, attention) "
                         "instead of the fused paged_decode_step")
    ap.add_argument("--layers", type=int, default=0,
                    help="layer caches to cycle (0: enough for 4x L2)")
    ap.add_argument("--workload", default="rollout",
                    choices=sorted(list(WORKLOAD_CHOICES) + ["prefill", "prefill-long",
                                                             "prefill-gemma-sliding",
                                                             "prefill-gemma-full"]),
                    help="rollout (the headline line) or one of the static decode layers")
    return ap.parse_args()


# ----------------------------------------------------------------- helpers --
def attn_bytes(seq_lens: np.ndarray, B, Hq, Hkv, D, ps, window: int = 0) -> int:
    """Algorithmic bytes of one paged_decode_attn call: K and V of every key
    the row attends to read once, q read, out written, one table entry per
    page touched."""
    L = seq_lens.astype(np.int64)
    n = np.minimum(L, window) if window > 0 else L
    lo = L - n
    pages = np.where(n > 0, (L + ps - 1) // ps - lo // ps, 0)
    return int(Hkv * n.sum() * D * 2 * 2 + B * Hq * D * 2 * 2 + pages.sum() * 4)


def schedule_sample(S: int, K: int, offset: float = 0.5) -> np.ndarray:
    """K step indices spread evenly over a schedule of S steps: step
    floor((i + offset) * S / K) for i < K. At K = S (offset in [0, 1)) every
    step appears once; K < S takes the middle step of each of K equal stretches;
    K > S repeats every step K/S times, to within one."""
    i = np.arange(K, dtype=np.float64)
    return np.minimum(np.floor((i + offset) * S / K), S - 1).astype(np.int64)


# name -> (workload, layer index, description)
WORKLOAD_CHOICES = {
    "rollout": ("rollout", 0, None),
    "qwen3": ("qwen3", 0, "Qwen3-4B-shaped decode layer: B=8, 32/8 heads, D=128, page 64, "
                          "L0 ~ U[64,1024], one token appended per step, q/k norm, theta 1e6"),
    "llama": ("llama", 0, "Llama-3.2-3B-shaped decode layer: B=16, 24/8 heads, D=128, page 64, "
                          "L ~ U[512,1024], theta 5e5, no q/k norm"),
    "gemma-sliding": ("gemma", 0, "Gemma-4-E2B sliding layer: B=64, 8/1 heads, D=256, window 512, "
                                  "page 64, L ~ U[256,2048], theta 1e4, q/k norm, v norm"),
    "gemma-full": ("gemma", 1, "Gemma-4-E2B full layer: B=64, 8/1 heads, D=512, page 64, "
                               "L ~ U[256,2048], theta 1e6 proportional RoPE on 128 dims, "
                               "q/k norm, v norm, K=V"),
}


def static_metadata(w, total_steps):
    """Per-step tables and row metadata for a fixed batch whose rows each
    append one token per step (host-only PageTable)."""
    import paged_kv_decode_pagetable_gb300 as pkv
    pt = pkv.PageTable(w.max_batch_size, w.page_size, w.n_pages, w.max_pages_per_seq)
    L0 = wl.static_lengths(w)
    slots = [pt.assign(int(L) + 1) for L in L0]
    tables, bidx, pos, lens = [], [], [], []
    for t in range(total_steps):
        p = (L0 + t).astype(np.int32)
        for s_, L in zip(slots, p):
            pt.reserve(s_, int(L) + 1)
        tables.append(pt.host_table().numpy())
        bidx.append(np.array(slots, np.int32))
        pos.append(p)
        lens.append(p + 1)
    return (np.stack(tables), np.stack(bidx), np.stack(pos), np.stack(lens))


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f), "measured"
    except OSError:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0}, "fallback"


def hold_stream():
    """Keeps the current stream busy for some tens of microseconds (torch's
    spin kernel), issued before a start event: the graph replay that follows
    is then already queued when the event fires, so the timed region holds
    the steps' device time and not the host's submission of the graph (which
    a replay of K steps would otherwise carry once, 10 us or so)."""
    torch.cuda._sleep(100000)


def profile_traffic(kernel_key: str, mean_alg_bytes: float | None = None):
    """DRAM bytes per launch from a committed ncu capture, or None when the
    kernel source changed since the capture. A record with a measured /
    algorithmic ratio is scaled to this run's mean launch (decode: the bytes
    vary from step to step); one with bytes per launch is a capture of the
    same fixed workload."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f).get(kernel_key)
    except (OSError, ValueError):
        return None
    if not rec:
        return None
    src = os.path.join(ROOT, "paged_kv_decode_pagetable_gb300", "csrc",
                       rec.get("source_file", "decode_attn.cu"))
    with open(src, "rb") as f:
        digest = hashlib.sha256(f.read()).hexdigest()[:16]
    if rec.get("source_sha256_16") != digest:
        return None
    if "dram_over_algorithmic" in rec and mean_alg_bytes is not None:
        return float(rec["dram_over_algorithmic"]) * mean_alg_bytes
    return float(rec["dram_bytes_per_launch"]) if "dram_bytes_per_launch" in rec else None


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, enabled: bool, index: int):
        self.proc = None
        if not enabled:
            return
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "20", "-i", str(index)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.05)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, mx, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in out.splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


def rollout_metadata(w, total_steps):
    """Runs the schedule through a host-only PageTable; per-step tables and
    row metadata (what the device would hold after each step's pt_* calls)."""
    import paged_kv_decode_pagetable_gb300 as pkv
    from paged_kv_decode_pagetable_gb300 import engine
    sched = wl.rollout_schedule(w, steps=total_steps)
    pt = pkv.PageTable(w.max_batch_size, w.page_size, w.n_pages, w.max_pages_per_seq)
    drv = engine.RolloutDriver(pt, sched)
    tables, bidx, pos, lens = [], [], [], []
    for _ in range(total_steps):
        m = drv.next_step()
        tables.append(pt.host_table().numpy())
        bidx.append(m.batch_idx)
        pos.append(m.input_pos)
        lens.append(m.seq_lens)
    return (np.stack(tables), np.stack(bidx), np.stack(pos), np.stack(lens))


def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend)
    return world, rank, local


def reduce_max(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    dev = torch.device("cuda", torch.cuda.current_device()) if torch.cuda.is_available() else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def reduce_sum(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    dev = torch.device("cuda", torch.cuda.current_device()) if torch.cuda.is_available() else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ------------------------------------------------------------ CPU oracle ----
class PagePool:
    """Random float32 pages (all kv heads) that sampled rows point into."""

    def __init__(self, w, rng, D=128, pages=64):
        self.pages = pages
        self.kc = rng.standard_normal((w.n_kv_heads, pages * w.page_size, D)).astype(np.float32)
        self.vc = rng.standard_normal((w.n_kv_heads, pages * w.page_size, D)).astype(np.float32)


def oracle_sample(w, lens_rows, rng, seconds, pool, D=128, window=0, min_rows=1):
    """Times the oracle's attention for rows with the given lengths (cycled),
    their pages drawn from `pool`, until `seconds` of CPU time have been spent
    inside the oracle; returns (bytes, seconds, rows)."""
    import oracle
    Hq, Hkv, ps = w.n_q_heads, w.n_kv_heads, w.page_size
    pool_pages, kc, vc = pool.pages, pool.kc, pool.vc
    total_bytes, elapsed, rows = 0, 0.0, 0
    i = 0
    while (elapsed < seconds or rows < min_rows) and rows < 10 ** 7:
        L = int(lens_rows[i % len(lens_rows)])
        i += 1
        nb = -(-L // ps)
        table = np.zeros((2, nb), np.int32)
        table[1] = rng.integers(0, pool_pages, size=nb)
        q = rng.standard_normal((1, Hq, D))
        t0 = time.perf_counter()
        oracle.decode_attention(q, kc, vc, table, [1], [L], window, D ** -0.5, ps)
        elapsed += time.perf_counter() - t0
        total_bytes += attn_bytes(np.array([L]), 1, Hq, Hkv, D, ps, window)
        rows += 1
    return total_bytes, elapsed, rows


# A process pool over (row, kv head): each task is the oracle's attention for
# one kv head of one row (its G query heads), on pages of a per-worker pool.
_POOL = {}


def _pool_init(seed, Hq, Hkv, ps, D, pages, window):
    rng = np.random.default_rng(seed)
    _POOL.update(
        kc=rng.standard_normal((Hkv, pages * ps, D)).astype(np.float32),
        vc=rng.standard_normal((Hkv, pages * ps, D)).astype(np.float32),
        rng=rng, G=Hq // Hkv, ps=ps, D=D, pages=pages, window=window)


def _pool_task(task):
    import oracle
    L, g = task
    P = _POOL
    rng, ps, D, G = P["rng"], P["ps"], P["D"], P["G"]
    nb = -(-L // ps)
    table = np.zeros((2, nb), np.int32)
    table[1] = rng.integers(0, P["pages"], size=nb)
    q = rng.standard_normal((1, G, D))
    oracle.decode_attention(q, P["kc"][g:g + 1], P["vc"][g:g + 1], table, [1], [L],
                            P["window"], D ** -0.5, ps)
    return L


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def oracle_pool_sample(w, lens_rows, seconds, rows_per_s, D=128, window=0):
    """The oracle on every host core: a spawn-started process pool over (row,
    kv head) tasks for rows with the given lengths (cycled), sized from the
    single-thread rate so that the pool works about `seconds` of wall time;
    pool start-up is not timed. Returns (bytes, seconds, rows, processes)."""
    import multiprocessing as mp
    n = host_cores()
    Hq, Hkv, ps = w.n_q_heads, w.n_kv_heads, w.page_size
    rows = max(n, int(rows_per_s * n * seconds))
    lens = [int(lens_rows[i % len(lens_rows)]) for i in range(rows)]
    tasks = [(L, g) for L in lens for g in range(Hkv)]
    ctx = mp.get_context("spawn")
    with ctx.Pool(n, initializer=_pool_init,
                  initargs=(w.seed(11), Hq, Hkv, ps, D, 64, window)) as pool:
        pool.map(_pool_task, [(int(lens_rows[0]), 0)] * (2 * n), chunksize=1)   # warm
        t0 = time.perf_counter()
        for _ in pool.imap_unordered(_pool_task, tasks, chunksize=max(1, Hkv // 2)):
            pass
        sec = time.perf_counter() - t0
    byts = sum(attn_bytes(np.array([L]), 1, Hq, Hkv, D, ps, window) for L in lens)
    return byts, sec, rows, n


def cpu_baselines(w, lens_rows, seconds, D=128, window=0, seed_salt=7):
    """Single-thread and all-core oracle legs on rows with the given lengths;
    the all-core leg is the reported cpu_baseline, the single-thread one rides
    along in it."""
    rng = np.random.default_rng(w.seed(seed_salt))
    b1, s1, n1 = oracle_sample(w, lens_rows, rng, seconds, PagePool(w, rng, D), D, window)
    one = b1 / s1 / 1e9
    bn, sn, nn, procs = oracle_pool_sample(w, lens_rows, seconds, n1 / s1, D, window)
    return {"value": bn / sn / 1e9, "unit": UNIT, "cores": procs, "kind": "oracle",
            "sample": f"{nn} rows with the lengths of the timed steps' rows (cycled), "
                      f"float64 NumPy, a spawn process pool of {procs} over (row, kv head), "
                      f"{sn:.1f} s wall",
            "single_thread": {"value": one, "cores": 1,
                              "sample": f"{n1} rows, one thread, {s1:.1f} s"}}


def rollout_lengths(w) -> np.ndarray:
    """seq_lens [S][B] of the rollout schedule's S steps, from the schedule
    alone (no allocator needed for lengths)."""
    sched = wl.rollout_schedule(w)
    length = [r.prompt_len for r in sched.first]
    out = []
    for t in range(sched.steps):
        for lane, r in sched.start[t]:
            length[lane] = r.prompt_len
        out.append(np.array(length) + 1)
        length = [L + 1 for L in length]
    return np.stack(out)


def run_reference(args, world, rank):
    """The CPU oracle as the reference arm: each step a bounded sample of the
    step's rows (two rows), on the same steps of the 512-step schedule that
    our arm times; warm-up steps untimed."""
    if rank != 0:
        return
    w = wl.ROLLOUT
    lens_all = rollout_lengths(w)
    S = len(lens_all)
    warm = schedule_sample(S, max(args.warmup, 1), 0.0)[:args.warmup]
    timed = schedule_sample(S, args.steps)
    rng = np.random.default_rng(w.seed(99))
    pool = PagePool(w, rng)
    tot_bytes, tot_s, rows = 0, 0.0, 0
    for j, t in enumerate(list(warm) + list(timed)):
        lens = lens_all[t]
        sample = lens[[(2 * t) % w.batch, (2 * t + 1) % w.batch]]
        b, s, n = oracle_sample(w, sample, rng, 0.0, pool, min_rows=2)
        if j >= len(warm):
            tot_bytes, tot_s, rows = tot_bytes + b, tot_s + s, rows + n
    value = tot_bytes / tot_s / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": tot_s / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD_DESC, "global_batch": w.batch,
                   "schedule_steps": S,
                   "timed_schedule_steps": f"{args.steps} steps spread evenly over the {S}",
                   "sample": "2 rows per step (of 64), oracle on host cores",
                   "parallelism": "replicas"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": f"{rows} rows over {args.steps} steps (2 rows/step), "
                                   "float64 NumPy, single thread"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- GPU arm ---
def pt_timing(w):
    """Host allocator cost over the rollout schedule: every pt_assign,
    pt_reserve and pt_free the schedule issues, timed one by one through the
    Python binding (ctypes call included), with the device mirror of the table
    on (row writes queued with cudaMemcpyAsync on the current stream) and off
    (host state only). µs per call: median and mean."""
    import paged_kv_decode_pagetable_gb300 as pkv
    from paged_kv_decode_pagetable_gb300 import engine

    class Timed:
        def __init__(self, pt):
            self.pt, self.t = pt, {"assign": [], "reserve": [], "free": []}

        def _run(self, name, *a):
            t0 = time.perf_counter_ns()
            r = getattr(self.pt, name)(*a)
            self.t[name].append(time.perf_counter_ns() - t0)
            return r

        def assign(self, L):
            return self._run("assign", L)

        def reserve(self, s, L):
            return self._run("reserve", s, L)

        def free(self, s):
            return self._run("free", s)

    out = {}
    for mode, device in (("device_mirror", torch.cuda.current_device()), ("host_only", None)):
        pt = pkv.PageTable(w.max_batch_size, w.page_size, w.n_pages, w.max_pages_per_seq,
                           device=device)
        tp = Timed(pt)
        drv = engine.RolloutDriver(tp, wl.rollout_schedule(w))
        for _ in range(w.steps):
            drv.next_step()
        torch.cuda.synchronize()
        out[mode] = {name: {"calls": len(v), "median_us": float(np.median(v)) / 1e3,
                            "mean_us": float(np.mean(v)) / 1e3}
                     for name, v in tp.t.items() if v}
    out["note"] = ("through the ctypes binding; device_mirror includes queueing the table-row "
                   "copy (cudaMemcpyAsync from pageable host memory)")
    return out


def run_ours(args, world, rank, local):
    import paged_kv_decode_pagetable_gb300 as pkv
    from paged_kv_decode_pagetable_gb300 import engine

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (the product path has no CPU fallback)")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pkv.load_library()
    wname, li, desc = WORKLOAD_CHOICES[args.workload]
    w = wl.WORKLOADS[wname]
    lay = w.layers[li]
    spec = engine.LayerSpec(lay.head_dim, lay.theta, lay.window, lay.qk_norm, True,
                            lay.rotary_dims, lay.v_norm, lay.k_eq_v)
    B, Hq, Hkv, D, ps = w.batch, w.n_q_heads, w.n_kv_heads, spec.head_dim, w.page_size
    W, K = args.warmup, args.steps
    rollout = wname == "rollout"
    if rollout:
        # the schedule always has its configured steps; warm-up and timed steps
        # are drawn evenly across it
        S = w.steps
        tables, bidx, pos, lens = rollout_metadata(w, S)
        warm_idx = schedule_sample(S, max(W, 1), 0.0)[:W]
        timed_idx = schedule_sample(S, K)
    else:
        # a fixed batch appends one token per step until the table rows are
        # full, then the same steps repeat (re-appending the same positions)
        S = min(W + K, w.max_seq - int(wl.static_lengths(w).max()))
        tables, bidx, pos, lens = static_metadata(w, S)
        warm_idx = np.arange(W) % S
        timed_idx = (W + np.arange(K)) % S
    step_bytes = np.array([attn_bytes(lens[t], B, Hq, Hkv, D, ps, spec.window)
                           for t in range(S)])
    d_tables = torch.from_numpy(tables).to(dev)
    d_bidx = torch.from_numpy(bidx).to(dev)
    d_pos = torch.from_numpy(pos).to(dev)
    d_lens = torch.from_numpy(lens).to(dev)

    props = torch.cuda.get_device_properties(dev)
    l2 = getattr(props, "L2_cache_size", 126 * 2 ** 20) or 126 * 2 ** 20
    kv_step = float(np.mean(step_bytes[timed_idx]))
    n_layers = args.layers or max(2, math.ceil(4 * l2 / kv_step))
    caches = [engine.alloc_cache(Hkv, w.n_pages, ps, D, dev, fill="randn") for _ in range(n_layers)]

    g = torch.Generator(device=dev)
    g.manual_seed(w.seed(rank))
    q = torch.randn((B, Hq, D), generator=g, device=dev).to(torch.bfloat16)
    k = torch.randn((B, Hkv, D), generator=g, device=dev).to(torch.bfloat16)
    v = torch.randn((B, Hkv, D), generator=g, device=dev).to(torch.bfloat16)
    gq = (1 + 0.1 * torch.randn(D, generator=g, device=dev)).to(torch.bfloat16)
    gk = (1 + 0.1 * torch.randn(D, generator=g, device=dev)).to(torch.bfloat16)
    out = torch.empty((B, Hq, D), dtype=torch.bfloat16, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    ws = engine.AttnWorkspace(B, Hq, Hkv, D, w.max_pages_per_seq, ps, spec.window, dev,
                              args.num_splits)

    class Geom:
        n_slots, max_pages_per_seq, page_size, n_pages = (w.n_slots, w.max_pages_per_seq, ps,
                                                          w.n_pages)
        dev_table = None

    # step j of a sequence runs schedule step t on layer cache j mod n_layers,
    # so consecutive calls read different caches
    def step(j, t):
        kc, vc = caches[j % n_layers]
        engine.decode_layer_step(spec, Geom, kc, vc, q, k, v, d_bidx[t], d_pos[t], d_lens[t], out,
                                 ws, gq, gk, w.eps, err=err, table=d_tables[t],
                                 fused=not args.chain)

    def attn_only(j, t):
        kc, vc = caches[j % n_layers]
        pkv.paged_decode_attn(q, kc, vc, d_tables[t], w.n_slots, w.max_pages_per_seq, ps,
                              w.n_pages, d_bidx[t], d_lens[t], spec.window, D ** -0.5, ws.splits,
                              ws.buf, out, err)

    def capture(fn, idx, layer=None):
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr):
            for j, t in enumerate(idx):
                fn(j if layer is None else layer, int(t))
        return gr

    stream = torch.cuda.current_stream()

    def time_graph(gr):
        gr.replay()                       # the first launch of a graph uploads it
        torch.cuda.synchronize()
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        hold_stream()
        a0.record(stream)
        gr.replay()
        a1.record(stream)
        torch.cuda.synchronize()
        return a0.elapsed_time(a1)

    # warm-up: W eager steps (first use of every kernel), then capture
    for j, t in enumerate(warm_idx):
        step(j, int(t))
    torch.cuda.synchronize()
    graph = capture(step, timed_idx)
    graph_attn = capture(attn_only, timed_idx)
    torch.cuda.synchronize()
    graph.replay()
    torch.cuda.synchronize()

    sampler = ClockSampler(not args.no_clocks, local)
    barrier(world)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    hold_stream()
    e0.record(stream)
    graph.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clocks = sampler.stop()
    t_step_ms = e0.elapsed_time(e1)
    del graph

    # attention kernels alone over the same steps
    t_attn_ms = time_graph(graph_attn)
    del graph_attn
    timed_bytes = float(step_bytes[timed_idx].sum())
    peaks, peak_kind = measured_peaks()
    peak = float(peaks.get("hbm_gbs", 6800.0))

    # hot L2: the same attention calls, all on one layer cache
    t_hot_ms = time_graph(capture(attn_only, timed_idx, layer=0))
    hot = {"attn_us_per_call": t_hot_ms / K * 1e3,
           "gbs": timed_bytes / (t_hot_ms * 1e-3) / 1e9,
           "frac": timed_bytes / (t_hot_ms * 1e-3) / 1e9 / peak,
           "note": "same steps, one layer cache: consecutive calls re-read mostly the same pages"}

    schedule = None
    if rollout:
        # the whole schedule once, and its attention by quarter
        all_idx = np.arange(S)
        t_full_ms = time_graph(capture(step, all_idx))
        t_full_attn_ms = time_graph(capture(attn_only, all_idx))
        full_bytes = float(step_bytes.sum())
        phases = []
        for qd in range(4):
            idx = all_idx[qd * S // 4:(qd + 1) * S // 4]
            ms = time_graph(capture(attn_only, idx))
            byts = float(step_bytes[idx].sum())
            phases.append({"steps": f"{int(idx[0])}-{int(idx[-1])}",
                           "mean_seq_len": float(lens[idx].mean()),
                           "mean_kv_mb": byts / len(idx) / 1e6,
                           "attn_us_per_call": ms / len(idx) * 1e3,
                           "frac": byts / (ms * 1e-3) / 1e9 / peak})
        sched = wl.rollout_schedule(w)
        schedule = {"steps": S, "us_per_step": t_full_ms / S * 1e3,
                    "attn_us_per_call": t_full_attn_ms / S * 1e3,
                    "attn_gbs": full_bytes / (t_full_attn_ms * 1e-3) / 1e9,
                    "attn_frac": full_bytes / (t_full_attn_ms * 1e-3) / 1e9 / peak,
                    "step_gbs": full_bytes / (t_full_ms * 1e-3) / 1e9,
                    "mean_kv_mb": full_bytes / S / 1e6,
                    "seq_len": f"{int(lens.min())}-{int(lens.max())}",
                    "slot_reuses": int(sum(len(f) for f in sched.finish)),
                    "timed_steps_with_reuse": int(sum(1 for t in timed_idx if sched.finish[t])),
                    "attn_by_quarter": phases}
    errv = pkv.pkv_read_error_word(err)
    if errv != 0:
        raise SystemExit(f"device error word {errv}")

    t_max = reduce_max(t_step_ms, world)
    value = reduce_sum(timed_bytes, world) / (t_max * 1e-3) / 1e9
    attn_gbs = timed_bytes / (t_attn_ms * 1e-3) / 1e9
    # the combine kernel runs only with a fixed split count; the automatic mode
    # merges cut rows inside the attention kernel
    combine = bool(ws.splits) and ws.max_parts > 1
    launches_per_step = (3 if args.chain else 1) + (1 if combine else 0)

    # ---- end to end through the public API: pinned host in, output back ----
    n_e2e = min(args.e2e_steps, K)
    e2e_idx = schedule_sample(S, n_e2e) if rollout else timed_idx[:n_e2e]
    e2e = run_e2e(args, w, spec, engine, pkv, caches, n_layers, tables, bidx, pos, lens,
                  step_bytes, gq, gk, ws, dev, world, warm_idx, e2e_idx)

    # ---- CPU oracle baselines on a bounded sample (rank 0, N=1 only) ----
    cpu, pt_us = None, None
    if rank == 0 and world == 1:
        rows = np.concatenate([lens[t] for t in timed_idx])
        cpu = cpu_baselines(w, rows, args.cpu_seconds, D, spec.window)
        if rollout:
            pt_us = pt_timing(w)

    if rank == 0:
        tl = lens[timed_idx]
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K,
            "warmup": W, "ms_per_step": t_max / K, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": desc or WORKLOAD_DESC, "global_batch": B * world,
                       "seq_len": f"{int(tl.min())}-{int(tl.max())}",
                       "timed_steps": (f"{K} steps spread evenly over the {S}-step schedule"
                                       if rollout else f"steps {W}.. of a fixed batch"),
                       "mean_kv_mb_per_step": timed_bytes / K / 1e6,
                       "num_splits": ws.splits or "auto (length-balanced parts)",
                       "max_parts_per_row": ws.max_parts, "layer_caches_cycled": n_layers,
                       "l2_policy": f"inputs larger than L2: {n_layers} layer caches of "
                                    f"{caches[0][0].numel() * 4 / 2**20:.0f} MiB cycled; "
                                    f"{kv_step / 2**20:.0f} MiB of K/V read per step",
                       "us_per_step": t_max / K * 1e3, "attn_us_per_call": t_attn_ms / K * 1e3,
                       "layer_step": ("qk_norm_rope + kv_append + paged_decode_attn"
                                      if args.chain else "paged_decode_step (fused)"),
                       "schedule": schedule, "hot_l2": hot, "pt_us": pt_us,
                       "parallelism": f"replicas x{world}"},
            "roofline": {"bound": "hbm", "achieved": attn_gbs, "peak": peak, "unit": "GB/s",
                         "frac": attn_gbs / peak, "peak_kind": peak_kind,
                         "kernel": f"decode_attn_kernel<{D}, false>"
                                   + (f" + combine_kernel<{D}>" if combine else ""),
                         "traffic": profile_traffic(f"{args.workload}_decode_attn_{D}",
                                                    timed_bytes / K)},
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": K * launches_per_step,
            "clocks": clocks,
        }
        print(json.dumps(line), flush=True)


def run_e2e(args, w, spec, engine, pkv, caches, n_layers, tables, bidx, pos, lens, step_bytes,
            gq, gk, ws, dev, world, warm_idx, idx):
    """The metric through the public API with host buffers: every step copies
    its q, k, v, page table and row metadata from pinned host memory to the
    device, runs the layer step, and copies the output back to pinned host
    memory. A step's inputs sit in one pinned staging buffer laid out as the
    device input buffer (q | k | v | table | metadata), so they travel in one
    copy. As in the pages' engine (capture_decode_cudagraph / replay), the
    steps are replayed from a CUDA graph captured over the API calls; the
    same steps issued eagerly from Python are reported as eager_value."""
    B, Hq, Hkv, D = w.batch, w.n_q_heads, w.n_kv_heads, spec.head_dim
    n = len(idx)
    ring = 8
    gen = torch.Generator().manual_seed(w.seed(3))
    nq, nkv = B * Hq * D * 2, B * Hkv * D * 2
    ntab, nmeta = tables[0].nbytes, 3 * B * 4
    offs = np.cumsum([0, nq, nkv, nkv, ntab, nmeta])      # 16-byte multiples at these shapes
    qkv = [torch.randn(B * (Hq + 2 * Hkv) * D, generator=gen).to(torch.bfloat16)
           for _ in range(ring)]
    seq = [int(t) for t in list(warm_idx[:8]) + list(idx)]
    h_in = []
    for j, t in enumerate(seq):
        buf = torch.empty(int(offs[-1]), dtype=torch.uint8).pin_memory()
        buf[offs[0]:offs[3]].view(torch.bfloat16).copy_(qkv[j % ring])
        buf[offs[3]:offs[4]].view(torch.int32).copy_(torch.from_numpy(tables[t]).reshape(-1))
        buf[offs[4]:offs[5]].view(torch.int32).copy_(
            torch.from_numpy(np.stack([bidx[t], pos[t], lens[t]])).reshape(-1))
        h_in.append(buf)
    h_out = [torch.empty((B, Hq, D), dtype=torch.bfloat16).pin_memory() for _ in range(ring)]
    d_in = torch.empty(int(offs[-1]), dtype=torch.uint8, device=dev)
    q = d_in[offs[0]:offs[1]].view(torch.bfloat16).view(B, Hq, D)
    k = d_in[offs[1]:offs[2]].view(torch.bfloat16).view(B, Hkv, D)
    v = d_in[offs[2]:offs[3]].view(torch.bfloat16).view(B, Hkv, D)
    d_table = d_in[offs[3]:offs[4]].view(torch.int32).view(tables.shape[1:])
    d_meta = d_in[offs[4]:offs[5]].view(torch.int32).view(3, B)
    out = torch.empty((B, Hq, D), dtype=torch.bfloat16, device=dev)

    class Geom:
        n_slots, max_pages_per_seq, page_size, n_pages = (w.n_slots, w.max_pages_per_seq,
                                                          w.page_size, w.n_pages)
        dev_table = None

    def one(j):
        d_in.copy_(h_in[j], non_blocking=True)
        kc, vc = caches[j % n_layers]
        engine.decode_layer_step(spec, Geom, kc, vc, q, k, v, d_meta[0], d_meta[1], d_meta[2],
                                 out, ws, gq, gk, w.eps, table=d_table, fused=not args.chain)
        h_out[j % ring].copy_(out, non_blocking=True)

    n_warm = len(seq) - n
    for j in range(n_warm):
        one(j)
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()

    def timed(fn):
        barrier(world)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        fn()
        e1.record(stream)
        torch.cuda.synchronize()
        return reduce_max(e0.elapsed_time(e1), world)

    ms_eager = timed(lambda: [one(j) for j in range(n_warm, n_warm + n)])
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for j in range(n_warm, n_warm + n):
            one(j)
    g.replay()
    torch.cuda.synchronize()
    ms = timed(g.replay)
    byts = reduce_sum(float(step_bytes[np.asarray(idx)].sum()), world)
    h2d = int(offs[-1])
    return {"value": byts / (ms * 1e-3) / 1e9, "unit": UNIT, "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(B * Hq * D * 2), "steps": n, "ms_per_step": ms / n,
            "mode": "CUDA graph of the API calls, host copies inside every step "
                    "(one copy in, one copy out)",
            "eager_value": byts / (ms_eager * 1e-3) / 1e9, "eager_ms_per_step": ms_eager / n}


def prefill_docs(long: bool = False, n_docs: int = 64, seed_salt: int = 31):
    """Packed prefill: n_docs prompts with the rollout's admission lengths
    U[100, 400] (long: 8 documents of 2048 tokens), laid one after another
    (document id per token)."""
    if long:
        lens = np.full(8, 2048, dtype=np.int64)
        return np.repeat(np.arange(8), lens).astype(np.int32), lens
    rng = np.random.default_rng(wl.ROLLOUT.seed(seed_salt))
    lens = wl.uniform_lengths(rng, n_docs, 100, 400)
    return np.repeat(np.arange(n_docs), lens).astype(np.int32), lens


def prefill_flops(lens, Hq: int, D: int, window: int = 0) -> float:
    """QK^T and PV over the kept (causal, same-document, within the window)
    pairs: 4 D Hq per pair. A document of n tokens keeps n(n+1)/2 pairs, or
    with a window W < n: W(W+1)/2 + (n - W) W."""
    lens = np.asarray(lens, dtype=np.float64)
    full = lens * (lens + 1) / 2
    if window > 0:
        W = float(window)
        full = np.where(lens > W, W * (W + 1) / 2 + (lens - W) * W, full)
    return float(4.0 * D * Hq * np.sum(full))


# prefill workloads: name -> (q heads, kv heads, head_dim, window, long documents)
PREFILL_CHOICES = {
    "prefill": (32, 8, 128, 0, False),
    "prefill-long": (32, 8, 128, 0, True),
    "prefill-gemma-sliding": (8, 1, 256, 512, False),
    "prefill-gemma-full": (8, 1, 512, 0, False),
}


def run_prefill(args, world, rank, local):
    """Document-causal prefill attention (prefill_attn) on 64 packed prompts
    (or 8 documents of 2048 tokens), with Qwen3-4B heads (32 q / 8 kv,
    head_dim 128) or the Gemma-4 E2B layers (8 q / 1 kv; sliding: head_dim 256,
    window 512; full: head_dim 512); tensor-core bound. A step is one layer's
    attention call; the block mask (prefill_block_mask) depends only on the
    documents and the window, is built once per batch for all layers, and is
    timed on its own."""
    import paged_kv_decode_pagetable_gb300 as pkv
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (the product path has no CPU fallback)")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pkv.load_library()
    Hq, Hkv, D, window, long = PREFILL_CHOICES[args.workload]
    docs, lens = prefill_docs(long)
    L = len(docs)
    g = torch.Generator(device=dev)
    g.manual_seed(wl.ROLLOUT.seed(rank + 40))
    sets = [(torch.randn((Hq, L, D), generator=g, device=dev).to(torch.bfloat16),
             torch.randn((Hkv, L, D), generator=g, device=dev).to(torch.bfloat16),
             torch.randn((Hkv, L, D), generator=g, device=dev).to(torch.bfloat16))
            for _ in range(2)]
    d_docs = torch.from_numpy(docs).to(dev)
    out = torch.empty((Hq, L, D), dtype=torch.bfloat16, device=dev)
    scale = D ** -0.5
    W, K = args.warmup, min(args.steps, 200)

    bm = pkv.prefill_block_mask(d_docs, window)

    def call(t):
        q, k, v = sets[t % 2]
        pkv.prefill_attn(q, k, v, bm, scale, out)

    for t in range(W):
        call(t)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for t in range(K):
            call(t)
    graph.replay()
    torch.cuda.synchronize()
    sampler = ClockSampler(not args.no_clocks, local)
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    stream = torch.cuda.current_stream()
    hold_stream()
    e0.record(stream)
    graph.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clocks = sampler.stop()
    own_ms = e0.elapsed_time(e1)
    ms = reduce_max(own_ms, world)
    # the block mask build, timed alone (graph of K builds)
    mgraph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(mgraph):
        for _ in range(K):
            pkv.prefill_block_mask(d_docs, window)
    mgraph.replay()
    torch.cuda.synchronize()
    hold_stream()
    e0.record(stream)
    mgraph.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    mask_us = e0.elapsed_time(e1) * 1e3 / K
    flops = prefill_flops(lens, Hq, D, window)
    n_blocks = int(bm.kv_num_blocks.sum().item() + bm.full_kv_num_blocks.sum().item())
    value = reduce_sum(flops * K, world) / (ms * 1e-3) / 1e12
    peaks, peak_kind = measured_peaks()
    peak = float(peaks.get("bf16_tflops", 1900.0))
    achieved = flops * K / (own_ms * 1e-3) / 1e12
    cpu = None
    if rank == 0 and world == 1:
        import oracle
        n = 1 if long else 3                       # a bounded sample: the first documents
        end = int(np.sum(lens[:n]))
        qs = sets[0][0][:, :end].float().cpu().numpy()
        ks = sets[0][1][:, :end].float().cpu().numpy()
        vs = sets[0][2][:, :end].float().cpu().numpy()
        t0 = time.perf_counter()
        oracle.prefill_attention(qs, ks, vs, docs[:end], scale, window=window)
        sec = time.perf_counter() - t0
        cpu = {"value": prefill_flops(lens[:n], Hq, D, window) / sec / 1e12, "unit": "TFLOP/s",
               "cores": 1, "kind": "oracle",
               "sample": f"the first {n} documents ({end} tokens), float64 NumPy, {sec:.1f} s"}
    if rank == 0:
        print(json.dumps({
            "metric": "document-causal prefill attention TFLOP/s", "value": value,
            "unit": "TFLOP/s", "n_gpus": world, "steps": K, "warmup": W, "ms_per_step": ms / K,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": (f"packed prefill: 8 documents of 2048 tokens ({L} tokens), "
                                    if long else
                                    f"packed prefill: 64 prompts U[100,400] ({L} tokens), ")
                                   + f"{Hq} q / {Hkv} kv heads, head_dim {D}"
                                   + (f", window {window}" if window else ""),
                       "global_batch": len(lens) * world, "tokens": L, "flops_per_call": flops,
                       "visited_blocks_per_head": n_blocks,
                       "block_flops_per_call": 4.0 * 64 * 64 * D * Hq * n_blocks,
                       "block_mask_us": mask_us, "attn_us_per_call": ms * 1e3 / K,
                       "l2_policy": "two input sets of ~200 MB (larger than L2) alternated",
                       "parallelism": f"replicas x{world}"},
            "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak,
                         "unit": "TFLOP/s", "frac": achieved / peak, "peak_kind": peak_kind,
                         "kernel": (f"prefill_tc_kernel<{D}>" if D <= 128
                                    else f"prefill_wide_kernel<{D}>") + " (tcgen05)",
                         "traffic": profile_traffic(f"{args.workload}_prefill_{D}")},
            "cpu_baseline": cpu, "gpu_launches": K, "clocks": clocks}), flush=True)


def main():
    args = parse_args()
    world, rank, local = dist_setup(args)
    try:
        if args.impl == "reference":
            run_reference(args, world, rank)
        elif args.workload in PREFILL_CHOICES:
            run_prefill(args, world, rank, local)
        else:
            run_ours(args, world, rank, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            if dist.is_initialized():
                dist.destroy_process_group()


if __name__ == "__main__":
    main()
