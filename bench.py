#!/usr/bin/env python
"""Throughput of one KV-cache compression event on GB300.

A step is one full compression event of the Qwen3-8B-shaped stack (16
sequences x 36 layers x 8 KV heads, head_dim 128, bf16, 32768 cached rows per
slice -> budget 4096, prompt 512 and recent 128 protected, 17 geometric
offsets): tri_score, tri_select_topk, tri_compact_kv on inputs resident in
HBM. Metric: KV tokens (cached rows of every slice before the event) scored +
selected + compacted per second.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gpu|reference]

--impl reference times the oracle (the plain fp64 CPU restatement under
oracle/) on the host cores instead, on a bounded sample of the same workload.
Under torchrun each rank runs its own batch on its own GPU (weak scaling, no
collective on the data path); rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "KV tokens scored+selected+compacted per second"
UNIT = "KV tokens/s"
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 7900.0


# ---------------------------------------------------------------------------
# multi-process plumbing (also exercised by the gloo tests on CPU)
# ---------------------------------------------------------------------------
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def init_dist(backend: str):
    import torch.distributed as dist

    ws, rank, _ = dist_env()
    if ws > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend, rank=rank, world_size=ws)
    return ws, rank


def barrier():
    import torch.distributed as dist

    if dist.is_available() and dist.is_initialized():
        dist.barrier()


def max_over_ranks(x: float, device=None) -> float:
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()):
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate(per_rank_units: int, world: int, max_seconds: float, steps: int) -> dict:
    """Whole-job throughput: units processed by all ranks / slowest rank's time."""
    total = per_rank_units * world * steps
    return {"value": total / max_seconds, "ms_per_step": 1e3 * max_seconds / steps}


# ---------------------------------------------------------------------------
# clocks sampled during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str, period_ms: int = 100):
        self.gpu = gpu_id
        self.period = period_ms
        self.proc = None
        self.lines = []
        self.marks = {}

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 f"-lms={self.period}"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (FileNotFoundError, OSError):
            self.proc = None
            return
        self.th = threading.Thread(target=self._read, daemon=True)
        self.th.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self, name):
        self.marks[name] = time.time()

    def stop(self):
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()

    def summary(self, t0_mark="t0", t1_mark="t1") -> dict:
        if not self.lines:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        t0, t1 = self.marks.get(t0_mark, 0), self.marks.get(t1_mark, 1e30)
        rows = [l for (t, l) in self.lines if t0 <= t <= t1 + 0.15]
        if len(rows) < 3:  # short timed region: fall back to every sample under load
            rows = [l for (_, l) in self.lines]
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            parts = [p.strip() for p in r.split(",")]
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
        sm.sort()
        med = sm[len(sm) // 2] if sm else None
        return {"sm_mhz": med, "sm_max_mhz": max(smax) if smax else None, "reasons": sorted(reasons),
                "samples": len(sm)}


def nvsmi_gpu_id(torch_index: int) -> str:
    """nvidia-smi id of a torch device: its UUID (indices may be remapped)."""
    import torch

    try:
        u = str(torch.cuda.get_device_properties(torch_index).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
        ids = [x for x in vis.split(",") if x.strip()]
        return ids[torch_index] if torch_index < len(ids) else str(torch_index)


def host_mem_available() -> int:
    try:
        with open("/proc/meminfo") as f:
            for line in f:
                if line.startswith("MemAvailable:"):
                    return int(line.split()[1]) * 1024
    except OSError:
        pass
    return 32 << 30


def measured_peak_gbs():
    try:
        with open(PEAKS_FILE) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


# ---------------------------------------------------------------------------
# the oracle on a bounded sample (CPU baseline and the reference arm)
# ---------------------------------------------------------------------------
def oracle_sample_inputs(w, n_slices: int, seed: int = 0):
    """Slices drawn like the workload (same recipe, CPU generator), with
    centres calibrated by the oracle from n_cal queries per query head."""
    import numpy as np
    import torch

    import oracle as orc
    from kv_cache_compression_tri_gb300 import synth

    sw = synth.scaled(w, n_seq=1, n_layers=1, n_kv_heads=n_slices, n_cal=min(w.n_cal, 1024))
    inp = synth.make_inputs(sw, "cpu", with_queries=not w.random)
    k = inp.k.view(n_slices, w.n_cap, w.head_dim)
    v = inp.v.view(n_slices, w.n_cap, w.head_dim)
    cen = None
    if not w.random:
        cen = orc.calibrate(inp.q.to(torch.float64).numpy(), sw.group)
    items = []
    for s in range(n_slices):
        items.append({
            "k64": k[s].to(torch.float64).numpy(),
            "kbytes": k[s].contiguous().view(torch.uint8).numpy().reshape(w.n_cap, -1).copy(),
            "vbytes": v[s].contiguous().view(torch.uint8).numpy().reshape(w.n_cap, -1).copy(),
            "centre": None if cen is None else (cen[0][s], cen[1][s], cen[2][s]),
            "p_cur": w.n_valid - 1, "slot": s,
        })
    return items


def oracle_time(w, items, threads: int):
    """Run oracle score + select + compact (or random select + compact) on the
    items with a thread pool (ctypes releases the GIL); returns seconds."""
    import concurrent.futures as cf

    import numpy as np

    import oracle as orc

    n, P, W, B = w.n_valid, w.n_prompt, w.n_recent, w.budget

    def one(it):
        if w.random:
            keep = orc.rand_select(0, 0, 0, 0, it["slot"], n, P, W, B)
        else:
            c, m, R = it["centre"]
            sc = np.full(n, -np.inf)
            sc[P:n - W] = orc.score_series(it["k64"][P:n - W], c, m, R, w.offsets, it["p_cur"], w.theta,
                                           pos=np.arange(P, n - W))
            keep = orc.select(sc, n, P, W, B)
        kb, vb = it["kbytes"].copy(), it["vbytes"].copy()
        orc.compact(kb, keep)
        orc.compact(vb, keep)
        return int(keep[-1])

    t0 = time.perf_counter()
    with cf.ThreadPoolExecutor(max_workers=threads) as ex:
        list(ex.map(one, items))
    return time.perf_counter() - t0


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


# ---------------------------------------------------------------------------
# reference arm: the oracle as the reference implementation
# ---------------------------------------------------------------------------
def run_reference(args, w):
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    import oracle

    oracle.build()
    cores = host_cores()
    n_sample = max(1, min(args.ref_slices, w.n_slices))
    items = oracle_sample_inputs(w, n_sample)
    for _ in range(args.warmup):
        oracle_time(w, items[: max(1, min(len(items), cores))], cores)
    times = [oracle_time(w, items, cores) for _ in range(args.steps)]
    sec = sum(times) / len(times)
    tokens = n_sample * w.n_valid
    value = tokens / sec
    sample = (f"{n_sample} slices of {w.name} per step ({w.n_valid} rows each, fp64 oracle: series score, "
              f"stable-sort select, byte-loop compaction of K and V)")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * sec, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(w, args.path),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def workload_config(w, path: str = "separate") -> dict:
    return {
        "workload": w.name, "n_seq": w.n_seq, "n_layers": w.n_layers, "n_kv_heads": w.n_kv_heads,
        "head_dim": w.head_dim, "n_cap": w.n_cap, "n_valid": w.n_valid, "budget": w.budget,
        "n_prompt": w.n_prompt, "n_recent": w.n_recent, "offsets": len(w.offsets),
        "rope_theta": w.theta, "storage": "bf16" if w.elem_bytes == 2 else "f32",
        "keys": "post-RoPE" if w.key_layout == "post" else "pre-RoPE",
        "path": (("rand_evict_compact" if path in ("separate", "paged") else "rand_evict + tri_compact_kv")
                 if w.random else
                 ("tri_compress (score, select, compact in one call)" if path == "compress" else
                  ("tri_score_heads + tri_select_topk_zmax + tri_compact_kv (GQA z-score + max, group %d)"
                   % w.group if path == "gqa" else
                   ("tri_score (every row) + tri_select_union + tri_compact_kv" if path == "union" else
                    ("tri_score + tri_select_topk + tri_compact_kv on a paged pool (16-row blocks)"
                     if path == "paged" else "tri_score + tri_select_topk + tri_compact_kv"))))),
        "parallelism": "one cache batch per GPU (weak scaling)",
    }


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------
def run_gpu(args, w):
    import numpy as np
    import torch

    ws, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    init_dist("nccl")

    from kv_cache_compression_tri_gb300 import _build

    if rank == 0 or not os.path.exists(_build.LIB):
        _build.build()
    barrier()
    import kv_cache_compression_tri_gb300 as tri
    from kv_cache_compression_tri_gb300 import synth

    tri.load_library()
    S, n, P, W, B = w.n_slices, w.n_valid, w.n_prompt, w.n_recent, w.budget
    d, e = w.head_dim, w.elem_bytes
    inp = synth.make_inputs(w, dev)
    centers = None
    gqa = (args.path == "gqa") and not w.random
    if not w.random:
        # the GQA path keeps one centre per query head
        centers = tri.calibrate_centers(inp.q, 1 if gqa else w.group)
        inp.q = None
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    # first B rows of every slice are all compaction can change: keep a copy
    k_head = inp.k[:, :, :, :B].clone()
    v_head = inp.v[:, :, :, :B].clone()
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    n_valid = torch.full((S,), n, dtype=torch.int32, device=dev)
    pos_out = torch.empty(S, w.n_cap, dtype=torch.int32, device=dev)
    union = args.path == "union" and not w.random
    paged = args.path == "paged"
    if paged:
        # the same rows in a block pool: 16-row blocks, one shuffled table per sequence
        L_, H_, d_, bs = w.n_layers, w.n_kv_heads, w.head_dim, 16
        mb = w.n_cap // bs
        perm = torch.randperm(w.n_seq * mb, generator=torch.Generator().manual_seed(1)).view(w.n_seq, mb)
        kp = torch.empty(w.n_seq * mb, L_, H_, bs, d_, dtype=w.dtype, device=dev)
        vp = torch.empty_like(kp)
        for sq in range(w.n_seq):
            idx = perm[sq].to(dev)
            kp[idx] = inp.k[sq].reshape(L_, H_, mb, bs, d_).permute(2, 0, 1, 3, 4)
            vp[idx] = inp.v[sq].reshape(L_, H_, mb, bs, d_).permute(2, 0, 1, 3, 4)
        del k_head, v_head
        inp.k = inp.v = None
        torch.cuda.empty_cache()
        table = perm.to(torch.int32).to(dev)
        head_blocks = table[:, : (B + bs - 1) // bs].reshape(-1).long()
        k_head, v_head = kp[head_blocks].clone(), vp[head_blocks].clone()
        kv = tri.PagedKVCache(kp, vp, table, n_valid, None, pos_out, status, post_rope=(w.key_layout == "post"))
    else:
        kv = tri.KVCache(inp.k, inp.v, n_valid, None, pos_out, status, post_rope=(w.key_layout == "post"))
    if union:
        k_head_pick = B - P - W
        uws = torch.empty(tri.select_union_workspace_bytes(kv, P, W, k_head_pick), dtype=torch.uint8, device=dev)
    fused = (args.path == "compress") and not w.random
    # Random Attention: rand_evict_compact (selection and compaction in one kernel,
    # faster there); scored paths: three kernels (the fused one is not faster for them)
    fused_sc = w.random and args.path in ("separate", "paged")
    scores = None if (fused or gqa) else torch.empty(S, w.n_cap, dtype=torch.float32, device=dev)
    if gqa:
        G = w.group
        scores_g = torch.empty(S, G, w.n_cap, dtype=torch.float32, device=dev)
        stats = torch.empty(S, G, 2, dtype=torch.float32, device=dev)
        hws = torch.empty(tri.score_heads_workspace_bytes(kv, G), dtype=torch.uint8, device=dev)
    keep = torch.empty(S, B, dtype=torch.int32, device=dev)
    cws = torch.empty(tri.compress_workspace_bytes(kv), dtype=torch.uint8, device=dev) if fused else None
    stream = torch.cuda.current_stream()

    def restore():
        if paged:
            kp[head_blocks] = k_head
            vp[head_blocks] = v_head
        else:
            inp.k[:, :, :, :B].copy_(k_head)
            inp.v[:, :, :, :B].copy_(v_head)
        n_valid.fill_(n)

    ev = lambda: torch.cuda.Event(enable_timing=True)

    def step(rec=None):
        if fused:
            # one entry point (tri_compress): its three kernels in one call
            if rec: rec[0].record(stream)
            tri.compress(kv, centers, w.theta, w.offsets, inp.p_cur, P, W, B, keep, workspace=cws)
            if rec:
                rec[1].record(stream)
                rec[2].record(stream)
                rec[3].record(stream)
            return
        if fused_sc:
            # Random Attention: the draw, selection and compaction in one kernel per slice
            if rec:
                rec[0].record(stream)
                rec[1].record(stream)
            tri.rand_evict_compact(kv, 0, 0, P, W, B, keep)
            if rec:
                rec[2].record(stream)
                rec[3].record(stream)
            return
        if w.random:
            if rec: rec[0].record(stream)
            tri.rand_evict(kv, 0, 0, P, W, B, keep)
            if rec: rec[1].record(stream)
        elif gqa:
            if rec: rec[0].record(stream)
            tri.score_heads(kv, centers, G, w.theta, w.offsets, inp.p_cur, scores_g, stats, workspace=hws)
            if rec: rec[1].record(stream)
            tri.select_topk_zmax(scores_g, stats, G, kv, P, W, B, keep)
        elif union:
            if rec: rec[0].record(stream)
            tri.score(kv, centers, w.theta, w.offsets, inp.p_cur, scores)  # statistics need every row
            if rec: rec[1].record(stream)
            tri.select_union(scores, kv, P, W, B, k_head_pick, keep, workspace=uws)
        else:
            if rec: rec[0].record(stream)
            tri.score(kv, centers, w.theta, w.offsets, inp.p_cur, scores, n_prompt=P, n_recent=W)
            if rec: rec[1].record(stream)
            tri.select_topk(scores, kv, P, W, B, keep)
        if rec: rec[2].record(stream)
        tri.compact_kv(kv, keep, B)
        if rec: rec[3].record(stream)

    for _ in range(args.warmup):
        step()
        torch.cuda.synchronize()
        restore()
    torch.cuda.synchronize()
    assert int(status.item()) == 0, f"device status {int(status.item())}"
    # moved rows per event (identical every step: same inputs)
    keep_h = keep.cpu().numpy()
    moved = int((keep_h != np.arange(B)[None, :]).sum())
    restore()

    clocks = ClockSampler(nvsmi_gpu_id(local))
    clocks.start()
    time.sleep(0.3)
    recs = [[ev() for _ in range(4)] for _ in range(args.steps)]
    l0 = tri.launch_count()
    torch.cuda.synchronize()
    barrier()
    torch.cuda.synchronize()
    clocks.mark("t0")
    w0 = time.perf_counter()
    for i in range(args.steps):
        step(recs[i])
        restore()
    torch.cuda.synchronize()
    barrier()
    torch.cuda.synchronize()
    w1 = time.perf_counter()
    clocks.mark("t1")
    launches = tri.launch_count() - l0
    time.sleep(0.3)
    clocks.stop()
    assert int(status.item()) == 0, f"device status {int(status.item())}"

    step_ms = [recs[i][0].elapsed_time(recs[i][3]) for i in range(args.steps)]
    k1_ms = [recs[i][0].elapsed_time(recs[i][1]) for i in range(args.steps)]
    k2_ms = [recs[i][1].elapsed_time(recs[i][2]) for i in range(args.steps)]
    k3_ms = [recs[i][2].elapsed_time(recs[i][3]) for i in range(args.steps)]
    dev_sec = sum(step_ms) / 1e3
    max_sec = max_over_ranks(dev_sec, device=dev)
    agg = aggregate(S * n, ws, max_sec, args.steps)

    # algorithmic bytes
    cand_rows = S * n if (gqa or union) else S * (n - P - W)  # their statistics cover every cached row
    score_bytes = 0 if w.random else cand_rows * d * e
    compact_bytes = moved * (4 * d * e + 8)
    step_bytes = score_bytes + compact_bytes
    mean = lambda xs: sum(xs) / len(xs)
    peak, peak_kind = measured_peak_gbs()
    if w.random and fused_sc:
        dom_name, dom_ms, dom_bytes = "select_compact_kernel", mean(k2_ms), compact_bytes
    elif w.random:
        dom_name, dom_ms, dom_bytes = "compact_kernel", mean(k3_ms), compact_bytes
    else:
        heads_kernel = "score_heads_tc_kernel" if w.dtype == torch.bfloat16 else "score_heads_kernel"
        dom_name, dom_ms, dom_bytes = (heads_kernel if gqa else "score_kernel"), mean(k1_ms), score_bytes
    achieved = dom_bytes / (dom_ms * 1e-3) / 1e9
    traffic = known_traffic(w.name, dom_name)
    result = {
        "metric": METRIC, "value": agg["value"], "unit": UNIT, "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": agg["ms_per_step"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": dict(workload_config(w, args.path), l2="inputs larger than L2 (K+V %.1f GB); the first %d rows of every "
                       "slice are restored between steps (%.1f GB written, also flushes L2)" % (
                           2 * S * w.n_cap * d * e / 1e9, B, 2 * S * B * d * e / 1e9)),
        "gbs": step_bytes / (dev_sec / args.steps) / 1e9,
        "hbm_frac_of_8tbs": step_bytes / (dev_sec / args.steps) / 1e9 / 8000.0,
        "algorithmic_bytes_per_step": step_bytes,
        "kernel_ms": ({"compress": round(mean(k1_ms), 4)} if fused else
                      ({"rand_evict_compact": round(mean(k2_ms), 4)} if fused_sc else
                       {("score_heads" if gqa else "score") if not w.random else "rand_select": round(mean(k1_ms), 4),
                        "select": round(mean(k2_ms), 4), "compact": round(mean(k3_ms), 4)})),
        "moved_rows_per_step": moved,
        "roofline": {"kernel": dom_name, "bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_kind": peak_kind, "traffic": traffic,
                     "bytes_per_launch": dom_bytes},
        "clocks": clocks.summary(),
        "gpu_launches": launches,
        "wall_ms_per_step_incl_restore": 1e3 * (w1 - w0) / args.steps,
    }
    del scores, cws
    torch.cuda.empty_cache()
    if not args.no_e2e and not (gqa or union or paged):
        result["e2e"] = run_e2e(args, w, tri, synth, inp, centers, dev, stream)
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(args, w)
    if ws == 1 and not args.no_extra and w.name == "qwen3_8b_stack" and args.path == "separate":
        del inp, centers, k_head, v_head, kv, keep, pos_out
        torch.cuda.empty_cache()
        result["other_workloads"] = measure_other(args, tri, synth, dev)
    if rank == 0:
        print(json.dumps(result), flush=True)
    return 0


def measure_other(args, tri, synth, dev):
    """The other 32K-token workloads, timed like the main one (CUDA events
    around each event, first B rows restored between events): Random
    Attention on the stack, the stack with per-query-head GQA scoring
    (z-score + max), and the large-batch periodic workload
    (its 32768-row event, then 16 rounds of +128 rows -> 2048 with explicit
    positions, the appended rows drawn outside the timed region)."""
    import numpy as np
    import torch

    out = {}
    peak, _ = measured_peak_gbs()
    steps = max(3, min(args.steps, 10))
    ev = lambda: torch.cuda.Event(enable_timing=True)

    def timed(fn, restore):
        ts = []
        for i in range(args.warmup + steps):
            restore()
            a, b = ev(), ev()
            a.record()
            fn()
            b.record()
            torch.cuda.synchronize()
            if i >= args.warmup:
                ts.append(a.elapsed_time(b))
        return sum(ts) / len(ts)

    # ---- Random Attention on the stack --------------------------------------
    w = synth.WORKLOADS["random_stack"]
    S, n, P, W, B = w.n_slices, w.n_valid, w.n_prompt, w.n_recent, w.budget
    inp = synth.make_inputs(w, dev, with_queries=False)
    kh, vh = inp.k[:, :, :, :B].clone(), inp.v[:, :, :, :B].clone()
    nv = torch.full((S,), n, dtype=torch.int32, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    kv = tri.KVCache(inp.k, inp.v, nv, None, torch.empty(S, w.n_cap, dtype=torch.int32, device=dev), st)
    keep = torch.empty(S, B, dtype=torch.int32, device=dev)

    def restore_r():
        inp.k[:, :, :, :B].copy_(kh)
        inp.v[:, :, :, :B].copy_(vh)
        nv.fill_(n)

    ms = timed(lambda: tri.rand_evict_compact(kv, 0, 0, P, W, B, keep), restore_r)
    moved = int((keep.cpu().numpy() != np.arange(B)[None, :]).sum())
    by = moved * (4 * w.head_dim * w.elem_bytes + 8)
    assert int(st.item()) == 0
    out[w.name] = {"value": S * n / (ms / 1e3), "unit": UNIT, "ms_per_event": ms, "gbs": by / ms / 1e6,
                   "hbm_frac_of_8tbs": by / ms / 1e6 / 8000.0, "frac_of_measured_peak": by / ms / 1e6 / peak,
                   "algorithmic_bytes": by}
    del inp, kh, vh, kv, keep
    torch.cuda.empty_cache()

    # ---- GQA on the stack: per-query-head scores, z-score + max --------------
    w = synth.WORKLOADS["qwen3_8b_stack"]
    S, n, P, W, B, G = w.n_slices, w.n_valid, w.n_prompt, w.n_recent, w.budget, w.group
    inp = synth.make_inputs(w, dev)
    cq = tri.calibrate_centers(inp.q, 1)  # one row per query head
    inp.q = None
    torch.cuda.empty_cache()
    kh, vh = inp.k[:, :, :, :B].clone(), inp.v[:, :, :, :B].clone()
    nv = torch.full((S,), n, dtype=torch.int32, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    kv = tri.KVCache(inp.k, inp.v, nv, None, torch.empty(S, w.n_cap, dtype=torch.int32, device=dev), st)
    scores_g = torch.empty(S, G, w.n_cap, dtype=torch.float32, device=dev)
    stats = torch.empty(S, G, 2, dtype=torch.float32, device=dev)
    hws = torch.empty(tri.score_heads_workspace_bytes(kv, G), dtype=torch.uint8, device=dev)
    keep = torch.empty(S, B, dtype=torch.int32, device=dev)
    kms = []

    def gqa_event():
        e = [ev() for _ in range(4)]
        e[0].record()
        tri.score_heads(kv, cq, G, w.theta, w.offsets, inp.p_cur, scores_g, stats, workspace=hws)
        e[1].record()
        tri.select_topk_zmax(scores_g, stats, G, kv, P, W, B, keep)
        e[2].record()
        tri.compact_kv(kv, keep, B)
        e[3].record()
        kms.append(e)

    def restore_g():
        inp.k[:, :, :, :B].copy_(kh)
        inp.v[:, :, :, :B].copy_(vh)
        nv.fill_(n)

    ms = timed(gqa_event, restore_g)
    kt = [[x[0].elapsed_time(x[1]), x[1].elapsed_time(x[2]), x[2].elapsed_time(x[3])]
          for x in kms[args.warmup:]]
    moved = int((keep.cpu().numpy() != np.arange(B)[None, :]).sum())
    score_by = S * n * w.head_dim * w.elem_bytes  # every cached row is scored (statistics over all keys)
    by = score_by + moved * (4 * w.head_dim * w.elem_bytes + 8)
    assert int(st.item()) == 0
    k_ms = [sum(x[j] for x in kt) / len(kt) for j in range(3)]
    out["qwen3_8b_stack_gqa"] = {
        "value": S * n / (ms / 1e3), "unit": UNIT, "ms_per_event": ms, "gbs": by / ms / 1e6,
        "hbm_frac_of_8tbs": by / ms / 1e6 / 8000.0, "frac_of_measured_peak": by / ms / 1e6 / peak,
        "algorithmic_bytes": by, "group": G,
        "kernel_ms": {"score_heads": round(k_ms[0], 4), "select_zmax": round(k_ms[1], 4),
                      "compact": round(k_ms[2], 4)},
        "score_heads_gbs": score_by / k_ms[0] / 1e6}
    del inp, kh, vh, kv, keep, scores_g, stats, hws
    torch.cuda.empty_cache()

    # ---- the stack with one keep list per (seq, layer): union across heads ---
    w = synth.WORKLOADS["qwen3_8b_stack"]
    S, n, P, W, B = w.n_slices, w.n_valid, w.n_prompt, w.n_recent, w.budget
    k_head = B - P - W  # every head picks as many as are kept
    inp = synth.make_inputs(w, dev)
    c = tri.calibrate_centers(inp.q, w.group)
    inp.q = None
    torch.cuda.empty_cache()
    kh, vh = inp.k[:, :, :, :B].clone(), inp.v[:, :, :, :B].clone()
    nv = torch.full((S,), n, dtype=torch.int32, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    kv = tri.KVCache(inp.k, inp.v, nv, None, torch.empty(S, w.n_cap, dtype=torch.int32, device=dev), st)
    scores = torch.empty(S, w.n_cap, dtype=torch.float32, device=dev)
    keep = torch.empty(S, B, dtype=torch.int32, device=dev)
    uws = torch.empty(tri.select_union_workspace_bytes(kv, P, W, k_head), dtype=torch.uint8, device=dev)
    kms = []

    def union_event():
        e = [ev() for _ in range(4)]
        e[0].record()
        tri.score(kv, c, w.theta, w.offsets, inp.p_cur, scores)  # the statistics need every row
        e[1].record()
        tri.select_union(scores, kv, P, W, B, k_head, keep, workspace=uws)
        e[2].record()
        tri.compact_kv(kv, keep, B)
        e[3].record()
        kms.append(e)

    def restore_u():
        inp.k[:, :, :, :B].copy_(kh)
        inp.v[:, :, :, :B].copy_(vh)
        nv.fill_(n)

    ms = timed(union_event, restore_u)
    kt = [[x[0].elapsed_time(x[1]), x[1].elapsed_time(x[2]), x[2].elapsed_time(x[3])] for x in kms[args.warmup:]]
    k_ms = [sum(x[j] for x in kt) / len(kt) for j in range(3)]
    moved = int((keep.cpu().numpy() != np.arange(B)[None, :]).sum())
    score_by = S * n * w.head_dim * w.elem_bytes
    by = score_by + moved * (4 * w.head_dim * w.elem_bytes + 8)
    assert int(st.item()) == 0
    out["qwen3_8b_stack_union"] = {
        "value": S * n / (ms / 1e3), "unit": UNIT, "ms_per_event": ms, "gbs": by / ms / 1e6,
        "hbm_frac_of_8tbs": by / ms / 1e6 / 8000.0, "frac_of_measured_peak": by / ms / 1e6 / peak,
        "algorithmic_bytes": by, "k_head": k_head, "heads_per_list": w.n_kv_heads,
        "kernel_ms": {"score": round(k_ms[0], 4), "select_union": round(k_ms[1], 4), "compact": round(k_ms[2], 4)}}
    del inp, kh, vh, kv, keep, scores, uws
    torch.cuda.empty_cache()

    # ---- the stack in a paged pool (16-row blocks, shuffled block tables) ---
    w = synth.WORKLOADS["qwen3_8b_stack"]
    S, n, P, W, B = w.n_slices, w.n_valid, w.n_prompt, w.n_recent, w.budget
    L, H, d, bs = w.n_layers, w.n_kv_heads, w.head_dim, 16
    inp = synth.make_inputs(w, dev)
    c = tri.calibrate_centers(inp.q, w.group)
    inp.q = None
    mb = w.n_cap // bs
    nb = w.n_seq * mb
    perm = torch.randperm(nb, generator=torch.Generator().manual_seed(1)).view(w.n_seq, mb)
    table = perm.to(torch.int32).to(dev)
    kp = torch.empty(nb, L, H, bs, d, dtype=w.dtype, device=dev)
    vp = torch.empty_like(kp)
    for sq in range(w.n_seq):  # move each sequence into its blocks, then drop the contiguous copy
        idx = perm[sq].to(dev)
        kp[idx] = inp.k[sq].reshape(L, H, mb, bs, d).permute(2, 0, 1, 3, 4)
        vp[idx] = inp.v[sq].reshape(L, H, mb, bs, d).permute(2, 0, 1, 3, 4)
    p_cur = inp.p_cur.clone()
    del inp
    torch.cuda.empty_cache()
    head_blocks = table[:, : (B + bs - 1) // bs].reshape(-1).long()  # the blocks compaction rewrites
    kh, vh = kp[head_blocks].clone(), vp[head_blocks].clone()
    nv = torch.full((S,), n, dtype=torch.int32, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    kv = tri.PagedKVCache(kp, vp, table, nv, None, torch.empty(S, w.n_cap, dtype=torch.int32, device=dev), st)
    scores = torch.empty(S, w.n_cap, dtype=torch.float32, device=dev)
    keep = torch.empty(S, B, dtype=torch.int32, device=dev)
    kms = []

    def paged_event():
        e = [ev() for _ in range(4)]
        e[0].record()
        tri.score(kv, c, w.theta, w.offsets, p_cur, scores, n_prompt=P, n_recent=W)
        e[1].record()
        tri.select_topk(scores, kv, P, W, B, keep)
        e[2].record()
        tri.compact_kv(kv, keep, B)
        e[3].record()
        kms.append(e)

    def restore_b():
        kp[head_blocks] = kh
        vp[head_blocks] = vh
        nv.fill_(n)

    ms = timed(paged_event, restore_b)
    kt = [[x[0].elapsed_time(x[1]), x[1].elapsed_time(x[2]), x[2].elapsed_time(x[3])] for x in kms[args.warmup:]]
    k_ms = [sum(x[j] for x in kt) / len(kt) for j in range(3)]
    moved = int((keep.cpu().numpy() != np.arange(B)[None, :]).sum())
    score_by = S * (n - P - W) * d * w.elem_bytes
    by = score_by + moved * (4 * d * w.elem_bytes + 8)
    assert int(st.item()) == 0
    out["qwen3_8b_stack_paged"] = {
        "value": S * n / (ms / 1e3), "unit": UNIT, "ms_per_event": ms, "gbs": by / ms / 1e6,
        "hbm_frac_of_8tbs": by / ms / 1e6 / 8000.0, "frac_of_measured_peak": by / ms / 1e6 / peak,
        "algorithmic_bytes": by, "block_size": bs, "layout": "[blocks][layers][kv heads][16 rows][d], shuffled tables",
        "kernel_ms": {"score": round(k_ms[0], 4), "select": round(k_ms[1], 4), "compact": round(k_ms[2], 4)}}
    del kp, vp, kh, vh, kv, keep, scores, table
    torch.cuda.empty_cache()

    # ---- the stack with post-RoPE keys (the engine layout) ------------------
    w = synth.WORKLOADS["qwen3_8b_stack_post_rope"]
    S, n, P, W, B = w.n_slices, w.n_valid, w.n_prompt, w.n_recent, w.budget
    inp = synth.make_inputs(w, dev)
    c = tri.calibrate_centers(inp.q, w.group)
    inp.q = None
    torch.cuda.empty_cache()
    kh, vh = inp.k[:, :, :, :B].clone(), inp.v[:, :, :, :B].clone()
    nv = torch.full((S,), n, dtype=torch.int32, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    kv = tri.KVCache(inp.k, inp.v, nv, None, torch.empty(S, w.n_cap, dtype=torch.int32, device=dev), st,
                     post_rope=True)
    scores = torch.empty(S, w.n_cap, dtype=torch.float32, device=dev)
    keep = torch.empty(S, B, dtype=torch.int32, device=dev)
    kms = []

    def post_event():
        e = [ev() for _ in range(4)]
        e[0].record()
        tri.score(kv, c, w.theta, w.offsets, inp.p_cur, scores, n_prompt=P, n_recent=W)
        e[1].record()
        tri.select_topk(scores, kv, P, W, B, keep)
        e[2].record()
        tri.compact_kv(kv, keep, B)
        e[3].record()
        kms.append(e)

    def restore_q():
        inp.k[:, :, :, :B].copy_(kh)
        inp.v[:, :, :, :B].copy_(vh)
        nv.fill_(n)

    ms = timed(post_event, restore_q)
    kt = [[x[0].elapsed_time(x[1]), x[1].elapsed_time(x[2]), x[2].elapsed_time(x[3])] for x in kms[args.warmup:]]
    k_ms = [sum(x[j] for x in kt) / len(kt) for j in range(3)]
    moved = int((keep.cpu().numpy() != np.arange(B)[None, :]).sum())
    score_by = S * (n - P - W) * w.head_dim * w.elem_bytes
    by = score_by + moved * (4 * w.head_dim * w.elem_bytes + 8)
    assert int(st.item()) == 0
    out[w.name] = {
        "value": S * n / (ms / 1e3), "unit": UNIT, "ms_per_event": ms, "gbs": by / ms / 1e6,
        "hbm_frac_of_8tbs": by / ms / 1e6 / 8000.0, "frac_of_measured_peak": by / ms / 1e6 / peak,
        "algorithmic_bytes": by,
        "kernel_ms": {"score": round(k_ms[0], 4), "select": round(k_ms[1], 4), "compact": round(k_ms[2], 4)},
        "score_gbs": score_by / k_ms[0] / 1e6, "score_frac_of_measured_peak": score_by / k_ms[0] / 1e6 / peak}
    del inp, kh, vh, kv, keep, scores
    torch.cuda.empty_cache()

    # ---- large-batch periodic -----------------------------------------------
    w = synth.WORKLOADS["periodic_large_batch"]
    S, n, P, W, B, R, d, e = (w.n_slices, w.n_valid, w.n_prompt, w.n_recent, w.budget, w.round_rows,
                              w.head_dim, w.elem_bytes)
    inp = synth.make_inputs(w, dev)
    c = tri.calibrate_centers(inp.q, w.group)
    inp.q = None
    torch.cuda.empty_cache()
    kh, vh = inp.k[:, :, :, :B].clone(), inp.v[:, :, :, :B].clone()
    nv = torch.full((S,), n, dtype=torch.int32, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    pos = torch.empty(S, w.n_cap, dtype=torch.int32, device=dev)
    kv = tri.KVCache(inp.k, inp.v, nv, None, pos, st)
    scores = torch.empty(S, w.n_cap, dtype=torch.float32, device=dev)
    keep = torch.empty(S, B, dtype=torch.int32, device=dev)
    p_cur = inp.p_cur.clone()

    def event():
        tri.score(kv, c, w.theta, w.offsets, p_cur, scores, n_prompt=P, n_recent=W)
        tri.select_topk(scores, kv, P, W, B, keep)
        tri.compact_kv(kv, keep, B)

    def restore_p():
        inp.k[:, :, :, :B].copy_(kh)
        inp.v[:, :, :, :B].copy_(vh)
        nv.fill_(n)
        kv.pos = None

    ms = timed(event, restore_p)
    moved = int((keep.cpu().numpy() != np.arange(B)[None, :]).sum())
    by = S * (n - P - W) * d * e + moved * (4 * d * e + 8)
    assert int(st.item()) == 0
    res = {"pass_32k": {"value": S * n / (ms / 1e3), "unit": UNIT, "ms_per_event": ms, "gbs": by / ms / 1e6,
                        "hbm_frac_of_8tbs": by / ms / 1e6 / 8000.0, "frac_of_measured_peak": by / ms / 1e6 / peak,
                        "algorithmic_bytes": by}}
    # rounds continue from the state the last timed pass left; in steady state
    # only B + R rows of each slice are in use, so the rounds see a cache view
    # of capacity B + R (same storage and slice stride, positions and scores
    # laid out [S][B + R])
    cap = B + R
    pos2 = pos[:, :cap].clone()
    nv2 = torch.full((S,), B, dtype=torch.int32, device=dev)
    kv2 = tri.KVCache(inp.k[:, :, :, :cap], inp.v[:, :, :, :cap], nv2, pos2, pos2, st)
    cws2 = torch.empty(tri.compress_workspace_bytes(kv2), dtype=torch.uint8, device=dev)
    # untimed warm-up of the rounds' kernel (the same instantiation: dtype,
    # head_dim, explicit positions, one CTA per slice) on a one-slice cache of
    # its own, so that loading the kernel's code is not timed in round 1
    wk = inp.k[:1, :1, :1, :cap].clone(memory_format=torch.contiguous_format)
    wv = inp.v[:1, :1, :1, :cap].clone(memory_format=torch.contiguous_format)
    wpos = torch.arange(cap, dtype=torch.int32, device=dev)[None, :].contiguous()
    wkv = tri.KVCache(wk, wv, torch.full((1,), cap, dtype=torch.int32, device=dev), wpos, wpos, st)
    tri.compress(wkv, c, w.theta, w.offsets, p_cur[:1], P, W, B, keep[:1])
    torch.cuda.synchronize()
    del wk, wv, wpos, wkv
    rms, rby = [], []
    # clocks while the rounds run (each round is one ~1.3 ms launch between
    # host-side appends, so a clock that sags between launches shows here)
    rclk = ClockSampler(nvsmi_gpu_id(dev.index if dev.index is not None else torch.cuda.current_device()))
    rclk.start()
    time.sleep(0.3)
    rclk.mark("r0")
    for rnd in range(1, w.rounds + 1):
        kn, vn = synth.append_rows(inp, rnd, R)
        inp.k[:, :, :, B:B + R] = kn
        inp.v[:, :, :, B:B + R] = vn
        first = n + R * (rnd - 1)
        pos2[:, B:B + R] = torch.arange(first, first + R, dtype=torch.int32, device=dev)[None, :]
        nv2.fill_(B + R)
        p_cur.fill_(first + R - 1)
        del kn, vn
        a, b = ev(), ev()
        torch.cuda.synchronize()
        a.record()
        # short slices (one score CTA each): one kernel scores, selects and
        # compacts each slice, so a slice's latency-bound selection overlaps
        # other slices' traffic
        tri.compress(kv2, c, w.theta, w.offsets, p_cur, P, W, B, keep, workspace=cws2)
        b.record()
        torch.cuda.synchronize()
        rms.append(a.elapsed_time(b))
        mv = int((keep.cpu().numpy() != np.arange(B)[None, :]).sum())
        rby.append(S * (B + R - P - W) * (d * e + 4) + mv * (4 * d * e + 8))
    rclk.mark("r1")
    rclk.stop()
    assert int(st.item()) == 0
    mr = sum(rms) / len(rms)
    mb = sum(rby) / len(rby)
    res["rounds"] = {"count": w.rounds, "value": S * (B + R) / (mr / 1e3), "unit": UNIT, "ms_per_round": mr,
                     "ms_each": [round(x, 4) for x in rms], "clocks": rclk.summary("r0", "r1"),
                     "gbs": mb / mr / 1e6, "hbm_frac_of_8tbs": mb / mr / 1e6 / 8000.0,
                     "view": "capacity B + 128 rows per slice (steady state)",
                     "path": "tri_compress (one kernel: each slice scored, selected and compacted by one CTA)"}
    out[w.name] = res
    del inp, kh, vh, kv, kv2, keep, scores, cws2, pos, pos2
    torch.cuda.empty_cache()
    return out


# the files each kernel is built from (its traffic record is tied to their hash)
KERNEL_SOURCES = {"score_kernel": ["score.cu", "score_core.cuh", "score_common.cuh", "tri_internal.cuh"],
                  "compress_slice_kernel": ["compress.cu", "score_core.cuh", "score_common.cuh", "select_core.cuh",
                                            "compact_core.cuh", "tri_internal.cuh"],
                  "select_kernel": ["select_core.cuh", "tri_internal.cuh"],
                  "compact_kernel": ["compact_core.cuh", "tri_internal.cuh"],
                  "score_heads_kernel": ["score_heads.cu", "score_common.cuh", "tri_internal.cuh"],
                  "score_heads_tc_kernel": ["score_heads_tc.cu", "score_common.cuh", "umma.cuh", "tri_internal.cuh"],
                  "select_compact_kernel": ["select_compact.cu", "select_core.cuh", "compact_core.cuh",
                                            "tri_internal.cuh"]}


def kernel_sources_sha1(kernel: str) -> str:
    """sha1 of the concatenated source files a kernel is built from."""
    import hashlib

    h = hashlib.sha1()
    for name in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "kv_cache_compression_tri_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def known_traffic(workload: str, kernel: str):
    """DRAM bytes (read + write) per launch from the committed ncu summary
    (profiles/traffic.json), or None when there is none or the kernel's
    source has changed since the counters were taken."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            rec = json.load(f).get(workload, {}).get(kernel)
        sha = kernel_sources_sha1(kernel)
    except (OSError, ValueError, KeyError):
        return None
    if not rec or not sha.startswith(rec.get("source_sha1_prefix", "-")):
        return None
    return rec["bytes"]


def run_e2e(args, w, tri, synth, inp, centers, dev, stream):
    """Same metric through the public API with host buffers: each step copies
    the cache in from pinned host memory, compresses it, and reads the
    compacted rows and keep lists back (sequence by sequence, overlapped)."""
    import torch

    S, n, P, W, B = w.n_slices, w.n_valid, w.n_prompt, w.n_recent, w.budget
    LH = w.n_layers * w.n_kv_heads
    per_seq = 2 * LH * w.n_cap * w.head_dim * w.elem_bytes + 2 * LH * B * w.head_dim * w.elem_bytes + LH * B * 4
    avail = host_mem_available()
    n_seq = max(1, min(w.n_seq, int(0.5 * avail) // per_seq, args.e2e_max_seqs))
    Se = n_seq * LH
    # Host buffers: one pinned block per (sequence, layer) and tensor. The
    # pinned-memory allocator rounds every request up to a power of two, and a
    # (sequence, layer) of K is 2^26 bytes here, so blocks of that size waste
    # nothing (one tensor for the batch would take up to twice its size).
    # Memory page-locked after allocation (cudaHostRegister) gave well under
    # half the copy rate here (1.1e8 against 2.9e8 KV tokens/s end to end).
    L_ = w.n_layers

    def blocks(rows):
        return [[torch.empty(w.n_kv_heads, rows, w.head_dim, dtype=w.dtype, pin_memory=True) for _ in range(L_)]
                for _ in range(n_seq)]

    hk, hv = blocks(w.n_cap), blocks(w.n_cap)
    for c in range(n_seq):
        for l in range(L_):
            hk[c][l].copy_(inp.k[c, l])
            hv[c][l].copy_(inp.v[c, l])
    out_k, out_v = blocks(B), blocks(B)
    out_keep = torch.empty(Se, B, dtype=torch.int32, pin_memory=True)
    dk, dv = inp.k[:n_seq], inp.v[:n_seq]
    n_valid = torch.full((Se,), n, dtype=torch.int32, device=dev)
    pos_out = torch.empty(Se, w.n_cap, dtype=torch.int32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    keep = torch.empty(Se, B, dtype=torch.int32, device=dev)
    p_cur = inp.p_cur[:n_seq]

    fused = not w.random  # scored workloads go through the single public call (tri_compress)
    # Pipelined by sequence on three streams: the copy-in of sequence c + 1
    # runs while sequence c is compressed and sequence c - 1 is copied out
    # (the link carries both directions at once). A sequence's buffers are
    # rewritten only after the previous step has copied its result out.
    LHs = w.n_layers * w.n_kv_heads
    views = []
    for c in range(n_seq):
        sl = slice(c * LHs, (c + 1) * LHs)
        kvc = tri.KVCache(dk[c:c + 1], dv[c:c + 1], n_valid[sl], None, pos_out[sl], status,
                          post_rope=(w.key_layout == "post"))
        views.append((kvc, sl))
    cws = torch.empty(tri.compress_workspace_bytes(views[0][0]), dtype=torch.uint8, device=dev) if fused else None
    s_in, s_cmp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(n_seq)]
    ev_cmp = [torch.cuda.Event() for _ in range(n_seq)]
    ev_out = [torch.cuda.Event() for _ in range(n_seq)]
    started = [False]

    def one():
        for c, (kvc, sl) in enumerate(views):
            with torch.cuda.stream(s_in):
                if started[0]:
                    s_in.wait_event(ev_out[c])  # the previous step has read this sequence's result
                for l in range(L_):
                    dk[c, l].copy_(hk[c][l], non_blocking=True)
                    dv[c, l].copy_(hv[c][l], non_blocking=True)
                ev_in[c].record(s_in)
            with torch.cuda.stream(s_cmp):
                s_cmp.wait_event(ev_in[c])
                n_valid[sl].fill_(n)
                if w.random:
                    tri.rand_evict(kvc, 0, 0, P, W, B, keep[sl])
                    tri.compact_kv(kvc, keep[sl], B)
                else:
                    tri.compress(kvc, centers, w.theta, w.offsets, p_cur[c:c + 1], P, W, B, keep[sl],
                                 workspace=cws)
                ev_cmp[c].record(s_cmp)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_cmp[c])
                for l in range(L_):
                    out_k[c][l].copy_(dk[c, l, :, :B], non_blocking=True)
                    out_v[c][l].copy_(dv[c, l, :, :B], non_blocking=True)
                out_keep[sl].copy_(keep[sl], non_blocking=True)
                ev_out[c].record(s_out)
        started[0] = True

    for _ in range(max(1, args.warmup)):
        one()
    torch.cuda.synchronize()
    steps = max(1, min(args.steps, args.e2e_steps))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0 = time.perf_counter()
    e0.record(s_in)
    for _ in range(steps):
        one()
    s_in.wait_stream(s_out)
    e1.record(s_in)
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    sec = max(e0.elapsed_time(e1) / 1e3, wall)
    h2d = 2 * sum(t.numel() * t.element_size() for row in hk for t in row)
    d2h = 2 * sum(t.numel() * t.element_size() for row in out_k for t in row) + out_keep.numel() * 4
    assert int(status.item()) == 0
    res = {"value": Se * n * steps / sec, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
           "steps": steps, "n_seq": n_seq,
           "pipeline": "per sequence: copy-in, compress and copy-out on three streams, overlapped; host buffers "
                       "pinned per (sequence, layer)"}
    if n_seq != w.n_seq:
        res["note"] = f"host-buffer leg runs {n_seq} of {w.n_seq} sequences (pinned host memory bound)"
    del hk, hv, out_k, out_v, out_keep
    return res


def cpu_baseline(args, w):
    cores = host_cores()
    items = oracle_sample_inputs(w, args.cpu_slices)
    oracle_time(w, items[:1], 1)  # warm the library
    sec = oracle_time(w, items, cores)
    tokens = len(items) * w.n_valid
    return {"value": tokens / sec, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{len(items)} slices drawn like {w.name} ({w.n_valid} rows each), fp64 oracle "
                      f"score/select/compact, {cores} threads, {sec:.1f} s"}


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["gpu", "reference", "ours"], default="gpu")
    ap.add_argument("--workload", default="qwen3_8b_stack")
    ap.add_argument("--path", choices=["separate", "compress", "gqa", "union", "paged"], default="separate",
                    help="separate: tri_score + tri_select_topk + tri_compact_kv (an event after each; "
                         "rand_evict_compact for Random Attention); "
                         "compress: the single tri_compress call; gqa: per-query-head scores, "
                         "z-score + max selection, compaction; union: one keep list per (seq, layer) "
                         "(tri_select_union); paged: the separate calls on a paged copy of the cache "
                         "(16-row blocks, shuffled tables)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra", action="store_true", help="skip the other 32K-token workloads")
    ap.add_argument("--e2e-steps", type=int, default=3)
    ap.add_argument("--e2e-max-seqs", type=int, default=16)
    ap.add_argument("--cpu-slices", type=int, default=32)
    ap.add_argument("--ref-slices", type=int, default=16)
    args = ap.parse_args(argv)
    from kv_cache_compression_tri_gb300 import synth

    w = synth.WORKLOADS[args.workload]
    if args.impl == "reference":
        return run_reference(args, w)
    return run_gpu(args, w)


if __name__ == "__main__":
    sys.exit(main())
