"""Benchmark of one verification round per layer on GB300.

Workload: the DFlash2-style block verification configuration (K = 8 verify
queries per request at positions S..S+7, batch 128, S = 102400, int8
indexer with 4 heads of 128 summed, top-k 2048, GQA 16/1 with d = 128 in
bf16, hot cache 4096 rows per request, optional residency 0, queries of a
request sharing ~60% of their top rows), synthetic and seeded.  A step is
one whole round: select (indexer + top-k), resolve (union, probe,
compaction, shared host gather), attend (ring write, attention over the
union, merge, hot-cache install) and commit.  Metric: verified query-tokens
per second per layer = N * K / step time.  ``--workload`` times the other
configurations (diagnostics); ``--sweep`` runs the load-adaptive sweep
(optional residency 0/5/25/100% of history x K = 1/2/4/8, shared against
per-query retrieval) on the same shapes.

Each timed step starts from the same state (the snapshot taken after the
previous-step round), restored outside the timed region, and the L2 cache is
flushed (a 512 MiB write) before every step, also outside it.

Multi-GPU: requests are independent, so every rank runs its own batch of
requests on its own GPU (weak scaling, no collective on the data path); the
step time is the maximum over ranks.

--impl reference times the oracle (the plain CPU restatement in ``oracle/``)
on the host cores: each step is one request's round, a bounded sample of the
same workload, and the steps run on a pool of processes, one per core.
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOAD = "cfg3"


def wl_configs():
    import workload as wl
    return wl.CONFIGS.keys()


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--workload", default=WORKLOAD, choices=sorted(wl_configs()),
                    help="configuration to time (the headline is %s)" % WORKLOAD)
    ap.add_argument("--attn-pass", type=int, default=0, choices=[0, 1, 2, 3],
                    help="attention pass after a shared resolve: 0 auto, 1 per query, 2 union "
                         "(tensor cores where the shape allows), 3 union on mma.sync")
    ap.add_argument("--sweep", action="store_true",
                    help="the load-adaptive sweep on the DFlash2-style shapes: optional residency "
                         "0/5/25/100%% x K = 1/2/4/8, shared against per-query retrieval; one JSON "
                         "line per point, then a summary line")
    ap.add_argument("--layers", type=int, default=0,
                    help="layer-group diagnostic: one index producer and LAYERS-1 follower payload "
                         "layers on --chi shared staging arenas, timed on one stream and pipelined "
                         "(resolves with their host gathers on a copy stream while the previous "
                         "layer attends on a compute stream); prints one JSON line")
    ap.add_argument("--chi", type=int, default=2, help="staging arenas of the layer group")
    ap.add_argument("--round-groups", type=int, default=3,
                    help="issue each round as one dhs_round call with the requests split into "
                         "this many groups on internal streams (0: the four separate calls)")
    ap.add_argument("--groups", type=int, default=0,
                    help="request-group diagnostic: the workload's requests split into GROUPS "
                         "contexts on as many streams, each running its own round, so that one "
                         "group's host gather can overlap another's indexer; prints one JSON line")
    ap.add_argument("--batch", type=int, default=0,
                    help="requests per GPU (default: the configuration's); a smaller batch is a "
                         "cut of the workload for profiling, not a bench line")
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ---------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while timing."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu: int):
        self.gpu = gpu
        self.proc = None
        import tempfile
        self.path = os.path.join(tempfile.mkdtemp(prefix="dhs_clocks_"), "clocks_gpu%d.csv" % gpu)

    def start(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "20"], stdout=self.f,
                stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            p = [x.strip() for x in line.split(",")]
            if len(p) < 9:
                continue
            try:
                sm.append(float(p[1]))
                smax.append(float(p[2]))
            except ValueError:
                continue
            for n, v in zip(names, p[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": float(max(smax)),
                "samples": len(sm), "reasons": sorted(reasons)}


# ---------------------------------------------------------------- CPU baseline
def oracle_requests(rec, slots):
    """Run round 0 (previous step) on the oracle for ``slots``; return the oracle."""
    import oracle
    cfg = oracle.Config(n_slots=rec.N, k_max=rec.kmax, topk=rec.topk, s_max=rec.s_max,
                        idx_heads=rec.H_idx, idx_dim=rec.d_idx, q_heads=rec.Hq, Hkv=rec.Hkv,
                        qk_dim=rec.qk_dim, v_dim=rec.v_dim, kv_layout=rec.kv_layout,
                        budget=rec.B, ring_window=rec.W, page_rows=rec.p,
                        opt_rows_max=rec.opt_rows_max)
    o = oracle.Oracle(cfg)
    for r in slots:
        o.bind(r, rec.host_rows(r, r + 1)[0], rec.index_keys(r, r + 1)[0], rec.S)
    return o


def oracle_round_inputs(rec, rnd, slots):
    N, Km = rec.N, rec.kmax
    qi = np.zeros((N, Km, rec.idx_row), np.int8)
    qa = np.zeros((N, Km, rec.Hq, rec.qk_dim), np.uint16)
    bl = np.zeros((N, Km, rec.row_elems), np.uint16)
    for r in slots:
        qi[r] = rec.index_queries(rnd, r, r + 1)[0]
        qa[r] = rec.attn_queries(rnd, r, r + 1)[0]
        bl[r] = rec.block_rows(rnd, r, r + 1)[0]
    return qi, qa, bl


def oracle_step(o, rec, rnd, slots):
    kr = np.zeros(rec.N, np.int32)
    kr[slots] = rec.K
    qi, qa, bl = oracle_round_inputs(rec, rnd, slots)
    sel = o.select(qi, kr)
    o.resolve(sel)
    o.attend(qa, bl)
    acc = rec.accepted(rnd)
    acc_s = np.zeros(rec.N, np.int32)
    acc_s[slots] = acc[slots]
    o.commit(acc_s)


def _oracle_request_round(job):
    """One bounded sample of the workload on the oracle: request ``r``'s
    previous-step round (untimed; it leaves the hot cache as the workload
    describes), then its timed verification round.  Runs in a worker
    process; returns (request, seconds of the timed round)."""
    rec, r = job
    o = oracle_requests(rec, [r])
    oracle_step(o, rec, 0, [r])
    t0 = time.perf_counter()
    oracle_step(o, rec, 1, [r])
    return r, time.perf_counter() - t0


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def oracle_pool(rec, n_jobs, workers):
    """Run ``n_jobs`` request-rounds of the oracle (requests taken in order,
    cyclically) on ``workers`` processes started with ``spawn`` (each one
    single-threaded: numpy's thread pools are limited to one thread), all
    running at once.  Returns the per-job timed seconds and the wall time of
    the whole pool."""
    import multiprocessing as mp
    keep = {k: os.environ.get(k) for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS",
                                           "MKL_NUM_THREADS")}
    for k in keep:
        os.environ[k] = "1"
    try:
        ctx = mp.get_context("spawn")
        t0 = time.perf_counter()
        with ctx.Pool(workers) as pool:
            res = list(pool.imap_unordered(_oracle_request_round,
                                           [(rec, i % rec.N) for i in range(n_jobs)]))
        wall = time.perf_counter() - t0
    finally:
        for k, v in keep.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
    return [dt for _, dt in res], wall


def cpu_baseline(rec, rounds_per_core=2):
    """Time the oracle on the host cores: request-rounds of the workload
    (round 1, from the state round 0 leaves) on one single-threaded process
    per core, all running together, ``rounds_per_core`` each.  The value is
    the cores' summed rate: query-tokens of the timed rounds / mean timed
    round time x cores.  Set-up (input generation, round 0) is not timed."""
    cores = host_cores()
    times, wall = oracle_pool(rec, rounds_per_core * cores, cores)
    per = float(np.mean(times))
    return {"value": round(cores * rec.K / per, 2), "unit": "query-tokens/s", "cores": cores,
            "kind": "oracle",
            "single_thread_value": round(rec.K / per, 3),
            "sample": "%d request-rounds of the workload (K=%d, S=%d; requests 0..%d), one "
                      "single-threaded numpy process per host core (int64 scores, float64 "
                      "attention), all cores busy together; value = cores x K / mean timed "
                      "round" % (len(times), rec.K, rec.S, min(rec.N, len(times)) - 1),
            "seconds_timed": round(float(np.sum(times)), 2), "wall_s": round(wall, 2)}


# ---------------------------------------------------------------- algorithmic bytes
def algorithmic_bytes(rec, counts, k_per_req):
    """Bytes each step must move (not the work it avoids), per kernel and family.

    select family: index keys of the domain (read once for all K queries), the
    int8 queries and the int32 top-k lists.  attend family: each distinct
    selected row once, the block rows, bf16 queries and outputs, int32
    locations.  Per kernel: index_score reads keys and queries; topk reads the
    int32 scores and writes the lists; union_probe reads the lists and two
    row maps per union row and writes locations and the union and miss lists;
    gather moves the distinct missing rows over the host link (their writes
    to staging and to promoted hot slots are HBM-side); attn (per-query
    pass) and attn_union (union pass) are the attend family plus the block
    rows written into the draft ring; commit copies accepted rows.
    """
    K = int(k_per_req.max())
    n_act = int((k_per_req > 0).sum())
    rb = rec.row_bytes
    keys = n_act * rec.S * rec.idx_row
    qbytes = n_act * K * rec.idx_row
    lists = 4 * n_act * K * rec.topk
    select = keys + qbytes + lists
    U = int(counts[:, 0].sum())
    M = int(counts[:, 1].sum())
    qo = 2 * n_act * K * rec.Hq * (rec.qk_dim + rec.v_dim)
    attend = U * rb + n_act * K * rb + qo + lists
    kernel = {
        "index_score": keys + qbytes,
        "topk": 4 * n_act * K * rec.S + lists,
        "union_probe": 2 * lists + 8 * U + 4 * (U + M),
        "gather": M * rb,
        "attn": attend + n_act * K * rb,
        "attn_union": attend + n_act * K * rb,
    }
    return {"select": select, "attn": attend, "gather": M * rb, "union": U, "misses": M,
            "kernel_bytes": kernel}


# ncu --set full summaries per workload: DRAM traffic per launch of each
# kernel, captured on the whole workload or on a cut of its requests (the
# summary states "captured requests: n"; traffic grows with the requests, so
# it is scaled to the full batch).
NCU_SUMMARIES = {
    "cfg2": os.path.join(ROOT, "profiles", "kernels_cfg2_ncu_full.md"),
    "cfg3": os.path.join(ROOT, "profiles", "kernels_cfg3_batch16_ncu_full.md"),
}
NCU_SUMMARY = NCU_SUMMARIES["cfg3"]
NCU_NAMES = {"index_score": "k_index_score", "topk": "k_topk", "union_probe": "k_union_probe",
             "gather": "k_gather", "attn": "k_attn<", "attn_union": "k_uattn",
             "commit": "k_commit"}


def csrc_hash() -> str:
    """sha256 over the kernel sources (file name, then bytes; sorted), 16 hex digits."""
    import glob
    import hashlib
    h = hashlib.sha256()
    for f in sorted(glob.glob(os.path.join(ROOT, "hierarchical_sparse_kv_int8_gb300", "csrc", "*"))):
        h.update(os.path.basename(f).encode())
        h.update(open(f, "rb").read())
    return h.hexdigest()[:16]


def ncu_traffic(name, path=None, full_requests=None):
    """DRAM bytes (read + write) per launch of kernel ``name`` from a committed
    ncu --set full summary (default NCU_SUMMARY), scaled from the captured
    requests to ``full_requests`` when both are known; None when the summary
    is missing or the kernel sources have changed since it was captured."""
    import re
    path = path or NCU_SUMMARY
    if name not in NCU_NAMES or not os.path.exists(path):
        return None
    text = open(path).read()
    m = re.search(r"csrc-sha256: ([0-9a-f]+)", text)
    if not m or m.group(1) != csrc_hash():
        return None
    scale_req = 1.0
    mc = re.search(r"captured requests: (\d+)", text)
    if mc and full_requests:
        scale_req = full_requests / float(mc.group(1))
    scale = {"byte": 1.0, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9}
    for sec in text.split("\n## ")[1:]:
        if not sec.startswith(NCU_NAMES[name]):
            continue
        ms = re.search(r"captured requests: (\d+)", sec)  # a section captured on its own cut
        if ms and full_requests:
            scale_req = full_requests / float(ms.group(1))
        rd = re.search(r"DRAM read: ([0-9.]+) (\w+)", sec)
        wr = re.search(r"DRAM write: ([0-9.]+) (\w+)", sec)
        if rd and wr and rd.group(2) in scale and wr.group(2) in scale:
            return int(scale_req * (float(rd.group(1)) * scale[rd.group(2)] +
                                    float(wr.group(1)) * scale[wr.group(2)]))
    return None


def measure_h2d(torch, stream, nbytes=256 << 20):
    """Host-to-device link bandwidth: best of 5 pinned 256 MiB copies."""
    h = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
    d = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    best = 0.0
    for _ in range(6):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        d.copy_(h, non_blocking=True)
        b.record(stream)
        stream.synchronize()
        best = max(best, nbytes / (a.elapsed_time(b) * 1e-3) / 1e9)
    del h, d
    return best


# ---------------------------------------------------------------- native arm
def run_native(args):
    import torch
    import workload as wl
    import hierarchical_sparse_kv_int8_gb300 as dhs
    from hierarchical_sparse_kv_int8_gb300.runner import Runner

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    dhs.build()
    rec = wl.CONFIGS[args.workload]
    if args.batch:
        rec = rec.scaled(N=args.batch)
    if world > 1:
        rec = rec.scaled(seed=rec.seed + rank)   # each rank serves its own requests
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        run = Runner(rec, stream=stream, attn_pass=args.attn_pass,
                     round_groups=max(0, args.round_groups))
        kr = rec.k_per_req()
        # previous decode step: leaves the hot cache holding its selection
        run.load_round(0)
        run.round(kr, rec.accepted(0))
        run.load_round(1)
        snap = run.ctx.snapshot(stream)
        acc1 = rec.accepted(1)
        flush = torch.empty(512 << 20, dtype=torch.uint8, device="cuda")
        stream.synchronize()
        h2d_peak = measure_h2d(torch, stream)

        def step():
            if args.round_groups:
                run.round_fused(kr, acc1)
                return
            run.select(kr)
            run.resolve(True)
            run.attend()
            run.commit(acc1)

        for _ in range(args.warmup):
            run.ctx.restore(snap, stream)
            step()
        stream.synchronize()
        counts = run.export("counts", torch.int32, (rec.N, 4)).cpu().numpy()
        st_before = run.ctx.stats(stream)

        # Eager (one C-ABI call at a time) step time, for reference.
        ev0 = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]
        for i in range(args.steps):
            run.ctx.restore(snap, stream)
            flush.fill_(i & 0xFF)
            ev0[i][0].record(stream)
            step()
            ev0[i][1].record(stream)
        stream.synchronize()
        eager_ms = float(np.mean([a.elapsed_time(b) for a, b in ev0]))

        # The timed step is the same round captured once as a CUDA graph (the
        # state is restored before every launch, so the round is identical),
        # through the library's capture, which keeps the launches' priorities
        # that order the request groups (a plain graph ignores them).
        def capture(timing):
            run.ctx.set_timing(timing)
            run.ctx.restore(snap, stream)
            stream.synchronize()
            with dhs.Graph.capture(stream) as g:
                step()
            stream.synchronize()
            return g
        graph = capture(False)
        graph_timed = capture(True)
        # clocks are sampled from just before the warm-up to the end of the
        # timed steps (nvidia-smi needs a moment to start)
        sampler = ClockSampler(local)
        sampler.start()
        time.sleep(0.3)
        for _ in range(args.warmup):
            run.ctx.restore(snap, stream)
            graph.replay()
        stream.synchronize()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(args.steps)]
        barrier(world)
        stream.synchronize()
        for i in range(args.steps):
            run.ctx.restore(snap, stream)
            flush.fill_(i & 0xFF)
            ev[i][0].record(stream)
            graph.replay()
            ev[i][1].record(stream)
        stream.synchronize()
        clocks = sampler.stop()
        barrier(world)
        # per-kernel durations: the same steps, replayed from the graph that
        # carries an event pair around every kernel
        run.ctx.set_timing(True)
        for i in range(args.steps):
            run.ctx.restore(snap, stream)
            flush.fill_(i & 0xFF)
            graph_timed.replay()
            stream.synchronize()
            run.ctx.timing_accumulate_graph()
        kt = run.ctx.kernel_times()
        run.ctx.set_timing(False)
        ms_steps = [a.elapsed_time(b) for a, b in ev]
        ms_local = float(np.mean(ms_steps))
        st_after = run.ctx.stats(stream)

        # end to end through the host-buffer entry point
        hq = torch.from_numpy(rec.index_queries(1, 0, rec.N)).pin_memory()
        hqa = torch.from_numpy(rec.attn_queries(1, 0, rec.N).view(np.int16)).pin_memory()
        hbl = torch.from_numpy(rec.block_rows(1, 0, rec.N).view(np.int16)).pin_memory()
        hout = torch.empty((rec.N, rec.kmax, rec.Hq, rec.v_dim), dtype=torch.int16).pin_memory()
        hlse = torch.empty((rec.N, rec.kmax, rec.Hq), dtype=torch.float32).pin_memory()
        e2e_times = []
        for i in range(args.warmup + args.steps):
            run.ctx.restore(snap, stream)
            flush.fill_(i & 0xFF)
            stream.synchronize()
            t0 = time.perf_counter()
            run.ctx.round_host(hq, kr, hqa, hbl, acc1, hout, hlse, stream)
            t1 = time.perf_counter()
            if i >= args.warmup:
                e2e_times.append(t1 - t0)
        e2e_ms_local = 1e3 * float(np.mean(e2e_times))
        h2d = hq.numel() + hqa.numel() * 2 + hbl.numel() * 2
        d2h = hout.numel() * 2 + hlse.numel() * 4

    ms = max_over_ranks(ms_local, world)
    e2e_ms = max_over_ranks(e2e_ms_local, world)
    tokens = int(kr.sum())
    value = world * tokens / (ms * 1e-3)
    e2e_value = world * tokens / (e2e_ms * 1e-3)

    # roofline of every kernel and of the dominant one (largest share of the
    # timed region): algorithmic bytes per launch / average launch duration
    ab = algorithmic_bytes(rec, counts, kr)
    per = {name: (n, t) for name, (n, t) in kt.items() if n > 0}
    dom = max(per, key=lambda k: per[k][1])
    peaks = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json"))) \
        if os.path.exists(os.path.join(ROOT, "MEASURED_PEAKS.json")) else None
    hbm_peak = peaks["hbm_gbs"] if peaks else 6800.0
    hbm_src = "MEASURED_PEAKS.json hbm_gbs (copy, burst)" if peaks else "fallback 6.8 TB/s"
    roofs = {}
    # a kernel may run several times per step (once per request group): its
    # achieved rate is the round's algorithmic bytes over its event time per
    # step, which equals the bytes of one launch over that launch's time;
    # algorithmic bytes and ncu traffic are reported per launch
    for name, (n_l, t_l) in per.items():
        byts = ab["kernel_bytes"].get(name)
        if byts is None:
            continue
        avg_ms = t_l / n_l
        step_ms = t_l / args.steps
        ach = byts / (step_ms * 1e-3) / 1e9
        link = name == "gather"
        peak = h2d_peak if link else hbm_peak
        roofs[name] = {"kernel": name, "bound": "h2d" if link else "hbm",
                       "achieved": round(ach, 1), "peak": round(peak, 1), "unit": "GB/s",
                       "frac": round(ach / peak, 4),
                       "traffic": (ncu_traffic(name, NCU_SUMMARIES[args.workload],
                                               rec.N * args.steps / n_l)
                                   if args.workload in NCU_SUMMARIES else None),
                       "algorithmic_bytes": int(byts * args.steps / n_l),
                       "avg_launch_ms": round(avg_ms, 5),
                       "launches_per_step": round(n_l / args.steps, 3),
                       "ms_per_step": round(step_ms, 5),
                       "peak_source": ("host link: pinned host-to-device copy measured in this run"
                                       if link else hbm_src)}
    if "gather" in roofs:
        roofs["gather"]["traffic_note"] = (
            "DRAM bytes from ncu; the gather's algorithmic bytes cross the host link, "
            "not DRAM, and its staging and hot-slot writes stay in L2 during the launch")
    roof = roofs.get(dom)
    sel_t = sum(per[k][1] / args.steps for k in ("index_score", "topk") if k in per)
    att_t = sum(per[k][1] / args.steps for k in ("attn", "attn_union") if k in per)
    sa_bytes = ab["select"] + ab["attn"]
    families = {
        "select": {"achieved": round(ab["select"] / (sel_t * 1e-3) / 1e9, 1), "unit": "GB/s",
                   "frac_of_hbm": round(ab["select"] / (sel_t * 1e-3) / 1e9 / hbm_peak, 4),
                   "algorithmic_bytes": ab["select"], "ms": round(sel_t, 5)},
        "attend": {"achieved": round(ab["attn"] / (att_t * 1e-3) / 1e9, 1), "unit": "GB/s",
                   "frac_of_hbm": round(ab["attn"] / (att_t * 1e-3) / 1e9 / hbm_peak, 4),
                   "algorithmic_bytes": ab["attn"], "ms": round(att_t, 5)},
        # steps 1 and 5 together: indexer + top-k + attention bytes over the
        # sum of their average launch times
        "select+attend": {
            "achieved": round(sa_bytes / ((sel_t + att_t) * 1e-3) / 1e9, 1), "unit": "GB/s",
            "frac_of_hbm": round(sa_bytes / ((sel_t + att_t) * 1e-3) / 1e9 / hbm_peak, 4),
            "algorithmic_bytes": sa_bytes, "ms": round(sel_t + att_t, 5),
            "peak": round(hbm_peak, 1), "peak_source": hbm_src},
    }
    if "gather" in roofs:
        families["shared gather"] = {
            "achieved": roofs["gather"]["achieved"], "unit": "GB/s",
            "frac_of_h2d": roofs["gather"]["frac"], "h2d_peak": round(h2d_peak, 1)}
    breakdown = {k: {"launches": n, "avg_us": round(1e3 * t / n, 2),
                     "share": round(t / sum(v[1] for v in per.values()), 4)}
                 for k, (n, t) in per.items()}
    # every kernel of the round is timed (the control words travel as kernel
    # parameters, so no upload launch is needed)
    launches_per_step = sum(n for n, _ in per.values()) / args.steps
    # dhs_round forms request groups for the tensor-core union pass only
    groups = (args.round_groups if args.round_groups > 1 and "attn_union" in per
              and args.attn_pass != 3 else 1)
    if groups > 1:
        # the timed graph issues every kernel once per request group
        launches_per_step *= groups
    line = {
        "metric": "verified query-tokens/s per layer (select+resolve+attend)",
        "value": round(value, 1), "unit": "query-tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16+int8",
        "data": "synthetic (seeded; shapes of the %s configuration)" % rec.name,
        "config": dict(workload_config(rec),
                       l2="flushed (512 MiB write) before every step",
                       state="restored from snapshot before every step (untimed)",
                       attention_pass="union" if "attn_union" in per else "per_query",
                       round=("one dhs_round call, requests in %d groups on internal streams"
                              % groups if args.round_groups
                              else "dhs_select, dhs_resolve, dhs_attend, dhs_commit")),
        "e2e": {"value": round(e2e_value, 1), "unit": "query-tokens/s",
                "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
                "ms_per_step": round(e2e_ms, 5),
                "api": "dhs_round_host (pinned host inputs and outputs)"},
        "gpu_launches": int(round(launches_per_step * args.steps)),
        "eager_ms_per_step": round(eager_ms, 5),
        "launch": ("CUDA graph of one round (one dhs_round call: select, resolve, attend, commit "
                   "per request group, the %d groups overlapping on internal streams of "
                   "decreasing priority, a group's indexer after the previous group's top-k and "
                   "its attention after the next group's top-k; captured with dhs_graph_*, which "
                   "instantiates it with "
                   "the launches' priorities honoured), replayed per step; kernel times (roofline, families, kernels) from a second replay of "
                   "the same steps issued as one request group (each kernel over the whole batch, "
                   "none overlapping) with an event pair around every kernel" % groups)
                  if args.round_groups else
                  "CUDA graph of one round (select, resolve, attend, commit), replayed per step; "
                  "kernel times from a second replay of the same steps with per-kernel events",
        "roofline": roof,
        "roofline_all": roofs,
        "families": families,
        "kernels": breakdown,
        "workload_stats": {"union_rows": ab["union"], "misses": ab["misses"],
                           "hot_hits": int(counts[:, 3].sum()),
                           "host_bytes_per_step": ab["gather"]},
        "clocks": clocks,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(rec)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


# ---------------------------------------------------------------- reference arm
def run_sweep(args):
    """The load-adaptive sweep on the DFlash2-style shapes.

    One context with an optional pool for the whole history serves every
    point.  For each optional-residency fraction (whole pages, seeded) every
    slot is bound again and its optional rows set; for each K the
    previous-step round runs with K queries per request (it leaves the hot
    cache), its state is snapshotted, and round 1 is timed from that state
    with shared retrieval and with per-query retrieval (each missing
    selection fetched on its own).  Per point: the host-fetched fraction of
    the selected rows (rows fetched / valid selections, one round), the
    selections per fetched row, and verify-query throughput N * K / step time
    (CUDA events around each eager round, state restored and L2 flushed
    before every step, outside the timed region)."""
    import torch
    import workload as wl
    import hierarchical_sparse_kv_int8_gb300 as dhs
    from hierarchical_sparse_kv_int8_gb300.runner import Runner

    torch.cuda.set_device(0)
    dhs.build()
    base_rec = wl.sweep_recipe(1.0)
    if args.batch:
        base_rec = base_rec.scaled(N=args.batch)
    stream = torch.cuda.Stream()
    points = []
    steps = max(1, args.steps)
    with torch.cuda.stream(stream):
        run = Runner(base_rec, stream=stream)
        flush = torch.empty(512 << 20, dtype=torch.uint8, device="cuda")
        for opt in wl.SWEEP_OPT:
            rec = wl.sweep_recipe(opt).scaled(N=base_rec.N)
            run.rebind()
            run.set_residency(rec.residency_rows)
            base = run.ctx.snapshot(stream)
            for K in wl.SWEEP_K:
                kr = np.full(rec.N, K, np.int32)
                run.ctx.restore(base, stream)
                run.load_round(0)
                run.round(kr, rec.accepted(0, kr))
                run.load_round(1)
                snap = run.ctx.snapshot(stream)
                acc = rec.accepted(1, kr)
                for shared in (True, False):
                    # one round for the counters
                    run.ctx.restore(snap, stream)
                    run.ctx.reset_stats(stream)
                    run.round(kr, acc, shared)
                    st = run.ctx.stats(stream)
                    for i in range(args.warmup):
                        run.ctx.restore(snap, stream)
                        run.round(kr, acc, shared)
                    ev = []
                    for i in range(steps):
                        run.ctx.restore(snap, stream)
                        flush.fill_(i & 0xFF)
                        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                        a.record(stream)
                        run.round(kr, acc, shared)
                        b.record(stream)
                        ev.append((a, b))
                    stream.synchronize()
                    ms = float(np.median([a.elapsed_time(b) for a, b in ev]))
                    sel = max(1, st["selections"])
                    pt = {"sweep_point": True, "workload": rec.name, "optional_residency": opt,
                          "K": K, "retrieval": "shared" if shared else "per_query",
                          "selections": st["selections"], "union_rows": st["union_rows"],
                          "misses": st["misses"], "miss_selections": st["miss_selections"],
                          "host_rows_fetched": st["host_rows_fetched"],
                          "host_fetched_frac": round(st["host_rows_fetched"] / sel, 5),
                          "selections_per_fetched_row": (
                              round(st["miss_selections"] / st["host_rows_fetched"], 4)
                              if st["host_rows_fetched"] else None),
                          "opt_hits": st["opt_hits"], "hot_hits": st["hot_hits"],
                          "ring_hits": st["ring_hits"], "direct_only": st["direct_only"],
                          "ms_per_step": round(ms, 5),
                          "query_tokens_per_s": round(rec.N * K / (ms * 1e-3), 1)}
                    points.append(pt)
                    print(json.dumps(pt), flush=True)
                run.ctx.snapshot_free(snap)
            run.ctx.snapshot_free(base)
    # shared against per-query retrieval, per (residency, K)
    pairs = {}
    for p in points:
        pairs.setdefault((p["optional_residency"], p["K"]), {})[p["retrieval"]] = p
    summary = []
    for (opt, K), d in sorted(pairs.items()):
        sh, pq = d["shared"], d["per_query"]
        summary.append({
            "optional_residency": opt, "K": K,
            "host_fetched_frac_shared": sh["host_fetched_frac"],
            "host_fetched_frac_per_query": pq["host_fetched_frac"],
            "fetch_reduction": (round(1 - sh["host_rows_fetched"] / pq["host_rows_fetched"], 4)
                                if pq["host_rows_fetched"] else None),
            "query_tokens_per_s_shared": sh["query_tokens_per_s"],
            "query_tokens_per_s_per_query": pq["query_tokens_per_s"]})
    print(json.dumps({"sweep": "load-adaptive (optional residency x K x retrieval)",
                      "workload": base_rec.name, "batch": base_rec.N, "S": base_rec.S,
                      "steps": steps, "warmup": args.warmup,
                      "timing": "median of CUDA-event times around eager rounds; state restored "
                                "and L2 flushed before every step (untimed)",
                      "points": summary}), flush=True)


def run_layers(args):
    """Layer-group pipelining on the workload's shapes (a diagnostic).

    Layer 0 produces the positions (indexer + top-k); layers 1..L-1 are
    follower payload layers with their own host rows, hot caches and rings
    that take those positions.  All stage in ``chi`` shared arenas (layer l
    in arena l mod chi).  A step is every layer's resolve and attention plus
    the commits.  Sequential: all on one stream, layer after layer.
    Pipelined: resolves on a copy stream, each layer's attention on a
    compute stream one layer behind, so a layer's host gather overlaps the
    previous layer's attention; a resolve into an arena waits on the GPU for
    its previous user's attention.  Both start every step from the same
    snapshot, with the L2 flushed (untimed)."""
    import torch
    import workload as wl
    import hierarchical_sparse_kv_int8_gb300 as dhs
    from hierarchical_sparse_kv_int8_gb300.runner import Runner

    torch.cuda.set_device(0)
    dhs.build()
    base = wl.CONFIGS[args.workload].scaled(N=args.batch or 32)
    L, chi = max(2, args.layers), max(1, args.chi)
    recs = [base.scaled(seed=base.seed + l) for l in range(L)]
    comp, copy = torch.cuda.Stream(), torch.cuda.Stream()
    arenas = dhs.Arenas(chi, base.N, base.kmax, base.topk, base.row_elems)
    runs = [Runner(recs[0], arenas=arenas, arena=0, stream=comp)]
    for l in range(1, L):
        runs.append(Runner(recs[l], arenas=arenas, arena=l % chi, role=dhs.ROLE_FOLLOWER,
                           keys=runs[0].keys, stream=comp))
    kr = base.k_per_req()
    for rnd in range(2):  # the previous step, then the timed step's inputs
        for run in runs:
            run.load_round(rnd)
        torch.cuda.synchronize()
        if rnd == 0:
            p = runs[0]
            p.ctx.select(p.q_idx, kr, p.topk, None, comp)
            for l, run in enumerate(runs):
                if l:
                    run.topk = p.topk
                    run.ctx.adopt(kr, None, comp)
                run.ctx.resolve(run.topk, run.loc, True, comp)
                run.ctx.attend(run.q, run.block, run.loc, run.out, run.lse, comp)
            for run in runs:
                run.ctx.commit(base.accepted(0, kr), comp)
    torch.cuda.synchronize()
    snaps = [run.ctx.snapshot(comp) for run in runs]
    acc = base.accepted(1, kr)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device="cuda")

    def step(pipelined):
        p = runs[0]
        p.ctx.select(p.q_idx, kr, p.topk, None, comp)
        cs = copy if pipelined else comp
        if pipelined:
            ev = torch.cuda.Event()
            ev.record(comp)
            copy.wait_event(ev)
        for l, run in enumerate(runs):
            if l:
                run.topk = p.topk
                run.ctx.adopt(kr, None, cs)
            run.ctx.resolve(run.topk, run.loc, True, cs)
            if not pipelined:
                run.ctx.attend(run.q, run.block, run.loc, run.out, run.lse, comp)
            elif l:
                prev = runs[l - 1]
                prev.ctx.attend(prev.q, prev.block, prev.loc, prev.out, prev.lse, comp)
        if pipelined:
            last = runs[-1]
            last.ctx.attend(last.q, last.block, last.loc, last.out, last.lse, comp)
        for run in runs:
            run.ctx.commit(acc, comp)

    res = {}
    for mode in ("sequential", "pipelined"):
        times = []
        for i in range(args.warmup + args.steps):
            for run, sn in zip(runs, snaps):
                run.ctx.restore(sn, comp)
            flush.fill_(i & 0xFF)
            torch.cuda.synchronize()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(comp)
            step(mode == "pipelined")
            b.record(comp)   # every layer's work ends in its commit, on this stream
            torch.cuda.synchronize()
            if i >= args.warmup:
                times.append(a.elapsed_time(b))
        res[mode] = float(np.median(times))
    # the gathers alone: per-kernel times of one sequential step
    for run in runs:
        run.ctx.set_timing(True)
    for run, sn in zip(runs, snaps):
        run.ctx.restore(sn, comp)
    torch.cuda.synchronize()
    step(False)
    torch.cuda.synchronize()
    per = {}
    for run in runs:
        for name, (n, ms) in run.ctx.kernel_times().items():
            if n:
                per[name] = per.get(name, 0.0) + ms
        run.ctx.set_timing(False)
    dedicated = L * base.N * base.kmax * base.topk * base.row_bytes
    line = {"diagnostic": "layer-group pipelining (producer + follower payload layers)",
            "workload": base.name, "batch": base.N, "K": base.K, "layers": L, "chi": chi,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step_sequential": round(res["sequential"], 4),
            "ms_per_step_pipelined": round(res["pipelined"], 4),
            "speedup": round(res["sequential"] / res["pipelined"], 3),
            "kernel_ms_one_sequential_step": {k: round(v, 4) for k, v in per.items()},
            "gather_ms_hidden": round(res["sequential"] - res["pipelined"], 4),
            "gather_ms_total": round(per.get("gather", 0.0), 4),
            "staging_bytes_shared_arenas": arenas.nbytes(),
            "staging_bytes_one_arena_per_layer": dedicated,
            "staging_ratio": round(dedicated / arenas.nbytes(), 2)}
    print(json.dumps(line), flush=True)
    for run in runs:
        run.ctx.close()
    arenas.close()


def run_groups(args):
    """The round of the workload's requests as G independent request groups
    (a diagnostic).  Requests are independent, so the round of N requests is
    G rounds of N/G requests, each on its own context and stream: one group's
    host gather (host link) may then run while another group's indexer
    (HBM) runs.  One stream, G streams and the one-context round are timed
    from the same snapshots, with the L2 flushed before every step."""
    import torch
    import workload as wl
    import hierarchical_sparse_kv_int8_gb300 as dhs
    from hierarchical_sparse_kv_int8_gb300.runner import Runner

    torch.cuda.set_device(0)
    dhs.build()
    rec = wl.CONFIGS[args.workload]
    if args.batch:
        rec = rec.scaled(N=args.batch)
    G = max(1, args.groups)
    assert rec.N % G == 0
    n = rec.N // G
    streams = [torch.cuda.Stream() for _ in range(G)]
    main = torch.cuda.Stream()
    runs = []
    for g in range(G):
        sub = rec.scaled(N=n, req0=g * n)
        runs.append(Runner(sub, stream=streams[g]))
    kr = runs[0].rec.k_per_req()
    for rnd in range(2):
        for run in runs:
            run.load_round(rnd)
        torch.cuda.synchronize()
        if rnd == 0:
            for run in runs:
                run.round(kr, run.rec.accepted(0, kr))
    torch.cuda.synchronize()
    snaps = [run.ctx.snapshot(run.stream) for run in runs]
    accs = [run.rec.accepted(1, kr) for run in runs]
    flush = torch.empty(512 << 20, dtype=torch.uint8, device="cuda")
    torch.cuda.synchronize()

    def step(parallel):
        ev0 = torch.cuda.Event()
        ev0.record(main)
        for g, run in enumerate(runs):
            s = run.stream if parallel else main
            s.wait_event(ev0)
            run.ctx.select(run.q_idx, kr, run.topk, None, s)
            run.ctx.resolve(run.topk, run.loc, True, s)
            run.ctx.attend(run.q, run.block, run.loc, run.out, run.lse, s)
            run.ctx.commit(accs[g], s)
            if parallel:
                e = torch.cuda.Event()
                e.record(s)
                main.wait_event(e)

    res = {}
    for mode in ("one_stream", "parallel"):
        times = []
        for i in range(args.warmup + args.steps):
            for run, sn in zip(runs, snaps):
                run.ctx.restore(sn, run.stream)
            flush.fill_(i & 0xFF)
            torch.cuda.synchronize()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(main)
            step(mode == "parallel")
            b.record(main)
            torch.cuda.synchronize()
            if i >= args.warmup:
                times.append(a.elapsed_time(b))
        res[mode] = float(np.median(times))
    tokens = rec.N * rec.K
    line = {"diagnostic": "request groups on parallel streams", "workload": rec.name,
            "batch": rec.N, "groups": G, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step_one_stream": round(res["one_stream"], 4),
            "ms_per_step_parallel": round(res["parallel"], 4),
            "query_tokens_per_s_one_stream": round(tokens / (res["one_stream"] * 1e-3), 1),
            "query_tokens_per_s_parallel": round(tokens / (res["parallel"] * 1e-3), 1)}
    print(json.dumps(line), flush=True)


def workload_config(rec):
    """The ``config`` object of both arms' lines: the workload and its shapes."""
    return {"workload": rec.name, "batch": rec.N, "K": rec.K, "S": rec.S, "topk": rec.topk,
            "idx_heads": rec.H_idx, "d_idx": rec.d_idx, "q_heads": rec.Hq,
            "kv_heads": rec.Hkv, "head_dim": rec.qk_dim, "hot_cache_rows": rec.B,
            "ring_window": rec.W, "optional_residency": rec.opt_frac}


def run_reference(args):
    """The oracle on the host cores.  Each step is one request's verification
    round (its previous-step round runs first, untimed), a bounded sample of
    the workload; the steps run on a spawn pool of one single-threaded
    process per core, all cores busy together, and the first ``warmup``
    rounds to finish are dropped.  The host's cores serve the whole node, so
    under torchrun rank 0 alone runs and the value covers every core of the
    node, whatever the number of ranks."""
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import workload as wl
    rec = wl.CONFIGS[args.workload]
    if args.batch:
        rec = rec.scaled(N=args.batch)
    cores = host_cores()
    times, wall = oracle_pool(rec, args.warmup + args.steps, cores)
    times = times[args.warmup:] if len(times) > args.warmup else times
    mean = float(np.mean(times))
    ms = 1e3 * mean / cores          # pool time per request-round, all cores busy
    value = rec.K / (ms * 1e-3)
    line = {
        "impl": "reference",
        "metric": "verified query-tokens/s per layer (select+resolve+attend)",
        "value": round(value, 2), "unit": "query-tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 3),
        "higher_is_better": True, "scaling": "none", "vs_baseline": None, "dtype": "int64+f64",
        "per_rank": False,
        "reference_scope": "every host core of the node, run by rank 0 alone; the host's "
                           "cores are shared by all ranks, so the value does not grow with "
                           "n_gpus",
        "data": "synthetic (seeded; shapes of the %s configuration)" % rec.name,
        "config": workload_config(rec),
        "cpu_baseline": {"value": round(value, 2), "unit": "query-tokens/s", "cores": cores,
                         "kind": "oracle", "single_thread_value": round(rec.K / mean, 3),
                         "sample": "one request's verification round per step (%d timed), "
                                   "one single-threaded numpy process per host core" % len(times),
                         "wall_s": round(wall, 2)},
        "e2e": {"value": round(value, 2), "unit": "query-tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    a = parse()
    if a.impl == "reference":
        run_reference(a)
    elif a.sweep:
        run_sweep(a)
    elif a.layers:
        run_layers(a)
    elif a.groups:
        run_groups(a)
    else:
        run_native(a)
