#!/usr/bin/env python3
"""Benchmark of the sparse KV-cache offloading decode step on GB300.

One step = one decode step of every layer for every request: append the new
token, select blocks (shared top-k over block summaries), recall the missing
blocks from pinned host memory into the device pool, and run GQA sparse decode
attention; recall of layer l+1 overlaps attention of layer l (two streams).

Workloads follow the PulseInfer pages ("PulseInfer Guide: I/O-Centric Sparse
KV Cache Offloading": Llama-3-8B/70B shapes at 32k-128k context, paged blocks,
top-k budgets) with seeded synthetic data from ``synth``.

Reported (one JSON line, rank 0):
  value     sparse decode tokens/s (requests x steps / device time), inputs in HBM
  recall    UVA gather GB/s against the pinned host->device copy peak measured here
  roofline  the dominant kernel (by time) against its bound, plus every kernel
  e2e       the same step through pi_decode_step_host with host buffers
  cpu_baseline  the CPU oracle on a bounded sample of the same workload

``--impl reference`` times the CPU oracle alone (no GPU) on the same workload.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

CONFIGS = {
    "c1": dict(workload="small: 1 layer, batch 1, 8 q / 2 KV heads, d 64, 4096 tokens, blocks of 16, "
                        "top-32 + 4 recent, 64-slot pool",
               layers=1, batch=1, hq=8, hkv=2, head_dim=64, block_tokens=16, ntok=4096, k=32, window=4,
               pool_slots=64, rho=0.9, heavy=0.0),
    "c2": dict(workload="llama3-8b-shape: 32 layers, batch 8, 32 q / 8 KV heads, d 128, 32768 tokens, blocks of 64, "
                        "top-32 + 2 recent, pool 25% of blocks, AR(1) rho 0.9 queries, 5% heavy-hitter blocks",
               layers=32, batch=8, hq=32, hkv=8, head_dim=128, block_tokens=64, ntok=32768, k=32, window=2,
               pool_slots=128, rho=0.9, heavy=0.05),
    "c3": dict(workload="variable-recall stress: llama3-8b shape, 32 layers, batch 32, 65536 tokens, blocks of 64, "
                        "top-k drawn per (layer, step) from 16..128 + 2 recent, per-request resident fraction "
                        "10..60% (pool = max(fraction x blocks, 130)), AR(1) rho 0.8 queries",
               layers=32, batch=32, hq=32, hkv=8, head_dim=128, block_tokens=64, ntok=65536, k=128, window=2,
               pool_slots=0, rho=0.8, heavy=0.05, k_range=(16, 128), frac_range=(0.10, 0.60)),
    "c4": dict(workload="llama3-70b-slice: 8 of 80 layers, batch 16, 64 q / 8 KV heads, d 128, 131072 tokens, "
                        "blocks of 64, top-64 + 4 recent, pool 10% of blocks",
               layers=8, batch=16, hq=64, hkv=8, head_dim=128, block_tokens=64, ntok=131072, k=64, window=4,
               pool_slots=205, rho=0.9, heavy=0.0),
}
METRIC = "KV recall GB/s vs measured H2D peak; sparse decode tokens/s (1 GB300)"
KINDS = ["append", "select", "plan", "gather", "attention"]


def log(*a):
    print("[bench]", *a, file=sys.stderr, flush=True)


# ------------------------------------------------------------------ helpers
def host_mem_available() -> int:
    try:
        for line in open("/proc/meminfo"):
            if line.startswith("MemAvailable:"):
                return int(line.split()[1]) * 1024
    except OSError:
        pass
    return 1 << 40


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


def measure_h2d_peak(torch, dev, numa_out=None) -> float:
    """Pinned host -> device cudaMemcpyAsync of 1 GiB, best of 10 (GB/s). numa_out
    (a dict) receives the NUMA placement of the pinned buffer's pages."""
    n = 1 << 30
    h = torch.empty(n, dtype=torch.uint8, pin_memory=True)
    h.fill_(1)
    if numa_out is not None:
        numa_out.update(numa_pages({"h2d_probe_buffer": (h.data_ptr(), n)}))
    d = torch.empty(n, dtype=torch.uint8, device=dev)
    s = torch.cuda.Stream()
    best = 0.0
    with torch.cuda.stream(s):
        for _ in range(10):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(s)
            d.copy_(h, non_blocking=True)
            e1.record(s)
            e1.synchronize()
            best = max(best, n / (e0.elapsed_time(e1) * 1e-3) / 1e9)
    del h, d
    return best


def numa_pages(ranges):
    """NUMA nodes holding the pages of each named host range {name: (address,
    bytes)}: page counts per node from /proc/self/numa_maps over the mappings
    that overlap the range (read-only queries). {name: {"N0": pages, ...}}."""
    out = {}
    try:
        maps = []
        for line in open("/proc/self/maps"):
            a, b = line.split()[0].split("-")
            maps.append((int(a, 16), int(b, 16)))
        nodes_of = {}
        for line in open("/proc/self/numa_maps"):
            f = line.split()
            nodes_of[int(f[0], 16)] = {kv.split("=")[0]: int(kv.split("=")[1]) for kv in f[1:]
                                       if kv.startswith("N") and "=" in kv and kv[1:].split("=")[0].isdigit()}
        for name, (addr, nbytes) in ranges.items():
            tot = {}
            for a, b in maps:
                if a < addr + nbytes and b > addr:
                    for k_, v_ in nodes_of.get(a, {}).items():
                        tot[k_] = tot.get(k_, 0) + v_
            out[name] = tot
    except (OSError, ValueError, IndexError):
        pass
    return out


def gpu_numa_affinity(gpu_index: int):
    """The GPU's NUMA affinity column of `nvidia-smi topo -m` (a query), or None."""
    try:
        txt = subprocess.run(["nvidia-smi", "topo", "-m"], capture_output=True, text=True, timeout=20).stdout
    except (OSError, subprocess.TimeoutExpired):
        return None
    lines = [l_ for l_ in txt.splitlines() if l_.strip()]
    head = next((l_ for l_ in lines if "NUMA Affinity" in l_), None)
    row = next((l_ for l_ in lines if l_.split() and l_.split()[0] == f"GPU{gpu_index}"), None)
    if head is None or row is None:
        return None
    cols = [c.strip() for c in head.replace("\x1b[4m", "").replace("\x1b[0m", "").split("\t") if c.strip()]
    vals = [c.strip() for c in row.split("\t") if c.strip()]
    try:
        return vals[1:][cols.index("NUMA Affinity")]
    except (ValueError, IndexError):
        return None


def reduce_max(value: float, world: int, device=None) -> float:
    """Max of a per-rank float over all ranks (identity at world 1)."""
    if world <= 1:
        return float(value)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def rank_seed(seed: int, rank: int) -> int:
    """Each rank serves its own requests (data parallel over requests)."""
    return seed + 1000 * rank


def weak_scaling_tokens_per_s(world: int, batch: int, steps: int, elapsed_max_s: float) -> float:
    """Whole-job throughput: every rank decodes `batch` tokens per step; time is the slowest rank's."""
    return world * batch * steps / elapsed_max_s


# ------------------------------------------------------------------ CPU oracle leg
def oracle_unit_step(orc, region, kmean, ntok, q, k, W, sob, bos, pool_copy, k_new, v_new, hkv, B):
    """One (request, layer) of one decode step on the CPU oracle: append, select,
    plan, recall copy, attention. Returns the new token count."""
    b, tp = divmod(ntok, B)
    region[b, :, 0, tp] = k_new
    region[b, :, 1, tp] = v_new
    ntok += 1
    kmean[b] = orc.block_summary(region[b], tp + 1)
    nb = -(-ntok // B)
    sel = orc.select_shared(q, kmean[:nb], k, W)
    res = orc.recall_plan(sel, sob, bos)
    _, mb, ms, _ = res
    for blk, slot in zip(mb, ms):
        pool_copy[slot] = region[blk]
    orc.attention(q, region, sel, ntok, hkv)
    return ntok


class OracleSample:
    """A bounded sample of (request, layer) units of the workload for the CPU oracle."""

    def __init__(self, cfg, seed, units, max_blocks, region_source=None):
        import oracle as orc
        import synth
        self.orc, self.synth, self.cfg, self.seed = orc, synth, cfg, seed
        self.units = units
        self.B, self.hkv = cfg["block_tokens"], cfg["hkv"]
        self.state = {}
        nb0 = -(-cfg["ntok"] // cfg["block_tokens"])
        for (r, l) in units:
            if region_source is not None:
                reg = np.array(region_source(l, r))
            else:
                reg = synth.kv_region(seed, l, r, cfg["ntok"], max_blocks, cfg["hkv"], cfg["block_tokens"],
                                      cfg["head_dim"], cfg["heavy"], 2.0)
            km = np.zeros((max_blocks, cfg["hkv"], cfg["head_dim"]), dtype=np.float32)
            km[:nb0] = orc.region_summaries(reg, cfg["ntok"])
            P_unit = cfg["pool_slots"] or (cfg["k"] + cfg["window"])
            sob = np.full(max_blocks, -1, dtype=np.int32)
            resident = []
            if "frac_range" in cfg:
                # the variable-recall workload: per-request pool size and preloaded
                # residency drawn exactly as the GPU run draws them
                lo, hi = cfg["frac_range"]
                f = synth.uniform_real(seed, synth.KIND_FRAC, r, 0, 0, lo, hi)
                P_unit = max(int(math.ceil(f * nb0)), cfg["k"] + cfg["window"])
                resident = synth.sample_sorted(seed, synth.KIND_RESIDENT, l, r, nb0, int(round(f * nb0)))
            bos = np.full(P_unit, -1, dtype=np.int32)
            pool = np.zeros((P_unit,) + reg.shape[1:], dtype=np.uint16)
            for s_, b_ in enumerate(resident):
                sob[b_], bos[s_] = s_, b_
                pool[s_] = reg[b_]
            self.state[(r, l)] = dict(region=reg, kmean=km, ntok=cfg["ntok"], sob=sob, bos=bos, pool=pool)

    def budget(self, step_idx, l):
        """Top-k of layer l at decode step step_idx (drawn per (layer, step) in the
        variable-recall workload, as the GPU run draws it)."""
        if "k_range" in self.cfg:
            lo, hi = self.cfg["k_range"]
            return self.synth.uniform_int(self.seed, self.synth.KIND_BUDGET, step_idx, l, 0, lo, hi)
        return self.cfg["k"]

    def step(self, qs_step, step_idx, budget_s=None):
        """Run every unit (or until budget_s elapses). Returns (units done, seconds)."""
        t0 = time.perf_counter()
        done = 0
        for (r, l) in self.units:
            st = self.state[(r, l)]
            kn, vn = self.synth.token_kv(self.seed, l, r, self.cfg["ntok"] + step_idx, self.hkv, self.cfg["head_dim"])
            st["ntok"] = oracle_unit_step(self.orc, st["region"], st["kmean"], st["ntok"], qs_step[l, r],
                                          self.budget(step_idx, l),
                                          self.cfg["window"], st["sob"], st["bos"], st["pool"], kn, vn, self.hkv,
                                          self.B)
            done += 1
            if budget_s is not None and time.perf_counter() - t0 > budget_s:
                break
        return done, time.perf_counter() - t0


def cpu_baseline(cfg, seed, qs, max_blocks, region_source, budget_s=15.0, n_units=16):
    """Oracle on a bounded sample: n_units (request, layer) pairs stepped through
    consecutive decode steps until about budget_s seconds of oracle work."""
    L, R = cfg["layers"], cfg["batch"]
    rng = np.random.default_rng(seed + 17)
    all_units = [(r, l) for r in range(R) for l in range(L)]
    pick = [all_units[i] for i in sorted(rng.choice(len(all_units), size=min(n_units, len(all_units)),
                                                    replace=False))]
    samp = OracleSample(cfg, seed, pick, max_blocks, region_source)
    done, secs, steps = 0, 0.0, 0
    while secs < budget_s and steps < qs.shape[0]:
        d, t = samp.step(qs[steps], steps)
        done += d
        secs += t
        steps += 1
    per_unit = secs / max(done, 1)
    tok_s = 1.0 / (per_unit * L)   # one token of one request needs L units
    return {"value": tok_s, "unit": "tok/s", "cores": 1, "kind": "oracle",
            "sample": f"{len(pick)} (request, layer) units x {steps} decode steps = {done} unit-steps (append, "
                      f"select, plan, recall copy, fp64 attention), {secs:.1f} s single-threaded; "
                      f"tokens/s = 1 / (s per unit-step x {L} layers)"}


def _oracle_worker(args):
    """One process of the all-cores oracle leg: its own (request, layer) units,
    stepped through decode steps until the budget; returns (unit-steps, seconds)."""
    cfg, seed, units, max_blocks, budget_s, n_steps = args
    import synth
    qs = synth.q_ar1(seed, cfg["layers"], cfg["batch"], cfg["hq"], cfg["head_dim"], n_steps, cfg["rho"])
    samp = OracleSample(cfg, seed, units, max_blocks)
    done, secs, steps = 0, 0.0, 0
    while secs < budget_s and steps < n_steps:
        d, t = samp.step(qs[steps], steps, budget_s - secs)
        done += d
        secs += t
        steps += 1
    return done, secs


def cpu_baseline_all_cores(cfg, seed, max_blocks, budget_s=10.0, units_per_proc=2, procs=None):
    """The same oracle on every host core: one spawned process per core, each
    stepping its own (request, layer) units (the units are independent). Returns
    tokens/s from the summed unit-steps over the slowest process's time."""
    import multiprocessing as mp
    procs = procs or os.cpu_count() or 1
    L, R = cfg["layers"], cfg["batch"]
    rng = np.random.default_rng(seed + 29)
    all_units = [(r, l) for r in range(R) for l in range(L)]
    n = min(len(all_units), procs * units_per_proc)
    pick = [all_units[i] for i in sorted(rng.choice(len(all_units), size=n, replace=False))]
    groups = [pick[i::procs] for i in range(procs) if pick[i::procs]]
    n_steps = 64
    t0 = time.perf_counter()
    with mp.get_context("spawn").Pool(len(groups)) as pool_:
        res = pool_.map(_oracle_worker, [(cfg, seed, g, max_blocks, budget_s, n_steps) for g in groups])
    wall = time.perf_counter() - t0
    done = sum(d for d, _ in res)
    slowest = max(t for _, t in res)
    return {"value": done / slowest / L, "unit": "tok/s", "cores": len(groups), "kind": "oracle",
            "sample": f"{len(pick)} (request, layer) units over {len(groups)} spawned processes (one per core), "
                      f"{done} unit-steps in {slowest:.1f} s of the slowest process ({wall:.1f} s wall including "
                      f"start-up and input generation); tokens/s = unit-steps / s / {L} layers"}


# ------------------------------------------------------------------ measured traffic
# Host-link and DRAM bytes per recalled block of the UVA gather, from one ncu
# capture (counters syslts__t_sectors_srcunit_tex_aperture_sysmem_op_read_lookup_miss.sum
# x 32 B and dram__bytes_read.sum + dram__bytes_write.sum, divided by the blocks
# the captured launches recalled), valid only for the kernel sources whose hash
# is recorded with it: a changed kernel reports null until it is captured again.
GATHER_SOURCES = ["pi_gather.cuh", "pi_recall.cu"]
GATHER_TRAFFIC = {
    # ncu --set full of two gather launches of the variable-recall workload (2 layers,
    # batch 8): 999424 and 1302528 host-link read sectors for 122 and 159 recalled
    # 256 KiB blocks; DRAM 0.29 and 1.21 MB (the blocks land in L2)
    "sha": "9a4d8195ce0349e6", "block_bytes": 262144, "host_link_bytes_per_block": 262144.0,
    "dram_bytes_per_block": 1499648 / 281, "capture": "profiles/gather_kernel_uva_variable_recall.md"}


def sources_sha(names):
    import hashlib
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "sparse_kv_cache_block_gb300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def gather_traffic(blocks_per_launch: float, block_bytes: int):
    """traffic of one gather launch scaled from the capture by the blocks it
    recalls (the kernel reads each missing block once), or None with the reason."""
    sha = sources_sha(GATHER_SOURCES)
    rec = GATHER_TRAFFIC
    if not rec or rec.get("block_bytes") != block_bytes:
        return None, {"reason": "no capture of this kernel at this block size", "sources_sha": sha}
    if rec["sha"] != sha:
        return None, {"reason": "kernel changed since the capture", "sources_sha": sha, "captured_sha": rec["sha"]}
    return rec["host_link_bytes_per_block"] * blocks_per_launch, {
        "counter": "host-link read sectors x 32 B (syslts sysmem read misses), per launch, scaled from the capture by "
                   "recalled blocks", "dram_bytes_per_launch": rec["dram_bytes_per_block"] * blocks_per_launch,
        "capture": rec["capture"], "sources_sha": sha}


# ------------------------------------------------------------------ main arm
def run_ours(args, cfg, rank, world, local_rank, extra=False):
    """One configuration end to end. extra = True (the additional configurations
    of the same line): no e2e pass, no CPU legs, no eviction variant."""
    import torch

    import synth
    import sparse_kv_cache_block_gb300 as pi

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    pi.build()
    pi.load()
    L, R, Hq, Hkv, D, B = (cfg[k] for k in ("layers", "batch", "hq", "hkv", "head_dim", "block_tokens"))
    K, Wm = args.steps, args.warmup
    prewarm_cap = 400  # warm-up runs at least W steps and at least args.warmup_s seconds, at most this many
    total_steps = prewarm_cap + Wm + 4 * K + 4 + ((4 * args.pin_layers + 12 + Wm) if args.admission else 0)
    ntok0 = cfg["ntok"]
    max_blocks = -(-(ntok0 + total_steps) // B) + 1
    seed = rank_seed(args.seed, rank)
    method = {"uva": pi.PI_RECALL_UVA, "memcpy": pi.PI_RECALL_MEMCPY, "staged": pi.PI_RECALL_STAGED}[args.method]

    numa = {}
    h2d_peak = measure_h2d_peak(torch, dev, numa)
    log(f"rank {rank}: pinned H2D peak {h2d_peak:.1f} GB/s")

    region_bytes = max_blocks * 2 * Hkv * B * D * 2
    full_host = region_bytes * L * R
    budget = 0.6 * host_mem_available() / max(1, world if world > 1 else 1)
    host_layers = L
    if full_host > budget:
        host_layers = max(1, int(budget // (region_bytes * R)))
        log(f"rank {rank}: host store for {host_layers} of {L} layers (aliased) to fit host memory")
    nb0 = -(-ntok0 // B)
    fracs = None
    slots_per_req = None
    if "frac_range" in cfg:
        lo, hi = cfg["frac_range"]
        fracs = [synth.uniform_real(seed, synth.KIND_FRAC, r, 0, 0, lo, hi) for r in range(R)]
        slots_per_req = [max(int(math.ceil(f * nb0)), cfg["k"] + cfg["window"]) for f in fracs]
    pool = pi.Pool(L, R, Hq, Hkv, D, B, max_blocks, cfg["pool_slots"] or cfg["k"] + cfg["window"], cfg["k"],
                   cfg["window"], host_layers=(host_layers if host_layers < L else 0), gather_ctas=args.gather_ctas,
                   pool_slots_per_req=slots_per_req, gather_depth=args.gather_depth, host_alloc=args.host_alloc,
                   evict_policy=(pi.PI_EVICT_LRU if args.evict == "lru" else pi.PI_EVICT_ASCENDING),
                   select_mode=(pi.PI_CONSENSUS if args.select == "consensus" else pi.PI_SHARED),
                   pin_layers=(args.pin_layers if args.admission else 0))
    if args.select == "consensus":
        pool.set_consensus_lambda(args.consensus_lambda)
    if args.schedule == "dependent":
        pool.set_schedule(True, args.groups)
    pool.set_copy_streams(args.copy_streams)
    if args.fused:
        pool.set_fused(True, args.fused_ctas)
    if args.select_ahead >= 0 or args.two_streams:
        pool.set_pipeline(max(args.select_ahead, 0) if args.select_ahead >= 0 else 1, not args.two_streams)
    if args.gather_placement == "shared" or args.gather_ctas or args.gather_depth:
        pool.set_gather(args.gather_ctas, args.gather_depth or 8, args.gather_placement == "exclusive")
    if args.attn_splits:
        pool.set_attention(args.attn_splits)
    if not args.attn_cluster:
        pool.set_attention_cluster(False)
    t0 = time.time()
    for hl in range(host_layers):
        for r in range(R):
            synth.fill_kv(pool.host_kv_ptr(hl, r), seed, hl, r, ntok0, max_blocks, Hkv, B, D, cfg["heavy"], 2.0)
    for l in range(L):
        pool.update_summaries(l, [ntok0] * R)
    if fracs is not None:
        for l in range(L):
            for r in range(R):
                n_res = int(round(fracs[r] * nb0))
                pool.preload(l, r, synth.sample_sorted(seed, synth.KIND_RESIDENT, l, r, nb0, n_res))
    torch.cuda.synchronize()
    # prefill summaries (row a-1) of layer 0 again, timed: every key of the layer is
    # read over the host link through the mapping (the same values are rewritten)
    pre_ms = []
    for _ in range(3):
        e_p0, e_p1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e_p0.record()
        pool.update_summaries(0, [ntok0] * R)
        e_p1.record()
        torch.cuda.synchronize()
        pre_ms.append(e_p0.elapsed_time(e_p1))
    pre_bytes = R * ntok0 * Hkv * D * 2
    prefill = {"bytes": pre_bytes, "us": 1e3 * min(pre_ms), "us_all": [1e3 * x for x in pre_ms],
               "host_link_gbs": pre_bytes / (min(pre_ms) / 1e3) / 1e9,
               "note": "pi_update_summaries over one layer (keys of every request read through the mapping), "
                       "CUDA events, best of 3"}
    numa.update(numa_pages({"host_store": (pool.host_kv_ptr(0, 0), host_layers * R * pool.region_bytes)}))
    numa["gpu_numa_affinity"] = gpu_numa_affinity(local_rank)
    log(f"rank {rank}: host store {host_layers * R * region_bytes / 2**30:.1f} GiB filled + summarised in "
        f"{time.time() - t0:.1f} s")

    qs = synth.q_ar1(seed, L, R, Hq, D, total_steps, cfg["rho"])
    kn = np.empty((total_steps, L, R, Hkv, D), dtype=np.uint16)
    vn = np.empty_like(kn)
    for s in range(total_steps):
        for l in range(L):
            for r in range(R):
                kn[s, l, r], vn[s, l, r] = synth.token_kv(seed, l % host_layers, r, ntok0 + s, Hkv, D)
    if "k_range" in cfg:
        lo, hi = cfg["k_range"]
        kbs = np.array([[[synth.uniform_int(seed, synth.KIND_BUDGET, s_, l, 0, lo, hi)] * R for l in range(L)]
                        for s_ in range(total_steps)], dtype=np.int32)
    else:
        kbs = np.full((total_steps, L, R), cfg["k"], dtype=np.int32)
    kb = kbs[0]
    q_d = torch.from_numpy(qs.view(np.int16)).to(dev)
    kn_d = torch.from_numpy(kn.view(np.int16)).to(dev)
    vn_d = torch.from_numpy(vn.view(np.int16)).to(dev)
    kb_d = torch.from_numpy(kbs).to(dev)
    out = torch.empty((L, R, Hq, D), dtype=torch.int16, device=dev)
    lse = torch.empty((L, R, Hq), dtype=torch.float32, device=dev)
    compute, copy = torch.cuda.Stream(), torch.cuda.Stream()
    step = 0

    def run_step(stats=False):
        nonlocal step
        r_ = pool.decode_step(q_d[step], kn_d[step], vn_d[step], kb_d[step], out, lse, method=method,
                              compute=compute, copy=copy, stats=stats)
        step += 1
        return r_

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    # warm-up (the pool starts empty: step 0 recalls every selected block). The
    # first ~0.3 s of pipelined steps after the host-side setup run slower than the
    # steady state on this machine (measured), so warm-up lasts at least W steps and
    # at least --warmup-s seconds; the JSON reports the steps actually run.
    warm_stats = []
    for _ in range(min(Wm, 3)):
        warm_stats.append(run_step(stats=True))
    admission = None
    t_w = time.time()
    warm_steps = len(warm_stats)
    while warm_steps < Wm or (time.time() - t_w < args.warmup_s and warm_steps < prewarm_cap):
        run_step()
        warm_steps += 1
        if warm_steps % 8 == 0:
            torch.cuda.synchronize()
    torch.cuda.synchronize()
    assert pool.device_status() == pi.PI_OK

    if args.admission:
        # IO-adaptive admission in the steady state: one decision per window of two
        # steps from the link utilisation the window measured (recalled bytes /
        # window time / H2D peak), until three windows in a row change nothing
        decisions = []
        quiet = 0
        for _ in range(2 * args.pin_layers + 6):
            ea, eb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            ea.record(compute)
            got = [run_step(stats=True) for _ in range(2)]
            eb.record(compute)
            torch.cuda.synchronize()
            util = sum(g_["bytes"] for g_ in got) / (ea.elapsed_time(eb) / 1e3) / (h2d_peak * 1e9)
            layer_, pinned_ = pool.admission(util)
            decisions.append({"util": round(util, 3), "layer": layer_, "pinned": pinned_})
            quiet = quiet + 1 if layer_ < 0 else 0
            if quiet >= 3:
                break
        for _ in range(Wm):  # settle after the last change
            run_step()
        torch.cuda.synchronize()
        pinned_layers = [l for l in range(L) if pool.slots(0, l) > pool.slots_per_req[0]]
        admission = {"pin_layers": args.pin_layers, "pinned": pinned_layers, "decisions": decisions}
        log(f"rank {rank}: admission pinned layers {pinned_layers} after {len(decisions)} windows")

    # ---- pass A: headline, device time over K steps, no per-kernel events; the
    # device's recall counters (read after the timed region) give the blocks these
    # very steps recalled, so the link floor below is pass A's own
    barrier()
    pool.recall_totals(reset=True)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local_rank) as clocks:
        e0.record(compute)
        for _ in range(K):
            run_step()
        e1.record(compute)
        torch.cuda.synchronize()
    recalled_a, hits_a = pool.recall_totals(reset=True)
    barrier()
    elapsed = e0.elapsed_time(e1) / 1e3
    elapsed_max = reduce_max(elapsed, world, dev)
    tok_s = weak_scaling_tokens_per_s(world, R, K, elapsed_max)

    # ---- pass B: per-kernel CUDA-event durations inside the same pipelined step
    pool.set_timing(K)
    stats_b = []
    e2, e3 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e2.record(compute)
    ntok_b = []
    for _ in range(K):
        ntok_b.append(ntok0 + step + 1)
        stats_b.append(run_step(stats=True))
    e3.record(compute)
    torch.cuda.synchronize()
    timing = pool.get_timing()
    pool.set_timing(0)
    pass_b_s = e2.elapsed_time(e3) / 1e3
    assert pool.device_status() == pi.PI_OK

    BB = 2 * Hkv * B * D * 2
    recalled = sum(s["fragments"] for s in stats_b)
    selected = sum(s["selected"] for s in stats_b)
    alg = {}
    alg["gather"] = recalled * BB                                           # bytes over the host link
    alg["attention"] = selected * BB + K * L * (2 * R * Hq * D * 2 + R * Hq * 4)
    sel_bytes = 0
    for nt in ntok_b:
        nb = -(-nt // B)
        sel_bytes += L * R * (max(nb - cfg["window"], 0) * Hkv * D * 4 + Hq * D * 2 + (cfg["k"] + cfg["window"] + 1) * 4)
    alg["select"] = sel_bytes
    alg["append"] = K * L * R * (2 * Hkv * D * 2 * 3 + Hkv * D * 4 * 3)
    alg["plan"] = K * L * R * (cfg["k"] + cfg["window"]) * 4 * 4
    kernels = {}
    peaks = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json"))) if os.path.exists(
        os.path.join(ROOT, "MEASURED_PEAKS.json")) else {}
    hbm_peak = peaks.get("hbm_gbs", 6800.0)
    for k_ in KINDS:
        tm = timing[k_]
        if tm["launches"] == 0 or tm["total_ms"] <= 0:
            continue
        # launches of one kind may overlap (gathers on two copy streams): the
        # achieved rate divides by the union of their intervals, which equals the
        # sum of their durations when they do not overlap
        busy = tm.get("busy_ms") or tm["total_ms"]
        gbs = alg[k_] / (busy / 1e3) / 1e9
        bound, peak = ("h2d", h2d_peak) if k_ == "gather" else ("hbm", hbm_peak)
        kernels[k_] = {"launches": tm["launches"], "avg_us": 1e3 * tm["total_ms"] / tm["launches"],
                       "busy_us_per_launch": 1e3 * busy / tm["launches"],
                       "share": None, "bytes_per_launch": alg[k_] / tm["launches"], "achieved_gbs": gbs,
                       "bound": bound, "peak_gbs": peak, "frac": gbs / peak}
    tot_ms = sum(timing[k_]["total_ms"] for k_ in KINDS)
    for k_ in kernels:
        kernels[k_]["share"] = timing[k_]["total_ms"] / tot_ms
    dom = max(kernels, key=lambda k_: timing[k_]["total_ms"])
    dk = kernels[dom]
    traffic, traffic_note = (gather_traffic(recalled / max(timing["gather"]["launches"], 1), BB) if dom == "gather"
                             else (None, {"reason": "no traffic record for this kernel"}))
    roofline = {"kernel": dom, "bound": dk["bound"], "achieved": dk["achieved_gbs"], "peak": dk["peak_gbs"],
                "unit": "GB/s", "frac": dk["frac"], "traffic": traffic, "traffic_note": traffic_note,
                "peak_source": ("pinned host->device cudaMemcpyAsync measured in this run" if dk["bound"] == "h2d"
                                else "MEASURED_PEAKS.json hbm_gbs (measured copy)"),
                "kernels": kernels}

    # ---- pass C: end to end through the host-buffer entry point
    e2e = None
    if not args.no_e2e and not extra:
        qh = torch.from_numpy(qs.view(np.int16)).pin_memory()
        knh = torch.from_numpy(kn.view(np.int16)).pin_memory()
        vnh = torch.from_numpy(vn.view(np.int16)).pin_memory()
        kbh = torch.from_numpy(kbs).pin_memory()
        outh = torch.empty((L, R, Hq, D), dtype=torch.int16).pin_memory()
        lseh = torch.empty((L, R, Hq), dtype=torch.float32).pin_memory()
        barrier()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(K):
            pool.decode_step_host(qh[step], knh[step], vnh[step], kbh[step], outh, lseh, method=method,
                                  compute=compute, copy=copy)
            step += 1
        t_e2e = reduce_max(time.perf_counter() - t0, world, dev)
        h2d_b = L * R * Hq * D * 2 + 2 * L * R * Hkv * D * 2 + L * R * 4
        d2h_b = L * R * Hq * D * 2 + L * R * Hq * 4
        e2e = {"value": weak_scaling_tokens_per_s(world, R, K, t_e2e), "unit": "tok/s", "h2d_bytes_per_step": h2d_b,
               "d2h_bytes_per_step": d2h_b, "api": "pi_decode_step_host (pinned host buffers)"}
    assert pool.device_status() == pi.PI_OK

    # ---- pass D: attention and selection each launched alone, back to back on one
    # stream over the layers in turn (each launch reads another layer's blocks and
    # summaries, so nothing is served from L2), on the last step's selection
    torch.cuda.synchronize()
    sel_v, nsel_v, tab_v = pool.view_step()
    q_last, kb_last = q_d[step - 1], kb_d[step - 1]
    out_i = torch.empty_like(out)
    lse_i = torch.empty_like(lse)
    sel_i = torch.empty((R * pool.U, cfg["k"] + cfg["window"]), dtype=torch.int32, device=dev)
    nsel_i = torch.empty((R * pool.U,), dtype=torch.int32, device=dev)
    n_iso = max(2 * L, 16)

    host_issue_us = []

    def timed(fn):
        for i in range(L):
            fn(i)
        torch.cuda.synchronize()
        ea, eb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ea.record(compute)
        th = time.perf_counter()
        for i in range(n_iso):
            fn(i % L)
        th = time.perf_counter() - th
        eb.record(compute)
        torch.cuda.synchronize()
        host_issue_us.append(1e6 * th / n_iso)
        return ea.elapsed_time(eb) / 1e3 / n_iso

    # device pointers resolved up front, so the host issues launches faster than
    # the GPU retires them (the timing is the GPU's, not Python's)
    qp = [q_last[l].data_ptr() for l in range(L)]
    kbp = [kb_last[l].data_ptr() for l in range(L)]
    selp = [sel_v[l].data_ptr() for l in range(L)]
    tabp = [tab_v[l].data_ptr() for l in range(L)]
    nselp = [nsel_v[l].data_ptr() for l in range(L)]
    outp = [out_i[l].data_ptr() for l in range(L)]
    lsep = [lse_i[l].data_ptr() for l in range(L)]
    seli, nseli, cs_ = sel_i.data_ptr(), nsel_i.data_ptr(), compute.cuda_stream
    t_att = timed(lambda l: pool.sparse_decode(l, qp[l], selp[l], tabp[l], nselp[l], outp[l], lsep[l], stream=cs_))
    t_sel = timed(lambda l: pool.select_topk(l, qp[l], kbp[l], seli, nseli, stream=cs_))
    assert pool.device_status() == pi.PI_OK
    att_b = (int(nsel_v.sum().item()) * BB + L * (2 * R * Hq * D * 2 + R * Hq * 4)) / L
    nb_now = -(-(ntok0 + step) // B)
    sel_b = R * (max(nb_now - cfg["window"], 0) * Hkv * D * 4 + Hq * D * 2 + (cfg["k"] + cfg["window"] + 1) * 4)
    roofline["isolated"] = {
        k_: {"avg_us": 1e6 * t_, "bytes_per_launch": b_, "achieved_gbs": b_ / t_ / 1e9, "bound": "hbm",
             "peak_gbs": hbm_peak, "frac": b_ / t_ / 1e9 / hbm_peak}
        for k_, t_, b_ in (("attention", t_att, att_b), ("select", t_sel, sel_b))}
    roofline["isolated"]["attention"]["host_issue_us"] = host_issue_us[0]
    roofline["isolated"]["select"]["host_issue_us"] = host_issue_us[1]
    roofline["isolated"]["note"] = ("each kernel alone, back to back over the layers on one stream (no L2 reuse), "
                                    "CUDA events; the select launch here is the standalone one (no fused plan)")

    # ---- the other eviction policy on the same pool: flush, warm up, time K steps
    variant = None
    if not args.no_variant and fracs is None and not extra:
        other = "lru" if args.evict == "ascending" else "ascending"
        pool.flush()
        pool.set_evict(pi.PI_EVICT_LRU if other == "lru" else pi.PI_EVICT_ASCENDING)
        for _ in range(Wm):
            run_step()
        vstats = []
        torch.cuda.synchronize()
        e4, e5 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e4.record(compute)
        for _ in range(K):
            run_step()
        e5.record(compute)
        torch.cuda.synchronize()
        v_s = reduce_max(e4.elapsed_time(e5) / 1e3, world, dev)
        for _ in range(2):
            vstats.append(run_step(stats=True))
        assert pool.device_status() == pi.PI_OK
        variant = {"evict": other, "value": weak_scaling_tokens_per_s(world, R, K, v_s), "unit": "tok/s",
                   "ms_per_step": 1e3 * v_s / K,
                   "recall_blocks_per_step": sum(v["fragments"] for v in vstats) / len(vstats),
                   "note": "same pool and inputs after a flush and warm-up; not the headline"}

    # ---- CPU oracle baseline on a bounded sample (rank 0, N = 1)
    cpu = None
    cpu_all = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline and not extra:
        # the live host store has the appended tokens of the GPU steps; the oracle
        # sample starts from a fresh prefill region of the same seed instead
        cpu = cpu_baseline(cfg, seed, qs, max_blocks, None, budget_s=args.cpu_budget)
        if args.cpu_all_cores:
            cpu_all = cpu_baseline_all_cores(cfg, seed, max_blocks, budget_s=min(args.cpu_budget, 10.0))

    recall_gbs = kernels.get("gather", {}).get("achieved_gbs")
    line = {
        "metric": METRIC, "value": tok_s, "unit": "tok/s", "n_gpus": world, "steps": K, "warmup": Wm,
        "ms_per_step": 1e3 * elapsed_max / K, "higher_is_better": True, "warmup_steps_run": warm_steps, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic (seeded; shapes of the pages' Llama-3 long-context workloads)",
        "config": {"workload": cfg["workload"], "layers": L, "batch": R, "hq": Hq, "hkv": Hkv, "head_dim": D,
                   "block_tokens": B, "context": ntok0, "top_k": cfg["k"], "window": cfg["window"],
                   "pool_slots": cfg["pool_slots"] or (f"per request {min(slots_per_req)}..{max(slots_per_req)}"
                                                       if slots_per_req else None),
                   "recall": args.method, "evict": args.evict, "host_layers": host_layers,
                   "select": (args.select if args.select == "shared"
                              else f"consensus (lambda {args.consensus_lambda})"),
                   "select_ahead": ("library default" if args.select_ahead < 0 else (args.select_ahead or "all")),
                   "streams": 2 if args.two_streams else 3,
                   "admission": admission,
                   "copy_streams": args.copy_streams,
                   "select_gather": ((f"fused, {args.fused_ctas or 'a quarter of the SMs'} CTAs per launch")
                                     if args.fused else "separate launches"),
                   "schedule": ("queries known up front, selections run ahead" if args.schedule == "ahead" else
                                f"dependent queries, {args.groups} interleaved request group(s)"),
                   "gather_ctas": args.gather_ctas or "default",
                   "gather_depth": args.gather_depth or 8, "gather_placement": args.gather_placement,
                   "attn_splits": args.attn_splits or "one wave",
                   "attn_merge": "cluster" if args.attn_cluster else "global", "host_alloc": ["cudaHostAlloc", "mmap+THP+register"][args.host_alloc],
                   "parallelism": f"replicas{world}" if world > 1 else "single",
                   "l2": "inputs larger than L2 (host store and pool far exceed 129 MB)"},
        "recall": {"gbs": recall_gbs, "h2d_peak_gbs": h2d_peak,
                   "frac_of_h2d_peak": (recall_gbs / h2d_peak) if recall_gbs else None,
                   "bytes_per_step": recalled * BB / K, "blocks_per_step": recalled / K,
                   "selected_per_step": selected / K,
                   "pipelined_link_gbs": recalled * BB / pass_b_s / 1e9,
                   # the timed steps themselves (pass A): their recalled bytes over the
                   # pinned H2D peak is the least time the host link allows per step
                   "pass_a": {"blocks_per_step": recalled_a / K, "hits_per_step": hits_a / K,
                              "bytes_per_step": recalled_a * BB / K,
                              "link_floor_ms_per_step": 1e3 * recalled_a * BB / K / (h2d_peak * 1e9),
                              "link_gbs": recalled_a * BB / elapsed_max / 1e9,
                              "frac_of_link_floor": (recalled_a * BB / (h2d_peak * 1e9)) / elapsed_max}},
        "roofline": roofline,
        "evict_variant": variant,
        "cpu_baseline": cpu,
        "cpu_baseline_all_cores": cpu_all,
        "e2e": e2e,
        # kernels of the library per step, counted by the per-kernel timing of pass B
        # (same steps: append, selection with the fused plan, gather, attention per layer)
        "gpu_launches": int(round(sum(timing[k_]["launches"] for k_ in KINDS) / max(K, 1))) * K,
        "clocks": clocks.summary(),
        "kernel_timing": "per-kernel CUDA events over a second run of K pipelined steps (pass B)",
        "pass_b_tok_s": world * R * K / pass_b_s,
        "warmup_recall_blocks": [w["fragments"] for w in warm_stats],
        "numa": numa,
        "prefill_summaries": prefill,
    }
    pool.close()
    return line


def run_fragmentation_sweep(args):
    """Block size 16/32/64/128 at an equal 2048-token budget per (request, layer):
    shared top-k vs per-KV-head top-k, 0 % resident (pool flushed every step), each
    recall arm; recall GB/s and transfer counts per step. Emits one JSON line per
    (block size, selection, arm) and a final summary line."""
    import torch

    import synth
    import sparse_kv_cache_block_gb300 as pi

    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    pi.build()
    pi.load()
    L, R, Hq, Hkv, D, N = 32, 64, 32, 8, 128, 32768
    if args.layers:
        L = args.layers
    if args.batch:
        R = args.batch
    budget_tokens = 2048
    host_layers = max(1, min(L, args.sweep_host_layers))
    h2d_peak = measure_h2d_peak(torch, dev)
    methods = {"uva": pi.PI_RECALL_UVA, "memcpy": pi.PI_RECALL_MEMCPY, "staged": pi.PI_RECALL_STAGED}
    arms = [m for m in args.sweep_methods.split(",") if m]
    rows = []
    s_ = torch.cuda.Stream()
    for B in (int(b) for b in args.sweep_blocks.split(",")):
        k = budget_tokens // B
        max_blocks = N // B + 1
        qs = synth.q_ar1(args.seed, L, R, Hq, D, 2, 0.9)
        for mode_name, mode in (("shared", pi.PI_SHARED), ("headwise", pi.PI_HEADWISE)):
            pool = pi.Pool(L, R, Hq, Hkv, D, B, max_blocks, k, k, 0, select_mode=mode,
                           host_layers=(host_layers if host_layers < L else 0), gather_ctas=args.gather_ctas)
            t0 = time.time()
            for hl in range(host_layers):
                for r in range(R):
                    synth.fill_kv(pool.host_kv_ptr(hl, r), args.seed, hl, r, N, max_blocks, Hkv, B, D, 0.0, 0.0)
            for l in range(L):
                pool.update_summaries(l, [N] * R)
            torch.cuda.synchronize()
            log(f"B={B} {mode_name}: host store {host_layers * R * pool.region_bytes / 2**30:.1f} GiB ready in "
                f"{time.time() - t0:.1f} s")
            U = Hkv if mode == pi.PI_HEADWISE else 1
            sel = torch.empty((L, R * U, k), dtype=torch.int32, device=dev)
            nsel = torch.empty((L, R * U), dtype=torch.int32, device=dev)
            table = torch.empty_like(sel)
            kb = torch.full((R,), k, dtype=torch.int32, device=dev)
            q_d = torch.from_numpy(qs.view(np.int16)).to(dev)
            with torch.cuda.stream(s_):
                for l in range(L):
                    pool.select_topk(l, q_d[0, l], kb, sel[l], nsel[l], stream=s_)
            torch.cuda.synchronize()
            for arm in arms:
                res = None
                for rep in range(2):  # rep 0 warms up
                    pool.flush(-1, stream=s_)
                    torch.cuda.synchronize()
                    tot = {"bytes": 0, "fragments": 0, "runs": 0, "api_calls": 0, "host_wait_ms": 0.0,
                           "cpu_gather_ms": 0.0}
                    ms = 0.0
                    for l in range(L):
                        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                        h0 = time.perf_counter()
                        e0.record(s_)
                        st = pool.recall(l, sel[l], nsel[l], table[l], method=methods[arm], stats=True, stream=s_)
                        e1.record(s_)
                        e1.synchronize()
                        wall = time.perf_counter() - h0
                        # the memcpy and staged arms block on the host for part of the call:
                        # count the whole call (host wall clock) for them, device time for UVA
                        ms += e0.elapsed_time(e1) if arm == "uva" else 1e3 * wall
                        for kk in tot:
                            tot[kk] += st[kk]
                    res = (ms, tot)
                ms, tot = res
                assert pool.device_status() == pi.PI_OK
                row = {"sweep": "fragmentation", "block_tokens": B, "k": k, "selection": mode_name, "recall": arm,
                       "layers": L, "batch": R, "bytes_per_step": tot["bytes"], "fragments_per_step": tot["fragments"],
                       "runs_per_step": tot["runs"], "api_calls_per_step": tot["api_calls"],
                       "recall_ms_per_step": ms, "recall_gbs": tot["bytes"] / (ms / 1e3) / 1e9,
                       "h2d_peak_gbs": h2d_peak, "frac_of_h2d_peak": tot["bytes"] / (ms / 1e3) / 1e9 / h2d_peak,
                       "host_wait_ms": tot["host_wait_ms"], "cpu_gather_ms": tot["cpu_gather_ms"],
                       "host_layers": host_layers}
                rows.append(row)
                print(json.dumps(row), flush=True)
            pool.close()
            del sel, nsel, table
            torch.cuda.empty_cache()
    return rows


def run_mass_diagnostic(args):
    """Attention mass each query head keeps under the shared, the consensus and
    the per-KV-head selection at one budget (guide, "SoloHead Sparse Selection",
    "2. High Attention Mass Preservation"), with the blocks each selection moves
    and the mass kernel's host-link rate. Llama-3-8B shape at 32768 tokens
    (batch 8, top-32 + 2 recent, 5 % heavy-hitter blocks shifted by 2 u_g), AR(1)
    queries over a few steps, two query recipes: "random" (the benchmark's own
    queries: attention close to uniform) and "aligned" (each head's query plus
    1.5 sqrt(D) u_g, its group's heavy-hitter direction, so that every head
    attends to the heavy blocks: the premise the guide states for SoloHead).
    Synthetic keys: the comparison between the rankings is the result, not the
    absolute mass. One JSON line."""
    import torch

    import synth
    import sparse_kv_cache_block_gb300 as pi

    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    pi.build()
    pi.load()
    L = args.layers or 2
    R = args.batch or 8
    Hq, Hkv, D, B, N, k, W, steps = 32, 8, 128, 64, 32768, 32, 2, 4
    G, nb, cap = Hq // Hkv, N // B, k + W
    qs = synth.q_ar1(args.seed, L, R, Hq, D, steps, 0.9)
    qa = synth.bf16_to_f32(qs).astype(np.float64)
    for l in range(L):
        for r in range(R):
            for g in range(Hkv):
                qa[:, l, r, g * G:(g + 1) * G] += 1.5 * math.sqrt(D) * synth.direction(args.seed, l, r, g, D)
    recipes = {"random": qs, "aligned": synth.f32_to_bf16(qa.astype(np.float32))}
    kb = torch.full((R,), k, dtype=torch.int32, device=dev)
    pools = {}
    for name, mode in (("one_set", pi.PI_SHARED), ("headwise", pi.PI_HEADWISE)):
        pool = pi.Pool(L, R, Hq, Hkv, D, B, nb + 1, cap, k, W, select_mode=mode)
        for l in range(L):
            for r in range(R):
                synth.fill_kv(pool.host_kv_ptr(l, r), args.seed, l, r, N, nb + 1, Hkv, B, D, 0.05, 2.0)
            pool.update_summaries(l, [N] * R)
        pools[name] = pool
    torch.cuda.synchronize()
    rankings = (("shared", "one_set", pi.PI_SHARED, 1), ("consensus", "one_set", pi.PI_CONSENSUS, 1),
                ("headwise", "headwise", pi.PI_HEADWISE, Hkv))
    mass_ms = []
    out = {}
    for recipe, qbits in recipes.items():
        q_d = torch.from_numpy(np.ascontiguousarray(qbits).view(np.int16)).to(dev)
        masses = {name: [] for name, *_ in rankings}
        union_blocks = []
        for st in range(steps):
            for l in range(L):
                for name, pname, mode, U in rankings:
                    pool = pools[pname]
                    sel = torch.empty((R * U, cap), dtype=torch.int32, device=dev)
                    nsel = torch.empty((R * U,), dtype=torch.int32, device=dev)
                    mass = torch.empty((R, Hq), dtype=torch.float32, device=dev)
                    pool.select_topk(l, q_d[st, l], kb, sel, nsel, mode=mode)
                    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    e0.record()
                    pool.attention_mass(l, q_d[st, l], sel, nsel, mass, per_head=U > 1)
                    e1.record()
                    e1.synchronize()
                    mass_ms.append(e0.elapsed_time(e1))
                    masses[name].append(mass.cpu().numpy())
                    if U > 1:
                        sh, nh = sel.cpu().numpy().reshape(R, U, cap), nsel.cpu().numpy().reshape(R, U)
                        for r in range(R):
                            union_blocks.append(len(set(int(b) for g in range(U) for b in sh[r, g, :nh[r, g]])))
        stats = {}
        for name in masses:
            m = np.stack(masses[name])
            stats[name] = {"mean": float(m.mean()), "min": float(m.min()), "p01": float(np.quantile(m, 0.01))}
        out[recipe] = {"mass": stats,
                       "shared_over_headwise": stats["shared"]["mean"] / stats["headwise"]["mean"],
                       "consensus_over_headwise": stats["consensus"]["mean"] / stats["headwise"]["mean"],
                       "headwise_union_blocks": float(np.mean(union_blocks)),
                       "whole_block_volume_saved_vs_headwise_union": 1.0 - cap / float(np.mean(union_blocks))}
    for pool in pools.values():
        assert pool.device_status() == pi.PI_OK
        pool.close()
    mass_bytes = R * Hkv * N * D * 2
    warm = mass_ms[len(rankings):]  # the first calls allocate scratch and warm the mapping
    row = {"diagnostic": "attention_mass", "workload": "llama3-8b-shape", "layers": L, "batch": R, "context": N,
           "block_tokens": B, "k": k, "window": W, "steps": steps, "heavy_frac": 0.05, "data": "synthetic",
           "uniform_share": cap / nb, "shared_blocks": cap, "headwise_fragments": cap * Hkv, "recipes": out,
           "mass_kernel": {"bytes_per_call": mass_bytes, "ms_per_call": float(np.median(warm)),
                           "host_link_gbs": mass_bytes / (float(np.median(warm)) / 1e3) / 1e9}}
    print(json.dumps(row), flush=True)
    return row


def run_reference(args, cfg):
    """The CPU oracle as it stands, on a bounded sample of the workload per step."""
    import synth
    L, R = cfg["layers"], cfg["batch"]
    K, Wm = args.steps, args.warmup
    total = Wm + K + 1
    max_blocks = -(-(cfg["ntok"] + total) // cfg["block_tokens"]) + 1
    qs = synth.q_ar1(args.seed, L, R, cfg["hq"], cfg["head_dim"], total, cfg["rho"])
    rng = np.random.default_rng(args.seed + 17)
    all_units = [(r, l) for r in range(R) for l in range(L)]
    n_units = min(args.ref_units, len(all_units))
    pick = [all_units[i] for i in sorted(rng.choice(len(all_units), size=n_units, replace=False))]
    samp = OracleSample(cfg, args.seed, pick, max_blocks)
    for s in range(Wm):
        samp.step(qs[s], s)
    secs = 0.0
    done = 0
    for s in range(Wm, Wm + K):
        d, t = samp.step(qs[s], s)
        done += d
        secs += t
    tok_s = 1.0 / (secs / done * L)
    sample = (f"{n_units} (request, layer) units per step x {K} steps, single-threaded oracle; "
              f"tokens/s = 1 / (s per unit x {L} layers)")
    return {"impl": "reference", "metric": METRIC, "value": tok_s, "unit": "tok/s", "n_gpus": 1, "steps": K,
            "warmup": Wm, "ms_per_step": 1e3 * secs / K, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": cfg["workload"], "layers": L, "batch": R},
            "cpu_baseline": {"value": tok_s, "unit": "tok/s", "cores": 1, "kind": "oracle", "sample": sample},
            "e2e": {"value": tok_s, "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def extra_summary(lx):
    """The figures of an additional configuration kept in the headline line."""
    roof = lx["roofline"]
    iso = roof.get("isolated", {})
    return {"workload": lx["config"]["workload"], "value": lx["value"], "unit": lx["unit"],
            "ms_per_step": lx["ms_per_step"], "steps": lx["steps"], "warmup_steps_run": lx["warmup_steps_run"],
            "recall": lx["recall"], "clocks": lx["clocks"], "gpu_launches": lx["gpu_launches"],
            "prefill_summaries": lx["prefill_summaries"],
            "roofline": {"kernel": roof["kernel"], "bound": roof["bound"], "achieved": roof["achieved"],
                         "peak": roof["peak"], "unit": roof["unit"], "frac": roof["frac"], "traffic": roof["traffic"],
                         "kernels": {k_: {kk: v_[kk] for kk in ("avg_us", "busy_us_per_launch", "share", "frac")}
                                     for k_, v_ in roof["kernels"].items()},
                         "isolated": {k_: {kk: v_[kk] for kk in ("avg_us", "bytes_per_launch", "achieved_gbs", "frac")}
                                      for k_, v_ in iso.items() if isinstance(v_, dict)}}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--warmup-s", type=float, default=1.5,
                    help="warm-up also lasts at least this many seconds of pipelined steps")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default="c3", choices=sorted(CONFIGS),
                    help="headline workload (default: the variable-recall stress, the largest single-GPU one)")
    ap.add_argument("--extra-configs", default="c2,c4",
                    help="workloads also run after the headline and reported under extra_configs of the same line "
                         "(no e2e pass, CPU legs or eviction variant); empty: none")
    ap.add_argument("--method", default="uva", choices=["uva", "memcpy", "staged"])
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--gather-ctas", type=int, default=0)
    ap.add_argument("--gather-depth", type=int, default=0)
    ap.add_argument("--gather-placement", default="exclusive", choices=["exclusive", "shared"],
                    help="gather on a quarter of the SMs with 1024-thread CTAs (library default) or one CTA per SM")
    ap.add_argument("--evict", default="ascending", choices=["ascending", "lru"],
                    help="pool eviction policy of the headline passes")
    ap.add_argument("--no-variant", action="store_true", help="skip the extra pass under the other eviction policy")
    ap.add_argument("--two-streams", action="store_true",
                    help="attention on the compute stream (default: on the pool's own stream, so selection runs "
                         "ahead and consecutive steps overlap)")
    ap.add_argument("--select-ahead", type=int, default=-1,
                    help="layers selected ahead of attention in the step (0 = all; -1 = library default)")
    ap.add_argument("--host-alloc", type=int, default=0, choices=[0, 1],
                    help="0 cudaHostAlloc, 1 mmap + transparent huge pages + cudaHostRegister")
    ap.add_argument("--attn-splits", type=int, default=0,
                    help="attention CTAs per (request, KV head); 0 = one wave at the kernel's occupancy")
    ap.add_argument("--schedule", default="ahead", choices=["ahead", "dependent"],
                    help="dependent: a request's selection of layer l+1 waits for its attention of layer l")
    ap.add_argument("--groups", type=int, default=2, help="request groups interleaved under --schedule dependent")
    ap.add_argument("--fused", action="store_true",
                    help="selection, plan and gather of a layer as one launch on the copy stream")
    ap.add_argument("--fused-ctas", type=int, default=0, help="CTAs of a fused launch (0: a quarter of the SMs)")
    ap.add_argument("--copy-streams", type=int, default=2, choices=[1, 2],
                    help="2 (default): odd layers' gathers on a second copy stream; 1: one copy stream")
    ap.add_argument("--admission", action="store_true",
                    help="IO-adaptive admission during warm-up: pin layers whole in HBM while the link is saturated")
    ap.add_argument("--pin-layers", type=int, default=8, help="layers with room reserved for pinning (admission)")
    ap.add_argument("--select", default="shared", choices=["shared", "consensus"],
                    help="block ranking: mean-key shared score, or the consensus score (max + lambda x mean per group)")
    ap.add_argument("--consensus-lambda", type=float, default=0.5)
    ap.add_argument("--attn-cluster", type=int, default=1, choices=[0, 1],
                    help="1: a unit's 2..8 attention splits merge through DSMEM in one cluster; 0: global merge")
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--ref-units", type=int, default=4)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-all-cores", type=int, default=1, choices=[0, 1],
                    help="also time the oracle with one process per host core (reported separately)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--layers", type=int, default=0, help="override the layer count (small profiling cases)")
    ap.add_argument("--batch", type=int, default=0, help="override the batch (small profiling cases)")
    ap.add_argument("--sweep", default="", choices=["", "fragmentation", "mass"],
                    help="fragmentation: block-size sweep of shared vs head-wise recall; mass: attention mass "
                         "kept by each ranking (neither is the headline line)")
    ap.add_argument("--sweep-blocks", default="16,32,64,128")
    ap.add_argument("--sweep-methods", default="uva,memcpy,staged")
    ap.add_argument("--sweep-host-layers", type=int, default=2)
    args = ap.parse_args()
    if args.warmup < 3:
        log("warm-up raised to 3 steps (minimum)")
        args.warmup = 3
    cfg = dict(CONFIGS[args.config])
    if args.layers:
        cfg["layers"] = args.layers
        cfg["workload"] += f" [layers overridden to {args.layers}]"
    if args.batch:
        cfg["batch"] = args.batch
        cfg["workload"] += f" [batch overridden to {args.batch}]"
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.sweep == "fragmentation":
        rows = run_fragmentation_sweep(args)
        print(json.dumps({"sweep": "fragmentation", "rows": len(rows)}), flush=True)
        return
    if args.sweep == "mass":
        run_mass_diagnostic(args)
        return
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args, cfg)), flush=True)
        return
    if world > 1:
        import torch
        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group("nccl")
    line = run_ours(args, cfg, rank, world, local_rank)
    extras = {}
    for name in [c for c in args.extra_configs.split(",") if c and c != args.config]:
        import torch
        torch.cuda.empty_cache()
        cx = dict(CONFIGS[name])
        if args.layers:
            cx["layers"] = args.layers
        if args.batch:
            cx["batch"] = args.batch
        lx = run_ours(args, cx, rank, world, local_rank, extra=True)
        extras[name] = extra_summary(lx)
    if extras:
        line["extra_configs"] = extras
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
