"""Test-side drivers: build seeded workloads with ``synth`` and run the oracle
model next to the CUDA library. Inputs for both sides come from ``synth``
only; expected values come from ``oracle`` only."""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

import oracle
import synth


@dataclass
class Workload:
    layers: int
    batch: int
    hq: int
    hkv: int
    head_dim: int
    block_tokens: int
    ntok: list                 # prefill tokens per request
    k: int                     # top-k budget (k_max)
    window: int
    pool_slots: int
    steps: int = 1
    rho: float = 0.9
    heavy_frac: float = 0.0
    heavy_shift: float = 2.0
    seed: int = 0
    host_layers: int = 0
    select_mode: int = 0       # 0 shared, 1 head-wise, 2 consensus (one set per request)
    lam: float = 0.5           # consensus: weight of the group mean
    max_blocks: int = 0        # 0: enough for the prefill plus `steps` appended tokens
    slots_per_req: list | None = None
    evict_policy: int = 0      # 0 lowest free slot first, 1 least recently selected first

    def __post_init__(self):
        if self.max_blocks == 0:
            self.max_blocks = max(-(-(n + self.steps) // self.block_tokens) for n in self.ntok) + 1
        if self.host_layers == 0:
            self.host_layers = self.layers

    @property
    def hl(self):
        return self.host_layers

    def host_layer(self, l):
        return l % self.host_layers


def fill_pool_host(pool, w: Workload):
    """Fill the pinned host store through the synth generator (one region per host layer)."""
    for hl in range(w.hl):
        for r in range(w.batch):
            synth.fill_kv(pool.host_kv_ptr(hl, r), w.seed, hl, r, w.ntok[r], w.max_blocks, w.hkv, w.block_tokens,
                          w.head_dim, w.heavy_frac, w.heavy_shift)


def regions(w: Workload):
    """Independent host copies of every (host layer, request) region for the oracle."""
    return {(hl, r): synth.kv_region(w.seed, hl, r, w.ntok[r], w.max_blocks, w.hkv, w.block_tokens, w.head_dim,
                                     w.heavy_frac, w.heavy_shift)
            for hl in range(w.hl) for r in range(w.batch)}


def queries(w: Workload, steps: int | None = None):
    """[steps][L][R][Hq][D] bf16 bits (AR(1) across steps)."""
    return synth.q_ar1(w.seed, w.layers, w.batch, w.hq, w.head_dim, steps or w.steps, w.rho)


def new_tokens(w: Workload, step: int):
    """k_new, v_new [L][R][Hkv][D] of decode step `step` (token position ntok[r] + step).
    Aliased layers carry the same token (same host layer)."""
    k = np.empty((w.layers, w.batch, w.hkv, w.head_dim), dtype=np.uint16)
    v = np.empty_like(k)
    for l in range(w.layers):
        for r in range(w.batch):
            k[l, r], v[l, r] = synth.token_kv(w.seed, w.host_layer(l), r, w.ntok[r] + step, w.hkv, w.head_dim)
    return k, v


class OracleModel:
    """The oracle's own state for a multi-step decode: host regions (its copy),
    summaries, slot maps and token counts per (request, layer)."""

    def __init__(self, w: Workload, regs=None):
        self.w = w
        self.reg = regs if regs is not None else regions(w)
        self.ntok = {(r, l): w.ntok[r] for r in range(w.batch) for l in range(w.layers)}
        U = w.hkv if w.select_mode == 1 else 1
        self.U = U
        self.kmean = {}
        for r in range(w.batch):
            for l in range(w.layers):
                km = np.zeros((w.max_blocks, w.hkv, w.head_dim), dtype=np.float32)
                nb = -(-w.ntok[r] // w.block_tokens)
                km[:nb] = oracle.region_summaries(self.reg[(w.host_layer(l), r)], w.ntok[r])
                self.kmean[(r, l)] = km
        P = w.slots_per_req or [w.pool_slots] * w.batch
        self.P = P
        self.sob = {(r, l, u): np.full(w.max_blocks, -1, dtype=np.int32)
                    for r in range(w.batch) for l in range(w.layers) for u in range(U)}
        self.bos = {(r, l, u): np.full(P[r], -1, dtype=np.int32)
                    for r in range(w.batch) for l in range(w.layers) for u in range(U)}
        self.stamp = {(r, l, u): np.full(P[r], -1, dtype=np.int32)
                      for r in range(w.batch) for l in range(w.layers) for u in range(U)}
        self.epoch = {(r, l, u): 0 for r in range(w.batch) for l in range(w.layers) for u in range(U)}
        self.pinned = set()  # layers held whole in HBM

    def preload(self, l, r, blocks):
        for s, b in enumerate(blocks):
            self.sob[(r, l, 0)][b] = s
            self.bos[(r, l, 0)][s] = b
            self.stamp[(r, l, 0)][s] = 0

    def pin(self, l, capacity):
        """Layer l held whole in HBM: every request's slot list grows to `capacity`."""
        self.pinned.add(l)
        for key in self.bos:
            if key[1] == l and len(self.bos[key]) < capacity:
                extra = capacity - len(self.bos[key])
                self.bos[key] = np.concatenate([self.bos[key], np.full(extra, -1, dtype=np.int32)])
                self.stamp[key] = np.concatenate([self.stamp[key], np.full(extra, -1, dtype=np.int32)])

    def unpin(self, l):
        """Layer l back to P_r slots: blocks held beyond them leave the maps."""
        self.pinned.discard(l)
        for key in list(self.bos):
            if key[1] != l:
                continue
            P = self.P[key[0]]
            for s in range(P, len(self.bos[key])):
                b = self.bos[key][s]
                if b >= 0:
                    self.sob[key][b] = -1
            self.bos[key] = self.bos[key][:P].copy()
            self.stamp[key] = self.stamp[key][:P].copy()

    def flush(self):
        for key in self.sob:
            self.sob[key][:] = -1
            self.bos[key][:] = -1
            self.stamp[key][:] = -1
            self.epoch[key] = 0

    def _plan(self, sel, r, l, u):
        key = (r, l, u)
        if self.w.evict_policy == 1:
            self.epoch[key] += 1
            return oracle.recall_plan_lru(sel, self.sob[key], self.bos[key], self.stamp[key], self.epoch[key])
        return oracle.recall_plan(sel, self.sob[key], self.bos[key], empty_first=l in self.pinned)

    def append(self, l, k_new, v_new):
        w = self.w
        for r in range(w.batch):
            t = self.ntok[(r, l)]
            b, tp = divmod(t, w.block_tokens)
            reg = self.reg[(w.host_layer(l), r)]
            reg[b, :, 0, tp] = k_new[r]
            reg[b, :, 1, tp] = v_new[r]
            self.ntok[(r, l)] = t + 1
            self.kmean[(r, l)][b] = oracle.block_summary(reg[b], tp + 1)

    def nb(self, r, l):
        return -(-self.ntok[(r, l)] // self.w.block_tokens)

    def select(self, l, q, kreq):
        """q [R][Hq][D]; kreq [R]. Shared: list of arrays; head-wise: list of lists."""
        w = self.w
        out = []
        for r in range(w.batch):
            nb = self.nb(r, l)
            k = max(0, min(int(kreq[r]), w.k))
            km = self.kmean[(r, l)][:nb]
            if w.select_mode == 2:
                out.append(oracle.select_consensus(q[r], km, k, w.window, w.lam))
            elif self.U == 1:
                out.append(oracle.select_shared(q[r], km, k, w.window))
            else:
                out.append(oracle.select_headwise(q[r], km, k, w.window))
        return out

    def recall(self, l, sels):
        """Returns tables: shared [R] arrays, head-wise [R][Hkv] arrays."""
        tables = []
        for r, s in enumerate(sels):
            if self.U == 1:
                res = self._plan(s, r, l, 0)
                assert res is not None
                tables.append(res[0])
            else:
                tt = []
                for g in range(self.U):
                    res = self._plan(s[g], r, l, g)
                    assert res is not None
                    tt.append(res[0])
                tables.append(tt)
        return tables

    def attention(self, l, q, sels, want_logits=False):
        w = self.w
        outs, lses, lgs = [], [], []
        for r in range(w.batch):
            o, ls, lg = oracle.attention(q[r], self.reg[(w.host_layer(l), r)], sels[r], self.ntok[(r, l)], w.hkv,
                                         want_logits)
            outs.append(o)
            lses.append(ls)
            lgs.append(lg)
        return np.stack(outs), np.stack(lses), lgs


def bf16_to_f32(x):
    return synth.bf16_to_f32(np.asarray(x, dtype=np.uint16))


def padded(sel_list, cap, fill=-1):
    a = np.full((len(sel_list), cap), fill, dtype=np.int32)
    for i, s in enumerate(sel_list):
        a[i, : len(s)] = s
    return a


OUT_ATOL = 2e-2     # bf16 outputs, max abs error
LSE_RTOL = 1e-3     # fp32 log-sum-exp, relative
LOGIT_RTOL = 1e-3   # fp32 logits, relative to max(|z|, 1)
