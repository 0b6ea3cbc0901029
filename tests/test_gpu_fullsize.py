"""Full-size parity in the benchmark's launch configuration.

Each workload runs pipelined decode steps through pi_decode_step exactly as
bench.py launches it (compute + copy streams, UVA gather). Sampled (request,
layer) units are checked against the oracle element by element; properties
that hold at any size (selection size, table validity and uniqueness, map
inverses, finite outputs) are checked on every unit.

Workloads:
* Llama-3-8B shape: 32 layers, batch 8, 32 q / 8 KV heads, d 128, 32768 tokens
  in blocks of 64, top-32 + 2 recent, 128-slot pool, 5 % heavy-hitter blocks,
  AR(1) rho 0.9 queries.
* Llama-3-70B slice: 8 layers, batch 16, 64 q / 8 KV heads, 131072 tokens,
  top-64 + 4 recent, 205-slot pool (10 % of blocks).
* Variable-recall stress: 8B shape, batch 32, 65536 tokens, top-k drawn per
  (layer, step) from 16..128 + 2 recent, per-request resident fraction 10..60 %
  (pool = max(fraction x blocks, 130), preloaded), AR(1) rho 0.8; the host store
  holds 4 layers and layer l reads host layer l % 4 (host capacity).
"""
import math

import numpy as np
import pytest

import oracle
import synth
from _helpers import LSE_RTOL, OUT_ATOL, bf16_to_f32

torch = pytest.importorskip("torch")
pi = pytest.importorskip("sparse_kv_cache_block_gb300")

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

SHAPES = {
    "llama8b_32k": dict(L=32, R=8, HQ=32, HKV=8, D=128, B=64, NTOK=32768, K=32, W=2, P=128, RHO=0.9, HEAVY=0.05,
                        STEPS=3, SAMPLE=[(0, 0), (3, 7), (7, 31), (5, 16), (1, 23)], HOST_LAYERS=0),
    "llama70b_slice_128k": dict(L=8, R=16, HQ=64, HKV=8, D=128, B=64, NTOK=131072, K=64, W=4, P=205, RHO=0.9,
                                HEAVY=0.0, STEPS=2, SAMPLE=[(0, 0), (15, 7), (9, 3)], HOST_LAYERS=0),
    "variable_recall_64k": dict(L=32, R=32, HQ=32, HKV=8, D=128, B=64, NTOK=65536, K=128, W=2, P=0, RHO=0.8,
                                HEAVY=0.05, STEPS=3, SAMPLE=[(0, 0), (31, 13), (17, 30)], HOST_LAYERS=4,
                                K_RANGE=(16, 128), FRAC_RANGE=(0.10, 0.60)),
}
SEED = 0


class UnitOracle:
    """Oracle state of one (request, layer): its own copy of the host region."""

    def __init__(self, c, r, l, max_blocks, P, preload=None):
        self.c, self.r, self.l = c, r, l
        hl = l % (c["HOST_LAYERS"] or c["L"])
        self.reg = synth.kv_region(SEED, hl, r, c["NTOK"], max_blocks, c["HKV"], c["B"], c["D"], c["HEAVY"], 2.0)
        self.ntok = c["NTOK"]
        self.kmean = np.zeros((max_blocks, c["HKV"], c["D"]), dtype=np.float32)
        nb = -(-c["NTOK"] // c["B"])
        self.kmean[:nb] = oracle.region_summaries(self.reg, c["NTOK"])
        self.sob = np.full(max_blocks, -1, dtype=np.int32)
        self.bos = np.full(P, -1, dtype=np.int32)
        if preload is not None:
            for s, b in enumerate(preload):
                self.sob[b] = s
                self.bos[s] = b

    def step(self, q, k_new, v_new, k):
        c = self.c
        b, tp = divmod(self.ntok, c["B"])
        self.reg[b, :, 0, tp] = k_new
        self.reg[b, :, 1, tp] = v_new
        self.ntok += 1
        self.kmean[b] = oracle.block_summary(self.reg[b], tp + 1)
        nb = -(-self.ntok // c["B"])
        sel = oracle.select_shared(q, self.kmean[:nb], k, c["W"])
        table, _, _, _ = oracle.recall_plan(sel, self.sob, self.bos)
        out, lse, _ = oracle.attention(q, self.reg, sel, self.ntok, c["HKV"])
        return sel, table, out, lse


@pytest.mark.parametrize("name", list(SHAPES))
def test_full_size_sampled_parity(name):
    c = SHAPES[name]
    pi.build()
    L, R, HKV, D, B, NTOK = c["L"], c["R"], c["HKV"], c["D"], c["B"], c["NTOK"]
    HL = c["HOST_LAYERS"] or L
    max_blocks = -(-(NTOK + c["STEPS"]) // B) + 1
    nb0 = -(-NTOK // B)
    slots = None
    if "FRAC_RANGE" in c:
        lo, hi = c["FRAC_RANGE"]
        fracs = [synth.uniform_real(SEED, synth.KIND_FRAC, r, 0, 0, lo, hi) for r in range(R)]
        slots = [max(int(math.ceil(f * nb0)), c["K"] + c["W"]) for f in fracs]
    P_of = (lambda r: slots[r]) if slots else (lambda r: c["P"])
    with pi.Pool(L, R, c["HQ"], HKV, D, B, max_blocks, c["P"] or c["K"] + c["W"], c["K"], c["W"],
                 host_layers=(HL if HL < L else 0), pool_slots_per_req=slots) as pool:
        for hl in range(HL):
            for r in range(R):
                synth.fill_kv(pool.host_kv_ptr(hl, r), SEED, hl, r, NTOK, max_blocks, HKV, B, D, c["HEAVY"], 2.0)
        for l in range(L):
            pool.update_summaries(l, [NTOK] * R)
        pre = {}
        if slots:
            for l in range(L):
                for r in range(R):
                    pre[(r, l)] = synth.sample_sorted(SEED, synth.KIND_RESIDENT, l, r, nb0, int(round(fracs[r] * nb0)))
                    pool.preload(l, r, pre[(r, l)])
        torch.cuda.synchronize()
        units = {(r, l): UnitOracle(c, r, l, max_blocks, P_of(r), pre.get((r, l))) for (r, l) in c["SAMPLE"]}
        qs = synth.q_ar1(SEED, L, R, c["HQ"], D, c["STEPS"], c["RHO"])
        compute, copy = torch.cuda.Stream(), torch.cuda.Stream()
        for s in range(c["STEPS"]):
            if "K_RANGE" in c:
                lo, hi = c["K_RANGE"]
                kbud = np.array([[synth.uniform_int(SEED, synth.KIND_BUDGET, s, l, 0, lo, hi)] * R for l in range(L)],
                                dtype=np.int32)
            else:
                kbud = np.full((L, R), c["K"], dtype=np.int32)
            kn = np.empty((L, R, HKV, D), dtype=np.uint16)
            vn = np.empty_like(kn)
            for l in range(L):
                for r in range(R):
                    kn[l, r], vn[l, r] = synth.token_kv(SEED, l % HL, r, NTOK + s, HKV, D)
            out = torch.empty((L, R, c["HQ"], D), dtype=torch.int16, device="cuda")
            lse = torch.empty((L, R, c["HQ"]), dtype=torch.float32, device="cuda")
            pool.decode_step(torch.from_numpy(qs[s].view(np.int16)).cuda(), torch.from_numpy(kn.view(np.int16)).cuda(),
                             torch.from_numpy(vn.view(np.int16)).cuda(), torch.from_numpy(kbud).cuda(), out, lse,
                             compute=compute, copy=copy)
            torch.cuda.synchronize()
            assert pool.device_status() == pi.PI_OK
            sel_v, nsel_v, tab_v = (t.cpu().numpy() for t in pool.view_step())
            sob = pool.view_slot_of_block().cpu().numpy()
            bos = pool.view_block_of_slot().cpu().numpy()
            out_np = out.cpu().numpy().view(np.uint16)
            lse_np = lse.cpu().numpy()
            # properties on every unit
            for l in range(L):
                for r in range(R):
                    n = int(nsel_v[l, r, 0])
                    assert n == min(int(kbud[l, r]), -(-(NTOK + s + 1) // B) - c["W"]) + c["W"]
                    t = tab_v[l, r, 0, :n]
                    assert np.all((t >= 0) & (t < P_of(r))) and len(set(t.tolist())) == n
                    bs, sb = bos[r, l, 0, :P_of(r)], sob[r, l, 0]
                    occ = np.nonzero(bs >= 0)[0]
                    assert np.all(sb[bs[occ]] == occ)
                    assert (sb >= 0).sum() == occ.size
            assert np.all(np.isfinite(lse_np))
            # element by element on the sampled units
            poolv = pool.view_pool()
            for (r, l), u in units.items():
                sel, table, ref_out, ref_lse = u.step(qs[s][l, r], kn[l, r], vn[l, r], int(kbud[l, r]))
                assert np.array_equal(sel_v[l, r, 0, : len(sel)], sel)
                assert np.array_equal(tab_v[l, r, 0, : len(sel)], table)
                assert np.array_equal(sob[r, l, 0], u.sob) and np.array_equal(bos[r, l, 0, :P_of(r)], u.bos)
                for i, b in enumerate(sel):
                    gs = pool.global_slot(r, l, int(table[i]))
                    assert np.array_equal(poolv[gs].cpu().numpy().view(np.uint16), u.reg[b])
                err = np.max(np.abs(bf16_to_f32(out_np[l, r]) - bf16_to_f32(ref_out)))
                assert err <= OUT_ATOL
                rel = np.abs(lse_np[l, r] - ref_lse) / np.maximum(np.abs(ref_lse), 1.0)
                assert rel.max() <= LSE_RTOL
