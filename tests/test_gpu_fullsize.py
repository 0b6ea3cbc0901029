"""Full-size parity in the benchmark's launch configuration.

The Llama-3-8B-shaped workload (32 layers, batch 8, 32 q / 8 KV heads, d 128,
32768 tokens in blocks of 64, top-32 + 2 recent, a 128-slot pool per request
and layer, 5 % heavy-hitter blocks, AR(1) rho 0.9 queries) runs three
pipelined decode steps through pi_decode_step exactly as bench.py launches it
(compute + copy streams, UVA gather). Sampled (request, layer) units are checked
against the oracle element by element; properties that hold at any size
(selection size, table validity and uniqueness, map inverses, finite outputs)
are checked on every unit.
"""
import numpy as np
import pytest

import oracle
import synth
from _helpers import LSE_RTOL, OUT_ATOL, bf16_to_f32

torch = pytest.importorskip("torch")
pi = pytest.importorskip("sparse_kv_cache_block_gb300")

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

L, R, HQ, HKV, D, B, NTOK, K, W, P = 32, 8, 32, 8, 128, 64, 32768, 32, 2, 128
STEPS, SEED, RHO, HEAVY = 3, 0, 0.9, 0.05
SAMPLE = [(0, 0), (3, 7), (7, 31), (5, 16), (1, 23)]


class UnitOracle:
    """Oracle state of one (request, layer): its own copy of the host region."""

    def __init__(self, r, l, max_blocks):
        self.r, self.l = r, l
        self.reg = synth.kv_region(SEED, l, r, NTOK, max_blocks, HKV, B, D, HEAVY, 2.0)
        self.ntok = NTOK
        self.kmean = np.zeros((max_blocks, HKV, D), dtype=np.float32)
        self.kmean[: NTOK // B] = oracle.region_summaries(self.reg, NTOK)
        self.sob = np.full(max_blocks, -1, dtype=np.int32)
        self.bos = np.full(P, -1, dtype=np.int32)

    def step(self, q, k_new, v_new):
        b, tp = divmod(self.ntok, B)
        self.reg[b, :, 0, tp] = k_new
        self.reg[b, :, 1, tp] = v_new
        self.ntok += 1
        self.kmean[b] = oracle.block_summary(self.reg[b], tp + 1)
        nb = -(-self.ntok // B)
        sel = oracle.select_shared(q, self.kmean[:nb], K, W)
        table, _, _, _ = oracle.recall_plan(sel, self.sob, self.bos)
        out, lse, _ = oracle.attention(q, self.reg, sel, self.ntok, HKV)
        return sel, table, out, lse


def test_llama8b_shape_full_size_sampled_parity():
    pi.build()
    max_blocks = -(-(NTOK + STEPS) // B) + 1
    with pi.Pool(L, R, HQ, HKV, D, B, max_blocks, P, K, W) as pool:
        for l in range(L):
            for r in range(R):
                synth.fill_kv(pool.host_kv_ptr(l, r), SEED, l, r, NTOK, max_blocks, HKV, B, D, HEAVY, 2.0)
        for l in range(L):
            pool.update_summaries(l, [NTOK] * R)
        torch.cuda.synchronize()
        units = {(r, l): UnitOracle(r, l, max_blocks) for (r, l) in SAMPLE}
        qs = synth.q_ar1(SEED, L, R, HQ, D, STEPS, RHO)
        compute, copy = torch.cuda.Stream(), torch.cuda.Stream()
        kb = torch.full((L, R), K, dtype=torch.int32, device="cuda")
        for s in range(STEPS):
            kn = np.empty((L, R, HKV, D), dtype=np.uint16)
            vn = np.empty_like(kn)
            for l in range(L):
                for r in range(R):
                    kn[l, r], vn[l, r] = synth.token_kv(SEED, l, r, NTOK + s, HKV, D)
            out = torch.empty((L, R, HQ, D), dtype=torch.int16, device="cuda")
            lse = torch.empty((L, R, HQ), dtype=torch.float32, device="cuda")
            pool.decode_step(torch.from_numpy(qs[s].view(np.int16)).cuda(), torch.from_numpy(kn.view(np.int16)).cuda(),
                             torch.from_numpy(vn.view(np.int16)).cuda(), kb, out, lse, compute=compute, copy=copy)
            torch.cuda.synchronize()
            assert pool.device_status() == pi.PI_OK
            sel_v, nsel_v, tab_v = (t.cpu().numpy() for t in pool.view_step())
            sob = pool.view_slot_of_block().cpu().numpy()
            bos = pool.view_block_of_slot().cpu().numpy()
            out_np = out.cpu().numpy().view(np.uint16)
            lse_np = lse.cpu().numpy()
            # properties on every unit
            assert np.all(nsel_v == K + W)
            for l in range(L):
                for r in range(R):
                    t = tab_v[l, r, 0, : K + W]
                    assert np.all((t >= 0) & (t < P)) and len(set(t.tolist())) == K + W
                    bs, sb = bos[r, l, 0], sob[r, l, 0]
                    occ = np.nonzero(bs >= 0)[0]
                    assert np.all(sb[bs[occ]] == occ)
                    assert (sb >= 0).sum() == occ.size
            assert np.all(np.isfinite(lse_np))
            # element-by-element on the sampled units
            poolv = pool.view_pool()
            for (r, l), u in units.items():
                sel, table, ref_out, ref_lse = u.step(qs[s][l, r], kn[l, r], vn[l, r])
                assert np.array_equal(sel_v[l, r, 0, : len(sel)], sel)
                assert np.array_equal(tab_v[l, r, 0, : len(sel)], table)
                assert np.array_equal(sob[r, l, 0], u.sob) and np.array_equal(bos[r, l, 0, :P], u.bos)
                for i, b in enumerate(sel):
                    gs = pool.global_slot(r, l, int(table[i]))
                    assert np.array_equal(poolv[gs].cpu().numpy().view(np.uint16), u.reg[b])
                err = np.max(np.abs(bf16_to_f32(out_np[l, r]) - bf16_to_f32(ref_out)))
                assert err <= OUT_ATOL
                rel = np.abs(lse_np[l, r] - ref_lse) / np.maximum(np.abs(ref_lse), 1.0)
                assert rel.max() <= LSE_RTOL
