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
* Fragmentation sweep shapes: 8 KV heads, d 128, batch 64, 32768 tokens in
  blocks of 16 or 128 at an equal 2048-token budget (top-128 or top-16, no
  recent window), shared or per-KV-head selection, pool of k slots flushed
  before the recall (0 % resident); per-layer select and recall calls as the
  sweep makes them, UVA gather and per-run cudaMemcpyAsync arms.

Bars beyond the path's own gates (max-abs 2e-2 on bf16 outputs, 1e-3 relative
on the log-sum-exp): every output element within 2^-7 |ref| + 2e-3 (2^-7 |ref|
covers the two bf16 roundings of the output, the GPU's and the oracle's; 2e-3
covers the bf16 rounding of the softmax weights in the PV product, at most
2^-9 times the weighted mean of |V|, about 0.8 for N(0, 1) values); every
head's log-sum-exp within 1e-5 relative (fp32 logits of 128 products and fp32
row sums: a few 1e-7 relative; dropping one token of a 2 176-token selection
moves it by about 6e-5); and, for one sampled (request, layer) per shape, every
fp32 logit within 1e-5 max(|z|, 1).
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
OUT_REL, OUT_ABS = 2.0 ** -7, 2e-3   # per-element output bound: OUT_REL |ref| + OUT_ABS
LSE_TIGHT = 1e-5                       # per-head log-sum-exp, relative
LOGIT_TIGHT = 1e-5                     # fp32 logits of one sampled unit, relative to max(|z|, 1)


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

    def step(self, q, k_new, v_new, k, want_logits=False):
        c = self.c
        b, tp = divmod(self.ntok, c["B"])
        self.reg[b, :, 0, tp] = k_new
        self.reg[b, :, 1, tp] = v_new
        self.ntok += 1
        self.kmean[b] = oracle.block_summary(self.reg[b], tp + 1)
        nb = -(-self.ntok // c["B"])
        sel = oracle.select_shared(q, self.kmean[:nb], k, c["W"])
        table, _, _, _ = oracle.recall_plan(sel, self.sob, self.bos)
        out, lse, lg = oracle.attention(q, self.reg, sel, self.ntok, c["HKV"], want_logits)
        return sel, table, out, lse, lg


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
        worst = {"out_abs": 0.0, "lse_rel": 0.0, "logit_rel": None, "logits_compared": 0}
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
            # element by element on the sampled units; the first sampled unit of the
            # last step also has its fp32 logits compared (a second attention launch
            # over the step's own selection and table, with the debug logits)
            poolv = pool.view_pool()
            last = s == c["STEPS"] - 1
            for i_u, ((r, l), u) in enumerate(units.items()):
                with_logits = last and i_u == 0
                sel, table, ref_out, ref_lse, ref_lg = u.step(qs[s][l, r], kn[l, r], vn[l, r], int(kbud[l, r]),
                                                              with_logits)
                assert np.array_equal(sel_v[l, r, 0, : len(sel)], sel)
                assert np.array_equal(tab_v[l, r, 0, : len(sel)], table)
                assert np.array_equal(sob[r, l, 0], u.sob) and np.array_equal(bos[r, l, 0, :P_of(r)], u.bos)
                for i, b in enumerate(sel):
                    gs = pool.global_slot(r, l, int(table[i]))
                    assert np.array_equal(poolv[gs].cpu().numpy().view(np.uint16), u.reg[b])
                got = bf16_to_f32(out_np[l, r]).astype(np.float64)
                ref = bf16_to_f32(ref_out).astype(np.float64)
                dev_abs = np.abs(got - ref)
                assert dev_abs.max() <= OUT_ATOL
                assert np.all(dev_abs <= OUT_REL * np.abs(ref) + OUT_ABS), float((dev_abs - OUT_REL * np.abs(ref)).max())
                rel = np.abs(lse_np[l, r] - ref_lse) / np.maximum(np.abs(ref_lse), 1.0)
                assert rel.max() <= LSE_RTOL
                assert rel.max() <= LSE_TIGHT, float(rel.max())
                worst["out_abs"] = max(worst["out_abs"], float(dev_abs.max()))
                worst["lse_rel"] = max(worst["lse_rel"], float(rel.max()))
                if with_logits:
                    cap = c["K"] + c["W"]
                    sel_d, nsel_d, tab_d = pool.view_step()
                    lg = torch.full((R, c["HQ"], cap, B), float("nan"), device="cuda")
                    o2 = torch.empty((R, c["HQ"], D), dtype=torch.int16, device="cuda")
                    l2 = torch.empty((R, c["HQ"]), dtype=torch.float32, device="cuda")
                    q_l = torch.from_numpy(np.ascontiguousarray(qs[s][l]).view(np.int16)).cuda()
                    pool.sparse_decode(l, q_l, sel_d[l], tab_d[l], nsel_d[l], o2, l2, lg)
                    torch.cuda.synchronize()
                    assert pool.device_status() == pi.PI_OK
                    lg_r = lg[r].cpu().numpy().astype(np.float64)
                    m = ~np.isnan(ref_lg)
                    got_lg = lg_r[:, : ref_lg.shape[1]][m]
                    assert not np.isnan(got_lg).any()
                    lrel = np.abs(got_lg - ref_lg[m]) / np.maximum(np.abs(ref_lg[m]), 1.0)
                    assert lrel.max() <= LOGIT_TIGHT, float(lrel.max())
                    worst["logit_rel"] = float(lrel.max())
                    worst["logits_compared"] = int(m.sum())
        print(f"{name}: largest |out - ref| {worst['out_abs']:.3e}, lse relative {worst['lse_rel']:.3e}, "
              f"logit relative {worst['logit_rel']:.3e} over {worst['logits_compared']} logits")


# ------------------------------------------------------------------ fragmentation sweep shapes
FRAG_SAMPLE = [(0, 0), (63, 1), (31, 0), (17, 1)]  # (request, layer) checked element by element


@pytest.mark.parametrize("B,mode,method", [(16, "shared", "uva"), (16, "headwise", "uva"), (128, "shared", "uva"),
                                           (128, "headwise", "uva"), (128, "headwise", "memcpy"),
                                           (16, "shared", "memcpy")],
                         ids=["B16_shared_uva", "B16_headwise_uva", "B128_shared_uva", "B128_headwise_uva",
                              "B128_headwise_memcpy", "B16_shared_memcpy"])
def test_fragmentation_sweep_shapes_parity(B, mode, method):
    """The sweep's shapes ("PulseInfer Guide", "1. The Small-Packet PCIe DMA Tax":
    small head-wise fragments against whole shared blocks): batch 64, 32 q / 8 KV
    heads, d 128, 32768 tokens, top-(2048/B) with no recent window, a pool of k
    slots flushed before the recall (0 % resident), 2 layers over one host layer.
    Per-layer select and recall calls as the sweep makes them. Every unit: nsel =
    k, table = 0..n-1 (every block missing, free slots taken in order), maps
    inverse; sampled units: selections, tables, maps and every recalled byte
    bit-exact against the oracle."""
    L, R, HQ, HKV, D, N = 2, 64, 32, 8, 128, 32768
    k = 2048 // B
    nb = N // B
    max_blocks = nb + 1
    pm = pi.PI_HEADWISE if mode == "headwise" else pi.PI_SHARED
    meth = {"uva": pi.PI_RECALL_UVA, "memcpy": pi.PI_RECALL_MEMCPY}[method]
    pi.build()
    with pi.Pool(L, R, HQ, HKV, D, B, max_blocks, k, k, 0, select_mode=pm, host_layers=1) as pool:
        U = pool.U
        for r in range(R):
            synth.fill_kv(pool.host_kv_ptr(0, r), SEED, 0, r, N, max_blocks, HKV, B, D, 0.0, 0.0)
        for l in range(L):
            pool.update_summaries(l, [N] * R)
        torch.cuda.synchronize()
        qs = synth.q_ar1(SEED, L, R, HQ, D, 1, 0.9)[0]
        sel = torch.full((L, R * U, k), -7, dtype=torch.int32, device="cuda")
        nsel = torch.full((L, R * U), -7, dtype=torch.int32, device="cuda")
        table = torch.full((L, R * U, k), -7, dtype=torch.int32, device="cuda")
        kb = torch.full((R,), k, dtype=torch.int32, device="cuda")
        q_d = torch.from_numpy(qs.view(np.int16)).cuda()
        for l in range(L):
            pool.select_topk(l, q_d[l], kb, sel[l], nsel[l])
        pool.flush(-1)
        frags = 0
        for l in range(L):
            st = pool.recall(l, sel[l], nsel[l], table[l], method=meth, stats=True)
            frags += st["fragments"]
        torch.cuda.synchronize()
        assert pool.device_status() == pi.PI_OK
        assert frags == L * R * U * k  # every selected unit was missing
        sel_np, nsel_np, tab_np = sel.cpu().numpy(), nsel.cpu().numpy(), table.cpu().numpy()
        sob = pool.view_slot_of_block().cpu().numpy()
        bos = pool.view_block_of_slot().cpu().numpy()
        # properties on every unit
        assert np.all(nsel_np == k)
        assert np.all(tab_np == np.arange(k, dtype=np.int32))
        for l in range(L):
            for r in range(R):
                for u in range(U):
                    s_ = sel_np[l, r * U + u]
                    assert np.all(np.diff(s_) > 0) and s_[0] >= 0 and s_[-1] < nb
                    assert np.array_equal(bos[r, l, u, :k], s_)
                    assert np.array_equal(np.nonzero(sob[r, l, u] >= 0)[0], s_)
        # element by element on the sampled units
        poolv = pool.view_pool()
        reg_cache = {}
        for (r, l) in FRAG_SAMPLE:
            if r not in reg_cache:
                reg = synth.kv_region(SEED, 0, r, N, max_blocks, HKV, B, D, 0.0, 0.0)
                reg_cache[r] = (reg, oracle.region_summaries(reg, N))
            reg, km = reg_cache[r]
            if U == 1:
                want = [oracle.select_shared(qs[l, r], km, k, 0)]
            else:
                want = oracle.select_headwise(qs[l, r], km, k, 0)
            for u in range(U):
                s_ref = want[u]
                assert np.array_equal(sel_np[l, r * U + u], s_ref), (r, l, u)
                sob_o = np.full(max_blocks, -1, dtype=np.int32)
                bos_o = np.full(k, -1, dtype=np.int32)
                t_ref, _, _, _ = oracle.recall_plan(s_ref, sob_o, bos_o)
                assert np.array_equal(tab_np[l, r * U + u], t_ref)
                assert np.array_equal(sob[r, l, u], sob_o) and np.array_equal(bos[r, l, u, :k], bos_o)
                for i, b in enumerate(s_ref):
                    got = poolv[pool.global_slot(r, l, int(t_ref[i]))].cpu().numpy().view(np.uint16)
                    if U == 1:
                        assert np.array_equal(got, reg[b]), (r, l, i, b)
                    else:
                        assert np.array_equal(got[u], reg[b, u]), (r, l, u, i, b)
        print(f"B={B} {mode} {method}: {frags} fragments recalled, {len(FRAG_SAMPLE)} units checked byte for byte")
