"""CUDA path vs the CPU oracle, element by element, through the C ABI.

Bars: selected block ids, nsel, block tables, slot maps and recalled bytes are
bit-exact; block summaries are bit-exact (they decide the selection); attention
outputs (bf16) within max-abs 2e-2, log-sum-exp and logits (fp32) within 1e-3
relative.
"""
import numpy as np
import pytest

import oracle
import synth
from _helpers import (LOGIT_RTOL, LSE_RTOL, OUT_ATOL, OracleModel, Workload, bf16_to_f32, fill_pool_host,
                      new_tokens, queries)

torch = pytest.importorskip("torch")
pi = pytest.importorskip("sparse_kv_cache_block_gb300")

pytestmark = pytest.mark.gpu

METHODS = [pi.PI_RECALL_UVA, pi.PI_RECALL_MEMCPY, pi.PI_RECALL_STAGED]


@pytest.fixture(scope="module", autouse=True)
def _built():
    pi.build()
    pi.load()


def make_pool(w: Workload, **kw):
    return pi.Pool(w.layers, w.batch, w.hq, w.hkv, w.head_dim, w.block_tokens, w.max_blocks, w.pool_slots, w.k,
                   w.window, select_mode=w.select_mode, host_layers=(w.host_layers if w.host_layers != w.layers else 0),
                   pool_slots_per_req=w.slots_per_req, evict_policy=w.evict_policy, **kw)


def prefill(pool, w: Workload):
    fill_pool_host(pool, w)
    for l in range(w.layers):
        pool.update_summaries(l, w.ntok)
    torch.cuda.synchronize()


def dev(a, dtype=None):
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    t = torch.from_numpy(a)
    return t.cuda() if dtype is None else t.to(dtype).cuda()


def check_kmean(pool, om, w):
    km = pool.view_kmean().cpu().numpy()
    for r in range(w.batch):
        for l in range(w.layers):
            nb = om.nb(r, l)
            assert np.array_equal(km[r, l, :nb].view(np.uint32), om.kmean[(r, l)][:nb].view(np.uint32)), (r, l)


def check_selection(sel_dev, nsel_dev, ref, U):
    sel = sel_dev.cpu().numpy()
    nsel = nsel_dev.cpu().numpy().reshape(-1)
    cap = sel.shape[-1]
    sel = sel.reshape(-1, cap)
    units = [s for s in ref] if U == 1 else [sg for s in ref for sg in s]
    for u, want in enumerate(units):
        assert nsel[u] == len(want), (u, nsel[u], len(want))
        assert np.array_equal(sel[u, : len(want)], want), (u, sel[u, : len(want)], want)


def check_tables_maps_bytes(pool, om, w, l, sels, tables, table_dev):
    tab = table_dev.cpu().numpy().reshape(-1, w.k + w.window)
    U = om.U
    sob = pool.view_slot_of_block().cpu().numpy()
    bos = pool.view_block_of_slot().cpu().numpy()
    poolv = pool.view_pool()
    for r in range(w.batch):
        for u in range(U):
            want_t = tables[r] if U == 1 else tables[r][u]
            got = tab[r * U + u, : len(want_t)]
            assert np.array_equal(got, want_t), (r, u, got, want_t)
            n_slots = len(om.bos[(r, l, u)])
            assert np.array_equal(sob[r, l, u], om.sob[(r, l, u)]), (r, l, u)
            assert np.array_equal(bos[r, l, u, :n_slots], om.bos[(r, l, u)]), (r, l, u)
            if w.evict_policy == 1:
                st = pool.view_slot_stamp().cpu().numpy()
                assert np.array_equal(st[r, l, u, :n_slots], om.stamp[(r, l, u)]), (r, l, u)
            s_list = sels[r] if U == 1 else sels[r][u]
            reg = om.reg[(w.host_layer(l), r)]
            for i, b in enumerate(s_list):
                gs = pool.global_slot(r, l, int(want_t[i]))
                got_bytes = poolv[gs].cpu().numpy().view(np.uint16)
                if U == 1:
                    assert np.array_equal(got_bytes, reg[b]), (r, l, i, b)
                else:
                    assert np.array_equal(got_bytes[u], reg[b, u]), (r, l, u, i, b)


def check_attention(out_dev, lse_dev, ref_out, ref_lse, logits_dev=None, ref_logits=None):
    out = bf16_to_f32(out_dev.cpu().numpy().view(np.uint16))
    ref = bf16_to_f32(ref_out)
    err = np.max(np.abs(out - ref))
    assert err <= OUT_ATOL, f"max abs err {err}"
    if lse_dev is not None:
        lse = lse_dev.cpu().numpy().astype(np.float64)
        fin = np.isfinite(ref_lse)
        assert np.array_equal(np.isfinite(lse), fin)
        rel = np.abs(lse[fin] - ref_lse[fin]) / np.maximum(np.abs(ref_lse[fin]), 1.0)
        assert rel.size == 0 or rel.max() <= LSE_RTOL, rel.max()
    if logits_dev is not None:
        lg = logits_dev.cpu().numpy().astype(np.float64)
        for r, rl in enumerate(ref_logits):
            m = ~np.isnan(rl)
            cap = rl.shape[1]
            got = lg[r][:, :cap][m]
            want = rl[m]
            assert not np.isnan(got).any()
            assert np.all(np.abs(got - want) <= LOGIT_RTOL * np.maximum(np.abs(want), 1.0))
    return err


def run_layer(pool, om, w, l, q, kreq, method, logits=True):
    """select -> recall -> attention for one layer, each checked against the oracle."""
    R, U, cap = w.batch, om.U, w.k + w.window
    q_dev = dev(q)
    kreq_dev = dev(np.asarray(kreq, dtype=np.int32))
    sel = torch.full((R * U, cap), -7, dtype=torch.int32, device="cuda")
    nsel = torch.full((R * U,), -7, dtype=torch.int32, device="cuda")
    pool.select_topk(l, q_dev, kreq_dev, sel, nsel)
    ref_sel = om.select(l, q, kreq)
    check_selection(sel, nsel, ref_sel, U)
    table = torch.full((R * U, cap), -7, dtype=torch.int32, device="cuda")
    stats = pool.recall(l, sel, nsel, table, method=method, stats=True)
    ref_tab = om.recall(l, ref_sel)
    check_tables_maps_bytes(pool, om, w, l, ref_sel, ref_tab, table)
    out = torch.empty((R, w.hq, w.head_dim), dtype=torch.int16, device="cuda")
    lse = torch.empty((R, w.hq), dtype=torch.float32, device="cuda")
    lg = torch.full((R, w.hq, cap, w.block_tokens), float("nan"), device="cuda") if logits else None
    pool.sparse_decode(l, q_dev, sel, table, nsel, out, lse, lg)
    ref_out, ref_lse, ref_lg = om.attention(l, q, ref_sel, want_logits=logits)
    check_attention(out, lse, ref_out, ref_lse, lg, ref_lg if logits else None)
    torch.cuda.synchronize()
    assert pool.device_status() == pi.PI_OK
    return stats, ref_sel


C1 = Workload(layers=1, batch=1, hq=8, hkv=2, head_dim=64, block_tokens=16, ntok=[4096], k=32, window=4,
              pool_slots=64, steps=1, seed=0)


@pytest.mark.parametrize("method", METHODS)
def test_small_config_layer_calls(method):
    """1 layer, batch 1, 8 q / 2 KV heads, d 64, 4096 tokens in 256 blocks of 16,
    top-32 + 4 recent, empty 64-slot pool, one step: every output checked."""
    w = C1
    with make_pool(w) as pool:
        prefill(pool, w)
        om = OracleModel(w)
        check_kmean(pool, om, w)
        q = queries(w)[0]
        stats, ref_sel = run_layer(pool, om, w, 0, q[0], [w.k] * w.batch, method)
        assert stats["fragments"] == 36 and stats["bytes"] == 36 * pool.block_bytes
        if method == pi.PI_RECALL_MEMCPY:
            assert stats["api_calls"] == stats["runs"]
        # a second identical recall hits everything and moves nothing
        sel = torch.tensor(np.array(ref_sel[0], dtype=np.int32)[None], device="cuda")
        nsel = torch.tensor([len(ref_sel[0])], dtype=torch.int32, device="cuda")
        table = torch.empty((1, w.k + w.window), dtype=torch.int32, device="cuda")
        st2 = pool.recall(0, sel, nsel, table, method=method, stats=True)
        assert st2["fragments"] == 0 and st2["hits"] == 36


@pytest.mark.parametrize("method,evict,ahead,placement", [(m, 0, 1, "default") for m in METHODS] +
                         [(pi.PI_RECALL_UVA, 1, 1, "default"), (pi.PI_RECALL_MEMCPY, 1, 1, "default"),
                          (pi.PI_RECALL_UVA, 0, 0, "default"), (pi.PI_RECALL_UVA, 1, 0, "default"),
                          (pi.PI_RECALL_UVA, 0, 1, "few"), (pi.PI_RECALL_UVA, 1, 1, "shared"),
                          (pi.PI_RECALL_UVA, 0, 1, "shared"), (pi.PI_RECALL_UVA, 0, -1, "default"),
                          (pi.PI_RECALL_UVA, 1, -1, "default"), (pi.PI_RECALL_MEMCPY, 0, -1, "default"),
                          (pi.PI_RECALL_UVA, 0, -1, "one_copy"), (pi.PI_RECALL_UVA, 1, 1, "one_copy"),
                          (pi.PI_RECALL_UVA, 0, -1, "fused"), (pi.PI_RECALL_UVA, 1, -1, "fused"),
                          (pi.PI_RECALL_UVA, 0, -1, "fused_few"), (pi.PI_RECALL_UVA, 1, 1, "fused"),
                          (pi.PI_RECALL_UVA, 0, -1, "fused_one_copy")])
def test_multistep_pipeline_8b_shape(method, evict, ahead, placement):
    """Llama-3-8B-shaped heads (32 q / 8 KV, d 128, blocks of 64), 2 layers, 2
    requests with ragged tails, heavy-hitter blocks, AR(1) queries, 4 pipelined
    decode steps with token append; all per-layer results checked each step,
    under both eviction policies."""
    w = Workload(layers=2, batch=2, hq=32, hkv=8, head_dim=128, block_tokens=64, ntok=[4000, 2500], k=8, window=2,
                 pool_slots=14, steps=4, rho=0.9, heavy_frac=0.05, heavy_shift=2.0, seed=3, evict_policy=evict)
    L, R = w.layers, w.batch
    with make_pool(w) as pool:
        pool.set_pipeline(max(ahead, 0), attention_stream=(ahead < 0))  # -1: attention on its own stream (default)
        if placement == "few":
            pool.set_gather(5, 8, True)  # few exclusive CTAs: every CTA loops over many chunks
        elif placement == "shared":
            pool.set_gather(0, 8, False)  # one 256-thread CTA per SM beside other kernels
        elif placement == "one_copy":
            pool.set_copy_streams(1)  # every gather on the caller's copy stream (the default uses two)
        elif placement.startswith("fused"):
            # selection, plan and gather of a layer in one launch; "few": 3 CTAs, many items each
            pool.set_fused(True, 3 if placement == "fused_few" else 0)
            if placement == "fused_one_copy":
                pool.set_copy_streams(1)
        prefill(pool, w)
        om = OracleModel(w)
        qs = queries(w)
        compute = torch.cuda.Stream()
        copy = torch.cuda.Stream()
        for step in range(w.steps):
            kn, vn = new_tokens(w, step)
            kbud = np.full((L, R), w.k, dtype=np.int32)
            kbud[1, 0] = 3  # a smaller budget for one (layer, request)
            out = torch.empty((L, R, w.hq, w.head_dim), dtype=torch.int16, device="cuda")
            lse = torch.empty((L, R, w.hq), dtype=torch.float32, device="cuda")
            q_dev, k_dev, v_dev, b_dev = dev(qs[step]), dev(kn), dev(vn), dev(kbud)
            torch.cuda.synchronize()
            st = pool.decode_step(q_dev, k_dev, v_dev, b_dev, out, lse, method=method, compute=compute, copy=copy,
                                  stats=True)
            torch.cuda.synchronize()
            assert pool.device_status() == pi.PI_OK
            sel_v, nsel_v, tab_v = pool.view_step()
            for l in range(L):
                om.append(l, kn[l], vn[l])
                ref_sel = om.select(l, qs[step][l], kbud[l])
                check_selection(sel_v[l], nsel_v[l], ref_sel, 1)
                ref_tab = om.recall(l, ref_sel)
                check_tables_maps_bytes(pool, om, w, l, ref_sel, ref_tab, tab_v[l])
                ref_out, ref_lse, _ = om.attention(l, qs[step][l], ref_sel)
                check_attention(out[l], lse[l], ref_out, ref_lse)
            check_kmean(pool, om, w)
            assert st["selected"] == sum(int(nsel_v[l].sum()) for l in range(L))


@pytest.mark.parametrize("mode", [pi.PI_SHARED, pi.PI_CONSENSUS], ids=["shared", "consensus"])
def test_selection_form_changes_during_decode(mode):
    """A pool whose candidate count crosses 1024 during the decode (1024 at the
    first step, 1025 from the second): the selection runs as one cluster per
    request, then as the last-CTA form, with the token append folded into the
    first and done by the append kernel in the second; every layer of every step
    against the oracle, with preloaded residency and per-request budgets."""
    B = 16
    ntok = (1024 + 2) * B - 1  # 1026 blocks (the last one holds 15 tokens): 1024 candidates
    w = Workload(layers=2, batch=3, hq=8, hkv=2, head_dim=64, block_tokens=B, ntok=[ntok, ntok - 400, ntok], k=24,
                 window=2, pool_slots=40, steps=4, rho=0.9, heavy_frac=0.05, seed=91, select_mode=mode,
                 slots_per_req=[40, 60, 40])
    L, R = w.layers, w.batch
    with make_pool(w) as pool:
        prefill(pool, w)
        om = OracleModel(w)
        for l in range(L):
            blocks = synth.sample_sorted(w.seed, synth.KIND_RESIDENT, l, 0, 1026, 30)
            pool.preload(l, 0, blocks)
            om.preload(l, 0, blocks)
        qs = queries(w)
        for step in range(w.steps):
            kn, vn = new_tokens(w, step)
            kbud = np.full((L, R), w.k, dtype=np.int32)
            kbud[1, 2] = 5
            out = torch.empty((L, R, w.hq, w.head_dim), dtype=torch.int16, device="cuda")
            lse = torch.empty((L, R, w.hq), dtype=torch.float32, device="cuda")
            pool.decode_step(dev(qs[step]), dev(kn), dev(vn), dev(kbud), out, lse)
            torch.cuda.synchronize()
            assert pool.device_status() == pi.PI_OK
            sel_v, nsel_v, tab_v = pool.view_step()
            for l in range(L):
                om.append(l, kn[l], vn[l])
                ref_sel = om.select(l, qs[step][l], kbud[l])
                check_selection(sel_v[l], nsel_v[l], ref_sel, 1)
                ref_tab = om.recall(l, ref_sel)
                check_tables_maps_bytes(pool, om, w, l, ref_sel, ref_tab, tab_v[l])
                ref_out, ref_lse, _ = om.attention(l, qs[step][l], ref_sel)
                check_attention(out[l], lse[l], ref_out, ref_lse)
            check_kmean(pool, om, w)
        assert om.nb(0, 0) - w.window == 1025  # the last steps ran with more than 1024 candidates


@pytest.mark.parametrize("evict", [0, 1])
def test_headwise_arm(evict):
    """Per-KV-head selection (the fragmenting comparison arm): own top-k per head,
    fragment-granular recall into per-head sub-slots, attention per head."""
    w = Workload(layers=1, batch=2, hq=16, hkv=4, head_dim=128, block_tokens=32, ntok=[2000, 1500], k=6, window=0,
                 pool_slots=6, steps=1, seed=5, select_mode=1, evict_policy=evict)
    with make_pool(w) as pool:
        prefill(pool, w)
        om = OracleModel(w)
        q = queries(w)[0][0]
        for method in METHODS:
            stats, ref_sel = run_layer(pool, om, w, 0, q, [w.k] * w.batch, method)
            if method == METHODS[0]:
                assert stats["bytes"] == stats["fragments"] * pool.frag_bytes
            pool.flush()
            torch.cuda.synchronize()
            om.flush()


def test_select_all_equals_dense_attention():
    """k >= number of candidates: every block is selected and the sparse result is
    dense attention over all tokens (independent numpy fp64 routine)."""
    w = Workload(layers=1, batch=2, hq=8, hkv=2, head_dim=64, block_tokens=16, ntok=[1000, 777], k=70, window=4,
                 pool_slots=74, steps=1, seed=11)
    with make_pool(w) as pool:
        prefill(pool, w)
        om = OracleModel(w)
        q = queries(w)[0][0]
        _, ref_sel = run_layer(pool, om, w, 0, q, [w.k] * w.batch, pi.PI_RECALL_UVA, logits=False)
        for r in range(w.batch):
            nb = om.nb(r, 0)
            assert list(ref_sel[r]) == list(range(nb))
        # dense: recompute with the library's output against numpy directly
        q_dev = dev(q)
        sel = torch.tensor(np.stack([np.pad(s, (0, w.k + w.window - len(s)), constant_values=-1) for s in ref_sel]),
                           dtype=torch.int32, device="cuda")
        nsel = torch.tensor([len(s) for s in ref_sel], dtype=torch.int32, device="cuda")
        table = torch.empty_like(sel)
        pool.recall(0, sel, nsel, table)
        out = torch.empty((w.batch, w.hq, w.head_dim), dtype=torch.int16, device="cuda")
        pool.sparse_decode(0, q_dev, sel, table, nsel, out)
        got = bf16_to_f32(out.cpu().numpy().view(np.uint16))
        for r in range(w.batch):
            reg = om.reg[(0, r)]
            n = w.ntok[r]
            K = np.stack([oracle.bf16_to_f64(reg[:, g, 0].reshape(-1, w.head_dim)[:n]) for g in range(w.hkv)])
            V = np.stack([oracle.bf16_to_f64(reg[:, g, 1].reshape(-1, w.head_dim)[:n]) for g in range(w.hkv)])
            dout, _ = oracle.dense_attention_fp64(oracle.bf16_to_f64(q[r]), K, V)
            assert np.max(np.abs(got[r] - dout)) <= OUT_ATOL


def test_edge_cases_tiny_and_degenerate():
    """Token counts 1, 16, 17, 40 (nb <= W, exact block, ragged), budgets 0, 1, 5,
    large; pool exactly k+W slots; per-request slot counts."""
    w = Workload(layers=1, batch=4, hq=8, hkv=2, head_dim=64, block_tokens=16, ntok=[1, 16, 17, 40], k=5, window=4,
                 pool_slots=9, steps=1, seed=7, slots_per_req=[9, 9, 12, 20])
    with make_pool(w) as pool:
        prefill(pool, w)
        om = OracleModel(w)
        check_kmean(pool, om, w)
        q = queries(w)[0][0]
        for kreq in ([0, 1, 5, 100], [5, 5, 5, 5], [2, 0, 3, 1]):
            for method in METHODS:
                run_layer(pool, om, w, 0, q, kreq, method)


@pytest.mark.parametrize("evict", [0, 1])
def test_preload_then_recall_counts_hits(evict):
    """Initial residency (a seeded sample) placed in slots 0.. ; later recalls only
    move what is missing, evicting unselected blocks; three queries in a row."""
    w = Workload(layers=1, batch=2, hq=32, hkv=8, head_dim=128, block_tokens=64, ntok=[6000, 6000], k=12, window=2,
                 pool_slots=40, steps=3, seed=9, heavy_frac=0.05, evict_policy=evict)
    with make_pool(w) as pool:
        prefill(pool, w)
        om = OracleModel(w)
        for r in range(w.batch):
            nb = -(-w.ntok[r] // w.block_tokens)
            blocks = synth.sample_sorted(w.seed, synth.KIND_RESIDENT, 0, r, nb, 30)
            pool.preload(0, r, blocks)
            om.preload(0, r, blocks)
        for step in range(w.steps):
            q = queries(w)[step][0]
            stats, ref_sel = run_layer(pool, om, w, 0, q, [w.k] * w.batch, pi.PI_RECALL_UVA)
            assert stats["hits"] + stats["fragments"] == sum(len(s) for s in ref_sel)


def test_recall_totals_accumulate_across_steps():
    """pi_pool_recall_totals (blocks recalled and hits, summed over layers on the
    device): over 4 decode steps without statistics they equal the sums of what
    the per-step statistics report for the same steps on a second pool (the two
    pools make the same selections); a reset zeroes them."""
    w = Workload(layers=2, batch=2, hq=32, hkv=8, head_dim=128, block_tokens=64, ntok=[4000, 2500], k=8, window=2,
                 pool_slots=14, steps=4, rho=0.9, heavy_frac=0.05, heavy_shift=2.0, seed=5)
    L, R = w.layers, w.batch
    qs = queries(w)
    sums = [0, 0]
    totals = None
    for use_stats in (True, False):
        with make_pool(w) as pool:
            prefill(pool, w)
            pool.recall_totals(reset=True)
            compute, copy = torch.cuda.Stream(), torch.cuda.Stream()
            for step in range(w.steps):
                kn, vn = new_tokens(w, step)
                kbud = np.full((L, R), w.k, dtype=np.int32)
                out = torch.empty((L, R, w.hq, w.head_dim), dtype=torch.int16, device="cuda")
                lse = torch.empty((L, R, w.hq), dtype=torch.float32, device="cuda")
                st = pool.decode_step(dev(qs[step]), dev(kn), dev(vn), dev(kbud), out, lse, compute=compute,
                                      copy=copy, stats=use_stats)
                torch.cuda.synchronize()
                if use_stats:
                    sums[0] += st["fragments"]
                    sums[1] += st["hits"]
            if not use_stats:
                totals = pool.recall_totals(reset=True)
                assert pool.recall_totals() == (0, 0)
            assert pool.device_status() == pi.PI_OK
    assert sums[0] > 0 and sums[1] > 0
    assert totals == (sums[0], sums[1])


def test_decode_step_host_matches_device_inputs():
    w = Workload(layers=2, batch=2, hq=16, hkv=4, head_dim=128, block_tokens=32, ntok=[3000, 2100], k=6, window=2,
                 pool_slots=10, steps=2, seed=13)
    L, R = w.layers, w.batch
    qs = queries(w)
    res = []
    for host_path in (False, True):
        with make_pool(w) as pool:
            prefill(pool, w)
            outs = []
            for step in range(w.steps):
                kn, vn = new_tokens(w, step)
                kb = np.full((L, R), w.k, dtype=np.int32)
                if host_path:
                    out = np.empty((L, R, w.hq, w.head_dim), dtype=np.uint16)
                    lse = np.empty((L, R, w.hq), dtype=np.float32)
                    pool.decode_step_host(np.ascontiguousarray(qs[step]), kn, vn, kb, out, lse)
                    outs.append((out.copy(), lse.copy()))
                else:
                    out = torch.empty((L, R, w.hq, w.head_dim), dtype=torch.int16, device="cuda")
                    lse = torch.empty((L, R, w.hq), dtype=torch.float32, device="cuda")
                    pool.decode_step(dev(qs[step]), dev(kn), dev(vn), dev(kb), out, lse)
                    torch.cuda.synchronize()
                    outs.append((out.cpu().numpy().view(np.uint16), lse.cpu().numpy()))
            res.append(outs)
    for (a, la), (b, lb) in zip(res[0], res[1]):
        assert np.array_equal(a, b) and np.array_equal(la, lb)


def test_injected_recall_fault_leaves_maps_unchanged():
    w = C1
    with make_pool(w) as pool:
        prefill(pool, w)
        om = OracleModel(w)
        q = queries(w)[0][0]
        pool.set_fault("recall_fail@2")
        run_layer(pool, om, w, 0, q, [w.k], pi.PI_RECALL_UVA)           # call 1 succeeds
        torch.cuda.synchronize()
        sob0 = pool.view_slot_of_block().cpu().clone()
        bos0 = pool.view_block_of_slot().cpu().clone()
        q2 = queries(Workload(**{**w.__dict__, "seed": 99}))[0][0]
        sel = torch.empty((1, w.k + w.window), dtype=torch.int32, device="cuda")
        nsel = torch.empty((1,), dtype=torch.int32, device="cuda")
        pool.select_topk(0, dev(q2), dev(np.array([w.k], dtype=np.int32)), sel, nsel)
        table = torch.empty_like(sel)
        with pytest.raises(pi.PiError) as ei:
            pool.recall(0, sel, nsel, table)                                 # call 2 fails
        assert ei.value.status == pi.PI_ERR_FAULT_INJECTED
        torch.cuda.synchronize()
        assert torch.equal(pool.view_slot_of_block().cpu(), sob0)
        assert torch.equal(pool.view_block_of_slot().cpu(), bos0)
        pool.recall(0, sel, nsel, table)                                     # call 3 succeeds
        torch.cuda.synchronize()
        assert pool.device_status() == pi.PI_OK


def test_out_of_range_block_id_is_flagged_not_faulted():
    """A selection naming a block past max_blocks: the plan kernel's own bounds
    check skips it and records PI_ERR_DEVICE in the status word."""
    w = C1
    with make_pool(w) as pool:
        prefill(pool, w)
        sel = torch.tensor([[0, 1, w.max_blocks + 5]], dtype=torch.int32, device="cuda")
        nsel = torch.tensor([3], dtype=torch.int32, device="cuda")
        table = torch.empty((1, w.k + w.window), dtype=torch.int32, device="cuda")
        pool.recall(0, sel, nsel, table)
        torch.cuda.synchronize()
        assert pool.device_status() == pi.PI_ERR_DEVICE
        assert table[0, 2].item() == -1
        pool.clear_device_status()
        assert pool.device_status() == pi.PI_OK


def test_invalid_arguments_return_status():
    w = C1
    with pytest.raises(pi.PiError) as ei:
        pi.Pool(1, 1, 8, 3, 64, 16, 256, 64, 32, 4)   # Hq % Hkv != 0
    assert ei.value.status == pi.PI_ERR_INVALID
    with pytest.raises(pi.PiError):
        pi.Pool(1, 1, 8, 2, 64, 16, 256, 10, 32, 4)   # pool smaller than k + W
    with make_pool(w) as pool:
        with pytest.raises(pi.PiError):
            pool.select_topk(0, torch.zeros(1, 8, 64, dtype=torch.int16, device="cuda"),
                             torch.zeros(1, dtype=torch.int32, device="cuda"), torch.zeros(1, 36, dtype=torch.int32,
                                                                                           device="cuda"),
                             torch.zeros(1, dtype=torch.int32, device="cuda"), mode=pi.PI_HEADWISE)


def test_bounded_wait_times_out_into_status_word():
    """A wait on a barrier phase that nothing completes gives up after its limit,
    records PI_ERR_TIMEOUT, and leaves the context usable (a normal call follows)."""
    w = C1
    with make_pool(w) as pool:
        assert pool.selftest_bounded_wait(20_000_000) == pi.PI_ERR_TIMEOUT
        pool.clear_device_status()
        prefill(pool, w)
        om = OracleModel(w)
        run_layer(pool, om, w, 0, queries(w)[0][0], [w.k], pi.PI_RECALL_UVA)


@pytest.mark.parametrize("hq,hkv", [(64, 8), (16, 8), (8, 8), (32, 4)], ids=["G8_70b", "G2", "G1", "G8_4kv"])
def test_query_group_sizes(hq, hkv):
    """Group sizes 1, 2 and 8 (the Llama-3-70B slice: 64 q / 8 KV heads fills every
    column of the mma's N = 8), ragged tails, two layers."""
    w = Workload(layers=2, batch=2, hq=hq, hkv=hkv, head_dim=128, block_tokens=64, ntok=[5000, 3001], k=16, window=4,
                 pool_slots=24, steps=1, seed=31 + hq + hkv, heavy_frac=0.05)
    with make_pool(w) as pool:
        prefill(pool, w)
        om = OracleModel(w)
        check_kmean(pool, om, w)
        q = queries(w)[0]
        for l in range(w.layers):
            run_layer(pool, om, w, l, q[l], [w.k, 7], pi.PI_RECALL_UVA)


@pytest.mark.parametrize("splits,cluster", [(0, 1), (1, 1), (3, 1), (3, 0), (8, 1), (14, 1)],
                         ids=["one_wave_global", "one_cta", "three_cluster", "three_global", "seven_cluster",
                              "fourteen_global"])
@pytest.mark.parametrize("D,B", [(64, 16), (64, 32), (64, 64), (64, 128), (128, 16), (128, 32), (128, 64), (128, 128)])
def test_attention_every_shape_and_split(D, B, splits, cluster):
    """The attention kernel at every head size and block size it is built for,
    under split counts that take each merge (one CTA writes directly; 2..8 splits
    merge in a cluster through DSMEM, or through the global partial buffer; more
    than 8 always through the buffer); ragged tails, a request shorter than one
    block, one budget of 0, logits checked."""
    w = Workload(layers=1, batch=3, hq=16, hkv=4, head_dim=D, block_tokens=B, ntok=[3000, 1777, 70], k=12, window=2,
                 pool_slots=14, steps=1, seed=41 + D + B)
    with make_pool(w) as pool:
        pool.set_attention(splits)
        pool.set_attention_cluster(bool(cluster))
        prefill(pool, w)
        om = OracleModel(w)
        run_layer(pool, om, w, 0, queries(w)[0][0], [w.k, 5, 0], pi.PI_RECALL_UVA)


@pytest.mark.parametrize("splits,cluster", [(2, 1), (3, 1), (8, 1), (2, 0)],
                         ids=["two_push", "three_pull", "eight_pull", "two_global"])
def test_attention_cluster_merges_group_of_eight(splits, cluster):
    """Llama-3-70B heads (64 q / 8 KV, G = 8 fills the mma's N), d 128, blocks of 64:
    two splits merge by pushing their partials into the first CTA's shared memory,
    three and eight pull slices from their peers (the push region would lower the
    CTAs per SM), and two without a cluster through the global buffer; ragged
    tails, a short request, a budget of 0."""
    w = Workload(layers=1, batch=3, hq=64, hkv=8, head_dim=128, block_tokens=64, ntok=[6000, 2300, 100], k=14,
                 window=2, pool_slots=16, steps=1, seed=61 + splits)
    with make_pool(w) as pool:
        pool.set_attention(splits)
        pool.set_attention_cluster(bool(cluster))
        prefill(pool, w)
        om = OracleModel(w)
        run_layer(pool, om, w, 0, queries(w)[0][0], [w.k, 9, 0], pi.PI_RECALL_UVA)


@pytest.mark.parametrize("splits", [0, 1], ids=["one_wave", "one_cta"])
def test_empty_selection_gives_zero_output(splits):
    """No recent window and a budget of 0: nothing is selected for that request;
    its output is zero and its log-sum-exp is -inf, the others are unaffected."""
    w = Workload(layers=1, batch=3, hq=32, hkv=8, head_dim=128, block_tokens=64, ntok=[2000, 900, 4100], k=6,
                 window=0, pool_slots=6, steps=1, seed=47)
    with make_pool(w) as pool:
        pool.set_attention(splits)
        prefill(pool, w)
        om = OracleModel(w)
        run_layer(pool, om, w, 0, queries(w)[0][0], [6, 0, 3], pi.PI_RECALL_UVA)


@pytest.mark.parametrize("hq,hkv,D,lam", [(8, 2, 64, 0.5), (32, 8, 128, 0.5), (32, 8, 128, 1.0), (64, 8, 128, 0.0),
                                          (16, 8, 128, 0.5), (8, 8, 128, 0.5), (12, 3, 64, 0.25)],
                         ids=["C1_shape", "8B", "8B_lam1", "70B_max_only", "G2", "G1", "G4_odd_hkv_d64"])
def test_consensus_selection_layer_calls(hq, hkv, D, lam):
    """Consensus-ranked shared selection (guide, "SoloHead Sparse Selection",
    "1. Consensus Scoring Mechanism"): selected ids bit-exact against the oracle,
    then recall and attention over them; ragged tails, a short request."""
    w = Workload(layers=1, batch=3, hq=hq, hkv=hkv, head_dim=D, block_tokens=64 if D == 128 else 16,
                 ntok=[4000, 2500, 90], k=12, window=2, pool_slots=16, steps=1, seed=51 + hq + D, heavy_frac=0.05,
                 select_mode=pi.PI_CONSENSUS, lam=lam)
    with make_pool(w) as pool:
        pool.set_consensus_lambda(lam)
        prefill(pool, w)
        om = OracleModel(w)
        check_kmean(pool, om, w)
        run_layer(pool, om, w, 0, queries(w)[0][0], [w.k, 5, 3], pi.PI_RECALL_UVA)


def test_consensus_worked_example_on_the_gpu():
    """The guide's SoloHead example through the library: three query heads of one
    KV head, block b's keys all equal to the unit vector e_b (so its summary is e_b
    exactly) and q_h[b] = the fixture's S(h, b); lambda = 1 selects the page's four
    consensus blocks, lambda = 0 (the largest head score alone) does not."""
    import test_oracle_pins as pins
    heads, _, top4, lam = pins._consensus_fixture()
    nb, D, B = 105, 128, 16
    w = Workload(layers=1, batch=1, hq=3, hkv=1, head_dim=D, block_tokens=B, ntok=[nb * B], k=4, window=0,
                 pool_slots=8, steps=1, select_mode=pi.PI_CONSENSUS, lam=lam)
    q_bits, _ = pins._one_hot_problem(heads, nb=nb, D=D)
    with make_pool(w) as pool:
        region = np.zeros((w.max_blocks, 1, 2, B, D), dtype=np.uint16)
        one = synth.f32_to_bf16(np.ones(1, dtype=np.float32))[0]
        for b in range(nb):
            region[b, 0, 0, :, b] = one
        host = pool.host_kv(0, 0)
        host[...] = region.reshape(host.shape)
        pool.update_summaries(0, [nb * B])
        torch.cuda.synchronize()
        sel = torch.empty((1, 4), dtype=torch.int32, device="cuda")
        nsel = torch.empty((1,), dtype=torch.int32, device="cuda")
        kreq = torch.tensor([4], dtype=torch.int32, device="cuda")
        for lam_, want_page in ((lam, True), (0.0, False)):
            pool.set_consensus_lambda(lam_)
            pool.select_topk(0, dev(q_bits[None]), kreq, sel, nsel)
            torch.cuda.synchronize()
            got = sorted(sel[0, : int(nsel[0])].cpu().tolist())
            assert (got == sorted(top4)) == want_page, (lam_, got)
            assert got == list(oracle.select_consensus(q_bits, np.eye(nb, D, dtype=np.float32)[:, None, :], 4, 0,
                                                       lam_))


@pytest.mark.parametrize("evict", [0, 1])
def test_consensus_multistep_pipeline(evict):
    """A consensus pool through pi_decode_step: 3 pipelined steps with appends,
    selections, tables, maps, bytes and attention checked against the oracle."""
    w = Workload(layers=2, batch=2, hq=32, hkv=8, head_dim=128, block_tokens=64, ntok=[4000, 2500], k=8, window=2,
                 pool_slots=14, steps=3, rho=0.9, heavy_frac=0.05, heavy_shift=2.0, seed=57, evict_policy=evict,
                 select_mode=pi.PI_CONSENSUS)
    L, R = w.layers, w.batch
    with make_pool(w) as pool:
        prefill(pool, w)
        om = OracleModel(w)
        qs = queries(w)
        for step in range(w.steps):
            kn, vn = new_tokens(w, step)
            kbud = np.full((L, R), w.k, dtype=np.int32)
            out = torch.empty((L, R, w.hq, w.head_dim), dtype=torch.int16, device="cuda")
            lse = torch.empty((L, R, w.hq), dtype=torch.float32, device="cuda")
            pool.decode_step(dev(qs[step]), dev(kn), dev(vn), dev(kbud), out, lse)
            torch.cuda.synchronize()
            assert pool.device_status() == pi.PI_OK
            sel_v, nsel_v, tab_v = pool.view_step()
            for l in range(L):
                om.append(l, kn[l], vn[l])
                ref_sel = om.select(l, qs[step][l], kbud[l])
                check_selection(sel_v[l], nsel_v[l], ref_sel, 1)
                ref_tab = om.recall(l, ref_sel)
                check_tables_maps_bytes(pool, om, w, l, ref_sel, ref_tab, tab_v[l])
                ref_out, ref_lse, _ = om.attention(l, qs[step][l], ref_sel)
                check_attention(out[l], lse[l], ref_out, ref_lse)


def test_selection_modes_accepted_per_pool():
    """A shared pool ranks by either score per call; a head-wise pool only per
    head; mismatches return PI_ERR_STATE; lambda must be finite and >= 0."""
    w = C1
    with make_pool(w) as pool:
        prefill(pool, w)
        q = dev(queries(w)[0][0])
        kreq = torch.tensor([w.k], dtype=torch.int32, device="cuda")
        sel = torch.empty((1, w.k + w.window), dtype=torch.int32, device="cuda")
        nsel = torch.empty((1,), dtype=torch.int32, device="cuda")
        om = OracleModel(w)
        for mode in (pi.PI_SHARED, pi.PI_CONSENSUS):
            pool.select_topk(0, q, kreq, sel, nsel, mode=mode)
            torch.cuda.synchronize()
            km = om.kmean[(0, 0)][: om.nb(0, 0)]
            qn = queries(w)[0][0][0]
            want = (oracle.select_shared(qn, km, w.k, w.window) if mode == pi.PI_SHARED
                    else oracle.select_consensus(qn, km, w.k, w.window, 0.5))
            assert np.array_equal(sel[0, : int(nsel[0])].cpu().numpy(), want)
        with pytest.raises(pi.PiError) as ei:
            pool.select_topk(0, q, kreq, sel, nsel, mode=pi.PI_HEADWISE)
        assert ei.value.status == pi.PI_ERR_STATE
        for bad in (-1.0, float("nan"), float("inf")):
            with pytest.raises(pi.PiError):
                pool.set_consensus_lambda(bad)


def _run_steps(w, setup, method=pi.PI_RECALL_UVA):
    """Decode w.steps pipelined steps on a fresh pool configured by setup(pool);
    returns every step's outputs and library state (host copies)."""
    L, R = w.layers, w.batch
    qs = queries(w)
    res = []
    with make_pool(w) as pool:
        setup(pool)
        prefill(pool, w)
        for step in range(w.steps):
            kn, vn = new_tokens(w, step)
            kbud = np.full((L, R), w.k, dtype=np.int32)
            kbud[-1, 0] = max(1, w.k // 2)
            out = torch.empty((L, R, w.hq, w.head_dim), dtype=torch.int16, device="cuda")
            lse = torch.empty((L, R, w.hq), dtype=torch.float32, device="cuda")
            compute = torch.cuda.Stream()
            pool.decode_step(dev(qs[step]), dev(kn), dev(vn), dev(kbud), out, lse, method=method, compute=compute)
            torch.cuda.synchronize()
            assert pool.device_status() == pi.PI_OK
            sel_v, nsel_v, tab_v = pool.view_step()
            res.append(dict(out=out.cpu().numpy(), lse=lse.cpu().numpy(), sel=sel_v.cpu().numpy(),
                            nsel=nsel_v.cpu().numpy(), tab=tab_v.cpu().numpy(),
                            sob=pool.view_slot_of_block().cpu().numpy(), bos=pool.view_block_of_slot().cpu().numpy(),
                            pool=pool.view_pool().cpu().numpy()))
    return res


@pytest.mark.parametrize("mode,evict", [(pi.PI_SHARED, 0), (pi.PI_SHARED, 1), (pi.PI_CONSENSUS, 0)],
                         ids=["shared", "shared_lru", "consensus"])
def test_dependent_schedule_gives_identical_results(mode, evict):
    """Interruptible layer-wise scheduling (guide, "Interruptible Layer-Wise
    Scheduling"): with dependent queries and 1, 2 or 3 interleaved request groups
    the decode step computes what the default schedule computes: selections,
    tables, slot maps and pool bytes bit for bit, attention outputs within the
    tolerances (a launch over fewer requests uses more splits, so the summation
    order differs), every step; the default run is itself checked against the
    oracle."""
    w = Workload(layers=3, batch=5, hq=32, hkv=8, head_dim=128, block_tokens=64, ntok=[4000, 2500, 3100, 700, 5000],
                 k=8, window=2, pool_slots=12, steps=3, rho=0.9, heavy_frac=0.05, seed=61, evict_policy=evict,
                 select_mode=mode)
    base = _run_steps(w, lambda pool: None)
    om = OracleModel(w)
    qs = queries(w)
    for step in range(w.steps):
        kn, vn = new_tokens(w, step)
        kbud = np.full((w.layers, w.batch), w.k, dtype=np.int32)
        kbud[-1, 0] = max(1, w.k // 2)
        for l in range(w.layers):
            om.append(l, kn[l], vn[l])
            ref_sel = om.select(l, qs[step][l], kbud[l])
            for r in range(w.batch):
                assert np.array_equal(base[step]["sel"][l, r, 0, : len(ref_sel[r])], ref_sel[r])
            om.recall(l, ref_sel)
            ref_out, ref_lse, _ = om.attention(l, qs[step][l], ref_sel)
            assert np.max(np.abs(bf16_to_f32(base[step]["out"][l].view(np.uint16)) - bf16_to_f32(ref_out))) <= OUT_ATOL
    for groups in (1, 2, 3):
        got = _run_steps(w, lambda pool, g=groups: pool.set_schedule(True, g))
        for s in range(w.steps):
            for key in ("sel", "nsel", "tab", "sob", "bos", "pool"):
                assert np.array_equal(got[s][key], base[s][key]), (groups, s, key)
            err = np.max(np.abs(bf16_to_f32(got[s]["out"].view(np.uint16)) - bf16_to_f32(base[s]["out"].view(np.uint16))))
            assert err <= OUT_ATOL, (groups, s, err)
            rel = np.abs(got[s]["lse"] - base[s]["lse"]) / np.maximum(np.abs(base[s]["lse"]), 1.0)
            assert rel.max() <= LSE_RTOL, (groups, s)


@pytest.mark.parametrize("mode,evict", [(pi.PI_SHARED, 0), (pi.PI_SHARED, 1), (pi.PI_CONSENSUS, 0),
                                        (pi.PI_HEADWISE, 0)], ids=["shared", "shared_lru", "consensus", "headwise"])
def test_fused_select_gather_gives_identical_results(mode, evict):
    """Selection, recall plan and gather of a layer as one launch: selections,
    tables, slot maps and pool bytes bit for bit equal to the unfused decode step,
    and the outputs too (the attention launches are the same), with the default
    grid, with 3 CTAs (every CTA takes many items), on one copy stream; under the
    dependent schedule with 2 or 3 request groups (their launches of a layer run
    at the same time on the groups' streams) the outputs are within the
    tolerances (launches over fewer requests split differently)."""
    w = Workload(layers=3, batch=5, hq=32, hkv=8, head_dim=128, block_tokens=64, ntok=[4000, 2500, 3100, 700, 5000],
                 k=8, window=2, pool_slots=12, steps=3, rho=0.9, heavy_frac=0.05, seed=67, evict_policy=evict,
                 select_mode=mode)
    base = _run_steps(w, lambda pool: None)
    setups = {"fused": lambda pool: pool.set_fused(True),
              "fused_3_ctas": lambda pool: pool.set_fused(True, 3),
              "fused_one_copy": lambda pool: (pool.set_fused(True), pool.set_copy_streams(1)),
              "fused_dependent_2": lambda pool: (pool.set_fused(True), pool.set_schedule(True, 2)),
              "fused_dependent_3": lambda pool: (pool.set_fused(True, 2), pool.set_schedule(True, 3))}
    for name, setup in setups.items():
        got = _run_steps(w, setup)
        for s in range(w.steps):
            for key in ("sel", "nsel", "tab", "sob", "bos", "pool"):
                assert np.array_equal(got[s][key], base[s][key]), (name, s, key)
            if not name.startswith("fused_dependent"):
                assert np.array_equal(got[s]["out"], base[s]["out"]), (name, s)
                assert np.array_equal(got[s]["lse"], base[s]["lse"]), (name, s)
            else:
                err = np.max(np.abs(bf16_to_f32(got[s]["out"].view(np.uint16)) -
                                    bf16_to_f32(base[s]["out"].view(np.uint16))))
                assert err <= OUT_ATOL, (name, s, err)


def test_schedule_arguments():
    w = C1
    with make_pool(w) as pool:
        for dep, g in ((2, 1), (1, 0), (1, 9), (1, 2)):  # batch 1: at most one group
            with pytest.raises(pi.PiError) as ei:
                pool.set_schedule(bool(dep) if dep < 2 else dep, g)
            assert ei.value.status == pi.PI_ERR_INVALID
        pool.set_schedule(True, 1)
        prefill(pool, w)
        L, R = w.layers, w.batch
        q = dev(queries(w)[0])
        kn, vn = new_tokens(w, 0)
        out = torch.empty((L, R, w.hq, w.head_dim), dtype=torch.int16, device="cuda")
        with pytest.raises(pi.PiError) as ei:
            pool.decode_step(q, dev(kn), dev(vn), dev(np.full((L, R), w.k, dtype=np.int32)), out,
                             method=pi.PI_RECALL_MEMCPY)
        assert ei.value.status == pi.PI_ERR_INVALID
        pool.set_schedule(False, 1)


@pytest.mark.parametrize("evict", [0, 1])
def test_headwise_pool_through_the_decode_step(evict):
    """The per-KV-head arm through pi_decode_step: per-head selections, fragment
    recall into per-head sub-slots and per-head attention, 3 pipelined steps with
    appends, checked against the oracle every layer and step."""
    w = Workload(layers=2, batch=2, hq=16, hkv=4, head_dim=128, block_tokens=32, ntok=[2000, 1500], k=6, window=2,
                 pool_slots=10, steps=3, seed=67, select_mode=1, evict_policy=evict, heavy_frac=0.05)
    L, R = w.layers, w.batch
    with make_pool(w) as pool:
        prefill(pool, w)
        om = OracleModel(w)
        qs = queries(w)
        for step in range(w.steps):
            kn, vn = new_tokens(w, step)
            kbud = np.full((L, R), w.k, dtype=np.int32)
            out = torch.empty((L, R, w.hq, w.head_dim), dtype=torch.int16, device="cuda")
            lse = torch.empty((L, R, w.hq), dtype=torch.float32, device="cuda")
            pool.decode_step(dev(qs[step]), dev(kn), dev(vn), dev(kbud), out, lse)
            torch.cuda.synchronize()
            assert pool.device_status() == pi.PI_OK
            sel_v, nsel_v, tab_v = pool.view_step()
            for l in range(L):
                om.append(l, kn[l], vn[l])
                ref_sel = om.select(l, qs[step][l], kbud[l])
                check_selection(sel_v[l], nsel_v[l], ref_sel, om.U)
                ref_tab = om.recall(l, ref_sel)
                check_tables_maps_bytes(pool, om, w, l, ref_sel, ref_tab, tab_v[l])
                ref_out, ref_lse, _ = om.attention(l, qs[step][l], ref_sel)
                check_attention(out[l], lse[l], ref_out, ref_lse)


@pytest.mark.parametrize("evict", [0, 1])
def test_pinned_layers_and_admission(evict):
    """IO-adaptive admission (guide, "2. IO-Adaptive Offloading Admission"): a
    pinned layer keeps room for every block, so blocks once recalled stay; a
    released layer drops what it held beyond P_r; every step matches the oracle
    run with the same residency changes. Then the controller's decisions: pin in
    the order 0, L-1, ... above 0.85 utilisation, release the last pinned below
    0.5, nothing in between; layers without reserved room cannot be pinned."""
    w = Workload(layers=3, batch=2, hq=32, hkv=8, head_dim=128, block_tokens=64, ntok=[3000, 2000], k=8, window=2,
                 pool_slots=12, steps=4, rho=0.5, heavy_frac=0.05, seed=71, evict_policy=evict)
    L, R = w.layers, w.batch
    cap = max(w.pool_slots, w.max_blocks)
    with make_pool(w, pin_layers=2) as pool:
        prefill(pool, w)
        om = OracleModel(w)
        with pytest.raises(pi.PiError) as ei:
            pool.pin_layer(1, True)
        assert ei.value.status == pi.PI_ERR_INVALID
        pool.pin_layer(0, True)
        om.pin(0, cap)
        assert pool.slots(0, 0) == cap and pool.slots(0, 1) == w.pool_slots
        qs = queries(w)
        held = [set() for _ in range(R)]
        for step in range(w.steps):
            if step == 2:
                pool.pin_layer(0, False)
                om.unpin(0)
                pool.pin_layer(2, True)
                om.pin(2, cap)
            kn, vn = new_tokens(w, step)
            kbud = np.full((L, R), w.k, dtype=np.int32)
            out = torch.empty((L, R, w.hq, w.head_dim), dtype=torch.int16, device="cuda")
            lse = torch.empty((L, R, w.hq), dtype=torch.float32, device="cuda")
            pool.decode_step(dev(qs[step]), dev(kn), dev(vn), dev(kbud), out, lse)
            torch.cuda.synchronize()
            assert pool.device_status() == pi.PI_OK
            sel_v, nsel_v, tab_v = pool.view_step()
            for l in range(L):
                om.append(l, kn[l], vn[l])
                ref_sel = om.select(l, qs[step][l], kbud[l])
                check_selection(sel_v[l], nsel_v[l], ref_sel, 1)
                ref_tab = om.recall(l, ref_sel)
                check_tables_maps_bytes(pool, om, w, l, ref_sel, ref_tab, tab_v[l])
                ref_out, ref_lse, _ = om.attention(l, qs[step][l], ref_sel)
                check_attention(out[l], lse[l], ref_out, ref_lse)
            if step < 2:  # while pinned, layer 0 never lets a block go
                sob = pool.view_slot_of_block().cpu().numpy()
                for r in range(R):
                    now = set(np.nonzero(sob[r, 0, 0] >= 0)[0].tolist())
                    assert held[r] <= now
                    held[r] = now
        # controller decisions (layer 2 pinned, layer 0 released at this point)
        assert pool.admission(0.90) == (0, True)
        assert pool.admission(0.95) == (-1, False)   # 0 and 2 pinned, 1 has no room
        assert pool.admission(0.70) == (-1, False)
        assert pool.admission(0.30) == (0, False)    # the last pinned goes first
        assert pool.admission(0.30) == (2, False)
        assert pool.admission(0.10) == (-1, False)
        assert pool.slots(1, 2) == w.pool_slots


@pytest.mark.parametrize("mode", [pi.PI_SHARED, pi.PI_CONSENSUS], ids=["shared", "consensus"])
def test_large_selection_sizes(mode):
    """Beyond the register-resident fast paths: 4 375 candidate blocks (more than
    the 4 096 a selection CTA keeps in registers, so keys are read from the score
    buffer), a budget of 1 100 blocks (more than the 512 one attention CTA takes,
    so at least three splits), a second request with a budget of 300."""
    w = Workload(layers=1, batch=2, hq=8, hkv=2, head_dim=64, block_tokens=16, ntok=[70000, 33000], k=1100, window=4,
                 pool_slots=1104, steps=1, seed=73, select_mode=mode)
    with make_pool(w) as pool:
        prefill(pool, w)
        om = OracleModel(w)
        run_layer(pool, om, w, 0, queries(w)[0][0], [1100, 300], pi.PI_RECALL_UVA, logits=False)


@pytest.mark.parametrize("mode", [pi.PI_SHARED, pi.PI_CONSENSUS], ids=["shared", "consensus"])
@pytest.mark.parametrize("ncands", [[1, 31, 300, 701, 1024], [1500, 2000]], ids=["cluster_form", "last_cta_form"])
def test_selection_ties_and_signed_zeros(ncands, mode):
    """Every block's keys are one constant from {-1, -1/2, -0, +0, 1/2, 1} (exact
    in bf16) and the query is all ones, so every score is an exact multiple of
    its block's constant: five distinct scores among up to 2 000 candidates, and
    blocks of -0 keys tie with blocks of +0 keys. At every budget from 0 to all
    candidates the selection must be the oracle's (equal scores by lower index),
    in both launch forms: up to 1 024 candidates a
    cluster per request with the one-warp top-k (1, 31, 300, 701 and 1 024
    candidates: one, one, two and four registers per lane, and the full 32), above
    that the last CTA of each request. Ragged last blocks."""
    hq, hkv, D, B, W, lam = 32, 8, 128, 16, 2, 0.5
    R = len(ncands)
    ntok = [B * (n + W) - 5 for n in ncands]
    nbs = [-(-t // B) for t in ntok]
    assert nbs == [n + W for n in ncands]
    mb = max(nbs) + 2
    kmax = max(ncands)
    pool = pi.Pool(1, R, hq, hkv, D, B, mb, kmax + W, kmax, W, select_mode=mode, host_layers=1)
    try:
        if mode == pi.PI_CONSENSUS:
            pool.set_consensus_lambda(lam)
        rng = np.random.default_rng(101 + R)
        vals = np.array([0xBF80, 0xBF00, 0x8000, 0x0000, 0x3F00, 0x3F80], dtype=np.uint16)
        kms = []
        for r in range(R):
            reg = pool.host_kv(0, r)
            reg[:] = vals[rng.integers(0, len(vals), size=mb)][:, None, None, None, None]
            kms.append(oracle.region_summaries(reg.copy(), ntok[r]))
        pool.update_summaries(0, ntok)
        torch.cuda.synchronize()
        q = np.full((R, hq, D), 0x3F80, dtype=np.uint16)
        for k in sorted({0, 1, 17, 31, 32, 33, 64, 300, 701, kmax}):
            sel = torch.full((R, kmax + W), -7, dtype=torch.int32, device="cuda")
            nsel = torch.full((R,), -7, dtype=torch.int32, device="cuda")
            pool.select_topk(0, dev(q), dev(np.full(R, k, dtype=np.int32)), sel, nsel, mode=mode)
            if mode == pi.PI_CONSENSUS:
                ref = [oracle.select_consensus(q[r], kms[r], k, W, lam) for r in range(R)]
            else:
                ref = [oracle.select_shared(q[r], kms[r], k, W) for r in range(R)]
            check_selection(sel, nsel, ref, 1)
        assert pool.device_status() == pi.PI_OK
    finally:
        pool.close()


@pytest.mark.parametrize("mode", [pi.PI_SHARED, pi.PI_CONSENSUS], ids=["shared", "consensus"])
@pytest.mark.parametrize("hq", [32, 64], ids=["G4_llama8b", "G8_llama70b"])
def test_gpu_selection_matches_exact_arithmetic(mode, hq):
    """The GPU's selection against the formula evaluated exactly, not only
    against the oracle's fp32 order: for every request whose exact ranking no
    rounding within the bound can change, the GPU's top-k is the exact top-k
    (mean-key score: sum over heads of q_h . kmean; consensus: per group the
    largest head score plus lambda x the mean, summed over groups). 12 requests of
    256 blocks of 16 tokens, 8 KV heads, d 128, 5 % heavy-hitter blocks."""
    import test_oracle_pins as pins
    hkv, B, D, nb, k, W, lam = 8, 16, 128, 256, 32, 2, 0.5
    w = Workload(layers=1, batch=12, hq=hq, hkv=hkv, head_dim=D, block_tokens=B, ntok=[nb * B] * 12, k=k, window=W,
                 pool_slots=k + W, steps=1, seed=37, heavy_frac=0.05, select_mode=mode, lam=lam)
    with make_pool(w) as pool:
        if mode == pi.PI_CONSENSUS:
            pool.set_consensus_lambda(lam)
        prefill(pool, w)
        om = OracleModel(w)
        q = queries(w)[0][0]
        sel = torch.full((w.batch, k + W), -7, dtype=torch.int32, device="cuda")
        nsel = torch.full((w.batch,), -7, dtype=torch.int32, device="cuda")
        pool.select_topk(0, dev(q), dev(np.full(w.batch, k, dtype=np.int32)), sel, nsel, mode=mode)
        torch.cuda.synchronize()
        assert pool.device_status() == pi.PI_OK
        check_selection(sel, nsel, om.select(0, q, [k] * w.batch), 1)
        got = sel.cpu().numpy()
        ncand = nb - W
        decided = 0
        for r in range(w.batch):
            km = om.kmean[(r, 0)][:ncand]
            if mode == pi.PI_CONSENSUS:
                exact, bound = pins.exact_consensus(q[r], km, lam)
            else:
                s64, a64 = pins._exact_scores(q[r], km)
                G = hq // hkv
                bound = ((G - 1) + hkv * D // 32 + 5 + 1) * 2.0 ** -24 * a64 * 1.01
                exact = s64
            top, ok = pins._decided_by_exact_arithmetic(exact, bound, k)
            if ok:
                # the W recent blocks are the highest ids; the top-k are the rest
                assert sorted(top) == sorted(int(b) for b in got[r] if 0 <= b < ncand), r
                decided += 1
        assert decided >= w.batch // 2
        print(f"{decided}/{w.batch} requests decided by exact arithmetic")


@pytest.mark.parametrize("fused", [False, True], ids=["separate", "fused"])
@pytest.mark.parametrize("mode", [pi.PI_SHARED, pi.PI_CONSENSUS, pi.PI_HEADWISE], ids=["shared", "consensus", "headwise"])
def test_features_together(mode, fused):
    """Dependent-query schedule with two request groups, a pinned layer, the
    least-recently-selected rule and each ranking, three pipelined steps, with
    selection and gather as separate launches or fused (2 CTAs per launch): every
    layer and step against the oracle run with the same residency."""
    w = Workload(layers=3, batch=3, hq=16, hkv=4, head_dim=128, block_tokens=32, ntok=[2500, 1800, 900], k=6,
                 window=2, pool_slots=9, steps=3, rho=0.7, heavy_frac=0.05, seed=79, evict_policy=1,
                 select_mode=mode)
    L, R = w.layers, w.batch
    cap = max(w.pool_slots, w.max_blocks)
    with make_pool(w, pin_layers=1) as pool:
        pool.set_schedule(True, 2)
        if fused:
            pool.set_fused(True, 2)
        prefill(pool, w)
        om = OracleModel(w)
        pool.pin_layer(0, True)
        om.pin(0, cap)
        qs = queries(w)
        for step in range(w.steps):
            kn, vn = new_tokens(w, step)
            kbud = np.full((L, R), w.k, dtype=np.int32)
            out = torch.empty((L, R, w.hq, w.head_dim), dtype=torch.int16, device="cuda")
            lse = torch.empty((L, R, w.hq), dtype=torch.float32, device="cuda")
            pool.decode_step(dev(qs[step]), dev(kn), dev(vn), dev(kbud), out, lse)
            torch.cuda.synchronize()
            assert pool.device_status() == pi.PI_OK
            sel_v, nsel_v, tab_v = pool.view_step()
            for l in range(L):
                om.append(l, kn[l], vn[l])
                ref_sel = om.select(l, qs[step][l], kbud[l])
                check_selection(sel_v[l], nsel_v[l], ref_sel, om.U)
                ref_tab = om.recall(l, ref_sel)
                check_tables_maps_bytes(pool, om, w, l, ref_sel, ref_tab, tab_v[l])
                ref_out, ref_lse, _ = om.attention(l, qs[step][l], ref_sel)
                check_attention(out[l], lse[l], ref_out, ref_lse)


MASS_ATOL = 1e-4   # fp32 logits (128 fused products) and fp32 sums over <= 32768 tokens per head


def _mass_case(w, l, kreq, sel=None, nsel=None, expect_status=pi.PI_OK):
    """Select (or take the given selection), then the attention mass of every head
    on the GPU against the fp64 oracle."""
    R, U, cap = w.batch, (w.hkv if w.select_mode == pi.PI_HEADWISE else 1), w.k + w.window
    with make_pool(w) as pool:
        prefill(pool, w)
        om = OracleModel(w)
        q = queries(w)[0][l]
        if sel is None:
            sel_d = torch.full((R * U, cap), -7, dtype=torch.int32, device="cuda")
            nsel_d = torch.full((R * U,), -7, dtype=torch.int32, device="cuda")
            pool.select_topk(l, dev(q), dev(np.asarray(kreq, dtype=np.int32)), sel_d, nsel_d)
            ref_sel = om.select(l, q, kreq)
            check_selection(sel_d, nsel_d, ref_sel, U)
        else:
            sel_d, nsel_d = dev(sel), dev(nsel)
            ref_sel = [[sel[r * U + g, :nsel[r * U + g]] for g in range(U)] if U > 1 else sel[r, :nsel[r]]
                       for r in range(R)]
        mass = torch.full((R, w.hq), float("nan"), dtype=torch.float32, device="cuda")
        pool.attention_mass(l, dev(q), sel_d, nsel_d, mass, per_head=U > 1)
        torch.cuda.synchronize()
        assert pool.device_status() == expect_status
        got = mass.cpu().numpy()
        for r in range(R):
            want = oracle.attention_mass(q[r], om.reg[(w.host_layer(l), r)], ref_sel[r], w.ntok[r], w.hkv)
            assert np.max(np.abs(got[r] - want)) <= MASS_ATOL, (r, got[r], want)
        return got


@pytest.mark.parametrize("mode", [pi.PI_SHARED, pi.PI_CONSENSUS, pi.PI_HEADWISE], ids=["shared", "consensus", "headwise"])
@pytest.mark.parametrize("hq,hkv,D,B", [(32, 8, 128, 64), (8, 2, 64, 16), (64, 8, 128, 64), (12, 3, 64, 32)],
                         ids=["8B", "C1_shape", "70B_G8", "G4_odd_hkv"])
def test_attention_mass_matches_oracle(mode, hq, hkv, D, B):
    """Attention mass each head keeps under the library's own selection (guide,
    "SoloHead Sparse Selection", "2. High Attention Mass Preservation"): GPU fp32
    against the fp64 oracle within MASS_ATOL; ragged tails, a one-block request,
    the second layer of an aliased host store."""
    w = Workload(layers=2, batch=3, hq=hq, hkv=hkv, head_dim=D, block_tokens=B, ntok=[5000, 2500, 40], k=12,
                 window=2, pool_slots=16, seed=61 + hq + D, heavy_frac=0.05, select_mode=mode, host_layers=1)
    _mass_case(w, 1, [w.k, 5, 3])


def test_attention_mass_degenerate_selections():
    """Every block -> 1; nothing -> 0; a repeated id counts once; one id past the
    context is skipped and flagged in the status word, not read."""
    w = Workload(layers=1, batch=3, hq=8, hkv=2, head_dim=64, block_tokens=16, ntok=[1000, 300, 37], k=70,
                 window=0, pool_slots=70, seed=62)
    cap = w.k
    sel = np.full((3, cap), -1, dtype=np.int32)
    nsel = np.array([63, 0, 4], dtype=np.int32)
    sel[0, :63] = np.arange(63)
    sel[2, :4] = [1, 1, 2, 0]
    got = _mass_case(w, 0, None, sel, nsel)
    assert np.all(np.abs(got[0] - 1.0) <= MASS_ATOL) and np.all(got[1] == 0.0)
    sel[2, :4] = [1, 1, 2, 9]     # request 2 holds 3 blocks: block 9 is past its context
    with make_pool(w) as pool:
        prefill(pool, w)
        q = queries(w)[0][0]
        mass = torch.empty((3, w.hq), dtype=torch.float32, device="cuda")
        pool.attention_mass(0, dev(q), dev(sel), dev(nsel), mass)
        torch.cuda.synchronize()
        assert pool.device_status() == pi.PI_ERR_DEVICE
        want = oracle.attention_mass(q[2], synth.kv_region(w.seed, 0, 2, 37, w.max_blocks, 2, 16, 64),
                                     np.array([1, 2]),
                                     37, w.hkv)
        assert np.max(np.abs(mass[2].cpu().numpy() - want)) <= MASS_ATOL


def test_attention_mass_full_context_8b_shape():
    """Two requests of the Llama-3-8B shape at 32768 tokens (512 blocks, top-32 +
    2): every head against the oracle, shared selection."""
    w = Workload(layers=1, batch=2, hq=32, hkv=8, head_dim=128, block_tokens=64, ntok=[32768, 32768], k=32,
                 window=2, pool_slots=128, seed=63, heavy_frac=0.05)
    _mass_case(w, 0, [32, 32])
