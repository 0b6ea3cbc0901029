"""Pins of the CPU oracle to things other than itself (no GPU needed).

Each group below checks one oracle function against brute force, a closed
form, an invariant the definition fixes, or a value printed on the pages, so
that a dropped term, a wrong sign or index, or a transposed operand fails.
"""
import itertools
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
import synth

GOLD = os.path.join(os.path.dirname(__file__), "golden")
rng = np.random.default_rng(1234)


def bf16_bits(x):
    return synth.f32_to_bf16(np.asarray(x, dtype=np.float32))


def f32_of_bf16(bits):
    return synth.bf16_to_f32(bits)


# ------------------------------------------------------------------ bf16 rounding
def test_bf16_rne_known_values():
    assert oracle.bf16_rne(1.0) == 0x3F80
    assert oracle.bf16_rne(-2.0) == 0xC000
    assert oracle.bf16_rne(1.0 + 2.0 ** -8) == 0x3F80      # tie -> even
    assert oracle.bf16_rne(1.0 + 3 * 2.0 ** -8) == 0x3F82  # tie -> even (up)
    assert oracle.bf16_rne(1.0 + 2.0 ** -8 + 2.0 ** -30) == 0x3F81  # just above the tie
    assert oracle.bf16_rne(0.0) == 0 and oracle.bf16_rne(-0.0) == 0x8000
    assert oracle.bf16_rne(1e39) == 0x7F80
    assert oracle.bf16_rne(2.0 ** -133) == 0x0001           # smallest bf16 subnormal


def test_bf16_rne_matches_independent_fp32_path():
    # for fp32-representable inputs the direct fp64 rounding must equal the
    # generator's independent fp32 bit-trick rounding
    x = rng.standard_normal(4000).astype(np.float32) * np.float32(3.0)
    a = np.array([oracle.bf16_rne(float(v)) for v in x], dtype=np.uint16)
    assert np.array_equal(a, synth.f32_to_bf16(x))


# ------------------------------------------------------------------ a-1 summaries
def _block(hkv, B, D, fill=None):
    blk = np.zeros((hkv, 2, B, D), dtype=np.uint16)
    if fill is not None:
        blk[...] = fill
    return blk


def test_summary_constant_block_is_exact():
    for n in (1, 3, 16, 64):
        blk = _block(2, 64, 8, bf16_bits(0.3)[()])
        km = oracle.block_summary(blk, n)
        # exact for power-of-two n; within 1 ulp-ish for others
        ref = np.float32(f32_of_bf16(bf16_bits(0.3)))
        if n & (n - 1) == 0:
            assert np.all(km == ref)
        else:
            assert np.all(np.abs(km - ref) <= 4 * np.spacing(ref))


def test_summary_uses_keys_of_its_head_and_valid_tokens_only():
    hkv, B, D = 3, 16, 8
    blk = _block(hkv, B, D)
    for g in range(hkv):
        blk[g, 0, :5] = bf16_bits(float(g + 1))     # K of head g = g+1 on valid tokens
        blk[g, 0, 5:] = bf16_bits(1000.0)           # tokens past n_valid must be ignored
        blk[g, 1] = bf16_bits(-77.0)                # V must be ignored
    km = oracle.block_summary(blk, 5)
    for g in range(hkv):
        assert np.all(km[g] == np.float32(g + 1))


def test_summary_exact_rational_mean():
    # small multiples of 1/8: every partial sum is exact in fp32, so the result is
    # the correctly rounded exact mean
    B, D = 32, 4
    vals = rng.integers(-40, 40, size=(B, D)) / 8.0
    blk = _block(1, B, D)
    blk[0, 0] = bf16_bits(vals)
    for n in (1, 7, 32):
        km = oracle.block_summary(blk, n)
        for d in range(D):
            exact = Fraction(sum(Fraction(int(v * 8), 8) for v in vals[:n, d]), n)
            assert km[0, d] == np.float32(float(exact))


def test_summary_error_bound_random():
    B, D = 64, 128
    x = rng.standard_normal((B, D)).astype(np.float32)
    blk = _block(1, B, D)
    blk[0, 0] = bf16_bits(x)
    xf = f32_of_bf16(blk[0, 0]).astype(np.float64)
    km = oracle.block_summary(blk, B)
    u = 2.0 ** -24
    for d in range(D):
        exact = xf[:, d].sum() / B
        bound = (B - 1) * u * np.abs(xf[:, d]).sum() / B + u * abs(exact) + 1e-30
        assert abs(km[0, d] - exact) <= bound


def test_region_summaries_tail_block():
    reg = synth.kv_region(3, 0, 0, 100, 8, 2, 16, 8)
    km = oracle.region_summaries(reg, 100)
    assert km.shape == (7, 2, 8)
    # tail block 6 holds 4 tokens
    direct = f32_of_bf16(reg[6, :, 0, :4]).astype(np.float64).mean(axis=1)
    assert np.allclose(km[6], direct, rtol=1e-6, atol=1e-7)


# ------------------------------------------------------------------ a-2 score
def test_score_integer_inputs_equal_per_head_definition():
    """Exact small integers: the grouped fp32 score must equal the per-head integer
    sum  sum_h q_h . kmean[b, h // G]  computed with Python ints."""
    hq, hkv, D = 8, 2, 32
    G = hq // hkv
    q = rng.integers(-3, 4, size=(hq, D))
    km = rng.integers(-3, 4, size=(hkv, D))
    exact = sum(int(q[h, d]) * int(km[h // G, d]) for h in range(hq) for d in range(D))
    qs = oracle.qsum(bf16_bits(q.astype(np.float32)), hkv)
    s = oracle.score(qs, km.astype(np.float32))
    assert s == float(exact)


def test_score_one_hot_picks_element():
    E = 256
    km = rng.standard_normal(E).astype(np.float32)
    for e in (0, 5, 127, 128, 200, 255):
        qs = np.zeros(E, dtype=np.float32)
        qs[e] = 1.0
        assert oracle.score(qs, km) == km[e]


def test_score_error_bound_random():
    for E in (64, 128, 1024):
        qs = rng.standard_normal(E).astype(np.float32)
        km = (rng.standard_normal(E) / 8).astype(np.float32)
        exact = float(np.dot(qs.astype(np.float64), km.astype(np.float64)))
        bound = E * 2.0 ** -24 * float(np.abs(qs.astype(np.float64) * km).sum())
        assert abs(oracle.score(qs, km) - exact) <= bound


# ------------------------------------------------------------------ a-2 top-k
def _brute_topk(scores, k):
    """Among all k-subsets of the candidates, the one with the largest score sum
    (exact rationals); ties broken by the lexicographically smallest index tuple."""
    n = len(scores)
    best, best_key = None, None
    fr = [Fraction(float(s)) for s in scores]
    for comb in itertools.combinations(range(n), k):
        key = (-sum(fr[i] for i in comb), comb)
        if best_key is None or key < best_key:
            best, best_key = comb, key
    return list(best)


@pytest.mark.parametrize("seed", range(40))
def test_topk_matches_brute_force_with_ties(seed):
    r = np.random.default_rng(seed)
    nb = int(r.integers(1, 11))
    W = int(r.integers(0, 3))
    k = int(r.integers(0, nb + 2))
    scores = r.integers(-2, 3, size=nb).astype(np.float32)  # many ties
    sel = oracle.select_topk(scores, nb, k, W)
    ncand = max(nb - W, 0)
    kk = min(k, ncand)
    want = sorted(_brute_topk(scores[:ncand], kk) + list(range(ncand, nb)))
    assert list(sel) == want


def test_topk_invariant_random_large():
    for seed in range(20):
        r = np.random.default_rng(100 + seed)
        nb, W, k = 513, 2, 32
        scores = r.standard_normal(nb).astype(np.float32)
        scores[r.integers(0, nb, 50)] = scores[0]  # some ties
        sel = oracle.select_topk(scores, nb, k, W)
        assert list(sel) == sorted(sel) and len(sel) == k + W
        assert set(range(nb - W, nb)) <= set(sel)
        T = [b for b in sel if b < nb - W]
        rest = [b for b in range(nb - W) if b not in set(T)]
        worst_in = max(T, key=lambda b: (-scores[b], b))
        best_out = min(rest, key=lambda b: (-scores[b], b))
        assert (-scores[worst_in], worst_in) < (-scores[best_out], best_out)


def test_topk_zero_query_takes_lowest_indices():
    q = np.zeros((8, 64), dtype=np.uint16)
    km = rng.standard_normal((256, 2, 64)).astype(np.float32)
    sel = oracle.select_shared(q, km, 32, 4)
    assert list(sel) == list(range(32)) + [252, 253, 254, 255]


def test_topk_negative_zero_ties_plus_zero():
    scores = np.array([0.0, -0.0, 0.0, -1.0], dtype=np.float32)
    assert list(oracle.select_topk(scores, 4, 2, 0)) == [0, 1]
    scores = np.array([-0.0, 0.0, -1.0], dtype=np.float32)
    assert list(oracle.select_topk(scores, 3, 1, 0)) == [0]


def test_topk_degenerate_sizes():
    s = np.arange(10, dtype=np.float32)
    assert list(oracle.select_topk(s, 10, 100, 2)) == list(range(10))  # k >= candidates
    assert list(oracle.select_topk(s, 3, 5, 4)) == [0, 1, 2]           # nb <= W
    assert list(oracle.select_topk(s, 10, 0, 2)) == [8, 9]             # k = 0
    assert list(oracle.select_topk(s, 0, 4, 2)) == []                  # empty


def test_headwise_equals_shared_when_one_kv_head():
    q = bf16_bits(rng.standard_normal((4, 128)))
    km = rng.standard_normal((300, 1, 128)).astype(np.float32)
    hw = oracle.select_headwise(q, km, 20, 2)
    sh = oracle.select_shared(q, km, 20, 2)
    assert list(hw[0]) == list(sh)


def test_headwise_uses_its_own_head():
    # head 1 summaries favour blocks 0..4; head 0 favours 10..14
    hq, hkv, D, nb = 4, 2, 64, 20
    q = bf16_bits(np.ones((hq, D)))
    km = np.zeros((nb, hkv, D), dtype=np.float32)
    km[10:15, 0] = 1.0
    km[0:5, 1] = 1.0
    hw = oracle.select_headwise(q, km, 5, 0)
    assert list(hw[0]) == list(range(10, 15)) and list(hw[1]) == list(range(0, 5))


def test_fragmentation_worked_example():
    """PulseInfer Guide, "SoloHead Sparse Selection": 3 heads x 3 blocks -> 7 unique."""
    sets, union = [], None
    with open(os.path.join(GOLD, "solohead_fragmentation.txt")) as f:
        for line in f:
            if line.startswith("head"):
                sets.append([int(x) for x in line.split(":")[1].split()])
            elif line.startswith("union_blocks"):
                union = int(line.split(":")[1])
    assert oracle.union_fragments(sets) == union == 7


# ------------------------------------------------------------------ sizes
def test_kv_and_block_sizes_printed_on_pages():
    vals = {}
    with open(os.path.join(GOLD, "kv_sizes.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                k, v = line.split()
                vals[k] = float(v)
    b8 = oracle.kv_cache_bytes(int(vals["kv8b_layers"]), int(vals["kv8b_hkv"]), int(vals["kv8b_d"]), int(vals["kv8b_seq"]))
    assert round(b8 / 1e9, 1) == vals["kv8b_gb_printed"]
    b70 = oracle.kv_cache_bytes(int(vals["kv70b_layers"]), int(vals["kv70b_hkv"]), int(vals["kv70b_d"]), int(vals["kv70b_seq"]))
    assert b70 / 1e9 > vals["kv70b_gb_printed_lower_bound"] and round(b70 / 1e9, 1) == 41.9
    assert oracle.block_bytes(int(vals["block_hkv"]), int(vals["block_tokens"]), int(vals["block_d"])) == 65536
    # Llama-3-70B slice of 8 layers, batch 16, 131072 tokens: "~69 GB" of host KV
    assert round(16 * oracle.kv_cache_bytes(8, 8, 128, 131072) / 1e9, 1) == 68.7


# ------------------------------------------------------------------ a-3 plan
def test_plan_hand_worked_example():
    # pool of 4 slots holding blocks 5, 7, 9 in slots 0..2; select [1, 7, 8]
    sob = np.full(16, -1, dtype=np.int32)
    bos = np.array([5, 7, 9, -1], dtype=np.int32)
    for s, b in enumerate(bos):
        if b >= 0:
            sob[b] = s
    table, mb, ms, ev = oracle.recall_plan(np.array([1, 7, 8]), sob, bos)
    # missing [1, 8]; free slots ascending [0 (5 unselected), 2 (9 unselected), 3 (empty)]
    assert list(mb) == [1, 8] and list(ms) == [0, 2] and list(ev) == [5, 9]
    assert list(table) == [0, 1, 2]
    assert list(bos) == [1, 7, 8, -1]
    assert sob[5] == -1 and sob[9] == -1 and sob[1] == 0 and sob[7] == 1 and sob[8] == 2


def test_plan_pool_too_small_leaves_maps():
    sob = np.full(8, -1, dtype=np.int32)
    bos = np.full(2, -1, dtype=np.int32)
    assert oracle.recall_plan(np.array([0, 1, 2]), sob, bos) is None
    assert np.all(sob == -1) and np.all(bos == -1)


def test_plan_invariants_random_sequence():
    r = np.random.default_rng(7)
    nb, P = 200, 40
    sob = np.full(nb, -1, dtype=np.int32)
    bos = np.full(P, -1, dtype=np.int32)
    for step in range(60):
        sel = np.sort(r.choice(nb, size=int(r.integers(0, P + 1)), replace=False)).astype(np.int32)
        before = {int(b): int(s) for s, b in enumerate(bos) if b >= 0}
        out = oracle.recall_plan(sel, sob, bos)
        assert out is not None
        table, mb, ms, ev = out
        assert set(mb) == set(int(b) for b in sel) - set(before)          # only missing move
        for b in sel:                                                    # hits stay put
            if int(b) in before:
                assert sob[b] == before[int(b)]
        assert all(e not in set(sel.tolist()) for e in ev if e >= 0)      # evict unselected only
        assert list(table) == [sob[b] for b in sel]
        for s in range(P):                                               # maps inverse
            if bos[s] >= 0:
                assert sob[bos[s]] == s
        assert (sob >= 0).sum() == (bos >= 0).sum()


def test_plan_lru_hand_worked_example():
    # 4 slots hold 5 (last selected at epoch 3), 7 (epoch 1), 9 (epoch 2); slot 3 empty.
    sob = np.full(16, -1, dtype=np.int32)
    bos = np.array([5, 7, 9, -1], dtype=np.int32)
    stamp = np.array([3, 1, 2, -1], dtype=np.int32)
    for s, b in enumerate(bos):
        if b >= 0:
            sob[b] = s
    # epoch 4 selects [1, 8, 9]: 9 hits; 1 and 8 miss. Free: slot 3 (empty, first),
    # then slot 1 (block 7, epoch 1) before slot 0 (block 5, epoch 3).
    table, mb, ms, ev = oracle.recall_plan_lru(np.array([1, 8, 9]), sob, bos, stamp, 4)
    assert list(mb) == [1, 8] and list(ms) == [3, 1] and list(ev) == [-1, 7]
    assert list(table) == [3, 1, 2]
    assert list(bos) == [5, 8, 9, 1] and list(stamp) == [3, 4, 4, 4]


def test_plan_lru_evicts_least_recently_selected_invariant():
    r = np.random.default_rng(11)
    nb, P = 120, 24
    sob = np.full(nb, -1, dtype=np.int32)
    bos = np.full(P, -1, dtype=np.int32)
    stamp = np.full(P, -1, dtype=np.int32)
    for epoch in range(1, 80):
        sel = np.sort(r.choice(nb, size=int(r.integers(1, P + 1)), replace=False)).astype(np.int32)
        before_bos, before_stamp = bos.copy(), stamp.copy()
        out = oracle.recall_plan_lru(sel, sob, bos, stamp, epoch)
        assert out is not None
        table, mb, ms, ev = out
        S = set(sel.tolist())
        # every evicted slot is no more recent than any unselected resident that was kept
        kept_unsel = [before_stamp[s] for s in range(P) if before_bos[s] >= 0 and before_bos[s] not in S
                      and s not in set(ms.tolist())]
        for s in ms:
            if before_bos[s] >= 0:
                assert not any(k < before_stamp[s] for k in kept_unsel)
        assert all(stamp[t] == epoch for t in table)
        assert list(table) == [sob[b] for b in sel]
        for s in range(P):
            if bos[s] >= 0:
                assert sob[bos[s]] == s


# ------------------------------------------------------------------ a-5 attention
def _dense_inputs(reg, ntok, hkv, sel):
    B = reg.shape[3]
    Ks, Vs = [], []
    for g in range(hkv):
        kk, vv = [], []
        for b in sel:
            nv = min(B, ntok - b * B)
            kk.append(oracle.bf16_to_f64(reg[b, g, 0, :nv]))
            vv.append(oracle.bf16_to_f64(reg[b, g, 1, :nv]))
        Ks.append(np.concatenate(kk))
        Vs.append(np.concatenate(vv))
    return np.stack(Ks), np.stack(Vs)


@pytest.mark.parametrize("ntok", [4096, 1000, 17])
def test_attention_all_blocks_equals_dense(ntok):
    hq, hkv, B, D = 8, 2, 16, 64
    nbmax = -(-ntok // B) + 1
    reg = synth.kv_region(5, 0, 0, ntok, nbmax, hkv, B, D)
    q = synth.normal_bf16(5, synth.KIND_MISC, 0, 0, hq * D).reshape(hq, D)
    nb = -(-ntok // B)
    km = oracle.region_summaries(reg, ntok)
    sel = oracle.select_shared(q, km, nb, 4)        # k >= candidates: every block
    assert list(sel) == list(range(nb))
    out, lse, _ = oracle.attention(q, reg, sel, ntok, hkv)
    K, V = _dense_inputs(reg, ntok, hkv, sel)
    dout, dlse = oracle.dense_attention_fp64(oracle.bf16_to_f64(q), K, V)
    assert np.array_equal(out, np.array([[oracle.bf16_rne(v) for v in row] for row in dout], dtype=np.uint16))
    assert np.allclose(lse, dlse, rtol=1e-12, atol=1e-12)
    torch = pytest.importorskip("torch")
    G = hq // hkv
    qt = torch.tensor(oracle.bf16_to_f64(q)).reshape(1, hq, 1, D)
    kt = torch.tensor(K).repeat_interleave(G, 0).reshape(1, hq, -1, D)
    vt = torch.tensor(V).repeat_interleave(G, 0).reshape(1, hq, -1, D)
    ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt).reshape(hq, D).numpy()
    assert np.max(np.abs(oracle.bf16_to_f64(out) - ref)) <= 2.0 ** -8 * np.max(np.abs(ref)) + 1e-12


def test_attention_weights_sum_to_one_and_gqa_mapping():
    hq, hkv, B, D, ntok = 8, 2, 16, 64, 300
    reg = synth.kv_region(6, 0, 0, ntok, 20, hkv, B, D)
    for g in range(hkv):
        reg[:, g, 1] = np.where(np.arange(B)[None, :, None] >= 0, bf16_bits(float(g + 1)), 0)
    q = synth.normal_bf16(6, synth.KIND_MISC, 0, 0, hq * D).reshape(hq, D)
    sel = np.array([0, 3, 7, 18], dtype=np.int32)
    out, _, _ = oracle.attention(q, reg, sel, ntok, hkv)
    G = hq // hkv
    for h in range(hq):
        assert np.all(oracle.bf16_to_f64(out[h]) == h // G + 1)   # convex weights sum to 1


def test_attention_single_token_and_equal_logits():
    hq, hkv, B, D = 4, 1, 16, 64
    reg = synth.kv_region(8, 0, 0, 33, 4, hkv, B, D)
    q = synth.normal_bf16(8, synth.KIND_MISC, 0, 0, hq * D).reshape(hq, D)
    out, lse, lg = oracle.attention(q, reg, np.array([2], dtype=np.int32), 33, hkv, want_logits=True)
    assert np.array_equal(out, np.repeat(reg[2, 0, 1, 0][None], hq, 0))   # one valid token: out = V
    # logits of that token equal the plain dot product / sqrt(D)
    k = oracle.bf16_to_f64(reg[2, 0, 0, 0])
    for h in range(hq):
        assert math.isclose(lg[h, 0, 0], float(oracle.bf16_to_f64(q[h]) @ k) / 8.0, rel_tol=1e-12)
        assert math.isclose(lse[h], lg[h, 0, 0], rel_tol=1e-12)
    q0 = np.zeros((hq, D), dtype=np.uint16)
    sel = np.array([0, 1], dtype=np.int32)
    out, lse, _ = oracle.attention(q0, reg, sel, 33, hkv)
    mean = oracle.bf16_to_f64(reg[0:2, 0, 1].reshape(-1, D)).mean(axis=0)
    assert np.array_equal(out[0], np.array([oracle.bf16_rne(v) for v in mean], dtype=np.uint16))
    assert math.isclose(lse[0], math.log(32), rel_tol=1e-12)


def test_attention_ignores_tokens_past_ntok():
    hq, hkv, B, D, ntok = 8, 2, 16, 64, 40   # tail block 2 holds 8 tokens
    reg = synth.kv_region(9, 0, 0, ntok, 4, hkv, B, D)
    q = synth.normal_bf16(9, synth.KIND_MISC, 0, 0, hq * D).reshape(hq, D)
    sel = np.array([0, 2], dtype=np.int32)
    a, la, _ = oracle.attention(q, reg, sel, ntok, hkv)
    reg2 = reg.copy()
    reg2[2, :, :, 8:] = bf16_bits(50.0)
    b, lb, _ = oracle.attention(q, reg2, sel, ntok, hkv)
    assert np.array_equal(a, b) and np.array_equal(la, lb)


def test_attention_empty_selection():
    reg = synth.kv_region(1, 0, 0, 16, 2, 1, 16, 64)
    q = synth.normal_bf16(1, synth.KIND_MISC, 0, 0, 4 * 64).reshape(4, 64)
    out, lse, _ = oracle.attention(q, reg, np.zeros(0, dtype=np.int32), 16, 1)
    assert np.all(out == 0) and np.all(np.isneginf(lse))


def test_attention_headwise_selection_per_head():
    hq, hkv, B, D, ntok = 8, 2, 16, 64, 160
    reg = synth.kv_region(2, 0, 0, ntok, 10, hkv, B, D)
    q = synth.normal_bf16(2, synth.KIND_MISC, 0, 0, hq * D).reshape(hq, D)
    sels = [np.array([1, 4], dtype=np.int32), np.array([0, 2, 9], dtype=np.int32)]
    out, lse, _ = oracle.attention(q, reg, sels, ntok, hkv)
    for g in range(hkv):
        o1, l1, _ = oracle.attention(q, reg, sels[g], ntok, hkv)
        G = hq // hkv
        assert np.array_equal(out[g * G:(g + 1) * G], o1[g * G:(g + 1) * G])


# ------------------------------------------------------------------ consensus score
def _consensus_fixture():
    heads, top3, top4, lam = {}, {}, None, None
    with open(os.path.join(GOLD, "solohead_consensus_example.txt")) as f:
        for line in f:
            if line.startswith("scores head"):
                h = int(line.split(":")[0].split()[-1])
                heads[h] = {int(kv.split("=")[0]): int(kv.split("=")[1]) for kv in line.split(":")[1].split()}
            elif line.startswith("top3 head"):
                h = int(line.split(":")[0].split()[-1])
                top3[h] = [int(x) for x in line.split(":")[1].split()]
            elif line.startswith("consensus_lambda"):
                lam = float(line.split(":")[1])
            elif line.startswith("consensus_top4"):
                top4 = [int(x) for x in line.split(":")[1].split()]
    return heads, top3, top4, lam


def _one_hot_problem(heads, nb=105, D=128):
    """q[h][b] = S(h, b) and kmean[b] = e_b (one KV head), so q_h . kmean[b] = S(h, b) exactly."""
    hq = len(heads)
    q = np.zeros((hq, D), dtype=np.float64)
    for h, sc in heads.items():
        for b, v in sc.items():
            q[h, b] = v
    km = np.zeros((nb, 1, D), dtype=np.float32)
    for b in range(nb):
        km[b, 0, b] = 1.0
    return synth.f32_to_bf16(q.astype(np.float32)), km


def test_consensus_worked_example_of_the_guide():
    heads, top3, top4, lam = _consensus_fixture()
    q, km = _one_hot_problem(heads)
    nb = km.shape[0]
    for h, want in top3.items():
        sc = np.array([oracle.head_score(q[h], km[b, 0]) for b in range(nb)], dtype=np.float32)
        assert list(oracle.select_topk(sc, nb, 3, 0)) == sorted(want)
    assert list(oracle.select_consensus(q, km, 4, 0, lam)) == sorted(top4)
    # the rule needs both terms: the largest head score alone, or the mean alone, picks another set
    max_only = np.array([max(heads[h].get(b, 0) for h in heads) for b in range(nb)], dtype=np.float32)
    mean_only = np.array([sum(heads[h].get(b, 0) for h in heads) / 3 for b in range(nb)], dtype=np.float32)
    assert list(oracle.select_topk(max_only, nb, 4, 0)) != sorted(top4)
    assert list(oracle.select_topk(mean_only, nb, 4, 0)) != sorted(top4)
    # the union a head-wise recall would move, against the consensus set
    assert oracle.union_fragments(list(top3.values())) == 7 and len(top4) == 4


@pytest.mark.parametrize("hq,hkv,D", [(8, 8, 128), (16, 8, 128), (32, 8, 128), (64, 8, 128), (8, 2, 64), (12, 3, 64)])
@pytest.mark.parametrize("lam", [0.0, 0.25, 0.5, 1.0])
def test_consensus_score_exact_small_integers(hq, hkv, D, lam):
    """Small integer queries and quarter-integer summaries keep every product and
    sum exact in fp32 (G a power of two keeps the mean exact), so the oracle must
    equal the formula evaluated in exact rational arithmetic: per group the largest
    head score plus lam times their mean, summed over groups."""
    from fractions import Fraction
    G = hq // hkv
    if G & (G - 1):
        pytest.skip("mean exact only for power-of-two groups")
    rng = np.random.default_rng(hq * 131 + hkv * 7 + D + int(lam * 4))
    nb = 40
    qi = rng.integers(-3, 4, size=(hq, D))
    ki = rng.integers(-8, 9, size=(nb, hkv, D))
    q = synth.f32_to_bf16(qi.astype(np.float32))
    km = (ki / 4.0).astype(np.float32)
    want = []
    for b in range(nb):
        tot = Fraction(0)
        for g in range(hkv):
            s_h = [Fraction(int(np.dot(qi[g * G + j], ki[b, g])), 4) for j in range(G)]
            tot += max(s_h) + Fraction(lam).limit_denominator() * sum(s_h) / G
        want.append(tot)
    got = [Fraction(oracle.consensus_score(q, km[b], lam)) for b in range(nb)]
    assert got == want
    # the selection is the (score desc, index asc) order of those exact scores
    order = sorted(range(nb - 2), key=lambda b: (-want[b], b))[:7]
    assert list(oracle.select_consensus(q, km, 7, 2, lam)) == sorted(order + [nb - 2, nb - 1])


def test_consensus_one_head_per_group_is_the_scaled_shared_score():
    """G = 1: max = mean = the head's score, so consensus = (1 + lam) x shared score;
    with exact inputs the two selections coincide."""
    rng = np.random.default_rng(5)
    hkv, D, nb = 8, 128, 60
    qi = rng.integers(-3, 4, size=(hkv, D))
    ki = rng.integers(-8, 9, size=(nb, hkv, D))
    q = synth.f32_to_bf16(qi.astype(np.float32))
    km = (ki / 4.0).astype(np.float32)
    s_shared, sc_shared = oracle.select_shared(q, km, 10, 2, return_scores=True)
    s_cons, sc_cons = oracle.select_consensus(q, km, 10, 2, 0.5, return_scores=True)
    assert np.array_equal(sc_cons, (1.5 * sc_shared).astype(np.float32))
    assert np.array_equal(s_shared, s_cons)


def test_consensus_score_close_to_fp64_formula_on_gaussian_inputs():
    """Realistic values: the fp32 score agrees with the formula in fp64 within a
    few fp32 rounding steps of the operands' magnitude."""
    rng = np.random.default_rng(9)
    hq, hkv, D, nb = 32, 8, 128, 30
    q = synth.f32_to_bf16(rng.standard_normal((hq, D)).astype(np.float32))
    km = rng.standard_normal((nb, hkv, D)).astype(np.float32)
    qf = synth.bf16_to_f32(q).astype(np.float64)
    G = hq // hkv
    for b in range(nb):
        tot = 0.0
        for g in range(hkv):
            s_h = qf[g * G:(g + 1) * G] @ km[b, g].astype(np.float64)
            tot += s_h.max() + 0.5 * s_h.mean()
        got = oracle.consensus_score(q, km[b], 0.5)
        assert abs(got - tot) <= 1e-4 * (1.0 + np.abs(qf).sum() * 0.1)


# ------------------------------------------------------------------ pinned-layer plan
def test_pinned_plan_takes_empty_slots_first_hand_example():
    """Slots [7, -, 3, -, 9], selection {3, 4, 5}: the lowest-free-slot rule puts 4
    in slot 0 (evicting 7) and 5 in slot 1; a layer held whole in HBM puts them in
    the empty slots 1 and 3 and evicts nothing."""
    def maps():
        bos = np.array([7, -1, 3, -1, 9], dtype=np.int32)
        sob = np.full(12, -1, dtype=np.int32)
        for s, b in enumerate(bos):
            if b >= 0:
                sob[b] = s
        return sob, bos
    sel = np.array([3, 4, 5], dtype=np.int32)
    sob, bos = maps()
    t, mb, ms, ev = oracle.recall_plan(sel, sob, bos)
    assert list(mb) == [4, 5] and list(ms) == [0, 1] and list(ev) == [7, -1] and list(t) == [2, 0, 1]
    sob, bos = maps()
    t, mb, ms, ev = oracle.recall_plan(sel, sob, bos, empty_first=True)
    assert list(mb) == [4, 5] and list(ms) == [1, 3] and list(ev) == [-1, -1] and list(t) == [2, 1, 3]
    assert list(bos) == [7, 4, 3, 5, 9] and sob[7] == 0 and sob[9] == 4


def test_pinned_plan_never_evicts_while_room_is_left():
    """Random selections over a layer with room for every block: a block, once
    placed, stays; the table maps every selected block to its slot."""
    rng = np.random.default_rng(3)
    nb, P = 60, 60
    sob = np.full(nb, -1, dtype=np.int32)
    bos = np.full(P, -1, dtype=np.int32)
    placed = {}
    for _ in range(40):
        sel = np.sort(rng.choice(nb, size=9, replace=False)).astype(np.int32)
        t, mb, ms, ev = oracle.recall_plan(sel, sob, bos, empty_first=True)
        assert np.all(ev == -1)
        for b, s in zip(mb, ms):
            placed[int(b)] = int(s)
        for b, s in placed.items():
            assert sob[b] == s and bos[s] == b
        assert np.array_equal(t, sob[sel])


# ------------------------------------------------------------------ attention mass kept by a selection
# Guide, "SoloHead Sparse Selection", "2. High Attention Mass Preservation".

def test_mass_every_block_is_one_and_none_is_zero():
    hq, hkv, B, D, ntok = 8, 2, 16, 64, 1000      # ragged tail: 63 blocks, 8 tokens in the last
    reg = synth.kv_region(21, 0, 0, ntok, 64, hkv, B, D, 0.05, 2.0)
    q = synth.normal_bf16(21, synth.KIND_MISC, 0, 0, hq * D).reshape(hq, D)
    nb = -(-ntok // B)
    m = oracle.attention_mass(q, reg, np.arange(nb), ntok, hkv)
    assert np.all(np.abs(m - 1.0) < 1e-12)
    assert np.all(oracle.attention_mass(q, reg, np.zeros(0, dtype=np.int32), ntok, hkv) == 0.0)
    assert np.all(oracle.attention_mass(q, reg, np.arange(nb), 0, hkv) == 0.0)


def test_mass_zero_query_is_the_token_share():
    """q = 0: every logit is 0, the softmax is uniform, and a selection keeps
    exactly its share of the valid tokens (the tail block counts its valid ones)."""
    hq, hkv, B, D, ntok = 4, 2, 16, 64, 200      # 13 blocks; the tail (block 12) holds 8 tokens
    reg = synth.kv_region(22, 0, 0, ntok, 13, hkv, B, D)
    q = np.zeros((hq, D), dtype=np.uint16)
    for sel, tokens in (([0, 5], 32), ([12], 8), ([3, 12, 3], 24), ([0, 1, 2, 3, 4, 5, 6, 7, 8, 9, 10, 11], 192)):
        m = oracle.attention_mass(q, reg, np.array(sel, dtype=np.int32), ntok, hkv)
        assert np.all(np.abs(m - tokens / ntok) < 1e-15), (sel, m)


def test_mass_two_token_closed_form_and_gqa_mapping():
    """Two tokens of one block each, head_dim 4, two KV groups of two heads.
    Group 0 holds (c e0, 0), group 1 (0, c e0); every q_h = 2 e0, so the logits
    are (c, 0) for heads 0, 1 and (0, c) for heads 2, 3 (scale 1/sqrt(4)). Block 0
    keeps sigmoid(c) of heads 0, 1 and sigmoid(-c) of heads 2, 3: a wrong scale,
    sign or head-to-group map changes one of the four values."""
    hq, hkv, B, D, ntok = 4, 2, 1, 4, 2
    reg = np.zeros((2, hkv, 2, B, D), dtype=np.uint16)
    c = 1.5
    reg[0, 0, 0, 0, 0] = bf16_bits([c])[0]
    reg[1, 1, 0, 0, 0] = bf16_bits([c])[0]
    q = np.zeros((hq, D), dtype=np.uint16)
    q[:, 0] = bf16_bits([2.0])[0]
    sig = 1.0 / (1.0 + math.exp(-c))
    m = oracle.attention_mass(q, reg, np.array([0], dtype=np.int32), ntok, hkv)
    assert np.allclose(m, [sig, sig, 1 - sig, 1 - sig], rtol=0, atol=1e-15)
    # per-head sets: group 0 keeps block 1, group 1 keeps block 1
    m = oracle.attention_mass(q, reg, [np.array([1]), np.array([1])], ntok, hkv)
    assert np.allclose(m, [1 - sig, 1 - sig, sig, sig], rtol=0, atol=1e-15)


def test_mass_is_additive_over_disjoint_selections():
    hq, hkv, B, D, ntok = 8, 2, 16, 64, 700
    reg = synth.kv_region(23, 0, 0, ntok, 44, hkv, B, D, 0.1, 2.0)
    q = synth.normal_bf16(23, synth.KIND_MISC, 0, 0, hq * D).reshape(hq, D)
    nb = -(-ntok // B)
    rs = np.random.default_rng(23)
    for _ in range(5):
        perm = rs.permutation(nb)
        s1, s2 = np.sort(perm[:10]), np.sort(perm[10:25])
        m1 = oracle.attention_mass(q, reg, s1, ntok, hkv)
        m2 = oracle.attention_mass(q, reg, s2, ntok, hkv)
        m12 = oracle.attention_mass(q, reg, np.sort(np.concatenate([s1, s2])), ntok, hkv)
        assert np.all(np.abs(m1 + m2 - m12) < 1e-12)
        assert np.all((m1 > 0) & (m1 < 1) & (m12 >= m1))


@pytest.mark.parametrize("ntok", [1000, 33])
def test_mass_equals_sparse_over_dense_softmax_normaliser(ntok):
    """log(mass) = lse over the selected tokens - lse over all tokens: the sparse
    attention oracle (C, over the selection) against the independent numpy fp64
    dense attention (over the whole context)."""
    hq, hkv, B, D = 8, 2, 16, 64
    nb = -(-ntok // B)
    reg = synth.kv_region(24, 0, 0, ntok, nb + 1, hkv, B, D, 0.05, 2.0)
    q = synth.normal_bf16(24, synth.KIND_MISC, 0, 0, hq * D).reshape(hq, D)
    sel = np.array(sorted({0, nb - 1, nb // 2}), dtype=np.int32)
    _, lse_sel, _ = oracle.attention(q, reg, sel, ntok, hkv)
    K, V = _dense_inputs(reg, ntok, hkv, np.arange(nb))
    _, lse_all = oracle.dense_attention_fp64(oracle.bf16_to_f64(q), K, V)
    m = oracle.attention_mass(q, reg, sel, ntok, hkv)
    assert np.allclose(np.log(m), lse_sel - lse_all, rtol=0, atol=1e-10)


def test_mass_per_head_sets_equal_sparse_over_dense_softmax_normaliser():
    """Per-KV-head sets: each head's log(mass) is the lse over its group's set
    (C sparse-attention oracle, head-wise selection) minus the dense lse."""
    hq, hkv, B, D, ntok = 8, 2, 16, 64, 500
    nb = -(-ntok // B)
    reg = synth.kv_region(25, 0, 0, ntok, nb + 1, hkv, B, D, 0.05, 2.0)
    q = synth.normal_bf16(25, synth.KIND_MISC, 0, 0, hq * D).reshape(hq, D)
    sets = [np.array([0, 4, nb - 1], dtype=np.int32), np.array([2, 3, 9, 17], dtype=np.int32)]
    _, lse_sel, _ = oracle.attention(q, reg, sets, ntok, hkv)
    K, V = _dense_inputs(reg, ntok, hkv, np.arange(nb))
    _, lse_all = oracle.dense_attention_fp64(oracle.bf16_to_f64(q), K, V)
    m = oracle.attention_mass(q, reg, sets, ntok, hkv)
    assert np.allclose(np.log(m), lse_sel - lse_all, rtol=0, atol=1e-10)
    # a head of group 0 does not see group 1's set
    m_swapped = oracle.attention_mass(q, reg, sets[::-1], ntok, hkv)
    assert not np.allclose(m, m_swapped)


# ------------------------------------------------------------------ selection against exact arithmetic
def _exact_scores(q, km):
    """score(b) = sum over query heads h of q_h . kmean[b, h // G] in fp64 (the
    bf16 queries and fp32 summaries are exact there), and sum |q_h| . |kmean|."""
    qf = oracle.bf16_to_f64(q)
    hq, D = qf.shape
    nb, hkv, _ = km.shape
    G = hq // hkv
    kmf = km.astype(np.float64)
    s = np.einsum("hd,bhd->b", qf, np.repeat(kmf, G, axis=1))
    a = np.einsum("hd,bhd->b", np.abs(qf), np.abs(np.repeat(kmf, G, axis=1)))
    return s, a


def _decided_by_exact_arithmetic(exact, bound, k):
    """The exact top-k (score desc, index asc) and whether rounding within `bound`
    cannot change it: every member's lowest possible fp32 score stays above every
    other candidate's highest possible one."""
    n = len(exact)
    order = sorted(range(n), key=lambda b: (-exact[b], b))
    top, rest = order[:k], order[k:]
    if not rest or not top:
        return top, True
    lo = min(exact[b] - bound[b] for b in top)
    hi = max(exact[b] + bound[b] for b in rest)
    return top, lo > hi


def test_selection_matches_exact_arithmetic_outside_the_rounding_margin():
    """The fp32 score of every candidate lies within its rounding bound of the
    exact score (query-group sums: G - 1 roundings; the canonical dot: E/32
    sequential fused multiply-adds per lane, then a 5-level tree), and wherever
    no candidate's bound interval can cross the exact k-th/(k+1)-th boundary the
    fp32 top-k is the exact top-k. Llama-3-8B heads (32 q / 8 KV, d 128: E =
    1024), 256 blocks of 16 tokens, 5 % heavy-hitter blocks, 12 (request, layer)
    units. Also reports the margin diagnostic: the fraction of units whose
    k-th/(k+1)-th gap is below 1e-6 relative (where fp32 and exact arithmetic may
    disagree)."""
    hq, hkv, B, D, nb, k, W = 32, 8, 16, 128, 256, 32, 2
    ntok = nb * B
    G, E = hq // hkv, hkv * D
    u = 2.0 ** -24
    close = decided = 0
    units = 12
    for unit in range(units):
        reg = synth.kv_region(31, unit % 3, unit, ntok, nb, hkv, B, D, 0.05, 2.0)
        km = oracle.region_summaries(reg, ntok)
        q = synth.normal_bf16(31, synth.KIND_MISC, unit, 1, hq * D).reshape(hq, D)
        sel, s32 = oracle.select_shared(q, km, k, W, return_scores=True)
        s64, a64 = _exact_scores(q, km)
        ncand = nb - W
        bound = ((G - 1) + E // 32 + 5 + 1) * u * a64[:ncand] * 1.01
        assert np.all(np.abs(s32.astype(np.float64) - s64[:ncand]) <= bound)
        top, ok = _decided_by_exact_arithmetic(s64[:ncand], bound, k)
        if ok:
            assert sorted(top) == sorted(int(b) for b in sel[:k])
            decided += 1
        order = sorted(range(ncand), key=lambda b: (-s64[b], b))
        gap = s64[order[k - 1]] - s64[order[k]]
        if gap <= 1e-6 * max(abs(s64[order[k - 1]]), 1e-30):
            close += 1
    assert decided >= units // 2  # the comparison is not vacuous
    print(f"margin diagnostic: {close}/{units} units with a k-th/(k+1)-th gap below 1e-6 relative; "
          f"{decided}/{units} decided by exact arithmetic")


# ------------------------------------------------------------------ consensus against exact arithmetic
def exact_consensus(q, km, lam):
    """The consensus score of the guide ("SoloHead Sparse Selection", "1. Consensus
    Scoring Mechanism"), evaluated exactly, and a bound on any fp32 evaluation
    that follows the fixed operation count of this library's reading.

    Exact: S(h, b) = q_h . kmean[b, h // G] (bf16 x fp32 products are exact in
    fp64; the fp64 sum of 128 of them is within 2^-46 of exact, far below the
    fp32 bounds), c_g = max_h S + lam x (sum_h S) / G per group, score = sum_g c_g,
    with lam taken as the fp32 value the library uses.

    Bound: one standard rounding bound per operation, |fl(x op y) - (x op y)| <=
    u |x op y| with u = 2^-24, carried through in order:
      head score  4 fused multiply-adds per partial, then log2(D/4) additions:
                  e_S <= (4 + log2(D/4)) u A_h, A_h = sum_d |q_hd| |kmean_gd|;
      max         no rounding: e_M <= max_h e_S;
      head sum    log2(P) pairwise levels (P = pow2(G)):
                  e_sum <= sum_h e_S + log2(P) u sum_h (|S| + e_S);
      mean        exact for a power-of-two G, else one division;
      lam x mean, max + that: one rounding each;
      groups      Hkv - 1 sequential additions.
    Returns (exact [nb], bound [nb]) in fp64."""
    qf = oracle.bf16_to_f64(q)
    hq, D = qf.shape
    nb, hkv, _ = km.shape
    G = hq // hkv
    P = 1 << (G - 1).bit_length()
    lam = float(np.float32(lam))
    u = 2.0 ** -24
    slack = 1.01
    kmf = np.repeat(km.astype(np.float64), G, axis=1)           # [nb][Hq][D]
    S = np.einsum("hd,bhd->bh", qf, kmf).reshape(nb, hkv, G)
    A = np.einsum("hd,bhd->bh", np.abs(qf), np.abs(kmf)).reshape(nb, hkv, G)
    eS = (4 + int(math.log2(D // 4))) * u * A * slack
    M = S.max(axis=2)
    eM = eS.max(axis=2)
    Ssum = S.sum(axis=2)
    esum = eS.sum(axis=2) + int(math.log2(P)) * u * (np.abs(S) + eS).sum(axis=2) * slack
    mean = Ssum / G
    emean = esum / G
    if P != G:
        emean = emean + u * (np.abs(mean) + emean) * slack
    t = lam * mean
    et = lam * emean + u * (np.abs(t) + lam * emean) * slack
    c = M + t
    ec = eM + et + u * (np.abs(c) + eM + et) * slack
    exact = c.sum(axis=1)
    bound = ec.sum(axis=1) + (hkv - 1) * u * (np.abs(c) + ec).sum(axis=1) * slack
    return exact, bound


def test_exact_consensus_equals_rational_arithmetic_on_integers():
    """The exact reference itself, on inputs whose fp64 evaluation is exact: the
    same value as the formula in rational arithmetic (so the reference is the
    guide's formula and not a restatement of the fp32 order)."""
    rng_ = np.random.default_rng(77)
    for hq, hkv, D in ((32, 8, 128), (64, 8, 128), (12, 3, 64)):
        G = hq // hkv
        nb = 9
        qi = rng_.integers(-3, 4, size=(hq, D))
        ki = rng_.integers(-8, 9, size=(nb, hkv, D))
        q = synth.f32_to_bf16(qi.astype(np.float32))
        km = (ki / 4.0).astype(np.float32)
        exact, bound = exact_consensus(q, km, 0.5)
        for b in range(nb):
            tot = Fraction(0)
            for g in range(hkv):
                s_h = [Fraction(int(np.dot(qi[g * G + j], ki[b, g])), 4) for j in range(G)]
                tot += max(s_h) + Fraction(1, 2) * sum(s_h) / G
            assert Fraction(exact[b]) == tot
            assert bound[b] > 0.0


@pytest.mark.parametrize("hq", [32, 64], ids=["G4_llama8b", "G8_llama70b"])
def test_consensus_selection_matches_exact_arithmetic_outside_the_rounding_margin(hq):
    """The consensus ranking pinned to the formula rather than to its own fp32
    order: every fp32 consensus score lies within its rounding bound of the exact
    score, and wherever no candidate's bound interval can cross the exact
    k-th/(k+1)-th boundary the fp32 top-k is the exact top-k. Llama-3-8B (G = 4)
    and 70B (G = 8) heads, 8 KV heads, d 128, 256 blocks of 16 tokens, 5 %
    heavy-hitter blocks, lambda 0.5, 12 (request, layer) units each. Reports the
    margin diagnostic and how many units exact arithmetic decides."""
    hkv, B, D, nb, k, W, lam = 8, 16, 128, 256, 32, 2, 0.5
    ntok = nb * B
    close = decided = 0
    units = 12
    worst = 0.0
    for unit in range(units):
        reg = synth.kv_region(37, unit % 3, unit, ntok, nb, hkv, B, D, 0.05, 2.0)
        km = oracle.region_summaries(reg, ntok)
        q = synth.normal_bf16(37, synth.KIND_MISC, unit, hq, hq * D).reshape(hq, D)
        sel, s32 = oracle.select_consensus(q, km, k, W, lam, return_scores=True)
        ncand = nb - W
        exact, bound = exact_consensus(q, km[:ncand], lam)
        err = np.abs(s32.astype(np.float64) - exact)
        assert np.all(err <= bound), (unit, float((err / bound).max()))
        worst = max(worst, float((err / bound).max()))
        top, ok = _decided_by_exact_arithmetic(exact, bound, k)
        if ok:
            assert sorted(top) == sorted(int(b) for b in sel[:k])
            decided += 1
        order = sorted(range(ncand), key=lambda b: (-exact[b], b))
        gap = exact[order[k - 1]] - exact[order[k]]
        if gap <= 1e-6 * max(abs(exact[order[k - 1]]), 1e-30):
            close += 1
    assert decided >= units // 2  # the comparison is not vacuous
    print(f"consensus G={hq // hkv}: margin diagnostic {close}/{units} units with a k-th/(k+1)-th gap below 1e-6 "
          f"relative; {decided}/{units} decided by exact arithmetic; largest error / bound {worst:.3f}")
