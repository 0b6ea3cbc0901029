"""CPU oracle of the sparse KV-cache offloading decode path.

TEST INFRASTRUCTURE ONLY. Only the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg (and its ``--impl reference`` arm) may import it;
the CUDA library never does, and the two share no code. The arithmetic lives
in ``pi_oracle.c`` (plain loops, ``-ffp-contract=off``); this module wraps it
with ctypes and adds an independent fp64 dense attention in numpy.

What each function follows (page title, section):

* block summaries, the shared top-k and the head-wise arm: "PulseInfer Guide:
  I/O-Centric Sparse KV Cache Offloading", "SoloHead Sparse Selection" (one
  block set shared by every head instead of one per head). The pages leave the
  block score undefined; the score used here (per-KV-head mean key, summed
  q_h . kmean over all query heads, fp32, ties to the lower block index, plus
  the W most recent blocks) is this library's fixed reading.
* pool plan and recall: same guide, "The Gather-Scatter I/O Engine" (recalled
  blocks land in pool page slots) and the abstract of "PulseInfer: I/O-Centric
  Sparse KV Cache Offloading for Efficient Long-Context LLM Decoding" (blocks
  stay in CPU DRAM and only selected ones are recalled on demand).
* attention: textbook scaled dot-product attention restricted to the tokens of
  the selected blocks, in fp64 (the guide's "PulseInfer Architectural
  Foundations": attention runs over the recalled pool blocks).
* attention mass kept by a selection (a diagnostic): same guide, "SoloHead
  Sparse Selection", "2. High Attention Mass Preservation"; fp64 dense softmax
  over the whole context, summed over the selected blocks' tokens.

Parity pins (tests/test_oracle_pins.py) tie every function to something other
than itself: brute force, closed forms, invariants and the worked example of
the guide's "SoloHead Sparse Selection" section.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(_HERE, "liboracle.so")


def build(force: bool = False) -> str:
    """Compile pi_oracle.c into liboracle.so (gcc -O2 -ffp-contract=off)."""
    src = os.path.join(_HERE, "pi_oracle.c")
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(src):
        tmp = _SO + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-ffp-contract=off", "-fPIC", "-shared", "-o", tmp, src, "-lm"])
        os.replace(tmp, _SO)
    return _SO


_lib = None


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_SO)
        i32, vp, f32 = ctypes.c_int, ctypes.c_void_p, ctypes.c_float
        L.or_bf16_rne.restype = ctypes.c_uint16
        L.or_bf16_rne.argtypes = [ctypes.c_double]
        L.or_block_summary.restype = None
        L.or_block_summary.argtypes = [vp, i32, i32, i32, i32, vp]
        L.or_region_summaries.restype = None
        L.or_region_summaries.argtypes = [vp, i32, i32, i32, i32, vp]
        L.or_qsum.restype = None
        L.or_qsum.argtypes = [vp, i32, i32, i32, vp]
        L.or_score.restype = f32
        L.or_score.argtypes = [vp, vp, i32]
        L.or_select_topk.restype = i32
        L.or_select_topk.argtypes = [vp, i32, i32, i32, vp]
        L.or_select_shared.restype = i32
        L.or_select_shared.argtypes = [vp, vp, i32, i32, i32, i32, i32, i32, vp, vp]
        L.or_head_score.restype = f32
        L.or_head_score.argtypes = [vp, vp, i32]
        L.or_consensus_score.restype = f32
        L.or_consensus_score.argtypes = [vp, vp, i32, i32, i32, f32]
        L.or_select_consensus.restype = i32
        L.or_select_consensus.argtypes = [vp, vp, i32, i32, i32, i32, i32, i32, f32, vp, vp]
        L.or_select_headwise.restype = None
        L.or_select_headwise.argtypes = [vp, vp, i32, i32, i32, i32, i32, i32, i32, vp, vp]
        L.or_recall_plan_pinned.restype = i32
        L.or_recall_plan_pinned.argtypes = [vp, i32, vp, vp, i32, vp, vp, vp, vp]
        L.or_recall_plan.restype = i32
        L.or_recall_plan.argtypes = [vp, i32, vp, vp, i32, vp, vp, vp, vp]
        L.or_recall_plan_lru.restype = i32
        L.or_recall_plan_lru.argtypes = [vp, i32, vp, vp, vp, i32, i32, vp, vp, vp, vp]
        L.or_attention.restype = None
        L.or_attention.argtypes = [vp, vp, vp, i32, vp, i32, i32, i32, i32, i32, i32, vp, vp, vp, i32]
        _lib = L
    return _lib


def _p(a: np.ndarray | None):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# --------------------------------------------------------------------- bf16
def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def bf16_rne(x: float) -> int:
    """fp64 -> bf16 bits, round to nearest even."""
    return int(lib().or_bf16_rne(float(x)))


# --------------------------------------------------------------------- a-1
def block_summary(blk: np.ndarray, n_valid: int) -> np.ndarray:
    """blk [Hkv][2][B][D] bf16 -> kmean [Hkv][D] fp32 (sequential fp32 sum / n)."""
    blk = _c(blk, np.uint16)
    hkv, _, B, D = blk.shape
    out = np.empty((hkv, D), dtype=np.float32)
    lib().or_block_summary(_p(blk), hkv, B, D, n_valid, _p(out))
    return out


def region_summaries(region: np.ndarray, ntok: int) -> np.ndarray:
    """region [max_blocks][Hkv][2][B][D] -> kmean [nb][Hkv][D] for nb = ceil(ntok / B)."""
    region = _c(region, np.uint16)
    _, hkv, _, B, D = region.shape
    nb = -(-ntok // B)
    out = np.empty((max(nb, 1), hkv, D), dtype=np.float32)
    lib().or_region_summaries(_p(region), ntok, hkv, B, D, _p(out))
    return out[:nb]


# --------------------------------------------------------------------- a-2
def qsum(q: np.ndarray, hkv: int) -> np.ndarray:
    q = _c(q, np.uint16)
    hq, D = q.shape
    out = np.empty((hkv, D), dtype=np.float32)
    lib().or_qsum(_p(q), hq, hkv, D, _p(out))
    return out


def score(qs: np.ndarray, km: np.ndarray) -> float:
    qs = _c(qs, np.float32).ravel()
    km = _c(km, np.float32).ravel()
    assert qs.size == km.size and qs.size % 4 == 0
    return float(np.float32(lib().or_score(_p(qs), _p(km), qs.size)))


def select_topk(scores: np.ndarray, nb: int, k: int, W: int) -> np.ndarray:
    scores = _c(scores, np.float32)
    sel = np.empty(max(nb, 1), dtype=np.int32)
    n = lib().or_select_topk(_p(scores), nb, k, W, _p(sel))
    return sel[:n].copy()


def select_shared(q: np.ndarray, kmean: np.ndarray, k: int, W: int, return_scores: bool = False):
    """q [Hq][D] bf16, kmean [nb][Hkv][D] fp32 -> ascending selected block ids."""
    q = _c(q, np.uint16)
    kmean = _c(kmean, np.float32)
    nb, hkv, D = kmean.shape
    hq = q.shape[0]
    sel = np.empty(max(nb, 1), dtype=np.int32)
    sc = np.empty(max(nb, 1), dtype=np.float32)
    n = lib().or_select_shared(_p(q), _p(kmean), nb, hq, hkv, D, k, W, _p(sel), _p(sc))
    if return_scores:
        return sel[:n].copy(), sc[: max(nb - W, 0)].copy()
    return sel[:n].copy()


def head_score(qh: np.ndarray, kmg: np.ndarray) -> float:
    """S(h, b) = q_h . kmean[b, group(h)] in the library's fixed fp32 order
    (guide, "SoloHead Sparse Selection"). qh [D] bf16 bits, kmg [D] fp32."""
    qh = _c(qh, np.uint16).ravel()
    kmg = _c(kmg, np.float32).ravel()
    assert qh.size == kmg.size and qh.size in (64, 128)
    return float(np.float32(lib().or_head_score(_p(qh), _p(kmg), qh.size)))


def consensus_score(q: np.ndarray, km_b: np.ndarray, lam: float) -> float:
    """Consensus score of one block (guide, "SoloHead Sparse Selection",
    "1. Consensus Scoring Mechanism"): per GQA group, the largest per-head score
    plus lam times their mean; summed over the groups. q [Hq][D] bf16 bits,
    km_b [Hkv][D] fp32."""
    q = _c(q, np.uint16)
    km_b = _c(km_b, np.float32)
    hkv, D = km_b.shape
    return float(np.float32(lib().or_consensus_score(_p(q), _p(km_b), q.shape[0], hkv, D, float(lam))))


def select_consensus(q: np.ndarray, kmean: np.ndarray, k: int, W: int, lam: float, return_scores: bool = False):
    """Shared block set of one (request, layer) ranked by consensus scores: the
    top-k rule of select_shared over consensus_score (same ties, same recent
    window, ascending output)."""
    q = _c(q, np.uint16)
    kmean = _c(kmean, np.float32)
    nb, hkv, D = kmean.shape
    sel = np.empty(max(nb, 1), dtype=np.int32)
    sc = np.empty(max(nb, 1), dtype=np.float32)
    n = lib().or_select_consensus(_p(q), _p(kmean), nb, q.shape[0], hkv, D, k, W, float(lam), _p(sel), _p(sc))
    if return_scores:
        return sel[:n].copy(), sc[: max(nb - W, 0)].copy()
    return sel[:n].copy()


def select_headwise(q: np.ndarray, kmean: np.ndarray, k: int, W: int):
    """Per-KV-head top-k (comparison arm). Returns list of Hkv ascending arrays."""
    q = _c(q, np.uint16)
    kmean = _c(kmean, np.float32)
    nb, hkv, D = kmean.shape
    hq = q.shape[0]
    cap = max(nb, 1)
    sel = np.empty((hkv, cap), dtype=np.int32)
    nsel = np.empty(hkv, dtype=np.int32)
    lib().or_select_headwise(_p(q), _p(kmean), nb, hq, hkv, D, k, W, cap, _p(sel), _p(nsel))
    return [sel[g, : nsel[g]].copy() for g in range(hkv)]


# --------------------------------------------------------------------- a-3
def recall_plan(sel: np.ndarray, slot_of_block: np.ndarray, block_of_slot: np.ndarray, empty_first: bool = False):
    """Updates the two maps in place. Returns (table, miss_blocks, miss_slots, evicted)
    or None when the pool is too small (maps untouched). empty_first: the rule of a
    layer held whole in HBM (guide, "2. IO-Adaptive Offloading Admission"): empty
    slots are taken before slots holding an unselected block."""
    sel = _c(sel, np.int32)
    assert slot_of_block.dtype == np.int32 and block_of_slot.dtype == np.int32
    assert slot_of_block.flags["C_CONTIGUOUS"] and block_of_slot.flags["C_CONTIGUOUS"]
    n = sel.size
    P = block_of_slot.size
    table = np.empty(max(n, 1), dtype=np.int32)
    mb = np.empty(max(n, 1), dtype=np.int32)
    ms = np.empty(max(n, 1), dtype=np.int32)
    ev = np.empty(max(n, 1), dtype=np.int32)
    fn = lib().or_recall_plan_pinned if empty_first else lib().or_recall_plan
    nm = fn(_p(sel), n, _p(slot_of_block), _p(block_of_slot), P, _p(table), _p(mb), _p(ms), _p(ev))
    if nm < 0:
        return None
    return table[:n].copy(), mb[:nm].copy(), ms[:nm].copy(), ev[:nm].copy()


def recall_plan_lru(sel: np.ndarray, slot_of_block: np.ndarray, block_of_slot: np.ndarray, stamp: np.ndarray,
                    epoch: int):
    """Least-recently-selected variant: free slots taken by (stamp, slot)
    ascending; selected slots stamped with `epoch`. Updates maps and stamps in
    place; returns (table, miss_blocks, miss_slots, evicted) or None."""
    sel = _c(sel, np.int32)
    for a in (slot_of_block, block_of_slot, stamp):
        assert a.dtype == np.int32 and a.flags["C_CONTIGUOUS"]
    n = sel.size
    P = block_of_slot.size
    table = np.empty(max(n, 1), dtype=np.int32)
    mb = np.empty(max(n, 1), dtype=np.int32)
    ms = np.empty(max(n, 1), dtype=np.int32)
    ev = np.empty(max(n, 1), dtype=np.int32)
    nm = lib().or_recall_plan_lru(_p(sel), n, _p(slot_of_block), _p(block_of_slot), _p(stamp), P, int(epoch),
                                  _p(table), _p(mb), _p(ms), _p(ev))
    if nm < 0:
        return None
    return table[:n].copy(), mb[:nm].copy(), ms[:nm].copy(), ev[:nm].copy()


# --------------------------------------------------------------------- a-5
def attention(q: np.ndarray, region: np.ndarray, sel, ntok: int, hkv: int, want_logits: bool = False):
    """Sparse decode attention of one (request, layer), fp64.

    q [Hq][D] bf16 bits; region [max_blocks][Hkv][2][B][D] bf16 bits; sel either one
    ascending array (shared) or a list of Hkv arrays (head-wise).
    Returns (out bf16 bits [Hq][D], lse fp64 [Hq], logits fp64 [Hq][cap][B] or None)."""
    q = _c(q, np.uint16)
    region = _c(region, np.uint16)
    hq, D = q.shape
    B = region.shape[3]
    if isinstance(sel, (list, tuple)):
        cap = max(1, max(len(s) for s in sel))
        sel_a = np.zeros((hkv, cap), dtype=np.int32)
        ns = np.zeros(hkv, dtype=np.int32)
        for g, s in enumerate(sel):
            sel_a[g, : len(s)] = s
            ns[g] = len(s)
        sel_stride, ns_stride = cap, 1
    else:
        sel_a = _c(sel, np.int32)
        cap = max(1, sel_a.size)
        ns = np.array([sel_a.size], dtype=np.int32)
        sel_stride, ns_stride = 0, 0
        if sel_a.size == 0:
            sel_a = np.zeros(1, dtype=np.int32)
    out = np.empty((hq, D), dtype=np.uint16)
    lse = np.empty(hq, dtype=np.float64)
    logits = np.full((hq, cap, B), np.nan, dtype=np.float64) if want_logits else None
    lib().or_attention(_p(q), _p(region), _p(sel_a), sel_stride, _p(ns), ns_stride, ntok, hq, hkv, B, D,
                       _p(out), _p(lse), _p(logits), cap)
    return out, lse, logits


def dense_attention_fp64(q: np.ndarray, K: np.ndarray, V: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """Independent textbook GQA attention in numpy fp64 (no blocks, no selection).

    q [Hq][D], K/V [Hkv][N][D] as float64. Returns (out [Hq][D] fp64, lse [Hq])."""
    hq, D = q.shape
    hkv = K.shape[0]
    G = hq // hkv
    out = np.empty((hq, D))
    lse = np.empty(hq)
    for h in range(hq):
        g = h // G
        z = K[g] @ q[h] / math.sqrt(D)
        m = z.max()
        p = np.exp(z - m)
        out[h] = (p @ V[g]) / p.sum()
        lse[h] = m + math.log(p.sum())
    return out, lse


def attention_mass(q: np.ndarray, region: np.ndarray, sel, ntok: int, hkv: int) -> np.ndarray:
    """Share of each query head's full attention that a block selection keeps, fp64.

    Guide, "SoloHead Sparse Selection", "2. High Attention Mass Preservation": a
    selection is judged by the softmax weight its blocks hold. Definition written
    out: for head h (KV group g = h // G), z_t = q_h . K_t / sqrt(D) over every
    valid token t of the context, p = softmax(z), mass[h] = sum of p_t over the
    tokens of the selected blocks. q [Hq][D] bf16 bits; region [max_blocks][Hkv][2][B][D]
    bf16 bits; sel one array of block ids (shared by all heads) or a list of Hkv
    arrays (head h uses sel[h // G]); a repeated id counts once. No tokens: 0."""
    qf = bf16_to_f64(_c(q, np.uint16))
    region = _c(region, np.uint16)
    hq, D = qf.shape
    B = region.shape[3]
    G = hq // hkv
    mass = np.zeros(hq)
    if ntok <= 0:
        return mass
    nb = -(-ntok // B)
    per_head = isinstance(sel, (list, tuple))
    for h in range(hq):
        g = h // G
        K = bf16_to_f64(region[:nb, g, 0]).reshape(nb * B, D)[:ntok]
        z = K @ qf[h] / math.sqrt(D)
        p = np.exp(z - z.max())
        member = np.zeros(ntok, dtype=bool)
        for b in set(int(x) for x in (sel[g] if per_head else sel)):
            member[b * B:min(ntok, (b + 1) * B)] = True
        mass[h] = p[member].sum() / p.sum()
    return mass


def union_fragments(per_head_sets) -> int:
    """Blocks a head-wise selection moves: the size of the union of the heads' sets."""
    u = set()
    for s in per_head_sets:
        u.update(int(b) for b in s)
    return len(u)


def block_bytes(hkv: int, block_tokens: int, head_dim: int, elem_bytes: int = 2) -> int:
    """Bytes of one paged KV block for all KV heads, K and V."""
    return 2 * hkv * block_tokens * head_dim * elem_bytes


def kv_cache_bytes(layers: int, hkv: int, head_dim: int, seq: int, elem_bytes: int = 2) -> int:
    """Whole-sequence KV cache bytes: K and V for every layer, KV head and token."""
    return 2 * layers * hkv * head_dim * seq * elem_bytes
