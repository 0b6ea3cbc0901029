"""pi_sparse_decode_noalloc: sparse decode attention for callers that cannot
allocate device memory (for example engines that reserve all HBM in their own
arena at start-up and forbid any later cudaMalloc). It reads a paged KV buffer
the caller owns and keeps its scratch in a fixed array inside the library.

Checked here through the C ABI against the oracle, element by element, on two
calls in a row with different queries (the second call reuses the array the
first one left behind), within the attention tolerance of the other tests; that
the calls leave free device memory unchanged; and that the status word the
array holds reports an out-of-range table entry and an out-of-range selection
count, then reads clean again after a good call. This file is collected last on
purpose.
"""
import ctypes

import numpy as np
import pytest

import oracle
from _helpers import LSE_RTOL, OUT_ATOL, OracleModel, Workload, bf16_to_f32, fill_pool_host, queries

torch = pytest.importorskip("torch")
pi = pytest.importorskip("sparse_kv_cache_block_gb300")

pytestmark = pytest.mark.gpu

CASES = [
    Workload(layers=2, batch=3, hq=32, hkv=8, head_dim=128, block_tokens=64, ntok=[3000, 2100, 4096], k=12,
             window=2, pool_slots=20, steps=2, seed=21, heavy_frac=0.05),
    Workload(layers=1, batch=2, hq=8, hkv=2, head_dim=64, block_tokens=16, ntok=[4096, 999], k=32, window=4,
             pool_slots=40, steps=2, seed=22),
]


def _dev(a):
    a = np.ascontiguousarray(a)
    return torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a).cuda()


def _check_against_oracle(out, lse, ref_out, ref_lse):
    got = bf16_to_f32(out.cpu().numpy().view(np.uint16))
    want = bf16_to_f32(ref_out)
    assert np.max(np.abs(got - want)) <= OUT_ATOL
    la = lse.cpu().numpy().astype(np.float64)
    assert np.all(np.abs(la - ref_lse) <= LSE_RTOL * np.maximum(np.abs(ref_lse), 1.0))


def _setup(w, layer):
    """A pool used only as the caller's paged buffer: the oracle's selection is
    recalled into it, and the caller's table gives each block's global slot."""
    pool = pi.Pool(w.layers, w.batch, w.hq, w.hkv, w.head_dim, w.block_tokens, w.max_blocks, w.pool_slots, w.k,
                   w.window)
    fill_pool_host(pool, w)
    for l in range(w.layers):
        pool.update_summaries(l, w.ntok)
    om = OracleModel(w)
    qs = queries(w, steps=2)
    R, cap = w.batch, w.k + w.window
    ref_sel = om.select(layer, qs[0][layer], [w.k] * R)
    sel_np = np.full((R, cap), -1, dtype=np.int32)
    for r, s_ in enumerate(ref_sel):
        sel_np[r, : len(s_)] = s_
    sel = torch.from_numpy(sel_np).cuda()
    nsel = torch.tensor([len(s_) for s_ in ref_sel], dtype=torch.int32, device="cuda")
    table = torch.full((R, cap), -1, dtype=torch.int32, device="cuda")
    pool.recall(layer, sel, nsel, table)
    torch.cuda.synchronize()
    tab = table.cpu().numpy()
    gtab = np.full_like(tab, -1)
    for r, s_ in enumerate(ref_sel):
        gtab[r, : len(s_)] = [pool.global_slot(r, layer, int(x)) for x in tab[r, : len(s_)]]
    ntok = torch.tensor(w.ntok, dtype=torch.int32, device="cuda")
    return pool, om, qs, ref_sel, sel, nsel, gtab, ntok


def _call(lib, kv, w, q, sel, gtab_d, nsel, ntok, out, lse):
    return lib.pi_sparse_decode_noalloc(kv.data_ptr(), kv.shape[0], w.batch, w.hq, w.hkv, w.head_dim,
                                        w.block_tokens, w.k + w.window, q.data_ptr(), sel.data_ptr(),
                                        gtab_d.data_ptr(), nsel.data_ptr(), ntok.data_ptr(), out.data_ptr(),
                                        lse.data_ptr(), torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("w", CASES, ids=["d128_b64", "d64_b16"])
def test_noalloc_matches_oracle_twice(w):
    pi.build()
    lib = pi.load()
    layer = w.layers - 1
    R = w.batch
    pool, om, qs, ref_sel, sel, nsel, gtab, ntok = _setup(w, layer)
    with pool:
        gtab_d = torch.from_numpy(gtab).cuda()
        kv = pool.view_pool()
        outs = []
        for call, qi in enumerate((0, 1)):
            q_np = qs[qi][layer]
            q = _dev(q_np)
            out = torch.full((R, w.hq, w.head_dim), 0x7FC0, dtype=torch.int16, device="cuda")
            lse = torch.full((R, w.hq), float("nan"), dtype=torch.float32, device="cuda")
            torch.cuda.synchronize()
            free_before = torch.cuda.mem_get_info()[0]
            st = _call(lib, kv, w, q, sel, gtab_d, nsel, ntok, out, lse)
            assert st == pi.PI_OK, lib.pi_status_str(st)
            assert pi.sparse_decode_noalloc_status() == pi.PI_OK
            if call == 1:  # the first call's set-up is done; later calls take no device memory
                assert torch.cuda.mem_get_info()[0] == free_before
            ref_out, ref_lse, _ = om.attention(layer, q_np, ref_sel)
            _check_against_oracle(out, lse, ref_out, ref_lse)
            outs.append(out.clone())
        assert not torch.equal(outs[0], outs[1])  # two different queries, both matched
        assert pool.device_status() == pi.PI_OK


def test_noalloc_reports_out_of_range_entries_then_reads_clean():
    """One table entry past the caller's slots and one selection count above cap
    are skipped and reported through the status word; a good call afterwards
    clears it. The other requests' outputs still match the oracle."""
    w = CASES[1]
    pi.build()
    lib = pi.load()
    layer, R = 0, w.batch
    pool, om, qs, ref_sel, sel, nsel, gtab, ntok = _setup(w, layer)
    with pool:
        kv = pool.view_pool()
        q_np = qs[0][layer]
        q = _dev(q_np)
        out = torch.empty((R, w.hq, w.head_dim), dtype=torch.int16, device="cuda")
        lse = torch.empty((R, w.hq), dtype=torch.float32, device="cuda")
        ref_out, ref_lse, _ = om.attention(layer, q_np, ref_sel)
        # request 1's third block points one slot past the end of the buffer
        bad = gtab.copy()
        bad[1, 2] = kv.shape[0]
        assert _call(lib, kv, w, q, sel, torch.from_numpy(bad).cuda(), nsel, ntok, out, lse) == pi.PI_OK
        assert pi.sparse_decode_noalloc_status() == pi.PI_ERR_DEVICE
        got = bf16_to_f32(out.cpu().numpy().view(np.uint16))
        assert np.max(np.abs(got[0] - bf16_to_f32(ref_out[0]))) <= OUT_ATOL  # request 0 untouched by it
        # a selection count above cap
        bad_n = nsel.clone()
        bad_n[0] = w.k + w.window + 1
        gtab_d = torch.from_numpy(gtab).cuda()
        assert _call(lib, kv, w, q, sel, gtab_d, bad_n, ntok, out, lse) == pi.PI_OK
        assert pi.sparse_decode_noalloc_status() == pi.PI_ERR_DEVICE
        # a good call clears the word when it starts
        assert _call(lib, kv, w, q, sel, gtab_d, nsel, ntok, out, lse) == pi.PI_OK
        assert pi.sparse_decode_noalloc_status() == pi.PI_OK
        _check_against_oracle(out, lse, ref_out, ref_lse)


def test_noalloc_rejects_sizes_beyond_its_fixed_scratch():
    lib = pi.load()
    dummy = ctypes.c_void_p(256)
    # batch * KV heads above 1024
    assert lib.pi_sparse_decode_noalloc(dummy, 10, 200, 64, 8, 128, 64, 34, dummy, dummy, dummy, dummy, dummy, dummy,
                                        None, None) == pi.PI_ERR_INVALID
    # more than 512 selected blocks per request
    assert lib.pi_sparse_decode_noalloc(dummy, 10, 2, 32, 8, 128, 64, 600, dummy, dummy, dummy, dummy, dummy, dummy,
                                        None, None) == pi.PI_ERR_INVALID
