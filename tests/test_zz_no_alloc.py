"""pi_sparse_decode_noalloc: sparse decode attention for callers that cannot
allocate device memory (for example engines that reserve all HBM in their own
arena at start-up and forbid any later cudaMalloc). It reads a paged KV buffer
the caller owns and keeps its scratch in a fixed array inside the library.

Checked here through the C ABI against the existing pool-based entry point
(pi_sparse_decode) on the same selection, within the attention tolerance of
the other tests, on two calls in a row; and that it leaves free device memory
unchanged. This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest

from _helpers import LSE_RTOL, OUT_ATOL, Workload, bf16_to_f32, fill_pool_host, queries

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


def _close(out_a, lse_a, out_b, lse_b):
    a = bf16_to_f32(out_a.cpu().numpy().view(np.uint16))
    b = bf16_to_f32(out_b.cpu().numpy().view(np.uint16))
    assert np.max(np.abs(a - b)) <= OUT_ATOL
    la, lb = lse_a.cpu().numpy().astype(np.float64), lse_b.cpu().numpy().astype(np.float64)
    assert np.all(np.abs(la - lb) <= LSE_RTOL * np.maximum(np.abs(lb), 1.0))


@pytest.mark.parametrize("w", CASES, ids=["d128_b64", "d64_b16"])
def test_noalloc_matches_pool_entry_point_twice(w):
    pi.build()
    lib = pi.load()
    layer = w.layers - 1
    cap = w.k + w.window
    R = w.batch
    with pi.Pool(w.layers, R, w.hq, w.hkv, w.head_dim, w.block_tokens, w.max_blocks, w.pool_slots, w.k,
                 w.window) as pool:
        fill_pool_host(pool, w)
        for l in range(w.layers):
            pool.update_summaries(l, w.ntok)
        qs = queries(w, steps=2)
        kreq = torch.full((R,), w.k, dtype=torch.int32, device="cuda")
        sel = torch.full((R, cap), -1, dtype=torch.int32, device="cuda")
        nsel = torch.empty((R,), dtype=torch.int32, device="cuda")
        table = torch.full((R, cap), -1, dtype=torch.int32, device="cuda")
        pool.select_topk(layer, _dev(qs[0][layer]), kreq, sel, nsel)
        pool.recall(layer, sel, nsel, table)
        torch.cuda.synchronize()
        # the caller's view: one flat buffer of slots and a table of global slot indices
        tab = table.cpu().numpy()
        gtab = np.full_like(tab, -1)
        ns = nsel.cpu().numpy()
        for r in range(R):
            gtab[r, : ns[r]] = [pool.global_slot(r, layer, int(s)) for s in tab[r, : ns[r]]]
        gtab_d = torch.from_numpy(gtab).cuda()
        ntok_d = pool.view_ntok()[:, layer].contiguous()
        kv = pool.view_pool()
        n_slots = kv.shape[0]
        outs = []
        for call, qi in enumerate((0, 1)):
            q = _dev(qs[qi][layer])
            ref_out = torch.empty((R, w.hq, w.head_dim), dtype=torch.int16, device="cuda")
            ref_lse = torch.empty((R, w.hq), dtype=torch.float32, device="cuda")
            pool.sparse_decode(layer, q, sel, table, nsel, ref_out, ref_lse)
            out = torch.full((R, w.hq, w.head_dim), 0x7FC0, dtype=torch.int16, device="cuda")
            lse = torch.full((R, w.hq), float("nan"), dtype=torch.float32, device="cuda")
            torch.cuda.synchronize()
            free_before = torch.cuda.mem_get_info()[0]
            st = lib.pi_sparse_decode_noalloc(kv.data_ptr(), n_slots, R, w.hq, w.hkv, w.head_dim, w.block_tokens,
                                              cap, q.data_ptr(), sel.data_ptr(), gtab_d.data_ptr(), nsel.data_ptr(),
                                              ntok_d.data_ptr(), out.data_ptr(), lse.data_ptr(),
                                              torch.cuda.current_stream().cuda_stream)
            assert st == pi.PI_OK, lib.pi_status_str(st)
            torch.cuda.synchronize()
            if call == 1:  # the first call's set-up is done; later calls take no device memory
                assert torch.cuda.mem_get_info()[0] == free_before
            _close(out, lse, ref_out, ref_lse)
            outs.append(out.clone())
        assert not torch.equal(outs[0], outs[1])  # two different queries, both matched
        assert pool.device_status() == pi.PI_OK


def test_noalloc_rejects_sizes_beyond_its_fixed_scratch():
    lib = pi.load()
    dummy = ctypes.c_void_p(256)
    # batch * KV heads above 1024
    assert lib.pi_sparse_decode_noalloc(dummy, 10, 200, 64, 8, 128, 64, 34, dummy, dummy, dummy, dummy, dummy, dummy,
                                        None, None) == pi.PI_ERR_INVALID
    # more than 512 selected blocks per request
    assert lib.pi_sparse_decode_noalloc(dummy, 10, 2, 32, 8, 128, 64, 600, dummy, dummy, dummy, dummy, dummy, dummy,
                                        None, None) == pi.PI_ERR_INVALID
