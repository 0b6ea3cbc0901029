"""GB300 sparse KV-cache offloading decode path (PulseInfer-style), Python binding.

The work happens in libpi.so (hand-written CUDA for sm_103a behind the C ABI of
include/pi.h). This package only marshals arguments: torch tensors become raw
device pointers, torch streams become cudaStream_t handles, library-owned
device state is exposed as zero-copy torch views.
"""
from __future__ import annotations

import ctypes

import numpy as np

from . import _lib
from ._lib import (PI_EVICT_ASCENDING, PI_EVICT_LRU, PI_ERR_CUDA, PI_ERR_DEVICE, PI_ERR_FAULT_INJECTED, PI_ERR_HOST_ALLOC, PI_ERR_INVALID, PI_ERR_OOM,
                   PI_ERR_POOL_FULL, PI_ERR_STATE, PI_ERR_TIMEOUT, PI_HEADWISE, PI_OK, PI_RECALL_MEMCPY,
                   PI_RECALL_STAGED, PI_RECALL_UVA, PI_SHARED, PI_CONSENSUS, PiError, check, declared_functions, load, pi_config,
                   pi_pool_views, pi_recall_stats, pi_step_stats)
from .build import build

__all__ = ["Pool", "PiError", "build", "load", "declared_functions", "PI_SHARED", "PI_HEADWISE", "PI_CONSENSUS", "PI_RECALL_UVA",
           "PI_RECALL_MEMCPY", "PI_RECALL_STAGED"]


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, np.ndarray):
        return t.ctypes.data
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(s) -> int | None:
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


class _DevView:
    """__cuda_array_interface__ over library-owned device memory (no copy)."""

    def __init__(self, ptr: int, shape, typestr: str):
        self.__cuda_array_interface__ = {"shape": tuple(shape), "typestr": typestr, "data": (ptr, False),
                                         "version": 3, "strides": None}


def device_view(ptr: int, shape, dtype: str):
    import torch
    typestr = {"int32": "<i4", "float32": "<f4", "uint8": "|u1", "int16": "<i2"}[dtype]
    return torch.as_tensor(_DevView(ptr, shape, typestr), device="cuda")


def sparse_decode_noalloc(kv_slots, n_slots: int, batch: int, hq: int, hkv: int, head_dim: int,
                          block_tokens: int, cap: int, q, sel, slot_table, nsel, ntok, out, lse=None, stream=None):
    """pi_sparse_decode_noalloc: attention over a caller-owned paged KV buffer
    that allocates nothing (its scratch is a fixed array inside the library).
    Returns the pi_status code (0 = ok) without raising."""
    return load().pi_sparse_decode_noalloc(_ptr(kv_slots), int(n_slots), batch, hq, hkv, head_dim, block_tokens, cap,
                                           _ptr(q), _ptr(sel), _ptr(slot_table), _ptr(nsel), _ptr(ntok), _ptr(out),
                                           _ptr(lse), _stream(stream))


def sparse_decode_noalloc_status(stream=None) -> int:
    """pi_sparse_decode_noalloc_status: the device-side outcome of the last
    no-allocation call on the current device (synchronizes the stream). Returns
    the pi_status code without raising."""
    return load().pi_sparse_decode_noalloc_status(_stream(stream))


class Pool:
    """One pi_pool: pinned host KV store + device block pool + summaries + maps."""

    def __init__(self, layers: int, batch: int, hq: int, hkv: int, head_dim: int, block_tokens: int,
                 max_blocks: int, pool_slots: int, k_max: int, window: int, select_mode: int = PI_SHARED,
                 host_layers: int = 0, staging_blocks: int = 0, gather_ctas: int = 0, pool_slots_per_req=None,
                 gather_depth: int = 0, host_alloc: int = 0, evict_policy: int = 0, pin_layers: int = 0):
        self.lib = load()
        cfg = pi_config(layers, batch, hq, hkv, head_dim, block_tokens, max_blocks, pool_slots, k_max, window,
                        select_mode, host_layers, staging_blocks, gather_ctas, gather_depth, evict_policy, host_alloc,
                        pin_layers, None)
        self._slots_arr = None
        if pool_slots_per_req is not None:
            self._slots_arr = (ctypes.c_int * batch)(*[int(x) for x in pool_slots_per_req])
            cfg.pool_slots_per_req = ctypes.cast(self._slots_arr, ctypes.POINTER(ctypes.c_int))
        h = ctypes.c_void_p()
        check(self.lib.pi_pool_create(ctypes.byref(cfg), ctypes.byref(h)), "pi_pool_create")
        self.h = h
        self.cfg = cfg
        self.L, self.R, self.Hq, self.Hkv, self.D, self.B = layers, batch, hq, hkv, head_dim, block_tokens
        self.max_blocks, self.k_max, self.W = max_blocks, k_max, window
        self.cap = k_max + window
        self.mode = select_mode
        self.U = hkv if select_mode == PI_HEADWISE else 1
        self.host_layers = host_layers if host_layers > 0 else layers
        v = pi_pool_views()
        check(self.lib.pi_pool_get_views(self.h, ctypes.byref(v)), "pi_pool_get_views")
        self._views = v
        self.p_max = v.p_max
        self.block_bytes = v.block_bytes
        self.frag_bytes = v.frag_bytes
        self.region_bytes = v.host_region_bytes
        self.slots_per_req = [v.slots_per_req[r] for r in range(batch)]
        self.slot_base = [[v.slot_base[r * layers + l] for l in range(layers)] for r in range(batch)]
        self.total_slots = v.total_slots

    # ---------------------------------------------------------------- lifetime
    def close(self):
        if getattr(self, "h", None):
            check(self.lib.pi_pool_destroy(self.h), "pi_pool_destroy")
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *a):
        self.close()

    # ---------------------------------------------------------------- host store
    def host_kv_ptr(self, layer: int, req: int) -> int:
        p = self.lib.pi_host_kv(self.h, layer, req)
        if not p:
            raise PiError(PI_ERR_INVALID, "pi_host_kv")
        return p

    def host_kv(self, layer: int, req: int) -> np.ndarray:
        """numpy view [max_blocks][Hkv][2][B][D] (uint16 bf16 bits) of the pinned region."""
        n = self.region_bytes // 2
        buf = (ctypes.c_uint16 * n).from_address(self.host_kv_ptr(layer, req))
        return np.frombuffer(buf, dtype=np.uint16).reshape(self.max_blocks, self.Hkv, 2, self.B, self.D)

    # ---------------------------------------------------------------- views
    def view_pool(self):
        return device_view(self._views.pool, (self.total_slots, self.Hkv, 2, self.B, self.D), "int16")

    def global_slot(self, r: int, l: int, s: int) -> int:
        return self.slot_base[r][l] + s

    def slots(self, r: int, l: int) -> int:
        """Slots (r, l) uses now: P_r, or every block of a pinned layer."""
        return self._views.slots_rl[r * self.L + l]

    def device_status_bits(self) -> int:
        """The raw bits of the device status word (synchronizes the device)."""
        import torch
        torch.cuda.synchronize()
        return int(device_view(self._views.dev_status, (1,), "int32").cpu()[0]) & 0xFFFFFFFF

    def view_kmean(self):
        return device_view(self._views.kmean, (self.R, self.L, self.max_blocks, self.Hkv, self.D), "float32")

    def view_ntok(self):
        return device_view(self._views.ntok, (self.R, self.L), "int32")

    def view_slot_of_block(self):
        return device_view(self._views.slot_of_block, (self.R, self.L, self.U, self.max_blocks), "int32")

    def view_block_of_slot(self):
        return device_view(self._views.block_of_slot, (self.R, self.L, self.U, self.p_max), "int32")

    def view_step(self):
        sel = device_view(self._views.step_sel, (self.L, self.R, self.U, self.cap), "int32")
        nsel = device_view(self._views.step_nsel, (self.L, self.R, self.U), "int32")
        tab = device_view(self._views.step_table, (self.L, self.R, self.U, self.cap), "int32")
        return sel, nsel, tab

    # ---------------------------------------------------------------- ops
    def update_summaries(self, layer: int, ntok, k_dev=None, block_begin: int = 0, block_end: int | None = None,
                         stream=None):
        arr = (ctypes.c_int * self.R)(*[int(x) for x in ntok])
        be = self.max_blocks if block_end is None else block_end
        check(self.lib.pi_update_summaries(self.h, layer, _ptr(k_dev), block_begin, be, ctypes.cast(arr, ctypes.c_void_p),
                                           _stream(stream)), "pi_update_summaries")

    def append_kv(self, layer: int, k_new, v_new, stream=None):
        check(self.lib.pi_append_kv(self.h, layer, _ptr(k_new), _ptr(v_new), _stream(stream)), "pi_append_kv")

    def select_topk(self, layer: int, q, k_per_req, sel, nsel, stream=None, mode: int | None = None):
        m = self.mode if mode is None else mode
        check(self.lib.pi_select_topk(self.h, layer, _ptr(q), _ptr(k_per_req), m, _ptr(sel), _ptr(nsel),
                                      _stream(stream)), "pi_select_topk")

    def recall(self, layer: int, sel, nsel, table, method: int = PI_RECALL_UVA, stats: bool = False, stream=None):
        st = pi_recall_stats() if stats else None
        check(self.lib.pi_recall(self.h, layer, _ptr(sel), _ptr(nsel), method, _ptr(table),
                                 ctypes.byref(st) if st is not None else None, _stream(stream)), "pi_recall")
        return st.as_dict() if st is not None else None

    def preload(self, layer: int, req: int, blocks, stream=None):
        arr = np.ascontiguousarray(blocks, dtype=np.int32)
        check(self.lib.pi_pool_preload(self.h, layer, req, arr.ctypes.data if arr.size else None, int(arr.size),
                                       _stream(stream)), "pi_pool_preload")

    def set_pipeline(self, select_ahead: int = 1, attention_stream: bool = True):
        check(self.lib.pi_pool_set_pipeline(self.h, select_ahead, int(attention_stream)), "pi_pool_set_pipeline")

    def set_attention(self, splits: int):
        check(self.lib.pi_pool_set_attention(self.h, splits), "pi_pool_set_attention")

    def set_schedule(self, dependent: bool, groups: int = 1):
        dep = dependent if isinstance(dependent, int) and not isinstance(dependent, bool) else int(bool(dependent))
        check(self.lib.pi_pool_set_schedule(self.h, dep, groups), "pi_pool_set_schedule")

    def set_fused(self, on: bool, ctas: int = 0):
        """Selection, plan and gather of a layer as one launch in the decode step."""
        check(self.lib.pi_pool_set_fused(self.h, int(bool(on)), ctas), "pi_pool_set_fused")

    def set_copy_streams(self, n: int):
        check(self.lib.pi_pool_set_copy_streams(self.h, n), "pi_pool_set_copy_streams")

    def pin_layer(self, layer: int, pinned: bool = True):
        check(self.lib.pi_pool_pin_layer(self.h, layer, int(bool(pinned))), "pi_pool_pin_layer")

    def admission(self, link_util: float):
        """One IO-adaptive admission decision; returns (layer changed or -1, pinned)."""
        layer, pinned = ctypes.c_int(), ctypes.c_int()
        check(self.lib.pi_pool_admission(self.h, float(link_util), ctypes.byref(layer), ctypes.byref(pinned)),
              "pi_pool_admission")
        return layer.value, bool(pinned.value)

    def recall_totals(self, reset: bool = False) -> tuple[int, int]:
        """(blocks recalled, hits) accumulated on the device since creation or the last reset."""
        m, h = ctypes.c_longlong(), ctypes.c_longlong()
        check(self.lib.pi_pool_recall_totals(self.h, ctypes.byref(m), ctypes.byref(h), int(bool(reset))),
              "pi_pool_recall_totals")
        return m.value, h.value

    def set_consensus_lambda(self, lam: float):
        check(self.lib.pi_pool_set_consensus_lambda(self.h, float(lam)), "pi_pool_set_consensus_lambda")

    def set_selection(self, cluster: bool = True, ctas_per_unit: int = 0):
        check(self.lib.pi_pool_set_selection(self.h, int(bool(cluster)), int(ctas_per_unit)), "pi_pool_set_selection")

    def set_attention_cluster(self, on: bool):
        check(self.lib.pi_pool_set_attention_cluster(self.h, int(bool(on))), "pi_pool_set_attention_cluster")

    def set_evict(self, policy: int):
        check(self.lib.pi_pool_set_evict(self.h, policy), "pi_pool_set_evict")

    def view_slot_stamp(self):
        return device_view(self._views.slot_stamp, (self.R, self.L, self.U, self.p_max), "int32")

    def set_gather(self, ctas: int, depth: int, exclusive: bool = False):
        check(self.lib.pi_pool_set_gather(self.h, ctas, depth, int(exclusive)), "pi_pool_set_gather")

    def flush(self, layer: int = -1, stream=None):
        check(self.lib.pi_pool_flush(self.h, layer, _stream(stream)), "pi_pool_flush")

    def sparse_decode(self, layer: int, q, sel, table, nsel, out, lse=None, logits=None, stream=None):
        check(self.lib.pi_sparse_decode(self.h, layer, _ptr(q), _ptr(sel), _ptr(table), _ptr(nsel), _ptr(out),
                                        _ptr(lse), _ptr(logits), _stream(stream)), "pi_sparse_decode")

    def attention_mass(self, layer: int, q, sel, nsel, mass, per_head: bool = False, stream=None):
        """Share of each head's full attention that the selection keeps: mass [R][Hq] fp32."""
        check(self.lib.pi_attention_mass(self.h, layer, _ptr(q), _ptr(sel), _ptr(nsel), int(bool(per_head)),
                                         _ptr(mass), _stream(stream)), "pi_attention_mass")

    def decode_step(self, q_all, k_new_all, v_new_all, k_budget, out_all, lse_all=None, method: int = PI_RECALL_UVA,
                    compute=None, copy=None, stats: bool = False):
        st = pi_step_stats() if stats else None
        check(self.lib.pi_decode_step(self.h, _ptr(q_all), _ptr(k_new_all), _ptr(v_new_all), _ptr(k_budget), method,
                                      _ptr(out_all), _ptr(lse_all), _stream(compute), _stream(copy),
                                      ctypes.byref(st) if st is not None else None), "pi_decode_step")
        if st is None:
            return None
        d = st.recall.as_dict()
        d["selected"] = st.selected
        return d

    def decode_step_host(self, q_all, k_new_all, v_new_all, k_budget, out_all, lse_all=None,
                         method: int = PI_RECALL_UVA, compute=None, copy=None):
        """Host (numpy or pinned CPU tensor) inputs and outputs; returns when outputs are on the host."""
        check(self.lib.pi_decode_step_host(self.h, _ptr(q_all), _ptr(k_new_all), _ptr(v_new_all), _ptr(k_budget),
                                           method, _ptr(out_all), _ptr(lse_all), _stream(compute), _stream(copy)),
              "pi_decode_step_host")

    def set_timing(self, max_steps: int):
        check(self.lib.pi_pool_set_timing(self.h, max_steps), "pi_pool_set_timing")

    def get_timing(self) -> dict:
        arr = (_lib.pi_kernel_timing * _lib.PI_K_KINDS)()
        check(self.lib.pi_pool_get_timing(self.h, arr), "pi_pool_get_timing")
        return {name: {"launches": arr[i].launches, "total_ms": arr[i].total_ms, "busy_ms": arr[i].busy_ms}
                for i, name in enumerate(_lib.KERNEL_KINDS)}

    def device_status(self) -> int:
        return self.lib.pi_get_device_status(self.h)

    def clear_device_status(self):
        check(self.lib.pi_clear_device_status(self.h), "pi_clear_device_status")

    def selftest_bounded_wait(self, limit_cycles: int) -> int:
        return self.lib.pi_selftest_bounded_wait(self.h, limit_cycles)

    def set_fault(self, spec: str):
        check(self.lib.pi_set_fault(self.h, spec.encode()), "pi_set_fault")
