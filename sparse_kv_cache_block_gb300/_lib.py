"""ctypes binding of libpi.so: the C ABI declared in include/pi.h, same names.

Argument marshalling only; every step of the decode path runs in the CUDA
library. There is no fallback: if libpi.so cannot be loaded, ``load()``
raises.
"""
from __future__ import annotations

import ctypes
import os
import re

from .build import LIB, ROOT

c_int, c_ll, c_double, c_void_p, c_char_p, c_size_t = (
    ctypes.c_int, ctypes.c_longlong, ctypes.c_double, ctypes.c_void_p, ctypes.c_char_p, ctypes.c_size_t)

PI_OK, PI_ERR_INVALID, PI_ERR_CUDA, PI_ERR_OOM, PI_ERR_HOST_ALLOC = 0, 1, 2, 3, 4
PI_ERR_POOL_FULL, PI_ERR_TIMEOUT, PI_ERR_DEVICE, PI_ERR_STATE, PI_ERR_FAULT_INJECTED = 5, 6, 7, 8, 9
PI_SHARED, PI_HEADWISE, PI_CONSENSUS = 0, 1, 2
PI_RECALL_UVA, PI_RECALL_MEMCPY, PI_RECALL_STAGED = 0, 1, 2
PI_EVICT_ASCENDING, PI_EVICT_LRU = 0, 1


class pi_config(ctypes.Structure):
    _fields_ = [("layers", c_int), ("batch", c_int), ("hq", c_int), ("hkv", c_int), ("head_dim", c_int),
                ("block_tokens", c_int), ("max_blocks", c_int), ("pool_slots", c_int), ("k_max", c_int),
                ("window", c_int), ("select_mode", c_int), ("host_layers", c_int), ("staging_blocks", c_int),
                ("gather_ctas", c_int), ("gather_depth", c_int), ("evict_policy", c_int), ("host_alloc", c_int),
                ("pin_layers", c_int), ("pool_slots_per_req", ctypes.POINTER(c_int))]


class pi_recall_stats(ctypes.Structure):
    _fields_ = [("bytes", c_ll), ("fragments", c_ll), ("runs", c_ll), ("api_calls", c_ll), ("hits", c_ll),
                ("host_wait_ms", c_double), ("cpu_gather_ms", c_double)]

    def as_dict(self):
        return {k: getattr(self, k) for k, _ in self._fields_}


class pi_step_stats(ctypes.Structure):
    _fields_ = [("recall", pi_recall_stats), ("selected", c_ll)]


class pi_pool_views(ctypes.Structure):
    _fields_ = [("pool", c_void_p), ("slot_base", ctypes.POINTER(c_ll)), ("slots_per_req", ctypes.POINTER(c_int)),
                ("kmean", c_void_p), ("ntok", c_void_p), ("slot_of_block", c_void_p), ("block_of_slot", c_void_p),
                ("p_max", c_int), ("step_sel", c_void_p), ("step_nsel", c_void_p), ("step_table", c_void_p),
                ("block_bytes", c_size_t), ("frag_bytes", c_size_t), ("host_region_bytes", c_size_t),
                ("slot_stamp", c_void_p), ("slots_rl", ctypes.POINTER(c_int)), ("capacity_rl", ctypes.POINTER(c_int)),
                ("total_slots", c_ll), ("dev_status", c_void_p)]


class pi_kernel_timing(ctypes.Structure):
    _fields_ = [("launches", c_ll), ("total_ms", c_double), ("busy_ms", c_double)]


PI_K_KINDS = 5
KERNEL_KINDS = ["append", "select", "plan", "gather", "attention"]

_P = c_void_p  # pi_pool*, device/host pointers, streams
_SIGS = {
    "pi_abi_version": (c_int, []),
    "pi_status_str": (c_char_p, [c_int]),
    "pi_pool_create": (c_int, [ctypes.POINTER(pi_config), ctypes.POINTER(c_void_p)]),
    "pi_pool_destroy": (c_int, [_P]),
    "pi_pool_get_config": (c_int, [_P, ctypes.POINTER(pi_config)]),
    "pi_pool_get_views": (c_int, [_P, ctypes.POINTER(pi_pool_views)]),
    "pi_host_kv": (c_void_p, [_P, c_int, c_int]),
    "pi_update_summaries": (c_int, [_P, c_int, _P, c_int, c_int, _P, _P]),
    "pi_append_kv": (c_int, [_P, c_int, _P, _P, _P]),
    "pi_select_topk": (c_int, [_P, c_int, _P, _P, c_int, _P, _P, _P]),
    "pi_recall": (c_int, [_P, c_int, _P, _P, c_int, _P, ctypes.POINTER(pi_recall_stats), _P]),
    "pi_pool_preload": (c_int, [_P, c_int, c_int, _P, c_int, _P]),
    "pi_pool_flush": (c_int, [_P, c_int, _P]),
    "pi_pool_set_gather": (c_int, [_P, c_int, c_int, c_int]),
    "pi_pool_set_pipeline": (c_int, [_P, c_int, c_int]),
    "pi_pool_set_attention": (c_int, [_P, c_int]),
    "pi_pool_set_attention_cluster": (c_int, [_P, c_int]),
    "pi_pool_set_selection": (c_int, [_P, c_int, c_int]),
    "pi_pool_set_schedule": (c_int, [_P, c_int, c_int]),
    "pi_pool_set_copy_streams": (c_int, [_P, c_int]),
    "pi_pool_pin_layer": (c_int, [_P, c_int, c_int]),
    "pi_pool_admission": (c_int, [_P, c_double, ctypes.POINTER(c_int), ctypes.POINTER(c_int)]),
    "pi_pool_recall_totals": (c_int, [_P, ctypes.POINTER(c_ll), ctypes.POINTER(c_ll), c_int]),
    "pi_pool_set_consensus_lambda": (c_int, [_P, ctypes.c_float]),
    "pi_pool_set_fused": (c_int, [_P, c_int, c_int]),
    "pi_admission_decide": (c_int, [c_int, _P, _P, c_int, ctypes.c_double, _P, _P]),
    "pi_pool_set_evict": (c_int, [_P, c_int]),
    "pi_sparse_decode": (c_int, [_P, c_int, _P, _P, _P, _P, _P, _P, _P, _P]),
    "pi_attention_mass": (c_int, [_P, c_int, _P, _P, _P, c_int, _P, _P]),
    "pi_sparse_decode_noalloc": (c_int, [_P, c_ll, c_int, c_int, c_int, c_int, c_int, c_int, _P, _P, _P, _P, _P,
                                         _P, _P, _P]),
    "pi_sparse_decode_noalloc_status": (c_int, [_P]),
    "pi_decode_step": (c_int, [_P, _P, _P, _P, _P, c_int, _P, _P, _P, _P, ctypes.POINTER(pi_step_stats)]),
    "pi_decode_step_host": (c_int, [_P, _P, _P, _P, _P, c_int, _P, _P, _P, _P]),
    "pi_pool_set_timing": (c_int, [_P, c_int]),
    "pi_pool_get_timing": (c_int, [_P, ctypes.POINTER(pi_kernel_timing)]),
    "pi_get_device_status": (c_int, [_P]),
    "pi_clear_device_status": (c_int, [_P]),
    "pi_set_fault": (c_int, [_P, c_char_p]),
    "pi_selftest_bounded_wait": (c_int, [_P, c_ll]),
}

_lib = None


def declared_functions() -> list[str]:
    """Names of the functions include/pi.h declares."""
    hdr = open(os.path.join(ROOT, "include", "pi.h")).read()
    hdr = re.sub(r"/\*.*?\*/", "", hdr, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\**\s*(pi_\w+)\s*\(", hdr, flags=re.M)))


def load(path: str | None = None):
    """Load libpi.so (build it first with sparse_kv_cache_block_gb300.build.build()).

    Raises OSError/FileNotFoundError when the library is absent: there is no
    fallback implementation."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or LIB
    if not os.path.exists(path):
        raise FileNotFoundError(f"libpi.so not built ({path}); run __graft_entry__.build()")
    lib = ctypes.CDLL(path)
    for name, (res, args) in _SIGS.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


class PiError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        msg = load().pi_status_str(status).decode()
        super().__init__(f"{what}: {msg} ({status})" if what else f"{msg} ({status})")


def check(status: int, what: str = "") -> None:
    if status != PI_OK:
        raise PiError(status, what)
