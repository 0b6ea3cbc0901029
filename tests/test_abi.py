"""The C-ABI library builds for sm_103a, loads, and exports every symbol that
include/pi.h declares (no GPU needed: no compute call is made)."""
import ctypes
import os
import subprocess

import pytest

import sparse_kv_cache_block_gb300 as pi
from sparse_kv_cache_block_gb300 import _lib


@pytest.fixture(scope="module")
def lib():
    pi.build()
    return pi.load()


def test_header_declares_the_boundary():
    names = set(pi.declared_functions())
    for n in ("pi_pool_create", "pi_pool_destroy", "pi_update_summaries", "pi_append_kv", "pi_select_topk",
              "pi_recall", "pi_sparse_decode", "pi_decode_step", "pi_decode_step_host", "pi_host_kv",
              "pi_get_device_status", "pi_status_str"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for n in pi.declared_functions():
        assert hasattr(lib, n), n
    out = subprocess.run(["nm", "-D", "--defined-only", pi.build()], capture_output=True, text=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    assert set(pi.declared_functions()) <= exported


def test_binding_covers_every_declared_function():
    assert set(pi.declared_functions()) == set(_lib._SIGS)


def test_host_only_calls(lib):
    assert lib.pi_abi_version() == 1
    assert lib.pi_status_str(pi.PI_ERR_POOL_FULL).decode().startswith("pool")
    assert lib.pi_pool_create(None, None) == pi.PI_ERR_INVALID
    assert lib.pi_pool_destroy(None) == pi.PI_ERR_INVALID
    assert lib.pi_host_kv(None, 0, 0) is None
    # every entry point checks its pool before touching the device
    null_calls = {
        "pi_select_topk": (None, 0, None, None, 0, None, None, None),
        "pi_recall": (None, 0, None, None, 0, None, None, None),
        "pi_sparse_decode": (None, 0, None, None, None, None, None, None, None, None),
        "pi_attention_mass": (None, 0, None, None, None, 0, None, None),
        "pi_pool_set_fused": (None, 1, 0),
        "pi_pool_set_schedule": (None, 1, 2),
        "pi_pool_set_copy_streams": (None, 2),
        "pi_pool_pin_layer": (None, 0, 1),
        "pi_pool_set_consensus_lambda": (None, 0.5),
        "pi_pool_set_attention_cluster": (None, 1),
        "pi_pool_recall_totals": (None, None, None, 0),
    }
    for name, args in null_calls.items():
        assert getattr(lib, name)(*args) == pi.PI_ERR_INVALID, name


def test_library_is_built_for_sm103a_only():
    import importlib
    b = importlib.import_module("sparse_kv_cache_block_gb300.build")
    assert b.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]


def test_struct_layouts_match_header():
    # the binding's structs must match the C layout compiled into the library
    hdr = open(os.path.join(os.path.dirname(pi.build()), "..", "include", "pi.h")).read()
    for field in ("gather_ctas", "pool_slots_per_req", "cpu_gather_ms", "host_region_bytes"):
        assert field in hdr
    assert ctypes.sizeof(_lib.pi_config) == 18 * 4 + 8
    assert ctypes.sizeof(_lib.pi_recall_stats) == 5 * 8 + 2 * 8


def test_missing_library_fails_loudly(tmp_path, monkeypatch):
    """No fallback: loading a library that is not there raises."""
    monkeypatch.setattr(_lib, "_lib", None)
    with pytest.raises(FileNotFoundError):
        _lib.load(str(tmp_path / "libpi.so"))


def test_product_path_never_touches_the_oracle():
    """The package and the bench's GPU leg stay independent of oracle/: no
    source file of the package names it."""
    pkg = os.path.dirname(_lib.__file__)
    for root, _, files in os.walk(pkg):
        if "_build" in root or "__pycache__" in root:
            continue
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                src = open(os.path.join(root, f)).read()
                assert "import oracle" not in src and "from oracle" not in src and "pi_oracle" not in src, f
