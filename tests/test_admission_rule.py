"""The IO-adaptive admission rule on the host (no device): the guide's
"Interruptible Layer-Wise Scheduling & Adaptive Admission", "2. IO-Adaptive
Offloading Admission" -- pin the next layer (most active first: 0, L-1, 1,
L-2, ...) while the link is saturated (utilisation above 0.85), release the
layer pinned last when it is quiet (below 0.5), otherwise leave residency
alone. The library's pool-level call applies exactly this decision."""
import ctypes

import pytest

import sparse_kv_cache_block_gb300 as pi


@pytest.fixture(scope="module")
def lib():
    pi.build()
    return pi.load()


def decide(lib, pinnable, pinned, last, util):
    L = len(pinnable)
    a = (ctypes.c_int * L)(*pinnable)
    b = (ctypes.c_int * L)(*pinned)
    layer, pin = ctypes.c_int(), ctypes.c_int()
    st = lib.pi_admission_decide(L, ctypes.cast(a, ctypes.c_void_p), ctypes.cast(b, ctypes.c_void_p), last, util,
                                 ctypes.byref(layer), ctypes.byref(pin))
    return st, layer.value, pin.value


def test_saturated_link_pins_the_most_active_layers_first(lib):
    L = 6
    pinned, order, last = [0] * L, [], -1
    for _ in range(L + 1):
        st, layer, pin = decide(lib, [1] * L, pinned, last, 0.9)
        assert st == pi.PI_OK
        if layer < 0:
            break
        assert pin == 1
        pinned[layer] = 1
        order.append(layer)
        last = layer
    assert order == [0, 5, 1, 4, 2, 3]
    assert decide(lib, [1] * L, pinned, last, 0.99) == (pi.PI_OK, -1, 0)  # every layer pinned


def test_only_layers_with_reserved_room_are_pinned(lib):
    # 8 layers, room for 3: the first ceil(3/2) = 2 and the last floor(3/2) = 1
    pinnable = [1, 1, 0, 0, 0, 0, 0, 1]
    pinned, order, last = [0] * 8, [], -1
    while True:
        st, layer, pin = decide(lib, pinnable, pinned, last, 0.86)
        if layer < 0:
            break
        pinned[layer] = 1
        order.append(layer)
        last = layer
    assert order == [0, 7, 1]


def test_thresholds_and_release(lib):
    pinnable, pinned = [1] * 4, [1, 0, 0, 1]
    assert decide(lib, pinnable, pinned, 3, 0.85) == (pi.PI_OK, -1, 0)   # at the threshold: no change
    assert decide(lib, pinnable, pinned, 3, 0.5) == (pi.PI_OK, -1, 0)
    assert decide(lib, pinnable, pinned, 3, 0.7) == (pi.PI_OK, -1, 0)
    assert decide(lib, pinnable, pinned, 3, 0.49) == (pi.PI_OK, 3, 0)    # the layer pinned last goes first
    assert decide(lib, pinnable, [0] * 4, -1, 0.1) == (pi.PI_OK, -1, 0)  # nothing pinned: nothing to release
    assert decide(lib, pinnable, pinned, 3, 0.851) == (pi.PI_OK, 1, 1)   # order 0, 3, 1, 2 with 0 and 3 held
    assert decide(lib, pinnable, pinned, 3, 0.0)[1:] == (3, 0)


def test_invalid_arguments(lib):
    assert decide(lib, [1, 1], [0, 0], -1, float("nan"))[0] == pi.PI_ERR_INVALID
    assert decide(lib, [1, 1], [0, 0], -1, -0.1)[0] == pi.PI_ERR_INVALID
    layer, pin = ctypes.c_int(), ctypes.c_int()
    assert lib.pi_admission_decide(0, None, None, -1, 0.9, ctypes.byref(layer), ctypes.byref(pin)) == pi.PI_ERR_INVALID
    a = (ctypes.c_int * 2)(1, 1)
    assert lib.pi_admission_decide(2, ctypes.cast(a, ctypes.c_void_p), None, -1, 0.9, ctypes.byref(layer),
                                   ctypes.byref(pin)) == pi.PI_ERR_INVALID


def test_stale_last_pinned_layer_is_rejected(lib):
    """A controller that names as pinned last a layer that is not pinned (or has
    no reserved room, or does not exist) gets PI_ERR_INVALID, not a release."""
    pinnable = [1, 1, 0, 1]
    assert decide(lib, pinnable, [1, 0, 0, 0], 1, 0.1)[0] == pi.PI_ERR_INVALID   # layer 1 is not pinned
    assert decide(lib, pinnable, [1, 0, 1, 0], 2, 0.1)[0] == pi.PI_ERR_INVALID   # layer 2 has no room
    assert decide(lib, pinnable, [1, 0, 0, 0], 4, 0.1)[0] == pi.PI_ERR_INVALID   # no layer 4
    assert decide(lib, pinnable, [1, 0, 0, 0], 1, 0.9)[0] == pi.PI_ERR_INVALID   # checked whatever the load
    assert decide(lib, pinnable, [1, 0, 0, 0], 0, 0.1) == (pi.PI_OK, 0, 0)
