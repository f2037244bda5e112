"""C-ABI boundary checks that need no GPU: the library builds, loads, exports
every function the header declares, and rejects bad arguments before touching
the device."""
import ctypes

import pytest

from quantized_linear_error_gb300 import build, spear


@pytest.fixture(scope="module")
def L():
    build.build()
    return spear.load()


def test_exports_every_header_function(L):
    names = spear.header_functions()
    assert {"spear_linear_create", "spear_linear_forward_decode", "spear_linear_forward_prefill",
            "spear_linear_destroy"} <= set(names)
    for n in names:
        assert hasattr(L, n), f"{n} declared in spear.h but not exported"


def test_status_strings(L):
    assert [spear.status_string(i) for i in range(6)] == [
        "SPEAR_OK", "SPEAR_ERR_INVALID_ARG", "SPEAR_ERR_UNSUPPORTED", "SPEAR_ERR_OOM", "SPEAR_ERR_CUDA",
        "SPEAR_ERR_TIMEOUT"]


def _desc(**kw):
    d = dict(K=256, N=64, group_size=128, qweight=16, scales=16, zeros=None, rank=0, A=None, B=None,
             alpha=1.0, gate=0, max_tokens=4, gate_hidden=0, gate_w1=None, gate_w2=None)
    d.update(kw)
    return spear.spear_linear_desc_t(*[d[f] for f, _ in spear.spear_linear_desc_t._fields_])


@pytest.mark.parametrize("bad", [dict(K=100), dict(K=0), dict(N=12), dict(group_size=64), dict(qweight=None),
                                 dict(scales=None), dict(rank=8), dict(rank=272), dict(rank=16),
                                 dict(max_tokens=0), dict(gate=7)])
def test_create_rejects_bad_descriptor(L, bad):
    h = ctypes.c_void_p(1234)
    assert L.spear_linear_create(ctypes.byref(_desc(**bad)), None, ctypes.byref(h)) == spear.SPEAR_ERR_INVALID_ARG
    assert h.value is None


def test_null_arguments(L):
    h = ctypes.c_void_p()
    assert L.spear_linear_create(None, None, ctypes.byref(h)) == spear.SPEAR_ERR_INVALID_ARG
    assert L.spear_linear_create(ctypes.byref(_desc()), None, None) == spear.SPEAR_ERR_INVALID_ARG
    for fn in (L.spear_linear_forward_decode, L.spear_linear_forward_prefill, L.spear_linear_forward):
        assert fn(None, 16, 32, 1, None) == spear.SPEAR_ERR_INVALID_ARG
    assert L.spear_linear_forward_host(None, 16, 32, 1, None) == spear.SPEAR_ERR_INVALID_ARG
    assert L.spear_linear_forward_host_batch(None, None, None, None, 1, None) == spear.SPEAR_ERR_INVALID_ARG
    nulls = (ctypes.c_void_p * 1)(None)
    ms = (ctypes.c_int32 * 1)(1)
    assert L.spear_linear_forward_host_batch(nulls, nulls, nulls, ms, 1, None) == spear.SPEAR_ERR_INVALID_ARG
    assert L.spear_linear_forward_host_batch(None, None, None, None, 0, None) == spear.SPEAR_OK
    assert L.spear_linear_forward_host_batch(None, None, None, None, -1, None) == spear.SPEAR_ERR_INVALID_ARG
    assert L.spear_linear_dequantize(None, 0, 16, None) == spear.SPEAR_ERR_INVALID_ARG
    assert L.spear_linear_check(None, None) == spear.SPEAR_ERR_INVALID_ARG
    assert L.spear_linear_debug_set(None, 0, 0) == spear.SPEAR_ERR_INVALID_ARG
    assert L.spear_linear_destroy(None) == spear.SPEAR_OK
    assert L.spear_linear_enable_concurrent_ec(None) == spear.SPEAR_ERR_INVALID_ARG
    assert L.spear_linear_forward_prefill_concurrent(None, 16, 32, 1, None, None) == spear.SPEAR_ERR_INVALID_ARG


_MLP = dict(gate=spear.SPEAR_GATE_MLP, rank=16, A=16, B=16, gate_hidden=8, gate_w1=16, gate_w2=32)


@pytest.mark.parametrize("bad", [dict(gate_hidden=0), dict(gate_hidden=65), dict(gate_w1=None), dict(gate_w2=None),
                                 dict(gate_w1=24), dict(rank=0, A=None, B=None)])
def test_create_rejects_bad_mlp_gate(L, bad):
    h = ctypes.c_void_p(1234)
    d = _desc(**{**_MLP, **bad})
    assert L.spear_linear_create(ctypes.byref(d), None, ctypes.byref(h)) == spear.SPEAR_ERR_INVALID_ARG
    assert h.value is None


def test_noalloc_entry_point_rejects_mlp_gate(L):
    """The allocation-free decode has no MLP gate: refused before any device work."""
    d = _desc(**_MLP)
    assert L.spear_linear_forward_decode_noalloc(ctypes.byref(d), 16, 32, 1, None) == spear.SPEAR_ERR_UNSUPPORTED


def test_grouped_create_rejects_incompatible_members(L):
    """Checked before any device work: members must share K, group size, rank
    and gate, have N a multiple of 16 and a stacked rank <= 256; the MLP gate
    is not supported for groups; 1..8 members."""
    base = dict(K=256, N=64, group_size=128, rank=16, A=16, B=16)
    cases = [([base, {**base, "K": 512}], spear.SPEAR_ERR_INVALID_ARG),
             ([base, {**base, "rank": 32, "A": 16, "B": 16}], spear.SPEAR_ERR_INVALID_ARG),
             ([base, {**base, "group_size": 0}], spear.SPEAR_ERR_INVALID_ARG),
             ([base, {**base, "N": 72}], spear.SPEAR_ERR_INVALID_ARG),
             ([base, {**base, "gate": 1}], spear.SPEAR_ERR_INVALID_ARG),
             ([{**base, "rank": 144}, {**base, "rank": 144}], spear.SPEAR_ERR_INVALID_ARG),
             ([{**base, **_MLP}, {**base, **_MLP}], spear.SPEAR_ERR_UNSUPPORTED),
             ([base] * 9, spear.SPEAR_ERR_INVALID_ARG)]
    for members, want in cases:
        arr = (spear.spear_linear_desc_t * len(members))(*[_desc(**m) for m in members])
        h = ctypes.c_void_p(1234)
        assert L.spear_linear_create_grouped(arr, len(members), None, ctypes.byref(h)) == want, members
        assert h.value is None
    h = ctypes.c_void_p()
    assert L.spear_linear_create_grouped(None, 2, None, ctypes.byref(h)) == spear.SPEAR_ERR_INVALID_ARG
    assert L.spear_linear_create_grouped(None, 0, None, ctypes.byref(h)) == spear.SPEAR_ERR_INVALID_ARG
