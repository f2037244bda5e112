"""The allocation-free decode entry point (spear_linear_forward_decode_noalloc).

It serves callers that cannot call cudaMalloc at all (memory fully reserved by
another allocator, or serving loops that must not allocate): everything comes
from the caller except a small static scratch array inside the library.
Checked through the C ABI against the fp64 oracle and against the handle-based
decode entry point, on two calls in a row (the scratch array keeps the
previous call's contents). Collected last so that a failure here cannot stop
the other GPU tests from running.
"""
import ctypes

import numpy as np
import pytest
import torch

from oracle import ref
from quantized_linear_error_gb300 import build, spear
from quantized_linear_error_gb300 import workload as wl

from .helpers import codes_equal_zeros, dev_bf16, host_f64, rel_err, with_spec

pytestmark = pytest.mark.gpu
TOL = 1e-2


@pytest.fixture(scope="module")
def L():
    build.build()
    return spear.load()


def _desc_and_tensors(w, zeros=True):
    sp = w.spec
    keep = {
        "q": torch.from_numpy(w.q).cuda(),
        "s": dev_bf16(w.s),
        "z": torch.from_numpy(w.z).cuda() if zeros else None,
        "A": dev_bf16(w.A) if sp.rank else None,
        "B": dev_bf16(w.B) if sp.rank else None,
    }
    ptr = lambda t: None if t is None else t.data_ptr()
    d = spear.spear_linear_desc_t(sp.K, sp.N, sp.group_size, ptr(keep["q"]), ptr(keep["s"]), ptr(keep["z"]),
                                  sp.rank, ptr(keep["A"]), ptr(keep["B"]), sp.alpha, sp.gate, 32)
    return d, keep


def _noalloc(L, d, x, N):
    M = x.shape[0]
    y = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    st = L.spear_linear_forward_decode_noalloc(ctypes.byref(d), x.data_ptr(), y.data_ptr(), M,
                                               torch.cuda.current_stream().cuda_stream)
    assert st == spear.SPEAR_OK, spear.status_string(st)
    torch.cuda.synchronize()
    return host_f64(y)


@pytest.mark.parametrize("spec,Ms", [
    (wl.LinearSpec("na/g128", 1024, 4104, 128, 64), (7, 32)),
    (wl.LinearSpec("na/pc", 640, 520, 0, 256), (16, 3)),
])
def test_matches_handle_decode_two_calls(L, spec, Ms):
    w = wl.make_weights(spec, 21)
    d, keep = _desc_and_tensors(w)
    lin = spear.from_weights(w, max_tokens=32)
    for call, M in enumerate(Ms):
        xb = wl.make_x(spec.K, M, w.outliers, call, f"na/{call}")
        x = dev_bf16(xb)
        y_ref = torch.empty((M, spec.N), dtype=torch.bfloat16, device="cuda")
        lin.forward_decode(x, y_ref)
        y = _noalloc(L, d, x, spec.N)
        e = rel_err(y, host_f64(y_ref))
        assert e <= TOL, f"call {call} M={M}: rel err {e:.3e} against the handle path"
        e = rel_err(y, ref.forward_w(w, xb))
        assert e <= TOL, f"call {call} M={M}: rel err {e:.3e} against the oracle"
    assert lin.check() == spear.SPEAR_OK


def _variant(name, w):
    if name == "zeros_null":
        return wl.LinearWeights(w.spec, w.q, w.s, None, w.A, w.B, w.outliers)
    if name == "gate_one":
        return with_spec(w, gate=wl.GATE_ONE)
    if name == "rank0":
        return wl.LinearWeights(with_spec(w, rank=0).spec, w.q, w.s, w.z, None, None, w.outliers)
    if name == "alpha0":
        return with_spec(w, alpha=0.0)
    if name == "ec_only":
        return codes_equal_zeros(w)
    if name == "alpha30":
        return with_spec(w, alpha=30.0)
    raise ValueError(name)


@pytest.mark.parametrize("variant", ["zeros_null", "gate_one", "rank0", "alpha0", "ec_only", "alpha30"])
def test_variants_against_oracle(L, variant):
    """Null zeros (z = 8), the constant gate, no compensator, alpha = 0, codes
    equal to zeros (the compensator alone) and alpha = 30, each on two calls
    in a row against the fp64 oracle."""
    w = _variant(variant, wl.make_weights(wl.LinearSpec("na/var", 768, 392, 128, 32), 23))
    d, keep = _desc_and_tensors(w, zeros=w.z is not None)
    for call, M in enumerate((5, 32)):
        xb = wl.make_x(w.spec.K, M, w.outliers, call, f"na/var{call}")
        y = _noalloc(L, d, dev_bf16(xb), w.spec.N)
        e = rel_err(y, ref.forward_w(w, xb))
        assert e <= TOL, f"{variant} call {call} M={M}: rel err {e:.3e}"


def test_rejects_sizes_beyond_scratch(L):
    w = wl.make_weights(wl.LinearSpec("na/big", 256, 64, 128, 16), 22)
    d, keep = _desc_and_tensors(w)
    x = torch.zeros((33, 256), dtype=torch.bfloat16, device="cuda")
    y = torch.zeros((33, 64), dtype=torch.bfloat16, device="cuda")
    assert L.spear_linear_forward_decode_noalloc(ctypes.byref(d), x.data_ptr(), y.data_ptr(), 33, None) == \
        spear.SPEAR_ERR_INVALID_ARG
    d.rank = 272
    assert L.spear_linear_forward_decode_noalloc(ctypes.byref(d), x.data_ptr(), y.data_ptr(), 4, None) == \
        spear.SPEAR_ERR_INVALID_ARG
    assert L.spear_linear_forward_decode_noalloc(None, x.data_ptr(), y.data_ptr(), 4, None) == \
        spear.SPEAR_ERR_INVALID_ARG
