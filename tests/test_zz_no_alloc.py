"""The allocation-free decode entry point (spear_linear_forward_decode_noalloc).

It serves callers that cannot call cudaMalloc at all (memory fully reserved by
another allocator, or allocation-free serving loops): everything comes from the
caller except a small static scratch array inside the library. Checked through
the C ABI against the handle-based decode entry point, on two calls in a row
(the scratch array keeps the previous call's contents). Collected last so that
a failure here cannot stop the other GPU tests from running.
"""
import ctypes

import numpy as np
import pytest
import torch

from quantized_linear_error_gb300 import build, spear
from quantized_linear_error_gb300 import workload as wl

from .helpers import dev_bf16, host_f64, rel_err

pytestmark = pytest.mark.gpu
TOL = 1e-2


@pytest.fixture(scope="module")
def L():
    build.build()
    return spear.load()


def _desc_and_tensors(w):
    sp = w.spec
    keep = {
        "q": torch.from_numpy(w.q).cuda(),
        "s": dev_bf16(w.s),
        "z": torch.from_numpy(w.z).cuda(),
        "A": dev_bf16(w.A) if sp.rank else None,
        "B": dev_bf16(w.B) if sp.rank else None,
    }
    ptr = lambda t: None if t is None else t.data_ptr()
    d = spear.spear_linear_desc_t(sp.K, sp.N, sp.group_size, ptr(keep["q"]), ptr(keep["s"]), ptr(keep["z"]),
                                  sp.rank, ptr(keep["A"]), ptr(keep["B"]), sp.alpha, sp.gate, 32)
    return d, keep


@pytest.mark.parametrize("spec,Ms", [
    (wl.LinearSpec("na/g128", 1024, 4104, 128, 64), (7, 32)),
    (wl.LinearSpec("na/pc", 640, 520, 0, 256), (16, 3)),
])
def test_matches_handle_decode_two_calls(L, spec, Ms):
    w = wl.make_weights(spec, 21)
    d, keep = _desc_and_tensors(w)
    lin = spear.from_weights(w, max_tokens=32)
    stream = torch.cuda.current_stream().cuda_stream
    for call, M in enumerate(Ms):
        x = dev_bf16(wl.make_x(spec.K, M, w.outliers, call, f"na/{call}"))
        y_ref = torch.empty((M, spec.N), dtype=torch.bfloat16, device="cuda")
        lin.forward_decode(x, y_ref)
        y = torch.full((M, spec.N), float("nan"), dtype=torch.bfloat16, device="cuda")
        st = L.spear_linear_forward_decode_noalloc(ctypes.byref(d), x.data_ptr(), y.data_ptr(), M, stream)
        assert st == spear.SPEAR_OK, spear.status_string(st)
        torch.cuda.synchronize()
        e = rel_err(host_f64(y), host_f64(y_ref))
        assert e <= TOL, f"call {call} M={M}: rel err {e:.3e}"
    assert lin.check() == spear.SPEAR_OK


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
