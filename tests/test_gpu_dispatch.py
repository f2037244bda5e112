"""The phase-dispatching entry points against the fp64 oracle.

spear_linear_forward sends M <= 32 to the decode kernel and larger M to the
prefill path ("SPEAR", section 2.2A: the two phases of one layer);
spear_linear_forward_host does the same from host buffers, with the copies
inside the call. Both are checked on handles with and without a compensator,
at token counts on both sides of the dispatch boundary, with the layer's
tolerance max |y - y_ref| / max |y_ref| <= 1e-2.
"""
import numpy as np
import pytest
import torch

from oracle import ref
from quantized_linear_error_gb300 import spear
from quantized_linear_error_gb300 import workload as wl

from .helpers import bits_of, codes_equal_zeros, dev_bf16, host_f64, rel_err

pytestmark = pytest.mark.gpu
TOL = 1e-2
SPECS = [
    wl.LinearSpec("dp/g128", 1024, 1032, 128, 64),
    wl.LinearSpec("dp/pc", 640, 520, 0, 32),
    wl.LinearSpec("dp/noec", 768, 392, 128, 0),
]
TOKENS = (1, 32, 33, 300)


@pytest.fixture(scope="module", params=SPECS, ids=lambda s: s.name)
def layer(request):
    w = wl.make_weights(request.param, 31)
    lin = spear.from_weights(w, max_tokens=max(TOKENS))
    yield w, lin
    lin.close()


@pytest.mark.parametrize("M", TOKENS)
def test_forward_device(layer, M):
    w, lin = layer
    xb = wl.make_x(w.spec.K, M, w.outliers, M, "dp/x")
    y = torch.full((M, w.spec.N), float("nan"), dtype=torch.bfloat16, device="cuda")
    lin.forward(dev_bf16(xb), y)
    assert lin.check() == spear.SPEAR_OK
    e = rel_err(host_f64(y), ref.forward_w(w, xb))
    assert e <= TOL, f"M={M}: rel err {e:.3e}"


@pytest.mark.parametrize("pinned", [True, False], ids=["pinned", "pageable"])
@pytest.mark.parametrize("M", TOKENS)
def test_forward_host(layer, M, pinned):
    w, lin = layer
    xb = wl.make_x(w.spec.K, M, w.outliers, M + 1, "dp/xh")
    xh = torch.from_numpy(np.ascontiguousarray(xb).view(np.int16)).view(torch.bfloat16)
    yh = torch.full((M, w.spec.N), float("nan"), dtype=torch.bfloat16)
    if pinned:
        xh, yh = xh.pin_memory(), yh.pin_memory()
    lin.forward_host(xh, yh)
    assert lin.check() == spear.SPEAR_OK
    e = rel_err(yh.double().numpy(), ref.forward_w(w, xb))
    assert e <= TOL, f"M={M}: rel err {e:.3e}"


def test_host_and_device_paths_agree_on_the_prefill_side(layer):
    """Above the boundary both calls run the same prefill kernels on the same
    handle. Without a compensator they are deterministic (partial tiles are
    added in CTA order), so the host entry point's result is the device
    entry point's bit for bit; with one, the pre-kernel sums z over its K
    splits with atomics in arbitrary order, so u' may differ by one bf16 ulp
    and y agrees to well inside the tolerance."""
    w, lin = layer
    M = 300
    xb = wl.make_x(w.spec.K, M, w.outliers, 5, "dp/agree")
    y = torch.empty((M, w.spec.N), dtype=torch.bfloat16, device="cuda")
    lin.forward(dev_bf16(xb), y)
    xh = torch.from_numpy(np.ascontiguousarray(xb).view(np.int16)).view(torch.bfloat16).pin_memory()
    yh = torch.empty((M, w.spec.N), dtype=torch.bfloat16).pin_memory()
    lin.forward_host(xh, yh)
    if w.spec.rank == 0:
        np.testing.assert_array_equal(bits_of(y), yh.view(torch.int16).numpy().view(np.uint16))
    else:
        assert rel_err(yh.double().numpy(), host_f64(y)) <= 1e-3


def test_compensator_dominant_through_the_dispatcher():
    """Codes equal to zeros (W_q = 0, y is the compensator alone) on both sides
    of the boundary: a dispatcher that dropped the compensator would fail."""
    w = codes_equal_zeros(wl.make_weights(SPECS[0], 32))
    lin = spear.from_weights(w, max_tokens=300)
    for M in (8, 300):
        xb = wl.make_x(w.spec.K, M, w.outliers, M, "dp/ec")
        y = torch.empty((M, w.spec.N), dtype=torch.bfloat16, device="cuda")
        lin.forward(dev_bf16(xb), y)
        e = rel_err(host_f64(y), ref.forward_w(w, xb))
        assert e <= TOL, f"M={M}: rel err {e:.3e}"
        xh = torch.from_numpy(np.ascontiguousarray(xb).view(np.int16)).view(torch.bfloat16).pin_memory()
        yh = torch.empty((M, w.spec.N), dtype=torch.bfloat16).pin_memory()
        lin.forward_host(xh, yh)
        e = rel_err(yh.double().numpy(), ref.forward_w(w, xb))
        assert e <= TOL, f"host M={M}: rel err {e:.3e}"
    assert lin.check() == spear.SPEAR_OK
    lin.close()


def test_host_entry_rejects_more_tokens_than_the_handle_holds(layer):
    w, lin = layer
    M = max(TOKENS) + 1
    xh = torch.zeros((M, w.spec.K), dtype=torch.bfloat16)
    yh = torch.zeros((M, w.spec.N), dtype=torch.bfloat16)
    with pytest.raises(spear.SpearError) as ei:
        lin.forward_host(xh, yh)
    assert ei.value.status == spear.SPEAR_ERR_INVALID_ARG


def test_host_batch_against_oracle():
    """spear_linear_forward_host_batch: several handles, one of them twice,
    token counts on both sides of the dispatch boundary, one synchronisation;
    every result against the oracle."""
    ws = [wl.make_weights(sp, 33) for sp in SPECS]
    lins = [spear.from_weights(w, max_tokens=300) for w in ws]
    plan = [(0, 1), (1, 32), (2, 300), (0, 33), (1, 8)]
    xs_bits, xs, ys = [], [], []
    for i, (li, M) in enumerate(plan):
        xb = wl.make_x(ws[li].spec.K, M, ws[li].outliers, i, "dp/batch")
        xs_bits.append(xb)
        xs.append(torch.from_numpy(np.ascontiguousarray(xb).view(np.int16)).view(torch.bfloat16).pin_memory())
        ys.append(torch.full((M, ws[li].spec.N), float("nan"), dtype=torch.bfloat16).pin_memory())
    spear.forward_host_batch([lins[li] for li, _ in plan], xs, ys)
    for i, (li, M) in enumerate(plan):
        e = rel_err(ys[i].double().numpy(), ref.forward_w(ws[li], xs_bits[i]))
        assert e <= TOL, f"call {i} (linear {li}, M={M}): rel err {e:.3e}"
    for lin in lins:
        assert lin.check() == spear.SPEAR_OK
        lin.close()
