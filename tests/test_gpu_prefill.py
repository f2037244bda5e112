"""Parity of the tensor-core prefill path against the fp64 oracle.

Same bound as decode: max |y_gpu - y_ref| / max |y_ref| <= 1e-2 per call,
also on compensator-dominant inputs (codes equal to zeros; alpha = 30). The
prefill weights are the exported bf16 dequantised values and u is rounded to
bf16 once, both far inside the bound.
"""
import numpy as np
import pytest

from oracle import ref
from quantized_linear_error_gb300 import spear
from quantized_linear_error_gb300 import workload as wl

from .helpers import codes_equal_zeros, rel_err, run, sample_rows, with_spec
from .test_gpu_decode import SMALL

pytestmark = pytest.mark.gpu
TOL = 1e-2


def _check(w, M, rows=None, lin=None, seed=0):
    sp = w.spec
    x = wl.make_x(sp.K, M, w.outliers, seed, sp.name)
    lin = lin or spear.from_weights(w, max_tokens=M)
    y = run(lin, x, "prefill")
    yr = ref.forward_w(w, x, rows)
    e = rel_err(y if rows is None else y[:, rows], yr)
    assert e <= TOL, f"{sp.name} M={M}: rel err {e:.3e}"
    return y


@pytest.mark.parametrize("M", [1, 33, 100, 256, 300, 513])
@pytest.mark.parametrize("sp", SMALL, ids=lambda s: s.name)
def test_small_shapes(sp, M):
    _check(wl.make_weights(sp, 11), M)


@pytest.mark.parametrize("sp", SMALL[:2] + SMALL[3:], ids=lambda s: s.name)
def test_compensator_dominant(sp):
    w = wl.make_weights(sp, 12)
    _check(codes_equal_zeros(w), 200)
    _check(with_spec(w, alpha=30.0), 130)
    _check(with_spec(codes_equal_zeros(w), gate=wl.GATE_ONE), 64)


def test_matches_decode_path():
    """Both phases compute the same layer: at M <= 32 they agree closely."""
    w = wl.make_weights(SMALL[3], 13)
    lin = spear.from_weights(w, max_tokens=32)
    x = wl.make_x(w.spec.K, 24, w.outliers, 0, "both")
    yd, yp = run(lin, x, "decode"), run(lin, x, "prefill")
    assert rel_err(yp, yd) <= 5e-3


@pytest.mark.parametrize("idx", range(3))
def test_config3_mlp(idx):
    sp = wl.config_linears(3)[idx]
    w = wl.make_weights(sp, 0)
    rows = sample_rows(sp.N, 96, idx)
    _check(w, 2048, rows)


@pytest.mark.parametrize("idx,M", [(0, 320), (4, 576), (6, 1088)])
def test_config5_linears(idx, M):
    """Shapes of the mixed serving step: decode tokens plus a prefill chunk."""
    sp = wl.llama7b_layer("c5/L0/")[idx]
    w = wl.make_weights(sp, 0)
    rows = sample_rows(sp.N, 96, idx)
    _check(w, M, rows)
    nw = wl.LinearWeights(with_spec(w, rank=0).spec, w.q, w.s, w.z, None, None, w.outliers)
    _check(nw, M, rows)


@pytest.mark.parametrize("M", [17, 100, 300])
@pytest.mark.parametrize("group_size,rank", [(128, 64), (0, 32), (128, 0)])
def test_split_over_k(M, group_size, rank):
    """Few row tiles: without a compensator the main kernel splits K (up to
    four splits) and the last split adds the others' fp32 partials in split
    order; with one it does not split. Both give the oracle's result."""
    sp = wl.LinearSpec(f"split/g{group_size}/r{rank}", 4096, 1024, group_size, rank)
    w = wl.make_weights(sp, 14)
    lin = spear.from_weights(w, max_tokens=512)
    y1 = _check(w, M, lin=lin)
    y2 = _check(w, M, lin=lin)  # counters and partials are reused by the next call
    if rank == 0:
        # the partials are added in split order: repeated calls agree bit for bit
        # (with a compensator, the pre-kernel's atomic split-K sum of z does not)
        np.testing.assert_array_equal(y1, y2)


def test_split_wait_times_out_and_recovers():
    """The K splits skip their "partial tile stored" arrival: the split that
    adds the partials waits out its 4 x 2 ms limit, writes nothing for its
    tile and latches TIMEOUT; check() reports it and resets the workspace, and
    the next call on the same handle is correct again. Nothing traps or hangs."""
    import torch

    from .helpers import dev_bf16
    sp = wl.LinearSpec("split/timeout", 4096, 1024, 128, 0)
    w = wl.make_weights(sp, 15)
    lin = spear.from_weights(w, max_tokens=512)
    M = 100
    x = dev_bf16(wl.make_x(sp.K, M, w.outliers, 0, sp.name))
    y = torch.empty((M, sp.N), dtype=torch.bfloat16, device="cuda")
    lin.debug_set(wait_ns=2_000_000, skip_arrive=True)
    lin.forward_prefill(x, y)
    assert lin.check() == spear.SPEAR_ERR_TIMEOUT
    lin.debug_set(0, False)
    _check(w, M, lin=lin)
    assert lin.check() == spear.SPEAR_OK
