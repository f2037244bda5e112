"""Parity of the fused decode kernel (M <= 32) against the fp64 oracle.

Tolerance: max |y_gpu - y_ref| / max |y_ref| <= 1e-2 per linear call, with
y_ref the unrounded fp64 result. Because the compensator term is only a few
percent of |y| on the workload distributions, the same bound is also applied
to runs where it dominates (codes equal to zeros, so W_q = 0; and alpha = 30),
which pins the projection, gate and up-projection on their own.
"""
import numpy as np
import pytest
import torch

from oracle import ref
from quantized_linear_error_gb300 import spear
from quantized_linear_error_gb300 import workload as wl

from .helpers import codes_equal_zeros, dev_bf16, host_f64, rel_err, run, sample_rows, with_spec

pytestmark = pytest.mark.gpu
TOL = 1e-2


def _check(w, M, rows=None, path="decode", tol=TOL, seed=0, lin=None):
    sp = w.spec
    x = wl.make_x(sp.K, M, w.outliers, seed, sp.name)
    lin = lin or spear.from_weights(w, max_tokens=max(M, 1))
    y = run(lin, x, path)
    yr = ref.forward_w(w, x, rows)
    yg = y if rows is None else y[:, rows]
    e = rel_err(yg, yr)
    assert e <= tol, f"{sp.name} M={M}: rel err {e:.3e}"
    return y, e


# ---------------------------------------------------------------- small shapes, full compare
SMALL = [
    wl.LinearSpec("s/g128", 256, 200, 128, 16),
    wl.LinearSpec("s/pc", 384, 328, 0, 32),
    wl.LinearSpec("s/noec", 512, 136, 128, 0),
    wl.LinearSpec("s/wide", 1024, 4104, 128, 64),
    wl.LinearSpec("s/pc_ec256", 640, 520, 0, 256),
]


@pytest.mark.parametrize("M", [1, 3, 8, 13, 16, 29, 32])
@pytest.mark.parametrize("sp", SMALL, ids=lambda s: s.name)
def test_small_shapes(sp, M):
    _check(wl.make_weights(sp, 1), M)


@pytest.mark.parametrize("sp", SMALL[:2] + SMALL[4:], ids=lambda s: s.name)
def test_compensator_dominant(sp):
    w = wl.make_weights(sp, 2)
    _check(codes_equal_zeros(w), 8)
    _check(with_spec(w, alpha=30.0), 5)


def test_gate_one_and_alpha_zero():
    w = wl.make_weights(SMALL[0], 3)
    _check(with_spec(w, gate=wl.GATE_ONE), 4)
    _check(with_spec(codes_equal_zeros(w), gate=wl.GATE_ONE), 4)
    # alpha = 0 adds an exact zero: identical to the handle without a compensator
    x = wl.make_x(w.spec.K, 6, w.outliers, 0, "a0")
    y0 = run(spear.from_weights(with_spec(w, alpha=0.0)), x, "decode")
    nw = wl.LinearWeights(with_spec(w, rank=0).spec, w.q, w.s, w.z, None, None, w.outliers)
    y1 = run(spear.from_weights(nw), x, "decode")
    np.testing.assert_array_equal(y0, y1)


def test_repeated_calls_reuse_workspace():
    """The fused kernel clears its z accumulators and counters itself, so a
    sequence of calls on one handle stays correct. z is summed with atomics in
    arbitrary order, so repeated calls may differ in the last bit of z and,
    rarely, by one bf16 ulp in y."""
    w = wl.make_weights(SMALL[3], 4)
    lin = spear.from_weights(w, max_tokens=32)
    ys = [_check(w, M, lin=lin)[0] for M in (7, 7, 32, 1, 7)]
    for a, b in ((ys[0], ys[1]), (ys[0], ys[4])):
        assert np.max(np.abs(a - b) / np.maximum(np.abs(a), 1e-3)) <= 2.0 ** -7


def test_unit_vector_input():
    sp = SMALL[1]
    w = wl.make_weights(sp, 5)
    x = np.zeros((2, sp.K), np.uint16)
    x[0, 17] = 0x3F80
    x[1, sp.K - 1] = 0xBF80
    lin = spear.from_weights(w)
    y = run(lin, x, "decode")
    assert rel_err(y, ref.forward_w(w, x)) <= TOL


# ---------------------------------------------------------------- workload sizes (sampled rows)
@pytest.mark.parametrize("M", [4])
def test_config1_full(M):
    _check(wl.make_weights(wl.config_linears(1)[0], 0), M)


@pytest.mark.parametrize("idx", range(7))
def test_config2_layer_set(idx):
    sp = wl.config_linears(2)[idx]
    w = wl.make_weights(sp, 0)
    lin = spear.from_weights(w, max_tokens=32)
    rows = sample_rows(sp.N, 384, idx)
    for M in (1, 8, 32):
        _check(w, M, rows, lin=lin)
    _check(codes_equal_zeros(w), 32, rows)


@pytest.mark.parametrize("idx", range(2))
def test_config4_per_channel(idx):
    sp = wl.config_linears(4)[idx]
    w = wl.make_weights(sp, 0)
    rows = sample_rows(sp.N, 256, idx)
    _check(w, 16, rows)
    _check(codes_equal_zeros(w), 16, rows)
    _check(with_spec(w, alpha=30.0), 16, rows)


@pytest.mark.parametrize("cfg,idx,M", [(2, 3, 16), (2, 6, 16), (4, 0, 32), (4, 1, 32)])
def test_stage_plans_late_b_and_half_stages(cfg, idx, M):
    """The plans that keep at least two stages: the o and down projections at
    16 tokens and config 4's down projection at 32 take one 128-channel unit
    per K warp and stage; config 4's up projection at 32 copies its B
    fragments (rank 256) into the stage area after the W loop. The plan is
    asserted through the host query, then the result against the oracle
    (compensator as is, and dominant)."""
    sp = wl.config_linears(cfg)[idx]
    w = wl.make_weights(sp, 5)
    n_sm = torch.cuda.get_device_properties(0).multi_processor_count
    d = spear.decode_schedule(sp.N, sp.K, M, n_sm, rank_b=sp.rank, group_size=sp.group_size)
    assert d["NS"] >= 2 and d["n_stages"] > 1
    rows = sample_rows(sp.N, 192, idx)
    lin = spear.from_weights(w, max_tokens=32)
    _check(w, M, rows, lin=lin)
    _check(codes_equal_zeros(w), M, rows)


# ---------------------------------------------------------------- boundary and bounded waits
def test_decode_rejects_too_many_tokens():
    w = wl.make_weights(SMALL[0], 6)
    lin = spear.from_weights(w, max_tokens=64)
    x = torch.zeros((33, w.spec.K), dtype=torch.bfloat16, device="cuda")
    y = torch.empty((33, w.spec.N), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(spear.SpearError) as ei:
        lin.forward_decode(x, y)
    assert ei.value.status == spear.SPEAR_ERR_INVALID_ARG
    lin.forward_decode(x[:0], y[:0])  # M = 0 is a no-op


def test_bounded_wait_times_out_and_recovers():
    """CTAs skip their arrival: every CTA's wait runs out after 2 ms, the kernel
    leaves the compensator out, check() reports TIMEOUT and resets the handle."""
    w = wl.make_weights(SMALL[3], 7)
    lin = spear.from_weights(w, max_tokens=8)
    x = dev_bf16(wl.make_x(w.spec.K, 8, w.outliers, 0, "to"))
    y = torch.empty((8, w.spec.N), dtype=torch.bfloat16, device="cuda")
    lin.debug_set(wait_ns=2_000_000, skip_arrive=True)
    lin.forward_decode(x, y)
    assert lin.check() == spear.SPEAR_ERR_TIMEOUT
    nw = wl.LinearWeights(with_spec(w, rank=0).spec, w.q, w.s, w.z, None, None, w.outliers)
    y_plain = run(spear.from_weights(nw), wl.make_x(w.spec.K, 8, w.outliers, 0, "to"), "decode")
    np.testing.assert_array_equal(host_f64(y), y_plain)
    lin.debug_set(0, False)
    _check(w, 8, lin=lin, seed=0)
