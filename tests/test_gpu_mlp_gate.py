"""Parity of the bottleneck-MLP gate (gamma(z) = sigmoid(W2 relu(W1 z)),
SPEAR section 2.1A) on both paths against the fp64 oracle, with the same
bound as the other gates: max |y_gpu - y_ref| / max |y_ref| <= 1e-2. The
compensator-dominant runs (codes equal to zeros, so W_q = 0) make the gate's
output the whole result."""
import numpy as np
import pytest

from oracle import ref
from quantized_linear_error_gb300 import spear
from quantized_linear_error_gb300 import workload as wl

from .helpers import codes_equal_zeros, rel_err, run, sample_rows, with_spec

pytestmark = pytest.mark.gpu
TOL = 1e-2
MLP = wl.GATE_MLP

SPECS = [
    wl.LinearSpec("m/g128", 256, 200, 128, 16, gate=MLP, gate_hidden=8),
    wl.LinearSpec("m/pc", 384, 328, 0, 32, gate=MLP, gate_hidden=16),
    wl.LinearSpec("m/r256h64", 640, 520, 0, 256, gate=MLP, gate_hidden=64),
    wl.LinearSpec("m/h1", 512, 136, 128, 16, gate=MLP, gate_hidden=1),
]


def _check(w, M, path, rows=None, seed=0):
    x = wl.make_x(w.spec.K, M, w.outliers, seed, w.spec.name)
    y = run(spear.from_weights(w, max_tokens=max(M, 1)), x, path)
    yr = ref.forward_w(w, x, rows)
    e = rel_err(y if rows is None else y[:, rows], yr)
    assert e <= TOL, f"{w.spec.name} {path} M={M}: rel err {e:.3e}"
    return y


@pytest.mark.parametrize("M", [1, 5, 8, 16, 32])
@pytest.mark.parametrize("sp", SPECS, ids=lambda s: s.name)
def test_decode(sp, M):
    _check(wl.make_weights(sp, 1), M, "decode")


@pytest.mark.parametrize("M", [1, 33, 300])
@pytest.mark.parametrize("sp", SPECS, ids=lambda s: s.name)
def test_prefill(sp, M):
    _check(wl.make_weights(sp, 1), M, "prefill")


@pytest.mark.parametrize("path,M", [("decode", 8), ("decode", 32), ("prefill", 300)])
@pytest.mark.parametrize("sp", SPECS[:3], ids=lambda s: s.name)
def test_compensator_dominant(sp, path, M):
    w = codes_equal_zeros(wl.make_weights(sp, 2))
    y = _check(w, M, path)
    # the MLP gate is really applied: the elementwise sigmoid gate gives another result
    ys = run(spear.from_weights(with_spec(w, gate=wl.GATE_SIGMOID), max_tokens=M), 
             wl.make_x(sp.K, M, w.outliers, 0, sp.name), path)
    assert rel_err(ys, y) > 5e-2


@pytest.mark.parametrize("M", [1, 8, 32])
def test_llama7b_q_projection_sampled_rows(M):
    sp = wl.LinearSpec("m/c2q", 4096, 4096, 128, 64, gate=MLP, gate_hidden=16)
    _check(wl.make_weights(sp, 0), M, "decode", rows=sample_rows(sp.N, 96))


def test_prefill_llama7b_q_projection_sampled_rows():
    sp = wl.LinearSpec("m/c2q", 4096, 4096, 128, 64, gate=MLP, gate_hidden=16)
    _check(wl.make_weights(sp, 0), 320, "prefill", rows=sample_rows(sp.N, 96))


@pytest.mark.parametrize("dominant", [False, True])
def test_prefill_gate_in_the_main_kernel_prologue(dominant):
    """4096 -> 11008 at 640 tokens: the projection runs as the main kernel's
    prologue, and the MLP gate is evaluated there on z staged in shared
    memory (W_q = 0 in the dominant case, so the gate decides the result)."""
    sp = wl.LinearSpec("m/c5gate", 4096, 11008, 128, 64, gate=MLP, gate_hidden=16)
    w = wl.make_weights(sp, 3)
    if dominant:
        w = codes_equal_zeros(w)
    _check(w, 640, "prefill", rows=sample_rows(sp.N, 96, 1))
