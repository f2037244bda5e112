"""Grouped handles (spear_linear_create_grouped): several linears that read
the same x (fused q/k/v, or gate/up) as one handle. Each member's slice of y
is checked against the fp64 oracle of that member alone, on both paths
(decode and prefill), with the layer's tolerance max |y - y_ref| / max |y_ref|
<= 1e-2 per member."""
import dataclasses

import numpy as np
import pytest
import torch

from oracle import ref
from quantized_linear_error_gb300 import spear
from quantized_linear_error_gb300 import workload as wl

from .helpers import codes_equal_zeros, dev_bf16, host_f64, rel_err

pytestmark = pytest.mark.gpu
TOL = 1e-2


def _members(seed, K=1024, Ns=(512, 256, 768), group=128, rank=32, alphas=(1.0, 0.5, 2.0), gate=wl.GATE_SIGMOID,
             null_zeros=(1,)):
    out = []
    for i, (N, a) in enumerate(zip(Ns, alphas)):
        w = wl.make_weights(wl.LinearSpec(f"grp/{seed}/{i}", K, N, group, rank, alpha=a, gate=gate), seed)
        if i in null_zeros:
            w = wl.LinearWeights(w.spec, w.q, w.s, None, w.A, w.B, w.outliers)
        out.append(w)
    return out


def _check(ws, lin, M, path, seed=0, tol=TOL):
    K = ws[0].spec.K
    xb = wl.make_x(K, M, ws[0].outliers, seed, "grp/x")
    y = torch.full((M, lin.N), float("nan"), dtype=torch.bfloat16, device="cuda")
    getattr(lin, f"forward_{path}")(dev_bf16(xb), y)
    assert lin.check() == spear.SPEAR_OK
    yh = host_f64(y)
    c0 = 0
    for i, w in enumerate(ws):
        yr = ref.forward_w(w, xb)
        e = rel_err(yh[:, c0:c0 + w.spec.N], yr)
        assert e <= tol, f"{path} M={M} member {i}: rel err {e:.3e}"
        c0 += w.spec.N
    assert c0 == lin.N


@pytest.mark.parametrize("M", [1, 5, 8, 16, 32])
def test_decode_three_members(M):
    ws = _members(40)
    lin = spear.grouped_from_weights(ws, max_tokens=32)
    _check(ws, lin, M, "decode", seed=M)


@pytest.mark.parametrize("M", [33, 300])
def test_prefill_three_members(M):
    ws = _members(41)
    lin = spear.grouped_from_weights(ws, max_tokens=300)
    _check(ws, lin, M, "prefill", seed=M)


@pytest.mark.parametrize("path,M", [("decode", 8), ("decode", 32), ("prefill", 200)])
def test_compensator_dominant_members(path, M):
    """Codes equal to zeros in every member: y is each member's compensator
    alone, so a member that used another member's u columns, B rows or alpha
    would fail."""
    ws = [codes_equal_zeros(w) if w.z is not None else w for w in _members(42, null_zeros=())]
    lin = spear.grouped_from_weights(ws, max_tokens=max(M, 32))
    _check(ws, lin, M, path, seed=M)


@pytest.mark.parametrize("path,M", [("decode", 4), ("prefill", 130)])
def test_per_channel_gate_one(path, M):
    ws = _members(43, K=640, Ns=(16, 528), group=0, rank=16, alphas=(1.0, 3.0), gate=wl.GATE_ONE, null_zeros=())
    lin = spear.grouped_from_weights(ws, max_tokens=max(M, 32))
    _check(ws, lin, M, path, seed=M)


def test_members_without_compensator():
    ws = _members(44, rank=0)
    lin = spear.grouped_from_weights(ws, max_tokens=300)
    for path, M in (("decode", 7), ("prefill", 257)):
        _check(ws, lin, M, path, seed=M)


@pytest.mark.parametrize("idx", [(0, 1, 2), (4, 5)])
def test_llama7b_fused_projections(idx):
    """The fused q/k/v (rank 3 x 64 = 192) and gate/up (2 x 64) projections of
    the decode layer set, sampled rows at M = 1, 8, 32 and the prefill path at
    M = 320."""
    specs = wl.config_linears(2)
    ws = [wl.make_weights(specs[i], 0) for i in idx]
    lin = spear.grouped_from_weights(ws, max_tokens=320)
    for path, M in (("decode", 1), ("decode", 8), ("decode", 32), ("prefill", 320)):
        _check(ws, lin, M, path, seed=M)


def test_grouped_matches_separate_handles_on_decode():
    """The grouped decode call and the members' own handles compute the same
    layer; they agree far inside the tolerance (only summation order and the
    atomics of z differ)."""
    ws = _members(45)
    lin = spear.grouped_from_weights(ws, max_tokens=32)
    xb = wl.make_x(ws[0].spec.K, 8, ws[0].outliers, 0, "grp/sep")
    x = dev_bf16(xb)
    y = torch.empty((8, lin.N), dtype=torch.bfloat16, device="cuda")
    lin.forward_decode(x, y)
    c0 = 0
    for w in ws:
        single = spear.from_weights(w, max_tokens=32)
        ys = torch.empty((8, w.spec.N), dtype=torch.bfloat16, device="cuda")
        single.forward_decode(x, ys)
        assert rel_err(host_f64(y[:, c0:c0 + w.spec.N]), host_f64(ys)) <= 2e-3
        c0 += w.spec.N
