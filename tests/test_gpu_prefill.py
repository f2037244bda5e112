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


@pytest.mark.parametrize("variant", ["plain", "ec_only", "gate_one", "alpha30"])
@pytest.mark.parametrize("K,N,M", [(4096, 4096, 1088), (4096, 11008, 640)])
def test_compensator_prologue_in_the_main_kernel(K, N, M, variant):
    """Shapes where the projection runs as the persistent kernel's prologue
    (one 128-token item over all of K, gated in tensor memory, u' written
    by one bulk copy; the owners' K-tail loads wait for the tile's flag),
    also with W_q = 0 so that the compensator is the whole result."""
    sp = wl.LinearSpec(f"pro/{K}x{N}", K, N, 128, 64)
    w = wl.make_weights(sp, 19)
    w = {"plain": w, "ec_only": codes_equal_zeros(w), "gate_one": with_spec(codes_equal_zeros(w), gate=wl.GATE_ONE),
         "alpha30": with_spec(w, alpha=30.0)}[variant]
    rows = sample_rows(N, 96, 3)
    lin = spear.from_weights(w, max_tokens=M)
    y1 = _check(w, M, rows, lin=lin)
    y2 = _check(w, M, rows, lin=lin)  # the "u' ready" flags are cleared for the next call
    # every sum is in a fixed order (the projection is not split over K): bit for bit
    np.testing.assert_array_equal(y1, y2)


@pytest.mark.parametrize("M", [17, 100, 300])
@pytest.mark.parametrize("group_size,rank", [(128, 64), (0, 32), (128, 0)])
def test_split_over_k(M, group_size, rank):
    """Few row tiles: the stream-K schedule splits every tile's K range over
    two to four CTAs, and each tile's owner adds the others' fp32 partials in
    CTA order (with a compensator the owner also runs the K-tail). Both give
    the oracle's result."""
    sp = wl.LinearSpec(f"split/g{group_size}/r{rank}", 4096, 1024, group_size, rank)
    w = wl.make_weights(sp, 14)
    lin = spear.from_weights(w, max_tokens=512)
    y1 = _check(w, M, lin=lin)
    y2 = _check(w, M, lin=lin)  # counters and partials are reused by the next call
    if rank == 0:
        # the partials are added in CTA order: repeated calls agree bit for bit
        # (with a compensator, the pre-kernel's atomic split-K sum of z does not)
        np.testing.assert_array_equal(y1, y2)


def test_split_wait_times_out_and_recovers():
    """The CTAs that run a tile's later K blocks skip their "partial tile
    stored" flag: the tile's owner waits out its 4 x 2 ms limit, writes
    nothing for its tile and latches TIMEOUT; check() reports it and resets the workspace, and
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


# ---------------------------------------------------------------- compensator on a concurrent stream
def _concurrent(w, M, lin=None, seed=0, graph=False):
    import torch

    from .helpers import dev_bf16, host_f64
    sp = w.spec
    lin = lin or spear.from_weights(w, max_tokens=M)
    lin.enable_concurrent_ec()
    xb = wl.make_x(sp.K, M, w.outliers, seed, sp.name)
    x = dev_bf16(xb)
    y = torch.full((M, sp.N), float("nan"), dtype=torch.bfloat16, device="cuda")
    s_main, s_ec = torch.cuda.Stream(), torch.cuda.Stream()
    if graph:
        lin.forward_prefill_concurrent(x, y, stream=s_main, ec_stream=s_ec)  # warm
        s_main.synchronize()
        y.fill_(float("nan"))
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s_main):
            lin.forward_prefill_concurrent(x, y, stream=s_main, ec_stream=s_ec)
        g.replay()
    else:
        lin.forward_prefill_concurrent(x, y, stream=s_main, ec_stream=s_ec)
    torch.cuda.synchronize()
    assert lin.check() == spear.SPEAR_OK
    return host_f64(y), ref.forward_w(w, xb)


@pytest.mark.parametrize("M", [33, 300])
@pytest.mark.parametrize("sp", [SMALL[0], SMALL[1], SMALL[3], SMALL[4]], ids=lambda s: s.name)
def test_concurrent_compensator_matches_oracle(sp, M):
    y, yr = _concurrent(wl.make_weights(sp, 16), M)
    assert rel_err(y, yr) <= TOL


@pytest.mark.parametrize("variant", ["ec_only", "alpha30", "gate_one"])
def test_concurrent_compensator_dominant(variant):
    w = wl.make_weights(SMALL[3], 17)
    w = {"ec_only": codes_equal_zeros(w), "alpha30": with_spec(w, alpha=30.0),
         "gate_one": with_spec(codes_equal_zeros(w), gate=wl.GATE_ONE)}[variant]
    y, yr = _concurrent(w, 130)
    assert rel_err(y, yr) <= TOL


def test_concurrent_compensator_in_a_graph_and_next_to_the_fused_path():
    """Captured into one CUDA graph (fork and join by events) and replayed;
    the result agrees with the fused path far inside the tolerance. The two
    forms split the projection z = A x over K differently, so a u' element
    (rounded to bf16 once) may differ by one bf16 ulp (2^-8 relative) between
    them, and y by a few 1e-3 of its largest value."""
    w = wl.make_weights(SMALL[3], 18)
    lin = spear.from_weights(w, max_tokens=300)
    y, yr = _concurrent(w, 300, lin=lin, graph=True)
    assert rel_err(y, yr) <= TOL
    yf = run(lin, wl.make_x(w.spec.K, 300, w.outliers, 0, w.spec.name), "prefill")
    assert rel_err(y, yf) <= 5e-3


def test_concurrent_compensator_grouped_and_plain_handles():
    from .test_gpu_grouped import _members
    ws = _members(46)
    lin = spear.grouped_from_weights(ws, max_tokens=200)
    lin.enable_concurrent_ec()
    import torch

    from .helpers import dev_bf16, host_f64
    xb = wl.make_x(ws[0].spec.K, 200, ws[0].outliers, 0, "conc/grp")
    y = torch.empty((200, lin.N), dtype=torch.bfloat16, device="cuda")
    lin.forward_prefill_concurrent(dev_bf16(xb), y, stream=torch.cuda.Stream(), ec_stream=torch.cuda.Stream())
    torch.cuda.synchronize()
    yh, c0 = host_f64(y), 0
    for w in ws:
        assert rel_err(yh[:, c0:c0 + w.spec.N], ref.forward_w(w, xb)) <= TOL
        c0 += w.spec.N
    # a handle without a compensator takes the plain path (nothing to enable)
    nw = wl.make_weights(SMALL[2], 19)
    yp, yr = _concurrent(nw, 100)
    assert rel_err(yp, yr) <= TOL


def test_concurrent_compensator_argument_errors():
    import torch
    w = wl.make_weights(SMALL[0], 20)
    lin = spear.from_weights(w, max_tokens=64)
    x = torch.zeros((40, w.spec.K), dtype=torch.bfloat16, device="cuda")
    y = torch.empty((40, w.spec.N), dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.Stream()
    with pytest.raises(spear.SpearError):  # not enabled
        lin.forward_prefill_concurrent(x, y, stream=s, ec_stream=torch.cuda.Stream())
    lin.enable_concurrent_ec()
    lin.enable_concurrent_ec()  # idempotent
    with pytest.raises(spear.SpearError):  # the same stream twice
        lin.forward_prefill_concurrent(x, y, stream=s, ec_stream=s)
