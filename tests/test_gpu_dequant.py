"""Bit-exact dequantisation on the GPU: both kernel-side layouts, unpacked by
the kernels' own code, must equal the oracle's bf16_RNE((q - z) * s) on every
element (workload weight formats, edge values, hand-derived roundings)."""
import numpy as np
import pytest
import torch

from oracle import ref
from quantized_linear_error_gb300 import spear
from quantized_linear_error_gb300 import workload as wl

from .helpers import bits_of, dev_bf16
from .test_oracle import _golden_cases, _pack

pytestmark = pytest.mark.gpu


def _gpu_dequant(q, s, z, K, N, group_size):
    lin = spear.SpearLinear(K, N, group_size, torch.from_numpy(q).cuda(), dev_bf16(s),
                            None if z is None else torch.from_numpy(z).cuda(), max_tokens=1)
    outs = []
    for path in (0, 1):
        o = torch.empty((N, K), dtype=torch.bfloat16, device="cuda")
        lin.dequantize(o, path)
        torch.cuda.synchronize()
        outs.append(bits_of(o))
    lin.close()
    return outs


@pytest.mark.parametrize("cfg,idx", [(1, 0), (2, 0), (2, 6), (3, 0), (4, 0), (4, 1)])
def test_workload_formats_bit_exact(cfg, idx):
    sp = wl.config_linears(cfg)[idx]
    w = wl.make_weights(wl.LinearSpec(sp.name, sp.K, sp.N, sp.group_size, 0), 0)
    expect = ref.dequant_bf16(w.q, w.s, w.z, sp.N, sp.K, sp.G)
    for path, got in enumerate(_gpu_dequant(w.q, w.s, w.z, sp.K, sp.N, sp.group_size)):
        bad = np.argwhere(got != expect)
        assert bad.size == 0, f"path {path}: {len(bad)} mismatches, first at {bad[0]}"


@pytest.mark.parametrize("K,N,group_size,zeros", [(256, 200, 128, True), (384, 136, 0, True),
                                                   (128, 8, 128, False), (512, 1000, 0, False)])
def test_ragged_shapes_bit_exact(K, N, group_size, zeros):
    rng = np.random.default_rng(K + N)
    G = K if group_size == 0 else group_size
    codes = rng.integers(0, 16, size=(N, K))
    s = wl.to_bf16_bits(rng.uniform(0.005, 0.02, size=(N, K // G)).astype(np.float32))
    z = rng.integers(0, 16, size=(N, K // G), dtype=np.uint8) if zeros else None
    q = _pack(codes)
    expect = ref.dequant_bf16(q, s, z, N, K, G)
    for got in _gpu_dequant(q, s, z, K, N, group_size):
        np.testing.assert_array_equal(got, expect)


def test_edge_values_and_golden_roundings():
    """Rows of codes/zeros at 0 and 15, extreme and full-significand scales,
    plus every hand-derived rounding of the golden fixture."""
    K, G = 128, 128
    cases = _golden_cases()
    rows = []
    for sb, qv, zv, _ in cases:
        rows.append((np.full(K, qv), sb, zv))
    for qv in (0, 15):
        for zv in (0, 15):
            for sb in (0x3BA4, 0x3CA4, 0x3BFF, 0x3C7F, 0x3F81, 0x7F7F, 0x0080):
                rows.append((np.full(K, qv), sb, zv))
    rows.append((np.arange(K) % 16, 0x3CA3, 7))
    N = (len(rows) + 7) // 8 * 8
    while len(rows) < N:
        rows.append((np.zeros(K, int), 0x3F80, 0))
    codes = np.stack([r[0] for r in rows])
    s = np.array([[r[1]] for r in rows], np.uint16)
    z = np.array([[r[2]] for r in rows], np.uint8)
    q = _pack(codes)
    expect = ref.dequant_bf16(q, s, z, N, K, G)
    for i, (sb, qv, zv, e) in enumerate(cases):
        assert expect[i, 0] == e
    for got in _gpu_dequant(q, s, z, K, N, 128):
        np.testing.assert_array_equal(got, expect)
