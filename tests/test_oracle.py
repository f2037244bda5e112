"""Pins for the CPU oracle (no GPU).

The oracle is checked against things fixed by the method's definition and by
mathematics rather than against itself:

* hand-derived bf16 roundings of the dequantised value (golden fixture);
* the closed form s = 1, z = 8 -> w = code - 8 on codes packed by the test;
* the pure-Python brute force (independent unpack, library bf16 cast,
  explicitly materialised effective weight per token);
* the reductions the SPEAR paper names (section 2.1A and section 1): alpha = 0
  gives the dequantised matmul, gamma = 1 gives the static low-rank correction
  W + alpha B A, both evaluated with numpy's matmul on independently unpacked
  weights;
* the gate against torch's SiLU and closed-form sigmoid values;
* the bottleneck-MLP gate against sigma(0) = 1/2, hand-derived sparse cases
  and its reduction to the elementwise sigmoid gate for W1 = W2 = I, z >= 0;
* special inputs: A = 0, B = 0, q = z (compensator alone), x = e_k.
"""
import math
from pathlib import Path

import numpy as np
import pytest
import torch

from oracle import brute, ref
from quantized_linear_error_gb300 import workload as wl

GOLDEN = Path(__file__).parent / "golden" / "dequant_rounding.txt"


def _pack(codes: np.ndarray) -> np.ndarray:
    """Pack codes [N][K] into bytes, even k in the low nibble."""
    c = codes.astype(np.uint8)
    return (c[:, 0::2] | (c[:, 1::2] << 4)).astype(np.uint8)


def _tiny(seed, N, K, G, r, M, zeros=True):
    rng = np.random.default_rng(seed)
    codes = rng.integers(0, 16, size=(N, K))
    ng = K // G
    s = wl.to_bf16_bits(rng.uniform(0.005, 0.02, size=(N, ng)).astype(np.float32))
    z = rng.integers(0, 16, size=(N, ng), dtype=np.uint8) if zeros else None
    A = wl.to_bf16_bits(rng.normal(0, 0.02, size=(r, K)).astype(np.float32)) if r else None
    B = wl.to_bf16_bits(rng.normal(0, 0.02, size=(N, r)).astype(np.float32)) if r else None
    x = wl.to_bf16_bits(rng.normal(0, 1, size=(M, K)).astype(np.float32))
    return codes, _pack(codes), s, z, A, B, x


def _f(bits):
    return wl.bf16_bits_to_f32(bits).astype(np.float64)


def _silu(v):
    return torch.nn.functional.silu(torch.from_numpy(np.asarray(v, np.float64))).numpy()


def _wd_brute(q, s, z, N, K, G):
    return np.array([[brute.dequant_value(q, s, z, n, k, G) for k in range(K)] for n in range(N)])


def _rel(a, b):
    return np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-300)


# ------------------------------------------------------------------ dequant
def _golden_cases():
    cases = []
    for line in GOLDEN.read_text().splitlines():
        line = line.split(";")[0].strip()
        if not line or line.startswith("#"):
            continue
        sb, q, z, e = line.split()
        cases.append((int(sb, 16), int(q), int(z), int(e, 16)))
    return cases


@pytest.mark.parametrize("s_bits,q,z,expected", _golden_cases())
def test_golden_rounding(s_bits, q, z, expected):
    qa = np.array([[q | (0 << 4)]], np.uint8)          # k = 0 in the low nibble
    sa = np.array([[s_bits]], np.uint16)
    za = np.array([[z]], np.uint8)
    got = ref.dequant_bf16(qa, sa, za, 1, 2, 2)[0, 0]
    assert got == expected, f"oracle {got:#06x} != {expected:#06x}"
    got_b = brute.dequant_bf16(qa, sa, za, 1, 2, 2)[0, 0]
    assert got_b == expected, f"brute {got_b:#06x} != {expected:#06x}"


def test_closed_form_unit_scale_symmetric():
    rng = np.random.default_rng(1)
    N, K, G = 24, 256, 128
    codes = rng.integers(0, 16, size=(N, K))
    s = np.full((N, K // G), 0x3F80, np.uint16)         # 1.0
    got = ref.dequant_f64(_pack(codes), s, None, N, K, G)   # zeros absent -> z = 8
    np.testing.assert_array_equal(got, codes - 8.0)
    got_bf = ref.dequant_bf16(_pack(codes), s, None, N, K, G)
    np.testing.assert_array_equal(_f(got_bf), codes - 8.0)


@pytest.mark.parametrize("N,K,G,zeros", [(8, 256, 128, True), (16, 128, 128, False),
                                          (5, 64, 64, True), (32, 384, 128, True)])
def test_dequant_matches_brute(N, K, G, zeros):
    _, q, s, z, *_ = _tiny(N * K + G, N, K, G, 0, 1, zeros)
    np.testing.assert_array_equal(ref.dequant_bf16(q, s, z, N, K, G), brute.dequant_bf16(q, s, z, N, K, G))
    np.testing.assert_array_equal(ref.dequant_f64(q, s, z, N, K, G), _wd_brute(q, s, z, N, K, G))


def test_dequant_edge_values():
    """Codes and zeros at 0 and 15, smallest and largest scales of the workload
    and full 8-bit significands so that rounding happens."""
    N, K, G = 4, 256, 128
    codes = np.zeros((N, K), int)
    codes[0], codes[1] = 0, 15
    codes[2] = np.arange(K) % 16
    codes[3] = 15 - np.arange(K) % 16
    z = np.array([[15, 0], [0, 15], [0, 15], [15, 7]], np.uint8)
    s = np.array([[0x3BA4, 0x3CA4], [0x3BFF, 0x3C7F], [0x3F81, 0x3F83], [0x3CA3, 0x3BA5]], np.uint16)
    q = _pack(codes)
    np.testing.assert_array_equal(ref.dequant_bf16(q, s, z, N, K, G), brute.dequant_bf16(q, s, z, N, K, G))


# ------------------------------------------------------------------ gate
def test_gate_closed_forms():
    l3 = math.log(3.0)
    u = ref.gate(np.array([0.0, l3, -l3, 40.0]), 0)
    np.testing.assert_allclose(u, [0.0, 0.75 * l3, -0.25 * l3, 40.0], rtol=1e-15, atol=1e-300)
    np.testing.assert_array_equal(ref.gate(np.array([-2.5, 3.0]), 1), [-2.5, 3.0])


def test_gate_is_silu():
    z = np.linspace(-30, 30, 1001)
    np.testing.assert_allclose(ref.gate(z, 0), _silu(z), rtol=1e-14, atol=1e-300)


def _bits(a):
    return wl.to_bf16_bits(np.asarray(a, np.float32))


def test_mlp_gate_with_zero_output_layer_is_one_half():
    """W2 = 0: every gate logit is 0 and sigma(0) = 1/2 exactly, whatever W1."""
    rng = np.random.default_rng(11)
    z = rng.normal(0, 3, size=(5, 16))
    W1 = _bits(rng.normal(0, 1, size=(4, 16)))
    u = ref.gate_mlp(z, W1, np.zeros((16, 4), np.uint16))
    np.testing.assert_array_equal(u, z / 2)


def test_mlp_gate_sparse_hand_cases():
    """r = h = 2, W1 = [[0, 1], [0, 0]] (t0 = relu(z1)), W2 = [[1, 0], [0, 0]]:
    gamma = (sigma(relu(z1)), 1/2). z = (2, 3) gives u = (2 sigma(3), 3/2);
    z = (2, -3) cuts the hidden unit: u = (1, -3/2)."""
    W1 = _bits([[0, 1], [0, 0]])
    W2 = _bits([[1, 0], [0, 0]])
    sig3 = 1.0 / (1.0 + math.exp(-3.0))
    np.testing.assert_allclose(ref.gate_mlp(np.array([[2.0, 3.0]]), W1, W2), [[2 * sig3, 1.5]], rtol=1e-15)
    np.testing.assert_array_equal(ref.gate_mlp(np.array([[2.0, -3.0]]), W1, W2), [[1.0, -1.5]])


def test_mlp_gate_relu_and_shapes():
    """r = 2, h = 1, W1 = [[1, -1]], W2 = [[2], [-1]]: t = relu(z0 - z1).
    z = (1, 3): t = 0, u = z / 2; z = (3, 1): t = 2, u = (3 sigma(4), sigma(-2))."""
    W1 = _bits([[1, -1]])
    W2 = _bits([[2], [-1]])
    np.testing.assert_array_equal(ref.gate_mlp(np.array([[1.0, 3.0]]), W1, W2), [[0.5, 1.5]])
    s4, sm2 = 1 / (1 + math.exp(-4.0)), 1 / (1 + math.exp(2.0))
    np.testing.assert_allclose(ref.gate_mlp(np.array([[3.0, 1.0]]), W1, W2), [[3 * s4, sm2]], rtol=1e-15)


def test_mlp_gate_identity_reduces_to_sigmoid_gate():
    """W1 = W2 = I (h = r): gamma_j = sigma(relu(z_j)), which for z >= 0 is the
    elementwise sigmoid gate, i.e. u = SiLU(z) (compared with the separate
    elementwise path of the oracle and with torch)."""
    rng = np.random.default_rng(12)
    z = np.abs(rng.normal(0, 2, size=(3, 16)))
    eye = _bits(np.eye(16))
    u = ref.gate_mlp(z, eye, eye)
    np.testing.assert_allclose(u, ref.gate(z, 0), rtol=1e-15)
    np.testing.assert_allclose(u, _silu(z), rtol=1e-14)


def test_ec_projection_matches_numpy():
    _, q, s, z, A, B, x = _tiny(3, 16, 256, 128, 8, 3)
    zz, uu = ref.ec(A, x, 0)
    np.testing.assert_allclose(zz, _f(x) @ _f(A).T, rtol=1e-13)
    np.testing.assert_allclose(uu, _silu(_f(x) @ _f(A).T), rtol=1e-13)


# ------------------------------------------------------------------ forward
@pytest.mark.parametrize("gate", [0, 1])
@pytest.mark.parametrize("N,K,G,r,M", [(16, 64, 32, 8, 3), (8, 48, 48, 4, 2), (12, 32, 16, 0, 2)])
def test_forward_matches_materialised_effective_weight(N, K, G, r, M, gate):
    _, q, s, z, A, B, x = _tiny(N + K + r, N, K, G, r, M)
    alpha = 1.7
    yb = brute.forward(q, s, z, K, G, A, B, alpha, gate, x)
    yc = ref.forward(q, s, z, K, G, A, B, alpha, gate, x)
    assert _rel(yc, yb) <= 1e-12


@pytest.mark.parametrize("N,K,G,r,h,M", [(16, 64, 32, 8, 3, 3), (8, 48, 48, 4, 5, 2)])
def test_forward_mlp_gate_matches_materialised_effective_weight(N, K, G, r, h, M):
    _, q, s, z, A, B, x = _tiny(N + K + r + h, N, K, G, r, M)
    rng = np.random.default_rng(N * h)
    # A x is small (std 0.02 sqrt(K)); scale the gate weights so the gate varies
    W1 = _bits(rng.normal(0, 4, size=(h, r)))
    W2 = _bits(rng.normal(0, 4, size=(r, h)))
    alpha = 1.3
    yb = brute.forward(q, s, z, K, G, A, B, alpha, 2, x, W1, W2)
    yc = ref.forward(q, s, z, K, G, A, B, alpha, 2, x, W1=W1, W2=W2)
    assert _rel(yc, yb) <= 1e-12


def test_alpha_zero_is_dequantised_matmul():
    N, K, G = 40, 256, 128
    _, q, s, z, A, B, x = _tiny(5, N, K, G, 16, 4)
    y = ref.forward(q, s, z, K, G, A, B, 0.0, 0, x)
    expect = _f(x) @ _wd_brute(q, s, z, N, K, G).T
    assert _rel(y, expect) <= 1e-12


def test_gate_one_is_static_low_rank_correction():
    N, K, G, alpha = 40, 256, 128, 3.0
    _, q, s, z, A, B, x = _tiny(6, N, K, G, 16, 4)
    y = ref.forward(q, s, z, K, G, A, B, alpha, 1, x)
    weff = _wd_brute(q, s, z, N, K, G) + alpha * _f(B) @ _f(A)
    assert _rel(y, _f(x) @ weff.T) <= 1e-12


def test_zero_projections_drop_compensator():
    N, K, G = 24, 128, 64
    _, q, s, z, A, B, x = _tiny(7, N, K, G, 8, 3)
    plain = _f(x) @ _wd_brute(q, s, z, N, K, G).T
    zA = np.zeros_like(A)
    zB = np.zeros_like(B)
    assert _rel(ref.forward(q, s, z, K, G, zA, B, 2.0, 0, x), plain) <= 1e-12
    assert _rel(ref.forward(q, s, z, K, G, A, zB, 2.0, 0, x), plain) <= 1e-12
    assert _rel(ref.forward(q, s, z, K, G, None, None, 2.0, 0, x), plain) <= 1e-12


def test_codes_equal_zeros_leave_compensator_alone():
    N, K, G, alpha = 24, 256, 128, 1.5
    rng = np.random.default_rng(8)
    zp = rng.integers(0, 16, size=(N, K // G), dtype=np.uint8)
    codes = np.repeat(zp, G, axis=1)                     # q == z everywhere
    _, _, s, _, A, B, x = _tiny(8, N, K, G, 8, 3)
    y = ref.forward(_pack(codes), s, zp, K, G, A, B, alpha, 0, x)
    expect = alpha * _silu(_f(x) @ _f(A).T) @ _f(B).T
    assert _rel(y, expect) <= 1e-12


def test_unit_vector_input_picks_a_column():
    N, K, G, alpha, k = 24, 128, 64, 2.0, 77
    _, q, s, z, A, B, _ = _tiny(9, N, K, G, 8, 1)
    x = np.zeros((1, K), np.uint16)
    x[0, k] = 0x3F80
    y = ref.forward(q, s, z, K, G, A, B, alpha, 0, x)[0]
    expect = _wd_brute(q, s, z, N, K, G)[:, k] + alpha * _f(B) @ _silu(_f(A)[:, k])
    assert _rel(y, expect) <= 1e-12


def test_row_subset_matches_full():
    w = wl.make_weights(wl.LinearSpec("t/rows", 512, 96, 128, 16), 3)
    x = wl.make_x(512, 5, w.outliers, 3, "t/rows")
    full = ref.forward_w(w, x)
    rows = np.array([0, 7, 95, 31, 31, 60])
    np.testing.assert_array_equal(ref.forward_w(w, x, rows), full[:, rows])


# ------------------------------------------------------------------ generator
def test_workload_generator_properties():
    sp = wl.LinearSpec("t/gen", 2048, 256, 128, 32)
    w = wl.make_weights(sp, 0)
    assert w.q.shape == (256, 1024) and w.s.shape == (256, 16) and w.z.shape == (256, 16)
    assert w.A.shape == (32, 2048) and w.B.shape == (256, 32)
    lo, hi = w.q & 0xF, w.q >> 4
    for part in (lo, hi):
        counts = np.bincount(part.ravel(), minlength=16)
        assert counts.min() > 0.9 * part.size / 16
    sf = _f(w.s)
    assert sf.min() >= 0.0049 and sf.max() <= 0.0201
    assert w.z.max() == 15 and w.z.min() == 0
    assert len(w.outliers) == 20 and len(set(w.outliers.tolist())) == 20
    x = wl.make_x(2048, 4, w.outliers, 0, "t/gen")
    xf = _f(x)
    assert np.abs(xf[:, w.outliers]).mean() > 10 * np.abs(np.delete(xf, w.outliers, axis=1)).mean()
    # determinism: same seed, same bytes
    w2 = wl.make_weights(sp, 0)
    assert np.array_equal(w.q, w2.q) and np.array_equal(w.A, w2.A)


def test_mlp_gate_generator():
    sp = wl.LinearSpec("t/mlp", 1024, 64, 128, 32, gate=wl.GATE_MLP, gate_hidden=8)
    w = wl.make_weights(sp, 0)
    assert w.W1.shape == (8, 32) and w.W2.shape == (32, 8)
    assert wl.make_weights(wl.LinearSpec("t/mlp", 1024, 64, 128, 32), 0).W1 is None
    assert sp.algorithmic_bytes(1) == wl.LinearSpec("t/mlp", 1024, 64, 128, 32).algorithmic_bytes(1) + 2 * 32 * 8 * 2


def test_config_shapes():
    assert [(l.K, l.N) for l in wl.config_linears(2)] == [
        (4096, 4096)] * 4 + [(4096, 11008)] * 2 + [(11008, 4096)]
    c5 = wl.config_linears(5)
    assert len(c5) == 224 and sum(l.rank > 0 for l in c5) == 28
    assert len(wl.ec_layer_indices(0)) == 4
    assert all(l.group_size == 0 and l.rank == 256 for l in wl.config_linears(4))


# ------------------------------------------------------------------ planted mistakes
PLANTS = {1: "nibble order swapped", 2: "zero point added, not subtracted", 3: "gate drops the z factor",
          4: "B indexed transposed", 5: "alpha ignored", 6: "rounding ties away from zero",
          7: "group index ignores the group size", 8: "sigmoid sign flipped", 9: "x reversed in A x",
          10: "MLP gate without the relu", 11: "MLP gate reads W1 transposed", 12: "MLP gate without the sigmoid"}

_PIN_TESTS = [
    lambda: [test_golden_rounding(*c) for c in _golden_cases()],
    test_closed_form_unit_scale_symmetric,
    lambda: [test_dequant_matches_brute(*a) for a in [(8, 256, 128, True), (5, 64, 64, True)]],
    test_dequant_edge_values,
    test_gate_closed_forms,
    test_gate_is_silu,
    test_ec_projection_matches_numpy,
    lambda: [test_forward_matches_materialised_effective_weight(16, 64, 32, 8, 3, g) for g in (0, 1)],
    test_alpha_zero_is_dequantised_matmul,
    test_gate_one_is_static_low_rank_correction,
    test_zero_projections_drop_compensator,
    test_codes_equal_zeros_leave_compensator_alone,
    test_unit_vector_input_picks_a_column,
    test_mlp_gate_with_zero_output_layer_is_one_half,
    test_mlp_gate_sparse_hand_cases,
    test_mlp_gate_relu_and_shapes,
    test_mlp_gate_identity_reduces_to_sigmoid_gate,
]


@pytest.mark.parametrize("plant", sorted(PLANTS))
def test_pins_reject_planted_mistake(plant):
    """Each planted oracle variant must fail at least one pin above."""
    failed = 0
    with ref.planted(plant):
        for t in _PIN_TESTS:
            try:
                t()
            except AssertionError:
                failed += 1
    assert failed > 0, f"no pin caught plant {plant}: {PLANTS[plant]}"
