"""Pins for the RTN quantiser and static SVD initialisation oracle (no GPU)."""
import numpy as np
import pytest

from oracle import rtn


def test_exact_grid_round_trips():
    """Values already on a 4-bit grid with a bf16-exact step come back exactly:
    w = (c - 8) * 0.5 with every code c in 0..15 present gives lo = -4,
    hi = 3.5, s = 0.5, z = 8 and q = c."""
    rng = np.random.default_rng(0)
    codes = np.stack([rng.permutation(np.tile(np.arange(16), 8)) for _ in range(6)])  # [6][128]
    w = ((codes.astype(np.float32) - 8) * 0.5).astype(np.float32)
    q, s, z = rtn.rtn_quantize(w, 128)
    np.testing.assert_array_equal(q, codes)
    assert np.all(rtn.bf16_bits_to_f32(s) == 0.5) and np.all(z == 8)


def test_all_zero_group_and_positive_group():
    """A group of zeros gets range 1e-8, z = 0 and codes 0 (so w_q = 0). A group
    of values in [0.25, 1.5] still has lo = 0 (the range includes zero), so
    s = bf16(1.5 / 15) = bf16(0.1) = 0x3DCD = 0.10009765625 (by hand: 0.1 =
    1.6 * 2^-4, mantissa 0.6 * 128 = 76.8 -> 77), z = 0, and the first and last
    codes are rint(0.25 / s) = rint(2.4976) = 2 and rint(1.5 / s) = 15."""
    w = np.zeros((2, 128), np.float32)
    w[1] = np.linspace(0.25, 1.5, 128, dtype=np.float32)
    q, s, z = rtn.rtn_quantize(w, 128)
    assert np.all(q[0] == 0) and z[0, 0] == 0
    assert s[1, 0] == 0x3DCD and z[1, 0] == 0
    assert q[1, 0] == 2 and q[1, -1] == 15


def test_error_is_at_most_half_a_step():
    """Unclipped codes are within s/2 of w (round to nearest); the range always
    contains 0 and both extremes, so no code is clipped by more than rounding."""
    rng = np.random.default_rng(1)
    for G in (128, 0):
        w = rng.normal(0, 0.02, size=(16, 512)).astype(np.float32)
        q, s, z = rtn.rtn_quantize(w, G)
        wq = rtn.dequant(q, s, z, G)
        Gs = 512 if G == 0 else G
        step = np.repeat(rtn.bf16_bits_to_f32(s).astype(np.float64), Gs, axis=1)
        # the bf16 rounding of s can stretch the grid by 2^-8 relative over 15 steps
        assert np.all(np.abs(wq - w) <= step * (0.5 + 15 * 2.0 ** -8) + 1e-12)


def test_bf16_rounding_ties_to_even():
    v = np.array([1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, 1.0 + 2.0 ** -9], np.float32)
    # 1 + 2^-8 is halfway between 1 and 1 + 2^-7: even is 1.0 (0x3F80)
    np.testing.assert_array_equal(rtn.bf16_rne_bits(v), [0x3F80, 0x3F82, 0x3F80])


def test_svd_init_recovers_an_exactly_low_rank_error():
    rng = np.random.default_rng(2)
    E = rng.normal(size=(40, 6)) @ rng.normal(size=(6, 96))
    A, B = rtn.svd_init(E, 6)
    assert A.shape == (6, 96) and B.shape == (40, 6)
    np.testing.assert_allclose(B @ A, E, rtol=0, atol=1e-10 * np.abs(E).max())


def test_svd_init_is_best_rank_r():
    """Eckart-Young: the residual of the rank-r truncation is the tail of the
    singular values, and no other rank-r product does better."""
    rng = np.random.default_rng(3)
    E = rng.normal(size=(30, 50))
    A, B = rtn.svd_init(E, 5)
    sv = np.linalg.svd(E, compute_uv=False)
    assert np.isclose(np.linalg.norm(E - B @ A), np.sqrt((sv[5:] ** 2).sum()))
    A2, B2 = rng.normal(size=(5, 50)), rng.normal(size=(30, 5))
    assert np.linalg.norm(E - B2 @ A2) > np.linalg.norm(E - B @ A)


@pytest.mark.parametrize("bad", ["no_zero_in_range", "z_sign"])
def test_pins_reject_planted_rtn_mistakes(bad, monkeypatch):
    """A quantiser that forgets to include 0 in the range or flips the zero
    point's sign must fail the round-trip pin."""
    orig = rtn.rtn_quantize

    def planted(w, group_size):
        with np.errstate(all="ignore"):
            return _planted(w, group_size)

    def _planted(w, group_size):
        q, s, z = orig(w, group_size)
        if bad == "z_sign":
            sf = rtn.bf16_bits_to_f32(s)
            G = w.shape[1] if group_size == 0 else group_size
            wg = w.reshape(w.shape[0], -1, G)
            z = np.clip(np.rint(np.minimum(wg.min(axis=2), 0) / sf), 0, 15).astype(np.uint8)
            q = np.clip(np.rint(wg / sf[:, :, None]) + z[:, :, None], 0, 15).reshape(w.shape).astype(np.uint8)
        else:
            G = w.shape[1] if group_size == 0 else group_size
            wg = w.reshape(w.shape[0], -1, G)
            lo, hi = wg.min(axis=2), wg.max(axis=2)
            s = rtn.bf16_rne_bits(((hi - lo) / np.float32(15)).astype(np.float32))
            sf = rtn.bf16_bits_to_f32(s)
            z = np.clip(np.rint(-lo / sf), 0, 15).astype(np.uint8)
            q = np.clip(np.rint(wg / sf[:, :, None]) + z[:, :, None], 0, 15).reshape(w.shape).astype(np.uint8)
        return q, s, z

    monkeypatch.setattr(rtn, "rtn_quantize", planted)
    failed = 0
    for t in (test_exact_grid_round_trips, test_all_zero_group_and_positive_group):
        try:
            t()
        except (AssertionError, FloatingPointError):
            failed += 1
    assert failed > 0


# ------------------------------------------------------------------ pack_codes
def test_pack_codes_hand_packed():
    """The user layout (even k in the low nibble of byte k / 2) by hand: codes
    [1, 2] are the byte 0x21; a row 0..15 is 0x10, 0x32, ..., 0xFE; 15 and 0
    give 0x0F (the high nibble is the odd channel)."""
    np.testing.assert_array_equal(rtn.pack_codes(np.array([[1, 2]])), [[0x21]])
    np.testing.assert_array_equal(rtn.pack_codes(np.arange(16)[None, :]),
                                  [[0x10, 0x32, 0x54, 0x76, 0x98, 0xBA, 0xDC, 0xFE]])
    np.testing.assert_array_equal(rtn.pack_codes(np.array([[15, 0], [0, 15]])), [[0x0F], [0xF0]])


def test_pack_codes_round_trip_by_bit_ops():
    """Unpacking each byte with its own shift and mask (written here, not
    taken from the oracle) gives back every code of a random matrix."""
    rng = np.random.default_rng(9)
    codes = rng.integers(0, 16, size=(7, 96))
    b = rtn.pack_codes(codes)
    assert b.dtype == np.uint8 and b.shape == (7, 48)
    back = np.empty_like(codes)
    for n in range(7):
        for j in range(48):
            back[n, 2 * j] = int(b[n, j]) & 0xF
            back[n, 2 * j + 1] = int(b[n, j]) >> 4
    np.testing.assert_array_equal(back, codes)


def test_pins_reject_planted_nibble_swap(monkeypatch):
    """A packer that puts the even channel in the high nibble must fail the
    hand-packed pin."""
    monkeypatch.setattr(rtn, "pack_codes",
                        lambda c: (np.asarray(c, np.uint8)[:, 1::2] | (np.asarray(c, np.uint8)[:, 0::2] << 4))
                        .astype(np.uint8))
    with pytest.raises(AssertionError):
        test_pack_codes_hand_packed()
    with pytest.raises(AssertionError):
        test_pack_codes_round_trip_by_bit_ops()
