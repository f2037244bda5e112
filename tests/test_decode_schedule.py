"""The decode launch plan, checked on the host (no GPU).

``spear_decode_schedule`` returns the plan ``spear_linear_forward_decode``
launches with, from the same host code. The decode kernel ("SPEAR", section
2.2A: the decode phase as one fused kernel) gives each CTA P 16-row tiles,
streams K in stages of KC channels through an NS-deep ring of shared memory
and waits, bounded, for every CTA's share of the compensator projection. What
makes a plan valid, and what these tests check over the decode shapes of the
workloads and small ragged ones at every token count:

- the grid covers every 16-row tile and is resident on the SMs at once (the
  grid-wide wait needs it);
- the consumer warps cover the tiles, the block fits 1024 threads, shared
  memory fits the opt-in limit, and the stage ring holds the partial sums
  that the reduction writes into it;
- stages are whole 256-channel layout runs, split evenly over the K warps
  (one or two 128-channel units each) unless one stage holds all of K, and
  the x box of a stage is at most 64 KB;
- there are at least two stages wherever K needs more than one (copy and
  compute overlap).
"""

import pytest

from quantized_linear_error_gb300 import build, spear

SMS = 152
SMEM_MAX = 227 * 1024

# (name, N, K, rank_b, n_members, group_size, gate_hidden)
SHAPES = [
    ("c1", 2048, 2048, 32, 1, 128, 0),
    ("c2/q", 4096, 4096, 64, 1, 128, 0),
    ("c2/qkv", 12288, 4096, 64, 3, 128, 0),
    ("c2/gateup", 22016, 4096, 64, 2, 128, 0),
    ("c2/up", 11008, 4096, 64, 1, 128, 0),
    ("c2/down", 4096, 11008, 64, 1, 128, 0),
    ("c2/q noec", 4096, 4096, 0, 1, 128, 0),
    ("c4/up", 28672, 8192, 256, 1, 0, 0),
    ("c4/down", 8192, 28672, 256, 1, 0, 0),
    ("mlp", 4096, 4096, 64, 1, 128, 16),
    ("mlp r256", 520, 640, 256, 1, 0, 64),
    ("ragged", 200, 256, 16, 1, 128, 0),
    ("one tile", 8, 128, 0, 1, 128, 0),
]
TOKENS = [1, 2, 5, 8, 9, 16, 17, 32]


@pytest.fixture(scope="module")
def lib():
    build.build()
    return spear.load()


@pytest.mark.parametrize("M", TOKENS)
@pytest.mark.parametrize("name,N,K,rb,n,gs,gh", SHAPES, ids=[s[0] for s in SHAPES])
def test_plan_is_valid(lib, name, N, K, rb, n, gs, gh, M):
    d = spear.decode_schedule(N, K, M, SMS, rank_b=rb, n_members=n, group_size=gs, gate_hidden=gh)
    tiles = (N + 15) // 16
    assert d["grid"] * d["P"] >= tiles and (d["grid"] - 1) * d["P"] < tiles
    assert d["grid"] <= SMS  # one CTA per SM, all resident
    assert d["MT"] == (1 if M <= 8 else 2 if M <= 16 else 4)
    assert d["P"] <= d["T"] * d["NW"]
    assert d["KW"] >= 1 and d["KW"] * ((d["P"] + d["T"] - 1) // d["T"]) <= d["NW"]
    assert d["threads"] == (d["NW"] + 5) * 32 <= 1024
    assert d["smem"] <= SMEM_MAX
    assert d["KC"] % 256 == 0
    units = d["KC"] // 128  # per stage; an even split is the fixed-offset path, else the round-robin one
    assert (units % d["KW"] == 0 and units // d["KW"] <= 2) or d["KC"] >= (K + 255) // 256 * 256
    assert d["bytes_x"] == d["KC"] * 8 * d["MT"] * 2 <= 64 * 1024
    assert d["n_stages"] == (K + d["KC"] - 1) // d["KC"]
    assert d["NS"] >= 1
    assert d["NS"] * d["stage_bytes"] >= d["P"] * d["KW"] * 32 * 4 * d["MT"] * 4  # the reduction's partials
    if d["n_stages"] > 1:
        assert d["NS"] >= 2, "a single stage leaves copies and compute serialised"


def test_large_compensator_leaves_room_for_stages(lib):
    """Rank 256 (config 4): the B fragments are staged after the W loop, so
    that the pipeline keeps several stages (with them resident for the whole
    call it had 1-3)."""
    for M in (1, 8, 16, 32):
        d = spear.decode_schedule(28672, 8192, M, SMS, rank_b=256, group_size=0)
        assert d["NS"] >= 4


def test_rejects_bad_shapes(lib):
    import ctypes
    L = spear.load()
    info = (ctypes.c_int32 * 13)()
    bad = [(0, 128, 0, 1, 128, 0, 1, SMS), (128, 100, 0, 1, 128, 0, 1, SMS), (128, 128, 8, 1, 128, 0, 1, SMS),
           (128, 128, 64, 9, 128, 0, 1, SMS), (128, 128, 64, 5, 128, 0, 1, SMS), (128, 128, 64, 1, 64, 0, 1, SMS),
           (128, 128, 64, 1, 128, 24, 1, SMS), (128, 128, 0, 1, 128, 16, 1, SMS), (128, 128, 64, 1, 128, 0, 0, SMS),
           (128, 128, 64, 1, 128, 0, 33, SMS), (128, 128, 64, 1, 128, 0, 1, 0)]
    for args in bad:
        assert L.spear_decode_schedule(*args, info) == spear.SPEAR_ERR_INVALID_ARG, args
    assert L.spear_decode_schedule(128, 128, 0, 1, 128, 0, 1, SMS, None) == spear.SPEAR_ERR_INVALID_ARG
    # more rows than 16 tiles per CTA on every SM
    assert L.spear_decode_schedule(16 * 16 * 4 + 16, 128, 0, 1, 128, 0, 1, 4, info) == spear.SPEAR_ERR_UNSUPPORTED


def test_random_shapes(lib):
    """A seeded sweep of shapes beyond the workloads: every plan valid, and
    two or more stages wherever K needs them at ranks up to 64 without the
    MLP gate (at rank 128-256 with a 64-wide gate, or 16 tiles per CTA at
    rank 256, the compensator's buffers can leave room for one)."""
    import random
    rng = random.Random(1)
    checked = 0
    for _ in range(600):
        N = rng.choice([8, 16, 136, 200, 520, 1032, 2048, 4096, 4104, 8192, 11008, 12288, 22016, 28672, 36864])
        K = 128 * rng.randint(1, 230)
        gs, n, M = rng.choice([0, 128]), rng.choice([1, 1, 2, 3, 4]), rng.randint(1, 32)
        rb = rng.choice([0, 16, 32, 64, 128, 256])
        gh = rng.choice([0, 0, 16, 64]) if rb and n == 1 else 0
        if N % n or n * rb > 256:
            continue
        try:
            d = spear.decode_schedule(N, K, M, SMS, rank_b=rb, n_members=n, group_size=gs, gate_hidden=gh)
        except spear.SpearError as e:
            assert e.status == spear.SPEAR_ERR_UNSUPPORTED  # more than 16 tiles per CTA
            continue
        checked += 1
        assert d["grid"] <= SMS and d["smem"] <= SMEM_MAX and d["NS"] >= 1 and d["threads"] <= 1024
        assert d["grid"] * d["P"] >= (N + 15) // 16 and d["KC"] % 256 == 0 and d["bytes_x"] <= 64 * 1024
        if rb <= 64 and gh == 0 and d["n_stages"] > 1:
            assert d["NS"] >= 2, (N, K, gs, n, rb, M, d)
    assert checked > 300


@pytest.mark.parametrize("sms", [16, 76, 132, 148])
def test_other_sm_counts(lib, sms):
    """Fewer SMs than the GB300's 152: more tiles per CTA, the same limits.
    UNSUPPORTED is allowed where a CTA would need more than 16 tiles or its
    buffers would not fit next to one stage; the decode layer set's shapes
    plan on 76 SMs and more wherever 16 tiles per CTA cover them."""
    for name, N, K, rb, n, gs, gh in SHAPES:
        for M in (1, 16, 32):
            try:
                d = spear.decode_schedule(N, K, M, sms, rank_b=rb, n_members=n, group_size=gs, gate_hidden=gh)
            except spear.SpearError as e:
                assert e.status == spear.SPEAR_ERR_UNSUPPORTED, name
                assert not (name.startswith("c2/") and sms >= 76 and (N + 15) // 16 <= 16 * sms), name
                continue
            assert d["grid"] <= sms and d["grid"] * d["P"] >= (N + 15) // 16, name
            assert d["smem"] <= SMEM_MAX and d["NS"] >= 1 and d["threads"] <= 1024, name
