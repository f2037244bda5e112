"""The prefill launch plan, checked on the host (no GPU).

``spear_prefill_schedule`` returns the plan ``spear_linear_forward_prefill``
launches with, from the same host code. The plan splits the work of a layer
("SPEAR", section 3.3: the weight contraction W_q x with the compensator's
output GEMM alpha B u' as a K-tail) into units of one 64-channel K block of
one output tile, shares the units between the CTAs of a persistent kernel
(stream-K), and gives the compensator's projection items (one per 128 tokens)
their weight in units. What makes such a split correct, and what these tests
check over the layer shapes of the workloads and small ragged ones:

- the ranges partition the units: starts[0] = 0, starts[G] = units, and
  every range non-empty;
- no range starts inside a tile's K-tail, so each tile's owner (the CTA that
  holds its first unit) runs the whole K-tail, and every W block of every
  tile is run exactly once;
- an owner only waits for CTAs with a larger index (no cycle of waits), and
  the most partial tiles an owner adds fit its stage memory;
- all CTAs are resident at once (one CTA per SM, G at most the SMs that a
  preceding pre-kernel leaves), shared memory and TMEM columns within limits;
- the prologue items' weight comes out of their CTAs' shares.
"""

import pytest

from quantized_linear_error_gb300 import build, spear

SMS = 152
SMEM_MAX = 227 * 1024

# (N, K, rank, M, gate_hidden): the prefill shapes of the workloads, then
# small and ragged ones (gate_hidden > 0: the bottleneck-MLP gate).
SHAPES = [
    (14336, 4096, 128, 2048, 0),      # Llama-3-8B gate / up
    (14336, 4096, 128, 2048, 16),     # the same with the bottleneck-MLP gate
    (4096, 14336, 128, 2048, 0),      # Llama-3-8B down
    (4096, 4096, 64, 320, 0),         # 32-layer stack, 64 decode + 256 prefill tokens
    (11008, 4096, 64, 320, 0),
    (4096, 11008, 64, 320, 0),
    (4096, 4096, 64, 576, 0),
    (11008, 4096, 64, 576, 0),
    (4096, 11008, 64, 576, 0),
    (4096, 4096, 64, 1088, 0),
    (11008, 4096, 64, 1088, 0),
    (4096, 11008, 64, 1088, 0),
    (4096, 4096, 0, 1088, 0),         # layers without a compensator
    (11008, 4096, 0, 576, 0),
    (28672, 8192, 256, 2048, 0),      # Llama-70B MLP at a prefill token count
    (8192, 28672, 256, 600, 0),
    (2048, 2048, 32, 40, 0),
    (2048, 2048, 32, 200, 0),
    (200, 192, 32, 33, 0),
    (128, 64, 0, 33, 0),
    (384, 640, 96, 1000, 64),
    (4096, 4096, 256, 4096, 0),
    (14336, 4096, 256, 2048, 64),     # MLP gate whose prologue buffers would not fit
]


@pytest.fixture(scope="module")
def lib():
    build.build()
    return spear.load()


def _plan(N, K, r, M, gh, sms=SMS, ws=True):
    return spear.prefill_schedule(N, K, r, M, sms, gate_hidden=gh, with_workspace=ws)


def _tiles(d, N, M):
    return ((N + 127) // 128) * ((M + d["TN"] - 1) // d["TN"])


def _walk(d):
    """Each CTA's segments, as the kernel walks its range: (tile, first unit
    in the tile, units). Returns per tile the owner and contributors, and the
    run count of every unit."""
    kpt, starts = d["kpt"], d["starts"]
    owner, contrib, runs = {}, {}, [0] * d["units"]
    for c in range(d["G"]):
        u, end = starts[c], starts[c + 1]
        while u < end:
            t, j0 = divmod(u, kpt)
            n = min(kpt - j0, end - u)
            if j0 == 0:
                assert t not in owner
                owner[t] = c
            else:
                contrib.setdefault(t, []).append(c)
            for k in range(u, u + n):
                runs[k] += 1
            u += n
    return owner, contrib, runs


@pytest.mark.parametrize("N,K,r,M,gate", SHAPES)
def test_ranges_partition_the_units(lib, N, K, r, M, gate):
    d = _plan(N, K, r, M, gate)
    tiles = _tiles(d, N, M)
    assert d["tail"] == (r + 63) // 64
    assert d["kpt"] == K // 64 + d["tail"]
    assert d["units"] == tiles * d["kpt"]
    s = d["starts"]
    assert s[0] == 0 and s[-1] == d["units"] and len(s) == d["G"] + 1
    assert all(b > a for a, b in zip(s, s[1:]))
    owner, contrib, runs = _walk(d)
    assert all(n == 1 for n in runs)
    assert sorted(owner) == list(range(tiles))


@pytest.mark.parametrize("N,K,r,M,gate", SHAPES)
def test_owner_runs_the_whole_tail_and_waits_only_forward(lib, N, K, r, M, gate):
    d = _plan(N, K, r, M, gate)
    for b in d["starts"][:-1]:
        j = b % d["kpt"]
        assert j == 0 or j >= d["tail"], "a range starts inside a K-tail"
    owner, contrib, _ = _walk(d)
    worst = 0
    for t, cs in contrib.items():
        assert all(c > owner[t] for c in cs)
        # a contributor's partial is the first segment of its range
        assert all(d["starts"][c] // d["kpt"] == t for c in cs)
        worst = max(worst, len(cs))
    assert worst == d["max_contrib"]
    # the owner copies each partial [256][128] fp32 into stage memory 32 columns at a time
    assert d["max_contrib"] * 32 * 512 <= d["NS"] * d["stage_bytes"] or d["G"] == 1


@pytest.mark.parametrize("N,K,r,M,gate", SHAPES)
def test_resources_and_residency(lib, N, K, r, M, gate):
    d = _plan(N, K, r, M, gate)
    assert d["TN"] % 16 == 0 and 16 <= d["TN"] <= 256
    assert (M + d["TN"] - 1) // d["TN"] == (M + 255) // 256  # fewest tiles of at most 256 tokens
    assert SMEM_MAX // 2 < d["smem"] <= SMEM_MAX  # one CTA per SM, within the opt-in limit
    assert d["NS"] >= 2
    assert d["tmem_a"] >= d["TN"] and d["tmem_a"] % 32 == 0
    assert d["tmem_a"] + 32 * d["NS"] <= 512
    assert d["G"] + d["pre_ctas"] <= SMS  # every CTA resident, next to the pre-kernel's
    if d["mode"] == 3:
        assert r > 0 and d["pro_items"] == 0 and d["pre_ctas"] >= 1
    else:
        assert d["pre_ctas"] == 0
        assert d["pro_items"] == ((M + 127) // 128 if r > 0 else 0)
        if r > 0:  # an item's u' rows (and the MLP gate's z rows and weights) fit next to the barriers
            need = 128 * r * 2 + (128 * (r + 8) * 4 + (gate * (r + 8) + r * (gate + 8)) * 2 if gate else 0)
            assert need + 1024 < d["smem"]


@pytest.mark.parametrize("N,K,r,M,gate", [s for s in SHAPES if s[2] > 0])
def test_prologue_items_take_their_weight_from_their_ctas(lib, N, K, r, M, gate):
    d = _plan(N, K, r, M, gate)
    if d["mode"] != 0 or d["pro_d"] == 0:
        pytest.skip("no weighted prologue items in this plan")
    G, s = d["G"], d["starts"]
    items = [0] * G
    for i in range(d["pro_items"]):
        items[i % G] += 1
    share = (d["units"] + d["pro_items"] * d["pro_d"]) / G
    for c in range(G):
        load = s[c + 1] - s[c] + items[c] * d["pro_d"]
        assert abs(load - share) <= d["tail"] + 1
    with_item = [s[c + 1] - s[c] for c in range(G) if items[c]]
    without = [s[c + 1] - s[c] for c in range(G) if not items[c]]
    if with_item and without:
        assert max(with_item) < min(without)


def test_projection_placement(lib):
    """Where the projection runs: in the prologue when an item weighs at most
    3/4 of a CTA's share; else in the split-K pre-kernel (measured choices on
    the 32-layer stack's shapes at 576 tokens)."""
    assert _plan(14336, 4096, 128, 2048, 0)["mode"] == 0
    assert _plan(11008, 4096, 64, 576, 0)["mode"] == 0
    assert _plan(4096, 4096, 64, 576, 0)["mode"] == 3
    assert _plan(4096, 11008, 64, 576, 0)["mode"] == 3
    assert _plan(4096, 4096, 0, 576, 0)["mode"] == 0
    # rank 256 with a 64-wide MLP gate: z rows, u' rows and the gate's
    # weights need more than 227 KB, so the pre-kernel runs instead
    assert _plan(14336, 4096, 256, 2048, 0)["mode"] == 0
    assert _plan(14336, 4096, 256, 2048, 64)["mode"] == 3


def test_without_partial_workspace_one_cta_per_tile(lib):
    """Handles sized for decode token counts hold no partial-tile workspace:
    then each CTA runs one whole tile and the projection is a pre-kernel."""
    for N, K, r, M in [(4096, 4096, 64, 300), (2048, 2048, 32, 40), (4096, 4096, 0, 600)]:
        d = _plan(N, K, r, M, 0, ws=False)
        tiles = _tiles(d, N, M)
        assert d["G"] == tiles
        assert d["starts"] == [c * d["kpt"] for c in range(tiles + 1)]
        assert d["max_contrib"] == 0
        assert d["mode"] == (3 if r > 0 else 0)


@pytest.mark.parametrize("sms", [1, 2, 7, 76, 132, 148, 152])
def test_other_sm_counts(lib, sms):
    for N, K, r, M, gate in [(4096, 4096, 64, 1088, 0), (14336, 4096, 128, 2048, 16), (200, 192, 32, 33, 0)]:
        d = _plan(N, K, r, M, gate, sms=sms)
        assert 1 <= d["G"] <= max(1, sms - d["pre_ctas"])
        owner, _, runs = _walk(d)
        assert all(n == 1 for n in runs)
        assert len(owner) == _tiles(d, N, M)


def test_rejects_bad_shapes(lib):
    import ctypes
    info = (ctypes.c_int32 * 14)()
    L = spear.load()
    for args in [(0, 64, 0, 0, 1, 152, 1), (128, 100, 0, 0, 1, 152, 1), (128, 64, 300, 0, 1, 152, 1),
                 (128, 64, 0, 0, 0, 152, 1), (128, 64, 0, 0, 1, 0, 1), (128, 64, 32, 24, 1, 152, 1),
                 (128, 64, 32, 80, 1, 152, 1)]:
        assert L.spear_prefill_schedule(*args, info, None, 0) == spear.SPEAR_ERR_INVALID_ARG
    assert L.spear_prefill_schedule(128, 64, 0, 0, 1, 152, 1, None, None, 0) == spear.SPEAR_ERR_INVALID_ARG
    starts = (ctypes.c_uint32 * 1)()
    assert L.spear_prefill_schedule(4096, 4096, 64, 0, 2048, 152, 1, info, starts, 1) == spear.SPEAR_ERR_INVALID_ARG


def test_random_shapes(lib):
    """A seeded sweep of shapes beyond the workloads, with and without the
    stream-K workspace: every split partitions the units without starting
    inside a K-tail; stream-K grids are resident next to the pre-kernel and
    their owners' partials fit; one-CTA-per-tile grids have no partials."""
    import random
    rng = random.Random(2)
    for _ in range(300):
        N = rng.choice([8, 136, 200, 520, 1032, 4096, 4104, 11008, 12288, 14336, 22016, 28672])
        K = 64 * rng.randint(1, 460)
        r = rng.choice([0, 16, 32, 64, 128, 192, 256])
        gh = rng.choice([0, 0, 16, 64]) if r else 0
        M, ws = rng.randint(33, 4096), rng.random() < 0.9
        d = spear.prefill_schedule(N, K, r, M, SMS, gate_hidden=gh, with_workspace=ws)
        s = d["starts"]
        assert s[0] == 0 and s[-1] == d["units"] and all(b > a for a, b in zip(s, s[1:]))
        assert all(b % d["kpt"] == 0 or b % d["kpt"] >= d["tail"] for b in s[:-1])
        assert d["smem"] <= SMEM_MAX and d["NS"] >= 2 and d["tmem_a"] + 32 * d["NS"] <= 512
        if ws:
            assert d["G"] + d["pre_ctas"] <= SMS
            assert d["max_contrib"] * 32 * 512 <= d["NS"] * d["stage_bytes"] or d["G"] == 1
        else:
            assert d["max_contrib"] == 0 and all(x % d["kpt"] == 0 for x in s)
