"""Seeded synthetic inputs for the W4 + input-adaptive error-compensator linear.

This module only draws random tensors. It holds none of the layer's arithmetic
(no unpacking, dequantisation, contraction or gate), so that the CPU oracle and
the CUDA path can both consume its output without sharing any method code.

Every tensor is drawn on the CPU from its own counter-based Philox stream whose
key is the first 8 bytes of SHA-256("{base_seed}/{name}"), so a tensor is
bit-identical on any machine and independent of which other tensors were drawn.

Distributions (the SPEAR linear, "SPEAR: A System for Post-Quantization
Error-Adaptive Recovery", section 2.1A, with the workload shapes of the
serving benchmarks it reports in section 3.2):

* ``q``: packed INT4 codes, uint8 ``[N][K/2]``; byte ``j`` of row ``n`` holds
  ``k = 2j`` in its low nibble and ``k = 2j+1`` in its high nibble. Every nibble
  is uniform on 0..15 (uniform random bytes).
* ``s``: bf16 scales ``[N][K/G]``, ``U(0.005, 0.02)`` rounded to bf16 (RNE).
* ``z``: uint8 zero points ``[N][K/G]``, uniform on 0..15.
* ``A``: bf16 ``[r][K]``, ``B``: bf16 ``[N][r]``, both ``N(0, 0.02)`` (0.02 is
  the standard deviation).
* ``x``: bf16 ``[M][K]``, ``N(0, 1)`` with ``round(0.01 K)`` channels (picked
  without replacement per linear, fixed across tokens) multiplied by 20 before
  the bf16 rounding.

bf16 tensors are carried as ``numpy.uint16`` bit patterns.
"""
from __future__ import annotations

import hashlib
from dataclasses import dataclass, field

import numpy as np
import torch

GATE_SIGMOID = 0
GATE_ONE = 1
GATE_MLP = 2


def stream(base_seed: int, name: str) -> np.random.Generator:
    """Independent Philox stream for the tensor called ``name``."""
    key = int.from_bytes(hashlib.sha256(f"{base_seed}/{name}".encode()).digest()[:8], "little")
    return np.random.Generator(np.random.Philox(key))


def to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns with round-to-nearest-even (torch's cast)."""
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to float32 (exact)."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def random_bytes(rng: np.random.Generator, n: int) -> np.ndarray:
    words = (n + 7) // 8
    return rng.bit_generator.random_raw(words).view(np.uint8)[:n].copy()


@dataclass(frozen=True)
class LinearSpec:
    """Shape and EC settings of one quantised linear (weights are N x K)."""
    name: str
    K: int
    N: int
    group_size: int = 128      # 0 means one group per output channel (G = K)
    rank: int = 0              # 0 means no error compensator
    alpha: float = 1.0
    gate: int = GATE_SIGMOID
    gate_hidden: int = 16      # hidden width h of the bottleneck-MLP gate (GATE_MLP only)

    @property
    def G(self) -> int:
        return self.K if self.group_size == 0 else self.group_size

    @property
    def n_groups(self) -> int:
        return self.K // self.G

    def algorithmic_bytes(self, M: int) -> int:
        """HBM bytes one forward must move at minimum: W4 codes, bf16 scales,
        4-bit zeros, the EC's A and B, x read once and y written once."""
        w = self.N * self.K // 2 + self.N * self.n_groups * 2 + (self.N * self.n_groups + 1) // 2
        ec = self.rank * (self.K + self.N) * 2
        if self.rank and self.gate == GATE_MLP:
            ec += 2 * self.rank * self.gate_hidden * 2
        return w + ec + M * self.K * 2 + M * self.N * 2

    def flops(self, M: int) -> int:
        """Multiply-adds x2 of the main contraction plus both EC projections
        (and the two layers of an MLP gate)."""
        mlp = 4 * M * self.rank * self.gate_hidden if self.rank and self.gate == GATE_MLP else 0
        return 2 * M * self.K * self.N + 2 * M * self.rank * (self.K + self.N) + mlp


@dataclass
class LinearWeights:
    spec: LinearSpec
    q: np.ndarray          # uint8 [N][K/2]
    s: np.ndarray          # uint16 (bf16) [N][K/G]
    z: np.ndarray          # uint8 [N][K/G]
    A: np.ndarray | None   # uint16 (bf16) [r][K]
    B: np.ndarray | None   # uint16 (bf16) [N][r]
    outliers: np.ndarray = field(default_factory=lambda: np.zeros(0, np.int64))
    W1: np.ndarray | None = None   # uint16 (bf16) [h][r], MLP gate only
    W2: np.ndarray | None = None   # uint16 (bf16) [r][h], MLP gate only


def outlier_channels(K: int, base_seed: int, name: str) -> np.ndarray:
    n_out = int(round(0.01 * K))
    rng = stream(base_seed, f"{name}/outliers")
    return np.sort(rng.permutation(K)[:n_out]).astype(np.int64)


def make_weights(spec: LinearSpec, base_seed: int = 0, prefix: str = "") -> LinearWeights:
    name = f"{prefix}{spec.name}"
    N, K, ng, r = spec.N, spec.K, spec.n_groups, spec.rank
    q = random_bytes(stream(base_seed, f"{name}/q"), N * K // 2).reshape(N, K // 2)
    s = to_bf16_bits(stream(base_seed, f"{name}/s").uniform(0.005, 0.02, size=(N, ng)).astype(np.float32))
    z = stream(base_seed, f"{name}/z").integers(0, 16, size=(N, ng), dtype=np.uint8)
    A = B = None
    if r > 0:
        A = to_bf16_bits(stream(base_seed, f"{name}/A").normal(0.0, 0.02, size=(r, K)).astype(np.float32))
        B = to_bf16_bits(stream(base_seed, f"{name}/B").normal(0.0, 0.02, size=(N, r)).astype(np.float32))
    W1 = W2 = None
    if r > 0 and spec.gate == GATE_MLP:
        # weights of unit gain per layer: hidden pre-activations and gate logits O(1)
        h = spec.gate_hidden
        W1 = to_bf16_bits(stream(base_seed, f"{name}/W1").normal(0.0, r ** -0.5, size=(h, r)).astype(np.float32))
        W2 = to_bf16_bits(stream(base_seed, f"{name}/W2").normal(0.0, h ** -0.5, size=(r, h)).astype(np.float32))
    return LinearWeights(spec, q, s, z, A, B, outlier_channels(K, base_seed, name), W1, W2)


def make_x(K: int, M: int, outliers: np.ndarray, base_seed: int = 0, name: str = "x") -> np.ndarray:
    """bf16 activations [M][K]: N(0,1) with the outlier channels scaled by 20."""
    x = stream(base_seed, f"{name}/x{M}").standard_normal(size=(M, K), dtype=np.float32)
    x[:, outliers] *= 20.0
    return to_bf16_bits(x)


# ---------------------------------------------------------------------------
# The five workloads. Names follow the projections of a Llama-style block.
# ---------------------------------------------------------------------------
def llama7b_layer(prefix: str = "", rank: int = 64, group_size: int = 128) -> list[LinearSpec]:
    d, f = 4096, 11008
    shapes = [("q", d, d), ("k", d, d), ("v", d, d), ("o", d, d),
              ("gate", d, f), ("up", d, f), ("down", f, d)]
    return [LinearSpec(f"{prefix}{n}", K, N, group_size, rank) for n, K, N in shapes]


def config_linears(cfg: int, base_seed: int = 0) -> list[LinearSpec]:
    """Linear specs of workload ``cfg`` (1..5)."""
    if cfg == 1:
        return [LinearSpec("c1/fc", 2048, 2048, 128, 32)]
    if cfg == 2:
        return llama7b_layer("c2/")
    if cfg == 3:
        return [LinearSpec("c3/gate", 4096, 14336, 128, 128), LinearSpec("c3/up", 4096, 14336, 128, 128),
                LinearSpec("c3/down", 14336, 4096, 128, 128)]
    if cfg == 4:
        return [LinearSpec("c4/up", 8192, 28672, 0, 256), LinearSpec("c4/down", 28672, 8192, 0, 256)]
    if cfg == 5:
        ec_layers = set(ec_layer_indices(base_seed))
        out = []
        for layer in range(32):
            out += llama7b_layer(f"c5/L{layer}/", rank=64 if layer in ec_layers else 0)
        return out
    raise ValueError(f"unknown workload {cfg}")


def ec_layer_indices(base_seed: int = 0, n_layers: int = 32, n_ec: int = 4) -> list[int]:
    """The decoder layers that carry an error compensator in the mixed serving step."""
    return sorted(int(i) for i in stream(base_seed, "c5/ec_layers").permutation(n_layers)[:n_ec])


CONFIG_TOKENS = {1: [4], 2: [1, 8, 32], 3: [2048], 4: [16], 5: [64 + 256, 64 + 512, 64 + 1024]}
