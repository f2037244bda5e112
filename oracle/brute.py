"""Pure-Python brute force for tiny shapes (test infrastructure only).

Unlike the C oracle, which applies the compensator in factored form, this file
builds the per-token effective weight of the SPEAR error compensator
("SPEAR: A System for Post-Quantization Error-Adaptive Recovery", section 2.1A,
"Mechanism"),

    W_eff(x) = W + alpha * B * diag(gamma(A x)) * A,

element by element and multiplies it with x. The 4-bit codes are pulled out of
the packed bytes with explicit bit operations, and the bf16 rounding of the
dequantised value uses torch's float32 -> bfloat16 cast instead of the C
oracle's hand-written rounding. Plain Python floats (IEEE double) throughout.
Intended for K, N <= 64, r <= 8, M <= 4.
"""
from __future__ import annotations

import math
import struct

import numpy as np
import torch


def bf16_value(bits: int) -> float:
    return struct.unpack("<f", struct.pack("<I", (int(bits) & 0xFFFF) << 16))[0]


def unpack_code(q_row: np.ndarray, k: int) -> int:
    byte = int(q_row[k >> 1])
    return (byte >> 4) & 0xF if k & 1 else byte & 0xF


def dequant_value(q, s, z, n, k, G) -> float:
    g = k // G
    zp = 8 if z is None else int(z[n][g])
    return float(unpack_code(q[n], k) - zp) * bf16_value(s[n][g])


def dequant_bf16(q, s, z, N, K, G) -> np.ndarray:
    """bf16 bits of each dequantised element via torch's RNE cast of the exact
    float32 product (|q - z| <= 15 times an 8-bit significand is exact)."""
    vals = np.array([[dequant_value(q, s, z, n, k, G) for k in range(K)] for n in range(N)], np.float32)
    return torch.from_numpy(vals).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def sigmoid(v: float) -> float:
    return 1.0 / (1.0 + math.exp(-v))


def mlp_gamma(zvec, W1, W2) -> list:
    """Bottleneck-MLP gate values gamma(z) = sigmoid(W2 relu(W1 z)) by plain
    loops (W1 bf16 bits [h][r], W2 bf16 bits [r][h])."""
    h, r = len(W1), len(zvec)
    t = [max(0.0, sum(bf16_value(W1[i][j]) * zvec[j] for j in range(r))) for i in range(h)]
    return [sigmoid(sum(bf16_value(W2[j][i]) * t[i] for i in range(h))) for j in range(r)]


def forward(q, s, z, K, G, A, B, alpha, gate, x, W1=None, W2=None) -> np.ndarray:
    """y [M][N] from the explicitly materialised effective weight per token."""
    N = len(q)
    M = len(x)
    r = 0 if A is None else len(A)
    W = [[dequant_value(q, s, z, n, k, G) for k in range(K)] for n in range(N)]
    Af = [[bf16_value(A[j][k]) for k in range(K)] for j in range(r)]
    Bf = [[bf16_value(B[n][j]) for j in range(r)] for n in range(N)]
    y = np.zeros((M, N))
    for m in range(M):
        xm = [bf16_value(v) for v in x[m]]
        zvec = [sum(Af[j][k] * xm[k] for k in range(K)) for j in range(r)]
        if gate == 2:
            gam = mlp_gamma(zvec, W1, W2)
        else:
            gam = [1.0 if gate == 1 else sigmoid(v) for v in zvec]
        weff = [[W[n][k] + alpha * sum(Bf[n][j] * gam[j] * Af[j][k] for j in range(r))
                 for k in range(K)] for n in range(N)]
        for n in range(N):
            y[m][n] = sum(weff[n][k] * xm[k] for k in range(K))
    return y
