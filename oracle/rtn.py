"""Oracle of the 4-bit round-to-nearest (RTN) quantiser and of the static
low-rank initialisation of the compensator.

Test infrastructure only (see the package docstring).

RTN is the quantisation backend the SPEAR paper reports its per-channel
results on ("SPEAR: A System for Post-Quantization Error-Adaptive Recovery",
section 3.1, "RTN, per-channel"); the paper does not spell the quantiser out,
so this follows the usual asymmetric min/max form. Per group of G input
channels of one output row:

    lo = min(0, min w), hi = max(0, max w), range = max(hi - lo, 1e-8)
    s  = bf16_RNE(range / 15)                       (the stored scale)
    z  = clamp(rint(-lo / s), 0, 15)                (the stored zero point)
    q  = clamp(rint(w / s) + z, 0, 15)              (the stored code)

so that w is approximated by (q - z) * s, the dequantisation the layer uses.
The codes are integers decided by floating point, so the steps are taken in
fp32 (IEEE division, round half to even) exactly as the GPU kernel takes them.

The static initialisation of the compensator from the quantisation error
E = W - W_q (the static low-rank correction the paper contrasts with in
section 1) is the truncated SVD E ~ U S V^T: B = U S^(1/2), A = S^(1/2) V^T.
"""
from __future__ import annotations

import numpy as np

F32 = np.float32


def bf16_rne_bits(v: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns, round to nearest even (finite inputs)."""
    u = np.ascontiguousarray(v, dtype=F32).view(np.uint32).astype(np.uint64)
    r = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return r.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, np.uint32) << 16).view(F32)


def rtn_quantize(w: np.ndarray, group_size: int):
    """w float32 [N][K] -> (codes uint8 [N][K], s bf16 bits [N][K/G], z uint8 [N][K/G])."""
    w = np.ascontiguousarray(w, dtype=F32)
    N, K = w.shape
    G = K if group_size == 0 else group_size
    wg = w.reshape(N, K // G, G)
    lo = np.minimum(wg.min(axis=2), F32(0))
    hi = np.maximum(wg.max(axis=2), F32(0))
    rng = np.maximum((hi - lo).astype(F32), F32(1e-8))
    s_bits = bf16_rne_bits((rng / F32(15)).astype(F32))
    s = bf16_bits_to_f32(s_bits)
    z = np.clip(np.rint((-lo) / s), 0, 15).astype(F32)
    q = np.clip(np.rint(wg / s[:, :, None]) + z[:, :, None], 0, 15)
    return q.reshape(N, K).astype(np.uint8), s_bits, z.astype(np.uint8)


def pack_codes(codes: np.ndarray) -> np.ndarray:
    """[N][K] codes -> [N][K/2] bytes, even k in the low nibble."""
    c = codes.astype(np.uint8)
    return (c[:, 0::2] | (c[:, 1::2] << 4)).astype(np.uint8)


def dequant(codes, s_bits, z, group_size):
    """fp64 (q - z) * s, [N][K]."""
    N, K = codes.shape
    G = K if group_size == 0 else group_size
    s = bf16_bits_to_f32(s_bits).astype(np.float64)
    return ((codes.astype(np.float64).reshape(N, K // G, G) - z[:, :, None]) * s[:, :, None]).reshape(N, K)


def svd_init(E: np.ndarray, rank: int):
    """(A [rank][K], B [N][rank]) fp64 with B A the best rank-`rank` approximation of E."""
    U, S, Vt = np.linalg.svd(np.asarray(E, np.float64), full_matrices=False)
    r = np.sqrt(S[:rank])
    return r[:, None] * Vt[:rank], U[:, :rank] * r[None, :]
