"""Offline set-up of a compensated 4-bit linear from full-precision weights.

1. RTN 4-bit quantisation on the GPU (``spear_quantize_rtn``, the backend of
   the per-channel results in "SPEAR: A System for Post-Quantization
   Error-Adaptive Recovery", section 3.1).
2. The exact dequantised weight W_q from the library's own unpack code (a
   rank-0 handle's dequantisation export).
3. The static initialisation of the compensator from the quantisation error
   E = W - W_q: the truncated SVD E ~ U S V^T gives B = U S^(1/2) and
   A = S^(1/2) V^T, so that with the constant gate the layer computes
   (W_q + B A) x, the static low-rank correction the paper contrasts with in
   section 1. With per-channel activation scales a (the RMS of each input
   channel over calibration tokens) the SVD is taken of E diag(a) and A is
   divided by a afterwards: the truncation then keeps the error directions
   that matter for the output (E x), which the activation outliers dominate.

This is a set-up step, not the layer's hot path: the SVD is a library call
(torch.linalg.svd). The paper calibrates the gate itself by minimising a KL
divergence against the full-precision model, which needs a model and data and
is not done here.
"""
from __future__ import annotations

import torch

from . import spear


def quantize_and_init(W: torch.Tensor, group_size: int = 128, rank: int = 64, act_scale: torch.Tensor | None = None,
                      stream=None):
    """W: CUDA fp32 [N][K]. Returns (qweight, scales, zeros, A bf16 [rank][K],
    B bf16 [N][rank], W_q fp32 [N][K]); A and B are None for rank 0."""
    N, K = W.shape
    q, s, z = spear.quantize_rtn(W, group_size, stream)
    lin = spear.SpearLinear(K, N, group_size, q, s, z, max_tokens=1, stream=stream)
    wq = torch.empty((N, K), dtype=torch.bfloat16, device=W.device)
    lin.dequantize(wq, 0, stream)
    torch.cuda.synchronize()
    lin.close()
    wq = wq.float()
    if rank == 0:
        return q, s, z, None, None, wq
    E = (W.float() - wq).double()
    if act_scale is not None:
        E = E * act_scale.double()[None, :]
    U, S, Vh = torch.linalg.svd(E, full_matrices=False)
    r = S[:rank].sqrt()
    A = r[:, None] * Vh[:rank]
    B = U[:, :rank] * r[None, :]
    if act_scale is not None:
        A = A / act_scale.double()[None, :]
    return q, s, z, A.to(torch.bfloat16).contiguous(), B.to(torch.bfloat16).contiguous(), wq
