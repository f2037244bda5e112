"""Shared helpers for the GPU parity tests (device marshalling and error metrics)."""
from __future__ import annotations

import numpy as np
import torch

from quantized_linear_error_gb300 import spear
from quantized_linear_error_gb300 import workload as wl


def dev_bf16(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def host_f64(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


def bits_of(t: torch.Tensor) -> np.ndarray:
    return t.cpu().view(torch.int16).numpy().view(np.uint16)


def rel_err(y: np.ndarray, ref: np.ndarray) -> float:
    """max |y - ref| / max |ref|: the layer's output tolerance metric."""
    return float(np.max(np.abs(y - ref)) / max(np.max(np.abs(ref)), 1e-30))


def sample_rows(N: int, n: int, seed: int = 0) -> np.ndarray:
    """Rows to check at full size: both ends, tile boundaries and a random set."""
    rng = np.random.default_rng(seed)
    fixed = {0, 1, 15, 16, 127, 128, N // 2, N - 129, N - 17, N - 16, N - 2, N - 1}
    rows = set(int(r) for r in fixed if 0 <= r < N)
    rows |= set(rng.choice(N, size=min(n, N), replace=False).tolist())
    return np.array(sorted(rows), dtype=np.int64)


def codes_equal_zeros(w: wl.LinearWeights) -> wl.LinearWeights:
    """Same linear with every code equal to its group's zero point (W_q = 0)."""
    sp = w.spec
    zfull = np.repeat(w.z, sp.G, axis=1).astype(np.uint8)           # [N][K]
    q = (zfull[:, 0::2] | (zfull[:, 1::2] << 4)).astype(np.uint8)
    return wl.LinearWeights(sp, q, w.s, w.z, w.A, w.B, w.outliers, w.W1, w.W2)


def with_spec(w: wl.LinearWeights, **kw) -> wl.LinearWeights:
    import dataclasses
    return wl.LinearWeights(dataclasses.replace(w.spec, **kw), w.q, w.s, w.z, w.A, w.B, w.outliers, w.W1, w.W2)


def run(lin: spear.SpearLinear, x_bits: np.ndarray, path: str) -> np.ndarray:
    x = dev_bf16(x_bits)
    y = torch.empty((x.shape[0], lin.N), dtype=torch.bfloat16, device="cuda")
    getattr(lin, f"forward_{path}")(x, y)
    st = lin.check()
    assert st == spear.SPEAR_OK, spear.status_string(st)
    return host_f64(y)
