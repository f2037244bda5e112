"""ctypes front end of the fp64 C oracle (``spear_ref.c``).

Test infrastructure only (see the package docstring). The formulas live in the
C file; this module only builds it, marshals numpy arrays and returns numpy
results.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from pathlib import Path

import numpy as np

_HERE = Path(__file__).resolve().parent
_SRC = _HERE / "spear_ref.c"
_BUILD = _HERE / "_build"
_libs: dict = {}
_active = 0


def build(force: bool = False, plant: int = 0) -> Path:
    """Compile the oracle (cc, -O2, OpenMP, no fast-math). ``plant`` > 0 builds
    a variant with one deliberate mistake, used only to show the pins catch it."""
    path = _BUILD / ("libspear_ref.so" if plant == 0 else f"libspear_ref_plant{plant}.so")
    _BUILD.mkdir(exist_ok=True)
    if force or not path.exists() or path.stat().st_mtime < _SRC.stat().st_mtime:
        tmp = path.with_suffix(f".{os.getpid()}.so")
        subprocess.check_call(["cc", "-O2", "-fopenmp", "-shared", "-fPIC", "-std=c11",
                               f"-DSPEAR_PLANT={plant}", "-o", str(tmp), str(_SRC), "-lm"])
        os.replace(tmp, path)
    return path


def lib():
    plant = _active
    if plant not in _libs:
        L = ctypes.CDLL(str(build(plant=plant)))
        P = ctypes.c_void_p
        I = ctypes.c_int
        L.oracle_dequant_bf16.argtypes = [P, P, P, I, I, I, P]
        L.oracle_dequant_f64.argtypes = [P, P, P, I, I, I, P]
        L.oracle_ec.argtypes = [P, P, I, I, I, I, P, P]
        L.oracle_gate.argtypes = [P, I, I, P]
        L.oracle_forward.argtypes = [P, P, P, I, I, I, P, P, I, ctypes.c_double, I, P, I, P, I, P, I, I, P, P]
        L.oracle_gate_mlp.argtypes = [P, I, I, I, P, P, P]
        L.oracle_max_threads.restype = I
        _libs[plant] = L
    return _libs[plant]


class planted:
    """Context manager: route this module's calls to planted variant ``n``."""

    def __init__(self, n: int):
        self.n = n

    def __enter__(self):
        global _active
        self.prev, _active = _active, self.n
        return self

    def __exit__(self, *exc):
        global _active
        _active = self.prev
        return False


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dt):
    return None if a is None else np.ascontiguousarray(a, dtype=dt)


def dequant_bf16(q, s, z, N, K, G):
    """bf16 bit patterns [N][K] of (q - z) * s, one round-to-nearest-even."""
    q, s, z = _c(q, np.uint8), _c(s, np.uint16), _c(z, np.uint8)
    out = np.empty((N, K), np.uint16)
    lib().oracle_dequant_bf16(_p(q), _p(s), _p(z), N, K, G, _p(out))
    return out


def dequant_f64(q, s, z, N, K, G):
    q, s, z = _c(q, np.uint8), _c(s, np.uint16), _c(z, np.uint8)
    out = np.empty((N, K), np.float64)
    lib().oracle_dequant_f64(_p(q), _p(s), _p(z), N, K, G, _p(out))
    return out


def ec(A, x, gate=0):
    """(z, u) double [M][r]: z = A x per token, u = gamma(z) * z."""
    A, x = _c(A, np.uint16), _c(x, np.uint16)
    r, K = A.shape
    M = x.shape[0]
    z = np.empty((M, r), np.float64)
    u = np.empty((M, r), np.float64)
    lib().oracle_ec(_p(A), _p(x), r, K, M, gate, _p(z), _p(u))
    return z, u


def gate(z, gate=0):
    z = _c(z, np.float64)
    u = np.empty_like(z)
    lib().oracle_gate(_p(z), z.size, gate, _p(u))
    return u


def gate_mlp(z, W1, W2):
    """u double [M][r] = sigmoid(W2 relu(W1 z)) * z per token; W1 bf16 [h][r], W2 bf16 [r][h]."""
    z = _c(np.atleast_2d(z), np.float64)
    W1, W2 = _c(W1, np.uint16), _c(W2, np.uint16)
    M, r = z.shape
    h = W1.shape[0]
    u = np.empty_like(z)
    lib().oracle_gate_mlp(_p(z), M, r, h, _p(W1), _p(W2), _p(u))
    return u


def forward(q, s, z, K, G, A, B, alpha, gate, x, rows=None, nthreads=0, W1=None, W2=None):
    """y double [M][len(rows)] (all N rows when rows is None). gate 2 (MLP)
    takes W1 bf16 [h][r] and W2 bf16 [r][h]."""
    q, s, z = _c(q, np.uint8), _c(s, np.uint16), _c(z, np.uint8)
    A, B, x = _c(A, np.uint16), _c(B, np.uint16), _c(x, np.uint16)
    W1, W2 = _c(W1, np.uint16), _c(W2, np.uint16)
    h = 0 if W1 is None else W1.shape[0]
    N = q.shape[0]
    r = 0 if A is None else A.shape[0]
    M = x.shape[0]
    rows_a = None if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    nrows = N if rows_a is None else rows_a.size
    y = np.empty((M, nrows), np.float64)
    lib().oracle_forward(_p(q), _p(s), _p(z), N, K, G, _p(A), _p(B), r, float(alpha), gate,
                         _p(x), M, _p(rows_a), nrows, _p(y), int(nthreads), h, _p(W1), _p(W2))
    return y


def forward_w(w, x, rows=None, nthreads=0):
    """Convenience: forward for a ``workload.LinearWeights``."""
    sp = w.spec
    return forward(w.q, w.s, w.z, sp.K, sp.G, w.A, w.B, sp.alpha, sp.gate, x, rows, nthreads,
                   getattr(w, "W1", None), getattr(w, "W2", None))


def max_threads() -> int:
    return lib().oracle_max_threads()
