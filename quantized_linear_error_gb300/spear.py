"""Thin ctypes binding of ``include/spear.h``.

Argument marshalling only: every step of the layer runs in the CUDA kernels of
``libspear_gb300.so``. The functions keep the C names; :class:`SpearLinear`
is a convenience owner of one handle that takes torch tensors for device
memory and streams. There is no CPU fallback: loading fails loudly when the
library has not been built.
"""
from __future__ import annotations

import ctypes
import re
from ctypes import POINTER, byref, c_char_p, c_double, c_float, c_int, c_int32, c_int64, c_void_p
from pathlib import Path

PKG = Path(__file__).resolve().parent
LIB_PATH = PKG / "libspear_gb300.so"
HEADER = PKG.parent / "include" / "spear.h"

SPEAR_OK, SPEAR_ERR_INVALID_ARG, SPEAR_ERR_UNSUPPORTED, SPEAR_ERR_OOM, SPEAR_ERR_CUDA, SPEAR_ERR_TIMEOUT = range(6)
SPEAR_GATE_SIGMOID, SPEAR_GATE_ONE, SPEAR_GATE_MLP = 0, 1, 2
DECODE_MAX_TOKENS = 32


class spear_linear_desc_t(ctypes.Structure):
    _fields_ = [("K", c_int32), ("N", c_int32), ("group_size", c_int32),
                ("qweight", c_void_p), ("scales", c_void_p), ("zeros", c_void_p),
                ("rank", c_int32), ("A", c_void_p), ("B", c_void_p),
                ("alpha", c_float), ("gate", c_int), ("max_tokens", c_int32),
                ("gate_hidden", c_int32), ("gate_w1", c_void_p), ("gate_w2", c_void_p)]


class SpearError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)}")


_lib = None


def header_functions() -> list[str]:
    """Names of the functions ``include/spear.h`` declares."""
    text = HEADER.read_text()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[\w\s\*]*?\b(spear_\w+)\s*\(", text, re.M)))


def load(path: Path | None = None):
    """Load the library (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    p = Path(path or LIB_PATH)
    if not p.exists():
        raise RuntimeError(f"{p} is missing: build it with quantized_linear_error_gb300.build.build()")
    L = ctypes.CDLL(str(p))
    H = c_void_p  # opaque handle / stream
    L.spear_linear_create.argtypes = [POINTER(spear_linear_desc_t), H, POINTER(c_void_p)]
    L.spear_linear_create_grouped.argtypes = [POINTER(spear_linear_desc_t), c_int32, H, POINTER(c_void_p)]
    L.spear_linear_create_grouped.restype = c_int
    L.spear_linear_forward_decode.argtypes = [H, c_void_p, c_void_p, c_int32, H]
    L.spear_linear_forward_prefill.argtypes = [H, c_void_p, c_void_p, c_int32, H]
    L.spear_linear_forward.argtypes = [H, c_void_p, c_void_p, c_int32, H]
    L.spear_linear_forward_prefill_concurrent.argtypes = [H, c_void_p, c_void_p, c_int32, H, H]
    L.spear_linear_forward_prefill_concurrent.restype = c_int
    L.spear_linear_enable_concurrent_ec.argtypes = [H]
    L.spear_linear_enable_concurrent_ec.restype = c_int
    L.spear_linear_forward_host.argtypes = [H, c_void_p, c_void_p, c_int32, H]
    L.spear_linear_forward_host_batch.argtypes = [c_void_p, c_void_p, c_void_p, c_void_p, c_int32, H]
    L.spear_linear_forward_host_batch.restype = c_int
    L.spear_linear_destroy.argtypes = [H]
    L.spear_linear_dequantize.argtypes = [H, c_int32, c_void_p, H]
    L.spear_linear_check.argtypes = [H, H]
    L.spear_linear_debug_set.argtypes = [H, c_int64, c_int32]
    L.spear_linear_forward_decode_noalloc.argtypes = [POINTER(spear_linear_desc_t), c_void_p, c_void_p, c_int32, H]
    L.spear_linear_forward_decode_noalloc.restype = c_int
    L.spear_sched_create.argtypes = [c_void_p, c_int32, c_void_p, c_int32, c_void_p, POINTER(c_void_p)]
    L.spear_sched_create.restype = c_int
    L.spear_sched_predict.argtypes = [H, c_int32, c_double]
    L.spear_sched_predict.restype = c_double
    L.spear_sched_pick_chunk.argtypes = [H, c_int32, c_double, c_double, c_void_p, c_int32, POINTER(c_int32)]
    L.spear_sched_pick_chunk.restype = c_int
    L.spear_sched_destroy.argtypes = [H]
    L.spear_sched_destroy.restype = c_int
    L.spear_quantize_rtn.argtypes = [c_void_p, c_int32, c_int32, c_int32, c_void_p, c_void_p, c_void_p, H]
    L.spear_quantize_rtn.restype = c_int
    L.spear_decode_schedule.argtypes = [c_int32] * 8 + [c_void_p]
    L.spear_decode_schedule.restype = c_int
    L.spear_prefill_schedule.argtypes = [c_int32] * 7 + [c_void_p, c_void_p, c_int32]
    L.spear_prefill_schedule.restype = c_int
    L.spear_status_string.argtypes = [c_int]
    L.spear_status_string.restype = c_char_p
    for name in ("spear_linear_create", "spear_linear_forward_decode", "spear_linear_forward_prefill",
                 "spear_linear_forward", "spear_linear_forward_host", "spear_linear_destroy",
                 "spear_linear_dequantize", "spear_linear_check", "spear_linear_debug_set"):
        getattr(L, name).restype = c_int
    _lib = L
    return L


def status_string(s: int) -> str:
    return load().spear_status_string(s).decode()


def _check(status: int, what: str) -> None:
    if status != SPEAR_OK:
        raise SpearError(status, what)


def _ptr(t) -> int | None:
    return None if t is None else t.data_ptr()


def _stream(stream) -> int:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


class SpearLinear:
    """Owner of one ``spear_linear_t``.

    ``qweight`` uint8 [N][K/2], ``scales`` bf16 [N][K/G], ``zeros`` uint8
    [N][K/G] or None, ``A`` bf16 [r][K], ``B`` bf16 [N][r] (None when r = 0),
    and for the MLP gate ``W1`` bf16 [h][r], ``W2`` bf16 [r][h]: CUDA tensors
    in the layout ``spear_linear_desc_t`` documents. The library copies them;
    the tensors may be freed after construction.
    """

    def __init__(self, K, N, group_size, qweight, scales, zeros=None, A=None, B=None,
                 alpha=1.0, gate=SPEAR_GATE_SIGMOID, max_tokens=32, stream=None, W1=None, W2=None):
        L = load()
        rank = 0 if A is None else int(A.shape[0])
        hidden = 0 if W1 is None else int(W1.shape[0])
        d = spear_linear_desc_t(int(K), int(N), int(group_size), _ptr(qweight), _ptr(scales), _ptr(zeros),
                                rank, _ptr(A), _ptr(B), float(alpha), int(gate), int(max_tokens),
                                hidden, _ptr(W1), _ptr(W2))
        h = c_void_p()
        _check(L.spear_linear_create(byref(d), _stream(stream), byref(h)), "spear_linear_create")
        self.h = h
        self.K, self.N, self.rank, self.max_tokens = int(K), int(N), rank, int(max_tokens)

    @classmethod
    def grouped(cls, members, max_tokens=32, stream=None):
        """One handle for linears sharing x (spear_linear_create_grouped).
        ``members``: list of dicts with the keyword arguments of the
        constructor (K, N, group_size, qweight, scales, zeros, A, B, alpha,
        gate). y of the handle is [M][sum of the members' N]."""
        L = load()
        n = len(members)
        arr = (spear_linear_desc_t * n)()
        for i, m in enumerate(members):
            A = m.get("A")
            arr[i] = spear_linear_desc_t(int(m["K"]), int(m["N"]), int(m["group_size"]), _ptr(m["qweight"]),
                                         _ptr(m["scales"]), _ptr(m.get("zeros")), 0 if A is None else int(A.shape[0]),
                                         _ptr(A), _ptr(m.get("B")), float(m.get("alpha", 1.0)),
                                         int(m.get("gate", SPEAR_GATE_SIGMOID)), int(max_tokens), 0, None, None)
        h = c_void_p()
        _check(L.spear_linear_create_grouped(arr, n, _stream(stream), byref(h)), "spear_linear_create_grouped")
        self = cls.__new__(cls)
        self.h = h
        self.K = int(members[0]["K"])
        self.N = sum(int(m["N"]) for m in members)
        self.rank = 0 if members[0].get("A") is None else int(members[0]["A"].shape[0]) * n
        self.max_tokens = int(max_tokens)
        return self

    def _io(self, fn, x, y, M, stream, what):
        _check(fn(self.h, _ptr(x), _ptr(y), int(M), _stream(stream)), what)

    def forward_decode(self, x, y, stream=None):
        self._io(load().spear_linear_forward_decode, x, y, x.shape[0], stream, "spear_linear_forward_decode")
        return y

    def forward_prefill(self, x, y, stream=None):
        self._io(load().spear_linear_forward_prefill, x, y, x.shape[0], stream, "spear_linear_forward_prefill")
        return y

    def enable_concurrent_ec(self) -> None:
        _check(load().spear_linear_enable_concurrent_ec(self.h), "spear_linear_enable_concurrent_ec")

    def forward_prefill_concurrent(self, x, y, stream=None, ec_stream=None):
        """Prefill with the compensator pre-kernel on ec_stream (a torch stream)."""
        _check(load().spear_linear_forward_prefill_concurrent(self.h, _ptr(x), _ptr(y), int(x.shape[0]),
                                                              _stream(stream), _stream(ec_stream)),
               "spear_linear_forward_prefill_concurrent")
        return y

    def forward(self, x, y, stream=None):
        self._io(load().spear_linear_forward, x, y, x.shape[0], stream, "spear_linear_forward")
        return y

    def forward_host(self, x_host, y_host, stream=None):
        self._io(load().spear_linear_forward_host, x_host, y_host, x_host.shape[0], stream,
                 "spear_linear_forward_host")
        return y_host

    def dequantize(self, out, path=0, stream=None):
        _check(load().spear_linear_dequantize(self.h, int(path), _ptr(out), _stream(stream)),
               "spear_linear_dequantize")
        return out

    def check(self, stream=None) -> int:
        return load().spear_linear_check(self.h, _stream(stream))

    def debug_set(self, wait_ns: int = 0, skip_arrive: bool = False) -> None:
        _check(load().spear_linear_debug_set(self.h, int(wait_ns), int(bool(skip_arrive))), "spear_linear_debug_set")

    def close(self) -> None:
        if getattr(self, "h", None) and self.h.value:
            load().spear_linear_destroy(self.h)
            self.h = c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def forward_host_batch(linears, xs_host, ys_host, stream=None) -> None:
    """spear_linear_forward_host_batch over (SpearLinear, host x, host y)
    triples: the forwards in order on `stream`, the copies on the first
    handle's copy streams overlapping them, one synchronisation at the end."""
    n = len(linears)
    hs = (c_void_p * n)(*[lin.h.value for lin in linears])
    xp = (c_void_p * n)(*[x.data_ptr() for x in xs_host])
    yp = (c_void_p * n)(*[y.data_ptr() for y in ys_host])
    ms = (c_int32 * n)(*[int(x.shape[0]) for x in xs_host])
    _check(load().spear_linear_forward_host_batch(hs, xp, yp, ms, n, _stream(stream)),
           "spear_linear_forward_host_batch")


def from_weights(w, device="cuda", max_tokens=32, alpha=None, gate=None, stream=None) -> SpearLinear:
    """Build a :class:`SpearLinear` from ``workload.LinearWeights`` (host numpy)."""
    import numpy as np
    import torch

    def dev(a, dt):
        return None if a is None else torch.from_numpy(np.ascontiguousarray(a)).view(dt).to(device)

    sp = w.spec
    q = dev(w.q, torch.uint8)
    s = dev(w.s.view(np.int16), torch.bfloat16)
    z = dev(w.z, torch.uint8)
    A = dev(w.A.view(np.int16), torch.bfloat16) if sp.rank else None
    B = dev(w.B.view(np.int16), torch.bfloat16) if sp.rank else None
    W1 = dev(w.W1.view(np.int16), torch.bfloat16) if getattr(w, "W1", None) is not None else None
    W2 = dev(w.W2.view(np.int16), torch.bfloat16) if getattr(w, "W2", None) is not None else None
    lin = SpearLinear(sp.K, sp.N, sp.group_size, q, s, z, A, B,
                      sp.alpha if alpha is None else alpha, sp.gate if gate is None else gate,
                      max_tokens, stream, W1, W2)
    return lin


def grouped_from_weights(ws, device="cuda", max_tokens=32, stream=None) -> SpearLinear:
    """A grouped :class:`SpearLinear` from several ``workload.LinearWeights``
    sharing K (host numpy); member i's outputs are columns
    [N_0 + ... + N_{i-1}, + N_i) of y."""
    import numpy as np
    import torch

    def dev(a, dt):
        return None if a is None else torch.from_numpy(np.ascontiguousarray(a)).view(dt).to(device)

    members, keep = [], []
    for w in ws:
        sp = w.spec
        m = {"K": sp.K, "N": sp.N, "group_size": sp.group_size, "qweight": dev(w.q, torch.uint8),
             "scales": dev(w.s.view(np.int16), torch.bfloat16), "zeros": dev(w.z, torch.uint8),
             "A": dev(w.A.view(np.int16), torch.bfloat16) if sp.rank else None,
             "B": dev(w.B.view(np.int16), torch.bfloat16) if sp.rank else None,
             "alpha": sp.alpha, "gate": sp.gate}
        members.append(m)
    return SpearLinear.grouped(members, max_tokens=max_tokens, stream=stream)


def quantize_rtn(w, group_size=128, stream=None):
    """RTN 4-bit quantisation of a CUDA fp32 tensor w [N][K] by the library's
    kernel: returns (qweight uint8 [N][K/2], scales bf16 [N][K/G], zeros uint8
    [N][K/G]) in the layout :class:`SpearLinear` takes."""
    import torch
    N, K = w.shape
    G = K if group_size == 0 else group_size
    w = w.contiguous()
    q = torch.empty((N, K // 2), dtype=torch.uint8, device=w.device)
    s = torch.empty((N, K // G), dtype=torch.bfloat16, device=w.device)
    z = torch.empty((N, K // G), dtype=torch.uint8, device=w.device)
    _check(load().spear_quantize_rtn(_ptr(w), int(N), int(K), int(group_size), _ptr(q), _ptr(s), _ptr(z),
                                     _stream(stream)), "spear_quantize_rtn")
    return q, s, z


DECODE_SCHEDULE_FIELDS = ("grid", "P", "NW", "T", "MT", "KW", "KC", "NS", "stage_bytes", "smem", "n_stages",
                          "threads", "bytes_x")


def decode_schedule(N: int, K: int, M: int, sm_count: int, rank_b: int = 0, n_members: int = 1,
                    group_size: int = 128, gate_hidden: int = 0) -> dict:
    """The decode launch plan for a handle of this shape (host only, no GPU):
    the fields of ``DECODE_SCHEDULE_FIELDS``."""
    L = load()
    info = (ctypes.c_int32 * len(DECODE_SCHEDULE_FIELDS))()
    _check(L.spear_decode_schedule(N, K, rank_b, n_members, group_size, gate_hidden, M, sm_count, info),
           "spear_decode_schedule")
    return dict(zip(DECODE_SCHEDULE_FIELDS, list(info)))


PREFILL_SCHEDULE_FIELDS = ("mode", "G", "TN", "kpt", "tail", "units", "pro_items", "pro_d", "NS",
                           "stage_bytes", "smem", "pre_ctas", "tmem_a", "max_contrib")


def prefill_schedule(N: int, K: int, rank: int, M: int, sm_count: int, gate_hidden: int = 0,
                     with_workspace: bool = True) -> dict:
    """The prefill launch plan for a layer of this shape (host only, no GPU):
    the fields of ``PREFILL_SCHEDULE_FIELDS`` plus ``starts``, the first unit
    of each main-kernel CTA's range (G + 1 entries)."""
    L = load()
    info = (ctypes.c_int32 * len(PREFILL_SCHEDULE_FIELDS))()
    _check(L.spear_prefill_schedule(N, K, rank, gate_hidden, M, sm_count, int(with_workspace), info, None, 0),
           "spear_prefill_schedule")
    out = dict(zip(PREFILL_SCHEDULE_FIELDS, list(info)))
    starts = (ctypes.c_uint32 * (out["G"] + 1))()
    _check(L.spear_prefill_schedule(N, K, rank, gate_hidden, M, sm_count, int(with_workspace), info, starts,
                                    out["G"] + 1), "spear_prefill_schedule")
    out["starts"] = list(starts)
    return out


class ChunkScheduler:
    """Owner of one ``spear_sched_t`` (host only): a latency table of measured
    step times over (compensator density, tokens per step)."""

    def __init__(self, densities, tokens, ms):
        import numpy as np
        self._d = np.ascontiguousarray(densities, dtype=np.float64)
        self._t = np.ascontiguousarray(tokens, dtype=np.int32)
        self._ms = np.ascontiguousarray(ms, dtype=np.float64)
        if self._ms.shape != (self._d.size, self._t.size):
            raise ValueError("ms must be [len(densities)][len(tokens)]")
        h = c_void_p()
        _check(load().spear_sched_create(self._d.ctypes.data, self._d.size, self._t.ctypes.data, self._t.size,
                                         self._ms.ctypes.data, byref(h)), "spear_sched_create")
        self.h = h

    def predict(self, M: int, density: float) -> float:
        return load().spear_sched_predict(self.h, int(M), float(density))

    def pick_chunk(self, n_decode: int, density: float, itl_ms: float, candidates) -> int:
        import numpy as np
        c = np.ascontiguousarray(candidates, dtype=np.int32)
        out = c_int32()
        _check(load().spear_sched_pick_chunk(self.h, int(n_decode), float(density), float(itl_ms), c.ctypes.data,
                                             c.size, byref(out)), "spear_sched_pick_chunk")
        return int(out.value)

    def close(self):
        if getattr(self, "h", None) and self.h.value:
            load().spear_sched_destroy(self.h)
            self.h = c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
