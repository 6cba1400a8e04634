"""KDA oracle: plain fp64 CPU recurrence (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. The CUDA library never does, and this
package imports nothing from it.

The arithmetic lives in ``kda_oracle.c`` (token-by-token, fp64, OpenMP over
sequences); this module only compiles it with the host C compiler and passes
buffers to it. It reads the exact bytes handed to the GPU: bf16 tensors are
passed as their raw 16-bit words and widened exactly inside the C code.

What the recurrence is and which passages of the orkas.ai page "Kimi K3
architecture" it follows is stated in the header of ``kda_oracle.c``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kda_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libkda_oracle.so")

F32 = 0
BF16 = 1

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``kda_oracle.c`` into a shared library (gcc, -O2, OpenMP)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)) or (
        os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-fopenmp", "-Wall",
               "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            vp, dp, fp = ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p
            L, I = ctypes.c_long, ctypes.c_int
            lib.kda_oracle_prefill.argtypes = [vp, vp, vp, I, fp, fp, fp, dp, dp,
                                               L, L, L, L, L, I]
            lib.kda_oracle_prefill.restype = I
            lib.kda_oracle_decode.argtypes = [vp, vp, vp, I, fp, fp, dp, dp,
                                              L, L, L, L, I]
            lib.kda_oracle_decode.restype = I
            lib.kda_oracle_max_threads.argtypes = []
            lib.kda_oracle_max_threads.restype = I
            _lib = lib
    return _lib


def _as_raw(x):
    """Return (contiguous numpy array, dtype code) holding the exact input bytes."""
    try:
        import torch
    except ImportError:  # pragma: no cover
        torch = None
    if torch is not None and isinstance(x, torch.Tensor):
        x = x.detach().to("cpu").contiguous()
        if x.dtype == torch.bfloat16:
            return x.view(torch.int16).numpy().view(np.uint16), BF16
        if x.dtype == torch.float32:
            return x.numpy(), F32
        raise TypeError(f"unsupported tensor dtype {x.dtype}")
    x = np.ascontiguousarray(x)
    if x.dtype == np.float32:
        return x, F32
    if x.dtype == np.uint16:  # raw bf16 words
        return x, BF16
    if x.dtype == np.float64:
        # fp64 inputs are accepted for the oracle's own pins: narrowed to fp32,
        # which is the widest input type the GPU path accepts.
        return x.astype(np.float32), F32
    raise TypeError(f"unsupported array dtype {x.dtype}")


def _as_f32(x):
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach().to("cpu", torch.float32).contiguous().numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(np.asarray(x, dtype=np.float32))


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def max_threads() -> int:
    return int(_load().kda_oracle_max_threads())


def prefill(q, k, v, g, beta, h0=None, *, nthreads: int = 0, want_o: bool = True,
            want_hT: bool = True):
    """fp64 recurrence over a whole sequence batch.

    q, k, g: [B, T, H, dk]; v: [B, T, H, dv]; beta: [B, T, H]; h0: [B, H, dk, dv]
    or None (zero state). q, k, v may be bf16 or fp32 (torch) / uint16 raw bf16
    or float32 (numpy); they must share one type. g, beta, h0 are fp32.
    Returns (o [B,T,H,dv] float64 or None, hT [B,H,dk,dv] float64 or None).
    """
    qa, qt = _as_raw(q)
    ka, kt = _as_raw(k)
    va, vt = _as_raw(v)
    if not (qt == kt == vt):
        raise TypeError("q, k and v must share one element type")
    if qa.ndim != 4 or ka.shape != qa.shape:
        raise ValueError("q and k must be [B, T, H, dk]")
    B, T, H, dk = qa.shape
    if va.ndim != 4 or va.shape[:3] != (B, T, H):
        raise ValueError("v must be [B, T, H, dv]")
    dv = va.shape[3]
    ga = _as_f32(g)
    ba = _as_f32(beta)
    if ga.shape != (B, T, H, dk) or ba.shape != (B, T, H):
        raise ValueError("g must be [B, T, H, dk] and beta [B, T, H]")
    ha = None
    if h0 is not None:
        ha = _as_f32(h0)
        if ha.shape != (B, H, dk, dv):
            raise ValueError("h0 must be [B, H, dk, dv]")
    o = np.empty((B, T, H, dv), np.float64) if want_o else None
    hT = np.empty((B, H, dk, dv), np.float64) if want_hT else None
    rc = _load().kda_oracle_prefill(_ptr(qa), _ptr(ka), _ptr(va), qt, _ptr(ga), _ptr(ba),
                                    _ptr(ha), _ptr(o), _ptr(hT), B, T, H, dk, dv,
                                    int(nthreads))
    if rc != 0:
        raise RuntimeError(f"kda_oracle_prefill failed with code {rc}")
    return o, hT


def decode(q, k, v, g, beta, S, *, nthreads: int = 0):
    """One in-place decode step in fp64.

    q, k, g: [N, H, dk]; v: [N, H, dv]; beta: [N, H]; S: [N, H, dk, dv] (any
    float type; copied to fp64). Returns (o [N,H,dv] float64, S_new float64).
    """
    qa, qt = _as_raw(q)
    ka, kt = _as_raw(k)
    va, vt = _as_raw(v)
    if not (qt == kt == vt):
        raise TypeError("q, k and v must share one element type")
    N, H, dk = qa.shape
    dv = va.shape[2]
    ga = _as_f32(g)
    ba = _as_f32(beta)
    try:
        import torch
        if isinstance(S, torch.Tensor):
            S = S.detach().to("cpu", torch.float64).numpy()
    except ImportError:  # pragma: no cover
        pass
    Sa = np.array(S, dtype=np.float64, copy=True, order="C")
    if Sa.shape != (N, H, dk, dv) or ga.shape != (N, H, dk) or ba.shape != (N, H):
        raise ValueError("decode shapes do not match")
    o = np.empty((N, H, dv), np.float64)
    rc = _load().kda_oracle_decode(_ptr(qa), _ptr(ka), _ptr(va), qt, _ptr(ga), _ptr(ba),
                                   _ptr(Sa), _ptr(o), N, H, dk, dv, int(nthreads))
    if rc != 0:
        raise RuntimeError(f"kda_oracle_decode failed with code {rc}")
    return o, Sa
