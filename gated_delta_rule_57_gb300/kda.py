"""Thin Python binding of the KDA C ABI (``include/kda.h``).

Argument marshalling only: every step of the computation runs in the CUDA
kernels of ``libkda.so``. PyTorch provides device memory and streams. There is
no CPU fallback: if the library is missing or a tensor is not on a CUDA
device, the call raises.
"""
from __future__ import annotations

import ctypes
import os
import re
import threading
from typing import Optional

import torch

from . import build as _build

KDA_OK = 0
KDA_ERR_INVALID_ARG = 1
KDA_ERR_UNSUPPORTED = 2
KDA_ERR_WORKSPACE = 3
KDA_ERR_CUDA = 4
KDA_ERR_DECAY_RANGE = 5
KDA_ERR_NONFINITE = 6
KDA_ERR_TIMEOUT = 7

KDA_BF16 = 0
KDA_F32 = 1

KDA_DEV_DECAY_RANGE = 0x1
KDA_DEV_NONFINITE = 0x2
KDA_DEV_TIMEOUT = 0x4

_DTYPE = {torch.bfloat16: KDA_BF16, torch.float32: KDA_F32}

_lock = threading.Lock()
_lib = None


class KdaError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__(what)


def header_functions():
    """Names of the functions declared in include/kda.h."""
    with open(os.path.join(_build.INCLUDE, "kda.h")) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return re.findall(r"\b(kda_\w+)\s*\(", text)


def lib(build_if_missing: bool = True) -> ctypes.CDLL:
    """Load libkda.so (building it first when it is missing or stale)."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.LIB_PATH
            if build_if_missing and _build.is_stale():
                _build.build()
            if not os.path.exists(path):
                raise RuntimeError(f"KDA CUDA library not built: {path} is missing")
            L = ctypes.CDLL(path)
            vp, I, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
            L.kda_abi_version.argtypes = []
            L.kda_abi_version.restype = I
            L.kda_status_string.argtypes = [I]
            L.kda_status_string.restype = ctypes.c_char_p
            L.kda_last_error_string.argtypes = []
            L.kda_last_error_string.restype = ctypes.c_char_p
            L.kda_chunk_fwd_workspace_size.argtypes = [I, I, I, I, I, I]
            L.kda_chunk_fwd_workspace_size.restype = sz
            L.kda_chunk_fwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, I, I, I, I, I, I, vp,
                                        sz, vp, vp]
            L.kda_chunk_fwd.restype = I
            L.kda_chunk_fwd_ckpt.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, I, I, I, I, I, I,
                                             I, vp, vp]
            L.kda_chunk_fwd_ckpt.restype = I
            L.kda_chunk_fwd_segmented.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, I, I, I, I, I,
                                                  I, I, I, vp, sz, vp, vp]
            L.kda_chunk_fwd_segmented.restype = I
            L.kda_chunk_fwd_segmented_workspace_size.argtypes = [I, I, I, I, I, I, I]
            L.kda_chunk_fwd_segmented_workspace_size.restype = sz
            L.kda_chunk_fwd_segmented_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, I, I,
                                                          I, I, I, I, I, I, vp, vp]
            L.kda_chunk_fwd_segmented_noalloc.restype = I
            L.kda_selftest_wait_timeout.argtypes = [ctypes.c_longlong, vp, vp]
            L.kda_selftest_wait_timeout.restype = I
            L.kda_chunk_fwd_segments_hint.argtypes = [I, I, I, I, I, I]
            L.kda_chunk_fwd_segments_hint.restype = I
            L.kda_chunk_fwd_segment_plan.argtypes = [I, I, I, I, I, I, I, I, ctypes.POINTER(I),
                                                     ctypes.POINTER(I)]
            L.kda_chunk_fwd_segment_plan.restype = I
            L.kda_chunk_fwd_segments_hint_decay.argtypes = [I, I, I, I, I, I,
                                                            ctypes.POINTER(ctypes.c_float), I,
                                                            ctypes.POINTER(I)]
            L.kda_chunk_fwd_segments_hint_decay.restype = I
            L.kda_chunk_fwd_decay_probe.argtypes = [vp, I, I, I, I, I, vp, vp]
            L.kda_chunk_fwd_decay_probe.restype = I
            L.kda_chunk_fwd_slice_transition.argtypes = [vp, vp, vp, vp, vp, I, I, I, I, I, vp,
                                                         vp]
            L.kda_chunk_fwd_slice_transition.restype = I
            L.kda_chunk_fwd_slice_correct.argtypes = [vp, vp, vp, vp, vp, vp, I, I, I, I, I, I, vp,
                                                      vp]
            L.kda_chunk_fwd_slice_correct.restype = I
            L.kda_state_scan.argtypes = [vp, vp, vp, vp, I, I, I, I, I, vp]
            L.kda_state_scan.restype = I
            L.kda_decode_step.argtypes = [vp, vp, vp, vp, vp, vp, vp, I, I, I, I, I, vp, vp]
            L.kda_decode_step.restype = I
            L.kda_decode_multi.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, I, I, I, I, I, I, I,
                                           vp, vp]
            L.kda_decode_multi.restype = I
            _lib = L
    return _lib


def status_string(code: int) -> str:
    return lib().kda_status_string(code).decode()


def _check(code: int):
    if code != KDA_OK:
        L = lib()
        raise KdaError(code, f"{status_string(code)}: {L.kda_last_error_string().decode()}")


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("KDA tensors must live on a CUDA device")
    if not t.is_contiguous():
        raise ValueError("KDA tensors must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def kda_chunk_fwd_workspace_size(B: int, T: int, H: int, dk: int, dv: int,
                                 io: torch.dtype = torch.bfloat16) -> int:
    n = lib().kda_chunk_fwd_workspace_size(B, T, H, dk, dv, _DTYPE[io])
    if n == ctypes.c_size_t(-1).value:
        raise KdaError(KDA_ERR_INVALID_ARG, "unsupported problem size")
    return int(n)


def kda_chunk_fwd(q, k, v, g, beta, h0=None, *, o=None, hT=None, want_hT: bool = True,
                  status: Optional[torch.Tensor] = None, workspace=None, stream=None):
    """KDA chunked forward. q, k, g: [B,T,H,dk]; v: [B,T,H,dv]; beta: [B,T,H].

    Returns (o, hT); hT is None when want_hT is False and no hT is given.
    `status` (a CUDA int32 tensor with one element) receives the OR of the
    KDA_DEV_* flags.
    """
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    io = _DTYPE.get(q.dtype)
    if io is None:
        raise TypeError(f"unsupported q dtype {q.dtype}")
    if o is None:
        o = torch.empty((B, T, H, dv), dtype=q.dtype, device=q.device)
    if hT is None and want_hT:
        hT = torch.empty((B, H, dk, dv), dtype=torch.float32, device=q.device)
    need = kda_chunk_fwd_workspace_size(B, T, H, dk, dv, q.dtype)
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    code = lib().kda_chunk_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(h0),
                               _ptr(o), _ptr(hT), B, T, H, dk, dv, io, _ptr(workspace),
                               ws_bytes, _ptr(status), _stream(stream))
    _check(code)
    return o, hT


def kda_chunk_fwd_segments_hint(B: int, T: int, H: int, dk: int, dv: int,
                                io: torch.dtype = torch.bfloat16) -> int:
    """Recommended segment count for kda_chunk_fwd_segmented on this device."""
    n = lib().kda_chunk_fwd_segments_hint(B, T, H, dk, dv, _DTYPE[io])
    if n < 0:
        raise KdaError(KDA_ERR_INVALID_ARG, "unsupported problem size")
    return int(n)


def kda_chunk_fwd_decay_probe(g, nsample: int = 16, out=None, stream=None):
    """Sampled decay statistic of g [B,T,H,dk] for kda_chunk_fwd_segments_hint_decay:
    a [B, nsample, H] fp32 device tensor (per head, the sum over a sampled
    chunk's tokens of the max over channels of g). The default sample is the
    one kda_chunk_fwd_segmented with nseg = 0 takes on the device, so the host
    planner then picks the same split."""
    B, T, H, dk = g.shape
    if out is None:
        out = torch.empty((B, nsample, H), dtype=torch.float32, device=g.device)
    _check(lib().kda_chunk_fwd_decay_probe(_ptr(g), B, T, H, dk, nsample, _ptr(out),
                                           _stream(stream)))
    return out


def kda_chunk_fwd_segments_hint_decay(B: int, T: int, H: int, dk: int, dv: int,
                                      io: torch.dtype = torch.bfloat16, probe=None):
    """(nseg, lead) for kda_chunk_fwd_segmented, planned with the decay
    statistic `probe` (kda_chunk_fwd_decay_probe's output; a device tensor is
    copied to the host first, which waits for it)."""
    p = torch.as_tensor(probe if probe is not None else [], dtype=torch.float32)
    p = p.detach().to("cpu").contiguous().reshape(-1)
    ld = ctypes.c_int(1)
    n = lib().kda_chunk_fwd_segments_hint_decay(
        B, T, H, dk, dv, _DTYPE[io],
        ctypes.cast(p.data_ptr(), ctypes.POINTER(ctypes.c_float)) if p.numel() else None,
        p.numel(), ctypes.byref(ld))
    if n < 0:
        raise KdaError(KDA_ERR_INVALID_ARG, "unsupported problem size")
    return int(n), int(ld.value)


def kda_chunk_fwd_segment_plan(B: int, T: int, H: int, dk: int, dv: int,
                               io: torch.dtype = torch.bfloat16, nseg: int = 1,
                               lead: Optional[int] = None):
    """The split kda_chunk_fwd_segmented uses for nseg (and lead; None: the
    library's choice) on this device: (segments, seg_chunks, lead). Segment 0
    spans lead * seg_chunks 64-token chunks, each later segment seg_chunks
    (the last may be shorter)."""
    sc, ld = ctypes.c_int(0), ctypes.c_int(0)
    n = lib().kda_chunk_fwd_segment_plan(B, T, H, dk, dv, _DTYPE[io], nseg,
                                         0 if lead is None else lead, ctypes.byref(sc),
                                         ctypes.byref(ld))
    if n < 0:
        raise KdaError(KDA_ERR_INVALID_ARG, "unsupported problem size or nseg")
    return int(n), int(sc.value), int(ld.value)


def kda_chunk_fwd_segmented_workspace_size(B: int, T: int, H: int, dk: int, dv: int,
                                           io: torch.dtype = torch.bfloat16,
                                           nseg: int = 1) -> int:
    n = lib().kda_chunk_fwd_segmented_workspace_size(B, T, H, dk, dv, _DTYPE[io], nseg)
    if n == ctypes.c_size_t(-1).value:
        raise KdaError(KDA_ERR_INVALID_ARG, "unsupported problem size or segment count")
    return int(n)


def kda_chunk_fwd_segmented(q, k, v, g, beta, h0=None, *, nseg=None,
                            lead: Optional[int] = None, o=None, hT=None, want_hT: bool = True,
                            status: Optional[torch.Tensor] = None, workspace=None, stream=None):
    """kda_chunk_fwd with each sequence split in time into `nseg` segments run
    in parallel, the first spanning `lead` segment lengths. nseg None: the
    library's shape-only hint for this device; nseg "decay" (or 0): planned
    on the device from kda_chunk_fwd_decay_probe's statistic of g (no host
    round trip; lead must be None). lead None: the library's choice for
    nseg. Returns (o, hT)."""
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    io = _DTYPE.get(q.dtype)
    if io is None:
        raise TypeError(f"unsupported q dtype {q.dtype}")
    if nseg is None:
        nseg = kda_chunk_fwd_segments_hint(B, T, H, dk, dv, q.dtype)
    elif nseg == "decay":
        nseg = 0
    if o is None:
        o = torch.empty((B, T, H, dv), dtype=q.dtype, device=q.device)
    if hT is None and want_hT:
        hT = torch.empty((B, H, dk, dv), dtype=torch.float32, device=q.device)
    need = kda_chunk_fwd_segmented_workspace_size(B, T, H, dk, dv, q.dtype, nseg)
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    code = lib().kda_chunk_fwd_segmented(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                                         _ptr(h0), _ptr(o), _ptr(hT), B, T, H, dk, dv, io, nseg,
                                         0 if lead is None else lead, _ptr(workspace), ws_bytes,
                                         _ptr(status), _stream(stream))
    _check(code)
    return o, hT


def kda_chunk_fwd_segmented_noalloc(q, k, v, g, beta, h0=None, *, nseg: int,
                                    lead: Optional[int] = None, o=None, hT=None,
                                    want_hT: bool = True, status: Optional[torch.Tensor] = None,
                                    stream=None):
    """kda_chunk_fwd_segmented with the library's static scratch (no workspace)."""
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    io = _DTYPE.get(q.dtype)
    if io is None:
        raise TypeError(f"unsupported q dtype {q.dtype}")
    if o is None:
        o = torch.empty((B, T, H, dv), dtype=q.dtype, device=q.device)
    if hT is None and want_hT:
        hT = torch.empty((B, H, dk, dv), dtype=torch.float32, device=q.device)
    code = lib().kda_chunk_fwd_segmented_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                                                 _ptr(h0), _ptr(o), _ptr(hT), B, T, H, dk, dv, io,
                                                 nseg, 0 if lead is None else lead, _ptr(status),
                                                 _stream(stream))
    _check(code)
    return o, hT


def kda_chunk_fwd_slice_transition(q, k, g, beta, *, M=None,
                                   status: Optional[torch.Tensor] = None, stream=None):
    """Transition of one time slice: M [B,H,dk,dk] = product of the slice's
    per-token transitions (the recurrence from the identity with v = 0)."""
    B, T, H, dk = q.shape
    io = _DTYPE.get(q.dtype)
    if io is None:
        raise TypeError(f"unsupported q dtype {q.dtype}")
    if M is None:
        M = torch.empty((B, H, dk, dk), dtype=torch.float32, device=q.device)
    _check(lib().kda_chunk_fwd_slice_transition(_ptr(q), _ptr(k), _ptr(g), _ptr(beta), _ptr(M),
                                                B, T, H, dk, io, _ptr(status), _stream(stream)))
    return M


def kda_chunk_fwd_slice_correct(q, k, g, beta, S_in, o, *,
                                status: Optional[torch.Tensor] = None, stream=None):
    """o += the outputs the incoming state S_in [B,H,dk,dv] contributes over
    the slice (the recurrence from S_in with v = 0). Returns o."""
    B, T, H, dk = q.shape
    dv = o.shape[-1]
    io = _DTYPE.get(q.dtype)
    if io is None:
        raise TypeError(f"unsupported q dtype {q.dtype}")
    _check(lib().kda_chunk_fwd_slice_correct(_ptr(q), _ptr(k), _ptr(g), _ptr(beta), _ptr(S_in),
                                             _ptr(o), B, T, H, dk, dv, io, _ptr(status),
                                             _stream(stream)))
    return o


def kda_state_scan(s0, m=None, *, x_in=None, hT=None, want_hT: bool = True, stream=None):
    """Prefix scan over slice summaries: s0 [n,B,H,dk,dv] (zero-start final
    states; slice 0's from the true initial state), m [n-1,B,H,dk,dk]
    (transitions of slices 1..). Returns (x_in [n-1,B,H,dk,dv] incoming
    states of slices 1.., hT [B,H,dk,dv])."""
    n, B, H, dk, dv = s0.shape
    if x_in is None and n > 1:
        x_in = torch.empty((n - 1, B, H, dk, dv), dtype=torch.float32, device=s0.device)
    if hT is None and want_hT:
        hT = torch.empty((B, H, dk, dv), dtype=torch.float32, device=s0.device)
    _check(lib().kda_state_scan(_ptr(s0), _ptr(m), _ptr(x_in), _ptr(hT), n, B, H, dk, dv,
                                _stream(stream)))
    return x_in, hT


def kda_selftest_wait_timeout(status: torch.Tensor, clocks: int = 1 << 20, stream=None):
    """Run the bounded-wait self-test: `status` (CUDA int32, one element)
    receives KDA_DEV_TIMEOUT when the wait gives up."""
    _check(lib().kda_selftest_wait_timeout(clocks, _ptr(status), _stream(stream)))


def kda_chunk_fwd_ckpt(q, k, v, g, beta, h0=None, *, ckpt_every: int, o=None, hT=None,
                       ckpt=None, want_hT: bool = True, status: Optional[torch.Tensor] = None,
                       stream=None):
    """kda_chunk_fwd that also returns the state every `ckpt_every` tokens.

    Returns (o, hT, ckpt) with ckpt [B, H, T // ckpt_every, dk, dv] fp32.
    """
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    io = _DTYPE.get(q.dtype)
    if io is None:
        raise TypeError(f"unsupported q dtype {q.dtype}")
    if o is None:
        o = torch.empty((B, T, H, dv), dtype=q.dtype, device=q.device)
    if hT is None and want_hT:
        hT = torch.empty((B, H, dk, dv), dtype=torch.float32, device=q.device)
    if ckpt is None:
        n = T // ckpt_every if ckpt_every > 0 else 0
        ckpt = torch.empty((B, H, max(n, 0), dk, dv), dtype=torch.float32, device=q.device)
    code = lib().kda_chunk_fwd_ckpt(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(h0),
                                    _ptr(o), _ptr(hT), _ptr(ckpt), int(ckpt_every), B, T, H, dk,
                                    dv, io, _ptr(status), _stream(stream))
    _check(code)
    return o, hT, ckpt


def kda_decode_step(q, k, v, g, beta, S, *, o=None, status: Optional[torch.Tensor] = None,
                    stream=None):
    """One in-place decode step. q, k, g: [N,H,dk]; v: [N,H,dv]; beta: [N,H];
    S: [N,H,dk,dv] fp32 (updated in place). Returns o [N,H,dv]."""
    N, H, dk = q.shape
    dv = v.shape[-1]
    io = _DTYPE.get(q.dtype)
    if io is None:
        raise TypeError(f"unsupported q dtype {q.dtype}")
    if o is None:
        o = torch.empty((N, H, dv), dtype=q.dtype, device=q.device)
    code = lib().kda_decode_step(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(S),
                                 _ptr(o), N, H, dk, dv, io, _ptr(status), _stream(stream))
    _check(code)
    return o


def kda_decode_multi(q, k, v, g, beta, S, *, ntok: Optional[torch.Tensor] = None,
                     commit: bool = False, o=None, want_o: bool = True,
                     status: Optional[torch.Tensor] = None, stream=None):
    """K cached tokens per sequence in one pass (speculative decoding).

    q, k, g: [N,K,H,dk]; v: [N,K,H,dv]; beta: [N,K,H]; S: [N,H,dk,dv] fp32.
    commit=False (verify): returns o [N,K,H,dv]; S is not modified.
    commit=True: S is advanced in place by ntok[n] tokens (int32 CUDA tensor
    [N], or all K when None); o is returned when want_o.
    """
    N, K, H, dk = q.shape
    dv = v.shape[-1]
    io = _DTYPE.get(q.dtype)
    if io is None:
        raise TypeError(f"unsupported q dtype {q.dtype}")
    if ntok is not None and (ntok.dtype != torch.int32 or ntok.numel() != N):
        raise ValueError("ntok must be an int32 tensor with N entries")
    if o is None and (want_o or not commit):
        o = torch.empty((N, K, H, dv), dtype=q.dtype, device=q.device)
    code = lib().kda_decode_multi(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(S),
                                  _ptr(o), _ptr(ntok), N, K, H, dk, dv, io, int(bool(commit)),
                                  _ptr(status), _stream(stream))
    _check(code)
    return o
