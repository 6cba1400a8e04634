"""Parity helpers shared by the GPU tests.

Tolerances (max-abs error relative to the largest reference magnitude over the
whole tensor; Frobenius for states):
  o,  bf16 I/O : max|o - o_ref| <= 2e-2 * max|o_ref|
  o,  fp32 I/O : max|o - o_ref| <= 1e-4 * max|o_ref|
  hT / S       : ||S - S_ref||_F <= 1e-2 * ||S_ref||_F (bf16 I/O), 1e-4 (fp32 I/O)
"""
import numpy as np
import torch

O_TOL = {torch.bfloat16: 2e-2, torch.float32: 1e-4}
S_TOL = {torch.bfloat16: 1e-2, torch.float32: 1e-4}


def to_np64(t):
    return t.detach().to("cpu", torch.float64).numpy()


def o_err(o_gpu, o_ref):
    o = to_np64(o_gpu)
    scale = max(np.abs(o_ref).max(), 1e-30)
    return float(np.abs(o - o_ref).max() / scale)


def s_err(s_gpu, s_ref):
    s = to_np64(s_gpu)
    return float(np.linalg.norm((s - s_ref).ravel()) / max(np.linalg.norm(s_ref.ravel()), 1e-30))


def assert_o(o_gpu, o_ref, dtype, what="o"):
    e = o_err(o_gpu, o_ref)
    assert np.isfinite(e) and e <= O_TOL[dtype], f"{what}: rel max err {e:.3e} > {O_TOL[dtype]}"
    return e


def assert_s(s_gpu, s_ref, dtype, what="hT"):
    e = s_err(s_gpu, s_ref)
    assert np.isfinite(e) and e <= S_TOL[dtype], f"{what}: rel Frobenius err {e:.3e} > {S_TOL[dtype]}"
    return e
