"""Pins for the fp64 oracle, each against something other than the oracle itself.

The oracle evaluates the KDA recurrence token by token with a rank-1 update
(see oracle/kda_oracle.c). These tests hold it to:
  - brute force: explicit dense transition matrices M_t = (I - b k k^T) Diag(e^g)
    and the unrolled sum S_t = (prod M) h0 + sum_s (prod_{r>s} M_r) b_s k_s v_s^T;
  - closed forms (beta = 0: pure per-channel decay; g = 0, beta = 1 with
    orthonormal keys: exact overwrite of a key's value);
  - structural identities (linearity in (v, h0), chaining through hT -> h0,
    composition of segment summaries, decode = one prefill token);
  - the numbers printed on the orkas.ai page "Kimi K3 architecture", section
    "A lower bound that deleted a GPU code path" (tests/golden/decay_bound.json);
  - mutants: plausible one-token mistakes planted in a copy of the oracle
    source must each fail the brute-force pin.
"""
import json
import math
import os
import re
import shutil
import subprocess

import numpy as np
import pytest
import torch

import oracle
from gated_delta_rule_57_gb300 import inputs

HERE = os.path.dirname(os.path.abspath(__file__))


def rand_case(seed, B, T, H, dk, dv, *, with_h0=True, g_lo=-5.0):
    rng = np.random.default_rng(seed)
    f = lambda *s: rng.standard_normal(s).astype(np.float32)  # noqa: E731
    q, k, v = f(B, T, H, dk), f(B, T, H, dk) * 0.5, f(B, T, H, dv)
    g = rng.uniform(g_lo, 0.0, (B, T, H, dk)).astype(np.float32)
    beta = rng.uniform(0.0, 1.0, (B, T, H)).astype(np.float32)
    h0 = f(B, H, dk, dv) * 0.5 if with_h0 else None
    return q, k, v, g, beta, h0


def brute_force(q, k, v, g, beta, h0):
    """Unrolled products of dense transition matrices (no token loop state)."""
    q, k, v, g, beta = (np.asarray(x, np.float64) for x in (q, k, v, g, beta))
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    o = np.zeros((B, T, H, dv))
    hT = np.zeros((B, H, dk, dv))
    for b in range(B):
        for h in range(H):
            S0 = np.zeros((dk, dv)) if h0 is None else np.asarray(h0[b, h], np.float64)
            M = [(np.eye(dk) - beta[b, t, h] * np.outer(k[b, t, h], k[b, t, h]))
                 @ np.diag(np.exp(g[b, t, h])) for t in range(T)]
            D = [beta[b, t, h] * np.outer(k[b, t, h], v[b, t, h]) for t in range(T)]
            S = S0
            for t in range(T):
                prod = np.eye(dk)
                S = np.zeros((dk, dv))
                for s in range(t, -1, -1):
                    S = S + prod @ D[s]
                    prod = prod @ M[s]
                S = S + prod @ S0
                o[b, t, h] = S.T @ q[b, t, h]
            hT[b, h] = S
    return o, hT


def rel_max(a, b):
    return np.abs(a - b).max() / max(np.abs(b).max(), 1e-300)


@pytest.mark.parametrize("shape", [(1, 12, 2, 8, 8), (2, 7, 1, 4, 6), (1, 1, 1, 3, 5),
                                   (1, 9, 3, 6, 2)])
@pytest.mark.parametrize("with_h0", [True, False])
def test_brute_force(shape, with_h0):
    case = rand_case(sum(shape) + with_h0, *shape, with_h0=with_h0)
    o, hT = oracle.prefill(*case)
    ob, hb = brute_force(*case)
    assert rel_max(o, ob) < 1e-12
    assert rel_max(hT, hb) < 1e-12


def test_beta_zero_is_pure_decay():
    q, k, v, g, beta, h0 = rand_case(3, 2, 20, 2, 8, 5)
    beta[:] = 0.0
    o, hT = oracle.prefill(q, k, v, g, beta, h0)
    Gam = np.cumsum(g.astype(np.float64), axis=1)  # [B, T, H, dk]
    for t in range(20):
        St = np.exp(Gam[:, t])[..., None] * h0.astype(np.float64)  # [B, H, dk, dv]
        ot = np.einsum("bhij,bhi->bhj", St, q[:, t].astype(np.float64))
        assert rel_max(o[:, t], ot) < 1e-12
    assert rel_max(hT, np.exp(Gam[:, -1])[..., None] * h0) < 1e-12


def _hadamard_keys():
    """8 exactly orthonormal keys (two 4x4 Hadamard blocks / 2), exact in fp32."""
    H4 = np.array([[1, 1, 1, 1], [1, -1, 1, -1], [1, 1, -1, -1], [1, -1, -1, 1]], np.float32)
    K = np.zeros((8, 8), np.float32)
    K[:4, :4] = H4 / 2
    K[4:, 4:] = H4 / 2
    return K


def test_overwrite_with_orthonormal_keys():
    """g = 0, beta = 1: writing (k, v) makes S^T k = v exactly; rewriting replaces."""
    K = _hadamard_keys()
    rng = np.random.default_rng(11)
    order = [0, 3, 5, 1, 7, 3, 0, 2]  # keys 3 and 0 are rewritten
    T = len(order)
    k = np.stack([K[i] for i in order])[None, :, None, :]
    q = k.copy()  # read back the key just written: o_t = S_t^T k_t
    v = rng.integers(-8, 8, (1, T, 1, 5)).astype(np.float32)
    g = np.zeros((1, T, 1, 8), np.float32)
    beta = np.ones((1, T, 1), np.float32)
    o, hT = oracle.prefill(q, k, v, g, beta)
    assert np.abs(o[0, :, 0] - v[0, :, 0]).max() < 1e-12
    latest = {}
    for t, i in enumerate(order):
        latest[i] = v[0, t, 0]
    S = sum(np.outer(K[i], val) for i, val in latest.items())
    assert np.abs(hT[0, 0] - S).max() < 1e-12
    # keys never written read back zero
    for i in set(range(8)) - set(order):
        assert np.abs(hT[0, 0].T @ K[i]).max() < 1e-12


def test_linear_in_v_and_h0():
    q, k, v1, g, beta, h1 = rand_case(5, 1, 16, 2, 6, 4)
    rng = np.random.default_rng(6)
    # dyadic values keep v1 + v2 and h1 + h2 exact in fp32
    v1 = (rng.integers(-64, 64, v1.shape) / 32).astype(np.float32)
    v2 = (rng.integers(-64, 64, v1.shape) / 32).astype(np.float32)
    h1 = (rng.integers(-64, 64, h1.shape) / 32).astype(np.float32)
    h2 = (rng.integers(-64, 64, h1.shape) / 32).astype(np.float32)
    oa, ha = oracle.prefill(q, k, v1, g, beta, h1)
    ob, hb = oracle.prefill(q, k, v2, g, beta, h2)
    oc, hc = oracle.prefill(q, k, v1 + v2, g, beta, h1 + h2)
    assert rel_max(oc, oa + ob) < 1e-12
    assert rel_max(hc, ha + hb) < 1e-12


def test_chaining_through_state():
    q, k, v, g, beta, h0 = rand_case(7, 2, 30, 2, 8, 8)
    o, hT = oracle.prefill(q, k, v, g, beta, h0)
    T1 = 13
    o1, h1 = oracle.prefill(q[:, :T1], k[:, :T1], v[:, :T1], g[:, :T1], beta[:, :T1], h0)
    # the intermediate state crosses the interface as fp32, as on the GPU
    o2, h2 = oracle.prefill(q[:, T1:], k[:, T1:], v[:, T1:], g[:, T1:], beta[:, T1:],
                            h1.astype(np.float32))
    assert rel_max(np.concatenate([o1, o2], axis=1), o) < 1e-6
    assert rel_max(h2, hT) < 1e-6


def test_segment_composition():
    """Two segments compose as (transition, zero-start state) pairs: the
    sequence-split scheme of section "The bill arrives in the serving stack"."""
    q, k, v, g, beta, h0 = rand_case(8, 1, 24, 1, 6, 5)
    _, hT = oracle.prefill(q, k, v, g, beta, h0)
    T1 = 10
    _, h1 = oracle.prefill(q[:, :T1], k[:, :T1], v[:, :T1], g[:, :T1], beta[:, :T1], h0)
    _, s2 = oracle.prefill(q[:, T1:], k[:, T1:], v[:, T1:], g[:, T1:], beta[:, T1:], None)
    M = np.eye(6)
    for t in range(T1, 24):
        kt = k[0, t, 0].astype(np.float64)
        M = (np.eye(6) - beta[0, t, 0] * np.outer(kt, kt)) @ np.diag(np.exp(g[0, t, 0].astype(np.float64))) @ M
    assert rel_max(M @ h1[0, 0] + s2[0, 0], hT[0, 0]) < 1e-12


def test_decode_equals_one_prefill_token():
    q, k, v, g, beta, h0 = rand_case(9, 3, 1, 2, 8, 8)
    o, hT = oracle.prefill(q, k, v, g, beta, h0)
    od, Sd = oracle.decode(q[:, 0], k[:, 0], v[:, 0], g[:, 0], beta[:, 0], h0)
    assert np.abs(od - o[:, 0]).max() == 0.0
    assert np.abs(Sd - hT).max() == 0.0


def test_reads_exact_bf16_bytes():
    q, k, v, g, beta, h0 = rand_case(10, 1, 9, 2, 8, 8)
    qb, kb, vb = (torch.from_numpy(x).to(torch.bfloat16) for x in (q, k, v))
    o1, h1 = oracle.prefill(qb, kb, vb, g, beta, h0)
    o2, h2 = oracle.prefill(qb.float(), kb.float(), vb.float(), g, beta, h0)
    assert np.array_equal(o1, o2) and np.array_equal(h1, h2)


def test_page_numbers_golden():
    with open(os.path.join(HERE, "golden", "decay_bound.json")) as f:
        facts = json.load(f)["facts"]
    g_min = -5.0
    assert round(100 * math.exp(g_min), 2) == facts["retained_per_step_percent"]
    lo, hi = facts["tile_log_decay_interval"]
    assert facts["tile_tokens"] * g_min == lo and hi == 0
    assert float(f"{math.exp(-lo):.1e}") == facts["reciprocal_bound"]
    bf16_max = float(torch.finfo(torch.bfloat16).max)
    assert float(f"{bf16_max:.1e}") == facts["bf16_max"]
    assert math.exp(-lo) < bf16_max


@pytest.mark.parametrize("w", [inputs.TINY_F32, inputs.PREFILL_T4K, inputs.PREFILL_B8_T8K])
def test_generated_decay_respects_tile_bound(w):
    """Every 16-token window of generated g sums above -80, so e^{-sum} < bf16 max."""
    x = inputs.prefill_inputs(w, B=1, T=min(w.T, 512), H=min(w.H, 32))
    g = x["g"].double()
    assert float(g.max()) <= 0.0 and float(g.min()) >= -5.0
    win = g.unfold(1, 16, 1).sum(-1)  # [B, T-15, H, dk]
    assert float(win.min()) > -80.0
    bf16_max = float(torch.finfo(torch.bfloat16).max)
    assert math.exp(-float(win.min())) < bf16_max


MUTANTS = [
    ("dropped decay", "double a = exp(gi[i]);", "double a = 1.0;"),
    ("decay index", "double a = exp(gi[i]);", "double a = exp(gi[0]);"),
    ("wrong sign", "u[j] = beta * (vi[j] - kv[j]);", "u[j] = beta * (vi[j] + kv[j]);"),
    ("dropped beta", "u[j] = beta * (vi[j] - kv[j]);", "u[j] = (vi[j] - kv[j]);"),
    ("read before write", "/* o_t = S_t^T q_t */", "/* o_t = S_t^T q_t */ for (i = 0; i < dk; i++) { double* rr = S + i * dv; for (j = 0; j < dv; j++) rr[j] -= ki[i] * u[j]; }"),
    ("key for query", "double qq = qi[i];", "double qq = ki[i];"),
    ("transposed update", "row[j] += kk * u[j];", "row[j] += ki[j % dk] * u[i % dv];"),
]


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutants_fail_brute_force(tmp_path, name, old, new):
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    src = open(os.path.join(os.path.dirname(oracle.__file__), "kda_oracle.c")).read()
    assert src.count(old) >= 1, name
    mut = src.replace(old, new, 1)
    (tmp_path / "kda_oracle.c").write_text(mut)
    so = tmp_path / "libmut.so"
    subprocess.run(["gcc", "-O1", "-std=c99", "-fPIC", "-shared", "-fopenmp", "-o", str(so),
                    str(tmp_path / "kda_oracle.c"), "-lm"], check=True)
    import ctypes
    lib = ctypes.CDLL(str(so))
    vp, L, I = ctypes.c_void_p, ctypes.c_long, ctypes.c_int
    lib.kda_oracle_prefill.argtypes = [vp] * 3 + [I] + [vp] * 5 + [L] * 5 + [I]
    q, k, v, g, beta, h0 = rand_case(21, 1, 8, 1, 6, 6)
    o = np.empty((1, 8, 1, 6))
    hT = np.empty((1, 1, 6, 6))
    p = lambda a: a.ctypes.data_as(vp)  # noqa: E731
    lib.kda_oracle_prefill(p(q), p(k), p(v), 0, p(g), p(beta), p(h0), p(o), p(hT), 1, 8, 1,
                           6, 6, 1)
    ob, hb = brute_force(q, k, v, g, beta, h0)
    assert rel_max(o, ob) > 1e-6 or rel_max(hT, hb) > 1e-6, f"mutant '{name}' survived"
