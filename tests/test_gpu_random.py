"""Randomised parity sweep: shapes drawn from a fixed seed, every path checked
against the fp64 oracle on the same inputs.

Each case draws a batch, a length (ragged or whole chunks), a head count and
an I/O type, then runs the call the shape selects (the tensor-core or fp32
path, the balanced schedule when the sequences outnumber the SMs, a time
split with a drawn segment count and first-segment length, a multi-token
verify and commit with drawn accepted lengths) and compares o and the final
state with the oracle's.
"""
import random

import pytest
import torch

import oracle
from gated_delta_rule_57_gb300 import inputs, kda
from helpers import assert_o, assert_s

pytestmark = pytest.mark.gpu
DEV = "cuda"


def draw(B, T, H, d, io, seed, h0):
    w = inputs.PrefillWorkload("random", B, T, H, d, d, io, seed,
                               h0_std=0.02 if h0 else None)
    return inputs.prefill_inputs(w, DEV)


def reference(x, **kw):
    xc = {n: (t.cpu() if t is not None else None) for n, t in x.items()}
    return oracle.prefill(xc["q"], xc["k"], xc["v"], xc["g"], xc["beta"], xc["h0"], **kw)


def cases(kind, n, seed):
    rng = random.Random(seed)
    out = []
    for i in range(n):
        if kind == "prefill":
            io, d = rng.choice([("bf16", 128), ("bf16", 64), ("f32", 64), ("f32", 128)])
            out.append((rng.randint(1, 3), rng.randint(1, 700), rng.randint(1, 5), d, io,
                        rng.random() < 0.5, 1000 + i))
        elif kind == "balanced":
            out.append((2, rng.randint(60, 420), rng.randint(77, 110), 128, "bf16",
                        rng.random() < 0.5, 2000 + i))
        elif kind == "segmented":
            T = rng.randint(129, 1500)
            nch = (T + 63) // 64
            out.append((rng.randint(1, 2), T, rng.randint(1, 4), rng.randint(2, nch),
                        rng.randint(0, min(4, nch)), rng.random() < 0.5, 3000 + i))
        else:
            io, d = rng.choice([("bf16", 128), ("f32", 128), ("bf16", 64), ("f32", 64)])
            out.append((rng.randint(1, 6), rng.randint(1, 10), rng.randint(1, 4), d, io,
                        4000 + i))
    return out


@pytest.mark.parametrize("B,T,H,d,io,h0,seed", cases("prefill", 10, 7))
def test_random_prefill(B, T, H, d, io, h0, seed):
    x = draw(B, T, H, d, io, seed, h0)
    o, hT = kda.kda_chunk_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"])
    torch.cuda.synchronize()
    o_ref, h_ref = reference(x)
    dt = inputs.io_dtype(io)
    assert_o(o, o_ref, dt)
    assert_s(hT, h_ref, dt)


@pytest.mark.parametrize("B,T,H,d,io,h0,seed", cases("balanced", 3, 8))
def test_random_balanced(B, T, H, d, io, h0, seed):
    """More sequences than SMs: with the workspace the balanced schedule runs
    (where the launcher takes it), bit-identical to one CTA per sequence."""
    x = draw(B, T, H, d, io, seed, h0)
    ws = torch.zeros(kda.kda_chunk_fwd_workspace_size(B, T, H, d, d, torch.bfloat16),
                     dtype=torch.uint8, device=DEV)
    o_b, h_b = kda.kda_chunk_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"],
                                 workspace=ws)
    o_p, h_p = kda.kda_chunk_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"])
    torch.cuda.synchronize()
    assert torch.equal(o_b, o_p) and torch.equal(h_b, h_p)
    sub = slice(0, 1)  # the oracle on the first batch row
    xs = {n: (t[sub] if t is not None else None) for n, t in x.items()}
    o_ref, h_ref = reference(xs)
    assert_o(o_b[sub], o_ref, torch.bfloat16)
    assert_s(h_b[sub], h_ref, torch.bfloat16)


@pytest.mark.parametrize("B,T,H,nseg,lead,h0,seed", cases("segmented", 8, 9))
def test_random_segmented(B, T, H, nseg, lead, h0, seed):
    """A drawn segment count and first-segment length (0: the library's)."""
    x = draw(B, T, H, 128, "bf16", seed, h0)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    o, hT = kda.kda_chunk_fwd_segmented(x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"],
                                        nseg=nseg, lead=lead or None, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    o_ref, h_ref = reference(x)
    assert_o(o, o_ref, torch.bfloat16)
    assert_s(hT, h_ref, torch.bfloat16)


@pytest.mark.parametrize("N,K,H,d,io,seed", cases("multi", 8, 10))
def test_random_multi_token(N, K, H, d, io, seed):
    """Verify all K drafts, then commit drawn accepted lengths 0..K."""
    x = draw(N, K, H, d, io, seed, True)
    rng = random.Random(seed)
    acc = [rng.randint(0, K) for _ in range(N)]
    S = x["h0"].clone()
    o = kda.kda_decode_multi(x["q"], x["k"], x["v"], x["g"], x["beta"], S)
    ntok = torch.tensor(acc, dtype=torch.int32, device=DEV)
    kda.kda_decode_multi(x["q"], x["k"], x["v"], x["g"], x["beta"], S, ntok=ntok, commit=True,
                         want_o=False)
    torch.cuda.synchronize()
    dt = inputs.io_dtype(io)
    o_ref, _ = reference(x)
    assert_o(o, o_ref, dt, "verify")
    xc = {n: t.cpu() for n, t in x.items()}
    for n, m in enumerate(acc):
        if m == 0:
            assert torch.equal(S[n], x["h0"][n])
            continue
        sl = slice(n, n + 1)
        _, h_ref = oracle.prefill(xc["q"][sl, :m], xc["k"][sl, :m], xc["v"][sl, :m],
                                  xc["g"][sl, :m], xc["beta"][sl, :m], xc["h0"][sl])
        assert_s(S[sl], h_ref, dt, f"state after {m} of {K} drafts")
