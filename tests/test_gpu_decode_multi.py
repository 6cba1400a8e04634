"""Multi-token decode (speculative verify / commit) against the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
from gated_delta_rule_57_gb300 import inputs, kda
from helpers import assert_o, assert_s

pytestmark = pytest.mark.gpu
DEV = "cuda"


def draft(N, K, H, d, io, seed):
    """K draft tokens per sequence ([N, K, H, d] = the prefill layout) and a state."""
    w = inputs.PrefillWorkload("draft", N, K, H, d, d, io, seed, h0_std=0.02)
    x = inputs.prefill_inputs(w, DEV)
    return x


@pytest.mark.parametrize("io,d", [("bf16", 128), ("f32", 64), ("bf16", 64)])
def test_verify_matches_oracle_and_keeps_state(io, d):
    x = draft(6, 5, 3, d, io, 21)
    S = x["h0"].clone()
    o = kda.kda_decode_multi(x["q"], x["k"], x["v"], x["g"], x["beta"], S)
    torch.cuda.synchronize()
    assert torch.equal(S, x["h0"])  # verify never writes the state
    xc = {n: t.cpu() for n, t in x.items()}
    o_ref, _ = oracle.prefill(xc["q"], xc["k"], xc["v"], xc["g"], xc["beta"], xc["h0"])
    assert_o(o, o_ref, inputs.io_dtype(io))


@pytest.mark.parametrize("io", ["bf16", "f32"])
def test_commit_accepted_prefix(io):
    """Per-sequence accepted lengths 0..K rebuild the state of that prefix."""
    N, K, H, d = 6, 5, 2, 128
    x = draft(N, K, H, d, io, 22)
    ntok = torch.tensor([0, 1, 2, 3, 5, 9], dtype=torch.int32, device=DEV)  # 9 clamps to K
    S = x["h0"].clone()
    kda.kda_decode_multi(x["q"], x["k"], x["v"], x["g"], x["beta"], S, ntok=ntok, commit=True,
                         want_o=False)
    torch.cuda.synchronize()
    xc = {n: t.cpu() for n, t in x.items()}
    for n, m in enumerate([0, 1, 2, 3, 5, 5]):
        sl = slice(n, n + 1)
        if m == 0:
            assert torch.equal(S[n], x["h0"][n])
            continue
        _, h_ref = oracle.prefill(xc["q"][sl, :m], xc["k"][sl, :m], xc["v"][sl, :m],
                                  xc["g"][sl, :m], xc["beta"][sl, :m], xc["h0"][sl])
        assert_s(S[sl], h_ref, inputs.io_dtype(io), f"state after {m} accepted tokens")


@pytest.mark.parametrize("io", ["bf16", "f32"])
def test_long_draft_crosses_token_blocks(io):
    """K = 19 drafts (more than one block of eight): verify outputs for all of
    them, and commits of accepted prefixes that end inside, at and past a
    block boundary."""
    N, K, H, d = 6, 19, 2, 128
    x = draft(N, K, H, d, io, 27)
    S = x["h0"].clone()
    o = kda.kda_decode_multi(x["q"], x["k"], x["v"], x["g"], x["beta"], S)
    torch.cuda.synchronize()
    assert torch.equal(S, x["h0"])
    xc = {n: t.cpu() for n, t in x.items()}
    o_ref, _ = oracle.prefill(xc["q"], xc["k"], xc["v"], xc["g"], xc["beta"], xc["h0"])
    assert_o(o, o_ref, inputs.io_dtype(io))
    acc = [7, 8, 9, 16, 17, 19]
    ntok = torch.tensor(acc, dtype=torch.int32, device=DEV)
    kda.kda_decode_multi(x["q"], x["k"], x["v"], x["g"], x["beta"], S, ntok=ntok, commit=True,
                         want_o=False)
    torch.cuda.synchronize()
    for n, m in enumerate(acc):
        sl = slice(n, n + 1)
        _, h_ref = oracle.prefill(xc["q"][sl, :m], xc["k"][sl, :m], xc["v"][sl, :m],
                                  xc["g"][sl, :m], xc["beta"][sl, :m], xc["h0"][sl])
        assert_s(S[sl], h_ref, inputs.io_dtype(io), f"state after {m} accepted tokens")


def test_decay_at_its_bound_over_long_drafts():
    """g = -5 everywhere (the strongest decay allowed) over 16 drafts."""
    N, K, H, d = 3, 16, 2, 128
    x = draft(N, K, H, d, "f32", 28)
    x["g"].fill_(-5.0)
    S = x["h0"].clone()
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    o = kda.kda_decode_multi(x["q"], x["k"], x["v"], x["g"], x["beta"], S, commit=True,
                             status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    xc = {n: t.cpu() for n, t in x.items()}
    o_ref, h_ref = oracle.prefill(xc["q"], xc["k"], xc["v"], xc["g"], xc["beta"], xc["h0"])
    assert_o(o, o_ref, torch.float32)
    assert_s(S, h_ref, torch.float32)


@pytest.mark.parametrize("io,K", [("bf16", 4), ("f32", 6)])
def test_commit_many_heads_mixed_lengths(io, K):
    """2400 heads (several waves of CTAs) with accepted lengths 0..K mixed,
    a run of sequences with none: those keep their state bit for bit, and
    sampled sequences match the oracle."""
    N, H, d = 600, 4, 128
    x = draft(N, K, H, d, io, 26 + K)
    gen = torch.Generator().manual_seed(27 + K)
    m_all = torch.randint(0, K + 1, (N,), generator=gen, dtype=torch.int32)
    m_all[:40] = 0  # a run of sequences with nothing to apply
    ntok = m_all.to(DEV)
    S = x["h0"].clone()
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    kda.kda_decode_multi(x["q"], x["k"], x["v"], x["g"], x["beta"], S, ntok=ntok, commit=True,
                         want_o=False, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    zero = (m_all == 0).nonzero().flatten().tolist()
    assert torch.equal(S[zero], x["h0"][zero])
    xc = {n: t.cpu() for n, t in x.items()}
    for n in [40, 41, 151, 152, 303, 455, 598, 599]:
        m = int(m_all[n])
        if m == 0:
            continue
        sl = slice(n, n + 1)
        _, h_ref = oracle.prefill(xc["q"][sl, :m], xc["k"][sl, :m], xc["v"][sl, :m],
                                  xc["g"][sl, :m], xc["beta"][sl, :m], xc["h0"][sl])
        assert_s(S[sl], h_ref, inputs.io_dtype(io), f"sequence {n}, {m} accepted tokens")


def test_commit_all_equals_single_steps():
    N, K, H, d = 4, 4, 3, 128
    x = draft(N, K, H, d, "bf16", 23)
    S_multi = x["h0"].clone()
    o_multi = kda.kda_decode_multi(x["q"], x["k"], x["v"], x["g"], x["beta"], S_multi,
                                   commit=True)
    S_step = x["h0"].clone()
    o_step = torch.stack([kda.kda_decode_step(x["q"][:, t].contiguous(), x["k"][:, t].contiguous(),
                                              x["v"][:, t].contiguous(), x["g"][:, t].contiguous(),
                                              x["beta"][:, t].contiguous(), S_step)
                          for t in range(K)], dim=1)
    torch.cuda.synchronize()
    assert (o_multi.float() - o_step.float()).abs().max() <= 1e-2 * o_step.float().abs().max()
    assert torch.allclose(S_multi, S_step, rtol=1e-4, atol=1e-6)


def test_workload_n256_k4():
    """The 256 x 32-head decode workload with 4 draft tokens: verify then commit."""
    x = draft(256, 4, 32, 128, "bf16", 24)
    S = x["h0"].clone()
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    o = kda.kda_decode_multi(x["q"], x["k"], x["v"], x["g"], x["beta"], S, status=status)
    kda.kda_decode_multi(x["q"], x["k"], x["v"], x["g"], x["beta"], S, commit=True,
                         want_o=False, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    xc = {n: t.cpu() for n, t in x.items()}
    o_ref, h_ref = oracle.prefill(xc["q"], xc["k"], xc["v"], xc["g"], xc["beta"], xc["h0"])
    assert_o(o, o_ref, torch.bfloat16)
    assert_s(S, h_ref, torch.bfloat16)


def test_multi_status_flags():
    x = draft(2, 3, 2, 128, "bf16", 25)
    x["g"][1, 2, 0, 7] = -9.0
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    kda.kda_decode_multi(x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"], status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & kda.KDA_DEV_DECAY_RANGE


@pytest.mark.parametrize("name", ["q", "k", "v"])
def test_multi_nonfinite_qkv_is_flagged(name):
    x = draft(2, 3, 2, 128, "bf16", 26)
    x[name][1, 2, 1, 40] = float("nan")
    for commit in (0, 1):
        status = torch.zeros(1, dtype=torch.int32, device=DEV)
        S = x["h0"].clone()
        kda.kda_decode_multi(x["q"], x["k"], x["v"], x["g"], x["beta"], S, commit=bool(commit),
                             status=status)
        torch.cuda.synchronize()
        assert int(status.item()) & kda.KDA_DEV_NONFINITE


@pytest.mark.parametrize("io,d,K", [("bf16", 128, 8), ("f32", 128, 7), ("bf16", 64, 3),
                                    ("f32", 64, 8)])
def test_commit_with_outputs(io, d, K):
    """A commit that also returns the outputs (every draft accepted, or a
    per-sequence prefix): o of the accepted tokens and the state after them."""
    N, H = 5, 3
    x = draft(N, K, H, d, io, 29)
    acc = [K, 1, K - 1, 2, K]
    ntok = torch.tensor(acc, dtype=torch.int32, device=DEV)
    S = x["h0"].clone()
    o = kda.kda_decode_multi(x["q"], x["k"], x["v"], x["g"], x["beta"], S, ntok=ntok,
                             commit=True)
    torch.cuda.synchronize()
    xc = {n: t.cpu() for n, t in x.items()}
    for n, m in enumerate(acc):
        sl = slice(n, n + 1)
        o_ref, h_ref = oracle.prefill(xc["q"][sl, :m], xc["k"][sl, :m], xc["v"][sl, :m],
                                      xc["g"][sl, :m], xc["beta"][sl, :m], xc["h0"][sl])
        assert_o(o[sl, :m], o_ref, inputs.io_dtype(io), f"o of the {m} accepted tokens")
        assert_s(S[sl], h_ref, inputs.io_dtype(io), f"state after {m} accepted tokens")


@pytest.mark.parametrize("io", ["bf16", "f32"])
def test_decay_at_its_bound_over_eight_drafts(io):
    """g = -5 on every channel of eight drafts: the block forms scale by
    e^{G} and e^{-G} with |G| up to 40, far inside fp32."""
    N, K, H, d = 3, 8, 2, 128
    x = draft(N, K, H, d, io, 30)
    x["g"].fill_(-5.0)
    S = x["h0"].clone()
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    o_v = kda.kda_decode_multi(x["q"], x["k"], x["v"], x["g"], x["beta"], S, status=status)
    o_c = kda.kda_decode_multi(x["q"], x["k"], x["v"], x["g"], x["beta"], S, commit=True,
                               status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    xc = {n: t.cpu() for n, t in x.items()}
    o_ref, h_ref = oracle.prefill(xc["q"], xc["k"], xc["v"], xc["g"], xc["beta"], xc["h0"])
    assert_o(o_v, o_ref, inputs.io_dtype(io), "verify")
    assert_o(o_c, o_ref, inputs.io_dtype(io), "commit")
    assert_s(S, h_ref, inputs.io_dtype(io))
