"""GPU parity of kda_chunk_fwd against the fp64 oracle (through the C ABI)."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from gated_delta_rule_57_gb300 import inputs, kda
from helpers import assert_o, assert_s

pytestmark = pytest.mark.gpu
DEV = "cuda"


def small(io, d, h0):
    return inputs.PrefillWorkload("small", 1, 1, 1, d, d, io, 0, h0_std=0.02 if h0 else None)


def run_case(w, *, B=None, T=None, H=None, seed=None, device_gen=False, h0_override=None):
    gen_dev = DEV if device_gen else "cpu"
    x = inputs.prefill_inputs(w, gen_dev, B=B, T=T, H=H, seed=seed)
    if h0_override is not None:
        x["h0"] = h0_override
    xd = {n: (t.to(DEV) if t is not None else None) for n, t in x.items()}
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    o, hT = kda.kda_chunk_fwd(xd["q"], xd["k"], xd["v"], xd["g"], xd["beta"], xd["h0"],
                              status=status)
    torch.cuda.synchronize()
    return x, o, hT, int(status.item())


def check_against_oracle(x, o, hT, dtype):
    o_ref, h_ref = oracle.prefill(x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"])
    eo = assert_o(o, o_ref, dtype)
    eh = assert_s(hT, h_ref, dtype)
    return eo, eh


def test_tiny_f32_workload():
    x, o, hT, st = run_case(inputs.TINY_F32)
    assert st == 0
    check_against_oracle(x, o, hT, torch.float32)


CASES = [
    # (B, T, H, d, io, h0): several chunks, ragged tails, tiny T, both head sizes
    (2, 200, 3, 128, "bf16", True),
    (1, 1, 2, 64, "bf16", False),
    (1, 15, 1, 128, "f32", True),
    (1, 17, 2, 64, "f32", False),
    (1, 250, 2, 64, "bf16", True),
    (3, 64, 2, 128, "bf16", False),
    (1, 129, 1, 128, "f32", True),
    (2, 333, 2, 128, "f32", False),
    (1, 1000, 4, 128, "bf16", True),
]


@pytest.mark.parametrize("B,T,H,d,io,h0", CASES)
def test_small_cases(B, T, H, d, io, h0):
    w = small(io, d, h0)
    x, o, hT, st = run_case(w, B=B, T=T, H=H, seed=B * 1000 + T + H + d)
    assert st == 0
    check_against_oracle(x, o, hT, inputs.io_dtype(io))


def test_workload_t4096_stress_heads():
    """Heads 16..31 decay at g = -4.99 everywhere: a 16-token tile reaches
    e^-79.84, the edge the bounded-reciprocal diagonal tiles must survive."""
    x, o, hT, st = run_case(inputs.PREFILL_T4K, device_gen=True)
    assert st == 0
    check_against_oracle(x, o, hT, torch.bfloat16)


@pytest.mark.slow
def test_workload_b8_t8192():
    x, o, hT, st = run_case(inputs.PREFILL_B8_T8K, device_gen=True)
    assert st == 0
    check_against_oracle(x, o, hT, torch.bfloat16)


@pytest.mark.parametrize("io,d", [("bf16", 128), ("bf16", 64), ("f32", 128)])
def test_empty_sequence_returns_h0(io, d):
    w = small(io, d, True)
    x = inputs.prefill_inputs(w, DEV, B=2, T=0, H=3)
    o, hT = kda.kda_chunk_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"])
    torch.cuda.synchronize()
    assert o.numel() == 0
    assert torch.equal(hT, x["h0"])
    _, hz = kda.kda_chunk_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], None)
    torch.cuda.synchronize()
    assert torch.count_nonzero(hz) == 0


@pytest.mark.parametrize("io", ["bf16", "f32"])
def test_hT_may_alias_h0(io):
    w = small(io, 64, True)
    x = inputs.prefill_inputs(w, DEV, B=2, T=100, H=2, seed=5)
    o1, h1 = kda.kda_chunk_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"])
    h = x["h0"].clone()
    o2, h2 = kda.kda_chunk_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], h, hT=h)
    torch.cuda.synchronize()
    assert h2.data_ptr() == h.data_ptr()
    assert torch.equal(o1, o2) and torch.equal(h1, h2)


@pytest.mark.parametrize("io", ["bf16", "f32"])
def test_chaining_matches_single_pass(io):
    """Prefill [0, T1) then [T1, T) with hT -> h0 equals one pass over [0, T)."""
    w = small(io, 128, True)
    x = inputs.prefill_inputs(w, DEV, B=2, T=300, H=2, seed=6)
    o, hT = kda.kda_chunk_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"])
    T1 = 137
    p1 = {n: x[n][:, :T1].contiguous() for n in ("q", "k", "v", "g", "beta")}
    p2 = {n: x[n][:, T1:].contiguous() for n in ("q", "k", "v", "g", "beta")}
    o1, h1 = kda.kda_chunk_fwd(p1["q"], p1["k"], p1["v"], p1["g"], p1["beta"], x["h0"])
    o2, h2 = kda.kda_chunk_fwd(p2["q"], p2["k"], p2["v"], p2["g"], p2["beta"], h1)
    torch.cuda.synchronize()
    dt = inputs.io_dtype(io)
    xc = {n: (t.cpu() if t is not None else None) for n, t in x.items()}
    o_ref, h_ref = oracle.prefill(xc["q"], xc["k"], xc["v"], xc["g"], xc["beta"], xc["h0"])
    assert_o(torch.cat([o1, o2], 1), o_ref, dt, "chained o")
    assert_s(h2, h_ref, dt, "chained hT")
    assert_o(o, o_ref, dt)


@pytest.mark.parametrize("io", ["bf16", "f32"])
@pytest.mark.parametrize("gval", [0.0, -5.0])
def test_decay_edges(io, gval):
    """g = 0 (no forgetting) and g = -5 (the bound itself) everywhere."""
    w = small(io, 128, True)
    x = inputs.prefill_inputs(w, "cpu", B=1, T=160, H=2, seed=7)
    x["g"].fill_(gval)
    xd = {n: t.to(DEV) for n, t in x.items()}
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    o, hT = kda.kda_chunk_fwd(xd["q"], xd["k"], xd["v"], xd["g"], xd["beta"], xd["h0"],
                              status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    check_against_oracle(x, o, hT, inputs.io_dtype(io))


@pytest.mark.parametrize("io", ["bf16", "f32"])
def test_beta_zero_pure_decay(io):
    w = small(io, 64, True)
    x = inputs.prefill_inputs(w, "cpu", B=1, T=70, H=2, seed=8)
    x["beta"].zero_()
    xd = {n: t.to(DEV) for n, t in x.items()}
    o, hT = kda.kda_chunk_fwd(xd["q"], xd["k"], xd["v"], xd["g"], xd["beta"], xd["h0"])
    torch.cuda.synchronize()
    ref = torch.exp(x["g"].double().sum(1))[..., None] * x["h0"].double()
    assert_s(hT, ref.numpy(), inputs.io_dtype(io))


@pytest.mark.parametrize("io", ["bf16", "f32"])
@pytest.mark.parametrize("bad,flag", [(-6.0, kda.KDA_DEV_DECAY_RANGE),
                                      (0.5, kda.KDA_DEV_DECAY_RANGE),
                                      (float("nan"), kda.KDA_DEV_NONFINITE)])
def test_status_flags(io, bad, flag):
    w = small(io, 64, False)
    x = inputs.prefill_inputs(w, DEV, B=1, T=40, H=2, seed=9)
    x["g"][0, 33, 1, 5] = bad
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    kda.kda_chunk_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], None, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & flag
    status.zero_()
    x["g"][0, 33, 1, 5] = -1.0
    kda.kda_chunk_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], None, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0


@pytest.mark.parametrize("io,d", [("bf16", 128), ("bf16", 64), ("f32", 128)])
@pytest.mark.parametrize("name", ["q", "k", "v"])
@pytest.mark.parametrize("bad", [float("nan"), float("inf")])
def test_nonfinite_qkv_is_flagged(io, d, name, bad):
    """A NaN or Inf in q, k or v (here in the second chunk of one head, on the
    tensor-core path for bf16, d = 64 or 128, and the CUDA-core path for fp32)
    sets KDA_DEV_NONFINITE."""
    w = small(io, d, True)
    x = inputs.prefill_inputs(w, DEV, B=2, T=150, H=2, seed=19)
    x[name][1, 97, 0, 11] = bad
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    kda.kda_chunk_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"], status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & kda.KDA_DEV_NONFINITE


@pytest.mark.parametrize("io,d,every", [("bf16", 128, 64), ("bf16", 128, 128), ("f32", 64, 64),
                                        ("f32", 128, 128), ("bf16", 64, 64)])
def test_state_checkpoints(io, d, every):
    """ckpt[b, h, j] is the state after token (j + 1) * every - 1 (oracle prefix)."""
    w = small(io, d, True)
    T = 330
    x = inputs.prefill_inputs(w, "cpu", B=2, T=T, H=2, seed=31)
    xd = {n: t.to(DEV) for n, t in x.items()}
    o, hT, ck = kda.kda_chunk_fwd_ckpt(xd["q"], xd["k"], xd["v"], xd["g"], xd["beta"], xd["h0"],
                                       ckpt_every=every)
    o2, h2 = kda.kda_chunk_fwd(xd["q"], xd["k"], xd["v"], xd["g"], xd["beta"], xd["h0"])
    torch.cuda.synchronize()
    assert ck.shape == (2, 2, T // every, d, d)
    assert torch.equal(o, o2) and torch.equal(hT, h2)  # checkpoints change nothing else
    dt = inputs.io_dtype(io)
    for j in range(T // every):
        n = (j + 1) * every
        _, h_ref = oracle.prefill(x["q"][:, :n], x["k"][:, :n], x["v"][:, :n], x["g"][:, :n],
                                  x["beta"][:, :n], x["h0"])
        assert_s(ck[:, :, j], h_ref, dt, f"checkpoint {j}")


def test_checkpoint_at_end_equals_hT():
    w = small("bf16", 128, True)
    x = inputs.prefill_inputs(w, DEV, B=1, T=256, H=3, seed=32)
    o, hT, ck = kda.kda_chunk_fwd_ckpt(x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"],
                                       ckpt_every=128)
    torch.cuda.synchronize()
    assert torch.equal(ck[:, :, -1], hT)


@pytest.mark.parametrize("io", ["bf16", "f32"])
def test_degenerate_inputs(io):
    """k = 0: the state only decays; v = 0 with h0 = 0: all zero; q = 0: o = 0."""
    w = small(io, 128, True)
    x = inputs.prefill_inputs(w, "cpu", B=1, T=150, H=2, seed=33)
    dt = inputs.io_dtype(io)
    xk = dict(x)
    xk["k"] = torch.zeros_like(x["k"])
    xd = {n: t.to(DEV) for n, t in xk.items()}
    o, hT = kda.kda_chunk_fwd(xd["q"], xd["k"], xd["v"], xd["g"], xd["beta"], xd["h0"])
    torch.cuda.synchronize()
    ref = torch.exp(x["g"].double().sum(1))[..., None] * x["h0"].double()
    assert_s(hT, ref.numpy(), dt, "k = 0 state")
    o_ref, _ = oracle.prefill(xk["q"], xk["k"], xk["v"], xk["g"], xk["beta"], xk["h0"])
    assert_o(o, o_ref, dt, "k = 0 output")
    xv = {n: t.to(DEV) for n, t in x.items()}
    xv["v"].zero_()
    o, hT = kda.kda_chunk_fwd(xv["q"], xv["k"], xv["v"], xv["g"], xv["beta"], None)
    torch.cuda.synchronize()
    assert torch.count_nonzero(o) == 0 and torch.count_nonzero(hT) == 0
    xq = {n: t.to(DEV) for n, t in x.items()}
    xq["q"].zero_()
    o, _ = kda.kda_chunk_fwd(xq["q"], xq["k"], xq["v"], xq["g"], xq["beta"], xq["h0"])
    torch.cuda.synchronize()
    assert torch.count_nonzero(o) == 0


@pytest.mark.parametrize("io", ["bf16", "f32"])
def test_exact_overwrite_orthonormal_keys(io):
    """g = 0, beta = 1 and exactly orthonormal keys (entries +-0.5, exact in
    bf16): writing (k, v) then reading with q = k returns v; rewriting a key
    replaces its value. Holds across chunk boundaries (T = 200)."""
    d, T = 128, 200
    H4 = torch.tensor([[1, 1, 1, 1], [1, -1, 1, -1], [1, 1, -1, -1], [1, -1, -1, 1]],
                      dtype=torch.float32) / 2
    K = torch.block_diag(*([H4] * (d // 4)))  # d exactly orthonormal rows
    gen = torch.Generator().manual_seed(34)
    idx = torch.randint(0, d, (T,), generator=gen)
    dt = inputs.io_dtype(io)
    k = K[idx][None, :, None, :].to(dt)
    q = k.clone()
    v = torch.randint(-4, 5, (1, T, 1, d), generator=gen).float().to(dt)
    g = torch.zeros(1, T, 1, d)
    beta = torch.ones(1, T, 1)
    o, hT = kda.kda_chunk_fwd(q.to(DEV), k.to(DEV), v.to(DEV), g.to(DEV), beta.to(DEV), None)
    torch.cuda.synchronize()
    assert_o(o, v.double().numpy(), dt, "read-back of the value just written")
    latest = {}
    for t in range(T):
        latest[int(idx[t])] = v[0, t, 0].double()
    S = sum(torch.outer(K[i].double(), val) for i, val in latest.items())
    assert_s(hT, S.numpy()[None, None], dt, "overwritten state")


def test_many_heads():
    """B*H = 2048 sequences (8 waves of CTAs) against the oracle on sampled heads."""
    w = inputs.PrefillWorkload("many", 16, 130, 128, 128, 128, "bf16", 35, h0_std=0.02)
    x = inputs.prefill_inputs(w, DEV)
    o, hT = kda.kda_chunk_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"])
    torch.cuda.synchronize()
    heads = [0, 77, 127]
    bsel = [0, 9, 15]
    sub = {n: x[n][bsel][:, :, heads].contiguous().cpu() for n in ("q", "k", "v", "g", "beta")}
    h0s = x["h0"][bsel][:, heads].contiguous().cpu()
    o_ref, h_ref = oracle.prefill(sub["q"], sub["k"], sub["v"], sub["g"], sub["beta"], h0s)
    assert_o(o[bsel][:, :, heads], o_ref, torch.bfloat16)
    assert_s(hT[bsel][:, heads], h_ref, torch.bfloat16)


def test_chunk_size_invariance():
    """The recurrence has no chunking: the tensor-core path (64-token chunks,
    bf16 operands) and the CUDA-core path (32-token chunks, fp32) on the same
    token values agree within the bf16 tolerance, and both match the oracle."""
    w = small("bf16", 128, True)
    x = inputs.prefill_inputs(w, DEV, B=2, T=300, H=2, seed=41)
    o64, h64 = kda.kda_chunk_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"])
    xf = {n: (t.float() if t is not None else None) for n, t in x.items()}
    o32, h32 = kda.kda_chunk_fwd(xf["q"], xf["k"], xf["v"], xf["g"], xf["beta"], xf["h0"])
    torch.cuda.synchronize()
    o32n = o32.double().cpu().numpy()
    assert_o(o64, o32n, torch.bfloat16, "C=64 vs C=32 o")
    assert_s(h64, h32.double().cpu().numpy(), torch.bfloat16, "C=64 vs C=32 hT")
    xc = {n: (t.cpu() if t is not None else None) for n, t in x.items()}
    o_ref, h_ref = oracle.prefill(xc["q"], xc["k"], xc["v"], xc["g"], xc["beta"], xc["h0"])
    assert_o(o32, o_ref, torch.float32, "C=32 o")
    assert_s(h32, h_ref, torch.float32, "C=32 hT")


@pytest.mark.parametrize("B,T,H,h0", [(1, 1, 2, True), (2, 129, 3, False), (1, 1000, 4, True),
                                      (3, 333, 2, True)])
def test_bf16_d64_on_tensor_cores(B, T, H, h0):
    """bf16 with d = 64 runs the tensor-core kernel at d = 128, channels 64..127
    read as zeros and clipped on store: outputs and final state against the
    oracle, ragged lengths, with and without h0."""
    w = inputs.PrefillWorkload("d64", B, T, H, 64, 64, "bf16", 80 + T, h0_std=0.02 if h0 else None)
    x = inputs.prefill_inputs(w, DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    o, hT = kda.kda_chunk_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"], status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    xc = {n: (t.cpu() if t is not None else None) for n, t in x.items()}
    o_ref, h_ref = oracle.prefill(xc["q"], xc["k"], xc["v"], xc["g"], xc["beta"], xc["h0"])
    assert_o(o, o_ref, torch.bfloat16)
    assert_s(hT, h_ref, torch.bfloat16)


def test_bf16_d64_balanced_and_aliased():
    """d = 64 with more sequences than SMs: the balanced schedule (handoffs in
    the 128 x 128 internal layout) gives the bits of one CTA per sequence, hT
    may alias h0, and a batch row matches the oracle."""
    B, T, H = 2, 1280, 80  # 160 sequences of 20 chunks
    w = inputs.PrefillWorkload("d64b", B, T, H, 64, 64, "bf16", 90, h0_std=0.02)
    x = inputs.prefill_inputs(w, DEV)
    ws = torch.zeros(kda.kda_chunk_fwd_workspace_size(B, T, H, 64, 64, torch.bfloat16),
                     dtype=torch.uint8, device=DEV)
    assert ws.numel() > 0
    o_b, h_b = kda.kda_chunk_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"], workspace=ws)
    o_p, h_p = kda.kda_chunk_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"])
    h = x["h0"].clone()
    o_a, h_a = kda.kda_chunk_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], h, hT=h)
    torch.cuda.synchronize()
    assert torch.equal(o_b, o_p) and torch.equal(h_b, h_p)
    assert torch.equal(o_a, o_p) and torch.equal(h_a, h_p) and h_a.data_ptr() == h.data_ptr()
    sub = {n: t[0:1, :, 0:4].contiguous().cpu() for n, t in x.items() if n != "h0"}
    o_ref, h_ref = oracle.prefill(sub["q"], sub["k"], sub["v"], sub["g"], sub["beta"],
                                  x["h0"][0:1, 0:4].contiguous().cpu())
    assert_o(o_b[0:1, :, 0:4], o_ref, torch.bfloat16)
    assert_s(h_b[0:1, 0:4], h_ref, torch.bfloat16)


@pytest.mark.parametrize("B,T,H,bal", [(2, 333, 3, False), (2, 1280, 80, True)])
def test_bf16_d64_equals_zero_padded_d128(B, T, H, bal):
    """bf16 d = 64 runs the d = 128 arithmetic on channels that the tensor maps
    fill with zeros, so it gives exactly the bits of the d = 128 kernel on the
    same inputs padded with zeros to 128 channels (g = 0 there), o and hT cut
    back to 64: one CTA per sequence and the balanced schedule."""
    w = inputs.PrefillWorkload("d64p", B, T, H, 64, 64, "bf16", 95 + T, h0_std=0.02)
    x = inputs.prefill_inputs(w, DEV)

    def pad(t, dims):
        out = torch.zeros(*t.shape[:-dims], *([128] * dims), dtype=t.dtype, device=DEV)
        out[(...,) + (slice(0, 64),) * dims] = t
        return out

    xp = {n: pad(x[n], 1) for n in ("q", "k", "v", "g")}
    h0p = pad(x["h0"], 2)

    def ws(d):
        if not bal:
            return None
        return torch.zeros(kda.kda_chunk_fwd_workspace_size(B, T, H, d, d, torch.bfloat16),
                           dtype=torch.uint8, device=DEV)

    def call(q, k, v, g, h0, d):
        o = torch.empty(B, T, H, d, dtype=torch.bfloat16, device=DEV)
        hT = torch.empty(B, H, d, d, dtype=torch.float32, device=DEV)
        w_ = ws(d)
        if w_ is None:  # one CTA per sequence: a workspace too small for the balanced schedule
            w_ = torch.empty(16, dtype=torch.uint8, device=DEV)
        return kda.kda_chunk_fwd(q, k, v, g, x["beta"], h0, o=o, hT=hT, workspace=w_)

    o64, h64 = call(x["q"], x["k"], x["v"], x["g"], x["h0"], 64)
    o128, h128 = call(xp["q"], xp["k"], xp["v"], xp["g"], h0p, 128)
    torch.cuda.synchronize()
    assert torch.equal(o64, o128[..., :64])
    assert torch.equal(h64, h128[..., :64, :64])
    assert torch.count_nonzero(o128[..., 64:]) == 0 and torch.count_nonzero(h128[..., 64:, :]) == 0
