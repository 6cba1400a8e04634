"""GPU parity of kda_decode_step against the fp64 oracle (through the C ABI)."""
import numpy as np
import pytest
import torch

import oracle
from gated_delta_rule_57_gb300 import inputs, kda
from helpers import assert_o, assert_s

pytestmark = pytest.mark.gpu
DEV = "cuda"


def run_steps(w, steps, **kw):
    x = inputs.decode_inputs(w, DEV, steps=steps, **kw)
    S = x["S"].clone()
    S_ref = x["S"].double().cpu().numpy()
    dt = inputs.io_dtype(w.io)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    for s in range(steps):
        o = kda.kda_decode_step(x["q"][s], x["k"][s], x["v"][s], x["g"][s], x["beta"][s], S,
                                status=status)
        torch.cuda.synchronize()
        o_ref, S_ref = oracle.decode(x["q"][s].cpu(), x["k"][s].cpu(), x["v"][s].cpu(),
                                     x["g"][s].cpu(), x["beta"][s].cpu(), S_ref)
        assert_o(o, o_ref, dt, f"o at step {s}")
    assert_s(S, S_ref, dt, "S")
    assert int(status.item()) == 0


def test_workload_n256_first_steps():
    run_steps(inputs.DECODE_N256, 3)


@pytest.mark.slow
def test_workload_n256_all_steps_sampled_sequences():
    """The decode workload over its whole horizon: 1000 consecutive in-place
    steps on the full 256 x 32 state with the workload's seeded inputs. Eight
    sequences (all 32 heads) are replayed by the oracle step by step; every
    step's output and the final state of those sequences are checked, so any
    drift of the fp32 state over the horizon shows."""
    w = inputs.DECODE_N256
    x = inputs.decode_inputs(w, DEV)
    seqs = torch.tensor([0, 37, 74, 111, 148, 185, 222, 255], device=DEV)
    S = x["S"].clone()
    dt = inputs.io_dtype(w.io)
    o_s = torch.empty(w.steps, len(seqs), w.H, w.dv, dtype=dt, device=DEV)
    o = torch.empty(w.N, w.H, w.dv, dtype=dt, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    for s in range(w.steps):
        kda.kda_decode_step(x["q"][s], x["k"][s], x["v"][s], x["g"][s], x["beta"][s], S, o=o,
                            status=status)
        o_s[s] = o[seqs]
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    sub = {n: x[n][:, seqs].cpu() for n in ("q", "k", "v", "g", "beta")}
    S_ref = x["S"][seqs].double().cpu().numpy()
    o_got = o_s.cpu()
    worst = 0.0
    for s in range(w.steps):
        o_ref, S_ref = oracle.decode(sub["q"][s], sub["k"][s], sub["v"][s], sub["g"][s],
                                     sub["beta"][s], S_ref)
        worst = max(worst, assert_o(o_got[s], o_ref, dt, f"o at step {s}"))
    es = assert_s(S[seqs], S_ref, dt, "S after the last step")
    print(f"\ndecode 1000 steps, 8 x 32 sampled heads: worst step o {worst:.3e}, final S {es:.3e}")


@pytest.mark.parametrize("io,d", [("bf16", 64), ("f32", 128), ("f32", 64)])
def test_small_decode(io, d):
    w = inputs.DecodeWorkload("small", 5, 3, d, d, io, 11, 4)
    run_steps(w, 4)


@pytest.mark.parametrize("io", ["bf16", "f32"])
def test_decode_continues_prefill(io):
    """Prefill T tokens, then decode token T: equals prefill of T + 1 tokens."""
    w = inputs.PrefillWorkload("small", 3, 41, 2, 128, 128, io, 12, h0_std=0.02)
    x = inputs.prefill_inputs(w, DEV)
    T = 40
    o_full, h_full = kda.kda_chunk_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"])
    part = {n: x[n][:, :T].contiguous() for n in ("q", "k", "v", "g", "beta")}
    _, S = kda.kda_chunk_fwd(part["q"], part["k"], part["v"], part["g"], part["beta"], x["h0"])
    last = {n: x[n][:, T].contiguous() for n in ("q", "k", "v", "g", "beta")}
    o_dec = kda.kda_decode_step(last["q"], last["k"], last["v"], last["g"], last["beta"], S)
    torch.cuda.synchronize()
    xc = {n: t.cpu() for n, t in x.items()}
    o_ref, h_ref = oracle.prefill(xc["q"], xc["k"], xc["v"], xc["g"], xc["beta"], xc["h0"])
    dt = inputs.io_dtype(io)
    assert_o(o_dec, o_ref[:, T], dt, "decoded token")
    assert_s(S, h_ref, dt, "state after decode")
    assert_o(o_full[:, T], o_ref[:, T], dt, "prefill token")


@pytest.mark.parametrize("bad,flag", [(-7.0, kda.KDA_DEV_DECAY_RANGE),
                                      (float("inf"), kda.KDA_DEV_NONFINITE)])
def test_decode_status_flags(bad, flag):
    w = inputs.DecodeWorkload("small", 4, 2, 128, 128, "bf16", 13, 1)
    x = inputs.decode_inputs(w, DEV)
    x["g"][0, 2, 1, 100] = bad
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    kda.kda_decode_step(x["q"][0], x["k"][0], x["v"][0], x["g"][0], x["beta"][0], x["S"],
                        status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & flag


@pytest.mark.parametrize("io", ["bf16", "f32"])
@pytest.mark.parametrize("name", ["q", "k", "v"])
def test_decode_nonfinite_qkv_is_flagged(io, name):
    w = inputs.DecodeWorkload("small", 4, 2, 128, 128, io, 14, 1)
    x = inputs.decode_inputs(w, DEV)
    x[name][0, 3, 1, 77] = float("inf")
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    kda.kda_decode_step(x["q"][0], x["k"][0], x["v"][0], x["g"][0], x["beta"][0], x["S"],
                        status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & kda.KDA_DEV_NONFINITE
