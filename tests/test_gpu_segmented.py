"""GPU parity of the time-segmented prefill (kda_chunk_fwd_segmented) against
the fp64 oracle, and against the single-pass kernel at sizes the oracle cannot
cover, through the C ABI."""
import numpy as np
import pytest
import torch

import oracle
from gated_delta_rule_57_gb300 import inputs, kda
from helpers import assert_o, assert_s, o_err, s_err

pytestmark = pytest.mark.gpu
DEV = "cuda"
BF16 = torch.bfloat16


def workload(h0):
    return inputs.PrefillWorkload("seg", 1, 1, 1, 128, 128, "bf16", 0, h0_std=0.02 if h0 else None)


def run_seg(x, nseg, **kw):
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    o, hT = kda.kda_chunk_fwd_segmented(x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"],
                                        nseg=nseg, status=status, **kw)
    torch.cuda.synchronize()
    return o, hT, int(status.item())


@pytest.mark.parametrize("B,T,H,nseg,h0", [
    (1, 1000, 2, 3, True),     # 16 chunks in 3 segments (ragged last chunk)
    (2, 640, 3, 10, False),    # one chunk per segment
    (1, 129, 1, 2, True),      # 3 chunks: 2 + 1, last segment a single ragged token
    (3, 2048, 2, 4, True),
    (1, 1000, 2, 7, True),     # 16 chunks, nseg 7 -> 6 non-empty segments
])
def test_segmented_matches_oracle(B, T, H, nseg, h0):
    x = inputs.prefill_inputs(workload(h0), DEV, B=B, T=T, H=H, seed=B * 1000 + T + nseg)
    o, hT, st = run_seg(x, nseg)
    assert st == 0
    xc = {n: (t.cpu() if t is not None else None) for n, t in x.items()}
    o_ref, h_ref = oracle.prefill(xc["q"], xc["k"], xc["v"], xc["g"], xc["beta"], xc["h0"])
    assert_o(o, o_ref, BF16)
    assert_s(hT, h_ref, BF16)


@pytest.mark.parametrize("T", [2048, 2000])
def test_long_first_segment_matches_oracle(T):
    """B=1, H=32, 32 chunks, nseg=8: the 224 short runs of the segment pass
    exceed the 120 SMs the first segments leave free, so the first segment
    spans several segment lengths (on 152 SMs: 12 chunks, then 3-chunk
    segments and a 2-chunk last one, ragged at T = 2000)."""
    n, sc, lead = kda.kda_chunk_fwd_segment_plan(1, T, 32, 128, 128, nseg=8)
    assert n == 8 and lead > 1, (n, sc, lead)
    assert (lead + n - 1) * sc >= 32 > (lead + n - 2) * sc
    x = inputs.prefill_inputs(workload(True), DEV, B=1, T=T, H=32, seed=15)
    o, hT, st = run_seg(x, 8)
    assert st == 0
    xc = {nm: (t.cpu() if t is not None else None) for nm, t in x.items()}
    o_ref, h_ref = oracle.prefill(xc["q"], xc["k"], xc["v"], xc["g"], xc["beta"], xc["h0"])
    assert_o(o, o_ref, BF16)
    assert_s(hT, h_ref, BF16)


def test_segmented_stress_heads_t4096():
    """The T = 4096 workload (half the heads at g = -4.99), five segments."""
    w = inputs.PREFILL_T4K
    x = inputs.prefill_inputs(w, DEV, H=4)
    o, hT, st = run_seg(x, 5)
    assert st == 0
    xc = {n: (t.cpu() if t is not None else None) for n, t in x.items()}
    o_ref, h_ref = oracle.prefill(xc["q"], xc["k"], xc["v"], xc["g"], xc["beta"], xc["h0"])
    assert_o(o, o_ref, BF16)
    assert_s(hT, h_ref, BF16)


def test_one_segment_is_the_single_pass():
    x = inputs.prefill_inputs(workload(True), DEV, B=2, T=700, H=2, seed=11)
    o1, h1 = kda.kda_chunk_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"])
    o2, h2, _ = run_seg(x, 1)
    assert torch.equal(o1, o2) and torch.equal(h1, h2)


def test_segmented_hT_may_alias_h0():
    x = inputs.prefill_inputs(workload(True), DEV, B=1, T=900, H=2, seed=12)
    o1, h1, _ = run_seg(x, 4)
    h = x["h0"].clone()
    x2 = dict(x, h0=h)
    o2, h2, _ = run_seg(x2, 4, hT=h)
    assert h2.data_ptr() == h.data_ptr()
    assert torch.equal(o1, o2) and torch.equal(h1, h2)


def test_segmented_status_flags():
    x = inputs.prefill_inputs(workload(False), DEV, B=1, T=500, H=1, seed=13)
    x["g"][0, 450, 0, 7] = -6.0  # in the last segment
    _, _, st = run_seg(x, 3)
    assert st & kda.KDA_DEV_DECAY_RANGE


@pytest.mark.parametrize("name", ["q", "k", "v"])
def test_segmented_nonfinite_qkv_is_flagged(name):
    x = inputs.prefill_inputs(workload(True), DEV, B=1, T=500, H=2, seed=16)
    x[name][0, 300, 1, 90] = float("nan")  # in a later segment
    _, _, st = run_seg(x, 3)
    assert st & kda.KDA_DEV_NONFINITE


def test_nan_crosses_zero_transitions():
    """g = -4.99 everywhere: every transition is exactly zero, so the scan
    takes X_{s+1} = S0_s without the product. A NaN in v in the first segment
    must still reach every later segment, as in the single pass (a zero
    transition times a NaN state is NaN): the same NaN entries in o and hT,
    the flag set, and the clean head against the oracle."""
    x = inputs.prefill_inputs(workload(False), DEV, B=1, T=1024, H=2, seed=17)
    x["g"].fill_(-4.99)
    x["v"][0, 5, 1, 40] = float("nan")
    o1, h1 = kda.kda_chunk_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"])
    o, hT, st = run_seg(x, 4)
    assert st & kda.KDA_DEV_NONFINITE
    assert torch.equal(torch.isnan(o), torch.isnan(o1))
    assert torch.equal(torch.isnan(hT), torch.isnan(h1))
    assert torch.isnan(o[0, -1, 1, 40]) and torch.isnan(hT[0, 1, :, 40]).all()
    sub = {n: x[n][:, :, :1].contiguous().cpu() for n in ("q", "k", "v", "g", "beta")}
    o_ref, h_ref = oracle.prefill(sub["q"], sub["k"], sub["v"], sub["g"], sub["beta"], None)
    assert_o(o[:, :, :1], o_ref, BF16)
    assert_s(hT[:, :1], h_ref, BF16)


@pytest.mark.slow
def test_t1m_benchmark_calls_against_oracle():
    """The long-context workload (B=1, T=2^20, H=32, the benchmark's seed)
    through the three calls the benchmark times: kda_chunk_fwd in one pass,
    kda_chunk_fwd_segmented with the segment count of
    kda_chunk_fwd_segments_hint and the library's first-segment length, and
    kda_chunk_fwd_segmented planned on the device from the decay probe
    (nseg = 0: more, shorter segments). The
    oracle recomputes four heads (two of them apart by half the head range)
    over the whole sequence, and every output and the final state of those
    heads is checked for both calls, so the transitions built over the long
    segments are checked against the definition, not against the one-pass
    kernel."""
    w = inputs.PREFILL_T1M
    x = inputs.prefill_inputs(w, DEV)
    heads = [0, 11, 22, 31]
    nseg = kda.kda_chunk_fwd_segments_hint(w.B, w.T, w.H, w.dk, w.dv)
    assert nseg > 1
    n_eff, sc, lead = kda.kda_chunk_fwd_segment_plan(w.B, w.T, w.H, w.dk, w.dv, nseg=nseg)
    ws = torch.empty(kda.kda_chunk_fwd_segmented_workspace_size(w.B, w.T, w.H, w.dk, w.dv,
                                                                nseg=nseg),
                     dtype=torch.uint8, device=DEV)
    o = torch.empty_like(x["v"])
    hT = torch.empty(w.B, w.H, w.dk, w.dv, dtype=torch.float32, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    got = {}
    kda.kda_chunk_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], None, o=o, hT=hT,
                      status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    got["single"] = (o[:, :, heads].cpu(), hT[:, heads].cpu())
    o.fill_(float("nan"))
    hT.fill_(float("nan"))
    kda.kda_chunk_fwd_segmented(x["q"], x["k"], x["v"], x["g"], x["beta"], None, nseg=nseg,
                                o=o, hT=hT, workspace=ws, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    got["segmented"] = (o[:, :, heads].cpu(), hT[:, heads].cpu())
    del ws
    ws = torch.empty(kda.kda_chunk_fwd_segmented_workspace_size(w.B, w.T, w.H, w.dk, w.dv,
                                                                nseg=0),
                     dtype=torch.uint8, device=DEV)
    probe = kda.kda_chunk_fwd_decay_probe(x["g"])
    nseg_d, lead_d = kda.kda_chunk_fwd_segments_hint_decay(w.B, w.T, w.H, w.dk, w.dv,
                                                           probe=probe)
    assert nseg_d > nseg, (nseg_d, lead_d)  # this decay empties a state within a few chunks
    o.fill_(float("nan"))
    hT.fill_(float("nan"))
    kda.kda_chunk_fwd_segmented(x["q"], x["k"], x["v"], x["g"], x["beta"], None, nseg="decay",
                                o=o, hT=hT, workspace=ws, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    got["segmented_decay"] = (o[:, :, heads].cpu(), hT[:, heads].cpu())
    sub = {n: x[n][:, :, heads].contiguous().cpu() for n in ("q", "k", "v", "g", "beta")}
    del x, o, hT, ws
    torch.cuda.empty_cache()
    o_ref, h_ref = oracle.prefill(sub["q"], sub["k"], sub["v"], sub["g"], sub["beta"], None,
                                  nthreads=len(heads))
    errs = {}
    for name, (og, hg) in got.items():
        errs[name] = (assert_o(og, o_ref, BF16, f"{name} o"),
                      assert_s(hg, h_ref, BF16, f"{name} hT"))
    print(f"\nT=2^20 H=32, heads {heads}: nseg {n_eff} (segment {sc} chunks, first {lead}x), "
          f"decay-planned nseg {nseg_d} (first {lead_d}x); "
          + "; ".join(f"{n}: o {e[0]:.3e} hT {e[1]:.3e}" for n, e in errs.items()))


def test_hint_and_workspace():
    n = kda.kda_chunk_fwd_segments_hint(1, 1 << 20, 32, 128, 128)
    assert n > 1  # 32 sequences on a GB300 leave most SMs idle
    assert kda.kda_chunk_fwd_segments_hint(8, 8192, 32, 128, 128) == 1  # 256 sequences
    assert kda.kda_chunk_fwd_segments_hint(1, 1 << 20, 32, 128, 128, torch.float32) == 1
    need = kda.kda_chunk_fwd_segmented_workspace_size(1, 1 << 20, 32, 128, 128, nseg=n)
    assert need == 32 * (3 * n - 2) * 128 * 128 * 4


def test_short_workspace_is_rejected():
    x = inputs.prefill_inputs(workload(False), DEV, B=1, T=640, H=1, seed=14)
    need = kda.kda_chunk_fwd_segmented_workspace_size(1, 640, 1, 128, 128, nseg=2)
    ws = torch.empty(need - 16, dtype=torch.uint8, device=DEV)
    with pytest.raises(kda.KdaError) as ei:
        run_seg(x, 2, workspace=ws)
    assert ei.value.code == kda.KDA_ERR_WORKSPACE


@pytest.mark.parametrize("B,T,H,dk,nsample", [
    (2, 1000, 3, 128, 8),     # ragged last chunk
    (1, 640, 2, 64, 40),      # more samples than chunks: chunks repeat
    (3, 64, 1, 128, 1),
    (1, 300, 19, 128, 5),     # heads over three CTAs, the last one partly idle
])
def test_decay_probe_matches_definition(B, T, H, dk, nsample):
    """d_probe[b, s, h] = sum over the tokens of chunk floor(s * nch / nsample)
    of max over channels of g[b, t, h]."""
    gen = torch.Generator(device=DEV).manual_seed(B * 100 + T)
    g = -5 * torch.sigmoid(torch.randn(B, T, H, dk, generator=gen, device=DEV))
    got = kda.kda_chunk_fwd_decay_probe(g, nsample=nsample)
    torch.cuda.synchronize()
    gd = g.double().cpu()
    nch = (T + 63) // 64
    for b in range(B):
        for s_ in range(nsample):
            c = s_ * nch // nsample
            want = gd[b, 64 * c:min(T, 64 * c + 64)].amax(dim=-1).sum(dim=0)  # [H]
            err = (got[b, s_].double().cpu() - want).abs().max().item()
            assert err <= 1e-5 * want.abs().max().item() + 1e-5, (b, s_, c)


def test_hint_decay_plans():
    """Strong decay (every run with v = 0 stops after a few chunks): more,
    shorter segments and a shorter first one than the shape-only hint; no
    decay information, or decay too weak to count on: the shape-only plan."""
    B, T, H = 1, 1 << 20, 32
    n0 = kda.kda_chunk_fwd_segments_hint(B, T, H, 128, 128)
    _, sc0, lead0 = kda.kda_chunk_fwd_segment_plan(B, T, H, 128, 128, nseg=n0)
    n, lead = kda.kda_chunk_fwd_segments_hint_decay(B, T, H, 128, 128, probe=[-20.0, -25.0])
    _, sc, _ = kda.kda_chunk_fwd_segment_plan(B, T, H, 128, 128, nseg=n, lead=lead)
    assert n > n0 and lead * sc < lead0 * sc0, (n, lead, sc, n0, lead0, sc0)
    for weak in ([], [0.0], [-20.0, float("nan")], [-1e-3]):
        n1, lead1 = kda.kda_chunk_fwd_segments_hint_decay(B, T, H, 128, 128, probe=weak)
        _, _, lead_shape = kda.kda_chunk_fwd_segment_plan(B, T, H, 128, 128, nseg=n1)
        assert n1 == n0 and lead1 == lead_shape, weak
    # many sequences: no split, whatever the decay
    assert kda.kda_chunk_fwd_segments_hint_decay(8, 8192, 32, 128, 128, probe=[-50.0]) == (1, 1)


@pytest.mark.parametrize("nseg,lead", [(6, 2), (7, 3), (16, 4)])
def test_explicit_lead_matches_oracle(nseg, lead):
    """B=1, T=2000 (32 chunks, ragged), H=4: a first segment of `lead`
    segment lengths, as kda_chunk_fwd_segment_plan reports it."""
    T = 2000
    n, sc, ld = kda.kda_chunk_fwd_segment_plan(1, T, 4, 128, 128, nseg=nseg, lead=lead)
    assert ld == lead and (ld + n - 1) * sc >= 32 > (ld + n - 2) * sc
    x = inputs.prefill_inputs(workload(True), DEV, B=1, T=T, H=4, seed=17 + nseg)
    o, hT, st = run_seg(x, nseg, lead=lead)
    assert st == 0
    xc = {nm: (t.cpu() if t is not None else None) for nm, t in x.items()}
    o_ref, h_ref = oracle.prefill(xc["q"], xc["k"], xc["v"], xc["g"], xc["beta"], xc["h0"])
    assert_o(o, o_ref, BF16)
    assert_s(hT, h_ref, BF16)


def test_decay_planned_call_matches_oracle():
    """nseg="decay" on the T = 4096 stress workload (half the heads at
    g = -4.99): probe, plan and segmented call, against the oracle."""
    w = inputs.PREFILL_T4K
    x = inputs.prefill_inputs(w, DEV)
    o, hT = kda.kda_chunk_fwd_segmented(x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"],
                                        nseg="decay")
    torch.cuda.synchronize()
    heads = [0, 7, 16, 31]
    sub = {n: x[n][:, :, heads].contiguous().cpu() for n in ("q", "k", "v", "g", "beta")}
    h0 = x["h0"][:, heads].contiguous().cpu() if x["h0"] is not None else None
    o_ref, h_ref = oracle.prefill(sub["q"], sub["k"], sub["v"], sub["g"], sub["beta"], h0)
    assert_o(o[:, :, heads], o_ref, BF16)
    assert_s(hT[:, heads], h_ref, BF16)


def test_slow_decay_runs_whole_segments():
    """Decay near zero (g = -0.01 on every channel) over chunks 10..29 and
    g = -4.99 elsewhere: the transition and correction runs of the slow
    stretch cannot stop early and run their whole segments, the others stop
    after a chunk or two. The probe tells the two apart (chunk 0 against
    chunk 16); under plans with several segment lengths the results match
    the oracle."""
    B, T, H = 1, 2000, 4  # 32 chunks
    x = inputs.prefill_inputs(workload(True), DEV, B=B, T=T, H=H, seed=31)
    x["g"].fill_(-4.99)
    x["g"][:, 640:1920] = -0.01  # chunks 10..29
    probe = kda.kda_chunk_fwd_decay_probe(x["g"], nsample=2)  # chunks 0 and 16
    torch.cuda.synchronize()
    assert probe[0, 0].max().item() < -300 and probe[0, 1].max().item() > -1
    for nseg, lead in ((8, 2), (6, 1)):
        o, hT, st = run_seg(x, nseg, lead=lead)
        assert st == 0
        xc = {nm: (t.cpu() if t is not None else None) for nm, t in x.items()}
        o_ref, h_ref = oracle.prefill(xc["q"], xc["k"], xc["v"], xc["g"], xc["beta"], xc["h0"])
        assert_o(o, o_ref, BF16, f"nseg {nseg} lead {lead}")
        assert_s(hT, h_ref, BF16, f"nseg {nseg} lead {lead}")


@pytest.mark.parametrize("B,T,H,stress", [(1, 4096, 32, True), (2, 3000, 5, False),
                                          (1, 900, 3, False)])
def test_device_plan_equals_host_plan(B, T, H, stress):
    """nseg = 0 (probe, planning kernel, passes reading the plan) gives exactly
    the bits of the explicit split the host's copy of the planner picks from
    the same probe, and matches the oracle."""
    w = inputs.PrefillWorkload("plan", B, T, H, 128, 128, "bf16", 50 + T, h0_std=0.02,
                               stress_heads=stress)
    x = inputs.prefill_inputs(w, DEV)
    o_d, h_d, st = run_seg(x, 0)
    assert st == 0
    n, lead = kda.kda_chunk_fwd_segments_hint_decay(B, T, H, 128, 128,
                                                    probe=kda.kda_chunk_fwd_decay_probe(x["g"]))
    if n > 1:
        o_h, h_h, _ = run_seg(x, n, lead=lead)
    else:
        o_h, h_h = kda.kda_chunk_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"])
        torch.cuda.synchronize()
    if n > 1:
        assert torch.equal(o_d, o_h) and torch.equal(h_d, h_h), (n, lead)
    xc = {nm: (t.cpu() if t is not None else None) for nm, t in x.items()}
    o_ref, h_ref = oracle.prefill(xc["q"], xc["k"], xc["v"], xc["g"], xc["beta"], xc["h0"])
    assert_o(o_d, o_ref, BF16)
    assert_s(h_d, h_ref, BF16)


@pytest.mark.parametrize("bad,flag", [(float("nan"), "KDA_DEV_NONFINITE"),
                                      (0.5, "KDA_DEV_DECAY_RANGE")])
def test_device_plan_with_bad_decay(bad, flag):
    """A NaN or a positive log-decay in g: the device-planned split still runs
    (a non-finite statistic makes the planner count whole-segment runs) and
    the status word reports the value."""
    B, T, H = 1, 2000, 4
    x = inputs.prefill_inputs(workload(True), DEV, B=B, T=T, H=H, seed=70)
    x["g"][0, 5, 2, 17] = bad  # inside chunk 0, which the probe samples
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    kda.kda_chunk_fwd_segmented(x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"], nseg=0,
                                status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & getattr(kda, flag)
