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


def test_segmented_t1m_against_single_pass():
    """T = 2^20 over two heads, eight segments: the segmented result against
    the single-pass kernel (the oracle covers the same heads in the
    single-pass test). Differences are rounding: o of later segments is the
    sum of two bf16-rounded parts."""
    w = inputs.PREFILL_T1M
    x = inputs.prefill_inputs(w, DEV, H=2)
    o1, h1 = kda.kda_chunk_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], None)
    o2, h2, st = run_seg(dict(x, h0=None), 8)
    assert st == 0
    eo = o_err(o2, o1.double().cpu().numpy())
    eh = s_err(h2, h1.double().cpu().numpy())
    assert eo <= 2e-2 and eh <= 1e-2, (eo, eh)


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
