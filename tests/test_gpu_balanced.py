"""The balanced schedule of the tensor-core prefill against the one-CTA-per-
sequence schedule (bit for bit) and the fp64 oracle.

With a workspace of kda_chunk_fwd_workspace_size bytes, B*H sequences that do
not fill whole waves of one CTA per SM run on one CTA per SM: CTA i takes
chunk steps [i W, (i + 1) W) of the sequences laid end to end, so a sequence
can be split between two CTAs, its head's final state handed to its tail
through the workspace. A workspace smaller than that size (or none) runs one
CTA per sequence. Both schedules do the same arithmetic in the same order.
"""
import numpy as np
import pytest
import torch

import oracle
from gated_delta_rule_57_gb300 import inputs, kda
from helpers import assert_o, assert_s

pytestmark = pytest.mark.gpu
DEV = "cuda"


def draw(B, T, H, seed):
    w = inputs.PrefillWorkload("balanced", B, T, H, 128, 128, "bf16", seed, h0_std=0.02)
    return inputs.prefill_inputs(w, DEV)


def plan(B, T, H):
    """The split the library chooses on this device (mirrors the host rule)."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    BH, nch = B * H, (T + 63) // 64
    if BH <= sms:
        return None
    W = (BH * nch + sms - 1) // sms
    plain = ((BH + sms - 1) // sms) * nch
    if (W + 4) * 100 >= plain * 97:
        return None
    split = sorted({(i * W) // nch for i in range(1, (BH * nch + W - 1) // W) if (i * W) % nch})
    return W, split


def run(x, ws, **kw):
    o, hT = kda.kda_chunk_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"],
                              workspace=ws, **kw)
    torch.cuda.synchronize()
    return o, hT


def test_balanced_equals_plain_and_oracle():
    B, T, H = 2, 2523, 100  # 200 sequences of 40 chunks, ragged last chunk
    pl = plan(B, T, H)
    if pl is None:
        pytest.skip("this device runs the problem in whole waves")
    W, split = pl
    x = draw(B, T, H, 61)
    need = kda.kda_chunk_fwd_workspace_size(B, T, H, 128, 128, torch.bfloat16)
    ws = torch.zeros(need, dtype=torch.uint8, device=DEV)
    o_b, h_b = run(x, ws)
    o_p, h_p = run(x, torch.empty(16, dtype=torch.uint8, device=DEV))  # too small: plain
    assert torch.equal(o_b, o_p) and torch.equal(h_b, h_p)
    # the handoff flags of exactly the split sequences were set
    flags = ws[B * H * 65536:B * H * 65536 + 4 * B * H].view(torch.int32).cpu().numpy()
    assert sorted(np.nonzero(flags)[0].tolist()) == split and len(split) > 0
    # the oracle over whole sequences that were split (head and tail on two CTAs)
    for s in split[:3] + split[-1:]:
        b, h = divmod(s, H)
        xc = {n: x[n][b:b + 1, :, h:h + 1].cpu() for n in ("q", "k", "v", "g", "beta")}
        o_ref, h_ref = oracle.prefill(xc["q"], xc["k"], xc["v"], xc["g"], xc["beta"],
                                      x["h0"][b:b + 1, h:h + 1].cpu())
        assert_o(o_b[b:b + 1, :, h:h + 1], o_ref, torch.bfloat16, f"o of split sequence {s}")
        assert_s(h_b[b:b + 1, h:h + 1], h_ref, torch.bfloat16, f"hT of split sequence {s}")


def test_balanced_hT_aliases_h0_and_no_hT():
    B, T, H = 1, 1280, 160  # 160 sequences of 20 chunks
    if plan(B, T, H) is None:
        pytest.skip("this device runs the problem in whole waves")
    x = draw(B, T, H, 62)
    o_p, h_p = run(x, torch.empty(16, dtype=torch.uint8, device=DEV))
    h = x["h0"].clone()
    o_a, h_a = kda.kda_chunk_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], h, hT=h)
    o_n, h_n = kda.kda_chunk_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"],
                                 want_hT=False)
    torch.cuda.synchronize()
    assert h_a.data_ptr() == h.data_ptr() and h_n is None
    assert torch.equal(o_a, o_p) and torch.equal(h_a, h_p) and torch.equal(o_n, o_p)


def test_balanced_status_flags():
    """A decay out of range in a split sequence is reported by the balanced schedule."""
    B, T, H = 2, 2523, 100
    pl = plan(B, T, H)
    if pl is None:
        pytest.skip("this device runs the problem in whole waves")
    s = pl[1][0]
    b, h = divmod(s, H)
    x = draw(B, T, H, 63)
    x["g"][b, T - 3, h, 5] = -7.0  # in the tail of a split sequence
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    kda.kda_chunk_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"], status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == kda.KDA_DEV_DECAY_RANGE
