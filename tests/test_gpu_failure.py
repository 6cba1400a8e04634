"""Failure detection on the GPU without a fault: a bounded mbarrier wait that
nothing completes gives up, reports KDA_DEV_TIMEOUT through the status word,
and the context keeps working (the kernels use the same bounded wait)."""
import pytest
import torch

import oracle
from gated_delta_rule_57_gb300 import inputs, kda
from helpers import assert_o, assert_s

pytestmark = pytest.mark.gpu
DEV = "cuda"


def test_wait_timeout_is_reported_and_context_survives():
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    kda.kda_selftest_wait_timeout(status, clocks=1 << 20)  # about half a millisecond
    torch.cuda.synchronize()
    assert int(status.item()) == kda.KDA_DEV_TIMEOUT
    # the same context still runs the prefill and gets it right
    w = inputs.PrefillWorkload("after", 1, 1, 1, 128, 128, "bf16", 31, h0_std=0.02)
    x = inputs.prefill_inputs(w, "cpu", B=1, T=200, H=2)
    xd = {n: t.to(DEV) for n, t in x.items()}
    st2 = torch.zeros(1, dtype=torch.int32, device=DEV)
    o, hT = kda.kda_chunk_fwd(xd["q"], xd["k"], xd["v"], xd["g"], xd["beta"], xd["h0"],
                              status=st2)
    torch.cuda.synchronize()
    assert int(st2.item()) == 0
    o_ref, h_ref = oracle.prefill(x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"])
    assert_o(o, o_ref, torch.bfloat16)
    assert_s(hT, h_ref, torch.bfloat16)


def test_wait_timeout_flags_accumulate():
    status = torch.full((1,), kda.KDA_DEV_DECAY_RANGE, dtype=torch.int32, device=DEV)
    kda.kda_selftest_wait_timeout(status, clocks=1 << 16)
    torch.cuda.synchronize()
    assert int(status.item()) == kda.KDA_DEV_DECAY_RANGE | kda.KDA_DEV_TIMEOUT
