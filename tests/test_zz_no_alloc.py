"""The entry point that allocates nothing: kda_chunk_fwd_segmented_noalloc runs
the segmented prefill with its scratch in the library's static device array."""
import pytest
import torch

import oracle
from gated_delta_rule_57_gb300 import inputs, kda
from helpers import assert_o, assert_s

pytestmark = pytest.mark.gpu
DEV = "cuda"


def workload():
    return inputs.PrefillWorkload("noalloc", 1, 1, 1, 128, 128, "bf16", 0, h0_std=0.02)


def test_matches_workspace_path_and_oracle():
    x = inputs.prefill_inputs(workload(), DEV, B=2, T=1000, H=3, seed=21)
    args = (x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"])
    o1, h1 = kda.kda_chunk_fwd_segmented(*args, nseg=4)
    o2, h2 = kda.kda_chunk_fwd_segmented_noalloc(*args, nseg=4)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(h1, h2)  # same kernels, other scratch
    xc = {n: t.cpu() for n, t in x.items()}
    o_ref, h_ref = oracle.prefill(xc["q"], xc["k"], xc["v"], xc["g"], xc["beta"], xc["h0"])
    assert_o(o2, o_ref, torch.bfloat16)
    assert_s(h2, h_ref, torch.bfloat16)


def test_allocates_no_device_memory():
    x = inputs.prefill_inputs(workload(), DEV, B=1, T=2048, H=4, seed=22)
    o = torch.empty_like(x["v"])
    hT = torch.empty(1, 4, 128, 128, device=DEV)
    args = (x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"])
    kda.kda_chunk_fwd_segmented_noalloc(*args, nseg=5, o=o, hT=hT)  # module loaded
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()  # device-wide, whoever allocates
    for _ in range(3):
        kda.kda_chunk_fwd_segmented_noalloc(*args, nseg=5, o=o, hT=hT)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0


def test_oversize_is_rejected_before_launch():
    # 1024 sequences x 2 segments need 1024 x 4 x 64 KB = 256 MB of scratch
    x = inputs.prefill_inputs(workload(), DEV, B=1, T=128, H=1024, seed=23)
    o = torch.zeros_like(x["v"])
    with pytest.raises(kda.KdaError) as ei:
        kda.kda_chunk_fwd_segmented_noalloc(x["q"], x["k"], x["v"], x["g"], x["beta"], None,
                                            nseg=2, o=o)
    assert ei.value.code == kda.KDA_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert torch.count_nonzero(o) == 0  # nothing ran


def test_one_segment_needs_no_scratch():
    x = inputs.prefill_inputs(workload(), DEV, B=1, T=300, H=2, seed=24)
    args = (x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"])
    o1, h1 = kda.kda_chunk_fwd(*args)
    o2, h2 = kda.kda_chunk_fwd_segmented_noalloc(*args, nseg=1)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(h1, h2)
