"""The entry point that allocates nothing, kda_chunk_fwd_segmented_noalloc.

Some callers cannot allocate device memory: a serving runtime that reserved
every byte up front, or an allocator plugin that must not call back into the
allocator running it. For them the segmented prefill keeps its scratch in a
fixed 48 MB array inside the library. These tests call it through the C ABI
and compare it with kda_chunk_fwd_segmented, which takes a caller-allocated
workspace and runs the same kernels: the outputs must agree bit for bit, on
two calls in a row (the array keeps the previous call's contents), and stay
within the bf16 tolerance of the fp64 oracle.

This file is collected last, so a run that stops at the first failure has
already run every other test; it also passes alone in a fresh process (the
first call on the device looks the array's address up).
"""
import pytest
import torch

import oracle
from gated_delta_rule_57_gb300 import inputs, kda
from helpers import assert_o, assert_s

pytestmark = pytest.mark.gpu
DEV = "cuda"
SCRATCH_BYTES = 48 << 20


def workload():
    return inputs.PrefillWorkload("noalloc", 1, 1, 1, 128, 128, "bf16", 0, h0_std=0.02)


def test_two_calls_match_workspace_path_and_oracle():
    x = inputs.prefill_inputs(workload(), DEV, B=2, T=1000, H=3, seed=21)
    args = (x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"])
    o1, h1 = kda.kda_chunk_fwd_segmented(*args, nseg=4)
    torch.cuda.synchronize()
    xc = {n: t.cpu() for n, t in x.items()}
    o_ref, h_ref = oracle.prefill(xc["q"], xc["k"], xc["v"], xc["g"], xc["beta"], xc["h0"])
    for _ in range(2):
        o2, h2 = kda.kda_chunk_fwd_segmented_noalloc(*args, nseg=4)
        torch.cuda.synchronize()
        assert torch.equal(o1, o2) and torch.equal(h1, h2)  # same kernels, other scratch
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


def test_problem_at_the_exact_limit():
    """B=1, H=48, T=768 in 6 segments needs 48 x (3*6 - 2) = 768 states of
    64 KB: exactly the 48 MB array. It runs and equals the workspace path bit
    for bit; one head more (784 states) is rejected before any launch."""
    x = inputs.prefill_inputs(workload(), DEV, B=1, T=768, H=49, seed=25)
    need = kda.kda_chunk_fwd_segmented_workspace_size(1, 768, 48, 128, 128, nseg=6)
    assert need == SCRATCH_BYTES
    sub = {n: (t[:, :, :48].contiguous() if n != "h0" else t[:, :48].contiguous())
           for n, t in x.items()}
    args = (sub["q"], sub["k"], sub["v"], sub["g"], sub["beta"], sub["h0"])
    o1, h1 = kda.kda_chunk_fwd_segmented(*args, nseg=6)
    o2, h2 = kda.kda_chunk_fwd_segmented_noalloc(*args, nseg=6)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(h1, h2)

    assert kda.kda_chunk_fwd_segmented_workspace_size(1, 768, 49, 128, 128, nseg=6) > need
    o = torch.zeros_like(x["v"])
    with pytest.raises(kda.KdaError) as ei:
        kda.kda_chunk_fwd_segmented_noalloc(x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"],
                                            nseg=6, o=o)
    assert ei.value.code == kda.KDA_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert torch.count_nonzero(o) == 0  # nothing ran


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


def test_argument_errors_come_first():
    """An oversize problem with a bad argument (o overlapping q) reports the
    argument, as kda_chunk_fwd_segmented does."""
    x = inputs.prefill_inputs(workload(), DEV, B=1, T=128, H=1024, seed=23)
    with pytest.raises(kda.KdaError) as ei:
        kda.kda_chunk_fwd_segmented_noalloc(x["q"], x["k"], x["v"], x["g"], x["beta"], None,
                                            nseg=2, o=x["q"])
    assert ei.value.code == kda.KDA_ERR_INVALID_ARG


def test_one_segment_needs_no_scratch():
    x = inputs.prefill_inputs(workload(), DEV, B=1, T=300, H=2, seed=24)
    args = (x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"])
    o1, h1 = kda.kda_chunk_fwd(*args)
    o2, h2 = kda.kda_chunk_fwd_segmented_noalloc(*args, nseg=1)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(h1, h2)
