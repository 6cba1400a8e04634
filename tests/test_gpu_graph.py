"""CUDA-graph capture of the library's calls.

No entry point synchronises or allocates (the scratch comes from the caller),
so a sequence of calls can be captured once into a CUDA graph and replayed:
a decode loop, a prefill on the balanced schedule (its flag clear is a memset
node, its launch a cooperative kernel node), a time-split prefill with a
preallocated workspace, and a speculative verify + commit round. Every replay
must give exactly the bits of the same calls run eagerly.
"""
import pytest
import torch

from gated_delta_rule_57_gb300 import inputs, kda

pytestmark = pytest.mark.gpu
DEV = "cuda"


def capture(fn):
    """Warm fn up on a side stream, then capture it into a graph."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    return g


def test_decode_loop_replays_bit_identical():
    w = inputs.DecodeWorkload("graph", 64, 8, 128, 128, "bf16", 41, 16)
    x = inputs.decode_inputs(w, DEV)
    steps = x["q"].shape[0]
    o_e = torch.empty(steps, w.N, w.H, w.dv, dtype=torch.bfloat16, device=DEV)
    S_e = x["S"].clone()
    for t in range(steps):
        kda.kda_decode_step(x["q"][t], x["k"][t], x["v"][t], x["g"][t], x["beta"][t], S_e,
                            o=o_e[t])
    o_g = torch.empty_like(o_e)
    S_g = x["S"].clone()

    def loop():
        for t in range(steps):
            kda.kda_decode_step(x["q"][t], x["k"][t], x["v"][t], x["g"][t], x["beta"][t], S_g,
                                o=o_g[t])

    g = capture(loop)
    S_g.copy_(x["S"])  # the warm-up ran the steps once
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(o_g, o_e) and torch.equal(S_g, S_e)
    # a second replay continues from the state the first one left
    g.replay()
    S2 = S_e.clone()
    for t in range(steps):
        kda.kda_decode_step(x["q"][t], x["k"][t], x["v"][t], x["g"][t], x["beta"][t], S2,
                            o=o_e[t])
    torch.cuda.synchronize()
    assert torch.equal(S_g, S2) and torch.equal(o_g, o_e)


def test_balanced_prefill_replays_bit_identical():
    B, T, H = 2, 1280, 80  # 160 sequences of 20 chunks: the balanced schedule
    w = inputs.PrefillWorkload("graph", B, T, H, 128, 128, "bf16", 42, h0_std=0.02)
    x = inputs.prefill_inputs(w, DEV)
    ws = torch.zeros(kda.kda_chunk_fwd_workspace_size(B, T, H, 128, 128), dtype=torch.uint8,
                     device=DEV)
    o_e, h_e = kda.kda_chunk_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"],
                                 workspace=ws)
    o_g, h_g = torch.empty_like(o_e), torch.empty_like(h_e)
    g = capture(lambda: kda.kda_chunk_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"],
                                          o=o_g, hT=h_g, workspace=ws))
    for _ in range(2):  # the flags are cleared inside the graph before every launch
        o_g.zero_()
        h_g.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(o_g, o_e) and torch.equal(h_g, h_e)


def test_segmented_prefill_replays_bit_identical():
    B, T, H, nseg = 1, 3000, 4, 6
    w = inputs.PrefillWorkload("graph", B, T, H, 128, 128, "bf16", 43, h0_std=0.02)
    x = inputs.prefill_inputs(w, DEV)
    ws = torch.empty(kda.kda_chunk_fwd_segmented_workspace_size(B, T, H, 128, 128, nseg=nseg),
                     dtype=torch.uint8, device=DEV)
    o_e, h_e = kda.kda_chunk_fwd_segmented(x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"],
                                           nseg=nseg, lead=2, workspace=ws)
    o_g, h_g = torch.empty_like(o_e), torch.empty_like(h_e)
    g = capture(lambda: kda.kda_chunk_fwd_segmented(x["q"], x["k"], x["v"], x["g"], x["beta"],
                                                    x["h0"], nseg=nseg, lead=2, o=o_g, hT=h_g,
                                                    workspace=ws))
    o_g.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(o_g, o_e) and torch.equal(h_g, h_e)


def test_speculative_round_replays_bit_identical():
    N, K, H = 16, 4, 8
    w = inputs.PrefillWorkload("graph", N, K, H, 128, 128, "bf16", 44, h0_std=0.02)
    x = inputs.prefill_inputs(w, DEV)
    ntok = torch.tensor([i % (K + 1) for i in range(N)], dtype=torch.int32, device=DEV)
    S_e = x["h0"].clone()
    o_e = kda.kda_decode_multi(x["q"], x["k"], x["v"], x["g"], x["beta"], S_e)
    kda.kda_decode_multi(x["q"], x["k"], x["v"], x["g"], x["beta"], S_e, ntok=ntok,
                         commit=True, want_o=False)
    o_g = torch.empty_like(o_e)
    S_g = x["h0"].clone()

    def rnd():
        kda.kda_decode_multi(x["q"], x["k"], x["v"], x["g"], x["beta"], S_g, o=o_g)
        kda.kda_decode_multi(x["q"], x["k"], x["v"], x["g"], x["beta"], S_g, ntok=ntok,
                             commit=True, want_o=False)

    g = capture(rnd)
    S_g.copy_(x["h0"])
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(o_g, o_e) and torch.equal(S_g, S_e)


def test_device_planned_split_replays_bit_identical():
    """nseg = 0: probe, planning kernel and the three passes, all captured."""
    B, T, H = 1, 4096, 8
    w = inputs.PrefillWorkload("graph", B, T, H, 128, 128, "bf16", 45, h0_std=0.02)
    x = inputs.prefill_inputs(w, DEV)
    ws = torch.empty(kda.kda_chunk_fwd_segmented_workspace_size(B, T, H, 128, 128, nseg=0),
                     dtype=torch.uint8, device=DEV)
    o_e, h_e = kda.kda_chunk_fwd_segmented(x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"],
                                           nseg=0, workspace=ws)
    o_g, h_g = torch.empty_like(o_e), torch.empty_like(h_e)
    g = capture(lambda: kda.kda_chunk_fwd_segmented(x["q"], x["k"], x["v"], x["g"], x["beta"],
                                                    x["h0"], nseg=0, o=o_g, hT=h_g,
                                                    workspace=ws))
    o_g.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(o_g, o_e) and torch.equal(h_g, h_e)
