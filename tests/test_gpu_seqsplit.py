"""GPU parity of the sequence-split building blocks (through the C ABI) and of
a sequence split across two processes that share one GPU and exchange their
slice summaries through gloo.

The two processes' kernels never wait on each other: each runs its slice,
then the summaries cross the host in one all-gather, then each runs its scan
and correction."""
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

import oracle
from gated_delta_rule_57_gb300 import inputs, kda
from helpers import assert_o, assert_s

pytestmark = pytest.mark.gpu
DEV = "cuda"
BF16 = torch.bfloat16
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _w(seed, h0=True):
    return inputs.PrefillWorkload("slice", 1, 1, 1, 128, 128, "bf16", seed,
                                  h0_std=0.02 if h0 else None)


def test_slice_transition_matches_oracle():
    """M = the recurrence from the identity with v = 0 (ragged T)."""
    x = inputs.prefill_inputs(_w(41, False), DEV, B=2, T=300, H=2)
    M = kda.kda_chunk_fwd_slice_transition(x["q"], x["k"], x["g"], x["beta"])
    torch.cuda.synchronize()
    xc = {n: x[n].cpu() for n in ("q", "k", "g", "beta")}
    eye = torch.eye(128).expand(2, 2, 128, 128).contiguous()
    _, m_ref = oracle.prefill(xc["q"], xc["k"], torch.zeros_like(xc["q"]), xc["g"], xc["beta"],
                              eye, want_o=False)
    assert_s(M, m_ref, BF16, "transition")


def test_empty_slice_transition_is_identity():
    x = inputs.prefill_inputs(_w(42, False), DEV, B=1, T=0, H=3)
    M = kda.kda_chunk_fwd_slice_transition(x["q"], x["k"], x["g"], x["beta"])
    torch.cuda.synchronize()
    assert torch.equal(M, torch.eye(128, device=DEV).expand(1, 3, 128, 128))


def test_slice_correction_matches_oracle():
    """o += the outputs of the run from S_in with v = 0."""
    x = inputs.prefill_inputs(_w(43), DEV, B=2, T=200, H=2)
    o = torch.zeros_like(x["v"])
    kda.kda_chunk_fwd_slice_correct(x["q"], x["k"], x["g"], x["beta"], x["h0"], o)
    torch.cuda.synchronize()
    xc = {n: x[n].cpu() for n in ("q", "k", "g", "beta", "h0")}
    o_ref, _ = oracle.prefill(xc["q"], xc["k"], torch.zeros_like(xc["q"]), xc["g"], xc["beta"],
                              xc["h0"], want_hT=False)
    assert_o(o, o_ref, BF16, "correction")


def test_state_scan_composes_in_order():
    """X_1 = S0_0, X_{s+1} = S0_s + M_s X_s over 4 slices, fp32 against fp64."""
    gen = torch.Generator(device="cpu").manual_seed(44)
    n, B, H = 4, 2, 3
    s0 = torch.randn(n, B, H, 128, 128, generator=gen) * 0.1
    m = torch.randn(n - 1, B, H, 128, 128, generator=gen) * 0.05
    x_in, hT = kda.kda_state_scan(s0.to(DEV), m.to(DEV))
    torch.cuda.synchronize()
    s0d, md = s0.double().numpy(), m.double().numpy()
    x = s0d[0]
    for s in range(1, n):
        assert np.abs(x_in[s - 1].double().cpu().numpy() - x).max() <= 1e-5 * np.abs(x).max()
        x = s0d[s] + np.einsum("bhij,bhjk->bhik", md[s - 1], x)
    assert np.abs(hT.double().cpu().numpy() - x).max() <= 1e-5 * np.abs(x).max()


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, cuts, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    import torch.distributed as dist
    from gated_delta_rule_57_gb300 import inputs as inp, seqsplit
    dist.init_process_group("gloo", rank=rank, world_size=world)
    torch.cuda.set_device(0)
    x = inp.prefill_inputs(_w(45), "cpu", B=2, T=cuts[-1], H=3)
    t0, t1 = cuts[rank], cuts[rank + 1]
    part = {n: x[n][:, t0:t1].contiguous().to(DEV) for n in ("q", "k", "v", "g", "beta")}
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    o, hT = seqsplit.kda_chunk_fwd_sequence_split(part["q"], part["k"], part["v"], part["g"],
                                                  part["beta"], x["h0"].to(DEV), status=status)
    torch.cuda.synchronize()
    out.put((rank, o.cpu(), hT.cpu(), int(status.item())))
    dist.destroy_process_group()


def test_two_processes_split_one_sequence():
    cuts = [0, 650, 1300]  # 11 + 11 chunks, ragged second slice end
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, cuts, out)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted((out.get(timeout=600) for _ in procs), key=lambda t: t[0])
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert all(r[3] == 0 for r in res)
    x = inputs.prefill_inputs(_w(45), "cpu", B=2, T=cuts[-1], H=3)
    o_ref, h_ref = oracle.prefill(x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"])
    o = torch.cat([r[1] for r in res], dim=1)
    assert_o(o, o_ref, BF16, "split o")
    for r in res:
        assert_s(r[2], h_ref, BF16, f"hT on rank {r[0]}")
