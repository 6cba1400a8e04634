"""A sequence split in time across ranks (seqsplit.py), host logic on CPU.

Two and three gloo ranks each take one time slice of the same seeded
sequences and run kda_chunk_fwd_sequence_split with the kernel steps replaced
by the fp64 oracle (run from a zero start, from the identity with v = 0, from
an incoming state with v = 0, and the composition X_{s+1} = S0_s + M_s X_s
written out in numpy). The concatenated outputs and the final state must
equal the oracle over the whole sequence, which checks the slice order, the
all-gather of the summaries, the order of composition in the scan and where
the correction is added. The GPU version of the same run is in
test_gpu_seqsplit.py.
"""
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


class OracleSteps:
    """CPU stand-in for the four kernel steps, from the fp64 oracle."""

    @staticmethod
    def zero_start(q, k, v, g, beta, h0, status=None):
        import oracle
        o, hT = oracle.prefill(q, k, v, g, beta, h0)
        return torch.from_numpy(o), torch.from_numpy(hT)

    @staticmethod
    def transition(q, k, g, beta, status=None):
        import oracle
        B, T, H, dk = q.shape
        eye = torch.eye(dk, dtype=torch.float32).expand(B, H, dk, dk).contiguous()
        _, m = oracle.prefill(q, k, torch.zeros_like(q), g, beta, eye, want_o=False)
        return torch.from_numpy(m)

    @staticmethod
    def scan(s0_all, m_rest):
        s0 = s0_all.numpy()
        x = s0[0]
        x_in = []
        for s in range(1, s0.shape[0]):
            x_in.append(x)
            x = s0[s] + np.einsum("bhij,bhjk->bhik", m_rest[s - 1].numpy(), x)
        xs = torch.from_numpy(np.stack(x_in)) if x_in else None
        return xs, torch.from_numpy(x)

    @staticmethod
    def correct(q, k, g, beta, x_in, o, status=None):
        import oracle
        oc, _ = oracle.prefill(q, k, torch.zeros_like(q), g, beta, x_in.float(), want_hT=False)
        return o + torch.from_numpy(oc)


def _inputs(B, T, H, d):
    from gated_delta_rule_57_gb300 import inputs
    w = inputs.PrefillWorkload("split", B, T, H, d, d, "f32", 31, h0_std=0.02)
    return inputs.prefill_inputs(w, "cpu")


def _worker(rank, world, port, cuts, shape, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    import torch.distributed as dist
    from gated_delta_rule_57_gb300 import seqsplit
    dist.init_process_group("gloo", rank=rank, world_size=world)
    x = _inputs(*shape)
    t0, t1 = cuts[rank], cuts[rank + 1]
    part = {n: x[n][:, t0:t1].contiguous() for n in ("q", "k", "v", "g", "beta")}
    o, hT = seqsplit.kda_chunk_fwd_sequence_split(part["q"], part["k"], part["v"], part["g"],
                                                  part["beta"], x["h0"], steps=OracleSteps)
    out.put((rank, o.numpy(), hT.numpy()))
    dist.destroy_process_group()


@pytest.mark.parametrize("cuts", [[0, 90, 150], [0, 40, 41, 150]])
def test_split_equals_whole_sequence(cuts):
    import oracle
    shape = (2, 150, 2, 16)
    world = len(cuts) - 1
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, cuts, shape, out))
             for r in range(world)]
    for p in procs:
        p.start()
    res = sorted((out.get(timeout=300) for _ in procs), key=lambda t: t[0])
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    x = _inputs(*shape)
    o_ref, h_ref = oracle.prefill(x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"])
    o = np.concatenate([r[1] for r in res], axis=1)
    assert o.shape == o_ref.shape
    assert np.abs(o - o_ref).max() <= 1e-5 * np.abs(o_ref).max()
    for r in res:  # every rank gets the final state
        assert np.linalg.norm(r[2] - h_ref) <= 1e-5 * np.linalg.norm(h_ref)
