"""One long sequence split in time across the ranks of a torch.distributed group.

The orkas.ai page "Kimi K3 architecture" (section "The bill arrives in the
serving stack", first bullet) describes how a sequence too long for one device
is split across several: the incoming state of a later slice is not a sum of
per-slice states, but each slice has two composable summaries, its cumulative
transition M and its final state S0 from a zero start; a prefix scan over
them, after one fixed-size all-gather of the summaries, gives every slice its
incoming state. Here rank r of the group holds time slice r of every sequence
(ranks in time order) and runs:

  1. its slice from a zero start (rank 0 from the sequence's h0): o_r, S0_r;
     ranks > 0 also the slice's transition M_r;
  2. one all-gather of the fixed-size pair (S0_r, M_r), 2 x B x H x dk x dv
     fp32 per rank;
  3. the scan over the gathered pairs: every slice's incoming state X_r and
     the sequence's final state hT;
  4. ranks > 0: o_r += the outputs X_r contributes over the slice.

Every step of the arithmetic runs in the library's kernels (``kda.py``); this
module only orders the calls and moves the summaries. The exchange uses the
group's backend: NCCL moves device tensors; with gloo the summaries go
through host memory.
"""
from __future__ import annotations

from typing import Optional

import torch
import torch.distributed as dist

from . import kda


class KernelSteps:
    """The four steps on the GPU, through the C ABI."""

    @staticmethod
    def zero_start(q, k, v, g, beta, h0, status=None):
        return kda.kda_chunk_fwd(q, k, v, g, beta, h0, status=status)

    @staticmethod
    def transition(q, k, g, beta, status=None):
        return kda.kda_chunk_fwd_slice_transition(q, k, g, beta, status=status)

    @staticmethod
    def scan(s0_all, m_rest):
        return kda.kda_state_scan(s0_all, m_rest if m_rest.shape[0] > 0 else None)

    @staticmethod
    def correct(q, k, g, beta, x_in, o, status=None):
        return kda.kda_chunk_fwd_slice_correct(q, k, g, beta, x_in, o, status=status)


def _all_gather(t: torch.Tensor, group) -> list:
    """All-gather of a fixed-size tensor; device tensors go through host
    memory when the group's backend is gloo."""
    backend = dist.get_backend(group)
    world = dist.get_world_size(group)
    src = t if (backend != "gloo" or not t.is_cuda) else t.cpu()
    out = [torch.empty_like(src) for _ in range(world)]
    dist.all_gather(out, src.contiguous(), group=group)
    return [o.to(t.device) for o in out]


def kda_chunk_fwd_sequence_split(q, k, v, g, beta, h0: Optional[torch.Tensor] = None, *,
                                 group=None, status: Optional[torch.Tensor] = None,
                                 steps=KernelSteps):
    """KDA prefill of sequences split in time across the ranks of `group`.

    Rank r passes its own time slice: q, k, g [B, T_r, H, dk], v [B, T_r, H, dv],
    beta [B, T_r, H] (slices in rank order; lengths may differ). h0 [B, H, dk, dv]
    is read on rank 0 only (None: zero state). Returns (o_r, hT): this rank's
    outputs and the sequences' final state (the same on every rank).
    """
    rank = dist.get_rank(group)
    world = dist.get_world_size(group)
    o, s0 = steps.zero_start(q, k, v, g, beta, h0 if rank == 0 else None, status)
    if rank > 0:
        m = steps.transition(q, k, g, beta, status)
    else:
        m = torch.zeros_like(s0)  # slice 0 needs no transition; keeps the exchange fixed-size
    gathered = _all_gather(torch.stack([s0, m]), group)
    s0_all = torch.stack([x[0] for x in gathered])
    m_rest = torch.stack([x[1] for x in gathered[1:]]) if world > 1 else s0_all[:0]
    x_in, hT = steps.scan(s0_all, m_rest)
    if rank > 0:
        o = steps.correct(q, k, g, beta, x_in[rank - 1], o, status)
    return o, hT
