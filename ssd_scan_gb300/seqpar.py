"""Sequence-parallel prefill: one sequence's rows split over the ranks of a
process group (one GPU each), chained by state passing.

TensorRT-Model-Connect #2207 "Implementation" gives the chunk form, in which
a chunk's total decay is the last element of its cumulative sum of a = dt A
and the state carries from chunk to chunk as h <- exp(min(gamma_S, 0)) h +
the chunk's own terms.  With a whole segment of rows in the role of the
chunk, every rank can scan its segment before it knows the state at its
start:

1. conv halo: rank k's conv state is the last W-1 raw rows of rank k-1's
   segment (rank 0: the sequence's conv state) -- an all-gather of W-1 rows;
2. pass 1: scan the segment from a zero SSM state -> its own contribution
   h_k, and its total decay Gamma_k (``ssd_segment_decay``);
3. exchange: all-gather (Gamma_k, h_k); every rank chains them in rank order,
   h_in_0 = h0, h_in_{k+1} = exp(min(Gamma_k, 0)) h_in_k + h_k
   (``ssd_state_combine``), so it knows its own h_in_k and the final state;
4. pass 2: scan the segment again from h_in_k -> its rows of y.

The second pass redoes the first one's work; its cost buys the parallelism
(each rank scans S/K rows twice instead of one rank scanning S).  The one
collective is the all-gather of [B,H,P,N] fp32 states (4 MiB per sequence at
the Nemotron-H shape) and of [B,H] decays and [B,W-1,Cdim] halos.

The per-rank steps are the CUDA library's by default (``cuda_ops``); they are
parameters so that the exchange can be exercised with other implementations
of the same three steps.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Callable

import torch


@dataclass
class SegmentOps:
    """The three per-rank steps.

    scan(xbc, dt, z, h0, conv_state) -> (y, h_final, conv_state_out)
        one prefill call over the rows of a segment (h0 None: zeros);
    decay(dt) -> gamma [B,H]: the segment's total decay;
    combine(gamma, h_prev, h_seg) -> exp(min(gamma, 0)) h_prev + h_seg.
    """
    scan: Callable
    decay: Callable
    combine: Callable


def cuda_ops(A, *, nheads, headdim, dstate, ngroups, conv_w=None, conv_b=None, dt_bias=None,
             D=None, dt_softplus=True, stream=None) -> SegmentOps:
    """The steps on this library's kernels (device tensors)."""
    import ssd_scan_gb300 as ssd

    def scan(xbc, dt, z, h0, conv_state):
        return ssd.chunk_scan(xbc, dt, A, nheads=nheads, headdim=headdim, dstate=dstate,
                              ngroups=ngroups, conv_w=conv_w, conv_b=conv_b,
                              conv_state=conv_state, dt_bias=dt_bias, D=D, z=z, ssm_state=h0,
                              dt_softplus=dt_softplus, stream=stream)

    def decay(dt):
        B, S, H = dt.shape
        g = torch.empty((B, H), dtype=torch.float32, device=dt.device)
        ssd.ssd_segment_decay(ssd.dims(B, S, H, headdim, dstate, ngroups),
                              ssd.SSD_DT_SOFTPLUS if dt_softplus else 0, dt, dt_bias, A, g,
                              stream)
        return g

    def combine(gamma, h_prev, h_seg):
        B, H = gamma.shape
        out = torch.empty_like(h_seg)
        ssd.ssd_state_combine(ssd.dims(B, 0, H, headdim, dstate, ngroups), gamma, h_prev,
                              h_seg, out, stream)
        return out

    return SegmentOps(scan, decay, combine)


def halo_rows(xbc, width):
    """The last width-1 raw rows of a segment: the next segment's conv state."""
    if xbc.shape[1] < width - 1:
        raise ValueError(f"a segment needs at least {width - 1} rows (conv width {width})")
    return xbc[:, xbc.shape[1] - (width - 1):].contiguous()


def pass1(ops: SegmentOps, xbc, dt, z, conv_state):
    """A segment from a zero state: (Gamma_k, h_k)."""
    _, h_k, _ = ops.scan(xbc, dt, z, None, conv_state)
    return ops.decay(dt), h_k


def chain(ops: SegmentOps, gammas, h_segs, h0):
    """h_in_0 = h0; h_in_{k+1} = combine(Gamma_k, h_in_k, h_k).  Returns the
    K+1 states h_in_0 .. h_in_K (the last one: the sequence's final state)."""
    h = [h0]
    for g, hk in zip(gammas, h_segs):
        h.append(ops.combine(g, h[-1], hk))
    return h


def sequence_parallel_scan(ops: SegmentOps, xbc, dt, z=None, h0=None, conv_state=None,
                           conv_width=4, group=None):
    """This rank's rows of one prefill, sequence-parallel over ``group``.

    xbc [B,S_k,Cdim], dt [B,S_k,H], z [B,S_k,H*P] or None: this rank's segment
    (the ranks' segments in rank order make up the sequences); h0, conv_state:
    the sequences' initial states, the same on every rank (None: zeros).
    Returns (y of this segment, the sequences' final SSM state, the final conv
    state), the last two the same on every rank."""
    import torch.distributed as dist

    rank, world = dist.get_rank(group), dist.get_world_size(group)
    conv = conv_width > 1
    # 1. conv halos
    cs_in = conv_state
    halos = None
    if conv:
        mine = halo_rows(xbc, conv_width)
        halos = [torch.empty_like(mine) for _ in range(world)]
        dist.all_gather(halos, mine, group=group)
        if rank > 0:
            cs_in = halos[rank - 1]
    # 2. pass 1 from a zero state
    g_k, h_k = pass1(ops, xbc, dt, z, cs_in)
    # 3. exchange and chain in rank order
    gs = [torch.empty_like(g_k) for _ in range(world)]
    hs = [torch.empty_like(h_k) for _ in range(world)]
    dist.all_gather(gs, g_k.contiguous(), group=group)
    dist.all_gather(hs, h_k.contiguous(), group=group)
    h_in = chain(ops, gs, hs, h0)
    # 4. pass 2 from this segment's initial state
    y, _, _ = ops.scan(xbc, dt, z, h_in[rank], cs_in)
    return y, h_in[world], (halos[world - 1] if conv else None)
