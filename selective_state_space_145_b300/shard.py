"""One selective scan split across ranks (torch.distributed): host-side partitioning and the
exchange step; every rank's arithmetic runs through a backend (the CUDA library on GPUs).

Two partitions of one problem:

* By channel. The channels d of a sequence are independent (they share only B and C, which
  every rank reads whole), so rank r scans the channel range partition(dim, W, r) of every
  sequence with no exchange; the outputs and final states are all-gathered along the channel
  axis.

* By sequence segment. Rank r holds tokens [t_r, t_{r+1}) of every sequence ("Mamba",
  ozercemkelahmet.com, "Deployment notes": long prompts are processed in chunks that pass the
  state on). The state after a segment is an affine map of the state before it, per (channel,
  state): h -> exp(A S) h + b, with S the segment's sum of Delta and b its end state from zero,
  and these maps compose associatively. One exchange step:
    1. the conv window each segment starts from (the last d_conv-1 raw inputs before it) is
       all-gathered as each rank's segment tail, and each rank rebuilds its own window;
    2. each rank computes its segment's aggregate (S_r, b_r);
    3. the aggregates are all-gathered (batch * dim * (dstate + 1) floats per rank);
    4. rank r composes the aggregates of segments 0 .. r-1 onto h0 and scans its segment from
       that state. The final state of the whole sequence is the last rank's, broadcast.
  Every rank walks its segment twice (the aggregate, then the scan), as the chunked scan does on
  one GPU with its carry pass.

The backend has three calls, named after the C entry points:
  scan(x, delta, A, B, C, D, z, delta_bias, conv_w, conv_b, conv_init, h0) -> (out, h_last)
  aggregate(x, delta, A, B, delta_bias, conv_w, conv_b, conv_init) -> (S, b)
  compose(S [nseg, batch, dim], b [nseg, batch, dim, dstate], A, h0) -> h
CudaBackend calls libssm; any object with the same methods can stand in (the CPU tests use the
fp64 oracle). Tensors are exchanged with all_gather, so they must live where the process group's
backend expects them (CUDA tensors for NCCL, CPU tensors for gloo).
"""

from __future__ import annotations

from typing import List, Optional, Sequence, Tuple

import torch
import torch.distributed as dist


def partition(n: int, world: int, rank: int) -> Tuple[int, int]:
    """The contiguous range [start, stop) of n items that rank `rank` of `world` owns; the ranges
    tile [0, n) in rank order and their sizes differ by at most one."""
    if world < 1 or not 0 <= rank < world or n < 0:
        raise ValueError(f"bad partition request n={n} world={world} rank={rank}")
    return n * rank // world, n * (rank + 1) // world


class CudaBackend:
    """The per-rank compute on this process's GPU, through libssm."""

    def scan(self, x, delta, A, B, C, D, z, delta_bias, conv_w, conv_b, conv_init, h0):
        from .ssm import ssm_selective_scan_fwd

        return ssm_selective_scan_fwd(x, delta, A, B, C, D, z, delta_bias, True, conv_w, conv_b, conv_init, h0)

    def aggregate(self, x, delta, A, B, delta_bias, conv_w, conv_b, conv_init):
        from .ssm import ssm_selective_scan_aggregate

        return ssm_selective_scan_aggregate(x, delta, A, B, delta_bias, True, conv_w, conv_b, conv_init)

    def compose(self, S, b, A, h0):
        from .ssm import ssm_scan_compose

        return ssm_scan_compose(S, b, A, h0)


def _world(group) -> Tuple[int, int]:
    return dist.get_world_size(group), dist.get_rank(group)


def _all_gather_padded(t: torch.Tensor, dim: int, sizes: Sequence[int], group) -> List[torch.Tensor]:
    """all_gather of tensors that differ only in their size along `dim` (sizes[r] on rank r)."""
    world = len(sizes)
    m = max(sizes) if sizes else 0
    shape = list(t.shape)
    shape[dim] = m
    pad = t.new_zeros(shape)
    pad.narrow(dim, 0, t.shape[dim]).copy_(t)
    bufs = [t.new_empty(shape) for _ in range(world)]
    dist.all_gather(bufs, pad, group=group)
    return [bufs[r].narrow(dim, 0, sizes[r]) for r in range(world)]


def scan_sharded_channels(x, delta, A, B, C, D=None, z=None, delta_bias=None, conv_w=None, conv_b=None,
                          conv_init=None, h0=None, group=None, backend=None, gather: bool = True):
    """Scan of the whole problem (every rank passes the full tensors) with rank r computing the
    channels partition(dim, W, r). Returns (out, h_last): the whole result when gather is True,
    else this rank's channel slice."""
    backend = backend or CudaBackend()
    world, rank = _world(group)
    dim = x.shape[1]
    d0, d1 = partition(dim, world, rank)
    ch = lambda t: None if t is None else t[:, d0:d1].contiguous()
    par = lambda t: None if t is None else t[d0:d1].contiguous()
    out, h_last = backend.scan(ch(x), ch(delta), par(A), B, C, par(D), ch(z), par(delta_bias), par(conv_w),
                               par(conv_b), ch(conv_init), ch(h0))
    if not gather:
        return out, h_last
    sizes = [partition(dim, world, r)[1] - partition(dim, world, r)[0] for r in range(world)]
    out_all = torch.cat(_all_gather_padded(out.contiguous(), 1, sizes, group), dim=1)
    h_all = torch.cat(_all_gather_padded(h_last.contiguous(), 1, sizes, group), dim=1)
    return out_all, h_all


def _window_before(conv_init: Optional[torch.Tensor], tails: Sequence[torch.Tensor], K1: int, like: torch.Tensor):
    """The last K1 raw inputs of the stream conv_init ++ tails[0] ++ tails[1] ++ ... (zeros where
    the stream is shorter), [batch, dim, K1]."""
    batch, dim = like.shape[0], like.shape[1]
    parts = [conv_init if conv_init is not None else like.new_zeros(batch, dim, K1)] + list(tails)
    stream = torch.cat(parts, dim=2)
    return stream[:, :, stream.shape[2] - K1:].contiguous()


def scan_sharded_sequence(x, delta, A, B, C, D=None, z=None, delta_bias=None, conv_w=None, conv_b=None,
                          conv_init=None, h0=None, group=None, backend=None):
    """Scan of one problem whose sequence is split into segments, one per rank in rank order:
    x, delta, z [batch, dim, L_r] and B, C [batch, dstate, L_r] are this rank's segment (the
    segments may differ in length); A, D, delta_bias, conv_w, conv_b and conv_init (the window
    before the whole sequence), h0 (the state before it) are the problem's. Returns (out, h_last):
    this rank's segment of the output, and the state after the whole sequence (on every rank)."""
    backend = backend or CudaBackend()
    world, rank = _world(group)
    batch, dim, L_r = x.shape
    N = A.shape[1]
    # segment lengths of all ranks
    lens_t = torch.tensor([L_r], dtype=torch.int64, device=x.device)
    lens = [torch.zeros_like(lens_t) for _ in range(world)]
    dist.all_gather(lens, lens_t, group=group)
    lens = [int(v.item()) for v in lens]
    # 1. the conv window before this rank's segment, from every earlier segment's raw tail
    seg_init = None
    if conv_w is not None and conv_w.shape[1] > 1:
        K1 = conv_w.shape[1] - 1
        tail = x[:, :, max(0, L_r - K1):]
        tails = _all_gather_padded(tail.contiguous(), 2, [min(K1, n) for n in lens], group)
        seg_init = _window_before(conv_init, tails[:rank], K1, x)
    # 2. this segment's aggregate, 3. everyone's
    S_r, b_r = backend.aggregate(x, delta, A, B, delta_bias, conv_w, conv_b, seg_init)
    S_all = [torch.empty_like(S_r) for _ in range(world)]
    b_all = [torch.empty_like(b_r) for _ in range(world)]
    dist.all_gather(S_all, S_r.contiguous(), group=group)
    dist.all_gather(b_all, b_r.contiguous(), group=group)
    # 4. the state before this segment, then the segment's scan from it
    if rank > 0:
        h_in = backend.compose(torch.stack(S_all[:rank]), torch.stack(b_all[:rank]), A, h0)
    else:
        h_in = h0
    out, h_last = backend.scan(x, delta, A, B, C, D, z, delta_bias, conv_w, conv_b, seg_init, h_in)
    # the state after the whole sequence is the last rank's
    h_final = h_last.contiguous() if rank == world - 1 else b_r.new_empty(batch, dim, N)
    last = world - 1 if group is None else dist.get_global_rank(group, world - 1)
    dist.broadcast(h_final, src=last, group=group)
    return out, h_final
