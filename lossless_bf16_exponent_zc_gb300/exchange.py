"""Zipped collectives over torch.distributed: the two-part exchange of [ZipCCL §2.D].

A compressed tensor travels as the two buffers of the ZC1 format: a main stream whose size follows from the
element count alone, and an escape stream whose size (n_esc, bytes 24..31 of the main stream's header) is
known only once the tensor is compressed.  The static part goes first -- sender and receiver both know its size
before anything moves -- then each side reads the escape counts from the headers it holds (the sender from its
own streams, the receiver from those that just arrived; one host read of 8 bytes per stream, batched) and the
dynamic part follows with exactly those sizes.

Only point-to-point sends and receives are used (torch.distributed.batch_isend_irecv), so the same code moves
device buffers over NCCL and host buffers over gloo.  The codec steps on either side run in libzc's kernels:
compression of all outgoing pieces in one batched launch (with the raw bypass, so an incompressible piece
travels as its own bytes), decompression of all incoming pieces in one batched launch, and, for the
reduce-scatter, the fused decode + fp32 sum in rank order + round to bf16 (+ re-encode) of zc_decompress_reduce.
Sizes handed to a receiver (recv_counts) are the caller's to know, as in any all-to-all: an MoE dispatch
exchanges its token counts first.
"""
from __future__ import annotations

from typing import Sequence

import torch
import torch.distributed as dist

from . import zc

N_ESC_OFFSET = 24  # a ZC1 main stream's header holds n_esc (u64, little-endian) at bytes 24..31


def headers_n_esc(mains: Sequence[torch.Tensor | None]) -> list[int]:
    """n_esc of several main streams with one host read (None -> 0)."""
    present = [m for m in mains if m is not None]
    if not present:
        return [0] * len(mains)
    raw = torch.stack([m[N_ESC_OFFSET:N_ESC_OFFSET + 8] for m in present]).cpu().numpy()
    vals = iter(int.from_bytes(row.tobytes(), "little") for row in raw)
    return [next(vals) if m is not None else 0 for m in mains]


def _peer(p: int, group) -> int:
    return p if group is None else dist.get_global_rank(group, p)


def _run(ops: list) -> None:
    if ops:
        for req in dist.batch_isend_irecv(ops):
            req.wait()


def exchange_streams(send_mains: Sequence[torch.Tensor], send_escs: Sequence[torch.Tensor],
                     recv_main_bytes: Sequence[int], group=None):
    """Send stream p (send_mains[p], send_escs[p]) to rank p and receive one stream from every rank.

    send_mains[p]: a whole main stream (ZC1 header included); send_escs[p]: its escape buffer (at least n_esc
    bytes); recv_main_bytes[p]: the main-stream size of the stream rank p sends here.  The main streams move
    first, then the escape streams, sized from the headers.  Returns (recv_mains, recv_escs, recv_n_esc), each
    indexed by source rank; recv_escs[p] holds exactly recv_n_esc[p] valid bytes (its buffer is at least 16).
    """
    rank, world = dist.get_rank(group), dist.get_world_size(group)
    if not (len(send_mains) == len(send_escs) == len(recv_main_bytes) == world):
        raise ValueError("one stream per rank, each way")
    dev = send_mains[rank].device
    recv_mains = [torch.empty(int(recv_main_bytes[p]), dtype=torch.uint8, device=dev) for p in range(world)]
    ops = []
    for p in range(world):
        if p == rank:
            recv_mains[p].copy_(send_mains[p])
            continue
        ops.append(dist.P2POp(dist.isend, send_mains[p].contiguous(), _peer(p, group), group))
        ops.append(dist.P2POp(dist.irecv, recv_mains[p], _peer(p, group), group))
    _run(ops)
    # the dynamic part's sizes: each side reads the headers it holds
    k_out = headers_n_esc(send_mains)
    k_in = headers_n_esc(recv_mains)
    recv_escs = [torch.empty(max(k_in[p], 16), dtype=torch.uint8, device=dev) for p in range(world)]
    ops = []
    for p in range(world):
        if p == rank:
            if k_in[p]:
                recv_escs[p][:k_in[p]].copy_(send_escs[p][:k_in[p]])
            continue
        if k_out[p]:
            ops.append(dist.P2POp(dist.isend, send_escs[p][:k_out[p]].contiguous(), _peer(p, group), group))
        if k_in[p]:
            ops.append(dist.P2POp(dist.irecv, recv_escs[p][:k_in[p]], _peer(p, group), group))
    _run(ops)
    return recv_mains, recv_escs, k_in


def _compress_pieces(pieces: Sequence[torch.Tensor], cb: torch.Tensor, status: torch.Tensor, ws=None):
    """Every outgoing piece compressed in one batched launch, with the raw bypass."""
    dev = pieces[0].device
    items = []
    for x in pieces:
        n = x.numel()
        mb, _ = zc.compressed_size(n)
        items.append(zc.BatchItem(bf16=x, main=torch.empty(mb, dtype=torch.uint8, device=dev),
                                  esc=torch.empty(max(zc.raw_spill(n), 16), dtype=torch.uint8, device=dev), cb=cb))
    if ws is None:
        ws = zc.workspace([x.numel() for x in pieces], device=dev)
    zc.compress_batched_adaptive(items, ws, status)
    return items


def zipped_all_to_all(chunks: Sequence[torch.Tensor], recv_counts: Sequence[int], cb: torch.Tensor,
                      status: torch.Tensor, ws: torch.Tensor | None = None, group=None) -> list[torch.Tensor]:
    """All-to-all of bf16 pieces, compressed on the wire: chunks[p] goes to rank p, and the piece rank p sends
    here (recv_counts[p] values) comes back decoded, bit for bit.  Device tensors, one codebook for all
    pieces (an MoE payload's histogram codebook, say); ws: a workspace for the pieces (zero-filled once)."""
    world = dist.get_world_size(group)
    if len(chunks) != world or len(recv_counts) != world:
        raise ValueError("one piece per rank, each way")
    items = _compress_pieces(chunks, cb, status, ws)
    recv_mains, recv_escs, k_in = exchange_streams([it.main for it in items], [it.esc for it in items],
                                                   [zc.compressed_size(int(c))[0] for c in recv_counts], group)
    dev = chunks[0].device
    outs = [zc.BatchItem(bf16=torch.empty(int(recv_counts[p]), dtype=torch.int16, device=dev), main=recv_mains[p],
                         esc=recv_escs[p], esc_bytes=k_in[p]) for p in range(world)]
    zc.decompress_batched(outs, status)
    return [o.bf16 for o in outs]


def zipped_reduce_scatter(x: torch.Tensor, cb_in: torch.Tensor, status: torch.Tensor,
                          out_cb: torch.Tensor | None = None, ws: torch.Tensor | None = None, group=None):
    """Reduce-scatter (sum) of a bf16 tensor of P * m values over P ranks, compressed on the wire: shard r
    (values r m .. (r + 1) m - 1) belongs to rank r.  Each rank compresses its P shards, sends shard r to rank
    r, and adds the P shards it receives in rank order 0..P-1 in fp32, rounding once to bf16
    (zc_decompress_reduce).  Returns (the reduced shard, its re-encoded main and escape streams when out_cb is
    given -- ready for a compressed all-gather -- else None, None)."""
    world = dist.get_world_size(group)
    if x.numel() % world:
        raise ValueError("the tensor must split into one shard per rank")
    m = x.numel() // world
    shards = [x[r * m:(r + 1) * m] for r in range(world)]
    if ws is None:
        ws = zc.workspace([m] * world, device=x.device)
    items = _compress_pieces(shards, cb_in, status, ws)
    mb, _ = zc.compressed_size(m)
    recv_mains, recv_escs, k_in = exchange_streams([it.main for it in items], [it.esc for it in items],
                                                   [mb] * world, group)
    out, out_main, out_esc = zc.decompress_reduce(recv_mains, recv_escs, m, status, out_cb=out_cb, ws=ws,
                                                  esc_bytes=k_in)
    return out, out_main, out_esc
