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
The all-gather sends one rank's streams to every rank (zipped_all_gather compresses first; all_gather_streams
takes streams a rank already holds, such as a reduce-scatter's re-encoded shard).
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


def all_gather_streams(main: torch.Tensor, esc: torch.Tensor, n: int, status: torch.Tensor,
                       out: torch.Tensor | None = None, group=None) -> torch.Tensor:
    """All-gather of a tensor already compressed: every rank holds the streams of its own n values (a ZC1 main
    stream and its escape buffer, coded or RAW), sends them to every rank and decodes the streams of all ranks
    in one batched launch.  Returns (or fills) world * n bf16 bit patterns (int16), rank r's values at
    [r n, (r + 1) n).  Every rank's piece has n values, so every main stream has the size the size law
    gives for n; the escape streams follow with the sizes their headers hold."""
    world = dist.get_world_size(group)
    mb, _ = zc.compressed_size(n)
    if main.numel() != mb:
        raise ValueError("the main stream does not hold n values")
    recv_mains, recv_escs, k_in = exchange_streams([main] * world, [esc] * world, [mb] * world, group)
    if out is None:
        out = torch.empty(world * n, dtype=torch.int16, device=main.device)
    elif out.numel() != world * n:
        raise ValueError("out must hold world * n values")
    zc.decompress_batched([zc.BatchItem(bf16=out[r * n:(r + 1) * n], main=recv_mains[r], esc=recv_escs[r],
                                        esc_bytes=k_in[r]) for r in range(world)], status)
    return out


def zipped_all_gather(x: torch.Tensor, cb: torch.Tensor, status: torch.Tensor, ws: torch.Tensor | None = None,
                      out: torch.Tensor | None = None, group=None) -> torch.Tensor:
    """All-gather of bf16 tensors of equal size, compressed on the wire: each rank compresses its x once (with
    the raw bypass, so an incompressible tensor travels as its own bytes), sends the streams to every rank, and
    every rank decodes all of them in one batched launch.  Returns world * x.numel() bf16 bit patterns (int16),
    rank r's tensor at [r n, (r + 1) n), bit for bit."""
    n = x.numel()
    (item,) = _compress_pieces([x.reshape(-1)], cb, status, ws)
    return all_gather_streams(item.main, item.esc, n, status, out=out, group=group)


# ------------------------------------------------------------------ the reduce-scatter switcher [ZipCCL §2.D]
def _max_over(value: float, group, device) -> float:
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX, group=group)
    return float(t.item())


def profile_link(group=None, small_bytes: int = 1 << 10, large_bytes: int = 1 << 24, reps: int = 5,
                 device=None) -> tuple[float, float]:
    """(bandwidth in GB/s per rank and direction, latency in us) of the group's point-to-point path, measured the
    way the zipped exchange moves data: every rank exchanges one message with every other rank at once
    (batch_isend_irecv), once with a small message (its time is the latency) and once with a large one (the extra
    bytes over the extra time give the bandwidth).  Each time is the median of `reps` exchanges after one untimed
    one, taken as the slowest rank's (so every rank gets the same model).  device: where the buffers live (the
    current CUDA device for NCCL, the CPU for gloo).  A group of one rank has no link: (inf, 0)."""
    import statistics
    import time
    rank, world = dist.get_rank(group), dist.get_world_size(group)
    if world == 1:
        return float("inf"), 0.0
    if device is None:
        device = torch.device("cuda", torch.cuda.current_device()) if dist.get_backend(group) == "nccl" else "cpu"
    on_gpu = torch.device(device).type == "cuda"

    def exchange_time(nbytes: int) -> float:
        send = [torch.zeros(nbytes, dtype=torch.uint8, device=device) for _ in range(world)]
        recv = [torch.empty(nbytes, dtype=torch.uint8, device=device) for _ in range(world)]
        ops = [op for p in range(world) if p != rank
               for op in (dist.P2POp(dist.isend, send[p], _peer(p, group), group),
                          dist.P2POp(dist.irecv, recv[p], _peer(p, group), group))]
        times = []
        for i in range(reps + 1):
            dist.barrier(group=group)
            if on_gpu:
                torch.cuda.synchronize()
            t0 = time.perf_counter()
            _run(ops)
            if on_gpu:
                torch.cuda.synchronize()
            if i:
                times.append(time.perf_counter() - t0)
        return _max_over(statistics.median(times), group, device)

    t_small = exchange_time(small_bytes)
    t_large = exchange_time(large_bytes)
    extra = (world - 1) * (large_bytes - small_bytes)  # bytes each rank sends beyond the small exchange
    bandwidth = extra / max(t_large - t_small, 1e-9) / 1e9
    return bandwidth, t_small * 1e6


def profile_codec(sample: torch.Tensor, cb: torch.Tensor, status: torch.Tensor, P: int = 8,
                  reps: int = 10) -> tuple[float, float, float]:
    """(compress GB/s, decode-reduce GB/s, ratio) of libzc on a sample of the caller's data (a bf16 device tensor):
    compress throughput of the sample's 2n bytes, zc_decompress_reduce throughput over P copies of its stream per
    byte of the P inputs (the figure the reduce-scatter model takes for the receiving side), and the ratio 2n /
    (main stream + escapes).  CUDA events on the current stream."""
    n = sample.numel()
    ws = zc.workspace(n, device=sample.device)
    main, esc = zc.compress(sample, cb, ws, status)
    k = zc.header_n_esc(main)

    def timed(fn) -> float:
        fn()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        for _ in range(reps):
            fn()
        e.record()
        e.synchronize()
        return s.elapsed_time(e) / reps * 1e-3  # seconds

    t_c = timed(lambda: zc.compress(sample, cb, ws, status, main=main, esc=esc))
    out = torch.empty(n, dtype=torch.int16, device=sample.device)
    t_d = timed(lambda: zc.decompress_reduce([main] * P, [esc] * P, n, status, out=out, esc_bytes=[k] * P))
    return 2 * n / t_c / 1e9, 2 * n * P / t_d / 1e9, 2 * n / (main.numel() + k)


class ReduceScatterSwitcher:
    """The reduce-scatter switcher of [ZipCCL §2.D]: it profiles the link (bandwidth, latency) and the codec
    (throughput, ratio on a sample of the caller's data) once, when it is made, and then for each tensor picks
    the native reduce-scatter (torch.distributed.reduce_scatter_tensor, summed the collective library's way) or
    the zipped one (zipped_reduce_scatter: fp32 sums in rank order, one rounding) by zc_reduce_scatter_choose's two
    time estimates.  link / codec: measured figures to use instead of profiling ((GB/s, us) and (GB/s, GB/s,
    ratio))."""

    def __init__(self, sample: torch.Tensor, cb: torch.Tensor, status: torch.Tensor, group=None,
                 link: tuple[float, float] | None = None, codec: tuple[float, float, float] | None = None):
        self.group, self.cb, self.status = group, cb, status
        self.world = dist.get_world_size(group)
        self.link = link if link is not None else profile_link(group, device=sample.device)
        self.codec = codec if codec is not None else profile_codec(sample, cb, status, P=max(self.world, 1))

    def zipped(self, nbytes: int) -> bool:
        """True when the zipped reduce-scatter of nbytes per rank is estimated to be faster (one rank: never)."""
        if self.world == 1:
            return False
        z, _, _ = zc.reduce_scatter_choose(int(nbytes), self.world, self.link[0], self.link[1], *self.codec)
        return z

    def __call__(self, x: torch.Tensor, out_cb: torch.Tensor | None = None, ws: torch.Tensor | None = None):
        """Reduce-scatter (sum) of x (bf16 bits, P * m values) over the group; returns this rank's shard."""
        if self.zipped(2 * x.numel()):
            return zipped_reduce_scatter(x, self.cb, self.status, out_cb=out_cb, ws=ws, group=self.group)[0]
        m = x.numel() // self.world
        out = torch.empty(m, dtype=torch.bfloat16, device=x.device)
        dist.reduce_scatter_tensor(out, x.view(torch.bfloat16), group=self.group)
        return out.view(torch.int16)
