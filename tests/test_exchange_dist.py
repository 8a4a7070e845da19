"""The zipped exchange's host logic on CPU [ZipCCL §2.D: static main streams first, escape streams sized from
n_esc after]: gloo ranks (world 2 and 4) exchange ZC1 streams written by the oracle through
exchange.exchange_streams -- the same code that moves device buffers over NCCL.  Every received main stream,
escape stream and escape count must equal what its sender wrote, byte for byte; pieces differ in size per
pair (ragged), and some are RAW (incompressible data) or have no escapes at all.  Then the reduce-scatter
semantics: rank r receives shard r of every rank, and the oracle's decode-reduce of what arrived must equal the
rank-order fp32 sum of the shards' values (torch), rounded to bf16.  Then the reduce-scatter switcher: its link
profile (timed exchanges) and its choice on a given model.  No kernel runs here; the device path (libzc compress
-> exchange -> zc_decompress_reduce, the codec profile) is checked on the GPU.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

DISJOINT = np.array([1, 2, 3, 4, 5, 6, 7], np.uint8)  # exponents no N(0, 1e-3) value has: every value escapes


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _values(src, dst, m, kind):
    import oracle
    import workloads
    rng = np.random.default_rng(1000 + 16 * src + dst)
    if kind == "exact":  # only codebook exponents: no escapes
        cb = oracle.codebook_from_sigma(1e-3)
        e = cb[rng.integers(0, 7, m)].astype(np.uint16)
        return ((rng.integers(0, 2, m).astype(np.uint16) << 15) | (e << 7) |
                rng.integers(0, 128, m).astype(np.uint16)).astype(np.uint16)
    return workloads.gaussian(m, sigma=1e-3, seed=1000 + 16 * src + dst)


def _stream(src, dst, m, kind):
    """(values, main, escapes) of the piece rank src sends rank dst."""
    import oracle
    x = _values(src, dst, m, kind)
    cb = DISJOINT if kind == "raw" else oracle.codebook_from_sigma(1e-3)
    main, esc, is_raw = oracle.compress_adaptive(x, cb)
    assert is_raw == (kind == "raw")
    return x, main, esc


def _kind(src, dst):
    return ("coded", "raw", "exact")[(src + 2 * dst) % 3]


def _piece_size(src, dst):
    # at least 3 tiles, so that a RAW image is larger than the coded form unless every value escapes
    return 4096 * (3 + (src + 3 * dst) % 3) + 37 * (src + 1) + 5 * dst


def _worker(rank, world, port, q):
    try:
        os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
        dist.init_process_group("gloo", rank=rank, world_size=world)
        import oracle
        from lossless_bf16_exponent_zc_gb300 import exchange
        # 1. pieces of different sizes and kinds, one per pair
        sends = [_stream(rank, p, _piece_size(rank, p), _kind(rank, p)) for p in range(world)]
        mains = [torch.from_numpy(s[1].copy()) for s in sends]
        escs = [torch.from_numpy(np.concatenate([s[2], np.zeros(16, np.uint8)])) for s in sends]
        rm, re, k = exchange.exchange_streams(mains, escs, [oracle.main_bytes(_piece_size(p, rank))
                                                            for p in range(world)])
        for p in range(world):
            x, main, esc = _stream(p, rank, _piece_size(p, rank), _kind(p, rank))
            assert np.array_equal(rm[p].numpy(), main), f"main stream from {p}"
            assert k[p] == esc.size and np.array_equal(re[p][:k[p]].numpy(), esc), f"escapes from {p}"
            assert np.array_equal(oracle.decompress(rm[p].numpy(), re[p][:k[p]].numpy(), x.size), x)
        # 2. reduce-scatter: equal shards of m values; rank r keeps shard r of everyone, summed in rank order
        m = 3 * 4096 + 1000
        shards = [_stream(rank, d, m, "raw" if (rank == 1 and d == 0) else "coded") for d in range(world)]
        mains = [torch.from_numpy(s[1].copy()) for s in shards]
        escs = [torch.from_numpy(np.concatenate([s[2], np.zeros(16, np.uint8)])) for s in shards]
        rm, re, k = exchange.exchange_streams(mains, escs, [oracle.main_bytes(m)] * world)
        y = oracle.decompress_reduce([t.numpy() for t in rm], [re[p][:k[p]].numpy() for p in range(world)], m)
        vals = [_values(p, rank, m, "coded") for p in range(world)]
        acc = torch.from_numpy(vals[0].view(np.int16)).view(torch.bfloat16).float()
        for v in vals[1:]:
            acc = acc + torch.from_numpy(v.view(np.int16)).view(torch.bfloat16).float()
        want = acc.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        assert np.array_equal(y, want), "reduced shard"
        # 3. the switcher's start-up profile of the link: finite, positive and the same on every rank
        bw, lat = exchange.profile_link(device="cpu", large_bytes=1 << 20, reps=3)
        assert np.isfinite(bw) and bw > 0 and np.isfinite(lat) and lat > 0
        got = [None] * world
        dist.all_gather_object(got, (bw, lat))
        assert all(g == (bw, lat) for g in got)
        # and its choice is zc_reduce_scatter_choose's on the model it holds (no device work)
        from lossless_bf16_exponent_zc_gb300 import zc
        codec = (800.0, 600.0, 1.4)
        for link in ((1.0, 5.0), (50.0, 5.0), (1e6, 1.0)):
            sw = exchange.ReduceScatterSwitcher(torch.empty(0), None, None, link=link, codec=codec)
            for nbytes in (1 << 10, 1 << 20, 1 << 28):
                assert sw.zipped(nbytes) == zc.reduce_scatter_choose(nbytes, world, *link, *codec)[0]
        slow = exchange.ReduceScatterSwitcher(torch.empty(0), None, None, link=(1.0, 5.0), codec=codec)
        fast = exchange.ReduceScatterSwitcher(torch.empty(0), None, None, link=(1e6, 1.0), codec=codec)
        assert slow.zipped(1 << 28) and not fast.zipped(1 << 28)
        dist.barrier()
        dist.destroy_process_group()
        q.put((rank, True, ""))
    except Exception:  # reported to the parent, which fails the test
        import traceback
        q.put((rank, False, traceback.format_exc()[-1500:]))


@pytest.mark.parametrize("world", [2, 4])
def test_zipped_exchange_gloo(world):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=300) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
    assert all(ok for _, ok, _ in out), out
    assert [p.exitcode for p in procs] == [0] * world
