"""The zipped collectives' device path: libzc's batched (adaptive) compression, the two-part exchange over
NCCL, and libzc's decoders on the receiving side [ZipCCL §2.D].  One rank in a spawned child process (a box
here has one GPU, so a rank exchanges with itself only; more ranks are covered on CPU by test_exchange_dist.py),
against the oracle byte for byte: the all-to-all and the all-gather return every piece bit for bit (the
all-gather also from streams the oracle wrote), the reduce-scatter's shard is the oracle's decode-reduce of the
same streams and its re-encoded streams are the oracle's.
"""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

pytestmark = pytest.mark.gpu


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _child(port, q):
    try:
        import torch
        import torch.distributed as dist
        import oracle
        import workloads
        from lossless_bf16_exponent_zc_gb300 import exchange, zc
        torch.cuda.set_device(0)
        os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK="0", WORLD_SIZE="1",
                          NCCL_NVLS_ENABLE="0")
        dist.init_process_group("nccl", rank=0, world_size=1, device_id=torch.device("cuda", 0))
        st = zc.new_status()
        # all-to-all of one piece (ragged, with escapes)
        n = 5 * 4096 + 333
        x = workloads.gradient(n=n, sigma=1e-3, seed=21)
        cb = oracle.codebook_from_sigma(1e-3)
        xt = torch.from_numpy(x.view(np.int16)).cuda()
        (y,) = exchange.zipped_all_to_all([xt], [n], zc.codebook_to_device(cb), st)
        torch.cuda.synchronize()
        assert zc.status_value(st) == 0, zc.status_string(zc.status_value(st))
        assert np.array_equal(y.cpu().numpy().view(np.uint16), x), "all-to-all piece"
        # an incompressible piece travels RAW and still comes back exact
        r = workloads.random_bits(3 * 4096 + 77, seed=22)
        (yr,) = exchange.zipped_all_to_all([torch.from_numpy(r.view(np.int16)).cuda()], [r.size],
                                           zc.codebook_to_device(cb), st)
        torch.cuda.synchronize()
        assert np.array_equal(yr.cpu().numpy().view(np.uint16), r), "RAW piece"
        # all-gather: compressed once, decoded from what arrived (coded and RAW tensors, bf16 dtype kept)
        g = exchange.zipped_all_gather(xt.view(torch.bfloat16), zc.codebook_to_device(cb), st)
        gr = exchange.zipped_all_gather(torch.from_numpy(r.view(np.int16)).cuda(), zc.codebook_to_device(cb), st)
        torch.cuda.synchronize()
        assert zc.status_value(st) == 0, zc.status_string(zc.status_value(st))
        assert np.array_equal(g.cpu().numpy().view(np.uint16), x), "all-gather"
        assert np.array_equal(gr.cpu().numpy().view(np.uint16), r), "all-gather of a RAW tensor"
        # all-gather of streams the oracle wrote (the receiving side decodes them)
        om_, oe_ = oracle.compress(x, cb)
        ga = exchange.all_gather_streams(torch.from_numpy(om_).cuda(),
                                         torch.from_numpy(np.concatenate([oe_, np.zeros(16, np.uint8)])).cuda(), n, st)
        torch.cuda.synchronize()
        assert zc.status_value(st) == 0 and np.array_equal(ga.cpu().numpy().view(np.uint16), x), "oracle streams"
        try:
            exchange.all_gather_streams(torch.from_numpy(om_).cuda(), torch.zeros(16, dtype=torch.uint8).cuda(),
                                        n + 4096, st)
            raise AssertionError("a main stream of another size was accepted")
        except ValueError:
            pass
        # reduce-scatter with a re-encoded output
        m = 7 * 4096 + 5
        s = workloads.gaussian(m, sigma=1e-3, seed=23)
        out_cb = oracle.codebook_from_sigma(1e-3)
        yt, om, oe = exchange.zipped_reduce_scatter(torch.from_numpy(s.view(np.int16)).cuda(),
                                                    zc.codebook_to_device(cb), st,
                                                    out_cb=zc.codebook_to_device(out_cb))
        torch.cuda.synchronize()
        assert zc.status_value(st) == 0, zc.status_string(zc.status_value(st))
        main, esc, _ = oracle.compress_adaptive(s, cb)
        oy, omain, oesc = oracle.decompress_reduce([main], [esc], m, out_cb=out_cb)
        assert np.array_equal(yt.cpu().numpy().view(np.uint16), oy), "reduced shard"
        k = zc.header_n_esc(om)
        assert np.array_equal(om.cpu().numpy(), omain) and np.array_equal(oe[:k].cpu().numpy(), oesc)
        # the switcher on one rank: no link, the codec profiled on a sample, the native path chosen
        bw, lat = exchange.profile_link()
        assert bw == float("inf") and lat == 0.0
        sample = torch.from_numpy(workloads.gaussian(1 << 20, sigma=1e-3, seed=24).view(np.int16)).cuda()
        cgbps, dgbps, ratio = exchange.profile_codec(sample, zc.codebook_to_device(cb), st, P=4, reps=3)
        sm, se = oracle.compress(sample.cpu().numpy().view(np.uint16), cb)
        assert cgbps > 0 and dgbps > 0 and abs(ratio - 2 * (1 << 20) / (sm.size + se.size)) < 1e-9
        sw = exchange.ReduceScatterSwitcher(sample, zc.codebook_to_device(cb), st)
        assert not sw.zipped(1 << 30)
        assert torch.equal(sw(sample), sample)  # one rank: its shard is the whole tensor
        torch.cuda.synchronize()
        assert zc.status_value(st) == 0
        dist.destroy_process_group()
        q.put((True, ""))
    except Exception:
        import traceback
        q.put((False, traceback.format_exc()[-2000:]))


def test_zipped_collectives_one_rank_nccl():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    p = ctx.Process(target=_child, args=(_free_port(), q))
    p.start()
    ok, msg = q.get(timeout=600)
    p.join(timeout=120)
    assert ok, msg
    assert p.exitcode == 0
