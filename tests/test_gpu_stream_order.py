"""Stream order holds for data across the library's programmatic dependent launches.

Every libzc kernel may be placed on the GPU while the kernel before it on the
stream is still running, and waits (griddepcontrol.wait) before it touches
global memory.  These chains enqueue many launches back to back with no host
synchronisation in between and check every result at the end, so a kernel
that read its input before the producer finished (read after write), or
overwrote a buffer that the previous kernel was still reading (write after
read), would show up as a wrong byte:

* a torch kernel writes the input right before each compress;
* compress -> decompress -> compress of the decoded tensor, six times over;
* histogram -> compress with the codebook the histogram just wrote;
* one main / escape buffer pair reused by every round of compress + decompress;
* decompress -> decompress_reduce -> re-encoded stream -> decompress;
* compress on one stream, decompress on another after an event;
* the benchmark's step (histogram, compress with the histogram's and with
  the sigma codebook, both decompressed) hundreds of times on one
  workspace, back to back and with a synchronisation after every call: the
  escape scan's per-launch state (epoch, counters) is handed from launch to
  launch, and a slip there shows up as escape offsets that no longer match
  the code planes, which the decoder reports.
"""
import math

import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu

N = 1 << 24  # 32 MB of bf16 per tensor: kernels long enough to overlap if ordering broke


def _inputs(k, seed):
    return [workloads.gaussian_on_device(N, 1e-3 * (1 + i), seed=seed + i) for i in range(k)]


def _check_status(zc, st):
    torch.cuda.synchronize()
    assert zc.status_value(st) == 0, zc.status_string(zc.status_value(st))


def test_torch_write_then_compress(zc):
    xs = _inputs(6, 100)
    buf = torch.empty_like(xs[0])
    cb = zc.codebook_to_device(oracle.codebook_from_sigma(2e-3))
    st, ws = zc.new_status(), zc.workspace(N)
    streams = []
    for x in xs:
        buf.copy_(x)  # a torch kernel writes the input, then the encoder reads it
        streams.append(zc.compress(buf, cb, ws, st))
        buf.zero_()  # and a torch kernel overwrites it right after
    outs = [zc.decompress(m, e, N, st) for m, e in streams]
    _check_status(zc, st)
    for x, y in zip(xs, outs):
        assert torch.equal(y, x)


def test_codec_chain(zc):
    (x,) = _inputs(1, 200)
    cb = zc.codebook_to_device(oracle.codebook_from_sigma(1e-3))
    st, ws = zc.new_status(), zc.workspace(N)
    y = x
    for _ in range(6):
        m, e = zc.compress(y, cb, ws, st)
        y = zc.decompress(m, e, N, st)
    _check_status(zc, st)
    assert torch.equal(y, x)


def test_histogram_then_compress(zc):
    xs = _inputs(4, 300)
    st, ws = zc.new_status(), zc.workspace(N)
    cbs, streams = [], []
    for x in xs:
        cb = torch.empty(7, dtype=torch.uint8, device="cuda")
        zc.histogram_topk(x, ws, st, cb_out=cb)  # writes cb; the encoder reads it next
        cbs.append(cb)
        streams.append(zc.compress(x, cb, ws, st))
    outs = [zc.decompress(m, e, N, st) for m, e in streams]
    _check_status(zc, st)
    for x, cb, (m, _), y in zip(xs, cbs, streams, outs):
        assert torch.equal(y, x)
        want_cb, _ = oracle.histogram_topk(x.cpu().numpy().view("u2"))
        assert bytes(cb.cpu().numpy()) == bytes(want_cb)
        assert bytes(m[32:39].cpu().numpy()) == bytes(want_cb)  # the encoder read the codebook just written


def test_buffers_reused_every_round(zc):
    xs = _inputs(6, 400)
    cb = zc.codebook_to_device(oracle.codebook_from_sigma(3e-3))
    st, ws = zc.new_status(), zc.workspace(N)
    main, esc = zc.compress(xs[0], cb, ws, st)
    outs = []
    for x in xs:
        zc.compress(x, cb, ws, st, main=main, esc=esc)  # overwrites what the last decompress read
        outs.append(zc.decompress(main, esc, N, st))
    _check_status(zc, st)
    for x, y in zip(xs, outs):
        assert torch.equal(y, x)


def test_reduce_chain(zc):
    P = 4
    xs = _inputs(P, 500)
    cb = zc.codebook_to_device(oracle.codebook_from_sigma(2e-3))
    cb_out = zc.codebook_to_device(oracle.codebook_from_sigma(2e-3 * math.sqrt(P)))
    st, ws = zc.new_status(), zc.workspace(N)
    shards = [zc.compress(x, cb, ws, st) for x in xs]
    y, om, oe = zc.decompress_reduce([m for m, _ in shards], [e for _, e in shards], N, st, out_cb=cb_out, ws=ws)
    z = zc.decompress(om, oe, N, st)  # decodes the stream the reduce just wrote
    _check_status(zc, st)
    assert torch.equal(z, y)
    # the reduction itself, on a slice the oracle finishes quickly
    k = 3 * 4096 + 5
    want = oracle.reduce([x[:k].cpu().numpy().view("u2") for x in xs])
    assert (y[:k].cpu().numpy().view("u2") == want).all()


def test_cross_stream_event(zc):
    xs = _inputs(3, 600)
    cb = zc.codebook_to_device(oracle.codebook_from_sigma(2e-3))
    st, ws = zc.new_status(), zc.workspace(N)
    s_enc, s_dec = torch.cuda.Stream(), torch.cuda.Stream()
    s_enc.wait_stream(torch.cuda.current_stream())
    outs = []
    for x in xs:
        with torch.cuda.stream(s_enc):
            m, e = zc.compress(x, cb, ws, st)
            ev = torch.cuda.Event()
            ev.record(s_enc)
        s_dec.wait_event(ev)
        with torch.cuda.stream(s_dec):
            outs.append(zc.decompress(m, e, N, st))
            m.record_stream(s_dec)
            e.record_stream(s_dec)
    torch.cuda.current_stream().wait_stream(s_dec)
    _check_status(zc, st)
    for x, y in zip(xs, outs):
        assert torch.equal(y, x)


def test_long_runs_of_the_benchmark_step(zc):
    n = 1 << 26
    # the benchmark's own tensor: N(0, 1e-3) with outliers and special values
    x = torch.from_numpy(workloads.gradient().view("int16")).cuda()
    cb_sig = zc.codebook_to_device(oracle.codebook_from_sigma(1e-3))
    cb_hist = torch.empty(7, dtype=torch.uint8, device="cuda")
    st, ws = zc.new_status(), zc.workspace(n)
    mb, eb = zc.compressed_size(n)
    ma, mb_ = torch.empty(mb, dtype=torch.uint8, device="cuda"), torch.empty(mb, dtype=torch.uint8, device="cuda")
    ea, eb_ = torch.empty(eb, dtype=torch.uint8, device="cuda"), torch.empty(eb, dtype=torch.uint8, device="cuda")
    ya, yb = torch.empty_like(x), torch.empty_like(x)

    def step():
        zc.histogram_topk(x, ws, st, cb_out=cb_hist)
        zc.compress(x, cb_hist, ws, st, main=ma, esc=ea)
        zc.compress(x, cb_sig, ws, st, main=mb_, esc=eb_)
        zc.decompress(ma, ea, n, st, out=ya)
        zc.decompress(mb_, eb_, n, st, out=yb)

    for _ in range(300):
        step()
    _check_status(zc, st)
    for _ in range(100):
        for call in (lambda: zc.histogram_topk(x, ws, st, cb_out=cb_hist),
                     lambda: zc.compress(x, cb_hist, ws, st, main=ma, esc=ea),
                     lambda: zc.compress(x, cb_sig, ws, st, main=mb_, esc=eb_),
                     lambda: zc.decompress(ma, ea, n, st, out=ya),
                     lambda: zc.decompress(mb_, eb_, n, st, out=yb)):
            call()
            _check_status(zc, st)
    assert torch.equal(ya, x) and torch.equal(yb, x)
    # the last streams are the ones a fresh workspace gives
    ws2, st2 = zc.workspace(n), zc.new_status()
    for cb, m in ((cb_hist, ma), (cb_sig, mb_)):
        rm, _ = zc.compress(x, cb, ws2, st2)
        _check_status(zc, st2)
        assert torch.equal(rm, m)
