"""Device-side error reporting: corrupt or inconsistent streams, escape overflow, bad codebooks and the
bounded inter-block wait.  Every failure is produced on the host (corrupted bytes, the workspace's hold hook);
nothing here faults or hangs the GPU: kernels finish and report through the status word."""
import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu


def dev(x):
    return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).cuda()


def _stream(zc, n=3 * 4096 + 100, seed=1):
    x = workloads.gradient(n=n, sigma=1e-3, seed=seed)
    cb = oracle.codebook_from_sigma(1e-3)
    st = zc.new_status()
    main, esc = zc.compress(dev(x), zc.codebook_to_device(cb), zc.workspace(n), st)
    torch.cuda.synchronize()
    assert zc.status_value(st) == 0
    return x, cb, main, esc


def _decode_status(zc, main, esc, n, esc_bytes=None):
    st = zc.new_status()
    out = torch.full((n,), 0x1234, dtype=torch.int16, device="cuda")
    zc.decompress(main, esc, n, st, out=out, esc_bytes=esc_bytes)
    torch.cuda.synchronize()
    return zc.status_value(st), out


def test_bad_magic_writes_nothing(zc):
    x, cb, main, esc = _stream(zc)
    bad = main.clone()
    bad[0] ^= 1
    code, out = _decode_status(zc, bad, esc, x.size)
    assert code == zc.ERR_BAD_HEADER
    assert bool((out == 0x1234).all())


def test_size_mismatch(zc):
    x, cb, main, esc = _stream(zc)
    code, _ = _decode_status(zc, main, esc, x.size + 1)   # same tile count, different n
    assert code == zc.ERR_SIZE_MISMATCH


def test_escape_count_beyond_buffer(zc):
    x, cb, main, esc = _stream(zc)
    n_esc = zc.header_n_esc(main)
    code, _ = _decode_status(zc, main, esc, x.size, esc_bytes=n_esc - 1)
    assert code == zc.ERR_BAD_HEADER


def test_corrupt_offset_table(zc):
    x, cb, main, esc = _stream(zc)
    bad = main.clone()
    bad[128 + 4:128 + 8] = torch.tensor(list((10 ** 6).to_bytes(4, "little")), dtype=torch.uint8, device="cuda")
    code, _ = _decode_status(zc, bad, esc, x.size)
    assert code == zc.ERR_CORRUPT_STREAM


def test_offsets_inconsistent_with_planes(zc):
    """Tile 1 claims one escape fewer than its planes hold: detected, and no read leaves the escape range."""
    x, cb, main, esc = _stream(zc)
    bad = main.clone()
    off = int.from_bytes(bad[128 + 8:128 + 12].cpu().numpy().tobytes(), "little")
    bad[128 + 8:128 + 12] = torch.tensor(list((off - 1).to_bytes(4, "little")), dtype=torch.uint8, device="cuda")
    code, _ = _decode_status(zc, bad, esc, x.size)
    assert code == zc.ERR_CORRUPT_STREAM


def test_duplicate_codebook_in_header(zc):
    x, cb, main, esc = _stream(zc)
    bad = main.clone()
    bad[33] = bad[32]
    code, _ = _decode_status(zc, bad, esc, x.size)
    assert code == zc.ERR_BAD_HEADER


def test_escape_overflow_keeps_exact_count(zc):
    x = workloads.gradient(n=5 * 4096 + 9, sigma=1e-3, seed=3)
    cb = oracle.codebook_from_sigma(1e-3)
    om, oe = oracle.compress(x, cb)
    cap = 48     # 16-byte multiple, far below the escape count
    st = zc.new_status()
    main = torch.empty(om.size, dtype=torch.uint8, device="cuda")
    esc = torch.zeros(cap, dtype=torch.uint8, device="cuda")
    zc.compress(dev(x), zc.codebook_to_device(cb), zc.workspace(x.size), st, main=main, esc=esc)
    torch.cuda.synchronize()
    assert zc.status_value(st) == zc.ERR_ESCAPE_OVERFLOW
    assert zc.header_n_esc(main) == oe.size
    assert np.array_equal(main.cpu().numpy(), om)
    assert np.array_equal(esc.cpu().numpy(), oe[:cap])


def test_duplicate_device_codebook(zc):
    x = workloads.gradient(n=4096, seed=4)
    st = zc.new_status()
    main = torch.full((zc.compressed_size(x.size)[0],), 0xAB, dtype=torch.uint8, device="cuda")
    zc.compress(dev(x), zc.codebook_to_device([1, 2, 3, 4, 5, 6, 6]), zc.workspace(x.size), st, main=main)
    torch.cuda.synchronize()
    assert zc.status_value(st) == zc.ERR_DUP_CODEBOOK
    assert bool((main == 0xAB).all())


def test_reduce_shard_size_mismatch(zc):
    a = _stream(zc, n=4096 * 2, seed=5)
    b = _stream(zc, n=4096 * 2 + 3, seed=6)
    st = zc.new_status()
    zc.decompress_reduce([a[2], b[2]], [a[3], b[3]], 4096 * 2, st)
    torch.cuda.synchronize()
    assert zc.status_value(st) in (zc.ERR_SIZE_MISMATCH, zc.ERR_BAD_HEADER)


def test_escape_scan_wait_is_bounded(zc):
    """The workspace's hold hook keeps the first scan unit (a group of 10 tiles) from publishing its escape
    count, so the scans that need it wait on a count nobody publishes: the wait gives up after about a second
    with ZC_ERR_TIMEOUT and the kernel returns.  The context stays usable and the counters are reset."""
    import time
    n = 40 * 4096
    x = workloads.gradient(n=n, seed=7)
    cb = oracle.codebook_from_sigma(1e-3)
    ws = zc.workspace(n)
    ws[0:4] = torch.tensor([1, 0, 0, 0], dtype=torch.uint8, device="cuda")   # hold unit 0
    st = zc.new_status()
    t0 = time.time()
    zc.compress(dev(x), zc.codebook_to_device(cb), ws, st)
    torch.cuda.synchronize()
    dt = time.time() - t0
    assert zc.status_value(st) == zc.ERR_TIMEOUT
    assert 0.5 < dt < 30
    hdr = ws[:8].cpu().numpy().view(np.uint32)
    assert hdr[0] == 0 and hdr[1] == 0          # hook and exit counter reset by the last CTA
    # the same workspace works again
    st2 = zc.new_status()
    main, esc = zc.compress(dev(x), zc.codebook_to_device(cb), ws, st2)
    torch.cuda.synchronize()
    assert zc.status_value(st2) == 0
    om, oe = oracle.compress(x, cb)
    assert np.array_equal(main.cpu().numpy(), om)


@pytest.mark.parametrize("m", [12 * 4096 + 5, 700 * 4096])
def test_reduce_escape_scan_wait_is_bounded(zc, m):
    """The hold hook on a re-encoding decode-reduce: group 0 publishes no output escape count, so the scans of
    the later groups give up after about a second with ZC_ERR_TIMEOUT and the launch returns; the hook and the
    exit counter are reset, and the same workspace then reduces again byte for byte as the oracle.  One size
    per launch shape: one tile per CTA (the teams share the copies), and four tiles per CTA in the all-coded
    launch."""
    import math
    import time
    P = 3
    shards = workloads.rs_shards(P=P, m=m, sigma=1e-3, seed=17)
    cb_in = oracle.codebook_from_sigma(1e-3)
    cb_out = oracle.codebook_from_sigma(1e-3 * math.sqrt(P))
    ws = zc.workspace(m)
    st = zc.new_status()
    streams = [zc.compress(dev(s), zc.codebook_to_device(cb_in), ws, st) for s in shards]
    torch.cuda.synchronize()
    assert zc.status_value(st) == 0
    mains, escs = [a for a, _ in streams], [b for _, b in streams]
    ws[0:4] = torch.tensor([1, 0, 0, 0], dtype=torch.uint8, device="cuda")   # hold group 0
    st = zc.new_status()
    t0 = time.time()
    zc.decompress_reduce(mains, escs, m, st, out_cb=zc.codebook_to_device(cb_out), ws=ws)
    torch.cuda.synchronize()
    dt = time.time() - t0
    assert zc.status_value(st) == zc.ERR_TIMEOUT
    assert 0.5 < dt < 30
    hdr = ws[:8].cpu().numpy().view(np.uint32)
    assert hdr[0] == 0 and hdr[1] == 0          # hook and exit counter reset
    st2 = zc.new_status()
    y, om, oe = zc.decompress_reduce(mains, escs, m, st2, out_cb=zc.codebook_to_device(cb_out), ws=ws)
    torch.cuda.synchronize()
    assert zc.status_value(st2) == 0
    omains, oescs = zip(*(oracle.compress(s, cb_in) for s in shards))
    oy, orm, ore = oracle.decompress_reduce(list(omains), list(oescs), m, cb_out)
    assert np.array_equal(y.cpu().numpy().view(np.uint16), oy)
    assert np.array_equal(om.cpu().numpy(), orm)
    assert np.array_equal(oe[:ore.size].cpu().numpy(), ore)


def test_adaptive_launch_after_a_bounded_wait(zc):
    """An adaptive launch ends at a grid barrier of its CTAs before the raw bypass.  With the hold hook its
    escape scan times out (ZC_ERR_TIMEOUT) yet every CTA still reaches the barrier, so the launch returns, the
    barrier's arrival count is back to 0, and the same workspace then compresses adaptively again, coded and
    RAW, byte for byte as the oracle."""
    n = 40 * 4096
    x = workloads.gradient(n=n, seed=8)
    cb = oracle.codebook_from_sigma(1e-3)
    ws = zc.workspace(n)
    ws[0:4] = torch.tensor([1, 0, 0, 0], dtype=torch.uint8, device="cuda")   # hold unit 0
    st = zc.new_status()
    zc.compress_adaptive(dev(x), zc.codebook_to_device(cb), ws, st)
    torch.cuda.synchronize()
    assert zc.status_value(st) == zc.ERR_TIMEOUT
    hdr = ws[:32].cpu().numpy().view(np.uint32)
    assert hdr[0] == 0 and hdr[1] == 0           # hook and exit counter reset
    assert hdr[5] == 0 and hdr[6] == 0           # RAW rewrite counter and barrier arrivals back to 0
    gen = int(hdr[7])
    for data, book in ((x, cb), (workloads.random_bits(n, seed=9), np.array([1, 2, 3, 4, 5, 6, 7], np.uint8))):
        st2 = zc.new_status()
        main, esc = zc.compress_adaptive(dev(data), zc.codebook_to_device(book), ws, st2)
        torch.cuda.synchronize()
        assert zc.status_value(st2) == 0
        om, oe, _ = oracle.compress_adaptive(data, book)
        assert np.array_equal(main.cpu().numpy(), om)
        assert np.array_equal(esc[:oe.size].cpu().numpy(), oe)
    hdr = ws[:32].cpu().numpy().view(np.uint32)
    assert hdr[6] == 0 and int(hdr[7]) == gen + 2  # one barrier per launch
