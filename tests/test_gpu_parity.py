"""GPU parity: libzc's CUDA kernels against the CPU oracle, byte for byte.

Every case runs the product path through the C ABI (the ctypes binding) and the
oracle on the same seeded inputs; compressed main and escape streams, decoded
tensors, histogram codebooks and reduced / re-encoded outputs must be
bit-identical (integer work: no tolerance).  Sizes span several tiles with
ragged tails; the five workload configurations run at full size.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu


def dev(x: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).cuda()


def host_u16(t: torch.Tensor) -> np.ndarray:
    return t.cpu().numpy().view(np.uint16)


def host_u8(t: torch.Tensor) -> np.ndarray:
    return t.cpu().numpy().view(np.uint8)


def gpu_compress(zc, x: np.ndarray, cb, ws=None):
    st = zc.new_status()
    ws = zc.workspace(x.size) if ws is None else ws
    main, esc = zc.compress(dev(x), zc.codebook_to_device(cb), ws, st)
    torch.cuda.synchronize()
    assert zc.status_value(st) == 0, zc.status_string(zc.status_value(st))
    n_esc = zc.header_n_esc(main)
    return host_u8(main), host_u8(esc)[:n_esc], main, esc


def assert_stream_equal(got_main, got_esc, want_main, want_esc):
    assert got_main.size == want_main.size
    d = np.nonzero(got_main != want_main)[0]
    assert d.size == 0, f"{d.size} main bytes differ, first at {d[:8]}: {got_main[d[:8]]} vs {want_main[d[:8]]}"
    assert got_esc.size == want_esc.size, (got_esc.size, want_esc.size)
    assert np.array_equal(got_esc, want_esc)


def roundtrip_check(zc, x, cb):
    gm, ge, main_t, esc_t = gpu_compress(zc, x, cb)
    om, oe = oracle.compress(x, cb)
    assert_stream_equal(gm, ge, om, oe)
    st = zc.new_status()
    out = zc.decompress(main_t, esc_t, x.size, st)
    torch.cuda.synchronize()
    assert zc.status_value(st) == 0, zc.status_string(zc.status_value(st))
    assert np.array_equal(host_u16(out), x)
    return gm, ge


# ------------------------------------------------------------------ small and ragged cases
def test_gaussian_2pow20_roundtrip(zc):
    """The 2^20-element N(0, 0.02) case with the sigma codebook."""
    x = workloads.gaussian()
    cb = oracle.codebook_from_sigma(0.02)
    assert np.array_equal(zc.codebook_from_sigma(0.02), cb)
    roundtrip_check(zc, x, cb)


@pytest.mark.parametrize("n", [1, 7, 31, 32, 255, 256, 257, 1023, 1024, 1025, 2047, 4095, 4096, 4097,
                               3 * 4096 + 5, 100_003, 1 << 18])
def test_ragged_sizes(zc, n):
    x = workloads.gradient(n=n, sigma=1e-3, seed=n % 1000 + 7)
    roundtrip_check(zc, x, oracle.codebook_from_sigma(1e-3))


def test_empty_tensor(zc):
    x = np.zeros(0, np.uint16)
    st = zc.new_status()
    ws = zc.workspace(0)
    cb = oracle.codebook_from_sigma(0.02)
    main, esc = zc.compress(torch.empty(0, dtype=torch.int16, device="cuda"), zc.codebook_to_device(cb), ws, st)
    torch.cuda.synchronize()
    om, oe = oracle.compress(x, cb)
    assert zc.status_value(st) == 0
    assert_stream_equal(host_u8(main), host_u8(esc)[:0], om, oe)


@pytest.mark.parametrize("cb", [
    [121, 120, 119, 122, 118, 117, 116],
    [255, 0, 127, 1, 254, 128, 126],
    [140, 141, 142, 143, 144, 145, 146],
])
def test_all_65536_patterns(zc, cb):
    x = workloads.all_bf16_patterns()
    roundtrip_check(zc, x, np.array(cb, np.uint8))
    # shuffled, so that every tile mixes NaN payloads, infinities, zeros and subnormals
    rng = np.random.default_rng(3)
    roundtrip_check(zc, rng.permutation(np.tile(x, 3)), np.array(cb, np.uint8))


def test_all_escape_and_no_escape(zc):
    cb = np.array([120, 121, 122, 123, 124, 125, 126], np.uint8)
    x = workloads.all_bf16_patterns()
    all_esc = x[~np.isin((x >> 7) & 0xFF, cb)]
    gm, ge = roundtrip_check(zc, all_esc, cb)
    assert ge.size == all_esc.size
    rng = np.random.default_rng(4)
    n = 5 * 4096 + 17
    e = cb[rng.integers(0, 7, n)].astype(np.uint16)
    none = (rng.integers(0, 2, n).astype(np.uint16) << 15) | (e << 7) | rng.integers(0, 128, n).astype(np.uint16)
    gm, ge = roundtrip_check(zc, none, cb)
    assert ge.size == 0


def test_worked_example_fixture(zc):
    import json, os
    with open(os.path.join(os.path.dirname(__file__), "golden", "worked_example_n1030.json")) as f:
        fx = json.load(f)
    x = np.full(fx["n"], int(fx["default_bits"], 16), np.uint16)
    for k, v in fx["elements"].items():
        x[int(k)] = int(v["bits"], 16)
    gm, ge = roundtrip_check(zc, x, np.array(fx["codebook"], np.uint8))
    assert ge.tolist() == fx["escapes"]


# ------------------------------------------------------------------ histogram
# sizes around the kernel's pieces: the tail of fewer than 8 values counted with plain loads, 32 KB chunks of
# 16384 values (one partial), one chunk per CTA of a full grid and one more; random bits fill all 256 bins
@pytest.mark.parametrize("n,kind", [(0, "g"), (1, "g"), (7, "g"), (8, "g"), (9, "g"), (4096 * 3 + 3, "g"),
                                    (16383, "g"), (16384, "g"), (16385, "g"), (16384 * 152 + 29, "g"),
                                    (16384 * 153, "g"), (1 << 20, "g"), (16384 * 5 + 13, "r")])
def test_histogram_small(zc, n, kind):
    if not n:
        x = np.zeros(0, np.uint16)
    else:
        x = workloads.gradient(n=n, seed=21) if kind == "g" else workloads.random_bits(n, seed=22)
    st = zc.new_status()
    ws = zc.workspace(n)
    hist = torch.zeros(256, dtype=torch.int32, device="cuda")
    xt = dev(x) if n else torch.empty(0, dtype=torch.int16, device="cuda")
    cb, _ = zc.histogram_topk(xt, ws, st, hist_out=hist)
    torch.cuda.synchronize()
    ocb, oh = oracle.histogram_topk(x)
    assert np.array_equal(host_u8(cb), ocb)
    assert np.array_equal(hist.cpu().numpy().astype(np.uint64), oh)
    # the workspace is left clean: a second call gives the same answer
    cb2, _ = zc.histogram_topk(xt, ws, st, hist_out=hist)
    torch.cuda.synchronize()
    assert np.array_equal(host_u8(cb2), ocb)
    assert np.array_equal(hist.cpu().numpy().astype(np.uint64), oh)


def test_histogram_ties(zc):
    """Equal counts: the smaller exponent ranks first."""
    e = np.repeat(np.array([200, 7, 90, 50, 51, 52, 53, 54], np.uint16), [5, 5, 1, 3, 3, 3, 3, 3])
    x = (e << 7).astype(np.uint16)
    st = zc.new_status()
    cb, _ = zc.histogram_topk(dev(x), zc.workspace(x.size), st)
    torch.cuda.synchronize()
    assert host_u8(cb).tolist() == oracle.histogram_topk(x)[0].tolist() == [7, 200, 50, 51, 52, 53, 54]


# ------------------------------------------------------------------ workload configurations at full size
@pytest.mark.slow
def test_config_gradient_64M_histogram_and_sigma(zc):
    """64M gradient tensor with outliers and special values; histogram vs sigma codebooks, both round-tripped."""
    x = workloads.gradient()
    st = zc.new_status()
    ws = zc.workspace(x.size)
    xt = dev(x)
    cb_dev, _ = zc.histogram_topk(xt, ws, st)
    torch.cuda.synchronize()
    ocb, _ = oracle.histogram_topk(x)
    assert np.array_equal(host_u8(cb_dev), ocb)
    for cb in (ocb, oracle.codebook_from_sigma(1e-3)):
        main, esc = zc.compress(xt, zc.codebook_to_device(cb), ws, st)
        out = zc.decompress(main, esc, x.size, st)
        torch.cuda.synchronize()
        assert zc.status_value(st) == 0
        om, oe = oracle.compress(x, cb)
        n_esc = zc.header_n_esc(main)
        assert_stream_equal(host_u8(main), host_u8(esc)[:n_esc], om, oe)
        assert np.array_equal(host_u16(out), x)


def _llama_items(zc, bucket):
    items = []
    for name, x, sigma in bucket:
        mb, eb = zc.compressed_size(x.size)
        items.append(zc.BatchItem(bf16=dev(x), main=torch.empty(mb, dtype=torch.uint8, device="cuda"),
                                  esc=torch.empty(max(eb, 16), dtype=torch.uint8, device="cuda"),
                                  cb=zc.codebook_to_device(oracle.codebook_from_sigma(sigma))))
    return items


@pytest.mark.parametrize("scale", [pytest.param(1.0, marks=pytest.mark.slow), 1 / 512])
def test_config_llama_bucket_batched(zc, scale):
    """Nine Llama-3-8B layer tensors, per-tensor sigma codebooks, one batched launch each way."""
    bucket = workloads.llama_bucket(scale=scale)
    items = _llama_items(zc, bucket)
    st = zc.new_status()
    ws = zc.workspace([x.size for _, x, _ in bucket])
    zc.compress_batched(items, ws, st)
    torch.cuda.synchronize()
    assert zc.status_value(st) == 0
    outs = []
    for it, (name, x, sigma) in zip(items, bucket):
        om, oe = oracle.compress(x, oracle.codebook_from_sigma(sigma))
        n_esc = zc.header_n_esc(it.main)
        assert_stream_equal(host_u8(it.main), host_u8(it.esc)[:n_esc], om, oe)
        outs.append(zc.BatchItem(bf16=torch.empty(x.size, dtype=torch.int16, device="cuda"), main=it.main,
                                 esc=it.esc))
    zc.decompress_batched(outs, st)
    torch.cuda.synchronize()
    assert zc.status_value(st) == 0
    for o, (name, x, sigma) in zip(outs, bucket):
        assert np.array_equal(host_u16(o.bf16), x), name


@pytest.mark.parametrize("adaptive", [False, True])
def test_batch_beyond_one_launch(zc, adaptive):
    """70 tensors in one call (three launches of at most 32 tensors on the stream): empty, one value, ragged,
    exactly one tile, several scan groups; a codebook per tensor (sigma from 1e-4 to 3e-2), every fifth tensor
    uniformly random bit patterns (RAW when adaptive).  Every stream against the oracle, byte for byte."""
    rng = np.random.default_rng(70)
    sizes = [0, 1, 4096, 4097, 8 * 4096 + 3, 10 * 4096, 21 * 4096 + 1] * 10
    xs, cbs = [], []
    for i, n in enumerate(sizes):
        sigma = float(10 ** rng.uniform(-4, math.log10(3e-2)))
        x = (rng.integers(0, 65536, n, dtype=np.uint16) if i % 5 == 4
             else workloads.gaussian(n=n, sigma=sigma, seed=700 + i) if n else np.zeros(0, np.uint16))
        xs.append(x)
        cbs.append(oracle.codebook_from_sigma(sigma))
    items = []
    for x, cb in zip(xs, cbs):
        mb, eb = zc.compressed_size(x.size)
        cap = max(zc.raw_spill(x.size), 16) if adaptive else max(eb, 16)
        items.append(zc.BatchItem(bf16=dev(x) if x.size else torch.empty(0, dtype=torch.int16, device="cuda"),
                                  main=torch.empty(mb, dtype=torch.uint8, device="cuda"),
                                  esc=torch.empty(cap, dtype=torch.uint8, device="cuda"),
                                  cb=zc.codebook_to_device(cb)))
    st = zc.new_status()
    ws = zc.workspace([x.size for x in xs])
    (zc.compress_batched_adaptive if adaptive else zc.compress_batched)(items, ws, st)
    torch.cuda.synchronize()
    assert zc.status_value(st) == 0, zc.status_string(zc.status_value(st))
    outs = []
    for i, (it, x, cb) in enumerate(zip(items, xs, cbs)):
        om, oe = oracle.compress_adaptive(x, cb)[:2] if adaptive else oracle.compress(x, cb)
        n_esc = zc.header_n_esc(it.main)
        assert_stream_equal(host_u8(it.main), host_u8(it.esc)[:n_esc], om, oe)
        outs.append(zc.BatchItem(bf16=torch.empty(x.size, dtype=torch.int16, device="cuda"), main=it.main,
                                 esc=it.esc))
    zc.decompress_batched(outs, st)
    torch.cuda.synchronize()
    assert zc.status_value(st) == 0, zc.status_string(zc.status_value(st))
    for o, x in zip(outs, xs):
        assert np.array_equal(host_u16(o.bf16), x)


@pytest.mark.slow
def test_config_moe_payload_chunks(zc):
    """16384 x 4096 Student-t payload: one histogram codebook, 8 Zipf-sized destination chunks batched."""
    x, counts = workloads.moe_payload()
    st = zc.new_status()
    xt = dev(x)
    ws = zc.workspace([c * 4096 for c in counts])
    cb_dev, _ = zc.histogram_topk(xt, ws, st)
    torch.cuda.synchronize()
    ocb, _ = oracle.histogram_topk(x)
    assert np.array_equal(host_u8(cb_dev), ocb)
    items, start = [], 0
    for c in counts:
        n = c * 4096
        mb, eb = zc.compressed_size(n)
        items.append(zc.BatchItem(bf16=xt[start:start + n], main=torch.empty(mb, dtype=torch.uint8, device="cuda"),
                                  esc=torch.empty(eb, dtype=torch.uint8, device="cuda"), cb=cb_dev))
        start += n
    zc.compress_batched(items, ws, st)
    torch.cuda.synchronize()
    assert zc.status_value(st) == 0
    start = 0
    outs = []
    for it, c in zip(items, counts):
        n = c * 4096
        om, oe = oracle.compress(x[start:start + n], ocb)
        mb = zc.compressed_size(n)[0]
        assert mb == om.size            # the fixed-size part is known before encoding
        n_esc = zc.header_n_esc(it.main)
        assert_stream_equal(host_u8(it.main), host_u8(it.esc)[:n_esc], om, oe)
        outs.append(zc.BatchItem(bf16=torch.empty(n, dtype=torch.int16, device="cuda"), main=it.main, esc=it.esc,
                                 esc_bytes=n_esc))
        start += n
    zc.decompress_batched(outs, st)
    torch.cuda.synchronize()
    assert zc.status_value(st) == 0
    assert np.array_equal(np.concatenate([host_u16(o.bf16) for o in outs]), x)


def _reduce_case(zc, P, m, sigma=1e-3, reencode=True, seed=5, cb_in=None, cb_out=None):
    shards = workloads.rs_shards(P=P, m=m, sigma=sigma, seed=seed)
    cb_in = oracle.codebook_from_sigma(sigma) if cb_in is None else cb_in
    cb_out = oracle.codebook_from_sigma(sigma * math.sqrt(P)) if cb_out is None else cb_out
    st = zc.new_status()
    ws = zc.workspace(m)
    mains, escs, omains, oescs = [], [], [], []
    for s in shards:
        main, esc = zc.compress(dev(s), zc.codebook_to_device(cb_in), ws, st)
        mains.append(main)
        escs.append(esc)
        om, oe = oracle.compress(s, cb_in)
        omains.append(om)
        oescs.append(oe)
    y, om_t, oe_t = zc.decompress_reduce(mains, escs, m, st, out_cb=zc.codebook_to_device(cb_out) if reencode else None,
                                         ws=ws if reencode else None)
    torch.cuda.synchronize()
    assert zc.status_value(st) == 0, zc.status_string(zc.status_value(st))
    if reencode:
        oy, orm, ore = oracle.decompress_reduce(omains, oescs, m, cb_out)
        n_esc = zc.header_n_esc(om_t)
        assert_stream_equal(host_u8(om_t), host_u8(oe_t)[:n_esc], orm, ore)
    else:
        oy = oracle.decompress_reduce(omains, oescs, m)
    assert np.array_equal(host_u16(y), oy)


@pytest.mark.parametrize("P,m", [(1, 5000), (2, 4096), (3, 3 * 4096 + 77), (5, 2 * 4096 + 1000), (8, 1 << 16),
                                 (16, 3 * 4096), (64, 9000), (33, 4097)])
@pytest.mark.parametrize("reencode", [True, False])
def test_decompress_reduce_small(zc, P, m, reencode):
    _reduce_case(zc, P, m, reencode=reencode, seed=P * 7 + m % 13)


@pytest.mark.parametrize("reencode", [True, False])
def test_decompress_reduce_launch_modes(zc, reencode):
    """Up to two tiles per SM, each CTA takes one tile per round (its four teams share the tile's copies: team t
    decodes copies t, t + 4, ...) in the RAW-capable kernel alone; above that four (one per team).  A
    grid of at most one CTA per SM runs the RAW-capable kernel alone; beyond it the all-coded kernel runs,
    followed by the RAW-capable one that leaves at once.  Sizes on both sides of both switches, element by
    element against the oracle."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    for m in (4096 * sms, 4096 * sms + 1, 2 * 4096 * sms, 2 * 4096 * sms + 7, 4096 * (4 * (sms - 1) - 1) + 55,
              4 * 4096 * sms + 4096 + 9):
        _reduce_case(zc, 3, m, reencode=reencode, seed=m % 101)


FAR_CODEBOOK = np.array([1, 2, 3, 4, 5, 6, 7], dtype=np.uint8)  # no N(0, 1e-3) value has these exponents


@pytest.mark.parametrize("far_in,far_out", [(True, False), (False, True), (True, True)])
def test_decompress_reduce_all_escape(zc, far_in, far_out):
    """Every input and/or every output value an escape: input tiles carry 4096 escape bytes, more than a
    stage holds (the rest is read from global memory), and every re-encoded block has more escapes than its
    staging buffer (written from the rounded tile instead)."""
    _reduce_case(zc, 3, 5 * 4096 + 123, seed=91, cb_in=FAR_CODEBOOK if far_in else None,
                 cb_out=FAR_CODEBOOK if far_out else None)


def test_decompress_reduce_special_values(zc):
    """Infinities of both signs (NaN sums), overflow to inf, signed zeros and subnormals across shards."""
    P, m = 4, 3 * 4096 + 11
    rng = np.random.default_rng(17)
    shards = []
    for r in range(P):
        x = workloads.gradient(n=m, sigma=1e-3, seed=40 + r)
        x[rng.integers(0, m, 300)] = 0x7F7F
        x[rng.integers(0, m, 50)] = 0xFF80
        x[rng.integers(0, m, 300)] = rng.integers(1, 128, 300).astype(np.uint16)
        x[rng.integers(0, m, 100)] = 0x8000
        shards.append(x)
    # fixed positions: +inf + -inf (NaN), max + max (overflow to inf), all -0, subnormal sums, a NaN payload
    shards[0][0], shards[1][0] = 0x7F80, 0xFF80
    shards[0][1], shards[1][1], shards[2][1], shards[3][1] = 0x7F7F, 0x7F7F, 0x0000, 0x0000
    for r in range(P):
        shards[r][2] = 0x8000
        shards[r][3] = 0x0001 + r
    shards[2][4] = 0xFFC3
    cb = oracle.codebook_from_sigma(1e-3)
    st = zc.new_status()
    ws = zc.workspace(m)
    mains, escs, om, oe = [], [], [], []
    for s in shards:
        a, b = zc.compress(dev(s), zc.codebook_to_device(cb), ws, st)
        mains.append(a); escs.append(b)
        c, d = oracle.compress(s, cb)
        om.append(c); oe.append(d)
    y, m_t, e_t = zc.decompress_reduce(mains, escs, m, st, out_cb=zc.codebook_to_device(cb), ws=ws)
    torch.cuda.synchronize()
    assert zc.status_value(st) == 0
    oy, orm, ore = oracle.decompress_reduce(om, oe, m, cb)
    assert np.array_equal(host_u16(y), oy)
    assert_stream_equal(host_u8(m_t), host_u8(e_t)[:zc.header_n_esc(m_t)], orm, ore)
    assert oy[0] == 0x7FC0 and oy[1] == 0x7F80 and oy[2] == 0x8000 and oy[3] == 0x000A and oy[4] == 0x7FC0


@pytest.mark.slow
def test_config_reduce_scatter_8x32M(zc):
    """P = 8 shards of 2^25 elements, shared input codebook, sqrt(8)*sigma output codebook."""
    _reduce_case(zc, 8, 1 << 25)


@pytest.mark.slow
def test_config_reduce_scatter_sweep_largest(zc):
    """The largest point of the shard-size sweep, as the benchmark runs it: P = 8 shards of 2^29 elements
    (1 GiB each), each the 2^25-element base shard repeated 16 times.  Checked on a seeded sample of tiles
    (the format is tile-local given the offset table): the reduced values against the oracle's reduction of
    the same input slices, each re-encoded tile's bytes and escapes against the oracle's encoding of that
    tile alone, and the escape offsets against each other."""
    P, m_base, reps = 8, 1 << 25, 16
    m = m_base * reps
    base = workloads.rs_shards(P=P, m=m_base)
    cb_in = oracle.codebook_from_sigma(workloads.RS_SIGMA)
    cb_out = oracle.codebook_from_sigma(workloads.RS_SIGMA * math.sqrt(P))
    st = zc.new_status()
    ws = zc.workspace(m)
    mains, escs = [], []
    for b in base:
        main, esc = zc.compress(dev(b).repeat(reps), zc.codebook_to_device(cb_in), ws, st)
        mains.append(main)
        escs.append(esc)
    y, om_t, oe_t = zc.decompress_reduce(mains, escs, m, st, out_cb=zc.codebook_to_device(cb_out), ws=ws)
    torch.cuda.synchronize()
    assert zc.status_value(st) == 0, zc.status_string(zc.status_value(st))
    ntiles = m // 4096
    R = -(-4 * ntiles // 128) * 128
    n_esc = zc.header_n_esc(om_t)
    rng = np.random.default_rng(29)
    tiles = sorted({0, 1, 8191, 8192, ntiles - 2, ntiles - 1, *rng.integers(0, ntiles, 58).tolist()})
    table = om_t[128:128 + 4 * ntiles].view(torch.int32)
    for t in tiles:
        tt = t % (m_base // 4096)
        xs = [b[4096 * tt:4096 * (tt + 1)] for b in base]
        want_y = oracle.reduce(xs)
        assert np.array_equal(host_u16(y[4096 * t:4096 * (t + 1)]), want_y), f"tile {t}"
        tm, te = oracle.compress(want_y, cb_out)
        got_tile = host_u8(om_t[128 + R + 5632 * t:128 + R + 5632 * (t + 1)])
        assert np.array_equal(got_tile, tm[256:256 + 5632]), f"re-encoded tile {t}"
        a = int(table[t].item()) & 0xFFFFFFFF
        b = int(table[t + 1].item()) & 0xFFFFFFFF if t + 1 < ntiles else n_esc
        assert b - a == te.size, f"escape count of tile {t}"
        assert np.array_equal(host_u8(oe_t[a:b]), te), f"escapes of tile {t}"


@pytest.mark.slow
def test_largest_tensor(zc):
    """The largest tensor the format allows, n = 2^32 - 1 values (8 GiB of bf16, a 5.6 GiB main stream, a
    ragged last tile): byte offsets far past 2^31 and 2^32 go through 64-bit address arithmetic, tile and
    group counts reach their u32 limits.  The input is drawn on the device (seeded,
    workloads.gaussian_on_device); the round trip is compared in full on the device, and 24 seeded tiles of
    the main and escape streams against the oracle's encoding of those tiles alone (the format is
    tile-local given the offset table)."""
    n = (1 << 32) - 1
    xt = workloads.gaussian_on_device(n, 1e-3, seed=31)
    cb = oracle.codebook_from_sigma(1e-3)
    st = zc.new_status()
    ws = zc.workspace(n)
    main, esc = zc.compress(xt, zc.codebook_to_device(cb), ws, st)
    y = zc.decompress(main, esc, n, st)
    torch.cuda.synchronize()
    assert zc.status_value(st) == 0, zc.status_string(zc.status_value(st))
    assert torch.equal(y, xt)
    del y
    ntiles = -(-n // 4096)
    R = -(-4 * ntiles // 128) * 128
    n_esc = zc.header_n_esc(main)
    table = main[128:128 + 4 * ntiles].view(torch.int32)
    rng = np.random.default_rng(31)
    tiles = sorted({0, (1 << 31) // 4096, ntiles - 2, ntiles - 1, *rng.integers(0, ntiles, 20).tolist()})
    for t in tiles:
        x_tile = host_u16(xt[4096 * t:min(n, 4096 * (t + 1))])
        tm, te = oracle.compress(x_tile, cb)
        got = host_u8(main[128 + R + 5632 * t:128 + R + 5632 * (t + 1)])
        assert np.array_equal(got, tm[256:256 + 5632]), f"tile {t}"
        a = int(table[t].item()) & 0xFFFFFFFF
        b = int(table[t + 1].item()) & 0xFFFFFFFF if t + 1 < ntiles else n_esc
        assert b - a == te.size and np.array_equal(host_u8(esc[a:b]), te), f"escapes of tile {t}"


@pytest.mark.slow
def test_largest_all_escape(zc):
    """n = 2^32 - 1 values, none of whose exponents is in the codebook: n_esc = n, the escape offsets run up
    to the u32 limit.  Round trip on the device; 16 seeded tiles of the main and escape streams against the
    oracle; then decode-reduce-re-encode of the stream with itself (P = 2, x + x = 2x exactly, again all
    escapes), its result and re-encoded stream checked on the same tiles."""
    n = (1 << 32) - 1
    xt = workloads.gaussian_on_device(n, 1e-3, seed=33)
    cb = FAR_CODEBOOK
    st = zc.new_status()
    ws = zc.workspace(n)
    main, esc = zc.compress(xt, zc.codebook_to_device(cb), ws, st)
    y = zc.decompress(main, esc, n, st)
    torch.cuda.synchronize()
    assert zc.status_value(st) == 0, zc.status_string(zc.status_value(st))
    assert zc.header_n_esc(main) == n
    assert torch.equal(y, xt)
    del y
    ntiles = -(-n // 4096)
    R = -(-4 * ntiles // 128) * 128
    rng = np.random.default_rng(33)
    tiles = sorted({0, ntiles // 2, ntiles - 2, ntiles - 1, *rng.integers(0, ntiles, 12).tolist()})

    def check_stream(m_t, e_t, x_of_tile, cbook):
        table = m_t[128:128 + 4 * ntiles].view(torch.int32)
        n_esc = zc.header_n_esc(m_t)
        for t in tiles:
            tm, te = oracle.compress(x_of_tile(t), cbook)
            assert np.array_equal(host_u8(m_t[128 + R + 5632 * t:128 + R + 5632 * (t + 1)]), tm[256:256 + 5632]), t
            a = int(table[t].item()) & 0xFFFFFFFF
            b = int(table[t + 1].item()) & 0xFFFFFFFF if t + 1 < ntiles else n_esc
            assert b - a == te.size and np.array_equal(host_u8(e_t[a:b]), te), f"escapes of tile {t}"

    def x_tile(t):
        return host_u16(xt[4096 * t:min(n, 4096 * (t + 1))])

    check_stream(main, esc, x_tile, cb)
    out, om, oe = zc.decompress_reduce([main, main], [esc, esc], n, st, out_cb=zc.codebook_to_device(cb), ws=ws)
    torch.cuda.synchronize()
    assert zc.status_value(st) == 0, zc.status_string(zc.status_value(st))
    assert zc.header_n_esc(om) == n
    for t in tiles:
        want = oracle.reduce([x_tile(t), x_tile(t)])
        assert np.array_equal(host_u16(out[4096 * t:min(n, 4096 * (t + 1))]), want), f"reduced tile {t}"
    check_stream(om, oe, lambda t: oracle.reduce([x_tile(t), x_tile(t)]), cb)


@pytest.mark.slow
def test_huge_reduce_byte_offsets_beyond_2pow31(zc):
    """Decode-reduce-re-encode of P = 2 shards of 2^31 + 777 values (2.8 GiB main streams, a 4 GiB result):
    24 seeded tiles of the result and of the re-encoded stream against the oracle's reduction of the same
    input slices and its encoding of each tile alone."""
    n = (1 << 31) + 777
    xs = [workloads.gaussian_on_device(n, 1e-3, seed=40 + r) for r in range(2)]
    cb_in = oracle.codebook_from_sigma(1e-3)
    cb_out = oracle.codebook_from_sigma(1e-3 * math.sqrt(2))
    st = zc.new_status()
    ws = zc.workspace(n)
    streams = [zc.compress(x, zc.codebook_to_device(cb_in), ws, st) for x in xs]
    y, om_t, oe_t = zc.decompress_reduce([m for m, _ in streams], [e for _, e in streams], n, st,
                                         out_cb=zc.codebook_to_device(cb_out), ws=ws)
    torch.cuda.synchronize()
    assert zc.status_value(st) == 0, zc.status_string(zc.status_value(st))
    del streams
    ntiles = -(-n // 4096)
    R = -(-4 * ntiles // 128) * 128
    n_esc = zc.header_n_esc(om_t)
    table = om_t[128:128 + 4 * ntiles].view(torch.int32)
    rng = np.random.default_rng(41)
    tiles = sorted({0, (1 << 31) // 4096 // 2, ntiles - 2, ntiles - 1, *rng.integers(0, ntiles, 20).tolist()})
    for t in tiles:
        lo, hi = 4096 * t, min(n, 4096 * (t + 1))
        want_y = oracle.reduce([host_u16(x[lo:hi]) for x in xs])
        assert np.array_equal(host_u16(y[lo:hi]), want_y), f"tile {t}"
        tm, te = oracle.compress(want_y, cb_out)
        got = host_u8(om_t[128 + R + 5632 * t:128 + R + 5632 * (t + 1)])
        assert np.array_equal(got, tm[256:256 + 5632]), f"re-encoded tile {t}"
        a = int(table[t].item()) & 0xFFFFFFFF
        b = int(table[t + 1].item()) & 0xFFFFFFFF if t + 1 < ntiles else n_esc
        assert b - a == te.size and np.array_equal(host_u8(oe_t[a:b]), te), f"escapes of tile {t}"


# ------------------------------------------------------------------ workspace reuse
def test_workspace_reused_without_rezeroing(zc):
    ws = zc.workspace(1 << 18)
    cb = oracle.codebook_from_sigma(1e-3)
    for i, n in enumerate([1 << 18, 4096 * 5 + 1, 100, 1 << 17, 1 << 18]):
        x = workloads.gradient(n=n, seed=200 + i)
        gm, ge, _, _ = gpu_compress(zc, x, cb, ws=ws)
        om, oe = oracle.compress(x, cb)
        assert_stream_equal(gm, ge, om, oe)
    hdr = host_u8(ws[:16]).view(np.uint32)
    assert hdr[0] == 0 and hdr[1] == 0 and hdr[2] == 5   # test hook, exit count reset; epoch = launches


def test_epoch_wraparound(zc):
    """The escape-scan epoch tag wraps after 2^32 - 1 launches; the wrap clears every flag first.

    The first launch leaves flags tagged with epoch 1 holding other escape
    counts; if the wrap did not clear them, the launch tagged 1 after the wrap
    would pick them up and write wrong escape offsets."""
    ws = zc.workspace(1 << 16)
    cb = oracle.codebook_from_sigma(1e-3)
    other = workloads.gradient(n=1 << 16, seed=301, outlier_frac=0.2)
    gpu_compress(zc, other, cb, ws=ws)         # flags tagged with epoch 1
    ws[8:12] = torch.tensor([0xFE, 0xFF, 0xFF, 0xFF], dtype=torch.uint8, device="cuda")  # epoch = 2^32 - 2
    x = workloads.gradient(n=1 << 16, seed=300)
    om, oe = oracle.compress(x, cb)
    for epoch_after in (0, 1, 2):              # launches tagged 2^32 - 1 (wrap), 1, 2
        gm, ge, _, _ = gpu_compress(zc, x, cb, ws=ws)
        assert_stream_equal(gm, ge, om, oe)
        assert int(host_u8(ws[8:12]).view(np.uint32)[0]) == epoch_after
