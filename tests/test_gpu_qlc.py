"""GPU parity of Quad Length Codes for FP8 e4m3 bytes ([QLC §3-§4]) against the oracle, byte for byte.

zq_compress's ZQ1 stream must equal the oracle's for the same bytes and table
(header, block offsets, lane counts, code words, padding), and zq_decompress
must return the input from streams written by either side.  Sizes span one
symbol to several scan groups with ragged runs; tables: the static widths, a
dynamic table with a 2-symbol region of 4-bit codes, and a degenerate
8-bit-only table; data: e4m3 FFN1 / gradient stand-ins, uniform bytes and
all 256 byte values.  The full-size case is 2^26 bytes.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu

DEFAULT = tuple(oracle.QLC_DEFAULT_WIDTHS)
DYNAMIC = (1, 3, 4, 5, 5, 5, 5, 8)
EIGHT = (8, 0, 0, 0, 0, 0, 0, 0)


def gpu_encode(zc, x, widths, sym, ws=None, cap=None, expect=0):
    xt = torch.from_numpy(np.ascontiguousarray(x)).cuda() if x.size else torch.empty(0, dtype=torch.uint8,
                                                                                     device="cuda")
    ws = zc.workspace(max(x.size, 1)) if ws is None else ws
    st = zc.new_status()
    out = torch.zeros(cap if cap is not None else zc.zq_max_bytes(x.size), dtype=torch.uint8, device="cuda")
    zc.zq_compress(xt, zc.zq_table(widths, sym), ws, st, out=out)
    torch.cuda.synchronize()
    assert zc.status_value(st) == expect, zc.status_string(zc.status_value(st))
    return out


def check(zc, x, widths, sym, ws=None):
    out = gpu_encode(zc, x, widths, sym, ws)
    want = oracle.qlc_compress(x, widths, sym)
    nbytes = zc.zq_stream_bytes(out)
    assert nbytes == want.size
    got = out[:nbytes].cpu().numpy()
    d = np.nonzero(got != want)[0]
    assert d.size == 0, f"{d.size} stream bytes differ, first at {d[:8]}"
    st = zc.new_status()
    y = zc.zq_decompress(out, x.size, st, in_bytes=nbytes)
    torch.cuda.synchronize()
    assert zc.status_value(st) == 0, zc.status_string(zc.status_value(st))
    assert np.array_equal(y.cpu().numpy(), x)


@pytest.mark.parametrize("n", [1, 15, 16, 17, 511, 4095, 4096, 4097, 8 * 4096 + 3, 100_003, (1 << 20) + 7])
@pytest.mark.parametrize("widths", [DEFAULT, DYNAMIC])
def test_ffn1_parity(zc, n, widths):
    x = workloads.fp8_ffn1(n, seed=n % 101 + 1)
    check(zc, x, widths, oracle.qlc_table_for(x))


@pytest.mark.parametrize("gen", ["gradient", "uniform", "all_bytes"])
@pytest.mark.parametrize("widths", [DEFAULT, DYNAMIC, EIGHT])
def test_other_data_parity(zc, gen, widths):
    n = 300_001
    if gen == "gradient":
        x = workloads.fp8_gradient(n, seed=11)
    elif gen == "uniform":
        x = np.random.default_rng(12).integers(0, 256, n).astype(np.uint8)
    else:
        x = np.random.default_rng(13).permutation(np.tile(np.arange(256, dtype=np.uint8), n // 256))
    sym = np.random.default_rng(14).permutation(256).astype(np.uint8) if gen == "all_bytes" else oracle.qlc_table_for(x)
    check(zc, x, widths, sym)


def test_empty(zc):
    x = np.zeros(0, np.uint8)
    sym = np.arange(256, dtype=np.uint8)
    out = gpu_encode(zc, x, DEFAULT, sym)
    want = oracle.qlc_compress(x, DEFAULT, sym)
    assert np.array_equal(out[:want.size].cpu().numpy(), want)


@pytest.mark.parametrize("n", [1, 4097, 250_000])
def test_decode_oracle_streams(zc, n):
    x = workloads.fp8_gradient(n, seed=n)
    s = oracle.qlc_compress(x, DYNAMIC, oracle.qlc_table_for(x))
    buf = torch.from_numpy(np.concatenate([s, np.zeros(16, np.uint8)])).cuda()
    st = zc.new_status()
    y = zc.zq_decompress(buf, n, st, in_bytes=s.size)
    torch.cuda.synchronize()
    assert zc.status_value(st) == 0 and np.array_equal(y.cpu().numpy(), x)


def test_workspace_shared_with_bf16_codec(zc):
    """The QLC encoder and the bf16 encoder share one workspace (same scan protocol, one epoch sequence)."""
    n = 1 << 18
    ws = zc.workspace(n)
    for i in range(3):
        x = workloads.fp8_ffn1(n - 4096 * i, seed=30 + i)
        check(zc, x, DEFAULT, oracle.qlc_table_for(x), ws=ws)
        g = workloads.gaussian(n, seed=40 + i)
        st = zc.new_status()
        main, esc = zc.compress(torch.from_numpy(g.view(np.int16)).cuda(),
                                zc.codebook_to_device(oracle.codebook_from_sigma(0.02)), ws, st)
        om, oe = oracle.compress(g, oracle.codebook_from_sigma(0.02))
        torch.cuda.synchronize()
        assert zc.status_value(st) == 0 and np.array_equal(main.cpu().numpy(), om)


def test_out_of_room(zc):
    n = 100_000
    x = np.random.default_rng(5).integers(0, 256, n).astype(np.uint8)
    sym = oracle.qlc_table_for(x)
    want = oracle.qlc_compress(x, DEFAULT, sym)
    out = gpu_encode(zc, x, DEFAULT, sym, cap=want.size - 64, expect=zc.ERR_OUT_OF_ROOM)
    assert zc.zq_stream_bytes(out) == want.size  # the header still counts the whole stream


def test_stream_errors(zc):
    n = 50_000
    x = workloads.fp8_ffn1(n, seed=9)
    s = oracle.qlc_compress(x, DEFAULT, oracle.qlc_table_for(x))
    cases = []
    bad = s.copy()
    bad[0] ^= 1
    cases.append((bad, n, zc.ERR_BAD_HEADER))
    bad = s.copy()
    bad[128 + 3] = bad[128 + 4]  # the rank table is no longer a permutation
    cases.append((bad, n, zc.ERR_BAD_HEADER))
    cases.append((s, n + 1, zc.ERR_SIZE_MISMATCH))
    bad = s.copy()
    bad[512] = 200  # lane 0's word count of block 0 no longer adds up
    cases.append((bad, n, zc.ERR_CORRUPT_STREAM))
    for stream, nn, code in cases:
        st = zc.new_status()
        zc.zq_decompress(torch.from_numpy(stream.copy()).cuda(), nn, st, in_bytes=stream.size)
        torch.cuda.synchronize()
        assert zc.status_value(st) == code, (code, zc.status_string(zc.status_value(st)))


def test_decode_stream_tail(zc):
    """The decoder stages a block with one bulk copy of whole 16-byte units; where the last block's copy would
    reach past in_bytes it takes plain loads instead.  Streams whose sizes cover every residue mod 16 decode from
    buffers that end exactly at the stream; a stream that does not start on 16 bytes is refused."""
    residues = set()
    for k in range(12):
        n = 3 * 4096 + 517 * k + 1
        x = workloads.fp8_ffn1(n, seed=60 + k)
        s = oracle.qlc_compress(x, DYNAMIC, oracle.qlc_table_for(x))
        residues.add(s.size % 16)
        st = zc.new_status()
        y = zc.zq_decompress(torch.from_numpy(s).cuda(), n, st, in_bytes=s.size)
        torch.cuda.synchronize()
        assert zc.status_value(st) == 0 and np.array_equal(y.cpu().numpy(), x)
    assert residues == {0, 4, 8, 12}
    buf = torch.zeros(s.size + 16, dtype=torch.uint8, device="cuda")
    with pytest.raises(zc.ZcError):
        zc.zq_decompress(buf[4:], n, zc.new_status(), in_bytes=s.size)


def test_corrupt_block_offset(zc):
    """A block offset past the payload is a corrupt stream; the blocks around it still decode."""
    n = 20 * 4096
    x = workloads.fp8_ffn1(n, seed=78)
    s = oracle.qlc_compress(x, DEFAULT, oracle.qlc_table_for(x))
    bad = s.copy()
    bad[384 + 4 * 7:384 + 4 * 8] = np.frombuffer(np.uint32(0x7FFFFFF0).tobytes(), np.uint8)
    st = zc.new_status()
    y = zc.zq_decompress(torch.from_numpy(bad).cuda(), n, st, in_bytes=bad.size)
    torch.cuda.synchronize()
    assert zc.status_value(st) == zc.ERR_CORRUPT_STREAM
    got = y.cpu().numpy()
    assert np.array_equal(got[:6 * 4096], x[:6 * 4096]) and np.array_equal(got[8 * 4096:], x[8 * 4096:])


@pytest.mark.parametrize("widths", [DEFAULT, DYNAMIC])
def test_several_rounds_and_a_partial_last_group(zc, widths):
    """4917 blocks (a ragged last one): 308 groups of 16 blocks over at most one CTA per SM, so CTAs code two or
    three groups each and the last group holds 5 blocks; the whole stream against the oracle's."""
    n = (16 * 152 * 2 + 16 * 3 + 5) * 4096 - 77
    x = workloads.fp8_gradient(n, seed=4917)
    check(zc, x, widths, oracle.qlc_table_for(x))


@pytest.mark.parametrize("n", [40 * 4096 + 9, (16 * 152 * 2 + 5) * 4096])
def test_escape_scan_wait_is_bounded(zc, n):
    """The workspace's hold hook on the QLC encoder: group 0 publishes no size, so the block-offset scans of the
    later groups give up after about a second with ZC_ERR_TIMEOUT and the launch returns; the hook and the exit
    counter are reset, and the same workspace then compresses again byte for byte as the oracle.  One size
    with one group per CTA, one with several."""
    import time
    x = workloads.fp8_ffn1(n, seed=77)
    sym = oracle.qlc_table_for(x)
    ws = zc.workspace(n)
    ws[0:4] = torch.tensor([1, 0, 0, 0], dtype=torch.uint8, device="cuda")   # hold group 0
    t0 = time.time()
    gpu_encode(zc, x, DEFAULT, sym, ws=ws, expect=zc.ERR_TIMEOUT)
    dt = time.time() - t0
    assert 0.5 < dt < 30
    hdr = ws[:8].cpu().numpy().view(np.uint32)
    assert hdr[0] == 0 and hdr[1] == 0          # hook and exit counter reset
    check(zc, x, DEFAULT, sym, ws=ws)


@pytest.mark.slow
def test_full_size_ffn1(zc):
    n = 1 << 26
    x = workloads.fp8_ffn1(n)
    check(zc, x, DEFAULT, oracle.qlc_table_for(x))


@pytest.mark.slow
def test_largest_stream(zc):
    """The largest QLC input, n = 2^32 - 1 bytes (payload word offsets past 2^30, byte offsets past 2^32):
    full round trip on the device and 16 seeded blocks against the oracle's coding of each block alone."""
    n = (1 << 32) - 1
    g = torch.Generator(device="cuda")
    g.manual_seed(77)
    xt = torch.randint(0, 256, (n,), dtype=torch.uint8, device="cuda", generator=g)
    xt = torch.where(xt < 192, torch.full_like(xt, 56) + (xt & 7), xt)  # a skewed byte distribution
    hist = sum(torch.bincount(xt[i:i + (1 << 28)], minlength=256) for i in range(0, n, 1 << 28)).cpu().numpy()
    sym = oracle.qlc_table_from_histogram(hist)
    st = zc.new_status()
    ws = zc.workspace(n)
    out = zc.zq_compress(xt, zc.zq_table(DEFAULT, sym), ws, st)
    y = zc.zq_decompress(out, n, st, in_bytes=zc.zq_stream_bytes(out))
    torch.cuda.synchronize()
    assert zc.status_value(st) == 0, zc.status_string(zc.status_value(st))
    assert torch.equal(y, xt)
    del y
    nb = -(-n // 4096)
    tbl = -(-4 * nb // 128) * 128
    offs = out[384:384 + 4 * nb].view(torch.int32)
    words = int.from_bytes(out[24:32].cpu().numpy().tobytes(), "little")
    rng = np.random.default_rng(78)
    for b in sorted({0, nb // 2, nb - 1, *rng.integers(0, nb, 13).tolist()}):
        x_blk = xt[4096 * b:min(n, 4096 * (b + 1))].cpu().numpy()
        want = oracle.qlc_compress(x_blk, DEFAULT, sym)  # one block: its words start at byte 512
        a = int(offs[b].item()) & 0xFFFFFFFF
        e = int(offs[b + 1].item()) & 0xFFFFFFFF if b + 1 < nb else words
        got = out[384 + tbl + 4 * a:384 + tbl + 4 * e].cpu().numpy()
        assert np.array_equal(got, want[512:]), f"block {b}"
