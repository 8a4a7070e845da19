"""GPU parity of the raw bypass: adaptive compression, and decoding / reducing RAW streams.

The adaptive encoder stores a tensor RAW (header flags bit 0: its own
little-endian bytes, tile region then escape stream) exactly when that is
strictly smaller than the coded form ([CCCL §3.3], [CCCL §5.2]).  Every case
runs libzc through the C ABI and compares, byte for byte, with the oracle on
the same seeded inputs: the main and escape streams written by
zc_compress_adaptive / zc_compress_batched_adaptive, the values decoded from
RAW streams the oracle wrote, and reductions over mixed RAW / coded shards.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu

DISJOINT = np.array([250, 251, 252, 253, 254, 249, 248], np.uint8)


def dev(x):
    return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).cuda()


def host_u8(t):
    return t.cpu().numpy().view(np.uint8)


def host_u16(t):
    return t.cpu().numpy().view(np.uint16)


def random_bits(n, seed):
    return np.random.default_rng(seed).integers(0, 65536, n, dtype=np.uint16)


def gpu_adaptive(zc, x, cb, cap=None, ws=None, expect_status=0):
    st = zc.new_status()
    ws = zc.workspace(x.size) if ws is None else ws
    esc = None
    if cap is not None:
        esc = torch.zeros(max(cap, 16), dtype=torch.uint8, device="cuda")
    n = x.size
    mb, _ = zc.compressed_size(n)
    main = torch.empty(mb, dtype=torch.uint8, device="cuda")
    if esc is None:
        esc = torch.empty(max(zc.raw_spill(n), 16), dtype=torch.uint8, device="cuda")
    cap_bytes = esc.numel() if cap is None else cap
    xt = dev(x) if n else None  # kept alive until the kernels have run
    cbt = zc.codebook_to_device(cb)
    rc = zc.load().zc_compress_adaptive(xt.data_ptr() if n else None, n, cbt.data_ptr(), main.data_ptr(),
                                        esc.data_ptr(), cap_bytes, ws.data_ptr(), ws.numel(), st.data_ptr(),
                                        torch.cuda.current_stream().cuda_stream)
    assert rc == 0, zc.status_string(rc)
    torch.cuda.synchronize()
    assert zc.status_value(st) == expect_status, zc.status_string(zc.status_value(st))
    n_esc = zc.header_n_esc(main)
    return host_u8(main), host_u8(esc)[:min(n_esc, cap_bytes)], main, esc


def check_against_oracle(zc, x, cb, cap=None, ws=None):
    gm, ge, main_t, esc_t = gpu_adaptive(zc, x, cb, cap, ws)
    om, oe, raw = oracle.compress_adaptive(x, cb, esc_capacity=cap)
    assert np.array_equal(gm, om), f"{np.count_nonzero(gm != om)} main bytes differ (raw={raw})"
    assert np.array_equal(ge, oe)
    st = zc.new_status()
    out = zc.decompress(main_t, esc_t, x.size, st)
    torch.cuda.synchronize()
    assert zc.status_value(st) == 0, zc.status_string(zc.status_value(st))
    assert np.array_equal(host_u16(out), x)
    return raw


@pytest.mark.parametrize("n", [1, 7, 2816, 2817, 4095, 4096, 4097, 3 * 4096 + 5, 100_003, (1 << 20) + 123])
def test_random_bits_go_raw(zc, n):
    x = random_bits(n, seed=n % 977)
    raw = check_against_oracle(zc, x, DISJOINT)
    assert raw == (n > 0)


@pytest.mark.parametrize("n", [4096, 40961])
def test_decision_threshold(zc, n):
    cb = np.array([127, 1, 2, 3, 4, 5, 6], np.uint8)
    s = oracle.raw_spill(n)
    rng = np.random.default_rng(17)
    for k, want_raw in ((s, False), (s + 1, True)):
        x = (127 << 7 | rng.integers(0, 128, n)).astype(np.uint16)
        pos = rng.choice(n, k, replace=False)
        x[pos] = (200 << 7) | (x[pos] & 0x7F)
        assert check_against_oracle(zc, x, cb) == want_raw


def test_gaussian_stays_coded_and_equals_plain(zc):
    x = workloads.gradient(n=(1 << 20) + 77, sigma=1e-3, seed=9)
    cb = oracle.codebook_from_sigma(1e-3)
    assert not check_against_oracle(zc, x, cb, cap=x.size)


def test_workspace_reused_across_adaptive_calls(zc):
    ws = zc.workspace(1 << 18)
    cb = oracle.codebook_from_sigma(0.02)
    for i in range(6):
        n = (1 << 18) - 1000 * i
        x = random_bits(n, seed=i) if i % 2 else workloads.gaussian(n, seed=i + 50)
        assert check_against_oracle(zc, x, DISJOINT if i % 2 else cb, ws=ws) == bool(i % 2)


def test_overflow_rescued_by_raw(zc):
    n = 3 * 4096 + 100
    x = random_bits(n, seed=3)
    s = oracle.raw_spill(n)
    assert check_against_oracle(zc, x, DISJOINT, cap=s)


def test_overflow_when_neither_fits(zc):
    n = 3 * 4096 + 100
    x = random_bits(n, seed=3)
    cap = oracle.raw_spill(n) - 2
    gm, ge, _, _ = gpu_adaptive(zc, x, DISJOINT, cap=cap, expect_status=zc.ERR_ESCAPE_OVERFLOW)
    om, oe, raw, rc = oracle.compress_adaptive(x, DISJOINT, esc_capacity=cap, allow_overflow=True)
    assert not raw and rc == oracle.ERR_ESCAPE_OVERFLOW
    assert np.array_equal(gm, om) and np.array_equal(ge, oe)


def test_empty_tensor(zc):
    x = np.zeros(0, np.uint16)
    cb = oracle.codebook_from_sigma(0.02)
    gm, ge, _, _ = gpu_adaptive(zc, x, cb)
    om, oe, raw = oracle.compress_adaptive(x, cb)
    assert not raw and np.array_equal(gm, om) and ge.size == 0


def test_batched_adaptive_mixed(zc):
    sizes = [4096 * 3 + 11, 1, 0, 65536, 2817, 200_000, 4096]
    xs, cbs = [], []
    for i, n in enumerate(sizes):
        if i % 2:
            xs.append(random_bits(n, seed=100 + i))
            cbs.append(DISJOINT)
        else:
            xs.append(workloads.gaussian(n, sigma=1e-2, seed=200 + i))
            cbs.append(oracle.codebook_from_sigma(1e-2))
    items = []
    for x, cb in zip(xs, cbs):
        n = x.size
        mb, _ = zc.compressed_size(n)
        items.append(zc.BatchItem(bf16=dev(x) if n else torch.empty(0, dtype=torch.int16, device="cuda"),
                                  main=torch.empty(mb, dtype=torch.uint8, device="cuda"),
                                  esc=torch.empty(max(n, 16), dtype=torch.uint8, device="cuda"),
                                  cb=zc.codebook_to_device(cb)))
    ws = zc.workspace(sizes)
    st = zc.new_status()
    zc.compress_batched_adaptive(items, ws, st)
    torch.cuda.synchronize()
    assert zc.status_value(st) == 0
    outs, kinds = [], []
    for it, x, cb in zip(items, xs, cbs):
        om, oe, raw = oracle.compress_adaptive(x, cb)
        kinds.append(raw)
        assert np.array_equal(host_u8(it.main), om)
        assert np.array_equal(host_u8(it.esc)[:oe.size], oe)
        outs.append(torch.empty(max(x.size, 1), dtype=torch.int16, device="cuda")[:x.size])
    # 2817 values (i = 4) spill only 2 bytes as RAW: its ~2% Gaussian escapes make RAW smaller
    assert kinds == [False, True, False, True, True, True, False]
    dec = [zc.BatchItem(bf16=o, main=it.main, esc=it.esc) for o, it in zip(outs, items)]
    zc.decompress_batched(dec, st)
    torch.cuda.synchronize()
    assert zc.status_value(st) == 0
    for o, x in zip(outs, xs):
        assert np.array_equal(host_u16(o), x)


@pytest.mark.parametrize("n", [1, 2816, 2817, 4097, 6000, 65536 + 3])
def test_decode_oracle_raw_streams(zc, n):
    """RAW streams written by the oracle decode on the GPU."""
    x = random_bits(n, seed=n)
    om, oe, raw = oracle.compress_adaptive(x, DISJOINT)
    assert raw
    main_t = torch.from_numpy(om.copy()).cuda()
    esc_t = torch.from_numpy(np.concatenate([oe, np.zeros(16, np.uint8)])).cuda()
    st = zc.new_status()
    out = zc.decompress(main_t, esc_t, n, st, esc_bytes=oe.size)
    torch.cuda.synchronize()
    assert zc.status_value(st) == 0
    assert np.array_equal(host_u16(out), x)


def test_raw_header_errors(zc):
    n = 6000
    x = random_bits(n, seed=5)
    om, oe, raw = oracle.compress_adaptive(x, DISJOINT)
    assert raw and oe.size > 0
    cases = []
    bad = om.copy()
    bad[6] = 2  # unknown flag
    cases.append((bad, oe, oe.size))
    bad = om.copy()
    bad[24] ^= 2  # n_esc is not the spill
    cases.append((bad, np.concatenate([oe, oe]), 2 * oe.size))
    cases.append((om, oe, oe.size - 1))  # escape stream shorter than the spill
    for m, e, eb in cases:
        assert oracle.decompress_status(m, e[:eb], n)[0] == oracle.ERR_HEADER
        st = zc.new_status()
        zc.decompress(torch.from_numpy(m.copy()).cuda(), torch.from_numpy(e.copy()).cuda(), n, st, esc_bytes=eb)
        torch.cuda.synchronize()
        assert zc.status_value(st) == zc.ERR_BAD_HEADER


@pytest.mark.parametrize("n", [4096 * 8 + 1234, 6913, 4096 * 250 + 3, 4096 * 400 + 5, 4096 * 700 + 77])
def test_reduce_over_raw_and_coded_shards(zc, n):
    """A zipped reduce-scatter receives whatever each sender chose: mixed RAW and coded shards.  Sizes for each
    launch mode: one tile per CTA and round (the teams share the copies; one or two rounds), four tiles per CTA
    in one launch, and the all-coded launch that leaves for the RAW-capable one."""
    P = 5
    cb_in = oracle.codebook_from_sigma(1e-3)
    cb_out = oracle.codebook_from_sigma(1e-3 * np.sqrt(P))
    xs = [workloads.gaussian(n, sigma=1e-3, seed=300 + r) for r in range(P)]
    streams = [oracle.compress_adaptive(x, DISJOINT if r in (1, 4) else cb_in) for r, x in enumerate(xs)]
    assert [s[2] for s in streams] == [False, True, False, False, True]
    y, om, oe = oracle.decompress_reduce([s[0] for s in streams], [s[1] for s in streams], n, out_cb=cb_out)
    mains = [torch.from_numpy(s[0].copy()).cuda() for s in streams]
    escs = [torch.from_numpy(np.concatenate([s[1], np.zeros(16, np.uint8)])).cuda() for s in streams]
    st = zc.new_status()
    ws = zc.workspace(n)
    out, out_main, out_esc = zc.decompress_reduce(mains, escs, n, st, out_cb=zc.codebook_to_device(cb_out), ws=ws,
                                                  esc_bytes=[s[1].size for s in streams])
    torch.cuda.synchronize()
    assert zc.status_value(st) == 0, zc.status_string(zc.status_value(st))
    assert np.array_equal(host_u16(out), y)
    assert np.array_equal(host_u8(out_main), om)
    assert np.array_equal(host_u8(out_esc)[:oe.size], oe)


@pytest.mark.slow
def test_full_size_raw_image(zc):
    """2^26 random-bit values (no exponent in the codebook): the RAW image at full size equals the input bytes."""
    n = 1 << 26
    x = random_bits(n, seed=26)
    gm, ge, main_t, esc_t = gpu_adaptive(zc, x, DISJOINT)
    img = x.view(np.uint8)
    ntiles = -(-n // 4096)
    R = -(-4 * ntiles // 128) * 128
    region = 5632 * ntiles
    assert oracle.header_fields(gm)["flags"] == 1
    assert not gm[128:128 + R].any()
    assert np.array_equal(gm[128 + R:], img[:region])
    assert np.array_equal(ge, img[region:])
    st = zc.new_status()
    out = zc.decompress(main_t, esc_t, n, st)
    torch.cuda.synchronize()
    assert zc.status_value(st) == 0
    assert np.array_equal(host_u16(out), x)
