"""Pins for the oracle's raw bypass (RAW streams, header flags bit 0).

[CCCL §3.3] keeps tiny tensors uncompressed and [CCCL §5.2] falls back to
sending the data as is when compression does not shrink it.  The reading
taken: a RAW stream keeps the main stream's size, holds the values' own
little-endian bytes (tile region first, the rest in the escape stream), and
the adaptive encoder picks it exactly when it is strictly smaller than the
coded form.  Pinned here against what that definition fixes by itself:

* the RAW image equals numpy's own byte view of the input (byte order,
  tile region / escape split, zero table and zero tail);
* the spill 2n - 5632 ceil(n/4096) from the closed form;
* the decision against numpy's count of exponents outside the codebook,
  including both sides of the threshold (escapes == spill stays coded,
  spill + 1 goes RAW);
* round trips of RAW streams, the overflow rescue and the header checks.
"""
import numpy as np
import pytest

import oracle
import workloads

DISJOINT = [250, 251, 252, 253, 254, 249, 248]  # exponents no test input below uses


def _spill(n):
    region = 5632 * ((n + 4095) // 4096)
    return max(0, 2 * n - region)


def _escapes(x, cb):
    e = (np.asarray(x, np.uint16) >> 7) & 0xFF
    return int(np.count_nonzero(~np.isin(e, np.asarray(cb))))


def _tables(n):
    ntiles = (n + 4095) // 4096
    R = -(-4 * ntiles // 128) * 128
    return ntiles, R


@pytest.mark.parametrize("n", [0, 1, 7, 2816, 2817, 4096, 4097, 10000, 65536])
def test_spill_closed_form(n):
    assert oracle.raw_spill(n) == _spill(n)


def _check_raw_image(x, main, esc):
    n = x.size
    ntiles, R = _tables(n)
    region = 5632 * ntiles
    img = x.astype("<u2").view(np.uint8)  # numpy's little-endian byte image
    h = oracle.header_fields(main)
    assert h["flags"] == 1 and h["n"] == n and h["ntiles"] == ntiles and h["n_esc"] == _spill(n)
    assert not main[128:128 + R].any(), "offset table of a RAW stream is zero"
    tiles = main[128 + R:]
    assert tiles.size == region
    k = min(2 * n, region)
    assert np.array_equal(tiles[:k], img[:k])
    assert not tiles[k:].any(), "tile region beyond the data is zero"
    assert np.array_equal(esc, img[k:])


def test_raw_image_all_patterns():
    x = np.arange(65536, dtype=np.uint16)
    cb = list(range(7))
    main, esc, raw = oracle.compress_adaptive(x, cb)
    assert _escapes(x, cb) > _spill(x.size) and raw
    _check_raw_image(x, main, esc)
    assert np.array_equal(oracle.decompress(main, esc, x.size), x)


@pytest.mark.parametrize("n", [1, 5, 2816, 2817, 4095, 4096, 4097, 12289])
def test_raw_image_ragged(n):
    rng = np.random.default_rng(n)
    x = rng.integers(0, 65536, n, dtype=np.uint16)
    main, esc, raw = oracle.compress_adaptive(x, DISJOINT)
    # uniform random bits: escapes are every value whose exponent is not in DISJOINT
    assert raw == (_escapes(x, DISJOINT) > _spill(n))
    if raw:
        _check_raw_image(x, main, esc)
    assert np.array_equal(oracle.decompress(main, esc, n), x)


def test_tiny_tensor_with_one_escape_goes_raw():
    # n = 1: the whole value fits in the tile region, spill 0, any escape makes RAW smaller
    x = np.array([0x3F80], np.uint16)  # 1.0, exponent 127
    main, esc, raw = oracle.compress_adaptive(x, DISJOINT)
    assert raw and esc.size == 0
    assert main[256] == 0x80 and main[257] == 0x3F
    assert np.array_equal(oracle.decompress(main, esc, 1), x)
    # the same value with a codebook that holds its exponent stays coded
    main2, esc2, raw2 = oracle.compress_adaptive(x, [127, 1, 2, 3, 4, 5, 6])
    assert not raw2 and esc2.size == 0 and oracle.header_fields(main2)["flags"] == 0


def _threshold_input(n, n_escapes):
    """n values with exponent 127 except n_escapes of them with exponent 200."""
    rng = np.random.default_rng(17)
    x = (127 << 7 | rng.integers(0, 128, n)).astype(np.uint16)
    pos = rng.choice(n, n_escapes, replace=False)
    x[pos] = (200 << 7) | (x[pos] & 0x7F)
    return x


@pytest.mark.parametrize("n", [4096, 20000, 40961])
def test_decision_threshold(n):
    cb = [127, 1, 2, 3, 4, 5, 6]
    s = _spill(n)
    assert s > 0
    at = _threshold_input(n, s)
    main, esc, raw = oracle.compress_adaptive(at, cb)
    assert not raw and esc.size == s, "escapes == spill: RAW is not smaller, stays coded"
    plain_main, plain_esc = oracle.compress(at, cb)
    assert np.array_equal(main, plain_main) and np.array_equal(esc, plain_esc)
    over = _threshold_input(n, s + 1)
    main, esc, raw = oracle.compress_adaptive(over, cb)
    assert raw
    _check_raw_image(over, main, esc)
    assert np.array_equal(oracle.decompress(main, esc, n), over)


def test_gaussian_stays_coded():
    x = workloads.gaussian(1 << 16)
    cb = oracle.codebook_from_sigma(workloads.GAUSSIAN_SIGMA)
    main, esc, raw = oracle.compress_adaptive(x, cb)
    plain_main, plain_esc = oracle.compress(x, cb)
    assert not raw
    assert np.array_equal(main, plain_main) and np.array_equal(esc, plain_esc)


def test_overflow_rescued_by_raw():
    n = 8192
    x = np.random.default_rng(3).integers(0, 65536, n, dtype=np.uint16)
    s = _spill(n)
    assert _escapes(x, DISJOINT) > s + 1000
    # the coded form needs far more than s escape bytes; RAW fits exactly
    main, esc, raw = oracle.compress_adaptive(x, DISJOINT, esc_capacity=s)
    assert raw and esc.size == s
    _check_raw_image(x, main, esc)
    # neither fits: the coded output and the overflow stand, as in plain compress
    got = oracle.compress_adaptive(x, DISJOINT, esc_capacity=s - 1, allow_overflow=True)
    assert got[2] is False and got[3] == oracle.ERR_ESCAPE_OVERFLOW
    want = oracle.compress(x, DISJOINT, esc_capacity=s - 1, allow_overflow=True)
    assert np.array_equal(got[0], want[0]) and np.array_equal(got[1], want[1])


def test_raw_header_checks():
    n = 6000  # spill 736
    x = np.random.default_rng(4).integers(0, 65536, n, dtype=np.uint16)
    main, esc, raw = oracle.compress_adaptive(x, DISJOINT)
    assert raw
    bad = main.copy()
    bad[6] = 2  # unknown flag bit
    assert oracle.decompress_status(bad, esc, n)[0] == oracle.ERR_HEADER
    bad = main.copy()
    bad[24] ^= 1  # n_esc differs from the spill
    assert oracle.decompress_status(bad, np.concatenate([esc, esc]), n)[0] == oracle.ERR_HEADER
    # the escape stream shorter than the spill
    assert oracle.decompress_status(main, esc[:-1], n)[0] == oracle.ERR_HEADER
    # a coded stream with the RAW flag set: its n_esc is not the spill
    cm, ce = oracle.compress(workloads.gaussian(4096), oracle.codebook_from_sigma(0.02))
    flip = cm.copy()
    flip[6] = 1
    assert oracle.decompress_status(flip, ce, 4096)[0] == oracle.ERR_HEADER  # n_esc != spill


def test_reduce_over_raw_and_coded_shards():
    # a zipped reduce-scatter receives whatever each sender chose: shards 1 and
    # 3 arrive RAW (disjoint codebook), 0 and 2 coded; the reduction equals
    # torch's fp32 adds in rank order rounded to bfloat16
    import torch

    n = 9000
    xs = [workloads.gaussian(n, sigma=1e-3, seed=40 + r) for r in range(4)]
    cb = oracle.codebook_from_sigma(1e-3)
    streams = [oracle.compress_adaptive(x, DISJOINT if r % 2 else cb) for r, x in enumerate(xs)]
    assert [s[2] for s in streams] == [False, True, False, True]
    y = oracle.decompress_reduce([s[0] for s in streams], [s[1] for s in streams], n)
    acc = torch.from_numpy(xs[0].view(np.int16).copy()).view(torch.bfloat16).float()
    for x in xs[1:]:
        acc = acc + torch.from_numpy(x.view(np.int16).copy()).view(torch.bfloat16).float()
    want = acc.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(y, want)
