"""Pins for the oracle's encoder and decoder against what the pages and the format fix.

* a hand-worked byte fixture (tests/golden/worked_example_n1030.json),
* bit-exact round trip of all 65,536 BF16 patterns under three codebooks
  (losslessness, [ZipCCL §2.B] and the bit-exact claim of [ZipCCL §5]),
* the size law 16 -> 11 bits per value plus 8 per escape [ZipCCL §2.B],
* an independent vectorised reader of the format (numpy unpackbits and a
  permutation table) on random data,
* escape counts against numpy's own count of exponents outside the codebook,
* error statuses for corrupted streams and escape overflow.
"""
import json
import os

import numpy as np
import pytest

import oracle
import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _h(s):
    return int(s, 16)


# ------------------------------------------------------------ hand-worked fixture
def _fixture():
    with open(os.path.join(GOLDEN, "worked_example_n1030.json")) as f:
        return json.load(f)


def _fixture_input(fx):
    x = np.full(fx["n"], _h(fx["default_bits"]), np.uint16)
    for k, v in fx["elements"].items():
        x[int(k)] = _h(v["bits"])
    return x


def _fixture_expected_main(fx):
    main = np.zeros(fx["main_bytes"], np.uint8)
    nz = fx["nonzero_bytes"]
    for off, v in nz["header"].items():
        main[int(off)] = _h(v)
    blocks = {0: 256, 1: 256 + 1408}
    for b, base in blocks.items():
        for off, v in nz[f"block{b}_sign_mantissa"].items():
            main[base + int(off)] = _h(v)
        for c in range(3):
            spec = dict(nz[f"block{b}_plane{c}"])
            pbase = base + 1024 + 128 * c
            if "default" in spec:
                main[pbase:pbase + 128] = _h(spec.pop("default"))
            for off, v in spec.items():
                main[pbase + int(off)] = _h(v)
    return main


def test_worked_example_bytes():
    fx = _fixture()
    x = _fixture_input(fx)
    main, esc = oracle.compress(x, fx["codebook"])
    expected = _fixture_expected_main(fx)
    assert main.size == fx["main_bytes"] == oracle.main_bytes(fx["n"])
    diff = np.nonzero(main != expected)[0]
    assert diff.size == 0, f"first differing bytes at {diff[:10]}: got {main[diff[:10]]}, want {expected[diff[:10]]}"
    assert esc.tolist() == fx["escapes"]


def test_worked_example_decodes():
    fx = _fixture()
    x = _fixture_input(fx)
    out = oracle.decompress(_fixture_expected_main(fx), np.array(fx["escapes"], np.uint8), fx["n"])
    assert np.array_equal(out, x)


def test_worked_example_element_fields():
    """The fixture's per-element e / sm / code columns agree with the IEEE bfloat16 field layout."""
    fx = _fixture()
    cb = fx["codebook"]
    for k, v in fx["elements"].items():
        u = _h(v["bits"])
        sign, e, m = u >> 15, (u >> 7) & 0xFF, u & 0x7F
        assert e == v["e"]
        assert (sign << 7 | m) == _h(v["sm"])
        assert v["code"] == (cb.index(e) + 1 if e in cb else 0)
        i = int(k) % 1024
        assert v["q"] == 4 * ((i // 8) % 32) + i // 256 and v["j"] == i % 8


# ------------------------------------------------------------ round trip, every pattern
def _codebooks():
    sigma_cb = oracle.codebook_from_sigma(0.02)
    return {
        "sigma_0.02": sigma_cb,
        "with_0_and_255": np.array([255, 0, 127, 1, 254, 128, 126], np.uint8),
        "high_window": np.array([140, 141, 142, 143, 144, 145, 146], np.uint8),
    }


@pytest.mark.parametrize("name", ["sigma_0.02", "with_0_and_255", "high_window"])
def test_roundtrip_all_65536_patterns(name):
    cb = _codebooks()[name]
    x = workloads.all_bf16_patterns()
    main, esc = oracle.compress(x, cb)
    exps = (x >> 7) & 0xFF
    assert esc.size == int(np.count_nonzero(~np.isin(exps, cb)))
    out = oracle.decompress(main, esc, x.size)
    assert np.array_equal(out, x)


def test_all_escape_tensor():
    """Data whose exponents avoid the codebook: every value escapes, still lossless."""
    cb = np.array([120, 121, 122, 123, 124, 125, 126], np.uint8)
    x = workloads.all_bf16_patterns()
    x = x[~np.isin((x >> 7) & 0xFF, cb)][:9000]
    main, esc = oracle.compress(x, cb)
    assert esc.size == x.size
    assert np.array_equal(esc, ((x >> 7) & 0xFF)[np.argsort(_plane_order_index(x.size), kind="stable")].astype(np.uint8))
    assert np.array_equal(oracle.decompress(main, esc, x.size), x)


def _plane_order_index(n):
    """Position of each element in the escape order when every element escapes."""
    perm = _block_perm()            # plane-bit position -> block element
    inv = np.empty(1024, np.int64)
    inv[perm] = np.arange(1024)
    idx = np.arange(n)
    return (idx // 1024) * 1024 + inv[idx % 1024]


# ------------------------------------------------------------ size law
@pytest.mark.parametrize("n", [0, 1, 7, 4095, 4096, 4097, 3 * 4096, 1 << 20])
def test_main_bytes_formula(n):
    ntiles = -(-n // 4096)
    table = -(-(4 * ntiles) // 128) * 128
    assert oracle.main_bytes(n) == 128 + table + 5632 * ntiles


def test_size_law_eleven_bits_per_value():
    """At zero escapes a full tile costs 11 bits per value: 5632 / 8192 = 0.6875 (a 31.25% saving)."""
    cb = oracle.codebook_from_sigma(0.02)
    rng = np.random.default_rng(7)
    n = 8 * 4096
    e = cb[rng.integers(0, 7, n)].astype(np.uint16)
    x = (rng.integers(0, 2, n).astype(np.uint16) << 15) | (e << 7) | rng.integers(0, 128, n).astype(np.uint16)
    main, esc = oracle.compress(x, cb)
    assert esc.size == 0
    payload = main.size - 128 - 128
    assert payload * 8 == 11 * n
    assert payload / (2 * n) == 0.6875


def test_size_identity_with_escapes():
    x = workloads.gradient(n=3 * 4096 + 123, seed=11)
    cb = oracle.codebook_from_sigma(1e-3)
    main, esc = oracle.compress(x, cb)
    n = x.size
    ntiles = -(-n // 4096)
    table = -(-(4 * ntiles) // 128) * 128
    # bits: 11 per value + 8 per escape + header, table and last-tile padding at 11 bits per padded slot
    assert (main.size + esc.size) * 8 == 11 * n + 8 * esc.size + 8 * (128 + table) + 11 * (ntiles * 4096 - n)


# ------------------------------------------------------------ independent vectorised reader
def _block_perm():
    """perm[p] = block element held by plane-bit position p = 8*q + j (column-major 4 x 32 byte matrix)."""
    q = np.arange(128).repeat(8)
    j = np.tile(np.arange(8), 128)
    return 256 * (q % 4) + 8 * (q // 4) + j


def numpy_reader(main, esc, n):
    """Decode a ZC1 stream with numpy reshapes -- a second formulation of the layout."""
    main = np.asarray(main, np.uint8)
    hdr = oracle.header_fields(main)
    cb = np.array(hdr["codebook"], np.uint8)
    ntiles = hdr["ntiles"]
    table = -(-(4 * ntiles) // 128) * 128
    offs = main[128:128 + 4 * ntiles].view("<u4").astype(np.int64)
    blocks = main[128 + table: 128 + table + 5632 * ntiles].reshape(ntiles * 4, 1408)
    sm = blocks[:, :1024]
    bits = np.unpackbits(blocks[:, 1024:].reshape(-1, 3, 128), axis=-1, bitorder="little")  # (B, 3, 1024) plane order
    perm = _block_perm()
    code_plane_order = bits[:, 0] | (bits[:, 1] << 1) | (bits[:, 2] << 2)
    code = np.empty_like(code_plane_order)
    code[:, perm] = code_plane_order
    code = code.reshape(-1)[:n]
    sm = sm.reshape(-1)[:n].astype(np.uint16)
    e = np.where(code > 0, cb[np.maximum(code, 1) - 1], 0).astype(np.uint16)
    # escapes: plane order inside each block, blocks in order; tile offsets must match the running count
    valid = np.zeros(ntiles * 4096, bool)
    valid[:n] = True
    is_esc_plane = (code_plane_order == 0) & valid.reshape(-1, 1024)[:, perm]
    esc_elem = (np.arange(ntiles * 4)[:, None] * 1024 + perm[None, :])[is_esc_plane]
    tile_counts = np.bincount(esc_elem // 4096, minlength=ntiles)
    assert np.array_equal(offs, np.concatenate([[0], np.cumsum(tile_counts)[:-1]]) if ntiles else offs)
    e[esc_elem] = esc[: esc_elem.size]
    return ((sm & 0x80) << 8) | (e << 7) | (sm & 0x7F)


@pytest.mark.parametrize("seed,n,sigma", [(1, 1 << 16, 0.02), (2, 3 * 4096 + 1000, 1e-3), (3, 777, 0.5)])
def test_numpy_reader_agrees(seed, n, sigma):
    x = workloads.gradient(n=n, sigma=sigma, seed=seed)
    cb = oracle.codebook_from_sigma(sigma)
    main, esc = oracle.compress(x, cb)
    assert np.array_equal(numpy_reader(main, esc, n), x)
    assert np.array_equal(oracle.decompress(main, esc, n), x)


def test_numpy_reader_on_fixture():
    fx = _fixture()
    x = _fixture_input(fx)
    main = _fixture_expected_main(fx)
    assert np.array_equal(numpy_reader(main, np.array(fx["escapes"], np.uint8), fx["n"]), x)


# ------------------------------------------------------------ header and edge cases
def test_header_fields():
    x = workloads.gaussian(n=5000, seed=3)
    cb = oracle.codebook_from_sigma(0.02)
    main, esc = oracle.compress(x, cb)
    h = oracle.header_fields(main)
    assert h == {"magic": 0x3142435A, "version": 1, "flags": 0, "n": 5000, "tile_elems": 4096,
                 "ntiles": 2, "n_esc": esc.size, "codebook": cb.tolist()}
    assert bytes(main[:4]) == b"ZCB1"


def test_empty_tensor():
    main, esc = oracle.compress(np.zeros(0, np.uint16), oracle.codebook_from_sigma(0.02))
    assert main.size == 128 and esc.size == 0
    assert oracle.decompress(main, esc, 0).size == 0


@pytest.mark.parametrize("n", [1, 7, 31, 32, 255, 256, 257, 1023, 1024, 1025, 4095, 4096, 4097])
def test_ragged_sizes_roundtrip(n):
    x = workloads.gradient(n=n, sigma=1e-3, seed=n)
    cb = oracle.codebook_from_sigma(1e-3)
    main, esc = oracle.compress(x, cb)
    assert np.array_equal(oracle.decompress(main, esc, n), x)
    assert np.array_equal(numpy_reader(main, esc, n), x)


def test_padding_is_not_escape():
    """Positions past n carry code 0 but are not escapes, even when exponent 0 is absent from the codebook."""
    cb = np.array([120, 121, 122, 123, 124, 125, 126], np.uint8)
    x = np.full(5, 0x3D80, np.uint16)   # e = 123
    main, esc = oracle.compress(x, cb)
    assert esc.size == 0


def test_duplicate_codebook_rejected():
    with pytest.raises(oracle.OracleError) as ei:
        oracle.compress(np.zeros(4, np.uint16), [1, 2, 3, 4, 5, 6, 6])
    assert ei.value.code == oracle.ERR_CODEBOOK


def test_escape_overflow_reported():
    x = workloads.gradient(n=4096, seed=5)
    cb = oracle.codebook_from_sigma(1e-3)
    _, esc_full = oracle.compress(x, cb)
    main, esc, rc = oracle.compress(x, cb, esc_capacity=esc_full.size - 1, allow_overflow=True)
    assert rc == oracle.ERR_ESCAPE_OVERFLOW


def test_corrupt_streams_rejected():
    x = workloads.gradient(n=3 * 4096, seed=6)
    cb = oracle.codebook_from_sigma(1e-3)
    main, esc = oracle.compress(x, cb)
    bad = main.copy(); bad[0] ^= 1
    assert oracle.decompress_status(bad, esc, x.size)[0] == oracle.ERR_HEADER
    assert oracle.decompress_status(main, esc, x.size + 1)[0] == oracle.ERR_SIZE
    bad = main.copy(); bad[128 + 4:128 + 8] = np.frombuffer((10 ** 6).to_bytes(4, "little"), np.uint8)
    assert oracle.decompress_status(bad, esc, x.size)[0] == oracle.ERR_CORRUPT
    assert oracle.decompress_status(main, esc[:-1], x.size)[0] == oracle.ERR_HEADER
    bad = main.copy(); bad[33] = bad[32]
    assert oracle.decompress_status(bad, esc, x.size)[0] == oracle.ERR_HEADER
