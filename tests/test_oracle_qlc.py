"""Pins for the oracle's Quad Length Codes (FP8 e4m3) encoder and decoder.

[QLC §3.1-§3.3]: a 3-bit prefix picks one of 8 regions of the frequency-ranked
symbol space, the region fixes how many bits follow; [QLC §4.1-§4.2]: one
table lookup per symbol each way.  Pinned against what the definition and
the mathematics fix by themselves:

* a hand-worked stream (tests/golden/qlc_worked_example_n6.json), whose first
  two codes are the article's lookup-table example (symbol 113 -> 000_000,
  symbol 24 -> 000_001);
* a second hand-worked stream of two blocks
  (tests/golden/qlc_worked_example_two_blocks.json): a lane coding two runs, a
  ragged last run, an 11-bit code across a word boundary, the lane-count bytes
  and the block offsets, compared byte for byte with the whole stream;
* an independent ZQ1 reader (numpy, written from the layout's prose: the lane
  -> run map from a reshape, bits from unpackbits) that must decode the
  oracle's multi-block ragged streams to their input;
* bit-exact round trips of all 256 byte values and of random data under the
  default and dynamic tables, ragged sizes;
* prefix-freeness: the code lengths of every valid table satisfy Kraft's
  inequality, and the four lengths of the default table are 6/7/8/11;
* Shannon's bound: no stream's payload is shorter than n times the empirical
  entropy of its bytes, and the frequency ranking never gives a rarer symbol
  a shorter code;
* table and stream errors.
"""
import json
import os

import numpy as np
import pytest

import oracle
import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
DEFAULT = oracle.QLC_DEFAULT_WIDTHS
DYNAMIC = (1, 3, 4, 5, 5, 5, 5, 8)  # a 2-symbol region of 4-bit codes, wider middle regions ([QLC §3.3])


def _fixture():
    with open(os.path.join(GOLDEN, "qlc_worked_example_n6.json")) as f:
        return json.load(f)


def test_worked_example_stream():
    fx = _fixture()
    sym = np.array([113, 24] + [v for v in range(256) if v not in (24, 113)], np.uint8)
    s = oracle.qlc_compress(np.array(fx["symbols"], np.uint8), fx["widths"], sym)
    assert s.size == fx["stream_bytes"]
    h = fx["header"]
    assert int.from_bytes(s[0:4].tobytes(), "little") == int(h["magic_le_u32"], 16)
    assert s[4] == h["version"] and int.from_bytes(s[8:16].tobytes(), "little") == h["n"]
    assert int.from_bytes(s[16:20].tobytes(), "little") == h["block_symbols"]
    assert int.from_bytes(s[20:24].tobytes(), "little") == h["nblocks"]
    assert int.from_bytes(s[24:32].tobytes(), "little") == h["payload_words"]
    assert list(s[64:72]) == fx["widths"] and np.array_equal(s[128:384], sym)
    assert int.from_bytes(s[384:388].tobytes(), "little") == fx["block_offsets"][0]
    words = s[512:].view("<u4")
    assert [f"0x{w:08X}" for w in words] == fx["payload_words_hex"]
    assert np.array_equal(oracle.qlc_decompress(s, fx["n"]), np.array(fx["symbols"], np.uint8))


def test_article_lookup_example_codes():
    """[QLC §4.1]: the most frequent symbol (113) gets rank 0, code 000_000; the next (24) rank 1, code 000_001."""
    hist = np.ones(256, np.uint64)
    hist[113], hist[24] = 1000, 500
    sym = oracle.qlc_table_from_histogram(hist)
    assert sym[0] == 113 and sym[1] == 24
    for symbol in (113, 24):
        assert oracle.qlc_code_length(DEFAULT, sym, symbol) == 6
    s = oracle.qlc_compress(np.array([113, 24], np.uint8), DEFAULT, sym)
    (word,) = s[512 + 32:512 + 36].view("<u4")  # lane 0 codes both: 000000 000001, then padding
    assert word >> 20 == 0b000000_000001


@pytest.mark.parametrize("widths", [DEFAULT, DYNAMIC, (8, 0, 0, 0, 0, 0, 0, 0), (0, 1, 2, 3, 4, 5, 6, 8)])
def test_roundtrip_all_symbols(widths):
    rng = np.random.default_rng(sum(widths))
    x = rng.permutation(np.tile(np.arange(256, dtype=np.uint8), 37))
    sym = rng.permutation(256).astype(np.uint8)
    assert oracle.qlc_table_is_valid(widths, sym)
    s = oracle.qlc_compress(x, widths, sym)
    assert np.array_equal(oracle.qlc_decompress(s, x.size), x)


@pytest.mark.parametrize("n", [0, 1, 31, 32, 33, 127, 4095, 4096, 4097, 3 * 4096 + 77, 50_000])
def test_roundtrip_ragged(n):
    x = workloads.fp8_ffn1(n, seed=n + 1) if n else np.zeros(0, np.uint8)
    sym = oracle.qlc_table_for(x)
    for widths in (DEFAULT, DYNAMIC):
        s = oracle.qlc_compress(x, widths, sym)
        assert np.array_equal(oracle.qlc_decompress(s, n), x)


def _lengths(widths, sym):
    return np.array([oracle.qlc_code_length(widths, sym, v) for v in range(256)])


@pytest.mark.parametrize("widths", [DEFAULT, DYNAMIC, (8, 0, 0, 0, 0, 0, 0, 0), (2, 2, 2, 2, 8, 8, 8, 8)])
def test_kraft_inequality(widths):
    sym = np.arange(256, dtype=np.uint8)
    L = _lengths(widths, sym)
    assert (L >= 3).all() and np.sum(2.0 ** -L) <= 1.0 + 1e-12


def test_default_table_has_four_lengths():
    """[QLC §3.1]: code lengths 6, 7, 8 and 11 bits only; [QLC §3.2]: the last region is ranks 88-255."""
    sym = np.arange(256, dtype=np.uint8)
    L = _lengths(DEFAULT, sym)
    assert set(L.tolist()) == {6, 7, 8, 11}
    assert (L[:40] == 6).all() and (L[40:56] == 7).all() and (L[56:88] == 8).all() and (L[88:] == 11).all()


@pytest.mark.parametrize("gen", ["ffn1", "gradient", "uniform"])
def test_entropy_bound_and_monotone_lengths(gen):
    n = 1 << 18
    x = {"ffn1": workloads.fp8_ffn1, "gradient": workloads.fp8_gradient}.get(
        gen, lambda n, seed=9: np.random.default_rng(seed).integers(0, 256, n).astype(np.uint8))(n)
    hist = np.bincount(x, minlength=256)
    p = hist[hist > 0] / n
    entropy_bits = -(p * np.log2(p)).sum() * n
    sym = oracle.qlc_table_from_histogram(hist)
    L = _lengths(DEFAULT, sym)
    payload_bits = int((hist * L).sum())
    assert payload_bits >= entropy_bits  # Shannon: no prefix code beats the entropy
    s = oracle.qlc_compress(x, DEFAULT, sym)
    nblocks = -(-n // 4096)
    overhead_bytes = 384 + 4 * nblocks + nblocks * (32 + 32 * 4)  # header, offsets, lane counts, padding
    assert payload_bits / 8 <= s.size <= payload_bits / 8 + overhead_bytes
    # a symbol that occurs more often never has a longer code
    order = np.argsort(-hist, kind="stable")
    assert (np.diff(L[order]) >= 0).all()


def test_table_errors():
    x = np.arange(100, dtype=np.uint8)
    sym = np.arange(256, dtype=np.uint8)
    with pytest.raises(oracle.OracleError):
        oracle.qlc_compress(x, (3, 3, 3, 3, 3, 3, 3, 3), sym)  # 8 x 8 = 64 < 256 ranks
    dup = sym.copy()
    dup[5] = 6
    with pytest.raises(oracle.OracleError):
        oracle.qlc_compress(x, DEFAULT, dup)
    with pytest.raises(oracle.OracleError):
        oracle.qlc_compress(x, (9, 0, 0, 0, 0, 0, 0, 0), sym)


def test_stream_errors():
    x = workloads.fp8_ffn1(10_000, seed=3)
    s = oracle.qlc_compress(x, DEFAULT, oracle.qlc_table_for(x))
    assert oracle.qlc_decompress_status(s, 10_001)[0] == oracle.Q_ERR_SIZE
    bad = s.copy()
    bad[0] ^= 1
    assert oracle.qlc_decompress_status(bad, 10_000)[0] == oracle.Q_ERR_HEADER
    assert oracle.qlc_decompress_status(s[:-4], 10_000)[0] == oracle.Q_ERR_HEADER  # payload cut short
    bad = s.copy()
    bad[512] = 255  # lane 0's word count of block 0 runs past the block
    assert oracle.qlc_decompress_status(bad, 10_000)[0] == oracle.Q_ERR_CORRUPT


# ---------------------------------------------------------------------------------------------
# An independent reader of the ZQ1 stream, written from the layout's prose alone (reading Q3):
# a 384-byte header, one u32 word offset per 4096-symbol block (padded to 128 bytes), the
# payload of u32 words; a block = 8 words whose byte l counts lane l's words, then the lanes'
# words in lane order; the block's symbols are 256 runs of 16 and lane l codes runs l, l + 32,
# ..., l + 224; codes are read most significant bit first from bit 31 of a lane's first word.
# It shares nothing with the oracle's C: the lane -> symbol map comes from a reshape, the bits
# from numpy's unpackbits on big-endian word bytes, and the prefix decode is a table of regions.

def _lane_positions() -> np.ndarray:
    """[lane, j] -> symbol index inside a block: the block as (run round m, lane l, offset p)."""
    block = np.arange(4096).reshape(8, 32, 16)      # run 32 m + l holds symbols 16 (32 m + l) + p
    return block.transpose(1, 0, 2).reshape(32, 128)  # lane l: its runs in order, 16 symbols each


def _zq1_read(stream: np.ndarray):
    """Decode a ZQ1 stream; returns (symbols, per-block lane word counts, block offsets)."""
    s = np.asarray(stream, np.uint8)
    assert s[:4].tobytes() == b"ZQB1" and s[4] == 1
    le = lambda a, b: int.from_bytes(s[a:b].tobytes(), "little")
    n, bsz, nb, nwords = le(8, 16), le(16, 20), le(20, 24), le(24, 32)
    assert bsz == 4096 and nb == -(-n // 4096)
    widths = [int(v) for v in s[64:72]]
    sym = s[128:384]
    table_bytes = -(-4 * nb // 128) * 128
    offsets = [le(384 + 4 * b, 388 + 4 * b) for b in range(nb)]
    payload = s[384 + table_bytes:].view("<u4")
    assert payload.size == nwords
    # region r covers ranks [starts[r], starts[r] + 2**widths[r])
    starts = np.concatenate([[0], np.cumsum([1 << w for w in widths])])
    pos = _lane_positions()
    out = np.zeros(n, np.uint8)
    counts = []
    for b in range(nb):
        off = offsets[b]
        end = offsets[b + 1] if b + 1 < nb else nwords
        lane_counts = payload[off:off + 8].astype("<u4").view(np.uint8)  # 32 bytes, byte l = lane l
        counts.append(lane_counts.tolist())
        assert off + 8 + int(lane_counts.sum(dtype=np.int64)) == end
        first = off + 8
        for lane in range(32):
            words = payload[first:first + int(lane_counts[lane])]
            first += int(lane_counts[lane])
            bits = np.unpackbits(words.astype(">u4").view(np.uint8))
            cursor = 0
            for j in range(128):
                i = 4096 * b + int(pos[lane, j])
                if i >= n:
                    break
                region = int("".join(map(str, bits[cursor:cursor + 3])), 2)
                cursor += 3
                w = widths[region]
                offset = int("".join(map(str, bits[cursor:cursor + w])), 2) if w else 0
                cursor += w
                out[i] = sym[starts[region] + offset]
            assert -(-cursor // 32) == words.size  # exactly the words the lane needs
            assert not bits[cursor:].any()          # zero padding
    return out, counts, offsets


def _two_block_fixture():
    with open(os.path.join(GOLDEN, "qlc_worked_example_two_blocks.json")) as f:
        return json.load(f)


def _fixture_stream(fx) -> np.ndarray:
    """The whole stream spelled out from the fixture's hand-derived fields."""
    h = fx["header"]
    nb = h["nblocks"]
    table_bytes = -(-4 * nb // 128) * 128
    out = np.zeros(384 + table_bytes + 4 * h["payload_words"], np.uint8)
    out[0:4] = np.frombuffer(int(h["magic_le_u32"], 16).to_bytes(4, "little"), np.uint8)
    out[4] = h["version"]
    out[8:16] = np.frombuffer(h["n"].to_bytes(8, "little"), np.uint8)
    out[16:20] = np.frombuffer(h["block_symbols"].to_bytes(4, "little"), np.uint8)
    out[20:24] = np.frombuffer(nb.to_bytes(4, "little"), np.uint8)
    out[24:32] = np.frombuffer(h["payload_words"].to_bytes(8, "little"), np.uint8)
    out[64:72] = fx["widths"]
    out[128:384] = np.arange(256)
    for b, off in enumerate(fx["block_offsets"]):
        out[384 + 4 * b:388 + 4 * b] = np.frombuffer(off.to_bytes(4, "little"), np.uint8)
    words = out[384 + table_bytes:].view("<u4")
    for k, v in fx["nonzero_payload_words_hex"].items():
        words[int(k)] = int(v, 16)
    return out


def _fixture_symbols(fx) -> np.ndarray:
    x = np.full(fx["n"], fx["background_symbol"], np.uint8)
    for m in fx["markers"]:
        x[m["index"]] = m["symbol"]
    return x


def test_two_block_worked_example_bytes():
    """Two blocks, a lane coding two runs, a ragged last run, an 11-bit code across a word boundary:
    the oracle's stream equals the hand-derived one byte for byte (lane counts and offsets included)."""
    fx = _two_block_fixture()
    x = _fixture_symbols(fx)
    s = oracle.qlc_compress(x, fx["widths"], np.arange(256, dtype=np.uint8))
    expect = _fixture_stream(fx)
    assert s.size == fx["stream_bytes"] == expect.size
    assert np.array_equal(s, expect)
    assert np.array_equal(oracle.qlc_decompress(expect, fx["n"]), x)


def test_two_block_worked_example_reader():
    """The independent reader decodes the hand-derived stream to the fixture's symbols."""
    fx = _two_block_fixture()
    out, counts, offsets = _zq1_read(_fixture_stream(fx))
    assert np.array_equal(out, _fixture_symbols(fx))
    assert counts == fx["lane_word_counts"] and offsets == fx["block_offsets"]


def test_lane_positions_cover_a_block():
    pos = _lane_positions()
    assert np.array_equal(np.sort(pos.ravel()), np.arange(4096))
    assert list(pos[1, 14:18]) == [30, 31, 16 * 33, 16 * 33 + 1]  # lane 1: end of run 1, start of run 33


@pytest.mark.parametrize("n", [1, 17, 4096 + 16 * 37 + 9, 3 * 4096 + 16 * 33 + 5, 5 * 4096])
@pytest.mark.parametrize("gen", ["ffn1", "uniform"])
def test_independent_reader_agrees(n, gen):
    """Multi-block, ragged oracle streams under the default and a dynamic table read back by the
    independent reader; a lane -> run assignment or lane-count layout other than reading Q3 fails."""
    rng = np.random.default_rng(n)
    x = workloads.fp8_ffn1(n, seed=n) if gen == "ffn1" else rng.integers(0, 256, n).astype(np.uint8)
    for widths, sym in ((DEFAULT, oracle.qlc_table_for(x)), (DYNAMIC, rng.permutation(256).astype(np.uint8))):
        s = oracle.qlc_compress(x, widths, sym)
        out, counts, offsets = _zq1_read(s)
        assert np.array_equal(out, x)
        assert offsets[0] == 0 and all(a < b for a, b in zip(offsets, offsets[1:]))
