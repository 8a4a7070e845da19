"""CPU-side checks of libzc: it loads, exports every entry point include/zc.h declares, and its host logic
(sigma closed form, sizes, argument validation) behaves -- no kernel is launched here."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle
from lossless_bf16_exponent_zc_gb300 import zc

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "zc.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(z[cq]_[a-z_]+)\s*\(", text)))


def test_library_exports_every_declared_symbol():
    lib = zc.load()
    names = declared_functions()
    assert {"zc_codebook_from_sigma", "zc_histogram_topk", "zc_compress", "zc_decompress", "zc_decompress_reduce",
            "zc_compressed_size", "zc_workspace_size", "zc_compress_batched", "zc_decompress_batched",
            "zc_status_string", "zc_version", "zc_compress_adaptive", "zc_compress_batched_adaptive",
            "zc_raw_spill", "zc_pipeline_workspace_size", "zc_pipelined_transfer",
            "zc_pipeline_plan_create", "zc_pipeline_plan_launch", "zc_pipeline_plan_destroy", "zq_default_widths",
            "zq_table_from_histogram", "zq_max_bytes", "zq_compress", "zq_decompress", "zc_transfer_pays",
            "zc_reduce_scatter_choose"} <= set(names)
    for name in names:
        assert hasattr(lib, name), name


def test_version_and_status_strings():
    assert zc.version().startswith("libzc")
    for i, name in enumerate(zc.STATUS_NAMES):
        assert zc.status_string(i) == name
    assert zc.status_string(999) == "ZC_ERR_UNKNOWN"


@pytest.mark.parametrize("sigma", list(np.exp(np.linspace(np.log(1e-6), np.log(10.0), 120))) + [1e-38, 1e30])
def test_sigma_closed_form_matches_oracle(sigma):
    assert np.array_equal(zc.codebook_from_sigma(sigma), oracle.codebook_from_sigma(sigma))


def test_sigma_rejects_bad_values():
    for s in (0.0, -1.0, float("nan"), float("inf")):
        with pytest.raises(zc.ZcError) as ei:
            zc.codebook_from_sigma(s)
        assert ei.value.code == zc.ERR_INVALID_ARG


@pytest.mark.parametrize("n", [0, 1, 4095, 4096, 4097, 1 << 20, 67108864, 218103808 // 9, (1 << 32) - 1])
def test_sizes_match_oracle(n):
    mb, eb = zc.compressed_size(n)
    assert mb == oracle.main_bytes(n) and eb == n


def test_too_large():
    with pytest.raises(zc.ZcError) as ei:
        zc.compressed_size(1 << 32)
    assert ei.value.code == zc.ERR_TOO_LARGE


def test_workspace_size_formula():
    assert zc.workspace_size(0) == 4096
    assert zc.workspace_size([4096, 4097, 1]) == 4096 + 16 * (1 + 2 + 1)
    assert zc.workspace_size(1 << 26) == 4096 + 16 * (1 << 14)


def _raw(name, *args):
    return getattr(zc.load(), name)(*args)


def test_argument_errors_are_synchronous():
    """Bad arguments are rejected on the host before anything is enqueued (no GPU needed)."""
    E = zc
    # null pointers
    assert _raw("zc_compress", None, 10, None, None, None, 0, None, 0, None, None) == E.ERR_INVALID_ARG
    assert _raw("zc_decompress", None, None, 0, 10, None, None, None) == E.ERR_INVALID_ARG
    assert _raw("zc_histogram_topk", None, 10, None, None, None, 0, None, None) == E.ERR_INVALID_ARG
    # misaligned pointers (never dereferenced)
    fake = 0x10000
    status = 0x20000
    assert _raw("zc_compress", fake + 2, 10, fake, fake, fake, 10, fake, 1 << 20, status, None) == E.ERR_ALIGNMENT
    assert _raw("zc_decompress", fake + 8, fake, 10, 10, fake, status, None) == E.ERR_ALIGNMENT
    assert _raw("zc_compress", fake, 10, fake, fake, fake, 10, fake, 1 << 20, status + 2, None) == E.ERR_ALIGNMENT
    # workspace too small
    assert _raw("zc_compress", fake, 1 << 20, fake, fake, fake, 10, fake, 4096, status, None) == E.ERR_WORKSPACE
    # n too large
    assert _raw("zc_compress", fake, 1 << 32, fake, fake, fake, 10, fake, 1 << 40, status, None) == E.ERR_TOO_LARGE
    # shard count out of range
    arr = (ctypes.c_void_p * 1)(fake)
    sz = (ctypes.c_uint64 * 1)(0)
    assert _raw("zc_decompress_reduce", 0, arr, arr, sz, 10, fake, None, None, None, 0, None, 0, status,
                None) == E.ERR_INVALID_ARG
    assert _raw("zc_decompress_reduce", 65, arr, arr, sz, 10, fake, None, None, None, 0, None, 0, status,
                None) == E.ERR_INVALID_ARG
    # neither output requested
    assert _raw("zc_decompress_reduce", 1, arr, arr, sz, 10, None, None, None, None, 0, None, 0, status,
                None) == E.ERR_INVALID_ARG
    # batched: empty batch
    assert _raw("zc_compress_batched", 0, None, None, 0, status, None) == E.ERR_INVALID_ARG


@pytest.mark.parametrize("n", [0, 1, 2816, 2817, 4096, 65536, (1 << 26) + 5])
def test_raw_spill_matches_oracle(n):
    assert zc.raw_spill(n) == oracle.raw_spill(n)


def test_adaptive_argument_errors_are_synchronous():
    E = zc
    assert _raw("zc_compress_adaptive", None, 10, None, None, None, 0, None, 0, None, None) == E.ERR_INVALID_ARG
    fake, status = 1 << 20, 1 << 21
    assert _raw("zc_compress_adaptive", fake + 2, 10, fake, fake, fake, 10, fake, 1 << 20, status,
                None) == E.ERR_ALIGNMENT
    assert _raw("zc_compress_adaptive", fake, 1 << 20, fake, fake, fake, 10, fake, 4096, status,
                None) == E.ERR_WORKSPACE
    assert _raw("zc_compress_batched_adaptive", 0, None, None, 0, status, None) == E.ERR_INVALID_ARG
    with pytest.raises(zc.ZcError):
        zc.raw_spill(1 << 32)


def test_pipeline_workspace_size():
    for c in (8, 4096, 4104, 1 << 20):
        ws = zc.pipeline_workspace_size(c)
        # the encoder's workspace plus two send and two receive slots of a main stream and escape bytes
        assert ws >= zc.workspace_size(c) + 4 * (oracle.main_bytes(c) + oracle.raw_spill(c))
    for bad in (0, 4, 4100):
        with pytest.raises(zc.ZcError) as e:
            zc.pipeline_workspace_size(bad)
        assert e.value.code == zc.ERR_INVALID_ARG
    fake, status = 1 << 20, 1 << 21
    assert _raw("zc_pipelined_transfer", fake, 10, fake, fake, 4100, fake, 1 << 30, status, None, None,
                None) == zc.ERR_INVALID_ARG
    assert _raw("zc_pipelined_transfer", fake + 2, 10, fake, fake, 4096, fake, 1 << 30, status, None, None,
                None) == zc.ERR_ALIGNMENT
    assert _raw("zc_pipelined_transfer", fake, 10, fake, fake, 4096, fake, 100, status, None, None,
                None) == zc.ERR_WORKSPACE


def test_pipeline_plan_argument_errors():
    """The plan applies zc_pipelined_transfer's checks before it captures anything; a failed create leaves
    *plan NULL, and NULL plans are rejected (launch) or accepted (destroy)."""
    import ctypes
    fake, status = 1 << 20, 1 << 21
    plan = ctypes.c_void_p(1234)
    assert _raw("zc_pipeline_plan_create", fake, 10, fake, fake, 4100, fake, 1 << 30, status, 1,
                ctypes.byref(plan)) == zc.ERR_INVALID_ARG
    assert plan.value is None
    assert _raw("zc_pipeline_plan_create", fake + 2, 10, fake, fake, 4096, fake, 1 << 30, status, 1,
                ctypes.byref(plan)) == zc.ERR_ALIGNMENT
    assert _raw("zc_pipeline_plan_create", fake, 10, fake, fake, 4096, fake, 100, status, 0,
                ctypes.byref(plan)) == zc.ERR_WORKSPACE
    assert _raw("zc_pipeline_plan_create", fake, 10, None, fake, 4096, fake, 1 << 30, status, 1,
                ctypes.byref(plan)) == zc.ERR_INVALID_ARG
    assert _raw("zc_pipeline_plan_create", fake, 10, fake, fake, 4096, fake, 1 << 30, status, 1,
                None) == zc.ERR_INVALID_ARG
    assert _raw("zc_pipeline_plan_launch", None, None) == zc.ERR_INVALID_ARG
    assert _raw("zc_pipeline_plan_destroy", None) == zc.OK


def test_qlc_host_functions_match_oracle():
    assert tuple(zc.zq_default_widths()) == tuple(oracle.QLC_DEFAULT_WIDTHS)
    rng = np.random.default_rng(7)
    for _ in range(5):
        h = rng.integers(0, 50, 256)
        t = zc.zq_table_from_histogram(h)
        assert np.array_equal(np.frombuffer(bytes(t.sym), np.uint8), oracle.qlc_table_from_histogram(h))
    for n in (0, 1, 4096, 4097, 10 ** 6):
        assert zc.zq_max_bytes(n) == oracle.qlc_max_bytes(n)
    with pytest.raises(zc.ZcError) as e:
        zc.zq_table_from_histogram(np.ones(256), widths=(3, 3, 3, 3, 3, 3, 3, 3))
    assert e.value.code == zc.ERR_CODEBOOK
    fake, status = 1 << 20, 1 << 21
    bad = zc.zq_table((3, 3, 3, 3, 3, 3, 3, 3), range(256))
    assert zc.load().zq_compress(fake, 100, ctypes.byref(bad), fake, 1 << 20, fake, 1 << 20, status,
                                 None) == zc.ERR_CODEBOOK


# ------------------------------------------------------------------ cost models (host arithmetic)
def test_transfer_cost_model_break_even():
    """[CCCL §2.2]: compressing pays while compress + decompress + sending the smaller data beats sending the
    raw data.  Latency appears on both sides, so the break-even link bandwidth is (1 - 1/ratio) / (1/c + 1/d)."""
    c, d, r = 2800.0, 2900.0, 1.43
    bw_star = (1 - 1 / r) / (1 / c + 1 / d)
    assert zc.transfer_pays(1 << 28, bw_star * 0.99, 7.0, c, d, r)[0]
    assert not zc.transfer_pays(1 << 28, bw_star * 1.01, 7.0, c, d, r)[0]
    # a ratio of 1 or less never pays, however fast the codec
    for ratio in (1.0, 0.9):
        assert not zc.transfer_pays(1 << 30, 0.001, 0.0, 1e12, 1e12, ratio)[0]
    # times in microseconds: 1 MB over 1 GB/s is 1000 us
    pays, t_raw, t_zip = zc.transfer_pays(10 ** 6, 1.0, 2.0, 1000.0, 500.0, 2.0)
    assert t_raw == pytest.approx(1002.0) and t_zip == pytest.approx(1.0 + 2.0 + 500.0 + 2.0) and pays


def test_reduce_scatter_switcher():
    """[ZipCCL §2.D] switcher: native ring (P - 1 steps of bytes / P) against compress + one all-to-all of the
    compressed shards + decompress-reduce.  With no latency the break-even bandwidth is
    (P - 1) / P * (1 - 1/ratio) / (1/c + 1/d)."""
    c, d, r, P = 2800.0, 1300.0, 1.43, 8
    bw_star = (P - 1) / P * (1 - 1 / r) / (1 / c + 1 / d)
    assert zc.reduce_scatter_choose(1 << 28, P, bw_star * 0.99, 0.0, c, d, r)[0]
    assert not zc.reduce_scatter_choose(1 << 28, P, bw_star * 1.01, 0.0, c, d, r)[0]
    # one rank: nothing to send, the native path costs nothing
    use, t_native, t_zip = zc.reduce_scatter_choose(1 << 20, 1, 10.0, 5.0, c, d, r)
    assert not use and t_native == 0.0 and t_zip > 0
    # many small messages: the ring pays P - 1 latencies, the all-to-all one
    use, t_native, t_zip = zc.reduce_scatter_choose(1 << 10, 64, 100.0, 20.0, c, d, r)
    assert use and t_native == pytest.approx(63 * (20.0 + (1 << 10) / 64 / 100e3))


def test_cost_model_argument_errors():
    for args in ((1, -1.0, 1.0, 1.0, 1.0, 1.0), (1, 1.0, -1.0, 1.0, 1.0, 1.0), (1, 1.0, 1.0, 0.0, 1.0, 1.0),
                 (1, 1.0, 1.0, 1.0, 1.0, 0.0), (1, float("nan"), 1.0, 1.0, 1.0, 1.0)):
        with pytest.raises(zc.ZcError) as e:
            zc.transfer_pays(*args)
        assert e.value.code == zc.ERR_INVALID_ARG
    with pytest.raises(zc.ZcError):
        zc.reduce_scatter_choose(1, 0, 1.0, 1.0, 1.0, 1.0, 1.0)
