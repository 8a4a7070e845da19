"""CPU oracle for lossless BF16 exponent coding -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
and reference legs may import this package.  The product library never does,
and nothing here imports the product library.

The arithmetic lives in ``zc_oracle.c`` (plain single-threaded C, one function
per step of the method, each citing the passage it follows).  This module only
compiles it on first use and marshals numpy arrays to it.

Every function here is pinned by the ``-m "not gpu"`` tests against something
other than itself: the 65,536-pattern round trip, the size law, a hand-worked
byte fixture, Monte-Carlo exponent frequencies, numpy ``bincount``, and torch
CPU sums (see tests/test_oracle_*.py).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "zc_oracle.c")
_QSRC = os.path.join(_HERE, "qlc_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
# ZC_SANITIZE=1: the same C built with AddressSanitizer and UndefinedBehaviorSanitizer
# (a process that loads it must load the ASan runtime first, LD_PRELOAD)
_SAN_LIB = os.path.join(_HERE, "liboracle_san.so")
_SAN_FLAGS = ["-fsanitize=address,undefined", "-fno-sanitize-recover=undefined", "-fno-omit-frame-pointer", "-g"]


def _sanitized() -> bool:
    return os.environ.get("ZC_SANITIZE") == "1"
_lock = threading.Lock()
_lib = None

TILE = 4096
HEADER = 128
TILE_BYTES = 5632

# status codes of zc_oracle.c
OK, ERR_ARG, ERR_CODEBOOK, ERR_ESCAPE_OVERFLOW, ERR_HEADER, ERR_CORRUPT, ERR_SIZE = range(7)


class OracleError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"oracle {what} failed with status {code}")
        self.code = code


def build(force: bool = False, sanitize: bool | None = None) -> str:
    """Compile zc_oracle.c into liboracle.so (plain C11, no fast-math, no FMA contraction).

    sanitize (default: ZC_SANITIZE=1 in the environment) builds liboracle_san.so
    instead, the same sources under AddressSanitizer and UndefinedBehaviorSanitizer."""
    san = _sanitized() if sanitize is None else sanitize
    lib = _SAN_LIB if san else _LIB
    with _lock:
        newest = max(os.path.getmtime(_SRC), os.path.getmtime(_QSRC))
        if force or not os.path.exists(lib) or os.path.getmtime(lib) < newest:
            tmp = lib + f".tmp{os.getpid()}"
            subprocess.check_call([
                "gcc", "-std=c11", "-O1" if san else "-O2", "-fPIC", "-shared", "-ffp-contract=off",
                "-fno-fast-math", "-Wall", "-Wextra"] + (_SAN_FLAGS if san else []) + [
                "-o", tmp, _SRC, _QSRC, "-lm",
            ])
            os.replace(tmp, lib)
    return lib


def _load():
    global _lib
    if _lib is not None:
        return _lib
    lib = ctypes.CDLL(build())
    u8p = ctypes.POINTER(ctypes.c_uint8)
    u16p = ctypes.POINTER(ctypes.c_uint16)
    u64p = ctypes.POINTER(ctypes.c_uint64)
    dp = ctypes.POINTER(ctypes.c_double)
    lib.zo_num_tiles.argtypes = [ctypes.c_uint64]
    lib.zo_num_tiles.restype = ctypes.c_uint64
    lib.zo_main_bytes.argtypes = [ctypes.c_uint64]
    lib.zo_main_bytes.restype = ctypes.c_uint64
    lib.zo_exponent_probability.argtypes = [ctypes.c_int, ctypes.c_double]
    lib.zo_exponent_probability.restype = ctypes.c_double
    lib.zo_codebook_from_sigma.argtypes = [ctypes.c_double, u8p, dp]
    lib.zo_codebook_from_sigma.restype = ctypes.c_int
    lib.zo_exponent_histogram.argtypes = [u16p, ctypes.c_uint64, u64p]
    lib.zo_exponent_histogram.restype = None
    lib.zo_topk_from_histogram.argtypes = [u64p, u8p]
    lib.zo_topk_from_histogram.restype = None
    lib.zo_compress.argtypes = [u16p, ctypes.c_uint64, u8p, u8p, u8p, ctypes.c_uint64, u64p]
    lib.zo_compress.restype = ctypes.c_int
    lib.zo_raw_spill.argtypes = [ctypes.c_uint64]
    lib.zo_raw_spill.restype = ctypes.c_uint64
    lib.zo_compress_adaptive.argtypes = [u16p, ctypes.c_uint64, u8p, u8p, u8p, ctypes.c_uint64, u64p,
                                         ctypes.POINTER(ctypes.c_int)]
    lib.zo_compress_adaptive.restype = ctypes.c_int
    lib.zo_decompress.argtypes = [u8p, u8p, ctypes.c_uint64, ctypes.c_uint64, u16p]
    lib.zqo_table_is_valid.argtypes = [u8p, u8p]
    lib.zqo_table_is_valid.restype = ctypes.c_int
    lib.zqo_table_from_histogram.argtypes = [u64p, u8p]
    lib.zqo_table_from_histogram.restype = None
    lib.zqo_code_length.argtypes = [u8p, u8p, ctypes.c_uint]
    lib.zqo_code_length.restype = ctypes.c_int
    lib.zqo_max_bytes.argtypes = [ctypes.c_uint64]
    lib.zqo_max_bytes.restype = ctypes.c_uint64
    lib.zqo_compress.argtypes = [u8p, ctypes.c_uint64, u8p, u8p, u8p, ctypes.c_uint64, u64p]
    lib.zqo_compress.restype = ctypes.c_int
    lib.zqo_decompress.argtypes = [u8p, ctypes.c_uint64, ctypes.c_uint64, u8p]
    lib.zqo_decompress.restype = ctypes.c_int
    lib.zo_decompress.restype = ctypes.c_int
    lib.zo_float_to_bf16_rne.argtypes = [ctypes.c_float]
    lib.zo_float_to_bf16_rne.restype = ctypes.c_uint16
    lib.zo_reduce.argtypes = [ctypes.c_int, ctypes.POINTER(u16p), ctypes.c_uint64, u16p]
    lib.zo_reduce.restype = None
    lib.zo_decompress_reduce.argtypes = [
        ctypes.c_int, ctypes.POINTER(u8p), ctypes.POINTER(u8p), u64p, ctypes.c_uint64, u16p,
        u8p, u8p, u8p, ctypes.c_uint64, u64p,
    ]
    lib.zo_decompress_reduce.restype = ctypes.c_int
    _lib = lib
    return lib


def _ptr(a: np.ndarray, ctype):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _u16(x) -> np.ndarray:
    x = np.ascontiguousarray(x)
    if x.dtype != np.uint16:
        x = x.view(np.uint16)
    return x.reshape(-1)


def _cb(cb) -> np.ndarray:
    a = np.ascontiguousarray(np.asarray(cb, dtype=np.uint8).reshape(-1))
    if a.size != 7:
        raise ValueError("codebook must have 7 entries")
    return a


# ---------------------------------------------------------------- sizes
def num_tiles(n: int) -> int:
    return int(_load().zo_num_tiles(n))


def main_bytes(n: int) -> int:
    return int(_load().zo_main_bytes(n))


# ---------------------------------------------------------------- codebooks
def exponent_probability(e: int, sigma: float) -> float:
    return float(_load().zo_exponent_probability(int(e), float(sigma)))


def codebook_from_sigma(sigma: float, return_probs: bool = False):
    cb = np.zeros(7, np.uint8)
    probs = np.zeros(256, np.float64)
    rc = _load().zo_codebook_from_sigma(float(sigma), _ptr(cb, ctypes.c_uint8), _ptr(probs, ctypes.c_double))
    if rc != OK:
        raise OracleError(rc, "codebook_from_sigma")
    return (cb, probs) if return_probs else cb


def exponent_histogram(x) -> np.ndarray:
    x = _u16(x)
    h = np.zeros(256, np.uint64)
    _load().zo_exponent_histogram(_ptr(x, ctypes.c_uint16), x.size, _ptr(h, ctypes.c_uint64))
    return h


def topk_from_histogram(hist) -> np.ndarray:
    h = np.ascontiguousarray(np.asarray(hist, dtype=np.uint64))
    cb = np.zeros(7, np.uint8)
    _load().zo_topk_from_histogram(_ptr(h, ctypes.c_uint64), _ptr(cb, ctypes.c_uint8))
    return cb


def histogram_topk(x):
    h = exponent_histogram(x)
    return topk_from_histogram(h), h


# ---------------------------------------------------------------- codec
def compress(x, cb, esc_capacity: int | None = None, allow_overflow: bool = False):
    """Return (main_stream uint8[main_bytes(n)], escapes uint8[n_esc])."""
    x = _u16(x)
    cb = _cb(cb)
    n = x.size
    cap = n if esc_capacity is None else int(esc_capacity)
    main = np.zeros(main_bytes(n), np.uint8)
    esc = np.zeros(max(cap, 1), np.uint8)
    n_esc = ctypes.c_uint64(0)
    rc = _load().zo_compress(_ptr(x, ctypes.c_uint16), n, _ptr(cb, ctypes.c_uint8), _ptr(main, ctypes.c_uint8),
                             _ptr(esc, ctypes.c_uint8), cap, ctypes.byref(n_esc))
    if rc == ERR_ESCAPE_OVERFLOW and allow_overflow:
        return main, esc[:min(cap, n_esc.value)].copy(), rc
    if rc != OK:
        raise OracleError(rc, "compress")
    return main, esc[: n_esc.value].copy()


def raw_spill(n: int) -> int:
    """Bytes of a RAW stream of n values that go to the escape stream (reading R12)."""
    return int(_load().zo_raw_spill(n))


def compress_adaptive(x, cb, esc_capacity: int | None = None, allow_overflow: bool = False):
    """Encode, then store RAW when that is strictly smaller (reading R12).

    Returns (main, escapes, raw) with raw = True for a RAW stream, or
    (main, escapes, raw, rc) with ``allow_overflow`` when neither form fits.
    """
    x = _u16(x)
    cb = _cb(cb)
    n = x.size
    cap = n if esc_capacity is None else int(esc_capacity)
    main = np.zeros(main_bytes(n), np.uint8)
    esc = np.zeros(max(cap, 1), np.uint8)
    n_esc = ctypes.c_uint64(0)
    raw = ctypes.c_int(0)
    rc = _load().zo_compress_adaptive(_ptr(x, ctypes.c_uint16), n, _ptr(cb, ctypes.c_uint8),
                                      _ptr(main, ctypes.c_uint8), _ptr(esc, ctypes.c_uint8), cap,
                                      ctypes.byref(n_esc), ctypes.byref(raw))
    if rc == ERR_ESCAPE_OVERFLOW and allow_overflow:
        return main, esc[:min(cap, n_esc.value)].copy(), bool(raw.value), rc
    if rc != OK:
        raise OracleError(rc, "compress_adaptive")
    return main, esc[: n_esc.value].copy(), bool(raw.value)


def decompress_status(main, esc, n: int):
    main = np.ascontiguousarray(main, dtype=np.uint8)
    esc_arr = np.ascontiguousarray(esc, dtype=np.uint8)
    esc_buf = esc_arr if esc_arr.size else np.zeros(1, np.uint8)
    out = np.zeros(max(n, 1), np.uint16)
    rc = _load().zo_decompress(_ptr(main, ctypes.c_uint8), _ptr(esc_buf, ctypes.c_uint8), esc_arr.size, n,
                               _ptr(out, ctypes.c_uint16))
    return rc, out[:n]


def decompress(main, esc, n: int) -> np.ndarray:
    rc, out = decompress_status(main, esc, n)
    if rc != OK:
        raise OracleError(rc, "decompress")
    return out


def float_to_bf16_rne(f: float) -> int:
    return int(_load().zo_float_to_bf16_rne(ctypes.c_float(f)))


def reduce(xs) -> np.ndarray:
    arrs = [_u16(a) for a in xs]
    n = arrs[0].size
    assert all(a.size == n for a in arrs)
    ptrs = (ctypes.POINTER(ctypes.c_uint16) * len(arrs))(*[_ptr(a, ctypes.c_uint16) for a in arrs])
    y = np.zeros(max(n, 1), np.uint16)
    _load().zo_reduce(len(arrs), ptrs, n, _ptr(y, ctypes.c_uint16))
    return y[:n]


def decompress_reduce(mains, escs, n: int, out_cb=None):
    """Decode P shards, sum in fp32 in rank order, round to bf16, optionally re-encode.

    Returns y (uint16[n]) or (y, main, esc) when ``out_cb`` is given.
    """
    P = len(mains)
    mains = [np.ascontiguousarray(m, dtype=np.uint8) for m in mains]
    escs_a = [np.ascontiguousarray(e, dtype=np.uint8) for e in escs]
    esc_bufs = [e if e.size else np.zeros(1, np.uint8) for e in escs_a]
    u8p = ctypes.POINTER(ctypes.c_uint8)
    mp = (u8p * P)(*[_ptr(m, ctypes.c_uint8) for m in mains])
    ep = (u8p * P)(*[_ptr(e, ctypes.c_uint8) for e in esc_bufs])
    eb = np.array([e.size for e in escs_a], np.uint64)
    y = np.zeros(max(n, 1), np.uint16)
    n_esc = ctypes.c_uint64(0)
    if out_cb is not None:
        cb = _cb(out_cb)
        om = np.zeros(main_bytes(n), np.uint8)
        oe = np.zeros(max(n, 1), np.uint8)
        rc = _load().zo_decompress_reduce(P, mp, ep, _ptr(eb, ctypes.c_uint64), n, _ptr(y, ctypes.c_uint16),
                                          _ptr(cb, ctypes.c_uint8), _ptr(om, ctypes.c_uint8),
                                          _ptr(oe, ctypes.c_uint8), n, ctypes.byref(n_esc))
        if rc != OK:
            raise OracleError(rc, "decompress_reduce")
        return y[:n], om, oe[: n_esc.value].copy()
    rc = _load().zo_decompress_reduce(P, mp, ep, _ptr(eb, ctypes.c_uint64), n, _ptr(y, ctypes.c_uint16),
                                      None, None, None, 0, ctypes.byref(n_esc))
    if rc != OK:
        raise OracleError(rc, "decompress_reduce")
    return y[:n]


def header_fields(main) -> dict:
    m = np.ascontiguousarray(main, dtype=np.uint8)
    b = m[:40].tobytes()
    return {
        "magic": int.from_bytes(b[0:4], "little"),
        "version": int.from_bytes(b[4:6], "little"),
        "flags": int.from_bytes(b[6:8], "little"),
        "n": int.from_bytes(b[8:16], "little"),
        "tile_elems": int.from_bytes(b[16:20], "little"),
        "ntiles": int.from_bytes(b[20:24], "little"),
        "n_esc": int.from_bytes(b[24:32], "little"),
        "codebook": list(b[32:39]),
    }


# ---------------------------------------------------------------- QLC (FP8 e4m3), qlc_oracle.c
QLC_DEFAULT_WIDTHS = (3, 3, 3, 3, 3, 4, 5, 8)  # reading Q2: code lengths 6/7/8/11
Q_OK, Q_ERR_ARG, Q_ERR_TABLE, Q_ERR_HEADER, Q_ERR_CORRUPT, Q_ERR_SIZE, Q_ERR_ROOM = range(7)


def _u8(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.uint8))


def qlc_table_from_histogram(hist) -> np.ndarray:
    """rank -> symbol, ordered by (count desc, symbol asc) (reading Q2)."""
    h = np.ascontiguousarray(np.asarray(hist, dtype=np.uint64).reshape(256))
    sym = np.zeros(256, np.uint8)
    _load().zqo_table_from_histogram(_ptr(h, ctypes.c_uint64), _ptr(sym, ctypes.c_uint8))
    return sym


def qlc_table_for(x) -> np.ndarray:
    return qlc_table_from_histogram(np.bincount(_u8(x), minlength=256))


def qlc_table_is_valid(widths, sym) -> bool:
    w, s = _u8(widths), _u8(sym)
    return bool(_load().zqo_table_is_valid(_ptr(w, ctypes.c_uint8), _ptr(s, ctypes.c_uint8)))


def qlc_code_length(widths, sym, symbol: int) -> int:
    w, s = _u8(widths), _u8(sym)
    return int(_load().zqo_code_length(_ptr(w, ctypes.c_uint8), _ptr(s, ctypes.c_uint8), int(symbol)))


def qlc_max_bytes(n: int) -> int:
    return int(_load().zqo_max_bytes(n))


def qlc_compress(x, widths, sym) -> np.ndarray:
    """Encode bytes x into a ZQ1 stream (reading Q3); returns the stream bytes."""
    x, w, s = _u8(x), _u8(widths), _u8(sym)
    cap = qlc_max_bytes(x.size)
    out = np.zeros(cap, np.uint8)
    nbytes = ctypes.c_uint64(0)
    xb = x if x.size else np.zeros(1, np.uint8)
    rc = _load().zqo_compress(_ptr(xb, ctypes.c_uint8), x.size, _ptr(w, ctypes.c_uint8), _ptr(s, ctypes.c_uint8),
                              _ptr(out, ctypes.c_uint8), cap, ctypes.byref(nbytes))
    if rc != Q_OK:
        raise OracleError(rc, "qlc_compress")
    return out[: nbytes.value].copy()


def qlc_decompress_status(stream, n: int):
    st = _u8(stream)
    sb = st if st.size else np.zeros(1, np.uint8)
    out = np.zeros(max(n, 1), np.uint8)
    rc = _load().zqo_decompress(_ptr(sb, ctypes.c_uint8), st.size, n, _ptr(out, ctypes.c_uint8))
    return rc, out[:n]


def qlc_decompress(stream, n: int) -> np.ndarray:
    rc, out = qlc_decompress_status(stream, n)
    if rc != Q_OK:
        raise OracleError(rc, "qlc_decompress")
    return out
