"""Thin Python binding of libzc (the C ABI in include/zc.h).

Argument marshalling only: every step runs in libzc's CUDA kernels on the
caller's current torch stream.  Tensors are passed as raw device pointers;
bfloat16 data may be given as ``torch.bfloat16``, ``torch.int16`` or
``torch.uint16`` tensors (the bits are what matters).  There is no CPU path:
if libzc cannot be loaded, every call raises.
"""
from __future__ import annotations

import ctypes
import functools
import os
from dataclasses import dataclass
from typing import Sequence

import numpy as np
import torch

from . import _build

TILE = 4096
HEADER_BYTES = 128
WORKSPACE_HEADER_BYTES = 4096
WORKSPACE_BYTES_PER_TILE = 16
MAX_SHARDS = 64

STATUS_NAMES = [
    "ZC_OK", "ZC_ERR_INVALID_ARG", "ZC_ERR_ALIGNMENT", "ZC_ERR_TOO_LARGE", "ZC_ERR_WORKSPACE",
    "ZC_ERR_CODEBOOK", "ZC_ERR_CUDA", "ZC_ERR_ESCAPE_OVERFLOW", "ZC_ERR_BAD_HEADER",
    "ZC_ERR_CORRUPT_STREAM", "ZC_ERR_SIZE_MISMATCH", "ZC_ERR_TIMEOUT", "ZC_ERR_DUP_CODEBOOK",
    "ZC_ERR_OUT_OF_ROOM",
]
for _i, _name in enumerate(STATUS_NAMES):
    globals()[_name[3:]] = _i   # OK, ERR_INVALID_ARG, ...


class ZcError(RuntimeError):
    def __init__(self, code: int, where: str):
        super().__init__(f"{where}: {status_string(code)} ({code})")
        self.code = code


class ZqTable(ctypes.Structure):
    _fields_ = [("width", ctypes.c_uint8 * 8), ("sym", ctypes.c_uint8 * 256)]


class LinkModel(ctypes.Structure):
    _fields_ = [("bandwidth_gbps", ctypes.c_double), ("latency_us", ctypes.c_double)]


class CodecModel(ctypes.Structure):
    _fields_ = [("compress_gbps", ctypes.c_double), ("decompress_gbps", ctypes.c_double), ("ratio", ctypes.c_double)]


class ZcTensor(ctypes.Structure):
    _fields_ = [("bf16", ctypes.c_void_p), ("main", ctypes.c_void_p), ("esc", ctypes.c_void_p),
                ("cb", ctypes.c_void_p), ("n", ctypes.c_uint64), ("esc_bytes", ctypes.c_uint64)]


_lib = None


def _sanitized() -> bool:
    """ZC_SANITIZE=1 selects the ASan/UBSan build of the host code (CPU-side checks only)."""
    return os.environ.get("ZC_SANITIZE") == "1"


def library_path() -> str:
    return _build.SAN_LIB if _sanitized() else _build.LIB


def load() -> ctypes.CDLL:
    """Load libzc.so (building it in-tree first if it is missing or stale)."""
    global _lib
    if _lib is not None:
        return _lib
    path = _build.build(sanitize=_sanitized())
    if not os.path.exists(path):
        raise RuntimeError(f"libzc not found at {path}")
    lib = ctypes.CDLL(path)
    vp, u64, i32 = ctypes.c_void_p, ctypes.c_uint64, ctypes.c_int
    u64p = ctypes.POINTER(ctypes.c_uint64)
    lib.zc_status_string.argtypes = [i32]
    lib.zc_status_string.restype = ctypes.c_char_p
    lib.zc_version.argtypes = []
    lib.zc_version.restype = ctypes.c_char_p
    lib.zc_codebook_from_sigma.argtypes = [ctypes.c_double, ctypes.POINTER(ctypes.c_uint8)]
    lib.zc_compressed_size.argtypes = [u64, u64p, u64p]
    lib.zc_workspace_size.argtypes = [u64p, i32, u64p]
    lib.zc_histogram_topk.argtypes = [vp, u64, vp, vp, vp, u64, vp, vp]
    lib.zc_compress.argtypes = [vp, u64, vp, vp, vp, u64, vp, u64, vp, vp]
    lib.zc_compress_adaptive.argtypes = [vp, u64, vp, vp, vp, u64, vp, u64, vp, vp]
    lib.zc_raw_spill.argtypes = [u64, u64p]
    lib.zc_decompress.argtypes = [vp, vp, u64, u64, vp, vp, vp]
    lib.zc_decompress_reduce.argtypes = [i32, ctypes.POINTER(vp), ctypes.POINTER(vp), u64p, u64, vp, vp, vp, vp,
                                         u64, vp, u64, vp, vp]
    lib.zc_compress_batched.argtypes = [i32, ctypes.POINTER(ZcTensor), vp, u64, vp, vp]
    lib.zc_compress_batched_adaptive.argtypes = [i32, ctypes.POINTER(ZcTensor), vp, u64, vp, vp]
    lib.zc_decompress_batched.argtypes = [i32, ctypes.POINTER(ZcTensor), vp, vp]
    lib.zq_default_widths.argtypes = [ctypes.POINTER(ctypes.c_uint8)]
    lib.zq_table_from_histogram.argtypes = [u64p, ctypes.POINTER(ctypes.c_uint8), ctypes.POINTER(ZqTable)]
    lib.zq_max_bytes.argtypes = [u64, u64p]
    lib.zq_compress.argtypes = [vp, u64, ctypes.POINTER(ZqTable), vp, u64, vp, u64, vp, vp]
    lib.zq_decompress.argtypes = [vp, u64, u64, vp, vp, vp]
    dp = ctypes.POINTER(ctypes.c_double)
    lib.zc_transfer_pays.argtypes = [u64, ctypes.POINTER(LinkModel), ctypes.POINTER(CodecModel),
                                     ctypes.POINTER(i32), dp, dp]
    lib.zc_reduce_scatter_choose.argtypes = [u64, i32, ctypes.POINTER(LinkModel), ctypes.POINTER(CodecModel),
                                             ctypes.POINTER(i32), dp, dp]
    lib.zc_pipeline_workspace_size.argtypes = [u64, u64p]
    lib.zc_pipelined_transfer.argtypes = [vp, u64, vp, vp, u64, vp, u64, vp, vp, vp, vp]
    lib.zc_pipeline_plan_create.argtypes = [vp, u64, vp, vp, u64, vp, u64, vp, i32, ctypes.POINTER(vp)]
    lib.zc_pipeline_plan_launch.argtypes = [vp, vp]
    lib.zc_pipeline_plan_destroy.argtypes = [vp]
    for name in ("zc_codebook_from_sigma", "zc_compressed_size", "zc_workspace_size", "zc_histogram_topk",
                 "zc_compress", "zc_compress_adaptive", "zc_raw_spill", "zc_decompress", "zc_decompress_reduce",
                 "zc_compress_batched", "zc_compress_batched_adaptive", "zc_decompress_batched",
                 "zc_pipeline_workspace_size", "zc_pipelined_transfer", "zc_pipeline_plan_create",
                 "zc_pipeline_plan_launch", "zc_pipeline_plan_destroy", "zq_default_widths",
                 "zq_table_from_histogram", "zq_max_bytes", "zq_compress", "zq_decompress", "zc_transfer_pays",
                 "zc_reduce_scatter_choose"):
        getattr(lib, name).restype = i32
    _lib = lib
    return lib


def status_string(code: int) -> str:
    return load().zc_status_string(int(code)).decode()


def version() -> str:
    return load().zc_version().decode()


def _check(code: int, where: str) -> None:
    if code != OK:  # noqa: F821 - defined from STATUS_NAMES
        raise ZcError(code, where)


def _ptr(t: torch.Tensor | None) -> int | None:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("libzc takes CUDA tensors")
    if not t.is_contiguous():
        raise ValueError("libzc takes contiguous tensors")
    return t.data_ptr()


def _current_raw_stream(device_index: int) -> int:
    """The current stream's cudaStream_t on a device (torch's raw query: no Stream object is built)."""
    raw = getattr(torch._C, "_cuda_getCurrentRawStream", None)
    if raw is not None:
        return raw(device_index)
    return torch.cuda.current_stream(device_index).cuda_stream


def _stream(stream: torch.cuda.Stream | None = None, like: torch.Tensor | None = None) -> int:
    """The cudaStream_t to launch on: the given stream, else the current stream of `like`'s device."""
    if stream is not None:
        return stream.cuda_stream
    index = like.device.index if like is not None and like.device.index is not None else torch.cuda.current_device()
    return _current_raw_stream(index)


def _nelem16(x: torch.Tensor) -> int:
    if x.element_size() != 2:
        raise ValueError("bfloat16 data must be a 2-byte dtype (bfloat16, int16 or uint16)")
    return x.numel()


# ------------------------------------------------------------------ host-side pure functions
def codebook_from_sigma(sigma: float) -> np.ndarray:
    cb = (ctypes.c_uint8 * 7)()
    _check(load().zc_codebook_from_sigma(float(sigma), cb), "zc_codebook_from_sigma")
    return np.frombuffer(bytes(cb), np.uint8).copy()


@functools.lru_cache(maxsize=4096)
def compressed_size(n: int) -> tuple[int, int]:
    m, e = ctypes.c_uint64(), ctypes.c_uint64()
    _check(load().zc_compressed_size(int(n), ctypes.byref(m), ctypes.byref(e)), "zc_compressed_size")
    return m.value, e.value


def raw_spill(n: int) -> int:
    """Escape bytes of a RAW stream of n values (the most an adaptive compression needs)."""
    out = ctypes.c_uint64()
    _check(load().zc_raw_spill(int(n), ctypes.byref(out)), "zc_raw_spill")
    return out.value


def workspace_size(ns: Sequence[int] | int) -> int:
    ns = [int(ns)] if isinstance(ns, (int, np.integer)) else [int(v) for v in ns]
    arr = (ctypes.c_uint64 * len(ns))(*ns)
    out = ctypes.c_uint64()
    _check(load().zc_workspace_size(arr, len(ns), ctypes.byref(out)), "zc_workspace_size")
    return out.value


def workspace(ns: Sequence[int] | int, device="cuda") -> torch.Tensor:
    """A zero-filled workspace (zero it again only after a call reported a device error)."""
    return torch.zeros(workspace_size(ns), dtype=torch.uint8, device=device)


def new_status(device="cuda") -> torch.Tensor:
    return torch.zeros(1, dtype=torch.int32, device=device)


def codebook_to_device(cb, device="cuda") -> torch.Tensor:
    return torch.as_tensor(np.asarray(cb, np.uint8).reshape(7), dtype=torch.uint8).to(device)


# ------------------------------------------------------------------ device entry points
def histogram_topk(x: torch.Tensor, ws: torch.Tensor, status: torch.Tensor, cb_out: torch.Tensor | None = None,
                   hist_out: torch.Tensor | None = None, stream=None):
    """Exact exponent histogram -> device codebook (7 x uint8) [+ 256 x int32 counts]."""
    n = _nelem16(x)
    if cb_out is None:
        cb_out = torch.empty(7, dtype=torch.uint8, device=x.device)
    rc = load().zc_histogram_topk(_ptr(x), n, _ptr(cb_out), _ptr(hist_out), _ptr(ws), ws.numel(), _ptr(status),
                                  _stream(stream, status))
    _check(rc, "zc_histogram_topk")
    return cb_out, hist_out


def compress(x: torch.Tensor, cb: torch.Tensor, ws: torch.Tensor, status: torch.Tensor,
             main: torch.Tensor | None = None, esc: torch.Tensor | None = None, stream=None):
    """Encode x into (main stream, escape buffer); the escape count is in the main header."""
    n = _nelem16(x)
    mb, eb = compressed_size(n)
    if main is None:
        main = torch.empty(mb, dtype=torch.uint8, device=x.device)
    if esc is None:
        esc = torch.empty(max(eb, 16), dtype=torch.uint8, device=x.device)
    rc = load().zc_compress(_ptr(x), n, _ptr(cb), _ptr(main), _ptr(esc), esc.numel(), _ptr(ws), ws.numel(),
                            _ptr(status), _stream(stream, status))
    _check(rc, "zc_compress")
    return main, esc


def compress_adaptive(x: torch.Tensor, cb: torch.Tensor, ws: torch.Tensor, status: torch.Tensor,
                      main: torch.Tensor | None = None, esc: torch.Tensor | None = None, stream=None):
    """compress with the raw bypass: the stream is stored RAW (header flags bit 0) when that is smaller.

    The default escape buffer is raw_spill(n) bytes, which never overflows.
    """
    n = _nelem16(x)
    mb, _ = compressed_size(n)
    if main is None:
        main = torch.empty(mb, dtype=torch.uint8, device=x.device)
    if esc is None:
        esc = torch.empty(max(raw_spill(n), 16), dtype=torch.uint8, device=x.device)
    rc = load().zc_compress_adaptive(_ptr(x), n, _ptr(cb), _ptr(main), _ptr(esc), esc.numel(), _ptr(ws),
                                     ws.numel(), _ptr(status), _stream(stream, status))
    _check(rc, "zc_compress_adaptive")
    return main, esc


def decompress(main: torch.Tensor, esc: torch.Tensor, n: int, status: torch.Tensor,
               out: torch.Tensor | None = None, esc_bytes: int | None = None, stream=None) -> torch.Tensor:
    if out is None:
        out = torch.empty(n, dtype=torch.int16, device=main.device)
    eb = esc.numel() if esc_bytes is None else int(esc_bytes)
    rc = load().zc_decompress(_ptr(main), _ptr(esc) if esc is not None else None, eb, int(n), _ptr(out),
                              _ptr(status), _stream(stream, status))
    _check(rc, "zc_decompress")
    return out


def decompress_reduce(mains: Sequence[torch.Tensor], escs: Sequence[torch.Tensor], n: int, status: torch.Tensor,
                      out: torch.Tensor | None = None, out_cb: torch.Tensor | None = None,
                      out_main: torch.Tensor | None = None, out_esc: torch.Tensor | None = None,
                      ws: torch.Tensor | None = None, want_out: bool = True, esc_bytes: Sequence[int] | None = None,
                      stream=None):
    P = len(mains)
    dev = mains[0].device
    if out is None and want_out:
        out = torch.empty(n, dtype=torch.int16, device=dev)
    if out_cb is not None:
        mb, eb = compressed_size(n)
        if out_main is None:
            out_main = torch.empty(mb, dtype=torch.uint8, device=dev)
        if out_esc is None:
            out_esc = torch.empty(max(eb, 16), dtype=torch.uint8, device=dev)
    mp = (ctypes.c_void_p * P)(*[_ptr(m) for m in mains])
    ep = (ctypes.c_void_p * P)(*[_ptr(e) for e in escs])
    sizes = [e.numel() for e in escs] if esc_bytes is None else list(esc_bytes)
    eb_arr = (ctypes.c_uint64 * P)(*sizes)
    rc = load().zc_decompress_reduce(P, mp, ep, eb_arr, int(n), _ptr(out), _ptr(out_cb), _ptr(out_main),
                                     _ptr(out_esc), out_esc.numel() if out_esc is not None else 0,
                                     _ptr(ws), ws.numel() if ws is not None else 0, _ptr(status), _stream(stream, status))
    _check(rc, "zc_decompress_reduce")
    return out, out_main, out_esc


@dataclass
class BatchItem:
    bf16: torch.Tensor
    main: torch.Tensor
    esc: torch.Tensor
    cb: torch.Tensor | None = None
    esc_bytes: int | None = None


def _descs(items: Sequence[BatchItem]):
    arr = (ZcTensor * len(items))()
    for i, it in enumerate(items):
        arr[i].bf16 = _ptr(it.bf16)
        arr[i].main = _ptr(it.main)
        arr[i].esc = _ptr(it.esc)
        arr[i].cb = _ptr(it.cb)
        arr[i].n = it.bf16.numel()
        arr[i].esc_bytes = it.esc.numel() if it.esc_bytes is None else int(it.esc_bytes)
    return arr


def compress_batched(items: Sequence[BatchItem], ws: torch.Tensor, status: torch.Tensor, stream=None) -> None:
    arr = _descs(items)
    _check(load().zc_compress_batched(len(items), arr, _ptr(ws), ws.numel(), _ptr(status), _stream(stream, status)),
           "zc_compress_batched")


def compress_batched_adaptive(items: Sequence[BatchItem], ws: torch.Tensor, status: torch.Tensor,
                              stream=None) -> None:
    arr = _descs(items)
    _check(load().zc_compress_batched_adaptive(len(items), arr, _ptr(ws), ws.numel(), _ptr(status),
                                               _stream(stream, status)), "zc_compress_batched_adaptive")


def decompress_batched(items: Sequence[BatchItem], status: torch.Tensor, stream=None) -> None:
    arr = _descs(items)
    _check(load().zc_decompress_batched(len(items), arr, _ptr(status), _stream(stream, status)), "zc_decompress_batched")


def transfer_pays(nbytes: int, bandwidth_gbps: float, latency_us: float, compress_gbps: float,
                  decompress_gbps: float, ratio: float) -> tuple[bool, float, float]:
    """(compress?, t_raw_us, t_zipped_us) for one message (zc_transfer_pays)."""
    link, codec = LinkModel(bandwidth_gbps, latency_us), CodecModel(compress_gbps, decompress_gbps, ratio)
    pays, tr, tz = ctypes.c_int(), ctypes.c_double(), ctypes.c_double()
    _check(load().zc_transfer_pays(int(nbytes), ctypes.byref(link), ctypes.byref(codec), ctypes.byref(pays),
                                   ctypes.byref(tr), ctypes.byref(tz)), "zc_transfer_pays")
    return bool(pays.value), tr.value, tz.value


def reduce_scatter_choose(nbytes: int, P: int, bandwidth_gbps: float, latency_us: float, compress_gbps: float,
                          decompress_gbps: float, ratio: float) -> tuple[bool, float, float]:
    """(zipped?, t_native_us, t_zipped_us) for a reduce-scatter of nbytes per rank over P ranks."""
    link, codec = LinkModel(bandwidth_gbps, latency_us), CodecModel(compress_gbps, decompress_gbps, ratio)
    z, tn, tz = ctypes.c_int(), ctypes.c_double(), ctypes.c_double()
    _check(load().zc_reduce_scatter_choose(int(nbytes), int(P), ctypes.byref(link), ctypes.byref(codec),
                                           ctypes.byref(z), ctypes.byref(tn), ctypes.byref(tz)),
           "zc_reduce_scatter_choose")
    return bool(z.value), tn.value, tz.value


def pipeline_workspace_size(chunk_elems: int) -> int:
    out = ctypes.c_uint64()
    _check(load().zc_pipeline_workspace_size(int(chunk_elems), ctypes.byref(out)), "zc_pipeline_workspace_size")
    return out.value


def pipeline_workspace(chunk_elems: int, device="cuda") -> torch.Tensor:
    """A zero-filled pipeline workspace (256-byte aligned, as the caching allocator returns)."""
    return torch.zeros(pipeline_workspace_size(chunk_elems), dtype=torch.uint8, device=device)


def pipelined_transfer(x: torch.Tensor, cb: torch.Tensor, chunk_elems: int, ws: torch.Tensor, status: torch.Tensor,
                       out: torch.Tensor | None = None, streams=None) -> torch.Tensor:
    """Zipped transfer of x into out through the compress / link / decompress pipeline.

    streams: (compress, link, decompress) torch streams; default: the current
    stream and two new ones.  out is ready once the current (compress) stream
    reaches this point.
    """
    n = _nelem16(x)
    if out is None:
        out = torch.empty(n, dtype=torch.int16, device=x.device)
    if streams is None:
        cur = torch.cuda.current_stream()
        streams = (cur, torch.cuda.Stream(device=x.device), torch.cuda.Stream(device=x.device))
    sc, sl, sd = (s.cuda_stream for s in streams)
    rc = load().zc_pipelined_transfer(_ptr(x), n, _ptr(cb), _ptr(out), int(chunk_elems), _ptr(ws), ws.numel(),
                                      _ptr(status), sc, sl, sd)
    _check(rc, "zc_pipelined_transfer")
    return out


class PipelinePlan:
    """zc_pipelined_transfer's launch sequence captured once into a CUDA graph; launch() replays it.

    The plan keeps the tensors it was made with alive: each launch reads x, cb and ws as they are when it runs
    (refill x in place for new data) and writes out and status.  Launches that share ws must be ordered."""

    def __init__(self, x: torch.Tensor, cb: torch.Tensor, chunk_elems: int, ws: torch.Tensor,
                 status: torch.Tensor, out: torch.Tensor | None = None, overlap: bool = True):
        n = _nelem16(x)
        if out is None:
            out = torch.empty(n, dtype=torch.int16, device=x.device)
        self.x, self.cb, self.ws, self.status, self.out = x, cb, ws, status, out
        self._plan = ctypes.c_void_p()
        with torch.cuda.device(x.device):
            rc = load().zc_pipeline_plan_create(_ptr(x), n, _ptr(cb), _ptr(out), int(chunk_elems), _ptr(ws),
                                                ws.numel(), _ptr(status), int(bool(overlap)),
                                                ctypes.byref(self._plan))
        _check(rc, "zc_pipeline_plan_create")

    def launch(self, stream=None) -> torch.Tensor:
        """Replays the pipeline on `stream` (default: the current stream of the plan's device, which must be the
        current device); returns out."""
        if self._plan is None:
            raise RuntimeError("the plan was closed")
        _check(load().zc_pipeline_plan_launch(self._plan, _stream(stream, self.status)), "zc_pipeline_plan_launch")
        return self.out

    def close(self) -> None:
        if self._plan is not None:
            _check(load().zc_pipeline_plan_destroy(self._plan), "zc_pipeline_plan_destroy")
            self._plan = None

    def __del__(self):
        try:
            self.close()
        except Exception:  # interpreter shutdown: nothing left to release into
            pass


def pipeline_plan(x: torch.Tensor, cb: torch.Tensor, chunk_elems: int, ws: torch.Tensor, status: torch.Tensor,
                  out: torch.Tensor | None = None, overlap: bool = True) -> PipelinePlan:
    return PipelinePlan(x, cb, chunk_elems, ws, status, out=out, overlap=overlap)


# ------------------------------------------------------------------ QLC for FP8 (e4m3) bytes
def zq_default_widths() -> np.ndarray:
    w = (ctypes.c_uint8 * 8)()
    _check(load().zq_default_widths(w), "zq_default_widths")
    return np.frombuffer(bytes(w), np.uint8).copy()


def zq_table_from_histogram(hist, widths=None) -> ZqTable:
    h = np.ascontiguousarray(np.asarray(hist, dtype=np.uint64).reshape(256))
    hp = h.ctypes.data_as(ctypes.POINTER(ctypes.c_uint64))
    wp = None
    if widths is not None:
        wp = (ctypes.c_uint8 * 8)(*[int(v) for v in widths])
    t = ZqTable()
    _check(load().zq_table_from_histogram(hp, wp, ctypes.byref(t)), "zq_table_from_histogram")
    return t


def zq_table(widths, sym) -> ZqTable:
    t = ZqTable()
    t.width[:] = [int(v) for v in widths]
    t.sym[:] = [int(v) for v in sym]
    return t


def zq_max_bytes(n: int) -> int:
    out = ctypes.c_uint64()
    _check(load().zq_max_bytes(int(n), ctypes.byref(out)), "zq_max_bytes")
    return out.value


def zq_compress(x: torch.Tensor, table: ZqTable, ws: torch.Tensor, status: torch.Tensor,
                out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """QLC-encode the bytes of x (uint8 / float8 tensor) into a ZQ1 stream buffer (zq_max_bytes(n) bytes)."""
    if x.element_size() != 1:
        raise ValueError("QLC codes 1-byte symbols (uint8 or float8 tensors)")
    n = x.numel()
    if out is None:
        out = torch.empty(zq_max_bytes(n), dtype=torch.uint8, device=x.device)
    rc = load().zq_compress(_ptr(x), n, ctypes.byref(table), _ptr(out), out.numel(), _ptr(ws), ws.numel(),
                            _ptr(status), _stream(stream, status))
    _check(rc, "zq_compress")
    return out


def zq_stream_bytes(stream_buf: torch.Tensor) -> int:
    """Bytes of the ZQ1 stream in stream_buf, from its header (a device-to-host read)."""
    h = stream_buf[:32].cpu().numpy()
    nblocks = int.from_bytes(h[20:24].tobytes(), "little")
    words = int.from_bytes(h[24:32].tobytes(), "little")
    return 384 + -(-4 * nblocks // 128) * 128 + 4 * words


def zq_decompress(stream_buf: torch.Tensor, n: int, status: torch.Tensor, out: torch.Tensor | None = None,
                  in_bytes: int | None = None, stream=None) -> torch.Tensor:
    if out is None:
        out = torch.empty(n, dtype=torch.uint8, device=stream_buf.device)
    nb = stream_buf.numel() if in_bytes is None else int(in_bytes)
    rc = load().zq_decompress(_ptr(stream_buf), nb, int(n), _ptr(out), _ptr(status), _stream(stream, status))
    _check(rc, "zq_decompress")
    return out


# ------------------------------------------------------------------ small host helpers
def header_n_esc(main: torch.Tensor) -> int:
    """Escape count from a main stream's header (a device-to-host read of 8 bytes)."""
    return int.from_bytes(main[24:32].cpu().numpy().tobytes(), "little")


def header_is_raw(main: torch.Tensor) -> bool:
    """Whether a main stream holds a RAW stream (header flags bit 0; a device-to-host read)."""
    return bool(int.from_bytes(main[6:8].cpu().numpy().tobytes(), "little") & 1)


def status_value(status: torch.Tensor) -> int:
    return int(status.item())
