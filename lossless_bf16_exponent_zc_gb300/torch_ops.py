"""PyTorch operators over libzc: ``torch.ops.zc.*``.

The codec as ordinary torch operators, so that training code and frameworks can
call it like any other op (the drop-in integration of [ZipCCL §3] and
[CCCL §4]) and graph tracers see it: each op has a fake implementation that
gives its outputs' shapes and dtypes without running it.  Every op calls the
C ABI through the binding in ``zc.py`` on the current stream; there is no CPU
path.

Ops (device tensors; bf16 data as bfloat16 / int16 / uint16):
  zc::compress(x, cb, ws, status, adaptive=False) -> (main, esc)
      main: zc_main_bytes(n) uint8; esc: the escape buffer (capacity n, or
      the RAW spill when adaptive); the escape count is in main's header.
  zc::decompress(main, esc, n, status) -> int16[n]
  zc::decompress_reduce(mains, escs, n, status) -> int16[n]
      the local stage of a zipped reduce-scatter (no re-encode).
  zc::pipelined_transfer(x, cb, chunk_elems, ws, status) -> int16[n]
      the chunked compress / link / decompress pipeline on three streams.
  zc::zq_compress(x, widths, sym, ws, status) -> uint8[zq_max_bytes(n)]
      Quad Length Codes of 1-byte symbols (uint8 / float8 e4m3), the table
      given as its 8 region widths and 256-entry rank -> symbol list.
  zc::zq_decompress(stream, n, status) -> uint8[n]
``ws`` and ``status`` are mutated (the workspace protocol and the device
status word), and declared so.
"""
from __future__ import annotations

import torch

from . import zc


@torch.library.custom_op("zc::compress", mutates_args=("ws", "status"))
def compress(x: torch.Tensor, cb: torch.Tensor, ws: torch.Tensor, status: torch.Tensor,
             adaptive: bool = False) -> tuple[torch.Tensor, torch.Tensor]:
    fn = zc.compress_adaptive if adaptive else zc.compress
    return fn(x.contiguous(), cb, ws, status)


@compress.register_fake
def _(x, cb, ws, status, adaptive=False):
    n = x.numel()
    main_bytes, max_esc = zc.compressed_size(n)  # host-side size law of the library
    esc = max(zc.raw_spill(n) if adaptive else max_esc, 16)
    return x.new_empty(main_bytes, dtype=torch.uint8), x.new_empty(esc, dtype=torch.uint8)


@torch.library.custom_op("zc::decompress", mutates_args=("status",))
def decompress(main: torch.Tensor, esc: torch.Tensor, n: int, status: torch.Tensor) -> torch.Tensor:
    return zc.decompress(main, esc, n, status)


@decompress.register_fake
def _(main, esc, n, status):
    return main.new_empty(n, dtype=torch.int16)


@torch.library.custom_op("zc::decompress_reduce", mutates_args=("status",))
def decompress_reduce(mains: list[torch.Tensor], escs: list[torch.Tensor], n: int,
                      status: torch.Tensor) -> torch.Tensor:
    out, _, _ = zc.decompress_reduce(list(mains), list(escs), n, status)
    return out


@decompress_reduce.register_fake
def _(mains, escs, n, status):
    return mains[0].new_empty(n, dtype=torch.int16)


@torch.library.custom_op("zc::pipelined_transfer", mutates_args=("ws", "status"))
def pipelined_transfer(x: torch.Tensor, cb: torch.Tensor, chunk_elems: int, ws: torch.Tensor,
                       status: torch.Tensor) -> torch.Tensor:
    return zc.pipelined_transfer(x.contiguous(), cb, chunk_elems, ws, status)


@pipelined_transfer.register_fake
def _(x, cb, chunk_elems, ws, status):
    return x.new_empty(x.numel(), dtype=torch.int16)


@torch.library.custom_op("zc::zq_compress", mutates_args=("ws", "status"))
def zq_compress(x: torch.Tensor, widths: list[int], sym: list[int], ws: torch.Tensor,
                status: torch.Tensor) -> torch.Tensor:
    return zc.zq_compress(x.contiguous(), zc.zq_table(widths, sym), ws, status)


@zq_compress.register_fake
def _(x, widths, sym, ws, status):
    return x.new_empty(zc.zq_max_bytes(x.numel()), dtype=torch.uint8)


@torch.library.custom_op("zc::zq_decompress", mutates_args=("status",))
def zq_decompress(stream: torch.Tensor, n: int, status: torch.Tensor) -> torch.Tensor:
    return zc.zq_decompress(stream, n, status)


@zq_decompress.register_fake
def _(stream, n, status):
    return stream.new_empty(n, dtype=torch.uint8)
