"""torch.ops.zc: the codec as PyTorch operators ([ZipCCL §3] drop-in use, [CCCL §4] framework integration).

CPU part (no GPU): the operators register, and a function built from them
traces into a graph with fake CUDA tensors (make_fx, tracing_mode="fake"):
output shapes and dtypes come from the library's host-side size law, the
workspace and status are marked as mutated.  GPU part: each operator's
outputs equal the binding's (and so the oracle's, byte for byte).
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from lossless_bf16_exponent_zc_gb300 import torch_ops  # noqa: F401  (registers torch.ops.zc)
from lossless_bf16_exponent_zc_gb300 import zc


def test_ops_registered():
    for name in ("compress", "decompress", "decompress_reduce", "pipelined_transfer", "zq_compress", "zq_decompress"):
        assert hasattr(torch.ops.zc, name)
    schema = torch.ops.zc.compress.default._schema
    mutated = {a.name for a in schema.arguments if a.alias_info is not None and a.alias_info.is_write}
    assert mutated == {"ws", "status"}


@pytest.mark.parametrize("n", [1, 4096, 100_003])
def test_fake_tracing(n):
    from torch.fx.experimental.proxy_tensor import make_fx
    from torch._subclasses.fake_tensor import FakeTensorMode

    def roundtrip(x, cb, ws, st):
        main, esc = torch.ops.zc.compress(x, cb, ws, st, True)
        return main, esc, torch.ops.zc.decompress(main, esc, x.numel(), st)

    with FakeTensorMode():
        x = torch.empty(n, dtype=torch.bfloat16, device="cuda")
        cb = torch.empty(7, dtype=torch.uint8, device="cuda")
        ws = torch.empty(zc.workspace_size(n), dtype=torch.uint8, device="cuda")
        st = torch.empty(1, dtype=torch.int32, device="cuda")
        main, esc, y = roundtrip(x, cb, ws, st)
        assert main.shape == (oracle.main_bytes(n),) and main.dtype == torch.uint8
        assert esc.shape == (max(oracle.raw_spill(n), 16),)
        assert y.shape == (n,) and y.dtype == torch.int16 and y.device.type == "cuda"
        g = make_fx(roundtrip, tracing_mode="fake")(x, cb, ws, st)
    targets = [str(node.target) for node in g.graph.nodes if node.op == "call_function"]
    assert any("zc.compress" in t for t in targets) and any("zc.decompress" in t for t in targets)


@pytest.mark.parametrize("n", [1, 4096, 100_003])
def test_fake_tracing_qlc(n):
    from torch.fx.experimental.proxy_tensor import make_fx
    from torch._subclasses.fake_tensor import FakeTensorMode
    widths = list(oracle.QLC_DEFAULT_WIDTHS)
    sym = list(range(256))

    def roundtrip(x, ws, st):
        s = torch.ops.zc.zq_compress(x, widths, sym, ws, st)
        return s, torch.ops.zc.zq_decompress(s, x.numel(), st)

    with FakeTensorMode():
        x = torch.empty(n, dtype=torch.uint8, device="cuda")
        ws = torch.empty(zc.workspace_size(n), dtype=torch.uint8, device="cuda")
        st = torch.empty(1, dtype=torch.int32, device="cuda")
        s, y = roundtrip(x, ws, st)
        assert s.shape == (zc.zq_max_bytes(n),) and s.dtype == torch.uint8
        assert y.shape == (n,) and y.dtype == torch.uint8 and y.device.type == "cuda"
        g = make_fx(roundtrip, tracing_mode="fake")(x, ws, st)
    targets = [str(node.target) for node in g.graph.nodes if node.op == "call_function"]
    assert any("zc.zq_compress" in t for t in targets) and any("zc.zq_decompress" in t for t in targets)


@pytest.mark.gpu
def test_qlc_ops_match_oracle(zc):
    x = workloads.fp8_ffn1(3 * 4096 + 777, seed=21)
    sym = oracle.qlc_table_for(x)
    widths = list(oracle.QLC_DEFAULT_WIDTHS)
    ws, st = zc.workspace(x.size), zc.new_status()
    xt = torch.from_numpy(x).cuda().view(torch.float8_e4m3fn)  # float8 tensors are coded by their bytes
    s = torch.ops.zc.zq_compress(xt, widths, [int(v) for v in sym], ws, st)
    want = oracle.qlc_compress(x, widths, sym)
    torch.cuda.synchronize()
    assert zc.status_value(st) == 0
    assert np.array_equal(s[:want.size].cpu().numpy(), want)
    y = torch.ops.zc.zq_decompress(s, x.size, st)
    torch.cuda.synchronize()
    assert zc.status_value(st) == 0 and np.array_equal(y.cpu().numpy(), x)


@pytest.mark.gpu
def test_ops_match_binding(zc):
    x = workloads.gradient(n=(1 << 20) + 333, sigma=1e-3, seed=12)
    xt = torch.from_numpy(x.view(np.int16)).cuda()
    cb = zc.codebook_to_device(oracle.codebook_from_sigma(1e-3))
    ws = zc.workspace(x.size)
    st = zc.new_status()
    main, esc = torch.ops.zc.compress(xt, cb, ws, st)
    om, oe = oracle.compress(x, cb.cpu().numpy())
    torch.cuda.synchronize()
    assert zc.status_value(st) == 0
    k = zc.header_n_esc(main)
    assert np.array_equal(main.cpu().numpy(), om) and np.array_equal(esc[:k].cpu().numpy(), oe)
    y = torch.ops.zc.decompress(main, esc, x.size, st)
    assert torch.equal(y, xt)
    # adaptive on random bits: RAW
    r = workloads.random_bits(50_000, seed=3)
    rm, re_ = torch.ops.zc.compress(torch.from_numpy(r.view(np.int16)).cuda(), cb, ws, st, True)
    om, oe, raw = oracle.compress_adaptive(r, cb.cpu().numpy())
    assert raw and np.array_equal(rm.cpu().numpy(), om) and np.array_equal(re_[:oe.size].cpu().numpy(), oe)
    # reduce and pipeline
    shards = [workloads.gaussian(20_000, sigma=1e-3, seed=40 + i) for i in range(3)]
    comp = [torch.ops.zc.compress(torch.from_numpy(s.view(np.int16)).cuda(), cb, zc.workspace(20_000), st)
            for s in shards]
    red = torch.ops.zc.decompress_reduce([c[0] for c in comp], [c[1] for c in comp], 20_000, st)
    want = oracle.reduce(shards)
    assert np.array_equal(red.cpu().numpy().view(np.uint16), want)
    pws = zc.pipeline_workspace(1 << 16)
    out = torch.ops.zc.pipelined_transfer(xt, cb, 1 << 16, pws, st)
    torch.cuda.synchronize()
    assert torch.equal(out, xt) and zc.status_value(st) == 0
