"""GPU checks of the zipped transfer pipeline (compress / link / decompress on three streams).

[CCCL §3.2] overlaps the compression of chunk k, the transfer of chunk k - 1
and the decompression of chunk k - 2 on separate streams with double-buffered
slots; [ZipCCL §2.D] sends the fixed-size main stream first and the
variable-size escape stream after it.  The pipeline as a whole is the identity
on the values (each chunk goes through the adaptive encoder, the link copies
and the decoder, all checked byte for byte against the oracle elsewhere), so
every case here compares the output with the input bit for bit: a missing
dependency between the streams shows up as corrupted values or a decoder
status.  Chunk counts from 1 to 256, ragged last chunks, chunk sizes that are
not a multiple of the 4096-value tile, incompressible chunks that travel RAW,
one stream for all three stages, and a reused workspace.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu


def dev(x):
    return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).cuda()


def run(zc, x, chunk, cb, ws=None, streams=None):
    xt = dev(x)
    ws = zc.pipeline_workspace(chunk) if ws is None else ws
    st = zc.new_status()
    out = zc.pipelined_transfer(xt, zc.codebook_to_device(cb), chunk, ws, st, streams=streams)
    torch.cuda.synchronize()
    assert zc.status_value(st) == 0, zc.status_string(zc.status_value(st))
    got = out.cpu().numpy().view(np.uint16)
    bad = np.nonzero(got != x)[0]
    assert bad.size == 0, f"{bad.size} values differ, first at {bad[:8]}"
    return ws


@pytest.mark.parametrize("n,chunk", [
    ((1 << 22) + 1234, 1 << 20),   # 5 chunks, ragged last
    (1 << 20, 1 << 22),            # one chunk larger than the tensor
    (3000, 1024),                  # chunks below one tile
    (100_000, 4104),               # chunk not a multiple of the tile size
    (1 << 21, 1 << 16),            # 32 chunks
])
def test_pipeline_identity(zc, n, chunk):
    x = workloads.gradient(n=n, sigma=1e-3, seed=n % 1009)
    run(zc, x, chunk, oracle.codebook_from_sigma(1e-3))


def test_pipeline_many_small_chunks(zc):
    """256 chunks of 2^14 values: the slot reuse waits are exercised 254 times."""
    x = workloads.gradient(n=1 << 22, sigma=1e-3, seed=77)
    run(zc, x, 1 << 14, oracle.codebook_from_sigma(1e-3))


def test_pipeline_raw_chunks(zc):
    """Chunks of random bit patterns (stored RAW) between Gaussian chunks."""
    chunk = 1 << 16
    parts = []
    for i in range(12):
        if i % 3 == 1:
            parts.append(workloads.random_bits(chunk, seed=i))
        else:
            parts.append(workloads.gaussian(chunk, sigma=1e-3, seed=100 + i))
    x = np.concatenate(parts + [workloads.random_bits(777, seed=99)])
    run(zc, x, chunk, oracle.codebook_from_sigma(1e-3))


def test_pipeline_one_stream(zc):
    x = workloads.gradient(n=(1 << 20) + 8, sigma=1e-3, seed=5)
    s = torch.cuda.current_stream()
    run(zc, x, 1 << 18, oracle.codebook_from_sigma(1e-3), streams=(s, s, s))


def test_pipeline_workspace_reused(zc):
    chunk = 1 << 17
    ws = zc.pipeline_workspace(chunk)
    for i in range(3):
        x = workloads.gradient(n=(1 << 20) - 4096 * i, sigma=1e-3, seed=200 + i)
        run(zc, x, chunk, oracle.codebook_from_sigma(1e-3), ws=ws)


def test_pipeline_empty(zc):
    x = np.zeros(0, np.uint16)
    ws = zc.pipeline_workspace(4096)
    st = zc.new_status()
    out = zc.pipelined_transfer(torch.empty(0, dtype=torch.int16, device="cuda"),
                                zc.codebook_to_device(oracle.codebook_from_sigma(1e-3)), 4096, ws, st)
    torch.cuda.synchronize()
    assert zc.status_value(st) == 0 and out.numel() == 0


def test_pipeline_argument_errors(zc):
    x = dev(workloads.gaussian(4096))
    cb = zc.codebook_to_device(oracle.codebook_from_sigma(0.02))
    st = zc.new_status()
    ws = zc.pipeline_workspace(4096)
    with pytest.raises(zc.ZcError) as e:
        zc.pipelined_transfer(x, cb, 4100, ws, st)  # not a multiple of 8
    assert e.value.code == zc.ERR_INVALID_ARG
    with pytest.raises(zc.ZcError) as e:
        zc.pipelined_transfer(x, cb, 8192, ws, st)  # workspace sized for 4096-value chunks
    assert e.value.code == zc.ERR_WORKSPACE


# ---------------------------------------------------------------- pipeline plans (the sequence as a CUDA graph)
def check_plan(zc, plan, x, stream=None):
    out = plan.launch(stream)
    torch.cuda.synchronize()
    assert zc.status_value(plan.status) == 0, zc.status_string(zc.status_value(plan.status))
    got = out.cpu().numpy().view(np.uint16)
    bad = np.nonzero(got != x)[0]
    assert bad.size == 0, f"{bad.size} values differ, first at {bad[:8]}"


@pytest.mark.parametrize("overlap", [True, False])
@pytest.mark.parametrize("n,chunk", [
    ((1 << 22) + 1234, 1 << 20),   # 5 chunks, ragged last
    (100_000, 4104),               # chunk not a multiple of the tile size
    (1 << 21, 1 << 16),            # 32 chunks
])
def test_plan_identity(zc, n, chunk, overlap):
    x = workloads.gradient(n=n, sigma=1e-3, seed=n % 997)
    plan = zc.pipeline_plan(dev(x), zc.codebook_to_device(oracle.codebook_from_sigma(1e-3)), chunk,
                            zc.pipeline_workspace(chunk), zc.new_status(), overlap=overlap)
    check_plan(zc, plan, x)
    plan.close()


def test_plan_replays_new_contents(zc):
    """One plan, replayed over new values written into the same input buffer: Gaussian, then chunks that travel
    RAW, then Gaussian again (the workspace's escape-scan state carries over between replays)."""
    chunk, n = 1 << 16, 12 * (1 << 16) + 777
    xt = torch.empty(n, dtype=torch.int16, device="cuda")
    plan = zc.pipeline_plan(xt, zc.codebook_to_device(oracle.codebook_from_sigma(1e-3)), chunk,
                            zc.pipeline_workspace(chunk), zc.new_status())
    side = torch.cuda.Stream()
    for i in range(4):
        if i == 1:
            x = np.concatenate([workloads.random_bits(n // 2, seed=i), workloads.gaussian(n - n // 2, sigma=1e-3)])
        else:
            x = workloads.gradient(n=n, sigma=1e-3, seed=300 + i)
        xt.copy_(dev(x))
        torch.cuda.synchronize()
        check_plan(zc, plan, x, stream=side if i == 3 else None)


def test_plan_empty(zc):
    ws = zc.pipeline_workspace(4096)
    plan = zc.pipeline_plan(torch.empty(0, dtype=torch.int16, device="cuda"),
                            zc.codebook_to_device(oracle.codebook_from_sigma(1e-3)), 4096, ws, zc.new_status())
    assert plan.launch().numel() == 0
    plan.close()
    with pytest.raises(RuntimeError):
        plan.launch()


def test_plan_first_call_in_a_fresh_process():
    """A plan made before any other libzc call: each kernel's one-time preparation (shared-memory limit,
    occupancy) then happens while the launch sequence is being captured.  Run in a fresh interpreter."""
    import subprocess
    import sys
    code = r'''
import numpy as np, torch, workloads, oracle
from lossless_bf16_exponent_zc_gb300 import zc
n, chunk = (1 << 20) + 24, 1 << 18
x = workloads.gradient(n=n, sigma=1e-3, seed=3)
xt = torch.from_numpy(x.view(np.int16)).cuda()
plan = zc.pipeline_plan(xt, zc.codebook_to_device(oracle.codebook_from_sigma(1e-3)), chunk,
                        zc.pipeline_workspace(chunk), zc.new_status())
out = plan.launch()
torch.cuda.synchronize()
assert zc.status_value(plan.status) == 0
assert np.array_equal(out.cpu().numpy().view(np.uint16), x)
print("ok")
'''
    import os
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "-c", code], cwd=root, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0 and r.stdout.strip().endswith("ok"), r.stdout[-2000:] + r.stderr[-2000:]
