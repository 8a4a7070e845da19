"""zc_compress_noalloc: the encoder for callers that cannot allocate device memory.

Such callers (framework hooks that only hand over the tensors to send, paths
that must never call cudaMalloc) pass no
workspace; the library keeps the scratch in a fixed device array of its own.
This file is collected last so that a run stopping at its first failure has
already run everything else, and it passes both alone in a fresh process and
after the other tests (the array keeps the previous call's contents).
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu


def _noalloc(lib):
    f = lib.zc_compress_noalloc
    vp, u64 = ctypes.c_void_p, ctypes.c_uint64
    f.argtypes = [vp, u64, vp, vp, vp, u64, vp, vp]
    f.restype = ctypes.c_int
    return f


def test_noalloc_matches_compress_two_calls_in_a_row(zc):
    f = _noalloc(zc.load())
    stream = torch.cuda.current_stream().cuda_stream
    cb = zc.codebook_to_device(oracle.codebook_from_sigma(1e-3))
    for seed, n in ((31, 23 * 4096 + 77), (32, 1 << 20)):   # two calls in a row, different sizes
        x = workloads.gradient(n=n, sigma=1e-3, seed=seed)
        xt = torch.from_numpy(x.view(np.int16)).cuda()
        mb, eb = zc.compressed_size(n)
        # the existing entry point, with its own workspace
        st_ref = zc.new_status()
        ref_main, ref_esc = zc.compress(xt, cb, zc.workspace(n), st_ref)
        # the new entry point through the C ABI, no workspace
        main = torch.full((mb,), 0xEE, dtype=torch.uint8, device="cuda")
        esc = torch.full((eb,), 0xEE, dtype=torch.uint8, device="cuda")
        st = zc.new_status()
        rc = f(xt.data_ptr(), n, cb.data_ptr(), main.data_ptr(), esc.data_ptr(), eb, st.data_ptr(), stream)
        assert rc == 0, zc.status_string(rc)
        torch.cuda.synchronize()
        assert zc.status_value(st) == 0 and zc.status_value(st_ref) == 0
        k = zc.header_n_esc(ref_main)
        assert torch.equal(main, ref_main)
        assert zc.header_n_esc(main) == k
        assert torch.equal(esc[:k], ref_esc[:k])
        out = zc.decompress(main, esc, n, zc.new_status())
        torch.cuda.synchronize()
        assert np.array_equal(out.cpu().numpy().view(np.uint16), x)


def test_noalloc_rejects_oversize_without_launching(zc):
    f = _noalloc(zc.load())
    fake = 0x10000
    rc = f(fake, (1 << 28) + 1, fake, fake, fake, 16, fake, None)
    assert rc == zc.ERR_WORKSPACE
