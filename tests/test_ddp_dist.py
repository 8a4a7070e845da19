"""The DDP hook's host side on CPU: two gloo ranks train a float32 model (not bf16 on the GPU, so the hook hands
each bucket to the process group's own all-reduce); the gradients must be the mean of what each rank computes
alone.  The zipped path (bf16 on the GPU) is checked in tests/test_gpu_ddp.py."""
import os
import socket

import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    try:
        os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
        dist.init_process_group("gloo", rank=rank, world_size=world)
        from torch.nn.parallel import DistributedDataParallel as DDP
        from lossless_bf16_exponent_zc_gb300 import ddp
        torch.manual_seed(3)
        ref = torch.nn.Sequential(torch.nn.Linear(50, 20), torch.nn.Tanh(), torch.nn.Linear(20, 3))
        model = DDP(torch.nn.Sequential(torch.nn.Linear(50, 20), torch.nn.Tanh(), torch.nn.Linear(20, 3)))
        model.module.load_state_dict(ref.state_dict())
        model.register_comm_hook(ddp.ZippedAllReduceState(device="cpu"), ddp.zipped_allreduce_hook)
        xs = [torch.randn(8, 50, generator=torch.Generator().manual_seed(10 + r)) for r in range(world)]
        model(xs[rank]).square().mean().backward()
        grads = []
        for r in range(world):  # what each rank computes alone
            ref.zero_grad()
            ref(xs[r]).square().mean().backward()
            grads.append([p.grad.clone() for p in ref.parameters()])
        for i, p in enumerate(model.module.parameters()):
            want = sum(g[i] for g in grads) / world
            assert torch.allclose(p.grad, want, rtol=1e-6, atol=1e-7), i
        dist.destroy_process_group()
        q.put((rank, True, ""))
    except Exception:
        import traceback
        q.put((rank, False, traceback.format_exc()[-1500:]))


def test_ddp_hook_native_path_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port, world = _free_port(), 2
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=300) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
    assert all(ok for _, ok, _ in out), out
