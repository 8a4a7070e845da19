"""The DDP communication hook (ddp.zipped_allreduce_hook) on one NCCL rank in a spawned child (a box here has one
GPU): bf16 gradient buckets go through the whole zipped path -- the bucket's histogram codebook, the zipped
reduce-scatter with its re-encoded output, the all-gather of the compressed shards, the batched decode -- and the
gradients must equal, bit for bit, those of the same model trained without DDP (one rank: the mean is the
gradient itself).  Buckets are kept small so a step has several, of sizes that need padding to whole 8-value
shards.  A float32 model takes the process group's own all-reduce."""
import os
import socket

import pytest
import torch.multiprocessing as mp

pytestmark = pytest.mark.gpu


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _child(port, q):
    try:
        import copy
        import torch
        import torch.distributed as dist
        from torch.nn.parallel import DistributedDataParallel as DDP
        from lossless_bf16_exponent_zc_gb300 import ddp
        torch.cuda.set_device(0)
        os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK="0", WORLD_SIZE="1",
                          NCCL_NVLS_ENABLE="0")
        dist.init_process_group("nccl", rank=0, world_size=1, device_id=torch.device("cuda", 0))
        for dtype in (torch.bfloat16, torch.float32):
            torch.manual_seed(5)
            ref = torch.nn.Sequential(torch.nn.Linear(1000, 517), torch.nn.GELU(), torch.nn.Linear(517, 333),
                                      torch.nn.GELU(), torch.nn.Linear(333, 7)).cuda().to(dtype)
            model = DDP(copy.deepcopy(ref), device_ids=[0], bucket_cap_mb=0.5)
            state = ddp.ZippedAllReduceState()
            model.register_comm_hook(state, ddp.zipped_allreduce_hook)
            for step in range(3):
                x = torch.randn(64, 1000, device="cuda", dtype=dtype)
                for m in (ref, model):
                    m.zero_grad(set_to_none=True)
                    m(x).float().square().mean().backward()
                torch.cuda.synchronize()
                state.check()
                for (name, a), b in zip(ref.named_parameters(), model.module.parameters()):
                    assert torch.equal(a.grad, b.grad), f"{dtype} step {step}: {name}"
        dist.destroy_process_group()
        q.put((True, ""))
    except Exception:
        import traceback
        q.put((False, traceback.format_exc()[-2000:]))


def test_zipped_allreduce_hook_one_rank():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    p = ctx.Process(target=_child, args=(_free_port(), q))
    p.start()
    ok, msg = q.get(timeout=600)
    p.join(timeout=120)
    assert ok, msg
    assert p.exitcode == 0
