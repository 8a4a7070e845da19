"""DDP communication hook: gradient buckets all-reduced compressed [ZipCCL §2.D].

A bf16 bucket is reduced as a zipped reduce-scatter (each rank compresses its P shards with the bucket's exact
histogram codebook, sends shard r to rank r, and rank r adds the P shards it receives in fp32 in rank order,
rounding once to bf16 and re-encoding the result) followed by a zipped all-gather of the re-encoded shards (every
rank sends its shard's streams to every rank and decodes all of them in one batched launch).  The sum is then
divided by the number of ranks, as DDP averages gradients.  Every codec step runs in libzc's kernels; the
exchanges are point-to-point sends (exchange.zipped_reduce_scatter, exchange.all_gather_streams).  Buckets of other dtypes go through the
process group's own all-reduce.

    state = ZippedAllReduceState()
    ddp_model.register_comm_hook(state, zipped_allreduce_hook)
    ...backward...
    state.check()        # raises if a kernel recorded a device error
"""
import torch
import torch.distributed as dist

from . import zc
from .exchange import all_gather_streams, zipped_reduce_scatter


class ZippedAllReduceState:
    """What the hook keeps between buckets: the process group, a device status word, and workspaces per size
    (zero-filled once, reused)."""

    def __init__(self, group=None, device=None):
        self.group = group
        self.device = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
        self.status = zc.new_status(device=self.device)
        self._ws: dict[tuple, torch.Tensor] = {}

    def workspace(self, sizes: tuple[int, ...]) -> torch.Tensor:
        ws = self._ws.get(sizes)
        if ws is None:
            ws = self._ws[sizes] = zc.workspace(list(sizes), device=self.device)
        return ws

    def check(self) -> None:
        code = zc.status_value(self.status)
        if code != 0:
            raise zc.ZcError(code, "zipped_allreduce_hook")


def zipped_allreduce(t: torch.Tensor, state: ZippedAllReduceState) -> torch.Tensor:
    """All-reduce (mean) of a bf16 CUDA tensor over state.group through the zipped reduce-scatter and all-gather;
    writes the result into t and returns it."""
    group = state.group
    world = dist.get_world_size(group)
    n = t.numel()
    m = -(-n // (8 * world)) * 8  # shard size: a multiple of 8 values, so every shard is 16-byte aligned
    src = t.view(torch.int16)
    if world * m == n:
        x = src
    else:
        x = torch.zeros(world * m, dtype=torch.int16, device=t.device)
        x[:n].copy_(src)
    cb, _ = zc.histogram_topk(x, state.workspace((world * m,)), state.status)
    _, om, oe = zipped_reduce_scatter(x, cb, state.status, out_cb=cb, ws=state.workspace((m,) * world),
                                      group=group)
    out = all_gather_streams(om, oe, m, state.status, group=group)
    t.copy_(out[:n].view(torch.bfloat16))
    if world > 1:
        t.div_(world)
    return t


def zipped_allreduce_hook(state: ZippedAllReduceState, bucket) -> torch.futures.Future[torch.Tensor]:
    """DDP communication hook (register_comm_hook(state, zipped_allreduce_hook))."""
    t = bucket.buffer()
    world = dist.get_world_size(state.group)
    if t.dtype != torch.bfloat16 or not t.is_cuda:
        t.div_(world)
        work = dist.all_reduce(t, group=state.group, async_op=True)
        return work.get_future().then(lambda f: f.value()[0])
    fut = torch.futures.Future()
    fut.set_result(zipped_allreduce(t, state))
    return fut
