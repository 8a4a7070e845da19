"""The benchmark's multi-rank path on CPU: world-size-2 gloo ranks agree on the max (time) and sum (bytes)
over ranks, as the replicas-only GPU run does over NCCL."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    mx = bench.max_over_ranks(1.5 + rank, world, device="cpu")
    sm = bench.sum_over_ranks(10.0 * (rank + 1), world, device="cpu")
    r, w, _ = bench.dist_env()
    q.put((rank, mx, sm, r, w))
    dist.destroy_process_group()


def test_rank_aggregation_gloo():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [o[1] for o in out] == [2.5, 2.5]
    assert [o[2] for o in out] == [30.0, 30.0]
    assert [(o[3], o[4]) for o in out] == [(0, 2), (1, 2)]


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks(3.0, 1) == 3.0
    assert bench.sum_over_ranks(3.0, 1) == 3.0


def test_reference_arm_line(capsys):
    import json
    import bench
    bench.main(["--impl", "reference", "--steps", "2", "--warmup", "1", "--n-log2", "16", "--ref-sample-log2", "14"])
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"
    host = line["cpu_baseline"]["host"]
    assert host["nproc"] >= 1 and host["machine"]


def test_host_info_reads_cpuinfo_fields(tmp_path, monkeypatch):
    """The CPU model comes from /proc/cpuinfo: "model name" on x86, implementer and part numbers on Arm."""
    import builtins
    import bench
    real_open = builtins.open
    arm = "processor\t: 0\nBogoMIPS\t: 2000.00\nCPU implementer\t: 0x41\nCPU part\t: 0xd4f\n"

    def fake_open(path, *a, **k):
        if path == "/proc/cpuinfo":
            p = tmp_path / "cpuinfo"
            p.write_text(arm)
            return real_open(p, *a, **k)
        return real_open(path, *a, **k)

    monkeypatch.setattr(builtins, "open", fake_open)
    assert bench.host_info()["cpu"] == "implementer 0x41 part 0xd4f"


def test_traffic_record_follows_code_not_comments(tmp_path, monkeypatch):
    """A measured DRAM traffic figure is tied to the kernel's code: comment and whitespace edits keep it, a
    code edit turns it into null."""
    import shutil
    import bench
    csrc = tmp_path / "lossless_bf16_exponent_zc_gb300" / "csrc"
    csrc.mkdir(parents=True)
    for f in bench.KERNEL_SOURCES["encode_kernel"]:
        shutil.copy(os.path.join(bench.ROOT, "lossless_bf16_exponent_zc_gb300", "csrc", f), csrc / f)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h0 = bench.source_hash("encode_kernel")
    main = csrc / bench.KERNEL_SOURCES["encode_kernel"][0]
    text = main.read_text()
    main.write_text("// a new comment line\n" + text.replace("\n", "  \n", 3) + "\n\n")
    assert bench.source_hash("encode_kernel") == h0
    monkeypatch.setitem(bench.MEASURED_TRAFFIC, "encode_kernel", (h0, 123))
    assert bench.measured_traffic("encode_kernel") == 123
    main.write_text(text + "\nconstexpr int kAnotherConstant = 1;\n")
    assert bench.source_hash("encode_kernel") != h0
    assert bench.measured_traffic("encode_kernel") is None
