"""Host-side logic of bench.py: the whole-job aggregation over ranks (max
time over ranks, all ranks' units) with world_size 2 on the gloo backend,
and the reference arm's JSON line at a tiny size."""
import json
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    local_ms = [2.0, 5.0][rank]
    max_ms, rate = bench.aggregate(local_ms, 1e9, world)
    out[rank] = (max_ms, rate)
    dist.destroy_process_group()


def test_aggregate_two_ranks_gloo():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    for r in range(2):
        max_ms, rate = out[r]
        assert max_ms == 5.0
        assert rate == pytest.approx(2 * 1e9 / 5e-3)


def test_aggregate_single_rank():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.aggregate(4.0, 8e9, 1) == (4.0, pytest.approx(2e12))


def test_reference_arm_line(capsys, monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "0")
    monkeypatch.setenv("WORLD_SIZE", "1")
    bench.main(["--impl", "reference", "--workload", "bf16_4096x4096x4096_f32out", "--shape", "64x64x128",
                "--steps", "3", "--warmup", "3", "--reference-seconds", "1"])
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "TFLOP/s" and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"


def test_kernel_hash_ignores_comments_only():
    """Recorded DRAM traffic stays attached to a kernel across comment edits, not code edits."""
    sys.path.insert(0, ROOT)
    import bench
    src = 'int a = 1; // note\n/* block\n comment */ asm("tcgen05.mma // not a comment");\n'
    assert bench.strip_comments(src) == bench.strip_comments(src.replace("note", "other note"))
    assert bench.strip_comments(src) == bench.strip_comments(src.replace("block", "a longer block"))
    assert "not a comment" in bench.strip_comments(src)
    assert bench.strip_comments(src) != bench.strip_comments(src.replace("a = 1", "a = 2"))
    for fam in bench.KERNEL_SOURCES:
        h = bench.kernel_source_hash(fam)
        assert len(h) == 16 and h == bench.kernel_source_hash(fam)
