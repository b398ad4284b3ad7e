"""The multi-rank host logic of bench.py on the CPU: two gloo ranks (127.0.0.1).

Each rank of `bench.py --gpus N` runs an independent replica; the job's time is the
slowest rank's and its value sums the replicas' work. The reference arm runs on rank 0
only and prints one JSON line; other ranks exit 0 without output."""
import io
import json
import os
import socket
import sys
from contextlib import redirect_stdout
from types import SimpleNamespace

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = 10.0 + 5.0 * rank  # rank 1 is the slower one
        total = bench.max_over_ranks(local_ms, world, torch.device("cpu"))
        value = bench.job_throughput_gbs(world, 28_000_000, 100, total)
        buf = io.StringIO()
        with redirect_stdout(buf):
            rc = bench.run_reference(SimpleNamespace(steps=1, warmup=0))
        q.put((rank, total, value, rc, buf.getvalue()))
    finally:
        dist.destroy_process_group()


def test_two_rank_aggregation_and_reference_arm():
    ctx = mp.get_context("spawn")
    q = ctx.SimpleQueue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=300)
        assert p.exitcode == 0
    out = {}
    while not q.empty():
        rank, total, value, rc, text = q.get()
        out[rank] = (total, value, rc, text)
    assert set(out) == {0, 1}
    for rank in (0, 1):
        total, value, rc, _ = out[rank]
        assert total == 15.0  # the slowest rank's time, on every rank
        assert value == pytest.approx(2 * 28_000_000 * 100 / 0.015 / 1e9)
        assert rc == 0
    lines = [l for l in out[0][3].splitlines() if l.strip()]
    assert len(lines) == 1
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference" and rec["n_gpus"] == 2 and rec["value"] > 0
    assert rec["cpu_baseline"]["kind"] == "oracle"
    assert out[1][3].strip() == ""  # rank 1 does no work and prints nothing
