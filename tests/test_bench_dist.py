"""Host-side multi-rank logic of bench.py, on CPU with the gloo backend (world size 2).

Each rank verifies its own batch (weak scaling); the only cross-rank steps are the barrier
around the timed region and the max of the ranks' times, and every rank draws its uniforms
from its own Philox counter range.
"""
import os
import socket
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench

    D = bench.Dist()
    D.init("gloo")
    D.barrier()
    local = 1.5 + 2.0 * rank  # each rank's own elapsed time
    out[rank] = (D.max(local, torch.device("cpu")), bench.rank_offset(D.rank), D.world)
    D.barrier()
    D.close()


def test_two_ranks_take_the_max_time_and_distinct_offsets():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.start_processes(_worker, args=(world, port, out), nprocs=world, start_method="spawn")
        res = dict(out)
    assert sorted(res) == [0, 1]
    # Every rank sees the slowest rank's time: the whole-job rate divides by it.
    assert res[0][0] == res[1][0] == 3.5
    # Disjoint Philox counter ranges (the offset's high word is the rank).
    assert res[0][1] != res[1][1]
    assert res[1][1] >> 32 == 1 and res[0][1] >> 32 == 0
    assert res[0][2] == res[1][2] == world


def test_single_process_dist_is_a_no_op():
    sys.path.insert(0, ROOT)
    import bench

    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        os.environ.pop(k, None)
    D = bench.Dist()
    D.init("gloo")
    assert D.world == 1 and D.pg is None
    assert D.max(2.25, torch.device("cpu")) == 2.25
    D.barrier()
    D.close()


def test_reference_arm_prints_one_contract_line():
    """`bench.py --impl reference` (the oracle on the host cores, a bounded sample) prints one JSON
    line with the contract's keys, its own e2e with no transfers, and a cpu_baseline equal to it."""
    import json
    import subprocess

    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "1", "--cpu-seconds", "1"], capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip().startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["value"] > 0 and d["steps"] == 1 and d["n_gpus"] == 1
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert d["e2e"]["value"] == d["value"] and d["e2e"]["unit"] == d["unit"]
    assert "workload" in d["config"]
