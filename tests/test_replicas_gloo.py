"""Several GPUs run independent replicas (no collective on the data path):
the bookkeeping of such a job, checked with two gloo ranks on the CPU.  The
job time is the slowest rank's, the throughput counts every rank's units, and
each rank draws inputs of its own."""
import json
import os
import socket
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_two_gloo_ranks_agree_on_the_slowest_rank(tmp_path):
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr=127.0.0.1", f"--master-port={_free_port()}", os.path.join(HERE, "replica_worker.py"),
           str(tmp_path)]
    env = {**os.environ, "OMP_NUM_THREADS": "1"}
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=300, env=env)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-2000:]
    res = [json.load(open(tmp_path / f"rank{i}.json")) for i in range(2)]
    for d in res:
        assert d["world"] == 2
        assert d["ms"] == 20.0  # the slower rank
        assert abs(d["value"] - 7 * 2 / 0.020) < 1e-9
    assert res[0]["digest"] != res[1]["digest"]  # inputs of their own
