"""Multi-rank host logic of bench.py on CPU (gloo, world size 2).

The retention path does not exchange data between GPUs: bench.py runs N independent
replicas (weak scaling) and the only collective is the max of the elapsed time over
ranks.  These tests run two CPU ranks over gloo and check that the aggregate
throughput is all ranks' units over the slowest rank's time, that the reference arm
prints only on rank 0, and that a rank that raises makes the job fail instead of
hanging the other rank.
"""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


WORKER = r"""
import json, os, sys, time
sys.path.insert(0, {root!r})
import bench
rank = int(os.environ["RANK"])
mode = sys.argv[1]
if mode == "aggregate":
    d = bench.Dist().init("gloo")
    # rank r reports an elapsed time of 10*(r+1) ms for 1000 units
    value, worst = bench.aggregate(d, 10.0 * (rank + 1), 1000.0)
    d.barrier()
    print(json.dumps({{"rank": rank, "value": value, "worst": worst}}))
    d.close()
elif mode == "fail":
    d = bench.Dist().init("gloo", timeout_s=60)
    if rank == 1:
        raise RuntimeError("rank 1 fails before the timing collective")
    try:
        bench.aggregate(d, 1.0, 1.0)
    except Exception as e:                       # the peer is gone: error, not a hang
        print(json.dumps({{"rank": rank, "error": type(e).__name__}}))
        sys.exit(3)
"""


def _launch(mode: str, timeout: float = 120.0):
    port = _free_port()
    procs = []
    for rank in range(2):
        env = dict(os.environ, RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE="2",
                   MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), CUDA_VISIBLE_DEVICES="")
        env["TORCH_DIST_INIT_BARRIER"] = "0"
        procs.append(subprocess.Popen([sys.executable, "-c", WORKER.format(root=ROOT), mode],
                                      env=env, stdout=subprocess.PIPE, stderr=subprocess.PIPE,
                                      text=True))
    outs = []
    for p in procs:
        try:
            out, err = p.communicate(timeout=timeout)
        except subprocess.TimeoutExpired:
            for q in procs:
                q.kill()
            raise
        outs.append((p.returncode, out, err))
    return outs


def test_two_rank_aggregate_is_total_units_over_slowest_rank():
    outs = _launch("aggregate")
    lines = []
    for rc, out, err in outs:
        assert rc == 0, err
        lines.append(json.loads(out.strip().splitlines()[-1]))
    for ln in lines:
        assert ln["worst"] == pytest.approx(20.0)
        # 2 ranks x 1000 units over the slowest rank's 20 ms
        assert ln["value"] == pytest.approx(2000.0 / 0.020)


def test_failed_rank_fails_the_job_without_hanging():
    outs = _launch("fail", timeout=300.0)
    rcs = [rc for rc, _, _ in outs]
    assert rcs[1] != 0                           # the failing rank exits with an error
    assert rcs[0] != 0                           # its peer gets an error, not a hang


def test_reference_arm_prints_only_on_rank_zero(tmp_path):
    """--impl reference: rank 0 times the oracle on a tiny step; other ranks exit 0 silently."""
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1", CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "1"], env=env, capture_output=True,
                       text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""
