"""The N > 1 path of the bench on CPU: two gloo ranks, each an independent replica.

The verification step shards by sequence and has no exchange step, so the ranks share no
data: each rank's accepted paths must equal a single-process run of its own batch, the
batches must differ between ranks, and the job's throughput must be every rank's tokens
over the slowest rank's time. The reference arm under torchrun prints one line from rank 0
and lets the other rank exit without work.
"""

import json
import os
import socket
import subprocess
import sys

import numpy as np
import pytest

import bench
import oracle
from speculative_decoding_tree_parent_gb300 import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _env(rank, ws, port):
    env = dict(os.environ, RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE=str(ws), MASTER_ADDR="127.0.0.1",
               MASTER_PORT=str(port), OMP_NUM_THREADS="1")
    env.pop("CUDA_VISIBLE_DEVICES", None)
    return env


def test_replica_seeds():
    assert bench.replica_seed(2, 0) is None           # rank 0 = the single-GPU workload itself
    seeds = {bench.replica_seed(2, r) for r in range(1, 8)}
    assert len(seeds) == 7 and None not in seeds
    assert bench.reduce_over_ranks(3.5, "max", 1) == 3.5
    assert bench.job_throughput(640, 2.0) == pytest.approx(320000.0)


@pytest.mark.timeout(240)
def test_two_gloo_ranks_are_independent_replicas(tmp_path):
    ws, port = 2, _free_port()
    outs = [tmp_path / f"rank{r}.json" for r in range(ws)]
    procs = [subprocess.Popen([sys.executable, os.path.join(ROOT, "tests", "replica_worker.py"), str(outs[r])],
                              env=_env(r, ws, port), cwd=ROOT, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)
             for r in range(ws)]
    logs = []
    try:
        for p in procs:
            logs.append(p.communicate(timeout=200)[0].decode(errors="replace"))
    finally:
        for p in procs:
            if p.poll() is None:
                p.kill()
    assert all(p.returncode == 0 for p in procs), logs
    res = [json.load(open(o)) for o in outs]

    # bookkeeping: max of the ranks' times, sum of their tokens, same view on every rank
    for r in res:
        assert r["ws"] == ws
        assert r["max_ms"] == max(x["own_ms"] for x in res)
        assert r["tokens_all"] == sum(x["own_tokens"] for x in res)
        assert r["value"] == pytest.approx(r["tokens_all"] * 3 / (r["max_ms"] / 1e3))

    # independence: each rank's result is the single-process oracle run of its own batch
    for rank, r in enumerate(res):
        inp = W.generate_index(1, seed=bench.replica_seed(1, rank))
        acc = oracle.greedy_accept(inp.parent, inp.draft_tokens, inp.target_logits, inp.qo_indptr, inp.path_cap)
        np.testing.assert_array_equal(np.asarray(r["accept_len"]), acc.accept_len)
        np.testing.assert_array_equal(np.asarray(r["path"]), acc.path)
        np.testing.assert_array_equal(np.asarray(r["out_tokens"]), acc.out_tokens)
    assert res[0]["parent_digest"] != res[1]["parent_digest"]   # the ranks drew different batches


@pytest.mark.timeout(300)
def test_reference_arm_under_torchrun_prints_once(tmp_path):
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "3"]
    env = dict(os.environ, OMP_NUM_THREADS="2")
    p = subprocess.run(cmd, cwd=ROOT, env=env, stdout=subprocess.PIPE, stderr=subprocess.PIPE, timeout=280)
    assert p.returncode == 0, p.stderr.decode(errors="replace")[-2000:]
    lines = [ln for ln in p.stdout.decode().splitlines() if ln.startswith("{")]
    assert len(lines) == 1, p.stdout.decode()
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["steps"] == 1
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["value"] == line["value"]
