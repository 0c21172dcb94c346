"""Host-side logic of bench.py on CPU: the multi-process replica path (gloo,
world size 2) and the algorithmic byte counts behind its roofline fractions.

The decode path shards by sequence with no exchange between GPUs, so N GPUs
run N replicas: each rank times its own steps, the job takes the slowest
rank's time (max over ranks after a barrier) and reports the tokens of all
ranks over it.  The reference arm runs on rank 0 only; the other ranks exit
without work.  These tests run those pieces as two gloo processes."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_env(rank, world, port):
    return {"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "RANK": str(rank),
            "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank)}


def _replica(rank, world, port, per_rank_ms, out):
    os.environ.update(_rank_env(rank, world, port))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    r, w, local = bench.dist_env()
    bench.dist_init(w, "gloo")
    bench.barrier()
    ms = bench.max_over_ranks(per_rank_ms[r])
    value = bench.job_value(w, 32, 100, ms)
    bench.barrier()
    out.put((r, w, local, ms, value))
    dist.destroy_process_group()


def test_replicas_take_the_slowest_rank_and_count_every_rank():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    per_rank_ms = [40.0, 55.0]
    procs = [ctx.Process(target=_replica, args=(r, 2, port, per_rank_ms, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[0] for r in res] == [0, 1] and all(r[1] == 2 and r[2] == r[0] for r in res)
    for _, _, _, ms, value in res:
        assert ms == 55.0                                  # the slowest rank's time, on every rank
        assert value == pytest.approx(2 * 32 * 100 / 0.055)  # both ranks' tokens over it


def test_single_process_is_the_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(12.5) == 12.5
    assert bench.job_value(1, 32, 2048, 70.0) == pytest.approx(32 * 2048 / 0.070)


def test_reference_arm_runs_on_rank_zero_only():
    # bench.py --impl reference under a 2-rank launch: rank 1 exits 0 and prints
    # nothing; rank 0 prints one JSON line marked impl=reference
    port = _free_port()
    outs = []
    procs = []
    for r in range(2):
        env = dict(os.environ, **_rank_env(r, 2, port))
        procs.append(subprocess.Popen([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                                       "--gpus", "2", "--steps", "1", "--warmup", "0"], cwd=ROOT, env=env,
                                      stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True))
    for p in procs:
        o, e = p.communicate(timeout=600)
        assert p.returncode == 0, e[-2000:]
        outs.append(o.strip())
    assert outs[1] == ""
    line = json.loads(outs[0].splitlines()[-1])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["e2e"]["h2d_bytes_per_step"] == 0


def test_algorithmic_bytes_match_the_scope_table():
    # bench.py's per-layer-step byte count (indexer + attention) against totals
    # worked out by hand from the entry sizes (132-byte indexer rows, 648-byte
    # compressed rows, 1152-byte window rows, q, output, indices and tables):
    # C4A 32K batch 32 54.83 MB, C128A 128K batch 64 39.72 MB (attention only),
    # C4A 1M batch 4 145.65 MB; they differ only in how table bytes are rounded
    sys.path.insert(0, ROOT)
    import bench
    w = bench.WORKLOADS
    ab = bench.algorithmic_bytes(w["c4a_32k_b32"], 32768)
    assert ab["indexer"] + ab["mla"] == pytest.approx(54.83e6, rel=2e-3)
    ab = bench.algorithmic_bytes(w["c128a_128k_b64"], 131072)
    assert ab["indexer"] == 0 and ab["mla"] == pytest.approx(39.72e6, rel=5e-3)
    ab = bench.algorithmic_bytes(w["c4a_1m_b4"], 1048576)
    assert ab["indexer"] + ab["mla"] == pytest.approx(145.65e6, rel=2e-3)


def test_reference_arm_names_what_it_cannot_time():
    # the reference arm times the headline workload only; for the others it
    # prints one line saying so and exits 0
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload",
                        "c128a_128k_b64"], cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and "headline" in line["unavailable"]
