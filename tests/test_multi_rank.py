"""Host side of the multi-process bench path, on CPU with gloo ranks.

Sequences are independent, so N GPUs run N replicas with no collective on
the data path; the only cross-rank steps are the barrier around the timed
region and the max-over-ranks of the elapsed time.  These run here as
world-size-2 gloo process groups on 127.0.0.1."""

import json
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out_dir):
    sys.path.insert(0, ROOT)
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dist.barrier()
        # rank r measured (r + 1) * 10 ms over 5 steps of 100 rows each
        ms = bench.max_over_ranks(dist, 10.0 * (rank + 1), torch.device("cpu"))
        rate = bench.job_rate(100, 5, world, ms)
        with open(os.path.join(out_dir, f"r{rank}.json"), "w") as f:
            json.dump({"ms": ms, "rate": rate}, f)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_job_rate_gloo(tmp_path):
    world = 2
    mp.spawn(_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world,
             join=True)
    got = [json.load(open(tmp_path / f"r{r}.json")) for r in range(world)]
    for g in got:
        assert g["ms"] == 20.0           # the slowest rank's time, on all ranks
        # 100 rows x 5 steps on each of 2 ranks in 20 ms
        assert g["rate"] == pytest.approx(100 * 5 * 2 / 0.020)


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(None, 3.5, None) == 3.5
    assert bench.job_rate(10, 4, 1, 2.0) == pytest.approx(20000.0)


def test_reference_arm_only_rank0_reports(capsys):
    sys.path.insert(0, ROOT)
    import bench

    class A:
        steps, warmup, workload = 1, 0, "chain_sample"
    assert bench.reference_arm(A(), 2, 1) is None
    assert capsys.readouterr().out == ""


def _records_worker(rank, world, port, out_dir):
    """Each rank records its own share of the rounds (oracle side), then
    the records are summed across ranks with an all-reduce."""
    sys.path.insert(0, ROOT)
    from oracle import stats
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        count, parent, path, conf, n, nb = _rounds_for_records()
        mine = slice(rank, None, world)           # rounds split over ranks
        st = stats.accept_stats(count[mine], parent[mine], path[mine],
                                conf[mine], n, nb)
        out = {}
        for f in ("len_hist", "node_tested", "node_accepted", "depth_tested",
                  "depth_accepted", "calib_tested", "calib_accepted"):
            t = torch.from_numpy(getattr(st, f).copy())
            dist.all_reduce(t)
            out[f] = t.tolist()
        t = torch.tensor([st.invalid], dtype=torch.int64)
        dist.all_reduce(t)
        out["invalid"] = int(t.item())
        with open(os.path.join(out_dir, f"rec{rank}.json"), "w") as fh:
            json.dump(out, fh)
    finally:
        dist.destroy_process_group()


def _rounds_for_records():
    import numpy as np
    rng = np.random.default_rng(5)
    B, n, nb = 41, 12, 6
    parent = np.array([[-1 if j == 0 or rng.random() < 0.3 else
                        int(rng.integers(0, j)) for j in range(n)]
                       for _ in range(B)], dtype=np.int32)
    count = np.zeros(B, dtype=np.int32)
    path = np.full((B, n), -1, dtype=np.int32)
    for b in range(B):
        j, chain = int(rng.integers(0, n)), []
        while j >= 0:
            chain.append(j)
            j = int(parent[b, j])
        count[b] = len(chain)
        path[b, :len(chain)] = chain[::-1]
    count[3] = n + 2                                # one invalid round
    conf = rng.random((B, n)).astype(np.float32)
    return count, parent, path, conf, n, nb


def test_acceptance_records_of_replicas_add_up_gloo(tmp_path):
    # replicas verify disjoint rounds; their acceptance records combine by a
    # sum (all-reduce) into exactly the records of all rounds together
    sys.path.insert(0, ROOT)
    from oracle import stats
    world = 2
    mp.spawn(_records_worker, args=(world, _free_port(), str(tmp_path)),
             nprocs=world, join=True)
    count, parent, path, conf, n, nb = _rounds_for_records()
    whole = stats.accept_stats(count, parent, path, conf, n, nb)
    for r in range(world):
        got = json.load(open(tmp_path / f"rec{r}.json"))
        for f, v in got.items():
            want = whole.invalid if f == "invalid" else getattr(whole, f).tolist()
            assert v == want, f


def _bench(args, env=None, timeout=240):
    import subprocess
    e = dict(os.environ)
    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK", "MASTER_ADDR",
              "MASTER_PORT"):
        e.pop(k, None)
    e.update(env or {})
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"),
                           *args], capture_output=True, text=True, env=e,
                          timeout=timeout, cwd=ROOT)


def test_bench_gpus_flag_launches_its_ranks():
    # outside torchrun, --gpus 2 launches two local ranks itself (the
    # reference arm runs on the host cores, so this needs no GPU); rank 0
    # prints the one line and reports both ranks
    r = _bench(["--gpus", "2", "--impl", "reference", "--workload",
                "chain_sample", "--steps", "1", "--warmup", "0",
                "--cpu-seconds", "0.3"])
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2
    assert d["config"]["workload"] == "chain_sample"


def test_bench_refuses_gpus_that_differ_from_world_size():
    r = _bench(["--gpus", "1", "--impl", "reference", "--workload",
                "chain_sample"], env={"WORLD_SIZE": "2", "RANK": "0",
                                      "LOCAL_RANK": "0"})
    assert r.returncode != 0
    assert "WORLD_SIZE" in (r.stderr + r.stdout)
