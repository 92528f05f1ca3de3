"""Multi-rank host logic of bench.py on CPU: world_size 2 over gloo.

The reduction does not shard: with N GPUs every rank reduces its own band
(replicas, no collective on the data path), and the reported value is all
ranks' bytes over the slowest rank's time.  These tests run the rank
bookkeeping, the replica seeds and the max/sum aggregation as two gloo
processes, each reducing its replica with the oracle (small band), and
check the `--impl reference` arm's rank > 0 early exit.
"""
import json
import os
import socket
import sys

import numpy as np
import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, outdir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    import band_inputs as bi
    import oracle
    r, wsz, local = bench.dist_env()
    dist.init_process_group("gloo", rank=r, world_size=wsz)
    w = bi.by_name("n256_bw8_tw7_f64")
    band = bi.make_band(w.n, w.bw, w.tw, w.dtype, w.dist, w.graded, bench.replica_seed(w, r))
    d, e = oracle.bidiagonal(band, w.n, w.bw, w.tw)
    ms = 10.0 + 5.0 * r            # per-rank time
    units = 1000.0 * (r + 1)       # per-rank bytes
    ms_max, units_sum = bench.aggregate(ms, units)
    dist.barrier()
    with open(os.path.join(outdir, f"rank{r}.json"), "w") as f:
        json.dump({"rank": r, "world": wsz, "local": local, "ms_max": ms_max, "units": units_sum,
                   "d0": float(d[0]), "sig": float(np.abs(d).sum() + np.abs(e).sum())}, f)
    dist.destroy_process_group()


def test_two_rank_replicas_aggregate(tmp_path):
    from oracle import build as build_oracle
    build_oracle()
    port = _free_port()
    mp.start_processes(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, join=True,
                       start_method="spawn")
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(2)]
    for r, x in enumerate(res):
        assert x["rank"] == r and x["world"] == 2 and x["local"] == r
        assert x["ms_max"] == pytest.approx(15.0)      # slowest rank's time
        assert x["units"] == pytest.approx(3000.0)     # all ranks' bytes
    # each replica reduced its own matrix
    assert res[0]["d0"] != res[1]["d0"] and res[0]["sig"] != res[1]["sig"]


def test_replica_seeds_distinct():
    import bench
    import band_inputs as bi
    for w in bi.WORKLOADS:
        seeds = {bench.replica_seed(w, r) for r in range(8)}
        assert len(seeds) == 8
        assert bench.replica_seed(w, 0) == w.seed


def test_aggregate_single_process_passthrough():
    import bench
    assert bench.aggregate(3.5, 42.0) == (3.5, 42.0)


def test_reference_arm_nonzero_rank_exits_without_work(monkeypatch, capsys):
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("LOCAL_RANK", "1")
    monkeypatch.setattr(sys, "argv", ["bench.py", "--impl", "reference", "--gpus", "2"])
    assert bench.main() == 0
    assert capsys.readouterr().out == ""
