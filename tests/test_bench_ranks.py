"""Host logic of the multi-GPU bench (CPU, gloo): the slowest replica's time
is what every rank reports, the reference arm runs on rank 0 only, and a
multi-stream round split by stream covers every stream once and gathers the
same results a single rank computes.

Batch-1 drafting does not shard across GPUs without a collective the method
does not have, so several GPUs run replicas; multi-stream rounds split their
streams into contiguous groups, one per rank. These tests cover the rank
handling with two gloo processes instead of GPUs."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, values, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench

    torch.distributed.init_process_group("gloo", rank=rank, world_size=world)
    got = bench.max_over_ranks(values[rank], world, "cpu")
    torch.distributed.barrier()
    torch.distributed.destroy_process_group()
    with open(os.path.join(out_dir, f"r{rank}.json"), "w") as f:
        json.dump(got, f)


def test_max_over_ranks_gloo(tmp_path):
    values = [3.25, 7.5]
    mp.start_processes(_rank_main, args=(2, _free_port(), values, str(tmp_path)), nprocs=2, start_method="spawn")
    for r in range(2):
        with open(tmp_path / f"r{r}.json") as f:
            assert json.load(f) == max(values)


def test_max_over_ranks_single():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.max_over_ranks(4.0, 1, "cpu") == 4.0


def test_reference_arm_other_ranks_exit_quietly():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference"], cwd=ROOT, env=env,
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""


def test_partition_streams_covers_each_stream_once():
    sys.path.insert(0, ROOT)
    import bench

    for S in (1, 7, 8, 32, 33):
        for world in (1, 2, 3, 4, 8):
            ranges = [bench.partition_streams(S, world, r) for r in range(world)]
            assert ranges[0][0] == 0 and ranges[-1][1] == S
            assert all(a[1] == b[0] for a, b in zip(ranges, ranges[1:]))  # contiguous, in rank order
            sizes = [hi - lo for lo, hi in ranges]
            assert max(sizes) - min(sizes) <= 1 and sum(sizes) == S


def _split_round(S, V, lo, hi, seed):
    """One round of streams [lo, hi) on the host: a stand-in drafter returns
    fixed ids per stream, the target logits are planted to accept a seeded
    length, and the oracle's greedy rule verifies."""
    import oracle as O
    import synthetic_inputs as SI

    ids = torch.tensor([[(97 * s + 13 * i + 5) % (V - 1) for i in range(15)] for s in range(S)], dtype=torch.int32)
    tl = SI.make_logits((S, 16, V), 2.0, seed)
    lengths = SI.make_accept_lengths(S, seed + 1)
    SI.plant_accepts(tl, ids, lengths)
    acc, toks = [], []
    for s in range(lo, hi):
        a, t = O.greedy_verify(ids[s].tolist(), O.to_f64(tl[s]))
        acc.append(a)
        toks.append(t)
    return acc, toks, [min(L, 15) for L in lengths]


def _split_rank_main(rank, world, port, S, V, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench

    torch.distributed.init_process_group("gloo", rank=rank, world_size=world)
    lo, hi = bench.partition_streams(S, world, rank)
    acc, toks, _ = _split_round(S, V, lo, hi, 11)
    got = bench.gather_streams(lo, acc, toks, world)
    torch.distributed.barrier()
    torch.distributed.destroy_process_group()
    with open(os.path.join(out_dir, f"split{rank}.json"), "w") as f:
        json.dump({"range": [lo, hi], "got": got}, f)


def test_stream_split_gather_gloo(tmp_path):
    """Two ranks each verify their contiguous half of a 7-stream round; rank 0
    gathers accept lengths and tokens in stream order, equal to one rank
    verifying all seven, and the planted accept lengths are recovered."""
    sys.path.insert(0, ROOT)
    import bench

    S, V = 7, 96
    mp.start_processes(_split_rank_main, args=(2, _free_port(), S, V, str(tmp_path)), nprocs=2,
                       start_method="spawn")
    with open(tmp_path / "split0.json") as f:
        r0 = json.load(f)
    with open(tmp_path / "split1.json") as f:
        r1 = json.load(f)
    assert r1["got"] is None and r0["range"][1] == r1["range"][0]
    acc, toks, planted = _split_round(S, V, 0, S, 11)
    assert bench.gather_streams(0, acc, toks, 1) == (acc, toks)
    assert r0["got"] == [acc, toks]
    assert acc == planted
