"""Host side of bench.py's multi-GPU mode (replicas): two gloo ranks on the CPU.

Requests are independent, so N GPUs run N replicas with no collective on the
data path; the only collectives are the timing ones: a barrier around the timed
region, the max over ranks of the elapsed time and the sum over ranks of the
verified positions.  value = sum of positions / max of times.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench
import workloads


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ["CUDA_VISIBLE_DEVICES"] = ""  # gloo on the CPU, also on a GPU machine
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world),
                      RANK=str(rank), LOCAL_RANK=str(rank))
    w, r, local = bench.dist_setup(world)
    assert (w, r, local) == (world, rank, rank)
    bench.barrier(w)
    t = 1.0 + 0.5 * rank            # this rank's timed seconds
    pos = 100 * (rank + 1)          # this rank's verified positions
    t_max = bench.max_over_ranks(t, w)
    all_pos = bench.sum_over_ranks(pos, w)
    # each rank draws its own batch (seeded by rank): replicas, not copies
    inp = workloads.make_inputs(1, rep=rank, device="cpu", B=2, K=2, V=64)
    tok = inp["tokens"].flatten().tolist()
    with open(os.path.join(out_dir, "rank%d.txt" % rank), "w") as f:
        f.write("%r %r %s\n" % (t_max, all_pos, " ".join(map(str, tok))))
    import torch.distributed as dist
    dist.destroy_process_group()


def test_two_gloo_ranks_timing_collectives(tmp_path):
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, str(tmp_path)))
             for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
    for p in procs:
        if p.is_alive():
            p.kill()
            pytest.fail("a gloo rank did not finish")
        assert p.exitcode == 0
    lines = [open(tmp_path / ("rank%d.txt" % r)).read().split() for r in range(world)]
    for ln in lines:
        assert float(ln[0]) == 1.5          # max over ranks of 1.0, 1.5
        assert float(ln[1]) == 300.0        # 100 + 200
    assert lines[0][2:] != lines[1][2:]     # different batches per rank
    # whole-job throughput as bench reports it
    assert 300.0 / 1.5 == 200.0


def test_logit_copies_cover_twice_l2():
    l2 = 126 << 20
    for alg in (1 << 20, 165_306_368, 723_876_864, 3_088_711_680):
        n = bench.logit_copies(alg, l2)
        assert n >= 2
        assert (n - 1) * alg >= 2 * l2      # bytes read between two uses of a copy
        assert n == 2 or (n - 2) * alg < 2 * l2  # and no more copies than needed


def test_early_exit_bytes():
    import torch
    T = torch.tensor([1.0, 0.0, 0.7, 0.5])          # sampled, greedy, sampled, sampled
    L = torch.tensor([4, 4, 1, 4], dtype=torch.int32)
    a = torch.tensor([3, 4, 1, 0], dtype=torch.int32)
    K, V, s = 4, 10, 2
    # one wave: each needed row once
    assert bench.early_exit_bytes(T, L, a, K, V, s, K) == workloads.algorithmic_bytes(T, L, V, s)
    # W = 2: wave 1 target 0..1 (+ draft 0..1 when sampled); request 2 (L = 1) ends in it
    # with target 0..1 and draft 0; requests 0 and 1 stay open (a >= 2) and read target
    # 2..4 (+ draft 2..3): 4 + 5, 2 + 3, 3, 4 rows
    assert bench.early_exit_bytes(T, L, a, K, V, s, 2) == (9 + 5 + 3 + 4) * V * s
