"""Host logic of bench.py that needs no GPU: the N>1 aggregation (max of the
step time over ranks, sum of tokens over ranks) on two gloo ranks, the
per-rank workload seeds of the weak-scaling run, and the algorithmic work
counts."""
import os
import socket

import pytest
import torch
import torch.multiprocessing as mp

import synth


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    bench.init_dist(world, "gloo")
    w, r, _ = bench.dist_env()
    step_ms = 10.0 + 5.0 * r            # rank 1 is the slow one
    mx = bench.reduce_max(step_ms, w, "cpu")
    tok = bench.reduce_sum(1000.0 + r, w, "cpu")
    cfg = bench.rank_config(synth.config_by_name("uniform_t4096_h4096"), r)
    bench.barrier(w)
    q.put((r, mx, tok, cfg.seed))
    torch.distributed.destroy_process_group()


def test_two_gloo_ranks_aggregate():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [o[1] for o in out] == [15.0, 15.0]
    assert [o[2] for o in out] == [2001.0, 2001.0]
    assert out[0][3] != out[1][3], "each rank draws its own batch"


def test_algorithmic_work_counts():
    import bench
    cfg = synth.config_by_name("zipf_t16384_h7168")
    w = bench.algorithmic_work(cfg, P=1000, M_pad=1280, nv=130)
    H, I = cfg.H, cfg.I
    assert w["gemm1"] == 2.0 * 1000 * 2 * I * H
    assert w["gemm2"] == 2.0 * 1000 * H * I
    assert w["combine"] == 2 * 1000 * H + 2 * 130 * H + 4 * 130 * cfg.K
    assert w["scatter"] == 130 * (H + (H // 128) * 4) + 4 * 130 * cfg.K + 1280 * (H + (H // 128) * 4 + 4)
    assert w["act_quant"] == 1280 * (4 * I + I + (I // 128) * 4)


def test_reference_arm_other_ranks_do_nothing():
    import bench
    res, rank = bench.run_reference(bench.parse_args(["--impl", "reference"]), 2, 1)
    assert res is None and rank == 1


def test_launches_per_step():
    """The gpu_launches claim: kernels one step launches in each mode."""
    import argparse
    import bench
    a = lambda **kw: argparse.Namespace(**{"fuse_layout_scatter": False, "masked_max_m": 0, **kw})  # noqa: E731
    big = synth.config_by_name("zipf_t16384_h7168")
    dec = synth.config_by_name("decode_t256_h7168_ue8m0")
    # layout 2 + scatter + gate_up(+act+quant) + down + combine
    assert bench.launches_per_step(a(), big, True) == 6
    assert bench.launches_per_step(a(), big, False) == 7            # + stand-alone act_quant
    assert bench.launches_per_step(a(masked_max_m=1152), big, True) == 8  # + two slab bridges
    assert bench.launches_per_step(a(fuse_layout_scatter=True), big, True) == 5
    # 256 x 8 pairs fit one 2048-pair chunk: the layout is one launch
    assert bench.launches_per_step(a(), dec, True) == 5
    assert bench.launches_per_step(a(fuse_layout_scatter=True), dec, True) == 5


def test_oracle_sample_on_a_thread_pool_matches_one_thread():
    """The all-cores CPU baseline runs the oracle's per-token path on a
    thread pool; the rows it returns are the single-threaded ones."""
    import bench
    cfg = synth.config_by_name("tiny_h512")
    d = synth.generate(cfg)
    toks = list(range(12))
    n1, _, y1 = bench._oracle_sample(cfg, d, 600.0, t_list=toks)
    n2, _, y2 = bench._oracle_sample(cfg, d, 600.0, t_list=toks, threads=4)
    assert n1 == n2 == len(toks)
    assert all((y1[t] == y2[t]).all() for t in toks)
