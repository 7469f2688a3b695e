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
    """The gpu_launches claim: kernels one step launches in each mode, on a
    152-SM GPU."""
    import argparse
    import bench
    a = lambda **kw: argparse.Namespace(**{"fuse_layout_scatter": True, "masked_max_m": 0, **kw})  # noqa: E731
    big = synth.config_by_name("zipf_t16384_h7168")
    dec = synth.config_by_name("decode_t256_h7168_ue8m0")
    pad = synth.config_by_name("padded_t32768_valid6000_h4096")
    sms = 152
    # fused layout+scatter (one cooperative launch) + gate_up(+act+quant) + down + combine
    assert bench.launches_per_step(a(), big, True, sms) == 4
    assert bench.launches_per_step(a(), pad, True, sms) == 4       # 128 chunks <= 2 x 152
    assert bench.launches_per_step(a(), big, False, sms) == 5      # + stand-alone act_quant
    assert bench.launches_per_step(a(masked_max_m=1152), big, True, sms) == 6  # + two slab bridges
    # two calls: one cooperative layout launch + the scatter
    assert bench.launches_per_step(a(fuse_layout_scatter=False), big, True, sms) == 5
    # 256 x 8 pairs fit one 2048-pair chunk: one-block layout + scatter either way
    assert bench.launches_per_step(a(), dec, True, sms) == 5
    assert bench.launches_per_step(a(fuse_layout_scatter=False), dec, True, sms) == 5


def test_front_launches_fall_back_past_the_cooperative_grid():
    """More chunks than the cooperative grid holds: the fused call becomes
    the two calls, and past three blocks per SM the layout takes two
    launches."""
    import bench
    sms = 152
    T, K, E, H = 2048 * 2 * sms // 8, 8, 32, 4096  # exactly 2 blocks per SM of chunks
    assert bench.front_launches(T, K, E, H, True, sms) == 1
    assert bench.front_launches(T + 256, K, E, H, True, sms) == 2   # layout coop + scatter
    T3 = 2048 * 3 * sms // 8
    assert bench.front_launches(T3, K, E, H, False, sms) == 2
    assert bench.front_launches(T3 + 256, K, E, H, False, sms) == 3  # count + rank + scatter
    assert bench.front_launches(T3 + 256, K, E, H, True, sms) == 3
    # shared memory limits the blocks per SM for very many experts
    assert bench.coop_blocks_per_sm(32, False) == 3 and bench.coop_blocks_per_sm(32, True) == 2
    assert bench.coop_blocks_per_sm(1024, False) == 2


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


def test_gate_up_traffic_ratio_inputs():
    """The stored per-byte DRAM ratios divide by gate_up_alg_bytes of the
    captured workloads (rows and experts as the layout gives them)."""
    import bench
    import oracle as orc
    for name, scale in (("uniform_t4096_h4096", "f32"), ("ue8m0_t2048_e16_h7168", "ue8m0")):
        cfg = synth.config_by_name(name)
        inp = orc.to_numpy_inputs(synth.generate(cfg))
        M_cap = orc.expanded_capacity(cfg.T * cfg.K, cfg.E, cfg.align)
        rl = orc.layout(inp["topk_ids"], cfg.E, cfg.align, inp["n_valid"], M_cap)
        ne = int(((rl["psum"] - rl["start"]) > 0).sum())
        alg = bench.gate_up_alg_bytes(cfg, int(rl["total"]), ne)
        assert cfg.scale_mode == scale
        assert 0.98 < bench.GATE_UP_DRAM_PER_ALG[scale] < 1.02
        assert alg in (604962816, 631476224)


def test_variant_lines_name_real_workloads_and_arguments():
    """Every variant line runs a known workload with argument overrides the
    bench parser defines."""
    import bench
    args = vars(bench.parse_args([]))
    for name, workload, over, _graph in bench.VARIANTS:
        synth.config_by_name(workload)
        assert set(over) <= set(args), (name, over)
