"""Benchmark of the expanded-layout MoE prefill layer on GB300.

One step = one pass of the whole layer (layout, expand-scatter, gate_up GEMM,
silu*mul + fp8 quant with the weight fold, down GEMM, combine) over one batch
of the Zipf-routed T=16384, H=7168, I=2048, E=32, top-8 workload (the
configuration the layer's targets are stated on), inputs resident in HBM.

Prints one JSON line. ``value`` is whole-job tokens/s (valid tokens of all
ranks / max-over-ranks median step time; ``ms_per_step`` is that median and
``ms_per_step_mean`` the mean); ``roofline`` is for the dominant kernel (the
gate_up GEMM) from CUDA events around its launches in the timed region;
``graph_replay`` times the same forward as one CUDA graph per step; ``e2e``
is the same metric through the package's HostPipeline with each step's
valid input rows copied from pinned host memory and its output rows copied
back; ``cpu_baseline`` is the CPU oracle on a sample of the same workload,
single-threaded and (``all_cores``) on a thread pool over the host cores;
``per_config`` holds the median step time and per-kernel split of the other
four workloads, measured in the same process after the headline one.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

import synth  # noqa: E402

METRIC = "MoE prefill layer tokens/s; scatter+combine HBM GB/s; grouped FP8 TFLOP/s"
WORKLOAD = synth.config_by_name("zipf_t16384_h7168")
L2_FLUSH_BYTES = 256 << 20           # > the 126 MB L2
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
FP8_PER_BF16 = 2.0                   # nominal dense fp8 : bf16 tensor rate
# DRAM bytes (read + write) per algorithmic byte of the dominant kernel
# (gate_up with act+quant in its epilogue), each from one ncu capture on a
# workload that holds a few GB of device memory:
#   python bench.py --workload W --steps 1 --warmup 3 --no-cpu-baseline
#   --no-e2e --no-per-config --no-graph-extra --no-variants, under ncu
#   --metrics dram__bytes_read.sum,dram__bytes_write.sum,gpu__time_duration.sum
#   --clock-control none -k regex:grouped_gemm -s 6 -c 2
# fp32 scales on uniform_t4096_h4096 (34816 expanded rows, 32 experts):
# 549653760 + 51582208 bytes against 604962816 algorithmic; ue8m0 scales on
# ue8m0_t2048_e16_h7168 (the ue8m0 workload's rows per expert, a quarter of
# its experts; 17408 rows, 16 experts): 597162496 + 33378560 against
# 631476224. A launch's traffic is reported as the ratio
# times its own algorithmic bytes (gate_up_alg_bytes). Update whenever that
# kernel changes.
GATE_UP_DRAM_PER_ALG = {
    "f32": (549653760 + 51582208) / 604962816,
    "ue8m0": (597162496 + 33378560) / 631476224,
}
GATE_UP_DRAM_SOURCE = ("ncu dram__bytes_read+write per algorithmic byte on uniform_t4096_h4096 "
                       "(fp32) / ue8m0_t2048_e16_h7168 (ue8m0), times this launch's bytes")


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=WORKLOAD.name)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--cpu-sample-seconds", type=float, default=15.0)
    ap.add_argument("--weighting", choices=["expanded", "gather"], default="expanded",
                    help="expanded: fold / output-row weighting (do_expand=True); gather: "
                         "weights applied in the combine (the do_expand=False A/B arrangement)")
    ap.add_argument("--masked-max-m", type=int, default=0,
                    help="decode variant: both GEMMs on per-expert slabs of this height")
    ap.add_argument("--graph", action="store_true",
                    help="time replays of a CUDA graph of the whole forward (no per-kernel split)")
    ap.add_argument("--fuse-layout-scatter", action=argparse.BooleanOptionalAction, default=True,
                    help="layout and expand-scatter as one moe_expand_layout_scatter call "
                         "(one cooperative launch); --no-fuse-layout-scatter: two calls")
    ap.add_argument("--unfused", action="store_true",
                    help="run gate_up and act+quant as two launches")
    ap.add_argument("--gemm-tile-n128", action="store_true",
                    help="force 128-column GEMM tiles (tuning comparison)")
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip the per-workload lines of the other four workloads")
    ap.add_argument("--per-config-steps", type=int, default=10)
    ap.add_argument("--no-variants", action="store_true",
                    help="skip the variant lines (gather weighting, masked slab, decode batch, "
                         "the layout and scatter as two calls)")
    ap.add_argument("--no-graph-extra", action="store_true",
                    help="skip the CUDA-graph replay timing added beside the eager step time")
    return ap.parse_args(argv)


# ------------------------------------------------------------------ ranks

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world: int, backend: str):
    if world > 1 and not torch.distributed.is_initialized():
        torch.distributed.init_process_group(backend=backend)


def barrier(world):
    if world > 1:
        torch.distributed.barrier()


def reduce_max(value: float, world: int, device) -> float:
    if world == 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def reduce_sum(value: float, world: int, device) -> float:
    if world == 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.SUM)
    return float(t.item())


def rank_config(cfg: synth.LayerConfig, rank: int) -> synth.LayerConfig:
    """Weak scaling: every rank gets its own batch of the same shape."""
    import dataclasses
    return dataclasses.replace(cfg, seed=cfg.seed + 1000 * rank) if rank else cfg


# ------------------------------------------------------------------ helpers

def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """nvidia-smi clock and throttle-reason samples while the timed region runs."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        self.device_index = device_index

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.device_index}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]
        return False

    def summary(self):
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in getattr(self, "lines", []):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


def gate_up_alg_bytes(cfg, M_pad: int, n_experts: int) -> int:
    """Bytes the gate_up launch (act+quant in its epilogue) must move: the
    expanded rows' codes and scales and the non-empty experts' W13 and its
    128x128 block scales read; the fp8 intermediate and its scales written."""
    H, I = cfg.H, cfg.I
    GH, GI = H // 128, I // 128
    if cfg.scale_mode == "f32":
        a_s, o_s, w_s = 4 * GH, 4 * GI, 4
    else:
        a_s, o_s, w_s = 4 * ((GH + 3) // 4), 4 * ((GI + 3) // 4), 1
    read = M_pad * (H + a_s) + n_experts * (2 * I * H + (2 * I // 128) * GH * w_s)
    return read + M_pad * (I + o_s)


def algorithmic_work(cfg, P: int, M_pad: int, nv: int):
    """Bytes or flops each step must move or compute (valid work only)."""
    H, I, K = cfg.H, cfg.I, cfg.K
    GH, GI = H // 128, I // 128
    sbytes = 4 if cfg.scale_mode == "f32" else 1
    M_cap_rows = M_pad
    return {
        "layout": 4 * cfg.T * K * 2 + 4 * M_cap_rows,
        "scatter": nv * (H + GH * sbytes) + 4 * nv * K + M_pad * (H + GH * sbytes + 4),
        "gemm1": 2.0 * P * (2 * I) * H,
        "act_quant": M_pad * (2 * 2 * I + I + GI * sbytes),
        "gemm2": 2.0 * P * H * I,
        "combine": 2 * P * H + 2 * nv * H + 4 * nv * K,
    }


# ------------------------------------------------------------------ our arm

def coop_blocks_per_sm(E: int, scatter: bool) -> int:
    """Resident blocks per SM of the cooperative layout kernel: 3 (40
    registers x 512 threads), 2 for the variant fused with the scatter (64
    registers), fewer when its 19*E ints of shared memory per block do not
    fit the SM's 228 KB (1 KB reserved per block)."""
    by_smem = (228 * 1024) // (19 * 4 * E + 1024 + 64)
    return max(0, min(2 if scatter else 3, by_smem))


def front_launches(T: int, K: int, E: int, H: int, fuse: bool, sms: int) -> int:
    """Kernels the layout and the expand-scatter launch. moe_expand_layout:
    1 (one block when all pairs fit one 2048-pair chunk; one cooperative
    launch when the grid holds every chunk), else 2. The scatter: 1. The
    fused call: 1 cooperative launch for 2+ chunks when its grid holds
    every chunk and the copy's 32-bit work counter suffices, else the two
    calls."""
    nb = max(1, -(-T * K // 2048))
    layout = 1 if nb == 1 or nb <= coop_blocks_per_sm(E, False) * sms else 2
    if fuse and nb > 1:
        cap = coop_blocks_per_sm(E, True) * sms
        nseg = -(-(H // 16) // 64)
        if nb <= cap and T * nseg + cap * 16 * 4 <= 2**32 - 1:
            return 1
    return layout + 1


def launches_per_step(args, cfg, fused: bool, sms: int) -> int:
    """Kernels one step launches: layout + scatter (front_launches); gate_up
    (with act+quant when fused, else + act_quant 1); down 1 (the masked slab
    adds its two bridges); combine 1."""
    front = front_launches(cfg.T, cfg.K, cfg.E, cfg.H, args.fuse_layout_scatter, sms)
    ffn = 4 if args.masked_max_m else (2 if fused else 3)
    return front + ffn + 1


KERNEL_NAMES = ["layout", "scatter", "gemm1", "act_quant", "gemm2", "combine"]


def make_step(args, cfg, layer, d, n_valid, mx, L, stream):
    """One layer pass as direct C-ABI calls on `stream`; step(ev) records
    events ev[0..6] around the six stages when given. Returns (step, fused)."""
    s = stream.cuda_stream
    lay = layer.lay
    ptr = lambda t: None if t is None else t.data_ptr()  # noqa: E731
    x_q, x_s, ids, w = d["x_q"], d["x_s"], d["topk_ids"], d["topk_w"]
    gflags = mx.MOE_GEMM_TILE_N128 if args.gemm_tile_n128 else 0
    # gate_up carries silu*mul, the quantiser and the fold in its epilogue
    fused = not args.unfused and gflags == 0

    def step(ev=None):
        def mark(i):
            if ev is not None:
                ev[i].record(stream)
        mark(0)
        if args.fuse_layout_scatter:
            # both in one call: its time is booked to "scatter"
            mark(1)
            mx.check(L.moe_expand_layout_scatter(
                ptr(ids), ptr(w), ptr(x_q), ptr(x_s), layer.sl, x_s.shape[1], cfg.T, cfg.H, cfg.K,
                cfg.E, cfg.align, ptr(n_valid), layer.M_cap, ptr(lay.psum), ptr(lay.start),
                ptr(lay.total), ptr(lay.m_indices), ptr(lay.src2dst), ptr(lay.tile_prefix),
                ptr(layer.xe), ptr(layer.xe_scale), layer.xe_scale.shape[1], ptr(layer.row_w),
                ptr(layer.ws), layer.ws.numel(), ptr(layer.status), s), "layout+scatter")
            mark(2)
        else:
            mx.check(L.moe_expand_layout(ptr(ids), cfg.T, cfg.K, cfg.E, cfg.align, ptr(n_valid),
                                         layer.M_cap, ptr(lay.psum), ptr(lay.start), ptr(lay.total),
                                         ptr(lay.m_indices), ptr(lay.src2dst), ptr(lay.tile_prefix),
                                         ptr(layer.ws), layer.ws.numel(), ptr(layer.status), s),
                     "layout")
            mark(1)
            mx.check(L.moe_expand_scatter(ptr(x_q), ptr(x_s), layer.sl, x_s.shape[1], ptr(w),
                                          ptr(lay.src2dst), ptr(lay.psum), ptr(lay.start),
                                          ptr(n_valid), cfg.T, cfg.H, cfg.K, cfg.E, cfg.align,
                                          layer.M_cap, ptr(layer.xe), ptr(layer.xe_scale),
                                          layer.xe_scale.shape[1], ptr(layer.row_w),
                                          ptr(layer.status), s), "scatter")
            mark(2)
        if layer.masked_max_m is not None:
            # decode variant: slab in, fused gate_up on the slab (segment
            # gemm1), down on the slab and back to expanded rows (gemm2)
            E, mm = cfg.E, layer.masked_max_m
            S = E * mm
            sll = layer.slab_lay
            mx.check(L.moe_expand_to_masked_slab(
                ptr(layer.xe), ptr(layer.xe_scale), layer.sl, layer.xe_scale.shape[1],
                ptr(lay.psum), ptr(lay.start), E, cfg.H, mm, ptr(layer.slab), ptr(layer.slab_scale),
                layer.slab_scale.shape[1], ptr(layer.masked_m), ptr(sll.start), ptr(sll.tile_prefix),
                ptr(sll.total), ptr(layer.status), s), "slab")
            mx.check(L.moe_grouped_gemm_act_quant(
                ptr(layer.slab), ptr(layer.slab_scale), layer.sl, layer.slab_scale.shape[1],
                ptr(sll.start), ptr(sll.tile_prefix), ptr(sll.total), ptr(layer.w13), ptr(layer.s13),
                None, 0, E, cfg.I, cfg.H, S, ptr(layer.slab_di), ptr(layer.slab_di_scale),
                layer.slab_di_scale.shape[1], ptr(layer.status), s), "gemm1+act_quant (slab)")
            mark(3)
            mark(4)
            mx.check(L.moe_grouped_gemm(
                ptr(layer.slab_di), ptr(layer.slab_di_scale), layer.sl, layer.slab_di_scale.shape[1],
                ptr(sll.start), ptr(sll.tile_prefix), ptr(sll.total), ptr(layer.w2), ptr(layer.s2),
                None, 0, E, cfg.H, cfg.I, S, ptr(layer.slab_out), ptr(layer.status), s),
                "gemm2 (slab)")
            mx.check(L.moe_masked_slab_to_expand(
                ptr(layer.slab_out), mm, ptr(lay.psum), ptr(lay.start), ptr(lay.total),
                ptr(layer.row_w), E, cfg.H, layer.M_cap, ptr(layer.down_out), s), "unslab")
            mark(5)
            mx.check(L.moe_combine(ptr(layer.down_out), ptr(lay.src2dst), None, ptr(n_valid), cfg.T,
                                   cfg.H, cfg.K, ptr(layer.y), s), "combine")
            mark(6)
            return
        if fused:
            mx.check(L.moe_grouped_gemm_act_quant(
                ptr(layer.xe), ptr(layer.xe_scale), layer.sl, layer.xe_scale.shape[1],
                ptr(lay.start), ptr(lay.tile_prefix), ptr(lay.total), ptr(layer.w13),
                ptr(layer.s13), ptr(layer.row_w), layer.flags & mx.MOE_FOLD_WEIGHT_INTO_SCALE,
                cfg.E, cfg.I, cfg.H, layer.M_cap, ptr(layer.down_in),
                ptr(layer.down_in_scale), layer.down_in_scale.shape[1], ptr(layer.status), s),
                "gemm1+act_quant")
            mark(3)
        else:
            mx.check(L.moe_grouped_gemm(ptr(layer.xe), ptr(layer.xe_scale), layer.sl,
                                        layer.xe_scale.shape[1], ptr(lay.start),
                                        ptr(lay.tile_prefix), ptr(lay.total), ptr(layer.w13),
                                        ptr(layer.s13), None, gflags, cfg.E, 2 * cfg.I, cfg.H,
                                        layer.M_cap, ptr(layer.gateup), ptr(layer.status), s),
                     "gemm1")
            mark(3)
            fold = layer.flags & mx.MOE_FOLD_WEIGHT_INTO_SCALE
            mx.check(L.moe_act_quant(ptr(layer.gateup), cfg.I, ptr(layer.row_w), fold, layer.sl,
                                     ptr(lay.total), layer.M_cap, ptr(layer.down_in),
                                     ptr(layer.down_in_scale), layer.down_in_scale.shape[1],
                                     ptr(layer.status), s), "act_quant")
        mark(4)
        mx.check(L.moe_grouped_gemm(ptr(layer.down_in), ptr(layer.down_in_scale), layer.sl,
                                    layer.down_in_scale.shape[1], ptr(lay.start),
                                    ptr(lay.tile_prefix), ptr(lay.total), ptr(layer.w2),
                                    ptr(layer.s2), ptr(layer.row_w),
                                    (layer.flags & mx.MOE_WEIGHT_OUTPUT_ROWS) | gflags, cfg.E, cfg.H, cfg.I,
                                    layer.M_cap, ptr(layer.down_out), ptr(layer.status), s), "gemm2")
        mark(5)
        gather_w = layer.row_w if layer.weighting == "gather" else None
        mx.check(L.moe_combine(ptr(layer.down_out), ptr(lay.src2dst), ptr(gather_w), ptr(n_valid), cfg.T,
                               cfg.H, cfg.K, ptr(layer.y), s), "combine")
        mark(6)

    return step, fused


def timed_steps(step, stream, steps: int, flush):
    """`steps` passes with L2 flushed between them (outside the events).
    Returns (per-step ms list, per-kernel ms lists)."""
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(7)] for _ in range(steps)]
    for k in range(steps):
        flush.fill_(k & 0xFF)          # evict the previous step's data from L2
        step(evs[k])
    torch.cuda.synchronize()
    per_kernel = {n: [ev[i].elapsed_time(ev[i + 1]) for ev in evs] for i, n in enumerate(KERNEL_NAMES)}
    return [ev[0].elapsed_time(ev[6]) for ev in evs], per_kernel


def n_experts(layer) -> int:
    """Experts with at least one row."""
    lay = layer.lay
    return int(((lay.psum - lay.start) > 0).sum().item())


def layer_work(layer, cfg, nv):
    lay = layer.lay
    psum = lay.psum.cpu().numpy()
    start = lay.start.cpu().numpy()
    P = int((psum - start).sum())
    M_pad = int(lay.total.item())
    return P, M_pad, algorithmic_work(cfg, P, M_pad, nv)


def kernel_split(per_kernel_ms, work, fused, args, hbm, fp8_peak):
    """Per stage: mean and median ms, achieved GB/s or TFLOP/s (from the
    mean, the average launch duration) and the fraction of the measured peak."""
    kernels = {}
    for n in KERNEL_NAMES:
        ms = statistics.mean(per_kernel_ms[n])
        med = statistics.median(per_kernel_ms[n])
        if fused and n == "act_quant":
            kernels[n] = {"ms": 0.0, "fused_into": "gemm1"}
            continue
        if args.fuse_layout_scatter and n == "layout":
            kernels[n] = {"ms": 0.0, "fused_into": "scatter"}
            continue
        w = work[n]
        if args.fuse_layout_scatter and n == "scatter":
            w = work["scatter"] + work["layout"]  # one call moves both
        if n.startswith("gemm"):
            ach = work[n] / (ms / 1e3) / 1e12
            kernels[n] = {"ms": round(ms, 4), "ms_median": round(med, 4), "achieved": round(ach, 1),
                          "unit": "TFLOP/s", "frac": round(ach / fp8_peak, 4), "work": work[n]}
        else:
            ach = w / (ms / 1e3) / 1e9
            kernels[n] = {"ms": round(ms, 4), "ms_median": round(med, 4), "achieved": round(ach, 1),
                          "unit": "GB/s", "frac": round(ach / hbm, 4), "work": w}
    return kernels


def run_workload(args, mx, L, cfg, dev, stream, flush, steps):
    """Builds the layer for one workload, warms up, times `steps` steps.
    Returns a dict of the timing plus the objects a caller may reuse."""
    d = synth.generate(cfg, device=dev)
    nv = d["n_valid"]
    n_valid = torch.tensor([nv], dtype=torch.int32, device=dev)
    layer = mx.ExpandedMoELayer(d["w13"], d["s13"], d["w2"], d["s2"], K=cfg.K, align=cfg.align,
                                scale_mode=cfg.scale_mode, max_tokens=cfg.T, weighting=args.weighting,
                                masked_max_m=args.masked_max_m or None,
                                fuse_layout_scatter=args.fuse_layout_scatter)
    step, fused = make_step(args, cfg, layer, d, n_valid, mx, L, stream)
    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    if layer.status.item() != 0:
        raise RuntimeError(f"device status {layer.status.item()} after warm-up ({cfg.name})")
    return dict(d=d, nv=nv, n_valid=n_valid, layer=layer, step=step, fused=fused)


def graph_replay_ms(layer, d, n_valid, stream, flush, steps: int):
    """Median time of one CUDA-graph replay of the whole forward (L2 flushed
    between replays, outside the events)."""
    cap = layer.capture(d["x_q"], d["x_s"], d["topk_ids"], d["topk_w"], n_valid)
    cap.replay()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    for k, (a, b) in enumerate(evs):
        flush.fill_(k & 0xFF)
        a.record(stream)
        cap.replay()
        b.record(stream)
    torch.cuda.synchronize()
    return statistics.median(a.elapsed_time(b) for a, b in evs)


def run_ours(args, world, rank, local):
    import expanded_layout_expert_gb300 as mx
    from expanded_layout_expert_gb300 import build as libbuild

    libbuild.build()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    init_dist(world, "nccl")
    cfg = rank_config(synth.config_by_name(args.workload), rank)
    L = mx.load()
    stream = torch.cuda.current_stream()
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    run = run_workload(args, mx, L, cfg, dev, stream, flush, args.steps)
    d, nv, n_valid, layer, fused = run["d"], run["nv"], run["n_valid"], run["layer"], run["fused"]
    step = run["step"]

    if args.graph:
        cap = layer.capture(d["x_q"], d["x_s"], d["topk_ids"], d["topk_w"], n_valid)
        cap.replay()
        torch.cuda.synchronize()

        def step(ev=None):  # noqa: F811  (the whole layer as one graph launch)
            if ev is not None:
                for i in range(6):
                    ev[i].record(stream)
            cap.replay()
            if ev is not None:
                ev[6].record(stream)

    barrier(world)
    torch.cuda.synchronize()
    t_wall0 = time.perf_counter()
    with ClockSampler(local) as clocks:
        step_list, per_kernel = timed_steps(step, stream, args.steps, flush)
    barrier(world)
    t_wall = time.perf_counter() - t_wall0
    if layer.status.item() != 0:
        raise RuntimeError(f"device status {layer.status.item()} in the timed region")
    step_med = statistics.median(step_list)
    step_mean = statistics.mean(step_list)

    P, M_pad, work = layer_work(layer, cfg, nv)
    step_ms_max = reduce_max(step_med, world, dev)
    tokens_all = reduce_sum(float(nv), world, dev)
    value = tokens_all / (step_ms_max / 1e3)

    peaks, peak_src = load_peaks()
    hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    fp8_peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])) * FP8_PER_BF16
    if args.graph:
        kernels = {"graph_replay": {"ms": round(step_med, 4)}}
        sc_gbs = gemm_tflops = float("nan")
        roofline = None
    else:
        kernels = kernel_split(per_kernel, work, fused, args, hbm, fp8_peak)
        pk = {n: statistics.mean(v) for n, v in per_kernel.items()}
        sc_bytes = work["scatter"] + work["combine"] + (work["layout"] if args.fuse_layout_scatter else 0)
        sc_gbs = sc_bytes / ((pk["scatter"] + pk["combine"]) / 1e3) / 1e9
        gemm_tflops = (work["gemm1"] + work["gemm2"]) / ((pk["gemm1"] + pk["gemm2"]) / 1e3) / 1e12
        roofline = {"bound": "tensor",
                    "kernel": "grouped_gemm (gate_up" + (" + act_quant epilogue)" if fused else ")"),
                    "achieved": kernels["gemm1"]["achieved"], "peak": round(fp8_peak, 1),
                    "unit": "TFLOP/s", "frac": kernels["gemm1"]["frac"],
                    "traffic": (round(GATE_UP_DRAM_PER_ALG[cfg.scale_mode] * gate_up_alg_bytes(
                        cfg, M_pad, n_experts(layer))) if fused else None),
                    "traffic_source": GATE_UP_DRAM_SOURCE if fused else None,
                    "peak_source": f"{peak_src}: bf16 burst x {FP8_PER_BF16:g} (nominal fp8:bf16)"}

    result = {
        "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": max(args.warmup, 3), "ms_per_step": round(step_ms_max, 4),
        "ms_per_step_mean": round(step_mean, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "fp8e4m3",
        "data": "synthetic (seeded generator; no dataset or trained weights)",
        "config": workload_config(cfg, nv, P, M_pad, layer, args, world),
        "scatter_combine_gbs": None if args.graph else round(sc_gbs, 1),
        "grouped_fp8_tflops": None if args.graph else round(gemm_tflops, 1),
        "kernels": kernels,
        "roofline": roofline,
        "gpu_launches": launches_per_step(
            args, cfg, fused, torch.cuda.get_device_properties(dev).multi_processor_count) * args.steps,
        "clocks": clocks.summary(),
        "wall_s_timed_region": round(t_wall, 3),
    }

    if not args.graph and not args.no_graph_extra:
        gms = graph_replay_ms(layer, d, n_valid, stream, flush, max(10, args.steps))
        result["graph_replay"] = {"ms_per_step": round(gms, 4),
                                  "tokens_per_s": round(nv / (gms / 1e3), 1),
                                  "steps": max(10, args.steps),
                                  "how": "one CUDA graph of the whole forward per step; "
                                         "median; L2 flushed between replays"}

    if not args.no_e2e:
        result["e2e"] = run_e2e(args, layer, d, dev, world)

    if rank == 0 and not args.no_cpu_baseline:
        result["cpu_baseline"], result["parity_sample"] = run_cpu_baseline(args, cfg, d, layer)

    if rank == 0 and not args.no_per_config and not args.graph:
        del run, step, layer, d
        torch.cuda.empty_cache()
        result["per_config"] = run_per_config(args, mx, L, dev, stream, flush, hbm, fp8_peak,
                                              exclude=cfg.name)
    if rank == 0 and not args.no_variants and not args.graph:
        result["variants"] = run_variants(args, mx, L, dev, stream, flush, hbm, fp8_peak)
    return result, rank


def workload_config(cfg, nv, P, M_pad, layer, args, world):
    return {"workload": cfg.name, "T": cfg.T, "n_valid": nv, "H": cfg.H, "I": cfg.I,
            "E": cfg.E, "top_k": cfg.K, "expert_alignment": cfg.align,
            "routing": (f"zipf(s={cfg.zipf_s}), {cfg.zipf_zero_experts} experts empty"
                        if cfg.routing == "zipf" else cfg.routing),
            "inactive_rows": cfg.inactive_frac, "scales": cfg.scale_mode,
            "weighting": args.weighting,
            "masked_max_m": args.masked_max_m or None,
            "cuda_graph": bool(args.graph),
            "layout_scatter": ("one call (moe_expand_layout_scatter)" if args.fuse_layout_scatter
                               else "2 calls"),
            "valid_pairs": P, "expanded_rows": M_pad, "M_cap": layer.M_cap,
            "l2": "flushed between steps (256 MiB write outside the timed events)",
            "parallelism": f"replicas x{world} (token-sharded, no collective)"}


def run_per_config(args, mx, L, dev, stream, flush, hbm, fp8_peak, exclude):
    """The other workloads, one after another in the same process: median
    step time and the per-kernel split of `--per-config-steps` steps each."""
    out = {}
    for cfg in synth.CONFIGS:
        if cfg.name == exclude:
            continue
        run = run_workload(args, mx, L, cfg, dev, stream, flush, args.per_config_steps)
        steps, per_kernel = timed_steps(run["step"], stream, args.per_config_steps, flush)
        if run["layer"].status.item() != 0:
            raise RuntimeError(f"device status {run['layer'].status.item()} ({cfg.name})")
        P, M_pad, work = layer_work(run["layer"], cfg, run["nv"])
        med = statistics.median(steps)
        out[cfg.name] = {
            "ms_per_step": round(med, 4), "ms_per_step_mean": round(statistics.mean(steps), 4),
            "tokens_per_s": round(run["nv"] / (med / 1e3), 1), "steps": args.per_config_steps,
            "n_valid": run["nv"], "valid_pairs": P, "expanded_rows": M_pad, "scales": cfg.scale_mode,
            "kernels": kernel_split(per_kernel, work, run["fused"], args, hbm, fp8_peak)}
        del run
        torch.cuda.empty_cache()
    return out


# (name, workload, argument overrides, with a graph replay)
VARIANTS = (
    ("gather_weighting", "zipf_t16384_h7168", {"weighting": "gather"}, False),
    ("layout_scatter_two_calls", "zipf_t16384_h7168", {"fuse_layout_scatter": False}, False),
    ("masked_slab_1152", "uniform_t4096_h4096", {"masked_max_m": 1152}, False),
    ("decode_batch", "decode_t256_h7168_ue8m0", {}, True),
    ("decode_batch_masked_slab_64", "decode_t256_h7168_ue8m0", {"masked_max_m": 64}, False),
)


def run_variants(args, mx, L, dev, stream, flush, hbm, fp8_peak):
    """The layer's variants, each on the workload it is meant for: median
    step time and per-kernel split of `--per-config-steps` steps (plus a
    CUDA-graph replay time for the decode batch)."""
    import argparse
    out = {}
    for name, wl, over, graph in VARIANTS:
        vargs = argparse.Namespace(**{**vars(args), **over})
        cfg = synth.config_by_name(wl)
        run = run_workload(vargs, mx, L, cfg, dev, stream, flush, args.per_config_steps)
        steps, per_kernel = timed_steps(run["step"], stream, args.per_config_steps, flush)
        if run["layer"].status.item() != 0:
            raise RuntimeError(f"device status {run['layer'].status.item()} ({name})")
        P, M_pad, work = layer_work(run["layer"], cfg, run["nv"])
        med = statistics.median(steps)
        out[name] = {"workload": wl, **{k: v for k, v in over.items()},
                     "ms_per_step": round(med, 4), "tokens_per_s": round(run["nv"] / (med / 1e3), 1),
                     "steps": args.per_config_steps,
                     "kernels": kernel_split(per_kernel, work, run["fused"], vargs, hbm, fp8_peak)}
        if graph:
            gms = graph_replay_ms(run["layer"], run["d"], run["n_valid"], stream, flush,
                                  max(10, args.per_config_steps))
            out[name]["graph_replay_ms"] = round(gms, 4)
        del run
        torch.cuda.empty_cache()
    return out


def run_e2e(args, layer, d, dev, world):
    """The same metric through the package's public API for host-resident
    batches (HostPipeline over ExpandedMoELayer.forward): every step copies its
    inputs from pinned host memory and its output y back to pinned host
    memory inside the timed region; the copies of neighbouring steps overlap
    the kernels on their own streams. The valid-row count is known on the
    host, so only the valid rows travel (the padded buffer's garbage tail
    stays where it is)."""
    nv = d["n_valid"]
    host = {k: d[k].cpu().pin_memory() for k in ("x_q", "x_s", "topk_ids", "topk_w")}
    nv_host = torch.tensor([nv], dtype=torch.int32).pin_memory()
    y_host = [torch.empty(layer.y.shape, dtype=layer.y.dtype).pin_memory() for _ in range(2)]

    def rows_bytes(t, n):
        if t.shape[0] == layer.T:                 # row-major [T, ...]
            return n * t[0].numel() * t.element_size()
        return t.shape[0] * n * t.element_size()  # column-major packed scales [W, T]
    h2d = sum(rows_bytes(t, nv) for t in host.values()) + 4
    d2h = rows_bytes(y_host[0], nv)
    import expanded_layout_expert_gb300 as mx
    pipe = mx.HostPipeline(layer)

    def one(k):
        pipe.submit(host["x_q"], host["x_s"], host["topk_ids"], host["topk_w"], nv_host,
                    y_host[k % 2], n_rows=nv)

    for k in range(3):
        one(k)
    pipe.synchronize()
    steps = max(5, args.steps // 2)
    # three timed runs of `steps` submits each; the median run is reported
    runs = []
    for _ in range(3):
        barrier(world)
        t0 = time.perf_counter()
        for k in range(steps):
            one(k)
        pipe.synchronize()
        runs.append(reduce_max(1e3 * (time.perf_counter() - t0) / steps, world, dev))
    ms = statistics.median(runs)
    tokens = reduce_sum(float(nv), world, dev)
    ok = torch.equal(y_host[(steps - 1) % 2][:nv], layer.y[:nv].cpu())
    return {"value": round(tokens / (ms / 1e3), 1), "unit": "tokens/s", "ms_per_step": round(ms, 4),
            "ms_per_step_runs": [round(r, 4) for r in runs],
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": steps,
            "output_matches_device_run": bool(ok),
            "api": "HostPipeline(ExpandedMoELayer), submit(..., n_rows=n_valid): pinned host "
                   "batches, the valid rows copied on their own streams overlapping the kernels; "
                   "host wall clock, all streams synchronised"}


def _oracle_sample(cfg, d, seconds: float, t_list=None, threads: int = 1):
    """The CPU oracle's per-token path on valid tokens of the workload for about
    `seconds`; returns (tokens, elapsed, {t: y_row}). With threads > 1 the
    tokens go to a thread pool (the oracle is C called through ctypes, which
    releases the GIL while it runs)."""
    import oracle
    inp = oracle.to_numpy_inputs({k: v for k, v in d.items()})
    nv = inp["n_valid"]
    ids = inp["topk_ids"][:nv]
    active = [int(t) for t in range(nv) if (ids[t] >= 0).any()]
    order = t_list if t_list is not None else active[:: max(1, len(active) // 997)]
    out = {}
    t0 = time.perf_counter()
    if threads <= 1:
        for t in order:
            out[t] = oracle.token_forward(inp, t)
            if time.perf_counter() - t0 > seconds:
                break
        return len(out), time.perf_counter() - t0, out
    import concurrent.futures as cf
    with cf.ThreadPoolExecutor(max_workers=threads) as ex:
        it = iter(order)
        pending = set()
        for _ in range(threads):
            t = next(it, None)
            if t is not None:
                pending.add(ex.submit(lambda t=t: (t, oracle.token_forward(inp, t))))
        while pending:
            done, pending = cf.wait(pending, return_when=cf.FIRST_COMPLETED)
            for f in done:
                t, y = f.result()
                out[t] = y
            if time.perf_counter() - t0 <= seconds:
                for _ in done:
                    t = next(it, None)
                    if t is not None:
                        pending.add(ex.submit(lambda t=t: (t, oracle.token_forward(inp, t))))
    return len(out), time.perf_counter() - t0, out


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        return os.cpu_count() or 1


def run_cpu_baseline(args, cfg, d, layer):
    import numpy as np
    n, secs, ys = _oracle_sample(cfg, d, args.cpu_sample_seconds)
    ts = sorted(ys)
    got = layer.y[ts].float().cpu().numpy().astype(np.float64)
    want = np.stack([((ys[t].astype(np.uint32) << 16).view(np.float32)).astype(np.float64) for t in ts])
    fro = float(np.linalg.norm(got - want) / max(np.linalg.norm(want), 1e-30))
    mx = float(np.abs(got - want).max())
    base = {"value": round(n / secs, 3), "unit": "tokens/s", "cores": 1, "kind": "oracle",
            "sample": f"{n} valid tokens of {cfg.name} through the oracle's per-token path "
                      f"(single-threaded C, fp64), {secs:.1f} s"}
    cores = host_cores()
    if cores > 1 and args.cpu_sample_seconds > 0:
        n2, secs2, _ = _oracle_sample(cfg, d, args.cpu_sample_seconds, threads=cores)
        base["all_cores"] = {"value": round(n2 / secs2, 3), "unit": "tokens/s", "cores": cores,
                             "kind": "oracle",
                             "sample": f"{n2} valid tokens of {cfg.name}, the same per-token path "
                                       f"on a pool of {cores} threads (one token each), "
                                       f"{secs2:.1f} s"}
    return base, {"tokens": n, "rel_fro": fro, "max_abs": mx}


# ------------------------------------------------------------------ reference arm

def run_reference(args, world, rank):
    if rank != 0:
        return None, rank
    cfg = synth.config_by_name(args.workload)
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    d = synth.generate(cfg, device=dev)
    d = {k: (v.cpu() if isinstance(v, torch.Tensor) else v) for k, v in d.items()}
    import oracle
    inp = oracle.to_numpy_inputs(d)
    nv = inp["n_valid"]
    ids = inp["topk_ids"][:nv]
    active = [int(t) for t in range(nv) if (ids[t] >= 0).any()]
    stride = max(1, len(active) // (args.steps + args.warmup + 1))
    tokens = active[::stride]
    for i in range(args.warmup):
        oracle.token_forward(inp, tokens[i % len(tokens)])
    times = []
    for i in range(args.steps):
        t0 = time.perf_counter()
        oracle.token_forward(inp, tokens[(args.warmup + i) % len(tokens)])
        times.append(time.perf_counter() - t0)
    ms = 1e3 * sum(times) / len(times)
    value = 1e3 / ms
    res = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "tokens/s",
           "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
           "ms_per_step": round(ms, 3), "higher_is_better": True, "scaling": "weak",
           "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded generator)",
           "config": {"workload": cfg.name, "T": cfg.T, "n_valid": nv, "H": cfg.H, "I": cfg.I,
                      "E": cfg.E, "top_k": cfg.K, "expert_alignment": cfg.align,
                      "step": "one valid token through the oracle's per-token path"},
           "cpu_baseline": {"value": round(value, 4), "unit": "tokens/s", "cores": 1,
                            "kind": "oracle",
                            "sample": f"{args.steps} valid tokens of {cfg.name}, one per step"},
           "e2e": {"value": round(value, 4), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}}
    return res, rank


def main(argv=None):
    args = parse_args(argv)
    world, rank, local = dist_env()
    if args.impl == "reference":
        res, rank = run_reference(args, world, rank)
    else:
        res, rank = run_ours(args, world, rank, local)
    if rank == 0 and res is not None:
        print(json.dumps(res), flush=True)
    if world > 1 and torch.distributed.is_initialized():
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
