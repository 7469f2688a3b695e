"""GPU parity: every step of the CUDA path against the CPU oracle, element by
element, on the parity workloads (tiny + mid-size shapes that span several
tiles, ragged scale words, alignment below the tile height, Zipf routing with
empty experts, inactive rows, and a padded buffer with a garbage tail).

Stage tests feed each GPU step the oracle's inputs for that step; the
end-to-end test runs the whole layer from the generator's inputs.
Layout and scatter must be bit-exact; floating-point stages are held to one
bf16 step (GEMMs, combine) or to the quantiser's own rounding (act+quant);
the final output to relative Frobenius error <= 1e-2 and max abs <= 5e-2.
"""
import numpy as np
import pytest
import torch

import synth
from parity_util import (assert_bf16_close, assert_final_close, bf16_val, e4m3_val, rel_fro, u16)

pytestmark = pytest.mark.gpu

NAMES = [c.name for c in synth.PARITY_CONFIGS]


@pytest.fixture(scope="module")
def mx():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from expanded_layout_expert_gb300 import build
    build.build()
    import expanded_layout_expert_gb300 as m
    assert m.load().moe_device_supported(torch.cuda.current_device()) == 1, "device is not sm_103"
    return m


@pytest.fixture(scope="module")
def cases(orc, mx):
    out = {}
    for cfg in synth.PARITY_CONFIGS:
        d = synth.generate(cfg, device="cpu")
        inp = orc.to_numpy_inputs(d)
        M_cap = orc.expanded_capacity(cfg.T * cfg.K, cfg.E, cfg.align)
        ref = orc.run_layer(inp, M_cap)
        g = {k: v.cuda() for k, v in d.items() if isinstance(v, torch.Tensor)}
        g["n_valid_dev"] = torch.tensor([d["n_valid"]], dtype=torch.int32, device="cuda")
        out[cfg.name] = dict(cfg=cfg, inp=inp, ref=ref, M_cap=M_cap, g=g,
                             sl=mx.scale_layout_of(cfg.scale_mode))
    return out


def _gpu_layout(mx, c, status=None):
    cfg, g = c["cfg"], c["g"]
    return mx.expand_layout(g["topk_ids"], cfg.E, cfg.align, c["M_cap"], n_valid=g["n_valid_dev"],
                            status=status)


def _pad_rows(a: np.ndarray, rows: int) -> np.ndarray:
    out = np.zeros((rows,) + a.shape[1:], a.dtype)
    out[: a.shape[0]] = a
    return out


@pytest.mark.parametrize("name", NAMES)
def test_layout_bit_exact(mx, cases, name):
    c = cases[name]
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    lay = _gpu_layout(mx, c, status)
    torch.cuda.synchronize()
    ref = c["ref"]["layout"]
    assert status.item() == 0
    assert int(lay.total.item()) == ref["total"]
    for k in ("psum", "start", "tile_prefix", "m_indices", "src2dst"):
        assert np.array_equal(getattr(lay, k).cpu().numpy(), ref[k]), k


def _poisoned_scatter_buffers(mx, M_cap, H, sl):
    """Expanded buffers holding garbage: 0xAB codes, NaN scale bits (fp32) or
    all-ones packed words (ue8m0), NaN weights."""
    xe = torch.full((M_cap, H), 0xAB, dtype=torch.uint8, device="cuda")
    xe_s = mx.new_scale(M_cap, H // 128, sl, "cuda")
    xe_s.view(torch.int32).fill_(0x7FC0DEAD if sl == 0 else -1)
    row_w = torch.full((M_cap,), float("nan"), dtype=torch.float32, device="cuda")
    return xe, xe_s, row_w


def _assert_scatter_equal(xe, xe_s, row_w, sl, rxe, rxs, rrw, tot, what):
    assert np.array_equal(xe.cpu().numpy()[:tot], rxe[:tot]), f"{what}: rows"
    assert np.array_equal(row_w.cpu().numpy().view(np.uint32)[:tot], rrw.view(np.uint32)[:tot]), \
        f"{what}: weights"
    xs = xe_s.cpu().numpy()
    if sl == 0:
        assert np.array_equal(xs[:tot].view(np.uint32), rxs[:tot].view(np.uint32)), f"{what}: scales"
    else:
        assert np.array_equal(xs[:, :tot], rxs[:, :tot]), f"{what}: packed scales"


def _rotated_routing(ids: np.ndarray, E: int) -> np.ndarray:
    """A second routing of the same tokens: every valid id moved to the next
    expert (the -1 entries stay), so the segment boundaries move."""
    return np.where(ids >= 0, (ids + 1) % E, ids).astype(np.int32)


@pytest.mark.parametrize("name", NAMES)
def test_scatter_bit_exact(mx, orc, cases, name):
    """The default moe_expand_scatter into buffers full of garbage: every row
    below the total, alignment gaps included, equals the oracle's scatter bit
    for bit (codes, scales or packed scale words, weights). Then the same
    buffers take a second routing, so that rows which held token data become
    gaps and must be zeroed (vLLM PR 54109, Motivation: the gaps are zeroed;
    deep_gemm.py, pre_permute_deepep_v2_to_deep_gemm: packed UE8M0 scales
    need zero padding lanes)."""
    c = cases[name]
    cfg, g, ref, inp = c["cfg"], c["g"], c["ref"], c["inp"]
    M_cap, sl, nv = c["M_cap"], c["sl"], inp["n_valid"]
    xe, xe_s, row_w = _poisoned_scatter_buffers(mx, M_cap, cfg.H, sl)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    lay = _gpu_layout(mx, c)
    mx.expand_scatter(g["x_q"], g["x_s"], sl, g["topk_w"], lay, n_valid=g["n_valid_dev"],
                      xe=xe, xe_scale=xe_s, row_w=row_w, status=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    _assert_scatter_equal(xe, xe_s, row_w, sl, ref["xe"], ref["xe_s"], ref["row_w"], ref["total"],
                          f"{name} first routing")

    ids2 = _rotated_routing(inp["topk_ids"], cfg.E)
    rl2 = orc.layout(ids2, cfg.E, cfg.align, nv, M_cap)
    assert rl2["rc"] == 0
    rxe2, rxs2, rrw2 = orc.scatter(inp["x_q"], inp["x_s"], inp["scale_layout"], inp["topk_w"], rl2,
                                   nv, cfg.E, cfg.align, M_cap)
    tot2 = rl2["total"]
    data1 = np.zeros(M_cap, bool)
    data1[ref["layout"]["src2dst"][:nv][ref["layout"]["src2dst"][:nv] >= 0]] = True
    gaps2 = np.ones(tot2, bool)
    gaps2[rl2["src2dst"][:nv][rl2["src2dst"][:nv] >= 0]] = False
    assert gaps2.sum() == 0 or (gaps2 & data1[:tot2]).any(), "no data row became a gap"
    lay2 = mx.expand_layout(torch.from_numpy(ids2).cuda(), cfg.E, cfg.align, M_cap,
                            n_valid=g["n_valid_dev"], status=status)
    mx.expand_scatter(g["x_q"], g["x_s"], sl, g["topk_w"], lay2, n_valid=g["n_valid_dev"],
                      xe=xe, xe_scale=xe_s, row_w=row_w, status=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    _assert_scatter_equal(xe, xe_s, row_w, sl, rxe2, rxs2, rrw2, tot2, f"{name} second routing")


@pytest.mark.parametrize("name", NAMES)
def test_layout_scatter_fused_bit_exact(mx, cases, name):
    """moe_expand_layout_scatter (the layout fused into the scatter): the
    oracle's layout and expanded rows bit for bit, into buffers filled with
    garbage first, so every row below the total must have been written."""
    c = cases[name]
    cfg, g, ref = c["cfg"], c["g"], c["ref"]
    H = cfg.H
    xe = torch.full((c["M_cap"], H), 0xAB, dtype=torch.uint8, device="cuda")
    xe_s = mx.new_scale(c["M_cap"], H // 128, c["sl"], "cuda")
    xe_s.view(torch.int32).fill_(0x7FC0DEAD)
    row_w = torch.full((c["M_cap"],), float("nan"), dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    lay, xe, xe_s, row_w = mx.expand_layout_scatter(
        g["x_q"], g["x_s"], c["sl"], g["topk_ids"], g["topk_w"], cfg.E, cfg.align, c["M_cap"],
        n_valid=g["n_valid_dev"], status=status, xe=xe, xe_scale=xe_s, row_w=row_w)
    torch.cuda.synchronize()
    assert status.item() == 0
    rl = ref["layout"]
    assert int(lay.total.item()) == rl["total"]
    for k in ("psum", "start", "tile_prefix", "m_indices", "src2dst"):
        assert np.array_equal(getattr(lay, k).cpu().numpy(), rl[k]), k
    tot = ref["total"]
    assert np.array_equal(xe.cpu().numpy()[:tot], ref["xe"][:tot])
    assert np.array_equal(row_w.cpu().numpy().view(np.uint32)[:tot], ref["row_w"].view(np.uint32)[:tot])
    xs = xe_s.cpu().numpy()
    if c["sl"] == 0:
        assert np.array_equal(xs[:tot].view(np.uint32), ref["xe_s"][:tot].view(np.uint32))
    else:
        assert np.array_equal(xs[:, :tot], ref["xe_s"][:, :tot])


# Inputs with several 2048-pair layout chunks (the parity workloads above fit
# one), top-k values that do not divide 2048 (chunks that split a token's
# pairs), empty experts, inactive rows and a garbage tail past n_valid.
MULTI_CHUNK = (
    synth.LayerConfig("chunks_k6_zipf", T=1000, H=512, I=128, E=16, K=6, align=64, seed=30,
                      routing="zipf", zipf_s=1.2, zipf_zero_experts=3, inactive_frac=0.05),
    synth.LayerConfig("chunks_k8_ue8m0", T=700, H=640, I=128, E=12, K=8, align=16, seed=31,
                      scale_mode=synth.SCALE_UE8M0),
    synth.LayerConfig("chunks_k5_padded", T=1600, H=512, I=128, E=10, K=5, align=128, seed=32,
                      n_valid=900, garbage_tail=True),
    # 1024 experts: the cooperative kernels' per-warp tables take 78 KB of
    # shared memory and each lane of the expert scan walks 32 experts
    synth.LayerConfig("chunks_e1024_k8", T=600, H=128, I=128, E=1024, K=8, align=16, seed=36,
                      routing="uniform", inactive_frac=0.05),
    # top-1 (one pair per token, lane 0 alone carries the rows in the copy)
    # and top-32 (every lane of a copy warp holds a destination row)
    synth.LayerConfig("chunks_k1", T=5000, H=256, I=128, E=8, K=1, align=32, seed=37,
                      routing="zipf", zipf_s=1.1, zipf_zero_experts=2, inactive_frac=0.05),
    synth.LayerConfig("chunks_k32_ue8m0", T=100, H=384, I=128, E=64, K=32, align=8, seed=38,
                      routing="uniform", scale_mode=synth.SCALE_UE8M0),
)


# More chunks than the cooperative grids hold on a 152-SM GPU: 313 chunks
# (past the fused kernel's two blocks per SM: the fused call becomes the
# two calls) and 469 (past the layout kernel's three: the layout takes its
# two-launch path).
MANY_CHUNKS = (
    synth.LayerConfig("chunks_313_k8", T=80000, H=128, I=128, E=8, K=8, align=16, seed=33,
                      routing="zipf", zipf_s=1.1, zipf_zero_experts=1, inactive_frac=0.02),
    synth.LayerConfig("chunks_469_k8_ue8m0", T=120000, H=128, I=128, E=8, K=8, align=32, seed=34,
                      scale_mode=synth.SCALE_UE8M0, n_valid=119000, garbage_tail=True),
)


@pytest.mark.parametrize("fused", [False, True], ids=["two_calls", "fused"])
@pytest.mark.parametrize("cfg", MULTI_CHUNK + MANY_CHUNKS,
                         ids=[c.name for c in MULTI_CHUNK + MANY_CHUNKS])
def test_layout_scatter_multi_chunk_bit_exact(mx, orc, cfg, fused):
    """Layout and scatter over several chunks against the oracle, bit for
    bit, through moe_expand_layout + moe_expand_scatter and through
    moe_expand_layout_scatter, into buffers full of garbage."""
    d = synth.generate(cfg, device="cpu")
    inp = orc.to_numpy_inputs(d)
    M_cap = orc.expanded_capacity(cfg.T * cfg.K, cfg.E, cfg.align)
    nv = inp["n_valid"]
    rl = orc.layout(inp["topk_ids"], cfg.E, cfg.align, nv, M_cap)
    assert rl["rc"] == 0
    sl = mx.scale_layout_of(cfg.scale_mode)
    rxe, rxs, rrw = orc.scatter(inp["x_q"], inp["x_s"], inp["scale_layout"], inp["topk_w"], rl, nv,
                                cfg.E, cfg.align, M_cap)
    g = {k: v.cuda() for k, v in d.items() if isinstance(v, torch.Tensor)}
    nvd = torch.tensor([nv], dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    xe, xe_s, row_w = _poisoned_scatter_buffers(mx, M_cap, cfg.H, sl)
    if fused:
        lay, xe, xe_s, row_w = mx.expand_layout_scatter(
            g["x_q"], g["x_s"], sl, g["topk_ids"], g["topk_w"], cfg.E, cfg.align, M_cap,
            n_valid=nvd, status=status, xe=xe, xe_scale=xe_s, row_w=row_w)
    else:
        lay = mx.expand_layout(g["topk_ids"], cfg.E, cfg.align, M_cap, n_valid=nvd, status=status)
        mx.expand_scatter(g["x_q"], g["x_s"], sl, g["topk_w"], lay, n_valid=nvd, xe=xe,
                          xe_scale=xe_s, row_w=row_w, status=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    tot = rl["total"]
    assert int(lay.total.item()) == tot
    for k in ("psum", "start", "tile_prefix", "m_indices", "src2dst"):
        assert np.array_equal(getattr(lay, k).cpu().numpy(), rl[k]), k
    assert np.array_equal(xe.cpu().numpy()[:tot], rxe[:tot])
    assert np.array_equal(row_w.cpu().numpy().view(np.uint32)[:tot], rrw.view(np.uint32)[:tot])
    xs = xe_s.cpu().numpy()
    if sl == 0:
        assert np.array_equal(xs[:tot].view(np.uint32), rxs[:tot].view(np.uint32))
    else:
        assert np.array_equal(xs[:, :tot], rxs[:, :tot])


@pytest.mark.parametrize("name", NAMES)
def test_layer_fused_layout_scatter_matches_default(mx, cases, name):
    """A layer built with fuse_layout_scatter=True gives the default layer's
    output bit for bit (same GEMM inputs)."""
    c = cases[name]
    cfg, g = c["cfg"], c["g"]
    nv = c["inp"]["n_valid"]
    ys = []
    for fuse in (False, True):
        layer = mx.ExpandedMoELayer(g["w13"], g["s13"], g["w2"], g["s2"], K=cfg.K, align=cfg.align,
                                    scale_mode=cfg.scale_mode, max_tokens=cfg.T,
                                    fuse_layout_scatter=fuse)
        y = layer.forward(g["x_q"], g["x_s"], g["topk_ids"], g["topk_w"], g["n_valid_dev"])
        torch.cuda.synchronize()
        assert layer.status.item() == 0
        ys.append(y[:nv].clone())
    assert torch.equal(ys[0], ys[1])


@pytest.mark.parametrize("tile_flag", [0, 16, 64], ids=["default", "bn128", "per_kblock"])
@pytest.mark.parametrize("name", NAMES)
def test_gate_up_gemm(mx, cases, name, tile_flag):
    c = cases[name]
    g, ref = c["g"], c["ref"]
    lay = _gpu_layout(mx, c)
    xe, xe_s, _ = mx.expand_scatter(g["x_q"], g["x_s"], c["sl"], g["topk_w"], lay,
                                    n_valid=g["n_valid_dev"])
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    gu = mx.grouped_gemm(xe, xe_s, c["sl"], lay, g["w13"], g["s13"], flags=tile_flag, status=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    tot = ref["total"]
    assert_bf16_close(u16(gu)[:tot], ref["gu"], f"{name} gate_up")
    assert (u16(gu)[tot:] == 0).all(), "rows past the total must be untouched"


@pytest.mark.parametrize("promo", [0, 64], ids=["default", "per_kblock"])
@pytest.mark.parametrize("name", NAMES)
def test_fused_gate_up_act_quant(mx, cases, name, promo):
    """gate_up with act+quant (and the fp32 path's weight fold) in its
    epilogue: bit-equal to the two stand-alone launches on every row < total
    (codes and scales; for ue8m0 every byte of a used packed word, the zero
    padding of a ragged last word included), and against the oracle's codes
    as the stand-alone act+quant is."""
    c = cases[name]
    g, ref = c["g"], c["ref"]
    lay = _gpu_layout(mx, c)
    xe, xe_s, row_w = mx.expand_scatter(g["x_q"], g["x_s"], c["sl"], g["topk_w"], lay,
                                        n_valid=g["n_valid_dev"])
    fold = mx.MOE_FOLD_WEIGHT_INTO_SCALE if c["sl"] == 0 else 0
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    di, di_s = mx.grouped_gemm_act_quant(xe, xe_s, c["sl"], lay, g["w13"], g["s13"],
                                         flags=fold | promo, row_w=row_w, status=status)
    poison = torch.full_like(di_s, -1)
    di2, di2_s = mx.grouped_gemm_act_quant(xe, xe_s, c["sl"], lay, g["w13"], g["s13"],
                                           flags=fold | promo, row_w=row_w, di_scale=poison,
                                           status=status)
    gu = mx.grouped_gemm(xe, xe_s, c["sl"], lay, g["w13"], g["s13"], flags=promo)
    du, du_s = mx.act_quant(gu, row_w, fold, c["sl"], lay.total)
    torch.cuda.synchronize()
    assert status.item() == 0
    tot = ref["total"]
    assert torch.equal(di[:tot], du[:tot])
    assert torch.equal(di2[:tot], du[:tot])
    if c["sl"] == 0:
        assert torch.equal(di_s[:tot].view(torch.int32), du_s[:tot].view(torch.int32))
        assert torch.equal(di2_s[:tot].view(torch.int32), du_s[:tot].view(torch.int32))
    else:
        assert torch.equal(di_s[:, :tot], du_s[:, :tot])
        assert torch.equal(di2_s[:, :tot], du_s[:, :tot])
    assert not di[tot:].any(), "rows past the total are untouched"
    dg, dr = di.cpu().numpy()[:tot], ref["di"]
    same = (dg == dr) | ((dg & 0x7F) == 0) & ((dr & 0x7F) == 0)
    assert same.mean() >= 0.999, f"{name}: {1 - same.mean():.2e} of fp8 codes differ"


def test_fused_gate_up_act_quant_rejects_fold_on_ue8m0(mx, cases):
    c = cases["mid_ue8m0"]
    g = c["g"]
    lay = _gpu_layout(mx, c)
    xe, xe_s, row_w = mx.expand_scatter(g["x_q"], g["x_s"], c["sl"], g["topk_w"], lay,
                                        n_valid=g["n_valid_dev"])
    with pytest.raises(mx.MoEError) as ei:
        mx.grouped_gemm_act_quant(xe, xe_s, c["sl"], lay, g["w13"], g["s13"],
                                  flags=mx.MOE_FOLD_WEIGHT_INTO_SCALE, row_w=row_w)
    assert ei.value.rc == -1


@pytest.mark.parametrize("name", NAMES)
def test_act_quant(mx, cases, name):
    c = cases[name]
    cfg, ref, M = c["cfg"], c["ref"], c["M_cap"]
    lay = _gpu_layout(mx, c)
    tot = ref["total"]
    gu = torch.from_numpy(_pad_rows(ref["gu"], M).view(np.int16)).view(torch.bfloat16).cuda()
    row_w = torch.from_numpy(ref["row_w"]).cuda()
    flags = mx.MOE_FOLD_WEIGHT_INTO_SCALE if c["sl"] == 0 else 0
    di, di_s = mx.act_quant(gu, row_w, flags, c["sl"], lay.total)
    torch.cuda.synchronize()
    dg, dr = di.cpu().numpy()[:tot], ref["di"]
    same = (dg == dr) | ((dg & 0x7F) == 0) & ((dr & 0x7F) == 0)
    assert same.mean() >= 0.999, f"{name}: {1 - same.mean():.2e} of fp8 codes differ"
    # where a code differs, it is by one e4m3 step (the silu in fp32 versus double)
    vg, vr = e4m3_val(dg), e4m3_val(dr)
    step = np.maximum(np.abs(vr), np.abs(vg)) / 8 + 2.0 ** -9
    assert (np.abs(vg - vr) <= step).all()
    sg = di_s.cpu().numpy()
    if c["sl"] == 0:
        sg = sg[:tot]
        sr = ref["di_s"]
        assert (sg == sr).mean() >= 0.99
        assert np.allclose(sg, sr, rtol=2.0 ** -7, atol=0)
    else:
        bg = sg[:, :tot].view(np.uint32)
        br = ref["di_s"].view(np.uint32)
        assert (bg == br).mean() >= 0.99


@pytest.mark.parametrize("promo", [0, 64], ids=["default", "per_kblock"])
@pytest.mark.parametrize("name", NAMES)
def test_down_gemm(mx, cases, name, promo):
    c = cases[name]
    g, ref, M = c["g"], c["ref"], c["M_cap"]
    lay = _gpu_layout(mx, c)
    di = torch.from_numpy(_pad_rows(ref["di"], M)).cuda()
    if c["sl"] == 0:
        di_s = torch.from_numpy(_pad_rows(ref["di_s"], M)).cuda()
        flags = 0
    else:
        s = np.zeros((ref["di_s"].shape[0], M), np.int32)
        s[:, : ref["di_s"].shape[1]] = ref["di_s"]
        di_s = torch.from_numpy(s).cuda()
        flags = mx.MOE_WEIGHT_OUTPUT_ROWS
    row_w = torch.from_numpy(ref["row_w"]).cuda()
    down = mx.grouped_gemm(di, di_s, c["sl"], lay, g["w2"], g["s2"], row_w=row_w, flags=flags | promo)
    torch.cuda.synchronize()
    tot = ref["total"]
    # ue8m0: the oracle rounds to bf16 before and after the weighting (the
    # pages' separate weighting pass over down_output); the kernel weights the
    # fp32 accumulator and rounds once, so the two differ by up to two bf16
    # steps (one step is 2^-8 relative)
    if c["sl"] == 0:
        assert_bf16_close(u16(down)[:tot], ref["down"], f"{name} down")
    else:
        assert_bf16_close(u16(down)[:tot], ref["down"], f"{name} down", ulps=2, rel=2.0 ** -8)


@pytest.mark.parametrize("name", NAMES)
def test_combine(mx, cases, name):
    c = cases[name]
    cfg, g, ref, M = c["cfg"], c["g"], c["ref"], c["M_cap"]
    lay = _gpu_layout(mx, c)
    down = torch.from_numpy(_pad_rows(ref["down"], M).view(np.int16)).view(torch.bfloat16).cuda()
    y = torch.full((cfg.T, cfg.H), float("nan"), dtype=torch.bfloat16, device="cuda")
    mx.combine(down, lay.src2dst, None, g["n_valid_dev"], y)
    torch.cuda.synchronize()
    nv = c["inp"]["n_valid"]
    assert_bf16_close(u16(y)[:nv], ref["y"][:nv], f"{name} combine")
    assert torch.isnan(y[nv:].float()).all(), "rows past n_valid must not be written"


@pytest.mark.parametrize("name", NAMES)
def test_weighted_combine(mx, cases, orc, name):
    """The gather-weighted combine (ep_gather's weighting) against the oracle's
    weighted sum on the oracle's unweighted down rows."""
    c = cases[name]
    cfg, g, ref, M = c["cfg"], c["g"], c["ref"], c["M_cap"]
    gref = c.setdefault("gather_ref", orc.run_layer(c["inp"], M, weighting="gather"))
    lay = _gpu_layout(mx, c)
    down = torch.from_numpy(_pad_rows(gref["down"], M).view(np.int16)).view(torch.bfloat16).cuda()
    row_w = torch.from_numpy(_pad_rows(gref["row_w"], M)).cuda()
    y = torch.full((cfg.T, cfg.H), float("nan"), dtype=torch.bfloat16, device="cuda")
    mx.combine(down, lay.src2dst, row_w, g["n_valid_dev"], y)
    torch.cuda.synchronize()
    nv = c["inp"]["n_valid"]
    assert_bf16_close(u16(y)[:nv], gref["y"][:nv], f"{name} weighted combine")
    assert torch.isnan(y[nv:].float()).all(), "rows past n_valid must not be written"


def _layer(mx, c, weighting="expanded"):
    cfg, g = c["cfg"], c["g"]
    return mx.ExpandedMoELayer(g["w13"], g["s13"], g["w2"], g["s2"], K=cfg.K, align=cfg.align,
                               scale_mode=cfg.scale_mode, max_tokens=cfg.T, weighting=weighting)


@pytest.mark.parametrize("name", NAMES)
def test_layer_gather_weighting_end_to_end(mx, cases, orc, name):
    """The do_expand=False arrangement (weights applied in the combine) against
    the oracle's layer with the same arrangement."""
    c = cases[name]
    g = c["g"]
    gref = c.setdefault("gather_ref", orc.run_layer(c["inp"], c["M_cap"], weighting="gather"))
    layer = _layer(mx, c, weighting="gather")
    y = layer.forward(g["x_q"], g["x_s"], g["topk_ids"], g["topk_w"], g["n_valid_dev"])
    torch.cuda.synchronize()
    assert layer.status.item() == 0
    nv = c["inp"]["n_valid"]
    assert_final_close(u16(y)[:nv], gref["y"][:nv], name)


@pytest.mark.parametrize("name", NAMES)
def test_layer_end_to_end(mx, cases, name):
    c = cases[name]
    g, ref = c["g"], c["ref"]
    layer = _layer(mx, c)
    y = layer.forward(g["x_q"], g["x_s"], g["topk_ids"], g["topk_w"], g["n_valid_dev"])
    torch.cuda.synchronize()
    assert layer.status.item() == 0
    nv = c["inp"]["n_valid"]
    fro, mxabs = assert_final_close(u16(y)[:nv], ref["y"][:nv], name)
    print(f"{name}: rel_fro {fro:.3e} max_abs {mxabs:.3e}")
    # a second call on the same buffers gives the same bits
    y2 = layer.forward(g["x_q"], g["x_s"], g["topk_ids"], g["topk_w"], g["n_valid_dev"]).clone()
    torch.cuda.synchronize()
    assert torch.equal(y2[:nv], y[:nv])


def test_poisoned_buffers_and_tail(mx, cases):
    """Garbage in every intermediate buffer and in the rows past n_valid
    (NaN codes, NaN scales, in-range ids) leaves the valid outputs
    bit-identical to a clean run (the padding-robustness test idea of vLLM
    PR 54109)."""
    c = cases["mid_padded"]
    g = c["g"]
    nv = c["inp"]["n_valid"]
    clean = _layer(mx, c).forward(g["x_q"], g["x_s"], g["topk_ids"], g["topk_w"],
                                  g["n_valid_dev"]).clone()
    layer = _layer(mx, c)
    for buf in (layer.xe, layer.down_in):
        buf.fill_(0x7F)
    for buf in (layer.gateup, layer.down_out, layer.y):
        buf.fill_(float("nan"))
    layer.xe_scale.fill_(float("nan")) if layer.xe_scale.dtype == torch.float32 else layer.xe_scale.fill_(-1)
    layer.row_w.fill_(float("nan"))
    x_q, x_s = g["x_q"].clone(), g["x_s"].clone()
    ids, w = g["topk_ids"].clone(), g["topk_w"].clone()
    x_q[nv:] = 0x7F
    x_s[nv:] = float("nan")
    ids[nv:] = torch.randint(0, c["cfg"].E, ids[nv:].shape, device="cuda", dtype=torch.int32)
    w[nv:] = float("inf")
    y = layer.forward(x_q, x_s, ids, w, g["n_valid_dev"])
    torch.cuda.synchronize()
    assert layer.status.item() == 0
    assert torch.equal(u16_t(y[:nv]), u16_t(clean[:nv]))
    assert torch.isnan(y[nv:].float()).all()


def u16_t(t):
    return t.view(torch.int16)


def test_device_checks_report_without_faulting(mx):
    E, K, T = 4, 2, 8
    ids = torch.tensor([[0, 1]] * T, dtype=torch.int32, device="cuda")
    ids[3, 1] = 9  # >= E in a valid row
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    lay = mx.expand_layout(ids, E, 4, 64, status=status)
    torch.cuda.synchronize()
    assert status.item() == mx._capi.MOE_ERR_DEVICE_CHECK
    assert lay.src2dst[3, 1].item() == -1
    # capacity smaller than the aligned total
    ids = torch.tensor([[0, 1], [2, 3]], dtype=torch.int32, device="cuda")
    status.zero_()
    lay = mx.expand_layout(ids, 4, 8, 16, status=status)
    torch.cuda.synchronize()
    assert status.item() == mx._capi.MOE_ERR_DEVICE_CHECK
    assert int(lay.total.item()) == 32
    s2d = lay.src2dst.cpu().numpy()
    assert ((s2d == -1) | (s2d < 16)).all()


def test_device_checks_on_several_chunks(mx):
    """The same checks through the cooperative layout and the fused layout +
    scatter (three 2048-pair chunks): an id >= E is flagged and its pair
    dropped; a capacity below the aligned total is flagged, and nothing is
    written at or past it."""
    E, K, T, H = 8, 2, 3000, 128
    g = torch.Generator().manual_seed(7)
    ids = torch.randint(0, E, (T, K), generator=g, dtype=torch.int32).cuda()
    ids[1234, 1] = E + 3
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    M_cap = mx.expanded_capacity(T, K, E, 16)
    lay = mx.expand_layout(ids, E, 16, M_cap, status=status)
    torch.cuda.synchronize()
    assert status.item() == mx._capi.MOE_ERR_DEVICE_CHECK
    assert lay.src2dst[1234, 1].item() == -1
    assert int((lay.src2dst >= 0).sum().item()) == T * K - 1
    # capacity below the total, through the fused call into guarded buffers
    ids[1234, 1] = 0
    small = 1024
    x = torch.randint(0, 256, (T, H), dtype=torch.uint8, device="cuda")
    xs = torch.ones(T, H // 128, dtype=torch.float32, device="cuda")
    w = torch.rand(T, K, device="cuda")
    xe = torch.full((small + 64, H), 0xAB, dtype=torch.uint8, device="cuda")
    xe_s = torch.full((small + 64, H // 128), float("nan"), device="cuda")
    rw = torch.full((small + 64,), float("nan"), device="cuda")
    status.zero_()
    lay, _, _, _ = mx.expand_layout_scatter(x, xs, mx.MOE_SCALE_F32_ROWMAJOR, ids, w, E, 16, small,
                                            status=status, xe=xe[:small], xe_scale=xe_s[:small],
                                            row_w=rw[:small])
    torch.cuda.synchronize()
    assert status.item() == mx._capi.MOE_ERR_DEVICE_CHECK
    assert int(lay.total.item()) > small
    s2d = lay.src2dst.cpu().numpy()
    assert ((s2d == -1) | (s2d < small)).all()
    assert (xe[small:] == 0xAB).all() and torch.isnan(rw[small:]).all()
    assert torch.isnan(xe_s[small:]).all()


@pytest.mark.parametrize("name", ["mid_f32", "mid_ue8m0_ragged", "wide_e160_k12"])
def test_grouped_ffn_fused_equals_three_launches(mx, cases, name):
    """moe_grouped_ffn's default (gate_up with act+quant fused) and its
    MOE_FFN_UNFUSED three-launch path give the same down_proj output bits."""
    c = cases[name]
    g = c["g"]
    lay = _gpu_layout(mx, c)
    xe, xe_s, row_w = mx.expand_scatter(g["x_q"], g["x_s"], c["sl"], g["topk_w"], lay,
                                        n_valid=g["n_valid_dev"])
    flags = mx.MOE_FOLD_WEIGHT_INTO_SCALE if c["sl"] == 0 else mx.MOE_WEIGHT_OUTPUT_ROWS
    outs = []
    for extra in (0, mx.MOE_FFN_UNFUSED):
        _, di, di_s, down = mx.grouped_ffn(xe, xe_s, c["sl"], lay, g["w13"], g["s13"], g["w2"],
                                           g["s2"], row_w, flags | extra)
        outs.append((di, di_s, down))
    torch.cuda.synchronize()
    tot = c["ref"]["total"]
    assert torch.equal(outs[0][0][:tot], outs[1][0][:tot])
    assert torch.equal(outs[0][2][:tot].view(torch.int16), outs[1][2][:tot].view(torch.int16))


@pytest.mark.parametrize("mode", ["expanded", "masked"])
def test_captured_forward_replays(mx, cases, mode):
    """A CUDA graph of the whole forward replays to the eager result, and
    again after the inputs are refilled in place with a new routing."""
    c = cases["mid_zipf_ragged"]
    cfg, g = c["cfg"], c["g"]
    kw = dict(K=cfg.K, align=cfg.align, scale_mode=cfg.scale_mode, max_tokens=cfg.T)
    if mode == "masked":
        kw["masked_max_m"] = cfg.T * cfg.K
    layer = mx.ExpandedMoELayer(g["w13"], g["s13"], g["w2"], g["s2"], **kw)
    x_q, x_s = g["x_q"].clone(), g["x_s"].clone()
    ids, w, nv = g["topk_ids"].clone(), g["topk_w"].clone(), g["n_valid_dev"].clone()
    want0 = layer.forward(x_q, x_s, ids, w, nv).clone()
    out = torch.zeros_like(layer.y)
    cap = layer.capture(x_q, x_s, ids, w, nv, out=out)
    y = cap.replay()
    torch.cuda.synchronize()
    n = c["inp"]["n_valid"]
    assert torch.equal(y[:n], want0[:n])
    perm = torch.randperm(cfg.T, generator=torch.Generator().manual_seed(3))
    ids.copy_(g["topk_ids"][perm.cuda()])
    want1 = layer.forward(x_q, x_s, ids, w, nv).clone()
    y = cap.replay()
    torch.cuda.synchronize()
    assert torch.equal(y[:n], want1[:n])
    assert not torch.equal(want0[:n], want1[:n])
    assert layer.status.item() == 0


def test_bounded_wait_times_out_and_the_context_survives(mx, cases):
    """A wait on a barrier nothing arrives at gives up after its limit with
    MOE_ERR_TIMEOUT on the status word; the other roles (a single thread and
    a warp in the warp-collective wait) leave on the abort flag well before
    their own (longer) limit; a warp-collective waiter alone gives up on its
    own limit, all lanes together; the device keeps working."""
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.full((8,), -1, dtype=torch.int64, device="cuda")
    limit = 2_000_000  # about 1 ms
    mx.check(mx.load().moe_selftest_bounded_wait(limit, status.data_ptr(), out.data_ptr(),
                                                  torch.cuda.current_stream().cuda_stream),
             "selftest")
    torch.cuda.synchronize()
    o = out.cpu().tolist()
    assert status.item() == mx._capi.MOE_ERR_TIMEOUT
    assert o[0] == 0 and o[1] >= limit
    assert o[2] == 0 and o[3] < 4 * limit, "the second waiter left on the abort flag"
    assert o[4] == 0 and o[5] < 4 * limit, "the waiting warp left on the abort flag"
    assert o[6] == 0 and o[7] >= limit, "a waiting warp gives up on its own limit"
    # the context is still usable: a whole layer runs and matches the oracle
    c = cases["tiny_h512"]
    g = c["g"]
    layer = _layer(mx, c)
    y = layer.forward(g["x_q"], g["x_s"], g["topk_ids"], g["topk_w"], g["n_valid_dev"])
    torch.cuda.synchronize()
    nv = c["inp"]["n_valid"]
    assert_final_close(u16(y)[:nv], c["ref"]["y"][:nv], "after timeout")


@pytest.mark.parametrize("T", [6, 3000], ids=["one_chunk", "three_chunks"])
def test_empty_and_all_inactive(mx, T):
    """No valid pair (every id -1), then no valid row (n_valid = 0): on one
    2048-pair chunk (the one-block layout) and on three (the cooperative
    layout and the fused layout + scatter)."""
    E, K, H, I = 4, 2, 256, 128
    dev = "cuda"
    ids = torch.full((T, K), -1, dtype=torch.int32, device=dev)
    lay = mx.expand_layout(ids, E, 32, 64)
    torch.cuda.synchronize()
    assert int(lay.total.item()) == 0 and (lay.m_indices == -1).all()
    assert (lay.tile_prefix == 0).all() and (lay.src2dst == -1).all()
    w13 = torch.zeros(E, 2 * I, H, dtype=torch.uint8, device=dev)
    s13 = torch.ones(E, 2 * I // 128, H // 128, dtype=torch.float32, device=dev)
    w2 = torch.zeros(E, H, I, dtype=torch.uint8, device=dev)
    s2 = torch.ones(E, H // 128, I // 128, dtype=torch.float32, device=dev)
    layer = mx.ExpandedMoELayer(w13, s13, w2, s2, K=K, align=32, scale_mode="f32", max_tokens=T)
    x = torch.full((T, H), 0x38, dtype=torch.uint8, device=dev)
    xs = torch.ones(T, H // 128, dtype=torch.float32, device=dev)
    layer.y.fill_(float("nan"))
    y = layer.forward(x, xs, ids, torch.zeros(T, K, device=dev))
    torch.cuda.synchronize()
    assert (y.float() == 0).all()
    # n_valid = 0: nothing is valid, nothing is written
    layer.y.fill_(float("nan"))
    nv = torch.zeros(1, dtype=torch.int32, device=dev)
    ids2 = torch.zeros(T, K, dtype=torch.int32, device=dev)
    y = layer.forward(x, xs, ids2, torch.ones(T, K, device=dev), nv)
    torch.cuda.synchronize()
    assert torch.isnan(y.float()).all()
    assert int(layer.lay.total.item()) == 0
    assert (layer.lay.src2dst == -1).all() and layer.status.item() == 0


@pytest.mark.parametrize("mode", ["expanded", "gather", "masked"])
def test_host_pipeline_matches_forward(mx, cases, mode):
    """HostPipeline (pinned host batches, copies on side streams, double
    buffers) gives every batch's forward output: four batches with different
    routings through the same two buffer sets, for each layer arrangement."""
    c = cases["mid_zipf_ragged"]
    cfg, g = c["cfg"], c["g"]
    if mode == "masked":
        layer = mx.ExpandedMoELayer(g["w13"], g["s13"], g["w2"], g["s2"], K=cfg.K,
                                    align=cfg.align, scale_mode=cfg.scale_mode,
                                    max_tokens=cfg.T, masked_max_m=cfg.T * cfg.K)
    else:
        layer = _layer(mx, c, weighting=mode)
    rng = np.random.default_rng(5)
    batches = []
    for b in range(4):
        ids = g["topk_ids"].cpu().numpy().copy()
        rng.shuffle(ids)  # a different token -> experts assignment per batch
        batches.append(dict(x_q=g["x_q"].cpu().pin_memory(), x_s=g["x_s"].cpu().pin_memory(),
                            ids=torch.from_numpy(ids).pin_memory(),
                            w=g["topk_w"].cpu().pin_memory(),
                            nv=torch.tensor([c["inp"]["n_valid"]], dtype=torch.int32).pin_memory()))
    want = []
    for bt in batches:
        y = layer.forward(bt["x_q"].cuda(), bt["x_s"].cuda(), bt["ids"].cuda(), bt["w"].cuda(),
                          bt["nv"].cuda())
        want.append(y.cpu().clone())
    pipe = mx.HostPipeline(layer)
    outs = [torch.zeros(cfg.T, cfg.H, dtype=torch.bfloat16).pin_memory() for _ in batches]
    for bt, o in zip(batches, outs):
        pipe.submit(bt["x_q"], bt["x_s"], bt["ids"], bt["w"], bt["nv"], o)
    pipe.synchronize()
    nv = c["inp"]["n_valid"]
    for k in range(len(batches)):
        assert torch.equal(outs[k][:nv], want[k][:nv]), k
    assert layer.status.item() == 0


@pytest.mark.parametrize("name", ["mid_padded", "mid_ue8m0_ragged"])
def test_host_pipeline_copies_only_the_valid_prefix(mx, cases, name):
    """HostPipeline.submit(..., n_rows=n) moves only rows [0, n) both ways
    (column-major packed scales by word row) and gives the forward's output
    on those rows; host rows past n are left as they were."""
    c = cases[name]
    cfg, g = c["cfg"], c["g"]
    nv = min(c["inp"]["n_valid"], cfg.T - 37)
    layer = _layer(mx, c)
    nvd = torch.tensor([nv], dtype=torch.int32, device="cuda")
    want = layer.forward(g["x_q"], g["x_s"], g["topk_ids"], g["topk_w"], nvd)[:nv].cpu().clone()
    host = [t.cpu().pin_memory() for t in (g["x_q"], g["x_s"], g["topk_ids"], g["topk_w"])]
    nv_h = torch.tensor([nv], dtype=torch.int32).pin_memory()
    pipe = mx.HostPipeline(layer)
    outs = []
    for _ in range(3):
        o = torch.full((cfg.T, cfg.H), float("nan"), dtype=torch.bfloat16).pin_memory()
        pipe.submit(*host, nv_h, o, n_rows=nv)
        outs.append(o)
    pipe.synchronize()
    for o in outs:
        assert torch.equal(o[:nv], want)
        assert torch.isnan(o[nv:].float()).all()
    assert layer.status.item() == 0


def test_one_workspace_serves_calls_of_different_sizes(mx, orc):
    """A workspace sized for the largest call, reused by smaller ones in
    between (three, one and 469 chunks: the cooperative layout, the one-block
    layout, the two-launch layout): every result equals the oracle's, so the
    barrier and ticket words the calls share start at zero every time."""
    E, K, align = 8, 2, 16
    sizes = (3000, 500, 480000, 3000, 700)
    ws = torch.zeros(max(mx.workspace_size(T, K, E) for T in sizes), dtype=torch.uint8,
                     device="cuda")
    g = torch.Generator().manual_seed(9)
    for T in sizes:
        ids = torch.randint(-1, E, (T, K), generator=g, dtype=torch.int32)
        M_cap = orc.expanded_capacity(T * K, E, align)
        rl = orc.layout(ids.numpy(), E, align, T, M_cap)
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        lay = mx.expand_layout(ids.cuda(), E, align, M_cap, ws=ws, status=status)
        torch.cuda.synchronize()
        assert status.item() == 0, T
        assert int(lay.total.item()) == rl["total"], T
        for k in ("psum", "start", "tile_prefix", "src2dst"):
            assert np.array_equal(getattr(lay, k).cpu().numpy().reshape(-1),
                                  np.asarray(rl[k]).reshape(-1)), (T, k)
