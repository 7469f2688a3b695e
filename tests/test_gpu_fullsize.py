"""The five workloads at full size, through ExpandedMoELayer (the launch
configuration the benchmark times):

* layout: bit-exact against the oracle on every row (the oracle's layout is
  cheap at any size);
* scatter: every expanded row equals its token's bytes, scale and weight, and
  every alignment gap is zero (a property checked on all rows on the device);
* the fused gate_up + act+quant of the forward equals the stand-alone
  launches on every row, bit for bit;
* gate_up rows and final outputs on sampled tokens against the oracle, which
  computes them one by one (the final output to rel-Frobenius <= 1e-2 and
  max abs <= 5e-2);
* rows past n_valid are never written, the status word stays clean.
"""
import numpy as np
import pytest
import torch

import synth
from parity_util import assert_bf16_close, assert_final_close, u16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mx():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from expanded_layout_expert_gb300 import build
    build.build()
    import expanded_layout_expert_gb300 as m
    return m


def _sample_tokens(ids, nv, n, seed):
    rng = np.random.default_rng(seed)
    active = np.flatnonzero((ids[:nv] >= 0).any(1))
    inactive = np.flatnonzero(~(ids[:nv] >= 0).any(1))
    pick = list(rng.choice(active, size=min(n, active.size), replace=False))
    if inactive.size:
        pick.append(int(inactive[0]))
    pick.append(int(active[-1]))
    return sorted(set(int(t) for t in pick))


@pytest.mark.parametrize("cfg", synth.CONFIGS, ids=lambda c: c.name)
def test_workload_full_size(mx, orc, cfg):
    dev = torch.device("cuda")
    d = synth.generate(cfg, device=dev)
    nv = d["n_valid"]
    n_valid = torch.tensor([nv], dtype=torch.int32, device=dev)
    layer = mx.ExpandedMoELayer(d["w13"], d["s13"], d["w2"], d["s2"], K=cfg.K, align=cfg.align,
                                scale_mode=cfg.scale_mode, max_tokens=cfg.T)
    layer.y.fill_(float("nan"))
    y = layer.forward(d["x_q"], d["x_s"], d["topk_ids"], d["topk_w"], n_valid)
    torch.cuda.synchronize()
    assert layer.status.item() == 0

    # layout, every row, against the oracle
    ids = d["topk_ids"].cpu().numpy()
    M_cap = orc.expanded_capacity(cfg.T * cfg.K, cfg.E, cfg.align)
    assert M_cap == layer.M_cap
    ref = orc.layout(ids, cfg.E, cfg.align, nv, M_cap)
    lay = layer.lay
    total = ref["total"]
    assert int(lay.total.item()) == total
    for k in ("psum", "start", "tile_prefix", "m_indices", "src2dst"):
        assert np.array_equal(getattr(lay, k).cpu().numpy(), ref[k]), k

    # scatter, every row, as a property on the device
    s2d = lay.src2dst
    valid = s2d >= 0
    t_idx = torch.arange(cfg.T, device=dev).unsqueeze(1).expand_as(s2d)[valid]
    rows = s2d[valid].long()
    assert torch.equal(layer.xe[rows], d["x_q"][t_idx])
    assert torch.equal(layer.row_w[rows], d["topk_w"][valid])
    if cfg.scale_mode == "f32":
        assert torch.equal(layer.xe_scale[rows].view(torch.int32), d["x_s"][t_idx].view(torch.int32))
    else:
        assert torch.equal(layer.xe_scale[:, rows], d["x_s"][:, t_idx])
    gap = torch.ones(total, dtype=torch.bool, device=dev)
    gap[rows] = False
    assert not layer.xe[:total][gap].any() and not layer.row_w[:total][gap].any()

    # the forward ran gate_up with act+quant fused; the two stand-alone
    # launches give the same codes and scales on every row
    gu = mx.grouped_gemm(layer.xe, layer.xe_scale, layer.sl, lay, layer.w13, layer.s13,
                         out=layer.gateup)
    fold = layer.flags & mx.MOE_FOLD_WEIGHT_INTO_SCALE
    du, du_s = mx.act_quant(gu, layer.row_w, fold, layer.sl, lay.total)
    torch.cuda.synchronize()
    assert torch.equal(du[:total], layer.down_in[:total])
    if cfg.scale_mode == "ue8m0":
        assert torch.equal(du_s[:, :total], layer.down_in_scale[:, :total])
    else:
        assert torch.equal(du_s[:total].view(torch.int32),
                           layer.down_in_scale[:total].view(torch.int32))

    # rows past n_valid untouched
    if nv < cfg.T:
        assert torch.isnan(y[nv:].float()).all()

    # sampled tokens through the oracle's per-token path
    inp = orc.to_numpy_inputs(d)
    toks = _sample_tokens(ids, nv, 4 if cfg.H >= 7168 else 8, cfg.seed)
    want = np.stack([orc.token_forward(inp, t) for t in toks])
    got = u16(y[toks])
    fro, mxabs = assert_final_close(got, want, cfg.name)
    print(f"{cfg.name}: {len(toks)} tokens rel_fro {fro:.3e} max_abs {mxabs:.3e}")

    # sampled gate_up rows against the oracle's GEMM on the token's own row
    s2d_h = s2d.cpu().numpy()
    pairs = [(t, k) for t in toks for k in range(cfg.K) if s2d_h[t, k] >= 0][:6]
    ref_rows = orc.gemm_rows(inp["x_q"], inp["x_s"], inp["scale_layout"], inp["x_s"].shape[1],
                             np.array([t for t, _ in pairs]), np.array([ids[t, k] for t, k in pairs]),
                             inp["w13"], inp["s13"])
    gu_rows = u16(layer.gateup[[int(s2d_h[t, k]) for t, k in pairs]])
    assert_bf16_close(gu_rows, ref_rows, f"{cfg.name} gate_up rows")


@pytest.mark.parametrize("cfg", synth.CONFIGS, ids=lambda c: c.name)
def test_fused_layout_scatter_full_size(mx, cfg):
    """moe_expand_layout_scatter at full size (in the benchmark's launch
    configuration) writes the same layout and the same expanded rows, bit for
    bit, as moe_expand_layout followed by moe_expand_scatter."""
    dev = torch.device("cuda")
    d = synth.generate(cfg, device=dev)
    nv = d["n_valid"]
    n_valid = torch.tensor([nv], dtype=torch.int32, device=dev)
    sl = mx.scale_layout_of(cfg.scale_mode)
    M_cap = int(mx.expanded_capacity(cfg.T, cfg.K, cfg.E, cfg.align))
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    lay = mx.expand_layout(d["topk_ids"], cfg.E, cfg.align, M_cap, n_valid=n_valid, status=status)
    xe, xs, rw = mx.expand_scatter(d["x_q"], d["x_s"], sl, d["topk_w"], lay, n_valid=n_valid,
                                   status=status)
    lay2, xe2, xs2, rw2 = mx.expand_layout_scatter(d["x_q"], d["x_s"], sl, d["topk_ids"],
                                                   d["topk_w"], cfg.E, cfg.align, M_cap,
                                                   n_valid=n_valid, status=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    total = int(lay.total.item())
    assert int(lay2.total.item()) == total
    for k in ("psum", "start", "tile_prefix", "m_indices", "src2dst"):
        assert torch.equal(getattr(lay, k), getattr(lay2, k)), k
    assert torch.equal(xe[:total], xe2[:total])
    assert torch.equal(rw[:total].view(torch.int32), rw2[:total].view(torch.int32))
    if cfg.scale_mode == "f32":
        assert torch.equal(xs[:total].view(torch.int32), xs2[:total].view(torch.int32))
    else:
        assert torch.equal(xs[:, :total], xs2[:, :total])
