"""The five workloads at full size, through ExpandedMoELayer (the launch
configuration the benchmark times), with every intermediate buffer filled
with garbage before the forward:

* layout: bit-exact against the oracle on every row (the oracle's layout is
  cheap at any size);
* scatter: every expanded row equals its token's bytes, scale and weight, and
  every alignment gap is zero (a property checked on all rows on the device);
* the fused gate_up + act+quant of the forward equals the stand-alone
  launches on every row, bit for bit;
* per non-empty expert, the first and the last valid row of its segment
  through gate_up, act+quant and down against the oracle, which computes
  those rows one by one from the layer's inputs (rows are independent, so an
  expanded row is the oracle's GEMM chain on its token and expert);
* the final output of at least 64 tokens (every active one if fewer), chosen
  to touch every expert,
  against the oracle's per-token path (rel-Frobenius <= 1e-2, max abs
  <= 5e-2);
* rows past n_valid are never written, the status word stays clean.

The oracle's calls run on a thread pool: they are C functions called
through ctypes, which releases the GIL.
"""
import concurrent.futures as cf
import os

import numpy as np
import pytest
import torch

import synth
from parity_util import assert_bf16_close, assert_final_close, bf16_val, rel_fro, u16

pytestmark = pytest.mark.gpu

N_TOKENS = 64


@pytest.fixture(scope="module")
def mx():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from expanded_layout_expert_gb300 import build
    build.build()
    import expanded_layout_expert_gb300 as m
    return m


@pytest.fixture(scope="module")
def pool():
    with cf.ThreadPoolExecutor(max_workers=max(1, os.cpu_count() or 1)) as ex:
        yield ex


def _sample_tokens(ids, nv, n, seed):
    """At least n valid tokens: one routed to each non-empty expert first,
    then random active tokens, plus the first inactive token and the last
    active one."""
    rng = np.random.default_rng(seed)
    live = ids[:nv]
    active = np.flatnonzero((live >= 0).any(1))
    inactive = np.flatnonzero(~(live >= 0).any(1))
    pick = set()
    for e in np.unique(live[live >= 0]):
        pick.add(int(rng.choice(np.flatnonzero((live == e).any(1)))))
    rest = np.setdiff1d(active, np.fromiter(pick, dtype=np.int64, count=len(pick)))
    need = max(0, n - len(pick))
    pick.update(int(t) for t in rng.choice(rest, size=min(need, rest.size), replace=False))
    if inactive.size:
        pick.add(int(inactive[0]))
    pick.add(int(active[-1]))
    return sorted(pick)


def _poison(layer):
    layer.xe.fill_(0xAB)
    layer.down_in.fill_(0x7F)
    layer.row_w.fill_(float("nan"))
    for s in (layer.xe_scale, layer.down_in_scale):
        if s.dtype == torch.float32:
            s.fill_(float("nan"))
        else:
            s.fill_(-1)
    for b in (layer.gateup, layer.down_out, layer.y):
        b.fill_(float("nan"))


def _oracle_row_chain(orc, inp, pairs, row_w, pool):
    """gate_up, act+quant (the fold on the fp32 path) and down of the
    expanded rows of the given (token, expert) pairs, each computed by the
    oracle from the layer's inputs. Returns (gu, di, di_s per row, down)."""
    sl = inp["scale_layout"]
    x_q, x_s = inp["x_q"], inp["x_s"]

    def one(i):
        t, e = pairs[i]
        gu = orc.gemm_rows(x_q, x_s, sl, x_s.shape[1], np.array([t]), np.array([e]),
                           inp["w13"], inp["s13"])
        w = np.array([row_w[i]], np.float32)
        di, di_s = orc.act_quant_rows(gu, w if sl == orc.SCALE_F32 else None, sl)
        down = orc.gemm_rows(di, di_s, sl, di_s.shape[1], np.array([0]), np.array([e]),
                             inp["w2"], inp["s2"])
        if sl != orc.SCALE_F32:
            down = orc.weight_rows(down, w)
        return gu[0], di[0], di_s, down[0]

    return list(pool.map(one, range(len(pairs))))


@pytest.mark.parametrize("cfg", synth.CONFIGS, ids=lambda c: c.name)
def test_workload_full_size(mx, orc, pool, cfg):
    dev = torch.device("cuda")
    d = synth.generate(cfg, device=dev)
    nv = d["n_valid"]
    n_valid = torch.tensor([nv], dtype=torch.int32, device=dev)
    layer = mx.ExpandedMoELayer(d["w13"], d["s13"], d["w2"], d["s2"], K=cfg.K, align=cfg.align,
                                scale_mode=cfg.scale_mode, max_tokens=cfg.T)
    _poison(layer)
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

    # scatter, every row, as a property on the device; the gaps held garbage
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
    if cfg.scale_mode == "f32":
        assert not layer.xe_scale[:total][gap].view(torch.int32).any()
    else:
        assert not layer.xe_scale[:, :total][:, gap].any()

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

    inp = orc.to_numpy_inputs(d)

    # per non-empty expert: the first and the last valid row of its segment
    start, psum = ref["start"], ref["psum"]
    row_tok = {}
    s2d_h = ref["src2dst"]
    for t, k in zip(*np.nonzero(s2d_h[:nv] >= 0)):
        row_tok[int(s2d_h[t, k])] = (int(t), int(k))
    pick_rows = []
    for e in range(cfg.E):
        if psum[e] > start[e]:
            pick_rows += sorted({int(start[e]), int(psum[e]) - 1})
    pairs = [(row_tok[r][0], int(ids[row_tok[r]])) for r in pick_rows]
    wts = [float(inp["topk_w"][row_tok[r]]) for r in pick_rows]
    chain = _oracle_row_chain(orc, inp, pairs, wts, pool)
    gu_ref = np.stack([c[0] for c in chain])
    assert_bf16_close(u16(gu[pick_rows]), gu_ref, f"{cfg.name} gate_up, first/last row per expert")
    di_ref = np.stack([c[1] for c in chain])
    di_got = layer.down_in[pick_rows].cpu().numpy()
    same = (di_got == di_ref) | ((di_got & 0x7F) == 0) & ((di_ref & 0x7F) == 0)
    assert same.mean() >= 0.999, f"{cfg.name}: {1 - same.mean():.2e} of fp8 codes differ"
    down_ref = np.stack([c[3] for c in chain])
    down_got = u16(layer.down_out[pick_rows])
    # rows whose codes all agree with the oracle's: the down GEMM alone, held
    # to the GEMM tolerance (ue8m0: weighting before vs after one rounding)
    exact = same.all(1)
    if exact.any():
        if cfg.scale_mode == "f32":
            assert_bf16_close(down_got[exact], down_ref[exact], f"{cfg.name} down rows")
        else:
            assert_bf16_close(down_got[exact], down_ref[exact], f"{cfg.name} down rows",
                              ulps=2, rel=2.0 ** -8)
    fro = rel_fro(bf16_val(down_got), bf16_val(down_ref))
    assert fro <= 1e-2, f"{cfg.name}: down rows rel_fro {fro:.3e}"
    print(f"{cfg.name}: {len(pick_rows)} expert rows ({int(exact.sum())} with identical codes), "
          f"down rel_fro {fro:.3e}")

    # final output of sampled tokens through the oracle's per-token path
    toks = _sample_tokens(ids, nv, N_TOKENS, cfg.seed)
    n_active = int((ids[:nv] >= 0).any(1).sum())
    assert len(toks) >= min(N_TOKENS, n_active)
    live = ids[toks]
    assert set(np.unique(live[live >= 0])) == set(np.unique(ids[:nv][ids[:nv] >= 0]))
    want = np.stack(list(pool.map(lambda t: orc.token_forward(inp, t), toks)))
    got = u16(y[toks])
    fro, mxabs = assert_final_close(got, want, cfg.name)
    print(f"{cfg.name}: {len(toks)} tokens rel_fro {fro:.3e} max_abs {mxabs:.3e}")


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
