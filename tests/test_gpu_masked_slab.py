"""GPU parity of the decode variant: the masked-slab bridges (bit-exact data
movement against a construction from the oracle's layout) and the whole layer
with the slab between the GEMMs against the oracle's row-weighted
arrangement; an expert with more rows than the slab holds is flagged and its
extra rows contribute nothing."""
import numpy as np
import pytest
import torch

import synth
from parity_util import assert_final_close, u16

pytestmark = pytest.mark.gpu

NAMES = ["mid_f32", "mid_ue8m0", "mid_zipf_ragged", "wide_e160_k12_ue8m0"]


@pytest.fixture(scope="module")
def mx():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from expanded_layout_expert_gb300 import build
    build.build()
    import expanded_layout_expert_gb300 as m
    return m


@pytest.fixture(scope="module")
def cases(orc):
    out = {}
    for name in NAMES:
        cfg = synth.config_by_name(name)
        d = synth.generate(cfg, device="cpu")
        inp = orc.to_numpy_inputs(d)
        M_cap = orc.expanded_capacity(cfg.T * cfg.K, cfg.E, cfg.align)
        ref = orc.run_layer(inp, M_cap, weighting="rows")
        g = {k: v.cuda() for k, v in d.items() if isinstance(v, torch.Tensor)}
        g["n_valid_dev"] = torch.tensor([d["n_valid"]], dtype=torch.int32, device="cuda")
        out[name] = dict(cfg=cfg, inp=inp, ref=ref, M_cap=M_cap, g=g)
    return out


def _counts(ref):
    lay = ref["layout"]
    return (lay["psum"] - lay["start"]).astype(np.int64), lay["start"].astype(np.int64)


@pytest.mark.parametrize("shrink", [False, True], ids=["fits", "overflow"])
@pytest.mark.parametrize("name", NAMES)
def test_expand_to_masked_slab(mx, cases, name, shrink):
    c = cases[name]
    cfg, ref = c["cfg"], c["ref"]
    sl = mx.scale_layout_of(cfg.scale_mode)
    cnt, start = _counts(ref)
    max_m = int(cnt.max()) + 5 if not shrink else max(1, int(cnt.max()) // 2)
    E, H, M = cfg.E, cfg.H, c["M_cap"]
    S = E * max_m
    xe = torch.zeros(M, H, dtype=torch.uint8)
    xe[: ref["total"]] = torch.from_numpy(ref["xe"][: ref["total"]])
    if sl == 0:
        xs = torch.zeros(M, H // 128, dtype=torch.float32)
        xs[: ref["total"]] = torch.from_numpy(ref["xe_s"][: ref["total"]])
    else:
        xs = torch.from_numpy(np.ascontiguousarray(ref["xe_s"]))
    xe, xs = xe.cuda(), xs.cuda()
    psum = torch.from_numpy(ref["layout"]["psum"]).cuda()
    st = torch.from_numpy(ref["layout"]["start"]).cuda()
    slab = torch.full((S, H), 0xAB, dtype=torch.uint8, device="cuda")
    ss = mx.new_scale(S, H // 128, sl, "cuda")
    ss.fill_(-7 if sl else 3.5)
    masked_m = torch.zeros(E, dtype=torch.int32, device="cuda")
    s_start = torch.zeros(E, dtype=torch.int32, device="cuda")
    s_tp = torch.zeros(E + 1, dtype=torch.int32, device="cuda")
    s_tot = torch.zeros(1, dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    L = mx.load()
    mx.check(L.moe_expand_to_masked_slab(xe.data_ptr(), xs.data_ptr(), sl, xs.shape[1], psum.data_ptr(),
                                         st.data_ptr(), E, H, max_m, slab.data_ptr(), ss.data_ptr(),
                                         ss.shape[1], masked_m.data_ptr(), s_start.data_ptr(),
                                         s_tp.data_ptr(), s_tot.data_ptr(), status.data_ptr(),
                                         torch.cuda.current_stream().cuda_stream), "slab")
    torch.cuda.synchronize()
    m = np.minimum(cnt, max_m)
    assert np.array_equal(masked_m.cpu().numpy(), m)
    assert np.array_equal(s_start.cpu().numpy(), np.arange(E) * max_m)
    tiles = (m + 127) // 128
    assert np.array_equal(s_tp.cpu().numpy(), np.concatenate([[0], np.cumsum(tiles)]))
    assert s_tot.item() == S
    assert status.item() == (-5 if (cnt > max_m).any() else 0)
    sb, ssh = slab.cpu().numpy(), ss.cpu().numpy()
    for e in range(E):
        used = min(int((m[e] + 127) // 128 * 128), max_m)
        rows = np.arange(e * max_m, e * max_m + m[e])
        src = start[e] + np.arange(m[e])
        assert np.array_equal(sb[rows], ref["xe"][src])
        assert not sb[e * max_m + m[e]: e * max_m + used].any(), "rest of the last tile is zero"
        assert (sb[e * max_m + used: (e + 1) * max_m] == 0xAB).all(), "unused rows untouched"
        if sl == 0:
            assert np.array_equal(ssh[rows].view(np.uint32), ref["xe_s"][src].view(np.uint32))
        else:
            assert np.array_equal(ssh[:, rows], ref["xe_s"][:, src])


@pytest.mark.parametrize("name", NAMES)
def test_masked_slab_to_expand(mx, cases, name):
    c = cases[name]
    cfg, ref, orc_M = c["cfg"], c["ref"], c["M_cap"]
    cnt, start = _counts(ref)
    max_m = max(1, int(cnt.max()) - 3)
    E, H = cfg.E, cfg.H
    rng = np.random.default_rng(3)
    slab_f = rng.standard_normal((E * max_m, H)).astype(np.float32)
    import oracle
    slab_bits = oracle.bf16_encode(slab_f.astype(np.float64))
    slab = torch.from_numpy(slab_bits.view(np.int16)).view(torch.bfloat16).cuda()
    w = ref["row_w"].astype(np.float32)
    out = torch.full((orc_M, H), float("nan"), dtype=torch.bfloat16, device="cuda")
    L = mx.load()
    psum = torch.from_numpy(ref["layout"]["psum"]).cuda()
    st = torch.from_numpy(ref["layout"]["start"]).cuda()
    tot = torch.tensor([ref["total"]], dtype=torch.int32, device="cuda")
    w_dev = torch.from_numpy(w).cuda()
    mx.check(L.moe_masked_slab_to_expand(slab.data_ptr(), max_m, psum.data_ptr(), st.data_ptr(),
                                         tot.data_ptr(), w_dev.data_ptr(), E, H, orc_M,
                                         out.data_ptr(), torch.cuda.current_stream().cuda_stream),
             "unslab")
    torch.cuda.synchronize()
    got = u16(out)
    want = np.zeros((ref["total"], H), np.uint16)
    vals = oracle.bf16_decode(slab_bits)
    for e in range(E):
        for j in range(min(int(cnt[e]), max_m)):
            r = start[e] + j
            prod = (vals[e * max_m + j].astype(np.float32) * w[r]).astype(np.float32)
            want[r] = oracle.bf16_encode(prod.astype(np.float64))
    assert np.array_equal(got[: ref["total"]], want)
    assert np.isnan(out[ref["total"]:].float().cpu().numpy()).all(), "rows past the total untouched"


@pytest.mark.parametrize("name", NAMES)
def test_masked_slab_layer_end_to_end(mx, cases, name):
    c = cases[name]
    cfg, g, ref = c["cfg"], c["g"], c["ref"]
    cnt, _ = _counts(ref)
    layer = mx.ExpandedMoELayer(g["w13"], g["s13"], g["w2"], g["s2"], K=cfg.K, align=cfg.align,
                                scale_mode=cfg.scale_mode, max_tokens=cfg.T,
                                masked_max_m=int(cnt.max()) + 3)
    y = layer.forward(g["x_q"], g["x_s"], g["topk_ids"], g["topk_w"], g["n_valid_dev"])
    torch.cuda.synchronize()
    assert layer.status.item() == 0
    nv = c["inp"]["n_valid"]
    assert_final_close(u16(y)[:nv], ref["y"][:nv], name)
