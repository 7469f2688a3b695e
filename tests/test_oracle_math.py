"""Pins for the oracle's grouped GEMM, activation + quantisation, weight fold
and whole-layer composition.

The GEMM is checked against torch.matmul in float64 on decoded fp8 values
(a library routine the oracle does not use), silu against
torch.nn.functional.silu, the quantiser against its error bound and the
amax -> 448 property, the fold against the closed-form identity "scaling the
per-row input scale by w equals multiplying the output by w", and the
expanded layer against the per-token path that expands nothing.
"""
import numpy as np
import pytest
import torch

import synth


def _dec(codes):
    return torch.from_numpy(np.ascontiguousarray(codes)).view(torch.float8_e4m3fn).to(torch.float64)


def _finite_codes(rng, shape):
    c = rng.integers(0, 256, size=shape, dtype=np.uint8)
    c[(c & 0x7F) == 0x7F] = 0x3C       # drop the two NaN codes
    return c


def _pack_colmajor(bytes_rows):
    rows, G = bytes_rows.shape
    W = (G + 3) // 4
    out = np.zeros((W, rows), np.uint32)
    for g in range(G):
        out[g // 4] |= bytes_rows[:, g].astype(np.uint32) << (8 * (g % 4))
    return out.view(np.int32)


def test_gemm_special_case_is_a_plain_matmul(orc):
    rng = np.random.default_rng(3)
    n, N, Kd = 7, 384, 640
    A = _finite_codes(rng, (n, Kd))
    W = _finite_codes(rng, (1, N, Kd))
    A_s = np.ones((n, Kd // 128), np.float32)
    W_s = np.ones((1, N // 128, Kd // 128), np.float32)
    out, f64 = orc.gemm_rows(A, A_s, orc.SCALE_F32, Kd // 128, np.arange(n), np.zeros(n),
                             W, W_s, want_f64=True)
    ref = (_dec(A) @ _dec(W[0]).T).numpy()
    assert np.array_equal(f64, ref)          # every partial sum is exact in double
    # bf16 output: the nearest bf16 of the exact value (within half a bf16 ulp)
    got = orc.bf16_decode(out)
    assert (np.abs(got - ref) <= 2.0 ** -8 * np.abs(ref)).all()
    assert np.array_equal(out, orc.bf16_encode(ref))


@pytest.mark.parametrize("layout", ["f32", "ue8m0"])
def test_gemm_block_scales_and_experts(orc, layout):
    rng = np.random.default_rng(4)
    E, N, Kd, M = 3, 256, 384, 11
    KB, NB = Kd // 128, N // 128
    A = _finite_codes(rng, (M, Kd))
    W = _finite_codes(rng, (E, N, Kd))
    rows = rng.permutation(M)[:9].astype(np.int64)
    experts = rng.integers(0, E, size=9).astype(np.int32)
    if layout == "f32":
        A_s = rng.uniform(0.5, 4, (M, KB)).astype(np.float32)
        W_s = rng.uniform(0.5, 4, (E, NB, KB)).astype(np.float32)
        sa, sw = A_s.astype(np.float64), W_s.astype(np.float64)
        out, f64 = orc.gemm_rows(A, A_s, orc.SCALE_F32, KB, rows, experts, W, W_s, want_f64=True)
    else:
        ab = rng.integers(120, 135, (M, KB)).astype(np.uint8)
        wb = rng.integers(120, 135, (E, NB, KB)).astype(np.uint8)
        sa, sw = 2.0 ** (ab.astype(np.float64) - 127), 2.0 ** (wb.astype(np.float64) - 127)
        packed = _pack_colmajor(ab)
        out, f64 = orc.gemm_rows(A, packed, orc.SCALE_UE8M0, M, rows, experts, W, wb, want_f64=True)
    Ad, Wd = _dec(A).numpy(), _dec(W).numpy()
    for i, (r, e) in enumerate(zip(rows, experts)):
        terms = np.zeros((KB, N))
        for kb in range(KB):
            blk = slice(kb * 128, kb * 128 + 128)
            part = Ad[r, blk] @ Wd[e][:, blk].T
            terms[kb] = sa[r, kb] * np.repeat(sw[e][:, kb], 128) * part
        ref = terms.sum(0)
        bound = 1e-14 * np.abs(terms).sum(0) + 1e-300
        assert (np.abs(f64[i] - ref) <= bound).all()


def test_silu_and_quantiser(orc):
    rng = np.random.default_rng(5)
    n, I = 6, 512
    g = rng.standard_normal((n, I)) * 3
    u = rng.standard_normal((n, I))
    g[1, :128] = 0.0                     # an all-zero group: amax clamps to 1e-10
    u[1, :128] = 0.0
    gu = torch.from_numpy(np.concatenate([g, u], 1).astype(np.float32)).to(torch.bfloat16)
    gu_bits = gu.view(torch.int16).numpy().view(np.uint16)
    gd, ud = gu.to(torch.float64)[:, :I], gu.to(torch.float64)[:, I:]
    h_ref = (torch.nn.functional.silu(gd) * ud).numpy()
    di, di_s = orc.act_quant_rows(gu_bits, None, orc.SCALE_F32)
    q = _dec(di).numpy()
    s = np.repeat(di_s.astype(np.float64), 128, axis=1)
    # |q*s - h| <= half an e4m3 step of h/s (2^-4 relative, 2^-10 absolute in
    # units of s) plus the bf16 rounding of h (2^-9 relative)
    err = np.abs(q * s - h_ref)
    assert (err <= (2.0 ** -4 + 2.0 ** -8) * np.abs(h_ref) + 2.0 ** -10 * s + 1e-30).all()
    # the largest |h| of each group lands on +-448 exactly
    grp = np.abs(q).reshape(n, I // 128, 128).max(-1)
    assert ((grp == 448.0) | (di_s == np.float32(1e-10) / np.float32(448.0))).all()
    assert di_s[1, 0] == np.float32(1e-10) / np.float32(448.0) and (di[1, :128] & 0x7F == 0).all()
    assert (np.abs(q) <= 448).all()


def test_ue8m0_quantiser_scale_is_pow2_ceiling(orc):
    rng = np.random.default_rng(6)
    n, I = 5, 640
    gu = torch.from_numpy((rng.standard_normal((n, 2 * I)) * 2).astype(np.float32)).to(torch.bfloat16)
    bits = gu.view(torch.int16).numpy().view(np.uint16)
    di_f, s_f = orc.act_quant_rows(bits, None, orc.SCALE_F32)
    di_u, s_u = orc.act_quant_rows(bits, None, orc.SCALE_UE8M0)
    G = I // 128
    words = s_u.view(np.uint32)
    b = np.stack([(words[g // 4] >> (8 * (g % 4))) & 0xFF for g in range(G)], 1)
    pow2 = 2.0 ** (b.astype(np.float64) - 127)
    assert (pow2 >= s_f).all() and (pow2 / 2 < s_f).all()
    assert (words[G // 4] >> (8 * (G % 4)) == 0).all()        # unused lanes zero
    assert (np.abs(_dec(di_u).numpy()) <= 448).all()


def test_weight_fold_identity(orc):
    """Scaling down_proj's per-row input scale by w equals multiplying its
    output by w: exact in real arithmetic, within fp32's rounding of s*w."""
    rng = np.random.default_rng(7)
    n, I, H, E = 6, 384, 256, 2
    gu = torch.from_numpy((rng.standard_normal((n, 2 * I)) * 2).astype(np.float32)).to(torch.bfloat16)
    bits = gu.view(torch.int16).numpy().view(np.uint16)
    w = rng.uniform(0.01, 0.9, n).astype(np.float32)
    di0, s0 = orc.act_quant_rows(bits, None, orc.SCALE_F32)
    di1, s1 = orc.act_quant_rows(bits, w, orc.SCALE_F32)
    assert np.array_equal(di0, di1)
    assert np.array_equal(s1, (s0 * w[:, None]).astype(np.float32))
    W2 = _finite_codes(rng, (E, H, I))
    S2 = rng.uniform(1e-3, 1e-2, (E, H // 128, I // 128)).astype(np.float32)
    ex = rng.integers(0, E, n).astype(np.int32)
    _, f0 = orc.gemm_rows(di0, s0, orc.SCALE_F32, I // 128, np.arange(n), ex, W2, S2, want_f64=True)
    _, f1 = orc.gemm_rows(di1, s1, orc.SCALE_F32, I // 128, np.arange(n), ex, W2, S2, want_f64=True)
    ref = f0 * w[:, None].astype(np.float64)
    # per element: each of the I/128 terms carries one fp32 rounding (2^-24)
    termsum = np.zeros_like(f0)
    q = _dec(di0).numpy()
    for i in range(n):
        for kb in range(I // 128):
            blk = slice(kb * 128, kb * 128 + 128)
            part = q[i, blk] @ _dec(W2[ex[i]]).numpy()[:, blk].T
            termsum[i] += np.abs(s1[i, kb] * np.repeat(S2[ex[i]][:, kb], 128) * part)
    assert (np.abs(f1 - ref) <= 2.0 ** -23 * termsum + 1e-300).all()
    rel = np.linalg.norm(f1 - ref) / np.linalg.norm(ref)
    assert rel <= 2.0 ** -23


@pytest.fixture(scope="module")
def layer_runs(orc):
    runs = {}
    for cfg in synth.PARITY_CONFIGS:
        inp = orc.to_numpy_inputs(synth.generate(cfg))
        M_cap = orc.expanded_capacity(cfg.T * cfg.K, cfg.E, cfg.align)
        runs[cfg.name] = (inp, orc.run_layer(inp, M_cap), M_cap)
    return runs


@pytest.mark.parametrize("name", [c.name for c in synth.PARITY_CONFIGS])
def test_expanded_layer_equals_per_token_path(orc, layer_runs, name):
    inp, out, _ = layer_runs[name]
    for t in range(inp["n_valid"]):
        assert np.array_equal(orc.token_forward(inp, t), out["y"][t]), t


def test_combine_sums_the_k_contributions(orc, layer_runs):
    inp, out, _ = layer_runs["mid_f32"]
    sub = dict(inp)
    for t in range(0, 40):
        ids = inp["topk_ids"][t]
        if (ids < 0).all():
            assert (out["y"][t] == 0).all()
            continue
        parts = []
        for k in range(ids.size):
            one = dict(sub)
            only = -np.ones_like(inp["topk_ids"])
            only[t, k] = ids[k]
            one["topk_ids"] = only
            parts.append(orc.bf16_decode(orc.token_forward(one, t)))
        assert np.array_equal(orc.bf16_encode(np.sum(parts, 0)), out["y"][t])


def test_inactive_tokens_give_zero(orc, layer_runs):
    inp, out, _ = layer_runs["mid_zipf_ragged"]
    off = (inp["topk_ids"][:inp["n_valid"]] < 0).all(1)
    assert off.sum() > 0
    assert (out["y"][:inp["n_valid"]][off] == 0).all()


def test_poisoned_tail_changes_nothing(orc, layer_runs):
    inp, out, M_cap = layer_runs["mid_padded"]
    nv = inp["n_valid"]
    bad = dict(inp)
    rng = np.random.default_rng(8)
    bad["x_q"] = inp["x_q"].copy()
    bad["x_q"][nv:] = 0x7F                       # NaN codes
    bad["x_s"] = inp["x_s"].copy()
    bad["x_s"][nv:] = np.float32(np.nan)
    bad["topk_ids"] = inp["topk_ids"].copy()
    bad["topk_ids"][nv:] = rng.integers(0, inp["cfg"].E, bad["topk_ids"][nv:].shape)
    bad["topk_w"] = inp["topk_w"].copy()
    bad["topk_w"][nv:] = np.float32(np.inf)
    out2 = orc.run_layer(bad, M_cap)
    assert np.array_equal(out2["y"][:nv], out["y"][:nv])
    for key in ("xe", "gu", "di", "down"):
        assert np.array_equal(out2[key], out[key])


def test_gather_weighting_differs_from_the_fold_only_in_the_stored_scale(orc, layer_runs):
    """The do_expand=False arrangement (weights applied while gathering) runs
    the same GEMMs on the same codes: gate_up is identical, the fp8 codes are
    identical, and the fold's stored scale is exactly fl(s * w)."""
    inp, out, M_cap = layer_runs["mid_f32"]
    g = orc.run_layer(inp, M_cap, weighting="gather")
    tot = out["total"]
    assert np.array_equal(g["gu"], out["gu"])
    assert np.array_equal(g["di"], out["di"])
    w = out["row_w"][:tot].astype(np.float32)
    folded = (g["di_s"].astype(np.float32) * w[:, None]).astype(np.float32)
    assert np.array_equal(folded.view(np.uint32), out["di_s"].view(np.uint32))
    nv = inp["n_valid"]
    a = orc.bf16_decode(g["y"][:nv])
    b = orc.bf16_decode(out["y"][:nv])
    assert np.linalg.norm(a - b) <= 1e-2 * np.linalg.norm(b)


def test_weighted_combine_invariants(orc, layer_runs):
    """Unit weights give the unweighted sum bit for bit; weights of 2 (exact
    in every format) give twice it bit for bit; a -1 pair adds nothing."""
    inp, out, _ = layer_runs["mid_zipf_ragged"]
    nv, T = inp["n_valid"], inp["topk_ids"].shape[0]
    s2d = out["layout"]["src2dst"]
    down = out["down"]
    ones = np.ones(out["row_w"].shape, np.float32)
    y0 = orc.combine(down, s2d, None, nv, T)
    assert np.array_equal(orc.combine(down, s2d, ones, nv, T), y0)
    y2 = orc.combine(down, s2d, 2 * ones, nv, T)
    assert np.array_equal(orc.bf16_decode(y2), 2 * orc.bf16_decode(y0))
    assert np.array_equal(y0, out["y"])


def test_gather_layer_equals_sum_of_weighted_single_pair_paths(orc, layer_runs):
    """Gather weighting on tiny inputs, against the definition pair by pair:
    y[t] = bf16(sum_k w[t,k] * f(x_t, e_k)), f the unweighted expert FFN taken
    as the layer output of that one pair with weight 1."""
    inp, out, M_cap = layer_runs["tiny_h512"]
    g = orc.run_layer(inp, M_cap, weighting="gather")
    ids, w = inp["topk_ids"], inp["topk_w"]
    for t in range(0, 12):
        if (ids[t] < 0).all():
            assert (g["y"][t] == 0).all()
            continue
        acc = np.zeros(inp["x_q"].shape[1])
        for k in range(ids.shape[1]):
            if ids[t, k] < 0:
                continue
            one = dict(inp)
            only = -np.ones_like(ids)
            only[t, k] = ids[t, k]
            one["topk_ids"] = only
            unit = inp["topk_w"].copy()
            unit[t, k] = 1.0
            one["topk_w"] = unit
            acc += float(w[t, k]) * orc.bf16_decode(orc.token_forward(one, t))
        assert np.array_equal(orc.bf16_encode(acc), g["y"][t]), t


def test_rows_weighting_pins(orc, layer_runs):
    """The decode arrangement (each down row weighted and rounded, then an
    unweighted sum): on ue8m0 it is the expanded layer itself; on fp32 scales
    it is, token by token, bf16(sum_k bf16(w_k * f(x_t, e_k))) with f the
    unweighted pair path, and its codes are the gather arrangement's."""
    inp, out, M_cap = layer_runs["mid_ue8m0"]
    r = orc.run_layer(inp, M_cap, weighting="rows")
    assert np.array_equal(r["y"], out["y"])
    inp, out, M_cap = layer_runs["tiny_h512"]
    r = orc.run_layer(inp, M_cap, weighting="rows")
    g = orc.run_layer(inp, M_cap, weighting="gather")
    assert np.array_equal(r["di"], g["di"]) and np.array_equal(r["di_s"], g["di_s"])
    ids, w = inp["topk_ids"], inp["topk_w"]
    for t in range(0, 12):
        acc = np.zeros(inp["x_q"].shape[1])
        for k in range(ids.shape[1]):
            if ids[t, k] < 0:
                continue
            one = dict(inp)
            only = -np.ones_like(ids)
            only[t, k] = ids[t, k]
            one["topk_ids"] = only
            unit = inp["topk_w"].copy()
            unit[t, k] = 1.0
            one["topk_w"] = unit
            f = orc.bf16_decode(orc.token_forward(one, t))
            acc += orc.bf16_decode(orc.bf16_encode(f * float(w[t, k])))
        assert np.array_equal(orc.bf16_encode(acc), r["y"][t]), t
