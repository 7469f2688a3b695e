"""Python access to the CPU oracle (moe_oracle.c).

TEST INFRASTRUCTURE ONLY: imported by tests/, by ``__graft_entry__.smoke()``
and by the CPU-baseline leg of ``bench.py``; the product package never
imports it. Arguments are numpy arrays; every function here is marshalling
around the C functions, plus ``run_layer`` which strings the C steps together
in the layer's order for shapes small enough to compute every row.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")

SCALE_F32 = 0
SCALE_UE8M0 = 1
BLOCK_M = 128

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile liboracle.so with gcc (C11, -O2, no fused multiply-add)."""
    os.makedirs(_BUILD, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH) or
             os.path.getmtime(_LIB_PATH) < max(os.path.getmtime(_SRC),
                                                os.path.getmtime(os.path.join(_HERE, "moe_oracle.h"))))
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math",
                               "-Wall", "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _declare(C.CDLL(build()))
    return _lib


P = C.c_void_p
I64 = C.c_int64
I32 = C.c_int


def _declare(L):
    L.orc_e4m3_decode.restype = C.c_double
    L.orc_e4m3_decode.argtypes = [C.c_uint8]
    L.orc_e4m3_encode.restype = C.c_uint8
    L.orc_e4m3_encode.argtypes = [C.c_float]
    L.orc_bf16_encode.restype = C.c_uint16
    L.orc_bf16_encode.argtypes = [C.c_double]
    L.orc_bf16_decode.restype = C.c_double
    L.orc_bf16_decode.argtypes = [C.c_uint16]
    L.orc_ue8m0_encode.restype = C.c_uint8
    L.orc_ue8m0_encode.argtypes = [C.c_float]
    L.orc_ue8m0_decode.restype = C.c_float
    L.orc_ue8m0_decode.argtypes = [C.c_uint8]
    for n in ("orc_e4m3_decode_array", "orc_e4m3_encode_array", "orc_bf16_encode_array",
              "orc_ue8m0_encode_array"):
        getattr(L, n).restype = None
        getattr(L, n).argtypes = [P, I64, P]
    L.orc_expanded_capacity.restype = I64
    L.orc_expanded_capacity.argtypes = [I64, I64, I64]
    L.orc_layout.restype = I32
    L.orc_layout.argtypes = [P, I64, I32, I32, I32, I64, I64, I32, P, P, P, P, P, P]
    L.orc_scatter.restype = I32
    L.orc_scatter.argtypes = [P, P, I32, I64, P, P, P, P, I64, I64, I32, I32, I32, I32,
                              P, P, I64, P]
    L.orc_gemm_rows.restype = I32
    L.orc_gemm_rows.argtypes = [P, I64, P, I32, I64, P, P, I64, P, P, I32, I32, I32, P, P]
    L.orc_act_quant_rows.restype = I32
    L.orc_act_quant_rows.argtypes = [P, I64, I32, P, I32, P, P, I64]
    L.orc_weight_rows.restype = I32
    L.orc_weight_rows.argtypes = [P, I64, I32, P]
    L.orc_combine.restype = I32
    L.orc_combine.argtypes = [P, P, P, I64, I64, I32, I32, P]
    L.orc_token_forward.restype = I32
    L.orc_token_forward.argtypes = [P, P, I32, I64, I64, P, P, I32, P, P, P, P, I32, I32, I32, P]
    return L


def _p(a):
    if a is None:
        return None
    assert isinstance(a, np.ndarray) and a.flags["C_CONTIGUOUS"], "contiguous numpy array expected"
    return a.ctypes.data


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def _check(rc, what):
    if rc != 0:
        raise RuntimeError(f"oracle {what} returned {rc}")


# ---- codecs -------------------------------------------------------------

def e4m3_decode(codes) -> np.ndarray:
    c = _c(codes, np.uint8)
    out = np.empty(c.shape, np.float64)
    lib().orc_e4m3_decode_array(_p(c), c.size, _p(out))
    return out


def e4m3_encode(values) -> np.ndarray:
    v = _c(values, np.float32)
    out = np.empty(v.shape, np.uint8)
    lib().orc_e4m3_encode_array(_p(v), v.size, _p(out))
    return out


def bf16_encode(values) -> np.ndarray:
    v = _c(values, np.float64)
    out = np.empty(v.shape, np.uint16)
    lib().orc_bf16_encode_array(_p(v), v.size, _p(out))
    return out


def bf16_decode(bits) -> np.ndarray:
    b = _c(bits, np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def ue8m0_encode(scales) -> np.ndarray:
    s = _c(scales, np.float32)
    out = np.empty(s.shape, np.uint8)
    lib().orc_ue8m0_encode_array(_p(s), s.size, _p(out))
    return out


def ue8m0_decode(b: int) -> float:
    return float(lib().orc_ue8m0_decode(int(b)))


def expanded_capacity(num_assignments: int, E: int, align: int) -> int:
    return int(lib().orc_expanded_capacity(num_assignments, E, align))


# ---- layer steps ---------------------------------------------------------

def layout(topk_ids, E, align, n_valid, M_cap, block_m=BLOCK_M):
    ids = _c(topk_ids, np.int32)
    T, K = ids.shape
    psum = np.zeros(E, np.int32)
    start = np.zeros(E, np.int32)
    total = np.zeros(1, np.int32)
    m_indices = np.full(M_cap, -7, np.int32)
    src2dst = np.full((T, K), -7, np.int32)
    tile_prefix = np.zeros(E + 1, np.int32)
    rc = lib().orc_layout(_p(ids), T, K, E, align, n_valid, M_cap, block_m, _p(psum), _p(start),
                          _p(total), _p(m_indices), _p(src2dst), _p(tile_prefix))
    return dict(rc=rc, psum=psum, start=start, total=int(total[0]), m_indices=m_indices,
                src2dst=src2dst, tile_prefix=tile_prefix)


def scatter(x_q, x_s, scale_layout, topk_w, lay, n_valid, E, align, M_cap):
    x_q = _c(x_q, np.uint8)
    T, H = x_q.shape
    K = lay["src2dst"].shape[1]
    G = H // 128
    if scale_layout == SCALE_F32:
        x_s = _c(x_s, np.float32)
        ld_xs = x_s.shape[1]
        xe_s = np.zeros((M_cap, G), np.float32)
        ld_xes = G
    else:
        x_s = _c(x_s, np.int32)
        ld_xs = x_s.shape[1]
        xe_s = np.zeros(((G + 3) // 4, M_cap), np.int32)
        ld_xes = M_cap
    xe = np.zeros((M_cap, H), np.uint8)
    row_w = np.zeros(M_cap, np.float32)
    w = _c(topk_w, np.float32)
    rc = lib().orc_scatter(_p(x_q), _p(x_s), scale_layout, ld_xs, _p(w), _p(lay["src2dst"]),
                           _p(lay["psum"]), _p(lay["start"]), n_valid, T, H, K, E, align,
                           _p(xe), _p(xe_s), ld_xes, _p(row_w))
    _check(rc, "scatter")
    return xe, xe_s, row_w


def gemm_rows(A, A_s, scale_layout, ld_as, rows, experts, W, W_s, want_f64=False):
    A = _c(A, np.uint8)
    lda = A.shape[1]
    rows = _c(rows, np.int64)
    experts = _c(experts, np.int32)
    W = _c(W, np.uint8)
    E, N, Kd = W.shape
    W_s = _c(W_s, np.float32 if scale_layout == SCALE_F32 else np.uint8)
    A_s = _c(A_s, np.float32 if scale_layout == SCALE_F32 else np.int32)
    out = np.zeros((rows.size, N), np.uint16)
    f64 = np.zeros((rows.size, N), np.float64) if want_f64 else None
    rc = lib().orc_gemm_rows(_p(A), lda, _p(A_s), scale_layout, ld_as, _p(rows), _p(experts),
                             rows.size, _p(W), _p(W_s), E, N, Kd, _p(out), _p(f64))
    _check(rc, "gemm_rows")
    return (out, f64) if want_f64 else out


def act_quant_rows(gu, row_w, scale_layout):
    gu = _c(gu, np.uint16)
    n, twoI = gu.shape
    I = twoI // 2
    G = I // 128
    di = np.zeros((n, I), np.uint8)
    if scale_layout == SCALE_F32:
        di_s = np.zeros((n, G), np.float32)
        ld = G
    else:
        di_s = np.zeros(((G + 3) // 4, n), np.int32)
        ld = n
    w = None if row_w is None else _c(row_w, np.float32)
    rc = lib().orc_act_quant_rows(_p(gu), n, I, _p(w), scale_layout, _p(di), _p(di_s), ld)
    _check(rc, "act_quant_rows")
    return di, di_s


def weight_rows(down, row_w):
    down = _c(down, np.uint16).copy()
    n, H = down.shape
    rc = lib().orc_weight_rows(_p(down), n, H, _p(_c(row_w, np.float32)))
    _check(rc, "weight_rows")
    return down


def combine(down, src2dst, row_w, n_valid, T):
    down = _c(down, np.uint16)
    H = down.shape[1]
    s2d = _c(src2dst, np.int32)
    K = s2d.shape[1]
    y = np.zeros((T, H), np.uint16)
    w = None if row_w is None else _c(row_w, np.float32)
    rc = lib().orc_combine(_p(down), _p(s2d), _p(w), n_valid, T, H, K, _p(y))
    _check(rc, "combine")
    return y


def token_forward(inp: dict, t: int) -> np.ndarray:
    """y[t] by the permutation-free path. ``inp`` holds numpy arrays."""
    sl = inp["scale_layout"]
    x_q, x_s = inp["x_q"], inp["x_s"]
    H = x_q.shape[1]
    E, twoI, _ = inp["w13"].shape
    I = twoI // 2
    ids = _c(inp["topk_ids"][t], np.int32)
    w = _c(inp["topk_w"][t], np.float32)
    y = np.zeros(H, np.uint16)
    rc = lib().orc_token_forward(_p(x_q), _p(x_s), sl, x_s.shape[1], t, _p(ids), _p(w), ids.size,
                                 _p(inp["w13"]), _p(inp["s13"]), _p(inp["w2"]), _p(inp["s2"]),
                                 E, H, I, _p(y))
    _check(rc, "token_forward")
    return y


def to_numpy_inputs(d: dict) -> dict:
    """Generator output (torch tensors) -> contiguous numpy arrays."""
    cfg = d["cfg"]
    out = {k: v.detach().cpu().contiguous().numpy() for k, v in d.items()
           if hasattr(v, "detach")}
    out["scale_layout"] = SCALE_UE8M0 if cfg.scale_mode == "ue8m0" else SCALE_F32
    out["n_valid"] = int(d["n_valid"])
    out["cfg"] = cfg
    return out


def run_layer(inp: dict, M_cap: int, weighting: str = "expanded") -> dict:
    """The whole expanded layer, every row, in the layer's order: layout,
    scatter, gate_up GEMM, activation + quant (+ fold), down GEMM, (ue8m0:
    output-row weighting), combine. Returns every intermediate.

    weighting "expanded": the top-k weight is folded into down_proj's fp32
    input scale, or on the ue8m0 path multiplies the down_proj output rows
    (SGLang PR 37261, Modifications/Core), and the combine sums unweighted.
    weighting "gather": the do_expand=False arrangement of the same PR's A/B
    baseline, where ep_gather applies the weights while summing
    (post_permute_deep_gemm_to_deepep_v2's non-expanded branch): no fold, no
    row weighting, y[t] = bf16(sum_k w[t,k] * down[row(t,k)]).
    weighting "rows": the decode masked-slab arrangement (masked_slab_to_expand
    takes the top-k weights): no fold on either scale layout, every down row
    multiplied by its weight and rounded to bf16, then the unweighted sum.
    On the ue8m0 path it is the same as "expanded"."""
    if weighting not in ("expanded", "gather", "rows"):
        raise ValueError(weighting)
    cfg = inp["cfg"]
    sl = inp["scale_layout"]
    nv = inp["n_valid"]
    T, H = inp["x_q"].shape
    lay = layout(inp["topk_ids"], cfg.E, cfg.align, nv, M_cap)
    _check(lay["rc"], "layout")
    xe, xe_s, row_w = scatter(inp["x_q"], inp["x_s"], sl, inp["topk_w"], lay, nv, cfg.E,
                              cfg.align, M_cap)
    total = lay["total"]
    rows = np.arange(total, dtype=np.int64)
    experts = lay["m_indices"][:total]
    ld_xes = xe_s.shape[1]
    gu = gemm_rows(xe, xe_s, sl, ld_xes, rows, experts, inp["w13"], inp["s13"])
    if weighting == "gather":
        di, di_s = act_quant_rows(gu, None, sl)
        down = gemm_rows(di, di_s, sl, di_s.shape[1], rows, experts, inp["w2"], inp["s2"])
        y = combine(down, lay["src2dst"], row_w, nv, T)
    elif weighting == "rows":
        di, di_s = act_quant_rows(gu, None, sl)
        down_u = gemm_rows(di, di_s, sl, di_s.shape[1], rows, experts, inp["w2"], inp["s2"])
        down = weight_rows(down_u, row_w[:total])
        y = combine(down, lay["src2dst"], None, nv, T)
    else:
        if sl == SCALE_F32:
            di, di_s = act_quant_rows(gu, row_w[:total], sl)
            down = gemm_rows(di, di_s, sl, di_s.shape[1], rows, experts, inp["w2"], inp["s2"])
        else:
            di, di_s = act_quant_rows(gu, None, sl)
            down_u = gemm_rows(di, di_s, sl, di_s.shape[1], rows, experts, inp["w2"], inp["s2"])
            down = weight_rows(down_u, row_w[:total])
        y = combine(down, lay["src2dst"], None, nv, T)
    return dict(layout=lay, xe=xe, xe_s=xe_s, row_w=row_w, gu=gu, di=di, di_s=di_s,
                down=down, y=y, total=total)
