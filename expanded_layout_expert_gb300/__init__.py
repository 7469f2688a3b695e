"""Expanded-layout MoE prefill layer on GB300 (sm_103a).

A thin binding over libmoe_expand.so (include/moe_expand.h): each function
marshals torch tensors (device memory, owned by the caller) and the current
CUDA stream into one C call; every step of the layer runs in the library's
CUDA kernels. ``ExpandedMoELayer`` strings the calls together with buffers
allocated once.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import torch

from . import _capi
from ._capi import (MOE_BLOCK_M, MOE_FFN_UNFUSED, MOE_FOLD_WEIGHT_INTO_SCALE,
                    MOE_GEMM_PER_KBLOCK_PROMOTION,
                    MOE_GEMM_TILE_N128,
                    MOE_SCALE_F32_ROWMAJOR, MOE_SCALE_UE8M0_PACKED_COLMAJOR,
                    MOE_WEIGHT_OUTPUT_ROWS, MoEError, check, load)

__all__ = [
    "expanded_capacity", "workspace_size", "expand_layout", "expand_scatter",
    "expand_layout_scatter", "grouped_gemm",
    "act_quant", "grouped_gemm_act_quant", "grouped_ffn", "combine", "ExpandedMoELayer",
    "HostPipeline", "CapturedForward", "Layout",
    "MoEError",
    "MOE_SCALE_F32_ROWMAJOR", "MOE_SCALE_UE8M0_PACKED_COLMAJOR", "MOE_FOLD_WEIGHT_INTO_SCALE",
    "MOE_WEIGHT_OUTPUT_ROWS", "MOE_GEMM_TILE_N128",
    "MOE_GEMM_PER_KBLOCK_PROMOTION", "MOE_FFN_UNFUSED", "MOE_BLOCK_M",
    "scale_layout_of",
]


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("contiguous tensor expected")
    return t.data_ptr()


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def scale_layout_of(mode: str) -> int:
    return MOE_SCALE_UE8M0_PACKED_COLMAJOR if mode == "ue8m0" else MOE_SCALE_F32_ROWMAJOR


def expanded_capacity(T: int, K: int, E: int, align: int) -> int:
    return int(load().moe_expanded_capacity(T, K, E, align))


def workspace_size(T: int, K: int, E: int) -> int:
    return int(load().moe_workspace_size(T, K, E))


@dataclasses.dataclass
class Layout:
    psum: torch.Tensor
    start: torch.Tensor
    total: torch.Tensor        # int32 [1], on the device
    m_indices: torch.Tensor
    src2dst: torch.Tensor
    tile_prefix: torch.Tensor
    E: int
    align: int
    M_cap: int


def new_scale(rows: int, G: int, layout: int, device) -> torch.Tensor:
    if layout == MOE_SCALE_F32_ROWMAJOR:
        return torch.zeros(rows, G, dtype=torch.float32, device=device)
    return torch.zeros((G + 3) // 4, rows, dtype=torch.int32, device=device)


def scale_ld(s: torch.Tensor, layout: int) -> int:
    return s.shape[1]


def expand_layout(topk_ids: torch.Tensor, E: int, align: int, M_cap: int,
                  n_valid: Optional[torch.Tensor] = None, ws: Optional[torch.Tensor] = None,
                  status: Optional[torch.Tensor] = None, out: Optional[Layout] = None,
                  stream=None) -> Layout:
    T, K = topk_ids.shape
    dev = topk_ids.device
    if out is None:
        out = Layout(psum=torch.empty(E, dtype=torch.int32, device=dev),
                     start=torch.empty(E, dtype=torch.int32, device=dev),
                     total=torch.empty(1, dtype=torch.int32, device=dev),
                     m_indices=torch.empty(M_cap, dtype=torch.int32, device=dev),
                     src2dst=torch.empty(T, K, dtype=torch.int32, device=dev),
                     tile_prefix=torch.empty(E + 1, dtype=torch.int32, device=dev),
                     E=E, align=align, M_cap=M_cap)
    if ws is None:
        ws = torch.zeros(workspace_size(T, K, E), dtype=torch.uint8, device=dev)
    rc = load().moe_expand_layout(_ptr(topk_ids), T, K, E, align, _ptr(n_valid), M_cap,
                                  _ptr(out.psum), _ptr(out.start), _ptr(out.total),
                                  _ptr(out.m_indices), _ptr(out.src2dst), _ptr(out.tile_prefix),
                                  _ptr(ws), ws.numel(), _ptr(status), _stream(stream))
    check(rc, "moe_expand_layout")
    return out


def expand_scatter(x_q: torch.Tensor, x_scale: torch.Tensor, scale_layout: int,
                   topk_w: torch.Tensor, lay: Layout, n_valid: Optional[torch.Tensor] = None,
                   xe: Optional[torch.Tensor] = None, xe_scale: Optional[torch.Tensor] = None,
                   row_w: Optional[torch.Tensor] = None, status: Optional[torch.Tensor] = None,
                   stream=None):
    T, H = x_q.shape
    K = topk_w.shape[1]
    dev = x_q.device
    if xe is None:
        xe = torch.zeros(lay.M_cap, H, dtype=torch.uint8, device=dev)
    if xe_scale is None:
        xe_scale = new_scale(lay.M_cap, H // 128, scale_layout, dev)
    if row_w is None:
        row_w = torch.zeros(lay.M_cap, dtype=torch.float32, device=dev)
    rc = load().moe_expand_scatter(_ptr(x_q), _ptr(x_scale), scale_layout, x_scale.shape[1],
                                   _ptr(topk_w), _ptr(lay.src2dst), _ptr(lay.psum),
                                   _ptr(lay.start), _ptr(n_valid), T, H, K, lay.E, lay.align,
                                   lay.M_cap, _ptr(xe), _ptr(xe_scale), xe_scale.shape[1],
                                   _ptr(row_w), _ptr(status), _stream(stream))
    check(rc, "moe_expand_scatter")
    return xe, xe_scale, row_w


def expand_layout_scatter(x_q: torch.Tensor, x_scale: torch.Tensor, scale_layout: int,
                          topk_ids: torch.Tensor, topk_w: torch.Tensor, E: int, align: int,
                          M_cap: int, n_valid: Optional[torch.Tensor] = None,
                          ws: Optional[torch.Tensor] = None, status: Optional[torch.Tensor] = None,
                          out: Optional[Layout] = None, xe: Optional[torch.Tensor] = None,
                          xe_scale: Optional[torch.Tensor] = None,
                          row_w: Optional[torch.Tensor] = None, stream=None):
    """The layout and the expand-scatter in one call (one cooperative
    launch when the grid holds every 2048-pair chunk); same outputs as
    expand_layout followed by expand_scatter. Returns (layout, xe, xe_scale,
    row_w)."""
    T, H = x_q.shape
    K = topk_ids.shape[1]
    dev = x_q.device
    if out is None:
        out = Layout(psum=torch.empty(E, dtype=torch.int32, device=dev),
                     start=torch.empty(E, dtype=torch.int32, device=dev),
                     total=torch.empty(1, dtype=torch.int32, device=dev),
                     m_indices=torch.empty(M_cap, dtype=torch.int32, device=dev),
                     src2dst=torch.empty(T, K, dtype=torch.int32, device=dev),
                     tile_prefix=torch.empty(E + 1, dtype=torch.int32, device=dev),
                     E=E, align=align, M_cap=M_cap)
    if ws is None:
        ws = torch.zeros(workspace_size(T, K, E), dtype=torch.uint8, device=dev)
    if xe is None:
        xe = torch.zeros(M_cap, H, dtype=torch.uint8, device=dev)
    if xe_scale is None:
        xe_scale = new_scale(M_cap, H // 128, scale_layout, dev)
    if row_w is None:
        row_w = torch.zeros(M_cap, dtype=torch.float32, device=dev)
    rc = load().moe_expand_layout_scatter(
        _ptr(topk_ids), _ptr(topk_w), _ptr(x_q), _ptr(x_scale), scale_layout, x_scale.shape[1], T,
        H, K, E, align, _ptr(n_valid), M_cap, _ptr(out.psum), _ptr(out.start), _ptr(out.total),
        _ptr(out.m_indices), _ptr(out.src2dst), _ptr(out.tile_prefix), _ptr(xe), _ptr(xe_scale),
        xe_scale.shape[1], _ptr(row_w), _ptr(ws), ws.numel(), _ptr(status), _stream(stream))
    check(rc, "moe_expand_layout_scatter")
    return out, xe, xe_scale, row_w


def grouped_gemm(A: torch.Tensor, A_scale: torch.Tensor, scale_layout: int, lay: Layout,
                 W: torch.Tensor, W_scale: torch.Tensor, row_w: Optional[torch.Tensor] = None,
                 flags: int = 0, out: Optional[torch.Tensor] = None,
                 status: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    M_cap, Kd = A.shape
    E, N, _ = W.shape
    if out is None:
        out = torch.zeros(M_cap, N, dtype=torch.bfloat16, device=A.device)
    rc = load().moe_grouped_gemm(_ptr(A), _ptr(A_scale), scale_layout, A_scale.shape[1],
                                 _ptr(lay.start), _ptr(lay.tile_prefix), _ptr(lay.total),
                                 _ptr(W), _ptr(W_scale), _ptr(row_w), flags, E, N, Kd, M_cap,
                                 _ptr(out), _ptr(status), _stream(stream))
    check(rc, "moe_grouped_gemm")
    return out


def act_quant(gu: torch.Tensor, row_w: Optional[torch.Tensor], flags: int, scale_layout: int,
              total: torch.Tensor, di: Optional[torch.Tensor] = None,
              di_scale: Optional[torch.Tensor] = None, status: Optional[torch.Tensor] = None,
              stream=None):
    M_cap, twoI = gu.shape
    I = twoI // 2
    if di is None:
        di = torch.zeros(M_cap, I, dtype=torch.uint8, device=gu.device)
    if di_scale is None:
        di_scale = new_scale(M_cap, I // 128, scale_layout, gu.device)
    rc = load().moe_act_quant(_ptr(gu), I, _ptr(row_w), flags, scale_layout, _ptr(total), M_cap,
                              _ptr(di), _ptr(di_scale), di_scale.shape[1], _ptr(status),
                              _stream(stream))
    check(rc, "moe_act_quant")
    return di, di_scale


def grouped_gemm_act_quant(A: torch.Tensor, A_scale: torch.Tensor, scale_layout: int, lay: Layout,
                           W13: torch.Tensor, W13_scale: torch.Tensor, flags: int = 0,
                           row_w: Optional[torch.Tensor] = None,
                           di: Optional[torch.Tensor] = None, di_scale: Optional[torch.Tensor] = None,
                           status: Optional[torch.Tensor] = None, stream=None):
    """gate_up GEMM with silu*mul and the fp8 quantiser (and, with
    MOE_FOLD_WEIGHT_INTO_SCALE, the weight fold) in its epilogue."""
    M_cap, H = A.shape
    E, twoI, _ = W13.shape
    I = twoI // 2
    if di is None:
        di = torch.zeros(M_cap, I, dtype=torch.uint8, device=A.device)
    if di_scale is None:
        di_scale = new_scale(M_cap, I // 128, scale_layout, A.device)
    rc = load().moe_grouped_gemm_act_quant(_ptr(A), _ptr(A_scale), scale_layout, A_scale.shape[1],
                                           _ptr(lay.start), _ptr(lay.tile_prefix), _ptr(lay.total),
                                           _ptr(W13), _ptr(W13_scale), _ptr(row_w), flags, E, I, H, M_cap,
                                           _ptr(di), _ptr(di_scale), di_scale.shape[1], _ptr(status),
                                           _stream(stream))
    check(rc, "moe_grouped_gemm_act_quant")
    return di, di_scale


def grouped_ffn(xe, xe_scale, scale_layout: int, lay: Layout, w13, s13, w2, s2, row_w, flags: int,
                gateup=None, down_in=None, down_in_scale=None, down_out=None, status=None,
                stream=None):
    M_cap, H = xe.shape
    E, twoI, _ = w13.shape
    I = twoI // 2
    dev = xe.device
    if gateup is None:
        gateup = torch.zeros(M_cap, twoI, dtype=torch.bfloat16, device=dev)
    if down_in is None:
        down_in = torch.zeros(M_cap, I, dtype=torch.uint8, device=dev)
    if down_in_scale is None:
        down_in_scale = new_scale(M_cap, I // 128, scale_layout, dev)
    if down_out is None:
        down_out = torch.zeros(M_cap, H, dtype=torch.bfloat16, device=dev)
    rc = load().moe_grouped_ffn(_ptr(xe), _ptr(xe_scale), xe_scale.shape[1], scale_layout,
                                _ptr(lay.start), _ptr(lay.tile_prefix), _ptr(lay.total),
                                _ptr(w13), _ptr(s13), _ptr(w2), _ptr(s2), _ptr(row_w), flags,
                                E, H, I, M_cap, _ptr(gateup), _ptr(down_in), _ptr(down_in_scale),
                                down_in_scale.shape[1], _ptr(down_out), _ptr(status),
                                _stream(stream))
    check(rc, "moe_grouped_ffn")
    return gateup, down_in, down_in_scale, down_out


def combine(down: torch.Tensor, src2dst: torch.Tensor, row_w: Optional[torch.Tensor],
            n_valid: Optional[torch.Tensor], out: torch.Tensor, stream=None) -> torch.Tensor:
    T, K = src2dst.shape
    H = down.shape[1]
    rc = load().moe_combine(_ptr(down), _ptr(src2dst), _ptr(row_w), _ptr(n_valid), T, H, K,
                            _ptr(out), _stream(stream))
    check(rc, "moe_combine")
    return out


class ExpandedMoELayer:
    """The whole expanded prefill layer for up to ``max_tokens`` token rows,
    with every intermediate buffer allocated once.

    forward(x_q, x_scale, topk_ids, topk_w, n_valid) -> y bf16 [T, H]
      x_q      uint8 [T, H] fp8 e4m3 codes
      x_scale  fp32 [T, H/128] (scale_mode "f32") or int32 [ceil(H/512), T]
               packed ue8m0 exponents (scale_mode "ue8m0")
      topk_ids int32 [T, K], -1 = no pair; topk_w fp32 [T, K]
      n_valid  optional int32 [1] device tensor: rows >= n_valid are padding
    weighting "expanded" (default): on the fp32 path the top-k weight is
    folded into down_proj's input scale; on the ue8m0 path it multiplies the
    down_proj output rows; the combine sums unweighted.
    weighting "gather": the do_expand=False arrangement (ep_gather): no fold,
    the combine multiplies each pair's row by its weight while summing.
    masked_max_m: the decode variant. Between the GEMMs each expert's rows
    sit in a fixed-height slab of masked_max_m rows (moe_expand_to_masked_slab
    / moe_masked_slab_to_expand); the weight multiplies each pair's down row
    on the way back (no fold); an expert with more rows than masked_max_m
    drops the extra ones and flags the status word.
    fuse_layout_scatter (default True): run the layout and the
    expand-scatter as one moe_expand_layout_scatter call (one cooperative
    launch when the grid holds every 2048-pair chunk) instead of
    moe_expand_layout + moe_expand_scatter; the outputs are the same bit for
    bit.
    """

    def __init__(self, w13, s13, w2, s2, *, K: int, align: int, scale_mode: str,
                 max_tokens: int, device=None, weighting: str = "expanded",
                 masked_max_m: Optional[int] = None, fuse_layout_scatter: bool = True):
        self.w13, self.s13, self.w2, self.s2 = w13, s13, w2, s2
        self.E, twoI, self.H = w13.shape
        self.I = twoI // 2
        self.K, self.align = K, align
        self.scale_mode = scale_mode
        self.sl = scale_layout_of(scale_mode)
        if weighting not in ("expanded", "gather"):
            raise ValueError(f"weighting must be 'expanded' or 'gather', got {weighting!r}")
        if masked_max_m is not None and weighting != "expanded":
            raise ValueError("the masked-slab path weights rows after the slab; use the default weighting")
        self.weighting = weighting
        self.masked_max_m = masked_max_m
        self.fuse_layout_scatter = bool(fuse_layout_scatter)
        if weighting == "gather" or masked_max_m is not None:
            self.flags = 0
        else:
            self.flags = MOE_WEIGHT_OUTPUT_ROWS if scale_mode == "ue8m0" else MOE_FOLD_WEIGHT_INTO_SCALE
        self.T = max_tokens
        dev = device if device is not None else w13.device
        self.device = dev
        self.M_cap = expanded_capacity(max_tokens, K, self.E, align)
        E, H, I, M = self.E, self.H, self.I, self.M_cap
        self.ws = torch.zeros(workspace_size(max_tokens, K, E), dtype=torch.uint8, device=dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        self.lay = Layout(psum=torch.zeros(E, dtype=torch.int32, device=dev),
                          start=torch.zeros(E, dtype=torch.int32, device=dev),
                          total=torch.zeros(1, dtype=torch.int32, device=dev),
                          m_indices=torch.zeros(M, dtype=torch.int32, device=dev),
                          src2dst=torch.zeros(max_tokens, K, dtype=torch.int32, device=dev),
                          tile_prefix=torch.zeros(E + 1, dtype=torch.int32, device=dev),
                          E=E, align=align, M_cap=M)
        self.xe = torch.zeros(M, H, dtype=torch.uint8, device=dev)
        self.xe_scale = new_scale(M, H // 128, self.sl, dev)
        self.row_w = torch.zeros(M, dtype=torch.float32, device=dev)
        self._gateup = None  # bf16 [M_cap, 2I], only for the stand-alone gate_up
        self.down_in = torch.zeros(M, I, dtype=torch.uint8, device=dev)
        self.down_in_scale = new_scale(M, I // 128, self.sl, dev)
        self.down_out = torch.zeros(M, H, dtype=torch.bfloat16, device=dev)
        self.y = torch.zeros(max_tokens, H, dtype=torch.bfloat16, device=dev)
        if masked_max_m is not None:
            # decode variant: fixed-height per-expert slabs between the GEMMs
            S = E * masked_max_m
            self.slab = torch.zeros(S, H, dtype=torch.uint8, device=dev)
            self.slab_scale = new_scale(S, H // 128, self.sl, dev)
            self.masked_m = torch.zeros(E, dtype=torch.int32, device=dev)
            self.slab_lay = Layout(psum=self.masked_m,
                                   start=torch.zeros(E, dtype=torch.int32, device=dev),
                                   total=torch.zeros(1, dtype=torch.int32, device=dev),
                                   m_indices=torch.zeros(0, dtype=torch.int32, device=dev),
                                   src2dst=torch.zeros(0, dtype=torch.int32, device=dev),
                                   tile_prefix=torch.zeros(E + 1, dtype=torch.int32, device=dev),
                                   E=E, align=1, M_cap=S)
            self.slab_di = torch.zeros(S, I, dtype=torch.uint8, device=dev)
            self.slab_di_scale = new_scale(S, I // 128, self.sl, dev)
            self.slab_out = torch.zeros(S, H, dtype=torch.bfloat16, device=dev)

    def forward(self, x_q, x_scale, topk_ids, topk_w, n_valid=None, stream=None,
                out: Optional[torch.Tensor] = None) -> torch.Tensor:
        """y (self.y, or ``out``: bf16 [T, H]; rows >= n_valid not written)."""
        T = x_q.shape[0]
        y = self.y if out is None else out
        if y.shape != (self.T, self.H) or y.dtype != torch.bfloat16 or not y.is_contiguous():
            raise ValueError("out must be a contiguous bf16 [T, H] tensor")
        if T != self.T:
            raise ValueError(f"layer was built for {self.T} token rows, got {T}")
        L = load()
        s = _stream(stream)
        lay = self.lay
        if self.fuse_layout_scatter:
            check(L.moe_expand_layout_scatter(
                _ptr(topk_ids), _ptr(topk_w), _ptr(x_q), _ptr(x_scale), self.sl, x_scale.shape[1],
                T, self.H, self.K, self.E, self.align, _ptr(n_valid), self.M_cap, _ptr(lay.psum),
                _ptr(lay.start), _ptr(lay.total), _ptr(lay.m_indices), _ptr(lay.src2dst),
                _ptr(lay.tile_prefix), _ptr(self.xe), _ptr(self.xe_scale), self.xe_scale.shape[1],
                _ptr(self.row_w), _ptr(self.ws), self.ws.numel(), _ptr(self.status), s),
                "moe_expand_layout_scatter")
        else:
            check(L.moe_expand_layout(_ptr(topk_ids), T, self.K, self.E, self.align,
                                      _ptr(n_valid), self.M_cap, _ptr(lay.psum), _ptr(lay.start),
                                      _ptr(lay.total), _ptr(lay.m_indices), _ptr(lay.src2dst),
                                      _ptr(lay.tile_prefix), _ptr(self.ws), self.ws.numel(),
                                      _ptr(self.status), s), "moe_expand_layout")
            check(L.moe_expand_scatter(_ptr(x_q), _ptr(x_scale), self.sl, x_scale.shape[1],
                                       _ptr(topk_w), _ptr(lay.src2dst), _ptr(lay.psum),
                                       _ptr(lay.start), _ptr(n_valid), T, self.H, self.K, self.E,
                                       self.align, self.M_cap, _ptr(self.xe), _ptr(self.xe_scale),
                                       self.xe_scale.shape[1], _ptr(self.row_w),
                                       _ptr(self.status), s), "moe_expand_scatter")
        if self.masked_max_m is not None:
            self._slab_ffn(L, s)
        else:
            self._expanded_ffn(L, s)
        gather_w = self.row_w if self.weighting == "gather" else None
        check(L.moe_combine(_ptr(self.down_out), _ptr(lay.src2dst), _ptr(gather_w), _ptr(n_valid),
                            T, self.H, self.K, _ptr(y), s), "moe_combine")
        return y

    def _expanded_ffn(self, L, s):
        lay = self.lay
        check(L.moe_grouped_ffn(_ptr(self.xe), _ptr(self.xe_scale), self.xe_scale.shape[1],
                                self.sl, _ptr(lay.start), _ptr(lay.tile_prefix), _ptr(lay.total),
                                _ptr(self.w13), _ptr(self.s13), _ptr(self.w2), _ptr(self.s2),
                                _ptr(self.row_w), self.flags, self.E, self.H, self.I, self.M_cap,
                                None, _ptr(self.down_in), _ptr(self.down_in_scale),
                                self.down_in_scale.shape[1], _ptr(self.down_out),
                                _ptr(self.status), s), "moe_grouped_ffn")

    def _slab_ffn(self, L, s):
        """Decode variant: expanded rows -> masked slab, both GEMMs on the slab
        (gate_up with act+quant fused), slab -> expanded rows with the top-k
        weights."""
        lay, sl_lay = self.lay, self.slab_lay
        E, H, I, m = self.E, self.H, self.I, self.masked_max_m
        S = E * m
        check(L.moe_expand_to_masked_slab(
            _ptr(self.xe), _ptr(self.xe_scale), self.sl, self.xe_scale.shape[1], _ptr(lay.psum),
            _ptr(lay.start), E, H, m, _ptr(self.slab), _ptr(self.slab_scale),
            self.slab_scale.shape[1], _ptr(self.masked_m), _ptr(sl_lay.start),
            _ptr(sl_lay.tile_prefix), _ptr(sl_lay.total), _ptr(self.status), s),
            "moe_expand_to_masked_slab")
        check(L.moe_grouped_gemm_act_quant(
            _ptr(self.slab), _ptr(self.slab_scale), self.sl, self.slab_scale.shape[1],
            _ptr(sl_lay.start), _ptr(sl_lay.tile_prefix), _ptr(sl_lay.total), _ptr(self.w13),
            _ptr(self.s13), None, 0, E, I, H, S, _ptr(self.slab_di), _ptr(self.slab_di_scale),
            self.slab_di_scale.shape[1], _ptr(self.status), s), "moe_grouped_gemm_act_quant")
        check(L.moe_grouped_gemm(
            _ptr(self.slab_di), _ptr(self.slab_di_scale), self.sl, self.slab_di_scale.shape[1],
            _ptr(sl_lay.start), _ptr(sl_lay.tile_prefix), _ptr(sl_lay.total), _ptr(self.w2),
            _ptr(self.s2), None, 0, E, H, I, S, _ptr(self.slab_out), _ptr(self.status), s),
            "moe_grouped_gemm")
        check(L.moe_masked_slab_to_expand(
            _ptr(self.slab_out), m, _ptr(lay.psum), _ptr(lay.start), _ptr(lay.total),
            _ptr(self.row_w), E, H, self.M_cap, _ptr(self.down_out), s),
            "moe_masked_slab_to_expand")

    def capture(self, x_q, x_scale, topk_ids, topk_w, n_valid=None,
                out: Optional[torch.Tensor] = None) -> "CapturedForward":
        """Records one forward on these device tensors into a CUDA graph.
        Replaying it reruns the whole layer (every kernel, no host work) on
        whatever the tensors hold at replay time: refill them in place, then
        call replay(). Run one eager forward first so the library has set up
        its per-device state; the captured launches must not be captured
        while another capture on the same device is in progress."""
        return CapturedForward(self, x_q, x_scale, topk_ids, topk_w, n_valid, out)

    @property
    def gateup(self) -> torch.Tensor:
        """bf16 [M_cap, 2I] buffer for the stand-alone gate_up GEMM (the
        layer's own forward fuses act+quant into gate_up and never needs it)."""
        if self._gateup is None:
            self._gateup = torch.zeros(self.M_cap, 2 * self.I, dtype=torch.bfloat16,
                                       device=self.device)
        return self._gateup

    # kernels one forward launches at most: layout + scatter 3 (1 when the
    # cooperative grid holds every 2048-pair chunk), gate_up with act+quant
    # fused 1, down 1, combine 1
    KERNELS_PER_FORWARD = 6


class HostPipeline:
    """Runs an ExpandedMoELayer on batches held in pinned host memory with the
    copies off the critical path: batch k+1's inputs go host->device on one
    copy stream and batch k's output device->host on another while the
    layer's kernels run batch k on the compute stream. Device inputs and
    outputs are double-buffered; every batch's copies still happen.

        pipe = HostPipeline(layer)
        for batch, y_host in ...:
            pipe.submit(x_q_h, x_s_h, ids_h, w_h, n_valid_h, y_host)
        pipe.synchronize()        # every y_host filled

    Host tensors must be pinned (page-locked) for the copies to be
    asynchronous, and a y_host may be read only after synchronize() (or after
    the submit two batches later has returned and its event completed).

    submit(..., n_rows=n) is for callers that know on the host how many
    leading rows of the batch are valid (n >= the n_valid the device word
    holds): only rows [0, n) of x_q, x_scale, topk_ids, topk_w go to the
    device and only rows [0, n) of y come back. The layer itself still takes
    the valid-row count from the device word; rows past it are never read,
    so what the device buffers hold there does not matter.
    """

    def __init__(self, layer: "ExpandedMoELayer", stream=None):
        self.layer = layer
        dev = layer.device
        self.comp = stream if stream is not None else torch.cuda.current_stream(dev)
        self.h2d = torch.cuda.Stream(dev)
        self.d2h = torch.cuda.Stream(dev)
        T, H, K = layer.T, layer.H, layer.K
        G = H // 128
        def bufs():
            xs = (torch.empty(T, G, dtype=torch.float32, device=dev) if layer.sl == 0 else
                  torch.empty((G + 3) // 4, T, dtype=torch.int32, device=dev))
            return dict(x_q=torch.empty(T, H, dtype=torch.uint8, device=dev), x_s=xs,
                        ids=torch.empty(T, K, dtype=torch.int32, device=dev),
                        w=torch.empty(T, K, dtype=torch.float32, device=dev),
                        nv=torch.empty(1, dtype=torch.int32, device=dev),
                        y=torch.zeros(T, H, dtype=torch.bfloat16, device=dev))
        self.bufs = [bufs(), bufs()]
        self.in_ready = [torch.cuda.Event() for _ in range(2)]
        self.done = [torch.cuda.Event() for _ in range(2)]
        self.out_copied = [torch.cuda.Event() for _ in range(2)]
        self.k = 0

    def submit(self, x_q, x_scale, topk_ids, topk_w, n_valid, y_host,
               n_rows: Optional[int] = None) -> None:
        i = self.k % 2
        b = self.bufs[i]
        if b["x_s"].shape != x_scale.shape:
            raise ValueError("x_scale shape does not match the layer's scale layout")
        T = self.layer.T
        n = T if n_rows is None else int(n_rows)
        if not 0 <= n <= T:
            raise ValueError(f"n_rows must be in [0, {T}], got {n}")
        with torch.cuda.stream(self.h2d):
            if self.k >= 2:
                self.h2d.wait_event(self.done[i])      # batch k-2 has read these inputs
            b["x_q"][:n].copy_(x_q[:n], non_blocking=True)
            if self.layer.sl == MOE_SCALE_F32_ROWMAJOR:
                b["x_s"][:n].copy_(x_scale[:n], non_blocking=True)
            elif n == T:
                b["x_s"].copy_(x_scale, non_blocking=True)
            else:
                for j in range(x_scale.shape[0]):      # column-major: one run per word row
                    b["x_s"][j, :n].copy_(x_scale[j, :n], non_blocking=True)
            b["ids"][:n].copy_(topk_ids[:n], non_blocking=True)
            b["w"][:n].copy_(topk_w[:n], non_blocking=True)
            b["nv"].copy_(n_valid, non_blocking=True)
            self.in_ready[i].record(self.h2d)
        self.comp.wait_event(self.in_ready[i])
        if self.k >= 2:
            self.comp.wait_event(self.out_copied[i])   # batch k-2's y has left this buffer
        self.layer.forward(b["x_q"], b["x_s"], b["ids"], b["w"], b["nv"], stream=self.comp,
                           out=b["y"])
        self.done[i].record(self.comp)
        with torch.cuda.stream(self.d2h):
            self.d2h.wait_event(self.done[i])
            y_host[:n].copy_(b["y"][:n], non_blocking=True)
            self.out_copied[i].record(self.d2h)
        self.k += 1

    def synchronize(self) -> None:
        self.h2d.synchronize()
        self.comp.synchronize()
        self.d2h.synchronize()


class CapturedForward:
    """A CUDA graph of one ExpandedMoELayer.forward over fixed device tensors
    (see ExpandedMoELayer.capture). replay() launches the recorded kernels on
    the current stream and returns the output tensor."""

    def __init__(self, layer: "ExpandedMoELayer", x_q, x_scale, topk_ids, topk_w, n_valid, out):
        self.layer = layer
        self.inputs = (x_q, x_scale, topk_ids, topk_w, n_valid)
        self.out = out if out is not None else layer.y
        side = torch.cuda.Stream(layer.device)
        side.wait_stream(torch.cuda.current_stream(layer.device))
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.stream(side):
            with torch.cuda.graph(self.graph, stream=side):
                layer.forward(x_q, x_scale, topk_ids, topk_w, n_valid, stream=side, out=self.out)
        torch.cuda.current_stream(layer.device).wait_stream(side)

    def replay(self) -> torch.Tensor:
        self.graph.replay()
        return self.out
