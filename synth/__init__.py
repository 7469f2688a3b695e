"""Seeded synthetic inputs for the expanded-layout MoE prefill layer.

This module makes inputs and nothing else. It is shared by the CPU oracle's
tests and by the CUDA path's tests and benchmark, and it holds none of the
layer's arithmetic: no layout, no scatter, no GEMM, no activation, no combine.
Random numbers are drawn with a seeded ``torch.Generator``; fp8 codes are made
with PyTorch's own ``float8_e4m3fn`` cast and power-of-two scales with
``torch.frexp`` (library routines, used only to give the inputs the form the
layer consumes).

Workloads (the five named configurations, plus smaller parity shapes):

* activations ``x ~ N(0, 1)`` quantised per 1x128 group with scale
  ``amax/448`` (fp32), or, on the ue8m0 workload, with that scale rounded up to
  a power of two and stored as a biased exponent byte, packed four groups per
  int32 in a column-major ``[ceil(G/4), T]`` array;
* expert weights ``W13 [E, 2I, H]`` and ``W2 [E, H, I] ~ N(0, 0.02)``, quantised
  per 128x128 block the same way (fp32 scales, or ue8m0 bytes);
* router logits ``~ N(0, 1)``; top-k ids by logit, weights = softmax over all E
  experts taken at the chosen ids (not renormalised).  Zipf routing draws
  expert popularity ``p_e ~ 1/rank^s`` over a seeded permutation, gives the
  least popular experts probability zero, and samples k experts without
  replacement by the Gumbel-top-k trick on ``log p_e``;
* inactive rows (all k ids = -1, weight 0) chosen by a seeded Bernoulli draw;
* the padded-receive workload fills rows past ``n_valid`` with random bytes,
  random scale bits (NaN and inf included), random in-range ids and random
  weights, which every consumer must ignore.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import torch

SCALE_F32 = "f32"
SCALE_UE8M0 = "ue8m0"


@dataclasses.dataclass(frozen=True)
class LayerConfig:
    name: str
    T: int          # token rows in the buffer
    H: int          # hidden size
    I: int          # expert intermediate size (gate and up halves each have I)
    E: int          # experts
    K: int          # top-k
    align: int      # expert_alignment of the expanded layout
    seed: int
    routing: str = "uniform"        # "uniform" | "zipf"
    inactive_frac: float = 0.0
    scale_mode: str = SCALE_F32     # "f32" | "ue8m0"
    n_valid: Optional[int] = None   # None -> all T rows valid
    zipf_s: float = 1.2
    zipf_zero_experts: int = 0
    garbage_tail: bool = False

    @property
    def valid_rows(self) -> int:
        return self.T if self.n_valid is None else self.n_valid

    @property
    def GH(self) -> int:
        return self.H // 128

    @property
    def GI(self) -> int:
        return self.I // 128

    def describe(self) -> dict:
        d = dataclasses.asdict(self)
        d["n_valid"] = self.valid_rows
        return d


# The five workloads, in order: tiny, uniform H=4096, Zipf H=7168,
# ue8m0 H=7168, padded receive buffer.
CONFIGS = (
    LayerConfig("tiny_h512", T=64, H=512, I=256, E=8, K=2, align=32, seed=0,
                routing="uniform", inactive_frac=0.10),
    LayerConfig("uniform_t4096_h4096", T=4096, H=4096, I=1536, E=32, K=8,
                align=128, seed=1, routing="uniform"),
    LayerConfig("zipf_t16384_h7168", T=16384, H=7168, I=2048, E=32, K=8,
                align=128, seed=2, routing="zipf", inactive_frac=0.05,
                zipf_s=1.2, zipf_zero_experts=4),
    LayerConfig("ue8m0_t8192_h7168", T=8192, H=7168, I=2048, E=64, K=8,
                align=128, seed=3, routing="uniform", scale_mode=SCALE_UE8M0),
    LayerConfig("padded_t32768_valid6000_h4096", T=32768, H=4096, I=1536, E=32,
                K=8, align=128, seed=4, routing="uniform", n_valid=6000,
                garbage_tail=True),
)

# A decode-sized batch (not one of the five layer workloads): few tokens per
# expert, for the masked-slab variant and graph-replay measurements.
EXTRA_CONFIGS = (
    LayerConfig("decode_t256_h7168_ue8m0", T=256, H=7168, I=2048, E=64, K=8, align=16,
                seed=20, routing="uniform", scale_mode=SCALE_UE8M0),
)

# Reduced copies of the ue8m0 workload for hardware-counter captures, which
# belong on a few GB of device memory: the same hidden and intermediate
# sizes, top-k and 1024 rows per expert (8 m blocks, so the GEMMs reuse an
# expert's weights exactly as at full size), with a quarter of the experts
# and of the tokens.
PROFILE_CONFIGS = (
    LayerConfig("ue8m0_t2048_e16_h7168", T=2048, H=7168, I=2048, E=16, K=8,
                align=128, seed=3, routing="uniform", scale_mode=SCALE_UE8M0),
)

# Shapes small enough for the oracle to run every row in seconds, still
# spanning several 128-row tiles, several N tiles and ragged tails.
PARITY_CONFIGS = (
    next(c for c in CONFIGS if c.name == "tiny_h512"),
    LayerConfig("mid_f32", T=200, H=1024, I=512, E=8, K=4, align=128, seed=10,
                routing="uniform", inactive_frac=0.10),
    LayerConfig("mid_ue8m0", T=192, H=1024, I=512, E=8, K=4, align=128,
                seed=11, routing="uniform", scale_mode=SCALE_UE8M0,
                inactive_frac=0.05),
    LayerConfig("mid_zipf_ragged", T=256, H=768, I=384, E=16, K=6, align=64,
                seed=12, routing="zipf", zipf_s=1.2, zipf_zero_experts=3,
                inactive_frac=0.05),
    LayerConfig("mid_ue8m0_ragged", T=160, H=768, I=384, E=12, K=3, align=16,
                seed=13, routing="uniform", scale_mode=SCALE_UE8M0),
    LayerConfig("mid_padded", T=512, H=1024, I=512, E=8, K=4, align=128,
                seed=14, routing="uniform", n_valid=150, garbage_tail=True),
    LayerConfig("small_h384", T=96, H=384, I=128, E=6, K=2, align=8, seed=15,
                routing="uniform", inactive_frac=0.10),
    # many experts (per-expert tables past the GEMM's shared-memory copy),
    # top-12 (not a power of two), most experts with a single short segment
    LayerConfig("wide_e160_k12", T=96, H=512, I=256, E=160, K=12, align=32, seed=16,
                routing="zipf", zipf_s=1.2, zipf_zero_experts=20, inactive_frac=0.05),
    LayerConfig("wide_e160_k12_ue8m0", T=80, H=512, I=256, E=160, K=12, align=16, seed=17,
                routing="uniform", scale_mode=SCALE_UE8M0),
    # ue8m0 with H % 256 != 0: the down GEMM takes 128-column tiles and the
    # per-K-block promotion kernel
    LayerConfig("small_h384_ue8m0", T=64, H=384, I=128, E=6, K=2, align=8, seed=18,
                routing="uniform", scale_mode=SCALE_UE8M0, inactive_frac=0.10),
    # the full workloads' hidden size: 56 K blocks in gate_up, so every row of
    # a long-K GEMM (accumulator ring and scale words wrapping many times) is
    # compared with the oracle
    LayerConfig("longk_h7168", T=64, H=7168, I=256, E=4, K=2, align=32, seed=19,
                routing="uniform", inactive_frac=0.05),
    LayerConfig("longk_h7168_ue8m0", T=48, H=7168, I=256, E=4, K=2, align=16, seed=21,
                routing="uniform", scale_mode=SCALE_UE8M0),
)


def config_by_name(name: str) -> LayerConfig:
    for c in CONFIGS + PARITY_CONFIGS + EXTRA_CONFIGS + PROFILE_CONFIGS:
        if c.name == name:
            return c
    raise KeyError(name)


def _pow2_ceil_exponent(s: torch.Tensor) -> torch.Tensor:
    """Integer e with 2**e the smallest power of two >= s (s > 0, normal)."""
    m, e = torch.frexp(s)
    return torch.where(m == 0.5, e - 1, e)


def _to_e4m3_bytes(v: torch.Tensor) -> torch.Tensor:
    return v.to(torch.float8_e4m3fn).view(torch.uint8)


def _pack_bytes_colmajor(b: torch.Tensor) -> torch.Tensor:
    """[rows, G] uint8 -> int32 [ceil(G/4), rows]: four groups per word, group
    4j in the low byte, unused lanes zero."""
    rows, G = b.shape
    W = (G + 3) // 4
    pad = torch.zeros(rows, W * 4, dtype=torch.int64, device=b.device)
    pad[:, :G] = b.to(torch.int64)
    pad = pad.view(rows, W, 4)
    word = pad[..., 0] | (pad[..., 1] << 8) | (pad[..., 2] << 16) | (pad[..., 3] << 24)
    word = torch.where(word >= 2**31, word - 2**32, word)
    return word.to(torch.int32).t().contiguous()


def quantise_rows(x: torch.Tensor, scale_mode: str):
    """Per 1x128 group: scale amax/448 (or its power-of-two ceiling), codes by
    PyTorch's e4m3 cast.  Returns (uint8 [T, H], scales)."""
    T, H = x.shape
    g = x.view(T, H // 128, 128)
    amax = g.abs().amax(dim=-1).clamp_min(1e-30)
    s = amax / 448.0
    if scale_mode == SCALE_UE8M0:
        e = _pow2_ceil_exponent(s)
        s = torch.ldexp(torch.ones_like(s), e)
        q = _to_e4m3_bytes(g / s.unsqueeze(-1)).view(T, H)
        return q, _pack_bytes_colmajor((e + 127).to(torch.uint8))
    q = _to_e4m3_bytes(g / s.unsqueeze(-1)).view(T, H)
    return q, s.contiguous()


def quantise_blocks(w: torch.Tensor, scale_mode: str):
    """Per 128x128 block of an [N, Kd] matrix."""
    N, Kd = w.shape
    b = w.view(N // 128, 128, Kd // 128, 128)
    amax = b.abs().amax(dim=(1, 3)).clamp_min(1e-30)
    s = amax / 448.0
    if scale_mode == SCALE_UE8M0:
        e = _pow2_ceil_exponent(s)
        s = torch.ldexp(torch.ones_like(s), e)
        byte = (e + 127).to(torch.uint8)
    q = _to_e4m3_bytes(b / s[:, None, :, None]).view(N, Kd)
    if scale_mode == SCALE_UE8M0:
        return q, byte
    return q, s


def _routing(cfg: LayerConfig, g: torch.Generator, device):
    T, E, K = cfg.T, cfg.E, cfg.K
    if cfg.routing == "zipf":
        perm = torch.randperm(E, generator=g, device=device)
        rank = torch.empty(E, dtype=torch.float64, device=device)
        rank[perm] = torch.arange(1, E + 1, dtype=torch.float64, device=device)
        p = rank.pow(-cfg.zipf_s)
        if cfg.zipf_zero_experts:
            p = torch.where(rank > E - cfg.zipf_zero_experts, torch.zeros_like(p), p)
        logp = torch.log(p / p.sum()).to(torch.float32)
        u = torch.rand(T, E, generator=g, device=device).clamp(1e-20, 1.0 - 1e-7)
        logits = logp.unsqueeze(0) - torch.log(-torch.log(u))
    else:
        logits = torch.randn(T, E, generator=g, device=device)
    probs = torch.softmax(logits, dim=-1)
    ids = logits.topk(K, dim=-1).indices
    w = probs.gather(1, ids)
    return ids.to(torch.int32), w.to(torch.float32)


def generate(cfg: LayerConfig, device="cpu", with_weights: bool = True) -> dict:
    """All inputs of one layer call, on ``device``."""
    device = torch.device(device)
    g = torch.Generator(device=device)
    g.manual_seed(cfg.seed)
    T, H, I, E, K = cfg.T, cfg.H, cfg.I, cfg.E, cfg.K
    nv = cfg.valid_rows

    x = torch.randn(T, H, generator=g, device=device)
    x_q, x_s = quantise_rows(x, cfg.scale_mode)
    del x
    ids, w = _routing(cfg, g, device)

    if cfg.inactive_frac > 0:
        off = torch.rand(T, generator=g, device=device) < cfg.inactive_frac
        ids = torch.where(off.unsqueeze(1), torch.full_like(ids, -1), ids)
        w = torch.where(off.unsqueeze(1), torch.zeros_like(w), w)

    if cfg.garbage_tail and nv < T:
        tail = T - nv
        x_q[nv:] = torch.randint(0, 256, (tail, H), generator=g, device=device,
                                 dtype=torch.int32).to(torch.uint8)
        ids[nv:] = torch.randint(0, E, (tail, K), generator=g, device=device,
                                 dtype=torch.int32)
        w[nv:] = torch.rand(tail, K, generator=g, device=device)
        bits = torch.randint(-2**31, 2**31 - 1, (tail, x_s.shape[1] if cfg.scale_mode == SCALE_F32 else x_s.shape[0]),
                             generator=g, device=device, dtype=torch.int64).to(torch.int32)
        if cfg.scale_mode == SCALE_F32:
            x_s[nv:] = bits.view(torch.float32)
        else:
            x_s[:, nv:] = bits.t()

    out = dict(cfg=cfg, n_valid=nv, x_q=x_q.contiguous(), x_s=x_s.contiguous(),
               topk_ids=ids.contiguous(), topk_w=w.contiguous())
    if with_weights:
        out.update(generate_weights(cfg, g, device))
    return out


def generate_weights(cfg: LayerConfig, g: torch.Generator, device) -> dict:
    E, H, I = cfg.E, cfg.H, cfg.I
    w13 = torch.empty(E, 2 * I, H, dtype=torch.uint8, device=device)
    w2 = torch.empty(E, H, I, dtype=torch.uint8, device=device)
    sdt = torch.uint8 if cfg.scale_mode == SCALE_UE8M0 else torch.float32
    s13 = torch.empty(E, 2 * I // 128, H // 128, dtype=sdt, device=device)
    s2 = torch.empty(E, H // 128, I // 128, dtype=sdt, device=device)
    for e in range(E):
        a = torch.randn(2 * I, H, generator=g, device=device) * 0.02
        w13[e], s13[e] = quantise_blocks(a, cfg.scale_mode)
        b = torch.randn(H, I, generator=g, device=device) * 0.02
        w2[e], s2[e] = quantise_blocks(b, cfg.scale_mode)
    return dict(w13=w13, s13=s13, w2=w2, s2=s2)
