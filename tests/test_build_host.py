"""Register allocation of the grouped-GEMM kernels, checked on the host from
ptxas's own report (no GPU). Each epilogue thread of the 256-column kernels
holds 128 fp32 accumulators and a 64-column staging batch in a 232-register
budget, and ptxas's choices there have flipped between builds before (a
change elsewhere in the kernel made it spill the accumulators and doubled a
launch's time), so every instantiation is held to a spill budget:

* the block-scaled (ue8m0) kernel and the 128-column promotion kernel: none;
* the 256-column promotion kernel: at most two 4-byte values (8 bytes stored,
  36 bytes loaded), which ptxas keeps in local memory across the tile loop
  (about one local load per epilogue warp and tile, measured with ncu).
"""
import re

import pytest

from expanded_layout_expert_gb300 import build


def _kernels(src, name):
    usage = build.ptxas_usage(src)
    out = {k: v for k, v in usage.items() if name in k}
    assert out, f"no {name} entry in {src}"
    return out


def test_block_scaled_gemm_kernels_do_not_spill():
    for k, v in _kernels("grouped_gemm_mx.cu", "grouped_gemm_mx_kernel").items():
        assert v["spill_st"] == 0 and v["spill_ld"] == 0 and v["stack"] == 0, (k, v)


def test_promotion_gemm_kernels_stay_within_their_spill_budget():
    ks = _kernels("grouped_gemm.cu", "grouped_gemm_kernel")
    assert len(ks) == 10   # BN x Staged x Fused x scale format instantiations
    for k, v in ks.items():
        bn = int(re.search(r"grouped_gemm_kernelILi(\d+)E", k).group(1))
        if bn == 128:
            assert v["spill_st"] == 0 and v["spill_ld"] == 0, (k, v)
        else:
            assert v["spill_st"] <= 8 and v["spill_ld"] <= 36, (k, v)
