"""ctypes declarations of libmoe_expand.so (include/moe_expand.h).

Loading fails loudly when the library has not been built: there is no
fallback of any kind.
"""
from __future__ import annotations

import ctypes as C
import os
import threading

from . import build as _build

MOE_OK = 0
MOE_ERR_INVALID_ARG = -1
MOE_ERR_UNSUPPORTED = -2
MOE_ERR_CUDA = -3
MOE_ERR_WORKSPACE = -4
MOE_ERR_DEVICE_CHECK = -5
MOE_ERR_TIMEOUT = -6

MOE_SCALE_F32_ROWMAJOR = 0
MOE_SCALE_UE8M0_PACKED_COLMAJOR = 1

MOE_FOLD_WEIGHT_INTO_SCALE = 1
MOE_WEIGHT_OUTPUT_ROWS = 2
MOE_GEMM_TILE_N128 = 16
MOE_GEMM_PER_KBLOCK_PROMOTION = 64
MOE_FFN_UNFUSED = 128

MOE_BLOCK_M = 128

ERROR_NAMES = {
    MOE_ERR_INVALID_ARG: "MOE_ERR_INVALID_ARG",
    MOE_ERR_UNSUPPORTED: "MOE_ERR_UNSUPPORTED",
    MOE_ERR_CUDA: "MOE_ERR_CUDA",
    MOE_ERR_WORKSPACE: "MOE_ERR_WORKSPACE",
    MOE_ERR_DEVICE_CHECK: "MOE_ERR_DEVICE_CHECK",
    MOE_ERR_TIMEOUT: "MOE_ERR_TIMEOUT",
}

# Every symbol include/moe_expand.h declares, with (restype, argtypes).
P, I32, I64, SZ = C.c_void_p, C.c_int, C.c_int64, C.c_size_t
SIGNATURES = {
    "moe_expanded_capacity": (I64, [I64, I32, I32, I32]),
    "moe_workspace_size": (SZ, [I64, I32, I32]),
    "moe_expand_layout": (I32, [P, I64, I32, I32, I32, P, I64, P, P, P, P, P, P, P, SZ, P, P]),
    "moe_expand_layout_noalloc": (I32, [P, I64, I32, I32, I32, P, I64, P, P, P, P, P, P, P, P]),
    "moe_expand_layout_noalloc_max_scratch": (SZ, []),
    "moe_expand_layout_scatter": (I32, [P, P, P, P, I32, I64, I64, I32, I32, I32, I32, P, I64,
                                        P, P, P, P, P, P, P, P, I64, P, P, SZ, P, P]),
    "moe_expand_scatter": (I32, [P, P, I32, I64, P, P, P, P, P, I64, I32, I32, I32, I32, I64,
                                 P, P, I64, P, P, P]),
    "moe_grouped_gemm": (I32, [P, P, I32, I64, P, P, P, P, P, P, I32, I32, I32, I32, I64, P, P, P]),
    "moe_act_quant": (I32, [P, I32, P, I32, I32, P, I64, P, P, I64, P, P]),
    "moe_grouped_gemm_act_quant": (I32, [P, P, I32, I64, P, P, P, P, P, P, I32, I32, I32, I32, I64,
                                         P, P, I64, P, P]),
    "moe_grouped_ffn": (I32, [P, P, I64, I32, P, P, P, P, P, P, P, P, I32, I32, I32, I32, I64,
                              P, P, P, I64, P, P, P]),
    "moe_combine": (I32, [P, P, P, P, I64, I32, I32, P, P]),
    "moe_expand_to_masked_slab": (I32, [P, P, I32, I64, P, P, I32, I32, I64, P, P, I64, P, P, P,
                                        P, P, P]),
    "moe_masked_slab_to_expand": (I32, [P, I64, P, P, P, P, I32, I32, I64, P, P]),
    "moe_gemm_set_trace": (I32, [P]),
    "moe_selftest_bounded_wait": (I32, [I64, P, P, P]),
    "moe_last_error_string": (C.c_char_p, []),
    "moe_device_supported": (I32, [I32]),
}

_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return _build.LIB


def load():
    """The loaded library; raises if it is missing."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.LIB
            if not os.path.exists(path):
                raise RuntimeError(
                    f"{path} is not built: run `python -m expanded_layout_expert_gb300.build` "
                    "(or __graft_entry__.build()) first")
            lib = C.CDLL(path)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib


class MoEError(RuntimeError):
    def __init__(self, rc: int, where: str):
        msg = load().moe_last_error_string().decode(errors="replace")
        super().__init__(f"{where}: {ERROR_NAMES.get(rc, rc)}: {msg}")
        self.rc = rc


def check(rc: int, where: str) -> None:
    if rc != MOE_OK:
        raise MoEError(rc, where)
