"""ctypes loader of ``libmoe_gb300.so`` with the C prototypes of ``include/moe_gb300.h``.

There is no fallback: if the library is missing or fails to load, every call raises.
"""
from __future__ import annotations

import ctypes
import os

from .build import LIB_PATH

_P = ctypes.c_void_p
_I = ctypes.c_int
_I64 = ctypes.c_int64
_F = ctypes.c_float
_SZ = ctypes.c_size_t
_U64 = ctypes.c_uint64

# name -> (restype, argtypes); mirrors include/moe_gb300.h
PROTOTYPES = {
    "moe_status_string": (ctypes.c_char_p, [_I]),
    "moe_version": (_I, []),
    "moe_padded_rows": (_I64, [_I64, _I, _I]),
    "moe_workspace_bytes": (_SZ, [_I64, _I, _I, _I]),
    "moe_device_status": (_I, [_P, _P, _P]),
    "moe_clear_device_status": (_I, [_P]),
    "moe_set_wait_limit_ns": (None, [_U64]),
    "moe_check_bounded_wait": (_I, [_U64, _P]),
    "moe_route": (_I, [_P, _P, _P, _I64, _I, _I, _I, _I, _F, _P, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "moe_permute": (_I, [_P, _P, _I64, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "moe_permute_noalloc": (_I, [_P, _P, _I64, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P]),
    "moe_expert_fwd": (_I, [_P, _P, _I, _I64, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P, _P, _SZ,
                            _P]),
    "moe_quantize_rows_fp8": (_I, [_P, _P, _I64, _I, _P, _P, _P]),
    "moe_permute_fp8": (_I, [_P, _P, _P, _P, _P, _I64, _I, _I, _I, _P, _P, _P]),
    "moe_expert_fwd_fp8": (_I, [_P, _P, _P, _I, _I64, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                                _P, _P, _P, _P, _P, _SZ, _P]),
    "moe_quantize_rows2_fp8": (_I, [_P, _P, _P, _I64, _I, _P, _P, _P]),
    "moe_quantize_cols_fp8": (_I, [_P, _P, _I, _I, _I, _P, _P, _P]),
    "moe_expert_bwd_fp8": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _I, _I64, _I, _I, _P, _P, _P, _P,
                                _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "moe_combine": (_I, [_P, _P, _P, _P, _I64, _I, _I, _P, _P]),
    "moe_bias_update": (_I, [_P, _I, _I64, _I, _F, _P, _P]),
    "moe_bias_update_proportional": (_I, [_P, _I, _I64, _I, _F, _P, _P]),
    "moe_combine_bwd": (_I, [_P, _P, _P, _P, _P, _P, _I64, _I, _I, _I, _P, _P, _P]),
    "moe_combine_bwd_fp8": (_I, [_P, _P, _P, _P, _P, _P, _I64, _I, _I, _I, _P, _P, _P, _P, _P]),
    "moe_expert_bwd": (_I, [_P, _P, _P, _P, _P, _P, _I, _I64, _I, _I, _P, _P, _P, _P, _P, _P, _P,
                            _P, _P, _P, _P, _I, _P, _P, _P, _SZ, _P]),
    "moe_row_gates": (_I, [_P, _P, _I64, _I, _I64, _P, _P]),
    "moe_gate_grad": (_I, [_P, _P, _I64, _I, _I, _P, _P]),
    "moe_route_bwd": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _I64, _I, _I, _I, _I, _F, _P, _P, _P,
                           _P, _P, _SZ, _P]),
    "moe_aux_loss": (_I, [_P, _P, _I64, _I, _I, _I, _I64, _F, _F, _P, _P, _P, _SZ, _P]),
    "moe_aux_loss_bwd": (_I, [_P, _P, _I64, _I, _I, _I64, _F, _F, _P, _P]),
    "moe_permute_bwd": (_I, [_P, _P, _P, _P, _P, _P, _I64, _I, _I, _I, _P, _P]),
    "moe_router_dx": (_I, [_P, _P, _I64, _I, _I, _P, _P, _SZ, _P]),
}

_lib = None


class MoELibraryError(RuntimeError):
    pass


def load(path: str | None = None) -> ctypes.CDLL:
    """Load the library once (building it first is the job of ``build_library``)."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or LIB_PATH
    if not os.path.exists(path):
        raise MoELibraryError(
            f"{path} is missing: build it with `python -m pretraining_sigmoid_softmax_gb300.build`")
    lib = ctypes.CDLL(path)
    for name, (res, args) in PROTOTYPES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib
