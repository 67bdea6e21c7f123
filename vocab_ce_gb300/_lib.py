"""ctypes declarations of libtpce's C ABI (include/tpce.h).

Loading is lazy; a missing or unloadable library raises immediately at first
use. There is no fallback implementation.
"""

from __future__ import annotations

import ctypes
import os
import threading

# the in-tree build; TPCE_LIBRARY may name another build of the same library
LIB_PATH = os.environ.get("TPCE_LIBRARY") or os.path.join(os.path.dirname(os.path.abspath(__file__)), "lib",
                                                           "libtpce.so")

STATUS = {
    0: "TPCE_OK", 1: "TPCE_ERR_INVALID", 2: "TPCE_ERR_SHAPE", 3: "TPCE_ERR_ALIGN",
    4: "TPCE_ERR_WORKSPACE", 5: "TPCE_ERR_CUDA", 6: "TPCE_ERR_TIMEOUT", 7: "TPCE_ERR_UNSUPPORTED",
}
TPCE_BF16 = 0
TPCE_F32 = 1
TPCE_COLUMN_PARALLEL = 0
TPCE_ROW_PARALLEL = 1

# every symbol include/tpce.h declares, with (restype, argtypes)
_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_I = ctypes.c_int
_SZ = ctypes.c_size_t
_F = ctypes.c_float
SIGNATURES = {
    "tpce_status_string": (ctypes.c_char_p, [_I]),
    "tpce_version": (_I, []),
    "tpce_last_error": (ctypes.c_char_p, []),
    "tpce_pad_vocab": (_I64, [_I64, _I, _I]),
    "tpce_mlp_workspace_bytes": (_SZ, [_I64, _I64, _I64, _I, _I]),
    "tpce_tail_workspace_bytes": (_SZ, []),
    "tpce_ce_workspace_bytes": (_SZ, [_I64, _I64, _I64, _I, _I, _I]),
    "tp_mlp_forward": (_I, [_P, _P, _P, _P, _P, _I64, _I64, _I64, _I, _I, _P, _P, _P, _P, _SZ, _P]),
    "tp_mlp_backward": (_I, [_P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _I, _I,
                             _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "tpce_swiglu_workspace_bytes": (_SZ, [_I64, _I64, _I64, _I, _I]),
    "tp_swiglu_forward": (_I, [_P, _P, _P, _P, _P, _I64, _I64, _I64, _I, _I, _P, _P, _P, _P, _SZ, _P]),
    "tp_swiglu_backward": (_I, [_P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _I, _I,
                                _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "tpce_linear_workspace_bytes": (_SZ, [_I64, _I64, _I64, _I, _I, _I]),
    "tp_linear_forward": (_I, [_P, _P, _P, _I64, _I64, _I64, _I, _I, _I, _P, _P, _SZ, _P]),
    "tp_linear_backward": (_I, [_P, _P, _P, _I64, _I64, _I64, _I, _I, _I, _P, _P, _P, _P, _SZ, _P]),
    "tpce_attn_workspace_bytes": (_SZ, [_I64, _I64, _I64, _I64, _I64, _I, _I]),
    "tp_attn_qkv_forward": (_I, [_P, _P, _P, _I64, _I64, _I64, _I64, _I64, _I, _I, _P, _P, _SZ, _P]),
    "tp_attn_qkv_backward": (_I, [_P, _P, _P, _I64, _I64, _I64, _I64, _I64, _I, _I, _P, _P, _P, _P, _SZ, _P]),
    "tp_attn_out_forward": (_I, [_P, _P, _P, _I64, _I64, _I64, _I64, _I, _I, _P, _P, _SZ, _P]),
    "tp_attn_out_backward": (_I, [_P, _P, _P, _I64, _I64, _I64, _I64, _I, _I, _P, _P, _P, _P, _SZ, _P]),
    "tp_mlp_forward_sp": (_I, [_P, _P, _P, _P, _P, _I64, _I64, _I64, _I, _I, _P, _P, _P, _P, _SZ, _P]),
    "tp_mlp_backward_sp": (_I, [_P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _I, _I,
                                _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "tp_swiglu_forward_sp": (_I, [_P, _P, _P, _P, _P, _I64, _I64, _I64, _I, _I, _P, _P, _P, _P, _SZ, _P]),
    "tp_swiglu_backward_sp": (_I, [_P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _I, _I,
                                   _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "tp_column_linear_forward_sp": (_I, [_P, _P, _P, _I64, _I64, _I64, _I, _I, _P, _P, _SZ, _P]),
    "tp_column_linear_backward_sp": (_I, [_P, _P, _P, _I64, _I64, _I64, _I, _I, _P, _P, _P, _P, _SZ, _P]),
    "tp_row_linear_forward_sp": (_I, [_P, _P, _P, _I64, _I64, _I64, _I, _I, _P, _P, _SZ, _P]),
    "tp_row_linear_backward_sp": (_I, [_P, _P, _P, _I64, _I64, _I64, _I, _I, _P, _P, _P, _P, _SZ, _P]),
    "tp_attn_qkv_forward_sp": (_I, [_P, _P, _P, _I64, _I64, _I64, _I64, _I64, _I, _I, _P, _P, _SZ, _P]),
    "tp_attn_qkv_backward_sp": (_I, [_P, _P, _P, _I64, _I64, _I64, _I64, _I64, _I, _I, _P, _P, _P, _P, _SZ, _P]),
    "tp_attn_out_forward_sp": (_I, [_P, _P, _P, _I64, _I64, _I64, _I64, _I, _I, _P, _P, _SZ, _P]),
    "tp_attn_out_backward_sp": (_I, [_P, _P, _P, _I64, _I64, _I64, _I64, _I, _I, _P, _P, _P, _P, _SZ, _P]),
    "vocab_parallel_ce": (_I, [_P, _P, _P, _I64, _I64, _I64, _I64, _I, _F, _I,
                               _P, _P, _P, _P, _P, _SZ, _P]),
    "vocab_parallel_ce_loss_static": (_I, [_P, _P, _P, _I64, _I64, _I64, _I64, _I, _I, _P, _P, _P]),
    "tpce_device_status": (_I, [_P, _I, ctypes.POINTER(ctypes.c_uint32)]),
    "tpce_debug_withhold_next_load": (_I, [_I]),
    "tpce_profile_enable": (_I, [_I]),
    "tpce_profile_count": (_I, []),
    "tpce_profile_get": (_I, [_I, ctypes.POINTER(ctypes.c_char_p), ctypes.POINTER(_I64),
                              ctypes.POINTER(ctypes.c_double)]),
}

_lock = threading.Lock()
_lib = None


class TpceError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: {STATUS.get(status, status)}" if what else STATUS.get(status, str(status)))


def lib() -> ctypes.CDLL:
    """The loaded library; raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"libtpce.so is not built ({LIB_PATH}); run "
                                   "`python -m vocab_ce_gb300.build` (nvcc, sm_103a)")
            L = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(L, name)
                fn.restype = res
                fn.argtypes = args
            _lib = L
        return _lib


def check(status: int, what: str) -> None:
    if status != 0:
        detail = (lib().tpce_last_error() or b"").decode(errors="replace")
        raise TpceError(status, f"{what} [{detail}]" if detail else what)
