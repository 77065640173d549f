"""ctypes declarations of include/dflash.h (argument marshalling only)."""
from __future__ import annotations

import ctypes as C
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libdflash.so")

DFLASH_OK = 0
DFLASH_EINVAL = -1
DFLASH_EGEOM = -2
DFLASH_ECAPACITY = -3
DFLASH_ERANGE = -4
DFLASH_ECUDA = -5
DFLASH_ENOMEM = -6
CODES = {DFLASH_EINVAL: "EINVAL", DFLASH_EGEOM: "EGEOM", DFLASH_ECAPACITY: "ECAPACITY", DFLASH_ERANGE: "ERANGE",
         DFLASH_ECUDA: "ECUDA", DFLASH_ENOMEM: "ENOMEM"}

QUANT_F32 = 0
QUANT_Q4G32 = 1

MAT_FC = 0
MAT_HEAD = 1
MAT_NAMES = ("q", "k", "v", "o", "gate", "up", "down")


def mat_layer(layer: int, which: str) -> int:
    return 2 + 7 * layer + MAT_NAMES.index(which)


class Geometry(C.Structure):
    _fields_ = [("hidden", C.c_int32), ("intermediate", C.c_int32), ("layers", C.c_int32), ("heads", C.c_int32),
                ("kv_heads", C.c_int32), ("head_dim", C.c_int32), ("vocab", C.c_int32), ("block", C.c_int32),
                ("n_taps", C.c_int32), ("mask_token", C.c_int32), ("window", C.c_int32), ("quant", C.c_int32),
                ("eps", C.c_float), ("rope_theta", C.c_double), ("windows", C.POINTER(C.c_int32)),
                ("no_rope", C.POINTER(C.c_int32)), ("conv_kernel", C.c_int32), ("conv_group", C.c_int32),
                ("selector_rank", C.c_int32), ("selector_top", C.c_int32)]


_FP = C.POINTER(C.c_float)
_FPP = C.POINTER(_FP)


class Weights(C.Structure):
    _fields_ = [("fc", _FP), ("hidden_norm", _FP), ("norm", _FP), ("embed", _FP), ("head", _FP),
                ("in_norm", _FPP), ("post_norm", _FPP), ("q_norm", _FPP), ("k_norm", _FPP), ("q", _FPP),
                ("k", _FPP), ("v", _FPP), ("o", _FPP), ("gate", _FPP), ("up", _FPP), ("down", _FPP),
                ("attn_conv_base", _FPP), ("attn_conv_proj", _FPP), ("mlp_conv_base", _FPP), ("mlp_conv_proj", _FPP),
                ("selector_projection", _FP), ("predecessor_codebook", C.c_void_p),
                ("successor_codebook", C.c_void_p)]


_VP = C.c_void_p
_SIGS = {
    "dflash_init": (C.c_int, [C.POINTER(Geometry), C.POINTER(Weights), C.c_int, _VP, C.POINTER(_VP)]),
    "dflash_free": (None, [_VP]),
    "dflash_last_error": (C.c_char_p, [_VP]),
    "dflash_geometry_of": (C.c_int, [_VP, C.POINTER(Geometry)]),
    "dflash_seq_new": (C.c_int, [_VP, C.c_int64, C.POINTER(_VP)]),
    "dflash_seq_free": (None, [_VP]),
    "dflash_seq_span": (C.c_int, [_VP, C.POINTER(C.c_int64), C.POINTER(C.c_int64)]),
    "dflash_ctx_append": (C.c_int, [_VP, _VP, C.c_int64, _VP, C.c_int64, C.c_int, _VP]),
    "dflash_ctx_queue": (C.c_int, [_VP, _VP, C.c_int64, _VP, C.c_int64, C.c_int, _VP]),
    "dflash_settle": (C.c_int, [_VP, _VP, _VP]),
    "dflash_truncate": (C.c_int, [_VP, C.c_int64]),
    "dflash_reset": (C.c_int, [_VP]),
    "dflash_block": (C.c_int, [_VP, C.POINTER(_VP), C.c_int32, _VP, C.POINTER(C.c_int64), C.c_int32, _VP, _VP,
                               C.c_int, _VP]),
    "dflash_profile_start": (C.c_int, [_VP]),
    "dflash_profile_stop": (C.c_int, [_VP]),
    "dflash_profile_entry": (C.c_int, [_VP, C.c_int32, C.POINTER(C.c_char_p), C.POINTER(C.c_int64),
                                       C.POINTER(C.c_double), C.POINTER(C.c_double)]),
    "dflash_launch_count": (C.c_int64, [_VP]),
    "dflash_debug_option": (C.c_int, [_VP, C.c_char_p, C.c_int64]),
    "dflash_debug_q4_codes": (C.c_int, [_VP, C.c_int32, _VP, _VP, _VP]),
    "dflash_debug_head_codes": (C.c_int, [_VP, _VP, _VP, _VP]),
    "dflash_debug_q4_groupsums": (C.c_int, [_VP, C.c_int32, _VP, C.c_int32, _VP, _VP]),
    "dflash_debug_q4_matmul": (C.c_int, [_VP, C.c_int32, _VP, _VP, C.c_int32, _VP, _VP]),
    "dflash_debug_wait_expiry": (C.c_int, [_VP, C.c_int64, _VP]),
    "dflash_debug_read_kv": (C.c_int, [_VP, _VP, C.c_int32, C.c_int64, C.c_int64, _VP, _VP, _VP]),
    "dflash_debug_trace": (C.c_int, [_VP, C.c_int32]),
    "dflash_debug_trace_force": (C.c_int, [_VP, C.c_int32, C.c_int32, _VP, _VP]),
    "dflash_debug_trace_site": (C.c_int, [_VP, C.c_int32, C.POINTER(C.c_int32), C.POINTER(C.c_int32), _VP, _VP, _VP]),
    "dflash_debug_attention": (C.c_int, [_VP, C.POINTER(_VP), C.c_int32, C.c_int32, C.POINTER(C.c_int64), C.c_int32,
                                         _VP, _VP, _VP]),
    "dflash_attention_noalloc": (C.c_int, [_VP, C.POINTER(_VP), C.c_int32, C.c_int32, C.POINTER(C.c_int64),
                                           C.c_int32, _VP, _VP, _VP]),
}


def load(path: str = LIB_PATH) -> C.CDLL:
    if not os.path.exists(path):
        raise ImportError(f"libdflash.so is not built ({path}); run __graft_entry__.build() or "
                          "python -m block_speculative_drafting_gb300.csrc.build")
    lib = C.CDLL(path)
    for name, (res, args) in _SIGS.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    return lib
