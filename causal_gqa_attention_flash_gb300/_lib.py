"""ctypes declarations of libgqa_attn.so: the C ABI of include/gqa_attn.h and the testing hooks of
include/gqa_attn_testing.h."""

from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
# GQA_ATTN_DEBUG=1 selects the checking build (every kernel checks its computed coordinates and
# reports a failed check as GQA_ERR_BOUNDS); it is read once, when the library is first loaded.
DEBUG = os.environ.get("GQA_ATTN_DEBUG", "0") == "1"
LIB_PATH = os.path.join(_HERE, "libgqa_attn_debug.so" if DEBUG else "libgqa_attn.so")

_c_int, _c_float, _vp, _sz = ctypes.c_int, ctypes.c_float, ctypes.c_void_p, ctypes.c_size_t

SIGNATURES = {
    "gqa_attn_fwd": (_c_int, [_vp, _vp, _vp, _vp, _vp] + [_c_int] * 6 + [_c_float, _vp]),
    "gqa_attn_fwd_cached": (_c_int, [_vp, _vp, _vp, _vp, _vp] + [_c_int] * 7 + [_c_float, _vp]),
    "gqa_attn_fwd_splitkv_workspace_size": (_sz, [_c_int] * 6),
    "gqa_attn_fwd_splitkv": (_c_int, [_vp] * 6 + [_sz] + [_c_int] * 7 + [_c_float, _vp]),
    "gqa_attn_fwd_varlen": (_c_int, [_vp] * 7 + [_c_int] * 8 + [_c_float, _vp]),
    "gqa_attn_bwd_workspace_size": (_sz, [_c_int] * 5),
    "gqa_attn_bwd_varlen_workspace_size": (_sz, [_c_int] * 4),
    "gqa_attn_bwd_deterministic": (_c_int, [_vp] * 10 + [_sz] + [_c_int] * 6 + [_c_float, _vp]),
    "gqa_attn_fwd_rope_workspace_size": (_sz, [_c_int] * 4),
    "gqa_attn_fwd_rope": (_c_int, [_vp] * 8 + [_sz] + [_c_int] * 6 + [_c_float, _vp]),
    "gqa_attn_bwd_rope_workspace_size": (_sz, [_c_int] * 5),
    "gqa_attn_bwd_rope": (_c_int, [_vp] * 12 + [_sz] + [_c_int] * 6 + [_c_float, _vp]),
    "gqa_attn_bwd_varlen": (_c_int, [_vp] * 10 + [_c_int] * 2 + [_vp, _sz] + [_c_int] * 5 + [_c_float, _vp]),
    "gqa_attn_bwd": (_c_int, [_vp] * 10 + [_sz] + [_c_int] * 6 + [_c_float, _vp]),
    "gqa_attn_get_error": (_c_int, [_vp]),
    "gqa_attn_strerror": (ctypes.c_char_p, [_c_int]),
    "gqa_attn_last_cuda_error": (_c_int, []),
    "gqa_attn_selftest_wait_timeout": (_c_int, [_c_int, _vp]),
    "gqa_attn_trace_arm": (_c_int, []),
    "gqa_attn_trace_collect": (_c_int, [ctypes.POINTER(_c_int), ctypes.POINTER(ctypes.c_double)]),
    "gqa_attn_bwd_noalloc": (_c_int, [_vp] * 9 + [_c_int] * 6 + [_c_float, _vp]),
    "gqa_attn_decode_workspace_size": (_sz, [_c_int] * 7),
    "gqa_attn_decode_fwd": (_c_int, [_vp] * 6 + [_sz] + [_c_int] * 7 + [_c_float, _c_int, _vp]),
}

_lib = None


def load() -> ctypes.CDLL:
    """Load the library once. Raises if it has not been built: there is no fallback."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with `python -m causal_gqa_attention_flash_gb300.build --all` "
                "(the CUDA library is the only implementation; there is no CPU fallback)")
        lib = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib
