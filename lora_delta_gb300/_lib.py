"""ctypes loader of ``liblora_delta.so`` with the C signatures of include/lora_delta.h.

Loading fails loudly when the library has not been built: there is no CPU or
PyTorch fallback anywhere in the package.
"""
from __future__ import annotations

import ctypes
import os

from .build import LIB

_c = ctypes
_vp = _c.c_void_p
_i = _c.c_int
_i64 = _c.c_int64
_sz = _c.c_size_t
_f = _c.c_float

# name -> (restype, argtypes); mirrors include/lora_delta.h
SIGNATURES = {
    "lora_status_string": (_c.c_char_p, [_i]),
    "lora_abi_version": (_i, []),
    "lora_set_wait_limit_ns": (_c.c_uint64, [_c.c_uint64]),
    "lora_scale": (_f, [_f, _i, _i]),
    "lora_pool_pack": (_i, [_vp, _vp, _vp, _vp, _i, _i, _i, _i, _vp]),
    "lora_workspace_size": (_sz, [_i, _i, _i, _i]),
    "lora_workspace_min_size": (_sz, [_i, _i, _i, _i]),
    "lora_route": (_i, [_vp, _vp, _vp, _i, _i, _vp, _vp]),
    "lora_route_scratch_size": (_sz, [_i, _i]),
    "lora_route_with_scratch": (_i, [_vp, _vp, _vp, _i, _i, _vp, _sz, _vp, _vp]),
    "lora_shrink": (_i, [_vp, _vp, _i, _i, _vp, _vp, _vp, _i, _i, _i, _vp, _sz, _vp, _vp]),
    "lora_expand": (_i, [_vp, _i64, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _vp, _sz,
                         _vp, _vp]),
    "lora_expand_gathered": (_i, [_vp, _i64, _vp, _i, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i,
                                  _i, _vp, _sz, _vp, _vp]),
    "lora_delta_fused": (_i, [_vp, _i64, _vp, _i, _i, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i,
                              _i, _vp, _sz, _vp, _vp]),
    "lora_delta_segmented": (_i, [_vp, _i64, _vp, _i, _i, _vp, _i, _vp, _vp, _vp, _vp, _i, _i,
                                  _i, _i, _vp, _sz, _vp, _vp]),
    "lora_delta_fused_floor": (_i, [_vp, _i64, _vp, _i, _i, _vp, _vp, _vp, _vp, _i, _i, _i, _i,
                                    _vp]),
    "lora_moe_workspace_size": (_sz, [_i, _i, _i, _i, _i, _i]),
    "lora_moe_fc1_delta": (_i, [_vp, _vp, _vp, _i64, _vp, _i64, _i, _vp, _vp, _i, _i, _i, _i, _i,
                                _i, _i, _f, _vp, _sz, _vp, _vp]),
    "lora_moe_w13_delta": (_i, [_vp, _vp, _vp, _i64, _vp, _i64, _i, _vp, _vp, _vp, _i, _vp,
                                _i, _i, _i, _i, _i, _i, _i, _f, _i, _vp, _sz, _vp, _vp]),
    "lora_moe_w2_delta": (_i, [_vp, _vp, _vp, _i64, _vp, _i64, _vp, _vp, _vp, _i, _vp, _vp,
                               _i, _i, _i, _i, _i, _i, _i, _f, _i, _vp, _sz, _vp, _vp]),
    "lora_moe_w2_delta_routed": (_i, [_vp, _vp, _vp, _i64, _vp, _i64, _vp, _i, _i, _i, _i, _i,
                                      _i, _i, _f, _i, _vp, _sz, _vp, _vp]),
    "lora_get_error": (_i, [_vp, _vp, _i, _vp]),
    "lora_noalloc_scratch_bytes": (_sz, []),
    "lora_delta_fused_noalloc": (_i, [_vp, _i64, _vp, _i, _i, _vp, _vp, _vp, _vp, _vp, _i, _i,
                                      _i, _i, _i, _vp, _vp]),
}

_LIB = None


class LibraryMissing(RuntimeError):
    pass


def lib() -> ctypes.CDLL:
    global _LIB
    if _LIB is not None:
        return _LIB
    if not os.path.exists(LIB):
        raise LibraryMissing(
            f"{LIB} is not built; run `python -c 'import __graft_entry__ as g; g.build()'` "
            "(there is no fallback path)")
    L = ctypes.CDLL(LIB)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(L, name)
        fn.restype = res
        fn.argtypes = args
    _LIB = L
    return L


def status_string(code: int) -> str:
    return lib().lora_status_string(code).decode()
