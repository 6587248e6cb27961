"""ctypes declarations for libpkv_attn.so (the C ABI declared in include/pkv_attn.h).

Argument marshalling only.  The library is loaded lazily on first use; if it is missing the call
fails loudly (there is no other implementation to fall back to).
"""

from __future__ import annotations

import ctypes as C
import os
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libpkv_attn.so")

PKV_OK = 0
PKV_EINVAL = -1
PKV_EUNSUPPORTED = -2
PKV_EWORKSPACE = -3
PKV_ECUDA = -4
PKV_EDEVICE = -5

PKV_BF16 = 0
PKV_FP8_E4M3 = 1
PKV_MODE_DECODE = 0
PKV_MODE_PREFILL = 1
PKV_MODE_MIXED = 2
PKV_MODE_RAGGED = 3
PKV_MODE_PAGED_RAGGED = 4

STATUS_NAMES = {0: "PKV_OK", -1: "PKV_EINVAL", -2: "PKV_EUNSUPPORTED", -3: "PKV_EWORKSPACE", -4: "PKV_ECUDA",
                -5: "PKV_EDEVICE"}


class PkvError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status
        self.message = message


class pkv_cache(C.Structure):
    _fields_ = [
        ("k", C.c_void_p),
        ("v", C.c_void_p),
        ("num_pages", C.c_int64),
        ("page_size", C.c_int32),
        ("num_kv_heads", C.c_int32),
        ("head_dim", C.c_int32),
        ("dtype", C.c_int32),
        ("stride_page", C.c_int64),
        ("stride_token", C.c_int64),
        ("stride_head", C.c_int64),
        ("k_scale", C.c_float),
        ("v_scale", C.c_float),
    ]


_i32p = C.POINTER(C.c_int32)


class pkv_plan_args(C.Structure):
    # the index arrays are host addresses (const int32_t*), set from ndarray.ctypes.data
    _fields_ = [
        ("batch_size", C.c_int32),
        ("qo_indptr", C.c_void_p),
        ("kv_indptr", C.c_void_p),
        ("kv_indices", C.c_void_p),
        ("last_page_len", C.c_void_p),
        ("num_qo_heads", C.c_int32),
        ("num_kv_heads", C.c_int32),
        ("head_dim", C.c_int32),
        ("page_size", C.c_int32),
        ("mode", C.c_int32),
        ("causal", C.c_int32),
        ("window_left", C.c_int32),
        ("sm_scale", C.c_float),
        ("q_dtype", C.c_int32),
        ("kv_dtype", C.c_int32),
        ("max_splits", C.c_int32),
        ("num_sms", C.c_int32),
    ]


class pkv_plan_info(C.Structure):
    _fields_ = [
        ("mode", C.c_int32),
        ("batch_size", C.c_int32),
        ("total_tokens", C.c_int64),
        ("num_work", C.c_int64),
        ("num_merge", C.c_int64),
        ("num_partials", C.c_int64),
        ("kv_chunk", C.c_int64),
        ("workspace_bytes", C.c_int64),
        ("max_page_id", C.c_int64),
        ("kv_tokens", C.c_int64),
        ("num_decode_work", C.c_int64),
        ("num_decodes", C.c_int64),
        ("num_decode_tokens", C.c_int64),
        ("num_prefills", C.c_int64),
        ("num_prefill_tokens", C.c_int64),
        ("num_prefill_partials", C.c_int64),
    ]


_SIGS = {
    "pkv_kv_store": (C.c_int, [C.c_void_p, C.c_void_p, C.c_void_p, C.c_int64, C.POINTER(pkv_cache), C.c_void_p]),
    "pkv_plan_create": (C.c_int, [C.POINTER(C.c_void_p)]),
    "pkv_plan_destroy": (None, [C.c_void_p]),
    "pkv_plan_workspace_size": (C.c_int, [C.POINTER(pkv_plan_args), C.POINTER(C.c_size_t)]),
    "pkv_attn_plan": (C.c_int, [C.c_void_p, C.POINTER(pkv_plan_args), C.c_void_p, C.c_size_t, C.c_void_p]),
    "pkv_attn_decode_run": (C.c_int, [C.c_void_p, C.c_void_p, C.POINTER(pkv_cache), C.c_void_p, C.c_void_p, C.c_void_p]),
    "pkv_attn_decode_run_noalloc": (C.c_int, [C.c_void_p, C.c_void_p, C.POINTER(pkv_cache), C.c_void_p, C.c_void_p, C.c_void_p]),
    "pkv_attn_prefill_run": (C.c_int, [C.c_void_p, C.c_void_p, C.POINTER(pkv_cache), C.c_void_p, C.c_void_p, C.c_void_p]),
    "pkv_attn_prefill_run_merge": (C.c_int, [C.c_void_p, C.c_void_p, C.POINTER(pkv_cache), C.c_void_p, C.c_void_p, C.c_void_p]),
    "pkv_attn_ragged_run": (C.c_int, [C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p]),
    "pkv_attn_paged_ragged_run": (C.c_int, [C.c_void_p, C.c_void_p, C.POINTER(pkv_cache), C.c_void_p, C.c_void_p,
                                            C.c_void_p, C.c_void_p, C.c_void_p]),
    "pkv_cascade_run": (C.c_int, [C.c_void_p, C.c_void_p, C.c_void_p, C.POINTER(pkv_cache), C.c_void_p, C.c_void_p,
                                  C.c_void_p]),
    "pkv_merge_state": (C.c_int, [C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_int64,
                                  C.c_int32, C.c_void_p]),
    "pkv_last_error": (C.c_char_p, []),
    "pkv_device_error": (C.c_int, [_i32p, C.c_int32, C.c_void_p]),
    "pkv_set_wait_limit": (C.c_int, [C.c_int64]),
    "pkv_test_hold_wait": (C.c_int, [C.c_int32]),
    "pkv_plan_info_get": (C.c_int, [C.c_void_p, C.POINTER(pkv_plan_info)]),
    "pkv_plan_work_items": (C.c_int, [C.c_void_p, _i32p, C.c_int64]),
    "pkv_block_table_to_csr": (C.c_int, [_i32p, C.c_int32, C.c_int32, _i32p, C.c_int32, _i32p, _i32p, C.c_int64, _i32p]),
    "pkv_token_table_to_page_table": (C.c_int, [_i32p, C.c_int32, C.c_int32, _i32p, C.c_int32, _i32p, C.c_int64]),
}

_lib = None
_lock = threading.Lock()


def lib():
    """The loaded library (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"{LIB_PATH} is missing: build it with `python -c 'import __graft_entry__ as g; g.build()'` "
                    "(there is no CPU fallback)")
            L = C.CDLL(LIB_PATH)
            for name, (res, args) in _SIGS.items():
                f = getattr(L, name)
                f.restype = res
                f.argtypes = args
            _lib = L
    return _lib


def check(status: int) -> None:
    if status != PKV_OK:
        raise PkvError(status, lib().pkv_last_error().decode())


def exported_symbols():
    return list(_SIGS)
