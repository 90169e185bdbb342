"""ctypes declarations of the C ABI in include/mac.h (libmac.so).

Loading fails loudly when the CUDA library has not been built: there is no
fallback implementation.
"""
import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "_build", "libmac.so")

MAC_OK = 0
STATUS = {0: "MAC_OK", -1: "MAC_ERR_INVALID_ARG", -2: "MAC_ERR_OOM", -3: "MAC_ERR_CUDA", -4: "MAC_ERR_CAPACITY",
          -5: "MAC_ERR_TIMEOUT", -6: "MAC_ERR_STATE"}

_vp, _i, _i64, _sz, _d, _f = (ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t, ctypes.c_double,
                              ctypes.c_float)
_pi32 = ctypes.POINTER(ctypes.c_int32)
_pu16 = ctypes.POINTER(ctypes.c_uint16)
_pf = ctypes.POINTER(ctypes.c_float)
_pi64 = ctypes.POINTER(ctypes.c_int64)
_psz = ctypes.POINTER(ctypes.c_size_t)


class MacConfig(ctypes.Structure):
    _fields_ = [("heads", _i), ("kv_heads", _i), ("head_dim", _i), ("ring_len", _i), ("band_r", _i),
                ("tau", _d), ("max_batch", _i), ("max_ctx", _i64), ("page_size", _i), ("num_pages", _i),
                ("sm_scale", _f), ("plan_mode", _i), ("amend_band", _i)]


class MacStats(ctypes.Structure):
    _fields_ = [("steps", ctypes.c_uint64), ("head_decisions", ctypes.c_uint64), ("hits", ctypes.c_uint64),
                ("kv_tokens_read", ctypes.c_uint64), ("kv_tokens_full", ctypes.c_uint64),
                ("removal_direct", ctypes.c_uint64), ("work_items", ctypes.c_uint64),
                ("device_error", ctypes.c_uint32), ("reserved", ctypes.c_uint32),
                ("tcgen05_steps", ctypes.c_uint64)]


class MacProfile(ctypes.Structure):
    _fields_ = [("match_plan_ms", _d), ("attention_ms", _d), ("combine_ms", _d), ("amend_ms", _d),
                ("steps", ctypes.c_uint64)]


_pcfg = ctypes.POINTER(MacConfig)
# Every entry point include/mac.h declares: name -> (restype, argtypes).
SIGNATURES = {
    "mac_query_sizes": (_i, [_pcfg, _psz, _psz, _psz]),
    "mac_create": (_i, [_pcfg, _vp, _sz, _vp, _sz, _vp, _sz, ctypes.POINTER(_vp)]),
    "mac_destroy": (_i, [_vp]),
    "mac_set_page_table": (_i, [_vp, _i, _vp, _i, _vp]),
    "mac_append_kv": (_i, [_vp, _i, _vp, _vp, _i64, _vp]),
    "mac_decode_step": (_i, [_vp, _i, _vp, _vp, _vp, _vp, _vp, _vp, _vp]),
    "mac_decode_step_host": (_i, [_vp, _i, _vp, _vp, _vp, _vp, _vp, _vp, _vp]),
    "mac_full_step": (_i, [_vp, _i, _vp, _vp, _vp, _vp, _vp, _vp]),
    "mac_join": (_i, [_vp, _vp]),
    "mac_sync": (_i, [_vp, _i]),
    "mac_get_stats": (_i, [_vp, ctypes.POINTER(MacStats)]),
    "mac_reset_stats": (_i, [_vp]),
    "mac_reset_request": (_i, [_vp, _i, _vp]),
    "mac_seed_ring": (_i, [_vp, _i, _i, _vp, _vp, _vp, _pi64, _vp]),
    "mac_set_profiling": (_i, [_vp, _i]),
    "mac_get_profile": (_i, [_vp, ctypes.POINTER(MacProfile)]),
    "mac_debug_force_decisions": (_i, [_vp, _vp, _i, _vp]),
    "mac_debug_get_decisions": (_i, [_vp, _i, _pi32, _pi32, _pf, _pf]),
    "mac_debug_read_ring": (_i, [_vp, _i, _pi32, _pu16, _pf, _pf, _pi64, _pi64]),
    "mac_attention_noalloc": (_i, [_i, _i, _i, _i, _i64, _vp, _vp, _pi32, _vp, _vp, _vp, _f, _vp]),
    "mac_status_string": (ctypes.c_char_p, [_i]),
    "mac_last_error": (ctypes.c_char_p, [_vp]),
}

_lib = None


class MacError(RuntimeError):
    def __init__(self, fn, status, detail=""):
        self.status = status
        super().__init__(f"{fn} -> {STATUS.get(status, status)}" + (f": {detail}" if detail else ""))


def lib():
    """The loaded CUDA library.  Raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"CUDA library not built ({LIB_PATH} missing); run "
                              "`python -c 'import __graft_entry__ as g; g.build()'`")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib
