"""fp64 CPU oracle of the MAC-Attention decode step.

TEST INFRASTRUCTURE ONLY.  Only the test suite, the package's ``smoke()``
check and ``bench.py``'s CPU-baseline / reference leg may import this module.
The CUDA library never calls it and shares no code with it.

This is a thin ``ctypes`` layer over ``mac_oracle.c`` (plain C, fp64), which
restates the method from "MAC-Attention" (arXiv 2604.00235): the Figure 2
caption (Match, Complete, Amend, the attention summary AS, the log-domain
merge and removal, the ring insert), the abstract (pre-RoPE L2 matching over
a short window, band recompute, stable merge) and the Figure 3 caption
(per-request rings, per-head spans).  Arrays cross as numpy; bf16 values
cross as their uint16 bit patterns.
"""
import ctypes
import os

import numpy as np

from . import build as _build

_lib = None

_d = ctypes.POINTER(ctypes.c_double)
_u16 = ctypes.POINTER(ctypes.c_uint16)
_i64 = ctypes.POINTER(ctypes.c_int64)
_i32 = ctypes.POINTER(ctypes.c_int32)


def _ptr(a, t):
    if a is None:
        return ctypes.cast(None, t)
    return a.ctypes.data_as(t)


def lib():
    """Load (building first if needed) the oracle shared library."""
    global _lib
    if _lib is not None:
        return _lib
    # MAC_ORACLE_LIB points the tests' mutation check at a deliberately broken copy
    path = os.environ.get("MAC_ORACLE_LIB") or _build.build()
    L = ctypes.CDLL(path)
    L.orc_bf16_to_double.restype = ctypes.c_double
    L.orc_bf16_to_double.argtypes = [ctypes.c_uint16]
    L.orc_num_threads.restype = ctypes.c_int
    L.orc_set_num_threads.restype = None
    L.orc_set_num_threads.argtypes = [ctypes.c_int]
    L.orc_attention_summary.restype = None
    L.orc_attention_summary.argtypes = [_d, _u16, _u16, ctypes.c_long, ctypes.c_long, ctypes.c_long,
                                        ctypes.c_int, ctypes.c_double, _d, _d]
    L.orc_merge.restype = None
    L.orc_merge.argtypes = [_d, ctypes.c_double, _d, ctypes.c_double, ctypes.c_int, _d, _d]
    L.orc_log1mexp.restype = ctypes.c_double
    L.orc_log1mexp.argtypes = [ctypes.c_double]
    L.orc_remove.restype = ctypes.c_double
    L.orc_remove.argtypes = [_d, ctypes.c_double, _d, ctypes.c_double, ctypes.c_int, _d, _d]
    L.orc_match.restype = ctypes.c_int
    L.orc_match.argtypes = [_u16, _u16, _i64, ctypes.c_int, ctypes.c_int, ctypes.c_double,
                            _d, _d, _d, ctypes.POINTER(ctypes.c_int)]
    L.orc_mac_create.restype = ctypes.c_void_p
    L.orc_mac_create.argtypes = [ctypes.c_int] * 6 + [ctypes.c_double, ctypes.c_double, ctypes.c_long,
                                                      _u16, _u16]
    L.orc_mac_destroy.restype = None
    L.orc_mac_destroy.argtypes = [ctypes.c_void_p]
    L.orc_mac_reset.restype = ctypes.c_int
    L.orc_mac_reset.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_long]
    L.orc_mac_direct_count.restype = ctypes.c_int64
    L.orc_mac_direct_count.argtypes = [ctypes.c_void_p]
    L.orc_mac_read_ring.restype = None
    L.orc_mac_read_ring.argtypes = [ctypes.c_void_p, _i64, _u16, _d, _d, _i64, _i64]
    L.orc_mac_step.restype = ctypes.c_int
    L.orc_mac_step.argtypes = [ctypes.c_void_p, ctypes.c_int, _u16, _u16, _u16, _u16, _d, _d,
                               _i32, _d, _d, _d, _i32, _i64]
    L.orc_mac_step_heads.restype = ctypes.c_int
    L.orc_mac_step_heads.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int, _u16, _u16, _u16,
                                     _u16, _d, _d, _i32, _d, _d, _d, _i32, _i64]
    L.orc_mac_seed.restype = ctypes.c_int
    L.orc_mac_seed.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, _u16, _d, _d, _i64]
    L.orc_full_step.restype = ctypes.c_int
    L.orc_full_step.argtypes = [ctypes.c_void_p, ctypes.c_int, _u16, _u16, _u16, _d, _d]
    _lib = L
    return L


def num_threads() -> int:
    """OpenMP threads the oracle's parallel loops use."""
    return lib().orc_num_threads()


def set_num_threads(n: int) -> None:
    """Threads for the oracle's following parallel loops."""
    lib().orc_set_num_threads(int(n))


def _u16c(a):
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError("bf16 arrays cross as uint16 bit patterns")
    return a


def bf16_to_f64(bits):
    """Exact value of bf16 bit patterns (uint16 array) as float64."""
    bits = np.asarray(bits, dtype=np.uint16)
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def attention_summary(q, K, V, lo, hi, scale):
    """AS over tokens [lo, hi) of one head: (o [d], lse).  q float64 [d];
    K, V uint16 (bf16 bits) [T, d]."""
    q = np.ascontiguousarray(q, dtype=np.float64)
    K, V = _u16c(K), _u16c(V)
    d = q.shape[0]
    assert K.shape[-1] == d and K.shape == V.shape and K.ndim == 2
    o = np.empty(d, np.float64)
    lse = np.empty(1, np.float64)
    lib().orc_attention_summary(_ptr(q, _d), _ptr(K, _u16), _ptr(V, _u16), d, lo, hi, d, scale,
                                _ptr(o, _d), _ptr(lse, _d))
    return o, float(lse[0])


def merge(oa, la, ob, lb):
    """Log-domain merge of two summaries of disjoint segments."""
    oa = np.ascontiguousarray(oa, np.float64)
    ob = np.ascontiguousarray(ob, np.float64)
    o = np.empty_like(oa)
    l = np.empty(1, np.float64)
    lib().orc_merge(_ptr(oa, _d), la, _ptr(ob, _d), lb, oa.shape[0], _ptr(o, _d), _ptr(l, _d))
    return o, float(l[0])


def remove(oab, lab, ob, lb):
    """Log-domain removal: summary of A from those of A u B and B.
    Returns (o, lse, 1 - e^delta)."""
    oab = np.ascontiguousarray(oab, np.float64)
    ob = np.ascontiguousarray(ob, np.float64)
    o = np.empty_like(oab)
    l = np.empty(1, np.float64)
    c = lib().orc_remove(_ptr(oab, _d), lab, _ptr(ob, _d), lb, oab.shape[0], _ptr(o, _d), _ptr(l, _d))
    return o, float(l[0]), c


def log1mexp(x: float) -> float:
    return lib().orc_log1mexp(x)


def match(q_pre, ring_q, ring_pos, tau):
    """Match one head: returns dict(slot, D, D2, qn2, hit)."""
    q_pre = _u16c(q_pre)
    ring_q = _u16c(ring_q)
    ring_pos = np.ascontiguousarray(ring_pos, np.int64)
    L, d = ring_q.shape
    D, D2, qn2 = (ctypes.c_double() for _ in range(3))
    hit = ctypes.c_int()
    slot = lib().orc_match(_ptr(q_pre, _u16), _ptr(ring_q, _u16), _ptr(ring_pos, _i64), L, d, tau,
                           ctypes.byref(D), ctypes.byref(D2), ctypes.byref(qn2), ctypes.byref(hit))
    return dict(slot=slot, D=D.value, D2=D2.value, qn2=qn2.value, hit=bool(hit.value))


class MacState:
    """Oracle state: per-request KV (caller-owned numpy arrays, written in
    place on append) and the per-request, per-head rings.

    K, V: uint16 (bf16 bits) arrays [B, t_max, Hkv, d]; kv_len[b] tokens of
    request b are valid after :meth:`reset`.
    """

    def __init__(self, K, V, heads, ring_len, band_r, tau, scale=None):
        if K.dtype != np.uint16 or V.dtype != np.uint16 or not K.flags.c_contiguous \
                or not V.flags.c_contiguous or K.shape != V.shape or K.ndim != 4:
            raise ValueError("K, V must be C-contiguous uint16 [B, t_max, Hkv, d]")
        self.K, self.V = K, V
        self.B, self.t_max, self.Hkv, self.d = K.shape
        self.H, self.L, self.r, self.tau = heads, ring_len, band_r, tau
        self.scale = (1.0 / np.sqrt(self.d)) if scale is None else scale
        self._h = lib().orc_mac_create(self.B, heads, self.Hkv, self.d, ring_len, band_r, tau,
                                       self.scale, self.t_max, _ptr(K, _u16), _ptr(V, _u16))
        if not self._h:
            raise ValueError("invalid oracle configuration")

    def __del__(self):
        h = getattr(self, "_h", None)
        if h:
            lib().orc_mac_destroy(h)
            self._h = None

    def reset(self, b, kv_len):
        if lib().orc_mac_reset(self._h, b, kv_len) != 0:
            raise ValueError("bad request or length")

    def seed(self, b, q_pre, o, lse, pos):
        """Insert n ring entries for request b: q_pre uint16 [n, H, d], o
        [n, H, d], lse [n, H], 1-based increasing positions [n]."""
        q_pre = _u16c(q_pre)
        o = np.ascontiguousarray(o, np.float64)
        lse = np.ascontiguousarray(lse, np.float64)
        pos = np.ascontiguousarray(pos, np.int64)
        n = pos.shape[0]
        assert q_pre.shape == (n, self.H, self.d) and o.shape == (n, self.H, self.d) and lse.shape == (n, self.H)
        if lib().orc_mac_seed(self._h, b, n, _ptr(q_pre, _u16), _ptr(o, _d), _ptr(lse, _d), _ptr(pos, _i64)) != 0:
            raise ValueError("bad seed entries")

    @property
    def direct_count(self):
        return lib().orc_mac_direct_count(self._h)

    def ring(self):
        B, H, L, d = self.B, self.H, self.L, self.d
        pos = np.empty((B, L), np.int64)
        q = np.empty((B, H, L, d), np.uint16)
        o = np.empty((B, H, L, d), np.float64)
        lse = np.empty((B, H, L), np.float64)
        kv_len = np.empty(B, np.int64)
        step = np.empty(B, np.int64)
        lib().orc_mac_read_ring(self._h, _ptr(pos, _i64), _ptr(q, _u16), _ptr(o, _d), _ptr(lse, _d),
                                _ptr(kv_len, _i64), _ptr(step, _i64))
        return dict(pos=pos, q=q, o=o, lse=lse, kv_len=kv_len, step=step)

    def step(self, q_pre, q_post, k_new, v_new, heads=None):
        """One MAC decode step.  q_pre, q_post uint16 [B', H, d]; k_new,
        v_new uint16 [B', Hkv, d].  Returns dict with out [B', H, d], lse
        [B', H] and the decisions.  ``heads=(lo, hi)`` evaluates only that
        range of query heads (a timing sample; other entries are undefined)."""
        q_pre, q_post, k_new, v_new = map(_u16c, (q_pre, q_post, k_new, v_new))
        Bp = q_pre.shape[0]
        H, d = self.H, self.d
        assert q_pre.shape == (Bp, H, d) and q_post.shape == (Bp, H, d)
        assert k_new.shape == (Bp, self.Hkv, d) and v_new.shape == (Bp, self.Hkv, d)
        out = np.empty((Bp, H, d), np.float64)
        lse = np.empty((Bp, H), np.float64)
        slot = np.empty((Bp, H), np.int32)
        D = np.empty((Bp, H), np.float64)
        D2 = np.empty((Bp, H), np.float64)
        qn2 = np.empty((Bp, H), np.float64)
        hit = np.empty((Bp, H), np.int32)
        p = np.empty((Bp, H), np.int64)
        h_lo, h_hi = (0, H) if heads is None else heads
        rc = lib().orc_mac_step_heads(self._h, Bp, h_lo, h_hi, _ptr(q_pre, _u16), _ptr(q_post, _u16), _ptr(k_new, _u16),
                                _ptr(v_new, _u16), _ptr(out, _d), _ptr(lse, _d), _ptr(slot, _i32),
                                _ptr(D, _d), _ptr(D2, _d), _ptr(qn2, _d), _ptr(hit, _i32), _ptr(p, _i64))
        if rc != 0:
            raise RuntimeError(f"oracle step failed ({rc})")
        return dict(out=out, lse=lse, slot=slot, D=D, D2=D2, qn2=qn2, hit=hit.astype(bool), p=p)

    def full_step(self, q_post, k_new, v_new):
        """Full-attention decode step (append, then AS_{1:m} for every head)."""
        q_post, k_new, v_new = map(_u16c, (q_post, k_new, v_new))
        Bp = q_post.shape[0]
        out = np.empty((Bp, self.H, self.d), np.float64)
        lse = np.empty((Bp, self.H), np.float64)
        rc = lib().orc_full_step(self._h, Bp, _ptr(q_post, _u16), _ptr(k_new, _u16), _ptr(v_new, _u16),
                                 _ptr(out, _d), _ptr(lse, _d))
        if rc != 0:
            raise RuntimeError(f"oracle full step failed ({rc})")
        return dict(out=out, lse=lse)


def decision_flags(D, D2, qn2, tau, rel=1e-4):
    """Cases where an fp32 decision may legitimately differ from the exact
    one: the best distance within ``rel`` (relative) of the threshold, or the
    two best distances within ``rel`` of each other."""
    D = np.asarray(D, np.float64)
    D2 = np.asarray(D2, np.float64)
    qn2 = np.asarray(qn2, np.float64)
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = np.sqrt(D / qn2)
        near_tau = np.isfinite(D) & (np.abs(ratio - tau) <= rel * max(tau, 1e-30))
        near_tie = np.isfinite(D2) & (np.abs(D2 - D) <= rel * np.maximum(D2, 1e-300))
    return near_tau | near_tie
