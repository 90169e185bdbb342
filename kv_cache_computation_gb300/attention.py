"""Python binding of the MAC-Attention decode-step library (include/mac.h).

Argument marshalling only: every step of the path runs in the CUDA library.
PyTorch supplies device memory (the three backing buffers, inputs, outputs)
and the current CUDA stream.
"""
from __future__ import annotations

import ctypes

import numpy as np
import torch

from . import _native as N


def _check(fn, status, handle=None):
    if status != N.MAC_OK:
        detail = ""
        if handle is not None and handle.value:
            detail = (N.lib().mac_last_error(handle) or b"").decode()
        raise N.MacError(fn, status, detail)


def _stream_ptr(stream=None, device=None):
    s = torch.cuda.current_stream(device) if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _dev(t: torch.Tensor, name, dtype, shape=None, device=None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, the handle lives on {device}")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    return ctypes.c_void_p(t.data_ptr())


def _host(t: torch.Tensor, name, dtype, shape=None):
    if not isinstance(t, torch.Tensor) or t.is_cuda or not t.is_pinned():
        raise TypeError(f"{name} must be a pinned (page-locked) CPU tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    return ctypes.c_void_p(t.data_ptr())


def make_config(heads, kv_heads, head_dim, ring_len, band_r, tau, max_batch, max_ctx, page_size=16,
                num_pages=0, sm_scale=0.0, plan_mode=0, amend_band=0) -> N.MacConfig:
    return N.MacConfig(heads, kv_heads, head_dim, ring_len, band_r, float(tau), max_batch, int(max_ctx),
                       page_size, num_pages, float(sm_scale), plan_mode, amend_band)


def query_sizes(cfg: N.MacConfig):
    """(kv_bytes, ring_bytes, scratch_bytes) for a configuration (host only)."""
    kv, ring, scr = ctypes.c_size_t(), ctypes.c_size_t(), ctypes.c_size_t()
    _check("mac_query_sizes", N.lib().mac_query_sizes(ctypes.byref(cfg), ctypes.byref(kv), ctypes.byref(ring),
                                                       ctypes.byref(scr)))
    return kv.value, ring.value, scr.value


class MacAttention:
    """One attention layer's MAC decode state on the current CUDA device.

    mac_create(heads, kv_heads, head_dim, ring_len, band r, tau) plus the
    capacity (max_batch requests of up to max_ctx tokens) and the KV layout
    (page_size 16 = paged, 0 = contiguous).  Tensors passed in must live on
    the handle's GPU, and calls are made with that GPU current (as in a
    one-process-per-GPU program).
    """

    def __init__(self, heads, kv_heads, head_dim=128, ring_len=16, band_r=64, tau=0.3, max_batch=1,
                 max_ctx=4096, page_size=16, num_pages=0, sm_scale=0.0, plan_mode=0, amend_band=0, device=None):
        self.cfg = make_config(heads, kv_heads, head_dim, ring_len, band_r, tau, max_batch, max_ctx, page_size,
                               num_pages, sm_scale, plan_mode, amend_band)
        self.heads, self.kv_heads, self.head_dim = heads, kv_heads, head_dim
        self.ring_len, self.max_batch, self.band_r, self.tau = ring_len, max_batch, band_r, tau
        self.device = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
        kv, ring, scr = query_sizes(self.cfg)
        self.sizes = dict(kv=kv, ring=ring, scratch=scr)
        self._h = ctypes.c_void_p()
        with torch.cuda.device(self.device):
            self._kv = torch.empty(max(kv, 256), dtype=torch.uint8, device=self.device)
            self._ring = torch.empty(max(ring, 256), dtype=torch.uint8, device=self.device)
            self._scratch = torch.empty(max(scr, 256), dtype=torch.uint8, device=self.device)
            h = ctypes.c_void_p()
            st = N.lib().mac_create(ctypes.byref(self.cfg), ctypes.c_void_p(self._kv.data_ptr()), kv,
                                    ctypes.c_void_p(self._ring.data_ptr()), ring,
                                    ctypes.c_void_p(self._scratch.data_ptr()), scr, ctypes.byref(h))
            _check("mac_create", st)
        self._h = h

    # -- lifetime -----------------------------------------------------------
    def close(self):
        if getattr(self, "_h", None) is not None and self._h.value:
            N.lib().mac_destroy(self._h)
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # -- KV -----------------------------------------------------------------
    def set_page_table(self, req: int, pages: torch.Tensor, stream=None):
        p = _dev(pages, "pages", torch.int32, device=self.device)
        _check("mac_set_page_table",
               N.lib().mac_set_page_table(self._h, req, p, pages.numel(), _stream_ptr(stream, self.device)),
               self._h)

    def append_kv(self, req: int, k: torch.Tensor, v: torch.Tensor, stream=None):
        n = k.shape[0]
        shape = (n, self.kv_heads, self.head_dim)
        _check("mac_append_kv",
               N.lib().mac_append_kv(self._h, req, _dev(k, "k", torch.bfloat16, shape, device=self.device),
                                     _dev(v, "v", torch.bfloat16, shape, device=self.device), n,
                                     _stream_ptr(stream, self.device)), self._h)

    def seed_ring(self, req: int, q_pre: torch.Tensor, o: torch.Tensor, lse: torch.Tensor, positions, stream=None):
        """Insert ring entries <q~, AS_{1:pos-r}> (e.g. from the prefill) for request req."""
        n = q_pre.shape[0]
        pos = np.ascontiguousarray(np.asarray(positions, dtype=np.int64))
        if pos.shape != (n,):
            raise ValueError("one position per entry")
        _check("mac_seed_ring",
               N.lib().mac_seed_ring(self._h, req, n,
                                     _dev(q_pre, "q_pre", torch.bfloat16, (n, self.heads, self.head_dim),
                                          device=self.device),
                                     _dev(o, "o", torch.float32, (n, self.heads, self.head_dim), device=self.device),
                                     _dev(lse, "lse", torch.float32, (n, self.heads), device=self.device),
                                     pos.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)),
                                     _stream_ptr(stream, self.device)), self._h)

    def reset_request(self, req: int, stream=None):
        _check("mac_reset_request", N.lib().mac_reset_request(self._h, req, _stream_ptr(stream, self.device)), self._h)

    # -- steps --------------------------------------------------------------
    def _outs(self, B, device, out, lse, want_lse):
        if out is None:
            out = torch.empty((B, self.heads, self.head_dim), dtype=torch.bfloat16, device=device)
        if lse is None and want_lse:
            lse = torch.empty((B, self.heads), dtype=torch.float32, device=device)
        lp = (_dev(lse, "lse", torch.float32, (B, self.heads), device=self.device) if lse is not None
              else ctypes.c_void_p(None))
        return out, lse, lp

    def decode_step(self, q_pre, q_post, k_new, v_new, out=None, lse=None, want_lse=True, stream=None):
        """One MAC decode step: Match, Complete, merge and Amend (Amend on the side
        stream when the handle was made with amend_band=1)."""
        B = q_pre.shape[0]
        qs, ks = (B, self.heads, self.head_dim), (B, self.kv_heads, self.head_dim)
        out, lse, lp = self._outs(B, q_pre.device, out, lse, want_lse)
        st = N.lib().mac_decode_step(self._h, B, _dev(q_pre, "q_pre", torch.bfloat16, qs, device=self.device),
                                     _dev(q_post, "q_post", torch.bfloat16, qs, device=self.device),
                                     _dev(k_new, "k_new", torch.bfloat16, ks, device=self.device),
                                     _dev(v_new, "v_new", torch.bfloat16, ks, device=self.device),
                                     _dev(out, "out", torch.bfloat16, qs, device=self.device), lp,
                                     _stream_ptr(stream, self.device))
        _check("mac_decode_step", st, self._h)
        return out, lse

    def decode_step_host(self, q_pre, q_post, k_new, v_new, out, lse=None, stream=None):
        """decode_step with pinned host tensors: the step's kernels read the
        inputs and write out (and lse) in place in host memory; the results
        are valid once `stream` has been synchronised."""
        B = q_pre.shape[0]
        qs, ks = (B, self.heads, self.head_dim), (B, self.kv_heads, self.head_dim)
        lp = _host(lse, "lse", torch.float32, (B, self.heads)) if lse is not None else ctypes.c_void_p(None)
        st = N.lib().mac_decode_step_host(self._h, B, _host(q_pre, "q_pre", torch.bfloat16, qs),
                                          _host(q_post, "q_post", torch.bfloat16, qs),
                                          _host(k_new, "k_new", torch.bfloat16, ks),
                                          _host(v_new, "v_new", torch.bfloat16, ks),
                                          _host(out, "out", torch.bfloat16, qs), lp, _stream_ptr(stream, self.device))
        _check("mac_decode_step_host", st, self._h)
        return out, lse

    def full_step(self, q_post, k_new, v_new, out=None, lse=None, want_lse=True, stream=None):
        """Full split-KV decode attention (no Match, no ring update)."""
        B = q_post.shape[0]
        qs, ks = (B, self.heads, self.head_dim), (B, self.kv_heads, self.head_dim)
        out, lse, lp = self._outs(B, q_post.device, out, lse, want_lse)
        st = N.lib().mac_full_step(self._h, B, _dev(q_post, "q_post", torch.bfloat16, qs, device=self.device),
                                   _dev(k_new, "k_new", torch.bfloat16, ks, device=self.device),
                                   _dev(v_new, "v_new", torch.bfloat16, ks, device=self.device),
                                   _dev(out, "out", torch.bfloat16, qs, device=self.device), lp,
                                   _stream_ptr(stream, self.device))
        _check("mac_full_step", st, self._h)
        return out, lse

    def join(self, stream=None):
        _check("mac_join", N.lib().mac_join(self._h, _stream_ptr(stream, self.device)), self._h)

    def sync(self, timeout_ms: int = 10000):
        _check("mac_sync", N.lib().mac_sync(self._h, timeout_ms), self._h)

    # -- observability --------------------------------------------------------
    def stats(self) -> dict:
        s = N.MacStats()
        _check("mac_get_stats", N.lib().mac_get_stats(self._h, ctypes.byref(s)), self._h)
        return {f: getattr(s, f) for f, _ in N.MacStats._fields_ if f != "reserved"}

    def reset_stats(self):
        _check("mac_reset_stats", N.lib().mac_reset_stats(self._h), self._h)

    def set_profiling(self, on: bool):
        _check("mac_set_profiling", N.lib().mac_set_profiling(self._h, int(bool(on))), self._h)

    def profile(self) -> dict:
        p = N.MacProfile()
        _check("mac_get_profile", N.lib().mac_get_profile(self._h, ctypes.byref(p)), self._h)
        return {f: getattr(p, f) for f, _ in N.MacProfile._fields_}

    # -- test hooks ---------------------------------------------------------
    def force_decisions(self, slots: torch.Tensor, stream=None):
        B = slots.shape[0]
        _check("mac_debug_force_decisions",
               N.lib().mac_debug_force_decisions(self._h, _dev(slots, "slots", torch.int32, (B, self.heads),
                                                                 device=self.device), B,
                                                 _stream_ptr(stream, self.device)), self._h)

    def decisions(self, batch: int) -> dict:
        n = batch * self.heads
        slot, hit = np.empty(n, np.int32), np.empty(n, np.int32)
        D, qn2 = np.empty(n, np.float32), np.empty(n, np.float32)
        c = lambda a, t: a.ctypes.data_as(ctypes.POINTER(t))
        _check("mac_debug_get_decisions",
               N.lib().mac_debug_get_decisions(self._h, batch, c(slot, ctypes.c_int32), c(hit, ctypes.c_int32),
                                               c(D, ctypes.c_float), c(qn2, ctypes.c_float)), self._h)
        sh = (batch, self.heads)
        return dict(slot=slot.reshape(sh), hit=hit.reshape(sh).astype(bool), D=D.reshape(sh), qn2=qn2.reshape(sh))

    def read_ring(self, req: int) -> dict:
        L, H, d = self.ring_len, self.heads, self.head_dim
        pos = np.empty(L, np.int32)
        q = np.empty((H, L, d), np.uint16)
        o = np.empty((H, L, d), np.float32)
        lse = np.empty((H, L), np.float32)
        kv_len, steps = ctypes.c_int64(), ctypes.c_int64()
        c = lambda a, t: a.ctypes.data_as(ctypes.POINTER(t))
        _check("mac_debug_read_ring",
               N.lib().mac_debug_read_ring(self._h, req, c(pos, ctypes.c_int32), c(q, ctypes.c_uint16),
                                           c(o, ctypes.c_float), c(lse, ctypes.c_float), ctypes.byref(kv_len),
                                           ctypes.byref(steps)), self._h)
        return dict(pos=pos, q=q, o=o, lse=lse, kv_len=kv_len.value, steps=steps.value)


def status_string(code: int) -> str:
    return N.lib().mac_status_string(code).decode()
