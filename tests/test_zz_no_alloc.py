"""mac_attention_noalloc: decode attention for callers that cannot allocate.

Some callers may not allocate device memory where they run attention (a
runtime with one arena planned at start-up, a latency-critical loop that must
not call cudaMalloc, a plug-in host that only hands over its buffers).  This
entry point keeps its scratch in a fixed array inside the library instead of
a caller-allocated buffer.  The test drives it through the C ABI and checks
every call against the fp64 oracle's full attention, element by element,
with the tolerance the other GPU tests use, over consecutive calls of
different shapes (the scratch regions move with the shape, so each call
finds the previous call's bytes under its own), at contexts long enough for
the attention kernel's shared page pools to engage, with every KV slot past
a request's length holding NaN.  It also checks that an oversized call is
refused.

Kept in a file of its own that pytest collects last, so a stop-at-first-
failure run has already run every other test when it gets here.
"""
import ctypes

import numpy as np
import pytest
import torch

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]

OUT_TOL, LSE_TOL = 5e-3, 1e-4


def _noalloc(lib, B, H, Hkv, ctx_stride, K, V, lens, q, out, lse):
    lens_c = (ctypes.c_int32 * B)(*lens)
    return lib.mac_attention_noalloc(B, H, Hkv, 128, ctx_stride, ctypes.c_void_p(K.data_ptr()),
                                     ctypes.c_void_p(V.data_ptr()), lens_c, ctypes.c_void_p(q.data_ptr()),
                                     ctypes.c_void_p(out.data_ptr()),
                                     ctypes.c_void_p(lse.data_ptr() if lse is not None else None), 0.0,
                                     ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _oracle_attention(K, V, lens, q_bits, H):
    """AS_{1:len}(q) per request and query head from the fp64 oracle.
    K, V uint16 [B, T, Hkv, d]; q_bits uint16 [B, H, d]."""
    import oracle
    B = K.shape[0]
    st = oracle.MacState(K.copy(), V.copy(), H, 1, 1, 0.0)
    idx = np.asarray(lens) - 1
    for b in range(B):
        st.reset(b, int(idx[b]))               # the last token is appended by the full step itself
    k_last = np.ascontiguousarray(K[np.arange(B), idx])
    v_last = np.ascontiguousarray(V[np.arange(B), idx])
    return st.full_step(q_bits, k_last, v_last)


def _call_case(lib, B, H, Hkv, lens, seed):
    from kv_cache_computation_gb300 import _native as N
    from kv_cache_computation_gb300 import workloads as W
    T = max(lens)
    ctx_stride = (T + 15) // 16 * 16 + 16
    cfg = W.DecodeConfig(f"noalloc_{B}x{H}x{Hkv}", B, H, Hkv, 128, T, 1, 1, 1, 0.0, paged=False, seed=seed)
    K, V = W.prefill_kv(cfg, device="cuda")
    g = torch.Generator(device="cuda").manual_seed(seed)
    q = torch.randn((B, H, 128), generator=g, device="cuda").to(torch.bfloat16)
    # the caller's cache: every slot NaN, then each request's tokens
    Kc = torch.full((B, Hkv, ctx_stride, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    Vc = torch.full_like(Kc, float("nan"))
    for b, n in enumerate(lens):
        Kc[b, :, :n] = K[b, :n].transpose(0, 1)
        Vc[b, :, :n] = V[b, :n].transpose(0, 1)
    out = torch.empty((B, H, 128), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((B, H), dtype=torch.float32, device="cuda")
    st = _noalloc(lib, B, H, Hkv, ctx_stride, Kc, Vc, lens, q, out, lse)
    assert st == 0, N.STATUS.get(st, st)
    torch.cuda.synchronize()
    ref = _oracle_attention(W.bf16_bits(K), W.bf16_bits(V), lens, W.bf16_bits(q), H)
    o = out.float().cpu().numpy().astype(np.float64)
    err = np.abs(o - ref["out"]).max(-1) / np.maximum(np.abs(ref["out"]).max(-1), 1e-30)
    assert np.isfinite(o).all(), "NaN from the slots past a request's length reached the output"
    assert err.max() <= OUT_TOL, f"{B}x{H}x{Hkv}: output error {err.max():.3g}"
    lerr = np.abs(lse.cpu().numpy().astype(np.float64) - ref["lse"]).max()
    assert lerr <= LSE_TOL, f"{B}x{H}x{Hkv}: lse error {lerr:.3g}"


def test_noalloc_matches_oracle_on_consecutive_calls_of_different_shapes():
    from kv_cache_computation_gb300 import build
    from kv_cache_computation_gb300 import _native as N
    build.build()
    lib = N.lib()
    # one request (8 groups, ~66-page work items), then eight ragged requests
    # (64 groups, ~250-page items), a 4-group call with an 8-head group and a
    # 45-token request, and the first shape again: every call's work items
    # are long enough for the shared page pools, whose claim counters sit
    # elsewhere in the array from one shape to the next
    _call_case(lib, 1, 32, 8, [39997], seed=11)
    _call_case(lib, 8, 32, 8, [20000 + 37 * b for b in range(8)], seed=12)
    _call_case(lib, 2, 32, 4, [30001, 45], seed=13)
    _call_case(lib, 1, 32, 8, [39997], seed=14)


def test_noalloc_refuses_what_its_scratch_cannot_hold():
    from kv_cache_computation_gb300 import build
    from kv_cache_computation_gb300 import _native as N
    build.build()
    lib = N.lib()
    # 64 requests of 256 query heads over 8 KV heads need more partial-summary
    # scratch than the fixed array holds on any grid: refused before any launch
    B, H, Hkv, ctx_stride = 64, 256, 8, 16
    K = torch.zeros((B, Hkv, ctx_stride, 128), dtype=torch.bfloat16, device="cuda")
    q = torch.zeros((B, H, 128), dtype=torch.bfloat16, device="cuda")
    out = torch.empty_like(q)
    st = _noalloc(lib, B, H, Hkv, ctx_stride, K, K, [16] * B, q, out, None)
    assert st == -4   # MAC_ERR_CAPACITY
    st = _noalloc(lib, 65, 32, 8, ctx_stride, K, K, [16] * 65, q, out, None)
    assert st == -1   # batch beyond 64
