"""mac_attention_noalloc: decode attention for callers that cannot allocate.

Some callers may not allocate device memory where they run attention (a
runtime with one arena planned at start-up, a latency-critical loop that must
not call cudaMalloc, a plug-in host that only hands over its buffers).  This
entry point keeps its scratch in a fixed array inside the library instead of
a caller-allocated buffer.  The test drives it through the C ABI and checks
it against mac_full_step -- the handle-based entry point computing the same
attention -- on two consecutive decode steps, with the tolerance the other
GPU tests use, and checks that an oversized call is refused.

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


def _rel_err(a, b):
    a = a.float().cpu().numpy().astype(np.float64)
    b = b.float().cpu().numpy().astype(np.float64)
    return (np.abs(a - b).max(axis=-1) / np.maximum(np.abs(b).max(axis=-1), 1e-30)).max()


def _noalloc(lib, B, H, Hkv, ctx_stride, K, V, lens, q, out, lse):
    lens_c = (ctypes.c_int32 * B)(*lens)
    return lib.mac_attention_noalloc(B, H, Hkv, 128, ctx_stride, ctypes.c_void_p(K.data_ptr()),
                                     ctypes.c_void_p(V.data_ptr()), lens_c, ctypes.c_void_p(q.data_ptr()),
                                     ctypes.c_void_p(out.data_ptr()),
                                     ctypes.c_void_p(lse.data_ptr() if lse is not None else None), 0.0,
                                     ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def test_noalloc_matches_full_step_on_two_calls():
    from kv_cache_computation_gb300 import MacAttention, build
    from kv_cache_computation_gb300 import _native as N
    from kv_cache_computation_gb300 import workloads as W
    build.build()
    lib = N.lib()
    B, H, Hkv, ctx, steps = 2, 32, 8, 700, 2
    cfg = W.DecodeConfig("noalloc_gqa32x8_ctx700_b2", B, H, Hkv, 128, ctx, steps, 4, 32, 0.3, paged=False)
    K0, V0 = W.prefill_kv(cfg)
    inp = W.decode_inputs(cfg)
    max_ctx = ctx + steps
    mac = MacAttention(H, Hkv, 128, 4, 32, 0.3, max_batch=B, max_ctx=max_ctx, page_size=0)
    ctx_stride = (max_ctx + 15) // 16 * 16
    # the caller's own KV cache in the same contiguous layout
    Kc = torch.zeros((B, Hkv, ctx_stride, 128), dtype=torch.bfloat16, device="cuda")
    Vc = torch.zeros_like(Kc)
    for b in range(B):
        mac.append_kv(b, K0[b].cuda().contiguous(), V0[b].cuda().contiguous())
        Kc[b, :, :ctx] = K0[b].transpose(0, 1).cuda()
        Vc[b, :, :ctx] = V0[b].transpose(0, 1).cuda()
    for t in range(steps):                       # two calls in a row, state carried over
        q = inp["q_post"][t].cuda().contiguous()
        kn = inp["k_new"][t].cuda().contiguous()
        vn = inp["v_new"][t].cuda().contiguous()
        ref_out, ref_lse = mac.full_step(q, kn, vn)
        Kc[:, :, ctx + t] = kn
        Vc[:, :, ctx + t] = vn
        out = torch.empty_like(ref_out)
        lse = torch.empty_like(ref_lse)
        st = _noalloc(lib, B, H, Hkv, ctx_stride, Kc, Vc, [ctx + t + 1] * B, q, out, lse)
        assert st == 0, N.STATUS.get(st, st)
        torch.cuda.synchronize()
        assert _rel_err(out, ref_out) <= OUT_TOL
        assert (lse - ref_lse).abs().max().item() <= LSE_TOL
    mac.close()


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
