"""GB300 (sm_103a) MAC-Attention decode-step attention.

Match-Amend-Complete decode attention (arXiv 2604.00235) behind the C ABI of
include/mac.h, with a thin Python binding:

    from kv_cache_computation_gb300 import MacAttention
    mac = MacAttention(heads=32, kv_heads=8, ring_len=16, band_r=64, tau=0.3,
                       max_batch=1, max_ctx=8192, page_size=0)
    mac.append_kv(0, k_prefill, v_prefill)
    out, lse = mac.decode_step(q_pre_rope, q_post_rope, k_new, v_new)

The CUDA library must be built first (``kv_cache_computation_gb300.build``);
there is no CPU fallback.
"""
from .attention import MacAttention, make_config, query_sizes, status_string  # noqa: F401
from ._native import MacError  # noqa: F401
