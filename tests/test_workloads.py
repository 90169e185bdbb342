"""The seeded synthetic input generators (no GPU): determinism and the
statistical shape of each stream."""
import math

import numpy as np
import pytest
import torch

from kv_cache_computation_gb300 import workloads as W


def _small(**kw):
    base = dict(name="t", batch=2, heads=8, kv_heads=2, head_dim=32, context=40, steps=30, ring_len=4,
                band_r=8, tau=0.3)
    base.update(kw)
    return W.DecodeConfig(**base)


def test_generation_is_deterministic_and_layer_dependent():
    cfg = _small()
    a = W.decode_inputs(cfg)
    b = W.decode_inputs(cfg)
    for k in a:
        assert torch.equal(a[k], b[k])
    c = W.decode_inputs(cfg, layer=1)
    assert not torch.equal(a["q_pre"], c["q_pre"])
    K1, V1 = W.prefill_kv(cfg)
    K2, V2 = W.prefill_kv(cfg)
    assert torch.equal(K1, K2) and torch.equal(V1, V2)
    assert K1.dtype == torch.bfloat16 and K1.shape == (2, 40, 2, 32)


def test_windows_agree_with_the_full_sequence():
    cfg = _small()
    full = W.decode_inputs(cfg)
    part = W.decode_inputs(cfg, steps=7, first_step=11)
    for k in part:
        assert torch.equal(part[k], full[k][11:18])


def test_ar1_lag1_correlation_matches_rho():
    cfg = _small(batch=4, heads=32, head_dim=128, steps=200, rho=0.9)
    q = W.decode_inputs(cfg)["q_pre"].double()
    x, y = q[:-1].flatten(), q[1:].flatten()
    corr = float(torch.corrcoef(torch.stack([x, y]))[0, 1])
    assert corr == pytest.approx(0.9, abs=0.01)
    assert float(q.std()) == pytest.approx(1.0, abs=0.05)


def test_per_head_rho_range():
    cfg = _small(rho_range=(0.5, 0.99), heads=64)
    r = W.head_rhos(cfg)
    assert r.min() >= 0.5 and r.max() <= 0.99 and r.std() > 0.05


def test_rope_is_a_rotation_and_identity_at_zero():
    x = torch.randn(5, 3, 64, dtype=torch.float64)
    pos = torch.tensor([0, 1, 7, 1000, 131071])
    y = W.rope(x, pos, 500000.0)
    torch.testing.assert_close(y.norm(dim=-1), x.norm(dim=-1), rtol=1e-12, atol=1e-12)
    torch.testing.assert_close(y[0], x[0], rtol=0, atol=0)
    # relative position property: <R(a)x, R(b)y> depends on a-b only
    u, v = torch.randn(1, 1, 64, dtype=torch.float64), torch.randn(1, 1, 64, dtype=torch.float64)
    d1 = (W.rope(u, torch.tensor([10]), 1e4) * W.rope(v, torch.tensor([3]), 1e4)).sum()
    d2 = (W.rope(u, torch.tensor([107]), 1e4) * W.rope(v, torch.tensor([100]), 1e4)).sum()
    assert float(d1) == pytest.approx(float(d2), rel=1e-10)


def test_forced_hit_stream_distances():
    cfg = _small(forced_hit_rate=0.5, steps=60, heads=8, kv_heads=2, head_dim=128, batch=3)
    d = W.decode_inputs(cfg)
    q = d["q_pre"].double()
    forced = d["forced"]
    assert not forced[0].any()
    rel = (q[1:] - q[:-1]).norm(dim=-1) / q[1:].norm(dim=-1)        # [S-1, B, H]
    f = forced[1:].repeat_interleave(cfg.group, dim=2)
    assert rel[f].max() < 0.03
    assert rel[~f].min() > 1.0
    assert 0.35 < float(forced[1:].double().mean()) < 0.65


def test_page_tables_are_a_permutation():
    pt = W.page_tables(4, 25, seed=3)
    assert pt.shape == (4, 25) and pt.dtype == torch.int32
    assert sorted(pt.flatten().tolist()) == list(range(100))
    assert not torch.equal(pt.flatten(), torch.arange(100, dtype=torch.int32))


def test_channel_scales_log_uniform():
    cfg = _small(channel_scale_range=(0.5, 2.0), head_dim=128, kv_heads=4)
    s = W.channel_scales(cfg, 0)
    assert s.shape == (2, 4, 128)
    assert s.min() >= 0.5 and s.max() <= 2.0
    assert abs(float(torch.log(s).mean())) < 0.1


def test_named_workloads():
    c1 = W.llama_gqa_4k_b1_contig()
    assert (c1.batch, c1.heads, c1.kv_heads, c1.context, c1.steps, c1.ring_len, c1.band_r, c1.paged) == \
        (1, 32, 8, 4096, 64, 16, 64, False)
    c3 = W.llama_gqa_128k_b1_hetero()
    assert c3.context == 131072 and c3.ring_len == 32 and c3.rho_range == (0.5, 0.99)
    c4 = W.qwen_moe_stack_120k_b4()
    assert c4.layers == 48 and c4.kv_heads == 4 and c4.context == 122880
    assert c3.kv_bytes_full_per_step(0) == 131073 * 8 * 128 * 4


def test_gap_stream_recurs_at_its_gap():
    """q~_t = q~_{t-gap} + 0.1 eps: the query of `gap` steps back is ~0.1
    away (relative), the one just before is an unrelated draw."""
    cfg = _small(gap=4, gap_noise=0.1, heads=4, kv_heads=2, head_dim=64, steps=40)
    q = W.decode_inputs(cfg)["q_pre"].double()
    rel = lambda a, b: ((a - b).norm(dim=-1) / a.norm(dim=-1)).mean().item()
    at_gap = [rel(q[t], q[t - 4]) for t in range(4, 40)]
    at_one = [rel(q[t], q[t - 1]) for t in range(4, 40)]
    assert max(at_gap) < 0.15 and min(at_one) > 1.0


def test_topic_stream_prefill_queries_lead_into_decode():
    """The topic stream's `lead` prefill queries are the process steps just
    before decode step 0: the same process with lead 0 and lead + S steps
    holds both, in order; queries revisit a few prototypes, so most decode
    queries have an earlier query within 0.2 (relative) among the previous
    lead + t ones."""
    lead, S = 24, 30
    a = _small(topics=4, topic_stay=0.9, topic_noise=0.05, lead=lead, steps=S, heads=4, kv_heads=2, head_dim=64)
    b = _small(topics=4, topic_stay=0.9, topic_noise=0.05, lead=0, steps=lead + S, heads=4, kv_heads=2, head_dim=64)
    qp, qq = W.prefill_queries(a)
    assert qp.shape == (lead, 2, 4, 64) and qq.shape == qp.shape
    dec_a = W.decode_inputs(a)["q_pre"]
    dec_b = W.decode_inputs(b)["q_pre"]
    assert torch.equal(dec_b[:lead], qp) and torch.equal(dec_b[lead:], dec_a)
    allq = dec_b.double()
    near = 0
    for t in range(lead, lead + S):
        d = ((allq[:t] - allq[t]).norm(dim=-1) / allq[t].norm(dim=-1)).min(dim=0).values
        near += (d < 0.2).float().mean().item()
    assert near / S > 0.8
