"""GPU parity at the full sizes of the benchmark workloads, in the launch
configuration bench.py times (persistent attention grid, balanced plan,
programmatic dependent launch, Amend in the merge epilogue).

Every decode step is checked against the fp64 oracle on all requests and
heads: Match decisions bit-exact except near-threshold / near-tie cases, the
outputs and LSE within the method's tolerances, and the rings.  The GPU runs
under the oracle's decisions so a flagged divergence cannot derail the chain.
"""
import numpy as np
import pytest
import torch

from kv_cache_computation_gb300 import workloads as W

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]


@pytest.fixture(scope="module", autouse=True)
def _built():
    from kv_cache_computation_gb300 import build
    build.build()


def _run(cfg, steps, page_size, ring_every=8):
    from gpu_harness import Pair
    p = Pair(cfg, page_size=page_size)
    hits = 0
    for t in range(steps):
        ref, _ = p.mac_step(t, force=True, check_ring=(t % ring_every == ring_every - 1))
        hits += int(ref["hit"].sum())
    st = p.mac.stats()
    assert st["device_error"] == 0
    return p, hits


def test_llama_layer_4k_contiguous_all_64_steps():
    cfg = W.llama_gqa_4k_b1_contig()
    p, hits = _run(cfg, cfg.steps, page_size=0)
    assert hits > 0


def test_llama_8x32k_paged_first_32_steps():
    cfg = W.llama_gqa_32k_b8_paged(steps=32)
    p, hits = _run(cfg, 32, page_size=16)
    assert hits > 0


@pytest.mark.parametrize("band_r", [32, 64, 128])
def test_llama_128k_heterogeneous_rho(band_r):
    cfg = W.llama_gqa_128k_b1_hetero(steps=24, band_r=band_r)
    p, hits = _run(cfg, 24, page_size=16, ring_every=12)
    # per-head rho ~ U[0.5, 0.99]: only the most correlated heads hit
    assert hits > 0


def test_qwen_stack_layer_4x120k_hits():
    """One layer of the 48-layer stack at full size (4 x 122880, 32 q / 4 KV
    heads, per-channel K/V scales), tau 0.45 so heads hit and miss."""
    cfg = W.qwen_moe_stack_120k_b4(steps=12, tau=0.45, layers=1)
    p, hits = _run(cfg, 12, page_size=16, ring_every=6)
    assert hits > 0


@pytest.mark.parametrize("kv_heads", [8, 1])
def test_forced_hit_sweep_largest_point(kv_heads):
    """The sweep's largest points, 32 requests x 131072 tokens (GQA 32/8,
    17 GB of KV; MQA 32/1), 90 % forced hits, every request on the GPU and
    four of them (the first and last two) on the oracle."""
    from gpu_harness import SampledPair
    cfg = W.sweep_point(131072, 32, 0.9, kv_heads, steps=6)
    p = SampledPair(cfg, requests=[0, 1, 30, 31])
    for t in range(cfg.steps):
        p.step(t, check_ring=(t == cfg.steps - 1))
    assert p.hits > 0
    assert p.mac.stats()["device_error"] == 0
