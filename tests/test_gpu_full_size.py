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


def _run(cfg, steps, page_size, ring_every=8, layer=0):
    from gpu_harness import Pair
    p = Pair(cfg, page_size=page_size, layer=layer)
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


@pytest.mark.parametrize("layer", [0, 47])
def test_qwen_stack_layer_4x120k_hits(layer):
    """The first and the last layer of the 48-layer stack at full size
    (4 x 122880, 32 q / 4 KV heads, the layer's own per-channel K/V scales
    and query streams), tau 0.45 so heads hit and miss."""
    cfg = W.qwen_moe_stack_120k_b4(steps=12, tau=0.45, layers=48)
    p, hits = _run(cfg, 12, page_size=16, ring_every=6, layer=layer)
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
    st = p.mac.stats()
    assert st["device_error"] == 0
    # groups of 32 heads at this size run on the tcgen05 kernel, others on mma.sync
    assert st["tcgen05_steps"] == (cfg.steps if kv_heads == 1 else 0)


def test_llama_128k_graph_replay_like_the_benchmark():
    """The benchmark's headline path at its full size: the decode loop of the
    128K workload captured into a CUDA graph and replayed, the GPU making its
    own decisions; every replayed step equals the oracle's."""
    import oracle
    from gpu_harness import Pair, check_out, KEYS
    cfg = W.llama_gqa_128k_b1_hetero(steps=14, band_r=64)
    p = Pair(cfg, page_size=16)
    for t in range(4):                           # eager steps first
        p.mac_step(t, force=False, check_ring=False)
    p.mac.sync()
    B, H, n = cfg.batch, cfg.heads, 10
    ins = [[p.inputs[k][t].cuda().contiguous() for k in KEYS] for t in range(4, 4 + n)]
    outs = [torch.empty((B, H, 128), dtype=torch.bfloat16, device="cuda") for _ in range(n)]
    lses = [torch.empty((B, H), dtype=torch.float32, device="cuda") for _ in range(n)]
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            for i in range(n):
                p.mac.decode_step(*ins[i], out=outs[i], lse=lses[i])
            p.mac.join()
    torch.cuda.synchronize()
    g.replay()
    torch.cuda.synchronize()
    hits = 0
    for i in range(n):
        ref = p.orc.step(*[W.bf16_bits(p.inputs[k][4 + i]) for k in KEYS])
        assert not oracle.decision_flags(ref["D"], ref["D2"], ref["qn2"], cfg.tau).any()
        hits += int(ref["hit"].sum())
        check_out(outs[i], lses[i], ref, f"graph step {i}")
    p.check_ring(4 + n - 1)
    assert hits > 0
    assert p.mac.stats()["device_error"] == 0
