"""GPU parity of the tcgen05 attention kernel against the fp64 oracle.

Groups of 32 query heads (MQA-shaped GQA) go through the tcgen05 kernel in
steps that hold at least 16384 KV tokens over all requests and KV heads;
smaller steps keep the mma.sync kernel.  These cases are sized to land on
either side of that line (the handle reports which kernel ran), with ragged
request lengths, several 128-token blocks per work item, items that start
and end inside a block, band items (a MAC step reads the band of every
request), paged and contiguous caches, and both Amend forms.
"""
import pytest
import torch

from kv_cache_computation_gb300 import workloads as W

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]


@pytest.fixture(scope="module", autouse=True)
def _built():
    from kv_cache_computation_gb300 import build
    build.build()


def cfg(**kw):
    base = dict(name="tc", batch=3, heads=32, kv_heads=1, head_dim=128, context=20000, steps=2, ring_len=4,
                band_r=64, tau=0.3, rho=0.995, paged=True)
    base.update(kw)
    return W.DecodeConfig(**base)


def _pair(c, **kw):
    from gpu_harness import Pair
    return Pair(c, **kw)


@pytest.mark.parametrize("page_size", [16, 0])
def test_full_steps_on_the_tensor_memory_kernel(page_size):
    # 3 ragged MQA requests, 33 104 tokens in the first step
    p = _pair(cfg(steps=3), contexts=[20000, 9001, 4100], page_size=page_size)
    for t in range(3):
        p.full_step(t)
    st = p.mac.stats()
    assert st["device_error"] == 0
    assert st["tcgen05_steps"] == 3


@pytest.mark.parametrize("amend_band", [0, 1])
@pytest.mark.parametrize("band_r", [64, 150])
def test_mac_chain_on_the_tensor_memory_kernel(band_r, amend_band):
    # 64 query heads over 2 KV heads (two groups of 32), 2 requests:
    # (9001 + 7778) x 2 = 33 558 tokens in the first step
    c = cfg(batch=2, heads=64, kv_heads=2, context=9000, steps=6, band_r=band_r)
    p = _pair(c, contexts=[9000, 7777], amend_band=amend_band)
    hits = 0
    for t in range(6):
        ref, _ = p.mac_step(t, force=True)
        hits += int(ref["hit"].sum())
    assert hits > 0
    st = p.mac.stats()
    assert st["device_error"] == 0
    assert st["tcgen05_steps"] == 6


def test_small_steps_of_32_head_groups_keep_the_mma_sync_kernel():
    p = _pair(cfg(batch=2, context=777, steps=2))
    for t in range(2):
        p.full_step(t)
    st = p.mac.stats()
    assert st["device_error"] == 0
    assert st["tcgen05_steps"] == 0


@pytest.mark.parametrize("amend_band", [0, 1])
def test_one_request_just_past_the_line(amend_band):
    # one MQA request of 17 000 tokens: the single group is cut into items of
    # about one 128-token block each, most starting and ending inside a block
    c = cfg(batch=1, context=17000, steps=4)
    p = _pair(c, amend_band=amend_band)
    p.full_step(0)
    for t in range(1, 4):
        p.mac_step(t, force=True)
    st = p.mac.stats()
    assert st["device_error"] == 0
    assert st["tcgen05_steps"] == 4


@pytest.mark.parametrize("amend_band", [0, 1])
def test_graph_captured_loop_on_the_tensor_memory_kernel(amend_band):
    """MQA steps of 2 x 9001+ tokens captured into a CUDA graph (programmatic
    dependent launches between the step's kernels) and replayed: every
    replayed step equals the oracle's, the GPU making its own decisions."""
    import oracle
    from gpu_harness import check_out, KEYS
    c = cfg(batch=2, context=9000, steps=11)
    p = _pair(c, amend_band=amend_band)
    for t in range(2):                           # eager steps first
        p.mac_step(t, force=False, check_ring=False)
    assert p.mac.stats()["tcgen05_steps"] == 2
    p.mac.sync()
    B, H = c.batch, c.heads
    ins = [[p.inputs[k][t].cuda().contiguous() for k in KEYS] for t in range(2, 10)]
    outs = [torch.empty((B, H, 128), dtype=torch.bfloat16, device="cuda") for _ in range(8)]
    lses = [torch.empty((B, H), dtype=torch.float32, device="cuda") for _ in range(8)]
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            for i in range(8):
                p.mac.decode_step(*ins[i], out=outs[i], lse=lses[i])
            p.mac.join()
    torch.cuda.synchronize()
    g.replay()
    torch.cuda.synchronize()
    for i in range(8):
        ref = p.orc.step(*[W.bf16_bits(p.inputs[k][i + 2]) for k in KEYS])
        assert not oracle.decision_flags(ref["D"], ref["D2"], ref["qn2"], c.tau).any()
        check_out(outs[i], lses[i], ref, f"graph step {i}")
    p.check_ring(9)
    assert p.mac.stats()["device_error"] == 0
