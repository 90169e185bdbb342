"""GPU parity of the CUDA path against the fp64 oracle, through the C ABI.

Shapes span several KV pages, several work items per group and a ragged
tail; edge cases cover empty prefill, single tokens, band wider than the
context, ring length 1, and every GQA/MQA group size.
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


def cfg(**kw):
    base = dict(name="t", batch=2, heads=32, kv_heads=8, head_dim=128, context=600, steps=12, ring_len=8,
                band_r=32, tau=0.3, rho=0.99, paged=True)
    base.update(kw)
    return W.DecodeConfig(**base)


def _pair(c, **kw):
    from gpu_harness import Pair
    return Pair(c, **kw)


@pytest.mark.parametrize("page_size", [16, 0])
@pytest.mark.parametrize("context", [1, 15, 300, 2049])
def test_full_step_matches_oracle(page_size, context):
    p = _pair(cfg(context=context, steps=3), page_size=page_size)
    for t in range(3):
        p.full_step(t)


@pytest.mark.parametrize("kv_heads", [32, 16, 8, 4, 2, 1])
def test_full_step_every_group_size(kv_heads):
    p = _pair(cfg(kv_heads=kv_heads, context=777, steps=2, batch=2))
    for t in range(2):
        p.full_step(t)


@pytest.mark.parametrize("amend_band", [0, 1])
@pytest.mark.parametrize("page_size", [16, 0])
@pytest.mark.parametrize("band_r,ring_len", [(32, 8), (64, 16), (16, 1), (150, 4)])
def test_mac_chain_under_oracle_decisions(page_size, band_r, ring_len, amend_band):
    p = _pair(cfg(band_r=band_r, ring_len=ring_len, steps=16), page_size=page_size, amend_band=amend_band)
    hits = 0
    for t in range(16):
        ref, _ = p.mac_step(t, force=True)
        hits += int(ref["hit"].sum())
    assert hits > 0
    st = p.mac.stats()
    assert st["device_error"] == 0 and st["steps"] == 16


def test_mac_chain_own_decisions():
    p = _pair(cfg(steps=16, rho=0.995, ring_len=6))
    hits = 0
    for t in range(16):
        ref, _ = p.mac_step(t, force=False)
        hits += int(ref["hit"].sum())
    assert hits > 0
    st = p.mac.stats()
    assert st["hits"] == hits and st["head_decisions"] == 16 * 2 * 32


@pytest.mark.parametrize("amend_band", [0, 1])
@pytest.mark.parametrize("kv_heads", [32, 8, 4, 1])
def test_mac_chain_group_sizes(kv_heads, amend_band):
    p = _pair(cfg(kv_heads=kv_heads, context=500, steps=10, rho=0.995, ring_len=4), amend_band=amend_band)
    for t in range(10):
        p.mac_step(t, force=True)


@pytest.mark.parametrize("kv_heads,ring_len", [(1, 16), (1, 17), (1, 32), (1, 33), (8, 16), (8, 17), (8, 32), (8, 33),
                                               (2, 20), (4, 9)])
def test_match_forms_at_their_ring_size_limits(kv_heads, ring_len):
    """Each form of Match on both sides of the ring sizes where it changes:
    up to 16 and up to 32 entries scanned in the Match block (8 or 16 loads
    per lane), longer rings through the scan kernel first.  Groups of 32
    heads (four Match blocks of 8), 16 heads (two of 8), 8 and 4 heads (one
    block).  The ring fills and wraps."""
    steps = ring_len + 6
    p = _pair(cfg(kv_heads=kv_heads, context=300, steps=steps, rho=0.995, ring_len=ring_len))
    hits = 0
    for t in range(steps):
        ref, _ = p.mac_step(t, force=True)
        hits += int(ref["hit"].sum())
    assert hits > 0


def test_heterogeneous_rho_and_lengths():
    c = cfg(batch=3, rho_range=(0.5, 0.999), steps=14, context=900, band_r=64)
    p = _pair(c, contexts=[900, 40, 333])
    for t in range(14):
        p.mac_step(t, force=True)


@pytest.mark.parametrize("amend_band", [0, 1])
def test_empty_prefill_and_band_wider_than_context(amend_band):
    p = _pair(cfg(context=0, steps=20, band_r=64, ring_len=4, rho=0.999), amend_band=amend_band)
    for t in range(20):
        p.mac_step(t, force=True)


def test_tau_zero_never_hits_and_is_full_attention():
    p = _pair(cfg(tau=0.0, steps=8, rho=0.9999))
    for t in range(8):
        ref, _ = p.mac_step(t, force=False)
        assert not ref["hit"].any()
    assert p.mac.stats()["hits"] == 0


@pytest.mark.parametrize("plan_mode", [0, 1])
def test_plan_modes_agree_with_oracle(plan_mode):
    c = cfg(batch=4, rho_range=(0.5, 0.999), steps=8, context=1500)
    p = _pair(c, plan_mode=plan_mode)
    for t in range(8):
        p.mac_step(t, force=True, check_ring=(t == 7))


def test_kv_bytes_accounting():
    c = cfg(steps=6, rho=0.999)
    p = _pair(c)
    for t in range(6):
        p.mac_step(t, force=True, check_ring=False)
    st = p.mac.stats()
    full = sum(2 * 8 * (600 + t + 1) for t in range(6))
    assert st["kv_tokens_full"] == full
    assert 0 < st["kv_tokens_read"] <= full


def test_capacity_and_argument_errors():
    from kv_cache_computation_gb300 import MacError
    c = cfg(steps=1, context=20)
    p = _pair(c)
    dev, _ = p.step_inputs(0)
    p.mac.decode_step(*dev)
    with pytest.raises(MacError) as e:
        p.mac.decode_step(*dev)                       # max_ctx = context + steps reached
    assert e.value.status == -4
    with pytest.raises(MacError):
        p.mac.append_kv(0, torch.zeros((1, 8, 128), dtype=torch.bfloat16, device="cuda"),
                        torch.zeros((1, 8, 128), dtype=torch.bfloat16, device="cuda"))
    with pytest.raises(TypeError):
        p.mac.decode_step(dev[0].float(), *dev[1:])
    p.mac.sync()
    assert p.mac.stats()["device_error"] == 0


def test_reset_request_restarts_cleanly():
    c = cfg(steps=6, batch=1, context=100)
    p = _pair(c, extra_steps=200)
    for t in range(3):
        p.mac_step(t, force=True, check_ring=False)
    p.mac.reset_request(0)
    p.mac.sync()
    r = p.mac.read_ring(0)
    assert r["kv_len"] == 0 and r["steps"] == 0 and not r["pos"].any()


def test_plan_fits_one_wave_of_the_grid():
    """Balanced planning keeps the long-segment items within one wave of the
    persistent grid when there are few groups; each group's band is one more
    item on top (a CTA that takes one starts its long item a band later)."""
    c = cfg(batch=1, context=20000, steps=3, rho=0.5)
    p = _pair(c)
    for t in range(3):
        p.mac_step(t, force=True, check_ring=False)
    st = p.mac.stats()
    grid = torch.cuda.get_device_properties(0).multi_processor_count * 2
    assert st["work_items"] / st["steps"] <= grid + c.batch * c.kv_heads


@pytest.mark.parametrize("amend_band", [0, 1])
def test_graph_captured_decode_loop_matches_oracle(amend_band):
    """A decode loop captured into a CUDA graph and replayed gives the same
    per-step outputs as the oracle (mac_sync before capture, mac_join at its
    end)."""
    import numpy as np
    from gpu_harness import check_out, KEYS
    import oracle
    c = cfg(steps=11, rho=0.995, ring_len=4, batch=2)
    p = _pair(c, amend_band=amend_band)
    for t in range(2):                           # eager steps first
        p.mac_step(t, force=False, check_ring=False)
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
        flag = oracle.decision_flags(ref["D"], ref["D2"], ref["qn2"], c.tau)
        assert not flag.any()
        check_out(outs[i], lses[i], ref, f"graph step {i}")
    p.check_ring(9)
    # eager steps continue after the replay (ordered behind it on this stream)
    out, lse = p.mac.decode_step(*[p.inputs[k][10].cuda().contiguous() for k in KEYS])
    p.mac.sync()
    assert out.isfinite().all()


@pytest.mark.parametrize("ring_len,n_seed", [(128, 100), (1024, 1100)])
def test_wide_ring_seeded_from_prefill(ring_len, n_seed):
    """Rings far longer than a warp (scanned by the grid-wide kernel), seeded
    with prefill entries: the last prefill queries of an AR(1) stream that
    leads into the decode stream, with summaries AS_{1:pos-r} from the
    oracle handed to both sides in fp32."""
    import math
    import numpy as np
    import oracle
    from conftest import bf16_value
    c = cfg(ring_len=ring_len, steps=10, context=1500, rho=0.995, band_r=32, batch=2)
    p = _pair(c)
    B, H, d, G = c.batch, c.heads, c.head_dim, c.group
    rng = np.random.default_rng(5)
    # prefill queries: AR(1) run backwards from the first decode query
    x = bf16_value(W.bf16_bits(p.inputs["q_pre"][0])).astype(np.float64)
    seeds = np.empty((n_seed, B, H, d))
    for i in range(n_seed - 1, -1, -1):
        x = c.rho * x + math.sqrt(1 - c.rho ** 2) * rng.standard_normal(x.shape)
        seeds[i] = x
    pos = np.arange(c.context - n_seed + 1, c.context + 1, dtype=np.int64)
    q_pre = torch.from_numpy(seeds).to(torch.bfloat16)
    q_post = W.to_bf16(W.rope(q_pre.double().reshape(n_seed, B * H, d), torch.from_numpy(pos - 1), c.rope_base)
                       ).reshape(n_seed, B, H, d)
    for b in range(B):
        qp = W.bf16_bits(q_pre[:, b].contiguous())
        o = np.zeros((n_seed, H, d), np.float64)
        lse = np.zeros((n_seed, H), np.float64)
        for i in range(n_seed):
            for h in range(H):
                o[i, h], lse[i, h] = oracle.attention_summary(
                    bf16_value(W.bf16_bits(q_post[i, b, h])), p.orc.K[b, :, h // G], p.orc.V[b, :, h // G],
                    0, max(0, pos[i] - c.band_r), 1 / math.sqrt(d))
        o32, l32 = o.astype(np.float32), lse.astype(np.float32)
        p.orc.seed(b, qp, o32.astype(np.float64), l32.astype(np.float64), pos)
        p.mac.seed_ring(b, q_pre[:, b].contiguous().cuda(), torch.from_numpy(o32).cuda(),
                        torch.from_numpy(l32).cuda(), pos)
    p.check_ring(-1)
    hits = 0
    for t in range(c.steps):
        ref, _ = p.mac_step(t, force=True, check_ring=(t == c.steps - 1))
        hits += int(ref["hit"].sum())
    assert hits > 0


@pytest.mark.parametrize("amend_band", [0, 1])
def test_host_buffer_step_is_the_device_step(amend_band):
    """mac_decode_step_host -- inputs and results in pinned host memory, read
    and written in place by the step's kernels -- gives bitwise the outputs,
    LSEs, decisions and rings of mac_decode_step on the same inputs, with
    Amend in the merge epilogue or on the side stream; the device path
    itself is checked against the oracle step by step."""
    from gpu_harness import check_out, KEYS
    c = cfg(steps=12, rho=0.995, ring_len=8)
    pd, ph = _pair(c, amend_band=amend_band), _pair(c, amend_band=amend_band)
    B, H, d = c.batch, c.heads, c.head_dim
    h_out = torch.empty((B, H, d), dtype=torch.bfloat16).pin_memory()
    h_lse = torch.empty((B, H), dtype=torch.float32).pin_memory()
    for t in range(c.steps):
        dev, host = pd.step_inputs(t)
        ref = pd.orc.step(*host)
        out_d, lse_d = pd.mac.decode_step(*dev)
        h_in = [ph.inputs[k][t].contiguous().pin_memory() for k in KEYS]
        ph.mac.decode_step_host(*h_in, out=h_out, lse=h_lse)
        pd.mac.sync()
        ph.mac.sync()
        torch.cuda.synchronize()
        check_out(out_d, lse_d, ref, f"step {t}")
        assert torch.equal(out_d.cpu().view(torch.int16), h_out.view(torch.int16)), f"step {t}: out differs"
        assert torch.equal(lse_d.cpu(), h_lse), f"step {t}: lse differs"
        dd, dh = pd.mac.decisions(B), ph.mac.decisions(B)
        for k in dd:
            np.testing.assert_array_equal(dd[k], dh[k])
    for b in range(B):
        rd, rh = pd.mac.read_ring(b), ph.mac.read_ring(b)
        for k in rd:
            np.testing.assert_array_equal(np.asarray(rd[k]), np.asarray(rh[k]))
    assert ph.mac.stats()["hits"] > 0 and ph.mac.stats()["device_error"] == 0


def test_host_buffer_step_refuses_pageable_memory():
    """Pageable host memory is refused before any launch: by the binding, and
    by the C entry point itself (MAC_ERR_INVALID_ARG, no step taken)."""
    import ctypes
    from gpu_harness import KEYS
    from kv_cache_computation_gb300 import _native as N
    c = cfg(steps=1)
    p = _pair(c)
    args = [p.inputs[k][0].contiguous() for k in KEYS]
    out = torch.empty((c.batch, c.heads, c.head_dim), dtype=torch.bfloat16)
    with pytest.raises(TypeError):
        p.mac.decode_step_host(*args, out=out)
    ptrs = [ctypes.c_void_p(a.data_ptr()) for a in args]
    st = N.lib().mac_decode_step_host(p.mac._h, c.batch, *ptrs, ctypes.c_void_p(out.data_ptr()), None, None)
    assert st == -1
    torch.cuda.synchronize()
    assert p.mac.stats()["steps"] == 0


@pytest.mark.parametrize("amend_band", [0, 1])
def test_band_holding_the_mass_takes_the_direct_form(amend_band):
    """Log-domain removal is ill-conditioned when the band [m-r+1, m] holds
    almost all of AS_{1:m}'s mass.  Each step's new key is 4x the sum of its
    KV group's post-RoPE queries (fresh random queries every step), so the
    new token outscores every other by a wide margin and 1 - e^delta falls
    far below 1/32: the GPU must then store AS_{1:m-r} in its direct form
    (counted in removal_direct), on hit and on miss steps, and the ring
    entries must still match the oracle's."""
    c = cfg(steps=14, rho=0.995, ring_len=4, band_r=8, context=300)
    p = _pair(c, amend_band=amend_band)
    gen = torch.Generator().manual_seed(31)
    B, H, Hkv, G, d = c.batch, c.heads, c.kv_heads, c.group, c.head_dim
    for t in range(c.steps):
        qp = W.to_bf16(torch.randn((B, H, d), generator=gen, dtype=torch.float64))
        p.inputs["q_post"][t] = qp
        p.inputs["k_new"][t] = W.to_bf16(4.0 * qp.double().reshape(B, Hkv, G, d).sum(2))
    hits = misses = 0
    for t in range(c.steps):
        ref, _ = p.mac_step(t, force=True)
        if c.context + t + 1 > c.band_r:
            hits += int(ref["hit"].sum())
            misses += int((~ref["hit"]).sum())
    assert hits > 0 and misses > 0
    st = p.mac.stats()
    assert st["device_error"] == 0
    # every (request, head) of every step past the band is ill-conditioned
    assert st["removal_direct"] == c.steps * B * H, st["removal_direct"]


@pytest.mark.parametrize("kv_heads,context", [(8, 3000), (1, 20000)])
def test_refused_page_is_reported_and_leaves_other_requests_exact(kv_heads, context):
    """A page-table entry outside the pool is refused on the device: the step
    completes, the bounds-check word reports it, and no other request's
    output moves.  GQA 32/8 runs the mma.sync kernel; MQA at 2 x 20001
    tokens the tcgen05 kernel."""
    from gpu_harness import check_out
    p = _pair(cfg(kv_heads=kv_heads, context=context, steps=1))
    bad = p.pages[0].clone()
    bad[5] = 1 << 30
    p.mac.set_page_table(0, bad.contiguous())
    dev, host = p.step_inputs(0)
    ref = p.orc.full_step(host[1], host[2], host[3])
    out, lse = p.mac.full_step(*dev[1:])
    torch.cuda.synchronize()
    st = p.mac.stats()
    assert st["device_error"] & 1
    assert st["tcgen05_steps"] == (1 if kv_heads == 1 else 0)
    check_out(out[1:], lse[1:], {"out": ref["out"][1:], "lse": ref["lse"][1:]}, "request 1")
    from kv_cache_computation_gb300 import _native as N
    with pytest.raises(N.MacError):   # the handle reports the refused page and stays failed
        p.mac.sync()
