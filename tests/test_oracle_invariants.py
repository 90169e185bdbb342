"""Invariants of the oracle's MAC step on realistic head sizes (no GPU).

"MAC-Attention", Figure 2 caption and abstract:
* with threshold 0 nothing ever hits, so every step is full attention;
* reusing the summary of an identical earlier query is exact: the reused
  prefix AS_{1:p-r} was computed with the same post-RoPE query;
* the stored ring entry, obtained by log-domain removal, equals the summary
  of tokens {1..m-r} computed directly;
* a hit never reads the KV prefix [1, p-r] yet the output still equals the
  definition (reused prefix merged with fresh band+tail attention).
"""
import math

import numpy as np
import pytest

import oracle
from conftest import bf16_value, bits


def _setup(rng, B=2, H=8, Hkv=2, d=64, ctx=300, steps=12, L=6, r=32, tau=0.3):
    t_max = ctx + steps + 4
    K = np.zeros((B, t_max, Hkv, d), np.uint16)
    V = np.zeros((B, t_max, Hkv, d), np.uint16)
    K[:, :ctx] = bits(rng.standard_normal((B, ctx, Hkv, d)))
    V[:, :ctx] = bits(rng.standard_normal((B, ctx, Hkv, d)))
    return K, V, dict(B=B, H=H, Hkv=Hkv, d=d, ctx=ctx, steps=steps, L=L, r=r, tau=tau)


def _stream(rng, c, rho):
    q = rng.standard_normal((c["B"], c["H"], c["d"]))
    for _ in range(c["steps"]):
        q = rho * q + math.sqrt(1 - rho * rho) * rng.standard_normal(q.shape)
        yield (bits(q), bits(q + 0.2 * rng.standard_normal(q.shape)),
               bits(rng.standard_normal((c["B"], c["Hkv"], c["d"]))),
               bits(rng.standard_normal((c["B"], c["Hkv"], c["d"]))))


def test_zero_threshold_is_full_attention_bitwise(rng):
    K, V, c = _setup(rng)
    K2, V2 = K.copy(), V.copy()
    mac = oracle.MacState(K, V, c["H"], c["L"], c["r"], 0.0)
    full = oracle.MacState(K2, V2, c["H"], c["L"], c["r"], 0.0)
    for b in range(c["B"]):
        mac.reset(b, c["ctx"])
        full.reset(b, c["ctx"])
    for qp, qq, kn, vn in _stream(rng, c, 0.999):
        a = mac.step(qp, qq, kn, vn)
        f = full.full_step(qq, kn, vn)
        assert not a["hit"].any()
        np.testing.assert_array_equal(a["out"], f["out"])
        np.testing.assert_array_equal(a["lse"], f["lse"])


def test_identical_query_reuse_is_exact(rng):
    K, V, c = _setup(rng, steps=8, tau=0.05, L=8)
    mac = oracle.MacState(K, V, c["H"], c["L"], c["r"], c["tau"])
    for b in range(c["B"]):
        mac.reset(b, c["ctx"])
    shape = (c["B"], c["H"], c["d"])
    kv = (c["B"], c["Hkv"], c["d"])
    saved = None
    for t in range(c["steps"]):
        if t == 6:
            qp, qq = saved                       # repeat step 2's queries exactly
        else:
            qp, qq = bits(rng.standard_normal(shape)), bits(rng.standard_normal(shape))
        if t == 2:
            saved = (qp, qq)
            p_expected = c["ctx"] + 3            # 1-based position of step 2's token
        kn, vn = bits(rng.standard_normal(kv)), bits(rng.standard_normal(kv))
        out = mac.step(qp, qq, kn, vn)
        if t < 6:
            assert not out["hit"].any()          # fresh random queries are far apart
        if t == 6:
            assert out["hit"].all()
            assert (out["p"] == p_expected).all() and (out["D"] == 0).all()
            m = c["ctx"] + 7
            for b in range(c["B"]):
                for h in range(c["H"]):
                    g = h // (c["H"] // c["Hkv"])
                    o_ref, l_ref = oracle.attention_summary(bf16_value(qq[b, h]), K[b, :, g], V[b, :, g], 0, m,
                                                            1 / math.sqrt(c["d"]))
                    np.testing.assert_allclose(out["out"][b, h], o_ref, rtol=0, atol=1e-12)
                    assert out["lse"][b, h] == pytest.approx(l_ref, abs=1e-12)


@pytest.mark.parametrize("rho", [0.5, 0.97, 0.995])
def test_ring_entry_equals_direct_prefix_summary(rng, rho):
    K, V, c = _setup(rng, tau=0.3, r=16, ctx=120, steps=10)
    mac = oracle.MacState(K, V, c["H"], c["L"], c["r"], c["tau"])
    for b in range(c["B"]):
        mac.reset(b, c["ctx"])
    s = 1 / math.sqrt(c["d"])
    G = c["H"] // c["Hkv"]
    prev_ring = None
    hits = 0
    for t, (qp, qq, kn, vn) in enumerate(_stream(rng, c, rho)):
        out = mac.step(qp, qq, kn, vn)
        ring = mac.ring()
        m = c["ctx"] + t + 1
        slot = t % c["L"]
        for b in range(c["B"]):
            for h in range(c["H"]):
                g = h // G
                q = bf16_value(qq[b, h])
                if out["hit"][b, h]:
                    hits += 1
                    e, p = out["slot"][b, h], out["p"][b, h]
                    pre = (prev_ring["o"][b, h, e], prev_ring["lse"][b, h, e])
                    mid = oracle.attention_summary(q, K[b, :, g], V[b, :, g], max(0, p - c["r"]), m - c["r"], s)
                    o_ref, l_ref = oracle.merge(*pre, *mid)
                else:
                    o_ref, l_ref = oracle.attention_summary(q, K[b, :, g], V[b, :, g], 0, m - c["r"], s)
                np.testing.assert_allclose(ring["o"][b, h, slot], o_ref, rtol=0, atol=1e-11)
                assert ring["lse"][b, h, slot] == pytest.approx(l_ref, abs=1e-11)
        prev_ring = ring
    if rho > 0.99:
        assert hits > 0


def test_hit_output_is_reused_prefix_merged_with_band_and_tail(rng):
    K, V, c = _setup(rng, tau=0.3, r=16, ctx=200, steps=10)
    mac = oracle.MacState(K, V, c["H"], c["L"], c["r"], c["tau"])
    for b in range(c["B"]):
        mac.reset(b, c["ctx"])
    s = 1 / math.sqrt(c["d"])
    G = c["H"] // c["Hkv"]
    prev = None
    hits = 0
    for t, (qp, qq, kn, vn) in enumerate(_stream(rng, c, 0.995)):
        out = mac.step(qp, qq, kn, vn)
        m = c["ctx"] + t + 1
        for b in range(c["B"]):
            for h in range(c["H"]):
                if not out["hit"][b, h]:
                    continue
                hits += 1
                e, p = out["slot"][b, h], out["p"][b, h]
                assert p < m and prev["pos"][b, e] == p
                # the reused entry's stored query is the one matched
                assert out["D"][b, h] < c["tau"] ** 2 * out["qn2"][b, h]
                tail = oracle.attention_summary(bf16_value(qq[b, h]), K[b, :, h // G], V[b, :, h // G],
                                                max(0, p - c["r"]), m, s)
                o_ref, l_ref = oracle.merge(prev["o"][b, h, e], prev["lse"][b, h, e], *tail)
                np.testing.assert_allclose(out["out"][b, h], o_ref, rtol=0, atol=1e-13)
                assert out["lse"][b, h] == pytest.approx(l_ref, abs=1e-13)
        prev = mac.ring()
    assert hits > 0


def test_early_positions_store_the_empty_summary(rng):
    # m <= r: AS_{1:m-r} is empty
    K, V, c = _setup(rng, ctx=3, steps=4, r=8)
    mac = oracle.MacState(K, V, c["H"], c["L"], c["r"], c["tau"])
    for b in range(c["B"]):
        mac.reset(b, c["ctx"])
    for t, (qp, qq, kn, vn) in enumerate(_stream(rng, c, 0.9)):
        mac.step(qp, qq, kn, vn)
        ring = mac.ring()
        assert (ring["lse"][:, :, t % c["L"]] == -math.inf).all()
        assert not ring["o"][:, :, t % c["L"]].any()


def test_ring_positions_and_wraparound(rng):
    K, V, c = _setup(rng, steps=13, L=5)
    mac = oracle.MacState(K, V, c["H"], c["L"], c["r"], c["tau"])
    for b in range(c["B"]):
        mac.reset(b, c["ctx"])
    for t, step in enumerate(_stream(rng, c, 0.5)):
        mac.step(*step)
    ring = mac.ring()
    # step t (0-based) wrote position ctx+t+1 at slot t % L; the last L steps survive
    for t in range(c["steps"] - c["L"], c["steps"]):
        assert (ring["pos"][:, t % c["L"]] == c["ctx"] + t + 1).all()
    assert (ring["kv_len"] == c["ctx"] + c["steps"]).all()
    assert (ring["step"] == c["steps"]).all()


def test_kv_capacity_is_enforced(rng):
    K, V, c = _setup(rng, steps=1)
    mac = oracle.MacState(K, V, c["H"], c["L"], c["r"], c["tau"])
    for b in range(c["B"]):
        mac.reset(b, K.shape[1])
    qp = bits(np.zeros((c["B"], c["H"], c["d"])))
    kv = bits(np.zeros((c["B"], c["Hkv"], c["d"])))
    with pytest.raises(RuntimeError):
        mac.step(qp, qp, kv, kv)


def test_seeded_ring_entries_are_matched_and_reused(rng):
    """Entries seeded from prefill queries behave exactly like decode-step
    entries: a later identical query reuses the seed's summary, and the output
    is that summary merged with fresh band+tail attention."""
    K, V, c = _setup(rng, ctx=300, steps=4, L=8, r=16, tau=0.05)
    mac = oracle.MacState(K, V, c["H"], c["L"], c["r"], c["tau"])
    s = 1 / math.sqrt(c["d"])
    G = c["H"] // c["Hkv"]
    for b in range(c["B"]):
        mac.reset(b, c["ctx"])
    n = 5
    pos = np.array([200, 230, 260, 280, 299], np.int64)
    qs = bits(rng.standard_normal((n, c["H"], c["d"])))
    qpost = bits(rng.standard_normal((n, c["H"], c["d"])))
    o = np.zeros((c["B"], n, c["H"], c["d"]))
    lse = np.zeros((c["B"], n, c["H"]))
    for b in range(c["B"]):
        for i in range(n):
            for h in range(c["H"]):
                o[b, i, h], lse[b, i, h] = oracle.attention_summary(bf16_value(qpost[i, h]), K[b, :, h // G],
                                                                    V[b, :, h // G], 0, pos[i] - c["r"], s)
        mac.seed(b, qs, o[b], lse[b], pos)
    ring = mac.ring()
    assert (ring["step"] == n).all() and sorted(ring["pos"][0][ring["pos"][0] > 0].tolist()) == pos.tolist()
    with pytest.raises(ValueError):
        mac.seed(0, qs[:2], o[0, :2], lse[0, :2], np.array([5, 5], np.int64))      # not increasing
    # a decode step whose pre- and post-RoPE queries equal seed 2's reuses it
    shape = (c["B"], c["H"], c["d"])
    kv = (c["B"], c["Hkv"], c["d"])
    qp = np.broadcast_to(qs[2], shape).copy()
    qq = np.broadcast_to(qpost[2], shape).copy()
    out = mac.step(qp, qq, bits(rng.standard_normal(kv)), bits(rng.standard_normal(kv)))
    assert out["hit"].all() and (out["p"] == pos[2]).all()
    m = c["ctx"] + 1
    for b in range(c["B"]):
        for h in range(c["H"]):
            tail = oracle.attention_summary(bf16_value(qq[b, h]), K[b, :, h // G], V[b, :, h // G],
                                            pos[2] - c["r"], m, s)
            o_ref, l_ref = oracle.merge(o[b, 2, h], lse[b, 2, h], *tail)
            np.testing.assert_allclose(out["out"][b, h], o_ref, atol=1e-13)
            # reusing an exact prefix summary with the same query is full attention
            full = oracle.attention_summary(bf16_value(qq[b, h]), K[b, :, h // G], V[b, :, h // G], 0, m, s)
            np.testing.assert_allclose(out["out"][b, h], full[0], atol=1e-12)
