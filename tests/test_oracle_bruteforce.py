"""Brute-force pin of the oracle's full MAC decode step on tiny shapes (no GPU).

An independent restatement of "MAC-Attention", Figure 2 (a)-(c), written
with explicit token sets and plain exponentials instead of log-domain
operators:

* AS of a set S for query q is (sum_j e^{z_j} v_j / Z, log Z), Z = sum_j e^{z_j};
* two summaries are combined by weighting each with e^{lse};
* the ring entry of step m is, by definition, the summary of tokens
  {1..m-r} as seen by the step (on a hit at p: the reused entry of p
  combined with tokens {p-r+1..m-r}); it is built directly here, never by
  removal, so a wrong sign or index in the oracle's removal fails.
"""
import math
from fractions import Fraction

import numpy as np
import pytest

import oracle
from conftest import bf16_value, bits


def as_set(q, K, V, S, scale):
    if not S:
        return [0.0] * len(q), -math.inf
    w = [math.exp(scale * sum(qi * ki for qi, ki in zip(q, K[j]))) for j in S]
    Z = sum(w)
    o = [sum(wj * V[j][i] for wj, j in zip(w, S)) / Z for i in range(len(q))]
    return o, math.log(Z)


def combine(a, b):
    (oa, la), (ob, lb) = a, b
    ea = 0.0 if la == -math.inf else math.exp(la)
    eb = 0.0 if lb == -math.inf else math.exp(lb)
    if ea + eb == 0.0:
        return [0.0] * len(oa), -math.inf
    return [(ea * x + eb * y) / (ea + eb) for x, y in zip(oa, ob)], math.log(ea + eb)


class BruteMac:
    """Per-request KV lists and per-(request, head) rings as Python lists."""

    def __init__(self, K0, V0, H, L, r, tau, scale):
        self.K = [[list(map(list, kv)) for kv in Kb] for Kb in K0]   # [b][t][g] -> d floats
        self.V = [[list(map(list, kv)) for kv in Vb] for Vb in V0]
        self.H, self.L, self.r, self.tau, self.scale = H, L, r, tau, scale
        self.B = len(K0)
        self.Hkv = len(K0[0][0])
        self.G = H // self.Hkv
        self.ring = [[[] for _ in range(H)] for _ in range(self.B)]  # entries: dict(pos, q, AS, t)
        self.steps = [0] * self.B

    def step(self, q_pre, q_post, k_new, v_new):
        B = len(q_pre)
        res = []
        for b in range(B):
            self.K[b].append([list(x) for x in k_new[b]])
            self.V[b].append([list(x) for x in v_new[b]])
            m = len(self.K[b])                     # 1-based position of the new token
            rb = []
            for h in range(self.H):
                g = h // self.G
                Kg = [kt[g] for kt in self.K[b]]
                Vg = [vt[g] for vt in self.V[b]]
                qt = [Fraction(x) for x in q_pre[b][h]]
                best = None
                for ent in self.ring[b][h]:
                    D = sum((a - Fraction(c)) ** 2 for a, c in zip(qt, ent["q"]))
                    if best is None or D < best[0] or (D == best[0] and ent["pos"] > best[1]["pos"]):
                        best = (D, ent)
                qn2 = sum(a * a for a in qt)
                hit = best is not None and best[0] < Fraction(self.tau) ** 2 * qn2
                q = q_post[b][h]
                # index sets are 0-based token indices; position P is index P-1
                if hit:
                    p = best[1]["pos"]
                    span = list(range(max(0, p - self.r), m))          # positions p-r+1..m
                    out = combine(best[1]["AS"], as_set(q, Kg, Vg, span, self.scale))
                    if m > self.r:
                        ent_as = combine(best[1]["AS"],
                                         as_set(q, Kg, Vg, list(range(max(0, p - self.r), m - self.r)), self.scale))
                    else:
                        ent_as = ([0.0] * len(q), -math.inf)
                else:
                    p = 0
                    out = as_set(q, Kg, Vg, list(range(m)), self.scale)
                    ent_as = as_set(q, Kg, Vg, list(range(m - self.r)), self.scale) if m > self.r \
                        else ([0.0] * len(q), -math.inf)
                rb.append(dict(out=out, hit=hit, p=p, ent=dict(pos=m, q=list(q_pre[b][h]), AS=ent_as)))
            for h in range(self.H):
                ring = self.ring[b][h]
                new = rb[h]["ent"]
                if len(ring) < self.L:
                    ring.append(new)
                else:
                    ring[self.steps[b] % self.L] = new
            self.steps[b] += 1
            res.append(rb)
        return res


def _tolist(a):
    return [[[float(x) for x in row] for row in mat] for mat in a]


@pytest.mark.parametrize("B,H,Hkv,L,r,tau", [(1, 2, 1, 3, 2, 0.6), (2, 4, 2, 3, 2, 0.5), (1, 2, 2, 2, 3, 0.7)])
def test_mac_steps_match_brute_force(B, H, Hkv, L, r, tau):
    rng = np.random.default_rng(7 + B + H + r)
    d, ctx, steps = 4, 2, 7
    t_max = ctx + steps
    scale = 0.5
    K = np.zeros((B, t_max, Hkv, d), np.uint16)
    V = np.zeros((B, t_max, Hkv, d), np.uint16)
    K[:, :ctx] = bits(rng.standard_normal((B, ctx, Hkv, d)))
    V[:, :ctx] = bits(rng.standard_normal((B, ctx, Hkv, d)))
    st = oracle.MacState(K, V, H, L, r, tau, scale)
    for b in range(B):
        st.reset(b, ctx)
    bf = BruteMac(_tolist_kv(K[:, :ctx]), _tolist_kv(V[:, :ctx]), H, L, r, tau, scale)
    qt = rng.standard_normal((B, H, d))
    n_hits = 0
    for t in range(steps):
        qt = qt + 0.15 * rng.standard_normal((B, H, d))       # slowly drifting queries: hits happen
        q_pre = bits(qt)
        q_post = bits(bf16_value(q_pre) + 0.3 * rng.standard_normal((B, H, d)))
        k_new = bits(rng.standard_normal((B, Hkv, d)))
        v_new = bits(rng.standard_normal((B, Hkv, d)))
        got = st.step(q_pre, q_post, k_new, v_new)
        exp = bf.step(_tolist(bf16_value(q_pre)), _tolist(bf16_value(q_post)),
                      _tolist(bf16_value(k_new)), _tolist(bf16_value(v_new)))
        ring = st.ring()
        for b in range(B):
            for h in range(H):
                e = exp[b][h]
                assert bool(got["hit"][b, h]) == e["hit"], (t, b, h)
                n_hits += e["hit"]
                if e["hit"]:
                    assert got["p"][b, h] == e["p"]
                np.testing.assert_allclose(got["out"][b, h], e["out"][0], rtol=0, atol=1e-12)
                assert got["lse"][b, h] == pytest.approx(e["out"][1], abs=1e-12)
                # the freshly inserted ring entry is AS_{1:m-r} by definition
                slot = t % L
                ent = e["ent"]
                assert ring["pos"][b, slot] == ent["pos"]
                np.testing.assert_array_equal(bf16_value(ring["q"][b, h, slot]), ent["q"])
                if ent["AS"][1] == -math.inf:
                    assert ring["lse"][b, h, slot] == -math.inf
                else:
                    np.testing.assert_allclose(ring["o"][b, h, slot], ent["AS"][0], rtol=0, atol=1e-11)
                    assert ring["lse"][b, h, slot] == pytest.approx(ent["AS"][1], abs=1e-11)
    assert n_hits > 0, "workload should exercise the hit path"


def _tolist_kv(A):
    return [[[[float(x) for x in bf16_value(A[b, t, g])] for g in range(A.shape[2])]
             for t in range(A.shape[1])] for b in range(A.shape[0])]


def test_band_holding_the_mass_takes_the_direct_form():
    """Removal is ill-conditioned when the band [m-r+1, m] carries almost all
    of AS_{1:m}'s mass (1 - e^delta near 0): the stored summary is then
    formed directly as the merge of its parts.  Each new key is a growing
    multiple of the (fixed) post-RoPE query direction, so the newest token's
    score exceeds every older one by 20: the prefix [1, m-r] holds about
    e^-40 of the mass.  The ring entry must still equal AS_{1:m-r} built from
    its token set, on hit steps (reused prefix merged with [p-r+1, m-r]) and
    on miss steps (tokens [1, m-r])."""
    B, H, Hkv, d, L, r, tau, scale = 1, 2, 1, 4, 3, 2, 0.3, 0.5
    ctx, steps = 3, 8
    rng = np.random.default_rng(2604)
    t_max = ctx + steps
    K = np.zeros((B, t_max, Hkv, d), np.uint16)
    V = np.zeros((B, t_max, Hkv, d), np.uint16)
    K[:, :ctx] = bits(rng.standard_normal((B, ctx, Hkv, d)))
    V[:, :ctx] = bits(rng.standard_normal((B, ctx, Hkv, d)))
    st = oracle.MacState(K, V, H, L, r, tau, scale)
    st.reset(0, ctx)
    bf = BruteMac(_tolist_kv(K[:, :ctx]), _tolist_kv(V[:, :ctx]), H, L, r, tau, scale)
    u = np.ones(d)
    q_post = bits(np.stack([u, 0.75 * u])[None])               # [1, H, d]: scores 2 alpha and 1.5 alpha
    qt = rng.standard_normal((B, H, d))
    reuse = {1, 2, 4, 5, 7}                                    # steps whose pre-RoPE query barely moves
    hit_steps = miss_steps = 0
    for t in range(steps):
        qt = qt + 0.01 * rng.standard_normal(qt.shape) if t in reuse else rng.standard_normal(qt.shape)
        q_pre = bits(qt)
        k_new = bits((10.0 * (t + 1)) * u[None, None])         # alpha_t = 10 (t + 1)
        v_new = bits(rng.standard_normal((B, Hkv, d)))
        before = st.direct_count
        got = st.step(q_pre, q_post, k_new, v_new)
        exp = bf.step(_tolist(bf16_value(q_pre)), _tolist(bf16_value(q_post)),
                      _tolist(bf16_value(k_new)), _tolist(bf16_value(v_new)))
        m = ctx + t + 1
        ring = st.ring()
        slot = t % L
        for h in range(H):
            e = exp[0][h]
            assert bool(got["hit"][0, h]) == e["hit"], (t, h)
            np.testing.assert_allclose(got["out"][0, h], e["out"][0], rtol=0, atol=1e-12)
            ent = e["ent"]["AS"]
            np.testing.assert_allclose(ring["o"][0, h, slot], ent[0], rtol=0, atol=1e-11)
            assert ring["lse"][0, h, slot] == pytest.approx(ent[1], abs=1e-11)
            if m > r:
                hit_steps += e["hit"]
                miss_steps += not e["hit"]
        if m > r:
            assert st.direct_count - before == H, f"step {t}: the removal should have been ill-conditioned"
    assert hit_steps > 0 and miss_steps > 0
