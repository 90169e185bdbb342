"""Seeded synthetic decode workloads for the MAC-Attention decode step.

This module only *generates inputs*; it holds none of the method's
arithmetic.  Both the CUDA path (tests, benchmark) and the fp64 oracle are fed
from it.  Everything is drawn from ``torch.Generator`` streams whose seeds are
derived from (base seed, layer, stream tag), so a workload is reproducible on
a given device.  The CPU and CUDA generators draw different numbers for the
same seed, so a caller that needs the same inputs on both sides generates
once and copies.

What is generated (the paper's workloads are LongBench v2 / RULER /
LongGenBench prompts run through trained models; none of that is available,
so seeded synthetic streams of the same shapes stand in for them):

* prefill K, V: i.i.d. N(0, 1) per element (optionally scaled per (kv-head,
  channel) by a log-uniform factor), K rotated by RoPE at its 0-based token
  index, both rounded to bf16;
* pre-RoPE decode queries q~_t: an AR(1) process per (request, head,
  channel), q~_t = rho q~_{t-1} + sqrt(1 - rho^2) eps_t, rounded to bf16 (rho
  may differ per head), or a forced-hit stream (per (request, KV group,
  step) Bernoulli), or a stream that recurs at a fixed gap (q~_t =
  q~_{t-gap} + noise), or a topic-revisiting stream (each (request, head)
  walks a Markov chain over a few prototype directions; q~_t is the current
  prototype plus noise), whose ``lead`` earliest steps can serve as prefill
  queries (``prefill_queries``);
* post-RoPE queries q_t = RoPE(q~_t) at the new token's index, in fp64,
  rounded to bf16;
* new tokens' K (RoPE'd) and V per step, i.i.d. N(0, 1);
* page tables: one random permutation of the page pool, cut per request.

RoPE here is the caller's (the model's) rotary embedding: rotate-half pairs
(i, i + d/2), angle = position * base^(-2i/d), no frequency scaling.  The
attention library never applies RoPE; it takes both queries.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional, Sequence

import torch

PAGE = 16

# stream tags for seed derivation
_T_K, _T_V, _T_Q0, _T_EPS, _T_KNEW, _T_VNEW, _T_RHO, _T_PAGES, _T_SCALE, _T_FORCE = range(10)


def derive_seed(base: int, *parts: int) -> int:
    """Mix integers into a 63-bit seed (splitmix64 finaliser over the parts)."""
    x = base & 0xFFFFFFFFFFFFFFFF
    for p in parts:
        x = (x + 0x9E3779B97F4A7C15 + (p & 0xFFFFFFFFFFFFFFFF)) & 0xFFFFFFFFFFFFFFFF
        z = x
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & 0xFFFFFFFFFFFFFFFF
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & 0xFFFFFFFFFFFFFFFF
        x = z ^ (z >> 31)
    return x & 0x7FFFFFFFFFFFFFFF


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def randn(shape, seed: int, device="cpu") -> torch.Tensor:
    """N(0, 1) in fp64 from a dedicated seeded stream."""
    return torch.randn(shape, generator=_gen(seed, device), device=device, dtype=torch.float64)


def rope(x: torch.Tensor, positions: torch.Tensor, base: float) -> torch.Tensor:
    """Rotate-half RoPE in fp64.  x [..., T, n, d] (or [T, n, d]) with the
    token axis at -3; positions [T] (0-based token indices)."""
    d = x.shape[-1]
    half = d // 2
    i = torch.arange(half, device=x.device, dtype=torch.float64)
    inv_freq = base ** (-2.0 * i / d)
    ang = positions.to(device=x.device, dtype=torch.float64)[:, None] * inv_freq[None, :]   # [T, half]
    cos = torch.cos(ang)[:, None, :]
    sin = torch.sin(ang)[:, None, :]
    x = x.to(torch.float64)
    x1, x2 = x[..., :half], x[..., half:]
    return torch.cat([x1 * cos - x2 * sin, x2 * cos + x1 * sin], dim=-1)


def to_bf16(x: torch.Tensor) -> torch.Tensor:
    """Round to bf16 (round-to-nearest-even)."""
    return x.to(torch.bfloat16)


def bf16_bits(x: torch.Tensor):
    """bf16 tensor -> numpy uint16 bit patterns (on the host)."""
    return x.detach().to("cpu").contiguous().view(torch.int16).numpy().view("uint16")


@dataclasses.dataclass
class DecodeConfig:
    """One synthetic decode workload (one attention layer unless ``layers`` > 1)."""
    name: str
    batch: int
    heads: int
    kv_heads: int
    head_dim: int
    context: int               # prefill tokens per request
    steps: int                 # decode steps
    ring_len: int
    band_r: int
    tau: float
    rho: float = 0.95          # AR(1) coefficient (ignored when rho_range or forced_hit_rate is set)
    rho_range: Optional[Sequence[float]] = None   # per-head rho ~ U[lo, hi]
    forced_hit_rate: Optional[float] = None        # per (request, kv group, step) Bernoulli
    paged: bool = True
    gap: Optional[int] = None          # q~_t = q~_{t-gap} + gap_noise eps (fresh N(0,1) before)
    gap_noise: float = 0.1
    topics: Optional[int] = None       # prototypes of the topic-revisiting stream
    topic_stay: float = 0.9            # probability of keeping the current prototype
    topic_noise: float = 0.1
    lead: int = 0                      # query-process steps before decode step 0 (prefill queries)
    layers: int = 1
    channel_scale_range: Optional[Sequence[float]] = None   # log-uniform per (layer, kv-head, channel)
    rope_base: float = 500000.0
    seed: int = 20260331

    @property
    def group(self) -> int:
        return self.heads // self.kv_heads

    @property
    def max_ctx(self) -> int:
        return self.context + self.steps

    def kv_bytes_full_per_step(self, step: int) -> int:
        """Bytes of K+V that full attention reads at decode step ``step``."""
        m = self.context + step + 1
        return self.batch * self.kv_heads * m * self.head_dim * 2 * 2


# Named workloads (sizes in the name).  Seeds follow base 20260331 + index.
def llama_gqa_4k_b1_contig(steps=64) -> DecodeConfig:
    """One Llama-3.1-8B-shaped layer (32 q / 8 kv heads, d 128), 4096-token
    context, 1 request, contiguous KV, rho 0.95, ring 16, r 64, tau 0.3."""
    return DecodeConfig("gqa32x8_d128_ctx4096_b1_contig_rho0.95", 1, 32, 8, 128, 4096, steps, 16, 64, 0.3,
                        rho=0.95, paged=False, seed=20260331 + 1)


def llama_gqa_32k_b8_paged(steps=256) -> DecodeConfig:
    """8 requests x 32768 tokens, paged (16) with a random page permutation."""
    return DecodeConfig("gqa32x8_d128_ctx32768_b8_paged16_rho0.95", 8, 32, 8, 128, 32768, steps, 16, 64, 0.3,
                        rho=0.95, paged=True, seed=20260331 + 2)


def llama_gqa_128k_b1_hetero(steps=512, band_r=64) -> DecodeConfig:
    """1 request x 131072 tokens, paged (16), per-head rho ~ U[0.5, 0.99],
    ring 32, r in {32, 64, 128}."""
    return DecodeConfig(f"gqa32x8_d128_ctx131072_b1_paged16_rhoU0.5-0.99_ring32_r{band_r}", 1, 32, 8, 128,
                        131072, steps, 32, band_r, 0.3, rho_range=(0.5, 0.99), paged=True, seed=20260331 + 3)


def qwen_moe_stack_120k_b4(steps=128, tau=0.3, layers=48) -> DecodeConfig:
    """Qwen3-30B-A3B-shaped attention stack: 48 layers x (32 q / 4 kv heads),
    4 requests x 122880 tokens, per-channel scale log-uniform in [0.5, 2]."""
    return DecodeConfig(f"qwen3moe_{layers}L_gqa32x4_d128_ctx122880_b4_paged16_rho0.9_tau{tau}", 4, 32, 4, 128,
                        122880, steps, 16, 64, tau, rho=0.9, paged=True, layers=layers,
                        channel_scale_range=(0.5, 2.0), seed=20260331 + 4)


def sweep_point(context, batch, hit_rate, kv_heads, steps=64) -> DecodeConfig:
    """One point of the context x batch x forced-hit-rate sweep (MQA kv_heads=1
    or GQA kv_heads=8, 32 q heads, d 128, paged 16, ring 16, r 64)."""
    kind = "mqa" if kv_heads == 1 else "gqa"
    return DecodeConfig(f"sweep_{kind}32x{kv_heads}_ctx{context}_b{batch}_hit{int(round(hit_rate * 100))}",
                        batch, 32, kv_heads, 128, context, steps, 16, 64, 0.3,
                        forced_hit_rate=hit_rate, paged=True, seed=20260331 + 5)


# ---------------------------------------------------------------------------
# generators
# ---------------------------------------------------------------------------
def channel_scales(cfg: DecodeConfig, layer: int, device="cpu") -> Optional[torch.Tensor]:
    """Per (kv-head, channel) scale for K and V, log-uniform in the range."""
    if cfg.channel_scale_range is None:
        return None
    lo, hi = cfg.channel_scale_range
    g = _gen(derive_seed(cfg.seed, layer, _T_SCALE), device)
    u = torch.rand((2, cfg.kv_heads, cfg.head_dim), generator=g, device=device, dtype=torch.float64)
    return torch.exp(math.log(lo) + u * (math.log(hi) - math.log(lo)))


def prefill_kv(cfg: DecodeConfig, layer: int = 0, device="cpu", chunk: int = 8192):
    """Prefill K (post-RoPE) and V, bf16 [B, context, Hkv, d]."""
    B, T, n, d = cfg.batch, cfg.context, cfg.kv_heads, cfg.head_dim
    K = torch.empty((B, T, n, d), dtype=torch.bfloat16, device=device)
    V = torch.empty((B, T, n, d), dtype=torch.bfloat16, device=device)
    sc = channel_scales(cfg, layer, device)
    for b in range(B):
        for c0 in range(0, T, chunk):
            c1 = min(T, c0 + chunk)
            k = randn((c1 - c0, n, d), derive_seed(cfg.seed, layer, _T_K, b, c0), device)
            v = randn((c1 - c0, n, d), derive_seed(cfg.seed, layer, _T_V, b, c0), device)
            if sc is not None:
                k = k * sc[0]
                v = v * sc[1]
            pos = torch.arange(c0, c1, device=device)
            K[b, c0:c1] = to_bf16(rope(k, pos, cfg.rope_base))
            V[b, c0:c1] = to_bf16(v)
    return K, V


def head_rhos(cfg: DecodeConfig, layer: int = 0) -> torch.Tensor:
    """AR(1) coefficient per head [H] (fp64, host)."""
    if cfg.rho_range is None:
        return torch.full((cfg.heads,), float(cfg.rho), dtype=torch.float64)
    lo, hi = cfg.rho_range
    g = _gen(derive_seed(cfg.seed, layer, _T_RHO), "cpu")
    return lo + (hi - lo) * torch.rand((cfg.heads,), generator=g, dtype=torch.float64)


def _query_process(cfg: DecodeConfig, layer: int, device, total: int):
    """Pre-RoPE queries (fp64 [total, B, H, d]) of the gap or topic stream,
    step 0 being the first of the ``lead`` prefill steps."""
    B, H, d = cfg.batch, cfg.heads, cfg.head_dim
    out = torch.empty((total, B, H, d), dtype=torch.float64, device=device)
    if cfg.gap is not None:
        for t in range(total):
            eps = randn((B, H, d), derive_seed(cfg.seed, layer, _T_EPS, t), device)
            out[t] = eps if t < cfg.gap else out[t - cfg.gap] + cfg.gap_noise * eps
        return out
    proto = randn((cfg.topics, B, H, d), derive_seed(cfg.seed, layer, _T_Q0), device)
    g = _gen(derive_seed(cfg.seed, layer, _T_FORCE), device)
    z = torch.randint(0, cfg.topics, (B, H), generator=g, device=device)
    bh = torch.arange(B * H, device=device)
    for t in range(total):
        if t > 0:
            move = torch.rand((B, H), generator=g, device=device, dtype=torch.float64) >= cfg.topic_stay
            z = torch.where(move, torch.randint(0, cfg.topics, (B, H), generator=g, device=device), z)
        base = proto.permute(1, 2, 0, 3).reshape(B * H, cfg.topics, d)[bh, z.reshape(-1)].reshape(B, H, d)
        out[t] = base + cfg.topic_noise * randn((B, H, d), derive_seed(cfg.seed, layer, _T_EPS, t), device)
    return out


def prefill_queries(cfg: DecodeConfig, layer: int = 0, device="cpu"):
    """The ``lead`` queries of the gap / topic stream that precede decode
    step 0, as prefill queries of tokens context - lead .. context - 1:
    q_pre, q_post bf16 [lead, B, H, d]."""
    n, B, H, d = cfg.lead, cfg.batch, cfg.heads, cfg.head_dim
    q = _query_process(cfg, layer, device, n)
    q_pre = to_bf16(q)
    pos = torch.arange(cfg.context - n, cfg.context, device=device)
    q_post = to_bf16(rope(q_pre.reshape(n, B * H, d), pos, cfg.rope_base).reshape(n, B, H, d))
    return q_pre, q_post


def decode_inputs(cfg: DecodeConfig, layer: int = 0, device="cpu", steps: Optional[int] = None,
                  first_step: int = 0):
    """Per-step inputs for decode steps [first_step, first_step + steps).

    Returns a dict of bf16 tensors: q_pre, q_post [S, B, H, d]; k_new, v_new
    [S, B, Hkv, d]; plus ``forced`` [S, B, Hkv] (bool, forced-hit draws) when
    the workload forces hits.  The query process is generated from step 0 so
    any window is consistent with the full sequence.
    """
    S = cfg.steps if steps is None else steps
    B, H, n, d = cfg.batch, cfg.heads, cfg.kv_heads, cfg.head_dim
    total = first_step + S
    sc = channel_scales(cfg, layer, device)
    q_pre = torch.empty((S, B, H, d), dtype=torch.bfloat16, device=device)
    q_post = torch.empty_like(q_pre)
    k_new = torch.empty((S, B, n, d), dtype=torch.bfloat16, device=device)
    v_new = torch.empty_like(k_new)
    forced = torch.zeros((S, B, n), dtype=torch.bool, device=device) if cfg.forced_hit_rate is not None else None

    q = randn((B, H, d), derive_seed(cfg.seed, layer, _T_Q0), device)        # latent q~_0
    rho = head_rhos(cfg, layer).to(device)[None, :, None]
    if cfg.forced_hit_rate is not None:
        gf = _gen(derive_seed(cfg.seed, layer, _T_FORCE), device)
    proc = None
    if cfg.gap is not None or cfg.topics is not None:
        proc = _query_process(cfg, layer, device, cfg.lead + total)
    for t in range(total):
        if proc is not None:
            q = proc[cfg.lead + t]
        elif t > 0:
            eps = randn((B, H, d), derive_seed(cfg.seed, layer, _T_EPS, t), device)
            if cfg.forced_hit_rate is None:
                q = rho * q + torch.sqrt(1.0 - rho * rho) * eps
            else:
                hit = torch.rand((B, n), generator=gf, device=device, dtype=torch.float64) < cfg.forced_hit_rate
                hit_h = hit.repeat_interleave(cfg.group, dim=1)[:, :, None]
                q = torch.where(hit_h, q + 0.01 * eps, eps)
        if t < first_step:
            continue
        s = t - first_step
        qb = to_bf16(q)
        pos = torch.full((1,), cfg.context + t, device=device)
        q_pre[s] = qb
        # RoPE over [B, H, d] with one position: view as [1, B*H, d]
        q_post[s] = to_bf16(rope(qb.reshape(1, B * H, d), pos, cfg.rope_base).reshape(B, H, d))
        kn = randn((B, n, d), derive_seed(cfg.seed, layer, _T_KNEW, t), device)
        vn = randn((B, n, d), derive_seed(cfg.seed, layer, _T_VNEW, t), device)
        if sc is not None:
            kn = kn * sc[0]
            vn = vn * sc[1]
        k_new[s] = to_bf16(rope(kn.reshape(1, B * n, d), pos, cfg.rope_base).reshape(B, n, d))
        v_new[s] = to_bf16(vn)
        if forced is not None and t > 0:
            forced[s] = hit
    out = dict(q_pre=q_pre, q_post=q_post, k_new=k_new, v_new=v_new)
    if forced is not None:
        out["forced"] = forced
    return out


def page_tables(batch: int, pages_per_request: int, seed: int, layer: int = 0) -> torch.Tensor:
    """int32 [batch, pages_per_request]: one random permutation of the pool's
    batch * pages_per_request pages, cut into consecutive runs per request."""
    g = _gen(derive_seed(seed, layer, _T_PAGES), "cpu")
    perm = torch.randperm(batch * pages_per_request, generator=g)
    return perm.to(torch.int32).reshape(batch, pages_per_request)
