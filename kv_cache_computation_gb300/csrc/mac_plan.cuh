// The work plan of the attention kernels (the prologue of every attention
// CTA; all CTAs derive the same plan), shared by the mma.sync and the tcgen05
// attention translation units.  Conventions: token index j (0-based) is the
// paper's position j+1; ranges [lo, hi) are half-open over indices.
#pragma once
#include "mac_device.cuh"

namespace macgpu {

namespace {

// ---------------------------------------------------------------------------
// Planning (prologue of every attention CTA; all CTAs derive the same plan).
// Per (request, kv-head) group the streamed span is [lo_g, m), lo_g being the
// smallest band+tail start of the group's heads.  In a MAC step Amend's band
// [m-r, m) is cut off as its own segment, so Complete yields the
// rectification term AS_{m-r+1:m} and the direct form of AS_{1:m-r} as
// by-products: one work item per group, at the head of the list (item g is
// group g's band).  The long segment [lo_g, m-r) (the whole span in a full
// step) is cut into chunks at multiples of C (a multiple of 16: page
// aligned); its items follow the bands, group after group.
//
// Balanced mode (Figure 3(b), "load-balanced planning"): every item costs at
// most C tokens, so the step finishes when the longest item does; the plan
// takes the smallest C for which the long items fit one wave of the
// persistent attention grid (or k waves when there are more long segments
// than CTAs), searched by bisection (aligned chunk counts are not strictly
// monotone in C, so it may settle on a slightly larger C that also fits).  The short band items either come on top -- a CTA that takes
// one starts its long item that much later, which idle CTAs or the page
// pools below absorb -- or are fitted into the wave, which lengthens every
// long item by about nb / (P - nb); band_wave_fit picks the cheaper.
// Longer spans thereby get proportionally more CTAs.  Equal mode gives every
// group the same number of items whatever its span (unbalanced baseline).
// ---------------------------------------------------------------------------
struct PlanShared {
    int lo[kPlanCache];
    int hi[kPlanCache];
    int off[kPlanCache + 1];
    int C;
    int total;
    long long T, Tf;
    ChunkDiv cd;            // chunk_div(C) (balanced mode)
};

// End of the long segment [lo, sp); the band is [sp, hi) (empty in a full step).
__device__ __forceinline__ int plan_split(const Layout &L, const StepArgs &a, int lo, int hi)
{
    return a.full_mode ? hi : max(lo, hi - L.band_r);
}

// Band items at the head of the work list: one per group in a MAC step.
__device__ __forceinline__ int plan_bands(const StepArgs &a, int nbg) { return a.full_mode ? 0 : nbg; }

// Whether the nb band items share one wave of P CTAs with the long items
// (TL long-segment tokens in all): fitting stretches a long item (about
// TL / P tokens) by nb / (P - nb); on top, a CTA with two items runs about
// band_r + 32 tokens longer (the band and an item's fixed cost).
__device__ __forceinline__ bool band_wave_fit(int nb, long long TL, int P, int band_r)
{
    return nb > 0 && 2 * nb < P && (long long)nb * TL <= (long long)(band_r + 32) * P * (P - nb);
}

__device__ __forceinline__ int plan_chunk(const Layout &L, const StepArgs &a, const PlanShared &ps, int nbg, int lo,
                                          int hi)
{
    if (a.plan_mode == 0) return ps.C;
    const int splits = a.plan_ctas / nbg > 1 ? a.plan_ctas / nbg : 1;
    return max(kMinChunk, round_up16(((long long)(hi - lo) + splits - 1) / splits));
}

// Up to 32 groups: one warp plans alone -- lane g holds group g; up to 8
// groups, 32 chunk candidates are counted at once (lane k counts candidate
// k), a ballot picks the smallest that fits; above that the chunk is found by
// bisection (each probe one warp sum of the groups' chunk counts); a shuffle
// scan gives the offsets.
__device__ bool cta_plan_small(const Layout &L, const StepArgs &a, PlanShared &ps)
{
    const int nbg = a.batch * L.Hkv;
    const int lane = threadIdx.x & 31;
    int lo = 0, hi = 0, sp = 0;
    if (lane < nbg) {
        hi = __ldcg(&L.m_cur[lane / L.Hkv]);
        lo = __ldcg(&L.grp_lo[lane]);
        sp = plan_split(L, a, lo, hi);
    }
    long long T = lane < nbg ? hi - lo : 0, Tf = lane < nbg ? hi : 0, TL = lane < nbg ? sp - lo : 0;
    int nseg = lane < nbg ? (sp > lo) : 0;   // long segments
    for (int o = 16; o; o >>= 1) {
        T += __shfl_xor_sync(0xffffffffu, T, o);
        Tf += __shfl_xor_sync(0xffffffffu, Tf, o);
        TL += __shfl_xor_sync(0xffffffffu, TL, o);
    }
    nseg = warp_sum_int(nseg);
    const int nb = plan_bands(a, nbg);
    if (lane < nbg) {
        ps.lo[lane] = lo;
        ps.hi[lane] = hi;
    }
    __syncwarp();
    int C = kMinChunk;
    ChunkDiv RC = {0u, 0};
    if (a.plan_mode == 0) {
        const int P = a.plan_ctas;
        int Q = (4 * nseg <= P) ? P : P * (1 + (2 * nseg + P - 1) / P);
        if (Q == P && band_wave_fit(nb, TL, P, L.band_r)) Q = P - nb;
        if (Q > L.item_cap - nb) Q = L.item_cap - nb;
        // A fitting chunk is at least T / Q (count(C) >= T / C), and
        // T / (Q - 2 nseg) fits (count(C) < T / C + 2 nseg).  Float quotients
        // (relative error < 2^-22) widened by 2^-20 bracket both.
        const float Tq = (float)TL;
        long long c_lo = (long long)(Tq / (float)Q * (1.f - 0x1p-20f)) / 16 * 16;
        long long c_hi = Q > 2 * nseg ? round_up16((long long)(Tq / (float)(Q - 2 * nseg) * (1.f + 0x1p-20f)) + 16)
                                      : (1ll << 30);
        if (c_lo < kMinChunk) c_lo = kMinChunk;
        if (c_hi < c_lo) c_hi = c_lo;
        if (nbg <= 8) {
            // few groups: lane k counts candidate c_lo + 16 * stride * k
            // (k = 0..31, the last one c_hi) over every group, a ballot picks
            // the smallest that fits
            for (;;) {
                const long long span16 = (c_hi - c_lo) / 16;
                const long long stride = span16 <= 31 ? 1 : (span16 + 30) / 31;
                long long cand = c_lo + 16 * stride * lane;
                if (cand > c_hi) cand = c_hi;
                const ChunkDiv R = chunk_div((int)cand);
                int cnt = 0;
#pragma unroll 4
                for (int g = 0; g < nbg; g++) {
                    const int glo = ps.lo[g], ghi = ps.hi[g], gsp = plan_split(L, a, glo, ghi);
                    cnt += n_chunks_c(glo, gsp, R);
                }
                const unsigned fit = __ballot_sync(0xffffffffu, cnt <= Q);
                const int k = fit ? __ffs(fit) - 1 : 31;
                const long long ck = __shfl_sync(0xffffffffu, cand, k);
                if (stride == 1 || k == 0) {
                    c_hi = ck;
                    RC.m = __shfl_sync(0xffffffffu, R.m, k);
                    RC.k = __shfl_sync(0xffffffffu, R.k, k);
                    break;
                }
                c_hi = ck;   // refine between the previous candidate and this one
                c_lo = __shfl_sync(0xffffffffu, cand, k - 1) + 16;
            }
            C = (int)c_hi;
        } else {
            // binary search over the multiples of 16 in [c_lo, c_hi], lane g
            // counting group g's chunks (one warp sum per probe): c_hi fits, and
            // the search only ever moves its upper end to a chunk that fits
            int lo16 = (int)(c_lo >> 4), hi16 = (int)(c_hi >> 4);
            while (lo16 < hi16) {
                const int mid = (lo16 + hi16) >> 1;
                const ChunkDiv R = chunk_div(mid << 4);
                const int cnt = warp_sum_int(lane < nbg ? n_chunks_c(lo, sp, R) : 0);
                if (cnt <= Q) hi16 = mid;
                else lo16 = mid + 1;
            }
            C = hi16 << 4;
            RC = chunk_div(C);
        }
    }
    // per-group counts and offsets
    int cnt = 0;
    if (lane < nbg) {
        if (a.plan_mode == 0) {
            cnt = n_chunks_c(lo, sp, RC);
        } else {
            cnt = n_chunks(lo, sp, plan_chunk(L, a, ps, nbg, lo, sp));
        }
    }
    int x = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    const int total = nb + __shfl_sync(0xffffffffu, x, 31);
    if (lane < nbg) ps.off[lane] = nb + x - cnt;
    if (lane == 0) {
        ps.off[nbg] = total;
        ps.total = total < L.item_cap ? total : L.item_cap;
        ps.C = C;
        ps.cd = RC;
        ps.T = T;
        ps.Tf = Tf;
    }
    return true;
}

__device__ void cta_plan(const Layout &L, const StepArgs &a, PlanShared &ps)
{
    const int nbg = a.batch * L.Hkv;
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    if (nbg <= 32) {
        if (w == 0) cta_plan_small(L, a, ps);
        __syncthreads();
        return;
    }
    for (int bg = threadIdx.x; bg < nbg; bg += blockDim.x) {
        ps.hi[bg] = __ldcg(&L.m_cur[bg / L.Hkv]);   // m: the length after this step's append
        ps.lo[bg] = __ldcg(&L.grp_lo[bg]);
    }
    __syncthreads();
    const int nb = plan_bands(a, nbg);
    if (w == 0) {
        long long T = 0, Tf = 0, TL = 0;
        int nseg = 0;   // long segments
        for (int bg = lane; bg < nbg; bg += 32) {
            const int lo = ps.lo[bg], hi = ps.hi[bg], sp = plan_split(L, a, lo, hi);
            T += hi - lo;
            Tf += hi;
            TL += sp - lo;
            nseg += sp > lo;
        }
        for (int o = 16; o; o >>= 1) {
            T += __shfl_xor_sync(0xffffffffu, T, o);
            Tf += __shfl_xor_sync(0xffffffffu, Tf, o);
            TL += __shfl_xor_sync(0xffffffffu, TL, o);
        }
        nseg = warp_sum_int(nseg);
        int C = kMinChunk;
        ChunkDiv RC = chunk_div(kMinChunk);
        if (a.plan_mode == 0) {
            auto count = [&](ChunkDiv R) {
                int c = 0;
                for (int bg = lane; bg < nbg; bg += 32) {
                    const int lo = ps.lo[bg], hi = ps.hi[bg], sp = plan_split(L, a, lo, hi);
                    c += n_chunks_c(lo, sp, R);
                }
                return warp_sum_int(c);
            };
            const long long P = a.plan_ctas;
            long long Q = (4ll * nseg <= P) ? P : P * (1 + (2ll * nseg + P - 1) / P);
            if (Q == P && band_wave_fit(nb, TL, (int)P, L.band_r)) Q = P - nb;
            if (Q > L.item_cap - nb) Q = L.item_cap - nb;
            // count(C) < TL/C + 2 nseg, so C >= TL / (Q - 2 nseg) always fits Q items
            long long c_lo = round_up16((TL + Q - 1) / Q);
            long long c_hi = Q > 2ll * nseg ? round_up16((TL + (Q - 2ll * nseg) - 1) / (Q - 2ll * nseg)) : (1ll << 30);
            if (c_lo < kMinChunk) c_lo = kMinChunk;
            if (c_hi < c_lo) c_hi = c_lo;
            // 32 candidates c_lo + 16 stride k (the last one c_hi, which fits):
            // lane k forms candidate k's reciprocal (one division for all),
            // a binary search over k counts the groups once per probe, and
            // a second round refines between neighbours when stride > 1.
            for (;;) {
                const long long span16 = (c_hi - c_lo) / 16;
                const long long stride = span16 <= 31 ? 1 : (span16 + 30) / 31;
                long long cand = c_lo + 16 * stride * lane;
                if (cand > c_hi) cand = c_hi;
                const ChunkDiv R = chunk_div((int)cand);
                int k0 = 0, k1 = (int)min(31ll, (span16 + stride - 1) / stride);   // the last distinct candidate
                while (k0 < k1) {
                    const int km = (k0 + k1) >> 1;
                    const ChunkDiv Rm = {__shfl_sync(0xffffffffu, R.m, km), __shfl_sync(0xffffffffu, R.k, km)};
                    if (count(Rm) <= Q) k1 = km;
                    else k0 = km + 1;
                }
                const long long ck = __shfl_sync(0xffffffffu, cand, k0);
                const long long cprev = __shfl_sync(0xffffffffu, cand, k0 > 0 ? k0 - 1 : 0);
                const ChunkDiv Rk = {__shfl_sync(0xffffffffu, R.m, k0), __shfl_sync(0xffffffffu, R.k, k0)};
                c_hi = ck;
                if (stride == 1 || k0 == 0) {
                    RC = Rk;
                    break;
                }
                c_lo = cprev + 16;
            }
            C = (int)c_hi;
        }
        if (lane == 0) {
            ps.C = C;
            ps.cd = RC;
            ps.T = T;
            ps.Tf = Tf;
        }
    }
    __syncthreads();
    // item offsets per group (block scan in rounds keeps the groups in order)
    int base = 0;
    for (int r0 = 0; r0 < nbg; r0 += blockDim.x) {
        const int bg = r0 + threadIdx.x;
        int cnt = 0;
        if (bg < nbg) {
            const int lo = ps.lo[bg], hi = ps.hi[bg], sp = plan_split(L, a, lo, hi);
            if (a.plan_mode == 0) {
                cnt = n_chunks_c(lo, sp, ps.cd);
            } else {
                cnt = n_chunks(lo, sp, plan_chunk(L, a, ps, nbg, lo, sp));
            }
        }
        int tot;
        const int off = base + block_exclusive_scan(cnt, &tot);
        if (bg < nbg) ps.off[bg] = nb + off;
        base += tot;
    }
    if (threadIdx.x == 0) {
        ps.off[nbg] = nb + base;
        ps.total = nb + base < L.item_cap ? nb + base : L.item_cap;
    }
    __syncthreads();
}

// Work item `it` of the plan: {group, lo, hi, segment}.  Items 0 .. nb - 1
// are the groups' bands (segment 1), then come the long segments' chunks
// (segment 0) group after group.
__device__ int4 plan_item(const Layout &L, const StepArgs &a, const PlanShared &ps, int nbg, int it)
{
    if (it < plan_bands(a, nbg)) {
        const int lo = ps.lo[it], hi = ps.hi[it];
        return make_int4(it, plan_split(L, a, lo, hi), hi, 1);
    }
    int g0 = 0, g1 = nbg - 1;   // the last group whose first long item is <= it
    while (g0 < g1) {
        const int mid = (g0 + g1 + 1) >> 1;
        if (ps.off[mid] <= it) g0 = mid;
        else g1 = mid - 1;
    }
    const int bg = g0, k = it - ps.off[bg];
    const int lo = ps.lo[bg], hi = ps.hi[bg], sp = plan_split(L, a, lo, hi);
    const int C = plan_chunk(L, a, ps, nbg, lo, sp);
    const ChunkDiv R = a.plan_mode == 0 ? ps.cd : chunk_div(C);
    const int c = div_c(lo, R) + k;
    return make_int4(bg, max(lo, c * C), min(sp, (c + 1) * C), 0);
}


}  // namespace

}  // namespace macgpu
