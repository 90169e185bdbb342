// sm_103a kernels of the MAC-Attention decode step.
//
// One decode step is four launches:
//   match_plan  (critical path) KV append of the new token; Match of each
//               query head's pre-RoPE query against its ring (Figure 2(a) of
//               the MAC-Attention paper); per-head band+tail spans; and, in
//               the last block, the span-proportional work list (Figure 3(b),
//               "load-balanced planning").
//   attention   (critical path) persistent split-KV attention over the work
//               list: each item streams 16-token KV pages of one KV head
//               through a cp.async shared-memory pipeline and evaluates all
//               query heads of the group with bf16 tensor-core tiles,
//               keeping fp32 online-softmax partials (Figure 2(b), Complete).
//   combine     (critical path) log-domain merge of the partials and, on a
//               hit, of the reused AS_{1:p-r} from the ring (Figure 2(b)).
//   amend       (side stream) recompute AS_{m-r+1:m}, log-domain removal to
//               AS_{1:m-r}, ring insert (Figure 2(c)).
//
// Conventions: token index j (0-based) is the paper's position j+1; ranges
// [lo, hi) are half-open over indices.  Scores are kept in log2 units
// (scaled by sm_scale * log2 e) inside the kernels; summaries that leave the
// kernels (ring, lse_out) use natural-log units.
#include "mac_internal.cuh"

#include <math_constants.h>

namespace macgpu {

namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ float4 load_bf16x4(const __nv_bfloat16 *p)
{
    uint2 u = *reinterpret_cast<const uint2 *>(p);
    __nv_bfloat162 a = *reinterpret_cast<__nv_bfloat162 *>(&u.x);
    __nv_bfloat162 b = *reinterpret_cast<__nv_bfloat162 *>(&u.y);
    float2 fa = __bfloat1622float2(a), fb = __bfloat1622float2(b);
    return make_float4(fa.x, fa.y, fb.x, fb.y);
}

// Element offset of the 16-token block `pg` of (request b, kv-head g).  Both
// layouts keep the block's 16 x 128 bf16 keys (and values) contiguous (4 KB).
__device__ __forceinline__ size_t kv_block(const Layout &L, int b, int g, int pg, bool &ok)
{
    if (pg < 0 || pg >= L.pages_per_req) {
        ok = false;
        return 0;
    }
    if (L.paged) {
        int phys = L.page_table[(size_t)b * L.pages_per_req + pg];
        if ((unsigned)phys >= (unsigned)L.num_pages) {
            ok = false;
            return 0;
        }
        return ((size_t)phys * L.Hkv + g) * (kPage * kD);
    }
    return (((size_t)b * L.Hkv + g) * L.ctx_stride + (size_t)pg * kPage) * kD;
}

// Programmatic dependent launch: a dependent grid may start while its
// predecessor in the stream still runs; it waits here until the predecessor
// has completed and its memory is visible.  Both are no-ops in a plain launch.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory"); }

__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(dst), "l"(src) : "memory");
}

// Bulk prefetch of `bytes` (multiple of 16, 16-byte aligned) into L2.
__device__ __forceinline__ void prefetch_l2_bulk(const void *src, uint32_t bytes)
{
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;\n" ::"l"(src), "r"(bytes) : "memory");
}

__device__ __forceinline__ void cp_async_commit()
{
    asm volatile("cp.async.commit_group;\n" ::: "memory");
}

template <int N>
__device__ __forceinline__ void cp_async_wait()
{
    asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

__device__ __forceinline__ void named_bar(int id, int nthreads)
{
    asm volatile("bar.sync %0, %1;\n" ::"r"(id), "r"(nthreads) : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t &a0, uint32_t &a1, uint32_t &a2, uint32_t &a3, uint32_t addr)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(a0), "=r"(a1), "=r"(a2), "=r"(a3)
                 : "r"(addr)
                 : "memory");
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t &a0, uint32_t &a1, uint32_t &a2, uint32_t &a3, uint32_t addr)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(a0), "=r"(a1), "=r"(a2), "=r"(a3)
                 : "r"(addr)
                 : "memory");
}

__device__ __forceinline__ uint32_t movmatrix_t(uint32_t x)
{
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;\n" : "=r"(y) : "r"(x));
    return y;
}

// D += A(16x16 bf16, row) * B(16x8 bf16, col), fp32 accumulate
__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t bf16x2_bits(__nv_bfloat162 v)
{
    return *reinterpret_cast<uint32_t *>(&v);
}

// log(1 - e^x), x <= 0: Maechler (2012), "Accurately computing
// log(1 - exp(-|a|))" -- log(-expm1(x)) above -ln 2, log1p(-exp(x)) below.
__device__ __forceinline__ float log1mexp_f(float x)
{
    return x > -kLn2 ? logf(-expm1f(x)) : log1pf(-expf(x));
}

// number of chunks of [a, b) when cut at multiples of C
__device__ __forceinline__ int n_chunks(int a, int b, int C)
{
    return b > a ? (b - 1) / C - a / C + 1 : 0;
}

// Division by a chunk size C = 16 c (4 <= c <= 2^26) shared by many
// dividends 0 <= x < 2^30, as one 32 x 32 -> 64-bit multiply: with
// l = ceil(log2 c), k = 26 + l and m = ceil(2^k / c) (below 2^28),
// floor((x >> 4) m / 2^k) = floor((x >> 4) / c) = floor(x / C), because
// (x >> 4) < 2^26 keeps the excess of the rounded-up m below 2^-l <= 1/c while
// the fractional part of (x >> 4) / c is at most 1 - 1/c (division by
// invariant integers using multiplication, Granlund and Montgomery 1994).
struct ChunkDiv {
    unsigned m;
    int k;
};

__device__ __forceinline__ ChunkDiv chunk_div(int C)
{
    const unsigned c = (unsigned)C >> 4;
    const int k = 26 + (32 - __clz(c - 1));
    return {(unsigned)(((1ull << k) + c - 1) / c), k};
}

__device__ __forceinline__ int div_c(int x, ChunkDiv d)
{
    return (int)(((unsigned long long)((unsigned)x >> 4) * d.m) >> d.k);
}

// Number of C-aligned chunks [c C, (c + 1) C) that meet [a, b).
__device__ __forceinline__ int n_chunks_c(int a, int b, ChunkDiv d)
{
    return b > a ? div_c(b - 1, d) - div_c(a, d) + 1 : 0;
}

// x rounded up to a multiple of 16, clamped to 2^30 (the longest request)
__device__ __forceinline__ int round_up16(long long x)
{
    const long long r = (x + 15) / 16 * 16;
    return (int)(r < (1ll << 30) ? r : (1ll << 30));
}

// Block-wide exclusive scan of one int per thread (blockDim a multiple of 32,
// up to 1024).  Returns the exclusive prefix; *total gets the sum.
__device__ int block_exclusive_scan(int v, int *total)
{
    __shared__ int warp_tot[32];
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = blockDim.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) warp_tot[w] = x;
    __syncthreads();
    if (w == 0) {
        int t = lane < nw ? warp_tot[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int y = __shfl_up_sync(0xffffffffu, t, o);
            if (lane >= o) t += y;
        }
        if (lane < nw) warp_tot[lane] = t;   // inclusive warp prefix
    }
    __syncthreads();
    int before = (w > 0 ? warp_tot[w - 1] : 0) + x - v;
    *total = warp_tot[nw - 1];
    __syncthreads();
    return before;
}

__device__ __forceinline__ int warp_sum_int(int v)
{
#pragma unroll
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ float warp_max(float v)
{
#pragma unroll
    for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// acc += a . b over 8 bf16 pairs (4 words each), in fp32 (comparison build)
__device__ __forceinline__ void dot8_bf16(float &acc, uint4 a, uint4 b)
{
    const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, bw[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
    for (int i = 0; i < 4; i++) {
        acc = fmaf(__uint_as_float(aw[i] << 16), __uint_as_float(bw[i] << 16), acc);
        acc = fmaf(__uint_as_float(aw[i] & 0xffff0000u), __uint_as_float(bw[i] & 0xffff0000u), acc);
    }
}

// ---------------------------------------------------------------------------
// Planning (prologue of every attention CTA; all CTAs derive the same plan).
// Per (request, kv-head) group the streamed span is [lo_g, m), lo_g being the
// smallest band+tail start of the group's heads.  Amend's band [m-r, m) is
// cut off as its own segment, so Complete yields the rectification term
// AS_{m-r+1:m} and the direct form of AS_{1:m-r} as by-products.  Chunks are
// cut at multiples of C (a multiple of 16: page aligned).
//
// Balanced mode (Figure 3(b), "load-balanced planning"): every item costs at
// most C tokens, so the step finishes when the longest item does; the plan
// takes the smallest C for which the items fit one wave of the persistent
// attention grid (or k waves when there are more segments than CTAs).
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

__device__ __forceinline__ int plan_split(const Layout &L, const StepArgs &a, int lo, int hi)
{
    return a.full_mode ? lo : max(lo, hi - L.band_r);
}

__device__ __forceinline__ int plan_chunk(const Layout &L, const StepArgs &a, const PlanShared &ps, int nbg, int lo,
                                          int hi)
{
    if (a.plan_mode == 0) return ps.C;
    const int splits = a.grid_ctas / nbg > 1 ? a.grid_ctas / nbg : 1;
    return max(kMinChunk, round_up16(((long long)(hi - lo) + splits - 1) / splits));
}

// Up to 32 groups: one warp plans alone -- lane g holds group g, 32 chunk
// candidates are counted at once (lane k counts candidate k), a ballot picks
// the smallest that fits, a shuffle scan gives the offsets.
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
    long long T = lane < nbg ? hi - lo : 0, Tf = lane < nbg ? hi : 0;
    int nseg = lane < nbg ? (sp > lo) + (hi > sp) : 0;
    for (int o = 16; o; o >>= 1) {
        T += __shfl_xor_sync(0xffffffffu, T, o);
        Tf += __shfl_xor_sync(0xffffffffu, Tf, o);
    }
    nseg = warp_sum_int(nseg);
    if (lane < nbg) {
        ps.lo[lane] = lo;
        ps.hi[lane] = hi;
    }
    __syncwarp();
    int C = kMinChunk;
    ChunkDiv RC = {0u, 0};
    if (a.plan_mode == 0) {
        const int P = a.grid_ctas;
        int Q = (4 * nseg <= P) ? P : P * (1 + (2 * nseg + P - 1) / P);
        if (Q > L.item_cap) Q = L.item_cap;
        // The smallest fitting chunk is at least T / Q (count(C) >= T / C)
        // and at most T / (Q - 2 nseg) (count(C) < T / C + 2 nseg).  Float
        // quotients (relative error < 2^-22) widened by 2^-20 bracket both.
        const float Tq = (float)T;
        long long c_lo = (long long)(Tq / (float)Q * (1.f - 0x1p-20f)) / 16 * 16;
        long long c_hi = Q > 2 * nseg ? round_up16((long long)(Tq / (float)(Q - 2 * nseg) * (1.f + 0x1p-20f)) + 16)
                                      : (1ll << 30);
        if (c_lo < kMinChunk) c_lo = kMinChunk;
        if (c_hi < c_lo) c_hi = c_lo;
        // candidates c_lo + 16 * stride * k, k = 0..31 (the last one is c_hi)
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
                cnt += n_chunks_c(glo, gsp, R) + n_chunks_c(gsp, ghi, R);
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
    }
    // per-group counts and offsets
    int cnt = 0;
    if (lane < nbg) {
        if (a.plan_mode == 0) {
            cnt = n_chunks_c(lo, sp, RC) + n_chunks_c(sp, hi, RC);
        } else {
            const int Cg = plan_chunk(L, a, ps, nbg, lo, hi);
            cnt = n_chunks(lo, sp, Cg) + n_chunks(sp, hi, Cg);
        }
    }
    int x = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    const int total = __shfl_sync(0xffffffffu, x, 31);
    if (lane < nbg) ps.off[lane] = x - cnt;
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
    if (w == 0) {
        long long T = 0, Tf = 0;
        int nseg = 0;
        for (int bg = lane; bg < nbg; bg += 32) {
            const int lo = ps.lo[bg], hi = ps.hi[bg], sp = plan_split(L, a, lo, hi);
            T += hi - lo;
            Tf += hi;
            nseg += (sp > lo) + (hi > sp);
        }
        for (int o = 16; o; o >>= 1) {
            T += __shfl_xor_sync(0xffffffffu, T, o);
            Tf += __shfl_xor_sync(0xffffffffu, Tf, o);
        }
        nseg = warp_sum_int(nseg);
        int C = kMinChunk;
        ChunkDiv RC = chunk_div(kMinChunk);
        if (a.plan_mode == 0) {
            auto count = [&](ChunkDiv R) {
                int c = 0;
                for (int bg = lane; bg < nbg; bg += 32) {
                    const int lo = ps.lo[bg], hi = ps.hi[bg], sp = plan_split(L, a, lo, hi);
                    c += n_chunks_c(lo, sp, R) + n_chunks_c(sp, hi, R);
                }
                return warp_sum_int(c);
            };
            const long long P = a.grid_ctas;
            long long Q = (4ll * nseg <= P) ? P : P * (1 + (2ll * nseg + P - 1) / P);
            if (Q > L.item_cap) Q = L.item_cap;
            // count(C) < T/C + 2 nseg, so C >= T / (Q - 2 nseg) always fits Q items
            long long c_lo = round_up16((T + Q - 1) / Q);
            long long c_hi = Q > 2ll * nseg ? round_up16((T + (Q - 2ll * nseg) - 1) / (Q - 2ll * nseg)) : (1ll << 30);
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
                cnt = n_chunks_c(lo, sp, ps.cd) + n_chunks_c(sp, hi, ps.cd);
            } else {
                const int C = plan_chunk(L, a, ps, nbg, lo, hi);
                cnt = n_chunks(lo, sp, C) + n_chunks(sp, hi, C);
            }
        }
        int tot;
        const int off = base + block_exclusive_scan(cnt, &tot);
        if (bg < nbg) ps.off[bg] = off;
        base += tot;
    }
    if (threadIdx.x == 0) {
        ps.off[nbg] = base;
        ps.total = base < L.item_cap ? base : L.item_cap;
    }
    __syncthreads();
}

// Work item `it` of the plan: {group, lo, hi, segment}.
__device__ int4 plan_item(const Layout &L, const StepArgs &a, const PlanShared &ps, int nbg, int it)
{
    int g0 = 0, g1 = nbg - 1;   // the last group whose first item is <= it
    while (g0 < g1) {
        const int mid = (g0 + g1 + 1) >> 1;
        if (ps.off[mid] <= it) g0 = mid;
        else g1 = mid - 1;
    }
    const int bg = g0, k = it - ps.off[bg];
    const int lo = ps.lo[bg], hi = ps.hi[bg], sp = plan_split(L, a, lo, hi);
    const int C = plan_chunk(L, a, ps, nbg, lo, hi);
    const ChunkDiv R = a.plan_mode == 0 ? ps.cd : chunk_div(C);
    const int nA = n_chunks_c(lo, sp, R);
    if (k < nA) {
        const int c = div_c(lo, R) + k;
        return make_int4(bg, max(lo, c * C), min(sp, (c + 1) * C), 0);
    }
    const int c = div_c(sp, R) + (k - nA);
    return make_int4(bg, max(sp, c * C), min(hi, (c + 1) * C), 1);
}

// ---------------------------------------------------------------------------
// match_plan: grid (lo_parts, Hkv, batch); block = part `part` of group g,
// nw = ceil(G / lo_parts) warps, warp w = query head g G + part nw + w.
// Leaves per group the span start lo_g (the parts of a split group take
// their minimum with atomicMin on a word Combine resets every step); the
// attention kernel plans from it.
// Match (Figure 2(a)): one warp per query head reads the head's ring
// queries coalesced, all loads in flight at once, and ends with one entry's
// distance per lane; a warp argmin then picks the nearest entry (ties to the
// larger position).
// ---------------------------------------------------------------------------
// One step of a transposing reduction over the 16 lanes of each half-warp:
// N per-lane values become N / 2, lane bit N / 2 choosing which half a lane
// keeps while it adds its partner's copy of that half.  After the steps for
// N = 16, 8, 4, 2, v[0] of lane l is the half-warp sum of value l & 15.
template <int N>
__device__ __forceinline__ void halve_sum(float (&v)[16], int lane)
{
    constexpr int O = N / 2;
    const bool up = (lane & O) != 0;
#pragma unroll
    for (int k = 0; k < O; k++) {
        const float send = up ? v[k] : v[k + O];
        const float keep = up ? v[k + O] : v[k];
        v[k] = keep + __shfl_xor_sync(0xffffffffu, send, O);
    }
}

// ---------------------------------------------------------------------------
// Wide rings (more than kSmallRing entries): warp w of a (split, head,
// request) block scans entries 32 w .. 32 w + 31 of the split with the
// Match kernel's coalesced layout (load i of lane l = column l & 15 of
// entries 2 i and 2 i + 1, then the transposing half-warp reduction); the
// block's best (distance, age) key goes into dec_key with a 64-bit atomic
// minimum.  Distances are non-negative, so their float bits order as
// unsigned integers; age 0 is the newest entry, so equal distances resolve
// to the most recent position.
// grid (ceil(L / kScanBlock), H, batch), block kScanBlock threads.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kScanBlock, 2) ring_scan_kernel(Layout L, StepArgs a)
{
    __shared__ __align__(16) uint4 sq[16];
    __shared__ unsigned long long s_best;
    pdl_launch_dependents();
    pdl_wait();   // launched early behind the previous step: read nothing before its completion
    const int h = blockIdx.y, b = blockIdx.z;
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const size_t bh = (size_t)b * L.H + h;
    const int e0 = blockIdx.x * kScanBlock + 32 * w;      // this warp's first entry
    const int e = e0 + 2 * (lane & 15) + (lane >> 4);     // the entry whose distance this lane ends with
    uint4 c[16];
    int pe = 0;
    if (e0 < L.ring_len) {
        const int nch = (L.ring_len - e0) * (kD / 8);      // 16-byte chunks of this warp's entries
        const uint4 *blk = reinterpret_cast<const uint4 *>(L.ring_q + (bh * L.ring_len + e0) * kD);
#pragma unroll
        for (int i = 0; i < 16; i++) c[i] = 32 * i + lane < nch ? blk[32 * i + lane] : make_uint4(0u, 0u, 0u, 0u);
        if (e < L.ring_len) pe = L.ring_pos[(size_t)b * L.ring_len + e];
    }
    if (threadIdx.x < 16) sq[threadIdx.x] = reinterpret_cast<const uint4 *>(a.q_pre + bh * kD)[threadIdx.x];
    if (threadIdx.x == 0) s_best = ~0ull;
    const int step = L.step_ctr[b];
    __syncthreads();
    if (e0 < L.ring_len) {
        const uint4 qq = sq[lane & 15];
        const uint32_t qa[4] = {qq.x, qq.y, qq.z, qq.w};
        float v[16];
#pragma unroll
        for (int i = 0; i < 16; i++) {
            const uint32_t ca[4] = {c[i].x, c[i].y, c[i].z, c[i].w};
            float acc = 0.f;
#pragma unroll
            for (int j = 0; j < 4; j++) {
                const float2 qf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&qa[j]));
                const float2 cf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&ca[j]));
                const float d0 = qf.x - cf.x, d1 = qf.y - cf.y;
                acc = fmaf(d0, d0, acc);
                acc = fmaf(d1, d1, acc);
            }
            v[i] = acc;
        }
        halve_sum<16>(v, lane);
        halve_sum<8>(v, lane);
        halve_sum<4>(v, lane);
        halve_sum<2>(v, lane);
        unsigned long long key = ~0ull;
        if (pe > 0) {
            const int age = ((step - 1 - e) % L.ring_len + L.ring_len) % L.ring_len;
            key = ((unsigned long long)__float_as_uint(v[0]) << 32) | (unsigned)age;
        }
#pragma unroll
        for (int o = 16; o; o >>= 1) {
            const unsigned long long ok = __shfl_xor_sync(0xffffffffu, key, o);
            key = ok < key ? ok : key;
        }
        if (lane == 0 && key != ~0ull) atomicMin(&s_best, key);
    }
    __syncthreads();
    if (threadIdx.x == 0 && s_best != ~0ull) atomicMin(&L.dec_key[bh], s_best);
}

// NI: 16-byte loads per lane for the ring's queries, 8 for rings of up to
// 16 entries, 16 for up to 32 (unused by the wide form).  SPLIT: the group
// is spread over L.lo_parts blocks (groups of more than kMatchWarps heads).
template <int MAX_THREADS, bool WIDE, int NI, bool SPLIT>
__global__ void __launch_bounds__(MAX_THREADS) match_plan_kernel(Layout L, StepArgs a)
{
    constexpr int NWM = MAX_THREADS / 32;
    __shared__ __align__(16) uint4 s_q[NWM][16];
    pdl_launch_dependents();
    pdl_wait();   // launched early behind the previous step: read nothing before its completion
    // block = part `part` of group g: its heads part * nw + w, w < nw
    const int part = SPLIT ? blockIdx.x : 0, g = blockIdx.y, b = blockIdx.z;
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = L.G, H = L.H;
    const int nw = blockDim.x >> 5;
    const int gh = part * nw + w;        // head within the group
    const bool active = !SPLIT || gh < G;
    const int h = g * G + gh;
    const size_t bh = (size_t)b * H + h;
    const int kvlen = L.kv_len[b];
    const int m = kvlen + 1;            // 1-based position of the new token (index kvlen)
    const int slot_new = a.full_mode ? 0 : L.step_ctr[b] % L.ring_len;

    // KV append of the new token: warp 0 moves K (lanes 0-15) and V (16-31).
    // Its loads go out first; the store follows once the Match loads are
    // in flight as well.
    const bool appender = w == 0 && part == 0;
    uint4 kv_val = make_uint4(0u, 0u, 0u, 0u);
    size_t kv_off = 0;
    bool kv_ok = true;
    if (appender) {
        kv_val = reinterpret_cast<const uint4 *>((lane < 16 ? a.k_new : a.v_new) + ((size_t)b * L.Hkv + g) * kD)[lane & 15];
        kv_off = kv_block(L, b, g, kvlen >> 4, kv_ok);
    }
    auto append_new = [&]() {
        if (!appender) return;
        if (kv_ok) {
            __nv_bfloat16 *dst = (lane < 16 ? L.k_pool : L.v_pool) + kv_off + (size_t)(kvlen & 15) * kD;
            reinterpret_cast<uint4 *>(dst)[lane & 15] = kv_val;
        } else if (lane == 0) {
            atomicOr(L.err, kErrPage);
        }
    };

    int lo_h = 0x7fffffff;
    if (!active) {
    } else if (!a.full_mode) {
        const int32_t *rpos = L.ring_pos + (size_t)b * L.ring_len;
        const __nv_bfloat16 *rq = L.ring_q + bh * L.ring_len * kD;
        // Every load that depends on nothing is issued first.  The ring's
        // queries are read coalesced: load i of lane l is 16-byte chunk
        // 32 i + l of the head's [L][128] block, i.e. column l & 15 of
        // entry 2 i + (l >> 4), so each lane needs column l & 15 of q~_m
        // alone.  A transposing reduction over each half-warp then leaves
        // lane l the distance of entry e_own.
        const int e_own = 2 * (lane & 15) + (lane >> 4);
        int pe0 = 0;
        uint4 c[NI];
        if (!WIDE) {
            const int nch = L.ring_len * kD / 8;
            const uint4 *blk = reinterpret_cast<const uint4 *>(rq);
#pragma unroll
            for (int i = 0; i < NI; i++) c[i] = 32 * i + lane < nch ? blk[32 * i + lane] : make_uint4(0u, 0u, 0u, 0u);
            if (e_own < L.ring_len) pe0 = rpos[e_own];
        }
        if (lane < 16) {
            s_q[w][lane] = reinterpret_cast<const uint4 *>(a.q_pre + bh * kD)[lane];
        } else {   // keep the post-RoPE query for Amend (the caller may reuse its buffer)
            reinterpret_cast<uint4 *>(L.q_stash + bh * kD)[lane - 16] =
                reinterpret_cast<const uint4 *>(a.q_post + bh * kD)[lane - 16];
        }
        append_new();
        __syncwarp();
        const float4 q4 = load_bf16x4(reinterpret_cast<const __nv_bfloat16 *>(s_q[w]) + 4 * lane);
        const float qn2 = warp_sum(q4.x * q4.x + q4.y * q4.y + q4.z * q4.z + q4.w * q4.w);
        int best = -1, best_pos = 0;
        float bestD = CUDART_INF_F;
        if (WIDE) {   // the scan kernel left the best (distance, age) key
            const unsigned long long key = L.dec_key[bh];
            if (key != ~0ull) {
                bestD = __uint_as_float((unsigned)(key >> 32));
                const int age = (int)(key & 0xffffffffu);
                best = ((L.step_ctr[b] - 1 - age) % L.ring_len + L.ring_len) % L.ring_len;
                best_pos = rpos[best];
            }
            __syncwarp();
            if (lane == 0) L.dec_key[bh] = ~0ull;   // ready for the next step
        } else {
            // D_e = ||q~_m - q~_e||^2 in fp32: this lane's column of every
            // chunk it loaded, then the half-warp sums
            const uint4 qq = s_q[w][lane & 15];
            const uint32_t qa[4] = {qq.x, qq.y, qq.z, qq.w};
            float v[16];
#pragma unroll
            for (int i = NI; i < 16; i++) v[i] = 0.f;   // entries past 2 NI: none
#pragma unroll
            for (int i = 0; i < NI; i++) {
                const uint32_t ca[4] = {c[i].x, c[i].y, c[i].z, c[i].w};
                float acc = 0.f;
#pragma unroll
                for (int j = 0; j < 4; j++) {
                    const float2 qf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&qa[j]));
                    const float2 cf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&ca[j]));
                    const float d0 = qf.x - cf.x, d1 = qf.y - cf.y;
                    acc = fmaf(d0, d0, acc);
                    acc = fmaf(d1, d1, acc);
                }
                v[i] = acc;
            }
            halve_sum<16>(v, lane);
            halve_sum<8>(v, lane);
            halve_sum<4>(v, lane);
            halve_sum<2>(v, lane);
            if (pe0 > 0) {
                best = e_own;
                bestD = v[0];
                best_pos = pe0;
            }
        }
#pragma unroll
        for (int o = 16; !WIDE && o; o >>= 1) {
            const float oD = __shfl_xor_sync(0xffffffffu, bestD, o);
            const int oe = __shfl_xor_sync(0xffffffffu, best, o);
            const int op = __shfl_xor_sync(0xffffffffu, best_pos, o);
            if (oe >= 0 && (best < 0 || oD < bestD || (oD == bestD && op > best_pos))) {
                best = oe;
                bestD = oD;
                best_pos = op;
            }
        }
        const int hit = best >= 0 && bestD < L.tau2 * qn2;
        int eff = a.force ? L.forced_slot[bh] : (hit ? best : -1);
        int p = 0;
        if (eff >= L.ring_len) eff = -2;
        if (eff >= 0) {
            p = eff == best ? best_pos : rpos[eff];
            if (p <= 0 || p >= m) eff = -2;
        }
        if (eff == -2) {   // a forced slot that holds no entry: treat as a miss, flag it
            if (lane == 0) atomicOr(L.err, kErrSlot);
            eff = -1;
            p = 0;
        }
        lo_h = eff >= 0 ? max(0, p - L.band_r) : 0;
        if (lane == 0) {
            L.dec_own_slot[bh] = best;
            L.dec_own_hit[bh] = hit;
            L.dec_D[bh] = bestD;
            L.dec_qn2[bh] = qn2;
            L.dec_slot[bh] = eff;
            L.dec_lo[bh] = lo_h;
            if (eff >= 0) atomicAdd(&L.stats[kStHits], 1ull);
        }
        // Stage q~_m into the slot this step's Amend completes (the old entry's
        // query has been read above).  Only this warp reads this head's ring
        // queries before that Amend has run.
        __syncwarp();
        if (lane < 16) reinterpret_cast<uint4 *>(L.ring_q + (bh * L.ring_len + slot_new) * kD)[lane] = s_q[w][lane];
    } else {
        lo_h = 0;
        if (lane == 0) {
            L.dec_slot[bh] = -1;
            L.dec_lo[bh] = 0;
        }
    }

    if (a.full_mode) append_new();
    if (g == 0 && part == 0 && threadIdx.x == 0) {
        L.m_cur[b] = m;
        L.slot_cur[b] = slot_new;
    }

    // span start of this block's heads, then of the group
    __shared__ int s_glo[NWM];
    if (lane == 0) s_glo[w] = lo_h;
    __syncthreads();
    if (threadIdx.x == 0) {
        int lo = s_glo[0];
        for (int i = 1; i < nw; i++) lo = min(lo, s_glo[i]);
        if (SPLIT) atomicMin(&L.grp_lo[(size_t)b * L.Hkv + g], lo);
        else L.grp_lo[(size_t)b * L.Hkv + g] = lo;
    }
}

// ---------------------------------------------------------------------------
// Split-KV attention.  CTA = NW warps arranged as NP page lanes x NH head
// tiles (NH = ceil(G/8)); the warps of one page lane share its S-stage
// shared-memory pipeline of 16-token pages (K 4 KB + V 4 KB, rows XOR
// swizzled in 16-byte chunks so ldmatrix is conflict-free).
//
// Per page and head tile (8 query heads of the group):
//   S^T[16 tok x 8 heads] = K[16 x 128] Q^T[128 x 8]   8 x mma m16n8k16
//   online softmax on the fragments (log2 units)
//   O^T[128 x 8] += V^T[128 x 16] P^T[16 x 8]          8 x 2 mma (P split
//   into bf16 hi + lo so P V keeps ~16 bits of P: the partials must be
//   fp32-accurate because Amend's removal amplifies their error)
//
// Copy addressing: thread t of a lane group copies the 16-byte chunks
// t + i * 32 NH of a page; its chunk column is fixed (t mod 16) and its rows
// step by 2 NH, so every offset is a per-thread constant computed once.
// ---------------------------------------------------------------------------
template <int NW, int S, int NH>
__global__ void __launch_bounds__(NW * 32) attention_kernel(Layout L, StepArgs a)
{
    extern __shared__ __align__(128) uint8_t smem[];
    constexpr int NP = NW / NH;
    constexpr int GT = NH * 32;              // threads per page lane
    constexpr int CPT = 256 / GT;            // 16-byte chunks of K (and of V) per thread per page
    const int G = L.G;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int ht = warp % NH, pl = warp / NH;
    const int gtid = threadIdx.x - pl * GT;
    uint8_t *lane_smem = smem + (size_t)pl * S * kStageBytes;
    // comparison build only: the query rows of the head tiles, past the stages and the lane-merge area
    uint8_t *q_tiles = smem + max((size_t)NP * S * kStageBytes, (size_t)NP * G * kD * 4 + (size_t)NP * G * 8);
    const uint32_t lane_smem_u32 = smem_u32(lane_smem);
    const int r4 = lane >> 2, c4 = lane & 3;
    const float sl2 = L.scale_log2;

    // per-thread copy offsets (bytes within a 4 KB page block / stage half)
    const int cch = gtid & 15, crow0 = gtid >> 4;   // chunk column, first row
    uint32_t dst_off[CPT];
#pragma unroll
    for (int i = 0; i < CPT; i++) {
        const int row = crow0 + i * (GT / 16);
        dst_off[i] = row * 256 + ((cch ^ (row & 7)) << 4);
    }
    const uint32_t src_off0 = crow0 * 256 + cch * 16;
    // ldmatrix row bases
    const int krow = (lane & 7) + ((lane >> 3) & 1) * 8;   // K tile row (token) this lane addresses
    const int vtok = (lane & 7) + 8 * (lane >> 4);         // V tile row (token) this lane addresses

    // Q^T fragments of group bg (head column 8 ht + r4) and the band+tail
    // starts dec_lo of this thread's two head columns (8 ht + 2 c4, + 1).
    auto load_group = [&](int bg, uint32_t (&qf)[8][2], int &d0, int &d1) {
        const int b = bg / L.Hkv, g = bg - b * L.Hkv;
        const size_t hrow = (size_t)b * L.H + (size_t)g * G;
        const int hn = 8 * ht + r4;
        if (hn < G) {
            const uint32_t *qrow = reinterpret_cast<const uint32_t *>(a.q_post + (hrow + hn) * kD);
#pragma unroll
            for (int kk = 0; kk < 8; kk++) {
                qf[kk][0] = qrow[8 * kk + c4];
                qf[kk][1] = qrow[8 * kk + 4 + c4];
            }
        } else {
#pragma unroll
            for (int kk = 0; kk < 8; kk++) qf[kk][0] = qf[kk][1] = 0u;
        }
        const int hc0 = 8 * ht + 2 * c4;
        d0 = hc0 < G ? L.dec_lo[hrow + hc0] : 0;
        d1 = hc0 + 1 < G ? L.dec_lo[hrow + hc0 + 1] : 0;
    };

    __shared__ PlanShared ps;
    __shared__ int s_pool[NP][8];   // per page lane: pool pages claimed, by lane step past its own pages
    pdl_launch_dependents();
    // Consecutive steps plan almost alike, so this CTA's first item is
    // likely the one it had in the previous step (a hint only: a stale or
    // unrelated entry costs bandwidth, never correctness).
    int spec_bg = -1;
    if (blockIdx.x < L.item_cap) {
        const int4 prev = L.items[blockIdx.x];
        if (prev.x >= 0 && prev.x < a.batch * L.Hkv && prev.y >= 0 && prev.y < prev.z) spec_bg = prev.x;
    }
    // While Match runs, HBM is idle: warm L2 with the first pages of that
    // item (every index is bounds-checked).
    if (kSpeculativePages > 0 && gtid == 0 && spec_bg >= 0) {
        const int4 prev = L.items[blockIdx.x];
        const int pb = prev.x / L.Hkv, pgrp = prev.x - pb * L.Hkv;
        {
            for (int k = 0; k < kSpeculativePages; k++) {
                const int pg = (prev.y >> 4) + pl + k * NP;
                if (pg * 16 >= prev.z) break;
                bool ok = true;
                const size_t off = kv_block(L, pb, pgrp, pg, ok);
                if (!ok) break;
                prefetch_l2_bulk(L.k_pool + off, 4096);
                prefetch_l2_bulk(L.v_pool + off, 4096);
            }
        }
    }
    pdl_wait();   // spans come from match_plan
    // the likely first item's queries load while the plan is made
    uint32_t q_spec[8][2];
    int d0_spec = 0, d1_spec = 0;
    if (spec_bg >= 0) load_group(spec_bg, q_spec, d0_spec, d1_spec);
    cta_plan(L, a, ps);
    const int nbg = a.batch * L.Hkv;
    const int n_items = ps.total;
    if (blockIdx.x == 0) {   // publish the plan for combine and the counters
        for (int i = threadIdx.x; i <= nbg; i += blockDim.x) L.grp_item_off[i] = min(ps.off[i], n_items);
        for (int i = threadIdx.x; i < n_items; i += blockDim.x) L.items[i] = plan_item(L, a, ps, nbg, i);
        if (threadIdx.x == 0) {
            *L.n_items = n_items;
            if (ps.off[nbg] > L.item_cap) atomicOr(L.err, kErrPos);
            atomicAdd(&L.stats[kStSteps], 1ull);
            atomicAdd(&L.stats[kStKvRead], (unsigned long long)ps.T);
            atomicAdd(&L.stats[kStKvFull], (unsigned long long)ps.Tf);
            atomicAdd(&L.stats[kStItems], (unsigned long long)n_items);
            if (!a.full_mode) atomicAdd(&L.stats[kStDecisions], (unsigned long long)a.batch * L.H);
        }
    }

    for (int it = blockIdx.x; it < n_items; it += gridDim.x) {
        const int4 item = plan_item(L, a, ps, nbg, it);
        const int bg = item.x, ilo = item.y, ihi = item.z;
        const int b = bg / L.Hkv, g = bg - b * L.Hkv;

        // Q^T fragments for head column n = r4 of this tile
        uint32_t qf[8][2];
        int d0, d1;
        if (it == (int)blockIdx.x && bg == spec_bg) {
#pragma unroll
            for (int kk = 0; kk < 8; kk++) {
                qf[kk][0] = q_spec[kk][0];
                qf[kk][1] = q_spec[kk][1];
            }
            d0 = d0_spec;
            d1 = d1_spec;
        } else {
            load_group(bg, qf, d0, d1);
        }
        if constexpr (kAttnCudaCore) {   // the item's query rows (bf16), 8 per head tile, zeros past G
            __syncthreads();
            for (int i = threadIdx.x; i < NH * 8 * 16; i += NW * 32) {
                const int hh = i >> 4, ch = i & 15;
                uint4 v = make_uint4(0u, 0u, 0u, 0u);
                if (hh < G)
                    v = reinterpret_cast<const uint4 *>(a.q_post + ((size_t)b * L.H + (size_t)g * G + hh) * kD)[ch];
                reinterpret_cast<uint4 *>(q_tiles)[i] = v;
            }
            __syncthreads();
        }
        // the item's segment of the group, [slo, shi): any page of it may be
        // computed here (see the pool below), so masks use its bounds
        const int glo = ps.lo[bg], ghi = ps.hi[bg], gsp = plan_split(L, a, glo, ghi);
        const int slo = item.w ? gsp : glo, shi = item.w ? ghi : gsp;
        // this thread's two head columns and their first valid token (columns
        // past the group's heads are computed and discarded: no mask)
        const int hc0 = 8 * ht + 2 * c4, hc1 = hc0 + 1;
        const int lo0 = max(slo, d0);
        const int lo1 = max(slo, d1);
        const int lo_max = max(lo0, lo1);

        float m0 = -CUDART_INF_F, m1 = -CUDART_INF_F, l0 = 0.f, l1 = 0.f;
        float acc[8][4];
#pragma unroll
        for (int i = 0; i < 8; i++) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;

        const int pg0 = ilo >> 4, pg1 = (ihi - 1) >> 4;
        const int npg = pg1 - pg0 + 1;

        // Pages.  Every long item of the segment keeps its last ~8 % of pages
        // back in a pool shared by the segment's CTAs (not for 32-head
        // groups, whose CTAs hold a single page lane): a CTA streams its own
        // other pages (this lane: pg0 + pl + k NP), then claims pool pages one
        // at a time, so the CTAs of a segment finish together whatever
        // bandwidth each one gets.  Items of the segment are the C-aligned
        // chunks c_first, c_first + 1, ... of [slo, shi).
        constexpr int KDF = NH <= 2 ? kDynFrac : 0;
        const int Cg = plan_chunk(L, a, ps, nbg, glo, ghi);
        const ChunkDiv Rg = a.plan_mode == 0 ? ps.cd : chunk_div(Cg);
        const int c_first = div_c(slo, Rg), n_seg = div_c(shi - 1, Rg) - c_first + 1;
        auto chunk_pages = [&](int j, int &p0, int &p1) {
            const int c = c_first + j;
            p0 = max(slo, c * Cg) >> 4;
            p1 = (min(shi, (c + 1) * Cg) - 1) >> 4;
        };
        auto kept_back = [&](int n) { return (KDF > 0 && n >= kDynMinPages) ? max(2, n * KDF / 128) : 0; };
        int fp0, fp1, lp0 = 0, lp1 = -1;
        chunk_pages(0, fp0, fp1);
        if (n_seg > 1) chunk_pages(n_seg - 1, lp0, lp1);
        const int a_first = kept_back(fp1 - fp0 + 1);
        const int a_mid = n_seg > 2 ? kept_back(Cg / 16) : 0;
        const int a_last = n_seg > 1 ? kept_back(lp1 - lp0 + 1) : 0;
        const int n_mid = n_seg > 2 ? (n_seg - 2) * a_mid : 0;
        const int pool = a_first + n_mid + a_last;
        const int k_self = div_c(ilo, Rg) - c_first;
        const int kept_self = k_self == 0 ? a_first : (k_self == n_seg - 1 ? a_last : a_mid);
        const bool dyn = pool > 0 && kept_self > 0;
        int *const claim_ctr = L.seg_claim + 2 * bg + item.w;
        // pool slot q -> page (-1 past the pool): the chunks' kept pages in order
        auto pool_page = [&](int q) -> int {
            if (q < 0 || q >= pool) return -1;
            int j = 0, kept = a_first;
            if (q >= a_first) {
                q -= a_first;
                if (q < n_mid) {
                    j = 1 + q / a_mid;
                    q -= (j - 1) * a_mid;
                    kept = a_mid;
                } else {
                    j = n_seg - 1;
                    q -= n_mid;
                    kept = a_last;
                }
            }
            int p0, p1;
            chunk_pages(j, p0, p1);
            return p1 - kept + 1 + q;
        };
        const int npg_own = npg - kept_self;
        const int npl = pl < npg_own ? (npg_own - pl + NP - 1) / NP : 0;   // this lane's own pages

        // L2 prefetch of the page kPrefetchAhead pages past the copy front:
        // raises the bytes in flight beyond what the shared-memory stages hold
        auto prefetch = [&](int k) {
            if (gtid != 0 || k >= npl) return;
            const int pg = pg0 + pl + k * NP;
            bool ok = true;
            const size_t off = kv_block(L, b, g, pg, ok);
            if (!ok) return;
            prefetch_l2_bulk(L.k_pool + off, 4096);
            prefetch_l2_bulk(L.v_pool + off, 4096);
        };
        auto issue_page = [&](int pg, int k) {   // page pg into the stage of lane step k
            const uint32_t st = lane_smem_u32 + (k % S) * kStageBytes;
            bool ok = true;
            const size_t off = kv_block(L, b, g, pg, ok);
            if (!ok) {
                if (gtid == 0) atomicOr(L.err, kErrPage);
                return;
            }
            const char *ksrc = reinterpret_cast<const char *>(L.k_pool + off) + src_off0;
            const char *vsrc = reinterpret_cast<const char *>(L.v_pool + off) + src_off0;
#pragma unroll
            for (int i = 0; i < CPT; i++) cp_async16(st + dst_off[i], ksrc + i * (GT / 16) * 256);
#pragma unroll
            for (int i = 0; i < CPT; i++) cp_async16(st + 4096 + dst_off[i], vsrc + i * (GT / 16) * 256);
        };

#pragma unroll
        for (int k = S - 1; k < S - 1 + kPrefetchAhead; k++) prefetch(k);
#pragma unroll
        for (int k = 0; k < S - 1; k++) {
            if (k < npl) issue_page(pg0 + pl + k * NP, k);
            cp_async_commit();
        }
        // lane steps: own pages first, then claimed pool pages; a claim goes
        // out one step before its page is issued (its result published in
        // s_pool by the lane's first thread before the step's barrier)
        int n_iss = min(npl, S - 1);   // pages this lane has issued
        bool more = dyn;               // the pool may still hold pages for this lane
        int pend = -2;                 // first thread: the slot claimed last step (-2: none)
        for (int k = 0; k < n_iss; k++) {
            cp_async_wait<S - 2>();
            if (gtid == 0 && pend != -2) {
                const int pgc = pool_page(pend);
                s_pool[pl][(n_iss - npl) & 7] = pgc;
                if (pgc >= 0) {
                    bool ok = true;
                    const size_t off = kv_block(L, b, g, pgc, ok);
                    if (ok) {
                        prefetch_l2_bulk(L.k_pool + off, 4096);
                        prefetch_l2_bulk(L.v_pool + off, 4096);
                    }
                }
            }
            named_bar(1 + pl, GT);
            if (n_iss == k + S - 1) {
                int pgn = -1;
                if (n_iss < npl) {
                    pgn = pg0 + pl + n_iss * NP;
                } else if (more) {
                    pgn = s_pool[pl][(n_iss - npl) & 7];
                    if (pgn < 0) more = false;
                }
                if (pgn >= 0) {
                    issue_page(pgn, n_iss);
                    n_iss++;
                }
            }
            cp_async_commit();
            prefetch(k + S - 1 + kPrefetchAhead);
            pend = -2;
            if (gtid == 0 && more && n_iss == k + S && k + S >= npl) pend = atomicAdd(claim_ctr, 1);

            const uint32_t Ks = lane_smem_u32 + (k % S) * kStageBytes;
            const uint32_t Vs = Ks + 4096;
            const int pg = k < npl ? pg0 + pl + k * NP : s_pool[pl][(k - npl) & 7];

            // S^T = K Q^T
            float s[4] = {0.f, 0.f, 0.f, 0.f};
            if constexpr (kAttnCudaCore) {
                const uint8_t *Kp = lane_smem + (k % S) * kStageBytes;
                const uint8_t *qa = q_tiles + (size_t)(8 * ht + 2 * c4) * 256, *qb = qa + 256;
                const int ra = r4, rb = r4 + 8;
#pragma unroll 4
                for (int ch = 0; ch < 16; ch++) {
                    const uint4 ka = *reinterpret_cast<const uint4 *>(Kp + ra * 256 + ((ch ^ (ra & 7)) << 4));
                    const uint4 kb = *reinterpret_cast<const uint4 *>(Kp + rb * 256 + ((ch ^ (rb & 7)) << 4));
                    const uint4 q0 = *reinterpret_cast<const uint4 *>(qa + ch * 16);
                    const uint4 q1 = *reinterpret_cast<const uint4 *>(qb + ch * 16);
                    dot8_bf16(s[0], ka, q0);
                    dot8_bf16(s[1], ka, q1);
                    dot8_bf16(s[2], kb, q0);
                    dot8_bf16(s[3], kb, q1);
                }
            } else {
                const uint32_t rbase = Ks + krow * 256;
#pragma unroll
                for (int kk = 0; kk < 8; kk++) {
                    const int ch = 2 * kk + (lane >> 4);
                    uint32_t a0, a1, a2, a3;
                    ldsm_x4(a0, a1, a2, a3, rbase + ((ch ^ (krow & 7)) << 4));
                    mma_bf16(s, a0, a1, a2, a3, qf[kk][0], qf[kk][1]);
                }
            }
            // s[0]: token r4 head hc0; s[1]: token r4 head hc1; s[2], s[3]: token r4+8
            float z0 = s[0] * sl2, z1 = s[1] * sl2, z2 = s[2] * sl2, z3 = s[3] * sl2;
            if (pg * 16 < lo_max || pg * 16 + 16 > shi) {
                const int j0 = pg * 16 + r4, j1 = j0 + 8;
                if (!(j0 >= lo0 && j0 < shi)) z0 = -CUDART_INF_F;
                if (!(j0 >= lo1 && j0 < shi)) z1 = -CUDART_INF_F;
                if (!(j1 >= lo0 && j1 < shi)) z2 = -CUDART_INF_F;
                if (!(j1 >= lo1 && j1 < shi)) z3 = -CUDART_INF_F;
            }
            float mx0 = fmaxf(z0, z2), mx1 = fmaxf(z1, z3);
#pragma unroll
            for (int o = 4; o < 32; o <<= 1) {
                mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
            }
            const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
            const float bs0 = mn0 == -CUDART_INF_F ? 0.f : mn0;
            const float bs1 = mn1 == -CUDART_INF_F ? 0.f : mn1;
            const float p0 = exp2f(z0 - bs0), p1 = exp2f(z1 - bs1);
            const float p2 = exp2f(z2 - bs0), p3 = exp2f(z3 - bs1);
            // rescale only when some running max moved (rare after the first pages)
            if (__any_sync(0xffffffffu, mn0 != m0 || mn1 != m1)) {
                const float al0 = exp2f(m0 - bs0), al1 = exp2f(m1 - bs1);
                l0 *= al0;
                l1 *= al1;
#pragma unroll
                for (int i = 0; i < 8; i++) {
                    acc[i][0] *= al0;
                    acc[i][1] *= al1;
                    acc[i][2] *= al0;
                    acc[i][3] *= al1;
                }
            }
            l0 += p0 + p2;
            l1 += p1 + p3;
            m0 = mn0;
            m1 = mn1;
            if constexpr (kAttnCudaCore) {   // O^T += V^T P^T with fp32 P gathered from the lanes that hold it
                const uint8_t *Vp = lane_smem + (k % S) * kStageBytes + 4096;
#pragma unroll 2
                for (int t = 0; t < 16; t++) {
                    const int src = (t & 7) * 4 + c4;
                    const float pa = __shfl_sync(0xffffffffu, t < 8 ? p0 : p2, src);
                    const float pb = __shfl_sync(0xffffffffu, t < 8 ? p1 : p3, src);
                    const uint8_t *vrow = Vp + t * 256 + r4 * 2;
#pragma unroll
                    for (int mt = 0; mt < 8; mt++) {
                        const float v0 = __uint_as_float((uint32_t)*reinterpret_cast<const uint16_t *>(
                                                             vrow + (((2 * mt) ^ (t & 7)) << 4)) << 16);
                        const float v1 = __uint_as_float((uint32_t)*reinterpret_cast<const uint16_t *>(
                                                             vrow + (((2 * mt + 1) ^ (t & 7)) << 4)) << 16);
                        acc[mt][0] = fmaf(v0, pa, acc[mt][0]);
                        acc[mt][1] = fmaf(v0, pb, acc[mt][1]);
                        acc[mt][2] = fmaf(v1, pa, acc[mt][2]);
                        acc[mt][3] = fmaf(v1, pb, acc[mt][3]);
                    }
                }
                continue;
            }
            // P^T fragments (hi + lo bf16 parts) via in-register transpose
            const __nv_bfloat162 h01 = __floats2bfloat162_rn(p0, p1);
            const __nv_bfloat162 h23 = __floats2bfloat162_rn(p2, p3);
            const float2 f01 = __bfloat1622float2(h01), f23 = __bfloat1622float2(h23);
            const __nv_bfloat162 e01 = __floats2bfloat162_rn(p0 - f01.x, p1 - f01.y);
            const __nv_bfloat162 e23 = __floats2bfloat162_rn(p2 - f23.x, p3 - f23.y);
            const uint32_t bh0 = movmatrix_t(bf16x2_bits(h01)), bh1 = movmatrix_t(bf16x2_bits(h23));
            const uint32_t bl0 = movmatrix_t(bf16x2_bits(e01)), bl1 = movmatrix_t(bf16x2_bits(e23));
            {
                const uint32_t vbase = Vs + vtok * 256;
#pragma unroll
                for (int mt = 0; mt < 8; mt++) {
                    const int ch = 2 * mt + ((lane >> 3) & 1);
                    uint32_t a0, a1, a2, a3;
                    ldsm_x4_t(a0, a1, a2, a3, vbase + ((ch ^ (vtok & 7)) << 4));
                    mma_bf16(acc[mt], a0, a1, a2, a3, bh0, bh1);
                    mma_bf16(acc[mt], a0, a1, a2, a3, bl0, bl1);
                }
            }
        }
        cp_async_wait<0>();
        __syncthreads();   // every page lane drained: stage memory is free

        // sum l over the 8 lanes that share a head column
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) {
            l0 += __shfl_xor_sync(0xffffffffu, l0, o);
            l1 += __shfl_xor_sync(0xffffffffu, l1, o);
        }
        if constexpr (NP == 1) {   // one page lane: the fragments are the item's partial
            const float NEG = -CUDART_INF_F;
            if (hc0 < G) {
                float *o0 = L.part_o + ((size_t)it * G + hc0) * kD;
                const bool none = m0 == NEG;
#pragma unroll
                for (int i = 0; i < 8; i++) {
                    o0[16 * i + r4] = none ? 0.f : acc[i][0];
                    o0[16 * i + r4 + 8] = none ? 0.f : acc[i][2];
                }
                if (r4 == 0) L.part_ml[(size_t)it * G + hc0] = make_float2(m0, none ? 0.f : l0);
            }
            if (hc1 < G) {
                float *o1 = L.part_o + ((size_t)it * G + hc1) * kD;
                const bool none = m1 == NEG;
#pragma unroll
                for (int i = 0; i < 8; i++) {
                    o1[16 * i + r4] = none ? 0.f : acc[i][1];
                    o1[16 * i + r4 + 8] = none ? 0.f : acc[i][3];
                }
                if (r4 == 0) L.part_ml[(size_t)it * G + hc1] = make_float2(m1, none ? 0.f : l1);
            }
            continue;   // the stage memory was drained above; nothing else is staged
        }
        // stage each page lane's partial in shared memory, then merge lanes
        float *red_o = reinterpret_cast<float *>(smem);                               // [NP][G][D]
        float2 *red_ml = reinterpret_cast<float2 *>(red_o + (size_t)NP * G * kD);     // [NP][G]
        if (hc0 < G) {
            float *o0 = red_o + ((size_t)pl * G + hc0) * kD;
#pragma unroll
            for (int i = 0; i < 8; i++) {
                o0[16 * i + r4] = acc[i][0];
                o0[16 * i + r4 + 8] = acc[i][2];
            }
            if (r4 == 0) red_ml[pl * G + hc0] = make_float2(m0, l0);
        }
        if (hc1 < G) {
            float *o1 = red_o + ((size_t)pl * G + hc1) * kD;
#pragma unroll
            for (int i = 0; i < 8; i++) {
                o1[16 * i + r4] = acc[i][1];
                o1[16 * i + r4 + 8] = acc[i][3];
            }
            if (r4 == 0) red_ml[pl * G + hc1] = make_float2(m1, l1);
        }
        __syncthreads();
        for (int idx = threadIdx.x; idx < G * kD; idx += NW * 32) {
            const int hh = idx / kD, dd = idx - hh * kD;
            float M = -CUDART_INF_F;
#pragma unroll
            for (int q = 0; q < NP; q++) M = fmaxf(M, red_ml[q * G + hh].x);
            float lsum = 0.f, osum = 0.f;
            if (M != -CUDART_INF_F) {
#pragma unroll
                for (int q = 0; q < NP; q++) {
                    const float2 ml = red_ml[q * G + hh];
                    const float wq = exp2f(ml.x - M);
                    lsum += ml.y * wq;
                    osum += red_o[((size_t)q * G + hh) * kD + dd] * wq;
                }
            }
            L.part_o[((size_t)it * G + hh) * kD + dd] = osum;
            if (dd == 0) L.part_ml[(size_t)it * G + hh] = make_float2(M, lsum);
        }
        __syncthreads();   // shared memory is reused by the next item's pipeline
    }
}

// ---------------------------------------------------------------------------
// combine: one block of NW warps per (request, head).  Merges the
// group's item partials -- segment 0 (before the amend band) and segment 1
// (the band) -- and, on a hit, the ring's AS_{1:p-r} (Figure 2(b),
// "log-domain merge").  Items are spread over the warps so every load is in
// flight at once: block-wide maxima per segment first, then each warp's
// weighted sums, then a shared-memory reduction.
//
// Epilogue: out (bf16) and lse_out; then, with amend_band 0, Amend itself
// (Figure 2(c)): the band segment is the rectification term AS_{m-r+1:m},
// AS_{1:m-r} = AS_{1:m} (-) band, and the ring insert.  With amend_band 1 the
// summaries are handed to the side-stream Amend kernel instead.
// ---------------------------------------------------------------------------

__device__ __forceinline__ void fma4(float4 &acc, float w, float4 v)
{
    acc.x = fmaf(w, v.x, acc.x);
    acc.y = fmaf(w, v.y, acc.y);
    acc.z = fmaf(w, v.z, acc.z);
    acc.w = fmaf(w, v.w, acc.w);
}

__device__ __forceinline__ float4 scale4(float4 v, float s)
{
    return make_float4(v.x * s, v.y * s, v.z * s, v.w * s);
}

// AS_{1:m-r} from AS_{1:m} and the band AS_{m-r+1:m} (natural-log lse) by
// log-domain removal; the direct form `pre` when 1 - e^delta is too small
// for fp32.  Returns whether the direct form was taken.
__device__ __forceinline__ bool remove_band(float lf, float4 of, float lb, float4 ob, float lpre, float4 opre,
                                            float &le, float4 &oe)
{
    const float delta = fminf(lb - lf, 0.f);
    const float cond = -expm1f(delta);   // 1 - e^delta
    if (cond < kRemovalMinCond) {
        le = lpre;
        oe = opre;
        return true;
    }
    const float wgt = expf(delta), inv_c = 1.f / cond;
    oe = make_float4((of.x - wgt * ob.x) * inv_c, (of.y - wgt * ob.y) * inv_c, (of.z - wgt * ob.z) * inv_c,
                     (of.w - wgt * ob.w) * inv_c);
    le = lf + log1mexp_f(delta);
    return false;
}

// KB partials per warp per round of loads: 4, or 16 when a group may hold
// hundreds of items (one request's single KV group spread over the grid).
// NW warps per block: kCombineWarps, or 2 when every head has a handful of
// items (many requests, where the grid is thousands of blocks).
constexpr int kCombineWarps = 8;

template <int KB, int NW>
__global__ void __launch_bounds__(NW * 32) combine_kernel(Layout L, StepArgs a)
{
    __shared__ float s_red[2][NW];
    __shared__ float s_l[2][NW];
    __shared__ float4 s_o[2][NW][32];
    const int gw = blockIdx.x;
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int b = gw / L.H, h = gw - b * L.H;
    const int g = h / L.G, hh = h - g * L.G;
    const int bg = b * L.Hkv + g;
    const float NEG = -CUDART_INF_F;
    pdl_launch_dependents();
    pdl_wait();   // partials come from the attention kernel
    if (hh == 0 && threadIdx.x == 0) {   // the group's page pools start empty next step
        L.seg_claim[2 * bg] = 0;
        L.seg_claim[2 * bg + 1] = 0;
        if (L.lo_parts > 1) L.grp_lo[bg] = 0x7fffffff;   // split Match groups meet by atomicMin
    }

    float m_ring = NEG;
    float4 o_ring = make_float4(0.f, 0.f, 0.f, 0.f);
    int m = 0, slot = 0;
    if (!a.full_mode && w == 0) {
        m = L.m_cur[b];   // for the epilogue, loaded alongside the rest
        slot = L.slot_cur[b];
        const int eff = L.dec_slot[gw];
        if (eff >= 0) {   // summary and weight in one round trip
            const size_t e = (size_t)gw * L.ring_len + eff;
            const float lse = L.ring_lse[e];
            const float4 o = *reinterpret_cast<const float4 *>(L.ring_o + e * kD + 4 * lane);
            if (lse != NEG) {
                m_ring = lse * kLog2e;
                o_ring = o;
            }
        }
    }
    const int off0 = L.grp_item_off[bg], off1 = L.grp_item_off[bg + 1];
    // One pass: each warp merges items w, w + NW, ... (segment 0
    // and segment 1 separately) online, rescaling its sums when a batch
    // raises a maximum; a shared-memory step then merges the warps.
    float mp = NEG, mb = NEG, lp = 0.f, lb = 0.f;
    float4 op = make_float4(0.f, 0.f, 0.f, 0.f), ob = op;
    if (w == 0 && m_ring != NEG) {   // the reused AS_{1:p-r}: weight 1 at its own maximum
        mp = m_ring;
        lp = 1.f;
        op = o_ring;
    }
    constexpr int kBatch = KB;
    for (int i0 = off0 + w; i0 < off1; i0 += kBatch * NW) {
        float2 ml[kBatch];
        int sg[kBatch];
        float4 ov[kBatch];
#pragma unroll
        for (int k = 0; k < kBatch; k++) {
            const int i = min(i0 + k * NW, off1 - 1);
            ml[k] = L.part_ml[(size_t)i * L.G + hh];
            sg[k] = L.items[i].w;
            ov[k] = *reinterpret_cast<const float4 *>(L.part_o + ((size_t)i * L.G + hh) * kD + 4 * lane);
            if (i0 + k * NW >= off1) ml[k].x = NEG;   // padding slot
        }
        float np = mp, nb = mb;
#pragma unroll
        for (int k = 0; k < kBatch; k++) {
            if (sg[k]) nb = fmaxf(nb, ml[k].x);
            else np = fmaxf(np, ml[k].x);
        }
        if (np != mp) {
            const float r = mp == NEG ? 0.f : exp2f(mp - np);
            lp *= r;
            op = scale4(op, r);
            mp = np;
        }
        if (nb != mb) {
            const float r = mb == NEG ? 0.f : exp2f(mb - nb);
            lb *= r;
            ob = scale4(ob, r);
            mb = nb;
        }
#pragma unroll
        for (int k = 0; k < kBatch; k++) {
            if (ml[k].x == NEG) continue;
            if (sg[k]) {
                const float wi = exp2f(ml[k].x - mb);
                lb = fmaf(ml[k].y, wi, lb);
                fma4(ob, wi, ov[k]);
            } else {
                const float wi = exp2f(ml[k].x - mp);
                lp = fmaf(ml[k].y, wi, lp);
                fma4(op, wi, ov[k]);
            }
        }
    }
    if (lane == 0) {
        s_red[0][w] = mp;
        s_red[1][w] = mb;
        s_l[0][w] = lp;
        s_l[1][w] = lb;
    }
    s_o[0][w][lane] = op;
    s_o[1][w][lane] = ob;
    __syncthreads();
    if (w != 0) return;
    float bp = NEG, bb = NEG;
#pragma unroll
    for (int i = 0; i < NW; i++) {
        bp = fmaxf(bp, s_red[0][i]);
        bb = fmaxf(bb, s_red[1][i]);
    }
    lp = lb = 0.f;
    op = ob = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int i = 0; i < NW; i++) {
        if (s_red[0][i] != NEG) {
            const float r = exp2f(s_red[0][i] - bp);
            lp = fmaf(s_l[0][i], r, lp);
            fma4(op, r, s_o[0][i][lane]);
        }
        if (s_red[1][i] != NEG) {
            const float r = exp2f(s_red[1][i] - bb);
            lb = fmaf(s_l[1][i], r, lb);
            fma4(ob, r, s_o[1][i][lane]);
        }
    }
    if (bp == NEG) bp = 0.f;
    if (bb == NEG) bb = 0.f;
    // AS_{1:m} = pre (+) band
    const float mf = fmaxf(lp > 0.f ? bp : NEG, lb > 0.f ? bb : NEG);
    const float wp = lp > 0.f ? exp2f(bp - mf) : 0.f, wb = lb > 0.f ? exp2f(bb - mf) : 0.f;
    const float lf = lp * wp + lb * wb;
    float4 of = scale4(op, wp);
    fma4(of, wb, ob);
    of = scale4(of, 1.f / lf);
    const float lse = (mf + log2f(lf)) * kLn2;
    const __nv_bfloat162 lo2 = __floats2bfloat162_rn(of.x, of.y), hi2 = __floats2bfloat162_rn(of.z, of.w);
    *reinterpret_cast<uint2 *>(a.out + (size_t)gw * kD + 4 * lane) = make_uint2(bf16x2_bits(lo2), bf16x2_bits(hi2));
    if (a.lse_out && lane == 0) a.lse_out[gw] = lse;
    if (a.full_mode) {
        if (h == 0 && lane == 0) L.kv_len[b] = L.m_cur[b];   // the full step has no Amend to commit the length
        return;
    }
    const float4 opre = lp > 0.f ? scale4(op, 1.f / lp) : make_float4(0.f, 0.f, 0.f, 0.f);
    const float lpre = lp > 0.f ? (bp + log2f(lp)) * kLn2 : NEG;
    if (L.amend_band == 1) {   // the side-stream Amend kernel recomputes the band
        *reinterpret_cast<float4 *>(L.as_full_o + (size_t)gw * kD + 4 * lane) = of;
        *reinterpret_cast<float4 *>(L.as_pre_o + (size_t)gw * kD + 4 * lane) = opre;
        if (lane == 0) {
            L.as_full_lse[gw] = lse;
            L.as_pre_lse[gw] = lpre;
        }
        return;
    }
    // Amend in the epilogue: the band segment is AS_{m-r+1:m}(q_m)
    float le = NEG;
    float4 oe = make_float4(0.f, 0.f, 0.f, 0.f);
    if (m > L.band_r) {
        const float4 oband = scale4(ob, 1.f / lb);
        const float lband = (bb + log2f(lb)) * kLn2;
        if (remove_band(lse, of, lband, oband, lpre, opre, le, oe) && lane == 0)
            atomicAdd(&L.stats[kStDirect], 1ull);
    }
    const size_t e = (size_t)gw * L.ring_len + slot;   // the matched entry was read above
    *reinterpret_cast<float4 *>(L.ring_o + e * kD + 4 * lane) = oe;
    if (lane == 0) {
        L.ring_lse[e] = le;
        if (h == 0) {   // nothing in this kernel reads these per-request words
            L.ring_pos[(size_t)b * L.ring_len + slot] = m;
            L.kv_len[b] = m;
            L.step_ctr[b] = L.step_ctr[b] + 1;
        }
    }
}

// ---------------------------------------------------------------------------
// amend (side stream, Figure 2(c)): grid (Hkv, batch), block G warps.
// Rectification term AS_{m-r+1:m} with q_m -- either the band summary
// Complete produced (amend_band 0) or recomputed here from the KV store
// through shared-memory tiles (amend_band 1) -- then AS_{1:m-r} =
// AS_{1:m} (-) band (log-domain removal), ring insert at the step's slot,
// and finally the step's position and length are committed.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(1024) amend_kernel(Layout L, StepArgs a)
{
    extern __shared__ __align__(16) uint8_t band_smem[];   // [kBandTile][kBandRow] K, then V; q per warp
    const int g = blockIdx.x, b = blockIdx.y;
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int h = g * L.G + w;
    const size_t gw = (size_t)b * L.H + h;
    const int m = L.m_cur[b];
    const int slot = L.slot_cur[b];
    const int r = L.band_r;
    const float NEG = -CUDART_INF_F;
    float4 oe = make_float4(0.f, 0.f, 0.f, 0.f);
    float le = NEG;
    if (m > r) {
        uint8_t *Ks = band_smem, *Vs = band_smem + kBandTile * kBandRow;
        uint4 *qs = reinterpret_cast<uint4 *>(band_smem + 2 * kBandTile * kBandRow) + w * 16;
        if (lane < 16) qs[lane] = reinterpret_cast<const uint4 *>(L.q_stash + gw * kD)[lane];
        bool ok = true;
        float M = NEG, Ls = 0.f;
        float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int t0 = m - r; t0 < m; t0 += kBandTile) {
            const int n = min(kBandTile, m - t0);
            __syncthreads();   // previous tile consumed
            for (int c = threadIdx.x; c < n * 32; c += blockDim.x) {
                const int tok = c >> 5, part = c & 31, isv = part >> 4, ch = part & 15;
                bool okc = true;
                const int j = t0 + tok;
                const size_t off = kv_block(L, b, g, j >> 4, okc) + (size_t)(j & 15) * kD;
                if (!okc) {
                    ok = false;
                    continue;
                }
                const uint4 v = reinterpret_cast<const uint4 *>((isv ? L.v_pool : L.k_pool) + off)[ch];
                *reinterpret_cast<uint4 *>((isv ? Vs : Ks) + tok * kBandRow + ch * 16) = v;
            }
            __syncthreads();
            // scores: lane owns tokens lane and lane+32 of the tile
            float z[2];
#pragma unroll
            for (int k = 0; k < 2; k++) {
                const int tok = lane + 32 * k;
                z[k] = NEG;
                if (tok < n) {
                    float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
                    for (int i = 0; i < 16; i++) {
                        const uint4 kk = *reinterpret_cast<const uint4 *>(Ks + tok * kBandRow + i * 16);
                        const uint4 qq = qs[i];
                        const uint32_t ka[4] = {kk.x, kk.y, kk.z, kk.w}, qa[4] = {qq.x, qq.y, qq.z, qq.w};
#pragma unroll
                        for (int jj = 0; jj < 4; jj++) {
                            const float2 kf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&ka[jj]));
                            const float2 qf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&qa[jj]));
                            acc[jj] = fmaf(kf.x, qf.x, acc[jj]);
                            acc[jj] = fmaf(kf.y, qf.y, acc[jj]);
                        }
                    }
                    z[k] = ((acc[0] + acc[1]) + (acc[2] + acc[3])) * L.scale_log2;
                }
            }
            const float tmax = warp_max(fmaxf(z[0], z[1]));
            const float Mn = fmaxf(M, tmax);
            const float al = exp2f(M - Mn);
            const float p0 = exp2f(z[0] - Mn), p1 = exp2f(z[1] - Mn);
            Ls = Ls * al + warp_sum(p0 + p1);
            O = scale4(O, al);
            for (int tok = 0; tok < n; tok++) {
                const float pt = __shfl_sync(0xffffffffu, tok < 32 ? p0 : p1, tok & 31);
                fma4(O, pt, load_bf16x4(reinterpret_cast<const __nv_bfloat16 *>(Vs + tok * kBandRow) + 4 * lane));
            }
            M = Mn;
        }
        if (!ok) {
            if (lane == 0) atomicOr(L.err, kErrPage);
        } else {
            const float lb = (M + log2f(Ls)) * kLn2;
            const float4 ob = scale4(O, 1.f / Ls);
            const float4 of = *reinterpret_cast<const float4 *>(L.as_full_o + gw * kD + 4 * lane);
            const float4 opre = *reinterpret_cast<const float4 *>(L.as_pre_o + gw * kD + 4 * lane);
            if (remove_band(L.as_full_lse[gw], of, lb, ob, L.as_pre_lse[gw], opre, le, oe) && lane == 0)
                atomicAdd(&L.stats[kStDirect], 1ull);
        }
    }
    const size_t e = gw * L.ring_len + slot;
    *reinterpret_cast<float4 *>(L.ring_o + e * kD + 4 * lane) = oe;
    if (lane == 0) L.ring_lse[e] = le;
    __syncthreads();
    if (g == 0 && threadIdx.x == 0) {
        L.ring_pos[(size_t)b * L.ring_len + slot] = m;
        L.kv_len[b] = m;
        L.step_ctr[b] = L.step_ctr[b] + 1;
    }
}

// ---------------------------------------------------------------------------
// seed: entries first..n-1 of a seeding call into request req's rings, entry
// i at slot (base_step + i) mod L, as if inserted by decode steps.  One warp
// per (entry, head); q [n][H][D] bf16, o [n][H][D] fp32, lse [n][H] fp32.
// ---------------------------------------------------------------------------
__global__ void seed_kernel(Layout L, int req, int first, int n, int base_step, const __nv_bfloat16 *q,
                            const float *o, const float *lse)
{
    const int gw = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    const int i = first + gw / L.H, h = gw % L.H;
    if (i >= n) return;
    const int slot = (base_step + i) % L.ring_len;
    const size_t src = (size_t)i * L.H + h;
    const size_t e = ((size_t)req * L.H + h) * L.ring_len + slot;
    if (lane < 16) reinterpret_cast<uint4 *>(L.ring_q + e * kD)[lane] = reinterpret_cast<const uint4 *>(q + src * kD)[lane];
    reinterpret_cast<float4 *>(L.ring_o + e * kD)[lane] = reinterpret_cast<const float4 *>(o + src * kD)[lane];
    if (lane == 0) {
        L.ring_lse[e] = lse[src];
        if (h == 0) L.ring_pos[(size_t)req * L.ring_len + slot] = L.seed_pos[i - first];
        if (gw == 0) L.step_ctr[req] = base_step + n;
    }
}

// ---------------------------------------------------------------------------
// append: n tokens of K and V [n][Hkv][D] at indices start.. of request req.
// ---------------------------------------------------------------------------
__global__ void append_kernel(Layout L, int req, int start, int n, const __nv_bfloat16 *k,
                              const __nv_bfloat16 *v)
{
    const size_t per = (size_t)n * L.Hkv * 16;   // 16-byte chunks of K (and of V)
    for (size_t idx = (size_t)blockIdx.x * blockDim.x + threadIdx.x; idx < 2 * per;
         idx += (size_t)gridDim.x * blockDim.x) {
        const int isv = idx >= per;
        const size_t c = isv ? idx - per : idx;
        const int t = (int)(c / ((size_t)L.Hkv * 16));
        const int rem = (int)(c - (size_t)t * L.Hkv * 16);
        const int g = rem >> 4, ch = rem & 15;
        const int tok = start + t;
        bool ok = true;
        const size_t off = kv_block(L, req, g, tok >> 4, ok);
        if (!ok) {
            atomicOr(L.err, kErrPage);
            continue;
        }
        const uint4 *src = reinterpret_cast<const uint4 *>((isv ? v : k) + ((size_t)t * L.Hkv + g) * kD) + ch;
        uint4 *dst = reinterpret_cast<uint4 *>((isv ? L.v_pool : L.k_pool) + off + (size_t)(tok & 15) * kD) + ch;
        *dst = *src;
    }
    if (blockIdx.x == 0 && threadIdx.x == 0) L.kv_len[req] = start + n;
}

}  // namespace

// ---------------------------------------------------------------------------
// launchers
// ---------------------------------------------------------------------------
static int head_tiles(int G) { return (G + 7) / 8; }

static size_t attention_smem(int G)
{
    const int NH = head_tiles(G), NP = kAttnWarps / NH;
    const size_t pipe = (size_t)NP * kAttnStages * kStageBytes;
    const size_t red = (size_t)NP * G * kD * 4 + (size_t)NP * G * 8;
    const size_t q_tiles = kAttnCudaCore ? (size_t)NH * 8 * kD * 2 : 0;   // after the stages
    return (pipe > red ? pipe : red) + q_tiles;
}

template <int NH>
static cudaError_t attention_config_nh(size_t smem, int *ctas_per_sm)
{
    auto k = attention_kernel<kAttnWarps, kAttnStages, NH>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(ctas_per_sm, k, kAttnWarps * 32, smem);
}

cudaError_t attention_kernel_config(int G, size_t *smem, int *ctas_per_sm)
{
    *smem = attention_smem(G);
    switch (head_tiles(G)) {
    case 1: return attention_config_nh<1>(*smem, ctas_per_sm);
    case 2: return attention_config_nh<2>(*smem, ctas_per_sm);
    default: return attention_config_nh<4>(*smem, ctas_per_sm);
    }
}



template <typename Kernel>
static cudaError_t launch_maybe_pdl(Kernel k, dim3 grid, dim3 block, size_t smem, cudaStream_t s, bool pdl,
                                    const Layout &L, const StepArgs &a)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, k, L, a);
}

cudaError_t launch_match_plan(const Layout &L, const StepArgs &a, cudaStream_t s)
{
    // One warp per query head, at most kMatchWarps heads per block (a group
    // of more heads is split over L.lo_parts blocks).  Rings of more than
    // kSmallRing entries go through the scan kernel first.
    constexpr int T = kMatchWarps * 32;
    const int nw = (L.G + L.lo_parts - 1) / L.lo_parts;
    const dim3 grid(L.lo_parts, L.Hkv, a.batch), block(nw * 32);
    const int form = a.full_mode || L.ring_len <= 16 ? 0 : L.ring_len <= kSmallRing ? 1 : 2;
    if (form == 2) {
        const dim3 sgrid((L.ring_len + kScanBlock - 1) / kScanBlock, L.H, a.batch);
        cudaError_t e = launch_maybe_pdl(ring_scan_kernel, sgrid, dim3(kScanBlock), 0, s, a.pdl, L, a);
        if (e != cudaSuccess) return e;
    }
    if (L.lo_parts == 1) {
        if (form == 0) return launch_maybe_pdl(match_plan_kernel<512, false, 8, false>, grid, block, 0, s, a.pdl, L, a);
        if (form == 1) return launch_maybe_pdl(match_plan_kernel<512, false, 16, false>, grid, block, 0, s, a.pdl, L, a);
        return launch_maybe_pdl(match_plan_kernel<512, true, 8, false>, grid, block, 0, s, a.pdl, L, a);
    }
    if (form == 0) return launch_maybe_pdl(match_plan_kernel<T, false, 8, true>, grid, block, 0, s, a.pdl, L, a);
    if (form == 1) return launch_maybe_pdl(match_plan_kernel<T, false, 16, true>, grid, block, 0, s, a.pdl, L, a);
    return launch_maybe_pdl(match_plan_kernel<T, true, 8, true>, grid, block, 0, s, a.pdl, L, a);
}

cudaError_t launch_seed(const Layout &L, int req, int first, int n, int base_step, const __nv_bfloat16 *q,
                        const float *o, const float *lse, cudaStream_t s)
{
    const int warps = (n - first) * L.H;
    seed_kernel<<<(warps + 7) / 8, 256, 0, s>>>(L, req, first, n, base_step, q, o, lse);
    return cudaGetLastError();
}

cudaError_t launch_attention(const Layout &L, const StepArgs &a, size_t smem, cudaStream_t s)
{
    const dim3 grid(a.grid_ctas), block(kAttnWarps * 32);
    switch (head_tiles(L.G)) {
    case 1: return launch_maybe_pdl(attention_kernel<kAttnWarps, kAttnStages, 1>, grid, block, smem, s, a.pdl, L, a);
    case 2: return launch_maybe_pdl(attention_kernel<kAttnWarps, kAttnStages, 2>, grid, block, smem, s, a.pdl, L, a);
    default: return launch_maybe_pdl(attention_kernel<kAttnWarps, kAttnStages, 4>, grid, block, smem, s, a.pdl, L, a);
    }
}

cudaError_t launch_combine(const Layout &L, const StepArgs &a, cudaStream_t s)
{
    // a group holds at most about grid / groups + 2 items
    const int nbg = a.batch * L.Hkv;
    const int per_group = (a.grid_ctas + nbg - 1) / nbg + 2;
    const dim3 grid(a.batch * L.H);
    // A few items per head (many requests): small blocks, so that the whole
    // grid is resident beside the attention CTAs when their wait releases.
    if (per_group <= 8) return launch_maybe_pdl(combine_kernel<4, 2>, grid, dim3(64), 0, s, a.pdl != 0, L, a);
    const dim3 block(kCombineWarps * 32);
    if (per_group > 128) return launch_maybe_pdl(combine_kernel<16, kCombineWarps>, grid, block, 0, s, a.pdl != 0, L, a);
    return launch_maybe_pdl(combine_kernel<4, kCombineWarps>, grid, block, 0, s, a.pdl != 0, L, a);
}

static size_t amend_smem(int G) { return (size_t)2 * kBandTile * kBandRow + (size_t)G * kD * 2; }

cudaError_t amend_kernel_config()
{
    return cudaFuncSetAttribute(amend_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)amend_smem(kMaxGroup));
}

cudaError_t launch_amend(const Layout &L, const StepArgs &a, cudaStream_t s)
{
    amend_kernel<<<dim3(L.Hkv, a.batch), L.G * 32, amend_smem(L.G), s>>>(L, a);
    return cudaGetLastError();
}

cudaError_t launch_append(const Layout &L, int req, int start, int n, const __nv_bfloat16 *k,
                          const __nv_bfloat16 *v, cudaStream_t s)
{
    const size_t chunks = (size_t)2 * n * L.Hkv * 16;
    size_t blocks = (chunks + 255) / 256;
    if (blocks > 4096) blocks = 4096;
    if (blocks < 1) blocks = 1;
    append_kernel<<<(unsigned)blocks, 256, 0, s>>>(L, req, start, n, k, v);
    return cudaGetLastError();
}

}  // namespace macgpu
