// sm_103a split-KV attention of the MAC-Attention decode step (Complete,
// Figure 2(b) of the MAC-Attention paper) and the span-proportional planner
// every CTA runs in its prologue (Figure 3(b), "load-balanced planning").
//
// Conventions: token index j (0-based) is the paper's position j+1; ranges
// [lo, hi) are half-open over indices.  Scores are kept in log2 units
// (scaled by sm_scale * log2 e) inside the kernels.
#include "mac_plan.cuh"

namespace macgpu {

namespace {

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
//
// Groups of 16 or 32 heads (HM = true) put the heads on the M axis instead:
// a warp owns a 16-head tile, so a page is read from shared memory by G / 16
// warps rather than G / 8, and the score fragments are already the A
// operand of P V (no transpose):
//   S[16 heads x 16 tok] = Q[16 x 128] K^T[128 x 16]     2 x 8 mma
//   O[16 heads x 128]   += P[16 x 16] V[16 x 128]        16 x 2 mma (hi + lo)
// with Q in registers as A fragments and K, V read by ldmatrix as B.
// ---------------------------------------------------------------------------
template <int NW, int S, int NH, bool HM, int MINB>
__global__ void __launch_bounds__(NW * 32, MINB) attention_kernel(Layout L, StepArgs a)
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

    // Query fragments of group bg and the band+tail starts dec_lo of this
    // thread's two heads: Q^T as B (head column 8 ht + r4; heads 8 ht + 2 c4,
    // + 1), or, with HM, Q as A (head rows 16 ht + r4, + 8: the two heads).
    using QFrag = uint32_t[8][HM ? 4 : 2];
    auto load_group = [&](int bg, QFrag &qf, int &d0, int &d1) {
        const int b = bg / L.Hkv, g = bg - b * L.Hkv;
        const size_t hrow = (size_t)b * L.H + (size_t)g * G;
        if constexpr (HM) {
            const int ha = 16 * ht + r4;
            const uint32_t *qa = reinterpret_cast<const uint32_t *>(a.q_post + (hrow + ha) * kD);
            const uint32_t *qb = reinterpret_cast<const uint32_t *>(a.q_post + (hrow + ha + 8) * kD);
#pragma unroll
            for (int kk = 0; kk < 8; kk++) {
                qf[kk][0] = qa[8 * kk + c4];
                qf[kk][1] = qb[8 * kk + c4];
                qf[kk][2] = qa[8 * kk + 4 + c4];
                qf[kk][3] = qb[8 * kk + 4 + c4];
            }
            d0 = L.dec_lo[hrow + ha];
            d1 = L.dec_lo[hrow + ha + 8];
            return;
        }
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
    QFrag q_spec;
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

        // query fragments of this warp's head tile
        QFrag qf;
        int d0, d1;
        if (it == (int)blockIdx.x && bg == spec_bg) {
#pragma unroll
            for (int kk = 0; kk < 8; kk++)
#pragma unroll
                for (int j = 0; j < (HM ? 4 : 2); j++) qf[kk][j] = q_spec[kk][j];
            d0 = d0_spec;
            d1 = d1_spec;
        } else {
            load_group(bg, qf, d0, d1);
        }
        if constexpr (kAttnCudaCore && !HM) {   // the item's query rows (bf16), 8 per head tile, zeros past G
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
        // this thread's two heads (columns, or rows with HM) and their first
        // valid token (columns past the group's heads are computed and
        // discarded: no mask)
        const int hc0 = HM ? 16 * ht + r4 : 8 * ht + 2 * c4, hc1 = HM ? hc0 + 8 : hc0 + 1;
        const int lo0 = max(slo, d0);
        const int lo1 = max(slo, d1);
        const int lo_max = max(lo0, lo1);

        float m0 = -CUDART_INF_F, m1 = -CUDART_INF_F, l0 = 0.f, l1 = 0.f;
        float up0 = -CUDART_INF_F, up1 = -CUDART_INF_F;   // HM: raw score above which a row's reference moves
        constexpr int NACC = HM ? 16 : 8;   // O^T m-tiles of 16 dims, or O n-tiles of 8 dims (HM)
        float acc[NACC][4];
#pragma unroll
        for (int i = 0; i < NACC; i++) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;

        const int pg0 = ilo >> 4, pg1 = (ihi - 1) >> 4;
        const int npg = pg1 - pg0 + 1;

        // Pages.  Every long item of the segment keeps its last ~8 % of pages
        // back in a pool shared by the segment's CTAs (not with four 8-head
        // tiles, whose CTAs hold a single page lane): a CTA streams its own
        // other pages (this lane: pg0 + pl + k NP), then claims pool pages one
        // at a time, so the CTAs of a segment finish together whatever
        // bandwidth each one gets.  Items of the segment are the C-aligned
        // chunks c_first, c_first + 1, ... of [slo, shi).
        constexpr int KDF = NH <= 2 ? kDynFrac : 0;
        const int Cg = plan_chunk(L, a, ps, nbg, glo, gsp);
        const ChunkDiv Rg = a.plan_mode == 0 ? ps.cd : chunk_div(Cg);
        const int c_first = div_c(slo, Rg), n_seg = div_c(shi - 1, Rg) - c_first + 1;
        auto chunk_pages = [&](int j, int &p0, int &p1) {
            const int c = c_first + j;
            p0 = max(slo, c * Cg) >> 4;
            p1 = (min(shi, (c + 1) * Cg) - 1) >> 4;
        };
        // (a band item is a segment of its own: nothing is kept back)
        auto kept_back = [&](int n) {
            return (KDF > 0 && item.w == 0 && n >= kDynMinPages) ? max(2, n * KDF / 128) : 0;
        };
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
            // value rows past the segment's end are staged as zeros: their
            // weight is exactly 0, and 0 x (whatever the slot holds) must not
            // turn into NaN (key rows there are masked by the score select)
            const int vrows = shi - pg * 16;
#pragma unroll
            for (int i = 0; i < CPT; i++) cp_async16(st + dst_off[i], ksrc + i * (GT / 16) * 256);
#pragma unroll
            for (int i = 0; i < CPT; i++)
                cp_async16_zfill(st + 4096 + dst_off[i], vsrc + i * (GT / 16) * 256,
                                 crow0 + i * (GT / 16) < vrows ? 16u : 0u);
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

            if constexpr (HM) {
                // S = Q K^T: n-tile j holds tokens 8 j .. 8 j + 7; this thread
                // has head rows r4 (sc[j][0..1]) and r4 + 8 (sc[j][2..3]) at
                // tokens 8 j + 2 c4, + 1
                // (even and odd k-steps accumulate apart: four independent
                // mma chains instead of two)
                float sc[2][2][4] = {};
                {
                    const uint32_t kbase = Ks + vtok * 256;
#pragma unroll
                    for (int kk = 0; kk < 8; kk++) {
                        const int ch = 2 * kk + ((lane >> 3) & 1);
                        uint32_t b0, b1, b2, b3;
                        ldsm_x4(b0, b1, b2, b3, kbase + ((ch ^ (vtok & 7)) << 4));
                        mma_bf16(sc[0][kk & 1], qf[kk][0], qf[kk][1], qf[kk][2], qf[kk][3], b0, b1);
                        mma_bf16(sc[1][kk & 1], qf[kk][0], qf[kk][1], qf[kk][2], qf[kk][3], b2, b3);
                    }
                }
                // raw scores (the scale sl2 > 0 is applied inside the exponent)
                float z[2][4];
#pragma unroll
                for (int j = 0; j < 2; j++)
#pragma unroll
                    for (int e = 0; e < 4; e++) z[j][e] = sc[j][0][e] + sc[j][1][e];
                if (pg * 16 < lo_max || pg * 16 + 16 > shi) {
#pragma unroll
                    for (int j = 0; j < 2; j++)
#pragma unroll
                        for (int e = 0; e < 2; e++) {
                            const int tok = pg * 16 + 8 * j + 2 * c4 + e;
                            if (!(tok >= lo0 && tok < shi)) z[j][e] = -CUDART_INF_F;
                            if (!(tok >= lo1 && tok < shi)) z[j][2 + e] = -CUDART_INF_F;
                        }
                }
                // The reference maximum of a row moves only when a page's
                // scores pass it by more than kLazyMax (log2 units), so weights
                // stay <= 2^8; only then (about once per item) is the row's
                // maximum reduced over its quad and the accumulators rescaled.
                float mx0 = fmaxf(fmaxf(z[0][0], z[0][1]), fmaxf(z[1][0], z[1][1]));
                float mx1 = fmaxf(fmaxf(z[0][2], z[0][3]), fmaxf(z[1][2], z[1][3]));
                if (__any_sync(0xffffffffu, mx0 > up0 || mx1 > up1)) {
#pragma unroll
                    for (int o = 1; o < 4; o <<= 1) {
                        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
                        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
                    }
                    const float mn0 = mx0 > up0 ? mx0 * sl2 : m0, mn1 = mx1 > up1 ? mx1 * sl2 : m1;
                    const float al0 = ex2_approx(m0 - (mn0 == -CUDART_INF_F ? 0.f : mn0));
                    const float al1 = ex2_approx(m1 - (mn1 == -CUDART_INF_F ? 0.f : mn1));
                    l0 *= al0;
                    l1 *= al1;
#pragma unroll
                    for (int i = 0; i < 16; i++) {
                        acc[i][0] *= al0;
                        acc[i][1] *= al0;
                        acc[i][2] *= al1;
                        acc[i][3] *= al1;
                    }
                    m0 = mn0;
                    m1 = mn1;
                    up0 = m0 == -CUDART_INF_F ? -CUDART_INF_F : (m0 + kLazyMax) / sl2;
                    up1 = m1 == -CUDART_INF_F ? -CUDART_INF_F : (m1 + kLazyMax) / sl2;
                }
                const float nb0 = m0 == -CUDART_INF_F ? 0.f : -m0, nb1 = m1 == -CUDART_INF_F ? 0.f : -m1;
                float pr[2][4];
#pragma unroll
                for (int j = 0; j < 2; j++) {
                    pr[j][0] = ex2_approx(fmaf(z[j][0], sl2, nb0));
                    pr[j][1] = ex2_approx(fmaf(z[j][1], sl2, nb0));
                    pr[j][2] = ex2_approx(fmaf(z[j][2], sl2, nb1));
                    pr[j][3] = ex2_approx(fmaf(z[j][3], sl2, nb1));
                }
                l0 += (pr[0][0] + pr[0][1]) + (pr[1][0] + pr[1][1]);
                l1 += (pr[0][2] + pr[0][3]) + (pr[1][2] + pr[1][3]);
                // P as the A operand (k = token): a0 rows r4 tokens 2 c4.., a1
                // row r4 + 8, a2 / a3 the same at tokens 8 + 2 c4..; hi + lo
                uint32_t ph[4], plo[4];
#pragma unroll
                for (int j = 0; j < 2; j++)
#pragma unroll
                    for (int rr = 0; rr < 2; rr++) {
                        const __nv_bfloat162 hv = __floats2bfloat162_rn(pr[j][2 * rr], pr[j][2 * rr + 1]);
                        const float2 fv = __bfloat1622float2(hv);
                        const __nv_bfloat162 lv =
                            __floats2bfloat162_rn(pr[j][2 * rr] - fv.x, pr[j][2 * rr + 1] - fv.y);
                        ph[2 * j + rr] = bf16x2_bits(hv);
                        plo[2 * j + rr] = bf16x2_bits(lv);
                    }
                // O += P V: ldmatrix.trans gives the B fragments of dim
                // n-tiles 2 np and 2 np + 1; four n-tiles per round, hi parts
                // then lo parts, so no mma waits on the one before it
                const uint32_t vbase = Vs + krow * 256;
#pragma unroll
                for (int np = 0; np < 8; np += 2) {
                    uint32_t b[2][4];
#pragma unroll
                    for (int u = 0; u < 2; u++) {
                        const int ch = 2 * (np + u) + (lane >> 4);
                        ldsm_x4_t(b[u][0], b[u][1], b[u][2], b[u][3], vbase + ((ch ^ (krow & 7)) << 4));
                    }
#pragma unroll
                    for (int u = 0; u < 4; u++)
                        mma_bf16(acc[2 * np + u], ph[0], ph[1], ph[2], ph[3], b[u >> 1][2 * (u & 1)],
                                 b[u >> 1][2 * (u & 1) + 1]);
#pragma unroll
                    for (int u = 0; u < 4; u++)
                        mma_bf16(acc[2 * np + u], plo[0], plo[1], plo[2], plo[3], b[u >> 1][2 * (u & 1)],
                                 b[u >> 1][2 * (u & 1) + 1]);
                }
                continue;
            }

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

        // sum l over the lanes that share a head: the 8 of a column, or (HM)
        // the 4 of a row
#pragma unroll
        for (int o = HM ? 1 : 4; o < (HM ? 4 : 32); o <<= 1) {
            l0 += __shfl_xor_sync(0xffffffffu, l0, o);
            l1 += __shfl_xor_sync(0xffffffffu, l1, o);
        }
        // HM: this thread's fragment of head row h (acc[i][2 half], + 1: dims
        // 8 i + 2 c4, + 1) into a [G][D] array, and the row's (max, sum)
        auto store_rows = [&](float *o_base, float2 *ml_base, bool zero_empty) {
#pragma unroll
            for (int half = 0; half < 2; half++) {
                const int h = half ? hc1 : hc0;
                const float mh = half ? m1 : m0, lh = half ? l1 : l0;
                const bool none = zero_empty && mh == -CUDART_INF_F;
                float *orow = o_base + (size_t)h * kD + 2 * c4;
#pragma unroll
                for (int i = 0; i < NACC; i++)
                    *reinterpret_cast<float2 *>(orow + 8 * i) =
                        none ? make_float2(0.f, 0.f) : make_float2(acc[i][2 * half], acc[i][2 * half + 1]);
                if (c4 == 0) ml_base[h] = make_float2(mh, none ? 0.f : lh);
            }
        };
        if constexpr (NP == 1) {   // one page lane: the fragments are the item's partial
            const float NEG = -CUDART_INF_F;
            if constexpr (HM) {
                store_rows(L.part_o + (size_t)it * G * kD, L.part_ml + (size_t)it * G, true);
                continue;
            }
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
        if constexpr (HM) {
            store_rows(red_o + (size_t)pl * G * kD, red_ml + pl * G, false);
        } else if (hc0 < G) {
            float *o0 = red_o + ((size_t)pl * G + hc0) * kD;
#pragma unroll
            for (int i = 0; i < 8; i++) {
                o0[16 * i + r4] = acc[i][0];
                o0[16 * i + r4 + 8] = acc[i][2];
            }
            if (r4 == 0) red_ml[pl * G + hc0] = make_float2(m0, l0);
        }
        if (!HM && hc1 < G) {
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

}  // namespace

// ---------------------------------------------------------------------------
// launchers
// ---------------------------------------------------------------------------
// Groups of 16 or 32 heads put the heads on the mma M axis (16-head tiles);
// smaller groups put them on N (8-head tiles).
static bool heads_on_m(int G) { return kHeadsOnM && !kAttnCudaCore && G % 16 == 0; }
static int head_tiles(int G) { return heads_on_m(G) ? G / 16 : (G + 7) / 8; }

// Pipeline stages per page lane: 32-head groups (two page lanes per CTA)
// take their own depth.
static int attention_stages(int G) { return heads_on_m(G) && G == 32 ? kHmStages32 : kAttnStages; }

static size_t attention_smem(int G)
{
    const int NH = head_tiles(G), NP = kAttnWarps / NH;
    const size_t pipe = (size_t)NP * attention_stages(G) * kStageBytes;
    const size_t red = (size_t)NP * G * kD * 4 + (size_t)NP * G * 8;
    const size_t q_tiles = kAttnCudaCore ? (size_t)NH * 8 * kD * 2 : 0;   // after the stages
    return (pipe > red ? pipe : red) + q_tiles;
}

template <int NH, bool HM, int S, int MINB>
static cudaError_t attention_config_nh(size_t smem, int *ctas_per_sm)
{
    auto k = attention_kernel<kAttnWarps, S, NH, HM, MINB>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(ctas_per_sm, k, kAttnWarps * 32, smem);
}

// 32-head groups go to the tcgen05 kernel unless it is switched off
static bool tensor_memory_path(int G) { return kTc32 && !kAttnCudaCore && G == 32; }
bool attention_tc_wanted(int G) { return tensor_memory_path(G); }

bool attention_wide(int G, int groups) { return heads_on_m(G) && G == 32 && groups >= kHmWideGroups; }

cudaError_t attention_kernel_config(int G, bool wide, bool tc, size_t *smem, int *ctas_per_sm)
{
    if (tc && tensor_memory_path(G)) return attention_tc_config(smem, ctas_per_sm);
    *smem = attention_smem(G);
    if (heads_on_m(G)) {
        if (G == 16) return attention_config_nh<1, true, kAttnStages, kHmMinCtas16>(*smem, ctas_per_sm);
        if (wide) return attention_config_nh<2, true, kHmStages32, kHmMinCtas32Wide>(*smem, ctas_per_sm);
        return attention_config_nh<2, true, kHmStages32, kHmMinCtas32>(*smem, ctas_per_sm);
    }
    switch (head_tiles(G)) {
    case 1: return attention_config_nh<1, false, kAttnStages, 1>(*smem, ctas_per_sm);
    case 2: return attention_config_nh<2, false, kAttnStages, 1>(*smem, ctas_per_sm);
    default: return attention_config_nh<4, false, kAttnStages, 1>(*smem, ctas_per_sm);
    }
}

cudaError_t launch_attention(const Layout &L, const StepArgs &a, const TcMaps *maps, size_t smem, cudaStream_t s)
{
    if (a.tc && tensor_memory_path(L.G) && L.tc && maps) return launch_attention_tc(L, a, *maps, smem, s);
    const dim3 grid(a.grid_ctas), block(kAttnWarps * 32);
    if (heads_on_m(L.G)) {
        if (L.G == 16)
            return launch_maybe_pdl(attention_kernel<kAttnWarps, kAttnStages, 1, true, kHmMinCtas16>, grid, block, smem, s,
                                    a.pdl, L, a);
        if (a.wide)
            return launch_maybe_pdl(attention_kernel<kAttnWarps, kHmStages32, 2, true, kHmMinCtas32Wide>, grid, block, smem,
                                    s, a.pdl, L, a);
        return launch_maybe_pdl(attention_kernel<kAttnWarps, kHmStages32, 2, true, kHmMinCtas32>, grid, block, smem, s,
                                a.pdl, L, a);
    }
    switch (head_tiles(L.G)) {
    case 1: return launch_maybe_pdl(attention_kernel<kAttnWarps, kAttnStages, 1, false, 1>, grid, block, smem, s, a.pdl, L, a);
    case 2: return launch_maybe_pdl(attention_kernel<kAttnWarps, kAttnStages, 2, false, 1>, grid, block, smem, s, a.pdl, L, a);
    default: return launch_maybe_pdl(attention_kernel<kAttnWarps, kAttnStages, 4, false, 1>, grid, block, smem, s, a.pdl, L, a);
    }
}

}  // namespace macgpu
