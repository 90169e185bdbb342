// sm_103a kernels of the MAC-Attention decode step other than the split-KV
// attention (which, with its planner, is in mac_attention.cu).
//
// A decode step is three launches on the critical path, chained by
// programmatic dependent launch:
//   match_plan  KV append of the new token; Match of each query head's
//               pre-RoPE query against its ring (Figure 2(a) of the
//               MAC-Attention paper); per-group band+tail span starts.
//               Rings longer than 32 entries are scanned first by
//               ring_scan, a grid-wide kernel.
//   attention   persistent split-KV attention (Figure 2(b), Complete) over
//               the work list every CTA plans in its prologue (Figure 3(b)).
//   combine     log-domain merge of the partials and, on a hit, of the
//               reused AS_{1:p-r} from the ring (Figure 2(b)); its epilogue
//               runs Amend's removal and ring insert (Figure 2(c)) unless
//   amend       recomputes the band on a side stream instead.
//
// Conventions: token index j (0-based) is the paper's position j+1; ranges
// [lo, hi) are half-open over indices.  Scores are kept in log2 units
// (scaled by sm_scale * log2 e) inside the kernels; summaries that leave the
// kernels (ring, lse_out) use natural-log units.
#include "mac_device.cuh"

namespace macgpu {

namespace {

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
// NW warps per block: kCombineWarps, or one warp taking every item in one
// round when each head has a handful of items (many requests, where the
// grid is thousands of blocks).
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
    float2 ml_band = make_float2(NEG, 0.f);
    float4 o_band = make_float4(0.f, 0.f, 0.f, 0.f);
    int m = 0, slot = 0;
    if (!a.full_mode && w == 0) {
        // the group's band item (item bg of a MAC step's plan) seeds the band sums
        ml_band = L.part_ml[(size_t)bg * L.G + hh];
        o_band = *reinterpret_cast<const float4 *>(L.part_o + ((size_t)bg * L.G + hh) * kD + 4 * lane);
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
    // One pass: each warp merges the group's long-segment items w, w + NW, ...
    // online, rescaling its sums when a batch raises a maximum; a
    // shared-memory step then merges the warps.  The band (segment 1) is
    // the single item bg, which seeds warp 0's band sums.
    float mp = NEG, mb = NEG, lp = 0.f, lb = 0.f;
    float4 op = make_float4(0.f, 0.f, 0.f, 0.f), ob = op;
    if (w == 0 && m_ring != NEG) {   // the reused AS_{1:p-r}: weight 1 at its own maximum
        mp = m_ring;
        lp = 1.f;
        op = o_ring;
    }
    if (w == 0 && ml_band.x != NEG) {
        mb = ml_band.x;
        lb = ml_band.y;
        ob = o_band;
    }
    constexpr int kBatch = KB;
    for (int i0 = off0 + w; i0 < off1; i0 += kBatch * NW) {
        float2 ml[kBatch];
        float4 ov[kBatch];
#pragma unroll
        for (int k = 0; k < kBatch; k++) {
            const int i = min(i0 + k * NW, off1 - 1);
            ml[k] = L.part_ml[(size_t)i * L.G + hh];
            ov[k] = *reinterpret_cast<const float4 *>(L.part_o + ((size_t)i * L.G + hh) * kD + 4 * lane);
            if (i0 + k * NW >= off1) ml[k].x = NEG;   // padding slot
        }
        float np = mp;
#pragma unroll
        for (int k = 0; k < kBatch; k++) np = fmaxf(np, ml[k].x);
        if (np != mp) {
            const float r = mp == NEG ? 0.f : exp2f(mp - np);
            lp *= r;
            op = scale4(op, r);
            mp = np;
        }
#pragma unroll
        for (int k = 0; k < kBatch; k++) {
            if (ml[k].x == NEG) continue;
            const float wi = exp2f(ml[k].x - mp);
            lp = fmaf(ml[k].y, wi, lp);
            fma4(op, wi, ov[k]);
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
        __shared__ long long s_page[kBandTile / kPage + 1];   // element offset of each page of a tile (-1: refused)
        for (int t0 = m - r; t0 < m; t0 += kBandTile) {
            const int n = min(kBandTile, m - t0);
            const int p_first = t0 >> 4, npages = ((t0 + n - 1) >> 4) - p_first + 1;
            __syncthreads();   // previous tile consumed
            if ((int)threadIdx.x < npages) {   // one page-table lookup per page of the tile
                bool okp = true;
                const size_t o = kv_block(L, b, g, p_first + threadIdx.x, okp);
                s_page[threadIdx.x] = okp ? (long long)o : -1ll;
            }
            __syncthreads();
            // 16-byte chunks c = token * 32 + part (parts 0-15 K, 16-31 V): each
            // thread issues eight loads before it stores any of them
            const int total = n * 32;
            for (int c0 = threadIdx.x; c0 < total; c0 += 8 * blockDim.x) {
                uint4 v[8];
                int dst[8];
#pragma unroll
                for (int u = 0; u < 8; u++) {
                    const int c = c0 + u * blockDim.x;
                    dst[u] = -1;
                    if (c < total) {
                        const int tok = c >> 5, part = c & 31, isv = part >> 4, ch = part & 15;
                        const int j = t0 + tok;
                        const long long po = s_page[(j >> 4) - p_first];
                        if (po < 0) {
                            ok = false;
                        } else {
                            v[u] = reinterpret_cast<const uint4 *>((isv ? L.v_pool : L.k_pool) + po +
                                                                   (size_t)(j & 15) * kD)[ch];
                            dst[u] = (isv ? kBandTile * kBandRow : 0) + tok * kBandRow + ch * 16;
                        }
                    }
                }
#pragma unroll
                for (int u = 0; u < 8; u++)
                    if (dst[u] >= 0) *reinterpret_cast<uint4 *>(band_smem + dst[u]) = v[u];
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

cudaError_t launch_combine(const Layout &L, const StepArgs &a, cudaStream_t s)
{
    // a group holds at most about plan slots / groups + 2 items
    const int nbg = a.batch * L.Hkv;
    const int per_group = (a.plan_ctas + nbg - 1) / nbg + 2;
    const dim3 grid(a.batch * L.H);
    // A few items per head (many requests): small blocks, so that the whole
    // grid is resident beside the attention CTAs when their wait releases.
    if (per_group <= 8) return launch_maybe_pdl(combine_kernel<8, 1>, grid, dim3(32), 0, s, a.pdl != 0, L, a);
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
