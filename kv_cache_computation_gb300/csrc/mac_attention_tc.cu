// sm_103a split-KV attention for 32-head groups (MQA-shaped GQA) on the
// 5th-generation tensor cores: tcgen05.mma with operands in shared memory and
// accumulators in tensor memory (Complete, Figure 2(b) of the MAC-Attention
// paper; the plan is the span-proportional one of Figure 3(b), made in every
// CTA's prologue as in the mma.sync kernel).
//
// One CTA of 4 warps per SM.  The KV stream is cut into blocks of 64 tokens
// (4 pages), staged by cp.async into shared memory in the 128-byte swizzled
// layout the tensor core reads: rows of 128 bytes, the 16-byte chunk c of
// row t at position c ^ (t mod 8), a 64-element column block per 8 KB.  Per
// block, one thread issues
//   S[128 x 64]  = Qr[128 x 128] K^T          (8 mma, M 128, N 64, K 16)
//   O[128 x 128] += P_hi[128 x 64] V + P_lo V  (8 mma, M 128, N 128; V is read
//                                                MN-major: tokens are its K)
// where Qr holds the group's 32 query heads four times (row 32 w + h is head
// h): warp w reads its own 32 TMEM lanes of S, i.e. all 32 heads, and does the
// softmax of the block's tokens 16 w .. 16 w + 15 with one thread per head --
// no cross-lane reduction.  Its P row carries those 16 tokens and zeros
// elsewhere, so O row 32 w + h accumulates head h over token quarter w with
// its own softmax reference; the four quarters of a head are merged when the
// item ends.  The reference of a row moves only when a block passes it by
// more than 2^8 (then the row of O is rescaled in tensor memory).
//
// Every wait on an mbarrier has an iteration limit; on expiry the kernel sets
// kErrTimeout, drains its copies, frees its tensor memory and returns.
#include "mac_plan.cuh"

namespace macgpu {

namespace {

constexpr int kTcTok = 64;                         // tokens per block (4 pages)
constexpr int kTcThreads = 128;
constexpr int kTcQBytes = 2 * 128 * 128;           // Qr: 2 column blocks x 128 rows x 128 B
constexpr int kTcPBytes = 128 * 128;               // one P part (hi or lo): 128 rows x 64 tokens x 2 B
constexpr int kTcStageBytes = 2 * 2 * kTcTok * 128;   // K and V blocks: 2 column blocks x 64 rows x 128 B each
constexpr int kTcTmemCols = 256;                   // S at column 0 (64 columns), O at column 128 (128 columns)
constexpr uint32_t kTcSpinLimit = 1u << 22;

// instruction descriptors (kind::f16): D f32, A and B bf16; N >> 3 at bit 17, M >> 4 at bit 24
constexpr uint32_t kIdescS = (1u << 4) | (1u << 7) | (1u << 10) | ((64u >> 3) << 17) | ((128u >> 4) << 24);
constexpr uint32_t kIdescO = (1u << 4) | (1u << 7) | (1u << 10) | (1u << 16) | ((128u >> 3) << 17) | ((128u >> 4) << 24);

// Shared-memory matrix descriptor, 128-byte swizzle: start address, leading
// and stride byte offsets (all >> 4), version 1, layout type 2.
__device__ __forceinline__ uint64_t tc_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo)
{
    return (uint64_t)((saddr >> 4) & 0x3FFF) | ((uint64_t)((lbo >> 4) & 0x3FFF) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFF) << 32) | ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t acc)
{
    asm volatile("{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
                 "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n"
                 :: "r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(acc)
                 : "memory");
}

__device__ __forceinline__ void tc_commit(uint32_t mbar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" :: "r"(mbar)
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory"); }
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory"); }

__device__ __forceinline__ void mbar_init(uint32_t mbar)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;\n" :: "r"(mbar) : "memory");
}

// Waits until the phase of the given parity has completed; false after the
// iteration limit.
__device__ __forceinline__ bool mbar_wait(uint32_t mbar, uint32_t parity)
{
    for (uint32_t i = 0; i < kTcSpinLimit; i++) {
        uint32_t ok;
        asm volatile("{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\nselp.u32 %0, 1, 0, p;\n}\n"
                     : "=r"(ok)
                     : "r"(mbar), "r"(parity)
                     : "memory");
        if (ok) return true;
    }
    return false;
}

// 32 lanes x 16 / 32 consecutive 32-bit columns of tensor memory, one lane per thread
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16])
{
    uint32_t r[16];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
                   "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
                 : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
#pragma unroll
    for (int i = 0; i < 16; i++) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32])
{
    uint32_t r[32];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
                 "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
                   "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
                   "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
                   "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
                 : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; i++) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float (&v)[32])
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
                 "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};\n"
                 :: "r"(taddr), "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
                    "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
                    "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
                    "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
                    "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
                    "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])),
                    "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])), "r"(__float_as_uint(v[20])),
                    "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
                    "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])),
                    "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])),
                    "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
                 : "memory");
    asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory");
}

// byte offset of the 16-byte chunk c (0..15) of row t in a swizzled tile of
// `rows` rows: column block c / 8 is rows x 128 bytes
__device__ __forceinline__ uint32_t sw128(int rows, int t, int c)
{
    return (uint32_t)((c >> 3) * rows * 128 + t * 128 + (((c & 7) ^ (t & 7)) << 4));
}

template <int S>
__global__ void __launch_bounds__(kTcThreads, 1) attention_tc_kernel(Layout L, StepArgs a)
{
    extern __shared__ __align__(1024) uint8_t tc_smem_raw[];
    uint8_t *sbase = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(tc_smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *sQ = sbase;                                   // Qr
    uint8_t *sP = sbase + kTcQBytes;                       // P hi, then P lo
    uint8_t *sStage = sbase + kTcQBytes + 2 * kTcPBytes;   // S stages: K block, then V block
    __shared__ PlanShared ps;
    __shared__ __align__(8) uint64_t mbar_s, mbar_o;
    __shared__ uint32_t s_tmem;
    __shared__ long long s_pgoff[kTcStages][4];   // element offsets of a block's pages (-1: past the item or refused)
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const float sl2 = L.scale_log2;
    const uint32_t mb_s = smem_u32(&mbar_s), mb_o = smem_u32(&mbar_o);
    const uint32_t sQ_u = smem_u32(sQ), sP_u = smem_u32(sP), sStage_u = smem_u32(sStage);

    pdl_launch_dependents();
    // warm L2 with the first pages of the item this CTA streamed in the
    // previous step (a hint; every index is bounds-checked)
    if (tid == 0 && blockIdx.x < L.item_cap) {
        const int4 prev = L.items[blockIdx.x];
        if (prev.x >= 0 && prev.x < a.batch * L.Hkv && prev.y >= 0 && prev.y < prev.z) {
            const int pb = prev.x / L.Hkv, pgrp = prev.x - pb * L.Hkv;
            for (int k = 0; k < 4 * kSpeculativePages; k++) {
                const int pg = (prev.y >> 4) + k;
                if (pg * 16 >= prev.z) break;
                bool ok = true;
                const size_t off = kv_block(L, pb, pgrp, pg, ok);
                if (!ok) break;
                prefetch_l2_bulk(L.k_pool + off, 4096);
                prefetch_l2_bulk(L.v_pool + off, 4096);
            }
        }
    }
    // P rows are zero outside their own token quarter: clear both parts once
    for (int i = tid; i < 2 * kTcPBytes / 16; i += kTcThreads)
        reinterpret_cast<uint4 *>(sP)[i] = make_uint4(0u, 0u, 0u, 0u);
    if (tid == 0) {
        mbar_init(mb_s);
        mbar_init(mb_o);
        asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n"
                     :: "r"(smem_u32(&s_tmem)), "r"(kTcTmemCols) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem;
    const uint32_t t_s = tmem, t_o = tmem + 128;                 // S columns 0..63, O columns 128..255
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;      // this warp's TMEM lanes

    pdl_wait();   // spans come from match_plan
    cta_plan(L, a, ps);
    const int nbg = a.batch * L.Hkv;
    const int n_items = ps.total;
    if (blockIdx.x == 0) {   // publish the plan for combine and the counters
        for (int i = tid; i <= nbg; i += blockDim.x) L.grp_item_off[i] = min(ps.off[i], n_items);
        for (int i = tid; i < n_items; i += blockDim.x) L.items[i] = plan_item(L, a, ps, nbg, i);
        if (tid == 0) {
            *L.n_items = n_items;
            if (ps.off[nbg] > L.item_cap) atomicOr(L.err, kErrPos);
            atomicAdd(&L.stats[kStSteps], 1ull);
            atomicAdd(&L.stats[kStKvRead], (unsigned long long)ps.T);
            atomicAdd(&L.stats[kStKvFull], (unsigned long long)ps.Tf);
            atomicAdd(&L.stats[kStItems], (unsigned long long)n_items);
            if (!a.full_mode) atomicAdd(&L.stats[kStDecisions], (unsigned long long)a.batch * L.H);
        }
    }

    uint32_t n_s = 0, n_o = 0;   // completions waited on each barrier
    bool fail = false;
    for (int it = blockIdx.x; it < n_items && !fail; it += gridDim.x) {
        const int4 item = plan_item(L, a, ps, nbg, it);
        const int bg = item.x, ilo = item.y, ihi = item.z;
        const int b = bg / L.Hkv, g = bg - b * L.Hkv;
        const int glo = ps.lo[bg], ghi = ps.hi[bg], gsp = plan_split(L, a, glo, ghi);
        const int slo = item.w ? gsp : glo;   // the item's segment starts here
        const size_t hrow = (size_t)b * L.H + (size_t)g * L.G;
        // this thread's head is `lane`; its tokens in this item are [lo_i, ihi)
        // (the last block's pages past the item are zero-filled and masked)
        const int lo_i = max(max(slo, ilo), L.dec_lo[hrow + lane]);

        // Qr: row r is head r mod 32
        for (int i = tid; i < 128 * 16; i += kTcThreads) {
            const int r = i >> 4, c = i & 15;
            const uint4 v = reinterpret_cast<const uint4 *>(a.q_post + (hrow + (r & 31)) * kD)[c];
            *reinterpret_cast<uint4 *>(sQ + sw128(128, r, c)) = v;
        }
        fence_async_smem();

        const int pg0 = ilo >> 4, npg = ((ihi - 1) >> 4) - pg0 + 1;
        const int nblk = (npg + 3) >> 2;
        // page-table lookup of page p of block j into s_pgoff[j % S][p] (one thread per page)
        auto lookup = [&](int j, int p) {
            long long o = -1;
            if (j < nblk && 4 * j + p < npg) {
                bool ok = true;
                const size_t off = kv_block(L, b, g, pg0 + 4 * j + p, ok);
                if (ok) o = (long long)off;
                else atomicOr(L.err, kErrPage);
            }
            s_pgoff[j % S][p] = o;
        };
        // block j into stage j % S: 4 pages x (K 256 + V 256 chunks), 16 chunks per
        // thread (chunks 4 p .. 4 p + 3 of a thread lie in page p); pages past the
        // item and value rows past its end are zero-filled
        auto issue_block = [&](int j) {
            uint8_t *sk = sStage + (j % S) * kTcStageBytes;
#pragma unroll
            for (int u = 0; u < 16; u++) {
                const int q = tid + kTcThreads * u;
                const int p = q >> 9, rem = q & 511, isv = rem >> 8, tp = (rem >> 4) & 15, c = rem & 15;
                const long long po = s_pgoff[j % S][p];
                const int t = 16 * p + tp;
                const bool valid = po >= 0 && (!isv || (pg0 + 4 * j + p) * 16 + tp < ihi);
                const __nv_bfloat16 *src = (isv ? L.v_pool : L.k_pool) + (po >= 0 ? po : 0) + (size_t)tp * kD + c * 8;
                cp_async16_zfill(smem_u32(sk + isv * (kTcStageBytes / 2) + sw128(kTcTok, t, c)), src, valid ? 16u : 0u);
            }
        };
        if (tid < 4 * S) lookup(tid >> 2, tid & 3);   // blocks 0 .. S - 1
        __syncthreads();
#pragma unroll
        for (int j = 0; j < S - 1; j++) {
            if (j < nblk) issue_block(j);
            cp_async_commit();
        }

        float m = -CUDART_INF_F, up = -CUDART_INF_F, l = 0.f;   // this row's softmax state (log2 units)
        for (int j = 0; j < nblk; j++) {
            cp_async_wait<S - 2>();
            fence_async_smem();
            __syncthreads();   // block j staged; every thread done with block j - 1
            if (j + S - 1 < nblk) issue_block(j + S - 1);
            cp_async_commit();
            // the next block to issue (j + S) reuses block j's offsets slot; its
            // lookups land while this block is computed
            if (tid < 4 && j + S < nblk) lookup(j + S, tid);
            const uint32_t stK = sStage_u + (j % S) * kTcStageBytes, stV = stK + kTcStageBytes / 2;
            if (tid == 0) {
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 8; kk++)
                    tc_mma(t_s, tc_desc(sQ_u + (kk >> 2) * (128 * 128) + (kk & 3) * 32, 16, 1024),
                           tc_desc(stK + (kk >> 2) * (kTcTok * 128) + (kk & 3) * 32, 16, 1024), kIdescS, kk > 0);
                tc_commit(mb_s);
            }
            if (__syncthreads_or(!mbar_wait(mb_s, n_s & 1))) {   // uniform across the block
                fail = true;
                break;
            }
            n_s++;
            tc_fence_after();
            // scores of head `lane`, tokens 16 warp .. 16 warp + 15 of the block
            float z[16];
            tmem_ld16(t_s + lane_base + 16 * warp, z);
            const int t0 = (pg0 + 4 * j) * 16 + 16 * warp;
            if (t0 < lo_i || t0 + 16 > ihi) {
#pragma unroll
                for (int e = 0; e < 16; e++)
                    if (!(t0 + e >= lo_i && t0 + e < ihi)) z[e] = -CUDART_INF_F;
            }
            float mx = z[0];
#pragma unroll
            for (int e = 1; e < 16; e++) mx = fmaxf(mx, z[e]);
            // the reference of a row moves when the block passes it: its sums are
            // rescaled (the row of O only once it holds data; the tensor-memory
            // accesses are warp-wide, so every lane takes part, with factor 1
            // where its row did not move)
            const bool move = mx > up;
            if (__any_sync(0xffffffffu, move)) {
                const float mn = move ? mx * sl2 : m;
                const float al = move ? ex2_approx(m - mn) : 1.f;
                l *= al;
                if (j > 0) {
#pragma unroll 1
                    for (int cb = 0; cb < 128; cb += 32) {
                        float o[32];
                        tmem_ld32(t_o + lane_base + cb, o);
#pragma unroll
                        for (int i = 0; i < 32; i++) o[i] *= al;
                        tmem_st32(t_o + lane_base + cb, o);
                    }
                }
                if (move) {
                    m = mn;
                    up = (m + kLazyMax) / sl2;
                }
            }
            const float nb = m == -CUDART_INF_F ? 0.f : -m;
            uint32_t ph[8], pl[8];
#pragma unroll
            for (int e = 0; e < 16; e += 2) {
                const float p0 = ex2_approx(fmaf(z[e], sl2, nb)), p1 = ex2_approx(fmaf(z[e + 1], sl2, nb));
                l += p0 + p1;
                const __nv_bfloat162 hv = __floats2bfloat162_rn(p0, p1);
                const float2 fv = __bfloat1622float2(hv);
                ph[e >> 1] = bf16x2_bits(hv);
                pl[e >> 1] = bf16x2_bits(__floats2bfloat162_rn(p0 - fv.x, p1 - fv.y));
            }
            // row tid of P: tokens 16 warp .. + 15 are chunks 2 warp, 2 warp + 1
            {
                const uint32_t c0 = (uint32_t)(((2 * warp) ^ (tid & 7)) << 4), c1 = (uint32_t)(((2 * warp + 1) ^ (tid & 7)) << 4);
                uint8_t *rowh = sP + tid * 128, *rowl = sP + kTcPBytes + tid * 128;
                *reinterpret_cast<uint4 *>(rowh + c0) = make_uint4(ph[0], ph[1], ph[2], ph[3]);
                *reinterpret_cast<uint4 *>(rowh + c1) = make_uint4(ph[4], ph[5], ph[6], ph[7]);
                *reinterpret_cast<uint4 *>(rowl + c0) = make_uint4(pl[0], pl[1], pl[2], pl[3]);
                *reinterpret_cast<uint4 *>(rowl + c1) = make_uint4(pl[4], pl[5], pl[6], pl[7]);
            }
            fence_async_smem();
            tc_fence_before();
            __syncthreads();
            if (tid == 0) {
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 4; kk++)
                    tc_mma(t_o, tc_desc(sP_u + kk * 32, 16, 1024), tc_desc(stV + kk * 2048, 8192, 1024), kIdescO,
                           (j > 0 || kk > 0) ? 1u : 0u);
#pragma unroll
                for (int kk = 0; kk < 4; kk++)
                    tc_mma(t_o, tc_desc(sP_u + kTcPBytes + kk * 32, 16, 1024), tc_desc(stV + kk * 2048, 8192, 1024),
                           kIdescO, 1u);
                tc_commit(mb_o);
            }
            if (__syncthreads_or(!mbar_wait(mb_o, n_o & 1))) {
                fail = true;
                break;
            }
            n_o++;
            tc_fence_after();
        }
        if (fail) break;

        // merge the four token quarters of each head: rows h, 32 + h, 64 + h,
        // 96 + h of O, through the (drained) stage buffers
        cp_async_wait<0>();
        __syncthreads();
        float *ex_o = reinterpret_cast<float *>(sStage);                  // [4][32][128]
        float2 *ex_ml = reinterpret_cast<float2 *>(sStage + 4 * 32 * 128 * 4);   // [4][32]
#pragma unroll 1
        for (int cb = 0; cb < 128; cb += 32) {
            float o[32];
            tmem_ld32(t_o + lane_base + cb, o);
            float4 *dst = reinterpret_cast<float4 *>(ex_o + ((size_t)warp * 32 + lane) * kD + cb);
#pragma unroll
            for (int i = 0; i < 8; i++) dst[i] = make_float4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
        }
        ex_ml[warp * 32 + lane] = make_float2(m, l);
        tc_fence_before();
        __syncthreads();
        for (int idx = tid; idx < 32 * kD; idx += kTcThreads) {
            const int hh = idx >> 7, dd = idx & 127;
            float M = -CUDART_INF_F;
#pragma unroll
            for (int q = 0; q < 4; q++) M = fmaxf(M, ex_ml[q * 32 + hh].x);
            float lsum = 0.f, osum = 0.f;
            if (M != -CUDART_INF_F) {
#pragma unroll
                for (int q = 0; q < 4; q++) {
                    const float2 ml = ex_ml[q * 32 + hh];
                    const float wq = ex2_approx(ml.x - M);
                    lsum += ml.y * wq;
                    osum += ex_o[((size_t)q * 32 + hh) * kD + dd] * wq;
                }
            }
            L.part_o[((size_t)it * L.G + hh) * kD + dd] = osum;
            if (dd == 0) L.part_ml[(size_t)it * L.G + hh] = make_float2(M, lsum);
        }
        __syncthreads();   // the stage buffers take the next item's blocks
        tc_fence_after();
    }
    if (fail && tid == 0) atomicOr(L.err, kErrTimeout);
    cp_async_wait<0>();
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" :: "r"(tmem), "r"(kTcTmemCols) : "memory");
    }
}

size_t attention_tc_smem() { return 1024 + kTcQBytes + 2 * kTcPBytes + (size_t)kTcStages * kTcStageBytes; }

}  // namespace

cudaError_t attention_tc_config(size_t *smem, int *ctas_per_sm)
{
    *smem = attention_tc_smem();
    auto k = attention_tc_kernel<kTcStages>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)*smem);
    if (e != cudaSuccess) return e;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(ctas_per_sm, k, kTcThreads, *smem);
}

cudaError_t launch_attention_tc(const Layout &L, const StepArgs &a, size_t smem, cudaStream_t s)
{
    return launch_maybe_pdl(attention_tc_kernel<kTcStages>, dim3(a.grid_ctas), dim3(kTcThreads), smem, s, a.pdl, L, a);
}

}  // namespace macgpu
