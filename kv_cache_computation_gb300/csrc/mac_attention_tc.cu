// sm_103a split-KV attention for 32-head groups (MQA-shaped GQA) on the
// 5th-generation tensor cores: tcgen05.mma with operands in shared memory and
// accumulators in tensor memory (Complete, Figure 2(b) of the MAC-Attention
// paper; the plan is the span-proportional one of Figure 3(b), made in every
// CTA's prologue as in the mma.sync kernel).
//
// One CTA of 11 warps per SM, for steps of at least 16384 KV tokens (the host
// picks this kernel or the mma.sync one per step).  The KV stream is cut into
// blocks of 128 tokens (8 pages); a block's keys and its values go through
// rings of their own in shared memory (kTcKStages and kTcVStages blocks), each
// filled by TMA from a loader warp of its own (two 16-row x 64-column boxes per
// page) in the 128-byte swizzled layout the tensor core reads: rows of 128
// bytes, the 16-byte chunk c of row t at c ^ (t mod 8), a 64-element column
// block per 16 KB.  Tokens are the M of both products and the group's 32 heads
// their N, so no work is spent on padding:
//   S^T[128 x 32]  = K[128 x 128] Q^T                 (8 mma, M 128, N 32, K 16)
//   O^T[128 x 64] += V^T[128 x 128] [P_hi P_lo]^T      (8 mma, M 128, N 64; V is
//                                                     read MN-major)
// issued by one thread of a warp of its own.  Softmax thread (t, w / 4) of
// warp w owns token row t of S^T (TMEM lane t) for kTcHalf heads.  All threads
// keep one softmax reference per head, which moves only when a block passes it
// by more than 2^8; the threads agree on the moves of a block through shared
// memory and a bounded mbarrier, and a move rescales O^T in tensor memory
// (thread d holds row d: head h in columns h and 32 + h).  P is kept as a bf16
// pair (hi, lo) per head, so the product P V keeps about 16 bits of P.  Each
// thread sums its own token's P per head; the 128 partial sums of a head are
// added when the item ends.  The roles walk the CTA's items independently, so
// the next item's copies and score products overlap the current item's merge.
//
// Every wait on an mbarrier has an iteration limit; on expiry the kernel sets
// kErrTimeout, lets its copies land, frees its tensor memory and returns.
#include "mac_plan.cuh"

#include <climits>
#include <cudaTypedefs.h>

namespace macgpu {

namespace {

constexpr int kTcTok = 128;                        // tokens per block (8 pages): the M of the score product
constexpr int kTcHeads = 32;                       // query heads of the group: the N of the score product
#ifndef MAC_TC_SOFTMAX_WARPS
#define MAC_TC_SOFTMAX_WARPS 8
#endif
constexpr int kTcSoftmaxWarps = MAC_TC_SOFTMAX_WARPS;   // warp w: TMEM lanes 32 (w mod 4) .., heads kTcHalf (w / 4) ..
constexpr int kTcHalf = kTcHeads * 4 / kTcSoftmaxWarps; // heads per softmax thread (8 or 16)
static_assert(kTcHalf == 8 || kTcHalf == 16, "8 or 16 softmax warps");
constexpr int kTcKStages = MAC_TC_K_STAGES;        // key blocks in the ring
constexpr int kTcVStages = MAC_TC_V_STAGES;        // value blocks in the ring
constexpr int kTcKWarp = kTcSoftmaxWarps, kTcVWarp = kTcKWarp + 1, kTcMmaWarp = kTcVWarp + 1;
constexpr int kTcThreads = (kTcMmaWarp + 1) * 32;
constexpr int kTcQBytes = 2 * kTcHeads * 128;      // Q: 2 column blocks x 32 rows x 128 B
constexpr int kTcPBytes = kTcTok * 128;            // P^T: 128 token rows x (32 hi + 32 lo) bf16; two buffers
constexpr int kTcBlockBytes = 2 * kTcTok * 128;    // a key (or value) block: 2 column blocks x 128 rows x 128 B
constexpr int kTcTmemCols = 128;                   // S^T buffers at columns 0 and 32, O^T at 64 .. 127
constexpr uint32_t kTcSpinLimit = 1u << 22;

// instruction descriptors (kind::f16): D f32, A and B bf16, bit 15 / 16: A / B
// MN-major; N >> 3 at bit 17, M >> 4 at bit 24
constexpr uint32_t kIdescS = (1u << 4) | (1u << 7) | (1u << 10) | ((32u >> 3) << 17) | ((128u >> 4) << 24);
constexpr uint32_t kIdescO =
    (1u << 4) | (1u << 7) | (1u << 10) | (1u << 15) | (1u << 16) | ((64u >> 3) << 17) | ((128u >> 4) << 24);

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

__device__ __forceinline__ void mbar_init(uint32_t mbar, int count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" :: "r"(mbar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t mbar)
{
    asm volatile("{\n.reg .b64 st;\nmbarrier.arrive.shared::cta.b64 st, [%0];\n}\n" :: "r"(mbar) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t mbar, uint32_t bytes)
{
    asm volatile("{\n.reg .b64 st;\nmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n}\n" :: "r"(mbar), "r"(bytes)
                 : "memory");
}

// 2-D tiled TMA load of the box at (x, y) of a tensor map into shared
// memory, completing bytes on the mbarrier.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int x, int y, uint32_t mbar)
{
    asm volatile("cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];\n"
                 :: "r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(mbar)
                 : "memory");
}

// Non-blocking test of the phase of the given parity.
__device__ __forceinline__ bool mbar_test(uint32_t mbar, uint32_t parity)
{
    uint32_t ok;
    asm volatile("{\n.reg .pred p;\nmbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\nselp.u32 %0, 1, 0, p;\n}\n"
                 : "=r"(ok)
                 : "r"(mbar), "r"(parity)
                 : "memory");
    return ok != 0;
}

// Bounded wait that does not give up when another role fails (for the
// copies and products in flight when the CTA winds down).
__device__ __forceinline__ void mbar_wait_bounded(uint32_t mbar, uint32_t parity)
{
    for (uint32_t i = 0; i < kTcSpinLimit; i++)
        if (mbar_test(mbar, parity)) return;
}

// Bounded wait that also gives up once another role has failed.  The lanes
// of a warp run it in step on the same barrier word and the same flag, so
// they leave it together with the same outcome before any warp-wide
// instruction that follows.
__device__ __forceinline__ bool mbar_wait_or_fail(uint32_t mbar, uint32_t parity, volatile int *fail)
{
    for (uint32_t i = 0; i < kTcSpinLimit; i++) {
        uint32_t ok;
        asm volatile("{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\nselp.u32 %0, 1, 0, p;\n}\n"
                     : "=r"(ok)
                     : "r"(mbar), "r"(parity)
                     : "memory");
        if (ok) return true;
        if ((i & 255) == 255 && *fail) return false;
    }
    *fail = 1;
    return false;
}


// byte offset of the 16-byte chunk c (0..15) of row t in a swizzled tile of
// `rows` rows: column block c / 8 is rows x 128 bytes
__device__ __forceinline__ uint32_t sw128(int rows, int t, int c)
{
    return (uint32_t)((c >> 3) * rows * 128 + t * 128 + (((c & 7) ^ (t & 7)) << 4));
}

// 32 lanes x N (8 or 16) consecutive 32-bit columns of tensor memory, one
// lane per thread; the load waits for its data, the store for its completion
template <int N>
__device__ __forceinline__ void tmem_ld(uint32_t taddr, float (&v)[N])
{
    static_assert(N == 8 || N == 16, "8 or 16 columns");
    uint32_t r[N];
    if constexpr (N == 8) {
        asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];\n"
                     : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
                     : "r"(taddr));
    } else {
        asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n"
                     : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
                       "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
                     : "r"(taddr));
    }
    asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
#pragma unroll
    for (int i = 0; i < N; i++) v[i] = __uint_as_float(r[i]);
}

template <int N>
__device__ __forceinline__ void tmem_st(uint32_t taddr, const float (&v)[N])
{
    static_assert(N == 8 || N == 16, "8 or 16 columns");
    uint32_t r[N];
#pragma unroll
    for (int i = 0; i < N; i++) r[i] = __float_as_uint(v[i]);
    if constexpr (N == 8) {
        asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};\n"
                     :: "r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
                     : "memory");
    } else {
        asm volatile("tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};\n"
                     :: "r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
                        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
                     : "memory");
    }
    asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory");
}

// order-preserving map of a float to an int (for atomicMax) and back
__device__ __forceinline__ int ord_key(float f)
{
    const int i = __float_as_int(f);
    return i >= 0 ? i : i ^ 0x7fffffff;
}
__device__ __forceinline__ float ord_val(int k) { return __int_as_float(k >= 0 ? k : k ^ 0x7fffffff); }

// Roles: warps 0 .. kTcSoftmaxWarps - 1 softmax (warp w: TMEM lanes
// 32 (w mod 4) .. + 31, i.e. token rows of S^T and rows of O^T, for heads
// kTcHalf (w / 4) .. + kTcHalf - 1), warp kTcKWarp / kTcVWarp loads the key /
// value blocks by TMA, warp kTcMmaWarp issues the tensor-core work.  Barriers:
// kfull / vfull (a stage's bytes landed), kempty / vempty (the block's score /
// P V product done), sfull / sempty and pfull / pempty per S^T and P buffer,
// mv (the softmax threads' agreement on a block's moves), qfull (an item's Q
// stored), red (the merge's partial sums stored), oempty (O^T read by the
// merge), done (every product issued complete).  Completion k of a barrier is
// awaited with parity k & 1; every role waits each completion in order, so no
// barrier runs two phases ahead of a waiter.
template <int KS, int VS>
__global__ void __launch_bounds__(kTcThreads, 1) attention_tc_kernel(const __grid_constant__ Layout L, StepArgs a, const __grid_constant__ TcMaps M)
{
    extern __shared__ __align__(1024) uint8_t tc_smem_raw[];
    uint8_t *sbase = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(tc_smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *sQ = sbase;                          // Q, K-major
    uint8_t *sP = sQ + kTcQBytes;                 // two P^T buffers, MN-major
    uint8_t *sK = sP + 2 * kTcPBytes;             // KS key blocks
    uint8_t *sV = sK + KS * kTcBlockBytes;        // VS value blocks
    __shared__ PlanShared ps;
    __shared__ __align__(8) uint64_t bar_kfull[KS], bar_kempty[KS], bar_vfull[VS], bar_vempty[VS];
    __shared__ __align__(8) uint64_t bar_sfull[2], bar_sempty[2], bar_pfull[2], bar_pempty[2], bar_mv;
    __shared__ __align__(8) uint64_t bar_qfull, bar_red, bar_oempty, bar_done;
    __shared__ uint32_t s_tmem;
    __shared__ int s_fail;
    __shared__ uint32_t s_any[3];        // heads whose reference a block moves (three blocks in turn)
    __shared__ int s_ref[3][kTcHeads];   // their new references (ord_key of the block maximum)
    __shared__ int s_lo[kTcHeads];       // first token each head reads in the item
    __shared__ float s_m[kTcHeads];
    __shared__ float s_l[4][kTcHeads];   // per head, the sums of P of the four token quarters
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const float sl2 = L.scale_log2;
    volatile int *fail = &s_fail;
    const uint32_t sQ_u = smem_u32(sQ), sP_u = smem_u32(sP), sK_u = smem_u32(sK), sV_u = smem_u32(sV);
    auto B_ = [](uint64_t &b) { return smem_u32(&b); };

    pdl_launch_dependents();
    if (tid == kTcKWarp * 32 && blockIdx.x < L.item_cap) {
        // warm L2 with the first pages of the item this CTA streamed in the
        // previous step (a hint; every index is bounds-checked)
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
    if (tid == 0) {
        for (int i = 0; i < KS; i++) {
            mbar_init(B_(bar_kfull[i]), 1);
            mbar_init(B_(bar_kempty[i]), 1);
        }
        for (int i = 0; i < VS; i++) {
            mbar_init(B_(bar_vfull[i]), 1);
            mbar_init(B_(bar_vempty[i]), 1);
        }
        for (int i = 0; i < 2; i++) {
            mbar_init(B_(bar_sfull[i]), 1);
            mbar_init(B_(bar_sempty[i]), kTcSoftmaxWarps * 32);
            mbar_init(B_(bar_pfull[i]), kTcSoftmaxWarps * 32);
            mbar_init(B_(bar_pempty[i]), 1);
        }
        mbar_init(B_(bar_mv), kTcSoftmaxWarps * 32);
        mbar_init(B_(bar_qfull), kTcSoftmaxWarps * 32);
        mbar_init(B_(bar_red), kTcSoftmaxWarps * 32);
        mbar_init(B_(bar_oempty), kTcSoftmaxWarps * 32);
        mbar_init(B_(bar_done), 1);
        asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
        s_fail = 0;
    }
    if (tid < 3 * kTcHeads) s_ref[tid / kTcHeads][tid % kTcHeads] = INT_MIN;
    if (tid < 3) s_any[tid] = 0u;
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n"
                     :: "r"(smem_u32(&s_tmem)), "r"(kTcTmemCols) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem;
    const uint32_t t_s = tmem, t_o = tmem + 64;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;

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

    // Each role walks the CTA's items on its own; the loads of an item start
    // while the softmax warps still finish the one before.  Barrier
    // completions count blocks (jbase + j) or items (k) of this CTA.
    struct ItemView {
        int b, g, ilo, ihi, slo, pg0, npg, nblk;
        size_t hrow;
    };
    auto view = [&](int it) {
        ItemView v;
        const int4 item = plan_item(L, a, ps, nbg, it);
        const int bg = item.x;
        v.b = bg / L.Hkv;
        v.g = bg - v.b * L.Hkv;
        v.ilo = item.y;
        v.ihi = item.z;
        const int glo = ps.lo[bg], gsp = plan_split(L, a, glo, ps.hi[bg]);
        v.slo = item.w ? gsp : glo;   // the item's segment starts here
        v.hrow = (size_t)v.b * L.H + (size_t)v.g * L.G;
        v.pg0 = v.ilo >> 4;
        v.npg = ((v.ihi - 1) >> 4) - v.pg0 + 1;
        v.nblk = (v.npg + 7) >> 3;
        return v;
    };

    if (warp == kTcKWarp || warp == kTcVWarp) {
        // block j of an item goes to stage (jbase + j) mod KS (VS) of the
        // ring; lanes 0-7 look up the pages of the blocks two ahead, lanes
        // 0-15 issue the copies: per page, its two 64-column halves
        const bool keys = warp == kTcKWarp;
        const int ns = keys ? KS : VS;
        uint64_t *full = keys ? bar_kfull : bar_vfull;
        uint64_t *empty = keys ? bar_kempty : bar_vempty;
        const CUtensorMap *map = keys ? &M.kmap : &M.vmap;
        const uint32_t ring = keys ? sK_u : sV_u;
        uint32_t jbase = 0, issued = 0;   // blocks of the previous items; blocks whose copies were issued
        bool ok = true;
        for (int it = blockIdx.x; it < n_items && ok; it += gridDim.x) {
            const ItemView v = view(it);
            auto fetch = [&](int j) {   // page-table entry of page 8 j + lane (-2: none)
                const int q = 8 * j + lane, pg = v.pg0 + q;
                if (lane >= 8 || q >= v.npg) return -2;
                if (pg >= L.pages_per_req) return -1;
                return L.paged ? L.page_table[(size_t)v.b * L.pages_per_req + pg] : pg;
            };
            auto resolve = [&](int e) {   // pool row of a fetched entry, -1 if none (refused: error bit)
                if (e == -2) return -1;
                const bool good = e >= 0 && (!L.paged || e < L.num_pages);
                if (!good) {
                    atomicOr(L.err, kErrPage);
                    return -1;
                }
                return L.paged ? (int)(((size_t)e * L.Hkv + v.g) * kPage)
                               : (int)(((size_t)v.b * L.Hkv + v.g) * L.ctx_stride + (size_t)e * kPage);
            };
            int e0 = fetch(0), e1 = fetch(1);
            for (int j = 0; j < v.nblk; j++) {
                const uint32_t jg = jbase + j, st = jg % ns, round = jg / ns;
                const int row = resolve(e0);
                e0 = e1;
                e1 = fetch(j + 2);
                bool go = true;   // lane 0 waits for the stage, the warp follows its outcome
                if (lane == 0 && round >= 1) go = mbar_wait_or_fail(B_(empty[st]), (round - 1) & 1, fail);
                if (!__shfl_sync(0xffffffffu, go, 0)) {
                    ok = false;
                    break;
                }
                const uint32_t have = __ballot_sync(0xffffffffu, lane < 8 && row >= 0);
                if (have != 0xffu) {
                    // a page past the item or refused by the table is not copied:
                    // its rows are zeroed (the generic writes fenced for the
                    // tensor cores' proxy before the stage is announced)
#pragma unroll 1
                    for (int p = 0; p < 8; p++) {
                        if (have >> p & 1u) continue;
                        uint8_t *z = (keys ? sK : sV) + st * kTcBlockBytes + p * 2048;
                        for (int i = lane; i < 2 * 2048 / 16; i += 32)
                            *reinterpret_cast<uint4 *>(z + (i >> 7) * (kTcTok * 128) + (i & 127) * 16) = make_uint4(0u, 0u, 0u, 0u);
                    }
                    fence_async_smem();
                    __syncwarp();
                }
                {   // lane 0 arms the stage's byte count, then lane 2 p + h copies half h of page p
                    const uint32_t f = B_(full[st]);
                    if (lane == 0) mbar_expect_tx(f, (uint32_t)__popc(have) * 2u * 2048u);
                    __syncwarp();
                    const int hf = lane & 1, rp = __shfl_sync(0xffffffffu, row, (lane >> 1) & 7);
                    if (lane < 16 && rp >= 0)
                        tma_load_2d(ring + st * kTcBlockBytes + hf * (kTcTok * 128) + (lane >> 1) * 2048, map, hf * 64, rp, f);
                }
                issued++;
            }
            jbase += v.nblk;
        }
        // before the CTA exits, the copies it issued have landed: the last
        // fill of each stage completes its full barrier (bounded wait)
        if (lane == 0) {
            for (int s = 0; s < ns; s++) {
                const uint32_t n = (issued + (uint32_t)(ns - 1 - s)) / (uint32_t)ns;
                if (n > 0) mbar_wait_bounded(B_(full[s]), (n - 1) & 1);
            }
        }
    } else if (warp == kTcMmaWarp) {
        if (lane == 0) {
            uint32_t jbase = 0;
            bool ok = true;
            int k = 0;
            for (int it = blockIdx.x; it < n_items && ok; it += gridDim.x, k++) {
                const int nblk = view(it).nblk;
                // Q of the item written; O^T read by the previous item's merge
                if (!mbar_wait_or_fail(B_(bar_qfull), k & 1, fail)) break;
                bool o_free = k == 0;
                // event loop: P V of the oldest block whose P is written goes
                // first (it frees a value stage and a P buffer); the score mma
                // of the next block goes as soon as its keys have landed and its
                // S^T buffer has been read
                int n1 = 0, n2 = 0;   // next block for the score mma, for P V
                uint32_t idle = 0;
                while (n2 < nblk) {
                    bool did = false;
                    if (n2 < n1) {
                        const uint32_t jg = jbase + n2, pb = jg & 1, vs = jg % VS;
                        if (!o_free) o_free = mbar_test(B_(bar_oempty), (k - 1) & 1);
                        if (o_free && mbar_test(B_(bar_pfull[pb]), (jg >> 1) & 1) && mbar_test(B_(bar_vfull[vs]), (jg / VS) & 1)) {
                            tc_fence_after();
                            const uint32_t vst = sV_u + vs * kTcBlockBytes, pst = sP_u + pb * kTcPBytes;
#pragma unroll
                            for (int kk = 0; kk < 8; kk++)
                                tc_mma(t_o, tc_desc(vst + kk * 2048, kTcTok * 128, 1024), tc_desc(pst + kk * 2048, kTcPBytes, 1024),
                                       kIdescO, (n2 > 0 || kk > 0) ? 1u : 0u);
                            tc_commit(B_(bar_pempty[pb]));
                            tc_commit(B_(bar_vempty[vs]));
                            n2++;
                            did = true;
                        }
                    }
                    if (!did && n1 < nblk) {
                        const uint32_t jg = jbase + n1, sb = jg & 1, ks = jg % KS;
                        if (mbar_test(B_(bar_kfull[ks]), (jg / KS) & 1) &&
                            (jg < 2 || mbar_test(B_(bar_sempty[sb]), ((jg >> 1) - 1) & 1))) {
                            tc_fence_after();
                            const uint32_t kst = sK_u + ks * kTcBlockBytes;
#pragma unroll
                            for (int kk = 0; kk < 8; kk++)
                                tc_mma(t_s + sb * 32, tc_desc(kst + (kk >> 2) * (kTcTok * 128) + (kk & 3) * 32, 16, 1024),
                                       tc_desc(sQ_u + (kk >> 2) * (kTcHeads * 128) + (kk & 3) * 32, 16, 1024), kIdescS,
                                       kk > 0 ? 1u : 0u);
                            tc_commit(B_(bar_sfull[sb]));
                            tc_commit(B_(bar_kempty[ks]));
                            n1++;
                            did = true;
                        }
                    }
                    if (did) {
                        idle = 0;
                    } else if (++idle > 16 * kTcSpinLimit || ((idle & 255) == 0 && *fail)) {
                        *fail = 1;
                        ok = false;
                        break;
                    }
                }
                jbase += nblk;
            }
            // every product issued is complete before the CTA frees its tensor memory
            tc_commit(B_(bar_done));
            mbar_wait_bounded(B_(bar_done), 0);
        }
    } else {
        // softmax: thread (t, w / 4) holds token t of each block for the heads
        // h0 .. h0 + kTcHalf - 1
        const int t = tid & (kTcTok - 1), h0 = (warp >> 2) * kTcHalf;
        // Q of an item (thread: chunks tid, tid + 32 x kTcSoftmaxWarps, ... of
        // the 32 x 16) and its heads' first tokens, fetched one item ahead into
        // registers and stored as soon as the previous item's score products
        // are done
        constexpr int kQPer = kTcHeads * 16 / (kTcSoftmaxWarps * 32);
        uint4 qn[kQPer];
        int lon = 0;
        auto fetch_q = [&](const ItemView &w) {
#pragma unroll
            for (int r = 0; r < kQPer; r++) {
                const int i = tid + r * kTcSoftmaxWarps * 32, h = i >> 4, c = i & 15;
                qn[r] = reinterpret_cast<const uint4 *>(a.q_post + (w.hrow + h) * kD)[c];
            }
            if (tid < kTcHeads) lon = max(max(w.slo, w.ilo), L.dec_lo[w.hrow + tid]);
        };
        auto store_q = [&]() {
#pragma unroll
            for (int r = 0; r < kQPer; r++) {
                const int i = tid + r * kTcSoftmaxWarps * 32, h = i >> 4, c = i & 15;
                *reinterpret_cast<uint4 *>(sQ + sw128(kTcHeads, h, c)) = qn[r];
            }
            if (tid < kTcHeads) s_lo[tid] = lon;
            fence_async_smem();
            mbar_arrive(B_(bar_qfull));
        };
        if (blockIdx.x < n_items) {
            fetch_q(view(blockIdx.x));
            store_q();
        }
        uint32_t jbase = 0;
        bool ok = true;
        int k = 0;
        for (int it = blockIdx.x; it < n_items && ok; it += gridDim.x, k++) {
            const ItemView v = view(it);
            if (!mbar_wait_or_fail(B_(bar_qfull), k & 1, fail)) break;
            const bool has_next = it + (int)gridDim.x < n_items;
            if (has_next) fetch_q(view(it + gridDim.x));
            float m[kTcHalf], l[kTcHalf];   // reference (log2 units), this thread's sum of P, per head
#pragma unroll
            for (int h = 0; h < kTcHalf; h++) {
                m[h] = -CUDART_INF_F;
                l[h] = 0.f;
            }
            int lo_max = 0;
#pragma unroll
            for (int h = 0; h < kTcHalf; h++) lo_max = max(lo_max, s_lo[h0 + h]);
            for (int j = 0; j < v.nblk; j++) {
                const uint32_t jg = jbase + j, sb = jg & 1, rb = jg % 3;
                if (!mbar_wait_or_fail(B_(bar_sfull[sb]), (jg >> 1) & 1, fail)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                float y[kTcHalf];
                tmem_ld(t_s + sb * 32 + h0 + lane_base, y);
                tc_fence_before();
                mbar_arrive(B_(bar_sempty[sb]));
                const int tok = (v.pg0 + 8 * j) * 16 + t;
                const bool edge = tok < lo_max || tok >= v.ihi;
                uint32_t mv = 0;   // heads whose reference this token passes by more than kLazyMax
#pragma unroll
                for (int h = 0; h < kTcHalf; h++) y[h] *= sl2;
                if (edge) {   // a token before a head's first or past the item's last
#pragma unroll
                    for (int h = 0; h < kTcHalf; h++)
                        if (!(tok >= s_lo[h0 + h] && tok < v.ihi)) y[h] = -CUDART_INF_F;
                }
#pragma unroll
                for (int h = 0; h < kTcHalf; h++)
                    if (y[h] - m[h] > kLazyMax) mv |= 1u << h;
                const uint32_t wmv = __reduce_or_sync(0xffffffffu, mv);
                if (wmv) {
                    if (__popc(wmv) > 2) {
                        // many heads moved (an item's first block): the warp's
                        // maxima by a transposing butterfly, lane 2 i ending
                        // with head i's, then one shared atomic per head
                        int kk[kTcHalf];
#pragma unroll
                        for (int h = 0; h < kTcHalf; h++) kk[h] = (mv >> h & 1u) ? ord_key(y[h]) : INT_MIN;
#pragma unroll
                        for (int w = kTcHalf / 2; w >= 1; w >>= 1) {
                            const bool upper = (lane & (2 * w)) != 0;
#pragma unroll
                            for (int i = 0; i < w; i++) {
                                const int send = upper ? kk[i] : kk[w + i];
                                const int keep = upper ? kk[w + i] : kk[i];
                                kk[i] = max(keep, __shfl_xor_sync(0xffffffffu, send, 2 * w));
                            }
                        }
                        kk[0] = max(kk[0], __shfl_xor_sync(0xffffffffu, kk[0], 1));
                        if (kTcHalf == 8) kk[0] = max(kk[0], __shfl_xor_sync(0xffffffffu, kk[0], 16));
                        const int hl = (lane >> 1) & (kTcHalf - 1);
                        if ((lane & 1) == 0 && lane < 2 * kTcHalf && (wmv >> hl & 1u)) atomicMax(&s_ref[rb][h0 + hl], kk[0]);
                    } else {
#pragma unroll
                        for (int h = 0; h < kTcHalf; h++) {
                            if (wmv >> h & 1u) {
                                const int key = __reduce_max_sync(0xffffffffu, (mv >> h & 1u) ? ord_key(y[h]) : INT_MIN);
                                if (lane == 0) atomicMax(&s_ref[rb][h0 + h], key);
                            }
                        }
                    }
                    if (lane == 0) atomicOr(&s_any[rb], wmv << h0);
                }
                mbar_arrive(B_(bar_mv));
                if (!mbar_wait_or_fail(B_(bar_mv), jg & 1, fail)) {
                    ok = false;
                    break;
                }
                const uint32_t U = (s_any[rb] >> h0) & ((1u << kTcHalf) - 1u);
                // the slot two blocks on was read before everyone arrived here,
                // and is written again only after everyone arrives next time
                if (tid < kTcHeads) s_ref[(jg + 2) % 3][tid] = INT_MIN;
                if (tid == kTcHeads) s_any[(jg + 2) % 3] = 0u;
                if (U) {
                    float al[kTcHalf];
#pragma unroll
                    for (int h = 0; h < kTcHalf; h++) {
                        al[h] = 1.f;
                        if (U >> h & 1u) {
                            const float mn = ord_val(s_ref[rb][h0 + h]);
                            al[h] = m[h] == -CUDART_INF_F ? 0.f : ex2_approx(m[h] - mn);
                            m[h] = mn;
                            l[h] *= al[h];
                        }
                    }
                    if (j > 0) {   // O^T row t, once the P V of the previous block is done
                        if (!mbar_wait_or_fail(B_(bar_pempty[(jg - 1) & 1]), ((jg - 1) >> 1) & 1, fail)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
#pragma unroll
                        for (int part = 0; part < 2; part++) {   // the hi and the lo products
                            float o[kTcHalf];
                            tmem_ld(t_o + 32 * part + h0 + lane_base, o);
#pragma unroll
                            for (int h = 0; h < kTcHalf; h++) o[h] *= al[h];
                            tmem_st(t_o + 32 * part + h0 + lane_base, o);
                        }
                    }
                }
                uint32_t ph[kTcHalf / 2], pl[kTcHalf / 2];
#pragma unroll
                for (int h = 0; h < kTcHalf; h += 2) {
                    const float p0 = y[h] == -CUDART_INF_F ? 0.f : ex2_approx(y[h] - m[h]);
                    const float p1 = y[h + 1] == -CUDART_INF_F ? 0.f : ex2_approx(y[h + 1] - m[h + 1]);
                    l[h] += p0;
                    l[h + 1] += p1;
                    const __nv_bfloat162 hv = __floats2bfloat162_rn(p0, p1);
                    const float2 fv = __bfloat1622float2(hv);
                    ph[h >> 1] = bf16x2_bits(hv);
                    pl[h >> 1] = bf16x2_bits(__floats2bfloat162_rn(p0 - fv.x, p1 - fv.y));
                }
                // P buffer jg & 1 is free once the P V of block jg - 2 is done
                const uint32_t pb = jg & 1;
                if (jg >= 2 && !mbar_wait_or_fail(B_(bar_pempty[pb]), ((jg >> 1) - 1) & 1, fail)) {
                    ok = false;
                    break;
                }
                {   // row t: chunks 0-3 hold P_hi of heads 0-31 (8 per chunk), chunks 4-7 P_lo
                    uint8_t *row = sP + pb * kTcPBytes + t * 128;
#pragma unroll
                    for (int q = 0; q < kTcHalf / 8; q++) {
                        const int c = (h0 >> 3) + q;
                        *reinterpret_cast<uint4 *>(row + ((c ^ (t & 7)) << 4)) =
                            make_uint4(ph[4 * q], ph[4 * q + 1], ph[4 * q + 2], ph[4 * q + 3]);
                        *reinterpret_cast<uint4 *>(row + (((c + 4) ^ (t & 7)) << 4)) =
                            make_uint4(pl[4 * q], pl[4 * q + 1], pl[4 * q + 2], pl[4 * q + 3]);
                    }
                }
                fence_async_smem();
                tc_fence_before();
                mbar_arrive(B_(bar_pfull[pb]));
            }
            if (!ok) break;
            // every score product of the item is done (its S^T has been read):
            // the next item's Q goes in while this one merges
            if (has_next) store_q();
            // merge: the item's last P V done, O^T holds the hi and lo products
            const uint32_t last = jbase + v.nblk - 1;
            if (!mbar_wait_or_fail(B_(bar_pempty[last & 1]), (last >> 1) & 1, fail)) break;
            {   // O^T row t for this thread's heads (hi + lo), then O^T is free for the next item
                tc_fence_after();
                float o[kTcHalf], o2[kTcHalf];
                tmem_ld(t_o + h0 + lane_base, o);
                tmem_ld(t_o + 32 + h0 + lane_base, o2);
                tc_fence_before();
                mbar_arrive(B_(bar_oempty));
#pragma unroll
                for (int h = 0; h < kTcHalf; h++) L.part_o[((size_t)it * L.G + h0 + h) * kD + t] = o[h] + o2[h];
            }
            if (t == 0) {
#pragma unroll
                for (int h = 0; h < kTcHalf; h++) s_m[h0 + h] = m[h];
            }
            // the warp's 32 partial sums of each of its kTcHalf heads: a
            // transposing butterfly halves the heads a lane holds at each step,
            // so lane 2 i (i < kTcHalf) ends with the sum of head i once the
            // lanes the butterfly did not pair are added
#pragma unroll
            for (int w = kTcHalf / 2; w >= 1; w >>= 1) {
                const bool upper = (lane & (2 * w)) != 0;
#pragma unroll
                for (int i = 0; i < w; i++) {
                    const float send = upper ? l[i] : l[w + i];
                    const float keep = upper ? l[w + i] : l[i];
                    l[i] = keep + __shfl_xor_sync(0xffffffffu, send, 2 * w);
                }
            }
            l[0] += __shfl_xor_sync(0xffffffffu, l[0], 1);
            if (kTcHalf == 8) l[0] += __shfl_xor_sync(0xffffffffu, l[0], 16);
            if ((lane & 1) == 0 && lane < 2 * kTcHalf) s_l[warp & 3][h0 + ((lane >> 1) & (kTcHalf - 1))] = l[0];
            mbar_arrive(B_(bar_red));
            if (!mbar_wait_or_fail(B_(bar_red), k & 1, fail)) break;
            if (tid < kTcHeads)
                L.part_ml[(size_t)it * L.G + tid] =
                    make_float2(s_m[tid], (s_l[0][tid] + s_l[1][tid]) + (s_l[2][tid] + s_l[3][tid]));
            jbase += v.nblk;
        }
    }
    __syncthreads();
    if (*fail && tid == 0) atomicOr(L.err, kErrTimeout);
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" :: "r"(tmem), "r"(kTcTmemCols) : "memory");
    }
}

size_t attention_tc_smem() { return 1024 + kTcQBytes + 2 * kTcPBytes + (size_t)(kTcKStages + kTcVStages) * kTcBlockBytes; }

using EncodeTiled = PFN_cuTensorMapEncodeTiled_v12000;

}  // namespace

cudaError_t attention_tc_config(size_t *smem, int *ctas_per_sm)
{
    *smem = attention_tc_smem();
    auto k = attention_tc_kernel<kTcKStages, kTcVStages>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)*smem);
    if (e != cudaSuccess) return e;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(ctas_per_sm, k, kTcThreads, *smem);
}

cudaError_t launch_attention_tc(const Layout &L, const StepArgs &a, const TcMaps &maps, size_t smem, cudaStream_t s)
{
    return launch_maybe_pdl(attention_tc_kernel<kTcKStages, kTcVStages>, dim3(a.grid_ctas), dim3(kTcThreads), smem, s,
                            a.pdl, L, a, maps);
}

cudaError_t attention_tc_maps(Layout &L, TcMaps &M, int64_t rows)
{
    static EncodeTiled encode = nullptr;   // the driver's tensor-map encoder, looked up once
    if (!encode) {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        const cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
        if (e != cudaSuccess) return e;
        if (q != cudaDriverEntryPointSuccess || !fn) return cudaErrorNotSupported;
        encode = reinterpret_cast<EncodeTiled>(fn);
    }
    if (rows < kPage || rows > 0x7fffffffll) return cudaErrorInvalidValue;
    // each pool viewed as rows of 128 bf16 (a token of one KV head); a box is
    // one page (16 rows) by 64 columns, written with the 128-byte swizzle
    const cuuint64_t dims[2] = {(cuuint64_t)kD, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)kD * 2};
    const cuuint32_t box[2] = {64, (cuuint32_t)kPage};
    const cuuint32_t estr[2] = {1, 1};
    CUtensorMap *maps[2] = {&M.kmap, &M.vmap};
    void *pools[2] = {L.k_pool, L.v_pool};
    for (int i = 0; i < 2; i++) {
        const CUresult r = encode(maps[i], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, pools[i], dims, strides, box, estr,
                                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    }
    L.tc = 1;
    return cudaSuccess;
}

}  // namespace macgpu
