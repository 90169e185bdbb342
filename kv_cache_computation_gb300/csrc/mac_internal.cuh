// Internal definitions shared by the host layer (mac_api.cu) and the kernels
// (mac_kernels.cu) of the MAC-Attention decode-step library.  Not part of the
// public ABI (include/mac.h).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace macgpu {

constexpr int kD = 128;                 // head_dim
constexpr int kPage = 16;               // tokens per KV page / per staged block
constexpr int kMaxRing = 4096;          // ring entries per (request, head)
constexpr int kSmallRing = 32;          // rings up to this size (one entry's distance per lane) are
                                        // scanned inside the Match kernel
constexpr int kScanBlock = 256;         // ring entries per block of the wide-ring scan
constexpr int kMaxGroup = 32;           // query heads per KV head
constexpr int kMatchWarps = 8;          // query heads (warps) per Match block at most

// Match blocks per group: groups of more than kMatchWarps heads are split
// so that no SM holds more than kMatchWarps heads' ring scans.
inline __host__ __device__ int match_parts(int G) { return (G + kMatchWarps - 1) / kMatchWarps; }
constexpr int kMaxCtas = 1024;          // upper bound of the attention grid
constexpr int kMaxGroupsPerStep = 1024; // max_batch * kv_heads (the plan is held in shared memory)
// attention pipeline shape (overridable at build time for tuning sweeps)
#ifndef MAC_ATTN_WARPS
#define MAC_ATTN_WARPS 4
#endif
#ifndef MAC_ATTN_STAGES
#define MAC_ATTN_STAGES 3
#endif
#ifndef MAC_PREFETCH_AHEAD
#define MAC_PREFETCH_AHEAD 2
#endif
constexpr int kAttnWarps = MAC_ATTN_WARPS;         // warps per attention CTA
constexpr int kAttnStages = MAC_ATTN_STAGES;       // pipeline stages per page lane
constexpr int kPrefetchAhead = MAC_PREFETCH_AHEAD; // pages per lane prefetched into L2 past the copy front
#ifndef MAC_SPECULATIVE_PAGES
#define MAC_SPECULATIVE_PAGES 2
#endif
constexpr int kSpeculativePages = MAC_SPECULATIVE_PAGES;  // pages per lane of the previous step's item warmed in L2
constexpr int kStageBytes = 2 * kPage * kD * 2;   // one K page + one V page (bf16): 8 KB
#ifndef MAC_DYN_FRAC
#define MAC_DYN_FRAC 10
#endif
// A work item of at least kDynMinPages pages leaves its last npg * kDynFrac /
// 128 pages (at least 2) to its segment's shared pool; 0 turns pools off.
constexpr int kDynFrac = MAC_DYN_FRAC;
constexpr int kDynMinPages = 32;
#ifndef MAC_ATTN_CUDA_CORE
#define MAC_ATTN_CUDA_CORE 0
#endif
// Comparison build: the page contractions S^T = K Q^T and O^T += V^T P^T on
// fp32 FMA instead of mma.sync (same tiles, same layouts, q staged in shared
// memory); selected at compile time, never at run time.
constexpr bool kAttnCudaCore = MAC_ATTN_CUDA_CORE != 0;
#ifndef MAC_ATTN_HEADS_ON_M
#define MAC_ATTN_HEADS_ON_M 1
#endif
// Groups of 16 and 32 heads take the heads-on-M attention tiles (0: the
// 8-head N tiles of smaller groups for every group size; comparison build).
constexpr bool kHeadsOnM = MAC_ATTN_HEADS_ON_M != 0;
// Resident CTAs per SM the heads-on-M kernel is register-budgeted for: 2
// (no spills) for 16-head groups and, with fewer than kHmWideGroups groups
// in the step, for 32-head groups; 3 (about 170 registers, a few bytes
// spilled; more warps to hide latency) for 32-head groups in steps of many
// groups, which stream the most pages per CTA.
#ifndef MAC_HM_MIN_CTAS_16
#define MAC_HM_MIN_CTAS_16 2
#endif
#ifndef MAC_HM_MIN_CTAS_32
#define MAC_HM_MIN_CTAS_32 2
#endif
#ifndef MAC_HM_MIN_CTAS_32_WIDE
#define MAC_HM_MIN_CTAS_32_WIDE 3
#endif
#ifndef MAC_HM_WIDE_GROUPS
#define MAC_HM_WIDE_GROUPS 32
#endif
constexpr int kHmMinCtas16 = MAC_HM_MIN_CTAS_16;
constexpr int kHmMinCtas32 = MAC_HM_MIN_CTAS_32;
constexpr int kHmMinCtas32Wide = MAC_HM_MIN_CTAS_32_WIDE;
constexpr int kHmWideGroups = MAC_HM_WIDE_GROUPS;
// 1: steps of 32-head groups that hold at least MAC_TC_MIN_TOKENS KV tokens
// (over all requests and KV heads) stream through the tcgen05 kernel
// (mac_attention_tc.cu; blocks of 128 tokens, key and value rings of
// MAC_TC_K_STAGES and MAC_TC_V_STAGES blocks); smaller steps, whose time is
// mostly the kernels' fixed costs, keep the mma.sync heads-on-M kernel.
// 0: the mma.sync kernel for every step (comparison build).
#ifndef MAC_ATTN_TC32
#define MAC_ATTN_TC32 1
#endif
#ifndef MAC_TC_MIN_TOKENS
#define MAC_TC_MIN_TOKENS 16384
#endif
constexpr long long kTcMinTokens = MAC_TC_MIN_TOKENS;
// Steps of at least MAC_TC_WAVE_TOKENS KV tokens per tcgen05 CTA are planned
// for MAC_TC_PLAN_WAVES items per CTA (the CTA overlaps consecutive items):
// when the groups do not divide the grid, items of one wave leave CTAs idle.
#ifndef MAC_TC_PLAN_WAVES
#define MAC_TC_PLAN_WAVES 2
#endif
#ifndef MAC_TC_WAVE_TOKENS
#define MAC_TC_WAVE_TOKENS 16384
#endif
constexpr int kTcPlanWaves = MAC_TC_PLAN_WAVES;
constexpr long long kTcWaveTokens = MAC_TC_WAVE_TOKENS;
#ifndef MAC_TC_K_STAGES
#define MAC_TC_K_STAGES 2
#endif
#ifndef MAC_TC_V_STAGES
#define MAC_TC_V_STAGES 3
#endif
constexpr bool kTc32 = MAC_ATTN_TC32 != 0;
#ifndef MAC_HM_STAGES_32
#define MAC_HM_STAGES_32 3
#endif
constexpr int kHmStages32 = MAC_HM_STAGES_32;   // pipeline stages per page lane, 32-head groups
constexpr float kLazyMax = 8.0f;   // heads-on-M attention: a page moves the softmax reference past this margin
constexpr float kRemovalMinCond = 1.0f / 32.0f;   // Amend: 1 - e^delta below this -> direct form
constexpr int kMinChunk = 64;           // smallest work-item span in tokens
constexpr int kPlanCache = 1024;        // groups the planner caches in shared memory
constexpr int kBandTile = 64;           // tokens per shared-memory tile of the Amend band recompute
constexpr int kBandRow = 272;           // padded bytes per staged K/V row (conflict-free per-lane rows)

// device error bits
enum : uint32_t { kErrPage = 1u, kErrSlot = 2u, kErrPos = 4u, kErrTimeout = 8u };

// device counters
enum { kStSteps = 0, kStDecisions, kStHits, kStKvRead, kStKvFull, kStDirect, kStItems, kStCount };

// Device-side view of one handle: dimensions and carved buffer pointers.
struct Layout {
    int H, Hkv, G, ring_len, band_r;
    int max_batch;
    int paged;
    int pages_per_req;        // page-table row length (paged) / blocks per request (contiguous)
    int num_pages;            // paged: pool pages
    int ctx_stride;           // contiguous: tokens reserved per (request, kv-head)
    int item_cap;
    int amend_band;           // 0: reuse Complete's band summary; 1: recompute it in Amend
    int tc;                   // the pools' TMA descriptors are made: the tcgen05 attention kernel can serve
    float tau2;               // tau^2 (fp32)
    float scale_log2;         // sm_scale * log2(e)

    __nv_bfloat16 *k_pool, *v_pool;
    int32_t *page_table;      // [max_batch][pages_per_req]

    // rings
    int32_t *ring_pos;        // [max_batch][L] 1-based position, 0 = empty
    __nv_bfloat16 *ring_q;    // [max_batch][H][L][D]
    float *ring_o;            // [max_batch][H][L][D]
    float *ring_lse;          // [max_batch][H][L]

    // per-request state
    int32_t *kv_len;          // [max_batch]
    int32_t *step_ctr;        // [max_batch]
    int32_t *m_cur;           // [max_batch] position m of the step in flight
    int32_t *slot_cur;        // [max_batch] ring slot the step in flight inserts into

    // decisions [max_batch * H]
    int32_t *dec_own_slot, *dec_own_hit, *dec_slot, *dec_lo;
    float *dec_D, *dec_qn2;
    int32_t *forced_slot;
    unsigned long long *dec_key;   // [max_batch * H] wide rings: min over entries of (D bits << 32 | age)
    int32_t *seed_pos;             // [L] positions of the entries a seeding call inserts
    __nv_bfloat16 *q_stash;   // [max_batch][H][D] post-RoPE query kept for Amend

    // plan
    int32_t *grp_lo;          // [max_batch * Hkv] first token any head of the group reads
    int32_t *seg_claim;       // [max_batch * Hkv * 2] pool pages claimed per group segment this step
    int32_t *grp_item_off;    // [max_batch * Hkv + 1]
    int4 *items;              // [item_cap] {b*Hkv+g, lo, hi, segment}
    int32_t *n_items;

    // partial summaries of work items: unnormalised o, (max, sum) in log2 units
    float *part_o;            // [item_cap][G][D]
    float2 *part_ml;          // [item_cap][G]

    // merged summaries kept for Amend
    float *as_full_o, *as_full_lse;   // AS_{1:m}
    float *as_pre_o, *as_pre_lse;     // AS_{1:m-r} formed directly (fallback of the removal)

    unsigned long long *stats;        // [kStCount]
    uint32_t *err;

    int lo_parts;   // Match blocks per group (match_parts(G)); above 1 they meet in grp_lo by atomicMin
                    // and Combine sets the word back to INT_MAX for the next step
};

// TMA descriptors of the K and V pools (rows of 128 bf16; box 16 rows x 64
// columns, 128-byte swizzle), a parameter of the tcgen05 attention kernel only.
struct TcMaps {
    CUtensorMap kmap, vmap;
};

struct StepArgs {
    int batch;
    const __nv_bfloat16 *q_pre, *q_post, *k_new, *v_new;
    __nv_bfloat16 *out;
    float *lse_out;
    int force;        // use forced_slot instead of the Match decision
    int full_mode;    // full attention, no Match / Amend
    int grid_ctas;    // attention CTAs
    int plan_ctas;    // work slots the plan fills: grid_ctas, or a multiple of it for a kernel
                      // whose CTAs overlap consecutive items
    int plan_mode;    // 0 balanced, 1 equal split per group
    int pdl;          // launch attention / combine as programmatic dependents
    int wide;         // attention: the variant for many groups (grid_ctas is its grid)
    int tc;           // attention: the tcgen05 kernel (grid_ctas is its grid)
};

// launchers (mac_kernels.cu)
cudaError_t launch_match_plan(const Layout &L, const StepArgs &a, cudaStream_t s);
cudaError_t launch_seed(const Layout &L, int req, int first, int n, int base_step, const __nv_bfloat16 *q,
                        const float *o, const float *lse, cudaStream_t s);
cudaError_t launch_attention(const Layout &L, const StepArgs &a, const TcMaps *maps, size_t smem, cudaStream_t s);
cudaError_t launch_combine(const Layout &L, const StepArgs &a, cudaStream_t s);
cudaError_t launch_amend(const Layout &L, const StepArgs &a, cudaStream_t s);
cudaError_t launch_append(const Layout &L, int req, int start, int n, const __nv_bfloat16 *k,
                          const __nv_bfloat16 *v, cudaStream_t s);
cudaError_t attention_kernel_config(int G, bool wide, bool tc, size_t *smem, int *ctas_per_sm);
bool attention_tc_wanted(int G);                                                        // mac_attention.cu
cudaError_t attention_tc_config(size_t *smem, int *ctas_per_sm);                        // mac_attention_tc.cu
cudaError_t attention_tc_maps(Layout &L, TcMaps &maps, int64_t pool_rows);              // mac_attention_tc.cu
cudaError_t launch_attention_tc(const Layout &L, const StepArgs &a, const TcMaps &maps, size_t smem, cudaStream_t s);
bool attention_wide(int G, int groups);   // whether a step of `groups` groups takes the wide variant
cudaError_t amend_kernel_config();

}  // namespace macgpu
