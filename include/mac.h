/*
 * mac.h -- C ABI of the GB300 (sm_103a) MAC-Attention decode-step library.
 *
 * MAC-Attention ("Match-Amend-Complete", arXiv 2604.00235) accelerates one
 * decode step of attention by reusing the attention summary of a recent,
 * similar query.  Per request and per query head, at decode position m:
 *
 *   Match    (paper, Figure 2(a); abstract "pre-RoPE L2 matching over a short
 *            local window"): compare the pre-RoPE query q~_m with a small
 *            ring of recent pre-RoPE queries; if the nearest one, at position
 *            p, passes an L2 threshold, fetch its attention summary
 *            AS_{1:p-r}; otherwise run full attention.
 *   Complete (Figure 2(b)): attention of the post-RoPE query q_m over the
 *            band+tail [p-r+1, m] only, merged in the log domain with the
 *            fetched AS_{1:p-r}; KV [1, p-r] is not read.
 *   Amend    (Figure 2(c), asynchronous): recompute the rectification term
 *            AS_{m-r+1:m}, obtain AS_{1:m-r} by log-domain removal from the
 *            step's AS_{1:m}, and insert <q~_m, AS_{1:m-r}> into the rings.
 *
 * An attention summary AS = (o, lse): o is the softmax-normalised attention
 * output over a token set, lse the log-sum-exp of its scaled scores.
 *
 * Conventions
 *  - Every pointer argument named dev_* is CUDA device memory on the current
 *    device; host_* pointers are host memory.
 *  - Tensors are dense, row-major, with no padding: queries and outputs
 *    [batch][heads][head_dim]; new/appended K, V [n][kv_heads][head_dim].
 *    bf16 values are IEEE bfloat16 bit patterns (uint16).  Device tensors
 *    must be 16-byte aligned (fp32 lse: 4-byte aligned).
 *  - A `stream` argument is a cudaStream_t passed as void* (NULL = the legacy
 *    default stream).  Calls marked "async" only enqueue work on it.
 *  - Request i of a batched call is request slot i of the handle.
 *  - Ownership: the caller owns every buffer it passes, including the three
 *    backing buffers handed to mac_create, which must outlive the handle.
 *    The library owns one side stream, its events and nothing else.
 *  - Errors: every call returns a mac_status; no exception or abort crosses
 *    the ABI.  A CUDA error is sticky: the handle returns MAC_ERR_CUDA from
 *    then on.  A handle is not thread-safe.
 *  - Stream capture: the step calls enqueue only kernels (and, with
 *    amend_band 1, event records and waits), so a decode loop can be
 *    captured into a CUDA graph.  Call mac_sync before beginning a capture
 *    and, with amend_band 1, mac_join on the capturing stream before ending
 *    it.  Host-side length checks run at capture time: a replayed graph
 *    advances the device state, not the checks.  Calls made after a replay
 *    must be ordered after it (same stream, or after synchronising).
 */
#ifndef MAC_H
#define MAC_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct mac_ctx *mac_handle;

typedef enum {
    MAC_OK = 0,
    MAC_ERR_INVALID_ARG = -1,  /* bad pointer, size, index or configuration   */
    MAC_ERR_OOM = -2,          /* a backing buffer is too small or misaligned  */
    MAC_ERR_CUDA = -3,         /* a CUDA call failed (sticky)                  */
    MAC_ERR_CAPACITY = -4,     /* KV store or page table of a request is full  */
    MAC_ERR_TIMEOUT = -5,      /* mac_sync gave up waiting                     */
    MAC_ERR_STATE = -6         /* a device-side bounds check fired (sticky)    */
} mac_status;

/* Configuration of one attention layer (one handle per layer). */
typedef struct {
    int heads;          /* query heads H                                        */
    int kv_heads;       /* KV heads H_kv; heads % kv_heads == 0 and the group   */
                        /* G = heads / kv_heads is one of 1, 2, 4, 8, 16, 32     */
    int head_dim;       /* d; must be 128                                        */
    int ring_len;       /* L: ring entries per (request, head), 1..4096; rings   */
                        /* over 32 entries are scanned by a separate grid-wide  */
                        /* kernel before Match decides                          */
    int band_r;         /* r: rectification band width in tokens, >= 1           */
    double tau;         /* L2 threshold, relative: hit iff                       */
                        /* ||q~_m - q~_e|| < tau * ||q~_m||; tau >= 0           */
    int max_batch;      /* request slots, >= 1; max_batch * kv_heads <= 1024    */
    int64_t max_ctx;    /* tokens per request, 1 .. 2^30                         */
    int page_size;      /* 0: contiguous KV per request; 16: paged KV            */
    int num_pages;      /* paged: pages in the pool (0: max_batch*ceil(max_ctx/16)) */
    float sm_scale;     /* score scale; 0 selects 1/sqrt(head_dim)               */
    int plan_mode;      /* 0: span-proportional work split (the paper's          */
                        /* load-balanced planning, Figure 3(b)); 1: equal split  */
                        /* per KV group regardless of span (unbalanced baseline) */
    int amend_band;     /* where Amend's rectification term AS_{m-r+1:m} comes   */
                        /* from: 0 = the band segment Complete already streams   */
                        /* (the band lies inside band+tail and inside [1, m]);   */
                        /* 1 = recomputed by the Amend kernel from the KV store  */
                        /* (Figure 2(c) as drawn).  Same value either way.       */
} mac_config;

/* Cumulative device counters (mac_get_stats). */
typedef struct {
    uint64_t steps;           /* mac_decode_step + mac_full_step calls          */
    uint64_t head_decisions;  /* (request, head) Match decisions               */
    uint64_t hits;            /* of which reuse the ring (hits)                 */
    uint64_t kv_tokens_read;  /* sum over (request, KV head) of tokens streamed */
    uint64_t kv_tokens_full;  /* same for full attention over [1, m]            */
    uint64_t removal_direct;  /* Amend removals too ill-conditioned for fp32    */
                              /* (1 - e^delta < 1/32), formed directly instead  */
    uint64_t work_items;      /* attention work items planned                   */
    uint32_t device_error;    /* bounds-check bits (0 = none; any set makes     */
                              /* mac_sync return MAC_ERR_STATE and the handle   */
                              /* sticky): 1 a page-table entry outside          */
                              /* the pool or a page past the table (its tokens  */
                              /* are not read; the request's output is then     */
                              /* wrong, other requests' are not touched); 2 a   */
                              /* forced slot that holds no entry (taken as a    */
                              /* miss); 4 more work                             */
                              /* items than the scratch holds; 8 a wait in the  */
                              /* tcgen05 kernel gave up (its CTA stopped early) */
    uint32_t reserved;
    uint64_t tcgen05_steps;   /* of the steps, those whose attention ran on the */
                              /* tcgen05 kernel (groups of 32 heads, steps of   */
                              /* at least 16384 KV tokens); the others ran on   */
                              /* the mma.sync kernel                            */
} mac_stats;

/* Accumulated GPU time per phase since profiling was enabled (ms). */
typedef struct {
    double match_plan_ms;     /* KV append + Match (+ the ring scan of long     */
                              /* rings)                                         */
    double attention_ms;      /* work plan + split-KV band+tail / full          */
                              /* attention kernel                               */
    double combine_ms;        /* log-domain merge kernel (with Amend's removal  */
                              /* and ring insert when amend_band is 0)          */
    double amend_ms;          /* Amend kernel (side stream, amend_band 1); 0    */
                              /* when Amend runs inside the merge kernel        */
    uint64_t steps;           /* steps timed                                    */
} mac_profile;

/* Bytes of the three backing buffers a configuration needs.  Pure host
 * arithmetic (no GPU needed).  kv: the K and V store; ring: the rings of
 * pre-RoPE queries and summaries (per request and head, L slots of bf16 q~,
 * fp32 o and fp32 lse -- 772 B per slot per query head at d = 128 -- plus
 * one int32 position per request and slot); scratch: decisions, work list,
 * partial summaries and counters.  MAC_ERR_INVALID_ARG for a bad config. */
mac_status mac_query_sizes(const mac_config *cfg, size_t *kv_bytes, size_t *ring_bytes,
                           size_t *scratch_bytes);

/* Create a handle over caller-allocated device buffers (each 256-byte
 * aligned and at least the size mac_query_sizes gives; MAC_ERR_OOM if not).
 * Zeroes the KV store; clears rings, lengths and counters; creates the side
 * stream and events.
 * Synchronous. */
mac_status mac_create(const mac_config *cfg, void *dev_kv, size_t kv_bytes, void *dev_ring,
                      size_t ring_bytes, void *dev_scratch, size_t scratch_bytes, mac_handle *out);

/* Wait for outstanding work, then release the stream and events.  The
 * backing buffers stay the caller's. */
mac_status mac_destroy(mac_handle h);

/* Paged mode: install request req's page table, n_pages int32 page indices
 * into the pool (each < num_pages), copied device-to-device.  Logical page i
 * holds tokens [16 i, 16 i + 16).  The caller's KV manager chooses the pages
 * (paper abstract: composes with paged-KV managers).  Async on stream. */
mac_status mac_set_page_table(mac_handle h, int req, const int32_t *dev_pages, int n_pages,
                              void *stream);

/* Append n_tokens tokens of post-RoPE K and of V (device bf16
 * [n_tokens][kv_heads][head_dim]) after request req's current length, e.g.
 * the prefill.  The rings are not touched.  MAC_ERR_CAPACITY if the request
 * would exceed max_ctx or its page table.  Async on stream. */
mac_status mac_append_kv(mac_handle h, int req, const void *dev_k, const void *dev_v, int64_t n_tokens,
                         void *stream);

/* One MAC decode step for requests 0..batch-1 (Figure 2 (a)->(b)->(c)):
 * appends k_new/v_new (device bf16 [batch][kv_heads][head_dim], post-RoPE)
 * at position m = length + 1, runs Match on q_pre (pre-RoPE, device bf16
 * [batch][heads][head_dim]), Complete with q_post (post-RoPE, same shape),
 * and writes out (device bf16 [batch][heads][head_dim]) and, if lse_out is
 * not NULL, the natural-log LSE of AS_{1:m} (device fp32 [batch][heads]).
 * Amend runs on the library's side stream after Complete; the next call on
 * this handle waits for it.  The inputs may be reused by later work on
 * `stream` (Amend keeps its own copies).  Async on stream. */
mac_status mac_decode_step(mac_handle h, int batch, const void *dev_q_pre, const void *dev_q_post,
                           const void *dev_k_new, const void *dev_v_new, void *dev_out, float *dev_lse_out,
                           void *stream);

/* mac_decode_step with its inputs and results in page-locked host memory
 * (cudaHostAlloc / cudaMallocHost / cudaHostRegister; same layouts and
 * alignment as above): the step's kernels read q_pre, q_post, k_new and v_new and write
 * out and lse_out in place over the host link (NVLink-C2C on Grace
 * systems), so the transfers ride inside the step's three launches instead
 * of separate copies.  The host buffers must stay untouched until the work
 * on `stream` is complete; results are valid after a stream/event sync.
 * MAC_ERR_INVALID_ARG if a buffer is not page-locked host memory the device
 * can address (pageable memory is refused, not staged).  Async on stream. */
mac_status mac_decode_step_host(mac_handle h, int batch, const void *host_q_pre, const void *host_q_post,
                                const void *host_k_new, const void *host_v_new, void *host_out,
                                float *host_lse_out, void *stream);

/* Full split-KV decode attention (the miss path for every head; no Match,
 * no ring update): append, then out = AS_{1:m}(q_post).  The in-library
 * baseline the MAC path is compared against.  Async on stream. */
mac_status mac_full_step(mac_handle h, int batch, const void *dev_q_post, const void *dev_k_new,
                         const void *dev_v_new, void *dev_out, float *dev_lse_out, void *stream);

/* Make `stream` wait (device-side) for the handle's outstanding Amend. */
mac_status mac_join(mac_handle h, void *stream);

/* Block until the outstanding Amend has finished, polling; MAC_ERR_TIMEOUT
 * after timeout_ms (< 0: wait forever).  Then checks the device bounds-check
 * word (MAC_ERR_STATE if set). */
mac_status mac_sync(mac_handle h, int timeout_ms);

/* Copy the device counters out (waits for the device first). */
mac_status mac_get_stats(mac_handle h, mac_stats *out);
mac_status mac_reset_stats(mac_handle h);

/* Seed request req's rings with n entries <q~, AS_{1:pos-r}> -- for example
 * the last prefill queries and the summaries the caller's prefill attention
 * produced -- so the first decode steps can already reuse them (the paper's
 * 512-2048-entry match windows, Figure 6 and Tables 5 and 7, reach back into
 * the prompt; the pages do not say how those entries are formed, so the
 * caller supplies them).  dev_q_pre bf16 [n][heads][head_dim] (pre-RoPE),
 * dev_o fp32 [n][heads][head_dim] (normalised output of AS_{1:pos-r}),
 * dev_lse fp32 [n][heads] (its natural-log LSE; -inf for the empty set),
 * host_pos int64 [n]: 1-based positions, strictly increasing, each <= the
 * request's length.  Entries are inserted in order exactly as decode steps
 * insert theirs (slot = step mod L, step + 1), so only the last L survive.
 * Seed before decoding (positions must grow with insertion order).
 * Synchronous (waits for stream). */
mac_status mac_seed_ring(mac_handle h, int req, int n, const void *dev_q_pre, const float *dev_o,
                         const float *dev_lse, const int64_t *host_pos, void *stream);

/* Forget request req: length 0, empty rings, step counter 0.  Async on
 * stream (after outstanding Amend). */
mac_status mac_reset_request(mac_handle h, int req, void *stream);

/* Per-phase GPU timing with CUDA events around each launch (adds event
 * records to every step; off by default).  mac_get_profile synchronises and
 * reports the totals since profiling was (re-)enabled. */
mac_status mac_set_profiling(mac_handle h, int enable);
mac_status mac_get_profile(mac_handle h, mac_profile *out);

/* ---- test hooks --------------------------------------------------------- */

/* Override the next decode step's decisions: dev_slot [batch][heads] int32,
 * -1 = miss, otherwise the ring slot to reuse (it must hold an entry, else
 * the step treats it as a miss and sets a bounds-check bit).  The Match
 * kernel still computes and records its own decision.  One-shot.  Async. */
mac_status mac_debug_force_decisions(mac_handle h, const int32_t *dev_slot, int batch, void *stream);

/* The last decode step's own Match results for requests 0..batch-1 (host
 * [batch][heads] each; NULL skips): nearest valid slot (-1 if the ring was
 * empty), its hit flag, its squared distance D and ||q~||^2 in fp32.
 * Synchronous. */
mac_status mac_debug_get_decisions(mac_handle h, int batch, int32_t *host_slot, int32_t *host_hit,
                                   float *host_D, float *host_qn2);

/* Copy request req's rings to the host (NULL skips): positions [L] (1-based,
 * 0 = empty), q~ [heads][L][head_dim] bf16 bits, o [heads][L][head_dim]
 * fp32, lse [heads][L] fp32; and its length and step counter.  Synchronous. */
mac_status mac_debug_read_ring(mac_handle h, int req, int32_t *host_pos, uint16_t *host_q, float *host_o,
                               float *host_lse, int64_t *kv_len, int64_t *steps);

/* ---- decode attention without any device allocation --------------------- */

/* No counterpart in the paper: this entry point exists for callers that may
 * not allocate device memory at the point where they run attention -- a
 * runtime that plans every byte of device memory in one arena at start-up
 * and forbids later allocations, a latency-critical loop that must not call
 * cudaMalloc (it can synchronise the device), or a plug-in host that hands
 * the library nothing but its input and output buffers.  Every handle-based
 * call above needs a scratch buffer allocated for mac_create; this one
 * needs none.
 *
 * It computes what mac_full_step computes (full split-KV decode attention,
 * out = AS_{1:len}(q) per request and query head) over a KV cache the caller
 * holds, without appending to it:
 *   dev_k, dev_v  bf16 [batch][kv_heads][ctx_stride][head_dim]; token j of
 *                 request b, KV head g starts at element
 *                 ((b * kv_heads + g) * ctx_stride + j) * head_dim
 *                 (the contiguous layout of a mac_create handle with
 *                 page_size 0, ctx_stride = max_ctx rounded up to 16)
 *   host_lens     host int32 [batch], tokens of each request, 1..ctx_stride;
 *                 slots past a request's length are never used, whatever
 *                 they hold (NaN included)
 *   dev_q         bf16 [batch][heads][head_dim], post-RoPE query
 *   dev_out       bf16 [batch][heads][head_dim]; dev_lse fp32 [batch][heads]
 *                 natural-log LSE, or NULL
 *   sm_scale      score scale, 0 selects 1/sqrt(head_dim)
 * Limits: head_dim 128, heads / kv_heads in {1, 2, 4, 8, 16, 32}, batch
 * 1..64, batch * kv_heads <= 1024, ctx_stride a multiple of 16.  Its work list and partial summaries
 * live in a fixed 16 MiB device array inside the library, which every GPU
 * that loads the library holds until the process exits; a call whose
 * scratch would exceed it returns MAC_ERR_CAPACITY and launches nothing.
 * The first call on each device looks up that array's device address and
 * the kernels' launch shapes (with that device current); make that first
 * call before any stream capture.  All calls on a device share the array
 * and overwrite it: calls whose GPU work can overlap (other streams, other
 * host threads) race and must be serialised by the caller.  Async on
 * stream; returns MAC_ERR_INVALID_ARG for bad arguments, MAC_ERR_CUDA if a
 * launch fails.  Every block index the kernels form is checked on the host
 * first (lengths within ctx_stride), so this call has no device-side error
 * to report and none is read back: MAC_OK means the work was launched. */
mac_status mac_attention_noalloc(int batch, int heads, int kv_heads, int head_dim, int64_t ctx_stride,
                                 const void *dev_k, const void *dev_v, const int32_t *host_lens,
                                 const void *dev_q, void *dev_out, float *dev_lse, float sm_scale,
                                 void *stream);

/* Human-readable text for a status code (static storage). */
const char *mac_status_string(mac_status s);

/* Text of the handle's sticky error, or "" (owned by the handle). */
const char *mac_last_error(mac_handle h);

#ifdef __cplusplus
}
#endif

#endif /* MAC_H */
