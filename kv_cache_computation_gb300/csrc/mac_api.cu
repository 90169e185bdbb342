// Host side of the MAC-Attention decode-step library: the C ABI declared in
// include/mac.h.  Validates arguments, carves the caller's three device
// buffers, keeps host mirrors of the per-request lengths for capacity checks,
// and enqueues the per-step launch chain:
//
//   main stream : [wait Amend of the previous step] match_plan -> attention
//                 -> combine -> record "complete"
//   side stream : wait "complete" -> amend -> record "amend done"
//
// Nothing on the step path synchronises with the host or allocates.
#include "../../include/mac.h"
#include "mac_internal.cuh"

#include <algorithm>
#include <chrono>
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <new>
#include <thread>
#include <vector>

using namespace macgpu;

namespace {

constexpr size_t kAlign = 256;

size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

struct Carver {
    size_t off = 0;
    bool overflow = false;
    size_t take(size_t bytes)
    {
        const size_t o = off;
        const size_t n = align_up(bytes);
        if (n < bytes || off + n < off) overflow = true;
        off += n;
        return o;
    }
};

struct Sizes {
    size_t kv_each = 0, kv = 0, ring = 0, scratch = 0;
    int G = 0, pages_per_req = 0, num_pages = 0, ctx_stride = 0, item_cap = 0;
    size_t r_pos, r_q, r_o, r_lse;
    size_t s_page, s_kvlen, s_step, s_mcur, s_slot, s_own_slot, s_own_hit, s_dslot, s_dlo, s_dD, s_dqn2,
        s_forced, s_dkey, s_seedpos, s_qstash, s_glo, s_segc, s_goff, s_items, s_nitems, s_po, s_pml, s_afo, s_afl, s_apo,
        s_apl, s_stats, s_err;
};

bool valid_group(int G) { return G == 1 || G == 2 || G == 4 || G == 8 || G == 16 || G == 32; }

mac_status compute_sizes(const mac_config *c, Sizes *z)
{
    if (!c) return MAC_ERR_INVALID_ARG;
    if (c->heads < 1 || c->kv_heads < 1 || c->heads % c->kv_heads) return MAC_ERR_INVALID_ARG;
    const int G = c->heads / c->kv_heads;
    if (!valid_group(G)) return MAC_ERR_INVALID_ARG;
    if (c->head_dim != kD) return MAC_ERR_INVALID_ARG;
    if (c->ring_len < 1 || c->ring_len > kMaxRing) return MAC_ERR_INVALID_ARG;
    if (c->band_r < 1) return MAC_ERR_INVALID_ARG;
    if (!(c->tau >= 0.0) || !std::isfinite(c->tau)) return MAC_ERR_INVALID_ARG;
    if (c->max_batch < 1 || c->max_ctx < 1 || c->max_ctx > (int64_t(1) << 30)) return MAC_ERR_INVALID_ARG;
    if ((int64_t)c->max_batch * c->kv_heads > kMaxGroupsPerStep) return MAC_ERR_INVALID_ARG;
    if (c->page_size != 0 && c->page_size != kPage) return MAC_ERR_INVALID_ARG;
    if (c->num_pages < 0) return MAC_ERR_INVALID_ARG;
    if (!(c->sm_scale >= 0.f) || !std::isfinite(c->sm_scale)) return MAC_ERR_INVALID_ARG;
    if (c->plan_mode != 0 && c->plan_mode != 1) return MAC_ERR_INVALID_ARG;
    if (c->amend_band != 0 && c->amend_band != 1) return MAC_ERR_INVALID_ARG;

    const size_t B = c->max_batch, H = c->heads, Hkv = c->kv_heads, L = c->ring_len;
    z->G = G;
    z->pages_per_req = (int)((c->max_ctx + kPage - 1) / kPage);
    z->ctx_stride = z->pages_per_req * kPage;
    if (c->page_size == kPage) {
        const int64_t np = c->num_pages ? c->num_pages : (int64_t)c->max_batch * z->pages_per_req;
        if (np > 0x7fffffff) return MAC_ERR_INVALID_ARG;
        z->num_pages = (int)np;
        z->kv_each = (size_t)z->num_pages * Hkv * kPage * kD * 2;
    } else {
        z->num_pages = 0;
        z->kv_each = B * Hkv * (size_t)z->ctx_stride * kD * 2;
    }
    z->kv = 2 * align_up(z->kv_each);

    Carver r;
    z->r_pos = r.take(B * L * 4);
    z->r_q = r.take(B * H * L * kD * 2);
    z->r_o = r.take(B * H * L * kD * 4);
    z->r_lse = r.take(B * H * L * 4);
    z->ring = r.off;

    z->item_cap = 2 * kMaxCtas + 4 * (int)(B * Hkv);
    const size_t cap = z->item_cap, BH = B * H, BG = B * Hkv;
    Carver s;
    z->s_page = s.take(B * (size_t)z->pages_per_req * 4);
    z->s_kvlen = s.take(B * 4);
    z->s_step = s.take(B * 4);
    z->s_mcur = s.take(B * 4);
    z->s_slot = s.take(B * 4);
    z->s_own_slot = s.take(BH * 4);
    z->s_own_hit = s.take(BH * 4);
    z->s_dslot = s.take(BH * 4);
    z->s_dlo = s.take(BH * 4);
    z->s_dD = s.take(BH * 4);
    z->s_dqn2 = s.take(BH * 4);
    z->s_forced = s.take(BH * 4);
    z->s_dkey = s.take(BH * 8);
    z->s_seedpos = s.take(L * 4);
    z->s_qstash = s.take(BH * kD * 2);
    z->s_glo = s.take(BG * 4);
    z->s_segc = s.take(BG * 2 * 4);
    z->s_goff = s.take((BG + 1) * 4);
    z->s_items = s.take(cap * sizeof(int4));
    z->s_nitems = s.take(4);
    z->s_po = s.take(cap * G * kD * 4);
    z->s_pml = s.take(cap * G * 8);
    z->s_afo = s.take(BH * kD * 4);
    z->s_afl = s.take(BH * 4);
    z->s_apo = s.take(BH * kD * 4);
    z->s_apl = s.take(BH * 4);
    z->s_stats = s.take(kStCount * 8);
    z->s_err = s.take(4);
    z->scratch = s.off;
    if (r.overflow || s.overflow) return MAC_ERR_INVALID_ARG;
    return MAC_OK;
}

}  // namespace

struct mac_ctx {
    mac_config cfg;
    Sizes sz;
    Layout lay;
    int device = 0;
    int grid_ctas = 0;
    int grid_ctas_wide = 0;   // grid of the attention variant for steps of many groups (0: none)
    size_t attn_smem = 0;
    int grid_ctas_tc = 0;     // grid of the tcgen05 attention kernel (0: not available)
    uint64_t tc_steps = 0;    // steps whose attention ran on it
    TcMaps tc_maps{};         // its TMA descriptors of the two pools
    size_t attn_smem_tc = 0;
    cudaStream_t side = nullptr;
    cudaEvent_t ev_complete = nullptr, ev_amend = nullptr;
    bool amend_pending = false;
    unsigned long long amend_capture_id = 0;   // capture the outstanding Amend was recorded in (0: none)
    bool force_next = false;
    std::vector<int64_t> kv_len, steps, n_pages;
    mac_status sticky = MAC_OK;
    char errbuf[256] = {0};
    // profiling: 6 events per step (match start, match end, attention end,
    // combine end, amend start, amend end)
    bool prof = false;
    std::vector<cudaEvent_t> prof_ev;
    std::vector<char> prof_amend;   // per profiled step: the side-stream Amend ran (its two events are set)
    size_t prof_steps = 0;
    double prof_acc[4] = {0, 0, 0, 0};
    uint64_t prof_done = 0;
};

namespace {

constexpr size_t kProfCap = 2048;

bool log_on()
{
    static int on = -1;
    if (on < 0) {
        const char *e = std::getenv("MAC_LOG");
        on = (e && e[0] == '1') ? 1 : 0;
    }
    return on == 1;
}

mac_status fail_cuda(mac_ctx *h, cudaError_t e, const char *where)
{
    if (h) {
        h->sticky = MAC_ERR_CUDA;
        std::snprintf(h->errbuf, sizeof h->errbuf, "%s: %s", where, cudaGetErrorString(e));
        if (log_on()) std::fprintf(stderr, "[mac] %s\n", h->errbuf);
    }
    return MAC_ERR_CUDA;
}

#define MAC_CUDA(h, call)                                                   \
    do {                                                                    \
        cudaError_t e_ = (call);                                            \
        if (e_ != cudaSuccess) return fail_cuda((h), e_, #call);            \
    } while (0)

mac_status check_handle(mac_ctx *h)
{
    if (!h) return MAC_ERR_INVALID_ARG;
    return h->sticky;
}

bool aligned16(const void *p) { return ((uintptr_t)p & 15) == 0; }

// Make stream s wait for the outstanding side-stream Amend.  During stream
// capture the wait is legal only for an Amend recorded in the same capture;
// one recorded before the capture began must already have been waited for
// (mac_sync before capturing), so it is skipped.  *waited tells whether a
// wait was enqueued.
mac_status wait_amend(mac_ctx *h, cudaStream_t s, bool *waited)
{
    *waited = false;
    if (!h->amend_pending) return MAC_OK;
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    unsigned long long id = 0;
    MAC_CUDA(h, cudaStreamGetCaptureInfo(s, &cs, &id));
    if (cs == cudaStreamCaptureStatusActive && id != h->amend_capture_id) return MAC_OK;
    if (cs != cudaStreamCaptureStatusActive && h->amend_capture_id != 0) {
        // the outstanding Amend belongs to a captured graph, which mac_join
        // closed into the capturing stream: work ordered after its replay is
        // already behind it, and the event cannot be waited on outside the graph
        h->amend_pending = false;
        h->amend_capture_id = 0;
        return MAC_OK;
    }
    MAC_CUDA(h, cudaStreamWaitEvent(s, h->ev_amend, 0));
    *waited = true;
    return MAC_OK;
}

#define MAC_WAIT_AMEND(h, s)                                                \
    do {                                                                    \
        bool w_;                                                            \
        mac_status st_ = wait_amend((h), (s), &w_);                         \
        if (st_ != MAC_OK) return st_;                                      \
    } while (0)

int64_t capacity(const mac_ctx *h, int req)
{
    int64_t cap = h->cfg.max_ctx;
    if (h->cfg.page_size == kPage) {
        const int64_t pc = h->n_pages[req] * kPage;
        if (pc < cap) cap = pc;
    }
    return cap;
}

void prof_reset(mac_ctx *h)
{
    h->prof_steps = 0;
    for (double &x : h->prof_acc) x = 0;
    h->prof_done = 0;
}

mac_status prof_collect(mac_ctx *h)
{
    for (size_t s = 0; s < h->prof_steps; s++) {
        cudaEvent_t *e = &h->prof_ev[s * 6];
        float t[4] = {0, 0, 0, 0};
        MAC_CUDA(h, cudaEventSynchronize(e[3]));
        MAC_CUDA(h, cudaEventElapsedTime(&t[0], e[0], e[1]));
        MAC_CUDA(h, cudaEventElapsedTime(&t[1], e[1], e[2]));
        MAC_CUDA(h, cudaEventElapsedTime(&t[2], e[2], e[3]));
        if (h->prof_amend[s]) {   // otherwise Amend ran inside Combine (or the step had none): 0
            MAC_CUDA(h, cudaEventSynchronize(e[5]));
            MAC_CUDA(h, cudaEventElapsedTime(&t[3], e[4], e[5]));
        }
        for (int i = 0; i < 4; i++) h->prof_acc[i] += t[i];
        h->prof_done++;
    }
    h->prof_steps = 0;
    return MAC_OK;
}

// The step chain shared by mac_decode_step and mac_full_step.
mac_status run_step(mac_ctx *h, int batch, const void *q_pre, const void *q_post, const void *k_new,
                    const void *v_new, void *out, float *lse_out, void *stream, bool full, bool host_io = false)
{
    mac_status st = check_handle(h);
    if (st != MAC_OK) return st;
    if (batch < 1 || batch > h->cfg.max_batch) return MAC_ERR_INVALID_ARG;
    if ((!full && !q_pre) || !q_post || !k_new || !v_new || !out) return MAC_ERR_INVALID_ARG;
    if ((!full && !aligned16(q_pre)) || !aligned16(q_post) || !aligned16(k_new) || !aligned16(v_new) ||
        !aligned16(out) || ((uintptr_t)lse_out & 3))
        return MAC_ERR_INVALID_ARG;
    for (int b = 0; b < batch; b++)
        if (h->kv_len[b] + 1 > capacity(h, b)) return MAC_ERR_CAPACITY;

    cudaStream_t s = (cudaStream_t)stream;
    bool waited = false;
    st = wait_amend(h, s, &waited);
    if (st != MAC_OK) return st;

    StepArgs a{};
    a.batch = batch;
    a.q_pre = (const __nv_bfloat16 *)q_pre;
    a.q_post = (const __nv_bfloat16 *)q_post;
    a.k_new = (const __nv_bfloat16 *)k_new;
    a.v_new = (const __nv_bfloat16 *)v_new;
    a.out = (__nv_bfloat16 *)out;
    a.lse_out = lse_out;
    a.force = (!full && h->force_next) ? 1 : 0;
    a.full_mode = full ? 1 : 0;
    long long tokens = 0;   // KV tokens the step holds, all requests and KV heads
    for (int b = 0; b < batch; b++) tokens += h->kv_len[b] + 1;
    tokens *= h->lay.Hkv;
    a.tc = (h->grid_ctas_tc > 0 && tokens >= kTcMinTokens) ? 1 : 0;
    a.wide = (!a.tc && h->grid_ctas_wide > 0 && attention_wide(h->lay.G, batch * h->lay.Hkv)) ? 1 : 0;
    a.grid_ctas = a.tc ? h->grid_ctas_tc : (a.wide ? h->grid_ctas_wide : h->grid_ctas);
    a.plan_ctas = (a.tc && tokens >= kTcWaveTokens * a.grid_ctas) ? kTcPlanWaves * a.grid_ctas : a.grid_ctas;
    a.plan_mode = h->cfg.plan_mode;
    h->force_next = false;

    cudaEvent_t *pe = nullptr;
    if (h->prof && h->prof_steps < kProfCap) {
        h->prof_amend[h->prof_steps] = (!full && h->cfg.amend_band == 1) ? 1 : 0;
        pe = &h->prof_ev[h->prof_steps++ * 6];
    }
    // Programmatic dependent launch overlaps each launch with its
    // predecessor's tail; event records between the kernels (profiling)
    // would sit between them, so it is used only when not profiling.
    a.pdl = pe ? 0 : 1;
    // Match follows the previous step's combine directly in the stream only
    // when no side-stream Amend wait sits between them

    if (pe) MAC_CUDA(h, cudaEventRecord(pe[0], s));
    {
        StepArgs am = a;
        am.pdl = (a.pdl && !waited) ? 1 : 0;
        MAC_CUDA(h, launch_match_plan(h->lay, am, s));
    }
    if (pe) MAC_CUDA(h, cudaEventRecord(pe[1], s));
    {
        // inputs in host memory: the attention kernel takes the queries
        // from the device copy Match keeps (q_stash, same layout)
        StepArgs aa = a;
        if (host_io) aa.q_post = h->lay.q_stash;
        MAC_CUDA(h, launch_attention(h->lay, aa, &h->tc_maps, a.tc ? h->attn_smem_tc : h->attn_smem, s));
    }
    if (pe) MAC_CUDA(h, cudaEventRecord(pe[2], s));
    MAC_CUDA(h, launch_combine(h->lay, a, s));
    if (pe) MAC_CUDA(h, cudaEventRecord(pe[3], s));
    if (!full && h->cfg.amend_band == 1) {
        // Amend recomputes the band: its own kernel on the side stream
        MAC_CUDA(h, cudaEventRecord(h->ev_complete, s));
        MAC_CUDA(h, cudaStreamWaitEvent(h->side, h->ev_complete, 0));
        if (pe) MAC_CUDA(h, cudaEventRecord(pe[4], h->side));
        MAC_CUDA(h, launch_amend(h->lay, a, h->side));
        if (pe) MAC_CUDA(h, cudaEventRecord(pe[5], h->side));
        MAC_CUDA(h, cudaEventRecord(h->ev_amend, h->side));
        h->amend_pending = true;
        cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
        unsigned long long id = 0;
        MAC_CUDA(h, cudaStreamGetCaptureInfo(h->side, &cs, &id));
        h->amend_capture_id = cs == cudaStreamCaptureStatusActive ? id : 0;
    }
    for (int b = 0; b < batch; b++) {
        h->kv_len[b] += 1;
        if (!full) h->steps[b] += 1;
    }
    h->tc_steps += a.tc ? 1 : 0;
    return MAC_OK;
}

}  // namespace

extern "C" {

const char *mac_status_string(mac_status s)
{
    switch (s) {
    case MAC_OK: return "ok";
    case MAC_ERR_INVALID_ARG: return "invalid argument";
    case MAC_ERR_OOM: return "backing buffer too small or misaligned";
    case MAC_ERR_CUDA: return "CUDA error";
    case MAC_ERR_CAPACITY: return "KV capacity of a request exhausted";
    case MAC_ERR_TIMEOUT: return "timed out";
    case MAC_ERR_STATE: return "device bounds check fired";
    }
    return "unknown status";
}

const char *mac_last_error(mac_handle h) { return h ? h->errbuf : ""; }

mac_status mac_query_sizes(const mac_config *cfg, size_t *kv_bytes, size_t *ring_bytes, size_t *scratch_bytes)
{
    Sizes z;
    const mac_status st = compute_sizes(cfg, &z);
    if (st != MAC_OK) return st;
    if (kv_bytes) *kv_bytes = z.kv;
    if (ring_bytes) *ring_bytes = z.ring;
    if (scratch_bytes) *scratch_bytes = z.scratch;
    return MAC_OK;
}

mac_status mac_create(const mac_config *cfg, void *dev_kv, size_t kv_bytes, void *dev_ring, size_t ring_bytes,
                      void *dev_scratch, size_t scratch_bytes, mac_handle *out)
{
    if (!out) return MAC_ERR_INVALID_ARG;
    *out = nullptr;
    Sizes z;
    const mac_status st = compute_sizes(cfg, &z);
    if (st != MAC_OK) return st;
    if (!dev_kv || !dev_ring || !dev_scratch) return MAC_ERR_INVALID_ARG;
    if (((uintptr_t)dev_kv | (uintptr_t)dev_ring | (uintptr_t)dev_scratch) & (kAlign - 1)) return MAC_ERR_OOM;
    if (kv_bytes < z.kv || ring_bytes < z.ring || scratch_bytes < z.scratch) return MAC_ERR_OOM;

    mac_ctx *h = new (std::nothrow) mac_ctx();
    if (!h) return MAC_ERR_OOM;
    h->cfg = *cfg;
    h->sz = z;
    h->kv_len.assign(cfg->max_batch, 0);
    h->steps.assign(cfg->max_batch, 0);
    h->n_pages.assign(cfg->max_batch, 0);
    if (cfg->page_size == 0)
        for (auto &n : h->n_pages) n = z.pages_per_req;

    auto fail = [&](cudaError_t e, const char *where) {
        fail_cuda(h, e, where);
        if (log_on()) std::fprintf(stderr, "[mac] create failed: %s\n", h->errbuf);
        if (h->side) cudaStreamDestroy(h->side);
        if (h->ev_complete) cudaEventDestroy(h->ev_complete);
        if (h->ev_amend) cudaEventDestroy(h->ev_amend);
        delete h;
        return MAC_ERR_CUDA;
    };
    cudaError_t e = cudaGetDevice(&h->device);
    if (e != cudaSuccess) return fail(e, "cudaGetDevice");
    cudaDeviceProp prop;
    e = cudaGetDeviceProperties(&prop, h->device);
    if (e != cudaSuccess) return fail(e, "cudaGetDeviceProperties");
    if (prop.major * 10 + prop.minor != 103) return fail(cudaErrorNoKernelImageForDevice, "device check (sm_103a required)");
    // 32-head groups: the tcgen05 kernel needs TMA descriptors of the two
    // pools; if they cannot be made, the mma.sync kernel serves every step
    Layout &L = h->lay;
    int per_sm = 0;
    if (attention_tc_wanted(z.G)) {
        char *kvp = (char *)dev_kv;
        L.k_pool = (__nv_bfloat16 *)kvp;
        L.v_pool = (__nv_bfloat16 *)(kvp + align_up(z.kv_each));
        size_t smem_tc = 0;
        if (attention_tc_maps(L, h->tc_maps, (int64_t)(z.kv_each / (kD * 2))) == cudaSuccess &&
            attention_kernel_config(z.G, false, true, &smem_tc, &per_sm) == cudaSuccess && per_sm >= 1) {
            h->attn_smem_tc = smem_tc;
            h->grid_ctas_tc = std::min(prop.multiProcessorCount * per_sm, kMaxCtas);
        } else {
            L.tc = 0;
        }
        cudaGetLastError();
    }
    e = attention_kernel_config(z.G, false, false, &h->attn_smem, &per_sm);
    if (e != cudaSuccess) return fail(e, "attention kernel configuration");
    if (per_sm < 1) return fail(cudaErrorInvalidConfiguration, "attention kernel occupancy");
    h->grid_ctas = std::min(prop.multiProcessorCount * per_sm, kMaxCtas);
    if (attention_wide(z.G, kMaxGroupsPerStep)) {
        size_t smem_w = 0;
        e = attention_kernel_config(z.G, true, false, &smem_w, &per_sm);
        if (e != cudaSuccess) return fail(e, "attention kernel configuration");
        if (per_sm < 1 || smem_w != h->attn_smem) return fail(cudaErrorInvalidConfiguration, "attention kernel occupancy");
        h->grid_ctas_wide = std::min(prop.multiProcessorCount * per_sm, kMaxCtas);
    }
    e = amend_kernel_config();
    if (e != cudaSuccess) return fail(e, "amend kernel configuration");

    char *kv = (char *)dev_kv, *rg = (char *)dev_ring, *sc = (char *)dev_scratch;
    L.H = cfg->heads;
    L.Hkv = cfg->kv_heads;
    L.G = z.G;
    L.lo_parts = match_parts(z.G);
    L.ring_len = cfg->ring_len;
    L.band_r = cfg->band_r;
    L.max_batch = cfg->max_batch;
    L.paged = cfg->page_size == kPage;
    L.pages_per_req = z.pages_per_req;
    L.num_pages = z.num_pages;
    L.ctx_stride = z.ctx_stride;
    L.item_cap = z.item_cap;
    L.tau2 = (float)(cfg->tau * cfg->tau);
    const double scale = cfg->sm_scale > 0.f ? (double)cfg->sm_scale : 1.0 / std::sqrt((double)kD);
    L.scale_log2 = (float)(scale * 1.4426950408889634);
    L.k_pool = (__nv_bfloat16 *)kv;
    L.v_pool = (__nv_bfloat16 *)(kv + align_up(z.kv_each));
    L.ring_pos = (int32_t *)(rg + z.r_pos);
    L.ring_q = (__nv_bfloat16 *)(rg + z.r_q);
    L.ring_o = (float *)(rg + z.r_o);
    L.ring_lse = (float *)(rg + z.r_lse);
    L.page_table = (int32_t *)(sc + z.s_page);
    L.kv_len = (int32_t *)(sc + z.s_kvlen);
    L.step_ctr = (int32_t *)(sc + z.s_step);
    L.m_cur = (int32_t *)(sc + z.s_mcur);
    L.slot_cur = (int32_t *)(sc + z.s_slot);
    L.dec_own_slot = (int32_t *)(sc + z.s_own_slot);
    L.dec_own_hit = (int32_t *)(sc + z.s_own_hit);
    L.dec_slot = (int32_t *)(sc + z.s_dslot);
    L.dec_lo = (int32_t *)(sc + z.s_dlo);
    L.dec_D = (float *)(sc + z.s_dD);
    L.dec_qn2 = (float *)(sc + z.s_dqn2);
    L.forced_slot = (int32_t *)(sc + z.s_forced);
    L.dec_key = (unsigned long long *)(sc + z.s_dkey);
    L.seed_pos = (int32_t *)(sc + z.s_seedpos);
    L.q_stash = (__nv_bfloat16 *)(sc + z.s_qstash);
    L.grp_lo = (int32_t *)(sc + z.s_glo);
    L.seg_claim = (int32_t *)(sc + z.s_segc);
    L.grp_item_off = (int32_t *)(sc + z.s_goff);
    L.items = (int4 *)(sc + z.s_items);
    L.n_items = (int32_t *)(sc + z.s_nitems);
    L.part_o = (float *)(sc + z.s_po);
    L.part_ml = (float2 *)(sc + z.s_pml);
    L.as_full_o = (float *)(sc + z.s_afo);
    L.as_full_lse = (float *)(sc + z.s_afl);
    L.as_pre_o = (float *)(sc + z.s_apo);
    L.as_pre_lse = (float *)(sc + z.s_apl);
    L.amend_band = cfg->amend_band;
    L.stats = (unsigned long long *)(sc + z.s_stats);
    L.err = (uint32_t *)(sc + z.s_err);

    // Zero the KV store: a page's slots past a request's last token are
    // streamed (and masked to probability 0) with the rest of the page, and
    // 0 x NaN from never-written memory would still reach the output.
    e = cudaMemset(dev_kv, 0, z.kv);
    if (e != cudaSuccess) return fail(e, "cudaMemset(kv)");
    // zero the scratch (lengths, counters, ticket, page table) and the ring positions
    e = cudaMemset(dev_scratch, 0, z.scratch);
    if (e != cudaSuccess) return fail(e, "cudaMemset(scratch)");
    e = cudaMemset(rg + z.r_pos, 0, (size_t)cfg->max_batch * cfg->ring_len * 4);
    if (e != cudaSuccess) return fail(e, "cudaMemset(ring positions)");
    e = cudaMemset(sc + z.s_dkey, 0xff, (size_t)cfg->max_batch * cfg->heads * 8);   // "no entry" keys
    if (e != cudaSuccess) return fail(e, "cudaMemset(match keys)");
    e = cudaMemset(sc + z.s_glo, 0x7f, (size_t)cfg->max_batch * cfg->kv_heads * 4);   // above any position
    if (e != cudaSuccess) return fail(e, "cudaMemset(group span starts)");
    int lo_prio = 0, hi_prio = 0;
    e = cudaDeviceGetStreamPriorityRange(&lo_prio, &hi_prio);
    if (e != cudaSuccess) return fail(e, "cudaDeviceGetStreamPriorityRange");
    e = cudaStreamCreateWithPriority(&h->side, cudaStreamNonBlocking, lo_prio);
    if (e != cudaSuccess) return fail(e, "cudaStreamCreateWithPriority");
    e = cudaEventCreateWithFlags(&h->ev_complete, cudaEventDisableTiming);
    if (e != cudaSuccess) return fail(e, "cudaEventCreate");
    e = cudaEventCreateWithFlags(&h->ev_amend, cudaEventDisableTiming);
    if (e != cudaSuccess) return fail(e, "cudaEventCreate");
    e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return fail(e, "cudaDeviceSynchronize");
    if (log_on())
        std::fprintf(stderr, "[mac] create H=%d Hkv=%d L=%d r=%d tau=%g B=%d ctx=%lld paged=%d grid=%d smem=%zu\n",
                     L.H, L.Hkv, L.ring_len, L.band_r, cfg->tau, L.max_batch, (long long)cfg->max_ctx, L.paged,
                     h->grid_ctas, h->attn_smem);
    *out = h;
    return MAC_OK;
}

mac_status mac_destroy(mac_handle h)
{
    if (!h) return MAC_ERR_INVALID_ARG;
    if (h->side) cudaStreamSynchronize(h->side);
    cudaDeviceSynchronize();
    for (cudaEvent_t e : h->prof_ev)
        if (e) cudaEventDestroy(e);
    if (h->ev_complete) cudaEventDestroy(h->ev_complete);
    if (h->ev_amend) cudaEventDestroy(h->ev_amend);
    if (h->side) cudaStreamDestroy(h->side);
    delete h;
    return MAC_OK;
}

mac_status mac_set_page_table(mac_handle h, int req, const int32_t *dev_pages, int n_pages, void *stream)
{
    const mac_status st = check_handle(h);
    if (st != MAC_OK) return st;
    if (h->cfg.page_size != kPage) return MAC_ERR_INVALID_ARG;
    if (req < 0 || req >= h->cfg.max_batch || n_pages < 0 || n_pages > h->sz.pages_per_req) return MAC_ERR_INVALID_ARG;
    if (n_pages > 0 && !dev_pages) return MAC_ERR_INVALID_ARG;
    if ((int64_t)n_pages * kPage < h->kv_len[req]) return MAC_ERR_CAPACITY;
    cudaStream_t s = (cudaStream_t)stream;
    MAC_WAIT_AMEND(h, s);
    if (n_pages > 0)
        MAC_CUDA(h, cudaMemcpyAsync(h->lay.page_table + (size_t)req * h->sz.pages_per_req, dev_pages,
                                    (size_t)n_pages * 4, cudaMemcpyDeviceToDevice, s));
    h->n_pages[req] = n_pages;
    return MAC_OK;
}

mac_status mac_append_kv(mac_handle h, int req, const void *dev_k, const void *dev_v, int64_t n_tokens, void *stream)
{
    const mac_status st = check_handle(h);
    if (st != MAC_OK) return st;
    if (req < 0 || req >= h->cfg.max_batch || n_tokens < 0) return MAC_ERR_INVALID_ARG;
    if (n_tokens == 0) return MAC_OK;
    if (!dev_k || !dev_v || !aligned16(dev_k) || !aligned16(dev_v)) return MAC_ERR_INVALID_ARG;
    if (h->kv_len[req] + n_tokens > capacity(h, req)) return MAC_ERR_CAPACITY;
    cudaStream_t s = (cudaStream_t)stream;
    MAC_WAIT_AMEND(h, s);
    MAC_CUDA(h, launch_append(h->lay, req, (int)h->kv_len[req], (int)n_tokens, (const __nv_bfloat16 *)dev_k,
                              (const __nv_bfloat16 *)dev_v, s));
    h->kv_len[req] += n_tokens;
    return MAC_OK;
}

mac_status mac_decode_step(mac_handle h, int batch, const void *dev_q_pre, const void *dev_q_post,
                           const void *dev_k_new, const void *dev_v_new, void *dev_out, float *dev_lse_out,
                           void *stream)
{
    return run_step(h, batch, dev_q_pre, dev_q_post, dev_k_new, dev_v_new, dev_out, dev_lse_out, stream, false);
}

// The device's address of page-locked host memory (the same address under
// unified addressing); nullptr for anything else.
static void *host_for_device(const void *p)
{
    if (!p) return nullptr;
    cudaPointerAttributes at{};
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        (void)cudaGetLastError();
        return nullptr;
    }
    return at.type == cudaMemoryTypeHost ? at.devicePointer : nullptr;
}

mac_status mac_decode_step_host(mac_handle h, int batch, const void *host_q_pre, const void *host_q_post,
                                const void *host_k_new, const void *host_v_new, void *host_out,
                                float *host_lse_out, void *stream)
{
    const mac_status st = check_handle(h);
    if (st != MAC_OK) return st;
    const void *q_pre = host_for_device(host_q_pre), *q_post = host_for_device(host_q_post);
    const void *k_new = host_for_device(host_k_new), *v_new = host_for_device(host_v_new);
    void *out = host_for_device(host_out);
    float *lse = (float *)host_for_device(host_lse_out);
    if (!q_pre || !q_post || !k_new || !v_new || !out || (host_lse_out && !lse)) {
        std::snprintf(h->errbuf, sizeof h->errbuf, "a host buffer is not page-locked memory the device can address");
        return MAC_ERR_INVALID_ARG;
    }
    return run_step(h, batch, q_pre, q_post, k_new, v_new, out, lse, stream, false, true);
}

mac_status mac_full_step(mac_handle h, int batch, const void *dev_q_post, const void *dev_k_new,
                         const void *dev_v_new, void *dev_out, float *dev_lse_out, void *stream)
{
    return run_step(h, batch, nullptr, dev_q_post, dev_k_new, dev_v_new, dev_out, dev_lse_out, stream, true);
}

mac_status mac_join(mac_handle h, void *stream)
{
    const mac_status st = check_handle(h);
    if (st != MAC_OK) return st;
    MAC_WAIT_AMEND(h, (cudaStream_t)stream);
    return MAC_OK;
}

mac_status mac_sync(mac_handle h, int timeout_ms)
{
    const mac_status st = check_handle(h);
    if (st != MAC_OK) return st;
    if (h->amend_pending && h->amend_capture_id != 0) {   // captured Amend: ordered by the graph's stream
        h->amend_pending = false;
        h->amend_capture_id = 0;
    }
    if (h->amend_pending) {
        const auto t0 = std::chrono::steady_clock::now();
        for (;;) {
            const cudaError_t e = cudaEventQuery(h->ev_amend);
            if (e == cudaSuccess) break;
            if (e != cudaErrorNotReady) return fail_cuda(h, e, "cudaEventQuery(amend)");
            if (timeout_ms >= 0 && std::chrono::steady_clock::now() - t0 > std::chrono::milliseconds(timeout_ms))
                return MAC_ERR_TIMEOUT;
            std::this_thread::sleep_for(std::chrono::microseconds(20));
        }
    }
    uint32_t err = 0;
    MAC_CUDA(h, cudaMemcpy(&err, h->lay.err, 4, cudaMemcpyDeviceToHost));
    if (err) {
        h->sticky = MAC_ERR_STATE;
        std::snprintf(h->errbuf, sizeof h->errbuf, "device bounds check fired (bits 0x%x)", err);
        return MAC_ERR_STATE;
    }
    return MAC_OK;
}

mac_status mac_get_stats(mac_handle h, mac_stats *out)
{
    if (!h || !out) return MAC_ERR_INVALID_ARG;
    if (h->sticky == MAC_ERR_CUDA) return MAC_ERR_CUDA;
    MAC_CUDA(h, cudaDeviceSynchronize());
    unsigned long long v[kStCount];
    uint32_t err = 0;
    MAC_CUDA(h, cudaMemcpy(v, h->lay.stats, sizeof v, cudaMemcpyDeviceToHost));
    MAC_CUDA(h, cudaMemcpy(&err, h->lay.err, 4, cudaMemcpyDeviceToHost));
    std::memset(out, 0, sizeof *out);
    out->steps = v[kStSteps];
    out->head_decisions = v[kStDecisions];
    out->hits = v[kStHits];
    out->kv_tokens_read = v[kStKvRead];
    out->kv_tokens_full = v[kStKvFull];
    out->removal_direct = v[kStDirect];
    out->work_items = v[kStItems];
    out->device_error = err;
    out->tcgen05_steps = h->tc_steps;
    return MAC_OK;
}

mac_status mac_reset_stats(mac_handle h)
{
    const mac_status st = check_handle(h);
    if (st != MAC_OK) return st;
    MAC_CUDA(h, cudaDeviceSynchronize());
    MAC_CUDA(h, cudaMemset(h->lay.stats, 0, kStCount * 8));
    h->tc_steps = 0;
    return MAC_OK;
}

mac_status mac_reset_request(mac_handle h, int req, void *stream)
{
    const mac_status st = check_handle(h);
    if (st != MAC_OK) return st;
    if (req < 0 || req >= h->cfg.max_batch) return MAC_ERR_INVALID_ARG;
    cudaStream_t s = (cudaStream_t)stream;
    MAC_WAIT_AMEND(h, s);
    MAC_CUDA(h, cudaMemsetAsync(h->lay.ring_pos + (size_t)req * h->cfg.ring_len, 0, (size_t)h->cfg.ring_len * 4, s));
    MAC_CUDA(h, cudaMemsetAsync(h->lay.kv_len + req, 0, 4, s));
    MAC_CUDA(h, cudaMemsetAsync(h->lay.step_ctr + req, 0, 4, s));
    h->kv_len[req] = 0;
    h->steps[req] = 0;
    return MAC_OK;
}

mac_status mac_seed_ring(mac_handle h, int req, int n, const void *dev_q_pre, const float *dev_o,
                         const float *dev_lse, const int64_t *host_pos, void *stream)
{
    const mac_status st = check_handle(h);
    if (st != MAC_OK) return st;
    if (req < 0 || req >= h->cfg.max_batch || n < 0) return MAC_ERR_INVALID_ARG;
    if (n == 0) return MAC_OK;
    if (!dev_q_pre || !dev_o || !dev_lse || !host_pos || !aligned16(dev_q_pre) || !aligned16(dev_o) ||
        ((uintptr_t)dev_lse & 3))
        return MAC_ERR_INVALID_ARG;
    for (int i = 0; i < n; i++)
        if (host_pos[i] < 1 || host_pos[i] > h->kv_len[req] || (i > 0 && host_pos[i] <= host_pos[i - 1]))
            return MAC_ERR_INVALID_ARG;
    const int L = h->cfg.ring_len;
    const int first = n > L ? n - L : 0;   // only the last L entries survive the insertion
    std::vector<int32_t> pos(n - first);
    for (int i = first; i < n; i++) pos[i - first] = (int32_t)host_pos[i];
    cudaStream_t s = (cudaStream_t)stream;
    MAC_WAIT_AMEND(h, s);
    MAC_CUDA(h, cudaMemcpyAsync(h->lay.seed_pos, pos.data(), pos.size() * 4, cudaMemcpyHostToDevice, s));
    MAC_CUDA(h, launch_seed(h->lay, req, first, n, (int)h->steps[req], (const __nv_bfloat16 *)dev_q_pre, dev_o,
                            dev_lse, s));
    MAC_CUDA(h, cudaStreamSynchronize(s));   // the position staging buffer is reused by the next call
    h->steps[req] += n;
    return MAC_OK;
}

mac_status mac_set_profiling(mac_handle h, int enable)
{
    const mac_status st = check_handle(h);
    if (st != MAC_OK) return st;
    if (enable && h->prof_ev.empty()) {
        h->prof_ev.resize(kProfCap * 6, nullptr);
        h->prof_amend.assign(kProfCap, 0);
        for (auto &e : h->prof_ev) MAC_CUDA(h, cudaEventCreate(&e));
    }
    MAC_CUDA(h, cudaDeviceSynchronize());
    h->prof = enable != 0;
    prof_reset(h);
    return MAC_OK;
}

mac_status mac_get_profile(mac_handle h, mac_profile *out)
{
    if (!out) return MAC_ERR_INVALID_ARG;
    mac_status st = check_handle(h);
    if (st != MAC_OK) return st;
    st = prof_collect(h);
    if (st != MAC_OK) return st;
    out->match_plan_ms = h->prof_acc[0];
    out->attention_ms = h->prof_acc[1];
    out->combine_ms = h->prof_acc[2];
    out->amend_ms = h->prof_acc[3];
    out->steps = h->prof_done;
    return MAC_OK;
}

mac_status mac_debug_force_decisions(mac_handle h, const int32_t *dev_slot, int batch, void *stream)
{
    const mac_status st = check_handle(h);
    if (st != MAC_OK) return st;
    if (!dev_slot || batch < 1 || batch > h->cfg.max_batch) return MAC_ERR_INVALID_ARG;
    cudaStream_t s = (cudaStream_t)stream;
    MAC_WAIT_AMEND(h, s);
    MAC_CUDA(h, cudaMemcpyAsync(h->lay.forced_slot, dev_slot, (size_t)batch * h->cfg.heads * 4,
                                cudaMemcpyDeviceToDevice, s));
    h->force_next = true;
    return MAC_OK;
}

mac_status mac_debug_get_decisions(mac_handle h, int batch, int32_t *host_slot, int32_t *host_hit, float *host_D,
                                   float *host_qn2)
{
    const mac_status st = check_handle(h);
    if (st != MAC_OK) return st;
    if (batch < 1 || batch > h->cfg.max_batch) return MAC_ERR_INVALID_ARG;
    MAC_CUDA(h, cudaDeviceSynchronize());
    const size_t n = (size_t)batch * h->cfg.heads * 4;
    if (host_slot) MAC_CUDA(h, cudaMemcpy(host_slot, h->lay.dec_own_slot, n, cudaMemcpyDeviceToHost));
    if (host_hit) MAC_CUDA(h, cudaMemcpy(host_hit, h->lay.dec_own_hit, n, cudaMemcpyDeviceToHost));
    if (host_D) MAC_CUDA(h, cudaMemcpy(host_D, h->lay.dec_D, n, cudaMemcpyDeviceToHost));
    if (host_qn2) MAC_CUDA(h, cudaMemcpy(host_qn2, h->lay.dec_qn2, n, cudaMemcpyDeviceToHost));
    return MAC_OK;
}

mac_status mac_debug_read_ring(mac_handle h, int req, int32_t *host_pos, uint16_t *host_q, float *host_o,
                               float *host_lse, int64_t *kv_len, int64_t *steps)
{
    const mac_status st = check_handle(h);
    if (st != MAC_OK) return st;
    if (req < 0 || req >= h->cfg.max_batch) return MAC_ERR_INVALID_ARG;
    MAC_CUDA(h, cudaDeviceSynchronize());
    const size_t L = h->cfg.ring_len, H = h->cfg.heads;
    if (host_pos) MAC_CUDA(h, cudaMemcpy(host_pos, h->lay.ring_pos + req * L, L * 4, cudaMemcpyDeviceToHost));
    if (host_q)
        MAC_CUDA(h, cudaMemcpy(host_q, h->lay.ring_q + req * H * L * kD, H * L * kD * 2, cudaMemcpyDeviceToHost));
    if (host_o)
        MAC_CUDA(h, cudaMemcpy(host_o, h->lay.ring_o + req * H * L * kD, H * L * kD * 4, cudaMemcpyDeviceToHost));
    if (host_lse)
        MAC_CUDA(h, cudaMemcpy(host_lse, h->lay.ring_lse + req * H * L, H * L * 4, cudaMemcpyDeviceToHost));
    int32_t v[2] = {0, 0};
    MAC_CUDA(h, cudaMemcpy(&v[0], h->lay.kv_len + req, 4, cudaMemcpyDeviceToHost));
    MAC_CUDA(h, cudaMemcpy(&v[1], h->lay.step_ctr + req, 4, cudaMemcpyDeviceToHost));
    if (kv_len) *kv_len = v[0];
    if (steps) *steps = v[1];
    return MAC_OK;
}

}  // extern "C"
