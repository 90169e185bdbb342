// Decode attention for callers that cannot allocate device memory.
//
// Every other entry point works through a handle whose scratch (work list,
// partial summaries) lives in a buffer the caller allocated for mac_create.
// Some callers cannot allocate at all: a serving runtime that carves every
// byte of device memory out of one arena planned at start-up and forbids
// later allocations; a latency-critical loop that must not call cudaMalloc
// because it can synchronise the device; a plug-in host that hands the
// library only its input and output buffers.  For them,
// mac_attention_noalloc runs the full split-KV decode attention of
// mac_full_step over a KV cache the caller already holds, using a scratch
// area that is part of this library's device image: a file-scope
// __device__ array of kNoallocScratchBytes, held by every GPU that loads the
// library until the process exits (16 MiB each).  No call here allocates.
//
// The array is shared by every call on a device and keeps the previous
// call's contents.  Where each region sits depends on the call's shape, so a
// call finds another call's bytes under every region: it writes the plan
// inputs, the page-pool claim counters and the stats / error words before
// the attention kernel reads them, and the attention kernel writes the work
// list and partials before Combine reads them.  Calls whose GPU work
// overlaps (different streams, or different host threads on one device)
// race on it and must be serialised by the caller.
#include "../../include/mac.h"
#include "mac_internal.cuh"

#include <mutex>

using namespace macgpu;

namespace {

constexpr size_t kNoallocScratchBytes = size_t(16) << 20;   // 16 MiB per device
constexpr int kNoallocMaxBatch = 64;
constexpr int kNoallocMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

struct DeviceSetup {
    bool done = false;
    unsigned char *scratch = nullptr;   // device address of g_noalloc_scratch
    int sm_count = 0;
    int ctas[6] = {0, 0, 0, 0, 0, 0};    // attention grid per group size 1, 2, 4, 8, 16, 32
    size_t smem[6] = {0, 0, 0, 0, 0, 0};
};
DeviceSetup g_setup[kNoallocMaxDevices];
std::mutex g_setup_mutex;

int group_index(int G)
{
    switch (G) {
    case 1: return 0;
    case 2: return 1;
    case 4: return 2;
    case 8: return 3;
    case 16: return 4;
    case 32: return 5;
    }
    return -1;
}

struct NoallocPlanArgs {
    int batch, kv_heads;
    int lens[kNoallocMaxBatch];
};

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

// Byte offsets of the scratch regions for one call.
struct NoallocCarve {
    size_t items, n_items, goff, glo, segc, dec_lo, m_cur, kv_len, stats, err, part_ml, part_o, total;
};

NoallocCarve carve(int batch, int heads, int kv_heads, int item_cap)
{
    const int G = heads / kv_heads;
    NoallocCarve c{};
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t o = off;
        off += align256(bytes);
        return o;
    };
    c.items = take((size_t)item_cap * sizeof(int4));
    c.n_items = take(4);
    c.goff = take(((size_t)batch * kv_heads + 1) * 4);
    c.glo = take((size_t)batch * kv_heads * 4);
    c.segc = take((size_t)batch * kv_heads * 2 * 4);
    c.dec_lo = take((size_t)batch * heads * 4);
    c.m_cur = take((size_t)batch * 4);
    c.kv_len = take((size_t)batch * 4);
    c.stats = take(kStCount * 8);
    c.err = take(4);
    c.part_ml = take((size_t)item_cap * G * 8);
    c.part_o = take((size_t)item_cap * G * kD * 4);
    c.total = off;
    return c;
}

// One block: the span of every (request, KV head) group is [0, len); the
// attention kernel plans its work items from these.  Each group's two
// page-pool claim counters start at zero (the attention kernel takes pool
// pages by atomicAdd on them).
__global__ void noalloc_prepare_kernel(Layout L, NoallocPlanArgs p)
{
    const int nbg = p.batch * p.kv_heads;
    for (int bg = threadIdx.x; bg < nbg; bg += blockDim.x) L.grp_lo[bg] = 0;
    for (int i = threadIdx.x; i < 2 * nbg; i += blockDim.x) L.seg_claim[i] = 0;
    for (int i = threadIdx.x; i < p.batch * L.H; i += blockDim.x) L.dec_lo[i] = 0;
    for (int b = threadIdx.x; b < p.batch; b += blockDim.x) L.m_cur[b] = p.lens[b];
}

mac_status setup_device(int dev, DeviceSetup **out)
{
    if (dev < 0 || dev >= kNoallocMaxDevices) return MAC_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    DeviceSetup &s = g_setup[dev];
    if (!s.done) {
        cudaDeviceProp prop;
        if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return MAC_ERR_CUDA;
        if (prop.major * 10 + prop.minor != 103) return MAC_ERR_CUDA;
        // Host code sees g_noalloc_scratch only as a stand-in symbol: the
        // device address comes from the runtime, with this device current.
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) return MAC_ERR_CUDA;
        s.scratch = (unsigned char *)ptr;
        s.sm_count = prop.multiProcessorCount;
        const int groups[6] = {1, 2, 4, 8, 16, 32};
        for (int i = 0; i < 6; i++) {
            int per_sm = 0;
            if (attention_kernel_config(groups[i], false, false, &s.smem[i], &per_sm) != cudaSuccess || per_sm < 1)
                return MAC_ERR_CUDA;
            s.ctas[i] = s.sm_count * per_sm < kMaxCtas ? s.sm_count * per_sm : kMaxCtas;
        }
        s.done = true;
    }
    *out = &s;
    return MAC_OK;
}

}  // namespace

extern "C" mac_status mac_attention_noalloc(int batch, int heads, int kv_heads, int head_dim, int64_t ctx_stride,
                                            const void *dev_k, const void *dev_v, const int32_t *host_lens,
                                            const void *dev_q, void *dev_out, float *dev_lse, float sm_scale,
                                            void *stream)
{
    if (batch < 1 || batch > kNoallocMaxBatch || heads < 1 || kv_heads < 1 || heads % kv_heads) return MAC_ERR_INVALID_ARG;
    const int G = heads / kv_heads, gi = group_index(G);
    if (gi < 0 || head_dim != kD || batch * kv_heads > kMaxGroupsPerStep) return MAC_ERR_INVALID_ARG;
    if (ctx_stride < kPage || ctx_stride % kPage || ctx_stride > (int64_t(1) << 30)) return MAC_ERR_INVALID_ARG;
    if (!dev_k || !dev_v || !host_lens || !dev_q || !dev_out) return MAC_ERR_INVALID_ARG;
    if ((((uintptr_t)dev_k | (uintptr_t)dev_v | (uintptr_t)dev_q | (uintptr_t)dev_out) & 15) || ((uintptr_t)dev_lse & 3))
        return MAC_ERR_INVALID_ARG;
    if (!(sm_scale >= 0.f)) return MAC_ERR_INVALID_ARG;
    NoallocPlanArgs pa{};
    pa.batch = batch;
    pa.kv_heads = kv_heads;
    for (int b = 0; b < batch; b++) {
        if (host_lens[b] < 1 || host_lens[b] > ctx_stride) return MAC_ERR_INVALID_ARG;
        pa.lens[b] = host_lens[b];
    }
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MAC_ERR_CUDA;
    DeviceSetup *s = nullptr;
    const mac_status st = setup_device(dev, &s);
    if (st != MAC_OK) return st;

    const int grid = s->ctas[gi];
    const int item_cap = grid + 2 * batch * kv_heads;
    const NoallocCarve c = carve(batch, heads, kv_heads, item_cap);
    if (c.total > kNoallocScratchBytes) return MAC_ERR_CAPACITY;   // beyond the fixed scratch: nothing launched

    unsigned char *sc = s->scratch;
    Layout L{};
    L.H = heads;
    L.Hkv = kv_heads;
    L.G = G;
    L.lo_parts = 1;   // grp_lo is written by noalloc_prepare_kernel
    L.ring_len = 1;
    L.band_r = 1;
    L.max_batch = batch;
    L.paged = 0;
    L.pages_per_req = (int)(ctx_stride / kPage);
    L.ctx_stride = (int)ctx_stride;
    L.item_cap = item_cap;
    L.scale_log2 = (float)((sm_scale > 0.f ? (double)sm_scale : 1.0 / 11.313708498984761) * 1.4426950408889634);
    L.k_pool = (__nv_bfloat16 *)dev_k;
    L.v_pool = (__nv_bfloat16 *)dev_v;
    L.items = (int4 *)(sc + c.items);
    L.n_items = (int32_t *)(sc + c.n_items);
    L.grp_item_off = (int32_t *)(sc + c.goff);
    L.grp_lo = (int32_t *)(sc + c.glo);
    L.seg_claim = (int32_t *)(sc + c.segc);
    L.dec_lo = (int32_t *)(sc + c.dec_lo);
    L.m_cur = (int32_t *)(sc + c.m_cur);
    L.kv_len = (int32_t *)(sc + c.kv_len);
    L.stats = (unsigned long long *)(sc + c.stats);
    L.err = (uint32_t *)(sc + c.err);
    L.part_ml = (float2 *)(sc + c.part_ml);
    L.part_o = (float *)(sc + c.part_o);

    StepArgs a{};
    a.batch = batch;
    a.q_post = (const __nv_bfloat16 *)dev_q;
    a.out = (__nv_bfloat16 *)dev_out;
    a.lse_out = dev_lse;
    a.full_mode = 1;
    a.grid_ctas = grid;
    a.plan_ctas = grid;
    a.plan_mode = 0;
    a.pdl = 0;

    cudaStream_t cs = (cudaStream_t)stream;
    // counters and the error word only accumulate: start them at zero
    if (cudaMemsetAsync(sc + c.stats, 0, c.err + 4 - c.stats, cs) != cudaSuccess) return MAC_ERR_CUDA;
    noalloc_prepare_kernel<<<1, 256, 0, cs>>>(L, pa);
    if (cudaGetLastError() != cudaSuccess) return MAC_ERR_CUDA;
    if (launch_attention(L, a, nullptr, s->smem[gi], cs) != cudaSuccess) return MAC_ERR_CUDA;
    if (launch_combine(L, a, cs) != cudaSuccess) return MAC_ERR_CUDA;
    return MAC_OK;
}
