// Device helpers shared by the kernel translation units of the MAC-Attention
// decode step (mac_kernels.cu: Match, Combine, Amend and the KV/ring writers;
// mac_attention.cu: the planner and the split-KV attention kernel), and the
// launch helper with programmatic dependent launch.
#pragma once
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

// 16-byte copy whose first src_bytes (0 or 16) come from src and the rest
// are written as zeros; nothing is read from src when src_bytes is 0.
__device__ __forceinline__ void cp_async16_zfill(uint32_t dst, const void *src, uint32_t src_bytes)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
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

// 2^x by the hardware approximation (ex2.approx.ftz: relative error about
// 2^-22, results below 2^-126 flushed to 0; 2^-inf = 0).
__device__ __forceinline__ float ex2_approx(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
    return y;
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
    // m = ceil(2^k / c), below 2^27: a float quotient (within 2 ulp, i.e. 32,
    // of the exact one) corrected by integer steps -- no 64-bit division,
    // which costs about a thousand cycles in the plan's critical path
    const unsigned long long p2 = 1ull << k;
    unsigned long long m = (unsigned long long)__fdividef(__int_as_float((127 + k) << 23), (float)c);
    while (m * c < p2) m++;
    while ((m - 1) * c >= p2) m--;
    return {(unsigned)m, k};
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

}  // namespace

template <typename Kernel, typename... Args>
static cudaError_t launch_maybe_pdl(Kernel k, dim3 grid, dim3 block, size_t smem, cudaStream_t s, bool pdl,
                                    const Args &...args)
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
    return cudaLaunchKernelEx(&cfg, k, args...);
}

}  // namespace macgpu
