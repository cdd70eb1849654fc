// KV writer (quantise + append into a device page) and ring refill kernels.
#include <cuda_fp16.h>
#include <math.h>

#include <map>
#include <mutex>
#include <utility>

#include "kvs_internal.h"

namespace kvs {
namespace {

// One warp per (token, kv head, 32-element block).  Encodes K as Q8_0 and V
// as Q4_0 with IEEE fp32 steps in a fixed order, so the codes match any
// other implementation of the same definition bit for bit:
//   Q8_0: d = max|x| / 127, id = 1/d (0 if d == 0), code = roundf(x * id)
//   Q4_0: m = the element of largest |x| (lowest index on ties), d = m / -8,
//         id = 1/d (0 if d == 0), code = min(15, trunc(x * id + 8.5))
// The KV writer of the V2 design ("SET_ROWS" with a runtime row base in the
// PR "port adaptive KV streaming") writes encoded rows at the page's token
// slot; here the slot is t0 + token.
__global__ void __launch_bounds__(256) quantize_kernel(const QuantizeParams p) {
    // a programmatic dependent launch: the rows and the page are touched only
    // once the kernels this launch depends on have completed
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int D = p.geom.D, NB = D / 32, Hk = p.geom.Hk, P = p.geom.P;
    const int64_t wid = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    tl_begin(p.tl);
    if (wid >= (int64_t)p.n * Hk * NB) return;
    const int b = (int)(wid % NB);
    const int g = (int)((wid / NB) % Hk);
    const int i = (int)(wid / ((int64_t)NB * Hk));
    const int t = p.t0 + i;
    const int64_t src = ((int64_t)i * Hk + g) * D + b * 32 + lane;
    uint8_t *hb = p.page + (int64_t)g * p.geom.head_bytes;

    // K -> Q8_0
    const float x = p.k[src];
    float amax = fabsf(x);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float d = __fdiv_rn(amax, 127.0f);
    const float id = (d != 0.0f) ? __fdiv_rn(1.0f, d) : 0.0f;
    const int qk = (int)roundf(__fmul_rn(x, id));
    hb[kq_byte(t, b * 32 + lane, NB)] = (uint8_t)(int8_t)qk;
    if (lane == 0) reinterpret_cast<__half *>(hb + p.geom.ks_off)[(int64_t)t * NB + b] = __float2half_rn(d);

    // V -> Q4_0
    const float y = p.v[src];
    float ay = fabsf(y);
    int idx = lane;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float ao = __shfl_xor_sync(0xffffffffu, ay, o);
        const int io = __shfl_xor_sync(0xffffffffu, idx, o);
        if (ao > ay || (ao == ay && io < idx)) {
            ay = ao;
            idx = io;
        }
    }
    const float mx = __shfl_sync(0xffffffffu, y, idx);
    const float dv = __fdiv_rn(mx, -8.0f);
    const float idv = (dv != 0.0f) ? __fdiv_rn(1.0f, dv) : 0.0f;
    const float u = __fadd_rn(__fmul_rn(y, idv), 8.5f);
    int c = __float2int_rz(u);
    c = c > 15 ? 15 : (c < 0 ? 0 : c);
    const int chi = __shfl_down_sync(0xffffffffu, c, 16);
    if (lane < 16) hb[p.geom.vq_off + vq_byte(t, b * 16 + lane, NB)] = (uint8_t)(c | (chi << 4));
    if (lane == 0) reinterpret_cast<__half *>(hb + p.geom.vs_off)[(int64_t)b * P + t] = __float2half_rn(dv);
    if (p.tl && lane == 0) atomicMax(&p.tl[1], tl_now());
}

// Zero token slots [t0, P) of every section of every head of one page.
__global__ void clear_tail_kernel(uint8_t *page, PageGeom g, int t0, unsigned long long *tl) {
    tl_begin(tl);
    const int64_t n = g.page_bytes;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t off = i % g.head_bytes;
        const int NB = g.D / 32;
        int64_t tok;
        if (off < g.ks_off) tok = off / (NB * 512) * 16 + (off / 32) % 16;               // K lines
        else if (off < g.vq_off) tok = (off - g.ks_off) / (g.D / 16);                     // K scales
        else if (off < g.vs_off) tok = (off - g.vq_off) / (NB * 512) * 32 + (off - g.vq_off) % 32;  // V lines
        else tok = ((off - g.vs_off) / 2) % g.P;                                          // V scales
        if (tok >= t0) page[i] = 0;
    }
    if (tl) {
        __syncthreads();
        tl_finish(tl);
    }
}

__device__ __forceinline__ uint4 ld_nc_u4(const void *p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// Host pages are read through their mapped device address, 16 bytes per
// load, kFillUnroll loads in flight per thread before the first store.  The
// grid covers the chunk's pages as one flat range and is capped at
// kFillMaxCtas: that keeps about 2 MiB of host reads in flight (far more
// than the host link's bandwidth x latency) while leaving the SMs to the
// attention launches that run beside the copy.
constexpr int kFillThreads = 512;
constexpr int kFillUnroll = 4;
constexpr int kFillMaxCtas = 64;

__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__global__ void __launch_bounds__(kFillThreads) fill_kernel(const __grid_constant__ FillParams p) {
    if (p.rec && threadIdx.x == 0) atomicMax(&p.rec[0], ~global_ns());  // earliest start, complemented
    tl_begin(p.tl);
    const uint32_t upp = (uint32_t)(p.page_bytes / 16);  // 16-byte units per page
    const uint32_t n = upp * (uint32_t)p.n;
    const uint32_t stride = gridDim.x * blockDim.x;
    for (uint32_t i0 = blockIdx.x * blockDim.x + threadIdx.x; i0 < n; i0 += kFillUnroll * stride) {
        uint4 v[kFillUnroll];
#pragma unroll
        for (int u = 0; u < kFillUnroll; ++u) {
            const uint32_t i = i0 + u * stride;
            if (i < n) {
                const uint32_t pg = i / upp;
                v[u] = ld_nc_u4(reinterpret_cast<const uint4 *>(p.src[pg]) + (i - pg * upp));
            }
        }
#pragma unroll
        for (int u = 0; u < kFillUnroll; ++u) {
            const uint32_t i = i0 + u * stride;
            if (i < n) {
                const uint32_t pg = i / upp;
                reinterpret_cast<uint4 *>(p.dst[pg])[i - pg * upp] = v[u];
            }
        }
    }
    if (p.rec || p.tl) {  // latest end: after every thread of this CTA has issued its stores
        __syncthreads();
        if (p.rec && threadIdx.x == 0) atomicMax(&p.rec[1], global_ns());
        tl_finish(p.tl);
    }
}

}  // namespace

cudaError_t launch_quantize(const QuantizeParams &p, cudaStream_t s) {
    if (p.n <= 0) return cudaSuccess;
    const int64_t warps = (int64_t)p.n * p.geom.Hk * (p.geom.D / 32);
    const int64_t blocks = (warps * 32 + 255) / 256;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3((unsigned)blocks);
    cfg.blockDim = dim3(256);
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, quantize_kernel, p);
    return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_clear_tail(uint8_t *page, const PageGeom &g, int t0, cudaStream_t s,
                              unsigned long long *tl) {
    if (t0 <= 0 && !tl) return cudaMemsetAsync(page, 0, (size_t)g.page_bytes, s);
    if (t0 >= g.P) return cudaSuccess;
    clear_tail_kernel<<<152, 256, 0, s>>>(page, g, t0 < 0 ? 0 : t0, tl);
    return cudaGetLastError();
}

cudaError_t launch_fill(const FillParams &p, cudaStream_t s, bool pdl) {
    if (p.n <= 0) return cudaSuccess;
    if (p.n > kMaxFillPages || p.page_bytes % 16 != 0) return cudaErrorInvalidValue;
    const int64_t units = p.page_bytes / 16 * p.n;
    if (units >= (int64_t)1 << 31) return cudaErrorInvalidValue;
    int64_t ctas = (units + (int64_t)kFillThreads * kFillUnroll - 1) / ((int64_t)kFillThreads * kFillUnroll);
    if (ctas > kFillMaxCtas) ctas = kFillMaxCtas;
    if (!pdl) {
        fill_kernel<<<(unsigned)ctas, kFillThreads, 0, s>>>(p);
        return cudaGetLastError();
    }
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3((unsigned)ctas);
    cfg.blockDim = dim3(kFillThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, fill_kernel, p);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

namespace {
std::mutex g_dev_mutex;
std::map<int, int> g_dev_sms;                        // device -> SM count
std::map<std::pair<const void *, int>, int> g_smem;  // (kernel, device) -> dynamic smem limit set
}  // namespace

int current_device_sms() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 1;
    std::lock_guard<std::mutex> lock(g_dev_mutex);
    auto it = g_dev_sms.find(dev);
    if (it != g_dev_sms.end()) return it->second;
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 1;
    g_dev_sms[dev] = n;
    return n;
}

cudaError_t ensure_smem_limit(const void *kernel, int bytes) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(g_dev_mutex);
    int &have = g_smem[std::make_pair(kernel, dev)];
    if (have >= bytes) return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess) have = bytes;
    return e;
}

}  // namespace kvs
