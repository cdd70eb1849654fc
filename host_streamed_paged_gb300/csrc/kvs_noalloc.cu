// kvs_attend_pages_noalloc: paged Q8_0/Q4_0 attention for callers that may
// not allocate device memory.
//
// Some callers cannot call cudaMalloc: code running inside a custom allocator
// or memory-pool callback, a plug-in that is handed a fixed memory budget by
// its host application, or a process that must not grow its device footprint
// once it is serving.  kvs_attend needs a caller-provided workspace for its
// split-K partials; this entry point instead keeps them in the file-scope
// device array below, so the caller passes only its pages, queries and
// outputs.
//
// The array is a fixed kNoallocScratchBytes (32 MiB) on every GPU that loads
// this library, held until the process exits.  Every call on a device shares
// it and it keeps the previous call's contents.  Its first 256 bytes hold the
// kernels' timeout flag, which a bounded device wait sets when it gives up;
// each call clears it on its stream (cudaMemsetAsync, which allocates
// nothing) before its first kernel, and the combine kernel reads it: if any
// wait of this call gave up, some partials were never written, and every
// element of out (and lse) becomes NaN instead of a value built from an
// earlier call's partials.  Then come the query fragments and the split
// partials, which each call writes before it reads them.  Calls whose work
// overlaps on the GPU (two streams, or two host threads) race on the array:
// order them on one stream.
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>
#include <string.h>

#include <mutex>
#include <string>

#include "kvs.h"
#include "kvs_internal.h"

namespace {

constexpr uint64_t kNoallocScratchBytes = 32ull << 20;
constexpr uint64_t kStatusBytes = 256;  // timeout flag at the start of the array
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

std::mutex g_setup_mutex;
void *g_scratch_addr[kMaxDevices] = {};

// Device address of g_noalloc_scratch on the current device, looked up once
// per device (the host-side symbol is not a device address).
kvs_status scratch_on_current_device(void **out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        kvs::set_thread_error(std::string("cudaGetDevice: ") + cudaGetErrorString(e));
        return KVS_ERR_CUDA;
    }
    if (dev < 0 || dev >= kMaxDevices) {
        kvs::set_thread_error("device index beyond the supported range");
        return KVS_ERR_UNSUPPORTED;
    }
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (!g_scratch_addr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || !p) {
            kvs::set_thread_error(std::string("cudaGetSymbolAddress(scratch): ") + cudaGetErrorString(e));
            return KVS_ERR_CUDA;
        }
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return KVS_OK;
}

}  // namespace

extern "C" kvs_status kvs_attend_pages_noalloc(const void *pages_dev, uint64_t pages_bytes,
                                               const uint32_t *page_slots, uint64_t n_pages,
                                               uint32_t page_tokens, uint32_t n_kv_head,
                                               uint32_t head_dim, const void *q_dev, int32_t q_dtype,
                                               uint32_t n_rows, uint32_t n_q_head, uint64_t pos0,
                                               float scale, float *out_dev, float *lse_dev,
                                               void *stream) {
    const uint32_t P = page_tokens, D = head_dim, Hk = n_kv_head;
    if (!(P == 32 || P == 64 || P == 128 || P == 256) || !(D == 64 || D == 128 || D == 256) || Hk == 0) {
        kvs::set_thread_error("page_tokens must be 32..256 (power of two), head_dim 64, 128 or 256");
        return KVS_ERR_UNSUPPORTED;
    }
    if (q_dtype != KVS_F32 && q_dtype != KVS_F16) {
        kvs::set_thread_error("q_dtype must be KVS_F32 or KVS_F16");
        return KVS_ERR_INVALID;
    }
    if (n_rows < 1 || n_q_head < Hk || n_q_head % Hk != 0) {
        kvs::set_thread_error("need n_rows >= 1 and n_q_head a positive multiple of n_kv_head");
        return KVS_ERR_INVALID;
    }
    if ((n_q_head / Hk) * n_rows > (uint32_t)kvs::decode_max_mma_rows()) {
        kvs::set_thread_error("n_rows * (n_q_head / n_kv_head) must be <= 64");
        return KVS_ERR_UNSUPPORTED;
    }
    if (!pages_dev || !page_slots || !q_dev || !out_dev) {
        kvs::set_thread_error("null pages, page table, q or out");
        return KVS_ERR_INVALID;
    }
    if (pos0 > (uint64_t)INT64_MAX - n_rows) {  // the last row's position must not wrap
        kvs::set_thread_error("pos0 + n_rows beyond the position range");
        return KVS_ERR_INVALID;
    }
    const uint64_t n_split = (pos0 + n_rows - 1) / P + 1;  // pages the rows can see
    if (n_split > n_pages) {
        kvs::set_thread_error("rows reach beyond the pages given");
        return KVS_ERR_CAPACITY;
    }
    const kvs::PageGeom geom = kvs::make_geom((int)P, (int)Hk, (int)D);
    const uint64_t per_split = (uint64_t)n_q_head * n_rows;
    const uint64_t qfrag = (uint64_t)kvs::qfrag_bytes((int)Hk, (int)D);
    const uint64_t split_bytes = per_split * (D + 2) * sizeof(float);  // one page's partials
    if (n_split > (kNoallocScratchBytes - kStatusBytes - qfrag) / split_bytes) {
        kvs::set_thread_error("needs " + std::to_string(n_split) + " pages x " + std::to_string(split_bytes) +
                              " bytes of split partials; the fixed scratch holds " +
                              std::to_string(kNoallocScratchBytes) + " (use kvs_attend with a workspace instead)");
        return KVS_ERR_CAPACITY;
    }
    for (uint64_t i = 0; i < n_split; ++i) {
        if (((uint64_t)page_slots[i] + 1) * (uint64_t)geom.page_bytes > pages_bytes) {
            kvs::set_thread_error("a page slot lies outside pages_bytes");
            return KVS_ERR_INVALID;
        }
    }
    void *scratch = nullptr;
    kvs_status s = scratch_on_current_device(&scratch);
    if (s != KVS_OK) return s;

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // the timeout flag must start at zero for this call
    cudaError_t ce = cudaMemsetAsync(scratch, 0, sizeof(int), st);
    if (ce != cudaSuccess) {
        kvs::set_thread_error(std::string("clearing the timeout flag: ") + cudaGetErrorString(ce));
        return KVS_ERR_CUDA;
    }
    kvs::DecodeParams dp;
    memset(&dp, 0, offsetof(kvs::DecodeParams, page));
    dp.arena = static_cast<const uint8_t *>(pages_dev);
    dp.geom = geom;
    dp.q = q_dev;
    dp.q_f16 = q_dtype == KVS_F16;
    dp.status = static_cast<int *>(scratch);
    uint8_t *qf_area = static_cast<uint8_t *>(scratch) + kStatusBytes;
    dp.qf = reinterpret_cast<const uint4 *>(qf_area);
    dp.part_o = reinterpret_cast<float *>(qf_area + qfrag);
    dp.part_ml = dp.part_o + n_split * per_split * D;
    dp.R = (int)n_rows;
    dp.row0 = 0;
    dp.Rg = (int)n_rows;  // one row group: G * n_rows <= 64
    dp.Hq = (int)n_q_head;
    dp.G = (int)(n_q_head / Hk);
    dp.pos0 = (long long)pos0;
    dp.scale_log2 = scale * 1.4426950408889634f;
    dp.prep_q = 1;  // the first launch also builds the query fragments
    for (uint64_t i0 = 0; i0 < n_split; i0 += kvs::kMaxItems) {
        const int n = (int)((n_split - i0) < (uint64_t)kvs::kMaxItems ? (n_split - i0) : kvs::kMaxItems);
        dp.n_items = n;
        for (int j = 0; j < n; ++j) {
            dp.page[j] = (uint32_t)(i0 + j);
            dp.slot[j] = page_slots[i0 + j];
        }
        cudaError_t e = kvs::launch_decode(dp, st);
        if (e != cudaSuccess) {
            kvs::set_thread_error(std::string("attention kernel launch: ") + cudaGetErrorString(e));
            return KVS_ERR_CUDA;
        }
        dp.prep_q = 0;
    }
    kvs::CombineParams cp;
    cp.part_o = dp.part_o;
    cp.part_ml = dp.part_ml;
    cp.status = dp.status;
    cp.out = out_dev;
    cp.lse = lse_dev;
    cp.R = (int)n_rows;
    cp.Hq = (int)n_q_head;
    cp.D = (int)D;
    cp.P = (int)P;
    cp.split_pages = 1;
    cp.pos0 = (long long)pos0;
    cp.tl = nullptr;
    cudaError_t e = kvs::launch_combine(cp, st);
    if (e != cudaSuccess) {
        kvs::set_thread_error(std::string("combine launch: ") + cudaGetErrorString(e));
        return KVS_ERR_CUDA;
    }
    return KVS_OK;
}
