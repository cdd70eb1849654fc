// Internal declarations shared by the kvs host runtime and its CUDA kernels.
// Nothing here is part of the C ABI (include/kvs.h is).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <string>

namespace kvs {

// Byte layout of one page (kvs_query_sizes in include/kvs.h states it).  Inside a
// head section, K codes sit in 16-token groups of one 32-byte line per
// (32-dim block, token) and V nibbles in 32-token chunks of one 32-byte line
// per (block, byte row); every tensor-core fragment is then one conflict-free
// 8-byte shared-memory load, and a whole head section is one bulk copy.
__host__ __device__ inline int64_t kq_byte(int64_t t, int d, int NB) {
    return ((t / 16 * NB + d / 32) * 16 + t % 16) * 32 + d % 32;
}
__host__ __device__ inline int64_t vq_byte(int64_t t, int row, int NB) {
    return ((t / 32 * NB + row / 16) * 16 + row % 16) * 32 + t % 32;
}

// Launch timeline (kvs_timeline_begin): a record is two words {~first CTA
// start, last CTA end} of %globaltimer (ns), each by atomic max from zero; a
// kernel given a null record pointer stamps nothing.
#ifdef __CUDACC__
__device__ __forceinline__ unsigned long long tl_now() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
// called by every CTA (thread 0 stamps)
__device__ __forceinline__ void tl_begin(unsigned long long *tl) {
    if (tl && threadIdx.x == 0) atomicMax(&tl[0], ~tl_now());
}
// called by thread 0 once the CTA's work is done
__device__ __forceinline__ void tl_finish(unsigned long long *tl) {
    if (tl && threadIdx.x == 0) atomicMax(&tl[1], tl_now());
}
#endif

struct PageGeom {
    int P;               // tokens per page
    int Hk;              // kv heads
    int D;               // head dim
    int64_t head_bytes;  // P*D*13/8: one kv head's section
    int64_t page_bytes;  // Hk*head_bytes
    int64_t ks_off;      // K scales  fp16 [P][D/32]   (K codes at 0, in kq_byte order)
    int64_t vq_off;      // V nibbles u8, P*D/2 bytes in vq_byte order (32-token chunks)
    int64_t vs_off;      // V scales  fp16 [D/32][P]
};

inline PageGeom make_geom(int P, int Hk, int D) {
    PageGeom g;
    g.P = P;
    g.Hk = Hk;
    g.D = D;
    g.ks_off = (int64_t)P * D;
    g.vq_off = g.ks_off + (int64_t)P * D / 16;
    g.vs_off = g.vq_off + (int64_t)P * D / 2;
    g.head_bytes = g.vs_off + (int64_t)P * D / 16;
    g.page_bytes = g.head_bytes * Hk;
    return g;
}

// ---------------------------------------------------------------- decode
// One item = one (page, device slot) pair; work units are (item, kv head),
// spread over persistent CTAs (at most one per SM).
constexpr int kMaxItems = 1024;

struct DecodeParams {
    const uint8_t *arena;  // slot 0 of the page-slot array
    PageGeom geom;
    const void *q;         // [R][Hq][D], fp32 or fp16
    int q_f16;
    float *part_o;         // [split][Hq][R][D]   split = logical page
    float *part_ml;        // [split][Hq][R][2]   (max in log2 units, sum)
    int *status;           // set to 1 if a bounded device wait timed out
    int R, Hq, G;          // R: query rows of the call (the partials' row stride)
    int row0, Rg;          // this launch's row group: query rows row0 .. row0 + Rg - 1
                           // (G * Rg <= 64 MMA rows; a call wider than that runs as groups)
    long long pos0;
    float scale_log2;      // scale * log2(e)
    int stages;            // shared-memory stages (set by launch_decode)
    const uint4 *qf;       // Q fragments [Hk][NT][D/16][32] (written by the Q prep kernel)
    int prep_q;            // launch_decode first (re)builds qf/qs from q
    int tile_mode;         // one CTA per (page, kv head, row tile) (ring chunks)
    int early_dependents;  // signal programmatic dependents (the chunk's refill) as soon as the
                           // page sections are in shared memory, before the softmax
    int max_sms;           // > 0: use at most this many SMs' worth of CTA slots (resident reads
                           // beside ring-chunk reads and refills); 0: every SM
    int qtiles, run_tiles; // set by launch_decode: fragment-layout row tiles, tiles to run
    int single_f16;        // Q and P' as single f16 operands (else f16 hi + lo pairs)
    int give_up_waits;     // test hook: every pipeline wait gives up at once, as if its copy
                           // never landed (the drain of copies in flight keeps its bound)
    unsigned long long *rec;  // ring-chunk read: the chunk's fill record (nullable, see FillParams)
    unsigned long long *acc;  // observation accumulator the first CTA adds the read to
    int rec_pages;            // pages of the chunk
    unsigned long long *tl;       // timeline record of the attention launch (nullable)
    unsigned long long *tl_prep;  // timeline record of the query-fragment launch (nullable)
    int n_items;
    uint32_t page[kMaxItems];
    uint32_t slot[kMaxItems];
};

// Returns cudaErrorInvalidValue for an unsupported (D, rows) combination.
// With p.prep_q set it first rebuilds the Q fragments (p.qf/p.qs) from p.q;
// n_items may then be 0 (Q prep only).
cudaError_t launch_decode(const DecodeParams &p, cudaStream_t s);
int decode_max_mma_rows();  // G*R bound served by launch_decode
// bytes of the Q-fragment area for Hk kv heads of head dim D
inline int64_t qfrag_bytes(int Hk, int D) {
    const int64_t qf = (int64_t)Hk * 8 * (D / 16) * 32 * 16;
    return (qf + 255) / 256 * 256;
}

// ---------------------------------------------------------------- prefill
// tcgen05 prefill: one split = up to kMaxPrefillSplitPages consecutive pages;
// grid = (splits, Hk * G * row tiles).  Q is fp16; D must be 256.
constexpr int kMaxPrefillSplits = 64;
constexpr int kMaxPrefillItems = 1024;
constexpr int kMaxPrefillSplitPages = 128;  // pages in one split of the tensor-core prefill path
struct PrefillParams {
    const uint8_t *arena;
    PageGeom geom;
    const void *q;     // fp16 [R][Hq][D]
    float *part_o;     // [split][Hq][R][D]
    float *part_ml;    // [split][Hq][R][2]
    int *status;       // set to 1 if a bounded device wait timed out
    int R, Hq, G;
    long long pos0;
    float scale_log2;
    unsigned long long *tl;  // timeline record (nullable)
    int n_splits;
    int split_begin[kMaxPrefillSplits + 1];  // item range of each split
    int split_id[kMaxPrefillSplits];         // logical split index (partials row)
    uint32_t page[kMaxPrefillItems];
    uint32_t slot[kMaxPrefillItems];
};
cudaError_t launch_prefill(const PrefillParams &p, cudaStream_t s);
int prefill_smem_bytes();

// ---------------------------------------------------------------- combine
struct CombineParams {
    const float *part_o;
    const float *part_ml;
    const int *status;  // nullable: when *status != 0 (a device wait gave up), every output is NaN
    float *out;   // [R][Hq][D]
    float *lse;   // [R][Hq] or null
    int R, Hq, D, P;
    int split_pages;  // pages per split (1 for decode, the prefill split otherwise)
    long long pos0;
    unsigned long long *tl;  // timeline record (nullable)
};
cudaError_t launch_combine(const CombineParams &p, cudaStream_t s);

// ---------------------------------------------------------------- append
// Quantise rows [n][Hk][D] of K (Q8_0) and V (Q4_0) into one page slot,
// token slots t0 .. t0+n-1 of that page.
struct QuantizeParams {
    const float *k;
    const float *v;
    uint8_t *page;  // device page base
    PageGeom geom;
    int t0, n;
    unsigned long long *tl;  // timeline record (nullable)
};
cudaError_t launch_quantize(const QuantizeParams &p, cudaStream_t s);

// Zero token slots [t0, P) of one device page (all sections of all heads).
cudaError_t launch_clear_tail(uint8_t *page, const PageGeom &g, int t0, cudaStream_t s,
                              unsigned long long *tl = nullptr);

// ---------------------------------------------------------------- ring fill
// Copy whole pages host -> device with SM loads (pinned host memory is
// directly addressable by the GPU).  One launch per ring chunk.
constexpr int kMaxFillPages = 64;
// Observation records.  A ring refill stamps its record {~start, end} (ns, by
// atomic max, from zero); the first CTA of the read of that chunk turns the
// record into counts in the accumulator and clears it.  A read that starts
// within kMissNs of its copy's end waited for the copy (a readiness miss).
constexpr int kObsRecords = 1024;               // records, indexed by chunk id
constexpr unsigned long long kMissNs = 4000;
struct ObsAccumulator {  // all fields start at zero
    unsigned long long reads, misses;
    unsigned long long occupancy_page_ns;  // sum of pages x (read start - fill end)
    unsigned long long fill_busy_ns;       // sum of fill durations
    unsigned long long first_fill_neg;     // ~(earliest fill start), by atomic max
    unsigned long long last_read;          // latest read start
    unsigned long long fill_bytes;         // page bytes of the accounted refills
};
struct FillParams {
    unsigned long long *rec;  // this refill's record (nullable)
    unsigned long long *tl;   // timeline record (nullable)
    int n;
    int64_t page_bytes;
    const uint8_t *src[kMaxFillPages];
    uint8_t *dst[kMaxFillPages];
};
// pdl: programmatic dependent launch (may start once the previous kernel on
// `s` has signalled its dependents; see decode_kernel)
cudaError_t launch_fill(const FillParams &p, cudaStream_t s, bool pdl = false);

// Per device and thread-safe: the SM count of the current device, and a raise
// of a kernel's dynamic shared-memory limit on the current device to at
// least `bytes` (made once per kernel and device).
int current_device_sms();
cudaError_t ensure_smem_limit(const void *kernel, int bytes);

// Message returned by kvs_last_error(NULL) on this thread.
void set_thread_error(const std::string &msg);

}  // namespace kvs
