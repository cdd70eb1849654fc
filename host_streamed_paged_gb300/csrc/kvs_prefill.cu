// Prefill-chunk attention on the 5th-generation tensor cores (tcgen05).
//
// A prefill ubatch (up to 256 query rows, fp16 Q) attends causally over the
// paged Q8_0-K / Q4_0-V history.  Here QK^T and PV are dense contractions
// (1536 query rows per kv head at 6 query heads per kv head), so they run as
// tcgen05.mma with fp32 accumulators in tensor memory.  Every query tile
// reads a staged span before its ring slot may be reused (Adaptive KV
// Streaming for llama.cpp, "Batch and micro-batch sizes"): one launch covers
// every query tile of a key split.
//
// CTA = (key split, kv head, 128-row tile of one query head); 64-key blocks
// flow through a warp-specialised pipeline:
//   warps 4-7 (producers) dequantise block j's K (Q8_0) and V (Q4_0) into
//     shared memory as f16 pairs hi + lo, in the 128-byte-swizzled K-major
//     layout tcgen05 reads: hi = rn(d * x), lo = rn(d * x - hi) by one f16x2
//     multiply and one fused multiply-add (d * x has at most 18 significant
//     bits, so hi + lo is exact);
//   warp 8 (one thread) issues S_j = Q K_j^T (hi + lo, M 128, N 64, K 256)
//     into one of two TMEM score buffers, S_{j+1} before O += P_j V_j (hi + lo,
//     M 128, N 256, K 64), so the tensor pipe has work while the softmax runs;
//   warps 0-3 (one thread per row, TMEM lane = row) read S_j, scale, mask, run
//     the online softmax and write P_j (f16) to shared memory; O in TMEM is
//     rescaled only when a row's running max grows by more than 2^8 (the
//     weights are then formed against the stale max, which is exact).
// K, V and P are single-buffered: a block's K is rewritten once S_j is done,
// its V and P once PV_j is done; the fences are mbarriers (producer and
// softmax arrivals, tcgen05.commit for the MMAs).  At the end warps 0-3 write
// the split's unnormalised partial (m, l, O) for the log-sum-exp combine
// shared with the decode path.  Every wait is bounded; on a timeout the CTA
// raises an abort flag that ends every role's loop, waits (bounded) for its
// MMAs in flight and records a status code.
#include <cuda_fp16.h>
#include <math.h>

#include "kvs_internal.h"

namespace kvs {
namespace {

constexpr int kPThreads = 288;    // 4 softmax warps, 4 producer warps, 1 MMA warp
constexpr int kBN = 64;           // keys per block
constexpr int kD = 256;           // head dim served by this kernel
constexpr int kTileRows = 128;    // MMA M
constexpr uint32_t kSpinLimit = 1u << 26;

// shared-memory carve (bytes, 1024-aligned tiles for the 128B swizzle)
constexpr int kQBytes = kTileRows * kD * 2;  // 64 KB: 4 atoms of 128 rows x 128 B
constexpr int kKBytes = kBN * kD * 2;        // 32 KB: 4 atoms of 64 rows x 128 B
constexpr int kVBytes = kD * kBN * 2;        // 32 KB: 1 atom of 256 rows x 128 B
constexpr int kPBytes = kTileRows * kBN * 2; // 16 KB: 1 atom of 128 rows x 128 B
constexpr int kOffQ = 0;
constexpr int kOffKh = kOffQ + kQBytes;
constexpr int kOffKl = kOffKh + kKBytes;
constexpr int kOffVh = kOffKl + kKBytes;
constexpr int kOffVl = kOffVh + kVBytes;
constexpr int kOffP = kOffVl + kVBytes;       // two P buffers
constexpr int kOffBar = kOffP + 2 * kPBytes;  // mbarriers (kNumBars x 8 B)
constexpr int kNumBars = 12;
constexpr int kOffTmem = kOffBar + kNumBars * 8;  // TMEM base address written by tcgen05.alloc
constexpr int kOffAbort = kOffTmem + 8;
constexpr int kSmemBytes = kOffAbort + 8 + 1024;  // + slack to align the base to 1024

constexpr uint32_t kTmemCols = 512;  // S buffers at [0, 64) and [64, 128), O at [128, 384)
constexpr uint32_t kColS = 0, kColO = 128;
// barrier indices; a "+ buffer" barrier has one phase per use of that buffer,
// so no waiter can fall two phases behind the barrier it waits on
constexpr int kBarKFull = 0, kBarVFull = 1, kBarKEmpty = 2;
constexpr int kBarPFull = 3;   // + P buffer (2)
constexpr int kBarODone = 5;   // + P buffer (2): PV_j done, committed on buffer j & 1
constexpr int kBarSFull = 7;   // + S buffer (2)
constexpr int kBarSEmpty = 9;  // + S buffer (2)
constexpr int kBarFinal = 11;

// byte offset of element (row, k) in a 128B-swizzled K-major tile whose rows
// are 128-byte lines of 64 f16 (one swizzle atom per 64 elements of k)
__device__ __forceinline__ uint32_t sw128(int rows, int row, int k) {
    const int atom = k >> 6, kk = k & 63;
    const int chunk = (kk >> 3) ^ (row & 7);
    return (uint32_t)(atom * rows * 128 + row * 128 + chunk * 16 + (kk & 7) * 2);
}

__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFF) >> 4);       // start address
    d |= (uint64_t)1 << 16;                        // leading byte offset (unused for SW128 K-major)
    d |= (uint64_t)(1024 >> 4) << 32;              // stride byte offset: 8 rows x 128 B
    d |= (uint64_t)1 << 46;                        // descriptor version for tcgen05
    d |= (uint64_t)2 << 61;                        // layout: 128-byte swizzle
    return d;
}

// kind::f16 instruction descriptor: D f32, A/B f16, both K-major
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N) {
    return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ uint32_t smem_u32(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count));
}

// bounded wait for phase `parity` of an mbarrier; false on timeout or once
// another role of the CTA has raised *abort (which this wait also raises)
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int *abort) {
    for (uint32_t i = 0; i < kSpinLimit; ++i) {
        uint32_t done;
        asm volatile(
            "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
            : "=r"(done)
            : "r"(bar), "r"(parity)
            : "memory");
        if (done) return true;
        if ((i & 255) == 255 && *abort) return false;
    }
    *abort = 1;
    return false;
}

// the same wait taken by every lane of a warp, with one warp-wide outcome
__device__ __forceinline__ bool mbar_wait_warp(uint32_t bar, uint32_t parity, volatile int *abort) {
    return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort));
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(idesc), "r"(acc));
}

__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void tc_before_sync() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_after_sync() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void proxy_fence() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// 32 lanes x 32 columns of fp32 from TMEM (one row per thread)
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float (&v)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])), "r"(__float_as_uint(v[3])),
        "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])), "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])),
        "r"(__float_as_uint(v[8])), "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
        "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])), "r"(__float_as_uint(v[15])),
        "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])), "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])),
        "r"(__float_as_uint(v[20])), "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
        "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])), "r"(__float_as_uint(v[27])),
        "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])), "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
        : "memory");
}

// 4 int8 (bytes of w) -> f16x2 (x0, x1), (x2, x3), exact (see kvs_decode.cu)
__device__ __forceinline__ void i8x4_to_f16(uint32_t w, uint32_t &a, uint32_t &b) {
    const uint32_t u = w ^ 0x80808080u;
    uint32_t bl, bh;
    asm("prmt.b32 %0, %1, %2, 0x4140;" : "=r"(bl) : "r"(u), "r"(0x64646464u));
    asm("prmt.b32 %0, %1, %2, 0x4342;" : "=r"(bh) : "r"(u), "r"(0x64646464u));
    asm("sub.f16x2 %0, %1, %2;" : "=r"(a) : "r"(bl), "r"(0x64806480u));
    asm("sub.f16x2 %0, %1, %2;" : "=r"(b) : "r"(bh), "r"(0x64806480u));
}

// x * d -> (hi, lo) with hi = rn(x d), lo = rn(x d - hi) (exact remainder)
__device__ __forceinline__ void mul_split(uint32_t x, uint32_t d, uint32_t &hi, uint32_t &lo) {
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(hi) : "r"(x), "r"(d));
    const uint32_t nh = hi ^ 0x80008000u;
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(lo) : "r"(x), "r"(d), "r"(nh));
}

__global__ void __launch_bounds__(kPThreads, 1) prefill_kernel(const __grid_constant__ PrefillParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int split_idx = blockIdx.x;
    const int G = p.G, R = p.R, rt = (R + kTileRows - 1) / kTileRows;
    const int g = blockIdx.y / (G * rt);
    const int tile = blockIdx.y % (G * rt);
    const int hl = tile / rt, r0 = (tile % rt) * kTileRows;
    const int h = g * G + hl;
    const int P = p.geom.P, bpp = P / kBN;  // blocks per page
    const int it0 = p.split_begin[split_idx], it1 = p.split_begin[split_idx + 1];
    const int split = p.split_id[split_idx];
    const long long last_pos = p.pos0 + ((r0 + kTileRows < R) ? (r0 + kTileRows) : R) - 1;  // tile's last row

    const uint32_t bar0 = smem_u32(smem + kOffBar);
    auto bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + kOffTmem);
    volatile int *abort = reinterpret_cast<volatile int *>(smem + kOffAbort);

    // blocks of this split the tile can see (pages ascend, so the first masked one ends the list)
    int nblk = 0;
    for (int j = 0; j < (it1 - it0) * bpp; ++j) {
        const long long kpos0 = (long long)p.page[it0 + j / bpp] * P + (j % bpp) * kBN;
        if (kpos0 > last_pos) break;
        nblk = j + 1;
    }
    auto page_base = [&](int j) {
        return p.arena + (int64_t)p.slot[it0 + j / bpp] * p.geom.page_bytes + (int64_t)g * p.geom.head_bytes;
    };

    if (tid == 0) {
        mbar_init(bar(kBarKFull), 4);
        mbar_init(bar(kBarVFull), 4);
        mbar_init(bar(kBarPFull), 4);
        mbar_init(bar(kBarPFull + 1), 4);
        mbar_init(bar(kBarKEmpty), 1);
        mbar_init(bar(kBarODone), 1);
        mbar_init(bar(kBarODone + 1), 1);
        mbar_init(bar(kBarSFull), 1);
        mbar_init(bar(kBarSFull + 1), 1);
        mbar_init(bar(kBarSEmpty), 4);
        mbar_init(bar(kBarSEmpty + 1), 4);
        mbar_init(bar(kBarFinal), 1);
        *abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                     "r"(kTmemCols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    // Q tile -> shared memory (f16, swizzled); rows past R are zero
    {
        const __half *q = reinterpret_cast<const __half *>(p.q);
        for (int c = tid; c < kTileRows * (kD / 8); c += kPThreads) {
            const int row = c / (kD / 8), k = (c % (kD / 8)) * 8;
            uint4 v = make_uint4(0, 0, 0, 0);
            if (r0 + row < R) v = *reinterpret_cast<const uint4 *>(q + ((int64_t)(r0 + row) * p.Hq + h) * kD + k);
            *reinterpret_cast<uint4 *>(smem + kOffQ + sw128(kTileRows, row, k)) = v;
        }
    }
    proxy_fence();
    tc_before_sync();
    __syncthreads();
    tc_after_sync();
    const uint32_t tmem = *tmem_slot;

    if (warp >= 4 && warp < 8) {
        // ------------------------------------------------------------ producers
        // Raw bytes of block j+1 are loaded into registers before the wait
        // for block j's slot, so their latency hides behind the pipeline.
        const int pt = tid - 128;  // 0..127
        uint2 rk[16], rv[8];
        __half sk[16];
        uint4 sv[8];
        auto load_k = [&](int j) {
            const uint8_t *hb = page_base(j);
            const int kb = (j % bpp) * kBN;
            const __half *ks = reinterpret_cast<const __half *>(hb + p.geom.ks_off);
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const int c = pt + 128 * i, key = c >> 5, k = (c & 31) * 8;
                rk[i] = *reinterpret_cast<const uint2 *>(hb + kq_byte(kb + key, k, kD / 32));
                sk[i] = ks[(kb + key) * (kD / 32) + (k >> 5)];
            }
        };
        auto load_v = [&](int j) {
            const uint8_t *hb = page_base(j);
            const int kb = (j % bpp) * kBN;
            const __half *vs = reinterpret_cast<const __half *>(hb + p.geom.vs_off);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int pc = pt + 128 * i, br = pc >> 3, k8 = (pc & 7) * 8;
                rv[i] = *reinterpret_cast<const uint2 *>(hb + p.geom.vq_off + vq_byte(kb + k8, br, kD / 32));
                sv[i] = *reinterpret_cast<const uint4 *>(vs + (br >> 4) * P + kb + k8);
            }
        };
        // K of block j+1 needs only S_j finished, V of block j needs PV_{j-1}
        // finished; S_j runs before PV_{j-1}, so K goes first.
        auto write_k = [&](int j) {
            const int kb = (j % bpp) * kBN;
            (void)kb;
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const int c = pt + 128 * i, key = c >> 5, k = (c & 31) * 8;
                const __half2 d2 = __halves2half2(sk[i], sk[i]);
                const uint32_t d = *reinterpret_cast<const uint32_t *>(&d2);
                uint32_t x[4], hi[4], lo[4];
                i8x4_to_f16(rk[i].x, x[0], x[1]);
                i8x4_to_f16(rk[i].y, x[2], x[3]);
#pragma unroll
                for (int e = 0; e < 4; ++e) mul_split(x[e], d, hi[e], lo[e]);
                const uint32_t off = sw128(kBN, key, k);
                *reinterpret_cast<uint4 *>(smem + kOffKh + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
                *reinterpret_cast<uint4 *>(smem + kOffKl + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
            }
            proxy_fence();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(kBarKFull));
        };
        // V: 128 byte rows (dim pairs) x 8 chunks of 8 keys -> [dim][key] tiles
        auto write_v = [&]() {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int pc = pt + 128 * i, br = pc >> 3, k8 = (pc & 7) * 8;
                const int dA = (br >> 4) * 32 + (br & 15), dB = dA + 16;
                const uint32_t w[2] = {rv[i].x, rv[i].y};
                const uint32_t dv[4] = {sv[i].x, sv[i].y, sv[i].z, sv[i].w};  // (k, k+1) scale pairs
                uint32_t ah[4], al[4], bh[4], bl[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    // keys 2e, 2e+1: bytes 2(e%2), 2(e%2)+1 of w[e/2], one per f16 half
                    uint32_t sp;
                    const uint32_t sel = (e & 1) ? 0x7372u : 0x7170u;
                    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(sp) : "r"(w[e >> 1]), "r"(0u), "r"(sel));
                    uint32_t lo_n, hi_n, xa, xb;
                    asm("lop3.b32 %0, %1, %2, %3, 0xea;" : "=r"(lo_n) : "r"(sp), "r"(0x000f000fu), "r"(0x64006400u));
                    asm("lop3.b32 %0, %1, %2, %3, 0xea;" : "=r"(hi_n) : "r"(sp >> 4), "r"(0x000f000fu), "r"(0x64006400u));
                    asm("sub.f16x2 %0, %1, %2;" : "=r"(xa) : "r"(lo_n), "r"(0x64086408u));  // code - 8
                    asm("sub.f16x2 %0, %1, %2;" : "=r"(xb) : "r"(hi_n), "r"(0x64086408u));
                    mul_split(xa, dv[e], ah[e], al[e]);
                    mul_split(xb, dv[e], bh[e], bl[e]);
                }
                const uint32_t oa = sw128(kD, dA, k8), ob = sw128(kD, dB, k8);
                *reinterpret_cast<uint4 *>(smem + kOffVh + oa) = make_uint4(ah[0], ah[1], ah[2], ah[3]);
                *reinterpret_cast<uint4 *>(smem + kOffVl + oa) = make_uint4(al[0], al[1], al[2], al[3]);
                *reinterpret_cast<uint4 *>(smem + kOffVh + ob) = make_uint4(bh[0], bh[1], bh[2], bh[3]);
                *reinterpret_cast<uint4 *>(smem + kOffVl + ob) = make_uint4(bl[0], bl[1], bl[2], bl[3]);
            }
            proxy_fence();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(kBarVFull));
        };
        if (nblk > 0) {
            load_k(0);
            load_v(0);
            write_k(0);
            if (nblk > 1) load_k(1);
        }
        for (int j = 0; j < nblk; ++j) {  // every exit is a warp-uniform wait outcome
            if (j + 1 < nblk) {
                if (!mbar_wait_warp(bar(kBarKEmpty), (uint32_t)(j & 1), abort)) break;  // S_j done
                write_k(j + 1);
                if (j + 2 < nblk) load_k(j + 2);
            }
            if (j >= 1 && !mbar_wait_warp(bar(kBarODone + ((j - 1) & 1)), (uint32_t)(((j - 1) >> 1) & 1), abort))
                break;  // PV_{j-1} done
            write_v();
            if (j + 1 < nblk) load_v(j + 1);
        }
    } else if (warp == 8) {
        // ------------------------------------------------------------ MMA issue (one thread)
        if (lane == 0) {
            // descriptors of the tile bases; a k-step adds its byte offset / 16
            const uint64_t dq = smem_desc(smem_u32(smem + kOffQ)), dkh = smem_desc(smem_u32(smem + kOffKh));
            const uint64_t dkl = smem_desc(smem_u32(smem + kOffKl)), dvh = smem_desc(smem_u32(smem + kOffVh));
            const uint64_t dvl = smem_desc(smem_u32(smem + kOffVl)), dp = smem_desc(smem_u32(smem + kOffP));
            const uint32_t id_s = idesc_f16(kTileRows, kBN), id_o = idesc_f16(kTileRows, kD);
            auto issue_s = [&](int j) {
                const uint32_t ts = tmem + kColS + (uint32_t)((j & 1) * kBN);
#pragma unroll
                for (int s = 0; s < kD / 16; ++s) {
                    const uint32_t ao = ((s >> 2) * (kTileRows * 128) + (s & 3) * 32) >> 4;
                    const uint32_t bo = ((s >> 2) * (kBN * 128) + (s & 3) * 32) >> 4;
                    mma_f16(ts, dq + ao, dkh + bo, id_s, s > 0);
                    mma_f16(ts, dq + ao, dkl + bo, id_s, 1);
                }
                mma_commit(bar(kBarSFull + (j & 1)));
                mma_commit(bar(kBarKEmpty));
            };
            bool ok = true;
            if (nblk > 0) {
                ok = mbar_wait(bar(kBarKFull), 0u, abort);
                if (ok) {
                    tc_after_sync();
                    issue_s(0);
                }
            }
            for (int j = 0; j < nblk && ok; ++j) {
                if (j + 1 < nblk) {
                    ok = mbar_wait(bar(kBarKFull), (uint32_t)((j + 1) & 1), abort);
                    if (ok && j + 1 >= 2) ok = mbar_wait(bar(kBarSEmpty + ((j + 1) & 1)), (uint32_t)(((j - 1) >> 1) & 1), abort);
                    if (!ok) break;
                    tc_after_sync();
                    issue_s(j + 1);
                }
                ok = mbar_wait(bar(kBarPFull + (j & 1)), (uint32_t)((j >> 1) & 1), abort) &&
                     mbar_wait(bar(kBarVFull), (uint32_t)(j & 1), abort);
                if (!ok) break;
                tc_after_sync();
                const uint64_t dpj = dp + (uint64_t)(((j & 1) * kPBytes) >> 4);
#pragma unroll
                for (int s = 0; s < kBN / 16; ++s) {
                    mma_f16(tmem + kColO, dpj + (s * 32 >> 4), dvh + (s * 32 >> 4), id_o, (j > 0 || s > 0) ? 1u : 0u);
                    mma_f16(tmem + kColO, dpj + (s * 32 >> 4), dvl + (s * 32 >> 4), id_o, 1);
                }
                mma_commit(bar(kBarODone + (j & 1)));
            }
            // every MMA this thread issued has finished before TMEM is read or freed
            mma_commit(bar(kBarFinal));
            volatile int no_abort = 0;
            mbar_wait(bar(kBarFinal), 0u, &no_abort);
        }
    } else {
        // ------------------------------------------------------------ softmax rows (warps 0-3)
        const int row = tid;
        const long long qpos = p.pos0 + r0 + row;
        const bool row_valid = r0 + row < R;
        const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
        float m_used = -INFINITY, l_sum = 0.f;
        bool ok = true;
        for (int j = 0; j < nblk && ok; ++j) {
            const long long kpos0 = (long long)p.page[it0 + j / bpp] * P + (j % bpp) * kBN;
            ok = mbar_wait_warp(bar(kBarSFull + (j & 1)), (uint32_t)((j >> 1) & 1), abort);
            if (!ok) break;
            tc_after_sync();
            float s[kBN];
            {
                float t32[32];
                const uint32_t ta = lane_base + kColS + (uint32_t)((j & 1) * kBN);
                tmem_ld32(ta, t32);
#pragma unroll
                for (int i = 0; i < 32; ++i) s[i] = t32[i];
                tmem_ld32(ta + 32, t32);
#pragma unroll
                for (int i = 0; i < 32; ++i) s[32 + i] = t32[i];
            }
            tc_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(kBarSEmpty + (j & 1)));
            // causal mask only where the block reaches past this row (keys i > lim)
            const long long lim64 = row_valid ? qpos - kpos0 : -1;
            if (lim64 < kBN - 1) {
                const int lim = (int)(lim64 < -1 ? -1 : lim64);
#pragma unroll
                for (int i = 0; i < kBN; ++i) s[i] = (i <= lim) ? s[i] : -INFINITY;
            }
            // raw-score max in four independent chains; scale > 0 keeps the order
            float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
            for (int i = 0; i < kBN; ++i) m4[i & 3] = fmaxf(m4[i & 3], s[i]);
            const float mx = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3])) * p.scale_log2;
            int need_rescale = 0;
            float alpha = 1.f;
            if (mx > m_used + 8.f || (m_used == -INFINITY && mx != -INFINITY)) {
                alpha = (m_used == -INFINITY) ? 0.f : exp2f(m_used - mx);
                need_rescale = 1;
                l_sum *= alpha;
                m_used = mx;
            }
            // weights 2^(s * scale - m) <= 2^8 (a masked s = -inf gives +0)
            const float mneg = (m_used == -INFINITY) ? 0.f : -m_used;
            float b4[4] = {0.f, 0.f, 0.f, 0.f};
            uint32_t pk[kBN / 2];
#pragma unroll
            for (int i = 0; i < kBN; i += 2) {
                float e0, e1;
                asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e0) : "f"(fmaf(s[i], p.scale_log2, mneg)));
                asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e1) : "f"(fmaf(s[i + 1], p.scale_log2, mneg)));
                const __half2 hp = __floats2half2_rn(e0, e1);
                // l sums the fp32 weights; their f16 roundings (<= 2^-12 relative,
                // independent per key) average out far below the tolerance
                b4[(i >> 1) & 3] += e0 + e1;
                pk[i / 2] = *reinterpret_cast<const uint32_t *>(&hp);
            }
            l_sum += (b4[0] + b4[1]) + (b4[2] + b4[3]);
            // a rescale of O needs PV_{j-1} done; P buffer j & 1 needs PV_{j-2} done
            if (j >= 1 && __any_sync(0xffffffffu, need_rescale)) {
                ok = mbar_wait_warp(bar(kBarODone + ((j - 1) & 1)), (uint32_t)(((j - 1) >> 1) & 1), abort);
                if (!ok) break;
                tc_after_sync();
                {
                    const uint32_t ta = lane_base + kColO;
                    for (int c = 0; c < kD; c += 32) {
                        float v[32];
                        tmem_ld32(ta + c, v);
#pragma unroll
                        for (int i = 0; i < 32; ++i) v[i] *= alpha;
                        tmem_st32(ta + c, v);
                    }
                    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
                }
            }
            if (j >= 2) {
                ok = mbar_wait_warp(bar(kBarODone + (j & 1)), (uint32_t)(((j - 2) >> 1) & 1), abort);
                if (!ok) break;
            }
            uint8_t *pbuf = smem + kOffP + (j & 1) * kPBytes;
#pragma unroll
            for (int c8 = 0; c8 < kBN / 8; ++c8)
                *reinterpret_cast<uint4 *>(pbuf + sw128(kTileRows, row, c8 * 8)) =
                    make_uint4(pk[4 * c8], pk[4 * c8 + 1], pk[4 * c8 + 2], pk[4 * c8 + 3]);
            proxy_fence();
            tc_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(kBarPFull + (j & 1)));
        }
        // the last PV, then the partial: unnormalised O, m (log2 units), l
        if (ok && nblk > 0)
            ok = mbar_wait_warp(bar(kBarODone + ((nblk - 1) & 1)), (uint32_t)(((nblk - 1) >> 1) & 1), abort);
        if (ok) {
            tc_after_sync();
            const uint32_t ta = lane_base + kColO;
            const int64_t base = (((int64_t)split * p.Hq + h) * R + (r0 + row));
            float v[32];
            for (int c = 0; c < kD; c += 32) {
                if (nblk > 0) tmem_ld32(ta + c, v);
                if (row_valid) {
                    float *dst = p.part_o + base * kD + c;
#pragma unroll
                    for (int i = 0; i < 32; i += 4)
                        *reinterpret_cast<float4 *>(dst + i) = nblk > 0 ? make_float4(v[i], v[i + 1], v[i + 2], v[i + 3])
                                                                        : make_float4(0.f, 0.f, 0.f, 0.f);
                }
            }
            if (row_valid) {
                p.part_ml[base * 2] = m_used;
                p.part_ml[base * 2 + 1] = l_sum;
            }
        }
    }
    tc_before_sync();
    __syncthreads();
    tc_after_sync();
    if (tid == 0 && *abort) atomicExch(p.status, 1);
    if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols));
}

}  // namespace

int prefill_smem_bytes() { return kSmemBytes; }

cudaError_t launch_prefill(const PrefillParams &p, cudaStream_t s) {
    if (p.geom.D != kD || p.n_splits < 1 || p.n_splits > kMaxPrefillSplits || p.R < 1 || p.R > 256 ||
        p.geom.P % kBN != 0)
        return cudaErrorInvalidValue;
    {
        cudaError_t e = ensure_smem_limit(reinterpret_cast<const void *>(prefill_kernel), kSmemBytes);
        if (e != cudaSuccess) return e;
    }
    const int rt = (p.R + kTileRows - 1) / kTileRows;
    dim3 grid(p.n_splits, p.geom.Hk * p.G * rt);
    prefill_kernel<<<grid, kPThreads, kSmemBytes, s>>>(p);
    return cudaGetLastError();
}

}  // namespace kvs
