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
// CTA pairs.  Two CTAs of a cluster share one M = 256 MMA (tcgen05
// cta_group::2): each holds one 128-row query tile (a query head's rows) as
// its half of A and keeps its own S and O accumulators in its tensor memory.
// B is split along N between the pair: for S = Q K^T each CTA dequantises 64
// of a block's 128 keys, for O += P V each CTA dequantises 128 of the 256
// dims of V.  So a dequantised K/V block serves 256 query rows, and each SM
// reads only half of every B operand from its shared memory (one M = 128 MMA
// would read the whole of it, which saturates shared-memory bandwidth on its
// own).  The grid puts a kv head's tile pairs fastest, so the pairs that read
// one (split, kv head) run together and share its pages through L2.
//
// Roles, per CTA (the leader, cluster rank 0, issues every MMA of the pair):
//   warps 4-7 (producers) dequantise their halves of block j's K (Q8_0) and
//     block j-1's V (Q4_0) into shared-memory stages (two each) and publish
//     both under one proxy fence, as f16 in the 128-byte-
//     swizzled K-major layouts tcgen05 reads: K[key][dim], V[dim][key], each
//     value rn(d * x) (the pages' own tensor-core path also runs on f16
//     dequantised values);
//   warp 8, lane 0 of the leader, issues S_j (M 256, N 128, K 256) into one of
//     two TMEM score buffers, then O += P_{j-1} V_{j-1} (M 256, N 256, K 128);
//   warps 0-3 (one thread per row, TMEM lane = row) read S_j, scale, mask, run
//     the online softmax and write P_j (f16) to shared memory; O is rescaled
//     only when a row's running max grows by more than 2^8 (the weights are
//     then formed against the stale max, which is exact).
// Fences are mbarriers in the leader (full barriers: arrivals from both CTAs)
// and in both CTAs (empty barriers: multicast tcgen05.commit).  Every wait is
// bounded; a timeout raises an abort flag in both CTAs that ends every role's
// loop, and the CTA records a status code.  At the end each CTA writes its
// tile's unnormalised partial (m, l, O) for the log-sum-exp combine.
#include <cuda_fp16.h>
#include <math.h>

#include "kvs_internal.h"

namespace kvs {
namespace {

constexpr int kPThreads = 320;    // 4 softmax warps, 4 producer warps, MMA issue / relay warps 8-9
constexpr int kBN = 128;          // keys per block (S MMA N)
constexpr int kHalfN = kBN / 2;   // keys of a block this CTA dequantises
constexpr int kD = 256;           // head dim served by this kernel (PV MMA N)
constexpr int kHalfD = kD / 2;    // dims of V this CTA dequantises
constexpr int kNB = kD / 32;      // 32-dim scale blocks
constexpr int kTileRows = 128;    // query rows per CTA (the pair's MMA M is 256)
constexpr uint32_t kSpinLimit = 1u << 26;

// shared-memory carve (bytes, 1024-aligned tiles for the 128B swizzle)
constexpr int kQBytes = kTileRows * kD * 2;   // 64 KB: 4 atoms (64 dims) of 128 rows x 128 B
constexpr int kKBytes = kHalfN * kD * 2;      // 32 KB per stage: 4 atoms (64 dims) of 64 key rows
constexpr int kVBytes = kHalfD * kBN * 2;     // 32 KB per stage: 2 atoms (64 keys) of 128 dim rows
constexpr int kOffQ = 0;
constexpr int kOffK = kOffQ + kQBytes;        // 2 stages
constexpr int kOffV = kOffK + 2 * kKBytes;    // 2 stages
constexpr int kOffBar = kOffV + 2 * kVBytes;  // mbarriers (kNumBars x 8 B)
constexpr int kNumBars = 16;
constexpr int kOffTmem = kOffBar + kNumBars * 8;  // TMEM base address written by tcgen05.alloc
constexpr int kOffAbort = kOffTmem + 8;
constexpr int kOffSlots = kOffAbort + 8;          // device slot of each page of the split
constexpr int kSmemBytes = kOffSlots + kMaxPrefillSplitPages * 4 + 1024;  // + slack to align the base

constexpr uint32_t kTmemCols = 512;  // S buffers at [0, 128) and [128, 256), O at [256, 512);
                                     // P_j (f16 pairs, 64 columns) overwrites S_j's first half
constexpr uint32_t kColO = 256;
// barrier indices.  Producers and softmax warps arrive on their own CTA's
// "Full" barriers with a CTA-scope release; in the peer, relay threads (warps
// 8 and 9) wait for those and pass each phase on to the leader's barrier with
// one cluster-scope release, so the leader's Full barriers count 4 local warps
// and 1 relay.  A cluster-scope release costs the arriving warp about a
// microsecond; the relays take it off the producers' and the softmax's paths.
// The other barriers are armed by multicast commits in both CTAs.  Each
// completes one phase per use of what it guards.
constexpr int kBarKVFull = 0;  // + j & 1 (2): producers wrote K_j (stage j & 1) and V_{j-1}
constexpr int kBarPFull = 4;   // + j & 1 (2): softmax wrote P_j (which also means S_j was read)
// Two barriers per Full kind (by the parity of j) keep a relay's wait from
// aliasing: the next phase of the barrier it waits on (j + 2) cannot complete
// before the leader has consumed phase j, which needs the relay's arrival.
constexpr int kBarKEmpty = 7;  // + stage (2): S_j done, K stage free
constexpr int kBarVEmpty = 9;  // + stage (2): PV_j done, V stage free
constexpr int kBarFinal = 11;  // every MMA of the CTA pair finished
constexpr int kBarSFull = 12;  // + S buffer (2): S_j in TMEM
constexpr int kBarODone = 14;  // + j & 1 (2): PV_j done, O stable (one barrier per parity of
                               // j, so a wait for PV_j may be skipped: the barrier's next
                               // phase, PV_{j+2}, needs P_{j+2}, which is not written yet)

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

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// shared::cluster address of local shared address `a` in CTA `rank` of the cluster
__device__ __forceinline__ uint32_t peer_addr(uint32_t a, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(rank));
    return r;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count));
}

// bounded wait (cluster-scope acquire) for phase `parity` of a local
// mbarrier; false on timeout or once *abort is raised (a timeout raises it)
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int *abort) {
    for (uint32_t i = 0; i < kSpinLimit; ++i) {
        uint32_t done;
        asm volatile(
            "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
            " selp.u32 %0, 1, 0, p;\n}\n"
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

// arrive (release, cluster scope) on an mbarrier given by its shared::cluster address
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cbar) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cbar) : "memory");
}

// arrive (release, CTA scope) on an mbarrier of this CTA
__device__ __forceinline__ void mbar_arrive_local(uint32_t bar) {
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// D (TMEM of both CTAs) = A (smem of both) * B (smem of both, N split) [+ D]
__device__ __forceinline__ void mma_pair(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(idesc), "r"(acc));
}

// D (TMEM of both CTAs) = A (TMEM of both: each CTA's 128 rows, f16 pairs per
// column) * B (smem of both, N split) [+ D]
__device__ __forceinline__ void mma_pair_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc,
                                            uint32_t acc) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc));
}

// arrive on barrier `bar` (same offset) of both CTAs once the pair's MMAs issued so far are done
__device__ __forceinline__ void mma_commit_both(uint32_t bar) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(bar),
        "h"((uint16_t)3)
        : "memory");
}

__device__ __forceinline__ void tc_before_sync() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_after_sync() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void proxy_fence() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// 32 lanes x 32 columns of fp32 from TMEM (one row per thread), no wait
__device__ __forceinline__ void tmem_ld32_nowait(uint32_t taddr, float *v) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float *v) {
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

// 4 int8 (bytes of w) -> f16x2 (x0, x1), (x2, x3), exact: the byte x + 128
// under exponent 0x64 is 1024 + 128 + x, minus 1152 (exponent-bias
// conversion, Kim et al. 2022, as in kvs_decode.cu)
__device__ __forceinline__ void i8x4_to_f16(uint32_t w, uint32_t &a, uint32_t &b) {
    const uint32_t u = w ^ 0x80808080u;
    uint32_t bl, bh;
    asm("prmt.b32 %0, %1, %2, 0x4140;" : "=r"(bl) : "r"(u), "r"(0x64646464u));
    asm("prmt.b32 %0, %1, %2, 0x4342;" : "=r"(bh) : "r"(u), "r"(0x64646464u));
    asm("sub.f16x2 %0, %1, %2;" : "=r"(a) : "r"(bl), "r"(0x64806480u));
    asm("sub.f16x2 %0, %1, %2;" : "=r"(b) : "r"(bh), "r"(0x64806480u));
}

__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

__device__ __forceinline__ uint32_t hmul2(uint32_t x, uint32_t d) {
    uint32_t r;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(x), "r"(d));
    return r;
}

// Two packed Q4_0 bytes (keys k, k+1, bytes `sel` of w) -> f16x2 of the low
// nibbles - 8 and of the high nibbles - 8.  Each nibble sits in the mantissa
// under exponent 0x64: low = 1024 + n, high = 1024 + 16 n, and
// (1024 + 16 n) / 16 - 72 = n - 8 exactly in one fused multiply-add.
__device__ __forceinline__ void u4x2_pair(uint32_t w, uint32_t sel, uint32_t &lo, uint32_t &hi) {
    uint32_t sp, tl, th;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(sp) : "r"(w), "r"(0u), "r"(sel));
    asm("lop3.b32 %0, %1, %2, %3, 0xea;" : "=r"(tl) : "r"(sp), "r"(0x000f000fu), "r"(0x64006400u));
    asm("lop3.b32 %0, %1, %2, %3, 0xea;" : "=r"(th) : "r"(sp), "r"(0x00f000f0u), "r"(0x64006400u));
    asm("sub.f16x2 %0, %1, %2;" : "=r"(lo) : "r"(tl), "r"(0x64086408u));                          // - 1032
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(hi) : "r"(th), "r"(0x2c002c00u), "r"(0xd480d480u));  // / 16 - 72
}

// 9 warps put 3 on one of the SM's four 16K-register partitions: 168 registers
// per thread is the most that still launches
__global__ void __cluster_dims__(2, 1, 1) __maxnreg__(168) prefill_kernel(const __grid_constant__ PrefillParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    tl_begin(p.tl);
    const uint32_t rank = cluster_rank();  // 0: leader (issues the MMAs), 1: peer
    const int split_idx = blockIdx.y;
    const int G = p.G, R = p.R, rt = (R + kTileRows - 1) / kTileRows;
    const int ntiles = G * rt, npairs = (ntiles + 1) / 2;
    const int g = blockIdx.x / (2 * npairs);
    const int pair = (blockIdx.x % (2 * npairs)) >> 1;
    // this CTA's tile and its partner's; a tile past the last is empty (no valid row)
    auto tile_rows = [&](int t, int &h, int &r0, int &nrows) {
        const int tt = t < ntiles ? t : 0;
        h = g * G + tt / rt;
        r0 = (tt % rt) * kTileRows;
        nrows = t < ntiles ? ((R - r0) < kTileRows ? (R - r0) : kTileRows) : 0;
    };
    int h, r0, nrows, h_o, r0_o, nrows_o;
    tile_rows(2 * pair + (int)rank, h, r0, nrows);
    tile_rows(2 * pair + 1 - (int)rank, h_o, r0_o, nrows_o);
    const int P = p.geom.P;
    const int it0 = p.split_begin[split_idx], it1 = p.split_begin[split_idx + 1];
    const int split = p.split_id[split_idx];
    const int n_keys = (it1 - it0) * P;                     // keys of this split
    const long long key_pos0 = (long long)p.page[it0] * P;  // the split's pages are consecutive

    const uint32_t bar0 = smem_u32(smem + kOffBar);
    auto bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };
    const uint32_t lead_bar0 = peer_addr(bar0, 0);  // the leader's barriers, shared::cluster
    auto lead_bar = [&](int i) { return lead_bar0 + 8u * (uint32_t)i; };
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + kOffTmem);
    volatile int *abort = reinterpret_cast<volatile int *>(smem + kOffAbort);
    const uint32_t peer_abort = peer_addr(smem_u32(smem + kOffAbort), rank ^ 1u);

    // 128-key blocks of this split the pair runs: enough for the later of the
    // two tiles (the other tile's extra blocks are fully masked)
    int nblk;
    {
        long long last = -1;
        if (nrows > 0) last = p.pos0 + r0 + nrows - 1;
        if (nrows_o > 0 && p.pos0 + r0_o + nrows_o - 1 > last) last = p.pos0 + r0_o + nrows_o - 1;
        const long long vis = last - key_pos0 + 1;  // keys at or before the pair's last row
        const int nv = vis <= 0 ? 0 : (int)((vis + kBN - 1) / kBN);
        nblk = (n_keys + kBN - 1) / kBN;
        if (nv < nblk) nblk = nv;
    }
    // page-head section holding split key `ks` (0 <= ks < n_keys); the split's
    // slots are copied to shared memory once (indexing the parameter block at
    // run time is slow)
    const uint32_t *slots = reinterpret_cast<const uint32_t *>(smem + kOffSlots);
    const int lgP = __ffs(P) - 1;  // P is a power of two
    const uint8_t *arena_g = p.arena + (int64_t)g * p.geom.head_bytes;
    auto head_of = [&](int ks) {
        return arena_g + (int64_t)slots[ks >> lgP] * p.geom.page_bytes;
    };
    auto raise_abort = [&]() {
        *abort = 1;
        asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(peer_abort), "r"(1) : "memory");
    };

    if (tid == 0) {
        for (int s = 0; s < 2; ++s) {
            mbar_init(bar(kBarKVFull + s), rank == 0 ? 5 : 4);
            mbar_init(bar(kBarKEmpty + s), 1);
            mbar_init(bar(kBarVEmpty + s), 1);
            mbar_init(bar(kBarSFull + s), 1);
        }
        mbar_init(bar(kBarPFull), rank == 0 ? 5 : 4);
        mbar_init(bar(kBarPFull + 1), rank == 0 ? 5 : 4);
        mbar_init(bar(kBarODone), 1);
        mbar_init(bar(kBarODone + 1), 1);
        mbar_init(bar(kBarFinal), 1);
        *abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    for (int i = tid; i < it1 - it0; i += kPThreads) reinterpret_cast<uint32_t *>(smem + kOffSlots)[i] = p.slot[it0 + i];
    if (warp == 0) {  // one warp of each CTA allocates the pair's tensor memory together
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                     "r"(kTmemCols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;");
    }
    // Q tile -> shared memory (f16, swizzled); rows past the tile's are zero.
    // All of a thread's loads are issued before its first store.
    {
        constexpr int kQChunks = kTileRows * (kD / 8), kQPer = (kQChunks + kPThreads - 1) / kPThreads;
        const __half *q = reinterpret_cast<const __half *>(p.q);
        uint4 v[kQPer];
#pragma unroll
        for (int i = 0; i < kQPer; ++i) {
            const int c = tid + i * kPThreads, row = c / (kD / 8), k = (c % (kD / 8)) * 8;
            v[i] = make_uint4(0, 0, 0, 0);
            if (c < kQChunks && row < nrows)
                v[i] = *reinterpret_cast<const uint4 *>(q + ((int64_t)(r0 + row) * p.Hq + h) * kD + k);
        }
#pragma unroll
        for (int i = 0; i < kQPer; ++i) {
            const int c = tid + i * kPThreads, row = c / (kD / 8), k = (c % (kD / 8)) * 8;
            if (c < kQChunks) *reinterpret_cast<uint4 *>(smem + kOffQ + sw128(kTileRows, row, k)) = v[i];
        }
    }
    proxy_fence();
    tc_before_sync();
    __syncthreads();
    cluster_sync();  // both CTAs' barriers and Q tiles are ready before any remote arrival or MMA
    tc_after_sync();
    const uint32_t tmem = *tmem_slot;

    if (warp >= 4 && warp < 8) {
        // ------------------------------------------------------------ producers
        // K: thread pt owns key row kr = pt % 64 of this CTA's half of the block
        // (keys rank * 64 + kr) and dims blocks kb0 .. kb0 + 3, kb0 = (pt / 64) * 4.
        // V: this CTA dequantises dims rank * 128 .. + 127, i.e. scale blocks
        // rank * 4 .. + 3; thread pt owns 32-key chunk vc of block vb and its byte
        // rows vq, vq + 8 (dims vb * 32 + row and + 16), so its 32 scales sit in
        // its own registers; lanes differ in vq, which keeps every 16-byte store
        // of a warp phase on its own banks under the swizzle.  Raw bytes of the
        // next block are loaded into registers ahead of the waits for its stage.
        const int pt = tid - 128;  // 0..127
        const int kr = pt & 63, kb0 = (pt >> 6) * 4;
        const int vbl = pt >> 5, vb = (int)rank * 4 + vbl, vc = (pt >> 3) & 3, vq = pt & 7;
        uint4 rk[8], rv[4], sv[4];
        uint2 sk;
        auto load_k = [&](int j) {
            const int ks = j * kBN + (int)rank * kHalfN + kr;
            if (ks < n_keys) {
                const uint8_t *hb = head_of(ks);
                const int t = ks & (P - 1);
#pragma unroll
                for (int b = 0; b < 4; ++b) {
                    // kq_byte in 32 bits: 16-token group, 32-dim block, token in the group
                    const uint4 *line =
                        reinterpret_cast<const uint4 *>(hb + (((t >> 4) * kNB + kb0 + b) * 16 + (t & 15)) * 32);
                    rk[2 * b] = line[0];
                    rk[2 * b + 1] = line[1];
                }
                sk = *reinterpret_cast<const uint2 *>(hb + p.geom.ks_off + (t * kNB + kb0) * 2);
            } else {  // beyond the split: zero keys (masked by the softmax)
#pragma unroll
                for (int i = 0; i < 8; ++i) rk[i] = make_uint4(0, 0, 0, 0);
                sk = make_uint2(0, 0);
            }
        };
        auto load_v = [&](int j) {
            const int ks = j * kBN + 32 * vc;  // a 32-key chunk never straddles a page (P % 64 == 0)
            if (ks < n_keys) {
                const uint8_t *hb = head_of(ks);
                const int t = ks & (P - 1);
                // vq_byte in 32 bits: 32-token chunk, byte row, token in the chunk
                const uint8_t *line0 = hb + p.geom.vq_off + (((t >> 5) * kNB + vb) * 16 + vq) * 32 + (t & 31);
#pragma unroll
                for (int i = 0; i < 2; ++i) {  // byte rows vq + 8 i: lines 8 i apart
                    rv[2 * i] = reinterpret_cast<const uint4 *>(line0 + i * 256)[0];
                    rv[2 * i + 1] = reinterpret_cast<const uint4 *>(line0 + i * 256)[1];
                }
                const uint4 *sc = reinterpret_cast<const uint4 *>(hb + p.geom.vs_off + (vb * P + t) * 2);
#pragma unroll
                for (int i = 0; i < 4; ++i) sv[i] = sc[i];
            } else {  // beyond the split: code 8 = value 0
#pragma unroll
                for (int i = 0; i < 4; ++i) rv[i] = make_uint4(0x88888888u, 0x88888888u, 0x88888888u, 0x88888888u);
#pragma unroll
                for (int i = 0; i < 4; ++i) sv[i] = make_uint4(0, 0, 0, 0);
            }
        };
        auto write_k = [&](int stage) {
            uint8_t *kt = smem + kOffK + stage * kKBytes;
            const uint32_t sc[2] = {sk.x, sk.y};  // scale pairs (blocks kb0 + 2i, kb0 + 2i + 1)
#pragma unroll
            for (int b = 0; b < 4; ++b) {
                uint32_t d;  // scale of block kb0 + b in both halves
                asm("prmt.b32 %0, %1, %1, %2;" : "=r"(d) : "r"(sc[b >> 1]), "r"((b & 1) ? 0x3232u : 0x1010u));
                const uint32_t w[8] = {rk[2 * b].x,     rk[2 * b].y,     rk[2 * b].z,     rk[2 * b].w,
                                       rk[2 * b + 1].x, rk[2 * b + 1].y, rk[2 * b + 1].z, rk[2 * b + 1].w};
                uint32_t o[16];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    uint32_t x0, x1;
                    i8x4_to_f16(w[i], x0, x1);
                    o[2 * i] = hmul2(x0, d);
                    o[2 * i + 1] = hmul2(x1, d);
                }
#pragma unroll
                for (int m = 0; m < 4; ++m)
                    *reinterpret_cast<uint4 *>(kt + sw128(kHalfN, kr, (kb0 + b) * 32 + 8 * m)) =
                        make_uint4(o[4 * m], o[4 * m + 1], o[4 * m + 2], o[4 * m + 3]);
            }
        };
        auto write_v = [&](int stage) {
            uint8_t *vt = smem + kOffV + stage * kVBytes;
            const uint32_t d2[16] = {sv[0].x, sv[0].y, sv[0].z, sv[0].w, sv[1].x, sv[1].y, sv[1].z, sv[1].w,
                                     sv[2].x, sv[2].y, sv[2].z, sv[2].w, sv[3].x, sv[3].y, sv[3].z, sv[3].w};
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const int rA = vbl * 32 + vq + 8 * i, rB = rA + 16;  // rows of this CTA's V tile (dims - rank * 128)
                const uint32_t w[8] = {rv[2 * i].x,     rv[2 * i].y,     rv[2 * i].z,     rv[2 * i].w,
                                       rv[2 * i + 1].x, rv[2 * i + 1].y, rv[2 * i + 1].z, rv[2 * i + 1].w};
                uint32_t oa[16], ob[16];
#pragma unroll
                for (int k2 = 0; k2 < 16; ++k2) {  // keys 2 k2, 2 k2 + 1 of the chunk; d2[k2] holds their scales
                    uint32_t lo, hi;
                    u4x2_pair(w[k2 >> 1], (k2 & 1) ? 0x4342u : 0x4140u, lo, hi);
                    oa[k2] = hmul2(lo, d2[k2]);
                    ob[k2] = hmul2(hi, d2[k2]);
                }
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    *reinterpret_cast<uint4 *>(vt + sw128(kHalfD, rA, 32 * vc + 8 * m)) =
                        make_uint4(oa[4 * m], oa[4 * m + 1], oa[4 * m + 2], oa[4 * m + 3]);
                    *reinterpret_cast<uint4 *>(vt + sw128(kHalfD, rB, 32 * vc + 8 * m)) =
                        make_uint4(ob[4 * m], ob[4 * m + 1], ob[4 * m + 2], ob[4 * m + 3]);
                }
            }
        };
        // Iteration j publishes K_j (stage j & 1, free once S_{j-2} is done) and
        // V_{j-1} (stage (j-1) & 1, free once PV_{j-3} is done) under one proxy
        // fence and one arrival: the MMA thread issues PV_{j-1} right after S_j,
        // so both are wanted at the same time (separate K and V publishes, with
        // a third relay in the peer, measured slower).
        if (nblk > 0) load_k(0);
        for (int j = 0; j <= nblk; ++j) {  // every exit is a warp-uniform wait outcome
            const bool wk = j < nblk, wv = j >= 1;
            if (wk && j >= 2 && !mbar_wait_warp(bar(kBarKEmpty + (j & 1)), (uint32_t)(((j - 2) >> 1) & 1), abort)) break;
            if (wv && j >= 3 &&
                !mbar_wait_warp(bar(kBarVEmpty + ((j - 1) & 1)), (uint32_t)(((j - 3) >> 1) & 1), abort))
                break;
            if (wk) write_k(j & 1);
            if (wv) write_v((j - 1) & 1);
            proxy_fence();
            __syncwarp();
            if (lane == 0) mbar_arrive_local(bar(kBarKVFull + (j & 1)));
            if (j + 1 < nblk) load_k(j + 1);
            if (j < nblk) load_v(j);
        }
    } else if (warp >= 8) {
        // ------------------------------------------------------------ relays (peer, one thread each)
        if (rank == 1 && lane == 0) {
            // warp 8 passes on the producers' phases (nblk + 1 of them), warp 9 the softmax's
            const int nph = warp == 8 ? nblk + 1 : nblk;
            bool ok = true;
            for (int j = 0; j < nph && ok; ++j) {
                const int b = (warp == 8 ? kBarKVFull : kBarPFull) + (j & 1);
                ok = mbar_wait(bar(b), (uint32_t)((j >> 1) & 1), abort);
                if (ok) mbar_arrive_cluster(lead_bar(b));
            }
        }
        // ------------------------------------------------------------ MMA issue (leader, one thread)
        if (rank == 0 && warp == 8 && lane == 0) {
            // descriptors of the tile bases; a k-step adds its byte offset / 16
            const uint64_t dq = smem_desc(smem_u32(smem + kOffQ)), dk = smem_desc(smem_u32(smem + kOffK));
            const uint64_t dv = smem_desc(smem_u32(smem + kOffV));
            const uint32_t id_s = idesc_f16(2 * kTileRows, kBN), id_o = idesc_f16(2 * kTileRows, kD);
            auto issue_s = [&](int j) {
                const uint32_t ts = tmem + (uint32_t)((j & 1) * kBN);
                const uint64_t dkj = dk + (uint64_t)(((j & 1) * kKBytes) >> 4);
#pragma unroll
                for (int s = 0; s < kD / 16; ++s) {  // 16 dims per k-step, 64 per swizzle atom
                    const uint64_t aq = (uint64_t)(((s >> 2) * (kTileRows * 128) + (s & 3) * 32) >> 4);
                    const uint64_t bk = (uint64_t)(((s >> 2) * (kHalfN * 128) + (s & 3) * 32) >> 4);
                    mma_pair(ts, dq + aq, dkj + bk, id_s, s > 0);
                }
                mma_commit_both(bar(kBarSFull + (j & 1)));
                mma_commit_both(bar(kBarKEmpty + (j & 1)));
            };
            auto issue_pv = [&](int j) {
                const uint64_t dvj = dv + (uint64_t)(((j & 1) * kVBytes) >> 4);
                // A = P_j in TMEM over S_j's buffer: 16 keys per k-step = 8 columns.  S_{j+2},
                // which overwrites that buffer, is issued after this in program order, and
                // the tensor pipe runs one thread's MMAs in order
                const uint32_t tp = tmem + (uint32_t)((j & 1) * kBN);
#pragma unroll
                for (int s = 0; s < kBN / 16; ++s) {  // 16 keys per k-step, 64 per swizzle atom of V
                    const uint64_t bv = (uint64_t)(((s >> 2) * (kHalfD * 128) + (s & 3) * 32) >> 4);
                    mma_pair_ta(tmem + kColO, tp + (uint32_t)(8 * s), dvj + bv, id_o, (j > 0 || s > 0) ? 1u : 0u);
                }
                mma_commit_both(bar(kBarVEmpty + (j & 1)));
                mma_commit_both(bar(kBarODone + (j & 1)));
            };
            bool ok = true;
            // S_j overwrites the buffer of S_{j-2} and P_{j-2}: P_{j-2} written means
            // S_{j-2} was read, and PV_{j-2} was issued before S_j
            for (int j = 0; j < nblk && ok; ++j) {
                ok = mbar_wait(bar(kBarKVFull + (j & 1)), (uint32_t)((j >> 1) & 1), abort);  // K_j, V_{j-1}
                if (!ok) break;
                tc_after_sync();
                issue_s(j);
                if (j >= 1) {
                    ok = mbar_wait(bar(kBarPFull + ((j - 1) & 1)), (uint32_t)(((j - 1) >> 1) & 1), abort);
                    if (!ok) break;
                    tc_after_sync();
                    issue_pv(j - 1);
                }
            }
            if (ok && nblk > 0) {
                ok = mbar_wait(bar(kBarPFull + ((nblk - 1) & 1)), (uint32_t)(((nblk - 1) >> 1) & 1), abort) &&
                     mbar_wait(bar(kBarKVFull + (nblk & 1)), (uint32_t)((nblk >> 1) & 1), abort);  // V_{nblk-1}
                if (ok) {
                    tc_after_sync();
                    issue_pv(nblk - 1);
                }
            }
            if (!ok) raise_abort();
            // every MMA of the pair has finished before either CTA reads or frees TMEM
            mma_commit_both(bar(kBarFinal));
        }
    } else {
        // ------------------------------------------------------------ softmax rows (warps 0-3)
        const int row = tid;
        const long long qpos = p.pos0 + r0 + row;
        const bool row_valid = row < nrows;
        const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
        float m_used = -INFINITY, l_sum = 0.f;
        bool ok = true;
        for (int j = 0; j < nblk && ok; ++j) {
            ok = mbar_wait_warp(bar(kBarSFull + (j & 1)), (uint32_t)((j >> 1) & 1), abort);
            if (!ok) break;
            tc_after_sync();
            float s[kBN];
            {
                const uint32_t ta = lane_base + (uint32_t)((j & 1) * kBN);
#pragma unroll
                for (int c = 0; c < kBN; c += 32) tmem_ld32_nowait(ta + c, s + c);
                tmem_wait_ld();
            }
            // keys i > lim are masked: after this row's position, or beyond the split
            {
                const long long kpos = key_pos0 + (long long)j * kBN;
                long long lim64 = row_valid ? qpos - kpos : -1;
                const int in_split = n_keys - j * kBN - 1;
                if (lim64 > in_split) lim64 = in_split;
                if (lim64 < kBN - 1) {
                    const int lim = (int)(lim64 < -1 ? -1 : lim64);
#pragma unroll
                    for (int i = 0; i < kBN; ++i) s[i] = (i <= lim) ? s[i] : -INFINITY;
                }
            }
            // raw-score max in four independent chains of three-input maxima; scale > 0
            // keeps the order
            float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
            for (int i = 0; i < kBN; i += 2) m4[(i >> 1) & 3] = fmax3(m4[(i >> 1) & 3], s[i], s[i + 1]);
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
            // P_j as f16 pairs into the first 64 columns of S_j's buffer (this
            // thread's row was read out of it above), each half stored as soon
            // as it is formed
            const uint32_t tp = lane_base + (uint32_t)((j & 1) * kBN);
#pragma unroll
            for (int half = 0; half < 2; ++half) {
#pragma unroll
                for (int i = half * (kBN / 2); i < (half + 1) * (kBN / 2); i += 2) {
                    float e0, e1;
                    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e0) : "f"(fmaf(s[i], p.scale_log2, mneg)));
                    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e1) : "f"(fmaf(s[i + 1], p.scale_log2, mneg)));
                    const __half2 hp = __floats2half2_rn(e0, e1);
                    // l sums the fp32 weights; their f16 roundings (<= 2^-12 relative,
                    // independent per key) average out far below the tolerance
                    b4[(i >> 1) & 3] += e0 + e1;
                    pk[i / 2] = *reinterpret_cast<const uint32_t *>(&hp);
                }
                tmem_st32(tp + 32 * half, reinterpret_cast<const float *>(pk + 32 * half));
            }
            l_sum += (b4[0] + b4[1]) + (b4[2] + b4[3]);
            // O is rescaled once PV_{j-1} is done (P_j's buffer is not the one PV_{j-1}
            // reads, so only a rescale waits for it)
            if (j >= 1 && __any_sync(0xffffffffu, need_rescale)) {
                ok = mbar_wait_warp(bar(kBarODone + ((j - 1) & 1)), (uint32_t)(((j - 1) >> 1) & 1), abort);
                if (!ok) {
                    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
                    break;
                }
                tc_after_sync();
                const uint32_t ta = lane_base + kColO;
#pragma unroll 1
                for (int c = 0; c < kD; c += 32) {
                    float v[32];
                    tmem_ld32_nowait(ta + c, v);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; ++i) v[i] *= alpha;
                    tmem_st32(ta + c, v);
                }
            }
            asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");  // P_j (and O) stored
            tc_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive_local(bar(kBarPFull + (j & 1)));
        }
        // the last PV, then the partial: unnormalised O, m (log2 units), l
        if (ok && nblk > 0)
            ok = mbar_wait_warp(bar(kBarODone + ((nblk - 1) & 1)), (uint32_t)(((nblk - 1) >> 1) & 1), abort);
        if (ok) {
            tc_after_sync();
            const uint32_t ta = lane_base + kColO;
            const int64_t base = (((int64_t)split * p.Hq + h) * R + (r0 + row));
            float v[32];
#pragma unroll 1
            for (int c = 0; c < kD; c += 32) {
                if (nblk > 0) {
                    tmem_ld32_nowait(ta + c, v);
                    tmem_wait_ld();
                }
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
    // A role that gave up tells the peer CTA, so that its waits end too.
    if (lane == 0 && *abort) raise_abort();
    // Both CTAs wait for the pair's last MMA before either may exit or free
    // tensor memory: an MMA in flight reads both CTAs' shared memory.  The
    // leader commits Final on every path, so this wait (bounded, and not cut
    // short by an abort) always ends.
    if (tid == 0) {
        volatile int no_abort = 0;
        if (!mbar_wait(bar(kBarFinal), 0u, &no_abort)) *abort = 1;
    }
    tc_before_sync();
    __syncthreads();
    cluster_sync();
    tc_after_sync();
    if (tid == 0 && *abort) atomicExch(p.status, 1);
    tl_finish(p.tl);
    if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols));
}

}  // namespace

int prefill_smem_bytes() { return kSmemBytes; }

cudaError_t launch_prefill(const PrefillParams &p, cudaStream_t s) {
    if (p.geom.D != kD || p.n_splits < 1 || p.n_splits > kMaxPrefillSplits || p.R < 1 || p.R > 256 ||
        p.geom.P % 64 != 0)
        return cudaErrorInvalidValue;
    for (int i = 0; i < p.n_splits; ++i)
        if (p.split_begin[i + 1] - p.split_begin[i] > kMaxPrefillSplitPages) return cudaErrorInvalidValue;
    {
        cudaError_t e = ensure_smem_limit(reinterpret_cast<const void *>(prefill_kernel), kSmemBytes);
        if (e != cudaSuccess) return e;
    }
    const int rt = (p.R + kTileRows - 1) / kTileRows;
    const int npairs = (p.G * rt + 1) / 2;
    dim3 grid(p.geom.Hk * 2 * npairs, p.n_splits);  // clusters of 2 along x
    prefill_kernel<<<grid, kPThreads, kSmemBytes, s>>>(p);
    return cudaGetLastError();
}

}  // namespace kvs
