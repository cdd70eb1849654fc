// Prefill-chunk attention on the 5th-generation tensor cores (tcgen05).
//
// A prefill ubatch (up to 256 query rows, fp16 Q) attends causally over the
// paged Q8_0-K / Q4_0-V history.  Here QK^T and PV are dense contractions
// (1536 query rows per kv head at 6 query heads per kv head), so they run as
// tcgen05.mma with fp32 accumulators in tensor memory; "each staged KV span is
// consumed by all query tiles before its ring slot is released" (Adaptive KV
// Streaming for llama.cpp, "Batch and micro-batch sizes") holds because one
// launch covers every query tile of a key split.
//
// CTA = (key split, kv head, 128-row tile of one query head).  Per 64-key
// block of the split:
//   1. all 8 warps dequantise the block's K (Q8_0) and V (Q4_0) into shared
//      memory as f16 pairs hi + lo (code * scale is exact in fp32; hi/lo keep
//      ~22 of its bits), in the 128-byte-swizzled K-major layout tcgen05 reads;
//   2. one thread issues S = Q K_hi^T + Q K_lo^T (M 128, N 64, K 256) into TMEM;
//   3. warps 0-3 (one thread per row, TMEM lane = row) read S, scale, mask,
//      run the online softmax and write P (f16) to shared memory; O in TMEM is
//      rescaled only when a row's running max grows by more than 2^8 (the
//      weights are then formed against the stale max, which is exact);
//   4. one thread issues O += P V_hi + P V_lo (M 128, N 256, K 64).
// At the end warps 0-3 write the split's unnormalised partial (m, l, O) for
// the log-sum-exp combine shared with the decode path.  Every mbarrier wait
// is bounded: on timeout the kernel records a status code and skips the rest.
#include <cuda_fp16.h>
#include <math.h>

#include "kvs_internal.h"

namespace kvs {
namespace {

constexpr int kPThreads = 256;
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
constexpr int kOffP = kOffVl + kVBytes;
constexpr int kOffBar = kOffP + kPBytes;      // 2 mbarriers
constexpr int kOffTmem = kOffBar + 16;        // TMEM base address written by tcgen05.alloc
constexpr int kSmemBytes = kOffTmem + 16 + 1024;  // + slack to align the base to 1024

constexpr uint32_t kTmemCols = 512;  // S at [0, 64), O at [64, 320)
constexpr uint32_t kColS = 0, kColO = 64;

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

// bounded wait for phase `parity` of an mbarrier; false on timeout
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
    for (uint32_t i = 0; i < kSpinLimit; ++i) {
        uint32_t done;
        asm volatile(
            "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
            : "=r"(done)
            : "r"(bar), "r"(parity)
            : "memory");
        if (done) return true;
    }
    return false;
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

// (x, y) fp32 -> f16x2 hi = rn(x, y), lo = rn(x - hi, y - hi)
__device__ __forceinline__ void split_f16(float x, float y, uint32_t &hi, uint32_t &lo) {
    const __half2 h = __floats2half2_rn(x, y);
    const float2 hf = __half22float2(h);
    const __half2 l = __floats2half2_rn(x - hf.x, y - hf.y);
    hi = *reinterpret_cast<const uint32_t *>(&h);
    lo = *reinterpret_cast<const uint32_t *>(&l);
}

__global__ void __launch_bounds__(kPThreads, 1) prefill_kernel(const __grid_constant__ PrefillParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    const int tid = threadIdx.x, warp = tid >> 5;
    const int split_idx = blockIdx.x;
    const int G = p.G, R = p.R, rt = (R + kTileRows - 1) / kTileRows;
    const int g = blockIdx.y / (G * rt);
    const int tile = blockIdx.y % (G * rt);
    const int hl = tile / rt, r0 = (tile % rt) * kTileRows;
    const int h = g * G + hl;
    const int P = p.geom.P;
    const int it0 = p.split_begin[split_idx], it1 = p.split_begin[split_idx + 1];
    const int split = p.split_id[split_idx];

    const uint32_t bar_s = smem_u32(smem + kOffBar), bar_o = bar_s + 8;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + kOffTmem);

    if (tid == 0) {
        mbar_init(bar_s, 1);
        mbar_init(bar_o, 1);
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

    // per-row running state (warps 0-3: row = tid)
    const int row = tid;
    const bool row_owner = tid < kTileRows;
    const long long qpos = p.pos0 + r0 + row;  // this row's position
    const bool row_valid = row_owner && (r0 + row < R);
    float m_used = -INFINITY, l_sum = 0.f;
    const long long last_pos = p.pos0 + ((r0 + kTileRows < R) ? (r0 + kTileRows) : R) - 1;  // tile's last row
    uint32_t phase_s = 0, phase_o = 0;
    bool ok = true;
    bool any_o = false;  // O written at least once

    for (int it = it0; it < it1 && ok; ++it) {
        const int page = (int)p.page[it];
        const uint8_t *hb = p.arena + (int64_t)p.slot[it] * p.geom.page_bytes + (int64_t)g * p.geom.head_bytes;
        for (int kb = 0; kb < P && ok; kb += kBN) {
            const long long kpos0 = (long long)page * P + kb;
            if (kpos0 > last_pos) break;  // every later key is masked for every row of the tile
            // ---- dequantise K block (64 keys x 256 dims) -> K_hi, K_lo
            const __half *ks = reinterpret_cast<const __half *>(hb + p.geom.ks_off);
            for (int c = tid; c < kBN * (kD / 8); c += kPThreads) {
                const int key = c / (kD / 8), k = (c % (kD / 8)) * 8;
                const uint2 raw = *reinterpret_cast<const uint2 *>(hb + kq_byte(kb + key, k, kD / 32));
                const float d = __half2float(ks[(kb + key) * (kD / 32) + k / 32]);
                const int8_t *b8 = reinterpret_cast<const int8_t *>(&raw);
                uint32_t hi[4], lo[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) split_f16((float)b8[2 * e] * d, (float)b8[2 * e + 1] * d, hi[e], lo[e]);
                const uint32_t off = sw128(kBN, key, k);
                *reinterpret_cast<uint4 *>(smem + kOffKh + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
                *reinterpret_cast<uint4 *>(smem + kOffKl + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
            }
            // ---- dequantise V block -> V_hi, V_lo as [dim][key] (K-major for the PV MMA)
            const __half *vs = reinterpret_cast<const __half *>(hb + p.geom.vs_off);
            for (int c = tid; c < kD * (kBN / 8); c += kPThreads) {
                const int dim = c / (kBN / 8), k = (c % (kBN / 8)) * 8;
                const int blk = dim >> 5, within = dim & 31;
                const int brow = blk * 16 + (within & 15);
                const int shift = within < 16 ? 0 : 4;
                const uint2 raw = *reinterpret_cast<const uint2 *>(hb + p.geom.vq_off + vq_byte(kb + k, brow, kD / 32));
                const uint8_t *b8 = reinterpret_cast<const uint8_t *>(&raw);
                uint32_t hi[4], lo[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float d0 = __half2float(vs[blk * P + kb + k + 2 * e]);
                    const float d1 = __half2float(vs[blk * P + kb + k + 2 * e + 1]);
                    const float x0 = (float)(((b8[2 * e] >> shift) & 15) - 8) * d0;
                    const float x1 = (float)(((b8[2 * e + 1] >> shift) & 15) - 8) * d1;
                    split_f16(x0, x1, hi[e], lo[e]);
                }
                const uint32_t off = sw128(kD, dim, k);
                *reinterpret_cast<uint4 *>(smem + kOffVh + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
                *reinterpret_cast<uint4 *>(smem + kOffVl + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
            }
            proxy_fence();
            tc_before_sync();
            __syncthreads();
            tc_after_sync();
            // ---- S = Q K^T (hi + lo)
            if (tid == 0) {
                const uint32_t qa = smem_u32(smem + kOffQ), kh = smem_u32(smem + kOffKh), kl = smem_u32(smem + kOffKl);
                const uint32_t id = idesc_f16(kTileRows, kBN);
#pragma unroll 1
                for (int s = 0; s < kD / 16; ++s) {
                    const uint32_t ao = (s >> 2) * (kTileRows * 128) + (s & 3) * 32;
                    const uint32_t bo = (s >> 2) * (kBN * 128) + (s & 3) * 32;
                    mma_f16(tmem + kColS, smem_desc(qa + ao), smem_desc(kh + bo), id, s > 0);
                    mma_f16(tmem + kColS, smem_desc(qa + ao), smem_desc(kl + bo), id, 1);
                }
                mma_commit(bar_s);
            }
            if (!mbar_wait(bar_s, phase_s)) ok = false;
            phase_s ^= 1;
            ok = __syncthreads_and(ok);
            tc_after_sync();
            // ---- softmax rows (warps 0-3), P -> shared memory
            int need_rescale = 0;
            float alpha = 1.f;
            if (row_owner && ok) {
                float s[kBN];
                const uint32_t ta = tmem + ((uint32_t)(warp * 32) << 16) + kColS;
                float t32[32];
                tmem_ld32(ta, t32);
#pragma unroll
                for (int i = 0; i < 32; ++i) s[i] = t32[i];
                tmem_ld32(ta + 32, t32);
#pragma unroll
                for (int i = 0; i < 32; ++i) s[32 + i] = t32[i];
                float mx = -INFINITY;
#pragma unroll
                for (int i = 0; i < kBN; ++i) {
                    const bool valid = row_valid && (kpos0 + i <= qpos);
                    s[i] = valid ? s[i] * p.scale_log2 : -INFINITY;
                    mx = fmaxf(mx, s[i]);
                }
                if (mx > m_used + 8.f || (m_used == -INFINITY && mx != -INFINITY)) {
                    alpha = (m_used == -INFINITY) ? 0.f : exp2f(m_used - mx);
                    need_rescale = 1;
                    l_sum *= alpha;
                    m_used = mx;
                }
                float bsum = 0.f;
                uint32_t pk[kBN / 2];
#pragma unroll
                for (int i = 0; i < kBN; i += 2) {
                    const float e0 = (s[i] == -INFINITY) ? 0.f : exp2f(s[i] - m_used);
                    const float e1 = (s[i + 1] == -INFINITY) ? 0.f : exp2f(s[i + 1] - m_used);
                    const __half2 hp = __floats2half2_rn(e0, e1);
                    const float2 hf = __half22float2(hp);
                    bsum += hf.x + hf.y;  // l sums exactly the weights the MMA uses
                    pk[i / 2] = *reinterpret_cast<const uint32_t *>(&hp);
                }
                l_sum += bsum;
#pragma unroll
                for (int c8 = 0; c8 < kBN / 8; ++c8)
                    *reinterpret_cast<uint4 *>(smem + kOffP + sw128(kTileRows, row, c8 * 8)) =
                        make_uint4(pk[4 * c8], pk[4 * c8 + 1], pk[4 * c8 + 2], pk[4 * c8 + 3]);
            }
            // rescale O rows whose max moved (warp-collective TMEM access)
            if (warp < 4 && ok && any_o && __any_sync(0xffffffffu, need_rescale)) {
                const uint32_t ta = tmem + ((uint32_t)(warp * 32) << 16) + kColO;
                for (int c = 0; c < kD; c += 32) {
                    float v[32];
                    tmem_ld32(ta + c, v);
#pragma unroll
                    for (int i = 0; i < 32; ++i) v[i] *= alpha;
                    tmem_st32(ta + c, v);
                }
                asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
            }
            proxy_fence();
            tc_before_sync();
            __syncthreads();
            tc_after_sync();
            // ---- O += P V (hi + lo)
            if (tid == 0 && ok) {
                const uint32_t pa = smem_u32(smem + kOffP), vh = smem_u32(smem + kOffVh), vl = smem_u32(smem + kOffVl);
                const uint32_t id = idesc_f16(kTileRows, kD);
#pragma unroll 1
                for (int s = 0; s < kBN / 16; ++s) {
                    mma_f16(tmem + kColO, smem_desc(pa + s * 32), smem_desc(vh + s * 32), id, (any_o || s > 0) ? 1u : 0u);
                    mma_f16(tmem + kColO, smem_desc(pa + s * 32), smem_desc(vl + s * 32), id, 1);
                }
                mma_commit(bar_o);
            }
            if (ok && !mbar_wait(bar_o, phase_o)) ok = false;
            phase_o ^= 1;
            any_o = true;
            ok = __syncthreads_and(ok);
            tc_after_sync();
        }
    }
    if (!ok && tid == 0) atomicExch(p.status, 1);
    // ---- partial out: unnormalised O, m (log2 units), l
    if (row_owner && ok) {
        const uint32_t ta = tmem + ((uint32_t)(warp * 32) << 16) + kColO;
        float v[32];
        const bool write = row_valid && (r0 + row < R);
        const int64_t base = (((int64_t)split * p.Hq + h) * R + (r0 + row));
        for (int c = 0; c < kD; c += 32) {
            tmem_ld32(ta + c, v);
            if (write) {
                float *dst = p.part_o + base * kD + c;
                if (any_o) {
#pragma unroll
                    for (int i = 0; i < 32; i += 4) *reinterpret_cast<float4 *>(dst + i) = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
                } else {
#pragma unroll
                    for (int i = 0; i < 32; i += 4) *reinterpret_cast<float4 *>(dst + i) = make_float4(0.f, 0.f, 0.f, 0.f);
                }
            }
        }
        if (write) {
            p.part_ml[base * 2] = m_used;
            p.part_ml[base * 2 + 1] = l_sum;
        }
    }
    tc_before_sync();
    __syncthreads();
    tc_after_sync();
    if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols));
}

}  // namespace

int prefill_smem_bytes() { return kSmemBytes; }

cudaError_t launch_prefill(const PrefillParams &p, cudaStream_t s) {
    if (p.geom.D != kD || p.n_splits < 1 || p.n_splits > kMaxPrefillSplits || p.R < 1 || p.R > 256 ||
        p.geom.P % kBN != 0)
        return cudaErrorInvalidValue;
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    const int rt = (p.R + kTileRows - 1) / kTileRows;
    dim3 grid(p.n_splits, p.geom.Hk * p.G * rt);
    prefill_kernel<<<grid, kPThreads, kSmemBytes, s>>>(p);
    return cudaGetLastError();
}

}  // namespace kvs
