// Split-K paged attention for 1..N query rows over a Q8_0-K / Q4_0-V page,
// and the log-sum-exp combine of the per-page partials.
//
// One CTA = one (page, kv head) work item.  Every query head of the kv
// head's group and every query row is served by that CTA, so each K/V byte
// is read from memory once per step ("Q8_0 K and Q4_0 V are converted in
// small tiles, not copied into another full FP16 cache", Adaptive KV
// Streaming for llama.cpp V2, "Keep the stock attention order").
//
// Arithmetic.  Scores and P.V run on the tensor cores (mma.sync m16n8k16,
// f16 operands, fp32 accumulation):
//   S^T[key][row] = sum_d K[key][d] * Q[row][d]     A = K codes (exact in f16),
//                                                   B = Q as f16 hi + f16 lo
//   O^T[dim][row] = sum_key V[key][dim] * P'[row][key]
//                                                   A = V codes - 8 (exact),
//                                                   B = P' = p * dV, hi + lo
// The Q8_0 scale multiplies each 32-dim block's partial dot in fp32; the
// Q4_0 scale is folded into P' per (key, 32-dim block).  Splitting the fp32
// operand into two f16 parts keeps ~22 significand bits, so the result
// tracks fp32 arithmetic (tested against the fp64 oracle at 1e-3 relative).
// Softmax over the page's keys runs in fp32 with exp2 on log2-scaled scores.
//
// Fragment orders.  The reduction index of each MMA is permuted so that one
// 64-bit load gives a thread its whole fragment:
//   QK: thread (gid, tig) of a k-step in 32-dim block b holds dims
//       32b + 8*tig + 4*s + {0..3} (s = k-step within the block), i.e. one
//       32-bit word of an 8-byte load of the key row.
//   PV: the page stores V dim-major (byte row = dim pair, column = token), a
//       thread's word holds 4 consecutive keys of one dim pair; the four MMA
//       k positions (2t, 2t+1, 2t+8, 2t+9) map to keys (+0, +2, +1, +3) and
//       the MMA rows (gid, gid+8) to the low/high nibble dims of that byte.
// The int8 -> f16 and nibble -> f16 conversions use the exponent-bias trick
// described by Kim et al., "Who Says Elephants Can't Run: Bringing Large
// Scale MoE Models into Cloud Scale Production" (2022): a small integer u
// placed in the mantissa under exponent 0x64 is the half 1024 + u.
#include <cuda_fp16.h>
#include <math.h>

#include "kvs_internal.h"

namespace kvs {
namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ void mma16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// 4 int8 (bytes x0..x3 of w) -> f16x2 (x0, x1) and (x2, x3), exact.
__device__ __forceinline__ void i8x4_to_f16(uint32_t w, uint32_t &lo, uint32_t &hi) {
    const uint32_t u = w ^ 0x80808080u;  // x + 128 as unsigned bytes
    uint32_t t0, t1;
    asm("prmt.b32 %0, %1, %2, 0x4140;" : "=r"(t0) : "r"(u), "r"(0x64646464u));
    asm("prmt.b32 %0, %1, %2, 0x4342;" : "=r"(t1) : "r"(u), "r"(0x64646464u));
    const uint32_t bias = 0x64806480u;  // half2(1152, 1152)
    asm("sub.f16x2 %0, %1, %2;" : "=r"(lo) : "r"(t0), "r"(bias));
    asm("sub.f16x2 %0, %1, %2;" : "=r"(hi) : "r"(t1), "r"(bias));
}

// 4 packed bytes (keys k0..k3, byte = lo | hi << 4) -> A fragment of (code - 8):
// a0 = (lo k0, lo k2), a1 = (hi k0, hi k2), a2 = (lo k1, lo k3), a3 = (hi k1, hi k3).
__device__ __forceinline__ void u4x8_to_frag(uint32_t w, uint32_t (&a)[4]) {
    const uint32_t magic = 0x64006400u, mask = 0x000f000fu, bias = 0x64086408u;  // 1032
    uint32_t t[4];
    asm("lop3.b32 %0, %1, %2, %3, 0xea;" : "=r"(t[0]) : "r"(w), "r"(mask), "r"(magic));
    asm("lop3.b32 %0, %1, %2, %3, 0xea;" : "=r"(t[1]) : "r"(w >> 4), "r"(mask), "r"(magic));
    asm("lop3.b32 %0, %1, %2, %3, 0xea;" : "=r"(t[2]) : "r"(w >> 8), "r"(mask), "r"(magic));
    asm("lop3.b32 %0, %1, %2, %3, 0xea;" : "=r"(t[3]) : "r"(w >> 12), "r"(mask), "r"(magic));
#pragma unroll
    for (int i = 0; i < 4; ++i) asm("sub.f16x2 %0, %1, %2;" : "=r"(a[i]) : "r"(t[i]), "r"(bias));
}

// (x, y) fp32 -> f16x2 hi = rn(x, y), lo = rn(x - hi, y - hi).
__device__ __forceinline__ void split_f16(float x, float y, uint32_t &hi, uint32_t &lo) {
    const __half2 h = __floats2half2_rn(x, y);
    const float2 hf = __half22float2(h);
    const __half2 l = __floats2half2_rn(x - hf.x, y - hf.y);
    hi = *reinterpret_cast<const uint32_t *>(&h);
    lo = *reinterpret_cast<const uint32_t *>(&l);
}

__device__ __forceinline__ uint2 ldg_nc_u2(const void *p) {
    uint2 v;
    asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];"
                 : "=r"(v.x), "=r"(v.y)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ void cp_async16(void *smem, const void *gmem) {
    const uint32_t s = (uint32_t)__cvta_generic_to_shared(smem);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(s), "l"(gmem));
}

__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.commit_group;\ncp.async.wait_group 0;" ::: "memory");
}

// Shared-memory carve of decode_kernel<D, NT> for page size P (bytes).
struct DecodeSmem {
    int qf, sc, rmax, rsum, sv, svs, red, total;
};
__host__ __device__ inline int align16(int x) { return (x + 15) & ~15; }
__host__ __device__ inline DecodeSmem decode_smem(int D, int NT, int P) {
    DecodeSmem s;
    const int MR = NT * 8, SP = P + 4, NB = D / 32;
    int parts = 8 / NB;
    if (parts > P / 32) parts = P / 32;
    s.qf = 0;
    s.sc = align16(s.qf + NT * (D / 16) * 32 * 16);
    s.rmax = align16(s.sc + MR * SP * 4);
    s.rsum = align16(s.rmax + MR * 4);
    s.sv = align16(s.rsum + MR * 4);
    s.svs = align16(s.sv + (D / 2) * (P + 32));
    s.red = align16(s.svs + (D / 32) * P * 2);
    s.total = align16(s.red + (parts - 1) * MR * D * 4);
    return s;
}

template <int D, int NT>
__global__ void __launch_bounds__(kThreads, 2) decode_kernel(const __grid_constant__ DecodeParams p) {
    extern __shared__ __align__(16) uint8_t smem[];
    constexpr int NB = D / 32;  // 32-dim scale blocks
    constexpr int KS = D / 16;  // QK k-steps
    constexpr int MR = NT * 8;  // MMA rows (query rows x heads, padded to 8)
    const int P = p.geom.P;
    const int SP = P + 4;   // score row stride, floats
    const int SVS = P + 32;  // V nibble row stride in shared memory, bytes
    const DecodeSmem L = decode_smem(D, NT, P);
    uint4 *qf = reinterpret_cast<uint4 *>(smem + L.qf);
    float *sc = reinterpret_cast<float *>(smem + L.sc);
    float *rmax = reinterpret_cast<float *>(smem + L.rmax);
    float *rsum = reinterpret_cast<float *>(smem + L.rsum);
    uint8_t *sv = smem + L.sv;
    __half *svs = reinterpret_cast<__half *>(smem + L.svs);
    float *red = reinterpret_cast<float *>(smem + L.red);

    const int item = blockIdx.x, g = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, gid = lane >> 2, tig = lane & 3;
    const uint32_t page = p.page[item];
    const uint8_t *hb =
        p.arena + (int64_t)p.slot[item] * p.geom.page_bytes + (int64_t)g * p.geom.head_bytes;
    const int G = p.G, R = p.R, rows = G * R;

    // Stage the V section (nibbles + scales) into shared memory asynchronously.
    {
        const uint8_t *gvq = hb + p.geom.vq_off;
        const int cpr = P / 16;  // 16-byte chunks per nibble row
        for (int c = threadIdx.x; c < (D / 2) * cpr; c += kThreads) {
            const int row = c / cpr, col = c - row * cpr;
            cp_async16(sv + row * SVS + col * 16, gvq + (int64_t)row * P + col * 16);
        }
        const uint8_t *gvs = hb + p.geom.vs_off;
        for (int c = threadIdx.x; c < (D / 32) * P * 2 / 16; c += kThreads)
            cp_async16(reinterpret_cast<uint8_t *>(svs) + c * 16, gvs + c * 16);
        asm volatile("cp.async.commit_group;" ::: "memory");
    }

    // Q fragments: qf[nt][ks][lane] = {b0_hi, b1_hi, b0_lo, b1_lo}.
    for (int e = threadIdx.x; e < NT * KS * 32; e += kThreads) {
        const int ln = e & 31, ks = (e >> 5) % KS, nt = e / (KS * 32);
        const int m = nt * 8 + (ln >> 2);
        const int d0 = 32 * (ks >> 1) + 8 * (ln & 3) + 4 * (ks & 1);
        float x[4] = {0.f, 0.f, 0.f, 0.f};
        if (m < rows) {
            const int r = m / G, h = g * G + (m - r * G);
            const int64_t off = ((int64_t)r * p.Hq + h) * D + d0;
            if (p.q_f16) {
                const __half *q = reinterpret_cast<const __half *>(p.q) + off;
                const uint2 raw = *reinterpret_cast<const uint2 *>(q);
                const float2 a = __half22float2(*reinterpret_cast<const __half2 *>(&raw.x));
                const float2 b = __half22float2(*reinterpret_cast<const __half2 *>(&raw.y));
                x[0] = a.x; x[1] = a.y; x[2] = b.x; x[3] = b.y;
            } else {
                const float4 v = *reinterpret_cast<const float4 *>(reinterpret_cast<const float *>(p.q) + off);
                x[0] = v.x; x[1] = v.y; x[2] = v.z; x[3] = v.w;
            }
        }
        uint32_t h0, l0, h1, l1;
        split_f16(x[0], x[1], h0, l0);
        split_f16(x[2], x[3], h1, l1);
        qf[e] = make_uint4(h0, h1, l0, l1);
    }
    __syncthreads();

    // Scores: warp w owns keys [32w, 32w + 32) as two 16-key MMA row tiles.
    const long long kpos0 = (long long)page * P;
    if (warp < P / 32) {
#pragma unroll 1
        for (int mt = 0; mt < 2; ++mt) {
            const int k0 = warp * 32 + mt * 16 + gid, k1 = k0 + 8;
            const uint8_t *kr0 = hb + (int64_t)k0 * D + 8 * tig;
            const uint8_t *kr1 = hb + (int64_t)k1 * D + 8 * tig;
            const __half *ks0 = reinterpret_cast<const __half *>(hb + p.geom.ks_off) + k0 * NB;
            const __half *ks1 = reinterpret_cast<const __half *>(hb + p.geom.ks_off) + k1 * NB;
            uint2 kv0[NB], kv1[NB];
#pragma unroll
            for (int b = 0; b < NB; ++b) {
                kv0[b] = ldg_nc_u2(kr0 + 32 * b);
                kv1[b] = ldg_nc_u2(kr1 + 32 * b);
            }
            float sk0[NB], sk1[NB];
#pragma unroll
            for (int b = 0; b < NB; b += 2) {
                const float2 a = __half22float2(*reinterpret_cast<const __half2 *>(ks0 + b));
                const float2 c = __half22float2(*reinterpret_cast<const __half2 *>(ks1 + b));
                sk0[b] = a.x; sk0[b + 1] = a.y;
                sk1[b] = c.x; sk1[b + 1] = c.y;
            }
            float S[NT][4];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) S[nt][0] = S[nt][1] = S[nt][2] = S[nt][3] = 0.f;
#pragma unroll
            for (int b = 0; b < NB; ++b) {
                float cb[NT][4];
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) cb[nt][0] = cb[nt][1] = cb[nt][2] = cb[nt][3] = 0.f;
#pragma unroll
                for (int s = 0; s < 2; ++s) {
                    uint32_t a[4];
                    i8x4_to_f16(s ? kv0[b].y : kv0[b].x, a[0], a[2]);
                    i8x4_to_f16(s ? kv1[b].y : kv1[b].x, a[1], a[3]);
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) {
                        const uint4 qv = qf[(nt * KS + 2 * b + s) * 32 + lane];
                        mma16816(cb[nt], a, qv.x, qv.y);
                        mma16816(cb[nt], a, qv.z, qv.w);
                    }
                }
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    S[nt][0] += cb[nt][0] * sk0[b];
                    S[nt][1] += cb[nt][1] * sk0[b];
                    S[nt][2] += cb[nt][2] * sk1[b];
                    S[nt][3] += cb[nt][3] * sk1[b];
                }
            }
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int key = (e < 2) ? k0 : k1;
                    const int m = nt * 8 + 2 * tig + (e & 1);
                    const bool ok = m < rows && kpos0 + key <= p.pos0 + m / G;
                    sc[m * SP + key] = ok ? S[nt][e] * p.scale_log2 : -INFINITY;
                }
            }
        }
    }
    __syncthreads();

    // Softmax over the page's keys, one row per warp at a time.
    const int split = (int)page;
    for (int m = warp; m < MR; m += 8) {
        float mx = -INFINITY;
        for (int k = lane; k < P; k += 32) mx = fmaxf(mx, sc[m * SP + k]);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        float sum = 0.f;
        if (mx == -INFINITY) {
            for (int k = lane; k < P; k += 32) sc[m * SP + k] = 0.f;
        } else {
            for (int k = lane; k < P; k += 32) {
                const float e = exp2f(sc[m * SP + k] - mx);
                sc[m * SP + k] = e;
                sum += e;
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
        }
        if (lane == 0) {
            rmax[m] = mx;
            rsum[m] = sum;
            if (m < rows) {
                const int r = m / G, h = g * G + (m - r * G);
                float *ml = p.part_ml + (((int64_t)split * p.Hq + h) * R + r) * 2;
                ml[0] = mx;
                ml[1] = sum;
            }
        }
    }
    cp_async_wait_all();
    __syncthreads();

    // O^T = V^T P'^T: warp -> (32-dim block b, key part).
    int parts = 8 / NB;
    if (parts > P / 32) parts = P / 32;
    const int b = warp % NB, part = warp / NB;
    float acc[2][NT][4];
#pragma unroll
    for (int i = 0; i < 2; ++i)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) acc[i][nt][0] = acc[i][nt][1] = acc[i][nt][2] = acc[i][nt][3] = 0.f;
    if (part < parts) {
        const int kspan = P / parts;
#pragma unroll 1
        for (int kb = part * kspan; kb < (part + 1) * kspan; kb += 32) {
            const uint2 v0 = *reinterpret_cast<const uint2 *>(sv + (b * 16 + gid) * SVS + kb + 8 * tig);
            const uint2 v1 = *reinterpret_cast<const uint2 *>(sv + (b * 16 + 8 + gid) * SVS + kb + 8 * tig);
            const uint4 dvr = *reinterpret_cast<const uint4 *>(svs + b * P + kb + 8 * tig);
#pragma unroll
            for (int s = 0; s < 2; ++s) {
                uint32_t a0[4], a1[4];
                u4x8_to_frag(s ? v0.y : v0.x, a0);
                u4x8_to_frag(s ? v1.y : v1.x, a1);
                const float2 dA = __half22float2(*reinterpret_cast<const __half2 *>(s ? &dvr.z : &dvr.x));
                const float2 dB = __half22float2(*reinterpret_cast<const __half2 *>(s ? &dvr.w : &dvr.y));
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    const float4 pv = *reinterpret_cast<const float4 *>(sc + (nt * 8 + gid) * SP + kb + 8 * tig + 4 * s);
                    uint32_t bh0, bl0, bh1, bl1;
                    split_f16(pv.x * dA.x, pv.z * dB.x, bh0, bl0);  // keys +0, +2
                    split_f16(pv.y * dA.y, pv.w * dB.y, bh1, bl1);  // keys +1, +3
                    mma16816(acc[0][nt], a0, bh0, bh1);
                    mma16816(acc[0][nt], a0, bl0, bl1);
                    mma16816(acc[1][nt], a1, bh0, bh1);
                    mma16816(acc[1][nt], a1, bl0, bl1);
                }
            }
        }
    }
    if (parts > 1) {
        if (part >= 1 && part < parts) {
            float *dst = red + (part - 1) * MR * D;
#pragma unroll
            for (int mt = 0; mt < 2; ++mt)
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int dim = 32 * b + mt * 8 + gid + ((e >= 2) ? 16 : 0);
                        const int m = nt * 8 + 2 * tig + (e & 1);
                        dst[m * D + dim] = acc[mt][nt][e];
                    }
        }
        __syncthreads();
        if (part == 0) {
            for (int q = 1; q < parts; ++q) {
                const float *src = red + (q - 1) * MR * D;
#pragma unroll
                for (int mt = 0; mt < 2; ++mt)
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int dim = 32 * b + mt * 8 + gid + ((e >= 2) ? 16 : 0);
                            const int m = nt * 8 + 2 * tig + (e & 1);
                            acc[mt][nt][e] += src[m * D + dim];
                        }
            }
        }
    }
    if (part == 0) {
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int m = nt * 8 + 2 * tig + (e & 1);
                    if (m < rows) {
                        const int dim = 32 * b + mt * 8 + gid + ((e >= 2) ? 16 : 0);
                        const int r = m / G, h = g * G + (m - r * G);
                        p.part_o[(((int64_t)split * p.Hq + h) * R + r) * D + dim] = acc[mt][nt][e];
                    }
                }
    }
}

template <int D, int NT>
cudaError_t launch_decode_t(const DecodeParams &p, cudaStream_t s) {
    const DecodeSmem L = decode_smem(D, NT, p.geom.P);
    static int configured = 0;
    if (configured < L.total) {
        cudaError_t e = cudaFuncSetAttribute(decode_kernel<D, NT>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, L.total);
        if (e != cudaSuccess) return e;
        configured = L.total;
    }
    dim3 grid(p.n_items, p.geom.Hk);
    decode_kernel<D, NT><<<grid, kThreads, L.total, s>>>(p);
    return cudaGetLastError();
}

template <int D>
cudaError_t launch_decode_d(const DecodeParams &p, int nt, cudaStream_t s) {
    switch (nt) {
        case 1: return launch_decode_t<D, 1>(p, s);
        case 2: return launch_decode_t<D, 2>(p, s);
        case 3: return launch_decode_t<D, 3>(p, s);
        case 4: return launch_decode_t<D, 4>(p, s);
        case 5: return launch_decode_t<D, 5>(p, s);
        case 6: return launch_decode_t<D, 6>(p, s);
        case 7:
        case 8: return launch_decode_t<D, 8>(p, s);
        default: return cudaErrorInvalidValue;
    }
}

// ------------------------------------------------------------------ combine

template <int D>
__global__ void __launch_bounds__(kThreads) combine_kernel(const CombineParams p) {
    constexpr int VPL = D / 32;  // values per lane
    __shared__ float wm[8], wl[8];
    __shared__ float wo[8][D];
    const int rh = blockIdx.x, r = rh / p.Hq, h = rh - r * p.Hq;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nsplit = (int)((p.pos0 + r) / ((long long)p.P * p.split_pages)) + 1;
    float M = -INFINITY, Lsum = 0.f, o[VPL];
#pragma unroll
    for (int i = 0; i < VPL; ++i) o[i] = 0.f;
    for (int s = warp; s < nsplit; s += 8) {
        const int64_t base = ((int64_t)s * p.Hq + h) * p.R + r;
        const float ms = p.part_ml[base * 2], ls = p.part_ml[base * 2 + 1];
        if (!(ls > 0.f)) continue;
        const float Mn = fmaxf(M, ms);
        const float a = exp2f(M - Mn), c = exp2f(ms - Mn);
        const float *src = p.part_o + base * D + lane * VPL;
        float v[VPL];
#pragma unroll
        for (int i = 0; i < VPL; i += 2) {
            const float2 t = *reinterpret_cast<const float2 *>(src + i);
            v[i] = t.x;
            v[i + 1] = t.y;
        }
#pragma unroll
        for (int i = 0; i < VPL; ++i) o[i] = o[i] * a + v[i] * c;
        Lsum = Lsum * a + ls * c;
        M = Mn;
    }
    if (lane == 0) {
        wm[warp] = M;
        wl[warp] = Lsum;
    }
#pragma unroll
    for (int i = 0; i < VPL; ++i) wo[warp][lane * VPL + i] = o[i];
    __syncthreads();
    if (warp == 0) {
        float Mt = -INFINITY;
        for (int w = 0; w < 8; ++w)
            if (wl[w] > 0.f) Mt = fmaxf(Mt, wm[w]);
        float Lt = 0.f, ot[VPL];
#pragma unroll
        for (int i = 0; i < VPL; ++i) ot[i] = 0.f;
        if (Mt != -INFINITY) {
            for (int w = 0; w < 8; ++w) {
                if (!(wl[w] > 0.f)) continue;
                const float c = exp2f(wm[w] - Mt);
                Lt += wl[w] * c;
#pragma unroll
                for (int i = 0; i < VPL; ++i) ot[i] += wo[w][lane * VPL + i] * c;
            }
        }
        float *dst = p.out + ((int64_t)r * p.Hq + h) * D + lane * VPL;
        const float inv = (Lt > 0.f) ? 1.f / Lt : 0.f;
#pragma unroll
        for (int i = 0; i < VPL; ++i) dst[i] = ot[i] * inv;
        if (p.lse && lane == 0)
            p.lse[(int64_t)r * p.Hq + h] = (Lt > 0.f) ? (Mt + log2f(Lt)) * 0.69314718055994531f : -INFINITY;
    }
}

}  // namespace

int decode_max_mma_rows() { return 64; }

cudaError_t launch_decode(const DecodeParams &p, cudaStream_t s) {
    const int rows = p.G * p.R;
    if (rows < 1 || rows > 64 || p.n_items < 1 || p.n_items > kMaxItems) return cudaErrorInvalidValue;
    const int nt = (rows + 7) / 8;
    switch (p.geom.D) {
        case 64: return launch_decode_d<64>(p, nt, s);
        case 128: return launch_decode_d<128>(p, nt, s);
        case 256: return launch_decode_d<256>(p, nt, s);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_combine(const CombineParams &p, cudaStream_t s) {
    const int blocks = p.R * p.Hq;
    if (blocks < 1) return cudaSuccess;
    switch (p.D) {
        case 64: combine_kernel<64><<<blocks, kThreads, 0, s>>>(p); break;
        case 128: combine_kernel<128><<<blocks, kThreads, 0, s>>>(p); break;
        case 256: combine_kernel<256><<<blocks, kThreads, 0, s>>>(p); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace kvs
