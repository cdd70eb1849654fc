// Split-K paged attention for 1..N query rows over a Q8_0-K / Q4_0-V page,
// and the log-sum-exp combine of the per-page partials.
//
// One work unit = one (page, kv head).  Every query head of the kv head's
// group and every query row is served by the same unit, so each K/V byte is
// read from memory once per step.  The codes are dequantised tile by tile
// in registers; no f16 copy of the cache is ever made (Adaptive KV Streaming
// for llama.cpp V2, "Keep the stock attention order").
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
// Softmax over the page's keys runs in fp32 with exp2 on log2-scaled scores;
// each weight p is split once into f16 hi + lo, and every 32-dim block forms
// its P' = (hi + lo) * dV with f16x2 arithmetic: rn(hi dV), the exact
// remainder of that product by a fused multiply-add, plus lo dV.
//
// Fragment orders.  The reduction index of each MMA is permuted so that one
// 64-bit load gives a thread its whole fragment:
//   QK: thread (gid, tig) of a k-step in 32-dim block b holds dims
//       32b + 8*tig + 4*s + {0..3} (s = k-step within the block), i.e. one
//       32-bit word of an 8-byte load of the key row.
//   PV: the page stores V by byte row (= dim pair) with 32 tokens per line, a
//       thread's word holds 4 consecutive keys of one dim pair; the four MMA
//       k positions (2t, 2t+1, 2t+8, 2t+9) map to keys (+0, +2, +1, +3) and
//       the MMA rows (gid, gid+8) to the low/high nibble dims of that byte.
// The int8 -> f16 and nibble -> f16 conversions use the exponent-bias trick
// described by Kim et al., "Who Says Elephants Can't Run: Bringing Large
// Scale MoE Models into Cloud Scale Production" (2022): a small integer u
// placed in the mantissa under exponent 0x64 is the half 1024 + u.  A K code
// x becomes 1152 + x that way and one f16x2 subtraction gives x exactly.
// High V nibbles are taken in mantissa bits 4-7 as 16 * (code - 8) and their
// output rows scaled by 1/16.
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

// 4 int8 (bytes x0..x3 of w) -> f16x2 (x0, x1) and (x2, x3), exact: the
// byte x + 128 under exponent 0x64 is 1024 + 128 + x, minus 1152 (0x6480).
__device__ __forceinline__ void i8x4_to_f16(uint32_t w, uint32_t &lo, uint32_t &hi) {
    const uint32_t u = w ^ 0x80808080u;
    uint32_t bl, bh;
    asm("prmt.b32 %0, %1, %2, 0x4140;" : "=r"(bl) : "r"(u), "r"(0x64646464u));
    asm("prmt.b32 %0, %1, %2, 0x4342;" : "=r"(bh) : "r"(u), "r"(0x64646464u));
    asm("sub.f16x2 %0, %1, %2;" : "=r"(lo) : "r"(bl), "r"(0x64806480u));
    asm("sub.f16x2 %0, %1, %2;" : "=r"(hi) : "r"(bh), "r"(0x64806480u));
}

// 4 packed bytes (keys k0..k3, byte = lo | hi << 4) -> A fragment:
// a0 = (lo k0, lo k2) - 8, a2 = (lo k1, lo k3) - 8 and, for the high nibbles,
// a1 = 16 * ((hi k0, hi k2) - 8), a3 = 16 * ((hi k1, hi k3) - 8): the nibble
// stays in mantissa bits 4-7, so the MMA rows it feeds come out 16 times too
// large and are scaled by 1/16 (exactly) at the end.
__device__ __forceinline__ void u4x8_to_frag16(uint32_t w, uint32_t (&a)[4]) {
    const uint32_t magic = 0x64006400u, lo = 0x000f000fu, hi = 0x00f000f0u;
    const uint32_t bias_lo = 0x64086408u;  // 1032 = 1024 + 8
    const uint32_t bias_hi = 0x64806480u;  // 1152 = 1024 + 16 * 8
    const uint32_t w8 = w >> 8;
    uint32_t t0, t1, t2, t3;
    asm("lop3.b32 %0, %1, %2, %3, 0xea;" : "=r"(t0) : "r"(w), "r"(lo), "r"(magic));
    asm("lop3.b32 %0, %1, %2, %3, 0xea;" : "=r"(t1) : "r"(w), "r"(hi), "r"(magic));
    asm("lop3.b32 %0, %1, %2, %3, 0xea;" : "=r"(t2) : "r"(w8), "r"(lo), "r"(magic));
    asm("lop3.b32 %0, %1, %2, %3, 0xea;" : "=r"(t3) : "r"(w8), "r"(hi), "r"(magic));
    asm("sub.f16x2 %0, %1, %2;" : "=r"(a[0]) : "r"(t0), "r"(bias_lo));
    asm("sub.f16x2 %0, %1, %2;" : "=r"(a[1]) : "r"(t1), "r"(bias_hi));
    asm("sub.f16x2 %0, %1, %2;" : "=r"(a[2]) : "r"(t2), "r"(bias_lo));
    asm("sub.f16x2 %0, %1, %2;" : "=r"(a[3]) : "r"(t3), "r"(bias_hi));
}

// (hi + lo) * d for f16x2 pairs: ph = rn(hi d), pl = rn(lo d + (hi d - ph)),
// where hi d - ph is formed exactly by a fused multiply-add
__device__ __forceinline__ void scale_split(uint32_t hi, uint32_t lo, uint32_t d, uint32_t &ph, uint32_t &pl) {
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(ph) : "r"(hi), "r"(d));
    uint32_t r;
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(r) : "r"(hi), "r"(d), "r"(ph ^ 0x80008000u));
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(pl) : "r"(lo), "r"(d), "r"(r));
}

// (x, y) fp32 -> f16x2 hi = rn(x, y), lo = rn(x - hi, y - hi).
__device__ __forceinline__ void split_f16(float x, float y, uint32_t &hi, uint32_t &lo) {
    const __half2 h = __floats2half2_rn(x, y);
    const float2 hf = __half22float2(h);
    const __half2 l = __floats2half2_rn(x - hf.x, y - hf.y);
    hi = *reinterpret_cast<const uint32_t *>(&h);
    lo = *reinterpret_cast<const uint32_t *>(&l);
}

__device__ __forceinline__ uint32_t smem_u32(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

constexpr uint32_t kSpinLimit = 1u << 26;

// bounded wait for phase `parity` of an mbarrier; false after `limit` polls
// one non-blocking test: has the phase of this parity completed?
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    return done != 0;
}

__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, uint32_t limit = kSpinLimit) {
    for (uint32_t i = 0; i < limit; ++i) {
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

// one page-head section (global, contiguous) -> shared stage, completion on `bar`
__device__ __forceinline__ void stage_load(uint32_t dst, const uint8_t *src, uint32_t bytes, uint32_t bar) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
    // in pieces of at most 64 KiB
    for (uint32_t off = 0; off < bytes; off += 65536u) {
        const uint32_t n = (bytes - off) < 65536u ? (bytes - off) : 65536u;
        asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                         dst + off),
                     "l"(src + off), "r"(n), "r"(bar)
                     : "memory");
    }
}

// Key parts of the P.V product.  A page's O^T is the ordered sum
// part 0 + part 1 + ... of per-key-range MMA chains, whatever the launch
// shape, so a page's partial is bitwise the same from every launch shape.
__host__ __device__ inline int pv_parts(int D, int P) {
    int parts = 8 / (D / 32);
    if (parts < 2) parts = 2;
    if (parts > P / 32) parts = P / 32;
    return parts < 1 ? 1 : parts;
}

// Shared-memory carve of decode_kernel<D, NT, W, SPL> (bytes; page size P, S stages).
struct DecodeSmem {
    int stage, sc, red, obuf, obs, rowoff, rowtab, bar, total, stages;  // obs: output row stride (floats)
};
__host__ __device__ inline int align_to(int x, int a) { return (x + a - 1) / a * a; }
__host__ __device__ inline DecodeSmem decode_smem(int D, int NT, int W, int P, int stages) {
    DecodeSmem s;
    const int MR = NT * 8, SP = P + 4;
    const bool in_reg = (W == D / 32);  // a warp keeps every key part of its dim block in registers
    const int head = P * D * 13 / 8;
    s.stages = stages;
    s.stage = 0;
    s.sc = align_to(stages * head, 128);
    s.red = align_to(s.sc + MR * SP * 4, 16);
    const int red_end = s.red + (in_reg ? 0 : (pv_parts(D, P) - 1) * MR * D * 4);
    // the output tile reuses the score buffer when it fits there; its row stride
    // is 4 mod 32 floats, so a warp's fragment writes fall on distinct banks
    s.obs = (SP >= D + 4) ? SP : D + 4;
    s.obuf = (SP >= D + 4) ? s.sc : align_to(red_end, 16);
    const int obuf_end = (SP >= D + 4) ? red_end : s.obuf + MR * s.obs * 4;
    s.rowoff = align_to(red_end > obuf_end ? red_end : obuf_end, 16);  // MR ints: partial row offsets
    s.rowtab = align_to(s.rowoff + MR * 4, 16);  // 64 int2 per CTA: (mg / G, (mg % G) * R + mg / G)
    s.bar = align_to(s.rowtab + 64 * 8, 16);
    s.total = s.bar + 32 * stages;  // per stage: K-piece and V-piece barriers
    return s;
}

// Persistent split-K attention over work units.  A unit is one (page, kv
// head) with all NT row tiles (resident pages), or, in tile mode, one (page,
// kv head, row tile) (NT = 1: ring chunks, where a chunk is a few pages and
// the time until its slots can be refilled matters more than throughput).
// Both shapes run the same arithmetic per row tile, for any warp count W.
// Units are ordered head-major; CTA c takes units [c*U/C, (c+1)*U/C).
// Page-head sections stream into `stages` shared-memory stages by bulk
// asynchronous copies, in two pieces with a barrier each: the K piece (codes
// and scales) and the V piece.  A stage's K piece is refilled with a later
// unit as soon as the scores are done, its V piece once P.V is done, so the
// copies of the next unit overlap the softmax, P.V and store of this one.
template <int D, int NT, int W, bool SPL>
__global__ void __launch_bounds__(W * 32, (NT == 1 && W == 8) ? 2 : 1)
    decode_kernel(const __grid_constant__ DecodeParams p) {
    extern __shared__ __align__(128) uint8_t smem[];
    // launched as a programmatic dependent: nothing is read before the grids
    // this launch depends on have completed and their writes are visible
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (p.rec && blockIdx.x == 0 && threadIdx.x == 0) {
        // a ring chunk's read: account its wait for the copy and clear the record
        unsigned long long t;
        asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
        volatile unsigned long long *rc = p.rec;
        const unsigned long long fs = ~rc[0], fe = rc[1];
        if (fe != 0 && rc[0] != 0) {
            const unsigned long long wait = t > fe ? t - fe : 0ull;
            ObsAccumulator *a = reinterpret_cast<ObsAccumulator *>(p.acc);
            atomicAdd(&a->reads, 1ull);
            if (wait < kMissNs) atomicAdd(&a->misses, 1ull);
            atomicAdd(&a->occupancy_page_ns, wait * (unsigned long long)p.rec_pages);
            atomicAdd(&a->fill_busy_ns, fe > fs ? fe - fs : 0ull);
            atomicAdd(&a->fill_bytes, (unsigned long long)p.rec_pages * (unsigned long long)p.geom.page_bytes);
            atomicMax(&a->first_fill_neg, ~fs);
            atomicMax(&a->last_read, t);
        }
        rc[0] = 0ull;
        rc[1] = 0ull;
    }
    tl_begin(p.tl);
    constexpr int NB = D / 32;  // 32-dim scale blocks
    constexpr int KS = D / 16;  // QK k-steps
    constexpr int MR = NT * 8;  // MMA rows (query rows x heads, padded to 8)
    constexpr int NTH = W * 32;
    constexpr bool kInReg = (W == NB);                 // see decode_smem
    constexpr int PM = kInReg ? 2 : 1;                 // key parts a warp accumulates
    constexpr int KPW = (NT == 1 && W == 8) ? 2 : 1;   // 16-key groups a warp scores at once
    const int P = p.geom.P;
    const int SP = P + 4;  // score row stride, floats
    const int parts = pv_parts(D, P);
    const DecodeSmem L = decode_smem(D, NT, W, P, p.stages);
    float *sc = reinterpret_cast<float *>(smem + L.sc);
    float *red = reinterpret_cast<float *>(smem + L.red);
    float *obuf = reinterpret_cast<float *>(smem + L.obuf);
    int *rowoff = reinterpret_cast<int *>(smem + L.rowoff);
    int2 *rowtab = reinterpret_cast<int2 *>(smem + L.rowtab);
    const uint32_t bar0 = smem_u32(smem + L.bar);
    const int head_bytes = (int)p.geom.head_bytes;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, gid = lane >> 2, tig = lane & 3;
    // this launch serves query rows row0 .. row0 + Rg - 1 of the call's R rows
    const int G = p.G, R = p.R, rows = G * p.Rg, row0 = p.row0;
    const int T = p.tile_mode ? p.run_tiles : 1;
    const int U = p.n_items * p.geom.Hk * T;
    const int u0 = (int)((int64_t)blockIdx.x * U / gridDim.x), u1 = (int)((int64_t)(blockIdx.x + 1) * U / gridDim.x);
    if (u0 >= u1) {
        tl_finish(p.tl);
        return;
    }
    const int S = L.stages;

    auto src_of = [&](int u) {
        const int gi = u / T, g = gi / p.n_items, item = gi - g * p.n_items;
        return p.arena + (int64_t)p.slot[item] * p.geom.page_bytes + (int64_t)g * p.geom.head_bytes;
    };
    // barrier 2s: K piece of stage s, 2s + 1: its V piece
    const uint32_t kbytes = (uint32_t)p.geom.vq_off, vbytes = (uint32_t)head_bytes - kbytes;
    auto load_piece = [&](int s, int unit, int v) {
        const uint32_t off = v ? kbytes : 0u;
        stage_load(smem_u32(smem + L.stage + s * head_bytes) + off, src_of(unit) + off, v ? vbytes : kbytes,
                   bar0 + 16 * (2 * s + v));
    };
    // bit j of `pending`: a load on barrier j is not consumed yet; bit j of
    // `pend_parity`: the phase that load completes
    uint32_t pending = 0u, pend_parity = 0u;
    for (int s = 0; s < S && u0 + s < u1; ++s) pending |= 1u << (2 * s);
    // rows x heads m (< 64): x = its query row r = row0 + m / G, y = h_local * R + r
    // with h_local = m % G; the partial of kv head g sits at row g * G * R + y
    for (int m = threadIdx.x; m < 64; m += NTH) rowtab[m] = make_int2(row0 + m / G, (m % G) * R + row0 + m / G);
    if (threadIdx.x == 0) {
        for (int s = 0; s < 2 * S; ++s) asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(bar0 + 16 * s));
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        // the first units' K pieces only: every CTA starts at once, and the
        // scores can begin as soon as K is in; their V pieces follow below
        for (int s = 0; s < S && u0 + s < u1; ++s) load_piece(s, u0 + s, 0);
    }
    __syncthreads();

    bool ok = true, triggered = false;
    const uint32_t limit = p.give_up_waits ? 0u : kSpinLimit;
    // unit u = (g * n_items + item) * T + tile, advanced incrementally
    int tile = u0 % T, item = (u0 / T) % p.n_items, g = u0 / T / p.n_items;
    for (int u = u0, i = 0; u < u1; ++u, ++i) {
        if (i > 0 && ++tile == T) {
            tile = 0;
            if (++item == p.n_items) item = 0, ++g;
        }
        const int stage = i % S;
        const uint32_t parity = (uint32_t)((i / S) & 1);
        const int mo = tile * 8;  // first query row x head of this unit's tiles
        const uint32_t page = p.page[item];
        const uint8_t *hs = smem + L.stage + stage * head_bytes;  // this unit's page-head section

        // Q fragments of kv head g (built by qprep_kernel): qf[tile][ks][lane]
        const uint4 *qf = p.qf + ((int64_t)g * p.qtiles + tile) * KS * 32;
        const uint2 *qf2 = reinterpret_cast<const uint2 *>(p.qf) + ((int64_t)g * p.qtiles + tile) * KS * 32;
        if (!mbar_wait(bar0 + 16 * (2 * stage), parity, limit)) ok = false;
        if (!__syncthreads_and(ok)) break;
        pending &= ~(1u << (2 * stage));
        if (i == 0) {  // the first units' V pieces, behind their K pieces
            for (int s = 0; s < S && u0 + s < u1; ++s) pending |= 2u << (2 * s);
            if (threadIdx.x == 0)
                for (int s = 0; s < S && u0 + s < u1; ++s) load_piece(s, u0 + s, 1);
        }

        // Scores: each warp takes KPW 16-key groups at a time as MMA row tiles.
        const long long kpos0 = (long long)page * P;
        // per stored row (nt, parity): the last visible key of this page, -1 if none
        int klim[NT][2];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int par = 0; par < 2; ++par) {
                const int mg = mo + nt * 8 + 2 * tig + par;
                const long long l = mg < rows ? p.pos0 - kpos0 + rowtab[mg].x : -1;
                klim[nt][par] = l < -1 ? -1 : (l > P ? P : (int)l);
            }
        const int NKG = P / 16;
        const __half *ksc = reinterpret_cast<const __half *>(hs + p.geom.ks_off);
#pragma unroll 1
        for (int kgb = 0; kgb < NKG; kgb += W * KPW) {
            if (kgb + warp >= NKG) break;
            int kg[KPW];
            bool kvalid[KPW];
#pragma unroll
            for (int q = 0; q < KPW; ++q) {
                kg[q] = kgb + warp + W * q;
                kvalid[q] = kg[q] < NKG;
                if (!kvalid[q]) kg[q] = kgb + warp;  // computed, never stored
            }
            float S_[KPW][NT][4];
#pragma unroll
            for (int q = 0; q < KPW; ++q)
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) S_[q][nt][0] = S_[q][nt][1] = S_[q][nt][2] = S_[q][nt][3] = 0.f;
#pragma unroll(NT == 1 ? NB : (NT == 2 ? 2 : 1))
            for (int b = 0; b < NB; ++b) {
                uint2 kv0[KPW], kv1[KPW];
                float sk0[KPW], sk1[KPW];
#pragma unroll
                for (int q = 0; q < KPW; ++q) {
                    const uint8_t *line = hs + ((kg[q] * NB + b) * 16) * 32 + 8 * tig;
                    kv0[q] = *reinterpret_cast<const uint2 *>(line + gid * 32);
                    kv1[q] = *reinterpret_cast<const uint2 *>(line + (gid + 8) * 32);
                    sk0[q] = __half2float(ksc[(16 * kg[q] + gid) * NB + b]);
                    sk1[q] = __half2float(ksc[(16 * kg[q] + gid + 8) * NB + b]);
                }
                float cb[KPW][NT][4];
#pragma unroll
                for (int q = 0; q < KPW; ++q)
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) cb[q][nt][0] = cb[q][nt][1] = cb[q][nt][2] = cb[q][nt][3] = 0.f;
#pragma unroll
                for (int s = 0; s < 2; ++s) {
                    uint32_t a[KPW][4];
#pragma unroll
                    for (int q = 0; q < KPW; ++q) {
                        i8x4_to_f16(s ? kv0[q].y : kv0[q].x, a[q][0], a[q][2]);
                        i8x4_to_f16(s ? kv1[q].y : kv1[q].x, a[q][1], a[q][3]);
                    }
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) {
                        if (SPL) {
                            const uint4 qv = qf[(nt * KS + 2 * b + s) * 32 + lane];
#pragma unroll
                            for (int q = 0; q < KPW; ++q) {
                                mma16816(cb[q][nt], a[q], qv.x, qv.y);
                                mma16816(cb[q][nt], a[q], qv.z, qv.w);
                            }
                        } else {
                            const uint2 qv = qf2[(nt * KS + 2 * b + s) * 32 + lane];
#pragma unroll
                            for (int q = 0; q < KPW; ++q) mma16816(cb[q][nt], a[q], qv.x, qv.y);
                        }
                    }
                }
                // the block's Q8_0 scale multiplies its fp32 partial dot
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int q = 0; q < KPW; ++q) {
                        S_[q][nt][0] = fmaf(cb[q][nt][0], sk0[q], S_[q][nt][0]);
                        S_[q][nt][1] = fmaf(cb[q][nt][1], sk0[q], S_[q][nt][1]);
                        S_[q][nt][2] = fmaf(cb[q][nt][2], sk1[q], S_[q][nt][2]);
                        S_[q][nt][3] = fmaf(cb[q][nt][3], sk1[q], S_[q][nt][3]);
                    }
            }
#pragma unroll
            for (int q = 0; q < KPW; ++q) {
                if (!kvalid[q]) continue;
                const int k0 = 16 * kg[q] + gid, k1 = k0 + 8;
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int key = (e < 2) ? k0 : k1;
                        const int m = nt * 8 + 2 * tig + (e & 1);
                        const bool valid = key <= klim[nt][e & 1];
                        sc[m * SP + key] = valid ? S_[q][nt][e] * p.scale_log2 : -INFINITY;
                    }
                }
            }
        }
        // scores written; the K piece is read.  On the last unit, if its V piece
        // has landed too, every page section this CTA reads is in shared memory:
        // a refill of those slots launched as this grid's programmatic dependent
        // may be scheduled now rather than after the softmax (when the launch asks)
        bool v_in = false;
        if (p.early_dependents && u == u1 - 1 && threadIdx.x == 0) v_in = mbar_test(bar0 + 16 * (2 * stage + 1), parity);
        if (__syncthreads_or(v_in)) {
            asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
            triggered = true;
        }
        if (u + S < u1) {
            pending |= 1u << (2 * stage);
            pend_parity = (pend_parity & ~(1u << (2 * stage))) | ((parity ^ 1u) << (2 * stage));
            if (threadIdx.x == 0) {
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                load_piece(stage, u + S, 0);
            }
        }

        // Softmax over the page's keys, one row per warp at a time.  Each lane
        // owns 4-key groups (at most two: P <= 256) and rewrites a group's four
        // fp32 scores in place as the PV B-fragment record of its weights e as
        // f16 pairs hi = rn(e), lo = rn(e - hi): {hi k0,k2 | hi k1,k3 | lo k0,k2 |
        // lo k1,k3}, the key order of the MMA's k positions (2t, 2t+1, 2t+8, 2t+9).
        const int split = (int)page;
        for (int m = warp; m < MR; m += W) {
            float4 sg[2];
            float mx = -INFINITY;
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                const int k4 = 4 * (lane + 32 * q);
                sg[q] = k4 < P ? *reinterpret_cast<const float4 *>(sc + m * SP + k4)
                               : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
                mx = fmaxf(fmaxf(mx, fmaxf(sg[q].x, sg[q].y)), fmaxf(sg[q].z, sg[q].w));
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
            float sum = 0.f;
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                const int k4 = 4 * (lane + 32 * q);
                if (k4 >= P) continue;
                float e[4] = {0.f, 0.f, 0.f, 0.f};
                if (mx != -INFINITY) {
                    // 2^x by the SFU's approximation (relative error about 2^-22; a
                    // masked key's -inf gives +0)
                    e[0] = ex2_approx(sg[q].x - mx);
                    e[1] = ex2_approx(sg[q].y - mx);
                    e[2] = ex2_approx(sg[q].z - mx);
                    e[3] = ex2_approx(sg[q].w - mx);
                }
                sum += (e[0] + e[1]) + (e[2] + e[3]);
                if (SPL) {
                    uint32_t h02, l02, h13, l13;
                    split_f16(e[0], e[2], h02, l02);
                    split_f16(e[1], e[3], h13, l13);
                    *reinterpret_cast<uint4 *>(sc + m * SP + k4) = make_uint4(h02, h13, l02, l13);
                } else {
                    const __half2 h02 = __floats2half2_rn(e[0], e[2]), h13 = __floats2half2_rn(e[1], e[3]);
                    *reinterpret_cast<uint2 *>(sc + m * SP + k4) =
                        make_uint2(*reinterpret_cast<const uint32_t *>(&h02), *reinterpret_cast<const uint32_t *>(&h13));
                }
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
            const int mg = mo + m;
            if (lane == 0 && mg < rows) {
                const int off = g * G * R + rowtab[mg].y;  // (h * R + r) of this row
                rowoff[m] = off;
                float *ml = p.part_ml + ((int64_t)split * p.Hq * R + off) * 2;
                ml[0] = mx;
                ml[1] = sum;
            }
        }
        if (!mbar_wait(bar0 + 16 * (2 * stage + 1), parity, limit)) ok = false;
        if (!__syncthreads_and(ok)) break;
        pending &= ~(2u << (2 * stage));
        // every page section this CTA reads is now in shared memory: a refill
        // of those slots launched as this grid's programmatic dependent may
        // start (it begins once every CTA has signalled or exited)
        if (u == u1 - 1 && !triggered) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

        // O^T = V^T P'^T over key parts: job j = (dim block j % NB, key part j / NB).
        // A warp owns every part of its block (kInReg) or one job.
        int b, part0;
        bool has_job;
        if (kInReg) {
            b = warp;
            part0 = 0;
            has_job = true;
        } else {
            b = warp % NB;
            part0 = warp / NB;
            has_job = part0 < parts;
        }
        const int kspan = P / parts;
        float acc[PM][2][NT][4];
#pragma unroll
        for (int pp = 0; pp < PM; ++pp)
#pragma unroll
            for (int i2 = 0; i2 < 2; ++i2)
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int e = 0; e < 4; ++e) acc[pp][i2][nt][e] = 0.f;
        if (has_job) {
            const __half *vsc = reinterpret_cast<const __half *>(hs + p.geom.vs_off);
#pragma unroll 1
            for (int i0 = 0; i0 < kspan; i0 += 32) {
#pragma unroll
                for (int pp = 0; pp < PM; ++pp) {
                    if (kInReg && pp >= parts) continue;
                    const int kb = (kInReg ? pp : part0) * kspan + i0;
                    const uint8_t *vl = hs + p.geom.vq_off + ((kb / 32 * NB + b) * 16) * 32 + 8 * tig;
                    const uint2 v0 = *reinterpret_cast<const uint2 *>(vl + gid * 32);
                    const uint2 v1 = *reinterpret_cast<const uint2 *>(vl + (gid + 8) * 32);
                    const uint4 dvr = *reinterpret_cast<const uint4 *>(vsc + b * P + kb + 8 * tig);
#pragma unroll
                    for (int s = 0; s < 2; ++s) {
                        uint32_t a0[4], a1[4];
                        u4x8_to_frag16(s ? v0.y : v0.x, a0);
                        u4x8_to_frag16(s ? v1.y : v1.x, a1);
                        // Q4_0 scales of keys (+0, +2) and (+1, +3) as f16 pairs
                        const uint32_t dlo = s ? dvr.z : dvr.x, dhi = s ? dvr.w : dvr.y;
                        uint32_t d02, d13;
                        asm("prmt.b32 %0, %1, %2, 0x5410;" : "=r"(d02) : "r"(dlo), "r"(dhi));
                        asm("prmt.b32 %0, %1, %2, 0x7632;" : "=r"(d13) : "r"(dlo), "r"(dhi));
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt) {
                            const float *rec = sc + (nt * 8 + gid) * SP + kb + 8 * tig + 4 * s;
                            if (SPL) {
                                const uint4 pr = *reinterpret_cast<const uint4 *>(rec);
                                // P' = (hi + lo) * d: hi * d rounded, its exact remainder, plus lo * d
                                uint32_t bh0, bl0, bh1, bl1;
                                scale_split(pr.x, pr.z, d02, bh0, bl0);  // keys +0, +2
                                scale_split(pr.y, pr.w, d13, bh1, bl1);  // keys +1, +3
                                mma16816(acc[pp][0][nt], a0, bh0, bh1);
                                mma16816(acc[pp][1][nt], a1, bh0, bh1);
                                mma16816(acc[pp][0][nt], a0, bl0, bl1);
                                mma16816(acc[pp][1][nt], a1, bl0, bl1);
                            } else {
                                // P' = rn(p * d), p already rounded to f16
                                const uint2 pr = *reinterpret_cast<const uint2 *>(rec);
                                uint32_t b0, b1;
                                asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(b0) : "r"(pr.x), "r"(d02));
                                asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(b1) : "r"(pr.y), "r"(d13));
                                mma16816(acc[pp][0][nt], a0, b0, b1);
                                mma16816(acc[pp][1][nt], a1, b0, b1);
                            }
                        }
                    }
                }
            }
        }
        if (kInReg && parts > 1) {
#pragma unroll
            for (int i2 = 0; i2 < 2; ++i2)
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int e = 0; e < 4; ++e) acc[0][i2][nt][e] += acc[PM - 1][i2][nt][e];
        }
        if (!kInReg && has_job && part0 >= 1) {
            float *dst = red + (part0 - 1) * MR * D;
#pragma unroll
            for (int mt = 0; mt < 2; ++mt)
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int dim = 32 * b + mt * 8 + gid + ((e >= 2) ? 16 : 0);
                        const int m = nt * 8 + 2 * tig + (e & 1);
                        dst[m * D + dim] = acc[0][mt][nt][e];
                    }
        }
        __syncthreads();  // every read of this stage (and of sc) is done
        if (u + S < u1) {
            pending |= 2u << (2 * stage);
            pend_parity = (pend_parity & ~(2u << (2 * stage))) | ((parity ^ 1u) << (2 * stage + 1));
            if (threadIdx.x == 0) {
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                load_piece(stage, u + S, 1);
            }
        }
        if (part0 == 0) {
            if (!kInReg) {
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
                                acc[0][mt][nt][e] += src[m * D + dim];
                            }
                }
            }
            // This warp owns dims 32 b .. 32 b + 31 of every row: it stages them in its
            // own columns of the output tile and stores them itself, 128 contiguous
            // bytes per row, so no CTA barrier separates staging and store.  Rows
            // gid + 8 (high-nibble dims) carried 16 * (code - 8).
            const int OS = L.obs;
#pragma unroll
            for (int mt = 0; mt < 2; ++mt)
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int dim = 32 * b + mt * 8 + gid + ((e >= 2) ? 16 : 0);
                        const int m = nt * 8 + 2 * tig + (e & 1);
                        obuf[m * OS + dim] = (e >= 2) ? acc[0][mt][nt][e] * 0.0625f : acc[0][mt][nt][e];
                    }
            __syncwarp();
            // the valid rows, at their partial rows (offsets from the table)
            const int urows = rows - mo < MR ? rows - mo : MR;
            const int64_t split_base = (int64_t)split * p.Hq * R;
            const int d4 = 32 * b + 4 * (lane & 7);
            for (int m = lane >> 3; m < urows; m += 4)
                *reinterpret_cast<float4 *>(p.part_o + (split_base + rowoff[m]) * D + d4) =
                    *reinterpret_cast<const float4 *>(obuf + m * OS + d4);
        }
        __syncthreads();  // obuf / sc free for the next unit
    }
    if (!ok) {
        // a wait gave up: before the CTA exits, wait (bounded again) for every
        // stage load still in flight, so no copy lands in reassigned memory
        if (threadIdx.x == 0) {
            for (int s = 0; s < 2 * S; ++s)
                if ((pending >> s) & 1u) mbar_wait(bar0 + 16 * s, (pend_parity >> s) & 1u);
            atomicExch(p.status, 1);
        }
        __syncthreads();
    }
    if (p.tl) {
        __syncthreads();
        tl_finish(p.tl);
    }
}

// Q fragments for every kv head, once per attend: qf [Hk][NT][KS][32] uint4
// = {b0_hi, b1_hi, b0_lo, b1_lo} of the QK B operand.  One CTA per (kv head,
// row tile): the kernel sits between two layers' reads, so its latency counts.
template <int D, int NT, bool SPL>
__global__ void __launch_bounds__(kThreads) qprep_kernel(const __grid_constant__ DecodeParams p) {
    asm volatile("griddepcontrol.wait;" ::: "memory");            // q and the previous readers of qf
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");  // attention may be scheduled
    tl_begin(p.tl_prep);
    constexpr int KS = D / 16;
    const int g = blockIdx.x, nt = blockIdx.y, G = p.G, rows = G * p.Rg;
    uint4 *qf = const_cast<uint4 *>(p.qf) + ((int64_t)g * NT + nt) * KS * 32;
    uint2 *qf2 = reinterpret_cast<uint2 *>(const_cast<uint4 *>(p.qf)) + ((int64_t)g * NT + nt) * KS * 32;
    for (int e = threadIdx.x; e < KS * 32; e += kThreads) {
        const int ln = e & 31, ks = e >> 5;
        const int m = nt * 8 + (ln >> 2);
        const int d0 = 32 * (ks >> 1) + 8 * (ln & 3) + 4 * (ks & 1);
        float x[4] = {0.f, 0.f, 0.f, 0.f};
        if (m < rows) {
            const int rl = m / G, r = p.row0 + rl, h = g * G + (m - rl * G);
            const int64_t off = ((int64_t)r * p.Hq + h) * D + d0;
            if (p.q_f16) {
                const uint2 raw = *reinterpret_cast<const uint2 *>(reinterpret_cast<const __half *>(p.q) + off);
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
        if (SPL)
            qf[e] = make_uint4(h0, h1, l0, l1);
        else
            qf2[e] = make_uint2(h0, h1);
    }
    if (p.tl_prep) {
        __syncthreads();
        tl_finish(p.tl_prep);
    }
}

// Launch as a programmatic dependent of the previous kernel on `s`: the grid
// may be scheduled once that kernel signals (griddepcontrol.launch_dependents)
// and waits in griddepcontrol.wait for its completion before touching memory.
template <typename K, typename A>
cudaError_t launch_pdl(K kernel, dim3 grid, dim3 block, int smem, cudaStream_t s, const A &arg) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = (size_t)smem;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, arg);
    return e != cudaSuccess ? e : cudaGetLastError();
}

template <int D, int NT, int W, bool SPL>
cudaError_t launch_decode_t(const DecodeParams &p_in, cudaStream_t s) {
    DecodeParams p = p_in;
    if (p.prep_q) {
        cudaError_t e = launch_pdl(qprep_kernel<D, NT, SPL>, dim3(p.geom.Hk, NT), dim3(kThreads), 0, s, p);
        if (e != cudaSuccess) return e;
        if (p.n_items == 0) return cudaSuccess;
    }
    const int maxsm = 232448;
    // W = 8, one row tile: one stage per CTA and two CTAs per SM when they fit
    // (the other CTA's copy overlaps this one's compute); otherwise one CTA
    // per SM with two stages
    int occ = (NT == 1 && W == 8) ? 2 : 1;
    const int n_sms = current_device_sms();
    DecodeSmem L = decode_smem(D, NT, W, p.geom.P, occ == 2 ? 1 : 2);
    if (occ == 2 && 2 * (L.total + 1024) > 233472) occ = 1, L = decode_smem(D, NT, W, p.geom.P, 2);
    if (L.total > maxsm) L = decode_smem(D, NT, W, p.geom.P, 1);
    if (L.total > maxsm) return cudaErrorInvalidValue;
    p.stages = L.stages;
    {
        cudaError_t e = ensure_smem_limit(reinterpret_cast<const void *>(decode_kernel<D, NT, W, SPL>), L.total);
        if (e != cudaSuccess) return e;
    }
    const int U = p.n_items * p.geom.Hk * (p.tile_mode ? p.run_tiles : 1);
    int max_ctas = occ * n_sms;
    if (p.max_sms > 0 && p.max_sms < n_sms) max_ctas = occ * p.max_sms;
    const int per_cta = (U + max_ctas - 1) / max_ctas;
    const int grid = (U + per_cta - 1) / per_cta;
    return launch_pdl(decode_kernel<D, NT, W, SPL>, dim3(grid), dim3(W * 32), L.total, s, p);
}

template <int D, bool SPL>
cudaError_t launch_decode_m(const DecodeParams &p, int nt, cudaStream_t s) {
    if (p.tile_mode) return launch_decode_t<D, 1, 8, SPL>(p, s);
    switch (nt) {
        case 1: return launch_decode_t<D, 1, 8, SPL>(p, s);
        case 2: return launch_decode_t<D, 2, 8, SPL>(p, s);
        case 3: return launch_decode_t<D, 3, 8, SPL>(p, s);
        case 4: return launch_decode_t<D, 4, 8, SPL>(p, s);
        case 5: return launch_decode_t<D, 5, 8, SPL>(p, s);
        case 6: return launch_decode_t<D, 6, 8, SPL>(p, s);
        case 8: return launch_decode_t<D, 8, 8, SPL>(p, s);
        default: return cudaErrorInvalidValue;
    }
}
template <int D>
cudaError_t launch_decode_d(const DecodeParams &p, int nt, cudaStream_t s) {
    return p.single_f16 ? launch_decode_m<D, false>(p, nt, s) : launch_decode_m<D, true>(p, nt, s);
}

// ------------------------------------------------------------------ combine

// One CTA per (row, q head, 64-dim slice), in one pass over the splits.
// Warp w takes splits w, w + NW, w + 2 NW, ... in that order, with
// kCombineUnroll splits' (m, l) pairs and partial rows in flight, and keeps
// a running max m_w: when a split's max exceeds it, the warp's sums are
// rescaled by 2^(m_w - m) before the split is added with weight 2^(m_s - m_w).
// The warps' (m_w, l_w, o_w) are then merged in warp order.  A fixed order:
// the result does not depend on timing.
constexpr int kCombineDims = 64;
constexpr int kCombineThreads = 512;
constexpr int kCombineUnroll = 8;

template <int D>
__global__ void __launch_bounds__(kCombineThreads, 3) combine_kernel(const CombineParams p) {
    constexpr int DS = D < kCombineDims ? D : kCombineDims;
    constexpr int VPL = DS / 32;  // dims per lane (2)
    constexpr int NW = kCombineThreads / 32;
    __shared__ float wm[NW], wl[NW];
    __shared__ float wo[NW][DS];
    // launched as a programmatic dependent of the layer's last read: nothing is
    // read before that grid (and every earlier dependency) has completed
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");  // the next call's Q prep may be scheduled
    tl_begin(p.tl);
    const int rh = blockIdx.x, r = rh / p.Hq, h = rh - r * p.Hq;
    const int d0 = blockIdx.y * DS;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (p.status && *reinterpret_cast<const volatile int *>(p.status) != 0) {
        // a bounded wait in an attention kernel gave up, so some partials were
        // never written: make the whole output visibly invalid
        if (warp == 0) {
            float *dst = p.out + ((int64_t)r * p.Hq + h) * D + d0 + lane * VPL;
#pragma unroll
            for (int i = 0; i < VPL; ++i) dst[i] = __int_as_float(0x7fc00000);
            if (p.lse && lane == 0 && blockIdx.y == 0) p.lse[(int64_t)r * p.Hq + h] = __int_as_float(0x7fc00000);
        }
        tl_finish(p.tl);
        return;
    }
    const int nsplit = (int)((p.pos0 + r) / ((long long)p.P * p.split_pages)) + 1;
    auto base_of = [&](int s) { return ((int64_t)s * p.Hq + h) * p.R + r; };

    float mw = -INFINITY, Lw = 0.f, o[VPL];
#pragma unroll
    for (int i = 0; i < VPL; ++i) o[i] = 0.f;
    for (int j0 = warp; j0 < nsplit; j0 += NW * kCombineUnroll) {
        // lane u < kCombineUnroll holds the (m, l) pair of split j0 + u NW
        float2 mlu = make_float2(0.f, 0.f);
        if (lane < kCombineUnroll && j0 + lane * NW < nsplit)
            mlu = *reinterpret_cast<const float2 *>(p.part_ml + base_of(j0 + lane * NW) * 2);
        float v[kCombineUnroll][VPL];
#pragma unroll
        for (int u = 0; u < kCombineUnroll; ++u) {
            const int j = j0 + u * NW;
            v[u][0] = v[u][1] = 0.f;
            if (j < nsplit) {
                const float2 t = *reinterpret_cast<const float2 *>(p.part_o + base_of(j) * D + d0 + lane * VPL);
                v[u][0] = t.x;
                v[u][1] = t.y;
            }
        }
#pragma unroll
        for (int u = 0; u < kCombineUnroll; ++u) {
            const float m = __shfl_sync(0xffffffffu, mlu.x, u), l = __shfl_sync(0xffffffffu, mlu.y, u);
            if (!(l > 0.f)) continue;  // past the end, or a split with no visible key
            if (m > mw) {
                const float c = exp2f(mw - m);  // 0 while nothing has been added
                Lw *= c;
                o[0] *= c;
                o[1] *= c;
                mw = m;
            }
            const float w = exp2f(m - mw);
            o[0] = fmaf(w, v[u][0], o[0]);
            o[1] = fmaf(w, v[u][1], o[1]);
            Lw = fmaf(w, l, Lw);
        }
    }
    if (lane == 0) {
        wm[warp] = mw;
        wl[warp] = Lw;
    }
#pragma unroll
    for (int i = 0; i < VPL; ++i) wo[warp][lane * VPL + i] = o[i];
    __syncthreads();
    if (warp == 0) {
        float M = -INFINITY;
        for (int w = 0; w < NW; ++w) M = fmaxf(M, wm[w]);
        float Lt = 0.f, ot[VPL];
#pragma unroll
        for (int i = 0; i < VPL; ++i) ot[i] = 0.f;
        if (M != -INFINITY) {
            for (int w = 0; w < NW; ++w) {
                if (wm[w] == -INFINITY) continue;
                const float c = exp2f(wm[w] - M);
                Lt = fmaf(c, wl[w], Lt);
#pragma unroll
                for (int i = 0; i < VPL; ++i) ot[i] = fmaf(c, wo[w][lane * VPL + i], ot[i]);
            }
        }
        float *dst = p.out + ((int64_t)r * p.Hq + h) * D + d0 + lane * VPL;
        const float inv = (Lt > 0.f) ? 1.f / Lt : 0.f;
#pragma unroll
        for (int i = 0; i < VPL; ++i) dst[i] = ot[i] * inv;
        if (p.lse && lane == 0 && blockIdx.y == 0)
            p.lse[(int64_t)r * p.Hq + h] = (Lt > 0.f) ? (M + log2f(Lt)) * 0.69314718055994531f : -INFINITY;
        tl_finish(p.tl);
    }
}

// Combine for calls with many (row, head) pairs and few splits (the prefill
// chunk: 6144 pairs over about 22 splits): one warp per (row, q head), each
// lane holding D / 32 dims, merging the splits in split order with a running
// max (a split whose max exceeds it rescales the sums by 2^(m_w - m) first).
// The split-strided form above would give each pair 4 CTAs of 512 threads
// with one or two splits per warp; here a pair is 32 threads.  A fixed order:
// the result depends on the call's shape only.
constexpr int kRowsCombineThreads = 256;
constexpr int kRowsCombineUnroll = 4;

template <int D>
__global__ void __launch_bounds__(kRowsCombineThreads) combine_rows_kernel(const CombineParams p) {
    constexpr int VPL = D / 32;
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    tl_begin(p.tl);
    const int lane = threadIdx.x & 31;
    const int rh = blockIdx.x * (kRowsCombineThreads / 32) + (threadIdx.x >> 5);
    if (rh < p.R * p.Hq) {
        const int r = rh / p.Hq, h = rh - r * p.Hq;
        float *dst = p.out + (int64_t)rh * D + lane * VPL;
        if (p.status && *reinterpret_cast<const volatile int *>(p.status) != 0) {
            // a bounded wait in an attention kernel gave up: the output is invalid
#pragma unroll
            for (int i = 0; i < VPL; ++i) dst[i] = __int_as_float(0x7fc00000);
            if (p.lse && lane == 0) p.lse[rh] = __int_as_float(0x7fc00000);
        } else {
            const int nsplit = (int)((p.pos0 + r) / ((long long)p.P * p.split_pages)) + 1;
            auto base_of = [&](int s) { return ((int64_t)s * p.Hq + h) * p.R + r; };
            float mw = -INFINITY, Lw = 0.f, o[VPL];
#pragma unroll
            for (int i = 0; i < VPL; ++i) o[i] = 0.f;
            for (int j0 = 0; j0 < nsplit; j0 += kRowsCombineUnroll) {
                float2 ml[kRowsCombineUnroll];
                float v[kRowsCombineUnroll][VPL];
#pragma unroll
                for (int u = 0; u < kRowsCombineUnroll; ++u) {
                    ml[u] = make_float2(0.f, 0.f);
#pragma unroll
                    for (int i = 0; i < VPL; ++i) v[u][i] = 0.f;
                    if (j0 + u < nsplit) {
                        const int64_t b = base_of(j0 + u);
                        ml[u] = *reinterpret_cast<const float2 *>(p.part_ml + b * 2);
                        const float *src = p.part_o + b * D + lane * VPL;
                        if (VPL % 4 == 0) {
#pragma unroll
                            for (int i = 0; i < VPL; i += 4) {
                                const float4 t = *reinterpret_cast<const float4 *>(src + i);
                                v[u][i] = t.x;
                                v[u][i + 1] = t.y;
                                v[u][i + 2] = t.z;
                                v[u][i + 3] = t.w;
                            }
                        } else {
#pragma unroll
                            for (int i = 0; i < VPL; i += 2) {
                                const float2 t = *reinterpret_cast<const float2 *>(src + i);
                                v[u][i] = t.x;
                                v[u][i + 1] = t.y;
                            }
                        }
                    }
                }
#pragma unroll
                for (int u = 0; u < kRowsCombineUnroll; ++u) {
                    const float m = ml[u].x, l = ml[u].y;
                    if (!(l > 0.f)) continue;  // past the end, or a split with no visible key
                    if (m > mw) {
                        const float c = exp2f(mw - m);  // 0 while nothing has been added
                        Lw *= c;
#pragma unroll
                        for (int i = 0; i < VPL; ++i) o[i] *= c;
                        mw = m;
                    }
                    const float w = exp2f(m - mw);
#pragma unroll
                    for (int i = 0; i < VPL; ++i) o[i] = fmaf(w, v[u][i], o[i]);
                    Lw = fmaf(w, l, Lw);
                }
            }
            const float inv = (Lw > 0.f) ? 1.f / Lw : 0.f;
            if (VPL % 4 == 0) {
#pragma unroll
                for (int i = 0; i < VPL; i += 4)
                    *reinterpret_cast<float4 *>(dst + i) = make_float4(o[i] * inv, o[i + 1] * inv, o[i + 2] * inv, o[i + 3] * inv);
            } else {
#pragma unroll
                for (int i = 0; i < VPL; ++i) dst[i] = o[i] * inv;
            }
            if (p.lse && lane == 0) p.lse[rh] = (Lw > 0.f) ? (mw + log2f(Lw)) * 0.69314718055994531f : -INFINITY;
        }
    }
    if (p.tl) {
        __syncthreads();
        tl_finish(p.tl);
    }
}

}  // namespace

int decode_max_mma_rows() { return 64; }

cudaError_t launch_decode(const DecodeParams &p, cudaStream_t s) {
    const int rows = p.G * p.Rg;
    if (rows < 1 || rows > 64 || p.row0 < 0 || p.row0 + p.Rg > p.R || (p.n_items < 1 && !p.prep_q) || p.n_items > kMaxItems) return cudaErrorInvalidValue;
    if (p.tile_mode && p.prep_q) return cudaErrorInvalidValue;
    const int nt = (rows + 7) / 8;
    DecodeParams q = p;
    q.qtiles = nt == 7 ? 8 : nt;  // row tiles of the fragment layout (the variant's)
    q.run_tiles = nt;
    switch (p.geom.D) {
        case 64: return launch_decode_d<64>(q, q.qtiles, s);
        case 128: return launch_decode_d<128>(q, q.qtiles, s);
        case 256: return launch_decode_d<256>(q, q.qtiles, s);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_combine(const CombineParams &p, cudaStream_t s) {
    const int blocks = p.R * p.Hq;
    if (blocks < 1) return cudaSuccess;
    // many (row, head) pairs over few splits: a warp per pair (chosen from the
    // call's shape alone, so any residency gives the same arithmetic)
    const long long max_split = (p.pos0 + p.R - 1) / ((long long)p.P * p.split_pages) + 1;
    if (blocks >= 512 && max_split <= 64) {
        const dim3 rgrid((blocks + kRowsCombineThreads / 32 - 1) / (kRowsCombineThreads / 32));
        switch (p.D) {
            case 64: return launch_pdl(combine_rows_kernel<64>, rgrid, dim3(kRowsCombineThreads), 0, s, p);
            case 128: return launch_pdl(combine_rows_kernel<128>, rgrid, dim3(kRowsCombineThreads), 0, s, p);
            case 256: return launch_pdl(combine_rows_kernel<256>, rgrid, dim3(kRowsCombineThreads), 0, s, p);
            default: return cudaErrorInvalidValue;
        }
    }
    const dim3 grid(blocks, p.D > kCombineDims ? p.D / kCombineDims : 1);
    switch (p.D) {
        case 64: return launch_pdl(combine_kernel<64>, grid, dim3(kCombineThreads), 0, s, p);
        case 128: return launch_pdl(combine_kernel<128>, grid, dim3(kCombineThreads), 0, s, p);
        case 256: return launch_pdl(combine_kernel<256>, grid, dim3(kCombineThreads), 0, s, p);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace kvs
