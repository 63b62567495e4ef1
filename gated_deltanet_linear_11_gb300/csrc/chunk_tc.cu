// chunk_tc.cu -- tensor-core chunked gated delta rule for dk = dv = 128, chunk 64, bf16.
//
// Recurrence: "Qwen3.5-27B GPTQ Garbage Inference -- Root Cause Analysis", "Why
// abliteration failed on Qwen3.5", item 3.  Chunk boundaries anchored at every sequence
// start ("[Feature] Add batch invariance support to GDN_ATTN backend - #45819", Birol's
// comment, part 3(a), and the PR's "Fixes: 2."), so nothing depends on the packed batch.
//
// Two kernels, both tcgen05 (MMA into TMEM, operands in 128B-swizzled shared memory fed
// by TMA):
//
//  chunk_prep (one CTA per (chunk, v-head), fully parallel):
//      P = [K;Q] K^T                                   (tcgen05, M=128 N=64 K=128)
//    with gamma the in-chunk inclusive log-decay sums and nk, nq the L2-norm factors
//    (1 when the flag is off):
//      A[r][s]  = beta_r e^{gamma_r-gamma_s} nk_r nk_s (k_r.k_s)          s < r
//      M[r][s]  = e^{gamma_r-gamma_s} nq_r nk_s (q_r.k_s)                  s <= r
//      Tinv     = (I + A)^{-1}   (fp32, blocked forward substitution on CUDA cores)
//      Lo       = Tinv - I,  Mt = M Tinv = M + M Lo   (tcgen05: M Lo accumulates onto
//                                                      the fp32 M held in TMEM)
//    and stores one workspace tile: the 128x64 bf16 X = [Lo ; Mt] (already swizzled)
//    followed by the chunk's fp32 gamma, beta, nk and nq.
//
//  chunk_state (one CTA per (sequence, v-head, dv tile), walks the chunks):
//      D1 = [K;Q] h                      (h: fp32 state in registers, bf16 copy as operand)
//      R  = diag(beta) (V - diag(e^gamma nk) K h)              (fp32, CUDA cores)
//      D2 = X R  = [Lo R ; Mt R]
//      Vn = R + Lo R                     (identity part of Tinv applied exactly in fp32)
//      O  = scale (diag(e^gamma nq) Q h + Mt R)
//      h <- e^{gamma_L} h + K^T diag(e^{gamma_L-gamma} nk) Vn
//    The last product takes diag(.)Vn as a bf16 hi + lo pair (one MMA pass over [hi | lo],
//    the halves summed in fp32) so the state keeps fp32-level accuracy; q/k L2 norms and
//    decays are per-token fp32 scalars applied outside the MMAs, so the raw bf16 inputs
//    are the only operands that are not split.
//    One CTA per (sequence, v-head, dv tile of 64, 48 or 32 columns).  Eight compute
//    warps: warps w and w+4 share TMEM lanes 32(w%4).. and take half the tile's columns
//    each; a ninth warp issues the MMAs (as a converged warp, one elected lane issuing) and
//    a tenth the TMA and bulk loads.
//    chunk_state_vconv_kernel is the same pass for the layer entry's opt-in fusion: it
//    reads the raw activations of V and applies the width-4 conv + SiLU itself.
//
// Every wait on an mbarrier is bounded in time; on expiry the CTA records GDN_ERR_TIMEOUT
// in the status word, stops issuing work, frees its TMEM and returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cstring>

#include "common.cuh"
#include "conv_taps.cuh"
#include "tc_ptx.cuh"
#include "tmap.cuh"

namespace gdn {

constexpr int kPrepThreads = 128;
constexpr int kC = 64;          // chunk
constexpr int kD = 128;         // dk = dv
constexpr uint32_t kXTile = 16384;            // bf16 [128 rows][64] swizzled
constexpr uint32_t kScal = 4 * kC * 4;        // gamma, beta, nk, nq (fp32 x 64 each)
constexpr uint32_t kWsTile = kXTile + kScal;  // one workspace tile per (slot, v-head)
constexpr uint64_t kWaitNs = 2000000000ull;   // 2 s bound on any single wait

struct TcMaps {
    CUtensorMap q, k, v, o;
    CUtensorMap o48, o32;   // O as 48- and 32-column plain (unswizzled) boxes
};

constexpr int kStateOrderMax = 256;

struct TcParams {
    const float *g, *beta;
    const int32_t *cu;
    const float *h0;
    float *hT;
    bf16 *o;
    int64_t o_tok;
    uint8_t *ws;
    int N, Hk, Hv;
    float scale;
    int l2norm;
    int ntiles;              // dv tiles per head in the state kernel: 2 or 3
    int32_t *status;
    // Context-parallel passes over a batch split into chunk-aligned ranges (cp = 0: the
    // plain scan, cu and h0/hT indexed by sequence).  cu then holds the ranges' bounds.
    //   cp = 1: grid z = 2 n_ranges.  z < n_ranges: range z from its first state (the
    //           sequence's initial state for a sequence's first range, else zero), end
    //           state to sA (to hT when the range is the whole sequence), O only for first
    //           ranges; the last of several ranges is skipped (no composition reads its
    //           end state).  z >= n_ranges: the transition map of range z - n_ranges (V
    //           taken as zero, start = I), to sP; first and last ranges need none.
    //   cp = 2: grid z = n_ranges.  Every range but a first from its start state in sS,
    //           O stored, a last range's end state to hT.
    int cp;
    int n_ranges;
    const int32_t *rtab;     // per range: its sequence | first << 30 | last << 29
    float *sA, *sP;
    const float *sS;
    // The layer's v-channel conv fused into the state pass (vconv = 1, plain scan only):
    // maps.v then views the raw activations, and each state CTA convolves its own V
    // columns (width 4, SiLU) one chunk ahead, writes them to y and, at the end, the
    // sequence's new conv state for those channels.
    int vconv;
    const bf16 *xr;          // raw activations [T][xc]
    bf16 *y;                 // conv output [T][xc]
    const bf16 *cw, *cb;     // taps [xc][4]; bias [xc] or null
    const bf16 *cs_in;       // conv states [N][3][xc], or null for zeros
    bf16 *cs_out;            // new conv states [N][3][xc], or null
    int64_t xc;              // channels per row
    int cv0;                 // first v channel
    // Plain scan: state CTAs take their sequences in this order (grid z -> sequence), the
    // longest first, so that the longest chains start in the first wave rather than in the
    // tail; n_order = 0 (more than kStateOrderMax sequences): grid z is the sequence.
    int n_order;
    uint16_t order[kStateOrderMax];
};

constexpr int32_t kRangeFirst = 1 << 30, kRangeLast = 1 << 29, kRangeSeq = (1 << 29) - 1;

__device__ __forceinline__ uint64_t now_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}

// Bounded wait on an mbarrier phase by every thread, then a CTA-wide agreement.
__device__ __forceinline__ bool wait_all(uint64_t *bar, uint32_t parity) {
    bool ok = tc::mbar_try_wait(bar, parity);
    if (!ok) {
        const uint64_t t0 = now_ns();
        while (!(ok = tc::mbar_try_wait(bar, parity)))
            if (now_ns() - t0 > kWaitNs) break;
    }
    return __syncthreads_and(ok ? 1 : 0) != 0;
}

// First chunk slot of sequence n: floor(cu[n] / 64) + n.  Distinct chunks of a packed
// batch get distinct slots below ceil(T / 64) + N.
__device__ __forceinline__ int slot0(const int32_t *cu, int n) { return cu[n] / kC + n; }

// Pack N consecutive floats to bf16 into 16-byte chunks c0.. of a swizzled tile row.
template <int N>
__device__ __forceinline__ void pack_row(uint8_t *tile, int row, int c0, const float (&v)[N]) {
#pragma unroll
    for (int c = 0; c < N / 8; ++c) {
        float f[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) f[e] = v[8 * c + e];
        *reinterpret_cast<uint4 *>(tile + tc::swz(row, c0 + c)) = pack8(f);
    }
}

__device__ __forceinline__ void tmem_row64(uint32_t taddr, float (&v)[64]) {
    float a[32], b[32];
    tc::tmem_ld32(taddr, a);
    tc::tmem_ld32(taddr + 32, b);
    tc::tmem_wait_ld();
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        v[i] = a[i];
        v[32 + i] = b[i];
    }
}

__device__ __forceinline__ void tmem_row32(uint32_t taddr, float (&v)[32]) {
    tc::tmem_ld32(taddr, v);
    tc::tmem_wait_ld();
}

// Packed fp32 pair arithmetic (two lanes per instruction), rounded like the scalar ops.
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
    float2 d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;"
        : "=l"(*reinterpret_cast<unsigned long long *>(&d))
        : "l"(*reinterpret_cast<const unsigned long long *>(&a)),
          "l"(*reinterpret_cast<const unsigned long long *>(&b)),
          "l"(*reinterpret_cast<const unsigned long long *>(&c)));
    return d;
}
__device__ __forceinline__ float2 add2(float2 a, float2 b) {
    float2 d;
    asm("add.rn.f32x2 %0, %1, %2;"
        : "=l"(*reinterpret_cast<unsigned long long *>(&d))
        : "l"(*reinterpret_cast<const unsigned long long *>(&a)),
          "l"(*reinterpret_cast<const unsigned long long *>(&b)));
    return d;
}
__device__ __forceinline__ float2 mul2(float2 a, float2 b) {
    float2 d;
    asm("mul.rn.f32x2 %0, %1, %2;"
        : "=l"(*reinterpret_cast<unsigned long long *>(&d))
        : "l"(*reinterpret_cast<const unsigned long long *>(&a)),
          "l"(*reinterpret_cast<const unsigned long long *>(&b)));
    return d;
}

// Sum of squares of one 128-element bf16 row held in a K-major tile of two 64-wide
// blocks (block stride `blk` bytes), fixed order.
__device__ __forceinline__ float row_sumsq(const uint8_t *tile, int row, uint32_t blk) {
    float acc = 0.f;
#pragma unroll
    for (int kb = 0; kb < 2; ++kb) {
#pragma unroll 2
        for (int c = 0; c < 8; ++c) {
            float f[8];
            unpack8(*reinterpret_cast<const uint4 *>(tile + kb * blk + tc::swz(row, c)), f);
#pragma unroll
            for (int e = 0; e < 8; ++e) acc = fmaf(f[e], f[e], acc);
        }
    }
    return acc;
}

constexpr float kLog2e = 1.4426950408889634f;

// 2^x by the hardware approximation (relative error about 2^-22; 0 for x = -inf).
__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// ------------------------------------------------------------------ Tinv (fp32)
// T = (I + A)^{-1} for a 64x64 strictly lower A, computed in place (T replaces A) by 16x16
// blocks.  With T_ii the inverses of the diagonal blocks (I + A_ii) and, for the two
// 32x32 halves, T0 = [[T00,0],[T10,T11]], T1 = [[T22,0],[T32,T33]]:
//     T10 = -T11 A10 T00,   T32 = -T33 A32 T22,
//     [T20 T21; T30 T31] = -T1 [A20 A21; A30 A31] T0.
// Each block of A is read for the last time before the block of T at the same place is
// written, with a barrier in between.  Every product is a 16x16 block computed by one
// warp whose lanes hold 2x4 register tiles (two A values and four B values per step feed
// eight FMAs).  All 128 threads call this; Y ([64][kLdY]) is a scratch for the 16- and
// 32-column intermediates.
constexpr int kLd = 66;
constexpr int kLdY = 34;

// acc += A[ar.., ac..] (16x16) * B[br.., bc..] (16x16) for this lane's 2x4 tile: rows
// 2 tr, 2 tr + 1 and columns 4 tc .. 4 tc + 3 of the block, k in increasing order.
// Partly unrolled: the prep kernel's code size shows up as instruction-fetch stalls.
template <int LA, int LB>
__device__ __forceinline__ void blk_mma(float (&acc)[2][4], const float (*A)[LA], int ar, int ac,
                                          const float (*B)[LB], int br, int bc, int tr, int tc) {
#pragma unroll 4
    for (int m = 0; m < 16; ++m) {
        const float a0 = A[ar + 2 * tr][ac + m], a1 = A[ar + 2 * tr + 1][ac + m];
        const float2 b01 = *reinterpret_cast<const float2 *>(&B[br + m][bc + 4 * tc]);
        const float2 b23 = *reinterpret_cast<const float2 *>(&B[br + m][bc + 4 * tc + 2]);
        acc[0][0] = fmaf(a0, b01.x, acc[0][0]); acc[0][1] = fmaf(a0, b01.y, acc[0][1]);
        acc[0][2] = fmaf(a0, b23.x, acc[0][2]); acc[0][3] = fmaf(a0, b23.y, acc[0][3]);
        acc[1][0] = fmaf(a1, b01.x, acc[1][0]); acc[1][1] = fmaf(a1, b01.y, acc[1][1]);
        acc[1][2] = fmaf(a1, b23.x, acc[1][2]); acc[1][3] = fmaf(a1, b23.y, acc[1][3]);
    }
}
template <int LD>
__device__ __forceinline__ void blk_store(float (*D)[LD], int dr, int dc, int tr, int tc,
                                            const float (&acc)[2][4], float sgn) {
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        *reinterpret_cast<float2 *>(&D[dr + 2 * tr + i][dc + 4 * tc]) = make_float2(sgn * acc[i][0], sgn * acc[i][1]);
        *reinterpret_cast<float2 *>(&D[dr + 2 * tr + i][dc + 4 * tc + 2]) = make_float2(sgn * acc[i][2], sgn * acc[i][3]);
    }
}

__device__ void tinv64_inplace(float (*AT)[kLd], float (*Y)[kLdY]) {
    const int tid = threadIdx.x;
    // lane = 8 tc + tr: a half-warp's float2 stores of a block hit 2-way bank conflicts at
    // most (4-way with lane = 4 tr + tc); the loads stay conflict-free either way
    const int w = tid >> 5, lane = tid & 31, tr = lane & 7, tc = lane >> 3;
    {   // diagonal blocks by forward substitution, one column per thread
        const int b = (tid >> 4) & 3, j = tid & 15, o = 16 * b;
        float x[16];
        if (tid < 64) {
#pragma unroll
            for (int r = 0; r < 16; ++r) x[r] = (r == j) ? 1.f : 0.f;
#pragma unroll
            for (int r = 1; r < 16; ++r) {
                float acc = x[r];
#pragma unroll
                for (int q = 0; q < r; ++q) acc = fmaf(-AT[o + r][o + q], x[q], acc);
                x[r] = acc;
            }
        }
        __syncthreads();
        if (tid < 64) {
#pragma unroll
            for (int r = 0; r < 16; ++r) AT[o + r][o + j] = x[r];
        }
    }
    __syncthreads();
    if (w < 2) {   // X = A10 T00 (warp 0) and A32 T22 (warp 1), into Y rows 32.. and 48..
        float acc[2][4] = {};
        const int o = 32 * w;
        blk_mma(acc, AT, o + 16, o, AT, o, o, tr, tc);
        blk_store(Y, 32 + 16 * w, 0, tr, tc, acc, 1.f);
    }
    __syncthreads();
    if (w < 2) {   // T10 = -T11 X over A10,  T32 = -T33 X over A32
        float acc[2][4] = {};
        const int o = 32 * w;
        blk_mma(acc, AT, o + 16, o + 16, Y, 32 + 16 * w, 0, tr, tc);
        blk_store(AT, o + 16, o, tr, tc, acc, -1.f);
    }
    __syncthreads();
    {   // Z = [A20 A21; A30 A31] T0 into Y[0:32][0:32]; warp w: block row w >> 1, column w & 1
        const int half = w >> 1, which = w & 1, ar = 32 + 16 * half;
        float acc[2][4] = {};
        if (which == 0) {
            blk_mma(acc, AT, ar, 0, AT, 0, 0, tr, tc);     // A_r0 T00
            blk_mma(acc, AT, ar, 16, AT, 16, 0, tr, tc);   // + A_r1 T10
        } else {
            blk_mma(acc, AT, ar, 16, AT, 16, 16, tr, tc);  // A_r1 T11
        }
        blk_store(Y, 16 * half, 16 * which, tr, tc, acc, 1.f);
    }
    __syncthreads();
    {   // [T20 T21; T30 T31] = -T1 Z; warp w: block row 2 + (w >> 1), column w & 1
        const int half = w >> 1, which = w & 1;
        float acc[2][4] = {};
        if (half == 0) {
            blk_mma(acc, AT, 32, 32, Y, 0, 16 * which, tr, tc);    // T22 Z2x
        } else {
            blk_mma(acc, AT, 48, 32, Y, 0, 16 * which, tr, tc);    // T32 Z2x
            blk_mma(acc, AT, 48, 48, Y, 16, 16 * which, tr, tc);   // + T33 Z3x
        }
        // the stores go to columns 0..31, which no thread reads in this step
        blk_store(AT, 32 + 16 * half, 16 * which, tr, tc, acc, -1.f);
    }
    __syncthreads();
}

// ================================================================ chunk_prep kernel

// One region, reused by lifetime.  The [K;Q] K-major tile fills bytes 0..32767 until
// P = [K;Q]K^T and the norms are taken.  Then the fp32 A, inverted in place into
// T = (I + A)^{-1}, sits at byte 0, and the inverse's scratch Y at kXOff; once the
// inverse is done, the bf16 tile X = [Lo ; M] (then [Lo ; Mt]) replaces Y at kXOff.
constexpr uint32_t kXOff = 17 * 1024;   // 1024-aligned, past A
static_assert(64 * kLd * 4 <= kXOff && 64 * kLdY * 4 <= kXTile, "prep region layout");

struct PrepSmem {
    uint8_t buf[kXOff + kXTile];
    float gam[64], bet[64], nk[64], nq[64];
    float c2[64];            // gamma_s log2(e) - log2(nk_s): the key-side exponent
    float carry;
    uint64_t bar_tma, bar_mma;
    uint32_t tmem;

    __device__ uint8_t *kq() { return buf; }
    __device__ float (*AT())[kLd] { return reinterpret_cast<float (*)[kLd]>(buf); }
    __device__ float (*Y())[kLdY] { return reinterpret_cast<float (*)[kLdY]>(buf + kXOff); }
    __device__ uint8_t *x() { return buf + kXOff; }
};
static_assert(sizeof(PrepSmem) + 1024 <= 44 * 1024, "five prep CTAs fit on one SM");

// One CTA per (chunk slot, v-head); five CTAs per SM.  TMEM (64 columns): P = [K;Q]K^T,
// whose M rows are then replaced by the fp32 M itself, onto which M Lo accumulates.
__global__ void __launch_bounds__(kPrepThreads, 5)
chunk_prep_kernel(const __grid_constant__ TcMaps maps, const __grid_constant__ TcParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    PrepSmem &S = *reinterpret_cast<PrepSmem *>(
        (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023));
    grid_dependents_launch();
    grid_dependency_wait();
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int slot = blockIdx.x, hv = blockIdx.y;
    const int hk = hv / (p.Hv / p.Hk);

    // slot -> (sequence n, chunk c): the last n with slot0(n) <= slot.
    int lo = 0, hi = p.N - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (slot0(p.cu, mid) <= slot) lo = mid; else hi = mid - 1;
    }
    const int n = lo;
    const int c = slot - slot0(p.cu, n);
    const int start = p.cu[n], len = p.cu[n + 1] - start;
    if (c < 0 || c * kC >= len) return;
    const int t0 = start + c * kC;
    const int L = min(kC, len - c * kC);

    // this chunk's gates (latency hidden behind the TMA and the first MMA)
    float gx = 0.f, bx = 0.f;
    if (tid < L) {
        gx = p.g[(size_t)(t0 + tid) * p.Hv + hv];
        bx = p.beta[(size_t)(t0 + tid) * p.Hv + hv];
    }

    if (warp == 0) {
        tc::tmem_alloc(&S.tmem, 64);
        tc::tmem_relinquish();
    }
    if (tid == 0) {
        tc::mbar_init(&S.bar_tma, 1);
        tc::mbar_init(&S.bar_mma, 1);
        tc::mbar_fence_init();
        tc::prefetch_tmap(&maps.k);
        tc::prefetch_tmap(&maps.q);
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = S.tmem;
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    const uint32_t colP = 0;
    bool ok = true;

    if (tid == 0) {
        tc::mbar_expect_tx(&S.bar_tma, 32768);
        tc::tma_load_3d(S.kq() + 0, &maps.k, &S.bar_tma, 0, hk, t0);
        tc::tma_load_3d(S.kq() + 16384, &maps.k, &S.bar_tma, 64, hk, t0);
        tc::tma_load_3d(S.kq() + 8192, &maps.q, &S.bar_tma, 0, hk, t0);
        tc::tma_load_3d(S.kq() + 16384 + 8192, &maps.q, &S.bar_tma, 64, hk, t0);
    }
    // inclusive scan of g by warps 0 and 1 (fixed order), while the loads fly
    float gs = gx;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, gs, off);
        if (lane >= off) gs += y;
    }
    if (tid == 31) S.carry = gs;
    ok = wait_all(&S.bar_tma, 0);
    if (ok && warp == 0) {
        tc::fence_after_sync();
        constexpr uint32_t id = tc::idesc_bf16(128, 64, 0, 0);
        const uint32_t base = tc::smem_u32(S.kq());
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
            const uint32_t off = (ks >> 2) * 16384 + (ks & 3) * 32;
            tc::mma_bf16_warp(tmem + colP, tc::sdesc(base + off, 16, 1024),
                              tc::sdesc(base + off, 16, 1024), id, ks > 0);
        }
        tc::mma_commit_warp(&S.bar_mma);
    }
    const int r = tid & 63;
    if (ok) {
        // L2-norm factors of this chunk's k rows (threads 0..63) and q rows (64..127)
        const float ss = row_sumsq(S.kq(), tid, 16384);
        const float f = p.l2norm ? rsqrtf(ss + 1e-6f) : 1.f;
        if (tid < 64) {
            const float nkr = r < L ? f : 0.f;
            const float gamr = tid >= 32 ? gs + S.carry : gs;
            S.nk[r] = nkr;
            S.gam[r] = gamr;
            S.bet[r] = bx;
            // e^{gamma_r - gamma_s} nk_s = 2^(gamma_r log2 e - c2_s); nk_s = 0 gives +inf here
            // and an exact 0 below
            S.c2[r] = nkr > 0.f ? gamr * kLog2e - __log2f(nkr) : __int_as_float(0x7f800000);
        } else {
            S.nq[r] = r < L ? f : 0.f;
        }
    }
    // (this wait also orders the norm reads of kq before the region is reused)
    if (ok) ok = wait_all(&S.bar_mma, 0);
    uint8_t *wtile = p.ws + ((size_t)slot * p.Hv + hv) * kWsTile;
    // Rows 0..31 of A and M have no entries past column 31 (warp-uniform).
    const bool low = r < 32;
    float (*AT)[kLd] = S.AT();
    if (ok) {
        tc::fence_after_sync();
        // A_rs = beta_r nk_r e^{gamma_r - gamma_s} nk_s P_rs (s < r); M_rs likewise with nq_r
        // (s <= r).  Two 32-column halves keep the register footprint small.
        const float g2r = S.gam[r] * kLog2e;
        const bool arow = tid < 64;                 // warp-uniform
        const float rowf = arow ? S.bet[r] * S.nk[r] : S.nq[r];
        const int lim = arow ? r : r + 1;           // entries s < lim
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
            float v[32];
            if (hf == 1 && low) {
#pragma unroll
                for (int i = 0; i < 32; ++i) v[i] = 0.f;
            } else {
                float pv[32];
                tmem_row32(tmem + lane_off + colP + 32 * hf, pv);
#pragma unroll
                for (int i = 0; i < 32; i += 4) {
                    const int s = 32 * hf + i;
                    const float4 c4 = *reinterpret_cast<const float4 *>(&S.c2[s]);
                    const float e[4] = {fast_exp2(g2r - c4.x), fast_exp2(g2r - c4.y),
                                        fast_exp2(g2r - c4.z), fast_exp2(g2r - c4.w)};
#pragma unroll
                    for (int u = 0; u < 4; ++u)
                        v[i + u] = (s + u < lim && r < L) ? rowf * pv[i + u] * e[u] : 0.f;
                }
            }
            if (arow) {
#pragma unroll
                for (int i = 0; i < 32; i += 2)
                    *reinterpret_cast<float2 *>(&AT[r][32 * hf + i]) = make_float2(v[i], v[i + 1]);
            } else {
                // fp32 M over the P half just read: M Lo accumulates onto it, giving
                // Mt = M + M Lo (rows with no entries in this half store zeros)
                tc::tmem_st32(tmem + lane_off + colP + 32 * hf, v);
            }
        }
        if (!arow) tc::tmem_wait_st();
        // per-token scalars for the state kernel
        float *ws_s = reinterpret_cast<float *>(wtile + kXTile);
        if (tid < 64) {
            ws_s[r] = S.gam[r];
            ws_s[64 + r] = S.bet[r];
            ws_s[128 + r] = S.nk[r];
        } else {
            ws_s[192 + r] = S.nq[r];
        }
    }
    __syncthreads();
    if (ok) tinv64_inplace(AT, S.Y());   // ends with a barrier
    // X = [Lo ; M] in bf16 over the inverse's scratch
    if (ok && tid < 64) {
        // Lo = T - I: the strictly lower part of T
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
            float lrow[32];
#pragma unroll
            for (int i = 0; i < 32; i += 2) {   // two columns per load
                const float2 t2 = *reinterpret_cast<const float2 *>(&AT[r][32 * hf + i]);
                lrow[i] = (32 * hf + i < r) ? t2.x : 0.f;
                lrow[i + 1] = (32 * hf + i + 1 < r) ? t2.y : 0.f;
            }
            pack_row<32>(S.x(), tid, 4 * hf, lrow);
        }
    } else if (ok) {
        tc::fence_after_sync();
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
            float m[32];
            tmem_row32(tmem + lane_off + colP + 32 * hf, m);
            pack_row<32>(S.x(), tid, 4 * hf, m);
        }
    }
    tc::fence_async_smem();
    tc::fence_before_sync();
    __syncthreads();
    if (ok && warp == 0) {
        tc::fence_after_sync();
        // D[128x64] += X[128 x 64] * Lo[64 x 64]  (B = rows 0..63 of X, MN-major).  Rows
        // 64..127 of D held the fp32 M, so they end as Mt; rows 0..63 are not used.
        constexpr uint32_t id = tc::idesc_bf16(128, 64, 0, 1);
        const uint32_t xb = tc::smem_u32(S.x());
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
            tc::mma_bf16_warp(tmem + colP, tc::sdesc(xb + ks * 32, 16, 1024),
                              tc::sdesc(xb + ks * 2048, 8192, 1024), id, true);
        tc::mma_commit_warp(&S.bar_mma);
    }
    if (ok) ok = wait_all(&S.bar_mma, 1);
    if (ok && tid >= 64) {
        tc::fence_after_sync();
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
            float mt[32];
            tmem_row32(tmem + lane_off + colP + 32 * hf, mt);
            pack_row<32>(S.x(), tid, 4 * hf, mt);             // over M, which the MMA has read
        }
    }
    // The finished [Lo ; Mt] tile leaves in one bulk copy: 128 threads writing their own
    // 128-byte rows would cost a load/store wavefront per row per instruction.
    tc::fence_async_smem();
    __syncthreads();
    if (ok && tid == 0) {
        tc::bulk_store(wtile, S.x(), kXTile);
        tc::bulk_commit();
        tc::bulk_wait_all();
    }
    if (!ok && tid == 0) report(p.status, GDN_ERR_TIMEOUT);
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tmem, 64);
}

// =============================================================== chunk_state kernel

constexpr uint32_t kXStage = 18432;  // workspace tile rounded up to 1024 bytes

struct StateSmem {
    uint8_t kq[2][32768];    // [K;Q] per stage
    uint8_t x[2][kXStage];   // [Lo ; Mt] + scalars per stage
    uint8_t v[2][8192];      // V tile [64 tokens][64 dv] per stage
    uint8_t hb[16384];       // bf16 h  [128 dk rows][64 dv]  (MN-major B)
    uint8_t rb[8192];        // bf16 R  [64 tokens][64 dv]    (MN-major B)
    uint8_t dvh[8192];       // bf16 hi of diag(dcy) Vn
    uint8_t dvl[8192];       // bf16 lo
    uint8_t ob[2][8192];     // bf16 O tile [64 tokens][64 dv] per stage, stored by TMA
    uint64_t bar_tma[2], bar_d1, bar_d2, bar_d3, bar_fin;
    uint32_t tmem;
    int abort;               // set by the first thread whose wait runs out
    // The fused-conv kernel only (the plain kernel's allocation ends before them):
    alignas(1024) uint8_t vc[2][8192];   // the convolved V tile per stage (V's layout)
    uint8_t xv[3][8192];     // raw V tiles, a ring of three chunks
    float taps[5][64];       // the tile's taps, oldest first, and biases
    uint64_t bar_x[3];
};
// shared memory of the plain state kernel: StateSmem up to the fused-conv fields
constexpr size_t kStateSmemPlain = offsetof(StateSmem, vc);
static_assert(offsetof(StateSmem, dvl) == offsetof(StateSmem, dvh) + 8192,
              "the [hi | lo] operand is one MN-major tile with a 8192-byte block stride");
static_assert(sizeof(StateSmem) + 1024 <= 227 * 1024, "one state CTA fits on an SM");

// Bounded wait by one thread.  Gives up (false) when the phase has not completed within
// kWaitNs, or as soon as another thread of the CTA has given up; the caller then skips
// its work but keeps reaching every barrier, so the CTA still drains and exits.
__device__ __forceinline__ bool wait_one(uint64_t *bar, uint32_t parity, volatile int *abort) {
    if (tc::mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = now_ns();
    for (;;) {
        if (tc::mbar_try_wait(bar, parity)) return true;
        if (*abort) return false;
        if (now_ns() - t0 > kWaitNs) {
            *abort = 1;
            return false;
        }
    }
}

// Bounded wait that ignores the abort flag: used on the way out, for work already issued.
__device__ __forceinline__ bool wait_bounded(uint64_t *bar, uint32_t parity) {
    const uint64_t t0 = now_ns();
    while (!tc::mbar_try_wait(bar, parity))
        if (now_ns() - t0 > kWaitNs) return false;
    return true;
}

__device__ __forceinline__ void issue_chunk_loads(StateSmem &S, const TcMaps &maps,
                                                  const TcParams &p, int stage, int t0,
                                                  int hk, int hv, int j0, int slot,
                                                  bool with_v) {
    uint64_t *bar = &S.bar_tma[stage];
    tc::mbar_expect_tx(bar, 32768 + (with_v ? 8192 : 0) + kWsTile);
    uint8_t *kq = S.kq[stage];
    tc::tma_load_3d(kq + 0, &maps.k, bar, 0, hk, t0);
    tc::tma_load_3d(kq + 16384, &maps.k, bar, 64, hk, t0);
    tc::tma_load_3d(kq + 8192, &maps.q, bar, 0, hk, t0);
    tc::tma_load_3d(kq + 16384 + 8192, &maps.q, bar, 64, hk, t0);
    if (with_v) tc::tma_load_3d(S.v[stage], &maps.v, bar, j0, hv, t0);
    const uint8_t *src = p.ws + ((size_t)slot * p.Hv + hv) * kWsTile;
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 :: "r"(tc::smem_u32(S.x[stage])), "l"(src), "r"(kWsTile),
                    "r"(tc::smem_u32(bar)) : "memory");
}

// ---------------------------------------------------------------- fused v conv
// (chunk_state_vconv_kernel only.)  The width-4 causal conv + SiLU of the tile's V
// channels, with gdn_conv1d_fwd's arithmetic for every element (bias, then the taps
// oldest first, fused multiply-adds in fp32, its SiLU, round to nearest bf16), read from
// the raw activation tile that the loader put in the ring S.xv.  The eight compute warps
// convolve chunk c+1 during chunk c, in the window after the barrier that publishes h,
// while the chain waits for its first products: compute thread t takes the channel pair
// t & 31 of the tokens 8 (t >> 5) .. +7, so a warp's row accesses are one 128-byte row,
// free of bank conflicts, and the taps are five pair loads.  The three inputs before a
// chunk come from the previous chunk's raw tile (still in the ring), or for a sequence's
// first chunk from its conv state (zeros without one).
constexpr int kVcTok = 8;                       // tokens per thread

// The tile's taps and biases, fp32 pairs [tap 0..3, bias][channel pair] (threads 0..63,
// one column each).
template <int NT>
__device__ __forceinline__ void vconv_load_taps(StateSmem &S, const TcParams &p, int hv, int j0) {
    const int col = threadIdx.x;
    if (col < NT) {
        const int64_t chn = p.cv0 + (int64_t)hv * kD + j0 + col;
        const uint2 w = *reinterpret_cast<const uint2 *>(p.cw + chn * 4);
        float *tp = reinterpret_cast<float *>(S.taps);
        tp[0 * 64 + col] = __uint_as_float(w.x << 16);
        tp[1 * 64 + col] = __uint_as_float(w.x & 0xffff0000u);
        tp[2 * 64 + col] = __uint_as_float(w.y << 16);
        tp[3 * 64 + col] = __uint_as_float(w.y & 0xffff0000u);
        tp[4 * 64 + col] = p.cb ? __bfloat162float(p.cb[chn]) : 0.f;
    }
}

// Two bf16 of a tile row (channels 2 cp, 2 cp + 1) as floats.
__device__ __forceinline__ float2 tile_pair(const uint8_t *tile, int row, int cp) {
    const uint32_t u = *reinterpret_cast<const uint32_t *>(tile + tc::swz(row, cp >> 2) + 4 * (cp & 3));
    return make_float2(__uint_as_float(u << 16), __uint_as_float(u & 0xffff0000u));
}

// Tokens r0 .. r0+7 of chunk cc, channel pair cp.
__device__ __forceinline__ void vconv_rows(StateSmem &S, const TcParams &p, int n, int cp,
                                           int r0, int cc, int64_t chn, int t0, int L) {
    const uint8_t *cur = S.xv[cc % 3], *prev = S.xv[(cc + 2) % 3];
    uint8_t *out = S.vc[cc & 1];
    float2 xw[kVcTok + 3];                 // rows r0-3 .. r0+7
#pragma unroll
    for (int i = 0; i < kVcTok + 3; ++i) {
        const int rho = r0 - 3 + i;
        if (rho >= 0) {
            xw[i] = tile_pair(cur, rho, cp);
        } else if (cc > 0) {
            xw[i] = tile_pair(prev, 64 + rho, cp);
        } else if (p.cs_in) {
            const uint32_t u = *reinterpret_cast<const uint32_t *>(
                p.cs_in + ((int64_t)n * 3 + 3 + rho) * p.xc + chn);
            xw[i] = make_float2(__uint_as_float(u << 16), __uint_as_float(u & 0xffff0000u));
        } else {
            xw[i] = make_float2(0.f, 0.f);
        }
    }
    const float2 *tp = reinterpret_cast<const float2 *>(S.taps);
    const float2 w0 = tp[0 * 32 + cp], w1 = tp[1 * 32 + cp], w2 = tp[2 * 32 + cp],
                 w3 = tp[3 * 32 + cp], b = tp[4 * 32 + cp];
#pragma unroll
    for (int k = 0; k < kVcTok; ++k) {
        const int r = r0 + k;
        float2 z = fma2(w0, xw[k], b);
        z = fma2(w1, xw[k + 1], z);
        z = fma2(w2, xw[k + 2], z);
        z = fma2(w3, xw[k + 3], z);
        const __nv_bfloat162 o2 = __floats2bfloat162_rn(silu(z.x), silu(z.y));
        const uint32_t ou = *reinterpret_cast<const uint32_t *>(&o2);
        *reinterpret_cast<uint32_t *>(out + tc::swz(r, cp >> 2) + 4 * (cp & 3)) = ou;
        if (r < L) *reinterpret_cast<uint32_t *>(p.y + (int64_t)(t0 + r) * p.xc + chn) = ou;
    }
}

// Chunk cc of sequence n (tokens t0.., L of them) into S.vc[cc & 1] and y.
template <int NT>
__device__ __forceinline__ void vconv_chunk(StateSmem &S, const TcParams &p, int n, int hv,
                                            int j0, int cc, int t0, int L) {
    const int t = threadIdx.x;
    const int cp = t & 31;
    if (2 * cp >= NT) return;
    const int64_t chn = p.cv0 + (int64_t)hv * kD + j0 + 2 * cp;
    vconv_rows(S, p, n, cp, kVcTok * (t >> 5), cc, chn, t0, L);
}

// The sequence's new conv state for the tile's channels: xs = [old state (3) ; x_seq],
// rows xs[len], xs[len+1], xs[len+2].  One thread per 8 channels writes its three rows in
// order, each after the old row len + j >= j it reads, so cs_out may alias cs_in.
template <int NT>
__device__ __forceinline__ void vconv_state_out(const TcParams &p, int n, int hv, int j0,
                                                int start, int len) {
    const int grp = threadIdx.x;
    if (!p.cs_out || grp >= NT / 8) return;
    const int64_t chn = p.cv0 + (int64_t)hv * kD + j0 + 8 * grp;
#pragma unroll
    for (int j = 0; j < 3; ++j) {
        const int m = len + j;
        uint4 u = make_uint4(0u, 0u, 0u, 0u);
        if (m >= 3)
            u = *reinterpret_cast<const uint4 *>(p.xr + (int64_t)(start + m - 3) * p.xc + chn);
        else if (p.cs_in)
            u = *reinterpret_cast<const uint4 *>(p.cs_in + ((int64_t)n * 3 + m) * p.xc + chn);
        *reinterpret_cast<uint4 *>(p.cs_out + ((int64_t)n * 3 + j) * p.xc + chn) = u;
    }
}

// NC consecutive TMEM columns of this thread's lane (NC = 32, 24 or 16).
template <int NC>
__device__ __forceinline__ void tmem_cols(uint32_t taddr, float (&v)[NC]) {
    if constexpr (NC == 32) {
        tc::tmem_ld32(taddr, v);
    } else if constexpr (NC == 24) {
        tc::tmem_ld16(taddr, v);
        tc::tmem_ld8(taddr + 16, v + 16);
    } else {
        static_assert(NC == 16, "column count");
        tc::tmem_ld16(taddr, v);
    }
    tc::tmem_wait_ld();
}

// h <- a h + (K^T hi + K^T lo) for this thread's NC columns: the two halves of the state
// update sit NT = 2 NC TMEM columns apart.
template <int NC>
__device__ __forceinline__ void fold_update(float (&h)[NC], float a, uint32_t taddr) {
    float u[NC], w[NC];
    tmem_cols<NC>(taddr, u);
    tmem_cols<NC>(taddr + 2 * NC, w);
    const float2 a2 = make_float2(a, a);
#pragma unroll
    for (int i = 0; i < NC; i += 2) {
        const float2 s = add2(make_float2(u[i], u[i + 1]), make_float2(w[i], w[i + 1]));
        const float2 r = fma2(a2, make_float2(h[i], h[i + 1]), s);
        h[i] = r.x;
        h[i + 1] = r.y;
    }
}

// Named barrier between the four warps that own TMEM lanes 0..63 (warps 0, 1, 4, 5: the
// rows that feed the state chain) and the issuer warp.  The other four compute warps only
// produce outputs and never wait on it.
constexpr int kComputeThreads = 256;        // warps 0..7: two per TMEM lane quarter
constexpr int kIssuerWarp = kComputeThreads / 32;   // warp 8: MMAs
constexpr int kLoaderWarp = kIssuerWarp + 1;        // warp 9: TMA and bulk loads
constexpr int kStateThreads = kComputeThreads + 64;

__device__ __forceinline__ void chain_barrier() {
    asm volatile("bar.sync 1, %0;" :: "n"(128 + 32) : "memory");
}

// Named barrier over the four output warps (2, 3, 6, 7); thread kOutLeader issues the
// tensor stores of the O tile.
constexpr int kOutLeader = 64;
__device__ __forceinline__ void out_barrier() {
    asm volatile("bar.sync 2, 128;" ::: "memory");
}

// The per-CTA program for one dv tile of NT columns starting at column j0 (NT = 64, 48
// or 32).  Warp 8 issues every MMA and warp 9 every TMA load, so no compute warp ever stalls
// behind an issue queue; warps 0..7 hold the fp32 state rows and do the elementwise work.
// Operand tiles are 64 columns wide in shared memory whatever NT is; an NT-wide MMA reads
// only the first NT columns.  [hi | lo] is one 2 NT-wide MN-major operand whose 64-column
// blocks are S.dvh and S.dvl.
// What one state CTA computes: the chunks of entry n of p.cu (a sequence, or a range of
// one) for one v-head, from a start state, optionally without V, storing O and/or the
// end state.
struct StateJob {
    int n;
    bool active;             // false: nothing to do (no chunks, no stores)
    bool identity;           // start from I (dk = dv) instead of h0
    bool with_v;             // false: V is taken as zero and its tiles are not loaded
    bool write_o;            // store the chunk outputs
    const float *h0;         // this head's start state [dk][dv], or null for zero
    float *hT;               // this head's end state [dk][dv], or null
};

template <int NT, bool VCONV>
__device__ __forceinline__ void state_cta(StateSmem &S, const TcMaps &maps, const TcParams &p,
                                          const CUtensorMap *omap, int j0, int hv,
                                          const StateJob &job) {
    const int n = job.n;
    constexpr int NC = NT / 2;               // columns per thread
    constexpr int NCH = NC / 8;              // 16-byte chunks per thread row
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int hk = hv / (p.Hv / p.Hk);
    const int start = p.cu[n], len = job.active ? p.cu[n + 1] - start : 0;
    const int nch = (len + kC - 1) / kC;
    const int s0 = slot0(p.cu, n);
    const uint32_t tmem = S.tmem;
    // TMEM columns: D1 [K;Q]h, D2 [Lo;Mt]R, and the state update as a hi | lo pair
    const uint32_t colD1 = 0, colD2 = 64, colS = 128;
    volatile int *abort = &S.abort;

    if (warp == kIssuerWarp) {
        // ------------------------------------------------------------ issuer warp
        // Shared-memory descriptors, built once; a byte offset o is added as o >> 4.
        // Stage b of a double buffer sits b * (buffer bytes) after stage 0.
        const uint64_t dKQ0 = tc::sdesc(tc::smem_u32(S.kq[0]), 16, 1024);      // [K;Q], K-major
        const uint64_t dKQt0 = tc::sdesc(tc::smem_u32(S.kq[0]), 16384, 1024);  // K^T, MN-major
        const uint64_t dX0 = tc::sdesc(tc::smem_u32(S.x[0]), 16, 1024);        // [Lo;Mt], K-major
        const uint64_t dH = tc::sdesc(tc::smem_u32(S.hb), 8192, 1024);
        const uint64_t dR = tc::sdesc(tc::smem_u32(S.rb), 8192, 1024);
        const uint64_t dVhl = tc::sdesc(tc::smem_u32(S.dvh), 8192, 1024);
        constexpr uint32_t id1 = tc::idesc_bf16(128, NT, 0, 1);
        constexpr uint32_t id3 = tc::idesc_bf16(128, 2 * NT, 1, 1);
        const bool leader = lane == 0;
        bool ok = true;   // meaningful in lane 0
        // lane 0's wait result, broadcast: go on issuing unless a wait ran out
        auto go = [&]() { return __shfl_sync(0xffffffffu, (ok && !*abort) ? 1 : 0, 0) != 0; };
        // A chunk's tiles are waited for before the barrier that publishes its h: for
        // chunk c+1 right after chunk c's state update is issued, while the compute warps
        // fold that update, so the wait stays off the chain.
        if (leader && nch > 0) ok = wait_one(&S.bar_tma[0], 0, abort);
        for (int c = 0; c < nch; ++c) {
            const int st = c & 1;
            __syncthreads();                                   // h published as bf16
            if (go()) {
                tc::fence_after_sync();
#pragma unroll
                for (int ks = 0; ks < 8; ++ks)
                    tc::mma_bf16_warp(tmem + colD1,
                                      dKQ0 + ((st * 32768 + (ks >> 2) * 16384 + (ks & 3) * 32) >> 4),
                                      dH + ((ks * 2048) >> 4), id1, ks > 0);
                tc::mma_commit_warp(&S.bar_d1);
            }
            __syncwarp();
            chain_barrier();                                   // R ready
            if (go()) {
                tc::fence_after_sync();
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    tc::mma_bf16_warp(tmem + colD2, dX0 + ((st * kXStage + ks * 32) >> 4),
                                      dR + ((ks * 2048) >> 4), id1, ks > 0);
                tc::mma_commit_warp(&S.bar_d2);
            }
            __syncwarp();
            chain_barrier();                                   // hi | lo of d Vn ready
            if (go()) {
                // K^T [hi | lo]: both halves of the update in one pass, summed in fp32 later
                tc::fence_after_sync();
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    tc::mma_bf16_warp(tmem + colS, dKQt0 + ((st * 32768 + ks * 2048) >> 4),
                                      dVhl + ((ks * 2048) >> 4), id3, ks > 0);
                tc::mma_commit_warp(&S.bar_d3);
            }
            __syncwarp();
            if (leader && ok && c + 1 < nch)
                ok = wait_one(&S.bar_tma[st ^ 1], ((c + 1) >> 1) & 1, abort);
        }
        // Nothing this warp started may still run when the CTA exits: wait (bounded) for
        // every MMA it issued.
        tc::mma_commit_warp(&S.bar_fin);
        if (leader) wait_bounded(&S.bar_fin, 0);
        __syncwarp();
        tc::fence_before_sync();
        __syncthreads();
        return;
    }
    if (warp == kLoaderWarp) {
        // ----------------------------------------------------------- loader warp
        // Chunks 0 and 1 are loaded up front; chunk c+1 (c >= 1) goes into stage (c+1)&1
        // after the barrier that publishes chunk c's h: every warp has then finished chunk
        // c-1, the stage's previous occupant (its last MMA, the state update, completed
        // before the compute warps folded it).  Issuing them costs the MMA issuer nothing.
        const bool leader = lane == 0;
        int issued = 0;                                        // chunks 0..issued-1 are loaded
        // With the fused conv V is not part of a stage: raw V tile j goes into ring slot
        // j % 3 two chunks ahead (j + 2 after the barrier that publishes chunk j's h), so
        // chunk c+1's tile is there when the output warps convolve it during chunk c, and
        // the slot it replaces (chunk j - 1's, the halo of chunk j's conv) is done with.
        const bool stage_v = job.with_v && !VCONV;
        int x_issued = 0;                                      // raw tiles 0..x_issued-1
        auto issue_x = [&](int j) {
            uint64_t *bar = &S.bar_x[j % 3];
            tc::mbar_expect_tx(bar, 8192);
            tc::tma_load_3d(S.xv[j % 3], &maps.v, bar, j0, hv, start + j * kC);
            x_issued = j + 1;
        };
        if (leader) {
            if (VCONV)
                for (int j = 0; j < 2 && j < nch; ++j) issue_x(j);
            for (int c = 0; c < 2 && c < nch; ++c) {
                issue_chunk_loads(S, maps, p, c, start + c * kC, hk, hv, j0, s0 + c, stage_v);
                issued = c + 1;
            }
        }
        for (int c = 0; c < nch; ++c) {
            __syncwarp();
            __syncthreads();                                   // h published as bf16
            if (VCONV && leader && c + 2 < nch && !*abort) issue_x(c + 2);
            if (leader && c >= 1 && c + 1 < nch && !*abort) {
                issue_chunk_loads(S, maps, p, (c + 1) & 1, start + (c + 1) * kC, hk, hv, j0,
                                  s0 + c + 1, stage_v);
                issued = c + 2;
            }
        }
        if (leader) {
            // wait (bounded) for the last load into each stage and ring slot before the
            // CTA may exit
            for (int s = 0; s < 2; ++s) {
                const int last = issued - 1 - ((issued - 1 - s) & 1);   // last chunk into stage s
                if (last >= 0) wait_bounded(&S.bar_tma[s], (last >> 1) & 1);
            }
            for (int s = 0; s < (VCONV ? 3 : 0); ++s) {
                int last = -1;                                  // last raw tile into slot s
                for (int j = s; j < x_issued; j += 3) last = j;
                if (last >= 0) wait_bounded(&S.bar_x[s], (last / 3) & 1);
            }
        }
        __syncwarp();
        tc::fence_before_sync();
        __syncthreads();
        return;
    }

    // ---------------------------------------------------------------- compute warps
    const int quad = warp & 3;           // TMEM lane quarter
    const int half = warp >> 2;          // which NC of the NT dv columns
    const int row = quad * 32 + lane;    // TMEM lane = tile row
    const bool chain = quad < 2;         // rows 0..63: tokens of the chain / dk rows 0..63
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    const uint32_t ch = half * NC;       // this thread's column offset in the tile
    const int c0 = half * NCH;           // ... in 16-byte chunks

    // fp32 master state in registers: dk row `row`, dv columns j0+ch .. +NC-1.
    float h[NC];
    if (job.identity) {
#pragma unroll
        for (int i = 0; i < NC; ++i) h[i] = row == j0 + (int)ch + i ? 1.f : 0.f;
    } else if (job.h0) {
        const float4 *src = reinterpret_cast<const float4 *>(job.h0 + (size_t)row * kD + j0 + ch);
#pragma unroll
        for (int i = 0; i < NC / 4; ++i) {
            const float4 f = src[i];
            h[4 * i] = f.x; h[4 * i + 1] = f.y; h[4 * i + 2] = f.z; h[4 * i + 3] = f.w;
        }
    } else {
#pragma unroll
        for (int i = 0; i < NC; ++i) h[i] = 0.f;
    }

    bool ok = true;
    const int r = row & 63;
    if (VCONV && nch > 0) {
        // the tile's taps, then chunk 0's V (chunk c+1's is made during chunk c)
        vconv_load_taps<NT>(S, p, hv, j0);
        asm volatile("bar.sync 3, %0;" :: "n"(kComputeThreads) : "memory");
        ok = wait_one(&S.bar_x[0], 0, abort);
        if (ok) vconv_chunk<NT>(S, p, n, hv, j0, 0, start, min(kC, len));
    }
    float aL_prev = 1.f;   // e^{gamma_L} of the previous chunk
    for (int c = 0; c < nch; ++c) {
        const int st = c & 1;
        const uint32_t ph = c & 1;
        const int t0 = start + c * kC;
        const int L = min(kC, len - c * kC);

        // --- A: fold the previous chunk's update into h, publish the bf16 copy.  This
        // chunk's tiles were requested a chunk ago: waiting for them here overlaps the
        // barrier query with the previous update's MMAs instead of following the barrier.
        if (ok) ok = wait_one(&S.bar_tma[st], (c >> 1) & 1, abort);
        // this row's per-token factors, formed while the previous update's MMAs run
        const float *sc = reinterpret_cast<const float *>(S.x[st] + kXTile);
        const float *gam = sc, *bet = sc + 64, *nk = sc + 128, *nq = sc + 192;
        const float gL = gam[L - 1];
        const float gr = gam[r];
        const float egr = __expf(gr);
        const float cr = egr * nk[r];                          // e^gamma nk   (chain rows)
        const float cq = egr * nq[r];                          // e^gamma nq   (output rows)
        const float dc = r < L ? __expf(gL - gr) * nk[r] : 0.f;   // e^{gamma_L-gamma} nk
        const float br = bet[r];
        const float aL = __expf(gL);
        if (c > 0 && ok) {
            ok = wait_one(&S.bar_d3, ph ^ 1, abort);
            if (ok) {
                tc::fence_after_sync();
                fold_update<NC>(h, aL_prev, tmem + lane_off + colS + ch);
            }
        }
        pack_row<NC>(S.hb, row, c0, h);
        tc::fence_async_smem();
        tc::fence_before_sync();
        __syncthreads();
        // this row's V columns, read ahead of the D1 wait (the chain rows' R needs them)
        uint4 vraw[NCH];
        if (chain) {
            const uint8_t *vt = VCONV ? S.vc[st] : S.v[st];
#pragma unroll
            for (int cc = 0; cc < NCH; ++cc)
                vraw[cc] = job.with_v ? *reinterpret_cast<const uint4 *>(vt + tc::swz(r, c0 + cc))
                                      : make_uint4(0u, 0u, 0u, 0u);
        }

        // the next chunk's V, while the chain waits for D1
        if (VCONV && c + 1 < nch && ok) {
            ok = wait_one(&S.bar_x[(c + 1) % 3], ((c + 1) / 3) & 1, abort);
            if (ok)
                vconv_chunk<NT>(S, p, n, hv, j0, c + 1, t0 + kC, min(kC, len - (c + 1) * kC));
        }

        // --- B: R = beta (V - e^gamma nk K h) on the chain rows; e^gamma nq Q h on the rest
        if (ok) ok = wait_one(&S.bar_d1, ph, abort);
        float keep[NC];
        {
            float d1[NC];
            if (ok) {
                tc::fence_after_sync();
                tmem_cols<NC>(tmem + lane_off + colD1 + ch, d1);
            } else {
#pragma unroll
                for (int j = 0; j < NC; ++j) d1[j] = 0.f;
            }
            if (chain) {
                // R = beta (v - c d1) two columns at a time; rows past the chunk's end are
                // exact zeros
                const float2 br2 = make_float2(br, br);
                const float2 ncr = make_float2(-cr, -cr);
                if (r < L) {
#pragma unroll
                    for (int cc = 0; cc < NCH; ++cc) {
                        const uint4 u = vraw[cc];
                        const uint32_t uw[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const int i = 8 * cc + 2 * q;
                            const float2 v2 = make_float2(__uint_as_float(uw[q] << 16),
                                                          __uint_as_float(uw[q] & 0xffff0000u));
                            const float2 x2 = mul2(br2, fma2(ncr, make_float2(d1[i], d1[i + 1]), v2));
                            keep[i] = x2.x;
                            keep[i + 1] = x2.y;
                        }
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < NC; ++j) keep[j] = 0.f;
                }
                pack_row<NC>(S.rb, r, c0, keep);
                tc::fence_async_smem();
                tc::fence_before_sync();
                chain_barrier();
            } else {
                const float2 cq2 = make_float2(cq, cq);
#pragma unroll
                for (int j = 0; j < NC; j += 2) {
                    const float2 k2 = mul2(cq2, make_float2(d1[j], d1[j + 1]));
                    keep[j] = k2.x;
                    keep[j + 1] = k2.y;
                }
            }
        }

        // --- C: Vn = R + Lo R -> d Vn as bf16 hi + lo; outputs on the other rows
        if (ok) ok = wait_one(&S.bar_d2, ph, abort);
        {
            float d2[NC];
            if (ok) {
                tc::fence_after_sync();
                tmem_cols<NC>(tmem + lane_off + colD2 + ch, d2);
            } else {
#pragma unroll
                for (int j = 0; j < NC; ++j) d2[j] = 0.f;
            }
            if (chain) {
                // hi = bf16(x) two at a time (the paired conversion issues at several times
                // the rate of the single one); lo = x - hi is exact in fp32
                uint32_t hp[NC / 2];
                float lo[NC];
                const float2 dc2 = make_float2(dc, dc), m1 = make_float2(-1.f, -1.f);
#pragma unroll
                for (int jj = 0; jj < NC / 2; ++jj) {
                    const float2 x2 = mul2(dc2, add2(make_float2(keep[2 * jj], keep[2 * jj + 1]),
                                                     make_float2(d2[2 * jj], d2[2 * jj + 1])));
                    const __nv_bfloat162 hb2 = __floats2bfloat162_rn(x2.x, x2.y);
                    hp[jj] = *reinterpret_cast<const uint32_t *>(&hb2);
                    const float2 l2 = fma2(m1, make_float2(__uint_as_float(hp[jj] << 16),
                                                           __uint_as_float(hp[jj] & 0xffff0000u)), x2);
                    lo[2 * jj] = l2.x;
                    lo[2 * jj + 1] = l2.y;
                }
#pragma unroll
                for (int cc = 0; cc < NCH; ++cc) {
                    // hi: elements ch + 8cc of [hi | lo]; lo: NT + ch + 8cc, in 64-wide blocks
                    *reinterpret_cast<uint4 *>(S.dvh + tc::swz(r, c0 + cc)) =
                        make_uint4(hp[4 * cc], hp[4 * cc + 1], hp[4 * cc + 2], hp[4 * cc + 3]);
                    const int el = NT + 8 * (c0 + cc);
                    float f[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) f[e] = lo[8 * cc + e];
                    *reinterpret_cast<uint4 *>((el >= 64 ? S.dvl : S.dvh) + tc::swz(r, (el & 63) >> 3)) =
                        pack8(f);
                }
                tc::fence_async_smem();
                tc::fence_before_sync();
                chain_barrier();
            } else if (!job.write_o) {
                // no outputs from this CTA
            } else if (L == kC) {
                // A full chunk's O tile goes out through shared memory with one tensor store,
                // keeping 64 scattered row writes per warp off the load/store pipeline that
                // the chain warps' shared-memory traffic shares.  Stage st was last stored
                // two chunks ago; allowing one group in flight covers the previous chunk.
                // A 64-wide tile uses the 128B-swizzled layout, narrower ones plain rows.
                uint8_t *ob = S.ob[st];
                if (tid == kOutLeader) tc::bulk_wait_read<1>();
                out_barrier();
#pragma unroll
                for (int cc = 0; cc < NCH; ++cc) {
                    float f[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) f[e] = p.scale * (keep[8 * cc + e] + d2[8 * cc + e]);
                    const uint32_t off = NT == 64 ? tc::swz(r, c0 + cc)
                                                  : (uint32_t)(r * NT * 2 + (c0 + cc) * 16);
                    *reinterpret_cast<uint4 *>(ob + off) = pack8(f);
                }
                tc::fence_async_smem();
                out_barrier();
                if (tid == kOutLeader && ok && !*abort) {
                    tc::tma_store_3d(omap, ob, j0, hv, t0);
                    tc::bulk_commit();
                }
            } else if (r < L && ok) {
                // the last, partial chunk of a sequence: rows past L belong to the next one
                uint4 *dst = reinterpret_cast<uint4 *>(p.o + (size_t)(t0 + r) * p.o_tok +
                                                       (size_t)hv * kD + j0 + ch);
#pragma unroll
                for (int cc = 0; cc < NCH; ++cc) {
                    float f[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) f[e] = p.scale * (keep[8 * cc + e] + d2[8 * cc + e]);
                    dst[cc] = pack8(f);
                }
            }
            tc::fence_before_sync();
        }
        aL_prev = aL;
    }
    if (ok && nch > 0) {
        ok = wait_one(&S.bar_d3, (nch - 1) & 1, abort);
        if (ok) {
            tc::fence_after_sync();
            fold_update<NC>(h, aL_prev, tmem + lane_off + colS + ch);
        }
    }
    if (tid == kOutLeader) tc::bulk_wait_all();   // O tiles written before the CTA exits
    tc::fence_before_sync();
    __syncthreads();
    if (VCONV && !*abort) vconv_state_out<NT>(p, n, hv, j0, start, len);
    if (!*abort && job.hT) {
        float4 *dst = reinterpret_cast<float4 *>(job.hT + (size_t)row * kD + j0 + ch);
#pragma unroll
        for (int i = 0; i < NC / 4; ++i)
            dst[i] = make_float4(h[4 * i], h[4 * i + 1], h[4 * i + 2], h[4 * i + 3]);
    }
    if (*abort && tid == 0) report(p.status, GDN_ERR_TIMEOUT);
    if (warp == 0) tc::tmem_dealloc(tmem, 256);
}

// One CTA per (sequence, v-head, dv tile).  The tiles of a head are either two of 64
// columns or, when that leaves SMs idle (p.ntiles == 3), 48 + 48 + 32 columns.
template <bool VCONV>
__device__ __forceinline__ void state_kernel_body(const TcMaps &maps, const TcParams &p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    StateSmem &S = *reinterpret_cast<StateSmem *>(
        (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023));
    grid_dependents_launch();
    const int tid = threadIdx.x, warp = tid >> 5;
    const int jt = blockIdx.x, hv = blockIdx.y;
    const int n = p.cp == 0 && (int)blockIdx.z < p.n_order ? (int)p.order[blockIdx.z] : (int)blockIdx.z;
    // TMEM, barriers and tensor-map prefetches touch no memory of the previous kernel, so
    // they run before the dependency wait below
    if (warp == 0) {
        tc::tmem_alloc(&S.tmem, 256);
        tc::tmem_relinquish();
    }
    if (tid == 0) {
        tc::mbar_init(&S.bar_tma[0], 1);
        tc::mbar_init(&S.bar_tma[1], 1);
        tc::mbar_init(&S.bar_d1, 1);
        tc::mbar_init(&S.bar_d2, 1);
        tc::mbar_init(&S.bar_d3, 1);
        tc::mbar_init(&S.bar_fin, 1);
        if (VCONV)
            for (int i = 0; i < 3; ++i) tc::mbar_init(&S.bar_x[i], 1);
        S.abort = 0;
        tc::mbar_fence_init();
        tc::prefetch_tmap(&maps.k);
        tc::prefetch_tmap(&maps.q);
        tc::prefetch_tmap(&maps.v);
        tc::prefetch_tmap(p.ntiles == 3 ? (jt < 2 ? &maps.o48 : &maps.o32) : &maps.o);
    }
    grid_dependency_wait();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const size_t hd = (size_t)kD * kD;                  // one head's state
    StateJob job;
    job.identity = false;
    job.with_v = true;
    job.write_o = true;
    job.active = true;
    if (p.cp == 0) {
        job.n = n;
        job.h0 = p.h0 ? p.h0 + ((size_t)n * p.Hv + hv) * hd : nullptr;
        job.hT = p.hT ? p.hT + ((size_t)n * p.Hv + hv) * hd : nullptr;
    } else {
        const bool trans = p.cp == 1 && n >= p.n_ranges;
        const int rr = trans ? n - p.n_ranges : n;
        const int32_t t = p.rtab[rr];
        const int seq = t & kRangeSeq;
        const bool first = (t & kRangeFirst) != 0, last = (t & kRangeLast) != 0;
        float *hT_seq = p.hT ? p.hT + ((size_t)seq * p.Hv + hv) * hd : nullptr;
        const size_t roff = ((size_t)rr * p.Hv + hv) * hd;
        job.n = rr;
        job.h0 = nullptr;
        job.hT = nullptr;
        if (p.cp == 1 && !trans) {
            // a later sequence's last range: its end state from zero would feed no
            // composition (nothing follows it), so the first pass skips it
            job.active = first || !last;
            job.h0 = first && p.h0 ? p.h0 + ((size_t)seq * p.Hv + hv) * hd : nullptr;
            job.hT = first && last ? hT_seq : (job.active ? p.sA + roff : nullptr);
            job.write_o = first;
        } else if (p.cp == 1) {
            job.active = !first && !last;
            job.identity = true;
            job.with_v = false;
            job.write_o = false;
            job.hT = job.active ? p.sP + roff : nullptr;
        } else {
            job.active = !first;
            job.h0 = job.active ? p.sS + roff : nullptr;
            job.hT = job.active && last ? hT_seq : nullptr;
        }
    }
    if (p.ntiles != 3)
        state_cta<64, VCONV>(S, maps, p, &maps.o, 64 * jt, hv, job);
    else if (jt < 2)
        state_cta<48, VCONV>(S, maps, p, &maps.o48, 48 * jt, hv, job);
    else
        state_cta<32, VCONV>(S, maps, p, &maps.o32, 96, hv, job);
}

__global__ void __launch_bounds__(kStateThreads, 1)
chunk_state_kernel(const __grid_constant__ TcMaps maps, const __grid_constant__ TcParams p) {
    state_kernel_body<false>(maps, p);
}

// The same with the layer's v-channel conv fused in (p.vconv = 1).
__global__ void __launch_bounds__(kStateThreads, 1)
chunk_state_vconv_kernel(const __grid_constant__ TcMaps maps, const __grid_constant__ TcParams p) {
    state_kernel_body<true>(maps, p);
}

// ====================================================== context-parallel composition
// A sequence split into chunk-aligned ranges: each range's end state is an affine map of
// its start state, h_end = P h_start + R (h in the [dk][dv] layout, P dk x dk), since
// every token's update h <- e^g (I - beta k k^T) h + beta k v^T is affine in h.  The
// first state pass gives R (start 0) and P (start I, V = 0) for every range; the start
// states follow in order, S_{r+1} = P_r S_r + R_r; the second pass reruns each range from
// its start.

// The split batch's tables, from the device copy of cu: range bounds, per range its
// sequence and first / last flags, and each sequence's first range.  One thread, in
// order; a range count that disagrees with the host's (a device cu that differs from the
// host copy) stops the tables and reports GDN_ERR_SEQLENS.
__global__ void cp_tables_kernel(const int32_t *cu, int N, int range_chunks, int n_ranges,
                                 int32_t *cu_split, int32_t *rtab, int32_t *seq_first,
                                 int32_t *status) {
    if (threadIdx.x != 0 || blockIdx.x != 0) return;
    int idx = 0;
    for (int n = 0; n < N; ++n) {
        const int start = cu[n], len = cu[n + 1] - start;
        const int nch = (len + kC - 1) / kC;
        const int R = max(1, (nch + range_chunks - 1) / range_chunks);
        seq_first[n] = idx;
        for (int r = 0; r < R; ++r) {
            if (idx >= n_ranges) {
                report(status, GDN_ERR_SEQLENS);
                return;
            }
            cu_split[idx] = start + (int)min((int64_t)r * range_chunks * kC, (int64_t)len);
            rtab[idx] = n | (r == 0 ? kRangeFirst : 0) | (r == R - 1 ? kRangeLast : 0);
            ++idx;
        }
    }
    if (idx != n_ranges) report(status, GDN_ERR_SEQLENS);
    cu_split[n_ranges] = cu[N];
}

// Start states of a sequence's ranges, in order: one CTA per (8 dv columns, v-head,
// sequence).  S = the first range's end state; for each later range r: its start is S,
// then S <- P_r S + R_r in fp32, each element as (((R + the k < 32 terms) + the
// 32 <= k < 64 terms) + the 64 <= k < 96 terms) + the k >= 96 terms, every part in
// increasing k.  The chain is sequential over ranges, so a step's latency is what counts:
// a thread takes two dk rows (i, i + 64) of one k quarter, so each broadcast read of S
// serves both rows; then every thread adds up the four quarters of 4 of the 1024 outputs.
// P (64 KiB) and this CTA's R columns (4 KiB) of the next two ranges are in flight
// (16-byte asynchronous copies into a three-deep ring) while the current step computes,
// and the products run as packed fp32 pairs (fma.rn.f32x2, rounded like two fmaf).  P
// rows are stored with their 16-byte groups permuted (group g of row i at g ^ (i & 7)),
// so the eight rows a quarter-warp reads at once fall on distinct banks.
constexpr int kComposeCols = 8;
constexpr int kComposeSplit = 4;                       // k quarters
constexpr int kComposeThreads = kComposeSplit * kD / 2;
constexpr int kComposeDepth = 3;                       // P / R ring slots
constexpr size_t kComposeSmem = (size_t)kComposeDepth * kD * kD * 4 +
                                (size_t)(1 + kComposeSplit + kComposeDepth) * kD * kComposeCols * 4;
static_assert(kComposeSmem <= 227 * 1024, "composition ring exceeds shared memory");
static_assert(kComposeThreads * 4 == kD * kComposeCols, "one float4 of S per thread");

__device__ __forceinline__ void cp_async16(void *smem, const void *gmem) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;"
                 :: "r"(tc::smem_u32(smem)), "l"(gmem) : "memory");
}

__global__ void __launch_bounds__(kComposeThreads, 1)
cp_compose_kernel(const float *sA, const float *sP, float *sS, const int32_t *seq_first,
                  int N, int Hv, int n_ranges) {
    extern __shared__ __align__(16) float csm[];
    float (*Psm)[kD][kD] = reinterpret_cast<float (*)[kD][kD]>(csm);
    float *after_p = csm + kComposeDepth * kD * kD;
    float (*Ssm)[kComposeCols] = reinterpret_cast<float (*)[kComposeCols]>(after_p);
    float (*Hsm)[kD][kComposeCols] =
        reinterpret_cast<float (*)[kD][kComposeCols]>(after_p + kD * kComposeCols);
    float (*Rsm)[kD][kComposeCols] =
        reinterpret_cast<float (*)[kD][kComposeCols]>(after_p + (1 + kComposeSplit) * kD * kComposeCols);
    grid_dependents_launch();
    grid_dependency_wait();
    const int j0 = blockIdx.x * kComposeCols, hv = blockIdx.y, n = blockIdx.z;
    const int i = threadIdx.x & (kD / 2 - 1), kq = threadIdx.x / (kD / 2);   // rows i, i + 64
    const int orow = threadIdx.x >> 1, ocol = 4 * (threadIdx.x & 1);         // the float4 it sums
    const int first = seq_first[n];
    const int R = (n + 1 < N ? seq_first[n + 1] : n_ranges) - first;
    if (R <= 1) return;
    const size_t hd = (size_t)kD * kD;
    auto head = [&](const float *base, int range) { return base + ((size_t)range * Hv + hv) * hd; };
    auto start = [&](int range) { return sS + ((size_t)range * Hv + hv) * hd + (size_t)orow * kD + j0 + ocol; };
    // Step r (1 <= r <= R - 2) reads P and R of range first + r from ring slot r % 3.  One
    // commit group per step, empty past the last map, so a wait for all but the newest
    // group always covers the step about to run.
    auto fetch = [&](int r) {
        if (r <= R - 2) {
            const int b = r % kComposeDepth;
            const float *P = head(sP, first + r);
            for (int c = threadIdx.x; c < kD * kD / 4; c += kComposeThreads) {
                const int row = c / (kD / 4), grp = c % (kD / 4);
                cp_async16(&Psm[b][row][4 * (grp ^ (row & 7))], P + (size_t)row * kD + 4 * grp);
            }
            cp_async16(&Rsm[b][orow][ocol], head(sA, first + r) + (size_t)orow * kD + j0 + ocol);
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
    };
    fetch(1);
    fetch(2);
    {   // the second range starts at the first one's end state
        const float4 v = *reinterpret_cast<const float4 *>(head(sA, first) + (size_t)orow * kD + j0 + ocol);
        *reinterpret_cast<float4 *>(&Ssm[orow][ocol]) = v;
        *reinterpret_cast<float4 *>(start(first + 1)) = v;
    }
    for (int r = 1; r <= R - 2; ++r) {
        asm volatile("cp.async.wait_group 1;" ::: "memory");
        __syncthreads();                       // S and step r's slot visible; slot (r+2)%3 free
        fetch(r + 2);
        const int b = r % kComposeDepth;
        float2 acc[2][kComposeCols / 2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int row = i + h * (kD / 2);
#pragma unroll
            for (int j = 0; j < kComposeCols / 2; ++j)
                acc[h][j] = kq == 0 ? *reinterpret_cast<const float2 *>(&Rsm[b][row][2 * j])
                                    : make_float2(0.f, 0.f);
        }
        const float *prow0 = Psm[b][i], *prow1 = Psm[b][i + kD / 2];
#pragma unroll
        for (int g = 0; g < kD / (4 * kComposeSplit); ++g) {
            const int grp = kq * (kD / (4 * kComposeSplit)) + g;
            const int off = 4 * (grp ^ (i & 7));          // rows i and i + 64 share i & 7
            const float4 pa = *reinterpret_cast<const float4 *>(prow0 + off);
            const float4 pb = *reinterpret_cast<const float4 *>(prow1 + off);
            const float ka[4] = {pa.x, pa.y, pa.z, pa.w}, kb[4] = {pb.x, pb.y, pb.z, pb.w};
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const float4 s0 = *reinterpret_cast<const float4 *>(&Ssm[4 * grp + u][0]);
                const float4 s1 = *reinterpret_cast<const float4 *>(&Ssm[4 * grp + u][4]);
                const float2 sv[4] = {make_float2(s0.x, s0.y), make_float2(s0.z, s0.w),
                                      make_float2(s1.x, s1.y), make_float2(s1.z, s1.w)};
                const float2 qa = make_float2(ka[u], ka[u]), qb = make_float2(kb[u], kb[u]);
#pragma unroll
                for (int j = 0; j < kComposeCols / 2; ++j) {
                    acc[0][j] = fma2(qa, sv[j], acc[0][j]);
                    acc[1][j] = fma2(qb, sv[j], acc[1][j]);
                }
            }
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            float *dst = Hsm[kq][i + h * (kD / 2)];
            *reinterpret_cast<float4 *>(dst) = make_float4(acc[h][0].x, acc[h][0].y, acc[h][1].x, acc[h][1].y);
            *reinterpret_cast<float4 *>(dst + 4) = make_float4(acc[h][2].x, acc[h][2].y, acc[h][3].x, acc[h][3].y);
        }
        __syncthreads();                       // every read of S and of this slot is done
        float4 v = *reinterpret_cast<const float4 *>(&Hsm[0][orow][ocol]);
#pragma unroll
        for (int q = 1; q < kComposeSplit; ++q) {
            const float4 w = *reinterpret_cast<const float4 *>(&Hsm[q][orow][ocol]);
            const float2 lo = add2(make_float2(v.x, v.y), make_float2(w.x, w.y));
            const float2 hi = add2(make_float2(v.z, v.w), make_float2(w.z, w.w));
            v = make_float4(lo.x, lo.y, hi.x, hi.y);
        }
        *reinterpret_cast<float4 *>(&Ssm[orow][ocol]) = v;
        *reinterpret_cast<float4 *>(start(first + r + 1)) = v;
    }
    asm volatile("cp.async.wait_group 0;" ::: "memory");   // nothing in flight at exit
}

// Self-test of the bounded waits: one CTA waits, with the helper the kernels above use,
// on an mbarrier phase that nothing completes.  The wait gives up after kWaitNs and the
// CTA reports GDN_ERR_TIMEOUT, as a kernel above does when a copy or an MMA it waits on
// never signals; then it returns, leaving the context usable.
__global__ void __launch_bounds__(128) wait_selftest_kernel(int32_t *status) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        tc::mbar_init(&bar, 1);   // one arrival expected; none comes
        tc::mbar_fence_init();
    }
    __syncthreads();
    if (!wait_all(&bar, 0) && threadIdx.x == 0) report(status, GDN_ERR_TIMEOUT);
}

}  // namespace gdn

// ======================================================================== host side

namespace gdn_host {

namespace {

constexpr int kMaxDevices = 64;

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() { return tensor_map_encoder(); }

// [T, H, 128] bf16 token-major view -> 3-D map (d, head, token), box (width, 1, 64): 64
// columns with the 128B swizzle, or a narrower plain (unswizzled) box for output tiles.
bool make_map(CUtensorMap *m, const void *ptr, int64_t T, int H, int64_t tok_stride,
              int width = 64) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)gdn::kD, (cuuint64_t)H, (cuuint64_t)(T > 0 ? T : 1)};
    cuuint64_t strides[2] = {(cuuint64_t)gdn::kD * 2, (cuuint64_t)tok_stride * 2};
    cuuint32_t box[3] = {(cuuint32_t)width, 1, 64};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(ptr), dims, strides,
                    box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    width == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Streaming multiprocessors of the current device (cached per device).
int sm_count() {
    static std::atomic<int> cached[kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
    int v = cached[dev].load(std::memory_order_relaxed);
    if (v == 0) {
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        cached[dev].store(v, std::memory_order_relaxed);
    }
    return v;
}

}  // namespace

bool chunk_tc_supported(int32_t dk, int32_t dv, int32_t chunk, int in_f32) {
    return dk == gdn::kD && dv == gdn::kD && chunk == gdn::kC && !in_f32;
}

size_t chunk_tc_workspace(int32_t N, int64_t T, int32_t Hk, int32_t Hv) {
    (void)Hk;
    const size_t slots = (size_t)((T + gdn::kC - 1) / gdn::kC) + (size_t)N + 1;
    return slots * (size_t)Hv * gdn::kWsTile;
}

gdn_status_t launch_wait_selftest(int32_t *status, cudaStream_t st) {
    gdn::wait_selftest_kernel<<<1, 128, 0, st>>>(status);
    return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

namespace {

// Tensor maps, kernel parameters and the one-time per-device kernel attributes shared by
// the plain and the context-parallel scans.  n_chains: CTAs per (head, dv tile) of the
// state pass, for the tiling choice.
gdn_status_t setup_scan(const ScanArgs &a, int64_t n_chains, gdn::TcMaps &maps,
                        gdn::TcParams &p, size_t &prep_smem, size_t &state_smem) {
    // with the fused v conv the V map views the raw activations' v channels
    const VConvArgs *vc = a.vconv;
    const void *vsrc = vc ? (const void *)((const gdn::bf16 *)vc->x + vc->cv0) : a.v;
    const int64_t vtok = vc ? vc->xc : a.v_tok;
    if (!make_map(&maps.q, a.q, a.T, a.Hk, a.q_tok) || !make_map(&maps.k, a.k, a.T, a.Hk, a.k_tok) ||
        !make_map(&maps.v, vsrc, a.T, a.Hv, vtok) || !make_map(&maps.o, a.o, a.T, a.Hv, a.o_tok) ||
        !make_map(&maps.o48, a.o, a.T, a.Hv, a.o_tok, 48) ||
        !make_map(&maps.o32, a.o, a.T, a.Hv, a.o_tok, 32))
        return GDN_ERR_CUDA;
    memset(&p, 0, sizeof(p));
    p.g = a.g;
    p.beta = a.beta;
    p.cu = a.cu;
    p.h0 = a.h0;
    p.hT = a.hT;
    p.o = (gdn::bf16 *)a.o;
    p.o_tok = a.o_tok;
    p.ws = (uint8_t *)a.ws;
    p.N = a.N;
    p.Hk = a.Hk;
    p.Hv = a.Hv;
    p.scale = a.scale;
    p.l2norm = (a.flags & GDN_QK_L2NORM) ? 1 : 0;
    p.status = a.status;
    if (vc) {
        p.vconv = 1;
        p.xr = (const gdn::bf16 *)vc->x;
        p.y = (gdn::bf16 *)vc->y;
        p.cw = (const gdn::bf16 *)vc->w;
        p.cb = (const gdn::bf16 *)vc->b;
        p.cs_in = (const gdn::bf16 *)vc->s_in;
        p.cs_out = (gdn::bf16 *)vc->s_out;
        p.xc = vc->xc;
        p.cv0 = vc->cv0;
    }
    // Three dv tiles per head (48 + 48 + 32 columns) when they still fit one wave on the
    // SMs, else two of 64.  So the tiling follows N and the device's SM count; it changes
    // how the columns are grouped, not the arithmetic of any column (every column's
    // products, reductions and roundings are the same whatever tile it sits in), which
    // keeps a sequence's bits the same alone and in a batch.  GDN_PREFILL_TILES2/3 force
    // one tiling; the GPU tests run the same sequences under both and compare the bits.
    const int sms = sm_count();
    if (a.flags & GDN_PREFILL_TILES2)
        p.ntiles = 2;
    else if (a.flags & GDN_PREFILL_TILES3)
        p.ntiles = 3;
    else
        p.ntiles = (sms > 0 && (int64_t)3 * a.Hv * n_chains <= sms) ? 3 : 2;

    prep_smem = sizeof(gdn::PrepSmem) + 1024;
    state_smem = (vc ? sizeof(gdn::StateSmem) : gdn::kStateSmemPlain) + 1024;
    // the shared-memory opt-in is a per-device attribute: set it once on each device
    static std::atomic<bool> attr_set[kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return GDN_ERR_CUDA;
    if (!attr_set[dev].load(std::memory_order_acquire)) {
        // five prep CTAs per SM need the largest shared-memory carveout
        if (cudaFuncSetAttribute(gdn::chunk_prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)prep_smem) != cudaSuccess ||
            cudaFuncSetAttribute(gdn::chunk_prep_kernel,
                                 cudaFuncAttributePreferredSharedMemoryCarveout, 100) != cudaSuccess ||
            cudaFuncSetAttribute(gdn::chunk_state_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)(gdn::kStateSmemPlain + 1024)) != cudaSuccess ||
            cudaFuncSetAttribute(gdn::chunk_state_vconv_kernel,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)(sizeof(gdn::StateSmem) + 1024)) != cudaSuccess ||
            cudaFuncSetAttribute(gdn::cp_compose_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)gdn::kComposeSmem) != cudaSuccess)
            return GDN_ERR_CUDA;
        attr_set[dev].store(true, std::memory_order_release);
    }
    return GDN_OK;
}

gdn_status_t launch_prep(const gdn::TcMaps &maps, const gdn::TcParams &p, int64_t T,
                         size_t prep_smem, cudaStream_t st) {
    const int slots = (int)((T + gdn::kC - 1) / gdn::kC) + p.N;
    if (slots <= 0) return GDN_OK;
    dim3 g1(slots, p.Hv);
    return launch_dependent(gdn::chunk_prep_kernel, g1, dim3(gdn::kPrepThreads), prep_smem, st,
                            maps, p) == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

gdn_status_t launch_state(const gdn::TcMaps &maps, const gdn::TcParams &p, int grid_z,
                          size_t state_smem, cudaStream_t st) {
    dim3 g2(p.ntiles, p.Hv, grid_z);
    return launch_dependent(p.vconv ? gdn::chunk_state_vconv_kernel : gdn::chunk_state_kernel, g2,
                            dim3(gdn::kStateThreads), state_smem, st, maps, p) == cudaSuccess
               ? GDN_OK : GDN_ERR_CUDA;
}

// Ranges of the context-parallel split: ceil(chunks / range_chunks) per sequence, at
// least one (an empty sequence is one empty range).  -1 when the count exceeds the
// launch limits.
int64_t cp_range_count(const int32_t *cu_host, int32_t N, int32_t range_chunks) {
    int64_t nr = 0;
    for (int32_t n = 0; n < N; ++n) {
        const int64_t len = (int64_t)cu_host[n + 1] - cu_host[n];
        const int64_t nch = (len + gdn::kC - 1) / gdn::kC;
        nr += std::max<int64_t>(1, (nch + range_chunks - 1) / range_chunks);
    }
    return 2 * nr > 65535 ? -1 : nr;
}

constexpr size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

struct CpLayout {
    size_t tiles, sA, sP, sS, cu_split, rtab, seq_first, total;
};

CpLayout cp_layout(int64_t nr, int32_t N, int64_t T, int32_t Hk, int32_t Hv) {
    CpLayout L;
    const size_t states = (size_t)nr * Hv * gdn::kD * gdn::kD * sizeof(float);
    L.tiles = 0;
    L.sA = align256(chunk_tc_workspace((int32_t)nr, T, Hk, Hv));
    L.sP = L.sA + align256(states);
    L.sS = L.sP + align256(states);
    L.cu_split = L.sS + align256(states);
    L.rtab = L.cu_split + align256((size_t)(nr + 1) * sizeof(int32_t));
    L.seq_first = L.rtab + align256((size_t)nr * sizeof(int32_t));
    L.total = L.seq_first + align256((size_t)N * sizeof(int32_t));
    return L;
}

}  // namespace

// Range length for one sequence of nch chunks over Hv v-heads alone on this device, by a
// cost count in chunk-times (one chunk of one state CTA's chain), kept in halves so that
// it stays integral: each state pass costs its waves of CTAs (one per SM, in the dv
// tiling the kernels pick) times the range length plus one (a CTA's start and end); the
// split adds 1.5 per range (the composition runs range after range, and each range's end
// state and transition map go through memory) and 12 in all (its extra launches).  The
// constants are fitted on the
// GB300 to 14 single-sequence shapes (4096 to 65536 tokens, 1 to 48 v-heads, each timed
// plainly and in two to seventeen range lengths): on every one the pick is the fastest
// of the timed choices.  0 when the plain scan is expected to be at least as fast.
int32_t cp_range_hint(int64_t seq_len, int32_t Hv, int32_t sms) {
    constexpr int64_t kCpCta = 2, kCpPerRange = 3, kCpFixed = 24;   // half chunk-times
    if (sms <= 0 || Hv <= 0 || seq_len <= 0) return 0;
    const int64_t nch = (seq_len + gdn::kC - 1) / gdn::kC;
    auto tiles = [&](int64_t chains) -> int64_t { return 3 * Hv * chains <= sms ? 3 : 2; };
    auto waves = [&](int64_t ctas) -> int64_t { return (ctas + sms - 1) / sms; };
    int64_t best = waves(tiles(1) * Hv) * (2 * nch + kCpCta);
    int32_t best_r = 0;
    // every range count the launches allow, each with the shortest range length that
    // gives it (a longer one only costs more)
    for (int64_t want = 2; want <= std::min<int64_t>(nch, 65535 / 2); ++want) {
        const int64_t r = (nch + want - 1) / want;
        const int64_t nr = (nch + r - 1) / r;
        if (nr != want) continue;               // this count is not reachable exactly
        const int64_t mid = nr > 2 ? nr - 2 : 0;
        const int64_t t = tiles(2 * nr);
        // first pass: every range but the last, and the middle ranges' transition maps
        const int64_t cost = (waves(t * Hv * (nr - 1 + mid)) + waves(t * Hv * (nr - 1))) * (2 * r + kCpCta) +
                             kCpPerRange * nr + kCpFixed;
        // ties go to the shorter range, never away from the plain scan
        if (cost < best || (cost == best && best_r != 0)) {
            best = cost;
            best_r = (int32_t)r;
        }
    }
    return best_r;
}

int32_t cp_range_hint(int64_t seq_len, int32_t Hv) {
    return cp_range_hint(seq_len, Hv, sm_count());
}

size_t chunk_tc_cp_workspace(const int32_t *cu_host, int32_t N, int64_t T, int32_t Hk,
                             int32_t Hv, int32_t range_chunks) {
    if (!cu_host || N <= 0 || range_chunks <= 0) return 0;
    const int64_t nr = cp_range_count(cu_host, N, range_chunks);
    if (nr < 0) return 0;
    return cp_layout(nr, N, T, Hk, Hv).total;
}

gdn_status_t launch_chunk_tc(const ScanArgs &a, const int32_t *cu_host, cudaStream_t st,
                             cudaEvent_t before_state) {
    if (a.N == 0) return GDN_OK;
    if (a.out_f32) return GDN_ERR_DTYPE;
    gdn::TcMaps maps;
    gdn::TcParams p;
    size_t prep_smem = 0, state_smem = 0;
    gdn_status_t s = setup_scan(a, a.N, maps, p, prep_smem, state_smem);
    if (s != GDN_OK) return s;
    // The state CTAs' sequence order: by chunk count, longest first (ties in batch order).
    // A chain's arithmetic does not depend on when it runs, so this changes no bits.
    if (a.N > 1 && a.N <= gdn::kStateOrderMax) {
        int32_t idx[gdn::kStateOrderMax];
        for (int32_t n = 0; n < a.N; ++n) idx[n] = n;
        auto chunks = [&](int32_t n) { return ((int64_t)cu_host[n + 1] - cu_host[n] + gdn::kC - 1) / gdn::kC; };
        std::stable_sort(idx, idx + a.N, [&](int32_t x, int32_t y) { return chunks(x) > chunks(y); });
        p.n_order = a.N;
        for (int32_t n = 0; n < a.N; ++n) p.order[n] = (uint16_t)idx[n];
    }
    if ((s = launch_prep(maps, p, a.T, prep_smem, st)) != GDN_OK) return s;
    if (before_state && cudaStreamWaitEvent(st, before_state, 0) != cudaSuccess)
        return GDN_ERR_CUDA;
    return launch_state(maps, p, a.N, state_smem, st);
}

gdn_status_t launch_chunk_tc_cp(const ScanArgs &a, const int32_t *cu_host, int32_t range_chunks,
                                cudaStream_t st) {
    if (a.N == 0) return GDN_OK;
    if (a.out_f32) return GDN_ERR_DTYPE;
    if (a.vconv) return GDN_ERR_UNSUPPORTED;
    if (range_chunks <= 0) return GDN_ERR_SHAPE;
    const int64_t nr = cp_range_count(cu_host, a.N, range_chunks);
    if (nr < 0) return GDN_ERR_SHAPE;
    const CpLayout L = cp_layout(nr, a.N, a.T, a.Hk, a.Hv);
    uint8_t *ws = (uint8_t *)a.ws;
    float *sA = (float *)(ws + L.sA), *sP = (float *)(ws + L.sP), *sS = (float *)(ws + L.sS);
    int32_t *cu_split = (int32_t *)(ws + L.cu_split), *rtab = (int32_t *)(ws + L.rtab);
    int32_t *seq_first = (int32_t *)(ws + L.seq_first);

    gdn::cp_tables_kernel<<<1, 32, 0, st>>>(a.cu, a.N, range_chunks, (int)nr, cu_split, rtab,
                                            seq_first, a.status);
    if (cudaGetLastError() != cudaSuccess) return GDN_ERR_CUDA;

    ScanArgs split = a;
    split.cu = cu_split;
    split.N = (int32_t)nr;
    gdn::TcMaps maps;
    gdn::TcParams p;
    size_t prep_smem = 0, state_smem = 0;
    gdn_status_t s = setup_scan(split, 2 * nr, maps, p, prep_smem, state_smem);
    if (s != GDN_OK) return s;
    p.rtab = rtab;
    p.n_ranges = (int)nr;
    p.sA = sA;
    p.sP = sP;
    p.sS = sS;
    // the workspace tiles depend only on q, k, g and beta: one prep pass serves both passes
    if ((s = launch_prep(maps, p, a.T, prep_smem, st)) != GDN_OK) return s;
    p.cp = 1;
    if ((s = launch_state(maps, p, (int)(2 * nr), state_smem, st)) != GDN_OK) return s;
    if (launch_dependent(gdn::cp_compose_kernel, dim3(gdn::kD / gdn::kComposeCols, a.Hv, a.N),
                         dim3(gdn::kComposeThreads), gdn::kComposeSmem, st, (const float *)sA,
                         (const float *)sP, sS, (const int32_t *)seq_first, (int)a.N, (int)a.Hv,
                         (int)nr) != cudaSuccess)
        return GDN_ERR_CUDA;
    p.cp = 2;
    return launch_state(maps, p, (int)nr, state_smem, st);
}

}  // namespace gdn_host
