// chunk_tc.cu -- tensor-core chunked gated delta rule for dk = dv = 128, chunk 64, bf16.
//
// Recurrence: "Qwen3.5-27B GPTQ Garbage Inference -- Root Cause Analysis", "Why
// abliteration failed on Qwen3.5", item 3.  Chunk boundaries anchored at every sequence
// start ("[Feature] Add batch invariance support to GDN_ATTN backend - #45819", Birol's
// comment, part 3(a), and the PR's "Fixes: 2."), so nothing depends on the packed batch.
//
// With gamma the in-chunk inclusive log-decay sums, nk, nq the L2-norm factors (1 when
// the flag is off) and h the [dk][dv] state entering a chunk, the chunk's WY/UT form is
//     A[r][s] = beta_r e^{gamma_r-gamma_s} nk_r nk_s (k_r.k_s)        s < r
//     M[r][s] = e^{gamma_r-gamma_s} nq_r nk_s (q_r.k_s)                s <= r
//     Tinv = (I + A)^{-1} = I + Lo,   a_s = beta_s e^{gamma_s} nk_s
//     W  = Tinv diag(a) K,            U = Tinv diag(beta) V
//     Vn = U - W h,                   O = scale (diag(e^gamma nq) Q h + M Vn)
//     h <- e^{gamma_L} h + K^T diag(e^{gamma_L-gamma} nk) Vn
// Everything that does not involve h is folded, per (chunk, v-head), into three operand
// tiles so that the state pass has one product before Vn and one after it:
//     WQ = [W ; Q'],  Q' = diag(e^gamma nq) Q - M W          (the rows that multiply h)
//     Z  = [-Lo diag(beta) ; Mt diag(beta)],  Mt = M Tinv     (the rows that multiply V)
// so that  [Z V + WQ h]  holds  beta V - Vn  in its first 64 rows and  O / scale  in the
// other 64  (Vn = beta V + Lo diag(beta) V - W h;  M Vn = Mt diag(beta) V - M W h).
//
// Two kernels, both tcgen05 (MMA into TMEM, operands in 128B-swizzled shared memory fed
// by TMA and bulk copies):
//
//  chunk_prep (one CTA per (chunk, v-head), fully parallel):
//      P = [K;Q] K^T  ->  A, M (fp32)  ->  Tinv (blocked forward substitution, CUDA
//      cores)  ->  Mt = M + M Lo  ->  [Lo a ; Mt a] K  ->  WQ, Z, and the per-token
//      scalars beta, d = e^{gamma_L-gamma} nk and e^{gamma_L}, stored as one workspace
//      tile.
//
//  chunk_state (one CTA per (sequence, v-head, dv tile), walks the chunks):
//      D  = Z V  (issued ahead, off the chain)  +  WQ h_bf16
//      Vn = beta V - D[0:64];   O = scale D[64:128]
//      h <- e^{gamma_L} h + K^T [hi | lo](d Vn)
//    The state update takes d Vn as a bf16 hi + lo pair (one MMA pass over [hi | lo], the
//    halves summed in fp32) and beta V enters Vn exactly in fp32, so the state keeps
//    fp32-level accuracy.  Eight compute warps: warps w and w+4 share TMEM lanes 32(w%4)..
//    and take half the tile's columns each; a ninth warp issues the MMAs and a tenth the
//    TMA and bulk loads.
//
// Every wait on an mbarrier is bounded in time; on expiry the CTA records GDN_ERR_TIMEOUT
// in the status word, stops issuing work, frees its TMEM and returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <atomic>

#include "common.cuh"
#include "tc_ptx.cuh"
#include "tmap.cuh"

namespace gdn {

constexpr int kPrepThreads = 128;
constexpr int kC = 64;          // chunk
constexpr int kD = 128;         // dk = dv
constexpr uint32_t kXTile = 16384;            // bf16 [128 rows][64] swizzled
// Workspace tile per (chunk slot, v-head)
constexpr uint32_t kWQBytes = 32768;          // [W ; Q'] bf16: two 64-column K blocks
constexpr uint32_t kZOff = kWQBytes;          // Z = [-Lo diag(beta) ; Mt diag(beta)] bf16
constexpr uint32_t kScalOff = kZOff + kXTile; // beta[64], d[64], e^{gamma_L} (fp32)
constexpr uint32_t kScalBytes = 528;
constexpr uint32_t kWsTile = kScalOff + kScalBytes;
static_assert(kWsTile % 16 == 0, "bulk copies move multiples of 16 bytes");
constexpr uint64_t kWaitNs = 2000000000ull;   // 2 s bound on any single wait

struct TcMaps {
    CUtensorMap q, k, v, o;
    CUtensorMap o48, o32;   // O as 48- and 32-column plain (unswizzled) boxes
};

struct TcParams {
    const float *g, *beta;
    const int32_t *cu;
    const float *h0;
    float *hT;
    bf16 *o;
    int64_t o_tok;
    const bf16 *q;           // q rows, read back by the prep kernel for Q'
    int64_t q_tok;
    uint8_t *ws;
    int N, Hk, Hv;
    float scale;
    int l2norm;
    int ntiles;              // dv tiles per head in the state kernel: 2 or 3
    int32_t *status;
};

__device__ __forceinline__ uint64_t now_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}

// Bounded wait on an mbarrier phase by thread 0, then a CTA-wide agreement.  The barrier
// orders everything the phase made visible to thread 0 before the other threads' reads,
// and only one thread polls the mbarrier's shared-memory word.
__device__ __forceinline__ bool wait_all(uint64_t *bar, uint32_t parity) {
    bool ok = true;
    if (threadIdx.x == 0) {
        ok = tc::mbar_try_wait(bar, parity);
        if (!ok) {
            const uint64_t t0 = now_ns();
            while (!(ok = tc::mbar_try_wait(bar, parity)))
                if (now_ns() - t0 > kWaitNs) break;
        }
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

// Packed fp32 pair arithmetic (two lanes per instruction).
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
// blocks (block stride `blk` bytes): four packed accumulators over fixed element
// positions, summed in a fixed order.
__device__ __forceinline__ float row_sumsq(const uint8_t *tile, int row, uint32_t blk,
                                           uint32_t park) {
    float2 acc[4] = {{0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}};
#pragma unroll
    for (int kb = 0; kb < 2; ++kb) {
        float raw[32];   // the 64 bf16 values of this block, as 32 packed words
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            const uint4 u = *reinterpret_cast<const uint4 *>(tile + kb * blk + tc::swz(row, c));
            raw[4 * c] = __uint_as_float(u.x); raw[4 * c + 1] = __uint_as_float(u.y);
            raw[4 * c + 2] = __uint_as_float(u.z); raw[4 * c + 3] = __uint_as_float(u.w);
            float f[8];
            unpack8(u, f);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 x = make_float2(f[2 * e], f[2 * e + 1]);
                acc[e] = fma2(x, x, acc[e]);
            }
        }
        tc::tmem_st32(park + 32 * kb, raw);
    }
    return ((acc[0].x + acc[0].y) + (acc[1].x + acc[1].y)) +
           ((acc[2].x + acc[2].y) + (acc[3].x + acc[3].y));
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
// written, with a barrier in between.  Every product is a 16x16 block computed by 64
// threads holding 2x2 register tiles.  All 128 threads call this; Y ([64][kLdY]) is a
// scratch for the 16- and 32-column intermediates.
constexpr int kLd = 66;
constexpr int kLdY = 34;

// acc += A[ar.., ac..] (16x16) * B[br.., bc..] (16x16) for this thread's 2x2 tile.
template <int LA, int LB>
__device__ __forceinline__ void blk_mma(float (&acc)[2][2], const float (*A)[LA], int ar, int ac,
                                        const float (*B)[LB], int br, int bc, int tr, int tc) {
    // partly unrolled: nine call sites, and the prep kernel's code size shows up as
    // instruction-fetch stalls
#pragma unroll 4
    for (int m = 0; m < 16; ++m) {
        const float a0 = A[ar + 2 * tr][ac + m], a1 = A[ar + 2 * tr + 1][ac + m];
        const float2 bb = *reinterpret_cast<const float2 *>(&B[br + m][bc + 2 * tc]);
        acc[0][0] = fmaf(a0, bb.x, acc[0][0]);
        acc[0][1] = fmaf(a0, bb.y, acc[0][1]);
        acc[1][0] = fmaf(a1, bb.x, acc[1][0]);
        acc[1][1] = fmaf(a1, bb.y, acc[1][1]);
    }
}

template <int LD>
__device__ __forceinline__ void blk_store(float (*D)[LD], int dr, int dc, int tr, int tc,
                                          const float (&acc)[2][2], float sgn) {
    *reinterpret_cast<float2 *>(&D[dr + 2 * tr][dc + 2 * tc]) = make_float2(sgn * acc[0][0], sgn * acc[0][1]);
    *reinterpret_cast<float2 *>(&D[dr + 2 * tr + 1][dc + 2 * tc]) = make_float2(sgn * acc[1][0], sgn * acc[1][1]);
}

__device__ void tinv64_inplace(float (*AT)[kLd], float (*Y)[kLdY]) {
    const int tid = threadIdx.x;
    const int half = tid >> 6, t = tid & 63, tr = t >> 3, tc = t & 7;
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
        __syncthreads();                       // every read of the A_ii is done
        if (tid < 64) {
#pragma unroll
            for (int r = 0; r < 16; ++r) AT[o + r][o + j] = x[r];
        }
    }
    __syncthreads();
    {   // X = A10 T00 (half 0) and A32 T22 (half 1), into Y rows 32.. and 48..
        float acc[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
        const int o = 32 * half;
        blk_mma(acc, AT, o + 16, o, AT, o, o, tr, tc);
        blk_store(Y, 32 + 16 * half, 0, tr, tc, acc, 1.f);
    }
    __syncthreads();
    {   // T10 = -T11 X over A10,  T32 = -T33 X over A32
        float acc[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
        const int o = 32 * half;
        blk_mma(acc, AT, o + 16, o + 16, Y, 32 + 16 * half, 0, tr, tc);
        blk_store(AT, o + 16, o, tr, tc, acc, -1.f);
    }
    __syncthreads();
    {   // Z = [A20 A21; A30 A31] T0 into Y[0:32][0:32]; half h makes block row h
        const int ar = 32 + 16 * half;
        float z0[2][2] = {{0.f, 0.f}, {0.f, 0.f}}, z1[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
        blk_mma(z0, AT, ar, 0, AT, 0, 0, tr, tc);     // A_r0 T00
        blk_mma(z0, AT, ar, 16, AT, 16, 0, tr, tc);   // + A_r1 T10
        blk_mma(z1, AT, ar, 16, AT, 16, 16, tr, tc);  // A_r1 T11
        blk_store(Y, 16 * half, 0, tr, tc, z0, 1.f);
        blk_store(Y, 16 * half, 16, tr, tc, z1, 1.f);
    }
    __syncthreads();
    {   // [T20 T21; T30 T31] = -T1 Z over A2x, A3x; half h makes block row 2 + h
        float w0[2][2] = {{0.f, 0.f}, {0.f, 0.f}}, w1[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
        if (half == 0) {
            blk_mma(w0, AT, 32, 32, Y, 0, 0, tr, tc);    // T22 Z20
            blk_mma(w1, AT, 32, 32, Y, 0, 16, tr, tc);   // T22 Z21
        } else {
            blk_mma(w0, AT, 48, 32, Y, 0, 0, tr, tc);    // T32 Z20
            blk_mma(w0, AT, 48, 48, Y, 16, 0, tr, tc);   // + T33 Z30
            blk_mma(w1, AT, 48, 32, Y, 0, 16, tr, tc);   // T32 Z21
            blk_mma(w1, AT, 48, 48, Y, 16, 16, tr, tc);  // + T33 Z31
        }
        // the stores go to columns 0..31, which no thread reads in this step
        blk_store(AT, 32 + 16 * half, 0, tr, tc, w0, -1.f);
        blk_store(AT, 32 + 16 * half, 16, tr, tc, w1, -1.f);
    }
    __syncthreads();
}

// ================================================================ chunk_prep kernel

// One 33 KB region, reused by lifetime:
//   [0, 32K)    the [K;Q] K-major tile, until P = [K;Q]K^T and the norms are taken;
//               then the fp32 A, inverted in place into T = (I + A)^{-1}, at byte 0 and
//               the inverse's scratch at kXOff; once T is dead, the Z tile (staged for
//               its bulk copy) and then the chunk's K tile again (two 64-column blocks at
//               0 and 8K), the B operand of Y K.
//   [17K, 33K)  X = [Lo ; M] (bf16, the A operand of M Lo), then Y = [Lo a ; Mt a].
// Finally the [W ; Q'] tile is staged over [0, 32K) for one bulk copy.
// TMEM (128 columns): columns 0..63 hold P, then M and Mt, then each 64-column half of
// [Lo a ; Mt a] K in turn; columns 64..127 hold, from the start, this thread's own row of
// the chunk's K (lanes 0..63) or Q (lanes 64..127) as packed bf16, for the epilogue.
constexpr uint32_t kXOff = 17 * 1024;   // 1024-aligned, past A
constexpr uint32_t kPrepRegion = kXOff + kXTile;
static_assert(64 * kLd * 4 <= kXOff && 64 * kLdY * 4 <= kXTile, "prep region layout");

struct PrepSmem {
    uint8_t buf[kPrepRegion];
    float gam[64], bet[64], nk[64], nq[64];
    float c2[64];            // gamma_s log2(e) - log2(nk_s): the key-side exponent
    float a[64];             // beta_s e^{gamma_s} nk_s
    float carry;
    uint64_t bar_tma, bar_mma;
    uint32_t tmem;

    __device__ uint8_t *kq() { return buf; }
    __device__ float (*AT())[kLd] { return reinterpret_cast<float (*)[kLd]>(buf); }
    __device__ float (*Y())[kLdY] { return reinterpret_cast<float (*)[kLdY]>(buf + kXOff); }
    __device__ uint8_t *x() { return buf + kXOff; }
};
static_assert(sizeof(PrepSmem) + 1024 <= 56 * 1024, "four prep CTAs fit on one SM");

// One CTA per (chunk slot, v-head); four CTAs per SM.
__global__ void __launch_bounds__(kPrepThreads, 4)
chunk_prep_kernel(const __grid_constant__ TcMaps maps, const __grid_constant__ TcParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    PrepSmem &S = *reinterpret_cast<PrepSmem *>(
        (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023));
    grid_dependents_launch();
    grid_dependency_wait();
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // Launched chunk-major in reverse: the first chunks of every head are prepared last,
    // so their tiles are the ones still in L2 when the state pass starts reading.
    const int hv = blockIdx.x, slot = gridDim.y - 1 - blockIdx.y;
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
        tc::tmem_alloc(&S.tmem, 128);
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
            tc::mma_bf16_warp(tmem, tc::sdesc(base + off, 16, 1024),
                              tc::sdesc(base + off, 16, 1024), id, ks > 0);
        }
        tc::mma_commit_warp(&S.bar_mma);
    }
    const int r = tid & 63;
    if (ok) {
        // L2-norm factors of this chunk's k rows (threads 0..63) and q rows (64..127)
        const float ss = row_sumsq(S.kq(), tid, 16384, tmem + lane_off + 64);
        tc::tmem_wait_st();
        const float f = p.l2norm ? rsqrtf(ss + 1e-6f) : 1.f;
        if (tid < 64) {
            const float nkr = r < L ? f : 0.f;
            const float gamr = tid >= 32 ? gs + S.carry : gs;
            S.nk[r] = nkr;
            S.gam[r] = gamr;
            S.bet[r] = bx;
            S.a[r] = bx * __expf(gamr) * nkr;
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
                tmem_row32(tmem + lane_off + 32 * hf, pv);
#pragma unroll
                for (int i = 0; i < 32; i += 4) {
                    const int s = 32 * hf + i;
                    const float4 c4 = *reinterpret_cast<const float4 *>(&S.c2[s]);
                    const float2 e0 = make_float2(fast_exp2(g2r - c4.x), fast_exp2(g2r - c4.y));
                    const float2 e1 = make_float2(fast_exp2(g2r - c4.z), fast_exp2(g2r - c4.w));
                    const float2 rf = make_float2(rowf, rowf);
                    const float2 w0 = mul2(mul2(rf, make_float2(pv[i], pv[i + 1])), e0);
                    const float2 w1 = mul2(mul2(rf, make_float2(pv[i + 2], pv[i + 3])), e1);
                    v[i] = (s < lim && r < L) ? w0.x : 0.f;
                    v[i + 1] = (s + 1 < lim && r < L) ? w0.y : 0.f;
                    v[i + 2] = (s + 2 < lim && r < L) ? w1.x : 0.f;
                    v[i + 3] = (s + 3 < lim && r < L) ? w1.y : 0.f;
                }
            }
            if (arow) {
#pragma unroll
                for (int i = 0; i < 32; i += 2)
                    *reinterpret_cast<float2 *>(&AT[r][32 * hf + i]) = make_float2(v[i], v[i + 1]);
            } else {
                // fp32 M over the P half just read: M Lo accumulates onto it, giving
                // Mt = M + M Lo (rows with no entries in this half store zeros)
                tc::tmem_st32(tmem + lane_off + 32 * hf, v);
            }
        }
        if (!arow) tc::tmem_wait_st();
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
            for (int i = 0; i < 32; i += 2) {
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
            tmem_row32(tmem + lane_off + 32 * hf, m);
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
            tc::mma_bf16_warp(tmem, tc::sdesc(xb + ks * 32, 16, 1024),
                              tc::sdesc(xb + ks * 2048, 8192, 1024), id, true);
        tc::mma_commit_warp(&S.bar_mma);
    }
    if (ok) ok = wait_all(&S.bar_mma, 1);

    // Y = [Lo diag(a) ; Mt diag(a)] over X (which the MMA has read), and the rows of
    // Z = [-Lo diag(beta) ; Mt diag(beta)], kept in registers until A is dead.
    uint32_t zrow[32];
    if (ok) {
        tc::fence_after_sync();
        const float zs = tid < 64 ? -1.f : 1.f;
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
            float src[32];
            if (tid < 64) {
#pragma unroll
                for (int i = 0; i < 32; i += 2) {
                    const float2 t2 = *reinterpret_cast<const float2 *>(&AT[r][32 * hf + i]);
                    src[i] = (32 * hf + i < r) ? t2.x : 0.f;
                    src[i + 1] = (32 * hf + i + 1 < r) ? t2.y : 0.f;
                }
            } else {
                tmem_row32(tmem + lane_off + 32 * hf, src);
            }
            float y[32];
#pragma unroll
            for (int i = 0; i < 32; i += 4) {
                const float4 a4 = *reinterpret_cast<const float4 *>(&S.a[32 * hf + i]);
                const float4 b4 = *reinterpret_cast<const float4 *>(&S.bet[32 * hf + i]);
                const float2 s0 = make_float2(src[i], src[i + 1]);
                const float2 s1 = make_float2(src[i + 2], src[i + 3]);
                const float2 y0 = mul2(s0, make_float2(a4.x, a4.y));
                const float2 y1 = mul2(s1, make_float2(a4.z, a4.w));
                const float2 z0 = mul2(mul2(s0, make_float2(zs, zs)), make_float2(b4.x, b4.y));
                const float2 z1 = mul2(mul2(s1, make_float2(zs, zs)), make_float2(b4.z, b4.w));
                y[i] = y0.x; y[i + 1] = y0.y; y[i + 2] = y1.x; y[i + 3] = y1.y;
                const __nv_bfloat162 p0 = __floats2bfloat162_rn(z0.x, z0.y);
                const __nv_bfloat162 p1 = __floats2bfloat162_rn(z1.x, z1.y);
                zrow[16 * hf + i / 2] = *reinterpret_cast<const uint32_t *>(&p0);
                zrow[16 * hf + i / 2 + 1] = *reinterpret_cast<const uint32_t *>(&p1);
            }
            pack_row<32>(S.x(), tid, 4 * hf, y);
        }
    }
    tc::fence_async_smem();
    tc::fence_before_sync();
    __syncthreads();                         // A is dead, Y is complete, Mt has been read
    // Z leaves through shared memory (over A) and one bulk copy; then the chunk's K tile
    // comes back into the same bytes (an L2 hit), the B operand of Y K.
    if (ok) {
#pragma unroll
        for (int cc = 0; cc < 8; ++cc)
            *reinterpret_cast<uint4 *>(S.buf + tc::swz(tid, cc)) =
                make_uint4(zrow[4 * cc], zrow[4 * cc + 1], zrow[4 * cc + 2], zrow[4 * cc + 3]);
    }
    tc::fence_async_smem();
    __syncthreads();
    if (ok && tid == 0) {
        tc::bulk_store(wtile + kZOff, S.buf, kXTile);
        tc::bulk_commit();
        tc::bulk_wait_read<0>();
        tc::mbar_expect_tx(&S.bar_tma, 16384);
        tc::tma_load_3d(S.buf + 0, &maps.k, &S.bar_tma, 0, hk, t0);
        tc::tma_load_3d(S.buf + 8192, &maps.k, &S.bar_tma, 64, hk, t0);
    }
    if (ok) {
        float *ws_s = reinterpret_cast<float *>(wtile + kScalOff);
        const float gL = S.gam[L - 1];
        if (tid < 64) {
            ws_s[r] = S.bet[r];
            ws_s[64 + r] = r < L ? __expf(gL - S.gam[r]) * S.nk[r] : 0.f;
        } else if (tid == 64) {
            ws_s[128] = __expf(gL);
        }
    }
    if (ok) ok = wait_all(&S.bar_tma, 1);
    // W = diag(a) K + (Lo a) K and Q' = diag(e^gamma nq) Q - (Mt a) K in two 64-column
    // halves of the dk columns: D[128 x 64] = Y[128 x 64 tokens] * K[64 tokens x 64]
    // (B = one 64-column block of the K tile, MN-major), then this thread's row of the
    // half, from registers to the workspace tile.
    const float rs = tid < 64 ? S.a[r] : __expf(S.gam[r]) * S.nq[r];
    uint32_t wq[2][32];                      // this thread's [W ; Q'] row, packed bf16
#pragma unroll
    for (int half = 0; half < 2; ++half) {
        if (ok && warp == 0) {
            tc::fence_after_sync();
            constexpr uint32_t id = tc::idesc_bf16(128, 64, 0, 1);
            const uint32_t yb = tc::smem_u32(S.x()), kb = tc::smem_u32(S.buf + half * 8192);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
                tc::mma_bf16_warp(tmem, tc::sdesc(yb + ks * 32, 16, 1024),
                                  tc::sdesc(kb + ks * 2048, 8192, 1024), id, ks > 0);
            tc::mma_commit_warp(&S.bar_mma);
        }
        if (ok) ok = wait_all(&S.bar_mma, half & 1);
        if (ok) {
            tc::fence_after_sync();
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                float dv[32], raw[16];
                tc::tmem_ld32(tmem + lane_off + 32 * j, *reinterpret_cast<float (*)[32]>(dv));
                tc::tmem_ld16(tmem + lane_off + 64 + 32 * half + 16 * j, raw);
                tc::tmem_wait_ld();
#pragma unroll
                for (int w = 0; w < 16; ++w) {
                    const float2 f = __bfloat1622float2(
                        *reinterpret_cast<const __nv_bfloat162 *>(&raw[w]));
                    const float2 d2 = make_float2(dv[2 * w], dv[2 * w + 1]);
                    const float2 x = fma2(make_float2(rs, rs), f,
                                          tid < 64 ? d2 : make_float2(-d2.x, -d2.y));
                    const __nv_bfloat162 p2 = __floats2bfloat162_rn(x.x, x.y);
                    wq[half][16 * j + w] = *reinterpret_cast<const uint32_t *>(&p2);
                }
            }
        }
        tc::fence_before_sync();
        __syncthreads();                     // this half's columns are read: TMEM free again
    }
    // Y and the K tile are dead: stage [W ; Q'] over them and send it in one bulk copy
    if (ok) {
#pragma unroll
        for (int half = 0; half < 2; ++half)
#pragma unroll
            for (int cc = 0; cc < 8; ++cc)
                *reinterpret_cast<uint4 *>(S.buf + half * 16384 + tc::swz(tid, cc)) =
                    make_uint4(wq[half][4 * cc], wq[half][4 * cc + 1], wq[half][4 * cc + 2],
                               wq[half][4 * cc + 3]);
    }
    tc::fence_async_smem();
    __syncthreads();
    if (ok && tid == 0) {
        tc::bulk_store(wtile, S.buf, kWQBytes);
        tc::bulk_commit();
    }
    if (tid == 0) tc::bulk_wait_all();      // the Z and [W ; Q'] copies have completed
    if (!ok && tid == 0) report(p.status, GDN_ERR_TIMEOUT);
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tmem, 128);
}

// =============================================================== chunk_state kernel

constexpr uint32_t kWsStage = (kWsTile + 1023) & ~1023u;  // workspace tile, 1024-aligned

struct StateSmem {
    uint8_t ws[2][kWsStage]; // [W ; Q'], Z and the scalars, per stage
    uint8_t k[2][16384];     // K tile [64 tokens][128 dk] as two 64-column blocks
    uint8_t v[2][8192];      // V tile [64 tokens][64 dv] per stage
    uint8_t hb[16384];       // bf16 h  [128 dk rows][64 dv]  (MN-major B)
    uint8_t dvh[8192];       // bf16 hi of diag(d) Vn
    uint8_t dvl[8192];       // bf16 lo
    uint8_t ob[2][8192];     // bf16 O tile [64 tokens][64 dv] per stage, stored by TMA
    uint64_t bar_ws[2];      // [W ; Q'] and Z of a stage have landed
    uint64_t bar_kv[2];      // K, V and the scalars of a stage have landed
    uint64_t bar_d1, bar_d3, bar_fin;
    uint32_t tmem;
    int abort;               // set by the first thread whose wait runs out
};
static_assert(offsetof(StateSmem, dvl) == offsetof(StateSmem, dvh) + 8192,
              "the [hi | lo] operand is one MN-major tile with a 8192-byte block stride");

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

__device__ __forceinline__ void bulk_load(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 :: "r"(tc::smem_u32(dst)), "l"(src), "r"(bytes), "r"(tc::smem_u32(bar)) : "memory");
}

// A stage's loads come in two groups with their own barriers: the [W ; Q'] and Z tiles
// (read only by MMAs, dead once the chunk's W h product completes), and the K and V tiles
// with the per-token scalars (read until the chunk's state update and by the compute
// warps).
__device__ __forceinline__ void issue_ws_loads(StateSmem &S, const TcParams &p, int stage,
                                               int hv, int slot) {
    uint64_t *bar = &S.bar_ws[stage];
    tc::mbar_expect_tx(bar, kScalOff);
    bulk_load(S.ws[stage], p.ws + ((size_t)slot * p.Hv + hv) * kWsTile, kScalOff, bar);
}
__device__ __forceinline__ void issue_kv_loads(StateSmem &S, const TcMaps &maps,
                                               const TcParams &p, int stage, int t0, int hk,
                                               int hv, int j0, int slot) {
    uint64_t *bar = &S.bar_kv[stage];
    tc::mbar_expect_tx(bar, 16384 + 8192 + kScalBytes);
    tc::tma_load_3d(S.k[stage] + 0, &maps.k, bar, 0, hk, t0);
    tc::tma_load_3d(S.k[stage] + 8192, &maps.k, bar, 64, hk, t0);
    tc::tma_load_3d(S.v[stage], &maps.v, bar, j0, hv, t0);
    bulk_load(S.ws[stage] + kScalOff, p.ws + ((size_t)slot * p.Hv + hv) * kWsTile + kScalOff,
              kScalBytes, bar);
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
// or 32).  Warp 8 issues every MMA and warp 9 every TMA and bulk load, so no compute warp
// ever stalls behind an issue queue; warps 0..7 hold the fp32 state rows and do the
// elementwise work.
// Operand tiles are 64 columns wide in shared memory whatever NT is; an NT-wide MMA reads
// only the first NT columns.  [hi | lo] is one 2 NT-wide MN-major operand whose 64-column
// blocks are S.dvh and S.dvl.
//
// TMEM columns: the chunk accumulator D, double-buffered at 0 and 64 so that the next
// chunk's Z V can be issued while the current D is still being read, and the state update
// [K^T hi | K^T lo] at 128.
template <int NT>
__device__ __forceinline__ void state_cta(StateSmem &S, const TcMaps &maps, const TcParams &p,
                                          const CUtensorMap *omap, int j0, int hv, int n) {
    constexpr int NC = NT / 2;               // columns per thread
    constexpr int NCH = NC / 8;              // 16-byte chunks per thread row
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int hk = hv / (p.Hv / p.Hk);
    const int start = p.cu[n], len = p.cu[n + 1] - start;
    const int nch = (len + kC - 1) / kC;
    const int s0 = slot0(p.cu, n);
    const size_t hoff = ((size_t)n * p.Hv + hv) * kD * kD;
    const uint32_t tmem = S.tmem;
    const uint32_t colS = 128;
    volatile int *abort = &S.abort;

    if (warp == kIssuerWarp) {
        // ------------------------------------------------------------ issuer warp
        // Lane 0 does the bounded waits; the whole warp then issues each MMA group in
        // converged code (one elected lane issues), which keeps the descriptors in uniform
        // registers.  Shared-memory descriptors are built once; a byte offset o is added as
        // o >> 4.  Stage b of a double buffer sits b * (buffer bytes) after stage 0.
        const uint64_t dWQ0 = tc::sdesc(tc::smem_u32(S.ws[0]), 16, 1024);          // K-major
        const uint64_t dZ0 = tc::sdesc(tc::smem_u32(S.ws[0] + kZOff), 16, 1024);   // K-major
        const uint64_t dKt0 = tc::sdesc(tc::smem_u32(S.k[0]), 8192, 1024);         // K^T, MN-major
        const uint64_t dV0 = tc::sdesc(tc::smem_u32(S.v[0]), 8192, 1024);          // MN-major
        const uint64_t dH = tc::sdesc(tc::smem_u32(S.hb), 8192, 1024);
        const uint64_t dVhl = tc::sdesc(tc::smem_u32(S.dvh), 8192, 1024);
        constexpr uint32_t id1 = tc::idesc_bf16(128, NT, 0, 1);
        constexpr uint32_t id3 = tc::idesc_bf16(128, 2 * NT, 1, 1);
        const bool leader = lane == 0;
        bool ok = true;   // meaningful in lane 0
        // lane 0's verdict, broadcast: go on issuing unless a wait ran out
        auto go = [&]() { return __shfl_sync(0xffffffffu, (ok && !*abort) ? 1 : 0, 0) != 0; };
        // D = Z V of chunk c into its stage's accumulator, once the chunk's tiles landed.
        // It needs nothing of the chain: chunk c's is issued right after chunk c-1's state
        // update, so it runs while the compute warps fold that update.
        auto issue_zv = [&](int c) {
            const int st = c & 1;
            if (leader) {
                if (ok) ok = wait_one(&S.bar_ws[st], (c >> 1) & 1, abort);
                if (ok) ok = wait_one(&S.bar_kv[st], (c >> 1) & 1, abort);
            }
            if (go()) {
                tc::fence_after_sync();
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    tc::mma_bf16_warp(tmem + 64 * st, dZ0 + ((st * kWsStage + ks * 32) >> 4),
                                      dV0 + ((st * 8192 + ks * 2048) >> 4), id1, ks > 0);
            }
            __syncwarp();
        };
        if (nch > 0) issue_zv(0);
        for (int c = 0; c < nch; ++c) {
            const int st = c & 1;
            const uint32_t colD = 64 * st;
            __syncthreads();                                   // h published as bf16
            if (go()) {
                tc::fence_after_sync();
                // D += [W ; Q'] h
#pragma unroll
                for (int ks = 0; ks < 8; ++ks)
                    tc::mma_bf16_warp(tmem + colD,
                                      dWQ0 + ((st * kWsStage + (ks >> 2) * 16384 + (ks & 3) * 32) >> 4),
                                      dH + ((ks * 2048) >> 4), id1, 1);
                tc::mma_commit_warp(&S.bar_d1);
            }
            __syncwarp();
            chain_barrier();                                   // hi | lo of d Vn ready
            if (go()) {
                // K^T [hi | lo]: both halves of the update in one pass, summed in fp32 later
                tc::fence_after_sync();
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    tc::mma_bf16_warp(tmem + colS, dKt0 + ((st * 16384 + ks * 2048) >> 4),
                                      dVhl + ((ks * 2048) >> 4), id3, ks > 0);
                tc::mma_commit_warp(&S.bar_d3);
            }
            __syncwarp();
            // The next chunk's accumulator (stage st^1) was last read in chunk c-1, whose
            // readers all passed this chunk's first barrier.
            if (c + 1 < nch) issue_zv(c + 1);
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
        // Chunks 0 and 1 are loaded up front; chunk c+2 goes into stage c&1 after chunk c.
        //  * Its [W ; Q'] and Z tiles leave as soon as chunk c's W h product completes: only
        //    that product and the Z V before it read them.
        //  * Its K, V and scalars leave after the barrier that publishes h for chunk c+1: by
        //    then every compute warp has finished its reads of stage c&1 and waited for
        //    chunk c's state update, the last MMA that reads K.
        // The loads thus leave one to one and a half chunks ahead, on a warp of their own
        // (issuing them costs the MMA issuer no time).
        const bool leader = lane == 0;
        int ws_issued = 0, kv_issued = 0;                      // chunks 0..n-1 are loaded
        if (leader) {
            for (int c = 0; c < 2 && c < nch; ++c) {
                issue_ws_loads(S, p, c, hv, s0 + c);
                issue_kv_loads(S, maps, p, c, start + c * kC, hk, hv, j0, s0 + c);
                ws_issued = kv_issued = c + 1;
            }
        }
        for (int c = 0; c < nch; ++c) {
            __syncwarp();
            __syncthreads();                                   // h published as bf16
            if (leader && c >= 1 && c + 1 < nch && !*abort) {
                issue_kv_loads(S, maps, p, (c + 1) & 1, start + (c + 1) * kC, hk, hv, j0,
                               s0 + c + 1);
                kv_issued = c + 2;
            }
            if (leader && c + 2 < nch && !*abort && wait_one(&S.bar_d1, c & 1, abort)) {
                issue_ws_loads(S, p, c & 1, hv, s0 + c + 2);
                ws_issued = c + 3;
            }
        }
        if (leader) {
            // wait (bounded) for the last load into each stage before the CTA may exit
            for (int s = 0; s < 2; ++s) {
                int last = ws_issued - 1 - ((ws_issued - 1 - s) & 1);   // last chunk into stage s
                if (last >= 0) wait_bounded(&S.bar_ws[s], (last >> 1) & 1);
                last = kv_issued - 1 - ((kv_issued - 1 - s) & 1);
                if (last >= 0) wait_bounded(&S.bar_kv[s], (last >> 1) & 1);
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
    if (p.h0) {
        const float4 *src = reinterpret_cast<const float4 *>(p.h0 + hoff + (size_t)row * kD + j0 + ch);
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
    float aL_prev = 1.f;   // e^{gamma_L} of the previous chunk
    for (int c = 0; c < nch; ++c) {
        const int st = c & 1;
        const uint32_t ph = c & 1;
        const int t0 = start + c * kC;
        const int L = min(kC, len - c * kC);
        const uint32_t colD = 64 * st;

        // --- A: fold the previous chunk's update into h, publish the bf16 copy.  This
        // chunk's tiles were requested a chunk ago: waiting for them here overlaps the
        // barrier query with the previous update's MMAs instead of following the barrier.
        if (ok) ok = wait_one(&S.bar_kv[st], (c >> 1) & 1, abort);
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
        const float *sc = reinterpret_cast<const float *>(S.ws[st] + kScalOff);
        const float aL = sc[128];

        // --- B: D = Z V + [W ; Q'] h
        if (ok) ok = wait_one(&S.bar_d1, ph, abort);
        float d1[NC];
        if (ok) {
            tc::fence_after_sync();
            tmem_cols<NC>(tmem + lane_off + colD + ch, d1);
        } else {
#pragma unroll
            for (int j = 0; j < NC; ++j) d1[j] = 0.f;
        }
        if (chain) {
            // Vn = beta V - D on the chain rows, then d Vn as bf16 hi + lo
            // x = d (beta V - D), formed as (-d) (D - beta V) two columns at a time: the
            // same roundings as d * fma(beta, v, -D) (negation is exact)
            const bool live = r < L;
            const float2 nb = make_float2(-sc[r], -sc[r]);
            const float2 nd = make_float2(-sc[64 + r], -sc[64 + r]);
            float x[NC];
            if (live) {
#pragma unroll
                for (int cc = 0; cc < NCH; ++cc) {
                    const uint4 u = *reinterpret_cast<const uint4 *>(S.v[st] + tc::swz(r, c0 + cc));
                    const uint32_t uw[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int i = 8 * cc + 2 * e;
                        const float2 v2 = make_float2(__uint_as_float(uw[e] << 16),
                                                      __uint_as_float(uw[e] & 0xffff0000u));
                        const float2 t = fma2(nb, v2, make_float2(d1[i], d1[i + 1]));
                        const float2 xx = mul2(nd, t);
                        x[i] = xx.x;
                        x[i + 1] = xx.y;
                    }
                }
            } else {
#pragma unroll
                for (int i = 0; i < NC; ++i) x[i] = 0.f;
            }
            // hi = bf16(x) two at a time (the paired conversion issues at several times
            // the rate of the single one); lo = x - hi is exact in fp32
            uint32_t hp[NC / 2];
            float lo[NC];
            const float2 m1 = make_float2(-1.f, -1.f);
#pragma unroll
            for (int jj = 0; jj < NC / 2; ++jj) {
                const __nv_bfloat162 hb2 = __floats2bfloat162_rn(x[2 * jj], x[2 * jj + 1]);
                hp[jj] = *reinterpret_cast<const uint32_t *>(&hb2);
                const float2 l2 = fma2(m1, make_float2(__uint_as_float(hp[jj] << 16),
                                                       __uint_as_float(hp[jj] & 0xffff0000u)),
                                       make_float2(x[2 * jj], x[2 * jj + 1]));
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
        } else if (L == kC) {
            // O = scale D on the output rows.  A full chunk's O tile goes out through shared
            // memory with one tensor store, keeping 64 scattered row writes per warp off the
            // load/store pipeline that the chain warps' shared-memory traffic shares.  Stage
            // st was last stored two chunks ago; allowing one group in flight covers the
            // previous chunk.  A 64-wide tile uses the 128B-swizzled layout, narrower ones
            // plain rows.
            uint8_t *ob = S.ob[st];
            if (tid == kOutLeader) tc::bulk_wait_read<1>();
            out_barrier();
#pragma unroll
            for (int cc = 0; cc < NCH; ++cc) {
                float f[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) f[e] = p.scale * d1[8 * cc + e];
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
                for (int e = 0; e < 8; ++e) f[e] = p.scale * d1[8 * cc + e];
                dst[cc] = pack8(f);
            }
        }
        tc::fence_before_sync();
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
    if (!*abort && p.hT) {
        float4 *dst = reinterpret_cast<float4 *>(p.hT + hoff + (size_t)row * kD + j0 + ch);
#pragma unroll
        for (int i = 0; i < NC / 4; ++i)
            dst[i] = make_float4(h[4 * i], h[4 * i + 1], h[4 * i + 2], h[4 * i + 3]);
    }
    if (*abort && tid == 0) report(p.status, GDN_ERR_TIMEOUT);
    if (warp == 0) tc::tmem_dealloc(tmem, 256);
}

// One CTA per (sequence, v-head, dv tile).  The tiles of a head are either two of 64
// columns or, when that leaves SMs idle (p.ntiles == 3), 48 + 48 + 32 columns.
__global__ void __launch_bounds__(kStateThreads, 1)
chunk_state_kernel(const __grid_constant__ TcMaps maps, const __grid_constant__ TcParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    StateSmem &S = *reinterpret_cast<StateSmem *>(
        (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023));
    grid_dependents_launch();
    const int tid = threadIdx.x, warp = tid >> 5;
    const int jt = blockIdx.x, hv = blockIdx.y, n = blockIdx.z;
    // TMEM, barriers and tensor-map prefetches touch no memory of the previous kernel, so
    // they run before the dependency wait below
    if (warp == 0) {
        tc::tmem_alloc(&S.tmem, 256);
        tc::tmem_relinquish();
    }
    if (tid == 0) {
        tc::mbar_init(&S.bar_ws[0], 1);
        tc::mbar_init(&S.bar_ws[1], 1);
        tc::mbar_init(&S.bar_kv[0], 1);
        tc::mbar_init(&S.bar_kv[1], 1);
        tc::mbar_init(&S.bar_d1, 1);
        tc::mbar_init(&S.bar_d3, 1);
        tc::mbar_init(&S.bar_fin, 1);
        S.abort = 0;
        tc::mbar_fence_init();
        tc::prefetch_tmap(&maps.k);
        tc::prefetch_tmap(&maps.v);
        tc::prefetch_tmap(p.ntiles == 3 ? (jt < 2 ? &maps.o48 : &maps.o32) : &maps.o);
    }
    grid_dependency_wait();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if (p.ntiles != 3)
        state_cta<64>(S, maps, p, &maps.o, 64 * jt, hv, n);
    else if (jt < 2)
        state_cta<48>(S, maps, p, &maps.o48, 48 * jt, hv, n);
    else
        state_cta<32>(S, maps, p, &maps.o32, 96, hv, n);
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

gdn_status_t launch_chunk_tc(const ScanArgs &a, const int32_t *cu_host, cudaStream_t st,
                             cudaEvent_t before_state) {
    (void)cu_host;
    if (a.N == 0) return GDN_OK;
    if (a.out_f32) return GDN_ERR_DTYPE;
    gdn::TcMaps maps;
    if (!make_map(&maps.q, a.q, a.T, a.Hk, a.q_tok) || !make_map(&maps.k, a.k, a.T, a.Hk, a.k_tok) ||
        !make_map(&maps.v, a.v, a.T, a.Hv, a.v_tok) || !make_map(&maps.o, a.o, a.T, a.Hv, a.o_tok) ||
        !make_map(&maps.o48, a.o, a.T, a.Hv, a.o_tok, 48) ||
        !make_map(&maps.o32, a.o, a.T, a.Hv, a.o_tok, 32))
        return GDN_ERR_CUDA;
    gdn::TcParams p;
    p.g = a.g;
    p.beta = a.beta;
    p.cu = a.cu;
    p.h0 = a.h0;
    p.hT = a.hT;
    p.o = (gdn::bf16 *)a.o;
    p.o_tok = a.o_tok;
    p.q = (const gdn::bf16 *)a.q;
    p.q_tok = a.q_tok;
    p.ws = (uint8_t *)a.ws;
    p.N = a.N;
    p.Hk = a.Hk;
    p.Hv = a.Hv;
    p.scale = a.scale;
    p.l2norm = (a.flags & GDN_QK_L2NORM) ? 1 : 0;
    p.status = a.status;
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
        p.ntiles = (sms > 0 && (int64_t)3 * a.Hv * a.N <= sms) ? 3 : 2;

    const size_t prep_smem = sizeof(gdn::PrepSmem) + 1024;
    const size_t state_smem = sizeof(gdn::StateSmem) + 1024;
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
                                 (int)state_smem) != cudaSuccess)
            return GDN_ERR_CUDA;
        attr_set[dev].store(true, std::memory_order_release);
    }
    const int64_t slots64 = (a.T + gdn::kC - 1) / gdn::kC + a.N;
    if (slots64 > 65535) return GDN_ERR_SHAPE;   // chunk slots index the grid's y dimension
    const int slots = (int)slots64;
    if (slots > 0) {
        dim3 g1(a.Hv, slots);
        if (launch_dependent(gdn::chunk_prep_kernel, g1, dim3(gdn::kPrepThreads), prep_smem, st,
                             maps, p) != cudaSuccess)
            return GDN_ERR_CUDA;
    }
    if (before_state && cudaStreamWaitEvent(st, before_state, 0) != cudaSuccess)
        return GDN_ERR_CUDA;
    dim3 g2(p.ntiles, a.Hv, a.N);
    if (launch_dependent(gdn::chunk_state_kernel, g2, dim3(gdn::kStateThreads), state_smem, st,
                         maps, p) != cudaSuccess)
        return GDN_ERR_CUDA;
    return GDN_OK;
}

}  // namespace gdn_host
