// decode.cu -- one-token gated delta rule step on a pool of fp32 states, and the fused
// decode step (conv update + gating + recurrent step in one kernel).
//
// Source: decode path of "[Feature] Add batch invariance support to GDN_ATTN backend -
// #45819" (per-sequence state update through ssm_state_indices into the state pool, and
// the fused_sigmoid_gating_delta_rule_update decode entry) with the fp32 recurrent state
// of Birol's comment, part 1, and the recurrence of "Qwen3.5-27B GPTQ Garbage Inference --
// Root Cause Analysis", "Why abliteration failed", item 3.
//
// Per (sequence n, v-head h) with state tile H[i][j] = S[j][i] (dk x dv, fp32):
//     hk = H^T k,  hq = H^T q          (one pass over H, both dots at once)
//     u  = beta (v - e^g hk)
//     o  = scale (e^g hq + u (k.q))    (= scale * S_t q_t with S_t the updated state)
//     H <- e^g H + k u^T               (written back from registers: H read once, written once)
//
// The kernel is HBM-bound (64 KiB read + 64 KiB written per (n, h) against ~1 KiB of
// activations).  One CTA of 256 threads owns one (n, h): thread t holds columns
// 4*(t%32)..+3 of rows 16*(t/32)..+15 as 16 float4 registers, so every warp load is one
// 512-byte state row.  The column reduction over the 8 row groups goes through shared
// memory in a fixed order, so results do not depend on the batch.
#include "common.cuh"
#include "conv_taps.cuh"

namespace gdn {

constexpr int kDecThreads = 256;
constexpr int kDecD = 128;
constexpr int kDecRowsPerThread = kDecD / (kDecThreads / 32);  // 16
constexpr int kDecGroups = kDecThreads / 32;                   // row groups

__device__ __forceinline__ void load_state_tile(float4 (&H)[kDecRowsPerThread], const float4 *tile) {
    const int cg = threadIdx.x & 31, rg = threadIdx.x >> 5;
#pragma unroll
    for (int r = 0; r < kDecRowsPerThread; ++r)
        H[r] = tile[(size_t)(rg * kDecRowsPerThread + r) * (kDecD / 4) + cg];
}

// Norm factors and k.q of one (q, k) pair held in shared memory, by warp 0 in a fixed
// order (lane-strided partials, xor tree); the caller synchronises before and after.
__device__ __forceinline__ void qk_scalars(const float *sq, const float *sk, int l2norm,
                                           float *sscal) {
    const int cg = threadIdx.x & 31;
    if ((threadIdx.x >> 5) == 0) {
        float a = 0.f, b = 0.f, c = 0.f;
#pragma unroll
        for (int i = 0; i < kDecD / 32; ++i) {
            const float qi = sq[cg + 32 * i], ki = sk[cg + 32 * i];
            a = fmaf(qi, qi, a);
            b = fmaf(ki, ki, b);
            c = fmaf(ki, qi, c);
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            a += __shfl_xor_sync(0xffffffffu, a, off);
            b += __shfl_xor_sync(0xffffffffu, b, off);
            c += __shfl_xor_sync(0xffffffffu, c, off);
        }
        if (cg == 0) {
            float nq = 1.f, nk = 1.f;
            if (l2norm) {
                nq = rsqrtf(a + 1e-6f);
                nk = rsqrtf(b + 1e-6f);
            }
            sscal[0] = nq;
            sscal[1] = nk;
            sscal[2] = c * nq * nk;  // k.q after normalisation
        }
    }
}

// One head's step given its state tile in registers: decay a = e^g, beta b.  Contains
// barriers: every thread of the CTA calls it.  Writes o[0..127] and the new tile.
template <typename Tout>
__device__ __forceinline__ void decode_head(float4 (&H)[kDecRowsPerThread], float4 *tile,
                                            const float *sq, const float *sk, const float *sv,
                                            float *su, float (*red)[kDecGroups][kDecD],
                                            float nq, float nk, float kq, float a, float b,
                                            float scale, Tout *orow) {
    const int tid = threadIdx.x, cg = tid & 31, rg = tid >> 5;
    // Partial column dots over this thread's 16 rows.
    float pk[4] = {0.f, 0.f, 0.f, 0.f}, pq[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int r = 0; r < kDecRowsPerThread; ++r) {
        const int i = rg * kDecRowsPerThread + r;
        const float ki = sk[i] * nk, qi = sq[i] * nq;
        pk[0] = fmaf(H[r].x, ki, pk[0]); pq[0] = fmaf(H[r].x, qi, pq[0]);
        pk[1] = fmaf(H[r].y, ki, pk[1]); pq[1] = fmaf(H[r].y, qi, pq[1]);
        pk[2] = fmaf(H[r].z, ki, pk[2]); pq[2] = fmaf(H[r].z, qi, pq[2]);
        pk[3] = fmaf(H[r].w, ki, pk[3]); pq[3] = fmaf(H[r].w, qi, pq[3]);
    }
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        red[0][rg][4 * cg + c] = pk[c];
        red[1][rg][4 * cg + c] = pq[c];
    }
    __syncthreads();
    if (tid < kDecD) {
        float hkj = 0.f, hqj = 0.f;
#pragma unroll
        for (int r = 0; r < kDecGroups; ++r) {
            hkj += red[0][r][tid];
            hqj += red[1][r][tid];
        }
        const float u = b * (sv[tid] - a * hkj);
        su[tid] = u;
        orow[tid] = from_f32<Tout>(scale * fmaf(u, kq, a * hqj));
    }
    __syncthreads();
    const float4 u4 = reinterpret_cast<const float4 *>(su)[cg];
#pragma unroll
    for (int r = 0; r < kDecRowsPerThread; ++r) {
        const int i = rg * kDecRowsPerThread + r;
        const float ki = sk[i] * nk;
        float4 h = H[r];
        h.x = fmaf(a, h.x, ki * u4.x);
        h.y = fmaf(a, h.y, ki * u4.y);
        h.z = fmaf(a, h.z, ki * u4.z);
        h.w = fmaf(a, h.w, ki * u4.w);
        tile[(size_t)i * (kDecD / 4) + cg] = h;
    }
}

template <typename Tin, typename Tout>
__global__ void __launch_bounds__(kDecThreads, 2)
recurrent_decode_kernel(const Tin *__restrict__ q, const Tin *__restrict__ k,
                        const Tin *__restrict__ v, Tout *__restrict__ o, int64_t q_tok,
                        int64_t k_tok, int64_t v_tok, int64_t o_tok,
                        const float *__restrict__ g, const float *__restrict__ beta,
                        float *__restrict__ state, int P, const int32_t *__restrict__ idx,
                        int Hk, int Hv, float scale, int l2norm, int32_t *status) {
    __shared__ float sq[kDecD], sk[kDecD], sv[kDecD], su[kDecD];
    __shared__ float red[2][kDecGroups][kDecD];
    __shared__ float sscal[4];

    const int hv = blockIdx.x;
    const int n = blockIdx.y;
    const int tid = threadIdx.x;
    const int slot = idx ? idx[n] : n;
    if (slot < 0 || slot >= P) {
        if (tid == 0) report(status, GDN_ERR_INDEX);
        return;
    }
    const int hk = hv / (Hv / Hk);

    // Issue the state loads first: they are the HBM traffic.
    float4 *tile = reinterpret_cast<float4 *>(state + ((size_t)slot * Hv + hv) * kDecD * kDecD);
    float4 H[kDecRowsPerThread];
    load_state_tile(H, tile);
    const float g_n = g[(size_t)n * Hv + hv], b = beta[(size_t)n * Hv + hv];

    if (tid < kDecD) {
        sq[tid] = to_f32(q[(size_t)n * q_tok + (size_t)hk * kDecD + tid]);
        sk[tid] = to_f32(k[(size_t)n * k_tok + (size_t)hk * kDecD + tid]);
        sv[tid] = to_f32(v[(size_t)n * v_tok + (size_t)hv * kDecD + tid]);
    }
    __syncthreads();
    qk_scalars(sq, sk, l2norm, sscal);
    __syncthreads();
    decode_head(H, tile, sq, sk, sv, su, red, sscal[0], sscal[1], sscal[2], expf(g_n), b,
                scale, o + (size_t)n * o_tok + (size_t)hv * kDecD);
}

// Fused decode step for one (sequence n, v-head hv), the recurrent kernel's unit: the
// conv of the channels this head reads (q and k of its k-head hk = hv / G, v of hv), the
// gates, and the recurrent step.  The gates come as raw logits:
//     beta = sigmoid(b_raw),   g = -softplus(a_raw),  so  e^g = 1 / (1 + e^{a_raw}).
// The conv output is rounded to bf16 exactly as the conv kernels store it, then used in
// fp32 like the unfused path's q/k/v.  The state tile is loaded first, so the HBM traffic
// starts before the conv.
// The conv state is shifted in place.  Each CTA shifts the rows of its own v channels;
// the q and k channels are read by the G CTAs of a k-head, so their rows are shifted by
// conv_shift_qk_kernel, launched after this kernel on the same stream.
__global__ void __launch_bounds__(kDecThreads, 2)
fused_decode_kernel(const bf16 *__restrict__ x, int C, const bf16 *__restrict__ w,
                    const bf16 *__restrict__ bias, bf16 *conv_state,
                    const float *__restrict__ a_raw, const float *__restrict__ b_raw,
                    float *__restrict__ state, int P, const int32_t *__restrict__ idx,
                    bf16 *__restrict__ o, int Hk, int Hv, float scale, int l2norm,
                    int32_t *status) {
    __shared__ float sq[kDecD], sk[kDecD], sv[kDecD], su[kDecD];
    __shared__ float red[2][kDecGroups][kDecD];
    __shared__ float sscal[4];
    const int hv = blockIdx.x, n = blockIdx.y, tid = threadIdx.x;
    const int slot = idx ? idx[n] : n;
    if (slot < 0 || slot >= P) {
        if (tid == 0) report(status, GDN_ERR_INDEX);
        return;
    }
    const int hk = hv / (Hv / Hk);
    float4 *tile = reinterpret_cast<float4 *>(state + ((size_t)slot * Hv + hv) * kDecD * kDecD);
    float4 H[kDecRowsPerThread];
    load_state_tile(H, tile);
    const float ar = a_raw[(size_t)n * Hv + hv], br = b_raw[(size_t)n * Hv + hv];

    // conv of 3 x 16 groups of 8 adjacent channels: q (hk), k (hk), v (hv)
    if (tid < 3 * (kDecD / 8)) {
        const int part = tid / (kDecD / 8), sub = tid % (kDecD / 8);
        const int qk_width = Hk * kDecD;
        const int c0 = part == 0 ? hk * kDecD + 8 * sub
                     : part == 1 ? qk_width + hk * kDecD + 8 * sub
                                 : 2 * qk_width + hv * kDecD + 8 * sub;
        float *dst = (part == 0 ? sq : part == 1 ? sk : sv) + 8 * sub;
        bf16 *cs = conv_state + (size_t)slot * 3 * C + c0;
        const uint4 r0 = *reinterpret_cast<const uint4 *>(cs);
        const uint4 r1 = *reinterpret_cast<const uint4 *>(cs + C);
        const uint4 r2 = *reinterpret_cast<const uint4 *>(cs + 2 * C);
        const uint4 rx = *reinterpret_cast<const uint4 *>(x + (size_t)n * C + c0);
        Taps tp;
        load_taps(tp, w, bias, c0);
        float s0[8], s1[8], s2[8], cur[8], yv[8];
        unpack8(r0, s0);
        unpack8(r1, s1);
        unpack8(r2, s2);
        unpack8(rx, cur);
        unpack8(conv_out(tp, s0, s1, s2, cur), yv);
#pragma unroll
        for (int e = 0; e < 8; ++e) dst[e] = yv[e];
        if (part == 2) {
            *reinterpret_cast<uint4 *>(cs) = r1;
            *reinterpret_cast<uint4 *>(cs + C) = r2;
            *reinterpret_cast<uint4 *>(cs + 2 * C) = rx;
        }
    }
    __syncthreads();
    qk_scalars(sq, sk, l2norm, sscal);
    __syncthreads();
    const float a = 1.f / (1.f + expf(ar));   // e^{-softplus(a_raw)}
    const float b = 1.f / (1.f + expf(-br));  // sigmoid(b_raw)
    decode_head(H, tile, sq, sk, sv, su, red, sscal[0], sscal[1], sscal[2], a, b, scale,
                o + ((size_t)n * Hv + hv) * kDecD);
}

// The q and k channels' conv-state shift of the fused step: rows <- [row1, row2, x].
// grid: (ceil(2 Hk 128 / (8 * 256)), N)
__global__ void __launch_bounds__(kDecThreads)
conv_shift_qk_kernel(const bf16 *__restrict__ x, int C, int qk_channels, bf16 *conv_state,
                     int P, const int32_t *__restrict__ idx) {
    const int n = blockIdx.y;
    const int c0 = (blockIdx.x * kDecThreads + threadIdx.x) * 8;
    if (c0 >= qk_channels) return;
    const int slot = idx ? idx[n] : n;
    if (slot < 0 || slot >= P) return;   // reported by fused_decode_kernel
    bf16 *cs = conv_state + (size_t)slot * 3 * C + c0;
    const uint4 r1 = *reinterpret_cast<const uint4 *>(cs + C);
    const uint4 r2 = *reinterpret_cast<const uint4 *>(cs + 2 * C);
    const uint4 rx = *reinterpret_cast<const uint4 *>(x + (size_t)n * C + c0);
    *reinterpret_cast<uint4 *>(cs) = r1;
    *reinterpret_cast<uint4 *>(cs + C) = r2;
    *reinterpret_cast<uint4 *>(cs + 2 * C) = rx;
}

}  // namespace gdn

namespace gdn_host {

gdn_status_t launch_decode(const DecodeArgs &a, cudaStream_t st) {
    if (a.N == 0) return GDN_OK;
    if (a.dk != gdn::kDecD || a.dv != gdn::kDecD) return GDN_ERR_UNSUPPORTED;
    dim3 grid(a.Hv, a.N);
    const int l2 = (a.flags & GDN_QK_L2NORM) ? 1 : 0;
#define GDN_DEC(TI, TO)                                                                    \
    gdn::recurrent_decode_kernel<TI, TO><<<grid, gdn::kDecThreads, 0, st>>>(              \
        (const TI *)a.q, (const TI *)a.k, (const TI *)a.v, (TO *)a.o, a.q_tok, a.k_tok,   \
        a.v_tok, a.o_tok, a.g, a.beta, a.state, a.P, a.idx, a.Hk, a.Hv, a.scale, l2,      \
        a.status)
    if (a.in_f32 != a.out_f32) return GDN_ERR_DTYPE;
    if (!a.in_f32) GDN_DEC(gdn::bf16, gdn::bf16);
    else GDN_DEC(float, float);
#undef GDN_DEC
    return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

gdn_status_t launch_fused_decode(const FusedDecodeArgs &a, cudaStream_t st) {
    if (a.N == 0) return GDN_OK;
    gdn::fused_decode_kernel<<<dim3(a.Hv, a.N), gdn::kDecThreads, 0, st>>>(
        (const gdn::bf16 *)a.x, a.C, (const gdn::bf16 *)a.w, (const gdn::bf16 *)a.bias,
        (gdn::bf16 *)a.conv_state, a.a_raw, a.b_raw, a.state, a.P, a.idx, (gdn::bf16 *)a.o,
        a.Hk, a.Hv, a.scale, (a.flags & GDN_QK_L2NORM) ? 1 : 0, a.status);
    const int qk = 2 * a.Hk * gdn::kDecD;
    gdn::conv_shift_qk_kernel<<<dim3((qk / 8 + gdn::kDecThreads - 1) / gdn::kDecThreads, a.N),
                                gdn::kDecThreads, 0, st>>>(
        (const gdn::bf16 *)a.x, a.C, qk, (gdn::bf16 *)a.conv_state, a.P, a.idx);
    return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

}  // namespace gdn_host
