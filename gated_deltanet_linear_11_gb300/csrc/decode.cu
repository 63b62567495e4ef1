// decode.cu -- one-token gated delta rule step on a pool of fp32 states.
//
// Source: decode path of "[Feature] Add batch invariance support to GDN_ATTN backend -
// #45819" (per-sequence state update through ssm_state_indices into the state pool) with
// the fp32 recurrent state of Birol's comment, part 1, and the recurrence of "Qwen3.5-27B
// GPTQ Garbage Inference -- Root Cause Analysis", "Why abliteration failed", item 3.
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

namespace gdn {

constexpr int kDecThreads = 256;
constexpr int kDecD = 128;
constexpr int kDecRowsPerThread = kDecD / (kDecThreads / 32);  // 16

template <typename Tin, typename Tout>
__global__ void __launch_bounds__(kDecThreads, 2)
recurrent_decode_kernel(const Tin *__restrict__ q, const Tin *__restrict__ k,
                        const Tin *__restrict__ v, Tout *__restrict__ o, int64_t q_tok,
                        int64_t k_tok, int64_t v_tok, int64_t o_tok,
                        const float *__restrict__ g, const float *__restrict__ beta,
                        float *__restrict__ state, int P, const int32_t *__restrict__ idx,
                        int Hk, int Hv, float scale, int l2norm, int32_t *status) {
    __shared__ float sq[kDecD], sk[kDecD], sv[kDecD], su[kDecD];
    __shared__ float red[2][kDecThreads / 32][kDecD];
    __shared__ float sscal[4];

    const int hv = blockIdx.x;
    const int n = blockIdx.y;
    const int tid = threadIdx.x;
    const int cg = tid & 31;
    const int rg = tid >> 5;
    const int slot = idx ? idx[n] : n;
    if (slot < 0 || slot >= P) {
        if (tid == 0) report(status, GDN_ERR_INDEX);
        return;
    }
    const int hk = hv / (Hv / Hk);

    // Issue the state loads first: they are the HBM traffic.
    float4 *tile = reinterpret_cast<float4 *>(state + ((size_t)slot * Hv + hv) * kDecD * kDecD);
    float4 H[kDecRowsPerThread];
#pragma unroll
    for (int r = 0; r < kDecRowsPerThread; ++r)
        H[r] = tile[(size_t)(rg * kDecRowsPerThread + r) * (kDecD / 4) + cg];

    if (tid < kDecD) {
        sq[tid] = to_f32(q[(size_t)n * q_tok + (size_t)hk * kDecD + tid]);
        sk[tid] = to_f32(k[(size_t)n * k_tok + (size_t)hk * kDecD + tid]);
        sv[tid] = to_f32(v[(size_t)n * v_tok + (size_t)hv * kDecD + tid]);
    }
    __syncthreads();
    // Warp 0: |q|^2, |k|^2, k.q in a fixed order (lane-strided partials, xor tree).
    if (rg == 0) {
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
    __syncthreads();
    const float nq = sscal[0], nk = sscal[1], kq = sscal[2];

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
    const float a = expf(g[(size_t)n * Hv + hv]);
    const float b = beta[(size_t)n * Hv + hv];
    __syncthreads();
    if (tid < kDecD) {
        float hkj = 0.f, hqj = 0.f;
#pragma unroll
        for (int r = 0; r < kDecThreads / 32; ++r) {
            hkj += red[0][r][tid];
            hqj += red[1][r][tid];
        }
        const float u = b * (sv[tid] - a * hkj);
        su[tid] = u;
        o[(size_t)n * o_tok + (size_t)hv * kDecD + tid] = from_f32<Tout>(scale * fmaf(u, kq, a * hqj));
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

}  // namespace gdn_host
