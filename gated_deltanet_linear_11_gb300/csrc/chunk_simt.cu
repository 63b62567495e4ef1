// chunk_simt.cu -- CUDA-core fp32 chunked gated delta rule (WY/UT form).
//
// Recurrence: "Qwen3.5-27B GPTQ Garbage Inference -- Root Cause Analysis", "Why
// abliteration failed on Qwen3.5", item 3.  Chunking: "[Feature] Add batch invariance
// support to GDN_ATTN backend - #45819", Birol's comment, part 3(a) -- chunks anchored at
// every sequence start, so a sequence's math never depends on the packed batch.
//
// This kernel carries every product in fp32 on the CUDA cores.  It serves the small head
// sizes and fp32 activations that the tensor-core kernel does not take, and it is the
// straightforward form the tensor-core kernel is checked against.
//
// One CTA owns one (sequence, v-head, dv tile of DVT columns) and walks the sequence's
// chunks in order.  For a chunk of L <= CH tokens with inclusive in-chunk log-decay sums
// gamma, L2-norm factors nk, nq (1 when the flag is off) and entering state h [DK][DVT]:
//   A[r][s] = beta_r e^{gamma_r - gamma_s} nk_r nk_s (k_r . k_s)       s < r
//   M[r][s] = e^{gamma_r - gamma_s} nq_r nk_s (q_r . k_s)              s <= r
//   R       = diag(beta) (V - diag(e^gamma nk) K h)
//   Vn      = (I + A)^{-1} R                    (blocked forward substitution)
//   O       = scale (diag(e^gamma nq) Q h + M Vn)
//   h      <- e^{gamma_{L-1}} h + K^T diag(e^{gamma_{L-1} - gamma} nk) Vn
// Only exponents gamma_r - gamma_s with s <= r are formed, so nothing overflows.
#include "common.cuh"

namespace gdn {

constexpr int kSimtThreads = 256;

template <int DK, int DVT, int CH>
struct SimtSmem {
    float K[CH][DK + 1];
    float Q[CH][DK + 1];
    float A[CH][CH + 1];
    float M[CH][CH + 1];
    float V[CH][DVT + 1];
    float H[DK][DVT + 1];
    float gam[CH], bet[CH], nk[CH], nq[CH], dec[CH];
};

template <typename Tin, typename Tout, int DK, int DVT, int CH>
__global__ void __launch_bounds__(kSimtThreads)
chunk_simt_kernel(const Tin *__restrict__ q, const Tin *__restrict__ k,
                  const Tin *__restrict__ v, Tout *__restrict__ o, int64_t q_tok,
                  int64_t k_tok, int64_t v_tok, int64_t o_tok, const float *__restrict__ g,
                  const float *__restrict__ beta, const int32_t *__restrict__ cu,
                  const float *h0, float *hT, int Hk, int Hv, int DV, float scale,
                  int l2norm) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    SimtSmem<DK, DVT, CH> &S = *reinterpret_cast<SimtSmem<DK, DVT, CH> *>(smem_raw);
    const int tid = threadIdx.x;
    const int j0 = blockIdx.x * DVT;
    const int hv = blockIdx.y;
    const int n = blockIdx.z;
    const int hk = hv / (Hv / Hk);
    const int start = cu[n], end = cu[n + 1];
    const size_t hoff = ((size_t)n * Hv + hv) * DK * DV;

    for (int p = tid; p < DK * DVT; p += kSimtThreads) {
        const int i = p / DVT, j = p % DVT;
        S.H[i][j] = h0 ? h0[hoff + (size_t)i * DV + j0 + j] : 0.f;
    }

    for (int c0 = start; c0 < end; c0 += CH) {
        const int L = min(CH, end - c0);
        __syncthreads();  // previous chunk fully consumed
        for (int p = tid; p < CH * DK; p += kSimtThreads) {
            const int r = p / DK, i = p % DK;
            float kv = 0.f, qv = 0.f;
            if (r < L) {
                kv = to_f32(k[(size_t)(c0 + r) * k_tok + (size_t)hk * DK + i]);
                qv = to_f32(q[(size_t)(c0 + r) * q_tok + (size_t)hk * DK + i]);
            }
            S.K[r][i] = kv;
            S.Q[r][i] = qv;
        }
        for (int p = tid; p < CH * DVT; p += kSimtThreads) {
            const int r = p / DVT, j = p % DVT;
            S.V[r][j] = r < L ? to_f32(v[(size_t)(c0 + r) * v_tok + (size_t)hv * DV + j0 + j]) : 0.f;
        }
        if (tid < CH) {
            S.gam[tid] = tid < L ? g[(size_t)(c0 + tid) * Hv + hv] : 0.f;
            S.bet[tid] = tid < L ? beta[(size_t)(c0 + tid) * Hv + hv] : 0.f;
        }
        __syncthreads();
        // L2-norm factors: one warp per row, lane-strided partials + xor tree.
        {
            const int warp = tid >> 5, lane = tid & 31;
            for (int r = warp; r < CH; r += kSimtThreads / 32) {
                float a = 0.f, b = 0.f;
                for (int i = lane; i < DK; i += 32) {
                    a = fmaf(S.K[r][i], S.K[r][i], a);
                    b = fmaf(S.Q[r][i], S.Q[r][i], b);
                }
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) {
                    a += __shfl_xor_sync(0xffffffffu, a, off);
                    b += __shfl_xor_sync(0xffffffffu, b, off);
                }
                if (lane == 0) {
                    const bool live = r < L;
                    S.nk[r] = !live ? 0.f : (l2norm ? rsqrtf(a + 1e-6f) : 1.f);
                    S.nq[r] = !live ? 0.f : (l2norm ? rsqrtf(b + 1e-6f) : 1.f);
                }
            }
        }
        // Inclusive cumulative log decay, one thread, fixed order.
        if (tid == 0) {
            float acc = 0.f;
            for (int r = 0; r < CH; ++r) {
                acc += S.gam[r];
                S.gam[r] = acc;
            }
        }
        __syncthreads();
        const float gL = S.gam[L - 1];
        if (tid < CH) S.dec[tid] = tid < L ? expf(gL - S.gam[tid]) * S.nk[tid] : 0.f;
        // A (strict lower, gated) and M (lower incl. diagonal, gated).
        for (int p = tid; p < CH * CH; p += kSimtThreads) {
            const int r = p / CH, s = p % CH;
            float a = 0.f, m = 0.f;
            if (r < L && s <= r) {
                float dkk = 0.f, dqk = 0.f;
                for (int i = 0; i < DK; ++i) {
                    dkk = fmaf(S.K[r][i], S.K[s][i], dkk);
                    dqk = fmaf(S.Q[r][i], S.K[s][i], dqk);
                }
                const float e = expf(S.gam[r] - S.gam[s]);
                if (s < r) a = S.bet[r] * e * S.nk[r] * S.nk[s] * dkk;
                m = e * S.nq[r] * S.nk[s] * dqk;
            }
            S.A[r][s] = a;
            S.M[r][s] = m;
        }
        // R = diag(beta) (V - diag(e^gamma nk) K h), in place in S.V.
        for (int p = tid; p < CH * DVT; p += kSimtThreads) {
            const int r = p / DVT, j = p % DVT;
            if (r < L) {
                float kh = 0.f;
                for (int i = 0; i < DK; ++i) kh = fmaf(S.K[r][i], S.H[i][j], kh);
                S.V[r][j] = S.bet[r] * (S.V[r][j] - expf(S.gam[r]) * S.nk[r] * kh);
            }
        }
        __syncthreads();
        // Vn = (I + A)^{-1} R by blocks of 16 rows: subtract the finished blocks in
        // parallel, then substitute inside the block (one thread per column).
        for (int b0 = 0; b0 < L; b0 += 16) {
            const int b1 = min(b0 + 16, L);
            if (b0 > 0) {
                for (int p = tid; p < 16 * DVT; p += kSimtThreads) {
                    const int r = b0 + p / DVT, j = p % DVT;
                    if (r < b1) {
                        float acc = S.V[r][j];
                        for (int s = 0; s < b0; ++s) acc = fmaf(-S.A[r][s], S.V[s][j], acc);
                        S.V[r][j] = acc;
                    }
                }
                __syncthreads();
            }
            if (tid < DVT) {
                for (int r = b0 + 1; r < b1; ++r) {
                    float acc = S.V[r][tid];
                    for (int s = b0; s < r; ++s) acc = fmaf(-S.A[r][s], S.V[s][tid], acc);
                    S.V[r][tid] = acc;
                }
            }
            __syncthreads();
        }
        // O = scale (diag(e^gamma nq) Q h + M Vn)
        for (int p = tid; p < CH * DVT; p += kSimtThreads) {
            const int r = p / DVT, j = p % DVT;
            if (r < L) {
                float qh = 0.f, mv = 0.f;
                for (int i = 0; i < DK; ++i) qh = fmaf(S.Q[r][i], S.H[i][j], qh);
                for (int s = 0; s <= r; ++s) mv = fmaf(S.M[r][s], S.V[s][j], mv);
                const float out = scale * fmaf(expf(S.gam[r]) * S.nq[r], qh, mv);
                o[(size_t)(c0 + r) * o_tok + (size_t)hv * DV + j0 + j] = from_f32<Tout>(out);
            }
        }
        __syncthreads();
        // h <- e^{gamma_L} h + K^T diag(dec) Vn
        const float aL = expf(gL);
        for (int p = tid; p < DK * DVT; p += kSimtThreads) {
            const int i = p / DVT, j = p % DVT;
            float acc = 0.f;
            for (int s = 0; s < L; ++s) acc = fmaf(S.K[s][i] * S.dec[s], S.V[s][j], acc);
            S.H[i][j] = fmaf(aL, S.H[i][j], acc);
        }
    }
    __syncthreads();
    if (hT) {
        for (int p = tid; p < DK * DVT; p += kSimtThreads) {
            const int i = p / DVT, j = p % DVT;
            hT[hoff + (size_t)i * DV + j0 + j] = S.H[i][j];
        }
    }
}

template <typename Tin, typename Tout, int DK, int DVT, int CH>
static gdn_status_t launch_simt_t(const gdn_host::ScanArgs &a, cudaStream_t st) {
    const size_t smem = sizeof(SimtSmem<DK, DVT, CH>);
    auto kern = chunk_simt_kernel<Tin, Tout, DK, DVT, CH>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
        cudaSuccess)
        return GDN_ERR_CUDA;
    dim3 grid(a.dv / DVT, a.Hv, a.N);
    kern<<<grid, kSimtThreads, smem, st>>>(
        (const Tin *)a.q, (const Tin *)a.k, (const Tin *)a.v, (Tout *)a.o, a.q_tok, a.k_tok,
        a.v_tok, a.o_tok, a.g, a.beta, a.cu, a.h0, a.hT, a.Hk, a.Hv, a.dv, a.scale,
        (a.flags & GDN_QK_L2NORM) ? 1 : 0);
    return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

template <typename Tin, typename Tout, int DK>
static gdn_status_t launch_simt_chunk(const gdn_host::ScanArgs &a, cudaStream_t st) {
    constexpr int DVT = DK < 32 ? DK : 32;
    switch (a.chunk) {
    case 16: return launch_simt_t<Tin, Tout, DK, DVT, 16>(a, st);
    case 32: return launch_simt_t<Tin, Tout, DK, DVT, 32>(a, st);
    case 64: return launch_simt_t<Tin, Tout, DK, DVT, 64>(a, st);
    default: return GDN_ERR_UNSUPPORTED;
    }
}

template <typename Tin, typename Tout>
static gdn_status_t launch_simt_dk(const gdn_host::ScanArgs &a, cudaStream_t st) {
    if (a.dk != a.dv) return GDN_ERR_UNSUPPORTED;
    switch (a.dk) {
    case 16: return launch_simt_chunk<Tin, Tout, 16>(a, st);
    case 32: return launch_simt_chunk<Tin, Tout, 32>(a, st);
    case 64: return launch_simt_chunk<Tin, Tout, 64>(a, st);
    case 128: return launch_simt_chunk<Tin, Tout, 128>(a, st);
    default: return GDN_ERR_UNSUPPORTED;
    }
}

}  // namespace gdn

namespace gdn_host {

gdn_status_t launch_chunk_simt(const ScanArgs &a, cudaStream_t st) {
    if (a.N == 0) return GDN_OK;
    // Outputs take the activation dtype: bf16 in -> bf16 out, fp32 in -> fp32 out.
    if (a.in_f32 != a.out_f32) return GDN_ERR_DTYPE;
    if (!a.in_f32) return gdn::launch_simt_dk<gdn::bf16, gdn::bf16>(a, st);
    return gdn::launch_simt_dk<float, float>(a, st);
}

}  // namespace gdn_host
