// conv1d.cu -- width-4 causal depthwise conv1d + SiLU, prefill and one-token update.
//
// Source: "[Feature] Add batch invariance support to GDN_ATTN backend - #45819", Birol's
// comment, part 3(a): conv over cat(conv_state, x), padding 0, groups = channels, SiLU of
// the last seq_len outputs, new conv state = the last three conv inputs.
//
// Both kernels are HBM-bound streams: every thread owns 8 adjacent channels (one 16-byte
// vector), so a warp moves 512 contiguous bytes per token row.  The four taps are summed
// in one fixed order (bias, then w0..w3 oldest to newest) in fp32, so the prefill and the
// decode update give the same bits for the same token, and no value depends on how the
// packed batch is tiled.
#include "common.cuh"
#include "conv_taps.cuh"

namespace gdn {

constexpr int kConvThreads = 128;   // threads per block, 8 channels each
constexpr int kConvTile = 16;       // tokens per thread (anchored at the sequence start)
constexpr int kConvGroup = 2;       // rows per commit group of the full-tile copy
static_assert(kConvTile % kConvGroup == 0 && kConvTile / kConvGroup <= 8, "copy groups");

// Wait until at most n of this thread's copy groups are still in flight (n is a constant
// once the caller's loop is unrolled, so the switch folds to one instruction).
__device__ __forceinline__ void cp_async_wait_upto(int n) {
    switch (n) {
    case 0: asm volatile("cp.async.wait_group 0;" ::: "memory"); break;
    case 1: asm volatile("cp.async.wait_group 1;" ::: "memory"); break;
    case 2: asm volatile("cp.async.wait_group 2;" ::: "memory"); break;
    case 3: asm volatile("cp.async.wait_group 3;" ::: "memory"); break;
    case 4: asm volatile("cp.async.wait_group 4;" ::: "memory"); break;
    case 5: asm volatile("cp.async.wait_group 5;" ::: "memory"); break;
    case 6: asm volatile("cp.async.wait_group 6;" ::: "memory"); break;
    default: asm volatile("cp.async.wait_group 7;" ::: "memory"); break;
    }
}

// Channels [c_begin, c_end) of the C-wide rows.
// grid: (ceil((c_end - c_begin) / (8*kConvThreads)), ceil(max_len / kConvTile) (>=1), N)
__global__ void __launch_bounds__(kConvThreads, 5)
conv1d_fwd_kernel(const bf16 *__restrict__ x, const bf16 *__restrict__ w,
                  const bf16 *__restrict__ bias, const int32_t *__restrict__ cu,
                  const bf16 *s_in, bf16 *s_out, bf16 *__restrict__ y, int C, int c_begin,
                  int c_end) {
    grid_dependents_launch();
    grid_dependency_wait();
    const int n = blockIdx.z;
    const int tile = blockIdx.y;
    const int c0 = c_begin + (blockIdx.x * kConvThreads + threadIdx.x) * 8;
    if (c0 >= c_end) return;
    const int start = cu[n];
    const int L = cu[n + 1] - start;
    const int t0 = tile * kConvTile;
    if (t0 >= L && tile > 0) return;

    __shared__ uint4 conv_tile_buf[kConvTile][kConvThreads];   // 32 KiB

    Taps tp;
    load_taps(tp, w, bias, c0);

    // Window of the three conv inputs before token t0 (state rows when t0 - 3 + j < 0).
    float win[3][8];
#pragma unroll
    for (int j = 0; j < 3; ++j) {
        const int p = t0 - 3 + j;
        if (p >= 0) {
            unpack8(*reinterpret_cast<const uint4 *>(x + (size_t)(start + p) * C + c0), win[j]);
        } else if (s_in) {
            unpack8(*reinterpret_cast<const uint4 *>(s_in + ((size_t)n * 3 + (3 + p)) * C + c0), win[j]);
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) win[j][i] = 0.f;
        }
    }

    const int cnt = min(kConvTile, L - t0);
    if (cnt == kConvTile) {
        // Full tile: every row goes to shared memory by an asynchronous 16-byte copy at
        // once (in commit groups of kConvGroup rows), so a CTA keeps its whole tile in
        // flight without holding registers and starts on the first rows while the rest
        // arrive; each thread reads back only the slots it copied itself.  Straight-line
        // code keeps the sliding window in renamed registers.
        const bf16 *xp = x + (size_t)(start + t0) * C + c0;
        bf16 *yp = y + (size_t)(start + t0) * C + c0;
        const uint32_t slot0 = (uint32_t)__cvta_generic_to_shared(&conv_tile_buf[0][threadIdx.x]);
#pragma unroll
        for (int i = 0; i < kConvTile; ++i) {
            asm volatile("cp.async.cg.shared.global [%0], [%1], 16;"
                         :: "r"(slot0 + (uint32_t)(i * kConvThreads * 16)), "l"(xp + (size_t)i * C)
                         : "memory");
            if (i % kConvGroup == kConvGroup - 1) asm volatile("cp.async.commit_group;" ::: "memory");
        }
#pragma unroll
        for (int i = 0; i < kConvTile; ++i) {
            if (i % kConvGroup == 0) cp_async_wait_upto(kConvTile / kConvGroup - 1 - i / kConvGroup);
            float cur[8];
            unpack8(conv_tile_buf[i][threadIdx.x], cur);
            *reinterpret_cast<uint4 *>(yp + (size_t)i * C) = conv_out(tp, win[0], win[1], win[2], cur);
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                win[0][e] = win[1][e];
                win[1][e] = win[2][e];
                win[2][e] = cur[e];
            }
        }
    } else {
        // Partial tile (the last of a sequence): a plain row loop.
#pragma unroll 1
        for (int i = 0; i < cnt; ++i) {
            float cur[8];
            unpack8(*reinterpret_cast<const uint4 *>(x + (size_t)(start + t0 + i) * C + c0), cur);
            *reinterpret_cast<uint4 *>(y + (size_t)(start + t0 + i) * C + c0) =
                conv_out(tp, win[0], win[1], win[2], cur);
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                win[0][e] = win[1][e];
                win[1][e] = win[2][e];
                win[2][e] = cur[e];
            }
        }
    }

    // The first tile of a sequence is the only reader of the old conv state, so it also
    // writes the new one.  xs = [old(3) ; x_seq]; the new state is xs[L], xs[L+1],
    // xs[L+2].  Row j is written after old row L+j >= j was read, so s_out == s_in is safe.
    if (tile == 0 && s_out) {
#pragma unroll
        for (int j = 0; j < 3; ++j) {
            const int m = L + j;
            uint4 val = make_uint4(0u, 0u, 0u, 0u);
            if (m >= 3) {
                val = *reinterpret_cast<const uint4 *>(x + (size_t)(start + m - 3) * C + c0);
            } else if (s_in) {
                val = *reinterpret_cast<const uint4 *>(s_in + ((size_t)n * 3 + m) * C + c0);
            }
            *reinterpret_cast<uint4 *>(s_out + ((size_t)n * 3 + j) * C + c0) = val;
        }
    }
}

constexpr int kUpdSeqs = 4;  // sequences per thread in the decode conv update

// Decode conv: one new token per sequence; the state rows shift in place.  Each thread
// owns 8 channels of kUpdSeqs sequences, so 4 x kUpdSeqs independent 16-byte loads are in
// flight per thread.  grid: (ceil(C / (8*kConvThreads)), ceil(N / kUpdSeqs))
__global__ void __launch_bounds__(kConvThreads)
conv1d_update_kernel(const bf16 *__restrict__ x, const bf16 *__restrict__ w,
                     const bf16 *__restrict__ bias, bf16 *state, int P,
                     const int32_t *__restrict__ idx, bf16 *__restrict__ y, int C, int N,
                     int32_t *status) {
    const int c0 = (blockIdx.x * kConvThreads + threadIdx.x) * 8;
    if (c0 >= C) return;
    const int n0 = blockIdx.y * kUpdSeqs;
    int slot[kUpdSeqs];
#pragma unroll
    for (int i = 0; i < kUpdSeqs; ++i) {
        const int n = n0 + i;
        slot[i] = -1;
        if (n < N) {
            const int sl = idx ? idx[n] : n;
            if (sl >= 0 && sl < P) slot[i] = sl;
            else if (c0 == 0) report(status, GDN_ERR_INDEX);
        }
    }
    uint4 r0[kUpdSeqs], r1[kUpdSeqs], r2[kUpdSeqs], rx[kUpdSeqs];
#pragma unroll
    for (int i = 0; i < kUpdSeqs; ++i) {
        if (slot[i] >= 0) {
            const bf16 *s = state + (size_t)slot[i] * 3 * C + c0;
            r0[i] = *reinterpret_cast<const uint4 *>(s);
            r1[i] = *reinterpret_cast<const uint4 *>(s + C);
            r2[i] = *reinterpret_cast<const uint4 *>(s + 2 * C);
            rx[i] = *reinterpret_cast<const uint4 *>(x + (size_t)(n0 + i) * C + c0);
        }
    }
    Taps tp;
    load_taps(tp, w, bias, c0);
#pragma unroll
    for (int i = 0; i < kUpdSeqs; ++i) {
        if (slot[i] >= 0) {
            float s0[8], s1[8], s2[8], cur[8];
            unpack8(r0[i], s0);
            unpack8(r1[i], s1);
            unpack8(r2[i], s2);
            unpack8(rx[i], cur);
            *reinterpret_cast<uint4 *>(y + (size_t)(n0 + i) * C + c0) = conv_out(tp, s0, s1, s2, cur);
            bf16 *s = state + (size_t)slot[i] * 3 * C + c0;
            *reinterpret_cast<uint4 *>(s) = r1[i];
            *reinterpret_cast<uint4 *>(s + C) = r2[i];
            *reinterpret_cast<uint4 *>(s + 2 * C) = rx[i];
        }
    }
}

}  // namespace gdn

namespace gdn_host {

gdn_status_t launch_conv1d_fwd(const void *x, int32_t C, const void *w, const void *bias,
                               const int32_t *cu, int32_t N, int32_t max_len,
                               const void *s_in, void *s_out, void *y, cudaStream_t st,
                               int32_t c_begin, int32_t c_end) {
    if (c_end < 0) c_end = C;
    if (N == 0 || c_end <= c_begin) return GDN_OK;
    const int tiles = max_len > 0 ? (max_len + gdn::kConvTile - 1) / gdn::kConvTile : 1;
    dim3 grid(((c_end - c_begin) / 8 + gdn::kConvThreads - 1) / gdn::kConvThreads, tiles, N);
    const cudaError_t e = launch_dependent(
        gdn::conv1d_fwd_kernel, grid, dim3(gdn::kConvThreads), 0, st, (const gdn::bf16 *)x,
        (const gdn::bf16 *)w, (const gdn::bf16 *)bias, cu, (const gdn::bf16 *)s_in,
        (gdn::bf16 *)s_out, (gdn::bf16 *)y, C, c_begin, c_end);
    return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

gdn_status_t launch_conv1d_update(const void *x, int32_t N, int32_t C, const void *w,
                                  const void *bias, void *state, int32_t P,
                                  const int32_t *idx, void *y, int32_t *status,
                                  cudaStream_t st) {
    if (N == 0) return GDN_OK;
    dim3 grid((C / 8 + gdn::kConvThreads - 1) / gdn::kConvThreads,
              (N + gdn::kUpdSeqs - 1) / gdn::kUpdSeqs);
    gdn::conv1d_update_kernel<<<grid, gdn::kConvThreads, 0, st>>>(
        (const gdn::bf16 *)x, (const gdn::bf16 *)w, (const gdn::bf16 *)bias,
        (gdn::bf16 *)state, P, idx, (gdn::bf16 *)y, C, N, status);
    return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

}  // namespace gdn_host
