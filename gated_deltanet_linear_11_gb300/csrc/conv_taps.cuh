// conv_taps.cuh -- the width-4 causal depthwise conv + SiLU of 8 adjacent channels, shared
// by the prefill conv, the decode conv update and the fused decode step so all three give
// the same bits for the same token.
//
// Source: "[Feature] Add batch invariance support to GDN_ATTN backend - #45819", Birol's
// comment, part 3(a): conv over cat(conv_state, x), groups = channels, SiLU of the output.
#pragma once

#include "common.cuh"

namespace gdn {

struct Taps {
    float w[8][4];
    float b[8];
};

__device__ __forceinline__ void load_taps(Taps &tp, const bf16 *w, const bf16 *bias, int c0) {
    const uint4 *wp = reinterpret_cast<const uint4 *>(w + (size_t)c0 * 4);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float f[8];
        unpack8(__ldg(wp + i), f);  // channels c0+2i, c0+2i+1, 4 taps each
        tp.w[2 * i][0] = f[0]; tp.w[2 * i][1] = f[1]; tp.w[2 * i][2] = f[2]; tp.w[2 * i][3] = f[3];
        tp.w[2 * i + 1][0] = f[4]; tp.w[2 * i + 1][1] = f[5]; tp.w[2 * i + 1][2] = f[6]; tp.w[2 * i + 1][3] = f[7];
    }
    if (bias) {
        unpack8(__ldg(reinterpret_cast<const uint4 *>(bias + c0)), tp.b);
    } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) tp.b[i] = 0.f;
    }
}

// y = silu(b + w0*x0 + w1*x1 + w2*x2 + w3*x3), x0 oldest.  Fixed evaluation order.
__device__ __forceinline__ uint4 conv_out(const Taps &tp, const float x0[8], const float x1[8],
                                          const float x2[8], const float x3[8]) {
    float r[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        float z = tp.b[i];
        z = fmaf(tp.w[i][0], x0[i], z);
        z = fmaf(tp.w[i][1], x1[i], z);
        z = fmaf(tp.w[i][2], x2[i], z);
        z = fmaf(tp.w[i][3], x3[i], z);
        r[i] = silu(z);
    }
    return pack8(r);
}

}  // namespace gdn
