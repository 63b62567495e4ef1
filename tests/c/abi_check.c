/*
 * abi_check.c -- the C ABI of libgdn.so driven from plain C99, with no Python and no
 * PyTorch in the process.
 *
 *   abi_check cpu   host-side entries only: version, status names, argument rejections,
 *                   workspace sizes and the range hint for an explicit SM count.
 *   abi_check gpu   a bf16 chunked prefill of two packed sequences through
 *                   gdn_chunk_prefill, checked against the same tokens stepped one at a
 *                   time through gdn_recurrent_decode: two different kernels of the
 *                   library, which compute the same recurrence
 *                   ("Qwen3.5-27B GPTQ Garbage Inference -- Root Cause Analysis",
 *                   "Why abliteration failed on Qwen3.5", item 3).
 *
 * Prints "ok" and exits 0, or prints the first failed check and exits 1.
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "gdn.h"

#define CHECK(cond)                                                        \
    do {                                                                   \
        if (!(cond)) {                                                     \
            fprintf(stderr, "%s:%d: check failed: %s\n", __FILE__, __LINE__, #cond); \
            exit(1);                                                       \
        }                                                                  \
    } while (0)

static gdn_tensor_t view3(void *ptr, int32_t dtype, int64_t T, int64_t H, int64_t D) {
    gdn_tensor_t t;
    memset(&t, 0, sizeof(t));
    t.ptr = ptr;
    t.ndim = 3;
    t.dtype = dtype;
    t.shape[0] = T; t.shape[1] = H; t.shape[2] = D;
    t.stride[0] = H * D; t.stride[1] = D; t.stride[2] = 1;
    return t;
}

static int cpu_checks(void) {
    CHECK(gdn_version() >= 100);
    for (int s = 0; s <= 11; ++s) {
        const char *name = gdn_status_string((gdn_status_t)s);
        CHECK(name != NULL && strncmp(name, "GDN_", 4) == 0);
    }
    CHECK(strncmp(gdn_status_string(GDN_ERR_NONFINITE), "GDN_ERR_NONFINITE", 17) == 0);

    /* host-side validation: nothing here touches a device */
    static uint16_t buf[4 * 12 * 32 * 128 + 64];
    void *p = (void *)(((uintptr_t)buf + 15) & ~(uintptr_t)15);
    const int32_t cu[3] = {0, 5, 12}, cu_bad[3] = {0, 7, 5};
    gdn_tensor_t q = view3(p, GDN_BF16, 12, 16, 128), k = q;
    gdn_tensor_t v = view3(p, GDN_BF16, 12, 32, 128), o = v;
    float gb[12 * 32];
    CHECK(gdn_chunk_prefill(NULL, &k, &v, gb, gb, cu, cu, 2, 64, 1.f, 0, NULL, &o, NULL, NULL,
                            0, NULL, NULL) == GDN_ERR_NULL);
    CHECK(gdn_chunk_prefill(&q, &k, &v, gb, gb, cu, cu_bad, 2, 64, 1.f, 0, NULL, &o, NULL,
                            NULL, 0, NULL, NULL) == GDN_ERR_SEQLENS);
    /* a head-first [H, T, D] buffer viewed as [T, H, D] (head stride > token stride), with
     * the genuine T = 12 < H = 16 case left legal */
    gdn_tensor_t hf = q;
    hf.stride[0] = 128; hf.stride[1] = 12 * 128;
    CHECK(gdn_chunk_prefill(&hf, &k, &v, gb, gb, cu, cu, 2, 64, 1.f, 0, NULL, &o, NULL, NULL,
                            0, NULL, NULL) == GDN_ERR_LAYOUT);
    gdn_tensor_t k_short = view3(p, GDN_BF16, 11, 16, 128);
    CHECK(gdn_chunk_prefill(&q, &k_short, &v, gb, gb, cu, cu, 2, 64, 1.f, 0, NULL, &o, NULL,
                            NULL, 0, NULL, NULL) == GDN_ERR_SHAPE);
    /* a tensor-core call without its workspace */
    CHECK(gdn_chunk_prefill(&q, &k, &v, gb, gb, cu, cu, 2, 64, 1.f, 0, NULL, &o, NULL, NULL,
                            0, NULL, NULL) == GDN_ERR_WORKSPACE);

    /* workspace: one 17408-byte tile per (chunk slot, v-head), slots = ceil(T/64) + N + 1 */
    CHECK(gdn_chunk_prefill_workspace_size(1, 4096, 16, 48, 128, 128, 64, 0) ==
          (size_t)(64 + 1 + 1) * 48 * 17408);
    CHECK(gdn_chunk_prefill_workspace_size(2, 12, 16, 32, 128, 128, 64, GDN_PREFILL_SIMT) == 0);
    /* the range hint on a 152-SM device: one 32768-token sequence over 6 v-heads splits
     * into 40-chunk ranges; the 27B layer's 4096 tokens over 48 v-heads stay plain */
    CHECK(gdn_chunk_prefill_cp_range_hint_for(32768, 6, 152) == 40);
    CHECK(gdn_chunk_prefill_cp_range_hint_for(4096, 48, 152) == 0);
    CHECK(gdn_selftest_bounded_wait(NULL, NULL) == GDN_ERR_NULL);
    return 0;
}

/* ------------------------------------------------------------------------ GPU part */

static uint32_t lcg = 12345u;
static float uniform(void) {   /* [0, 1) */
    lcg = lcg * 1664525u + 1013904223u;
    return (float)(lcg >> 8) / 16777216.0f;
}
static uint16_t to_bf16(float f) {   /* round to nearest even */
    uint32_t u;
    memcpy(&u, &f, 4);
    u += 0x7fffu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}
static float from_bf16(uint16_t h) {
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}
static void *dev_copy(const void *host, size_t bytes) {
    void *d = NULL;
    CHECK(cudaMalloc(&d, bytes) == cudaSuccess);
    CHECK(cudaMemcpy(d, host, bytes, cudaMemcpyHostToDevice) == 0);
    return d;
}

static int gpu_checks(void) {
    enum { Hk = 1, Hv = 2, D = 128, N = 2 };
    const int32_t lens[N] = {70, 60};
    const int32_t T = lens[0] + lens[1];
    const int32_t cu[N + 1] = {0, lens[0], T};
    const size_t nqk = (size_t)T * Hk * D, nv = (size_t)T * Hv * D, ng = (size_t)T * Hv;
    uint16_t *hq = malloc(nqk * 2), *hk = malloc(nqk * 2), *hv = malloc(nv * 2);
    float *hg = malloc(ng * 4), *hb = malloc(ng * 4);
    for (size_t i = 0; i < nqk; ++i) hq[i] = to_bf16(2.f * uniform() - 1.f);
    for (size_t i = 0; i < nqk; ++i) hk[i] = to_bf16(2.f * uniform() - 1.f);
    for (size_t i = 0; i < nv; ++i) hv[i] = to_bf16(2.f * uniform() - 1.f);
    for (size_t i = 0; i < ng; ++i) {
        hg[i] = -0.02f - 0.2f * uniform();   /* decays e^g in (0.8, 0.98) */
        hb[i] = 0.1f + 0.8f * uniform();
    }
    void *dq = dev_copy(hq, nqk * 2), *dk = dev_copy(hk, nqk * 2), *dv = dev_copy(hv, nv * 2);
    float *dg = dev_copy(hg, ng * 4), *db = dev_copy(hb, ng * 4);
    int32_t *dcu = dev_copy(cu, sizeof(cu));
    void *dout = NULL;
    float *dstate = NULL, *dpool = NULL;
    int32_t *dstatus = NULL;
    const size_t head = (size_t)D * D, sbytes = (size_t)N * Hv * head * 4;
    CHECK(cudaMalloc(&dout, nv * 2) == 0);
    CHECK(cudaMalloc((void **)&dstate, sbytes) == 0);
    CHECK(cudaMalloc((void **)&dpool, (size_t)Hv * head * 4) == 0);
    CHECK(cudaMalloc((void **)&dstatus, 4) == 0);
    CHECK(cudaMemset(dstatus, 0, 4) == 0);

    /* the chunked prefill, q/k L2-normalised, zero initial state */
    const size_t ws_bytes = gdn_chunk_prefill_workspace_size(N, T, Hk, Hv, D, D, 64, 0);
    void *ws = NULL;
    if (ws_bytes) CHECK(cudaMalloc(&ws, ws_bytes) == 0);
    gdn_tensor_t q = view3(dq, GDN_BF16, T, Hk, D), k = view3(dk, GDN_BF16, T, Hk, D);
    gdn_tensor_t v = view3(dv, GDN_BF16, T, Hv, D), o = view3(dout, GDN_BF16, T, Hv, D);
    CHECK(gdn_chunk_prefill(&q, &k, &v, dg, db, dcu, cu, N, 64, 1.f, GDN_QK_L2NORM, NULL, &o,
                            dstate, ws, ws_bytes, dstatus, NULL) == GDN_OK);
    CHECK(cudaDeviceSynchronize() == 0);
    uint16_t *o_pre = malloc(nv * 2);
    float *h_pre = malloc(sbytes), *h_rec = malloc((size_t)Hv * head * 4);
    CHECK(cudaMemcpy(o_pre, dout, nv * 2, cudaMemcpyDeviceToHost) == 0);
    CHECK(cudaMemcpy(h_pre, dstate, sbytes, cudaMemcpyDeviceToHost) == 0);

    /* the same tokens one at a time through the recurrent decode step, one sequence at a
     * time on a one-slot pool */
    float err_o = 0.f, err_h = 0.f, ref_h = 0.f;
    void *dout1 = NULL;
    CHECK(cudaMalloc(&dout1, (size_t)Hv * D * 2) == 0);
    uint16_t o1[Hv * D];
    for (int n = 0; n < N; ++n) {
        CHECK(cudaMemset(dpool, 0, (size_t)Hv * head * 4) == 0);
        for (int t = cu[n]; t < cu[n + 1]; ++t) {
            gdn_tensor_t q1 = view3((uint16_t *)dq + (size_t)t * Hk * D, GDN_BF16, 1, Hk, D);
            gdn_tensor_t k1 = view3((uint16_t *)dk + (size_t)t * Hk * D, GDN_BF16, 1, Hk, D);
            gdn_tensor_t v1 = view3((uint16_t *)dv + (size_t)t * Hv * D, GDN_BF16, 1, Hv, D);
            gdn_tensor_t out1 = view3(dout1, GDN_BF16, 1, Hv, D);
            CHECK(gdn_recurrent_decode(&q1, &k1, &v1, dg + (size_t)t * Hv, db + (size_t)t * Hv,
                                       dpool, 1, NULL, 1.f, GDN_QK_L2NORM, &out1, dstatus,
                                       NULL) == GDN_OK);
            CHECK(cudaMemcpy(o1, dout1, sizeof(o1), cudaMemcpyDeviceToHost) == 0);
            for (int i = 0; i < Hv * D; ++i) {
                const float a = from_bf16(o1[i]), b = from_bf16(o_pre[(size_t)t * Hv * D + i]);
                err_o = fmaxf(err_o, fabsf(a - b) / (1.f + fabsf(b)));
            }
        }
        CHECK(cudaMemcpy(h_rec, dpool, (size_t)Hv * head * 4, cudaMemcpyDeviceToHost) == 0);
        for (size_t i = 0; i < (size_t)Hv * head; ++i) {
            const float a = h_rec[i], b = h_pre[(size_t)n * Hv * head + i];
            err_h = fmaxf(err_h, fabsf(a - b));
            ref_h = fmaxf(ref_h, fabsf(b));
        }
    }
    int32_t status = -1;
    CHECK(cudaMemcpy(&status, dstatus, 4, cudaMemcpyDeviceToHost) == 0);
    printf("prefill vs recurrent decode: max output error %.3g, max state error %.3g "
           "(state max %.3g)\n", err_o, err_h, ref_h);
    CHECK(status == 0);
    CHECK(ref_h > 0.f && isfinite(err_o) && isfinite(err_h));
    CHECK(err_o < 2e-2f);
    CHECK(err_h < 2e-3f * ref_h + 1e-4f);
    cudaFree(dq); cudaFree(dk); cudaFree(dv); cudaFree(dg); cudaFree(db); cudaFree(dcu);
    cudaFree(dout); cudaFree(dout1); cudaFree(dstate); cudaFree(dpool); cudaFree(dstatus);
    if (ws) cudaFree(ws);
    free(hq); free(hk); free(hv); free(hg); free(hb); free(o_pre); free(h_pre); free(h_rec);
    return 0;
}

int main(int argc, char **argv) {
    if (argc != 2 || (strcmp(argv[1], "cpu") != 0 && strcmp(argv[1], "gpu") != 0)) {
        fprintf(stderr, "usage: %s cpu|gpu\n", argv[0]);
        return 2;
    }
    cpu_checks();
    if (strcmp(argv[1], "gpu") == 0) gpu_checks();
    printf("ok\n");
    return 0;
}
