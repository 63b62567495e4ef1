// api.cu -- the extern "C" boundary of libgdn.so: argument validation and dispatch.
//
// Every entry point validates its arguments on the host and returns a gdn_status_t
// before launching anything; nothing here allocates device memory.
#include <string.h>

#include <cmath>
#include <vector>

#include "common.cuh"

namespace {

bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

int elem_size(int32_t dt) { return dt == GDN_BF16 ? 2 : 4; }

// Token-major activation view: [T,H,D] or [1,T,H,D]; unit element stride, head stride
// D, token stride >= H*D and a multiple of 16 bytes, 16-byte aligned base.  A view whose
// head stride exceeds its token stride is head-first and is rejected (no T < H guess).
struct View {
    void *ptr;
    int64_t T, H, D, tok;
    int32_t dtype;
};

gdn_status_t view_of(const gdn_tensor_t *t, View &out) {
    if (!t) return GDN_ERR_NULL;
    int off;
    if (t->ndim == 3) {
        off = 0;
    } else if (t->ndim == 4) {
        if (t->shape[0] != 1) return GDN_ERR_LAYOUT;  // packed varlen uses B = 1
        off = 1;
    } else {
        return GDN_ERR_SHAPE;
    }
    if (t->dtype != GDN_BF16 && t->dtype != GDN_F32) return GDN_ERR_DTYPE;
    const int64_t T = t->shape[off], H = t->shape[off + 1], D = t->shape[off + 2];
    const int64_t st = t->stride[off], sh = t->stride[off + 1], sd = t->stride[off + 2];
    if (T < 0 || H <= 0 || D <= 0) return GDN_ERR_SHAPE;
    if (T == 0) {   // an empty view touches no memory: no storage or strides to check
        out.ptr = t->ptr;
        out.T = 0;
        out.H = H;
        out.D = D;
        out.tok = H * D;
        out.dtype = t->dtype;
        return GDN_OK;
    }
    if (!t->ptr) return GDN_ERR_NULL;
    if (T > 1 && H > 1 && sh > st) return GDN_ERR_LAYOUT;  // head-first
    if (sd != 1 || sh != D) return GDN_ERR_LAYOUT;
    if (T > 1 && st < H * D) return GDN_ERR_LAYOUT;
    if ((st * elem_size(t->dtype)) % 16 != 0 || !aligned16(t->ptr)) return GDN_ERR_LAYOUT;
    out.ptr = t->ptr;
    out.T = T;
    out.H = H;
    out.D = D;
    out.tok = T > 1 ? st : H * D;
    out.dtype = t->dtype;
    return GDN_OK;
}

// GDN_CHECK_INPUTS: n floats at each of two device arrays, copied to the host in order on
// `st` (waiting for it), must all be finite.
gdn_status_t check_finite(const float *a, const float *b, size_t n, cudaStream_t st) {
    if (n == 0) return GDN_OK;
    std::vector<float> h(n);
    for (const float *src : {a, b}) {
        if (cudaMemcpyAsync(h.data(), src, n * sizeof(float), cudaMemcpyDeviceToHost, st) !=
                cudaSuccess ||
            cudaStreamSynchronize(st) != cudaSuccess)
            return GDN_ERR_CUDA;
        for (size_t i = 0; i < n; ++i)
            if (!std::isfinite(h[i])) return GDN_ERR_NONFINITE;
    }
    return GDN_OK;
}

// GDN_CHECK_INPUTS: the device offsets, copied back on `st` (waiting for it), must equal
// the host copy that was validated.
gdn_status_t check_seqlens_copy(const int32_t *cu_dev, const int32_t *cu_host, int32_t N,
                                cudaStream_t st) {
    std::vector<int32_t> h((size_t)N + 1);
    if (cudaMemcpyAsync(h.data(), cu_dev, h.size() * sizeof(int32_t), cudaMemcpyDeviceToHost,
                        st) != cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess)
        return GDN_ERR_CUDA;
    return memcmp(h.data(), cu_host, h.size() * sizeof(int32_t)) == 0 ? GDN_OK : GDN_ERR_SEQLENS;
}

gdn_status_t check_seqlens(const int32_t *cu, int32_t N, int64_t T, int32_t *max_len) {
    if (!cu) return GDN_ERR_NULL;
    if (cu[0] != 0 || (int64_t)cu[N] != T) return GDN_ERR_SEQLENS;
    int32_t m = 0;
    for (int32_t n = 0; n < N; ++n) {
        if (cu[n + 1] < cu[n]) return GDN_ERR_SEQLENS;
        m = cu[n + 1] - cu[n] > m ? cu[n + 1] - cu[n] : m;
    }
    *max_len = m;
    return GDN_OK;
}

}  // namespace

extern "C" {

const char *gdn_status_string(gdn_status_t s) {
    switch (s) {
    case GDN_OK: return "GDN_OK";
    case GDN_ERR_NULL: return "GDN_ERR_NULL: a required pointer is NULL";
    case GDN_ERR_SHAPE: return "GDN_ERR_SHAPE: inconsistent sizes";
    case GDN_ERR_LAYOUT: return "GDN_ERR_LAYOUT: head-first or unsupported strides/alignment";
    case GDN_ERR_DTYPE: return "GDN_ERR_DTYPE: unsupported or mismatched element type";
    case GDN_ERR_SEQLENS: return "GDN_ERR_SEQLENS: cu_seqlens must rise from 0 to T";
    case GDN_ERR_UNSUPPORTED: return "GDN_ERR_UNSUPPORTED: no kernel for this shape";
    case GDN_ERR_CUDA: return "GDN_ERR_CUDA: a CUDA runtime call failed";
    case GDN_ERR_TIMEOUT: return "GDN_ERR_TIMEOUT: a bounded device wait gave up";
    case GDN_ERR_WORKSPACE: return "GDN_ERR_WORKSPACE: workspace missing or too small";
    case GDN_ERR_INDEX: return "GDN_ERR_INDEX: state index outside the pool";
    case GDN_ERR_NONFINITE: return "GDN_ERR_NONFINITE: a gate input is NaN or infinite";
    }
    return "GDN_ERR_UNKNOWN";
}

int32_t gdn_version(void) { return 100; }

gdn_status_t gdn_conv1d_fwd(const void *x, int64_t T, int32_t C, const void *w,
                            const void *bias, const int32_t *cu_seqlens_dev,
                            const int32_t *cu_seqlens_host, int32_t N,
                            const void *conv_state_in, void *conv_state_out, void *y,
                            void *stream) {
    gdn_host::CallRange nvtx_range("gdn_conv1d_fwd");
    if ((!x && T > 0) || !w || !cu_seqlens_dev || !cu_seqlens_host || (!y && T > 0))
        return GDN_ERR_NULL;
    if (N < 0 || T < 0 || C <= 0 || N > 65535) return GDN_ERR_SHAPE;
    if (C % 8 != 0) return GDN_ERR_UNSUPPORTED;
    if (!aligned16(x) || !aligned16(w) || !aligned16(bias) || !aligned16(y) ||
        !aligned16(conv_state_in) || !aligned16(conv_state_out))
        return GDN_ERR_LAYOUT;
    int32_t max_len = 0;
    gdn_status_t s = check_seqlens(cu_seqlens_host, N, T, &max_len);
    if (s != GDN_OK) return s;
    if ((max_len + 15) / 16 > 65535) return GDN_ERR_SHAPE;
    return gdn_host::launch_conv1d_fwd(x, C, w, bias, cu_seqlens_dev, N, max_len,
                                       conv_state_in, conv_state_out, y,
                                       (cudaStream_t)stream);
}

gdn_status_t gdn_conv1d_update(const void *x, int32_t N, int32_t C, const void *w,
                               const void *bias, void *conv_state, int32_t P,
                               const int32_t *state_idx, void *y, int32_t *status_dev,
                               void *stream) {
    gdn_host::CallRange nvtx_range("gdn_conv1d_update");
    if (N < 0 || C <= 0 || P < 0 || N > 65535) return GDN_ERR_SHAPE;
    if (N == 0) return GDN_OK;
    if (!x || !w || !conv_state || !y) return GDN_ERR_NULL;
    if (C % 8 != 0) return GDN_ERR_UNSUPPORTED;
    if (!state_idx && P < N) return GDN_ERR_SHAPE;
    if (!aligned16(x) || !aligned16(w) || !aligned16(bias) || !aligned16(y) ||
        !aligned16(conv_state))
        return GDN_ERR_LAYOUT;
    return gdn_host::launch_conv1d_update(x, N, C, w, bias, conv_state, P, state_idx, y,
                                          status_dev, (cudaStream_t)stream);
}

size_t gdn_chunk_prefill_workspace_size(int32_t N, int64_t T, int32_t Hk, int32_t Hv,
                                        int32_t dk, int32_t dv, int32_t chunk,
                                        uint32_t flags) {
    if ((flags & GDN_PREFILL_SIMT) || !gdn_host::chunk_tc_supported(dk, dv, chunk, 0))
        return 0;
    return gdn_host::chunk_tc_workspace(N, T, Hk, Hv);
}

}  // extern "C"

namespace {

// gdn_chunk_prefill with one extra hook: an event that the work reading v must wait on
// (the layer entry produces v on a second stream).
gdn_status_t chunk_prefill_impl(const gdn_tensor_t *q, const gdn_tensor_t *k,
                                const gdn_tensor_t *v, const float *g, const float *beta,
                                const int32_t *cu_seqlens_dev, const int32_t *cu_seqlens_host,
                                int32_t N, int32_t chunk, float scale, uint32_t flags,
                                const float *initial_state, const gdn_tensor_t *o,
                                float *final_state, void *workspace, size_t workspace_bytes,
                                int32_t *status_dev, void *stream, cudaEvent_t v_ready,
                                int32_t range_chunks = 0,
                                const gdn_host::VConvArgs *vconv = nullptr) {
    View Q, K, V, O;
    gdn_status_t s;
    if ((s = view_of(q, Q)) != GDN_OK) return s;
    if ((s = view_of(k, K)) != GDN_OK) return s;
    if ((s = view_of(v, V)) != GDN_OK) return s;
    if ((s = view_of(o, O)) != GDN_OK) return s;
    if ((Q.T > 0 && (!g || !beta)) || !cu_seqlens_dev || !cu_seqlens_host) return GDN_ERR_NULL;
    if (N < 0 || N > 65535) return GDN_ERR_SHAPE;
    if (K.T != Q.T || V.T != Q.T || O.T != Q.T || K.H != Q.H || K.D != Q.D ||
        O.H != V.H || O.D != V.D)
        return GDN_ERR_SHAPE;
    if (V.H % Q.H != 0) return GDN_ERR_SHAPE;
    if (Q.dtype != K.dtype || Q.dtype != V.dtype) return GDN_ERR_DTYPE;
    if (!aligned16(initial_state) || !aligned16(final_state)) return GDN_ERR_LAYOUT;
    int32_t max_len = 0;
    if ((s = check_seqlens(cu_seqlens_host, N, Q.T, &max_len)) != GDN_OK) return s;
    cudaStream_t st = (cudaStream_t)stream;
    if (Q.T == 0) {
        // no tokens: every sequence is empty and keeps its initial state
        if (final_state && N > 0) {
            const size_t bytes = (size_t)N * V.H * Q.D * V.D * sizeof(float);
            const cudaError_t e =
                initial_state ? cudaMemcpyAsync(final_state, initial_state, bytes,
                                                cudaMemcpyDeviceToDevice, st)
                              : cudaMemsetAsync(final_state, 0, bytes, st);
            if (e != cudaSuccess) return GDN_ERR_CUDA;
        }
        return GDN_OK;
    }
    if ((flags & GDN_CHECK_INPUTS) &&
        ((s = check_finite(g, beta, (size_t)Q.T * V.H, st)) != GDN_OK ||
         (s = check_seqlens_copy(cu_seqlens_dev, cu_seqlens_host, N, st)) != GDN_OK))
        return s;

    gdn_host::ScanArgs a;
    memset(&a, 0, sizeof(a));
    a.q = Q.ptr; a.k = K.ptr; a.v = V.ptr; a.o = O.ptr;
    a.q_tok = Q.tok; a.k_tok = K.tok; a.v_tok = V.tok; a.o_tok = O.tok;
    a.g = g; a.beta = beta; a.cu = cu_seqlens_dev;
    a.h0 = initial_state; a.hT = final_state;
    a.N = N; a.Hk = (int32_t)Q.H; a.Hv = (int32_t)V.H; a.dk = (int32_t)Q.D;
    a.dv = (int32_t)V.D; a.chunk = chunk; a.T = Q.T; a.max_len = max_len;
    a.scale = scale; a.flags = flags;
    a.in_f32 = Q.dtype == GDN_F32; a.out_f32 = O.dtype == GDN_F32;
    a.status = status_dev; a.ws = workspace; a.ws_bytes = workspace_bytes;
    a.vconv = vconv;

    const bool tc = !(flags & GDN_PREFILL_SIMT) &&
                    gdn_host::chunk_tc_supported(a.dk, a.dv, chunk, a.in_f32);
    // the fused v conv exists in the plain tensor-core scan only
    if (vconv && (!tc || a.out_f32 || range_chunks != 0)) return GDN_ERR_UNSUPPORTED;
    if (range_chunks != 0) {
        // the context-parallel scan exists on the tensor-core path only
        if (!tc || a.out_f32) return GDN_ERR_UNSUPPORTED;
        if (range_chunks < 0) return GDN_ERR_SHAPE;
        const size_t need = gdn_host::chunk_tc_cp_workspace(cu_seqlens_host, N, Q.T, a.Hk, a.Hv,
                                                            range_chunks);
        if (N > 0 && need == 0) return GDN_ERR_SHAPE;
        if (need > 0 && (!workspace || workspace_bytes < need || ((uintptr_t)workspace & 255u)))
            return GDN_ERR_WORKSPACE;
        return gdn_host::launch_chunk_tc_cp(a, cu_seqlens_host, range_chunks, st);
    }
    if (tc) {
        const size_t need = gdn_host::chunk_tc_workspace(N, Q.T, a.Hk, a.Hv);
        if (need > 0 && (!workspace || workspace_bytes < need || ((uintptr_t)workspace & 255u)))
            return GDN_ERR_WORKSPACE;
        return gdn_host::launch_chunk_tc(a, cu_seqlens_host, st, v_ready);
    }
    if (v_ready && cudaStreamWaitEvent(st, v_ready, 0) != cudaSuccess) return GDN_ERR_CUDA;
    return gdn_host::launch_chunk_simt(a, st);
}

}  // namespace

extern "C" {

gdn_status_t gdn_chunk_prefill(const gdn_tensor_t *q, const gdn_tensor_t *k,
                               const gdn_tensor_t *v, const float *g, const float *beta,
                               const int32_t *cu_seqlens_dev,
                               const int32_t *cu_seqlens_host, int32_t N, int32_t chunk,
                               float scale, uint32_t flags, const float *initial_state,
                               const gdn_tensor_t *o, float *final_state, void *workspace,
                               size_t workspace_bytes, int32_t *status_dev, void *stream) {
    gdn_host::CallRange nvtx_range("gdn_chunk_prefill");
    return chunk_prefill_impl(q, k, v, g, beta, cu_seqlens_dev, cu_seqlens_host, N, chunk,
                              scale, flags, initial_state, o, final_state, workspace,
                              workspace_bytes, status_dev, stream, nullptr);
}

size_t gdn_chunk_prefill_cp_workspace_size(const int32_t *cu_seqlens_host, int32_t N,
                                           int64_t T, int32_t Hk, int32_t Hv, int32_t dk,
                                           int32_t dv, int32_t chunk, int32_t range_chunks) {
    if (!gdn_host::chunk_tc_supported(dk, dv, chunk, 0)) return 0;
    return gdn_host::chunk_tc_cp_workspace(cu_seqlens_host, N, T, Hk, Hv, range_chunks);
}

int32_t gdn_chunk_prefill_cp_range_hint(int64_t seq_len, int32_t Hv) {
    return gdn_host::cp_range_hint(seq_len, Hv);
}

int32_t gdn_chunk_prefill_cp_range_hint_for(int64_t seq_len, int32_t Hv, int32_t sm_count) {
    return gdn_host::cp_range_hint(seq_len, Hv, sm_count);
}

gdn_status_t gdn_chunk_prefill_cp(const gdn_tensor_t *q, const gdn_tensor_t *k,
                                  const gdn_tensor_t *v, const float *g, const float *beta,
                                  const int32_t *cu_seqlens_dev,
                                  const int32_t *cu_seqlens_host, int32_t N, int32_t chunk,
                                  float scale, uint32_t flags, int32_t range_chunks,
                                  const float *initial_state, const gdn_tensor_t *o,
                                  float *final_state, void *workspace, size_t workspace_bytes,
                                  int32_t *status_dev, void *stream) {
    gdn_host::CallRange nvtx_range("gdn_chunk_prefill_cp");
    if (range_chunks <= 0) return GDN_ERR_SHAPE;
    return chunk_prefill_impl(q, k, v, g, beta, cu_seqlens_dev, cu_seqlens_host, N, chunk,
                              scale, flags, initial_state, o, final_state, workspace,
                              workspace_bytes, status_dev, stream, nullptr, range_chunks);
}

gdn_status_t gdn_recurrent_decode(const gdn_tensor_t *q, const gdn_tensor_t *k,
                                  const gdn_tensor_t *v, const float *g,
                                  const float *beta, float *state, int32_t P,
                                  const int32_t *state_idx, float scale, uint32_t flags,
                                  const gdn_tensor_t *o, int32_t *status_dev,
                                  void *stream) {
    gdn_host::CallRange nvtx_range("gdn_recurrent_decode");
    View Q, K, V, O;
    gdn_status_t s;
    if ((s = view_of(q, Q)) != GDN_OK) return s;
    if ((s = view_of(k, K)) != GDN_OK) return s;
    if ((s = view_of(v, V)) != GDN_OK) return s;
    if ((s = view_of(o, O)) != GDN_OK) return s;
    if (!g || !beta || !state) return GDN_ERR_NULL;
    if (K.T != Q.T || V.T != Q.T || O.T != Q.T || K.H != Q.H || K.D != Q.D ||
        O.H != V.H || O.D != V.D)
        return GDN_ERR_SHAPE;
    if (V.H % Q.H != 0 || P < 0 || Q.T > 65535) return GDN_ERR_SHAPE;
    if (!state_idx && P < Q.T) return GDN_ERR_SHAPE;
    if (Q.dtype != K.dtype || Q.dtype != V.dtype) return GDN_ERR_DTYPE;
    if (!aligned16(state)) return GDN_ERR_LAYOUT;
    if ((flags & GDN_CHECK_INPUTS) &&
        (s = check_finite(g, beta, (size_t)Q.T * V.H, (cudaStream_t)stream)) != GDN_OK)
        return s;
    gdn_host::DecodeArgs a;
    memset(&a, 0, sizeof(a));
    a.q = Q.ptr; a.k = K.ptr; a.v = V.ptr; a.o = O.ptr;
    a.q_tok = Q.tok; a.k_tok = K.tok; a.v_tok = V.tok; a.o_tok = O.tok;
    a.g = g; a.beta = beta; a.state = state; a.idx = state_idx;
    a.N = (int32_t)Q.T; a.P = P; a.Hk = (int32_t)Q.H; a.Hv = (int32_t)V.H;
    a.dk = (int32_t)Q.D; a.dv = (int32_t)V.D; a.scale = scale; a.flags = flags;
    a.in_f32 = Q.dtype == GDN_F32; a.out_f32 = O.dtype == GDN_F32;
    a.status = status_dev;
    return gdn_host::launch_decode(a, (cudaStream_t)stream);
}

gdn_status_t gdn_fused_decode(const void *x, int32_t N, int32_t Hk, int32_t Hv, int32_t dk,
                              int32_t dv, const void *conv_w, const void *conv_bias,
                              void *conv_state, const float *a_raw, const float *b_raw,
                              float *state, int32_t P, const int32_t *state_idx, float scale,
                              uint32_t flags, void *o, int32_t *status_dev, void *stream) {
    gdn_host::CallRange nvtx_range("gdn_fused_decode");
    if (N < 0 || P < 0 || N > 65535 || Hk <= 0 || Hv <= 0 || Hk > 65535) return GDN_ERR_SHAPE;
    if (Hv % Hk != 0) return GDN_ERR_SHAPE;
    if (dk != 128 || dv != 128) return GDN_ERR_UNSUPPORTED;
    if (N == 0) return GDN_OK;
    if (!x || !conv_w || !conv_state || !a_raw || !b_raw || !state || !o) return GDN_ERR_NULL;
    if (!state_idx && P < N) return GDN_ERR_SHAPE;
    const int64_t C = 2 * (int64_t)Hk * dk + (int64_t)Hv * dv;
    if (C > (int64_t)1 << 30) return GDN_ERR_SHAPE;
    if (!aligned16(x) || !aligned16(conv_w) || !aligned16(conv_bias) || !aligned16(conv_state) ||
        !aligned16(state) || !aligned16(o))
        return GDN_ERR_LAYOUT;
    if (flags & GDN_CHECK_INPUTS) {
        const gdn_status_t s = check_finite(a_raw, b_raw, (size_t)N * Hv, (cudaStream_t)stream);
        if (s != GDN_OK) return s;
    }
    gdn_host::FusedDecodeArgs a;
    memset(&a, 0, sizeof(a));
    a.x = x; a.w = conv_w; a.bias = conv_bias; a.conv_state = conv_state;
    a.a_raw = a_raw; a.b_raw = b_raw; a.state = state; a.idx = state_idx; a.o = o;
    a.N = N; a.P = P; a.Hk = Hk; a.Hv = Hv; a.C = (int32_t)C;
    a.scale = scale; a.flags = flags; a.status = status_dev;
    return gdn_host::launch_fused_decode(a, (cudaStream_t)stream);
}

gdn_status_t gdn_layer_prefill(const void *x, int64_t T, int32_t Hk, int32_t Hv,
                               int32_t dk, int32_t dv, const void *conv_w,
                               const void *conv_bias, const int32_t *cu_seqlens_dev,
                               const int32_t *cu_seqlens_host, int32_t N,
                               const void *conv_state_in, void *conv_state_out, void *y,
                               const float *g, const float *beta, float scale, uint32_t flags,
                               const float *initial_state, void *o, float *final_state,
                               void *workspace, size_t workspace_bytes, int32_t *status_dev,
                               void *side_stream, void *stream) {
    gdn_host::CallRange nvtx_range("gdn_layer_prefill");
    if (Hk <= 0 || Hv <= 0 || dk <= 0 || dv <= 0 || T < 0 || N < 0 || N > 65535)
        return GDN_ERR_SHAPE;
    const int64_t qk = (int64_t)Hk * dk, C64 = 2 * qk + (int64_t)Hv * dv;
    if (C64 > (int64_t)1 << 30) return GDN_ERR_SHAPE;
    const int32_t C = (int32_t)C64;
    // q, k, v: strided [T, H, D] views of the conv output y [T, C]; o: contiguous
    gdn_tensor_t tq, tk, tv, to;
    const gdn_tensor_t *views[4] = {&tq, &tk, &tv, &to};
    const void *ptrs[4] = {y, y ? (const uint8_t *)y + qk * 2 : nullptr,
                           y ? (const uint8_t *)y + 2 * qk * 2 : nullptr, o};
    const int64_t hs[4] = {Hk, Hk, Hv, Hv}, ds[4] = {dk, dk, dv, dv};
    for (int i = 0; i < 4; ++i) {
        gdn_tensor_t &t = *const_cast<gdn_tensor_t *>(views[i]);
        memset(&t, 0, sizeof(t));
        t.ptr = const_cast<void *>(ptrs[i]);
        t.ndim = 3;
        t.dtype = GDN_BF16;
        t.shape[0] = T; t.shape[1] = hs[i]; t.shape[2] = ds[i];
        t.stride[0] = i < 3 ? C : hs[i] * ds[i];
        t.stride[1] = ds[i];
        t.stride[2] = 1;
    }
    cudaStream_t st = (cudaStream_t)stream;
    if (T == 0) {
        gdn_status_t s = gdn_conv1d_fwd(x, T, C, conv_w, conv_bias, cu_seqlens_dev,
                                        cu_seqlens_host, N, conv_state_in, conv_state_out, y,
                                        stream);
        if (s != GDN_OK) return s;
        return chunk_prefill_impl(&tq, &tk, &tv, g, beta, cu_seqlens_dev, cu_seqlens_host, N,
                                  64, scale, flags, initial_state, &to, final_state, workspace,
                                  workspace_bytes, status_dev, stream, nullptr);
    }
    // the conv's own checks, on the whole width, before anything is launched
    if (!x || !conv_w || !cu_seqlens_dev || !cu_seqlens_host || !y) return GDN_ERR_NULL;
    if (C % 8 != 0 || qk % 8 != 0) return GDN_ERR_UNSUPPORTED;
    if (!aligned16(x) || !aligned16(conv_w) || !aligned16(conv_bias) || !aligned16(y) ||
        !aligned16(conv_state_in) || !aligned16(conv_state_out))
        return GDN_ERR_LAYOUT;
    int32_t max_len = 0;
    gdn_status_t s = check_seqlens(cu_seqlens_host, N, T, &max_len);
    if (s != GDN_OK) return s;
    if ((max_len + 15) / 16 > 65535) return GDN_ERR_SHAPE;
    if (flags & GDN_CHECK_INPUTS) {
        // before the conv launches; the scan below need not repeat it
        if (!g || !beta) return GDN_ERR_NULL;
        if ((s = check_finite(g, beta, (size_t)T * Hv, st)) != GDN_OK ||
            (s = check_seqlens_copy(cu_seqlens_dev, cu_seqlens_host, N, st)) != GDN_OK)
            return s;
        flags &= ~GDN_CHECK_INPUTS;
    }

    if (flags & GDN_LAYER_FUSED_VCONV) {
        // the q/k channels' conv, then the scan, whose state pass convolves each V tile
        // from x itself (and writes y's v channels and their conv states): the v channels
        // make no round trip through memory before the scan
        if ((flags & GDN_PREFILL_SIMT) || !gdn_host::chunk_tc_supported(dk, dv, 64, 0))
            return GDN_ERR_UNSUPPORTED;
        s = gdn_host::launch_conv1d_fwd(x, C, conv_w, conv_bias, cu_seqlens_dev, N, max_len,
                                        conv_state_in, conv_state_out, y, st, 0,
                                        (int32_t)(2 * qk));
        if (s != GDN_OK) return s;
        gdn_host::VConvArgs vc;
        vc.x = x;
        vc.y = y;
        vc.w = conv_w;
        vc.b = conv_bias;
        vc.s_in = conv_state_in;
        vc.s_out = conv_state_out;
        vc.xc = C;
        vc.cv0 = (int32_t)(2 * qk);
        return chunk_prefill_impl(&tq, &tk, &tv, g, beta, cu_seqlens_dev, cu_seqlens_host, N,
                                  64, scale, flags, initial_state, &to, final_state, workspace,
                                  workspace_bytes, status_dev, stream, nullptr, 0, &vc);
    }
    if (!side_stream) {
        // one stream: the conv over every channel, then the chunk scan
        s = gdn_host::launch_conv1d_fwd(x, C, conv_w, conv_bias, cu_seqlens_dev, N, max_len,
                                        conv_state_in, conv_state_out, y, st);
        if (s != GDN_OK) return s;
        return chunk_prefill_impl(&tq, &tk, &tv, g, beta, cu_seqlens_dev, cu_seqlens_host, N,
                                  64, scale, flags, initial_state, &to, final_state, workspace,
                                  workspace_bytes, status_dev, stream, nullptr);
    }
    // fork: the v channels' conv on the caller's side stream, the q/k channels' conv and
    // the chunk preparation (which reads only q and k) on `stream`; the state pass waits
    // for v.  Events live only for this call.
    cudaStream_t side = (cudaStream_t)side_stream;
    cudaEvent_t fork = nullptr, v_ready = nullptr;
    if (cudaEventCreateWithFlags(&fork, cudaEventDisableTiming) != cudaSuccess) return GDN_ERR_CUDA;
    if (cudaEventCreateWithFlags(&v_ready, cudaEventDisableTiming) != cudaSuccess) {
        cudaEventDestroy(fork);
        return GDN_ERR_CUDA;
    }
    s = GDN_OK;
    if (cudaEventRecord(fork, st) != cudaSuccess || cudaStreamWaitEvent(side, fork, 0) != cudaSuccess)
        s = GDN_ERR_CUDA;
    // the q/k conv is launched first so its blocks are dispatched ahead of the v conv's
    if (s == GDN_OK)
        s = gdn_host::launch_conv1d_fwd(x, C, conv_w, conv_bias, cu_seqlens_dev, N, max_len,
                                        conv_state_in, conv_state_out, y, st, 0,
                                        (int32_t)(2 * qk));
    if (s == GDN_OK)
        s = gdn_host::launch_conv1d_fwd(x, C, conv_w, conv_bias, cu_seqlens_dev, N, max_len,
                                        conv_state_in, conv_state_out, y, side,
                                        (int32_t)(2 * qk), C);
    if (s == GDN_OK && cudaEventRecord(v_ready, side) != cudaSuccess) s = GDN_ERR_CUDA;
    if (s == GDN_OK)
        s = chunk_prefill_impl(&tq, &tk, &tv, g, beta, cu_seqlens_dev, cu_seqlens_host, N, 64,
                               scale, flags, initial_state, &to, final_state, workspace,
                               workspace_bytes, status_dev, stream, v_ready);
    // the caller's stream joins the side stream even if a launch failed
    if (cudaStreamWaitEvent(st, v_ready, 0) != cudaSuccess && s == GDN_OK) s = GDN_ERR_CUDA;
    cudaEventDestroy(fork);
    cudaEventDestroy(v_ready);
    return s;
}

gdn_status_t gdn_selftest_bounded_wait(int32_t *status_dev, void *stream) {
    gdn_host::CallRange nvtx_range("gdn_selftest_bounded_wait");
    if (!status_dev) return GDN_ERR_NULL;
    return gdn_host::launch_wait_selftest(status_dev, (cudaStream_t)stream);
}

}  // extern "C"
