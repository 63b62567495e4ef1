// common.cuh -- small device helpers shared by the GDN kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>
#include <stdint.h>

#include "../../include/gdn.h"

namespace gdn {

typedef __nv_bfloat16 bf16;

// 8 bf16 packed in 16 bytes <-> 8 floats.
__device__ __forceinline__ void unpack8(const uint4 &u, float f[8]) {
    const __nv_bfloat162 *p = reinterpret_cast<const __nv_bfloat162 *>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float2 t = __bfloat1622float2(p[i]);
        f[2 * i] = t.x;
        f[2 * i + 1] = t.y;
    }
}

__device__ __forceinline__ uint4 pack8(const float f[8]) {
    uint4 u;
    __nv_bfloat162 *p = reinterpret_cast<__nv_bfloat162 *>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) p[i] = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
    return u;
}

// SiLU z / (1 + e^-z), with e^-z = 2^(-z log2 e) on the hardware base-2 exponential
// (ex2.approx, relative error about 2^-22) and the fast divide: the result is rounded to
// bf16, whose unit roundoff (2^-9) is far above either error.  For z below about -88,
// e^-z overflows to infinity and the result is a signed zero (the exact value is under
// 1e-36 in magnitude).
__device__ __forceinline__ float silu(float z) {
    constexpr float kMinusLog2e = -1.4426950408889634f;
    float e;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e) : "f"(z * kMinusLog2e));
    return __fdividef(z, 1.0f + e);
}

template <typename T> __device__ __forceinline__ float to_f32(T x);
template <> __device__ __forceinline__ float to_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ float to_f32<bf16>(bf16 x) { return __bfloat162float(x); }

template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ bf16 from_f32<bf16>(float x) { return __float2bfloat16_rn(x); }

// Record a device-side error without faulting: first writer wins.
__device__ __forceinline__ void report(int32_t *status, int32_t code) {
    if (status) atomicCAS(status, 0, code);
}

// Programmatic dependent launch.  The prefill kernels are launched so that they may start
// while the previous kernel of the stream drains; before touching global memory each
// grid waits until every prerequisite grid has completed and its writes are visible, and
// it lets its own dependents start launching as soon as all of its CTAs are running.
__device__ __forceinline__ void grid_dependency_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void grid_dependents_launch() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

}  // namespace gdn

namespace gdn_host {
// One NVTX range per call of the C ABI, named after the entry point, so that a timeline
// tool (Nsight Systems, or ncu's --nvtx filters) shows each call and the kernels it
// launched.  The NVTX v3 header needs no library: with no tool attached, a push or pop is
// one call through a pointer that the first use resolves.
struct CallRange {
    explicit CallRange(const char *name) { nvtxRangePushA(name); }
    ~CallRange() { nvtxRangePop(); }
    CallRange(const CallRange &) = delete;
    CallRange &operator=(const CallRange &) = delete;
};

// cudaLaunchKernelEx with programmatic stream serialization allowed.
template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                             cudaStream_t st, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}
}  // namespace gdn_host

// Host-side launch helpers (defined in api.cu).
namespace gdn_host {
// channels [c_begin, c_end) of the C-wide rows (c_end < 0: all)
gdn_status_t launch_conv1d_fwd(const void *x, int32_t C, const void *w, const void *bias,
                               const int32_t *cu, int32_t N, int32_t max_len,
                               const void *s_in, void *s_out, void *y, cudaStream_t st,
                               int32_t c_begin = 0, int32_t c_end = -1);
gdn_status_t launch_conv1d_update(const void *x, int32_t N, int32_t C, const void *w,
                                  const void *bias, void *state, int32_t P,
                                  const int32_t *idx, void *y, int32_t *status,
                                  cudaStream_t st);

// The layer's v-channel conv, fused into the tensor-core state pass: V is then computed
// from the raw activations x (its channels cv0.. of rows xc wide) instead of read.
struct VConvArgs {
    const void *x;           // raw activations [T][xc] bf16
    void *y;                 // conv output [T][xc] bf16: the state pass writes its v channels
    const void *w, *b;       // taps [xc][4] bf16; bias [xc] bf16 or null
    const void *s_in;        // conv states [N][3][xc] bf16, or null for zeros
    void *s_out;             // new conv states [N][3][xc] bf16, or null
    int64_t xc;
    int32_t cv0;
};

struct ScanArgs {
    const void *q, *k, *v;
    void *o;
    int64_t q_tok, k_tok, v_tok, o_tok;  // token strides in elements
    const float *g, *beta;
    const int32_t *cu;       // device [N+1]
    const float *h0;         // [N,Hv,dk,dv] or null
    float *hT;               // [N,Hv,dk,dv] or null
    int32_t N, Hk, Hv, dk, dv, chunk;
    int64_t T;
    int32_t max_len;         // longest sequence (host-computed)
    float scale;
    uint32_t flags;
    int in_f32, out_f32;     // dtypes
    int32_t *status;
    void *ws;
    size_t ws_bytes;
    const VConvArgs *vconv;  // null: V is read from v
};
gdn_status_t launch_chunk_simt(const ScanArgs &a, cudaStream_t st);
// before_state: an event the state kernel's launch waits on (the producer of v), or NULL
gdn_status_t launch_chunk_tc(const ScanArgs &a, const int32_t *cu_host, cudaStream_t st,
                             cudaEvent_t before_state = nullptr);
size_t chunk_tc_workspace(int32_t N, int64_t T, int32_t Hk, int32_t Hv);
// The context-parallel scan: each sequence in ranges of range_chunks chunks (cu_host: the
// host copy of cu).  Workspace bytes (0 when the arguments are invalid) and the launch.
size_t chunk_tc_cp_workspace(const int32_t *cu_host, int32_t N, int64_t T, int32_t Hk,
                             int32_t Hv, int32_t range_chunks);
// range length for one sequence of seq_len tokens alone on the current device, or on a
// device with sms SMs (0: plain)
int32_t cp_range_hint(int64_t seq_len, int32_t Hv);
int32_t cp_range_hint(int64_t seq_len, int32_t Hv, int32_t sms);
gdn_status_t launch_chunk_tc_cp(const ScanArgs &a, const int32_t *cu_host, int32_t range_chunks,
                                cudaStream_t st);
// one CTA whose bounded mbarrier wait runs out (GDN_ERR_TIMEOUT into *status)
gdn_status_t launch_wait_selftest(int32_t *status, cudaStream_t st);
bool chunk_tc_supported(int32_t dk, int32_t dv, int32_t chunk, int in_f32);

struct DecodeArgs {
    const void *q, *k, *v;
    void *o;
    int64_t q_tok, k_tok, v_tok, o_tok;
    const float *g, *beta;
    float *state;
    const int32_t *idx;
    int32_t N, P, Hk, Hv, dk, dv;
    float scale;
    uint32_t flags;
    int in_f32, out_f32;
    int32_t *status;
};
gdn_status_t launch_decode(const DecodeArgs &a, cudaStream_t st);

struct FusedDecodeArgs {
    const void *x, *w, *bias;   // x [N, C] bf16; w [C, 4] bf16; bias [C] bf16 or NULL
    void *conv_state;           // [P, 3, C] bf16, shifted in place
    const float *a_raw, *b_raw; // [N, Hv] fp32 gate logits
    float *state;               // [P, Hv, 128, 128] fp32, in place
    const int32_t *idx;         // [N] or NULL (identity)
    void *o;                    // [N, Hv, 128] bf16
    int32_t N, P, Hk, Hv, C;
    float scale;
    uint32_t flags;
    int32_t *status;
};
gdn_status_t launch_fused_decode(const FusedDecodeArgs &a, cudaStream_t st);
}  // namespace gdn_host
