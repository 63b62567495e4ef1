// noalloc.cu -- gdn_chunk_prefill_noalloc: the chunked prefill for callers that cannot
// allocate device memory.
//
// Some callers cannot call cudaMalloc at all: an engine whose allocator has reserved the
// whole device up front, a latency-critical loop where an allocation (and the device
// synchronisation it may imply) is not acceptable, or a host program that embeds only
// this library and has no device allocator of its own.  gdn_chunk_prefill asks those
// callers for a workspace; this entry point instead uses a fixed scratch array that lives
// in this library's device image, so the caller passes only inputs and outputs.
//
// The array is GDN_NOALLOC_SCRATCH_BYTES (128 MiB).  Every GPU that loads the library
// holds it until the process exits.  Host code cannot use the array's name as a device
// address: the first call on each device looks the address up with cudaGetSymbolAddress
// (with that device current) and caches it.
#include <mutex>

#include "common.cuh"

namespace {

// Scratch for the tensor-core prefill's per-chunk workspace tiles ([W ; Q'], Z and the
// per-token scalars).  Every byte the kernels read in a call is first written by the same
// call, so nothing is cleared.
__device__ __align__(256) uint8_t gdn_noalloc_scratch[GDN_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void *g_scratch_addr[kMaxDevices] = {nullptr};

gdn_status_t scratch_for_current_device(void **out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return GDN_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!g_scratch_addr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, gdn_noalloc_scratch) != cudaSuccess || !p) return GDN_ERR_CUDA;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return GDN_OK;
}

}  // namespace

extern "C" gdn_status_t gdn_chunk_prefill_noalloc(
    const gdn_tensor_t *q, const gdn_tensor_t *k, const gdn_tensor_t *v, const float *g,
    const float *beta, const int32_t *cu_seqlens_dev, const int32_t *cu_seqlens_host,
    int32_t N, int32_t chunk, float scale, uint32_t flags, const float *initial_state,
    const gdn_tensor_t *o, float *final_state, int32_t *status_dev, void *stream) {
    gdn_host::CallRange nvtx_range("gdn_chunk_prefill_noalloc");
    if (!q || !v || !cu_seqlens_host) return GDN_ERR_NULL;
    if (q->ndim < 3 || q->ndim > 4 || v->ndim != q->ndim) return GDN_ERR_SHAPE;
    const int off = q->ndim - 3;
    // fp32 activations always run on the CUDA-core kernel, which needs no scratch
    const size_t need = q->dtype == GDN_F32
        ? 0
        : gdn_chunk_prefill_workspace_size(
              N, q->shape[off], (int32_t)q->shape[off + 1], (int32_t)v->shape[off + 1],
              (int32_t)q->shape[off + 2], (int32_t)v->shape[off + 2], chunk, flags);
    if (need > (size_t)GDN_NOALLOC_SCRATCH_BYTES) return GDN_ERR_WORKSPACE;
    void *scratch = nullptr;
    if (need > 0) {
        const gdn_status_t s = scratch_for_current_device(&scratch);
        if (s != GDN_OK) return s;
    }
    return gdn_chunk_prefill(q, k, v, g, beta, cu_seqlens_dev, cu_seqlens_host, N, chunk,
                             scale, flags, initial_state, o, final_state, scratch, need,
                             status_dev, stream);
}
