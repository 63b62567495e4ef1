// chunk_tc.cu -- tensor-core (tcgen05 / TMEM / TMA) chunked gated delta rule.
// Placeholder: no shape is routed here yet.
#include "common.cuh"

namespace gdn_host {

bool chunk_tc_supported(int32_t, int32_t, int32_t, int) { return false; }

size_t chunk_tc_workspace(int32_t, int64_t, int32_t, int32_t) { return 0; }

gdn_status_t launch_chunk_tc(const ScanArgs &, const int32_t *, cudaStream_t) {
    return GDN_ERR_UNSUPPORTED;
}

}  // namespace gdn_host
