// Tensor-core path (not built yet: every geometry goes to the SIMT kernels).
#include "tc_decode.h"

namespace mla {

bool tc_decode_supported(const mla_dims&) { return false; }
cudaError_t tc_decode_workspace(int32_t, int32_t, const mla_dims&, size_t* bytes) {
    *bytes = 0;
    return cudaErrorNotSupported;
}
cudaError_t launch_decode_tc(void*, float*, const void*, const void*, const int32_t*,
                             const int32_t*, int32_t, int32_t, int32_t, const mla_dims&, float,
                             void*, int32_t*, cudaStream_t) {
    return cudaErrorNotSupported;
}
bool tc_gemm_supported(const mla_dims&, int32_t, bool) { return false; }
cudaError_t launch_absorb_tc(void*, const void*, const void*, const void*, int32_t,
                             const mla_dims&, cudaStream_t) {
    return cudaErrorNotSupported;
}
cudaError_t launch_decompress_tc(void*, const void*, const void*, int32_t, const mla_dims&,
                                 cudaStream_t) {
    return cudaErrorNotSupported;
}

}  // namespace mla
