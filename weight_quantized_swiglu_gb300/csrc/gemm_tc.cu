// gemm_tc.cu -- tensor-core prefill GEMM (placeholder until the tcgen05
// kernel lands: reports the GEMM family as unavailable).
#include "internal.h"

namespace qmlp {
bool gemm_supported(int, int) { return false; }
size_t gemm_tiles_bytes(int, int) { return 0; }
cudaError_t repack_nvfp4_gemm(const uint8_t*, const uint8_t*, const uint8_t*, const uint8_t*, int, int, bool,
                              uint8_t*, cudaStream_t) {
    return cudaErrorNotSupported;
}
cudaError_t launch_gemm(const GemmLaunch&, int, cudaStream_t) { return cudaErrorNotSupported; }
}  // namespace qmlp
