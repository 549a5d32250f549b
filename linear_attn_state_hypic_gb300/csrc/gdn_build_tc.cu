// gdn_build_tc.cu -- chunked GDN build on the tensor cores (placeholder: the
// dispatcher falls back to the CUDA-core build until this path exists).
#include "kernels.h"
namespace hypic {
bool gdn_build_tc_supported(const BuildParams&) { return false; }
cudaError_t launch_gdn_build_tc(const BuildParams&, void*, unsigned*, cudaStream_t) { return cudaErrorNotSupported; }
}  // namespace hypic
