// compose_tc.cu -- GDN chain composition on the tensor cores (placeholder).
#include "kernels.h"
namespace hypic {
bool compose_tc_supported(const ComposeParams&) { return false; }
cudaError_t launch_compose_tc(const ComposeParams&, unsigned*, cudaStream_t) { return cudaErrorNotSupported; }
}  // namespace hypic
