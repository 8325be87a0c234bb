// Gated DeltaNet forward: placeholder until the kernels land.
#include "common.cuh"

namespace llattn {
size_t gdn_workspace(const ll_shape&) { return 0; }
ll_status gdn_launch(const FwdArgs&) { return LL_ERR_UNSUPPORTED; }
}  // namespace llattn
