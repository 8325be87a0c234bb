// Tensor-core (tcgen05) forward: placeholder until the kernel lands.
#include "common.cuh"

namespace llattn {
bool fwd_tc_supported(const ll_shape&) { return false; }
size_t fwd_tc_workspace(const ll_shape&) { return 0; }
ll_status fwd_tc_launch(const FwdArgs&) { return LL_ERR_UNSUPPORTED; }
int fwd_tc_launches(const ll_shape&) { return 1; }
}  // namespace llattn
