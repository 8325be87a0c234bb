// Test hooks of the C ABI (include/ll_attn_test.h): the tensor-core forward
// with one node's publication withheld and a short wait limit, so a test can
// make a bounded wait expire without faulting or hanging the GPU.
#include "../../include/ll_attn_test.h"
#include "common.cuh"

using namespace llattn;

extern "C" ll_status ll_test_fwd_withhold_node(const ll_shape* s, const void* q, const void* k, const void* v,
                                               const float* log_alpha, const float* lam, void* o, void* workspace,
                                               size_t ws_bytes, long long node, unsigned long long timeout_ns,
                                               void* stream) {
  if (!s || s->Ls != 0) return LL_ERR_INVALID_ARG;
  if (ll_attn_fwd_workspace_size(s) == 0) return LL_ERR_INVALID_ARG;  // the shape checks of ll_attn_fwd
  if (!fwd_tc_supported(*s)) return LL_ERR_UNSUPPORTED;
  if (!q || !k || !v || !log_alpha || !lam || !o) return LL_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(log_alpha) || !aligned16(lam) ||
      !aligned16(o))
    return LL_ERR_INVALID_ARG;
  const long long nodes = (long long)s->B * s->H * (s->T / 128);
  if (node < 0 || node >= nodes) return LL_ERR_INVALID_ARG;
  if (timeout_ns < 100000ull || timeout_ns > 4000000000ull) return LL_ERR_INVALID_ARG;
  if (!workspace || ws_bytes < fwd_tc_workspace(*s)) return LL_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return LL_ERR_WORKSPACE;
  FwdArgs a{*s, q, k, v, log_alpha, lam, nullptr, o, nullptr, nullptr, workspace, ws_bytes,
            static_cast<cudaStream_t>(stream), err_word()};
  if (!a.err) return LL_ERR_CUDA;
  a.timeout_ns = timeout_ns;
  a.withhold_node = node;
  return fwd_tc_launch(a);
}
