// Launchers of the forms with one decay per level (internal; not part of the C ABI).
#pragma once

#include "common.cuh"

namespace llattn {

// the forward, log_alpha [B,H,T,L]; the workspace size is 0 (and the launch
// LL_ERR_UNSUPPORTED) beyond 4096 chunks
size_t fwd_level_decay_workspace(const ll_shape& s);
int fwd_level_decay_launches(const ll_shape& s);
ll_status fwd_level_decay_launch(const FwdArgs& a);

// the same on the tensor cores: bf16 io, d = 128, T a multiple of 128, L <= 16
bool fwd_tc_level_decay_supported(const ll_shape& s);
size_t fwd_tc_level_decay_workspace(const ll_shape& s);
int fwd_tc_level_decay_launches(const ll_shape& s);
ll_status fwd_tc_level_decay_launch(const FwdArgs& a);

// the decode step, log_alpha [B,H,Ls+1] (entry l for level l)
ll_status decode_level_decay_launch(int B, int H, int dk, int dv, int Ls, ll_dtype io, const int64_t* t,
                                    const void* q, const void* k, const void* v, const float* log_alpha,
                                    const float* lam, float* states, float* scales, void* o, cudaStream_t stream,
                                    unsigned* err);

}  // namespace llattn
