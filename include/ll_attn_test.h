/*
 * ll_attn_test.h -- test hooks of libllattn.so (not for production use).
 *
 * The pages have no counterpart of anything here.  These entry points exist
 * so that failure handling can be tested without a GPU fault: every wait of
 * a kernel on data another CTA publishes is bounded, and a wait that expires
 * must end the kernel cleanly with LL_ERR_TIMEOUT reported by
 * ll_last_device_error() and the CUDA context still usable.
 */
#ifndef LL_ATTN_TEST_H
#define LL_ATTN_TEST_H

#include "ll_attn.h"

#ifdef __cplusplus
extern "C" {
#endif

/* ll_attn_fwd on the tensor-core path (bf16 io, dk = dv = 128, T a multiple
 * of 128), with one Fenwick node never published and a short wait limit.
 *   shape, q, k, v, log_alpha, lam, o, workspace, ws_bytes, stream: as
 *              ll_attn_fwd (shape->Ls must be 0)
 *   node       index of the node to withhold, head-major over the 128-token
 *              tiles: bh * (T / 128) + tile, in [0, B*H*T/128)
 *   timeout_ns limit of every bounded wait of the kernel, in
 *              [100000, 4000000000] (0.1 ms .. 4 s)
 * Every tile that needs the withheld node (its later levels, the merges that
 * look back over it) waits for its publication word until the limit, then
 * the kernel records LL_ERR_TIMEOUT in the device error word, stops arming
 * copies, drains the ones in flight and runs to its end.  The returned status
 * covers the launch only; the output is unspecified.  Returns
 * LL_ERR_UNSUPPORTED for a shape off the tensor-core path and
 * LL_ERR_INVALID_ARG for a node or limit out of range, before any launch. */
LL_API ll_status ll_test_fwd_withhold_node(const ll_shape* shape, const void* q, const void* k, const void* v,
                                           const float* log_alpha, const float* lam, void* o, void* workspace,
                                           size_t ws_bytes, long long node, unsigned long long timeout_ns,
                                           void* stream);

#ifdef __cplusplus
}
#endif

#endif /* LL_ATTN_TEST_H */
