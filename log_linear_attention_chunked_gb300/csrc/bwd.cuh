// Launchers of the backward (internal; not part of the C ABI).
#pragma once

#include "common.cuh"

namespace llattn {

// Fenwick nodes F, G of the chunk states S and chunk log-decays tot (BH heads
// of N chunks, matrices of `mat` floats); shared by the forward and backward.
// With Ft (d_k = d_v = 128) the nodes are also written as 128-byte-swizzled
// bf16 tiles, the operand layout of the tensor-core kernels; with cum, the
// running sums over the chunks of their log-decay totals ([BH, N] float64).
// With Ft, f32_nodes = false leaves F unwritten where the kernel allows it
// (for the consumers of the bf16 tiles alone): that is every N up to
// kFenwickOnChipChunks, whose chain stays on chip; beyond it the kernel reads
// the children back from F, so F must be there.
constexpr int kFenwickOnChipChunks = 4096;
ll_status simt_fenwick_launch(const float* S, float* F, const double* tot, double* G, int N, int mat, int BH,
                              cudaStream_t stream, __nv_bfloat16* Ft = nullptr, double* cum = nullptr,
                              bool f32_nodes = true);

struct BwdArgs {
  ll_shape s;
  const void *q, *k, *v, *dout;
  const float *log_alpha, *lam;
  void *dq, *dk, *dv;
  float *dlog_alpha, *dlam;
  void* ws;
  size_t ws_bytes;
  cudaStream_t stream;
  unsigned* err;
};
size_t bwd_simt_workspace(const ll_shape& s);
int bwd_simt_launches(const ll_shape& s);
ll_status bwd_simt_launch(const BwdArgs& a);
// the tensor-core backward (bf16 io, d_k = d_v = 128, 128-token tiles) on
// buffers laid out by the CUDA-core backward's plan
struct BwdTcBuffers {
  __nv_bfloat16 *dqp, *dkp, *dvp;  // the in-tile parts of dq, dk, dv (bf16)
  float *S, *F, *R;
  __nv_bfloat16* Ft;  // the nodes F as bf16 tiles
  double *tot, *G, *cum;
  float* dc;
  unsigned* err;
};
bool bwd_tc_supported(const ll_shape& s);
ll_status bwd_tc_launch(const BwdArgs& a, const BwdTcBuffers& b);

}  // namespace llattn
