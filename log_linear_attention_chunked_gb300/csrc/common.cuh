// Shared host/device helpers of libllattn (internal; not part of the C ABI).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/ll_attn.h"

namespace llattn {

// Bits of the device error word (read back by ll_last_device_error).
enum : unsigned { kErrTimeout = 1u, kErrDeviceArg = 2u };

// Device address of the library's error word on the current device.
unsigned* err_word();

__device__ __forceinline__ void raise_error(unsigned* err, unsigned bit) { atomicOr(err, bit); }

__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T> __device__ __forceinline__ T from_f(float x);
template <> __device__ __forceinline__ float from_f<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

// bit length of a positive integer (0 for 0): the level of key s for query t
// is bit_length(t xor s).
__device__ __forceinline__ int bitlen(unsigned x) { return 32 - __clz(x); }

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

inline bool is_pow2_in(int x, int lo, int hi) { return x >= lo && x <= hi && (x & (x - 1)) == 0; }

inline int ilog2(int x) {
  int r = 0;
  while ((1 << (r + 1)) <= x) ++r;
  return r;
}

// Number of lambda levels a sequence of length T touches.
inline int levels_needed(int T) {
  if (T <= 1) return 1;
  int b = 0;
  unsigned x = (unsigned)(T - 1);
  while (x) { ++b; x >>= 1; }
  return b + 1;
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

#define LL_CUDA_OK(expr)                          \
  do {                                            \
    cudaError_t e_ = (expr);                      \
    if (e_ != cudaSuccess) return LL_ERR_CUDA;    \
  } while (0)

// ---- launchers implemented in the kernel translation units ----
struct FwdArgs {
  ll_shape s;
  const void *q, *k, *v;
  const float *log_alpha, *lam, *beta;
  void* o;
  float *state_out, *scale_out;
  void* ws;
  size_t ws_bytes;
  cudaStream_t stream;
  unsigned* err;
  // prefill continuation: the tokens are positions t0 .. t0+T-1 and the
  // decode states of position t0 (state_in/scale_in, Ls slots) carry the prefix
  long long t0 = 0;
  const float* state_in = nullptr;
  const float* scale_in = nullptr;
  // limit of every bounded device-side wait of the tensor-core forward
  // (0 = the library default); and the test hook of its expiry: the index of
  // one Fenwick node whose publication word is never written (-1 = none)
  uint64_t timeout_ns = 0;
  long long withhold_node = -1;
  // row stride (tokens) between the (b, h) slices of q, k, v, o, log_alpha
  // and lam when it differs from s.T (the tensor-core forward of the whole
  // tiles of a longer sequence); 0 = s.T
  int rows_per_head = 0;
};

size_t fwd_simt_workspace(const ll_shape& s);
size_t fwd_simt_cont_workspace(const ll_shape& s);
// the decode states of t0 + T after a continuation (both forward paths)
ll_status cont_export_launch(const float* pre_states, const float* pre_scales, const float* seg_states,
                             const float* seg_scales, const float* log_alpha, float* seg_decay, float* state_out,
                             float* scale_out, int BH, int T, int mat, int Ls, long long t0, cudaStream_t stream);
ll_status fwd_simt_launch(const FwdArgs& a);
int fwd_simt_launches(const ll_shape& s);

bool fwd_tc_supported(const ll_shape& s);
size_t fwd_tc_workspace(const ll_shape& s);
bool fwd_tc_cont_supported(const ll_shape& s, long long t0);
size_t fwd_tc_cont_workspace(const ll_shape& s);
ll_status fwd_tc_launch(const FwdArgs& a);
int fwd_tc_launches(const ll_shape& s);

ll_status decode_launch(int B, int H, int dk, int dv, int Ls, ll_dtype io, const int64_t* t, const void* q,
                        const void* k, const void* v, const float* log_alpha, const float* lam, float* states,
                        float* scales, void* o, cudaStream_t stream, unsigned* err);

ll_status gdn_decode_launch(int B, int H, int dk, int dv, int Ls, ll_dtype io, const int64_t* t, const void* q,
                            const void* k, const void* v, const float* log_alpha, const float* beta,
                            const float* lam, float* states, void* o, cudaStream_t stream, unsigned* err);
// Gated DeltaNet forward (reading A) on the tensor cores: bf16 io, d = 128,
// T a multiple of 128 (at most 256 chunks of 128 tokens)
bool gdn_tc_supported(const ll_shape& s);
size_t gdn_tc_workspace(const ll_shape& s);
ll_status gdn_tc_launch(const FwdArgs& a);
size_t gdn_workspace(const ll_shape& s);
ll_status gdn_launch(const FwdArgs& a);
size_t gdn_b_workspace(const ll_shape& s);
ll_status gdn_b_launch(const FwdArgs& a);

}  // namespace llattn
