// C ABI entry points of libllattn: argument checks, path selection, launch.
//
// Every check here runs on the host before anything is launched, so an
// invalid call never touches device memory.
#include <mutex>

#include "bwd.cuh"

namespace llattn {

__device__ unsigned g_err_word = 0;

static constexpr int kMaxDevices = 64;

unsigned* err_word() {
  static std::mutex mu;
  static unsigned* addr[kMaxDevices] = {nullptr};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_err_word) != cudaSuccess) return nullptr;
    addr[dev] = static_cast<unsigned*>(p);
  }
  return addr[dev];
}

static bool head_dim_ok(int d) { return is_pow2_in(d, 16, 128); }

// Shape checks shared by the forward entry points.
static ll_status check_shape(const ll_shape* s) {
  if (!s) return LL_ERR_INVALID_ARG;
  if (s->B < 1 || s->H < 1 || s->T < 1) return LL_ERR_INVALID_ARG;
  if (s->io != LL_F32 && s->io != LL_BF16) return LL_ERR_INVALID_ARG;
  if (!is_pow2_in(s->chunk, 16, 128)) return LL_ERR_INVALID_ARG;
  if (s->L < levels_needed(s->T) || s->L > 64) return LL_ERR_INVALID_ARG;
  if (s->Ls < 0 || s->Ls > 62) return LL_ERR_INVALID_ARG;
  if (!head_dim_ok(s->dk) || !head_dim_ok(s->dv)) return LL_ERR_UNSUPPORTED;
  // element counts must stay addressable with 64-bit offsets and 32-bit T
  return LL_OK;
}

}  // namespace llattn

using namespace llattn;

extern "C" {

int ll_version(void) { return 100; }

const char* ll_status_str(ll_status s) {
  switch (s) {
    case LL_OK: return "ok";
    case LL_ERR_INVALID_ARG: return "invalid argument";
    case LL_ERR_UNSUPPORTED: return "unsupported shape or dtype";
    case LL_ERR_CUDA: return "CUDA error";
    case LL_ERR_TIMEOUT: return "device-side wait timed out";
    case LL_ERR_WORKSPACE: return "workspace missing or too small";
    case LL_ERR_DEVICE: return "device-side argument check failed";
  }
  return "unknown status";
}

ll_status ll_last_device_error(void* stream) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  unsigned* ew = err_word();
  if (!ew) return LL_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return LL_ERR_CUDA;
  unsigned h = 0;
  if (cudaMemcpyFromSymbolAsync(&h, g_err_word, sizeof(h), 0, cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return LL_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return LL_ERR_CUDA;
  if (h) {
    unsigned zero = 0;
    if (cudaMemcpyToSymbolAsync(g_err_word, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice, st) != cudaSuccess)
      return LL_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return LL_ERR_CUDA;
  }
  if (h & kErrTimeout) return LL_ERR_TIMEOUT;
  if (h & kErrDeviceArg) return LL_ERR_DEVICE;
  return LL_OK;
}

size_t ll_attn_fwd_workspace_size(const ll_shape* s) {
  if (check_shape(s) != LL_OK) return 0;
  if (fwd_tc_supported(*s)) return fwd_tc_workspace(*s);
  return fwd_simt_workspace(*s);
}

int ll_attn_fwd_launches(const ll_shape* s) {
  if (check_shape(s) != LL_OK) return 0;
  if (fwd_tc_supported(*s)) return fwd_tc_launches(*s);
  return fwd_simt_launches(*s);
}

ll_status ll_attn_fwd(const ll_shape* s, const void* q, const void* k, const void* v, const float* log_alpha,
                      const float* lam, void* o, float* state_out, float* scale_out, void* workspace,
                      size_t ws_bytes, void* stream) {
  ll_status st = check_shape(s);
  if (st != LL_OK) return st;
  if (!q || !k || !v || !log_alpha || !lam || !o) return LL_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(log_alpha) || !aligned16(lam) ||
      !aligned16(o))
    return LL_ERR_INVALID_ARG;
  if ((state_out == nullptr) != (scale_out == nullptr)) return LL_ERR_INVALID_ARG;
  if (state_out) {
    if (s->Ls < 1 || !aligned16(state_out) || !aligned16(scale_out)) return LL_ERR_INVALID_ARG;
    int need = 0;
    for (unsigned x = (unsigned)s->T; x; x >>= 1) ++need;  // bit_length(T)
    if (s->Ls < need) return LL_ERR_INVALID_ARG;
  }
  const bool tc = fwd_tc_supported(*s);
  const size_t need_ws = tc ? fwd_tc_workspace(*s) : fwd_simt_workspace(*s);
  if (!workspace || ws_bytes < need_ws) return LL_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return LL_ERR_WORKSPACE;
  FwdArgs a{*s, q, k, v, log_alpha, lam, nullptr, o, state_out, scale_out, workspace, ws_bytes,
            static_cast<cudaStream_t>(stream), err_word()};
  if (!a.err) return LL_ERR_CUDA;
  return tc ? fwd_tc_launch(a) : fwd_simt_launch(a);
}

// Shape conditions of a prefill continuation at position t0 (beyond check_shape).
static ll_status check_cont(const ll_shape* s, long long t0) {
  ll_status st = check_shape(s);
  if (st != LL_OK) return st;
  if (t0 < 0 || t0 > (1ll << 61)) return LL_ERR_INVALID_ARG;
  const long long T = s->T, t1 = t0 + T;
  long long P = 1;
  while (P < T) P <<= 1;
  if (t0 % P != 0) return LL_ERR_INVALID_ARG;  // the segment must sit in one aligned block
  int bl = 0;
  for (long long x = t1; x; x >>= 1) ++bl;
  if (s->Ls < 1 || s->Ls < bl) return LL_ERR_INVALID_ARG;  // the levels of t1 need slots
  int need = 1;
  for (long long x = t1 - 1; x; x >>= 1) ++need;
  if (s->L < need) return LL_ERR_INVALID_ARG;  // the segment's keys reach levels up to bitlen(t1 - 1)
  return LL_OK;
}

size_t ll_attn_fwd_cont_workspace_size(const ll_shape* s, long long t0) {
  if (check_cont(s, t0) != LL_OK) return 0;
  return fwd_tc_cont_supported(*s, t0) ? fwd_tc_cont_workspace(*s) : fwd_simt_cont_workspace(*s);
}

ll_status ll_attn_fwd_cont(const ll_shape* s, long long t0, const float* state_in, const float* scale_in,
                           const void* q, const void* k, const void* v, const float* log_alpha, const float* lam,
                           void* o, float* state_out, float* scale_out, void* workspace, size_t ws_bytes,
                           void* stream) {
  ll_status st = check_cont(s, t0);
  if (st != LL_OK) return st;
  if (!state_in || !scale_in || !q || !k || !v || !log_alpha || !lam || !o) return LL_ERR_INVALID_ARG;
  if ((state_out == nullptr) != (scale_out == nullptr)) return LL_ERR_INVALID_ARG;
  if (!aligned16(state_in) || !aligned16(scale_in) || !aligned16(q) || !aligned16(k) || !aligned16(v) ||
      !aligned16(log_alpha) || !aligned16(lam) || !aligned16(o) || (state_out && !aligned16(state_out)) ||
      (scale_out && !aligned16(scale_out)))
    return LL_ERR_INVALID_ARG;
  if (state_out) {  // the new states are written while the old ones are read
    const size_t n = (size_t)s->B * s->H * s->Ls * s->dv * s->dk * sizeof(float);
    const size_t ns = (size_t)s->B * s->H * s->Ls * sizeof(float);
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(state_in), a1 = reinterpret_cast<uintptr_t>(state_out);
    const uintptr_t c0 = reinterpret_cast<uintptr_t>(scale_in), c1 = reinterpret_cast<uintptr_t>(scale_out);
    if (a0 < a1 + n && a1 < a0 + n) return LL_ERR_INVALID_ARG;
    if (c0 < c1 + ns && c1 < c0 + ns) return LL_ERR_INVALID_ARG;
  }
  const bool tc = fwd_tc_cont_supported(*s, t0);
  const size_t need_ws = tc ? fwd_tc_cont_workspace(*s) : fwd_simt_cont_workspace(*s);
  if (!workspace || ws_bytes < need_ws) return LL_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return LL_ERR_WORKSPACE;
  FwdArgs a{*s, q, k, v, log_alpha, lam, nullptr, o, state_out, scale_out, workspace, ws_bytes,
            static_cast<cudaStream_t>(stream), err_word()};
  if (!a.err) return LL_ERR_CUDA;
  a.t0 = t0;
  a.state_in = state_in;
  a.scale_in = scale_in;
  return tc ? fwd_tc_launch(a) : fwd_simt_launch(a);
}

ll_status ll_attn_decode_step(int B, int H, int dk, int dv, int Ls, ll_dtype io, const int64_t* t, const void* q,
                              const void* k, const void* v, const float* log_alpha, const float* lam,
                              float* states, float* scales, void* o, void* stream) {
  if (B < 1 || H < 1 || Ls < 1 || Ls > 62) return LL_ERR_INVALID_ARG;
  if (io != LL_F32 && io != LL_BF16) return LL_ERR_INVALID_ARG;
  if (!head_dim_ok(dk) || !head_dim_ok(dv)) return LL_ERR_UNSUPPORTED;
  if (!t || !q || !k || !v || !log_alpha || !lam || !states || !scales || !o) return LL_ERR_INVALID_ARG;
  if (!aligned16(t) || !aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(log_alpha) ||
      !aligned16(lam) || !aligned16(states) || !aligned16(scales) || !aligned16(o))
    return LL_ERR_INVALID_ARG;
  unsigned* ew = err_word();
  if (!ew) return LL_ERR_CUDA;
  return decode_launch(B, H, dk, dv, Ls, io, t, q, k, v, log_alpha, lam, states, scales, o,
                       static_cast<cudaStream_t>(stream), ew);
}

size_t ll_attn_bwd_workspace_size(const ll_shape* s) {
  if (check_shape(s) != LL_OK || s->Ls != 0) return 0;
  return bwd_simt_workspace(*s);
}

int ll_attn_bwd_launches(const ll_shape* s) {
  if (check_shape(s) != LL_OK || s->Ls != 0) return 0;
  return bwd_simt_launches(*s);
}

ll_status ll_attn_bwd(const ll_shape* s, const void* q, const void* k, const void* v, const float* log_alpha,
                      const float* lam, const void* dout, void* dq, void* dk, void* dv, float* dlog_alpha,
                      float* dlam, void* workspace, size_t ws_bytes, void* stream) {
  ll_status st = check_shape(s);
  if (st != LL_OK) return st;
  if (s->Ls != 0) return LL_ERR_INVALID_ARG;
  const void* in[6] = {q, k, v, log_alpha, lam, dout};
  const void* out[5] = {dq, dk, dv, dlog_alpha, dlam};
  for (const void* p : in)
    if (!p || !aligned16(p)) return LL_ERR_INVALID_ARG;
  for (const void* p : out)
    if (!p || !aligned16(p)) return LL_ERR_INVALID_ARG;
  // the gradients are written while the inputs are still read: no output may
  // overlap an input or another output
  const size_t es = s->io == LL_F32 ? 4 : 2;
  const size_t rows = (size_t)s->B * s->H * s->T;
  const size_t in_bytes[6] = {rows * s->dk * es, rows * s->dk * es, rows * s->dv * es, rows * 4, rows * s->L * 4,
                              rows * s->dv * es};
  const size_t out_bytes[5] = {rows * s->dk * es, rows * s->dk * es, rows * s->dv * es, rows * 4, rows * s->L * 4};
  auto overlap = [](const void* a, size_t na, const void* b, size_t nb) {
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + nb && y < x + na;
  };
  for (int i = 0; i < 5; ++i) {
    for (int j = 0; j < 6; ++j)
      if (overlap(out[i], out_bytes[i], in[j], in_bytes[j])) return LL_ERR_INVALID_ARG;
    for (int j = i + 1; j < 5; ++j)
      if (overlap(out[i], out_bytes[i], out[j], out_bytes[j])) return LL_ERR_INVALID_ARG;
  }
  const size_t need_ws = bwd_simt_workspace(*s);
  if (!workspace || ws_bytes < need_ws) return LL_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return LL_ERR_WORKSPACE;
  BwdArgs a{*s, q, k, v, dout, log_alpha, lam, dq, dk, dv, dlog_alpha, dlam, workspace, ws_bytes,
            static_cast<cudaStream_t>(stream), err_word()};
  if (!a.err) return LL_ERR_CUDA;
  return bwd_simt_launch(a);
}

size_t ll_gdn_fwd_b_workspace_size(const ll_shape* s) {
  if (check_shape(s) != LL_OK || s->Ls != 0 || s->T % s->chunk != 0) return 0;
  return gdn_b_workspace(*s);
}

ll_status ll_gdn_fwd_b(const ll_shape* s, const void* q, const void* k, const void* v, const float* log_alpha,
                       const float* beta, const float* lam, void* o, void* workspace, size_t ws_bytes,
                       void* stream) {
  ll_status st = check_shape(s);
  if (st != LL_OK) return st;
  if (s->T % s->chunk != 0) return LL_ERR_INVALID_ARG;  // whole chunks only
  if (s->Ls != 0) return LL_ERR_INVALID_ARG;
  if (!q || !k || !v || !log_alpha || !beta || !lam || !o) return LL_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(log_alpha) || !aligned16(beta) ||
      !aligned16(lam) || !aligned16(o))
    return LL_ERR_INVALID_ARG;
  const size_t need_ws = gdn_b_workspace(*s);
  if (need_ws == 0) return LL_ERR_UNSUPPORTED;
  if (!workspace || ws_bytes < need_ws) return LL_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return LL_ERR_WORKSPACE;
  FwdArgs a{*s, q, k, v, log_alpha, lam, beta, o, nullptr, nullptr, workspace, ws_bytes,
            static_cast<cudaStream_t>(stream), err_word()};
  if (!a.err) return LL_ERR_CUDA;
  return gdn_b_launch(a);
}

ll_status ll_gdn_decode_step(int B, int H, int dk, int dv, int Ls, ll_dtype io, const int64_t* t, const void* q,
                             const void* k, const void* v, const float* log_alpha, const float* beta,
                             const float* lam, float* states, void* o, void* stream) {
  if (B < 1 || H < 1 || Ls < 1 || Ls > 62) return LL_ERR_INVALID_ARG;
  if (io != LL_F32 && io != LL_BF16) return LL_ERR_INVALID_ARG;
  if (!head_dim_ok(dk) || !head_dim_ok(dv)) return LL_ERR_UNSUPPORTED;
  if (!t || !q || !k || !v || !log_alpha || !beta || !lam || !states || !o) return LL_ERR_INVALID_ARG;
  if (!aligned16(t) || !aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(log_alpha) ||
      !aligned16(beta) || !aligned16(lam) || !aligned16(states) || !aligned16(o))
    return LL_ERR_INVALID_ARG;
  unsigned* ew = err_word();
  if (!ew) return LL_ERR_CUDA;
  return gdn_decode_launch(B, H, dk, dv, Ls, io, t, q, k, v, log_alpha, beta, lam, states, o,
                           static_cast<cudaStream_t>(stream), ew);
}

size_t ll_gdn_fwd_workspace_size(const ll_shape* s) {
  if (check_shape(s) != LL_OK || s->Ls != 0 || s->T % s->chunk != 0) return 0;
  return gdn_workspace(*s);
}

ll_status ll_gdn_fwd(const ll_shape* s, const void* q, const void* k, const void* v, const float* log_alpha,
                     const float* beta, const float* lam, void* o, void* workspace, size_t ws_bytes,
                     void* stream) {
  ll_status st = check_shape(s);
  if (st != LL_OK) return st;
  if (s->T % s->chunk != 0) return LL_ERR_INVALID_ARG;  // whole chunks only
  if (s->Ls != 0) return LL_ERR_INVALID_ARG;
  if (!q || !k || !v || !log_alpha || !beta || !lam || !o) return LL_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(log_alpha) || !aligned16(beta) ||
      !aligned16(lam) || !aligned16(o))
    return LL_ERR_INVALID_ARG;
  const size_t need_ws = gdn_workspace(*s);
  if (need_ws == 0) return LL_ERR_UNSUPPORTED;
  if (!workspace || ws_bytes < need_ws) return LL_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return LL_ERR_WORKSPACE;
  FwdArgs a{*s, q, k, v, log_alpha, lam, beta, o, nullptr, nullptr, workspace, ws_bytes,
            static_cast<cudaStream_t>(stream), err_word()};
  if (!a.err) return LL_ERR_CUDA;
  return gdn_launch(a);
}

}  // extern "C"
