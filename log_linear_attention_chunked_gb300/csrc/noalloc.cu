// ll_attn_fwd_noalloc: the log-linear Mamba-2 forward without a caller-owned
// workspace.
//
// Some callers cannot hand the library a workspace and cannot allocate one:
// a host application that reserves all device memory for its own pool at
// start-up and forbids later cudaMalloc calls, a plugin loaded by such a
// runtime that has no allocator handle to pass down, or a latency-bound loop
// where a cudaMalloc (which may synchronise the device) is not acceptable.
// For them the scratch lives in a fixed-size array in this file, part of the
// library's device image: every GPU that loads the library holds it until the
// process exits.  The call never allocates or frees anything.
//
// The array is shared by every call on a device and keeps the last call's
// contents; the forward writes every scratch word it reads before reading it,
// so nothing needs clearing.  Calls whose execution overlaps on the GPU
// (different streams, or several host threads) race on the array.
//
// Host code must not use the name of the array as a pointer: on the host it
// is only a stand-in for the symbol.  The device address is looked up once per
// device with cudaGetSymbolAddress, on the first call made while that device
// is current; make that first call before capturing any stream.
#include <mutex>

#include "common.cuh"

static_assert(LL_NOALLOC_SCRATCH_BYTES % 256 == 0, "scratch size must keep 256-byte alignment");

// The scratch itself: file scope, internal linkage, one copy per device.
static __device__ __align__(256) unsigned char g_noalloc_scratch[LL_NOALLOC_SCRATCH_BYTES];

namespace llattn {

namespace {

constexpr size_t kNoAllocScratchBytes = LL_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

// Device address of g_noalloc_scratch on the current device (set-up runs once
// per device, with that device current).
ll_status scratch_address(void** out) {
  static std::mutex mu;
  static void* addr[kMaxDevices] = {nullptr};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return LL_ERR_CUDA;
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return LL_ERR_CUDA;
    addr[dev] = p;
  }
  *out = addr[dev];
  return LL_OK;
}

}  // namespace

}  // namespace llattn

using namespace llattn;

extern "C" ll_status ll_attn_fwd_noalloc(const ll_shape* s, const void* q, const void* k, const void* v,
                                         const float* log_alpha, const float* lam, void* o, float* state_out,
                                         float* scale_out, void* stream) {
  const size_t need = ll_attn_fwd_workspace_size(s);
  if (need == 0) return LL_ERR_INVALID_ARG;                  // invalid shape
  if (need > kNoAllocScratchBytes) return LL_ERR_WORKSPACE;  // shape too large for the fixed scratch
  void* scratch = nullptr;
  ll_status st = scratch_address(&scratch);
  if (st != LL_OK) return st;
  return ll_attn_fwd(s, q, k, v, log_alpha, lam, o, state_out, scale_out, scratch, kNoAllocScratchBytes, stream);
}
