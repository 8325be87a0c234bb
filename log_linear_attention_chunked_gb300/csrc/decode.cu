// One Fenwick-state decode step of log-linear Mamba-2 ("Log-Linear Attention"
// study note §3-3 recurrent form and §3-6 memory-efficient decoding; carry /
// merge as in the drawer analogy of the gist.science (zh) summary).
//
// Per (b, h), at position t, with stored slots i = level i+1 (true state =
// scale_i * S_i; non-empty slots are the set bits of t, decayed to t-1):
//   g_i   = scale_i * alpha_t                       (lazy decay of every level;
//           with one decay per level, alpha_t^(i+1) for slot i)
//   o_t   = lam_0 (q.k) v + sum_{i: bit i of t} lam_{i+1} g_i S_i q
//   j     = ctz(t+1): slots 0..j-1 are full and merge into the empty slot j:
//           S_j = v k^T + sum_{i<j} g_i S_i,  scale_j = 1,  scales 0..j-1 = 0,
//           scales of the non-empty slots above j become g_i.
// The step is bound by HBM: every non-empty state is read once and one state
// is written.  One CTA per (b, h); each warp owns rows of dv, each lane dk/32
// consecutive columns (128-bit loads for dk = 128), and all non-empty levels
// of a row are loaded before any is used so their loads are in flight together.
#include "level_decay.cuh"

namespace llattn {

namespace {

constexpr int kWarps = 8;
constexpr int kMaxSlots = 62;
constexpr int kBatchLoads = 8;  // level loads issued back to back per row

template <int DK> struct Vec;
template <> struct Vec<128> { using T = float4; static constexpr int n = 4; };
template <> struct Vec<64> { using T = float2; static constexpr int n = 2; };
template <> struct Vec<32> { using T = float; static constexpr int n = 1; };
template <> struct Vec<16> { using T = float; static constexpr int n = 1; };  // lanes 16..31 idle

template <typename V> __device__ __forceinline__ void unpack(const V& v, float* x);
template <> __device__ __forceinline__ void unpack<float4>(const float4& v, float* x) {
  x[0] = v.x; x[1] = v.y; x[2] = v.z; x[3] = v.w;
}
template <> __device__ __forceinline__ void unpack<float2>(const float2& v, float* x) { x[0] = v.x; x[1] = v.y; }
template <> __device__ __forceinline__ void unpack<float>(const float& v, float* x) { x[0] = v; }

template <typename V> __device__ __forceinline__ V pack(const float* x);
template <> __device__ __forceinline__ float4 pack<float4>(const float* x) { return make_float4(x[0], x[1], x[2], x[3]); }
template <> __device__ __forceinline__ float2 pack<float2>(const float* x) { return make_float2(x[0], x[1]); }
template <> __device__ __forceinline__ float pack<float>(const float* x) { return x[0]; }

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

template <typename IO, int DK>
__global__ void __launch_bounds__(kWarps * 32, 4) decode_kernel(int H, int dv, int Ls, const int64_t* __restrict__ tpos,
                                                             const IO* __restrict__ q, const IO* __restrict__ k,
                                                             const IO* __restrict__ v,
                                                             const float* __restrict__ log_alpha,
                                                             const float* __restrict__ lam, float* __restrict__ states,
                                                             float* __restrict__ scales, IO* __restrict__ o,
                                                             unsigned* __restrict__ err, int per_level) {
  using V = typename Vec<DK>::T;
  constexpr int NV = Vec<DK>::n;
  __shared__ int slot_of[kMaxSlots];
  __shared__ float coef[kMaxSlots];   // lam_{i+1} * g_i
  __shared__ float mcoef[kMaxSlots];  // g_i if slot i merges, else 0
  __shared__ float gdec[kMaxSlots];
  __shared__ int ns_sh;

  const int bh = blockIdx.x;
  const int b = bh / H;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long t = tpos[b];
  if (t < 0 || t + 1 >= (1ll << Ls)) {
    if (threadIdx.x == 0) raise_error(err, kErrDeviceArg);
    return;
  }
  const int j = __ffsll(t + 1) - 1;  // trailing ones of t
  // log_alpha is [B,H] or, with one decay per level, [B,H,Ls+1] (entry l for level l)
  const float* la_bh = log_alpha + (size_t)bh * (per_level ? Ls + 1 : 1);
  const float* lam_bh = lam + (size_t)bh * (Ls + 1);
  float* sc = scales + (size_t)bh * Ls;
  if (warp == 0) {  // the non-empty slots, compacted in order; one lane per slot, loads in parallel
    int n = 0;
    for (int base = 0; base < Ls; base += 32) {
      const int i = base + lane;
      const bool set = i < Ls && ((t >> i) & 1);
      float g = 0.f, lm = 0.f;
      if (set) {
        g = sc[i] * expf(la_bh[per_level ? i + 1 : 0]);
        lm = lam_bh[i + 1];
      }
      const unsigned m = __ballot_sync(0xffffffffu, set);
      if (set) {
        const int at = n + __popc(m & ((1u << lane) - 1u));
        slot_of[at] = i;
        coef[at] = lm * g;
        mcoef[at] = (i < j) ? g : 0.f;
        gdec[at] = g;
      }
      n += __popc(m);
    }
    if (lane == 0) ns_sh = n;
  }
  __syncthreads();
  const int ns = ns_sh;

  const bool active = (DK >= 32) || lane < DK;
  const int c0 = (DK >= 32 ? lane * NV : lane);
  float qv[NV], kv[NV];
  const IO* qb = q + (size_t)bh * DK;
  const IO* kb = k + (size_t)bh * DK;
#pragma unroll
  for (int u = 0; u < NV; ++u) {
    qv[u] = active ? to_f(qb[c0 + u]) : 0.f;
    kv[u] = active ? to_f(kb[c0 + u]) : 0.f;
  }
  float qk = 0.f;
#pragma unroll
  for (int u = 0; u < NV; ++u) qk = fmaf(qv[u], kv[u], qk);
  qk = warp_sum(qk);
  const float lam0 = lam_bh[0];
  const size_t mat = (size_t)dv * DK;
  float* st = states + (size_t)bh * Ls * mat;
  const IO* vb = v + (size_t)bh * dv;
  IO* ob = o + (size_t)bh * dv;

  for (int r = warp; r < dv; r += kWarps) {
    const float vr = to_f(vb[r]);
    float acc[NV], mrg[NV];
#pragma unroll
    for (int u = 0; u < NV; ++u) { acc[u] = 0.f; mrg[u] = vr * kv[u]; }
    for (int i0 = 0; i0 < ns; i0 += kBatchLoads) {
      V s[kBatchLoads];
#pragma unroll
      for (int u = 0; u < kBatchLoads; ++u)
        if (active && i0 + u < ns)
          s[u] = *reinterpret_cast<const V*>(st + (size_t)slot_of[i0 + u] * mat + (size_t)r * DK + c0);
#pragma unroll
      for (int u = 0; u < kBatchLoads; ++u) {
        if (i0 + u < ns) {
          float x[NV];
          if (active) unpack<V>(s[u], x);
          else {
#pragma unroll
            for (int w = 0; w < NV; ++w) x[w] = 0.f;
          }
          const float cf = coef[i0 + u], mf = mcoef[i0 + u];
#pragma unroll
          for (int w = 0; w < NV; ++w) {
            acc[w] = fmaf(cf, x[w], acc[w]);
            mrg[w] = fmaf(mf, x[w], mrg[w]);
          }
        }
      }
    }
    float dot = 0.f;
#pragma unroll
    for (int u = 0; u < NV; ++u) dot = fmaf(acc[u], qv[u], dot);
    dot = warp_sum(dot);
    if (active) *reinterpret_cast<V*>(st + (size_t)j * mat + (size_t)r * DK + c0) = pack<V>(mrg);
    if (lane == 0) ob[r] = from_f<IO>(fmaf(lam0 * qk, vr, dot));
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int i = 0; i < j; ++i) sc[i] = 0.f;
    sc[j] = 1.f;
    for (int n = 0; n < ns; ++n)
      if (slot_of[n] > j) sc[slot_of[n]] = gdec[n];
  }
}

template <typename IO, int DK>
ll_status launch(int B, int H, int dv, int Ls, const int64_t* t, const void* q, const void* k, const void* v,
                 const float* log_alpha, const float* lam, float* states, float* scales, void* o, cudaStream_t stream,
                 unsigned* err, int per_level) {
  decode_kernel<IO, DK><<<B * H, kWarps * 32, 0, stream>>>(
      H, dv, Ls, t, static_cast<const IO*>(q), static_cast<const IO*>(k), static_cast<const IO*>(v), log_alpha, lam,
      states, scales, static_cast<IO*>(o), err, per_level);
  LL_CUDA_OK(cudaGetLastError());
  return LL_OK;
}

template <typename IO>
ll_status launch_io(int B, int H, int dk, int dv, int Ls, const int64_t* t, const void* q, const void* k,
                    const void* v, const float* log_alpha, const float* lam, float* states, float* scales, void* o,
                    cudaStream_t stream, unsigned* err, int pl) {
  switch (dk) {
    case 128: return launch<IO, 128>(B, H, dv, Ls, t, q, k, v, log_alpha, lam, states, scales, o, stream, err, pl);
    case 64: return launch<IO, 64>(B, H, dv, Ls, t, q, k, v, log_alpha, lam, states, scales, o, stream, err, pl);
    case 32: return launch<IO, 32>(B, H, dv, Ls, t, q, k, v, log_alpha, lam, states, scales, o, stream, err, pl);
    case 16: return launch<IO, 16>(B, H, dv, Ls, t, q, k, v, log_alpha, lam, states, scales, o, stream, err, pl);
  }
  return LL_ERR_UNSUPPORTED;
}

}  // namespace

ll_status decode_launch(int B, int H, int dk, int dv, int Ls, ll_dtype io, const int64_t* t, const void* q,
                        const void* k, const void* v, const float* log_alpha, const float* lam, float* states,
                        float* scales, void* o, cudaStream_t stream, unsigned* err) {
  if ((long long)B * H > 0x7fffffffll) return LL_ERR_UNSUPPORTED;
  if (io == LL_F32)
    return launch_io<float>(B, H, dk, dv, Ls, t, q, k, v, log_alpha, lam, states, scales, o, stream, err, 0);
  return launch_io<__nv_bfloat16>(B, H, dk, dv, Ls, t, q, k, v, log_alpha, lam, states, scales, o, stream, err, 0);
}

ll_status decode_level_decay_launch(int B, int H, int dk, int dv, int Ls, ll_dtype io, const int64_t* t,
                                    const void* q, const void* k, const void* v, const float* log_alpha,
                                    const float* lam, float* states, float* scales, void* o, cudaStream_t stream,
                                    unsigned* err) {
  if ((long long)B * H > 0x7fffffffll) return LL_ERR_UNSUPPORTED;
  if (io == LL_F32)
    return launch_io<float>(B, H, dk, dv, Ls, t, q, k, v, log_alpha, lam, states, scales, o, stream, err, 1);
  return launch_io<__nv_bfloat16>(B, H, dk, dv, Ls, t, q, k, v, log_alpha, lam, states, scales, o, stream, err, 1);
}

}  // namespace llattn
