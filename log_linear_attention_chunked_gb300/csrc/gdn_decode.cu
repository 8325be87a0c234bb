// One Fenwick-state decode step of log-linear Gated DeltaNet, reading A
// ("Log-Linear Attention" study note §3-5 and §3-6, gist.science (de)
// Technische Zusammenfassung §2; the gated delta rule itself is the standard
// one, since the pages print no delta-rule equations).
//
// Per (b, h), at position t, with stored slots i = level i+1 holding true
// states (non-empty slots are the set bits of t, each after the transition
// of token t-1):
//   every non-empty level   S <- alpha_t S (I - beta_t k_t k_t^T)
//   level 0 (the token)     beta_t v_t k_t^T
//   o_t = lam_0 beta (k.q) v + sum_l lam_l S^(l) q
//   j = ctz(t+1): level 0 and slots 0..j-1 merge into slot j by addition.
// The transition acts on each row of a state by itself:
//   S[r,:] <- alpha (S[r,:] - beta (S[r,:].k) k),   and its q-dot is
//   alpha (S[r,:].q - beta (S[r,:].k)(k.q)),
// so a warp owns rows of d_v, each lane d_k/32 consecutive columns (128-bit
// accesses for d_k = 128), and the two dot products of a row are warp sums.
// Every non-empty state is read and written back (there is no scalar decay to
// defer), so the step is bound by HBM at about twice the bytes of the
// Mamba-2 step.
#include "common.cuh"

namespace llattn {

namespace {

constexpr int kWarps = 8;
constexpr int kMaxSlots = 62;
constexpr int kBatchLoads = 8;  // level loads issued back to back per row

template <int DK> struct GVec;
template <> struct GVec<128> { using T = float4; static constexpr int n = 4; };
template <> struct GVec<64> { using T = float2; static constexpr int n = 2; };
template <> struct GVec<32> { using T = float; static constexpr int n = 1; };
template <> struct GVec<16> { using T = float; static constexpr int n = 1; };  // lanes 16..31 idle

__device__ __forceinline__ void to_arr(const float4& v, float* x) { x[0] = v.x; x[1] = v.y; x[2] = v.z; x[3] = v.w; }
__device__ __forceinline__ void to_arr(const float2& v, float* x) { x[0] = v.x; x[1] = v.y; }
__device__ __forceinline__ void to_arr(const float& v, float* x) { x[0] = v; }
template <typename V> __device__ __forceinline__ V from_arr(const float* x);
template <> __device__ __forceinline__ float4 from_arr<float4>(const float* x) { return make_float4(x[0], x[1], x[2], x[3]); }
template <> __device__ __forceinline__ float2 from_arr<float2>(const float* x) { return make_float2(x[0], x[1]); }
template <> __device__ __forceinline__ float from_arr<float>(const float* x) { return x[0]; }

__device__ __forceinline__ void warp_sum2(float& a, float& b) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    a += __shfl_xor_sync(0xffffffffu, a, o);
    b += __shfl_xor_sync(0xffffffffu, b, o);
  }
}

template <typename IO, int DK>
__global__ void __launch_bounds__(kWarps * 32) gdn_decode_kernel(
    int H, int dv, int Ls, const int64_t* __restrict__ tpos, const IO* __restrict__ q, const IO* __restrict__ k,
    const IO* __restrict__ v, const float* __restrict__ log_alpha, const float* __restrict__ beta,
    const float* __restrict__ lam, float* __restrict__ states, IO* __restrict__ o, unsigned* __restrict__ err) {
  using V = typename GVec<DK>::T;
  constexpr int NV = GVec<DK>::n;
  __shared__ int slot_of[kMaxSlots];
  __shared__ float lam_of[kMaxSlots];
  __shared__ int merges[kMaxSlots];
  __shared__ int ns_sh;

  const int bh = blockIdx.x;
  const int b = bh / H;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long t = tpos[b];
  if (t < 0 || t + 1 >= (1ll << Ls)) {
    if (threadIdx.x == 0) raise_error(err, kErrDeviceArg);
    return;
  }
  const int j = __ffsll(t + 1) - 1;  // trailing ones of t: the carry slot
  const float* lam_bh = lam + (size_t)bh * (Ls + 1);
  if (warp == 0) {  // the non-empty slots, compacted in order; one lane per slot, loads in parallel
    int n = 0;
    for (int base = 0; base < Ls; base += 32) {
      const int i = base + lane;
      const bool set = i < Ls && ((t >> i) & 1);
      const float lm = set ? lam_bh[i + 1] : 0.f;
      const unsigned m = __ballot_sync(0xffffffffu, set);
      if (set) {
        const int at = n + __popc(m & ((1u << lane) - 1u));
        slot_of[at] = i;
        lam_of[at] = lm;
        merges[at] = i < j;
      }
      n += __popc(m);
    }
    if (lane == 0) ns_sh = n;
  }
  __syncthreads();
  const int ns = ns_sh;
  const float alpha = expf(log_alpha[bh]);
  const float bt = beta[bh];

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
  float kq = 0.f, kk = 0.f;
#pragma unroll
  for (int u = 0; u < NV; ++u) {
    kq = fmaf(kv[u], qv[u], kq);
    kk = fmaf(kv[u], kv[u], kk);
  }
  warp_sum2(kq, kk);
  const float lam0 = lam_bh[0];
  const size_t mat = (size_t)dv * DK;
  float* st = states + (size_t)bh * Ls * mat;
  const IO* vb = v + (size_t)bh * dv;
  IO* ob = o + (size_t)bh * dv;

  for (int r = warp; r < dv; r += kWarps) {
    const float vr = to_f(vb[r]);
    float mrg[NV];
#pragma unroll
    for (int u = 0; u < NV; ++u) mrg[u] = bt * vr * kv[u];  // the token's write, level 0
    float out = lam0 * bt * vr * kq;
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
          if (active) to_arr(s[u], x);
          else {
#pragma unroll
            for (int w = 0; w < NV; ++w) x[w] = 0.f;
          }
          float sk = 0.f, sq = 0.f;
#pragma unroll
          for (int w = 0; w < NV; ++w) {
            sk = fmaf(x[w], kv[w], sk);
            sq = fmaf(x[w], qv[w], sq);
          }
          warp_sum2(sk, sq);
          const float c = bt * sk;
          out = fmaf(lam_of[i0 + u] * alpha, fmaf(-c, kq, sq), out);
#pragma unroll
          for (int w = 0; w < NV; ++w) x[w] = alpha * fmaf(-c, kv[w], x[w]);
          if (merges[i0 + u]) {
#pragma unroll
            for (int w = 0; w < NV; ++w) mrg[w] += x[w];
          } else if (active) {
            *reinterpret_cast<V*>(st + (size_t)slot_of[i0 + u] * mat + (size_t)r * DK + c0) = from_arr<V>(x);
          }
        }
      }
    }
    if (active) *reinterpret_cast<V*>(st + (size_t)j * mat + (size_t)r * DK + c0) = from_arr<V>(mrg);
    if (lane == 0) ob[r] = from_f<IO>(out);
  }
}

template <typename IO, int DK>
ll_status launch(int B, int H, int dv, int Ls, const int64_t* t, const void* q, const void* k, const void* v,
                 const float* log_alpha, const float* beta, const float* lam, float* states, void* o,
                 cudaStream_t stream, unsigned* err) {
  gdn_decode_kernel<IO, DK><<<B * H, kWarps * 32, 0, stream>>>(
      H, dv, Ls, t, static_cast<const IO*>(q), static_cast<const IO*>(k), static_cast<const IO*>(v), log_alpha,
      beta, lam, states, static_cast<IO*>(o), err);
  LL_CUDA_OK(cudaGetLastError());
  return LL_OK;
}

template <typename IO>
ll_status launch_io(int B, int H, int dk, int dv, int Ls, const int64_t* t, const void* q, const void* k,
                    const void* v, const float* log_alpha, const float* beta, const float* lam, float* states,
                    void* o, cudaStream_t stream, unsigned* err) {
  switch (dk) {
    case 128: return launch<IO, 128>(B, H, dv, Ls, t, q, k, v, log_alpha, beta, lam, states, o, stream, err);
    case 64: return launch<IO, 64>(B, H, dv, Ls, t, q, k, v, log_alpha, beta, lam, states, o, stream, err);
    case 32: return launch<IO, 32>(B, H, dv, Ls, t, q, k, v, log_alpha, beta, lam, states, o, stream, err);
    case 16: return launch<IO, 16>(B, H, dv, Ls, t, q, k, v, log_alpha, beta, lam, states, o, stream, err);
  }
  return LL_ERR_UNSUPPORTED;
}

}  // namespace

ll_status gdn_decode_launch(int B, int H, int dk, int dv, int Ls, ll_dtype io, const int64_t* t, const void* q,
                            const void* k, const void* v, const float* log_alpha, const float* beta,
                            const float* lam, float* states, void* o, cudaStream_t stream, unsigned* err) {
  if ((long long)B * H > 0x7fffffffll) return LL_ERR_UNSUPPORTED;
  if (io == LL_F32)
    return launch_io<float>(B, H, dk, dv, Ls, t, q, k, v, log_alpha, beta, lam, states, o, stream, err);
  return launch_io<__nv_bfloat16>(B, H, dk, dv, Ls, t, q, k, v, log_alpha, beta, lam, states, o, stream, err);
}

}  // namespace llattn
