// Chunked log-linear Mamba-2 forward on CUDA cores (float32 FMA throughout).
//
// This is the exact-precision path (float32 io, 1e-5 budget) and the path for
// shapes the tensor-core kernel does not take.  Algorithm ("Log-Linear
// Attention" study note §3-4 parallel form, computed chunk-wise as in the
// gist.science (zh) summary §2.3: dense inside a chunk, O(log(T/C)) state
// passes between chunks):
//
//   chunk c (Ce tokens, cs = inclusive cumsum of log_alpha inside the chunk)
//   (1) intra   : o_i += sum_{j<=i in c} (q_i.k_j) exp(cs_i - cs_j) lam_i[bitlen(i^j)] v_j
//   (2) state   : S_c  = sum_{j in c} exp(cs_end - cs_j) v_j k_j^T          [dv x dk]
//   (3) Fenwick : F_c  = S_c + sum_{m < cto(c)} exp(dec_m) F_{c - 2^m}
//                 F_c covers the 2^cto(c) chunks ending at c, decayed to the
//                 end of chunk c; G_c is the sum of log_alpha over that block.
//   (4) inter   : for every set bit h of c, the level  log2(Ce)+1+h  bucket of
//                 every query in chunk c is the block of F_e,
//                 e = (c with bits 0..h cleared) + 2^h - 1, and
//                 o_i += lam_i[log2(Ce)+1+h] exp(cs_i + D_h) F_e q_i,
//                 D_h = sum of G over the lower set bits of c (decay from the
//                 end of e to the start of chunk c).
//   (5) export  : the level states of position T are F nodes of the Fenwick
//                 prefix query of N = T/Ce, decayed to token T-1.
//
// Ragged T (T not a multiple of Ce): the last chunk holds the r = T mod Ce
// remaining tokens; the kernels treat its missing rows as absent (zero keys
// and values, log_alpha 0, no output).  At position T the levels above
// log2(Ce) are the nodes of the floor(T/Ce) full chunks, decayed over the
// partial chunk too; the levels up to log2(Ce) are the buckets of r inside the
// partial chunk, written by their own kernel.
//
// Prefill continuation (the tokens are positions t0 .. t0+T-1, the prefix
// enters as the decode states of position t0, decayed to t0-1; t0 is a
// multiple of the smallest power of two P >= T, so the segment sits inside
// one aligned block of P positions):
//   every prefix bucket of t0 has a level above log2(P), which for every
//   query of the segment is the same level (a key's level only changes where
//   the query differs from t0 above it), so (4) adds, per non-empty slot l,
//   o_i += lam_i[l] g_l exp(cs_i + D) S_l q_i with D the decay of the whole
//   segment before the chunk; the segment's own levels are those of the
//   relative positions.
//   (6) the states of t1 = t0 + T: with b = bitlen(t1 xor t0), a prefix
//   bucket of level l goes to level max(l, b) (decayed over the segment), the
//   segment's buckets (its export at T) keep their level if T < P and go to
//   level b if T = P; buckets that land on one level add.
//
// Cumulative decays are kept in double: the inputs and outputs are float32 and
// the exponent of a decay factor must not lose the absolute accuracy that a
// float32 running sum would lose at long range.
#include <algorithm>

#include "bwd.cuh"
#include "sm100.cuh"

namespace llattn {

namespace {

constexpr int kThreads = 256;

// The SIMT kernels stage a chunk of q, k, v in shared memory; chunks longer
// than this many elements per operand are processed as shorter chunks (the
// result does not depend on the chunk length).
constexpr int kMaxChunkElems = 8192;

struct SimtPlan {
  int Ce, N, lc;  // effective chunk, #chunks, log2(Ce)
  size_t off_S, off_F, off_tot, off_G, off_O, total;
  size_t off_segS, off_segSc, off_segDec, total_cont;  // the segment's own export (continuation)
};

SimtPlan plan_of(const ll_shape& s) {
  SimtPlan p{};
  int d = std::max(s.dk, s.dv);
  p.Ce = s.chunk;
  while (p.Ce * d > kMaxChunkElems && p.Ce > 16) p.Ce >>= 1;
  p.N = (s.T + p.Ce - 1) / p.Ce;  // the last chunk may be partial
  p.lc = ilog2(p.Ce);
  const size_t BH = (size_t)s.B * s.H;
  const size_t mat = (size_t)s.dv * s.dk;
  size_t off = 0;
  p.off_S = off;   off = align_up(off + BH * p.N * mat * sizeof(float), 256);
  p.off_F = off;   off = align_up(off + BH * p.N * mat * sizeof(float), 256);
  p.off_tot = off; off = align_up(off + BH * p.N * sizeof(double), 256);
  p.off_G = off;   off = align_up(off + BH * p.N * sizeof(double), 256);
  p.off_O = off;
  if (s.io != LL_F32) off = align_up(off + BH * (size_t)s.T * s.dv * sizeof(float), 256);
  p.total = off;
  p.off_segS = off;  off = align_up(off + BH * (size_t)std::max(s.Ls, 1) * mat * sizeof(float), 256);
  p.off_segSc = off; off = align_up(off + BH * (size_t)std::max(s.Ls, 1) * sizeof(float), 256);
  p.off_segDec = off; off = align_up(off + BH * sizeof(float), 256);
  p.total_cont = off;
  return p;
}

// cs[i] = the sum of log_alpha over rows 0..i of the chunk (rows >= nv add 0),
// float64, for i < Ce <= 128; every thread of the CTA takes part (a scan over
// each warp, then the warps' totals); cs is complete after the caller's next
// __syncthreads
__device__ __forceinline__ void chunk_scan(double* cs, const float* log_alpha, size_t row0, int nv, int Ce) {
  __shared__ double wsum[4];
  const int t = threadIdx.x, lane = t & 31, w = t >> 5;
  double x = (t < Ce && t < nv) ? (double)log_alpha[row0 + t] : 0.0;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const double y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31 && w < 4) wsum[w] = x;
  __syncthreads();
  if (t < Ce) {
    for (int ww = 0; ww < w; ++ww) x += wsum[ww];
    cs[t] = x;
  }
}

// (1) + (2): one CTA per (chunk, head).
template <typename IO>
__global__ void __launch_bounds__(kThreads) simt_chunk_kernel(const IO* __restrict__ q, const IO* __restrict__ k,
                                                              const IO* __restrict__ v,
                                                              const float* __restrict__ log_alpha,
                                                              const float* __restrict__ lam, float* o_intra,
                                                              float* __restrict__ S, double* __restrict__ tot, int T,
                                                              int dk, int dv, int L, int Ce) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  const int c = blockIdx.x;
  const int N = gridDim.x;
  const size_t bh = blockIdx.y;
  const int tid = threadIdx.x;
  const int dkp = dk + 1, dvp = dv + 1, Cp = Ce + 1;

  double* cs = reinterpret_cast<double*>(smem_raw);
  float* wdec = reinterpret_cast<float*>(cs + Ce);
  float* qs = wdec + Ce;
  float* ks = qs + Ce * dkp;
  float* vs = ks + Ce * dkp;
  float* P = vs + Ce * dvp;

  const size_t t0 = (size_t)c * Ce;
  const size_t row0 = bh * T + t0;
  const int nv = min(Ce, T - (int)t0);  // rows present in this chunk
  chunk_scan(cs, log_alpha, row0, nv, Ce);
  if (tid == Ce - 1) tot[bh * N + c] = cs[Ce - 1];
  for (int x = tid; x < Ce * dk; x += kThreads) {
    int i = x / dk, f = x % dk;
    qs[i * dkp + f] = i < nv ? to_f(q[(row0 + i) * dk + f]) : 0.f;
    ks[i * dkp + f] = i < nv ? to_f(k[(row0 + i) * dk + f]) : 0.f;
  }
  for (int x = tid; x < Ce * dv; x += kThreads) {
    int i = x / dv, e = x % dv;
    vs[i * dvp + e] = i < nv ? to_f(v[(row0 + i) * dv + e]) : 0.f;
  }
  __syncthreads();
  for (int j = tid; j < Ce; j += kThreads) wdec[j] = expf((float)(cs[Ce - 1] - cs[j]));

  // masked scores P[i][j]
  for (int x = tid; x < Ce * Ce; x += kThreads) {
    int i = x / Ce, j = x % Ce;
    float p = 0.f;
    if (j <= i && i < nv) {
      float dot = 0.f;
      for (int f = 0; f < dk; ++f) dot = fmaf(qs[i * dkp + f], ks[j * dkp + f], dot);
      int lv = bitlen((unsigned)(i ^ j));
      p = dot * expf((float)(cs[i] - cs[j])) * lam[(row0 + i) * L + lv];
    }
    P[i * Cp + j] = p;
  }
  __syncthreads();

  // intra output
  for (int x = tid; x < nv * dv; x += kThreads) {
    int i = x / dv, e = x % dv;
    float acc = 0.f;
    for (int j = 0; j <= i; ++j) acc = fmaf(P[i * Cp + j], vs[j * dvp + e], acc);
    o_intra[(row0 + i) * dv + e] = acc;
  }

  // chunk state S_c[e][f] = sum_j wdec_j v_j[e] k_j[f]
  float* Sc = S + (bh * N + c) * (size_t)dv * dk;
  for (int x = tid; x < dv * dk; x += kThreads) {
    int e = x / dk, f = x % dk;
    float acc = 0.f;
    for (int j = 0; j < Ce; ++j) acc = fmaf(wdec[j] * vs[j * dvp + e], ks[j * dkp + f], acc);
    Sc[x] = acc;
  }
}

// (3): sequential over chunks, parallel over matrix elements and heads.
// Element (r, c) of a [128][128] bf16 tile in the 128-byte-swizzled layout of
// the tensor-core kernels: two [128][64] halves, 128-byte rows, the 16-byte
// chunks of a row permuted by XOR with (r mod 8).
__device__ __forceinline__ int swizzled_elem(int r, int c) {
  return (c >> 6) * 8192 + r * 64 + ((((c & 63) >> 3) ^ (r & 7)) << 3) + (c & 7);
}

// With Ft (d_k = d_v = 128 only) every node is also written as such a bf16
// tile; with cum, the running sums of the chunk totals (per head, float64).
__global__ void __launch_bounds__(kThreads) simt_fenwick_kernel(const float* __restrict__ S, float* __restrict__ F,
                                                                const double* __restrict__ tot,
                                                                double* __restrict__ G, int N, int mat,
                                                                __nv_bfloat16* __restrict__ Ft,
                                                                double* __restrict__ cum) {
  extern __shared__ double Gs[];  // [N]
  __shared__ double wsum[kThreads / 32];
  const size_t bh = blockIdx.y;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  // Running sums of the chunk totals (a block scan in rounds of kThreads
  // chunks), then the node totals as their differences: node i covers the
  // 2^cto(i) chunks ending at i, so G_i = cum_i - cum_{i - 2^cto(i)}.
  double carry = 0.0;
  for (int base = 0; base < N; base += kThreads) {
    const int i = base + threadIdx.x;
    double x = i < N ? tot[bh * N + i] : 0.0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const double y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) wsum[warp] = x;
    __syncthreads();
    double off = carry, round = carry;
    for (int w = 0; w < kThreads / 32; ++w) {
      if (w < warp) off += wsum[w];
      round += wsum[w];
    }
    x += off;
    if (i < N) {
      Gs[i] = x;
      if (cum && blockIdx.x == 0) cum[bh * N + i] = x;
    }
    carry = round;
    __syncthreads();
  }
  // top round first: a node reads a lower index, which a later round rewrites,
  // and within a round every read precedes the writes
  for (int base = ((N - 1) / kThreads) * kThreads; base >= 0; base -= kThreads) {
    const int i = base + threadIdx.x;
    double g = 0.0;
    if (i < N) {
      const int lo = i - (1 << (__ffs(~i) - 1));
      g = Gs[i] - (lo >= 0 ? Gs[lo] : 0.0);
    }
    __syncthreads();
    if (i < N) Gs[i] = g;
    __syncthreads();
  }
  if (blockIdx.x == 0)
    for (int i = threadIdx.x; i < N; i += kThreads) G[bh * N + i] = Gs[i];
  const int idx = blockIdx.x * kThreads + threadIdx.x;
  if (idx >= mat) return;
  const float* Sb = S + bh * N * (size_t)mat;
  float* Fb = F + bh * N * (size_t)mat;
  const int tel = Ft ? swizzled_elem(idx >> 7, idx & 127) : 0;
  // the chunk states do not depend on the chain: four are loaded ahead
  float s0 = Sb[idx], s1 = N > 1 ? Sb[(size_t)mat + idx] : 0.f, s2 = N > 2 ? Sb[2 * (size_t)mat + idx] : 0.f,
        s3 = N > 3 ? Sb[3 * (size_t)mat + idx] : 0.f;
  for (int i = 0; i < N; ++i) {
    float acc = s0;
    s0 = s1;
    s1 = s2;
    s2 = s3;
    s3 = i + 4 < N ? Sb[(size_t)(i + 4) * mat + idx] : 0.f;
    double dec = tot[bh * N + i];
    for (int m = 0; (i >> m) & 1; ++m) {
      const int j = i - (1 << m);
      acc = fmaf(expf((float)dec), Fb[(size_t)j * mat + idx], acc);
      dec += Gs[j];
    }
    Fb[(size_t)i * mat + idx] = acc;
    if (Ft) Ft[(bh * N + i) * (size_t)mat + tel] = __float2bfloat16_rn(acc);
  }
}

// (3) for N <= kFenFastN: the same nodes with the chain kept on chip.  The
// prologue also tabulates, in float, the decay of each child of each node
// (exp(cum_i - cum_{i - 2^m}) for child i - 2^m; node i's children start at
// entry i - popcount(i) of the table), and each thread keeps the latest node
// of every level (the children of the next nodes) in shared memory, so a
// step of the chain reads no node back from global memory and does no
// float64 arithmetic.
constexpr int kFenFastN = kFenwickOnChipChunks;
constexpr int kFenLv = 13;  // levels of N <= 4096
constexpr int kFenVec = 4;   // consecutive matrix elements per thread (dk dv is a multiple of 256)
constexpr int kFenRing = 8;  // ring slots of the chunk states streamed ahead
// dynamic shared memory: the prefix table, the child decays, then (16-byte
// aligned) the latest nodes of each level and the ring
constexpr size_t fen_smem(int N) {
  return (size_t)N * (sizeof(double) + sizeof(float)) + 16 +
         (size_t)(kFenLv + kFenRing) * kThreads * kFenVec * sizeof(float);
}

// Each thread follows kFenVec consecutive elements of the matrix.
__global__ void __launch_bounds__(kThreads) simt_fenwick_fast_kernel(const float* __restrict__ S,
                                                                     float* __restrict__ F,
                                                                     const double* __restrict__ tot,
                                                                     double* __restrict__ G, int N, int mat,
                                                                     __nv_bfloat16* __restrict__ Ft,
                                                                     double* __restrict__ cum, int write_f) {
  extern __shared__ double Gs[];                                  // [N]
  float* coef = reinterpret_cast<float*>(Gs + N);                 // [N] child decays
  // [kFenLv][kThreads][kFenVec] the latest node of each level, then the ring
  float* last = reinterpret_cast<float*>((reinterpret_cast<uintptr_t>(coef + N) + 15) & ~uintptr_t(15));
  __shared__ double wsum[kThreads / 32];
  const size_t bh = blockIdx.y;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  double carry = 0.0;
  for (int base = 0; base < N; base += kThreads) {  // running sums of the chunk totals
    const int i = base + threadIdx.x;
    double x = i < N ? tot[bh * N + i] : 0.0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const double y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) wsum[warp] = x;
    __syncthreads();
    double off = carry, round = carry;
    for (int w = 0; w < kThreads / 32; ++w) {
      if (w < warp) off += wsum[w];
      round += wsum[w];
    }
    x += off;
    if (i < N) {
      Gs[i] = x;
      if (cum && blockIdx.x == 0) cum[bh * N + i] = x;
    }
    carry = round;
    __syncthreads();
  }
  for (int i = threadIdx.x; i < N; i += kThreads) {  // the children's decays
    const int h = __ffs(~i) - 1, o = i - __popc(i);
    for (int m = 0; m < h; ++m) coef[o + m] = expf((float)(Gs[i] - Gs[i - (1 << m)]));
  }
  for (int base = ((N - 1) / kThreads) * kThreads; base >= 0; base -= kThreads) {  // node totals
    const int i = base + threadIdx.x;
    double g = 0.0;
    if (i < N) {
      const int lo = i - (1 << (__ffs(~i) - 1));
      g = Gs[i] - (lo >= 0 ? Gs[lo] : 0.0);
    }
    __syncthreads();
    if (i < N) Gs[i] = g;
    __syncthreads();
  }
  if (blockIdx.x == 0)
    for (int i = threadIdx.x; i < N; i += kThreads) G[bh * N + i] = Gs[i];
  constexpr int kVec = kFenVec, kD = kFenRing;
  const int e0 = (blockIdx.x * kThreads + threadIdx.x) * kVec;  // the thread's first element
  if (e0 >= mat) return;
  // the thread's elements of each chunk state stream through a ring of kD
  // slots in shared memory, kD - 1 chunks ahead, by per-thread asynchronous
  // copies (each thread reads back only what it copied); the addresses
  // advance by one matrix per chunk
  float* ring = last + kFenLv * kThreads * kVec;  // [kD][kThreads][kVec]
  const float* next = S + bh * N * (size_t)mat + e0;
  int issued = 0;
  auto stream_in = [&]() {  // the next chunk's elements (past the end: an empty group)
    if (issued < N) {
      sm100::cp_async16(ring + ((issued % kD) * kThreads + threadIdx.x) * kVec, next);
      next += mat;
    }
    ++issued;
    sm100::cp_async_commit();
  };
  float* fdst = F + bh * N * (size_t)mat + e0;
  __nv_bfloat16* tdst = Ft ? Ft + bh * N * (size_t)mat + swizzled_elem(e0 >> 7, e0 & 127) : nullptr;
  for (int k = 0; k < kD - 1; ++k) stream_in();
  for (int i = 0; i < N; ++i) {
    stream_in();  // into the slot of chunk i - 1, read in the iteration before
    sm100::cp_async_wait<kD - 1>();  // chunk i's copy has landed
    float acc[kVec];
    {
      const float4 x = *reinterpret_cast<const float4*>(ring + ((i % kD) * kThreads + threadIdx.x) * kVec);
      acc[0] = x.x; acc[1] = x.y; acc[2] = x.z; acc[3] = x.w;
    }
    const int h = __ffs(~i) - 1, o = i - __popc(i);
    for (int m = 0; m < h; ++m) {
      const float cf = coef[o + m];
      const float* lp = last + (m * kThreads + threadIdx.x) * kVec;
#pragma unroll
      for (int v = 0; v < kVec; ++v) acc[v] = fmaf(cf, lp[v], acc[v]);
    }
    const float4 a4 = make_float4(acc[0], acc[1], acc[2], acc[3]);
    *reinterpret_cast<float4*>(last + (h * kThreads + threadIdx.x) * kVec) = a4;
    if (write_f) *reinterpret_cast<float4*>(fdst) = a4;
    if (tdst) {  // four consecutive columns: 8 contiguous bytes of the swizzled tile
      const __nv_bfloat162 lo = __floats2bfloat162_rn(acc[0], acc[1]), hi = __floats2bfloat162_rn(acc[2], acc[3]);
      *reinterpret_cast<uint2*>(tdst) =
          make_uint2(*reinterpret_cast<const uint32_t*>(&lo), *reinterpret_cast<const uint32_t*>(&hi));
    }
    fdst += mat;
    if (tdst) tdst += mat;
  }
}

// (4): one CTA per (chunk, head); adds the inter-chunk levels to the intra
// result and writes o.
template <typename IO>
__global__ void __launch_bounds__(kThreads) simt_inter_kernel(const IO* __restrict__ q,
                                                              const float* __restrict__ log_alpha,
                                                              const float* __restrict__ lam,
                                                              const float* o_intra,
                                                              const float* __restrict__ F,
                                                              const double* __restrict__ G, IO* o, int T,
                                                              int dk, int dv, int L, int Ce, int lc,
                                                              const float* __restrict__ pre_states,
                                                              const float* __restrict__ pre_scales, int Ls,
                                                              long long t0) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  const int c = blockIdx.x;
  const int N = gridDim.x;
  const size_t bh = blockIdx.y;
  const int tid = threadIdx.x;
  const int dkp = dk + 1;
  double* cs = reinterpret_cast<double*>(smem_raw);
  float* w = reinterpret_cast<float*>(cs + Ce);
  float* qs = w + Ce;
  float* Fs = qs + Ce * dk;
  float* Oc = Fs + dv * dkp;

  const size_t row0 = bh * T + (size_t)c * Ce;
  const int nv = min(Ce, T - c * Ce);  // rows present in this chunk
  chunk_scan(cs, log_alpha, row0, nv, Ce);
  for (int x = tid; x < Ce * dk; x += kThreads) qs[x] = x < nv * dk ? to_f(q[row0 * dk + x]) : 0.f;
  for (int x = tid; x < Ce * dv; x += kThreads) Oc[x] = x < nv * dv ? o_intra[row0 * dv + x] : 0.f;
  __syncthreads();

  const size_t mat = (size_t)dv * dk;
  double D = 0.0;
  for (int h = 0; (c >> h) != 0; ++h) {
    if (!((c >> h) & 1)) continue;
    const int e = ((c >> (h + 1)) << (h + 1)) + (1 << h) - 1;
    const float* Fe = F + (bh * N + e) * mat;
    for (int x = tid; x < (int)mat; x += kThreads) Fs[(x / dk) * dkp + (x % dk)] = Fe[x];
    for (int i = tid; i < Ce; i += kThreads)
      w[i] = i < nv ? lam[(row0 + i) * L + lc + 1 + h] * expf((float)(cs[i] + D)) : 0.f;
    __syncthreads();
    for (int x = tid; x < Ce * dv; x += kThreads) {
      int i = x / dv, ev = x % dv;
      float acc = 0.f;
      for (int f = 0; f < dk; ++f) acc = fmaf(Fs[ev * dkp + f], qs[i * dk + f], acc);
      Oc[x] = fmaf(w[i], acc, Oc[x]);
    }
    D += G[bh * N + e];
    __syncthreads();
  }
  // continuation: the prefix levels of t0, one state each, decayed over D and cs
  if (pre_states) {
    for (int slot = 0; slot < Ls; ++slot) {
      if (!((t0 >> slot) & 1)) continue;
      const float* Pe = pre_states + (bh * Ls + slot) * mat;
      const float g = pre_scales[bh * Ls + slot];
      for (int x = tid; x < (int)mat; x += kThreads) Fs[(x / dk) * dkp + (x % dk)] = Pe[x];
      for (int i = tid; i < Ce; i += kThreads)
        w[i] = i < nv ? lam[(row0 + i) * L + slot + 1] * g * expf((float)(cs[i] + D)) : 0.f;
      __syncthreads();
      for (int x = tid; x < Ce * dv; x += kThreads) {
        int i = x / dv, ev = x % dv;
        float acc = 0.f;
        for (int f = 0; f < dk; ++f) acc = fmaf(Fs[ev * dkp + f], qs[i * dk + f], acc);
        Oc[x] = fmaf(w[i], acc, Oc[x]);
      }
      __syncthreads();
    }
  }
  for (int x = tid; x < nv * dv; x += kThreads) o[row0 * dv + x] = from_f<IO>(Oc[x]);
}

// (5): level states of position T (= N chunks), decayed to token T-1.
__global__ void __launch_bounds__(kThreads) simt_export_kernel(const float* __restrict__ F,
                                                               const double* __restrict__ G,
                                                               const double* __restrict__ tot,
                                                               float* __restrict__ state_out,
                                                               float* __restrict__ scale_out, int N, int Nq, int mat,
                                                               int Ls, int lc) {
  // N chunks in the arrays; the level states are those of the Nq full ones,
  // decayed over the partial chunk N - 1 as well when Nq < N
  const size_t bh = blockIdx.y;
  const int idx = blockIdx.x * kThreads + threadIdx.x;
  double D = Nq < N ? tot[bh * N + N - 1] : 0.0;
  for (int slot = 0; slot < Ls; ++slot) {
    const int h = slot + 1 - (lc + 1);  // level slot+1 = lc + 1 + h
    float val = 0.f, sc = 0.f;
    if (h >= 0 && h < 31 && ((Nq >> h) & 1)) {
      const int e = ((Nq >> (h + 1)) << (h + 1)) + (1 << h) - 1;
      if (idx < mat) val = expf((float)D) * F[(bh * N + e) * (size_t)mat + idx];
      sc = 1.f;
      D += G[bh * N + e];
    }
    if (idx < mat) state_out[(bh * Ls + slot) * (size_t)mat + idx] = val;
    if (blockIdx.x == 0 && threadIdx.x == 0) scale_out[bh * Ls + slot] = sc;
  }
}

// (5) for ragged T: the levels 1..log2(Ce) of position T are the buckets of
// r = T mod Ce inside the partial chunk; bucket l (bit l-1 of r) holds rows
// [r_hi, r_hi + 2^(l-1)), r_hi = r with bits below l cleared, decayed to T-1.
template <typename IO>
__global__ void __launch_bounds__(kThreads) simt_tail_export_kernel(const IO* __restrict__ k,
                                                                    const IO* __restrict__ v,
                                                                    const float* __restrict__ log_alpha,
                                                                    float* __restrict__ state_out,
                                                                    float* __restrict__ scale_out, int T, int dk,
                                                                    int dv, int Ls, int r) {
  __shared__ float dec[128];  // exp(cs[r-1] - cs[a]) for the partial chunk's rows (r < 128)
  const size_t bh = blockIdx.y;
  const int idx = blockIdx.x * kThreads + threadIdx.x;
  const size_t row0 = bh * T + (size_t)(T - r);
  if (threadIdx.x == 0) {
    double acc = 0.0;  // suffix sums: decay from row a to the last row
    for (int a = r - 1; a >= 0; --a) {
      dec[a] = expf((float)acc);
      acc += (double)log_alpha[row0 + a];
    }
  }
  __syncthreads();
  const int mat = dv * dk;
  for (int l = 1; l <= Ls && (1 << (l - 1)) <= r; ++l) {
    const int slot = l - 1;
    if (!((r >> slot) & 1)) continue;
    const int lo = (r >> l) << l, hi = lo + (1 << slot);
    if (idx < mat) {
      const int e = idx / dk, f = idx % dk;
      float acc = 0.f;
      for (int a = lo; a < hi; ++a)
        acc = fmaf(dec[a] * to_f(v[(row0 + a) * dv + e]), to_f(k[(row0 + a) * dk + f]), acc);
      state_out[(bh * Ls + slot) * (size_t)mat + idx] = acc;
    }
    if (blockIdx.x == 0 && threadIdx.x == 0) scale_out[bh * Ls + slot] = 1.f;
  }
}

template <typename IO>
ll_status launch_typed(const FwdArgs& a, const SimtPlan& p) {
  const ll_shape& s = a.s;
  unsigned char* ws = static_cast<unsigned char*>(a.ws);
  float* S = reinterpret_cast<float*>(ws + p.off_S);
  float* F = reinterpret_cast<float*>(ws + p.off_F);
  double* tot = reinterpret_cast<double*>(ws + p.off_tot);
  double* G = reinterpret_cast<double*>(ws + p.off_G);
  float* o_intra = (s.io == LL_F32) ? static_cast<float*>(a.o) : reinterpret_cast<float*>(ws + p.off_O);
  const int BH = s.B * s.H;
  const int Ce = p.Ce;
  const int mat = s.dv * s.dk;

  size_t sm1 = Ce * sizeof(double) + Ce * sizeof(float) +
               sizeof(float) * ((size_t)2 * Ce * (s.dk + 1) + (size_t)Ce * (s.dv + 1) + (size_t)Ce * (Ce + 1));
  LL_CUDA_OK(cudaFuncSetAttribute(simt_chunk_kernel<IO>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm1));
  simt_chunk_kernel<IO><<<dim3(p.N, BH), kThreads, sm1, a.stream>>>(
      static_cast<const IO*>(a.q), static_cast<const IO*>(a.k), static_cast<const IO*>(a.v), a.log_alpha, a.lam,
      o_intra, S, tot, s.T, s.dk, s.dv, s.L, Ce);
  LL_CUDA_OK(cudaGetLastError());

  const ll_status fs = simt_fenwick_launch(S, F, tot, G, p.N, mat, BH, a.stream);
  if (fs != LL_OK) return fs;

  size_t sm3 = Ce * sizeof(double) + Ce * sizeof(float) +
               sizeof(float) * ((size_t)Ce * s.dk + (size_t)s.dv * (s.dk + 1) + (size_t)Ce * s.dv);
  LL_CUDA_OK(cudaFuncSetAttribute(simt_inter_kernel<IO>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm3));
  simt_inter_kernel<IO><<<dim3(p.N, BH), kThreads, sm3, a.stream>>>(static_cast<const IO*>(a.q), a.log_alpha,
                                                                     a.lam, o_intra, F, G, static_cast<IO*>(a.o), s.T,
                                                                     s.dk, s.dv, s.L, Ce, p.lc, a.state_in, a.scale_in,
                                                                     s.Ls, a.t0);
  LL_CUDA_OK(cudaGetLastError());

  const int Nq = s.T / Ce, r = s.T % Ce;  // full chunks, rows of the partial one
  auto export_states = [&](float* st, float* sc) -> ll_status {
    simt_export_kernel<<<dim3((mat + kThreads - 1) / kThreads, BH), kThreads, 0, a.stream>>>(
        F, G, tot, st, sc, p.N, Nq, mat, s.Ls, p.lc);
    LL_CUDA_OK(cudaGetLastError());
    if (r > 0) {
      simt_tail_export_kernel<IO><<<dim3((mat + kThreads - 1) / kThreads, BH), kThreads, 0, a.stream>>>(
          static_cast<const IO*>(a.k), static_cast<const IO*>(a.v), a.log_alpha, st, sc, s.T, s.dk, s.dv, s.Ls, r);
      LL_CUDA_OK(cudaGetLastError());
    }
    return LL_OK;
  };
  if (a.state_out && a.state_in) {
    float* segS = reinterpret_cast<float*>(ws + p.off_segS);
    float* segSc = reinterpret_cast<float*>(ws + p.off_segSc);
    const ll_status es = export_states(segS, segSc);
    if (es != LL_OK) return es;
    const ll_status st = cont_export_launch(a.state_in, a.scale_in, segS, segSc, a.log_alpha,
                                            reinterpret_cast<float*>(ws + p.off_segDec), a.state_out, a.scale_out,
                                            BH, s.T, mat, s.Ls, a.t0, a.stream);
    if (st != LL_OK) return st;
  } else if (a.state_out) {
    return export_states(a.state_out, a.scale_out);
  }
  return LL_OK;
}

}  // namespace

ll_status simt_fenwick_launch(const float* S, float* F, const double* tot, double* G, int N, int mat, int BH,
                              cudaStream_t stream, __nv_bfloat16* Ft, double* cum, bool f32_nodes) {
  if (N <= kFenFastN) {
    if (mat % kFenVec != 0) return LL_ERR_UNSUPPORTED;  // head dims of 16..128 make it a multiple of 256
    const size_t smf = fen_smem(N);
    LL_CUDA_OK(cudaFuncSetAttribute(simt_fenwick_fast_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smf));
    const int per = kFenVec * kThreads;
    simt_fenwick_fast_kernel<<<dim3((mat + per - 1) / per, BH), kThreads, smf, stream>>>(S, F, tot, G, N, mat, Ft, cum,
                                                                                   f32_nodes || !Ft ? 1 : 0);
    LL_CUDA_OK(cudaGetLastError());
    return LL_OK;
  }
  const size_t sm = (size_t)N * sizeof(double);
  if (sm > 200 * 1024) return LL_ERR_UNSUPPORTED;  // chunk count beyond the on-chip prefix table
  LL_CUDA_OK(cudaFuncSetAttribute(simt_fenwick_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm));
  simt_fenwick_kernel<<<dim3((mat + kThreads - 1) / kThreads, BH), kThreads, sm, stream>>>(S, F, tot, G, N, mat, Ft, cum);
  LL_CUDA_OK(cudaGetLastError());
  return LL_OK;
}

size_t fwd_simt_workspace(const ll_shape& s) { return plan_of(s).total; }

size_t fwd_simt_cont_workspace(const ll_shape& s) { return plan_of(s).total_cont; }

int fwd_simt_launches(const ll_shape& s) { return s.Ls > 0 ? (s.T % plan_of(s).Ce ? 5 : 4) : 3; }

ll_status fwd_simt_launch(const FwdArgs& a) {
  SimtPlan p = plan_of(a.s);
  if (a.ws_bytes < (a.state_in ? p.total_cont : p.total)) return LL_ERR_WORKSPACE;
  if (a.s.io == LL_F32) return launch_typed<float>(a, p);
  return launch_typed<__nv_bfloat16>(a, p);
}

// (6): the decode states of t1 = t0 + T from the prefix states of t0 and the
// segment's own export at T (relative); shared by both forward paths.  First
// the segment's total decay per head (one block per head), then one thread
// per matrix element writes every slot once, summing the buckets that land
// on it.
constexpr int kDecThreads = 1024;

__global__ void __launch_bounds__(kDecThreads) segment_decay_kernel(const float* __restrict__ log_alpha,
                                                                    float* __restrict__ seg_decay, int T) {
  __shared__ double part[kDecThreads];
  const size_t bh = blockIdx.x;
  // four independent float64 chains per thread: the sum is latency-bound otherwise
  double g0 = 0.0, g1 = 0.0, g2 = 0.0, g3 = 0.0;
  int i = threadIdx.x;
  for (; i + 3 * kDecThreads < T; i += 4 * kDecThreads) {
    g0 += (double)log_alpha[bh * T + i];
    g1 += (double)log_alpha[bh * T + i + kDecThreads];
    g2 += (double)log_alpha[bh * T + i + 2 * kDecThreads];
    g3 += (double)log_alpha[bh * T + i + 3 * kDecThreads];
  }
  for (; i < T; i += kDecThreads) g0 += (double)log_alpha[bh * T + i];
  part[threadIdx.x] = (g0 + g1) + (g2 + g3);
  __syncthreads();
  for (int o = kDecThreads / 2; o > 0; o >>= 1) {
    if (threadIdx.x < o) part[threadIdx.x] += part[threadIdx.x + o];
    __syncthreads();
  }
  if (threadIdx.x == 0) seg_decay[bh] = expf((float)part[0]);
}

__global__ void __launch_bounds__(kThreads) cont_export_kernel(
    const float* __restrict__ pre_states, const float* __restrict__ pre_scales, const float* __restrict__ seg_states,
    const float* __restrict__ seg_scales, const float* __restrict__ seg_decay, float* __restrict__ state_out,
    float* __restrict__ scale_out, int T, int mat, int Ls, long long t0) {
  const size_t bh = blockIdx.y;
  const int idx = blockIdx.x * kThreads + threadIdx.x;
  const long long t1 = t0 + T;
  const int b = 64 - __clzll(t1 ^ t0);                         // bitlen(t1 xor t0)
  const long long P = 1ll << (64 - __clzll((long long)T - 1));  // smallest power of two >= T
  const float dec = seg_decay[bh];
  if (idx < mat) {
    for (int out = 0; out < Ls; ++out) {
      float acc = 0.f;
      if ((t1 >> out) & 1) {
        for (int slot = 0; slot < Ls; ++slot) {
          // prefix level slot+1 goes to max(slot+1, b), decayed over the segment
          if (((t0 >> slot) & 1) && (slot + 1 > b ? slot + 1 : b) == out + 1)
            acc = fmaf(pre_scales[bh * Ls + slot] * dec, pre_states[(bh * Ls + slot) * (size_t)mat + idx], acc);
          // the segment's level slot+1 keeps it if T < P, else goes to b
          if (((T >> slot) & 1) && (T < P ? slot + 1 : b) == out + 1)
            acc = fmaf(seg_scales[bh * Ls + slot], seg_states[(bh * Ls + slot) * (size_t)mat + idx], acc);
        }
      }
      state_out[(bh * Ls + out) * (size_t)mat + idx] = acc;
    }
  }
  if (blockIdx.x == 0 && threadIdx.x == 0)
    for (int out = 0; out < Ls; ++out) scale_out[bh * Ls + out] = ((t1 >> out) & 1) ? 1.f : 0.f;
}

ll_status cont_export_launch(const float* pre_states, const float* pre_scales, const float* seg_states,
                             const float* seg_scales, const float* log_alpha, float* seg_decay, float* state_out,
                             float* scale_out, int BH, int T, int mat, int Ls, long long t0, cudaStream_t stream) {
  segment_decay_kernel<<<BH, kDecThreads, 0, stream>>>(log_alpha, seg_decay, T);
  LL_CUDA_OK(cudaGetLastError());
  cont_export_kernel<<<dim3((mat + kThreads - 1) / kThreads, BH), kThreads, 0, stream>>>(
      pre_states, pre_scales, seg_states, seg_scales, seg_decay, state_out, scale_out, T, mat, Ls, t0);
  LL_CUDA_OK(cudaGetLastError());
  return LL_OK;
}

}  // namespace llattn
