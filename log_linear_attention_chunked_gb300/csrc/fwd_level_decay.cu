// Log-linear Mamba-2 with one decay per level, chunk-wise on the CUDA cores
// (float32 FMA, float64 running sums of the log decays).
//
// The memory of level l decays at its own rate alpha_t^(l): at every step r a
// key decays at the rate of the level it occupies then ("Log-Linear
// Attention" study note §7 "Follow-up design" names a learned memory decay
// per level; this is the recurrent form of §3-3 with one decay per level
// state):
//   o_t = sum_{s<=t} lam_t[l(t,s)] exp(sum_{r in (s,t]} log_alpha_r[l(r,s)]) (q_t.k_s) v_s
//
// Key s, at level l = bitlen(t xor s) for query t, spent the steps (s, t] on
// levels 1..l: on a level m < l exactly the 2^(m-1) steps of the block just
// above s's own aligned block of 2^(m-1) positions (when bit m-1 of s is
// clear, none otherwise), and on level l the steps from the start of t's
// aligned block of 2^(l-1) positions through t.  The log decay is thus a key
// part plus a query part of the same level,
//   K(s, l) = sum over those blocks below level l of the level's log decays
//   Q(t, l) = sum of log_alpha^(l) over [t with bits below l-1 cleared, t],
// and each chunk-wise step of the base form carries over level by level
// (chunk c of Ce = 2^lc tokens; levels above lc are inter-chunk, level
// lc+1+h belongs to node height h):
//   (1) intra   : o_i += sum_{j<=i} (q_i.k_j) exp(K(j,l) + Q(i,l)) lam_i[l] v_j, l = bitlen(i^j)
//   (2) state   : S_c = sum_j exp(K(j, lc+1)) v_j k_j^T  (K through the chunk's end)
//   (3) Fenwick : F_c = S_c + sum_{m<cto(c)} exp(D^(lc+1+m)(c-2^m, c]) F_{c-2^m},
//                 D^(l)(a, b] the level-l log decays of chunks a+1..b
//   (4) inter   : for set bit h of c (node e, level l = lc+1+h),
//                 o_i += lam_i[l] exp(D^(l)[c with bits below h cleared, c) + cs^(l)_i) F_e q_i
//   (5) export  : the node of level l of position T, decayed by D^(l) from
//                 the end of the node through T-1; for a ragged T the levels
//                 up to lc are the buckets of T mod Ce in the partial chunk.
#include <algorithm>

#include "level_decay.cuh"

namespace llattn {

namespace {

constexpr int kThreads = 256;
constexpr int kMaxChunkElems = 8192;
constexpr int kMaxChunks = 4096;  // Fenwick chain on chip: node heights 0..12
constexpr int kLv = 13;

struct LdPlan {
  int Ce, N, lc, Lx;  // chunk, #chunks, log2(Ce), inter-chunk levels (>= 1 slot)
  size_t off_S, off_F, off_tot, off_cum, off_O, total;
};

LdPlan plan_of(const ll_shape& s) {
  LdPlan p{};
  const int d = std::max(s.dk, s.dv);
  p.Ce = s.chunk;
  while (p.Ce * d > kMaxChunkElems && p.Ce > 16) p.Ce >>= 1;
  p.N = (s.T + p.Ce - 1) / p.Ce;
  p.lc = ilog2(p.Ce);
  p.Lx = std::max(s.L - p.lc - 1, 1);
  const size_t BH = (size_t)s.B * s.H, mat = (size_t)s.dv * s.dk;
  size_t off = 0;
  p.off_S = off;   off = align_up(off + BH * p.N * mat * sizeof(float), 256);
  p.off_F = off;   off = align_up(off + BH * p.N * mat * sizeof(float), 256);
  p.off_tot = off; off = align_up(off + BH * p.N * p.Lx * sizeof(double), 256);
  p.off_cum = off; off = align_up(off + BH * p.N * p.Lx * sizeof(double), 256);
  p.off_O = off;
  if (s.io != LL_F32) off = align_up(off + BH * (size_t)s.T * s.dv * sizeof(float), 256);
  p.total = off;
  return p;
}

// cs[i] = sum of la[(row0 + r) * L + lv] over rows r <= i of the chunk (rows
// >= nv add 0), float64, Ce <= 128; every thread takes part; cs is complete
// after the caller's next __syncthreads
__device__ __forceinline__ void level_scan(double* cs, const float* la, size_t row0, int nv, int Ce, int L, int lv) {
  __shared__ double wsum[4];
  const int t = threadIdx.x, lane = t & 31, w = t >> 5;
  double x = (t < Ce && t < nv) ? (double)la[(row0 + t) * L + lv] : 0.0;
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

// (1) + (2) and the chunk's totals of the inter-chunk levels; one CTA per (chunk, head).
template <typename IO>
__global__ void __launch_bounds__(kThreads) ld_chunk_kernel(const IO* __restrict__ q, const IO* __restrict__ k,
                                                            const IO* __restrict__ v, const float* __restrict__ la,
                                                            const float* __restrict__ lam, float* o_intra,
                                                            float* __restrict__ S, double* __restrict__ totL, int T,
                                                            int dk, int dv, int L, int Ce, int lc, int Lx) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  const int c = blockIdx.x, N = gridDim.x;
  const size_t bh = blockIdx.y;
  const int tid = threadIdx.x;
  const int dkp = dk + 1, dvp = dv + 1, Cp = Ce + 1;
  const int kq = lc + 1, kk = lc + 2;  // row lengths of the Q and K tables

  double* csl = reinterpret_cast<double*>(smem_raw);  // [lc][Ce] running sums of levels 1..lc
  double* Qf = csl + (size_t)lc * Ce;                 // [Ce][lc+1], entries 1..lc
  double* Kf = Qf + (size_t)Ce * kq;                  // [Ce][lc+2], entries 1..lc+1
  float* wdec = reinterpret_cast<float*>(Kf + (size_t)Ce * kk);
  float* qs = wdec + Ce;
  float* ks = qs + Ce * dkp;
  float* vs = ks + Ce * dkp;
  float* P = vs + Ce * dvp;

  const size_t row0 = bh * T + (size_t)c * Ce;
  const int nv = min(Ce, T - c * Ce);
  // one thread per level: the running sums of the in-chunk levels (zero for
  // levels >= L, which no key of this T reaches), the totals of the
  // inter-chunk ones
  for (int m = tid + 1; m < max(L, lc + 1); m += kThreads) {
    double acc = 0.0;
    if (m <= lc) {
      for (int i = 0; i < Ce; ++i) {
        if (i < nv && m < L) acc += (double)la[(row0 + i) * L + m];
        csl[(size_t)(m - 1) * Ce + i] = acc;
      }
    } else {
      for (int i = 0; i < nv; ++i) acc += (double)la[(row0 + i) * L + m];
      totL[(bh * N + c) * Lx + (m - lc - 1)] = acc;
    }
  }
  for (int x = tid; x < Ce * dk; x += kThreads) {
    const int i = x / dk, f = x % dk;
    qs[i * dkp + f] = i < nv ? to_f(q[(row0 + i) * dk + f]) : 0.f;
    ks[i * dkp + f] = i < nv ? to_f(k[(row0 + i) * dk + f]) : 0.f;
  }
  for (int x = tid; x < Ce * dv; x += kThreads) {
    const int i = x / dv, e = x % dv;
    vs[i * dvp + e] = i < nv ? to_f(v[(row0 + i) * dv + e]) : 0.f;
  }
  __syncthreads();
  for (int x = tid; x < Ce; x += kThreads) {
    for (int l = 1; l <= lc; ++l) {
      const int bs = (x >> (l - 1)) << (l - 1);
      const double* cl = csl + (size_t)(l - 1) * Ce;
      Qf[x * kq + l] = cl[x] - (bs > 0 ? cl[bs - 1] : 0.0);
    }
    double acc = 0.0;
    Kf[x * kk + 1] = 0.0;
    for (int m = 1; m <= lc; ++m) {
      if (!((x >> (m - 1)) & 1)) {  // the block above x's own at height m-1
        const int ss = ((x >> m) << m) + (1 << (m - 1)), se = ss + (1 << (m - 1)) - 1;
        const double* cl = csl + (size_t)(m - 1) * Ce;
        acc += cl[se] - cl[ss - 1];
      }
      Kf[x * kk + m + 1] = acc;
    }
  }
  __syncthreads();
  for (int j = tid; j < Ce; j += kThreads) wdec[j] = expf((float)Kf[j * kk + lc + 1]);

  for (int x = tid; x < Ce * Ce; x += kThreads) {
    const int i = x / Ce, j = x % Ce;
    float p = 0.f;
    if (j <= i && i < nv) {
      float dot = 0.f;
      for (int f = 0; f < dk; ++f) dot = fmaf(qs[i * dkp + f], ks[j * dkp + f], dot);
      const int lv = bitlen((unsigned)(i ^ j));
      const float dec = lv == 0 ? 1.f : expf((float)(Kf[j * kk + lv] + Qf[i * kq + lv]));
      p = dot * dec * lam[(row0 + i) * L + lv];
    }
    P[i * Cp + j] = p;
  }
  __syncthreads();
  for (int x = tid; x < nv * dv; x += kThreads) {
    const int i = x / dv, e = x % dv;
    float acc = 0.f;
    for (int j = 0; j <= i; ++j) acc = fmaf(P[i * Cp + j], vs[j * dvp + e], acc);
    o_intra[(row0 + i) * dv + e] = acc;
  }
  float* Sc = S + (bh * N + c) * (size_t)dv * dk;
  for (int x = tid; x < dv * dk; x += kThreads) {
    const int e = x / dk, f = x % dk;
    float acc = 0.f;
    for (int j = 0; j < Ce; ++j) acc = fmaf(wdec[j] * vs[j * dvp + e], ks[j * dkp + f], acc);
    Sc[x] = acc;
  }
}

// Running sums over the chunks of every inter-chunk level's totals, per head:
// cumL[bh][x][i] = sum_{c <= i} totL[bh][c][x].  One warp per level.
__global__ void __launch_bounds__(kThreads) ld_cum_kernel(const double* __restrict__ totL, double* __restrict__ cumL,
                                                          int N, int Lx) {
  const size_t bh = blockIdx.x;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int x = warp; x < Lx; x += kThreads / 32) {
    double carry = 0.0;
    for (int base = 0; base < N; base += 32) {
      const int i = base + lane;
      double y = i < N ? totL[(bh * N + i) * Lx + x] : 0.0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const double z = __shfl_up_sync(0xffffffffu, y, o);
        if (lane >= o) y += z;
      }
      y += carry;
      if (i < N) cumL[(bh * Lx + x) * N + i] = y;
      carry = __shfl_sync(0xffffffffu, y, 31);
    }
  }
}

// (3): the Fenwick nodes, the chain on chip.  The prologue tabulates each
// child's decay (node i's children start at entry i - popcount(i)); each
// thread then keeps the latest node of every height in shared memory.
__global__ void __launch_bounds__(kThreads) ld_fenwick_kernel(const float* __restrict__ S, float* __restrict__ F,
                                                              const double* __restrict__ cumL, int N, int mat,
                                                              int Lx) {
  extern __shared__ float fsm[];
  float* coef = fsm;      // [N]
  float* last = fsm + N;  // [kLv][kThreads]
  const size_t bh = blockIdx.y;
  const double* cb = cumL + bh * Lx * (size_t)N;
  for (int i = threadIdx.x; i < N; i += kThreads) {
    const int h = __ffs(~i) - 1, o = i - __popc(i);
    for (int m = 0; m < h; ++m)
      coef[o + m] = m < Lx ? expf((float)(cb[(size_t)m * N + i] - cb[(size_t)m * N + i - (1 << m)])) : 0.f;
  }
  __syncthreads();
  const int idx = blockIdx.x * kThreads + threadIdx.x;
  if (idx >= mat) return;
  const float* Sb = S + bh * N * (size_t)mat;
  float* Fb = F + bh * N * (size_t)mat;
  float s0 = Sb[idx], s1 = N > 1 ? Sb[(size_t)mat + idx] : 0.f, s2 = N > 2 ? Sb[2 * (size_t)mat + idx] : 0.f,
        s3 = N > 3 ? Sb[3 * (size_t)mat + idx] : 0.f;
  for (int i = 0; i < N; ++i) {
    float acc = s0;
    s0 = s1;
    s1 = s2;
    s2 = s3;
    s3 = i + 4 < N ? Sb[(size_t)(i + 4) * mat + idx] : 0.f;
    const int h = __ffs(~i) - 1, o = i - __popc(i);
    for (int m = 0; m < h; ++m) acc = fmaf(coef[o + m], last[m * kThreads + threadIdx.x], acc);
    last[h * kThreads + threadIdx.x] = acc;
    Fb[(size_t)i * mat + idx] = acc;
  }
}

// (4): one CTA per (chunk, head); adds the inter-chunk levels to the intra
// result and writes o.
template <typename IO>
__global__ void __launch_bounds__(kThreads) ld_inter_kernel(const IO* __restrict__ q, const float* __restrict__ la,
                                                            const float* __restrict__ lam, const float* o_intra,
                                                            const float* __restrict__ F,
                                                            const double* __restrict__ cumL, IO* o, int T, int dk,
                                                            int dv, int L, int Ce, int lc, int Lx) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  const int c = blockIdx.x, N = gridDim.x;
  const size_t bh = blockIdx.y;
  const int tid = threadIdx.x;
  const int dkp = dk + 1;
  double* cs = reinterpret_cast<double*>(smem_raw);
  float* w = reinterpret_cast<float*>(cs + Ce);
  float* qs = w + Ce;
  float* Fs = qs + Ce * dk;
  float* Oc = Fs + dv * dkp;

  const size_t row0 = bh * T + (size_t)c * Ce;
  const int nv = min(Ce, T - c * Ce);
  for (int x = tid; x < Ce * dk; x += kThreads) qs[x] = x < nv * dk ? to_f(q[row0 * dk + x]) : 0.f;
  for (int x = tid; x < Ce * dv; x += kThreads) Oc[x] = x < nv * dv ? o_intra[row0 * dv + x] : 0.f;
  const size_t mat = (size_t)dv * dk;
  for (int h = 0; (c >> h) != 0; ++h) {
    if (!((c >> h) & 1)) continue;
    const int e = ((c >> (h + 1)) << (h + 1)) + (1 << h) - 1;
    const int lv = lc + 1 + h;
    level_scan(cs, la, row0, nv, Ce, L, lv);
    const int cb = c & ~((1 << h) - 1);  // first chunk of c's block at height h
    const double* cl = cumL + (bh * Lx + h) * (size_t)N;
    const double D = cb < c ? cl[c - 1] - (cb > 0 ? cl[cb - 1] : 0.0) : 0.0;
    const float* Fe = F + (bh * N + e) * mat;
    for (int x = tid; x < (int)mat; x += kThreads) Fs[(x / dk) * dkp + (x % dk)] = Fe[x];
    __syncthreads();
    for (int i = tid; i < Ce; i += kThreads) w[i] = i < nv ? lam[(row0 + i) * L + lv] * expf((float)(cs[i] + D)) : 0.f;
    __syncthreads();
    for (int x = tid; x < Ce * dv; x += kThreads) {
      const int i = x / dv, ev = x % dv;
      float acc = 0.f;
      for (int f = 0; f < dk; ++f) acc = fmaf(Fs[ev * dkp + f], qs[i * dk + f], acc);
      Oc[x] = fmaf(w[i], acc, Oc[x]);
    }
    __syncthreads();
  }
  __syncthreads();
  for (int x = tid; x < nv * dv; x += kThreads) o[row0 * dv + x] = from_f<IO>(Oc[x]);
}

// (5): the level states of position T from the nodes of the Nq full chunks.
__global__ void __launch_bounds__(kThreads) ld_export_kernel(const float* __restrict__ F,
                                                             const double* __restrict__ cumL,
                                                             float* __restrict__ state_out,
                                                             float* __restrict__ scale_out, int N, int Nq, int mat,
                                                             int Ls, int lc, int Lx) {
  const size_t bh = blockIdx.y;
  const int idx = blockIdx.x * kThreads + threadIdx.x;
  for (int slot = 0; slot < Ls; ++slot) {
    const int h = slot - lc;  // level slot+1 = lc + 1 + h
    float val = 0.f, sc = 0.f;
    if (h >= 0 && h < 31 && ((Nq >> h) & 1)) {
      const int e = ((Nq >> (h + 1)) << (h + 1)) + (1 << h) - 1;
      const int cb = Nq & ~((1 << h) - 1);  // the node's keys sit at level slot+1 from chunk cb on
      double D = 0.0;
      if (cb < N) {
        const double* cl = cumL + (bh * Lx + h) * (size_t)N;
        D = cl[N - 1] - (cb > 0 ? cl[cb - 1] : 0.0);
      }
      if (idx < mat) val = expf((float)D) * F[(bh * N + e) * (size_t)mat + idx];
      sc = 1.f;
    }
    if (idx < mat) state_out[(bh * Ls + slot) * (size_t)mat + idx] = val;
    if (blockIdx.x == 0 && threadIdx.x == 0) scale_out[bh * Ls + slot] = sc;
  }
}

// (5) for a ragged T: levels 1..lc of position T are the buckets of r = T mod
// Ce in the partial chunk; bucket l (bit l-1 of r) holds rows [lo, lo + 2^(l-1)),
// lo = r with bits below l cleared.  Row a of it carries K(a, l) and then the
// level-l decays of rows lo + 2^(l-1) .. r-1.
template <typename IO>
__global__ void __launch_bounds__(kThreads) ld_tail_export_kernel(const IO* __restrict__ k,
                                                                  const IO* __restrict__ v,
                                                                  const float* __restrict__ la,
                                                                  float* __restrict__ state_out,
                                                                  float* __restrict__ scale_out, int T, int dk,
                                                                  int dv, int L, int Ls, int r, int lc) {
  __shared__ double csl[7 * 128];  // running sums of levels 1..lc over the partial chunk's rows
  __shared__ float dec[128];
  const size_t bh = blockIdx.y;
  const int idx = blockIdx.x * kThreads + threadIdx.x;
  const size_t row0 = bh * T + (size_t)(T - r);
  for (int m = threadIdx.x + 1; m <= lc; m += kThreads) {
    double acc = 0.0;
    for (int a = 0; a < r; ++a) {
      if (m < L) acc += (double)la[(row0 + a) * L + m];
      csl[(m - 1) * 128 + a] = acc;
    }
  }
  __syncthreads();
  for (int a = threadIdx.x; a < r; a += kThreads) {
    const int l = bitlen((unsigned)(r ^ a));  // a's level for query r (bit l-1 of r is set, of a clear)
    double g = 0.0;
    for (int m = 1; m < l; ++m) {
      if (!((a >> (m - 1)) & 1)) {
        const int ss = ((a >> m) << m) + (1 << (m - 1)), se = ss + (1 << (m - 1)) - 1;
        g += csl[(m - 1) * 128 + se] - csl[(m - 1) * 128 + ss - 1];
      }
    }
    const int hi = ((r >> l) << l) + (1 << (l - 1));  // the steps hi..r-1 at level l
    if (hi < r) g += csl[(l - 1) * 128 + r - 1] - csl[(l - 1) * 128 + hi - 1];
    dec[a] = expf((float)g);
  }
  __syncthreads();
  const int mat = dv * dk;
  for (int l = 1; l <= Ls && l <= lc; ++l) {
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
ll_status launch_typed(const FwdArgs& a, const LdPlan& p) {
  const ll_shape& s = a.s;
  unsigned char* ws = static_cast<unsigned char*>(a.ws);
  float* S = reinterpret_cast<float*>(ws + p.off_S);
  float* F = reinterpret_cast<float*>(ws + p.off_F);
  double* totL = reinterpret_cast<double*>(ws + p.off_tot);
  double* cumL = reinterpret_cast<double*>(ws + p.off_cum);
  float* o_intra = s.io == LL_F32 ? static_cast<float*>(a.o) : reinterpret_cast<float*>(ws + p.off_O);
  const int BH = s.B * s.H, Ce = p.Ce, mat = s.dv * s.dk;
  const size_t sm1 = sizeof(double) * ((size_t)p.lc * Ce + (size_t)Ce * (p.lc + 1) + (size_t)Ce * (p.lc + 2)) +
                     sizeof(float) * ((size_t)Ce + 2 * (size_t)Ce * (s.dk + 1) + (size_t)Ce * (s.dv + 1) +
                                      (size_t)Ce * (Ce + 1));
  LL_CUDA_OK(cudaFuncSetAttribute(ld_chunk_kernel<IO>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm1));
  ld_chunk_kernel<IO><<<dim3(p.N, BH), kThreads, sm1, a.stream>>>(
      static_cast<const IO*>(a.q), static_cast<const IO*>(a.k), static_cast<const IO*>(a.v), a.log_alpha, a.lam,
      o_intra, S, totL, s.T, s.dk, s.dv, s.L, Ce, p.lc, p.Lx);
  LL_CUDA_OK(cudaGetLastError());
  ld_cum_kernel<<<BH, kThreads, 0, a.stream>>>(totL, cumL, p.N, p.Lx);
  LL_CUDA_OK(cudaGetLastError());
  const size_t smf = sizeof(float) * ((size_t)p.N + (size_t)kLv * kThreads);
  LL_CUDA_OK(cudaFuncSetAttribute(ld_fenwick_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smf));
  ld_fenwick_kernel<<<dim3((mat + kThreads - 1) / kThreads, BH), kThreads, smf, a.stream>>>(S, F, cumL, p.N, mat,
                                                                                             p.Lx);
  LL_CUDA_OK(cudaGetLastError());
  const size_t sm3 = Ce * sizeof(double) + Ce * sizeof(float) +
                     sizeof(float) * ((size_t)Ce * s.dk + (size_t)s.dv * (s.dk + 1) + (size_t)Ce * s.dv);
  LL_CUDA_OK(cudaFuncSetAttribute(ld_inter_kernel<IO>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm3));
  ld_inter_kernel<IO><<<dim3(p.N, BH), kThreads, sm3, a.stream>>>(static_cast<const IO*>(a.q), a.log_alpha, a.lam,
                                                                  o_intra, F, cumL, static_cast<IO*>(a.o), s.T,
                                                                  s.dk, s.dv, s.L, Ce, p.lc, p.Lx);
  LL_CUDA_OK(cudaGetLastError());
  if (a.state_out) {
    const int Nq = s.T / Ce, r = s.T % Ce;
    ld_export_kernel<<<dim3((mat + kThreads - 1) / kThreads, BH), kThreads, 0, a.stream>>>(
        F, cumL, a.state_out, a.scale_out, p.N, Nq, mat, s.Ls, p.lc, p.Lx);
    LL_CUDA_OK(cudaGetLastError());
    if (r > 0) {
      ld_tail_export_kernel<IO><<<dim3((mat + kThreads - 1) / kThreads, BH), kThreads, 0, a.stream>>>(
          static_cast<const IO*>(a.k), static_cast<const IO*>(a.v), a.log_alpha, a.state_out, a.scale_out, s.T,
          s.dk, s.dv, s.L, s.Ls, r, p.lc);
      LL_CUDA_OK(cudaGetLastError());
    }
  }
  return LL_OK;
}

}  // namespace

size_t fwd_level_decay_workspace(const ll_shape& s) {
  const LdPlan p = plan_of(s);
  return p.N > kMaxChunks ? 0 : p.total;
}

int fwd_level_decay_launches(const ll_shape& s) {
  const LdPlan p = plan_of(s);
  return 4 + (s.Ls > 0 ? (s.T % p.Ce ? 2 : 1) : 0);
}

ll_status fwd_level_decay_launch(const FwdArgs& a) {
  const LdPlan p = plan_of(a.s);
  if (p.N > kMaxChunks) return LL_ERR_UNSUPPORTED;
  if (a.ws_bytes < p.total) return LL_ERR_WORKSPACE;
  if (a.s.io == LL_F32) return launch_typed<float>(a, p);
  return launch_typed<__nv_bfloat16>(a, p);
}

}  // namespace llattn
