// Backward of the chunked log-linear Mamba-2 forward on CUDA cores (float32 FMA).
//
// The gradient of O = (A . M) V, A = Q K^T, M = Gamma . H with
// Gamma(t,s) = exp(c_t - c_s), c the cumulative sum of log_alpha, and
// H(t,s) = lam_t[level(t,s)] ("Log-Linear Attention" study note §3-4 parallel
// form and §3-5 mask composition; the study note §4-5 / §6 and the
// gist.science (zh) summary §5 name this backward, with its lambda terms, as
// the hard part of an implementation but print no formulas).  With
// P = A . M and dP = dO V^T on the causal triangle:
//   dV = P^T dO,   dQ = (dP . M) K,   dK = (dP . M)^T Q,
//   dlam_t[l] = sum over keys s of level l of dP_ts A_ts Gamma_ts,
//   dc_t = sum_s dP_ts P_ts - sum_t' dP_t't P_t't
//        = sum_l lam_t[l] dlam_t[l] - v_t . dv_t    (o_t is linear in lam_t, and
//                                                    the column sum is v_t . dv_t),
//   dlog_alpha_r = sum over t >= r of dc_t.
//
// Chunk-wise (chunk c of Ce tokens; cs = cumulative log_alpha inside the
// chunk; F_e, G_e the forward's Fenwick nodes of keys, decayed to the end of
// chunk e):
//   (1) intra, one CTA per chunk: the dense Ce x Ce form of every gradient,
//       levels 0..log2(Ce) of dlam; also the chunk state S_c and the chunk's
//       total log-decay for (2), and it clears the chunk's key-side node R_c.
//   (2) Fenwick nodes F_e, G_e from S_c (the forward's kernel).
//   (3) query side, one CTA per chunk c; for every set bit h of c the node
//       e = (c with bits 0..h cleared) + 2^h - 1 holds the keys of level
//       lc+1+h of every query of c, and with D the decay from the end of e to
//       the start of c:
//         g_i = exp(cs_i + D) F_e^T do_i,   dq_i += lam_i[lc+1+h] g_i,
//         dlam_i[lc+1+h] = g_i . q_i,
//       and the chunk adds its queries to the key-side node of e,
//         R_e += sum_i lam_i[lc+1+h] exp(cs_i + D) do_i q_i^T,
//       so that R_e holds every query that sees the keys of e at that level,
//       decayed to the end of e.
//   (4) key side, one CTA per chunk c: the keys of c are in the block of e_h
//       for every clear bit h of c (e_h as above); with E_c the sum of the
//       R_{e_h} decayed from the end of e_h back to the end of c,
//         dv_j += exp(cs_end - cs_j) E_c k_j,   dk_j += exp(cs_end - cs_j) E_c^T v_j;
//       the rows of dk, dv are final here, so dc_j is formed here too.
//   (5) per head: dlog_alpha as suffix sums of dc (float64).
// Ragged T: the last chunk's missing rows are absent (zero inputs, log_alpha 0,
// no outputs), as in the forward.
#include <algorithm>

#include "bwd.cuh"

namespace llattn {

namespace {

constexpr int kThreads = 256;
constexpr int kSuffixThreads = 256;
constexpr int kSuffixRun = 8;
constexpr int kSuffixPart = kSuffixThreads * kSuffixRun;  // tokens per CTA of the suffix sums
constexpr int kMaxChunkElems = 8192;           // Ce * max(dk, dv), as in the forward
constexpr size_t kMaxSmem = 220 * 1024;        // dynamic shared memory of one CTA

size_t intra_smem(int Ce, int dk, int dv) {
  return Ce * sizeof(double) +
         sizeof(float) * ((size_t)Ce + 2 * (size_t)Ce * (dk + 1) + 2 * (size_t)Ce * (dv + 1) + 3 * (size_t)Ce * (Ce + 1));
}
size_t query_smem(int Ce, int dk, int dv) {
  return Ce * sizeof(double) +
         sizeof(float) * (2 * (size_t)Ce + 3 * (size_t)Ce * dk + (size_t)Ce * dv + (size_t)dv * (dk + 1));
}
size_t key_smem(int Ce, int dk, int dv) {
  return Ce * sizeof(double) +
         sizeof(float) * ((size_t)Ce + (size_t)Ce * (dk + 1) + 2 * (size_t)Ce * (dv + 1) + (size_t)dv * (dk + 1));
}

struct BwdPlan {
  int Ce, N, lc;
  size_t off_S, off_F, off_R, off_tot, off_G, off_dq, off_dk, off_dv, off_dc, off_Ft, off_cum, off_sfx, off_ptot, total;
};

BwdPlan plan_of(const ll_shape& s) {
  BwdPlan p{};
  const int d = std::max(s.dk, s.dv);
  p.Ce = s.chunk;
  if (bwd_tc_supported(s)) p.Ce = 128;  // the tensor-core kernels' tiles, whatever the chunk
  while (!bwd_tc_supported(s) && p.Ce > 16 && (p.Ce * d > kMaxChunkElems || intra_smem(p.Ce, s.dk, s.dv) > kMaxSmem ||
                       query_smem(p.Ce, s.dk, s.dv) > kMaxSmem || key_smem(p.Ce, s.dk, s.dv) > kMaxSmem))
    p.Ce >>= 1;
  p.N = (s.T + p.Ce - 1) / p.Ce;
  p.lc = ilog2(p.Ce);
  const size_t BH = (size_t)s.B * s.H;
  const size_t mat = (size_t)s.dv * s.dk;
  size_t off = 0;
  p.off_S = off;   off = align_up(off + BH * p.N * mat * sizeof(float), 256);
  // float32 nodes: the tensor-core path reads only their bf16 tiles, and the
  // Fenwick kernel writes F there only when its chain cannot stay on chip
  const bool need_f32_nodes = !bwd_tc_supported(s) || p.N > kFenwickOnChipChunks;
  p.off_F = off;   off = align_up(off + (need_f32_nodes ? BH * p.N * mat * sizeof(float) : 0), 256);
  // (the tensor-core path keeps its query kernel's item counter in the word after R)
  p.off_R = off;   off = align_up(off + BH * p.N * mat * sizeof(float) + (bwd_tc_supported(s) ? sizeof(unsigned) : 0), 256);
  p.off_tot = off; off = align_up(off + BH * p.N * sizeof(double), 256);
  p.off_G = off;   off = align_up(off + BH * p.N * sizeof(double), 256);
  p.off_dc = off;  off = align_up(off + BH * (size_t)s.T * sizeof(float), 256);
  p.off_Ft = off;
  if (bwd_tc_supported(s)) off = align_up(off + BH * p.N * mat * 2, 256);  // the nodes as bf16 tiles
  p.off_cum = off;
  off = align_up(off + BH * p.N * sizeof(double), 256);  // running sums of the chunk totals
  // the suffix sums of dc: each part's own (float64) and the parts' totals
  p.off_sfx = off;  off = align_up(off + BH * (size_t)s.T * sizeof(double), 256);
  p.off_ptot = off; off = align_up(off + BH * (size_t)((s.T + kSuffixPart - 1) / kSuffixPart) * sizeof(double), 256);
  p.off_dq = p.off_dk = p.off_dv = off;
  if (s.io != LL_F32) {  // partial sums of dq, dk, dv (float32 io accumulates in the outputs):
    // float32 on the CUDA cores, the in-tile parts in bf16 on the tensor-core path
    const size_t pe = bwd_tc_supported(s) ? 2 : sizeof(float);
    p.off_dq = off; off = align_up(off + BH * (size_t)s.T * s.dk * pe, 256);
    p.off_dk = off; off = align_up(off + BH * (size_t)s.T * s.dk * pe, 256);
    p.off_dv = off; off = align_up(off + BH * (size_t)s.T * s.dv * pe, 256);
  }
  p.total = off;
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

// (1) one CTA per (chunk, head)
template <typename IO>
__global__ void __launch_bounds__(kThreads) bwd_intra_kernel(
    const IO* __restrict__ q, const IO* __restrict__ k, const IO* __restrict__ v, const IO* __restrict__ dout,
    const float* __restrict__ log_alpha, const float* __restrict__ lam, float* __restrict__ dq32,
    float* __restrict__ dk32, float* __restrict__ dv32, float* __restrict__ dlam, float* __restrict__ S,
    double* __restrict__ tot, float* __restrict__ R, int T, int dk, int dv, int L, int Ce, int lc) {
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
  float* gs = vs + Ce * dvp;   // dO
  float* P = gs + Ce * dvp;    // A . M
  float* dA = P + Ce * Cp;     // dP . M
  float* X = dA + Ce * Cp;     // dP . A . Gamma: its level sums are dlam

  const size_t row0 = bh * T + (size_t)c * Ce;
  const int nv = min(Ce, T - c * Ce);
  chunk_scan(cs, log_alpha, row0, nv, Ce);
  if (tid == Ce - 1) tot[bh * N + c] = cs[Ce - 1];
  for (int x = tid; x < Ce * dk; x += kThreads) {
    const int i = x / dk, f = x % dk;
    qs[i * dkp + f] = i < nv ? to_f(q[(row0 + i) * dk + f]) : 0.f;
    ks[i * dkp + f] = i < nv ? to_f(k[(row0 + i) * dk + f]) : 0.f;
  }
  for (int x = tid; x < Ce * dv; x += kThreads) {
    const int i = x / dv, e = x % dv;
    vs[i * dvp + e] = i < nv ? to_f(v[(row0 + i) * dv + e]) : 0.f;
    gs[i * dvp + e] = i < nv ? to_f(dout[(row0 + i) * dv + e]) : 0.f;
  }
  __syncthreads();
  for (int j = tid; j < Ce; j += kThreads) wdec[j] = expf((float)(cs[Ce - 1] - cs[j]));
  for (int x = tid; x < Ce * Ce; x += kThreads) {
    const int i = x / Ce, j = x % Ce;
    float p = 0.f, da = 0.f, xx = 0.f;
    if (j <= i && i < nv) {
      float a = 0.f, g = 0.f;
      for (int f = 0; f < dk; ++f) a = fmaf(qs[i * dkp + f], ks[j * dkp + f], a);
      for (int e = 0; e < dv; ++e) g = fmaf(gs[i * dvp + e], vs[j * dvp + e], g);
      const float ex = expf((float)(cs[i] - cs[j]));
      const float lm = lam[(row0 + i) * L + bitlen((unsigned)(i ^ j))];
      p = a * ex * lm;
      da = g * ex * lm;
      xx = g * a * ex;
    }
    P[i * Cp + j] = p;
    dA[i * Cp + j] = da;
    X[i * Cp + j] = xx;
  }
  __syncthreads();
  for (int x = tid; x < nv * dk; x += kThreads) {
    const int i = x / dk, f = x % dk;
    float aq = 0.f, ak = 0.f;
    for (int j = 0; j <= i; ++j) aq = fmaf(dA[i * Cp + j], ks[j * dkp + f], aq);
    for (int r = i; r < nv; ++r) ak = fmaf(dA[r * Cp + i], qs[r * dkp + f], ak);  // i is the key row here
    dq32[(row0 + i) * dk + f] = aq;
    dk32[(row0 + i) * dk + f] = ak;
  }
  for (int x = tid; x < nv * dv; x += kThreads) {
    const int j = x / dv, e = x % dv;
    float acc = 0.f;
    for (int i = j; i < nv; ++i) acc = fmaf(P[i * Cp + j], gs[i * dvp + e], acc);
    dv32[(row0 + j) * dv + e] = acc;
  }
  // levels 0..lc: level l of query i (l >= 1, bit l-1 of i set) holds the keys
  // of the lower half of i's aligned block of 2^l rows
  const int nl = min(lc + 1, L);
  for (int x = tid; x < nv * nl; x += kThreads) {
    const int i = x / nl, l = x % nl;
    float acc = 0.f;
    if (l == 0) {
      acc = X[i * Cp + i];
    } else if ((i >> (l - 1)) & 1) {
      const int lo = (i >> l) << l;
      for (int j = lo; j < lo + (1 << (l - 1)); ++j) acc += X[i * Cp + j];
    }
    dlam[(row0 + i) * L + l] = acc;
  }
  // chunk state S_c[e][f] = sum_j wdec_j v_j[e] k_j[f]; the key-side node of c starts at 0
  const size_t mat = (size_t)dv * dk;
  float* Sc = S + (bh * N + c) * mat;
  float* Rc = R + (bh * N + c) * mat;
  for (int x = tid; x < (int)mat; x += kThreads) {
    const int e = x / dk, f = x % dk;
    float acc = 0.f;
    for (int j = 0; j < nv; ++j) acc = fmaf(wdec[j] * vs[j * dvp + e], ks[j * dkp + f], acc);
    Sc[x] = acc;
    Rc[x] = 0.f;
  }
}

// (3) one CTA per (chunk, head)
template <typename IO>
__global__ void __launch_bounds__(kThreads) bwd_query_kernel(
    const IO* __restrict__ q, const IO* __restrict__ dout, const float* __restrict__ log_alpha,
    const float* __restrict__ lam, const float* __restrict__ F, const double* __restrict__ G,
    const float* dq32, IO* dq, float* __restrict__ dlam, float* __restrict__ R, int T, int dk, int dv, int L,
    int Ce, int lc) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  const int c = blockIdx.x;
  const int N = gridDim.x;
  const size_t bh = blockIdx.y;
  const int tid = threadIdx.x;
  const int dkp = dk + 1;
  double* cs = reinterpret_cast<double*>(smem_raw);
  float* w = reinterpret_cast<float*>(cs + Ce);  // exp(cs_i + D)
  float* lw = w + Ce;                            // lam_i[level] exp(cs_i + D)
  float* qs = lw + Ce;                           // [Ce][dk]
  float* gq = qs + Ce * dk;                      // [Ce][dk] g_i[f] q_i[f]
  float* acc = gq + Ce * dk;                     // [Ce][dk] inter-chunk part of dq
  float* gs = acc + Ce * dk;                     // [Ce][dv] dO
  float* Fs = gs + Ce * dv;                      // [dv][dk + 1]

  const size_t row0 = bh * T + (size_t)c * Ce;
  const int nv = min(Ce, T - c * Ce);
  chunk_scan(cs, log_alpha, row0, nv, Ce);
  for (int x = tid; x < Ce * dk; x += kThreads) {
    qs[x] = x < nv * dk ? to_f(q[row0 * dk + x]) : 0.f;
    acc[x] = 0.f;
  }
  for (int x = tid; x < Ce * dv; x += kThreads) gs[x] = x < nv * dv ? to_f(dout[row0 * dv + x]) : 0.f;
  __syncthreads();

  const size_t mat = (size_t)dv * dk;
  double D = 0.0;
  for (int h = 0; (c >> h) != 0; ++h) {
    if (!((c >> h) & 1)) continue;
    const int e = ((c >> (h + 1)) << (h + 1)) + (1 << h) - 1;
    const int lv = lc + 1 + h;
    const float* Fe = F + (bh * N + e) * mat;
    for (int x = tid; x < (int)mat; x += kThreads) Fs[(x / dk) * dkp + (x % dk)] = Fe[x];
    for (int i = tid; i < Ce; i += kThreads) {
      const float wi = i < nv ? expf((float)(cs[i] + D)) : 0.f;
      w[i] = wi;
      lw[i] = i < nv ? wi * lam[(row0 + i) * L + lv] : 0.f;
    }
    __syncthreads();
    // g_i[f] = w_i sum_e F[e][f] do_i[e]
    for (int x = tid; x < Ce * dk; x += kThreads) {
      const int i = x / dk, f = x % dk;
      float a = 0.f;
      for (int ev = 0; ev < dv; ++ev) a = fmaf(Fs[ev * dkp + f], gs[i * dv + ev], a);
      acc[x] = fmaf(lw[i], a, acc[x]);
      gq[x] = w[i] * a * qs[x];
    }
    // this chunk's queries into the key-side node of e
    float* Re = R + (bh * N + e) * mat;
    for (int x = tid; x < (int)mat; x += kThreads) {
      const int ev = x / dk, f = x % dk;
      float a = 0.f;
      for (int i = 0; i < nv; ++i) a = fmaf(lw[i] * gs[i * dv + ev], qs[i * dk + f], a);
      atomicAdd(Re + x, a);
    }
    __syncthreads();
    for (int i = tid; i < nv; i += kThreads) {
      float a = 0.f;
      for (int f = 0; f < dk; ++f) a += gq[i * dk + f];
      dlam[(row0 + i) * L + lv] = a;
    }
    D += G[bh * N + e];
    __syncthreads();
  }
  // the levels above lc that hold no key of this chunk's queries
  const int nh = L - (lc + 1);
  for (int x = tid; x < nv * max(nh, 0); x += kThreads) {
    const int i = x / nh, h = x % nh;
    if (!(h < 31 && ((c >> h) & 1))) dlam[(row0 + i) * L + lc + 1 + h] = 0.f;
  }
  for (int x = tid; x < nv * dk; x += kThreads) dq[row0 * dk + x] = from_f<IO>(dq32[row0 * dk + x] + acc[x]);
}

// (4) one CTA per (chunk, head)
template <typename IO>
__global__ void __launch_bounds__(kThreads) bwd_key_kernel(
    const IO* __restrict__ k, const IO* __restrict__ v, const float* __restrict__ log_alpha,
    const float* __restrict__ lam, const float* __restrict__ dlam, const float* __restrict__ R,
    const double* __restrict__ cum, const float* dk32, const float* dv32, IO* dk, IO* dv,
    float* __restrict__ dc, int T, int dkd, int dvd, int L, int Ce) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  __shared__ float coef[32];
  __shared__ int ent[32];
  __shared__ int n_sh;
  const int c = blockIdx.x;
  const int N = gridDim.x;
  const size_t bh = blockIdx.y;
  const int tid = threadIdx.x;
  const int dkp = dkd + 1, dvp = dvd + 1;
  double* cs = reinterpret_cast<double*>(smem_raw);
  float* wdec = reinterpret_cast<float*>(cs + Ce);
  float* ks = wdec + Ce;       // [Ce][dk + 1]
  float* vs = ks + Ce * dkp;   // [Ce][dv + 1]
  float* dvs = vs + Ce * dvp;  // [Ce][dv + 1] final dv rows
  float* Es = dvs + Ce * dvp;  // [dv][dk + 1]

  const size_t row0 = bh * T + (size_t)c * Ce;
  const int nv = min(Ce, T - c * Ce);
  if (tid == 0) {
    // the nodes whose blocks hold the keys of c and that have queries after
    // them, with the log-decay from the end of c to the end of each
    int n = 0;
    for (int h = 0; h < 31 && n < 32; ++h) {
      if ((c >> h) & 1) continue;
      const int e = ((c >> (h + 1)) << (h + 1)) + (1 << h) - 1;
      if (e + 1 >= N) break;  // e grows with h: no later node has queries either
      ent[n] = e;
      coef[n] = expf((float)(cum[bh * N + e] - cum[bh * N + c]));
      ++n;
    }
    n_sh = n;
  }
  chunk_scan(cs, log_alpha, row0, nv, Ce);
  for (int x = tid; x < Ce * dkd; x += kThreads) {
    const int j = x / dkd, f = x % dkd;
    ks[j * dkp + f] = j < nv ? to_f(k[(row0 + j) * dkd + f]) : 0.f;
  }
  for (int x = tid; x < Ce * dvd; x += kThreads) {
    const int j = x / dvd, e = x % dvd;
    vs[j * dvp + e] = j < nv ? to_f(v[(row0 + j) * dvd + e]) : 0.f;
  }
  __syncthreads();
  const int n = n_sh;
  for (int j = tid; j < Ce; j += kThreads) wdec[j] = expf((float)(cs[Ce - 1] - cs[j]));
  const size_t mat = (size_t)dvd * dkd;
  if (n > 0) {
    for (int x = tid; x < (int)mat; x += kThreads) {
      float a = 0.f;
      for (int m = 0; m < n; ++m) a = fmaf(coef[m], R[(bh * N + ent[m]) * mat + x], a);
      Es[(x / dkd) * dkp + (x % dkd)] = a;
    }
  }
  __syncthreads();
  for (int x = tid; x < nv * dvd; x += kThreads) {
    const int j = x / dvd, e = x % dvd;
    float a = 0.f;
    if (n > 0)
      for (int f = 0; f < dkd; ++f) a = fmaf(Es[e * dkp + f], ks[j * dkp + f], a);
    const float r = fmaf(wdec[j], a, dv32[(row0 + j) * dvd + e]);
    dvs[j * dvp + e] = r;
    dv[(row0 + j) * dvd + e] = from_f<IO>(r);
  }
  for (int x = tid; x < nv * dkd; x += kThreads) {
    const int j = x / dkd, f = x % dkd;
    float a = 0.f;
    if (n > 0)
      for (int e = 0; e < dvd; ++e) a = fmaf(Es[e * dkp + f], vs[j * dvp + e], a);
    dk[(row0 + j) * dkd + f] = from_f<IO>(fmaf(wdec[j], a, dk32[(row0 + j) * dkd + f]));
  }
  __syncthreads();
  // dc_j = sum_l lam_j[l] dlam_j[l] - v_j . dv_j, one warp per row
  const int warp = tid >> 5, lane = tid & 31;
  for (int j = warp; j < Ce; j += kThreads / 32) {
    float a = 0.f;
    if (j < nv) {
      for (int l = lane; l < L; l += 32) a = fmaf(lam[(row0 + j) * L + l], dlam[(row0 + j) * L + l], a);
      for (int e = lane; e < dvd; e += 32) a = fmaf(-vs[j * dvp + e], dvs[j * dvp + e], a);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) a += __shfl_xor_sync(0xffffffffu, a, o);
    if (lane == 0) {
      if (j < nv) dc[row0 + j] = a;
    }
  }
}

// (5) dlog_alpha_r = sum_{t >= r} dc_t, in float64, in two passes over parts
// of kSuffixPart tokens (float64 arithmetic is scarce on this GPU: the parts
// spread it over the SMs).  First pass, one CTA per (part, head): each thread
// sums a run of kSuffixRun consecutive tokens (staged by coalesced loads,
// rows padded against bank conflicts), a suffix scan over the threads (warp
// shuffles, then over the warps) gives each run the sum of the part after it,
// and the thread writes its tokens' suffix sums inside the part (float64) and
// the part's total.  Second pass: each part adds the totals of the parts after
// it and rounds to float32.
__global__ void __launch_bounds__(kSuffixThreads) bwd_suffix_part_kernel(const float* __restrict__ dc,
                                                                         double* __restrict__ sfx,
                                                                         double* __restrict__ ptot, int T) {
  __shared__ float sbuf[kSuffixThreads * (kSuffixRun + 1)];
  __shared__ double wtot[kSuffixThreads / 32];
  const int part = blockIdx.x, P = gridDim.x;
  const size_t bh = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  constexpr int kWarps = kSuffixThreads / 32;
  const int start = part * kSuffixPart, n = min(kSuffixPart, T - start);
  for (int x = tid; x < kSuffixPart; x += kSuffixThreads)
    sbuf[(x / kSuffixRun) * (kSuffixRun + 1) + x % kSuffixRun] = x < n ? dc[bh * T + start + x] : 0.f;
  __syncthreads();
  const float* run = sbuf + tid * (kSuffixRun + 1);
  double sum = 0.0;
#pragma unroll
  for (int u = 0; u < kSuffixRun; ++u) sum += (double)run[u];
  double sw = sum;  // the runs from this lane to the end of the warp
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const double y = __shfl_down_sync(0xffffffffu, sw, o);
    if (lane + o < 32) sw += y;
  }
  if (lane == 0) wtot[warp] = sw;
  __syncthreads();
  if (tid == 0) {  // the warps from each one to the end of the part
    double acc = 0.0;
    for (int w = kWarps - 1; w >= 0; --w) {
      acc += wtot[w];
      wtot[w] = acc;
    }
    ptot[bh * P + part] = acc;
  }
  __syncthreads();
  double acc = (warp + 1 < kWarps ? wtot[warp + 1] : 0.0) + (sw - sum);  // the part after this run
  const int t0 = start + tid * kSuffixRun;
#pragma unroll
  for (int u = kSuffixRun - 1; u >= 0; --u) {
    acc += (double)run[u];
    if (tid * kSuffixRun + u < n) sfx[bh * T + t0 + u] = acc;
  }
}

__global__ void __launch_bounds__(256) bwd_suffix_apply_kernel(const double* __restrict__ sfx,
                                                               const double* __restrict__ ptot,
                                                               float* __restrict__ dla, int T) {
  __shared__ double off_s;
  const int part = blockIdx.x, P = gridDim.x;
  const size_t bh = blockIdx.y;
  if (threadIdx.x == 0) {
    double o = 0.0;
    for (int q = P - 1; q > part; --q) o += ptot[bh * P + q];
    off_s = o;
  }
  __syncthreads();
  const double o = off_s;
  const int start = part * kSuffixPart, n = min(kSuffixPart, T - start);
  for (int x = threadIdx.x; x < n; x += 256) dla[bh * T + start + x] = (float)(sfx[bh * T + start + x] + o);
}

ll_status suffix_launch(const float* dc, double* sfx, double* ptot, float* dla, int BH, int T, cudaStream_t stream) {
  const int P = (T + kSuffixPart - 1) / kSuffixPart;
  bwd_suffix_part_kernel<<<dim3(P, BH), kSuffixThreads, 0, stream>>>(dc, sfx, ptot, T);
  LL_CUDA_OK(cudaGetLastError());
  bwd_suffix_apply_kernel<<<dim3(P, BH), 256, 0, stream>>>(sfx, ptot, dla, T);
  LL_CUDA_OK(cudaGetLastError());
  return LL_OK;
}

// ------------------------------------------------ d_k = d_v = 128, 64-token chunks
// The same five steps with register tiles: every product is an outer-product
// loop over shared-memory tiles in which a thread keeps a 4 x 8 (or 8 x 8)
// block of the result in registers and reads one or two 128-bit words of each
// operand per step, instead of one output per thread with two loads per FMA.
namespace fast {

constexpr int kC = 64, kD = 128;
constexpr int kP = kD + 4;   // pitch of [rows][128] tiles: rows 16-byte aligned, 4 banks apart
constexpr int kPc = kC + 4;  // pitch of [rows][64] tiles

// 4 consecutive io elements as floats (16-byte aligned float rows, 8-byte bf16)
__device__ __forceinline__ float4 load4(const float* p) { return *reinterpret_cast<const float4*>(p); }
__device__ __forceinline__ float4 load4(const __nv_bfloat16* p) {
  const uint2 u = *reinterpret_cast<const uint2*>(p);
  const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
  const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
  return make_float4(a.x, a.y, b.x, b.y);
}
__device__ __forceinline__ void store4(float* p, float4 v) { *reinterpret_cast<float4*>(p) = v; }
__device__ __forceinline__ void store4(__nv_bfloat16* p, float4 v) {
  __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y), b = __floats2bfloat162_rn(v.z, v.w);
  uint2 u;
  u.x = *reinterpret_cast<unsigned*>(&a);
  u.y = *reinterpret_cast<unsigned*>(&b);
  *reinterpret_cast<uint2*>(p) = u;
}

// rows [0, nv) of a [64][128] io tile into shared [64][kP] floats; rows >= nv are 0
template <typename IO>
__device__ __forceinline__ void load_tile(float* dst, const IO* src, int nv, int tid) {
#pragma unroll 4
  for (int x = tid; x < kC * kD / 4; x += 256) {
    const int r = x >> 5, c4 = (x & 31) * 4;
    const float4 v = r < nv ? load4(src + (size_t)r * kD + c4) : make_float4(0.f, 0.f, 0.f, 0.f);
    store4(dst + r * kP + c4, v);
  }
}

// C[m][n] += sum_k At[k][m] B[k][n] for m = 4ty + i (64 rows), n = 4tx + j and
// 64 + 4tx + j (128 columns); optional per-k scale of At
template <bool kScale>
__device__ __forceinline__ void tn64x128(float (&c)[4][8], const float* At, int lda, const float* B, int K,
                                         const float* scale, int ty, int tx) {
#pragma unroll 4
  for (int k = 0; k < K; ++k) {
    float4 a = load4(At + k * lda + 4 * ty);
    if (kScale) {
      const float s = scale[k];
      a.x *= s; a.y *= s; a.z *= s; a.w *= s;
    }
    const float4 b0 = load4(B + k * kP + 4 * tx), b1 = load4(B + k * kP + 64 + 4 * tx);
    const float av[4] = {a.x, a.y, a.z, a.w};
    const float bv[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 8; ++j) c[i][j] = fmaf(av[i], bv[j], c[i][j]);
  }
}

// C[m][n] += sum_k s_k A[k][m] B[k][n] for m, n in {4t + i, 64 + 4t + i}: 128 x 128, TN
template <bool kScale>
__device__ __forceinline__ void tn128x128(float (&c)[8][8], const float* A, const float* B, int K,
                                          const float* scale, int ty, int tx) {
#pragma unroll 2
  for (int k = 0; k < K; ++k) {
    float4 a0 = load4(A + k * kP + 4 * ty), a1 = load4(A + k * kP + 64 + 4 * ty);
    if (kScale) {
      const float s = scale[k];
      a0.x *= s; a0.y *= s; a0.z *= s; a0.w *= s;
      a1.x *= s; a1.y *= s; a1.z *= s; a1.w *= s;
    }
    const float4 b0 = load4(B + k * kP + 4 * tx), b1 = load4(B + k * kP + 64 + 4 * tx);
    const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
    const float bv[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int j = 0; j < 8; ++j) c[i][j] = fmaf(av[i], bv[j], c[i][j]);
  }
}

// C[m][n] += sum_k A[m][k] B[n][k] (both k-contiguous, K = 128) for
// m = ty + 16 r (R rows), n = tx + 16 s (S columns)
template <int R, int S>
__device__ __forceinline__ void nt(float (&c)[R][S], const float* A, const float* B, int ty, int tx) {
#pragma unroll 2
  for (int k = 0; k < kD; k += 4) {
    float4 a[R], b[S];
#pragma unroll
    for (int r = 0; r < R; ++r) a[r] = load4(A + (ty + 16 * r) * kP + k);
#pragma unroll
    for (int s = 0; s < S; ++s) b[s] = load4(B + (tx + 16 * s) * kP + k);
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
      for (int s = 0; s < S; ++s) {
        c[r][s] = fmaf(a[r].x, b[s].x, c[r][s]);
        c[r][s] = fmaf(a[r].y, b[s].y, c[r][s]);
        c[r][s] = fmaf(a[r].z, b[s].z, c[r][s]);
        c[r][s] = fmaf(a[r].w, b[s].w, c[r][s]);
      }
  }
}

// rows 4ty + i of a 64 x 128 register tile to a float32 [.][128] array (rows < nv)
__device__ __forceinline__ void store_rows(float* dst, const float (&c)[4][8], int nv, int ty, int tx) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int m = 4 * ty + i;
    if (m < nv) {
      store4(dst + (size_t)m * kD + 4 * tx, make_float4(c[i][0], c[i][1], c[i][2], c[i][3]));
      store4(dst + (size_t)m * kD + 64 + 4 * tx, make_float4(c[i][4], c[i][5], c[i][6], c[i][7]));
    }
  }
}

constexpr size_t intra_smem() { return sizeof(float) * (4 * kC * kP + 4 * kC * kPc + kC) + sizeof(double) * kC; }
constexpr size_t query_smem() {
  return sizeof(float) * (2 * kC * kP + kD * kPc + kD * kP + 2 * kC) + sizeof(double) * kC;
}
constexpr size_t key_smem() { return sizeof(float) * (kC * kP + kD * kPc + kD * kP + kC) + sizeof(double) * kC; }

// (1) one CTA per (chunk, head)
template <typename IO>
__global__ void __launch_bounds__(256, 1) bwd_intra128_kernel(
    const IO* __restrict__ q, const IO* __restrict__ k, const IO* __restrict__ v, const IO* __restrict__ dout,
    const float* __restrict__ log_alpha, const float* __restrict__ lam, float* __restrict__ dq32,
    float* __restrict__ dk32, float* __restrict__ dv32, float* __restrict__ dlam, float* __restrict__ S,
    double* __restrict__ tot, float* __restrict__ R, int T, int L) {
  extern __shared__ __align__(16) float sm[];
  float* qs = sm;                 // [64][kP]
  float* ks = qs + kC * kP;
  float* vs = ks + kC * kP;
  float* gs = vs + kC * kP;       // dO
  float* P = gs + kC * kP;        // [64][kPc] A . M
  float* dA = P + kC * kPc;       // [64][kPc] dP . M
  float* dAt = dA + kC * kPc;     // its transpose
  float* X = dAt + kC * kPc;      // dP . A . Gamma
  float* wdec = X + kC * kPc;     // [64]
  double* cs = reinterpret_cast<double*>(wdec + kC);
  const int c = blockIdx.x, N = gridDim.x;
  const size_t bh = blockIdx.y;
  const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;
  const size_t row0 = bh * T + (size_t)c * kC;
  const int nv = min(kC, T - c * kC);
  chunk_scan(cs, log_alpha, row0, nv, kC);
  if (tid == kC - 1) tot[bh * N + c] = cs[kC - 1];
  load_tile(qs, q + row0 * kD, nv, tid);
  load_tile(ks, k + row0 * kD, nv, tid);
  load_tile(vs, v + row0 * kD, nv, tid);
  load_tile(gs, dout + row0 * kD, nv, tid);
  __syncthreads();
  if (tid < kC) wdec[tid] = expf((float)(cs[kC - 1] - cs[tid]));
  {
    float a[4][4] = {}, g[4][4] = {};
    nt<4, 4>(a, qs, ks, ty, tx);
    nt<4, 4>(g, gs, vs, ty, tx);
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int i = ty + 16 * r;
#pragma unroll
      for (int s = 0; s < 4; ++s) {
        const int j = tx + 16 * s;
        float p = 0.f, da = 0.f, xx = 0.f;
        if (j <= i && i < nv) {
          const float ex = expf((float)(cs[i] - cs[j]));
          const float lm = lam[(row0 + i) * L + bitlen((unsigned)(i ^ j))];
          p = a[r][s] * ex * lm;
          da = g[r][s] * ex * lm;
          xx = g[r][s] * a[r][s] * ex;
        }
        P[i * kPc + j] = p;
        dA[i * kPc + j] = da;
        dAt[j * kPc + i] = da;
        X[i * kPc + j] = xx;
      }
    }
  }
  __syncthreads();
  {
    float cq[4][8] = {};
    tn64x128<false>(cq, dAt, kPc, ks, kC, nullptr, ty, tx);  // dq = dA K
    store_rows(dq32 + row0 * kD, cq, nv, ty, tx);
  }
  {
    float ck[4][8] = {};
    tn64x128<false>(ck, dA, kPc, qs, kC, nullptr, ty, tx);  // dk = dA^T Q
    store_rows(dk32 + row0 * kD, ck, nv, ty, tx);
  }
  {
    float cv[4][8] = {};
    tn64x128<false>(cv, P, kPc, gs, kC, nullptr, ty, tx);  // dv = P^T dO
    store_rows(dv32 + row0 * kD, cv, nv, ty, tx);
  }
  // levels 0..6 of dlam (level l >= 1: the lower half of the aligned block of 2^l rows)
  const int nl = min(7, L);
  for (int x = tid; x < nv * nl; x += 256) {
    const int i = x / nl, l = x % nl;
    float acc = 0.f;
    if (l == 0) {
      acc = X[i * kPc + i];
    } else if ((i >> (l - 1)) & 1) {
      const int lo = (i >> l) << l;
      for (int j = lo; j < lo + (1 << (l - 1)); ++j) acc += X[i * kPc + j];
    }
    dlam[(row0 + i) * L + l] = acc;
  }
  {  // chunk state S_c = (wdec V)^T K; the key-side node of c starts at 0
    float cs8[8][8] = {};
    tn128x128<true>(cs8, vs, ks, kC, wdec, ty, tx);
    float* Sc = S + (bh * N + c) * (size_t)(kD * kD);
    float* Rc = R + (bh * N + c) * (size_t)(kD * kD);
    const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int e = (i < 4 ? 0 : 64) + 4 * ty + (i & 3);
      store4(Sc + e * kD + 4 * tx, make_float4(cs8[i][0], cs8[i][1], cs8[i][2], cs8[i][3]));
      store4(Sc + e * kD + 64 + 4 * tx, make_float4(cs8[i][4], cs8[i][5], cs8[i][6], cs8[i][7]));
      store4(Rc + e * kD + 4 * tx, z);
      store4(Rc + e * kD + 64 + 4 * tx, z);
    }
  }
}

// (3) one CTA per (chunk, head)
template <typename IO>
__global__ void __launch_bounds__(256, 1) bwd_query128_kernel(
    const IO* __restrict__ q, const IO* __restrict__ dout, const float* __restrict__ log_alpha,
    const float* __restrict__ lam, const float* __restrict__ F, const double* __restrict__ G, const float* dq32,
    IO* dq, float* __restrict__ dlam, float* __restrict__ R, int T, int L) {
  extern __shared__ __align__(16) float sm[];
  float* qs = sm;              // [64][kP]
  float* gs = qs + kC * kP;    // [64][kP] dO
  float* gT = gs + kC * kP;    // [128][kPc] dO transposed
  float* Fs = gT + kD * kPc;   // [128][kP]
  float* w = Fs + kD * kP;     // [64] exp(cs_i + D)
  float* lw = w + kC;          // [64] lam_i[level] exp(cs_i + D)
  double* cs = reinterpret_cast<double*>(lw + kC);
  const int c = blockIdx.x, N = gridDim.x;
  const size_t bh = blockIdx.y;
  const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;
  const size_t row0 = bh * T + (size_t)c * kC;
  const int nv = min(kC, T - c * kC);
  constexpr int lc = 6;
  chunk_scan(cs, log_alpha, row0, nv, kC);
  load_tile(qs, q + row0 * kD, nv, tid);
  load_tile(gs, dout + row0 * kD, nv, tid);
  __syncthreads();
  // transpose dO: a warp takes 32 consecutive rows of one 4-column group
  for (int x = tid; x < kC * kD / 4; x += 256) {
    const int i = x & 63, e4 = (x >> 6) * 4;
    const float4 t = load4(gs + i * kP + e4);
    gT[(e4 + 0) * kPc + i] = t.x;
    gT[(e4 + 1) * kPc + i] = t.y;
    gT[(e4 + 2) * kPc + i] = t.z;
    gT[(e4 + 3) * kPc + i] = t.w;
  }
  float acc[4][8] = {};
  const size_t mat = (size_t)kD * kD;
  double D = 0.0;
  for (int h = 0; (c >> h) != 0; ++h) {
    if (!((c >> h) & 1)) continue;
    const int e = ((c >> (h + 1)) << (h + 1)) + (1 << h) - 1;
    const int lv = lc + 1 + h;
    const float* Fe = F + (bh * N + e) * mat;
    for (int x = tid; x < kD * kD / 4; x += 256) {
      const int r = x >> 5, c4 = (x & 31) * 4;
      store4(Fs + r * kP + c4, load4(Fe + r * kD + c4));
    }
    if (tid < kC) {
      const float wi = tid < nv ? expf((float)(cs[tid] + D)) : 0.f;
      w[tid] = wi;
      lw[tid] = tid < nv ? wi * lam[(row0 + tid) * L + lv] : 0.f;
    }
    __syncthreads();
    {  // g_i = F^T do_i (unscaled): dq_i += lw_i g_i, dlam_i = w_i g_i . q_i
      float cg[4][8] = {};
      tn64x128<false>(cg, gT, kPc, Fs, kD, nullptr, ty, tx);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int m = 4 * ty + i;
        const float lwm = lw[m];
        float part = 0.f;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int n = (j < 4 ? 0 : 64) + 4 * tx + (j & 3);
          acc[i][j] = fmaf(lwm, cg[i][j], acc[i][j]);
          part = fmaf(cg[i][j], qs[m * kP + n], part);
        }
#pragma unroll
        for (int o = 8; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
        if (tx == 0 && m < nv) dlam[(row0 + m) * L + lv] = w[m] * part;
      }
    }
    {  // R_e += sum_i lw_i do_i q_i^T
      float cr[8][8] = {};
      tn128x128<true>(cr, gs, qs, kC, lw, ty, tx);
      float* Re = R + (bh * N + e) * mat;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int ev = (i < 4 ? 0 : 64) + 4 * ty + (i & 3);
        atomicAdd(reinterpret_cast<float4*>(Re + ev * kD + 4 * tx),
                  make_float4(cr[i][0], cr[i][1], cr[i][2], cr[i][3]));
        atomicAdd(reinterpret_cast<float4*>(Re + ev * kD + 64 + 4 * tx),
                  make_float4(cr[i][4], cr[i][5], cr[i][6], cr[i][7]));
      }
    }
    D += G[bh * N + e];
    __syncthreads();
  }
  // the levels above 6 that hold no key of this chunk's queries
  const int nh = L - (lc + 1);
  for (int x = tid; x < nv * max(nh, 0); x += 256) {
    const int i = x / nh, hh = x % nh;
    if (!(hh < 31 && ((c >> hh) & 1))) dlam[(row0 + i) * L + lc + 1 + hh] = 0.f;
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int m = 4 * ty + i;
    if (m < nv) {
      const size_t o = (row0 + m) * kD;
      const float4 p0 = load4(dq32 + o + 4 * tx), p1 = load4(dq32 + o + 64 + 4 * tx);
      store4(dq + o + 4 * tx, make_float4(p0.x + acc[i][0], p0.y + acc[i][1], p0.z + acc[i][2], p0.w + acc[i][3]));
      store4(dq + o + 64 + 4 * tx,
             make_float4(p1.x + acc[i][4], p1.y + acc[i][5], p1.z + acc[i][6], p1.w + acc[i][7]));
    }
  }
}

// (4) one CTA per (chunk, head)
template <typename IO>
__global__ void __launch_bounds__(256, 1) bwd_key128_kernel(
    const IO* __restrict__ k, const IO* __restrict__ v, const float* __restrict__ log_alpha,
    const float* __restrict__ lam, const float* __restrict__ dlam, const float* __restrict__ R,
    const double* __restrict__ cum, const float* dk32, const float* dv32, IO* dk, IO* dv, float* __restrict__ dc,
    int T, int L) {
  extern __shared__ __align__(16) float sm[];
  __shared__ float coef[32];
  __shared__ int ent[32];
  __shared__ int n_sh;
  __shared__ float dcrow[kC];
  float* ks = sm;              // [64][kP]
  float* vT = ks + kC * kP;    // [128][kPc] V transposed
  float* Es = vT + kD * kPc;   // [128][kP]; first the staging of V
  float* wdec = Es + kD * kP;  // [64]
  double* cs = reinterpret_cast<double*>(wdec + kC);
  const int c = blockIdx.x, N = gridDim.x;
  const size_t bh = blockIdx.y;
  const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;
  const size_t row0 = bh * T + (size_t)c * kC;
  const int nv = min(kC, T - c * kC);
  if (tid == 0) {
    int n = 0;
    for (int h = 0; h < 31 && n < 32; ++h) {
      if ((c >> h) & 1) continue;
      const int e = ((c >> (h + 1)) << (h + 1)) + (1 << h) - 1;
      if (e + 1 >= N) break;  // e grows with h: no later node has queries either
      ent[n] = e;
      coef[n] = expf((float)(cum[bh * N + e] - cum[bh * N + c]));  // the decay from the end of c to the end of e
      ++n;
    }
    n_sh = n;
  }
  chunk_scan(cs, log_alpha, row0, nv, kC);
  load_tile(ks, k + row0 * kD, nv, tid);
  load_tile(Es, v + row0 * kD, nv, tid);
  __syncthreads();
  for (int x = tid; x < kC * kD / 4; x += 256) {
    const int j = x & 63, e4 = (x >> 6) * 4;
    const float4 t = load4(Es + j * kP + e4);
    vT[(e4 + 0) * kPc + j] = t.x;
    vT[(e4 + 1) * kPc + j] = t.y;
    vT[(e4 + 2) * kPc + j] = t.z;
    vT[(e4 + 3) * kPc + j] = t.w;
  }
  if (tid < kC) wdec[tid] = expf((float)(cs[kC - 1] - cs[tid]));
  const int n = n_sh;
  __syncthreads();
  const size_t mat = (size_t)kD * kD;
  if (n > 0) {
    for (int x = tid; x < kD * kD / 4; x += 256) {
      const int r = x >> 5, c4 = (x & 31) * 4;
      float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int m = 0; m < n; ++m) {
        const float4 t = load4(R + (bh * N + ent[m]) * mat + r * kD + c4);
        const float cf = coef[m];
        a.x = fmaf(cf, t.x, a.x); a.y = fmaf(cf, t.y, a.y); a.z = fmaf(cf, t.z, a.z); a.w = fmaf(cf, t.w, a.w);
      }
      store4(Es + r * kP + c4, a);
    }
    __syncthreads();
  }
  {  // dv_j = dv32_j + wdec_j E k_j (rows j = ty + 16 r, columns e = tx + 16 s), and v_j . dv_j
    float cv[4][8] = {};
    if (n > 0) nt<4, 8>(cv, ks, Es, ty, tx);
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int j = ty + 16 * r;
      float vdv = 0.f;
#pragma unroll
      for (int s = 0; s < 8; ++s) {
        const int e = tx + 16 * s;
        if (j < nv) {
          const size_t o = (row0 + j) * kD + e;
          const float val = fmaf(wdec[j], cv[r][s], dv32[o]);
          dv[o] = from_f<IO>(val);
          vdv = fmaf(vT[e * kPc + j], val, vdv);
        }
      }
#pragma unroll
      for (int o = 8; o > 0; o >>= 1) vdv += __shfl_xor_sync(0xffffffffu, vdv, o);
      if (tx == 0) dcrow[j] = -vdv;
    }
  }
  {  // dk_j = dk32_j + wdec_j E^T v_j
    float ck[4][8] = {};
    if (n > 0) tn64x128<false>(ck, vT, kPc, Es, kD, nullptr, ty, tx);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int m = 4 * ty + i;
      if (m < nv) {
        const size_t o = (row0 + m) * kD;
        const float wm = wdec[m];
        const float4 p0 = load4(dk32 + o + 4 * tx), p1 = load4(dk32 + o + 64 + 4 * tx);
        store4(dk + o + 4 * tx, make_float4(fmaf(wm, ck[i][0], p0.x), fmaf(wm, ck[i][1], p0.y),
                                            fmaf(wm, ck[i][2], p0.z), fmaf(wm, ck[i][3], p0.w)));
        store4(dk + o + 64 + 4 * tx, make_float4(fmaf(wm, ck[i][4], p1.x), fmaf(wm, ck[i][5], p1.y),
                                                 fmaf(wm, ck[i][6], p1.z), fmaf(wm, ck[i][7], p1.w)));
      }
    }
  }
  __syncthreads();
  // dc_j = sum_l lam_j[l] dlam_j[l] - v_j . dv_j, one warp per row
  const int warp = tid >> 5, lane = tid & 31;
  for (int j = warp; j < kC; j += 8) {
    float a = 0.f;
    if (j < nv)
      for (int l = lane; l < L; l += 32) a = fmaf(lam[(row0 + j) * L + l], dlam[(row0 + j) * L + l], a);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) a += __shfl_xor_sync(0xffffffffu, a, o);
    if (lane == 0) {
      a += dcrow[j];
      if (j < nv) dc[row0 + j] = a;
      dcrow[j] = a;
    }
  }
}

}  // namespace fast

// d_k = d_v = 128 with 64-token chunks runs on the register-tiled kernels
bool fast_shape(const ll_shape& s, const BwdPlan& p) { return s.dk == 128 && s.dv == 128 && p.Ce == 64; }

template <typename IO>
ll_status launch_typed(const BwdArgs& a, const BwdPlan& p) {
  const ll_shape& s = a.s;
  unsigned char* ws = static_cast<unsigned char*>(a.ws);
  float* S = reinterpret_cast<float*>(ws + p.off_S);
  float* F = reinterpret_cast<float*>(ws + p.off_F);
  float* R = reinterpret_cast<float*>(ws + p.off_R);
  double* tot = reinterpret_cast<double*>(ws + p.off_tot);
  double* G = reinterpret_cast<double*>(ws + p.off_G);
  double* cum = reinterpret_cast<double*>(ws + p.off_cum);
  float* dc = reinterpret_cast<float*>(ws + p.off_dc);
  double* sfx = reinterpret_cast<double*>(ws + p.off_sfx);
  double* ptot = reinterpret_cast<double*>(ws + p.off_ptot);
  const bool f32 = s.io == LL_F32;
  float* dq32 = f32 ? static_cast<float*>(a.dq) : reinterpret_cast<float*>(ws + p.off_dq);
  float* dk32 = f32 ? static_cast<float*>(a.dk) : reinterpret_cast<float*>(ws + p.off_dk);
  float* dv32 = f32 ? static_cast<float*>(a.dv) : reinterpret_cast<float*>(ws + p.off_dv);
  const int BH = s.B * s.H;
  const int Ce = p.Ce;
  const int mat = s.dv * s.dk;
  const dim3 grid(p.N, BH);
  const IO* q = static_cast<const IO*>(a.q);
  const IO* k = static_cast<const IO*>(a.k);
  const IO* v = static_cast<const IO*>(a.v);
  const IO* dout = static_cast<const IO*>(a.dout);

  if (bwd_tc_supported(s)) {
    const BwdTcBuffers b{reinterpret_cast<__nv_bfloat16*>(dq32), reinterpret_cast<__nv_bfloat16*>(dk32),
                         reinterpret_cast<__nv_bfloat16*>(dv32), S, F, R, reinterpret_cast<__nv_bfloat16*>(ws + p.off_Ft), tot, G,
                         cum, dc, a.err};
    const ll_status st = bwd_tc_launch(a, b);
    if (st != LL_OK) return st;
    return suffix_launch(dc, sfx, ptot, a.dlog_alpha, BH, s.T, a.stream);
  }
  if (fast_shape(s, p)) {
    LL_CUDA_OK(cudaFuncSetAttribute(fast::bwd_intra128_kernel<IO>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)fast::intra_smem()));
    fast::bwd_intra128_kernel<IO><<<grid, 256, fast::intra_smem(), a.stream>>>(
        q, k, v, dout, a.log_alpha, a.lam, dq32, dk32, dv32, a.dlam, S, tot, R, s.T, s.L);
    LL_CUDA_OK(cudaGetLastError());
    const ll_status fs = simt_fenwick_launch(S, F, tot, G, p.N, mat, BH, a.stream, nullptr, cum);
    if (fs != LL_OK) return fs;
    LL_CUDA_OK(cudaFuncSetAttribute(fast::bwd_query128_kernel<IO>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)fast::query_smem()));
    fast::bwd_query128_kernel<IO><<<grid, 256, fast::query_smem(), a.stream>>>(
        q, dout, a.log_alpha, a.lam, F, G, dq32, static_cast<IO*>(a.dq), a.dlam, R, s.T, s.L);
    LL_CUDA_OK(cudaGetLastError());
    LL_CUDA_OK(cudaFuncSetAttribute(fast::bwd_key128_kernel<IO>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)fast::key_smem()));
    fast::bwd_key128_kernel<IO><<<grid, 256, fast::key_smem(), a.stream>>>(
        k, v, a.log_alpha, a.lam, a.dlam, R, cum, dk32, dv32, static_cast<IO*>(a.dk), static_cast<IO*>(a.dv), dc,
        s.T, s.L);
    LL_CUDA_OK(cudaGetLastError());
    return suffix_launch(dc, sfx, ptot, a.dlog_alpha, BH, s.T, a.stream);
  }

  const size_t sm1 = intra_smem(Ce, s.dk, s.dv);
  LL_CUDA_OK(cudaFuncSetAttribute(bwd_intra_kernel<IO>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm1));
  bwd_intra_kernel<IO><<<grid, kThreads, sm1, a.stream>>>(
      static_cast<const IO*>(a.q), static_cast<const IO*>(a.k), static_cast<const IO*>(a.v),
      static_cast<const IO*>(a.dout), a.log_alpha, a.lam, dq32, dk32, dv32, a.dlam, S, tot, R, s.T, s.dk, s.dv, s.L,
      Ce, p.lc);
  LL_CUDA_OK(cudaGetLastError());

  const ll_status fs = simt_fenwick_launch(S, F, tot, G, p.N, mat, BH, a.stream, nullptr, cum);
  if (fs != LL_OK) return fs;

  const size_t sm3 = query_smem(Ce, s.dk, s.dv);
  LL_CUDA_OK(cudaFuncSetAttribute(bwd_query_kernel<IO>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm3));
  bwd_query_kernel<IO><<<grid, kThreads, sm3, a.stream>>>(
      static_cast<const IO*>(a.q), static_cast<const IO*>(a.dout), a.log_alpha, a.lam, F, G, dq32,
      static_cast<IO*>(a.dq), a.dlam, R, s.T, s.dk, s.dv, s.L, Ce, p.lc);
  LL_CUDA_OK(cudaGetLastError());

  const size_t sm4 = key_smem(Ce, s.dk, s.dv);
  LL_CUDA_OK(cudaFuncSetAttribute(bwd_key_kernel<IO>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm4));
  bwd_key_kernel<IO><<<grid, kThreads, sm4, a.stream>>>(
      static_cast<const IO*>(a.k), static_cast<const IO*>(a.v), a.log_alpha, a.lam, a.dlam, R, cum, dk32, dv32,
      static_cast<IO*>(a.dk), static_cast<IO*>(a.dv), dc, s.T, s.dk, s.dv, s.L, Ce);
  LL_CUDA_OK(cudaGetLastError());

  return suffix_launch(dc, sfx, ptot, a.dlog_alpha, BH, s.T, a.stream);
}

}  // namespace

size_t bwd_simt_workspace(const ll_shape& s) { return plan_of(s).total; }

int bwd_simt_launches(const ll_shape&) { return 6; }

ll_status bwd_simt_launch(const BwdArgs& a) {
  const BwdPlan p = plan_of(a.s);
  if (a.ws_bytes < p.total) return LL_ERR_WORKSPACE;
  if ((size_t)p.N * sizeof(double) > 200 * 1024) return LL_ERR_UNSUPPORTED;  // the Fenwick kernel's prefix table
  if ((long long)a.s.B * a.s.H > 65535) return LL_ERR_UNSUPPORTED;            // heads on the grid's y axis
  if (a.s.io == LL_F32) return launch_typed<float>(a, p);
  return launch_typed<__nv_bfloat16>(a, p);
}

}  // namespace llattn
