// Log-Linear Gated DeltaNet forward, reading A (float32 FMA on CUDA cores).
//
// The pages ("Log-Linear Attention" study note §3-5; gist.science (de)
// Technische Zusammenfassung §2) only say that the hierarchical mask is
// combined with the delta rule.  Reading A: every Fenwick level state follows
// the gated delta transition S <- alpha_t S (I - beta_t k_t k_t^T), the write
// beta_t v_t k_t^T enters level 0, merges are additions; equivalently
// O = (C . M^H) V with C the gated-delta-rule coefficient matrix.
//
// Chunk c (Ce tokens; g = inclusive cumsum of log_alpha inside the chunk,
// G_ij = exp(g_i - g_j) for j <= i, e = exp(g)):
//   UT transform  Tinv = (I + diag(beta) SL(K K^T . G))^{-1}      (unit lower)
//                 U = Tinv diag(beta) V,   W = Tinv diag(beta e) K
//   intra         Aqk = (Q K^T . G) incl. diagonal,
//                 Cl = Aqk Tinv diag(beta),   o_i += sum_{j<=i} Cl_ij lam_i[bitlen(i^j)] v_j
//   transport     a level state X (dv x dk) at the chunk start contributes
//                 o_i += lam_i[level] (X q'_i) with Q' = diag(e) Q - Aqk W, and
//                 leaves the chunk as X (gamma I - W^T Kt), Kt = diag(exp(g_end - g)) K,
//                 gamma = exp(g_end)
//   local state   S_c = U^T Kt (the chunk's own tokens at the chunk end)
//   carry         after chunk c the levels of heights h < cto(c) and S_c add
//                 into height cto(c) (level log2(Ce) + 1 + h for height h).
// Kernel 1 does everything per chunk in parallel; kernel 2 scans the chunks
// of each head in order, each CTA owning a slice of the d_v rows of every
// level state (rows transform independently).
#include <algorithm>

#include "common.cuh"

namespace llattn {

namespace {

constexpr int kThreads = 256;
constexpr int kRows = 16;         // d_v rows of the level states per scan CTA
constexpr int kMaxHeights = 12;   // chunk counts up to 4096
constexpr size_t kSmemLimit = 227 * 1024;

size_t prep_smem_floats(int Ce, int dk, int dv) {
  return (size_t)2 * Ce * (dk + 1) + (size_t)Ce * (dv + 1) + (size_t)3 * Ce * (Ce + 1) + (size_t)Ce * dv +
         (size_t)Ce * dk + 4 * (size_t)Ce;
}

int heights_of(int N) {
  int h = 0;
  while ((1 << h) <= N) ++h;  // bit_length(N): heights 0..h-1 can be live
  return std::max(h, 1);
}

size_t scan_smem_floats(int Ce, int dk, int nh) {
  return (size_t)nh * kRows * dk + (size_t)2 * Ce * (dk + 1) + (size_t)Ce * dk + (size_t)2 * kRows * Ce +
         (size_t)Ce * kRows + (size_t)Ce * nh + (size_t)kRows * dk;
}

struct GdnPlan {
  int Ce, N, lc, nh;
  size_t off_Qp, off_W, off_Kt, off_S, off_lg, off_O, total;
  bool ok;
};

GdnPlan gdn_plan(const ll_shape& s) {
  GdnPlan p{};
  p.Ce = std::min(s.chunk, 64);
  while (p.Ce > 16 && prep_smem_floats(p.Ce, s.dk, s.dv) * 4 > kSmemLimit) p.Ce >>= 1;
  p.N = s.T / p.Ce;
  p.lc = ilog2(p.Ce);
  p.nh = heights_of(p.N);
  p.ok = prep_smem_floats(p.Ce, s.dk, s.dv) * 4 <= kSmemLimit && p.nh <= kMaxHeights &&
         scan_smem_floats(p.Ce, s.dk, p.nh) * 4 <= kSmemLimit && s.dv % kRows == 0;
  const size_t BH = (size_t)s.B * s.H;
  size_t off = 0;
  p.off_Qp = off; off = align_up(off + BH * s.T * (size_t)s.dk * 4, 256);
  p.off_W = off;  off = align_up(off + BH * s.T * (size_t)s.dk * 4, 256);
  p.off_Kt = off; off = align_up(off + BH * s.T * (size_t)s.dk * 4, 256);
  p.off_S = off;  off = align_up(off + BH * p.N * (size_t)s.dv * s.dk * 4, 256);
  p.off_lg = off; off = align_up(off + BH * p.N * 4, 256);
  p.off_O = off;  off = align_up(off + BH * s.T * (size_t)s.dv * 4, 256);
  p.total = off;
  return p;
}

// ---------------------------------------------------------------- kernel 1
template <typename IO>
__global__ void __launch_bounds__(kThreads) gdn_prep_kernel(const IO* __restrict__ q, const IO* __restrict__ k,
                                                            const IO* __restrict__ v,
                                                            const float* __restrict__ log_alpha,
                                                            const float* __restrict__ beta,
                                                            const float* __restrict__ lam, float* __restrict__ Qp,
                                                            float* __restrict__ Wg, float* __restrict__ Kt,
                                                            float* __restrict__ Sloc, float* __restrict__ loggam,
                                                            float* __restrict__ Oacc, int T, int dk, int dv, int L,
                                                            int Ce) {
  extern __shared__ __align__(16) float sm[];
  const int c = blockIdx.x, N = gridDim.x;
  const size_t bh = blockIdx.y;
  const int tid = threadIdx.x;
  const int dkp = dk + 1, dvp = dv + 1, Cp = Ce + 1;
  float* qs = sm;
  float* ks = qs + Ce * dkp;
  float* vs = ks + Ce * dkp;
  float* Lm = vs + Ce * dvp;     // beta_i (k_i.k_j) G_ij, strictly lower; later Cl
  float* Ti = Lm + Ce * Cp;      // Tinv
  float* Aq = Ti + Ce * Cp;      // Aqk
  float* Us = Aq + Ce * Cp;      // U  [Ce][dv]
  float* Ws = Us + Ce * dv;      // W  [Ce][dk]
  float* gs = Ws + Ce * dk;      // g
  float* bs = gs + Ce;           // beta
  float* es = bs + Ce;           // exp(g)
  float* ds = es + Ce;           // exp(g_end - g)

  const size_t row0 = bh * T + (size_t)c * Ce;
  if (tid == 0) {
    double acc = 0.0;
    for (int i = 0; i < Ce; ++i) {
      acc += (double)log_alpha[row0 + i];
      gs[i] = (float)acc;
    }
    loggam[bh * N + c] = (float)acc;
  }
  for (int x = tid; x < Ce * dk; x += kThreads) {
    const int i = x / dk, f = x % dk;
    qs[i * dkp + f] = to_f(q[(row0 + i) * dk + f]);
    ks[i * dkp + f] = to_f(k[(row0 + i) * dk + f]);
  }
  for (int x = tid; x < Ce * dv; x += kThreads) vs[(x / dv) * dvp + (x % dv)] = to_f(v[row0 * dv + x]);
  for (int i = tid; i < Ce; i += kThreads) bs[i] = beta[row0 + i];
  __syncthreads();
  for (int i = tid; i < Ce; i += kThreads) {
    es[i] = expf(gs[i]);
    ds[i] = expf(gs[Ce - 1] - gs[i]);
  }

  // L (strict lower, beta folded in) and Aqk (inclusive)
  for (int x = tid; x < Ce * Ce; x += kThreads) {
    const int i = x / Ce, j = x % Ce;
    float lk = 0.f, aq = 0.f;
    if (j <= i) {
      float dkk = 0.f, dqk = 0.f;
      for (int f = 0; f < dk; ++f) {
        const float kj = ks[j * dkp + f];
        dkk = fmaf(ks[i * dkp + f], kj, dkk);
        dqk = fmaf(qs[i * dkp + f], kj, dqk);
      }
      const float gij = expf(gs[i] - gs[j]);
      aq = dqk * gij;
      if (j < i) lk = bs[i] * dkk * gij;
    }
    Lm[i * Cp + j] = lk;
    Aq[i * Cp + j] = aq;
  }
  __syncthreads();

  // Tinv = (I + L)^{-1}: forward substitution, one column per thread
  for (int j = tid; j < Ce; j += kThreads) {
    for (int i = 0; i < Ce; ++i) {
      float x = (i == j) ? 1.f : 0.f;
      if (i > j) {
        for (int m = j; m < i; ++m) x = fmaf(-Lm[i * Cp + m], Ti[m * Cp + j], x);
      }
      Ti[i * Cp + j] = (i >= j) ? x : 0.f;
    }
  }
  __syncthreads();

  // U = Tinv diag(beta) V,  W = Tinv diag(beta e) K
  for (int x = tid; x < Ce * dv; x += kThreads) {
    const int i = x / dv, e = x % dv;
    float acc = 0.f;
    for (int j = 0; j <= i; ++j) acc = fmaf(Ti[i * Cp + j] * bs[j], vs[j * dvp + e], acc);
    Us[i * dv + e] = acc;
  }
  for (int x = tid; x < Ce * dk; x += kThreads) {
    const int i = x / dk, f = x % dk;
    float acc = 0.f;
    for (int j = 0; j <= i; ++j) acc = fmaf(Ti[i * Cp + j] * bs[j] * es[j], ks[j * dkp + f], acc);
    Ws[i * dk + f] = acc;
  }
  // Cl = Aqk Tinv diag(beta)  (into Lm)
  for (int x = tid; x < Ce * Ce; x += kThreads) {
    const int i = x / Ce, j = x % Ce;
    float acc = 0.f;
    if (j <= i) {
      for (int m = j; m <= i; ++m) acc = fmaf(Aq[i * Cp + m], Ti[m * Cp + j], acc);
      acc *= bs[j];
    }
    Lm[i * Cp + j] = acc;
  }
  __syncthreads();

  // intra output, masked by the within-chunk levels
  for (int x = tid; x < Ce * dv; x += kThreads) {
    const int i = x / dv, e = x % dv;
    const float* lrow = lam + (row0 + i) * L;
    float acc = 0.f;
    for (int j = 0; j <= i; ++j) acc = fmaf(Lm[i * Cp + j] * lrow[bitlen((unsigned)(i ^ j))], vs[j * dvp + e], acc);
    Oacc[(row0 + i) * dv + e] = acc;
  }
  // Q' = diag(e) Q - Aqk W,  Kt = diag(exp(g_end - g)) K,  W
  for (int x = tid; x < Ce * dk; x += kThreads) {
    const int i = x / dk, f = x % dk;
    float acc = es[i] * qs[i * dkp + f];
    for (int j = 0; j <= i; ++j) acc = fmaf(-Aq[i * Cp + j], Ws[j * dk + f], acc);
    Qp[(row0 + i) * dk + f] = acc;
    Kt[(row0 + i) * dk + f] = ds[i] * ks[i * dkp + f];
    Wg[(row0 + i) * dk + f] = Ws[i * dk + f];
  }
  // local chunk state S_c = U^T Kt
  float* Sc = Sloc + (bh * N + c) * (size_t)dv * dk;
  for (int x = tid; x < dv * dk; x += kThreads) {
    const int e = x / dk, f = x % dk;
    float acc = 0.f;
    for (int j = 0; j < Ce; ++j) acc = fmaf(Us[j * dv + e] * ds[j], ks[j * dkp + f], acc);
    Sc[x] = acc;
  }
}

// ---------------------------------------------------------------- kernel 2
template <typename IO>
__global__ void __launch_bounds__(kThreads) gdn_scan_kernel(const float* __restrict__ Qp, const float* __restrict__ Wg,
                                                            const float* __restrict__ Kt,
                                                            const float* __restrict__ Sloc,
                                                            const float* __restrict__ loggam,
                                                            const float* __restrict__ Oacc,
                                                            const float* __restrict__ lam, IO* __restrict__ o, int T,
                                                            int dk, int dv, int L, int Ce, int N, int lc, int nh) {
  extern __shared__ __align__(16) float sm[];
  const size_t bh = blockIdx.y;
  const int r0 = blockIdx.x * kRows;
  const int tid = threadIdx.x;
  const int dkp = dk + 1;
  float* X = sm;                         // [nh][kRows][dk] level states (rows r0..r0+kRows)
  float* Wsm = X + nh * kRows * dk;      // [Ce][dk+1]
  float* Qsm = Wsm + Ce * dkp;           // [Ce][dk+1]
  float* Ksm = Qsm + Ce * dkp;           // [Ce][dk]
  float* Y = Ksm + Ce * dk;              // [kRows][Ce]  X W^T
  float* Pq = Y + kRows * Ce;            // [kRows][Ce]  X Q'^T
  float* Oc = Pq + kRows * Ce;           // [Ce][kRows]
  float* lamc = Oc + Ce * kRows;         // [Ce][nh]
  float* Snew = lamc + Ce * nh;          // [kRows][dk]

  for (int c = 0; c < N; ++c) {
    const size_t row0 = bh * T + (size_t)c * Ce;
    const float gam = expf(loggam[bh * N + c]);
    for (int x = tid; x < Ce * dk; x += kThreads) {
      const int i = x / dk, f = x % dk;
      Wsm[i * dkp + f] = Wg[row0 * dk + x];
      Qsm[i * dkp + f] = Qp[row0 * dk + x];
      Ksm[x] = Kt[row0 * dk + x];
    }
    for (int x = tid; x < Ce * kRows; x += kThreads) Oc[x] = 0.f;
    for (int x = tid; x < Ce * nh; x += kThreads) {
      const int i = x / nh, h = x % nh;
      lamc[x] = (lc + 1 + h < L) ? lam[(row0 + i) * L + lc + 1 + h] : 0.f;
    }
    __syncthreads();

    for (int h = 0; h < nh; ++h) {
      if (!((c >> h) & 1)) continue;
      float* Xh = X + h * kRows * dk;
      // Y = X W^T and Pq = X Q'^T
      for (int x = tid; x < kRows * Ce; x += kThreads) {
        const int r = x / Ce, i = x % Ce;
        float y = 0.f, pq = 0.f;
        for (int f = 0; f < dk; ++f) {
          const float xv = Xh[r * dk + f];
          y = fmaf(xv, Wsm[i * dkp + f], y);
          pq = fmaf(xv, Qsm[i * dkp + f], pq);
        }
        Y[x] = y;
        Pq[x] = pq;
      }
      __syncthreads();
      for (int x = tid; x < Ce * kRows; x += kThreads) {
        const int i = x / kRows, r = x % kRows;
        Oc[x] = fmaf(lamc[i * nh + h], Pq[r * Ce + i], Oc[x]);
      }
      // X <- gamma X - Y Kt
      for (int x = tid; x < kRows * dk; x += kThreads) {
        const int r = x / dk, f = x % dk;
        float acc = gam * Xh[x];
        for (int i = 0; i < Ce; ++i) acc = fmaf(-Y[r * Ce + i], Ksm[i * dk + f], acc);
        Xh[x] = acc;
      }
      __syncthreads();
    }

    // output rows of this chunk for d_v rows r0..r0+kRows
    for (int x = tid; x < Ce * kRows; x += kThreads) {
      const int i = x / kRows, r = x % kRows;
      const size_t oi = (row0 + i) * dv + r0 + r;
      o[oi] = from_f<IO>(Oacc[oi] + Oc[x]);
    }
    // carry into height cto(c): S_c + the transported levels below it
    int jc = 0;
    while ((c >> jc) & 1) ++jc;
    if (jc < nh) {
      const float* Sc = Sloc + (bh * N + c) * (size_t)dv * dk + (size_t)r0 * dk;
      for (int x = tid; x < kRows * dk; x += kThreads) {
        float acc = Sc[x];
        for (int h = 0; h < jc; ++h) acc += X[h * kRows * dk + x];
        X[jc * kRows * dk + x] = acc;
      }
    }
    __syncthreads();
  }
}

template <typename IO>
ll_status launch_typed(const FwdArgs& a, const GdnPlan& p) {
  const ll_shape& s = a.s;
  unsigned char* ws = static_cast<unsigned char*>(a.ws);
  float* Qp = reinterpret_cast<float*>(ws + p.off_Qp);
  float* W = reinterpret_cast<float*>(ws + p.off_W);
  float* Kt = reinterpret_cast<float*>(ws + p.off_Kt);
  float* S = reinterpret_cast<float*>(ws + p.off_S);
  float* lg = reinterpret_cast<float*>(ws + p.off_lg);
  float* O = reinterpret_cast<float*>(ws + p.off_O);
  const int BH = s.B * s.H;
  const size_t sm1 = prep_smem_floats(p.Ce, s.dk, s.dv) * 4;
  LL_CUDA_OK(cudaFuncSetAttribute(gdn_prep_kernel<IO>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm1));
  gdn_prep_kernel<IO><<<dim3(p.N, BH), kThreads, sm1, a.stream>>>(
      static_cast<const IO*>(a.q), static_cast<const IO*>(a.k), static_cast<const IO*>(a.v), a.log_alpha, a.beta,
      a.lam, Qp, W, Kt, S, lg, O, s.T, s.dk, s.dv, s.L, p.Ce);
  LL_CUDA_OK(cudaGetLastError());
  const size_t sm2 = scan_smem_floats(p.Ce, s.dk, p.nh) * 4;
  LL_CUDA_OK(cudaFuncSetAttribute(gdn_scan_kernel<IO>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm2));
  gdn_scan_kernel<IO><<<dim3(s.dv / kRows, BH), kThreads, sm2, a.stream>>>(
      Qp, W, Kt, S, lg, O, a.lam, static_cast<IO*>(a.o), s.T, s.dk, s.dv, s.L, p.Ce, p.N, p.lc, p.nh);
  LL_CUDA_OK(cudaGetLastError());
  return LL_OK;
}

}  // namespace

size_t gdn_workspace(const ll_shape& s) {
  const GdnPlan p = gdn_plan(s);
  return p.ok ? p.total : 0;
}

ll_status gdn_launch(const FwdArgs& a) {
  const GdnPlan p = gdn_plan(a.s);
  if (!p.ok) return LL_ERR_UNSUPPORTED;
  if (a.ws_bytes < p.total) return LL_ERR_WORKSPACE;
  if (a.s.io == LL_F32) return launch_typed<float>(a, p);
  return launch_typed<__nv_bfloat16>(a, p);
}

}  // namespace llattn
