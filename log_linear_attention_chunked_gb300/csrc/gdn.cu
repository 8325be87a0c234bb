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
#include "sm100.cuh"

namespace llattn {

// the reading-B forward on the tensor cores (gdn_tc.cu): bf16, d = 128
size_t gdn_tc_b_workspace(const ll_shape& s);
ll_status gdn_tc_b_launch(const FwdArgs& a);

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

namespace fast {
using sm100::smem_u32;
using sm100::bulk_prefetch_l2;

constexpr int kDk = 128;
constexpr int kCe = 64;
constexpr int kR = 16;
constexpr int kSx = 132;   // row stride (floats) of X, W, Q', Kt tiles
constexpr int kSy = 68;    // Y rows
constexpr int kSp1 = 72;   // Y partial rows
constexpr int kSp2 = 136;  // X-update partial rows
constexpr int kSo = 17;    // output partials, [token][row]
constexpr int kMaxHeights = 8;

__host__ __device__ constexpr size_t smem_floats(int nh) {
  return (size_t)nh * kR * kSx + 3 * kCe * kSx + 4 * kR * kSp1 + 4 * kR * kSp2 + kR * kSy + (size_t)2 * nh * kCe;
}
static_assert(4 * kCe * kSo <= 4 * kR * kSp1, "output partials alias the Y partials");

}  // namespace fast

struct GdnPlan {
  int Ce, N, lc, nh;
  bool fast;       // d_k = 128, 64-token chunks: the register-tiled scan
  bool fast_prep;  // and d_v = 128: the register-tiled chunk preparation
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
  p.fast = s.dk == fast::kDk && p.Ce == fast::kCe && s.dv % fast::kR == 0 && p.nh <= fast::kMaxHeights &&
           fast::smem_floats(p.nh) * 4 <= kSmemLimit;
  p.fast_prep = p.fast && s.dv == fast::kDk;
  p.ok = prep_smem_floats(p.Ce, s.dk, s.dv) * 4 <= kSmemLimit && p.nh <= kMaxHeights && s.dv % kRows == 0 &&
         (p.fast || scan_smem_floats(p.Ce, s.dk, p.nh) * 4 <= kSmemLimit);
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

// ------------------------------------------- kernel 2, d_k = 128, 64-token chunks
// Same recurrence as gdn_scan_kernel, register-tiled for the float32 pipes.
// 256 threads own 16 d_v rows of every level state.  Per set height h:
//   phase 1  Y = X_h W^T and Pq = X_h Q'^T: thread tile 4 rows x 4 tokens for
//            both products over a quarter of d_k (split-K 4); the Y partials go
//            through shared memory, the Pq partials are weighted by lambda and
//            kept in registers until the chunk's output is written;
//   phase 2  X_h <- gamma X_h - Y Kt: thread tile 4 rows x 8 columns over a
//            quarter of the chunk's tokens, partials reduced in shared memory.
// Phase 2 of one height and phase 1 of the next share a barrier interval.
// Tiles are staged by cp.async into rows padded to 132 floats, so the 16-byte
// loads of a warp fall on distinct banks.  The next chunk's W and Q' stream in
// once phase 1 of the last height is done, its Kt once phase 2 is; Kt is
// waited for only before the next chunk's first phase 2.
namespace fast {
using sm100::smem_u32;
using sm100::bulk_prefetch_l2;

using sm100::cp_async16;
using sm100::cp_async4;
using sm100::cp_async_commit;
__device__ __forceinline__ void cp_async_wait0() { sm100::cp_async_wait<0>(); }
__device__ __forceinline__ void cp_async_wait1() { sm100::cp_async_wait<1>(); }

// 64 rows x 128 floats (contiguous in global) into a padded shared tile.
__device__ __forceinline__ void stage_tile(float* dst, const float* src, int tid) {
#pragma unroll
  for (int m = 0; m < 8; ++m) {
    const int x = tid + m * kThreads;  // float4 index
    const int i = x >> 5, f4 = x & 31;
    cp_async16(dst + i * kSx + 4 * f4, src + (size_t)x * 4);
  }
}

template <typename IO>
__global__ void __launch_bounds__(kThreads, 1) gdn_scan128_kernel(
    const float* __restrict__ Qp, const float* __restrict__ Wg, const float* __restrict__ Kt,
    const float* __restrict__ Sloc, const float* __restrict__ loggam, const float* __restrict__ Oacc,
    const float* __restrict__ lam, IO* __restrict__ o, int T, int dv, int L, int N, int lc, int nh) {
  extern __shared__ __align__(16) float sm[];
  const size_t bh = blockIdx.y;
  const int r0 = blockIdx.x * kR;
  const int tid = threadIdx.x;
  float* X = sm;                      // [nh][16][kSx]
  float* Wsm = X + nh * kR * kSx;     // [64][kSx]
  float* Qsm = Wsm + kCe * kSx;       // [64][kSx]
  float* Ksm = Qsm + kCe * kSx;       // [64][kSx]
  float* P1 = Ksm + kCe * kSx;        // [4][16][kSp1]; at the chunk end [4][64][kSo]
  float* P2 = P1 + 4 * kR * kSp1;     // [4][16][kSp2]
  float* Ysm = P2 + 4 * kR * kSp2;    // [16][kSy]
  float* lamc = Ysm + kR * kSy;       // [2][nh][64], by chunk parity

  const int ks = tid >> 6;            // split-K quarter
  const int u = tid & 63;
  const int rg = u & 3;               // rows rg + 4a
  const int cg = u >> 2;              // phase 1: tokens cg + 16j; phase 2: columns 4cg.., 64 + 4cg..

  float oc[4][4];   // lambda-weighted Pq partials of this chunk
  float gam = 1.f;

  auto phase1 = [&](int h, const float* lamh) {
    const float* Xh = X + h * kR * kSx;
    float y[4][4], p[4][4];
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int j = 0; j < 4; ++j) y[a][j] = p[a][j] = 0.f;
#pragma unroll
    for (int s = 0; s < 8; ++s) {
      const int f = ks * 32 + 4 * s;
      float4 xa[4], wa[4], qa[4];
#pragma unroll
      for (int a = 0; a < 4; ++a) xa[a] = *reinterpret_cast<const float4*>(Xh + (rg + 4 * a) * kSx + f);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        wa[j] = *reinterpret_cast<const float4*>(Wsm + (cg + 16 * j) * kSx + f);
        qa[j] = *reinterpret_cast<const float4*>(Qsm + (cg + 16 * j) * kSx + f);
      }
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          y[a][j] = fmaf(xa[a].x, wa[j].x, y[a][j]);
          y[a][j] = fmaf(xa[a].y, wa[j].y, y[a][j]);
          y[a][j] = fmaf(xa[a].z, wa[j].z, y[a][j]);
          y[a][j] = fmaf(xa[a].w, wa[j].w, y[a][j]);
          p[a][j] = fmaf(xa[a].x, qa[j].x, p[a][j]);
          p[a][j] = fmaf(xa[a].y, qa[j].y, p[a][j]);
          p[a][j] = fmaf(xa[a].z, qa[j].z, p[a][j]);
          p[a][j] = fmaf(xa[a].w, qa[j].w, p[a][j]);
        }
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float lj = lamh[cg + 16 * j];
#pragma unroll
      for (int a = 0; a < 4; ++a) {
        P1[(ks * kR + rg + 4 * a) * kSp1 + cg + 16 * j] = y[a][j];
        oc[a][j] = fmaf(lj, p[a][j], oc[a][j]);
      }
    }
  };
  auto reduce1 = [&]() {  // Y = sum of the four partials
    const int r = tid >> 4, i4 = tid & 15;
    float4 acc = *reinterpret_cast<const float4*>(P1 + r * kSp1 + 4 * i4);
#pragma unroll
    for (int q = 1; q < 4; ++q) {
      const float4 t = *reinterpret_cast<const float4*>(P1 + (q * kR + r) * kSp1 + 4 * i4);
      acc.x += t.x; acc.y += t.y; acc.z += t.z; acc.w += t.w;
    }
    *reinterpret_cast<float4*>(Ysm + r * kSy + 4 * i4) = acc;
  };
  auto phase2 = [&]() {
    float acc[4][8];
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int b = 0; b < 8; ++b) acc[a][b] = 0.f;
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      const int i = ks * 16 + 4 * s;
      float4 ya[4];
#pragma unroll
      for (int a = 0; a < 4; ++a) ya[a] = *reinterpret_cast<const float4*>(Ysm + (rg + 4 * a) * kSy + i);
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        const float4 k0 = *reinterpret_cast<const float4*>(Ksm + (i + t) * kSx + 4 * cg);
        const float4 k1 = *reinterpret_cast<const float4*>(Ksm + (i + t) * kSx + 64 + 4 * cg);
#pragma unroll
        for (int a = 0; a < 4; ++a) {
          const float yv = t == 0 ? ya[a].x : t == 1 ? ya[a].y : t == 2 ? ya[a].z : ya[a].w;
          acc[a][0] = fmaf(yv, k0.x, acc[a][0]);
          acc[a][1] = fmaf(yv, k0.y, acc[a][1]);
          acc[a][2] = fmaf(yv, k0.z, acc[a][2]);
          acc[a][3] = fmaf(yv, k0.w, acc[a][3]);
          acc[a][4] = fmaf(yv, k1.x, acc[a][4]);
          acc[a][5] = fmaf(yv, k1.y, acc[a][5]);
          acc[a][6] = fmaf(yv, k1.z, acc[a][6]);
          acc[a][7] = fmaf(yv, k1.w, acc[a][7]);
        }
      }
    }
#pragma unroll
    for (int a = 0; a < 4; ++a) {
      float* dst = P2 + (ks * kR + rg + 4 * a) * kSp2;
      *reinterpret_cast<float4*>(dst + 4 * cg) = make_float4(acc[a][0], acc[a][1], acc[a][2], acc[a][3]);
      *reinterpret_cast<float4*>(dst + 64 + 4 * cg) = make_float4(acc[a][4], acc[a][5], acc[a][6], acc[a][7]);
    }
  };
  auto reduce2 = [&](int h) {  // X_h <- gamma X_h - sum of the partials (this thread's 2 x 4 elements)
#pragma unroll
    for (int m = 0; m < 2; ++m) {
      const int e = tid + m * kThreads;
      const int r = e >> 5, f4 = e & 31;
      float* xp = X + h * kR * kSx + r * kSx + 4 * f4;
      float4 xv = *reinterpret_cast<const float4*>(xp);
      xv.x *= gam; xv.y *= gam; xv.z *= gam; xv.w *= gam;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float4 t = *reinterpret_cast<const float4*>(P2 + (q * kR + r) * kSp2 + 4 * f4);
        xv.x -= t.x; xv.y -= t.y; xv.z -= t.z; xv.w -= t.w;
      }
      *reinterpret_cast<float4*>(xp) = xv;
    }
  };
  // lambda of the levels above the chunk for chunk c1 (zero where the height is empty)
  auto stage_lam = [&](int c1) {
    float* dst = lamc + (c1 & 1) * nh * kCe;
    const size_t rowc = bh * T + (size_t)c1 * kCe;
    for (int x = tid; x < nh * kCe; x += kThreads) {
      const int h = x >> 6, i = x & 63;
      if (((c1 >> h) & 1) && lc + 1 + h < L) cp_async4(dst + x, lam + (rowc + i) * L + lc + 1 + h);
      else dst[x] = 0.f;
    }
  };

  for (int c = 0; c < N; ++c) {
    const size_t row0 = bh * T + (size_t)c * kCe;
    const bool more = c + 1 < N;
    gam = expf(loggam[bh * N + c]);
    float oa[4];  // this thread's four intra outputs: token e >> 4, row e & 15
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      const int e = tid + m * kThreads;
      oa[m] = Oacc[(row0 + (e >> 4)) * dv + r0 + (e & 15)];
    }
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int j = 0; j < 4; ++j) oc[a][j] = 0.f;

    int jc = 0;  // carry height cto(c)
    while ((c >> jc) & 1) ++jc;
    const float* Sc = Sloc + (bh * N + c) * (size_t)dv * kDk + (size_t)r0 * kDk;
    float4 sc[2];
    if (c > 0) {
      const float* lamh = lamc + (c & 1) * nh * kCe;
      int h = __ffs(c) - 1;
      phase1(h, lamh + h * kCe);
      cp_async_wait0();  // Kt of this chunk (and lambda)
      __syncthreads();
      if (more) {
        stage_lam(c + 1);
        cp_async_commit();
        if ((c >> (h + 1)) == 0) {
          stage_tile(Wsm, Wg + (row0 + kCe) * kDk, tid);
          stage_tile(Qsm, Qp + (row0 + kCe) * kDk, tid);
          cp_async_commit();
        }
      }
      reduce1();
      __syncthreads();
      while (true) {
        const int rest = c >> (h + 1);
        const int hn = rest ? h + __ffs(rest) : -1;
        if (hn < 0 && jc < nh) {
#pragma unroll
          for (int m = 0; m < 2; ++m) {
            const int e = tid + m * kThreads;
            sc[m] = *reinterpret_cast<const float4*>(Sc + (e >> 5) * kDk + 4 * (e & 31));
          }
        }
        phase2();
        if (hn >= 0) phase1(hn, lamh + hn * kCe);
        __syncthreads();
        if (hn < 0 && more) {
          stage_tile(Ksm, Kt + (row0 + kCe) * kDk, tid);
          cp_async_commit();
        }
        reduce2(h);
        if (hn < 0) break;
        if (more && (c >> (hn + 1)) == 0) {
          stage_tile(Wsm, Wg + (row0 + kCe) * kDk, tid);
          stage_tile(Qsm, Qp + (row0 + kCe) * kDk, tid);
          cp_async_commit();
        }
        reduce1();
        __syncthreads();
        h = hn;
      }
    } else if (jc < nh) {
#pragma unroll
      for (int m = 0; m < 2; ++m) {
        const int e = tid + m * kThreads;
        sc[m] = *reinterpret_cast<const float4*>(Sc + (e >> 5) * kDk + 4 * (e & 31));
      }
    }

    // carry into height cto(c): S_c + the transported levels below it (same
    // element ownership as the X update, so no barrier is needed)
    if (jc < nh) {
#pragma unroll
      for (int m = 0; m < 2; ++m) {
        const int e = tid + m * kThreads;
        const int r = e >> 5, f4 = e & 31;
        float4 acc = sc[m];
        for (int h = 0; h < jc; ++h) {
          const float4 t = *reinterpret_cast<const float4*>(X + h * kR * kSx + r * kSx + 4 * f4);
          acc.x += t.x; acc.y += t.y; acc.z += t.z; acc.w += t.w;
        }
        *reinterpret_cast<float4*>(X + jc * kR * kSx + r * kSx + 4 * f4) = acc;
      }
    }
    // output partials (the Y partials are free: their last reader passed a barrier)
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int j = 0; j < 4; ++j) P1[(ks * kCe + cg + 16 * j) * kSo + rg + 4 * a] = oc[a][j];
    if (c == 0 && more) {  // chunk 0 has no live level: nothing was staged yet
      stage_lam(1);
      stage_tile(Wsm, Wg + (row0 + kCe) * kDk, tid);
      stage_tile(Qsm, Qp + (row0 + kCe) * kDk, tid);
      cp_async_commit();
      stage_tile(Ksm, Kt + (row0 + kCe) * kDk, tid);
      cp_async_commit();
    }
    if (tid == 0) {
      if (c + 2 < N) {
        const size_t rn = row0 + 2 * kCe;
        bulk_prefetch_l2(Wg + rn * kDk, kCe * kDk * 4);
        bulk_prefetch_l2(Qp + rn * kDk, kCe * kDk * 4);
        bulk_prefetch_l2(Kt + rn * kDk, kCe * kDk * 4);
        bulk_prefetch_l2(Oacc + rn * dv, kCe * dv * 4);
      }
      if (more) bulk_prefetch_l2(Sc + (size_t)dv * kDk, kR * kDk * 4);
    }
    __syncthreads();
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      const int e = tid + m * kThreads;
      const int i = e >> 4, r = e & 15;
      float v = oa[m];
#pragma unroll
      for (int q = 0; q < 4; ++q) v += P1[(q * kCe + i) * kSo + r];
      o[(row0 + i) * dv + r0 + r] = from_f<IO>(v);
    }
    cp_async_wait1();  // all but the next chunk's Kt
    __syncthreads();
  }
  cp_async_wait0();
}

// ------------------------------------------- reading B: one state, pseudo-values out
// Reading B is log-linear Mamba-2 applied to the delta rule's pseudo-values
// u_t = beta_t (v_t - alpha_t S_{t-1} k_t), S the single gated-delta state.
// Per chunk, with S the state at the chunk start (S = 0 for chunk 0),
//   U_c = U - W S^T          (U = Tinv diag(beta) V and W from the preparation)
//   S  <- gamma S - (S W^T) Kt + S_c     (S_c = U^T Kt, the chunk's own state)
// This kernel runs that recurrence for 16 d_v rows per CTA and writes U_c in
// the io dtype, the values of the log-linear Mamba-2 forward that follows.
// Tiles and thread mapping as in gdn_scan128_kernel (one product in phase 1).
template <typename IO>
__global__ void __launch_bounds__(kThreads, 1) gdn_b_scan128_kernel(
    const float* __restrict__ Wg, const float* __restrict__ Kt, const float* __restrict__ Sloc,
    const float* __restrict__ loggam, const float* __restrict__ Ul, IO* __restrict__ U, int T, int dv, int N) {
  extern __shared__ __align__(16) float sm[];
  const size_t bh = blockIdx.y;
  const int r0 = blockIdx.x * kR;
  const int tid = threadIdx.x;
  float* X = sm;                     // [16][kSx] the state rows
  float* Wsm = X + kR * kSx;         // [64][kSx]
  float* Ksm = Wsm + kCe * kSx;      // [64][kSx]
  float* P1 = Ksm + kCe * kSx;       // [4][16][kSp1]
  float* P2 = P1 + 4 * kR * kSp1;    // [4][16][kSp2]
  float* Ysm = P2 + 4 * kR * kSp2;   // [16][kSy]
  const int ks = tid >> 6, u = tid & 63, rg = u & 3, cg = u >> 2;

  for (int c = 0; c < N; ++c) {
    const size_t row0 = bh * T + (size_t)c * kCe;
    const bool more = c + 1 < N;
    const float* Sc = Sloc + (bh * N + c) * (size_t)dv * kDk + (size_t)r0 * kDk;
    // this chunk's inputs from global memory, loaded before the products
    // that hide their latency: U (4 elements: token e >> 4, row e & 15) and
    // S_c (2 x 4 elements of the state rows)
    float ul[4];
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      const int e = tid + m * kThreads;
      ul[m] = Ul[(row0 + (e >> 4)) * dv + r0 + (e & 15)];
    }
    float4 scv[2];
#pragma unroll
    for (int m = 0; m < 2; ++m) {
      const int e = tid + m * kThreads;
      scv[m] = *reinterpret_cast<const float4*>(Sc + (e >> 5) * kDk + 4 * (e & 31));
    }
    const float gam = expf(loggam[bh * N + c]);
    if (tid == 0) {
      if (c + 2 < N) {
        const size_t rn = row0 + 2 * kCe;
        bulk_prefetch_l2(Wg + rn * kDk, kCe * kDk * 4);
        bulk_prefetch_l2(Kt + rn * kDk, kCe * kDk * 4);
      }
      if (more) {
        bulk_prefetch_l2(Ul + (row0 + kCe) * dv, kCe * dv * 4);
        bulk_prefetch_l2(Sc + (size_t)dv * kDk, kR * kDk * 4);
      }
    }
    if (c > 0) {
      // ---- Y = X W^T (split-K 4, partials through shared memory)
      float y[4][4];
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int j = 0; j < 4; ++j) y[a][j] = 0.f;
#pragma unroll
      for (int s8 = 0; s8 < 8; ++s8) {
        const int f = ks * 32 + 4 * s8;
        float4 xa[4], wa[4];
#pragma unroll
        for (int a = 0; a < 4; ++a) xa[a] = *reinterpret_cast<const float4*>(X + (rg + 4 * a) * kSx + f);
#pragma unroll
        for (int j = 0; j < 4; ++j) wa[j] = *reinterpret_cast<const float4*>(Wsm + (cg + 16 * j) * kSx + f);
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            y[a][j] = fmaf(xa[a].x, wa[j].x, y[a][j]);
            y[a][j] = fmaf(xa[a].y, wa[j].y, y[a][j]);
            y[a][j] = fmaf(xa[a].z, wa[j].z, y[a][j]);
            y[a][j] = fmaf(xa[a].w, wa[j].w, y[a][j]);
          }
      }
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int j = 0; j < 4; ++j) P1[(ks * kR + rg + 4 * a) * kSp1 + cg + 16 * j] = y[a][j];
      __syncthreads();
      if (more) {  // W is no longer read: the next chunk's streams in
        stage_tile(Wsm, Wg + (row0 + kCe) * kDk, tid);
        cp_async_commit();
      }
      {
        const int r = tid >> 4, i4 = tid & 15;
        float4 acc = *reinterpret_cast<const float4*>(P1 + r * kSp1 + 4 * i4);
#pragma unroll
        for (int q = 1; q < 4; ++q) {
          const float4 t = *reinterpret_cast<const float4*>(P1 + (q * kR + r) * kSp1 + 4 * i4);
          acc.x += t.x; acc.y += t.y; acc.z += t.z; acc.w += t.w;
        }
        *reinterpret_cast<float4*>(Ysm + r * kSy + 4 * i4) = acc;
      }
      if (more) cp_async_wait1();  // this chunk's Kt (the next W may still be in flight)
      else cp_async_wait0();
      __syncthreads();
    }
    // ---- U_c = U - Y^T for this CTA's rows
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      const int e = tid + m * kThreads;
      const int i = e >> 4, r = e & 15;
      U[(row0 + i) * dv + r0 + r] = from_f<IO>(c > 0 ? ul[m] - Ysm[r * kSy + i] : ul[m]);
    }
    if (c > 0) {
      // ---- partials of Y Kt
      float acc[4][8];
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int b = 0; b < 8; ++b) acc[a][b] = 0.f;
#pragma unroll
      for (int s4 = 0; s4 < 4; ++s4) {
        const int i = ks * 16 + 4 * s4;
        float4 ya[4];
#pragma unroll
        for (int a = 0; a < 4; ++a) ya[a] = *reinterpret_cast<const float4*>(Ysm + (rg + 4 * a) * kSy + i);
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          const float4 k0 = *reinterpret_cast<const float4*>(Ksm + (i + t) * kSx + 4 * cg);
          const float4 k1 = *reinterpret_cast<const float4*>(Ksm + (i + t) * kSx + 64 + 4 * cg);
#pragma unroll
          for (int a = 0; a < 4; ++a) {
            const float yv = t == 0 ? ya[a].x : t == 1 ? ya[a].y : t == 2 ? ya[a].z : ya[a].w;
            acc[a][0] = fmaf(yv, k0.x, acc[a][0]);
            acc[a][1] = fmaf(yv, k0.y, acc[a][1]);
            acc[a][2] = fmaf(yv, k0.z, acc[a][2]);
            acc[a][3] = fmaf(yv, k0.w, acc[a][3]);
            acc[a][4] = fmaf(yv, k1.x, acc[a][4]);
            acc[a][5] = fmaf(yv, k1.y, acc[a][5]);
            acc[a][6] = fmaf(yv, k1.z, acc[a][6]);
            acc[a][7] = fmaf(yv, k1.w, acc[a][7]);
          }
        }
      }
#pragma unroll
      for (int a = 0; a < 4; ++a) {
        float* dst = P2 + (ks * kR + rg + 4 * a) * kSp2;
        *reinterpret_cast<float4*>(dst + 4 * cg) = make_float4(acc[a][0], acc[a][1], acc[a][2], acc[a][3]);
        *reinterpret_cast<float4*>(dst + 64 + 4 * cg) = make_float4(acc[a][4], acc[a][5], acc[a][6], acc[a][7]);
      }
      __syncthreads();
    }
    if (more) {
      if (c == 0) {  // chunk 0 reads no tile: both of chunk 1's stream in now
        stage_tile(Wsm, Wg + (row0 + kCe) * kDk, tid);
        cp_async_commit();
      }
      stage_tile(Ksm, Kt + (row0 + kCe) * kDk, tid);  // Kt is no longer read
      cp_async_commit();
    }
    // ---- X <- gamma X - sum of the partials + S_c (this thread's 2 x 4 elements)
#pragma unroll
    for (int m = 0; m < 2; ++m) {
      const int e = tid + m * kThreads;
      const int r = e >> 5, f4 = e & 31;
      float* xp = X + r * kSx + 4 * f4;
      float4 xv = scv[m];
      if (c > 0) {
        const float4 x0 = *reinterpret_cast<const float4*>(xp);
        xv.x = fmaf(gam, x0.x, xv.x); xv.y = fmaf(gam, x0.y, xv.y);
        xv.z = fmaf(gam, x0.z, xv.z); xv.w = fmaf(gam, x0.w, xv.w);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float4 t = *reinterpret_cast<const float4*>(P2 + (q * kR + r) * kSp2 + 4 * f4);
          xv.x -= t.x; xv.y -= t.y; xv.z -= t.z; xv.w -= t.w;
        }
      }
      *reinterpret_cast<float4*>(xp) = xv;
    }
    if (more) cp_async_wait1();  // the next chunk's W (its Kt may still be in flight)
    __syncthreads();
  }
  cp_async_wait0();
}

constexpr size_t b_scan_smem_floats() { return kR * kSx + 2 * kCe * kSx + 4 * kR * kSp1 + 4 * kR * kSp2 + kR * kSy; }

}  // namespace fast

// ------------------------------------------- kernel 1, d_k = d_v = 128, 64-token chunks
// Same per-chunk quantities as gdn_prep_kernel, register-tiled.  The
// algebra is arranged so that every contraction is a plain product of two
// shared tiles:
//   Tb = Tinv diag(beta), Tbe = Tinv diag(beta e)
//   Cl = Aqk Tb, Cle = Aqk Tbe = Cl diag(e)
//   intra o = (Cl . lambda-mask) V,  U = Tb V,  W = Tbe K,  Q' = diag(e) Q - Cle K
//   S_c = U^T diag(exp(g_end - g)) K
// Tinv = (I + L)^{-1} is formed block-wise: the four 16 x 16 diagonal blocks by
// forward substitution, then the blocks below the diagonal one block-diagonal
// at a time, T_IJ = -T_II sum_{J <= M < I} L_IM T_MJ.
namespace fast {

constexpr int kSa = 68;  // row stride of the 64 x 64 tiles

__host__ __device__ constexpr size_t prep_smem_floats() {
  return 3 * kCe * kSx + 4 * kCe * kSa + 3 * 16 * 17 + 4 * kCe + kCe * 8;
}

__device__ __forceinline__ float4 ld4(const float* p) { return *reinterpret_cast<const float4*>(p); }
__device__ __forceinline__ void st4(float* p, float a, float b, float c, float d) {
  *reinterpret_cast<float4*>(p) = make_float4(a, b, c, d);
}
__device__ __forceinline__ float comp(const float4& v, int t) {
  return t == 0 ? v.x : t == 1 ? v.y : t == 2 ? v.z : v.w;
}

// 64 rows x 128 values of IO into a padded float32 tile
__device__ __forceinline__ void load_tile(float* dst, const float* src, int tid) {
#pragma unroll
  for (int m = 0; m < 8; ++m) {
    const int x = tid + m * kThreads;
    const int i = x >> 5, f4 = x & 31;
    *reinterpret_cast<float4*>(dst + i * kSx + 4 * f4) = ld4(src + (size_t)x * 4);
  }
}
__device__ __forceinline__ void load_tile(float* dst, const __nv_bfloat16* src, int tid) {
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    const int x = tid + m * kThreads;  // 8-element group
    const int i = x >> 4, f8 = x & 15;
    const uint4 raw = *reinterpret_cast<const uint4*>(src + (size_t)x * 8);
    const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.x));
    const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.y));
    const float2 cc = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.z));
    const float2 d = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.w));
    st4(dst + i * kSx + 8 * f8, a.x, a.y, b.x, b.y);
    st4(dst + i * kSx + 8 * f8 + 4, cc.x, cc.y, d.x, d.y);
  }
}

// C1 = A1 B, C2 = A2 B for this thread's rows 4ti..4ti+3 and columns
// 4tj..4tj+3, 64+4tj..64+4tj+3; A1, A2 are 64 x 64 lower-triangular tiles, B
// is 64 x 128, so the reduction stops at the warp's last row.
__device__ __forceinline__ void pair_product(const float* A1, const float* A2, const float* Bm, int ti, int tj,
                                             int mend, float (&c1)[4][8], float (&c2)[4][8]) {
#pragma unroll
  for (int r = 0; r < 4; ++r)
#pragma unroll
    for (int x = 0; x < 8; ++x) c1[r][x] = c2[r][x] = 0.f;
  for (int m = 0; m < mend; m += 4) {
    float4 a1[4], a2[4];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      a1[r] = ld4(A1 + (4 * ti + r) * kSa + m);
      a2[r] = ld4(A2 + (4 * ti + r) * kSa + m);
    }
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const float4 b0 = ld4(Bm + (m + t) * kSx + 4 * tj);
      const float4 b1 = ld4(Bm + (m + t) * kSx + 64 + 4 * tj);
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const float x = comp(a1[r], t), y = comp(a2[r], t);
        c1[r][0] = fmaf(x, b0.x, c1[r][0]); c1[r][1] = fmaf(x, b0.y, c1[r][1]);
        c1[r][2] = fmaf(x, b0.z, c1[r][2]); c1[r][3] = fmaf(x, b0.w, c1[r][3]);
        c1[r][4] = fmaf(x, b1.x, c1[r][4]); c1[r][5] = fmaf(x, b1.y, c1[r][5]);
        c1[r][6] = fmaf(x, b1.z, c1[r][6]); c1[r][7] = fmaf(x, b1.w, c1[r][7]);
        c2[r][0] = fmaf(y, b0.x, c2[r][0]); c2[r][1] = fmaf(y, b0.y, c2[r][1]);
        c2[r][2] = fmaf(y, b0.z, c2[r][2]); c2[r][3] = fmaf(y, b0.w, c2[r][3]);
        c2[r][4] = fmaf(y, b1.x, c2[r][4]); c2[r][5] = fmaf(y, b1.y, c2[r][5]);
        c2[r][6] = fmaf(y, b1.z, c2[r][6]); c2[r][7] = fmaf(y, b1.w, c2[r][7]);
      }
    }
  }
}

// C = A B for the same thread tile (reading B needs one product per pass)
__device__ __forceinline__ void single_product(const float* A, const float* Bm, int ti, int tj, int mend,
                                               float (&c1)[4][8]) {
#pragma unroll
  for (int r = 0; r < 4; ++r)
#pragma unroll
    for (int x = 0; x < 8; ++x) c1[r][x] = 0.f;
  for (int m = 0; m < mend; m += 4) {
    float4 a1[4];
#pragma unroll
    for (int r = 0; r < 4; ++r) a1[r] = ld4(A + (4 * ti + r) * kSa + m);
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const float4 b0 = ld4(Bm + (m + t) * kSx + 4 * tj);
      const float4 b1 = ld4(Bm + (m + t) * kSx + 64 + 4 * tj);
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const float x = comp(a1[r], t);
        c1[r][0] = fmaf(x, b0.x, c1[r][0]); c1[r][1] = fmaf(x, b0.y, c1[r][1]);
        c1[r][2] = fmaf(x, b0.z, c1[r][2]); c1[r][3] = fmaf(x, b0.w, c1[r][3]);
        c1[r][4] = fmaf(x, b1.x, c1[r][4]); c1[r][5] = fmaf(x, b1.y, c1[r][5]);
        c1[r][6] = fmaf(x, b1.z, c1[r][6]); c1[r][7] = fmaf(x, b1.w, c1[r][7]);
      }
    }
  }
}

// kB: reading B, which needs only U, W, Kt and S_c (no Q, Aqk, intra output
// or Q'), so the chunk's Q is not loaded and four of the products drop out.
template <typename IO, bool kB>
__global__ void __launch_bounds__(kThreads, 1) gdn_prep128_kernel(
    const IO* __restrict__ q, const IO* __restrict__ k, const IO* __restrict__ v,
    const float* __restrict__ log_alpha, const float* __restrict__ beta, const float* __restrict__ lam,
    float* __restrict__ Qp, float* __restrict__ Wg, float* __restrict__ Kt, float* __restrict__ Sloc,
    float* __restrict__ loggam, float* __restrict__ Oacc, float* __restrict__ Ug, int T, int L) {
  extern __shared__ __align__(16) float sm[];
  const int c = blockIdx.x, N = gridDim.x;
  const size_t bh = blockIdx.y;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  float* qs = sm;                   // [64][kSx]
  float* kk = qs + kCe * kSx;       // [64][kSx]
  float* vs = kk + kCe * kSx;       // [64][kSx]  V, later diag(exp(g_end - g)) U
  float* Lm = vs + kCe * kSx;       // [64][kSa]  L, later Cl . lambda-mask
  float* Aq = Lm + kCe * kSa;       // [64][kSa]  Aqk, later Cle
  float* Tb = Aq + kCe * kSa;       // [64][kSa]  Tinv, later Tinv diag(beta)
  float* Tbe = Tb + kCe * kSa;      // [64][kSa]
  float* Z = Tbe + kCe * kSa;       // [3][16][17]
  float* gs = Z + 3 * 16 * 17;      // g
  float* bs = gs + kCe;             // beta
  float* es = bs + kCe;             // exp(g)
  float* ds = es + kCe;             // exp(g_end - g)
  float* lamI = ds + kCe;           // [64][8] lambda of the in-chunk levels

  const size_t row0 = bh * T + (size_t)c * kCe;
  if constexpr (!kB) load_tile(qs, q + row0 * kDk, tid);
  load_tile(kk, k + row0 * kDk, tid);
  load_tile(vs, v + row0 * kDk, tid);
  if (warp == 0) {  // inclusive cumsum of log alpha (float64 across the warp)
    double a0 = log_alpha[row0 + lane], a1 = log_alpha[row0 + 32 + lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const double t0 = __shfl_up_sync(0xffffffffu, a0, o);
      const double t1 = __shfl_up_sync(0xffffffffu, a1, o);
      if (lane >= o) { a0 += t0; a1 += t1; }
    }
    a1 += __shfl_sync(0xffffffffu, a0, 31);
    const double gend = __shfl_sync(0xffffffffu, a1, 31);
    gs[lane] = (float)a0;
    gs[32 + lane] = (float)a1;
    es[lane] = expf((float)a0);
    es[32 + lane] = expf((float)a1);
    ds[lane] = expf((float)(gend - a0));
    ds[32 + lane] = expf((float)(gend - a1));
    if (lane == 0) loggam[bh * N + c] = (float)gend;
  } else if (warp == 1) {
    bs[lane] = beta[row0 + lane];
    bs[32 + lane] = beta[row0 + 32 + lane];
  }
  if constexpr (!kB)
    for (int x = tid; x < kCe * 8; x += kThreads) {
      const int i = x >> 3, l = x & 7;
      lamI[x] = l < L ? lam[(row0 + i) * L + l] : 0.f;
    }
  __syncthreads();

  // ---- L (strict lower, beta folded in) and Aqk (inclusive): rows ti + 16a, columns tj + 16b
  {
    const int ti = tid >> 4, tj = tid & 15;
    float a1[4][4], a2[4][4];
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int b = 0; b < 4; ++b) a1[a][b] = a2[a][b] = 0.f;
#pragma unroll 2
    for (int f = 0; f < kDk; f += 4) {
      float4 kI[4], qI[4], kJ[4];
#pragma unroll
      for (int a = 0; a < 4; ++a) {
        kI[a] = ld4(kk + (ti + 16 * a) * kSx + f);
        if constexpr (!kB) qI[a] = ld4(qs + (ti + 16 * a) * kSx + f);
        kJ[a] = ld4(kk + (tj + 16 * a) * kSx + f);
      }
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int b = 0; b < 4; ++b) {
          a1[a][b] = fmaf(kI[a].x, kJ[b].x, a1[a][b]); a1[a][b] = fmaf(kI[a].y, kJ[b].y, a1[a][b]);
          a1[a][b] = fmaf(kI[a].z, kJ[b].z, a1[a][b]); a1[a][b] = fmaf(kI[a].w, kJ[b].w, a1[a][b]);
          if constexpr (!kB) {
            a2[a][b] = fmaf(qI[a].x, kJ[b].x, a2[a][b]); a2[a][b] = fmaf(qI[a].y, kJ[b].y, a2[a][b]);
            a2[a][b] = fmaf(qI[a].z, kJ[b].z, a2[a][b]); a2[a][b] = fmaf(qI[a].w, kJ[b].w, a2[a][b]);
          }
        }
    }
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const int i = ti + 16 * a, j = tj + 16 * b;
        float lv = 0.f, av = 0.f;
        if (j <= i) {
          const float g = expf(gs[i] - gs[j]);
          av = a2[a][b] * g;
          if (j < i) lv = bs[i] * a1[a][b] * g;
        }
        Lm[i * kSa + j] = lv;
        if constexpr (!kB) Aq[i * kSa + j] = av;
      }
  }
  __syncthreads();

  // ---- Tinv: diagonal blocks by forward substitution (lane = column), upper blocks zero
  if (warp < 4) {
    if (lane < 16) {
      const int o = 16 * warp;
      float x[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        float s = (i == lane) ? 1.f : 0.f;
#pragma unroll
        for (int m = 0; m < i; ++m) s = fmaf(-Lm[(o + i) * kSa + o + m], x[m], s);
        x[i] = s;
      }
#pragma unroll
      for (int i = 0; i < 16; ++i) Tb[(o + i) * kSa + o + lane] = x[i];
    }
  } else {
    for (int x = tid - 128; x < kCe * kCe; x += 128) {
      const int i = x >> 6, j = x & 63;
      if ((i >> 4) < (j >> 4)) Tb[i * kSa + j] = 0.f;
    }
  }
  __syncthreads();
  for (int d = 1; d < 4; ++d) {
    const int nblk = 4 - d;
    for (int o = tid; o < nblk * 256; o += kThreads) {
      const int J = o >> 8, r = (o >> 4) & 15, cc = o & 15;
      const int row = 16 * (J + d) + r, col = 16 * J + cc;
      float s = 0.f;
      for (int m = 16 * J; m < 16 * (J + d); ++m) s = fmaf(Lm[row * kSa + m], Tb[m * kSa + col], s);
      Z[(J * 16 + r) * 17 + cc] = s;
    }
    __syncthreads();
    for (int o = tid; o < nblk * 256; o += kThreads) {
      const int J = o >> 8, r = (o >> 4) & 15, cc = o & 15;
      const int row = 16 * (J + d) + r;
      float s = 0.f;
#pragma unroll
      for (int m = 0; m < 16; ++m) s = fmaf(Tb[row * kSa + 16 * (J + d) + m], Z[(J * 16 + m) * 17 + cc], s);
      Tb[row * kSa + 16 * J + cc] = -s;
    }
    __syncthreads();
  }
  for (int x = tid; x < kCe * kCe; x += kThreads) {
    const int i = x >> 6, j = x & 63;
    const float t = Tb[i * kSa + j] * bs[j];
    Tb[i * kSa + j] = t;
    Tbe[i * kSa + j] = t * es[j];
  }
  __syncthreads();

  const int ti = tid >> 4, tj = tid & 15;
  const int mend = 8 * warp + 8;  // rows of this warp: 8 warp .. 8 warp + 7
  // ---- Cl = Aqk Tb (masked by the in-chunk levels, into Lm), Cle = Aqk Tbe (into Aq)
  if constexpr (!kB) {
    float c1[4][4], c2[4][4];
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
      for (int x = 0; x < 4; ++x) c1[r][x] = c2[r][x] = 0.f;
    for (int m = 0; m < mend; m += 4) {
      float4 a[4];
#pragma unroll
      for (int r = 0; r < 4; ++r) a[r] = ld4(Aq + (4 * ti + r) * kSa + m);
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        const float4 b1 = ld4(Tb + (m + t) * kSa + 4 * tj);
        const float4 b2 = ld4(Tbe + (m + t) * kSa + 4 * tj);
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          const float x = comp(a[r], t);
          c1[r][0] = fmaf(x, b1.x, c1[r][0]); c1[r][1] = fmaf(x, b1.y, c1[r][1]);
          c1[r][2] = fmaf(x, b1.z, c1[r][2]); c1[r][3] = fmaf(x, b1.w, c1[r][3]);
          c2[r][0] = fmaf(x, b2.x, c2[r][0]); c2[r][1] = fmaf(x, b2.y, c2[r][1]);
          c2[r][2] = fmaf(x, b2.z, c2[r][2]); c2[r][3] = fmaf(x, b2.w, c2[r][3]);
        }
      }
    }
    __syncthreads();  // every read of Aq is done
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int i = 4 * ti + r;
      float w[4];
#pragma unroll
      for (int x = 0; x < 4; ++x) {
        const int j = 4 * tj + x;
        w[x] = j <= i ? c1[r][x] * lamI[i * 8 + bitlen((unsigned)(i ^ j))] : 0.f;
      }
      st4(Lm + i * kSa + 4 * tj, w[0], w[1], w[2], w[3]);
      st4(Aq + i * kSa + 4 * tj, c2[r][0], c2[r][1], c2[r][2], c2[r][3]);
    }
    __syncthreads();
  }

  // ---- intra output and U = Tb V (kept as diag(exp(g_end - g)) U in place of V)
  {
    float c1[4][8], c2[4][8];
    if constexpr (kB) {
      single_product(Tb, vs, ti, tj, mend, c2);
    } else {
      pair_product(Lm, Tb, vs, ti, tj, mend, c1, c2);
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        float* orow = Oacc + (row0 + 4 * ti + r) * kDk;
        st4(orow + 4 * tj, c1[r][0], c1[r][1], c1[r][2], c1[r][3]);
        st4(orow + 64 + 4 * tj, c1[r][4], c1[r][5], c1[r][6], c1[r][7]);
      }
    }
    if (Ug) {  // the chunk's own pseudo-values U (reading B)
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        float* urow = Ug + (row0 + 4 * ti + r) * kDk;
        st4(urow + 4 * tj, c2[r][0], c2[r][1], c2[r][2], c2[r][3]);
        st4(urow + 64 + 4 * tj, c2[r][4], c2[r][5], c2[r][6], c2[r][7]);
      }
    }
    __syncthreads();  // every read of V is done
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const float dsr = ds[4 * ti + r];
      float* u = vs + (4 * ti + r) * kSx;
      st4(u + 4 * tj, dsr * c2[r][0], dsr * c2[r][1], dsr * c2[r][2], dsr * c2[r][3]);
      st4(u + 64 + 4 * tj, dsr * c2[r][4], dsr * c2[r][5], dsr * c2[r][6], dsr * c2[r][7]);
    }
  }
  // ---- W = Tbe K, Q' = diag(e) Q - Cle K, Kt = diag(exp(g_end - g)) K
  {
    float c1[4][8], c2[4][8];
    if constexpr (kB) single_product(Tbe, kk, ti, tj, mend, c1);
    else pair_product(Tbe, Aq, kk, ti, tj, mend, c1, c2);
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int i = 4 * ti + r;
      const float ei = es[i], di = ds[i];
      const size_t go = (row0 + i) * kDk;
#pragma unroll
      for (int hlf = 0; hlf < 2; ++hlf) {
        const int f = 64 * hlf + 4 * tj;
        const float4 kv = ld4(kk + i * kSx + f);
        const int o = 4 * hlf;
        st4(Wg + go + f, c1[r][o], c1[r][o + 1], c1[r][o + 2], c1[r][o + 3]);
        if constexpr (!kB) {
          const float4 qv = ld4(qs + i * kSx + f);
          st4(Qp + go + f, ei * qv.x - c2[r][o], ei * qv.y - c2[r][o + 1], ei * qv.z - c2[r][o + 2],
              ei * qv.w - c2[r][o + 3]);
        }
        st4(Kt + go + f, di * kv.x, di * kv.y, di * kv.z, di * kv.w);
      }
    }
  }
  __syncthreads();  // diag(exp(g_end - g)) U is in place

  // ---- S_c = U^T diag(exp(g_end - g)) K: rows 4ti.., 64+4ti..; columns 4tj.., 64+4tj..
  {
    float s[8][8];
#pragma unroll
    for (int r = 0; r < 8; ++r)
#pragma unroll
      for (int x = 0; x < 8; ++x) s[r][x] = 0.f;
#pragma unroll 2
    for (int j = 0; j < kCe; ++j) {
      const float4 u0 = ld4(vs + j * kSx + 4 * ti), u1 = ld4(vs + j * kSx + 64 + 4 * ti);
      const float4 k0 = ld4(kk + j * kSx + 4 * tj), k1 = ld4(kk + j * kSx + 64 + 4 * tj);
#pragma unroll
      for (int r = 0; r < 8; ++r) {
        const float uv = comp(r < 4 ? u0 : u1, r & 3);
        s[r][0] = fmaf(uv, k0.x, s[r][0]); s[r][1] = fmaf(uv, k0.y, s[r][1]);
        s[r][2] = fmaf(uv, k0.z, s[r][2]); s[r][3] = fmaf(uv, k0.w, s[r][3]);
        s[r][4] = fmaf(uv, k1.x, s[r][4]); s[r][5] = fmaf(uv, k1.y, s[r][5]);
        s[r][6] = fmaf(uv, k1.z, s[r][6]); s[r][7] = fmaf(uv, k1.w, s[r][7]);
      }
    }
    float* Sc = Sloc + (bh * N + c) * (size_t)kDk * kDk;
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      const int e = r < 4 ? 4 * ti + r : 64 + 4 * ti + (r - 4);
      st4(Sc + e * kDk + 4 * tj, s[r][0], s[r][1], s[r][2], s[r][3]);
      st4(Sc + e * kDk + 64 + 4 * tj, s[r][4], s[r][5], s[r][6], s[r][7]);
    }
  }
}

}  // namespace fast

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
  if (p.fast_prep && aligned16(a.q) && aligned16(a.k) && aligned16(a.v)) {
    const size_t sm1 = fast::prep_smem_floats() * 4;
    LL_CUDA_OK(cudaFuncSetAttribute(fast::gdn_prep128_kernel<IO, false>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm1));
    fast::gdn_prep128_kernel<IO, false><<<dim3(p.N, BH), kThreads, sm1, a.stream>>>(
        static_cast<const IO*>(a.q), static_cast<const IO*>(a.k), static_cast<const IO*>(a.v), a.log_alpha,
        a.beta, a.lam, Qp, W, Kt, S, lg, O, nullptr, s.T, s.L);
  } else {
    const size_t sm1 = prep_smem_floats(p.Ce, s.dk, s.dv) * 4;
    LL_CUDA_OK(cudaFuncSetAttribute(gdn_prep_kernel<IO>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm1));
    gdn_prep_kernel<IO><<<dim3(p.N, BH), kThreads, sm1, a.stream>>>(
        static_cast<const IO*>(a.q), static_cast<const IO*>(a.k), static_cast<const IO*>(a.v), a.log_alpha,
        a.beta, a.lam, Qp, W, Kt, S, lg, O, s.T, s.dk, s.dv, s.L, p.Ce);
  }
  LL_CUDA_OK(cudaGetLastError());
  if (p.fast) {
    const size_t sm2 = fast::smem_floats(p.nh) * 4;
    LL_CUDA_OK(cudaFuncSetAttribute(fast::gdn_scan128_kernel<IO>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)sm2));
    fast::gdn_scan128_kernel<IO><<<dim3(s.dv / fast::kR, BH), kThreads, sm2, a.stream>>>(
        Qp, W, Kt, S, lg, O, a.lam, static_cast<IO*>(a.o), s.T, s.dv, s.L, p.N, p.lc, p.nh);
  } else {
    const size_t sm2 = scan_smem_floats(p.Ce, s.dk, p.nh) * 4;
    LL_CUDA_OK(cudaFuncSetAttribute(gdn_scan_kernel<IO>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm2));
    gdn_scan_kernel<IO><<<dim3(s.dv / kRows, BH), kThreads, sm2, a.stream>>>(
        Qp, W, Kt, S, lg, O, a.lam, static_cast<IO*>(a.o), s.T, s.dk, s.dv, s.L, p.Ce, p.N, p.lc, p.nh);
  }
  LL_CUDA_OK(cudaGetLastError());
  return LL_OK;
}

}  // namespace

size_t gdn_workspace(const ll_shape& s) {
  if (gdn_tc_supported(s)) return gdn_tc_workspace(s);
  const GdnPlan p = gdn_plan(s);
  return p.ok ? p.total : 0;
}

ll_status gdn_launch(const FwdArgs& a) {
  if (gdn_tc_supported(a.s)) return gdn_tc_launch(a);  // bf16 io: the tensor cores
  const GdnPlan p = gdn_plan(a.s);
  if (!p.ok) return LL_ERR_UNSUPPORTED;
  if (a.ws_bytes < p.total) return LL_ERR_WORKSPACE;
  if (a.s.io == LL_F32) return launch_typed<float>(a, p);
  return launch_typed<__nv_bfloat16>(a, p);
}

// ---------------------------------------------------------------- reading B
// workspace: the preparation's buffers | U (float32) | U_c (io dtype, the
// forward's values) | the log-linear Mamba-2 forward's own workspace
namespace {

struct GdnBPlan {
  GdnPlan g;
  size_t off_Ul, off_Uio, off_fwd, fwd_bytes, total;
  bool ok;
};

GdnBPlan gdn_b_plan(const ll_shape& s) {
  GdnBPlan b{};
  b.g = gdn_plan(s);
  b.ok = b.g.ok && b.g.fast_prep;
  if (!b.ok) return b;
  const size_t BH = (size_t)s.B * s.H;
  const size_t esz = s.io == LL_F32 ? 4 : 2;
  size_t off = b.g.total;
  b.off_Ul = off;  off = align_up(off + BH * s.T * (size_t)s.dv * 4, 256);
  b.off_Uio = off; off = align_up(off + BH * s.T * (size_t)s.dv * esz, 256);
  b.fwd_bytes = fwd_tc_supported(s) ? fwd_tc_workspace(s) : fwd_simt_workspace(s);
  b.off_fwd = off; off = align_up(off + b.fwd_bytes, 256);
  b.total = off;
  return b;
}

template <typename IO>
ll_status launch_b_typed(const FwdArgs& a, const GdnBPlan& b) {
  const ll_shape& s = a.s;
  const GdnPlan& p = b.g;
  unsigned char* ws = static_cast<unsigned char*>(a.ws);
  float* Qp = reinterpret_cast<float*>(ws + p.off_Qp);
  float* W = reinterpret_cast<float*>(ws + p.off_W);
  float* Kt = reinterpret_cast<float*>(ws + p.off_Kt);
  float* S = reinterpret_cast<float*>(ws + p.off_S);
  float* lg = reinterpret_cast<float*>(ws + p.off_lg);
  float* O = reinterpret_cast<float*>(ws + p.off_O);
  float* Ul = reinterpret_cast<float*>(ws + b.off_Ul);
  IO* Uio = reinterpret_cast<IO*>(ws + b.off_Uio);
  const int BH = s.B * s.H;
  const size_t sm1 = fast::prep_smem_floats() * 4;
  LL_CUDA_OK(cudaFuncSetAttribute(fast::gdn_prep128_kernel<IO, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)sm1));
  fast::gdn_prep128_kernel<IO, true><<<dim3(p.N, BH), kThreads, sm1, a.stream>>>(
      static_cast<const IO*>(a.q), static_cast<const IO*>(a.k), static_cast<const IO*>(a.v), a.log_alpha, a.beta,
      a.lam, Qp, W, Kt, S, lg, O, Ul, s.T, s.L);
  LL_CUDA_OK(cudaGetLastError());
  const size_t sm2 = fast::b_scan_smem_floats() * 4;
  LL_CUDA_OK(cudaFuncSetAttribute(fast::gdn_b_scan128_kernel<IO>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)sm2));
  fast::gdn_b_scan128_kernel<IO><<<dim3(s.dv / fast::kR, BH), kThreads, sm2, a.stream>>>(W, Kt, S, lg, Ul, Uio, s.T,
                                                                                         s.dv, p.N);
  LL_CUDA_OK(cudaGetLastError());
  FwdArgs f = a;
  f.v = Uio;
  f.beta = nullptr;
  f.state_out = nullptr;
  f.scale_out = nullptr;
  f.ws = ws + b.off_fwd;
  f.ws_bytes = b.fwd_bytes;
  return fwd_tc_supported(s) ? fwd_tc_launch(f) : fwd_simt_launch(f);
}

}  // namespace

size_t gdn_b_workspace(const ll_shape& s) {
  if (gdn_tc_supported(s) && fwd_tc_supported(s)) return gdn_tc_b_workspace(s);  // bf16 io: the tensor cores
  const GdnBPlan b = gdn_b_plan(s);
  return b.ok ? b.total : 0;
}

ll_status gdn_b_launch(const FwdArgs& a) {
  if (gdn_tc_supported(a.s) && fwd_tc_supported(a.s)) return gdn_tc_b_launch(a);
  const GdnBPlan b = gdn_b_plan(a.s);
  if (!b.ok) return LL_ERR_UNSUPPORTED;
  if (a.ws_bytes < b.total) return LL_ERR_WORKSPACE;
  if (a.s.io == LL_F32) return launch_b_typed<float>(a, b);
  return launch_b_typed<__nv_bfloat16>(a, b);
}

}  // namespace llattn
