// Log-Linear Gated DeltaNet forward, reading A, on the 5th-generation tensor
// cores (tcgen05 with TMEM accumulators, TMA-staged bf16 operands): bf16 io,
// d_k = d_v = 128, 128-token chunks ("Log-Linear Attention" study note §3-5;
// gist.science (de) Technische Zusammenfassung §2; the gated delta rule and
// reading A as in the float32 path of gdn.cu).
//
// Chunk c (128 tokens, g = inclusive cumsum of log_alpha inside the chunk,
// e = exp(g), G_ij = exp(g_i - g_j) for j <= i):
//   Tinv = (I + diag(beta) SL(K K^T . G))^{-1}            (unit lower triangular)
//   U = Tinv diag(beta) V,  W = Tinv diag(beta e) K,  Aqk = (Q K^T . G) (j <= i)
//   intra  o_i = sum_{j <= i} (Aqk Tinv diag(beta))_ij lam_i[bitlen(i ^ j)] v_j
//   Q' = diag(e) Q - Aqk W,  Kt = diag(exp(g_end - g)) K,  gamma = exp(g_end)
//   a level state X (d_v x d_k) at the chunk start adds lam_i[8 + h] X q'_i to
//   o_i and leaves the chunk as gamma X - (X W^T) Kt; after chunk c the heights
//   below cto(c) and S_c = U^T Kt add into height cto(c) (level 8 + h).
// The result does not depend on the chunk length (the float32 path uses 64).
//
// Kernel 1 (gdn_tc_prep_kernel), one CTA per (chunk, head), 256 threads:
// K K^T and Q K^T, then U^T (as V^T Tb^T, so it leaves TMEM row by row), W
// and Aqk Tinv, then Aqk W and the masked intra product, each a 128x128x128
// UMMA with bf16 operands in 128-byte-swizzled shared tiles and float32
// accumulators in TMEM.  The triangular inverse runs on the CUDA cores in
// float32 (16x16 blocks: the diagonal blocks by forward substitution, then the
// block diagonals below them, T_IJ = -T_II sum_M L_IM T_MJ, one block per
// warp).  Writes W, Q', U^T (bf16) and the intra output (bf16) per chunk.
//
// Kernel 2 (gdn_tc_scan_kernel), one CTA per (32 d_v rows, head), 128
// threads, sequential over the chunks of its head.  Every level state is held
// transposed in TMEM as a float32 accumulator X^T [d_k lanes x 32 columns];
// per chunk and live height h the products are
//   Y^T = W X^T and Pq^T = Q' X^T        (M = 128 tokens, N = 32, K = d_k)
//   X^T <- gamma X^T + Kt^T (-Y^T)       (M = d_k, N = 32, K = 128 tokens)
// with X and -Y rounded to bf16 as operands (the state itself stays float32),
// and the carry X^T_cto += Kt^T U^T_slice.  The lambda-weighted Pq^T rows are
// summed in registers and added to the intra output.
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>

#include "common.cuh"
#include "sm100.cuh"

namespace llattn {

namespace {

using namespace sm100;

constexpr int kC = 128;                     // tokens per chunk (the MMA M)
constexpr int kD = 128;                     // d_k = d_v
constexpr uint32_t kHalf = kC * 64 * 2;     // [128 rows x 64] bf16 swizzled block: 16 KB
constexpr uint32_t kTileB = 2 * kHalf;      // 32 KB
constexpr int kSlice = 32;                  // d_v rows per scan CTA
constexpr uint32_t kHalf32 = kSlice * 128;  // [32 rows x 64] bf16 swizzled block: 4 KB
constexpr uint32_t kSliceB = 2 * kHalf32;   // 8 KB
constexpr int kMaxHeights = 8;              // chunk counts up to 256
constexpr float kLog2e = 1.4426950408889634f;
constexpr uint64_t kTimeoutNs = 4000000000ull;

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Bounded wait for the phase with parity `par` (every thread); records a
// timeout in the error word and returns.  The waits of these kernels are on
// their own copies and products only, which always complete.
__device__ __forceinline__ void wait_bar(uint64_t* bar, uint32_t par, unsigned* err) {
  if (mbar_try_wait(bar, par)) return;
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, par)) {
    if (globaltimer_ns() - t0 > kTimeoutNs) {
      atomicOr(err, kErrTimeout);
      return;
    }
  }
}

// byte offset of element (r, k) in a K-major 128-byte-swizzled tile of `rows`
// rows (64-element column blocks rows*128 bytes apart)
__device__ __forceinline__ uint32_t swz_off(int r, int k, int rows) {
  return (uint32_t)(k >> 6) * (uint32_t)rows * 128u + (uint32_t)r * 128u +
         ((uint32_t)(((k & 63) >> 3) ^ (r & 7)) << 4) + (uint32_t)(k & 7) * 2u;
}
// 16-byte chunk c8 (elements 8 c8 .. 8 c8 + 7) of row r of a 128-row tile
__device__ __forceinline__ uint32_t swz16(int r, int c8) {
  return (uint32_t)(c8 >> 3) * kHalf + (uint32_t)r * 128u + ((uint32_t)((c8 & 7) ^ (r & 7)) << 4);
}

// K-major operand of a 128-row tile, k-step kk of 16
__device__ __forceinline__ uint64_t desc_k(uint32_t tile, int kk) {
  return sw128_desc(tile + (kk >> 2) * kHalf + (kk & 3) * 32, 16, 1024);
}
// K-major operand of a 32-row tile (N = 32), k-step kk of 16
__device__ __forceinline__ uint64_t desc_k32(uint32_t tile, int kk) {
  return sw128_desc(tile + (kk >> 2) * kHalf32 + (kk & 3) * 32, 16, 1024);
}
// MN-major operand of a 128x128 tile (rows = K), k-step kk of 16 rows
__device__ __forceinline__ uint64_t desc_mn(uint32_t tile, int kk) { return sw128_desc(tile + kk * 2048, kHalf, 1024); }

__device__ __forceinline__ void mma_128(uint32_t d, uint32_t a, bool a_mn, uint32_t b, bool b_mn, uint32_t acc0) {
  const uint32_t id = idesc_bf16(128, 128, a_mn, b_mn);
#pragma unroll
  for (int kk = 0; kk < 8; ++kk)
    umma_bf16(d, a_mn ? desc_mn(a, kk) : desc_k(a, kk), b_mn ? desc_mn(b, kk) : desc_k(b, kk), id,
              kk > 0 ? 1u : acc0);
}

// ------------------------------------------------------------------ kernel 1
// shared memory (offsets from a 1024-aligned base)
constexpr uint32_t kPK = 0;                    // K tile; U^T staging after the W product
constexpr uint32_t kPQ = kPK + kTileB;         // Q tile
constexpr uint32_t kPV = kPQ + kTileB;         // V tile
constexpr uint32_t kPA = kPV + kTileB;         // Aqk (bf16); Q' staging at the end
constexpr int kBS = 20;                        // row stride (floats) of a 16x16 block: conflict-free 16-byte reads
constexpr uint32_t kPBlk = 36 * 16 * kBS * 4;  // 36 lower 16x16 blocks, float32
constexpr uint32_t kPL = kPA + kTileB;         // L, then T_II L_IM (blocks); then Tb; then Cm; then intra staging
constexpr uint32_t kPT = kPL + kPBlk;          // Tinv (blocks); then Tbe; then W
constexpr uint32_t kPTab = kPT + kPBlk;        // g[128], e[128], beta[128], quadrant totals[4]
constexpr uint32_t kPBars = kPTab + (3 * 128 + 4) * 4;
constexpr uint32_t kPrepSmem = kPBars + 4 * 8;
constexpr int kPrepThreads = 256;
static_assert(kPL % 1024 == 0 && kPT % 1024 == 0, "tile alignment");
static_assert(kPrepSmem <= 232448, "shared memory budget of one CTA");

// float offset of lower block (I, J), J <= I, in the block storage
__device__ __forceinline__ int blk(int I, int J) { return (I * (I + 1) / 2 + J) * 16 * kBS; }

struct PrepParams {
  const float* log_alpha;
  const float* beta;
  const float* lam;
  int T, L, Nc;
  unsigned* err;
  const __nv_bfloat16 *q, *k, *v;  // (the L2 prefetch of the next item's rows)
  int BH;
};

// kB: reading B's preparation, which needs only U and W (no Q, Aqk, Q' or
// intra output: no Q load, three products fewer, two stores fewer).
template <bool kB>
__global__ void __launch_bounds__(kPrepThreads, 1)
    gdn_tc_prep_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                       const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tw,
                       const __grid_constant__ CUtensorMap tqp, const __grid_constant__ CUtensorMap tut,
                       const __grid_constant__ CUtensorMap toi, PrepParams p) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  if (smem_u32(smem_raw) & 1023u) {
    if (threadIdx.x == 0) atomicOr(p.err, kErrDeviceArg);
    return;
  }
  unsigned char* s = smem_raw;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int q = warp & 3, hf = warp >> 2;
  const int i = 32 * q + lane;  // this thread's row (TMEM lane)
  float* gs = reinterpret_cast<float*>(s + kPTab);
  float* es = gs + 128;
  float* bs = es + 128;
  float* qtot = bs + 128;
  uint64_t* bars = reinterpret_cast<uint64_t*>(s + kPBars);  // 0: inputs, 1: products
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(s + kPBars + 3 * 8);
  float* Lp = reinterpret_cast<float*>(s + kPL);
  float* Tp = reinterpret_cast<float*>(s + kPT);
  const uint32_t sK = smem_u32(s + kPK), sQ = smem_u32(s + kPQ), sV = smem_u32(s + kPV), sA = smem_u32(s + kPA),
                 sL = smem_u32(s + kPL), sT = smem_u32(s + kPT);

  if (tid == 0) {
    mbar_init(bars + 0, 1);
    mbar_init(bars + 1, 1);
    fence_mbar_init();
  }
  __syncwarp();
  if (warp == 0) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tl = tmem + ((uint32_t)(32 * q) << 16);
  constexpr uint32_t kProducts = kB ? 2 : 3;  // product commits per item
  const int items = p.Nc * p.BH;
  // persistent: item w = (chunk w mod Nc, head w / Nc), one after another
  uint32_t k_it = 0;
  for (int w = blockIdx.x; w < items; w += gridDim.x, ++k_it) {
  const int c = w % p.Nc;
  const int bh = w / p.Nc;
  const int row0 = bh * p.T + c * kC;
  const uint32_t pb = k_it * kProducts;  // product commits before this item
  if (tid == 0) {
    bulk_wait_read0();  // the previous item's stores have read their tiles
    mbar_arrive_expect_tx(bars + 0, (kB ? 2 : 3) * kTileB);
    tma_load_2d(s + kPK, &tk, bars + 0, 0, row0);
    tma_load_2d(s + kPK + kHalf, &tk, bars + 0, 64, row0);
    if (!kB) {
      tma_load_2d(s + kPQ, &tq, bars + 0, 0, row0);
      tma_load_2d(s + kPQ + kHalf, &tq, bars + 0, 64, row0);
    }
    tma_load_2d(s + kPV, &tv, bars + 0, 0, row0);
    tma_load_2d(s + kPV + kHalf, &tv, bars + 0, 64, row0);
    const int wn = w + (int)gridDim.x;  // the next item's rows into L2 meanwhile
    if (wn < items) {
      const size_t rn = (size_t)(wn / p.Nc) * p.T + (size_t)(wn % p.Nc) * kC;
      bulk_prefetch_l2(p.k + rn * kD, kTileB);
      if (!kB) bulk_prefetch_l2(p.q + rn * kD, kTileB);
      bulk_prefetch_l2(p.v + rn * kD, kTileB);
    }
  }
  // inclusive cumsum of log_alpha over the chunk (both halves compute it)
  const float la = p.log_alpha[row0 + i];
  const float bt = p.beta[row0 + i];
  float x = la;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (hf == 0 && lane == 31) qtot[q] = x;
  __syncthreads();
  float off = 0.f;
  for (int qq = 0; qq < q; ++qq) off += qtot[qq];
  const float g_i = x + off;
  if (hf == 0) {
    gs[i] = g_i;
    es[i] = ex2(g_i * kLog2e);
    bs[i] = bt;
  }
  float lam8[8];  // lambda of the intra-chunk levels 0..7 of row i
#pragma unroll
  for (int l = 0; l < 8; ++l) lam8[l] = kB ? 0.f : p.lam[(size_t)(row0 + i) * p.L + l];
  __syncthreads();

  // ---- K K^T -> cols 0..127, Q K^T -> cols 128..255
  wait_bar(bars + 0, k_it & 1, p.err);
  if (tid == 0) {
    tc_fence_after();
    mma_128(tmem + 0, sK, false, sK, false, 0);
    if (!kB) mma_128(tmem + 128, sQ, false, sK, false, 0);
    umma_commit(bars + 1);
  }
  wait_bar(bars + 1, pb & 1, p.err);
  __syncwarp();
  tc_fence_after();
  // L_ij = beta_i (k_i.k_j) G_ij (j < i), packed lower blocks; Aqk_ij = (q_i.k_j) G_ij (j <= i), bf16 tile
  {
    const float g2i = g_i * kLog2e;
#pragma unroll
    for (int c32 = 0; c32 < 2; ++c32) {
      const int j0 = 64 * hf + 32 * c32;
      float kk[32], qk[32];
      tmem_ld32(tl + j0, kk);
      if (!kB) tmem_ld32(tl + 128 + j0, qk);
      tmem_ld_wait();
#pragma unroll
      for (int jj = 0; jj < 32; ++jj) {
        const int j = j0 + jj;
        const float gij = j <= i ? ex2(g2i - gs[j] * kLog2e) : 0.f;
        kk[jj] = j < i ? bt * kk[jj] * gij : 0.f;
        qk[jj] = qk[jj] * gij;
      }
      // L: the 16-wide segments of blocks (i/16, j/16) on or below the diagonal
#pragma unroll
      for (int b = 0; b < 2; ++b) {
        const int J = (j0 >> 4) + b, I = i >> 4;
        if (J <= I) {
          float4* dst = reinterpret_cast<float4*>(Lp + blk(I, J) + (i & 15) * kBS);
#pragma unroll
          for (int v = 0; v < 4; ++v)
            dst[v] = make_float4(kk[16 * b + 4 * v], kk[16 * b + 4 * v + 1], kk[16 * b + 4 * v + 2],
                                 kk[16 * b + 4 * v + 3]);
        }
      }
#pragma unroll
      for (int c8 = 0; c8 < 4 && !kB; ++c8) {
        uint4 w;
        w.x = pack_bf16x2(qk[8 * c8], qk[8 * c8 + 1]);
        w.y = pack_bf16x2(qk[8 * c8 + 2], qk[8 * c8 + 3]);
        w.z = pack_bf16x2(qk[8 * c8 + 4], qk[8 * c8 + 5]);
        w.w = pack_bf16x2(qk[8 * c8 + 6], qk[8 * c8 + 7]);
        *reinterpret_cast<uint4*>(s + kPA + swz16(i, (j0 >> 3) + c8)) = w;
      }
    }
  }
  fence_proxy_async_shared();
  __syncthreads();

  // ---- Tinv = (I + L)^{-1} in 16x16 blocks.  Row block I of (I + L) T = I
  // gives T_IJ = -T_II sum_{M=J}^{I-1} L_IM T_MJ for J < I.  First the
  // diagonal blocks by forward substitution (one column per thread), then
  // Lam_IM = T_II L_IM over L's blocks, then the block diagonals below, one
  // block per warp: T_IJ = -sum_{M=J}^{I-1} Lam_IM T_MJ.  In a block product
  // lane (r = lane / 2, c0 = 8 (lane % 2)) owns row r, columns c0 .. c0 + 7.
  if (tid < 128) {
    const int I = tid >> 4, cc = tid & 15;
    const float* Lb = Lp + blk(I, I);
    float* Tb = Tp + blk(I, I);
    float col[16];
#pragma unroll
    for (int r = 0; r < 16; ++r) {
      float acc = r == cc ? 1.f : 0.f;
      if (r > cc) {
#pragma unroll
        for (int m = 0; m < 16; ++m)
          if (m >= cc && m < r) acc = fmaf(-Lb[r * kBS + m], col[m], acc);
      }
      col[r] = acc;
      Tb[r * kBS + cc] = acc;
    }
  }
  __syncthreads();
  {
    const int r = lane >> 1, c0 = 8 * (lane & 1);
    // acc[x] += sum_k A[r][k] B[k][c0 + x] over one 16x16 block pair
    auto block_fma = [&](float* acc, const float* A, const float* B) {
#pragma unroll
      for (int k4 = 0; k4 < 4; ++k4) {
        const float4 a = *reinterpret_cast<const float4*>(A + r * kBS + 4 * k4);
        const float av[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const float4 b0 = *reinterpret_cast<const float4*>(B + (4 * k4 + kk) * kBS + c0);
          const float4 b1 = *reinterpret_cast<const float4*>(B + (4 * k4 + kk) * kBS + c0 + 4);
          acc[0] = fmaf(av[kk], b0.x, acc[0]); acc[1] = fmaf(av[kk], b0.y, acc[1]);
          acc[2] = fmaf(av[kk], b0.z, acc[2]); acc[3] = fmaf(av[kk], b0.w, acc[3]);
          acc[4] = fmaf(av[kk], b1.x, acc[4]); acc[5] = fmaf(av[kk], b1.y, acc[5]);
          acc[6] = fmaf(av[kk], b1.z, acc[6]); acc[7] = fmaf(av[kk], b1.w, acc[7]);
        }
      }
    };
    auto store_row = [&](float* dst, const float* acc, float sgn) {
      *reinterpret_cast<float4*>(dst + r * kBS + c0) = make_float4(sgn * acc[0], sgn * acc[1], sgn * acc[2], sgn * acc[3]);
      *reinterpret_cast<float4*>(dst + r * kBS + c0 + 4) =
          make_float4(sgn * acc[4], sgn * acc[5], sgn * acc[6], sgn * acc[7]);
    };
    // Lam_IM = T_II L_IM for the 28 blocks below the diagonal, in place of L_IM
    for (int b = warp; b < 28; b += kPrepThreads / 32) {
      int I = 1, M = b;
      while (M >= I) { M -= I; ++I; }  // b enumerates (I, M), M < I, row by row
      float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      block_fma(acc, Tp + blk(I, I), Lp + blk(I, M));
      __syncwarp();
      store_row(Lp + blk(I, M), acc, 1.f);
    }
    __syncthreads();
    for (int d = 1; d < 8; ++d) {
      if (warp < 8 - d) {
        const int J = warp, I = J + d;
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        for (int M = J; M < I; ++M) block_fma(acc, Lp + blk(I, M), Tp + blk(M, J));
        store_row(Tp + blk(I, J), acc, -1.f);
      }
      __syncthreads();
    }
  }

  // ---- Tb = Tinv diag(beta) (into L's space), Tbe = Tinv diag(beta e) (over Tinv)
  {
    float t[64];
#pragma unroll
    for (int jb = 0; jb < 4; ++jb) {
      const int I = i >> 4, J = 4 * hf + jb;
#pragma unroll
      for (int v = 0; v < 4; ++v) {
        float4 x4 = make_float4(0.f, 0.f, 0.f, 0.f);
        if (J <= I) x4 = *reinterpret_cast<const float4*>(Tp + blk(I, J) + (i & 15) * kBS + 4 * v);
        t[16 * jb + 4 * v] = x4.x;
        t[16 * jb + 4 * v + 1] = x4.y;
        t[16 * jb + 4 * v + 2] = x4.z;
        t[16 * jb + 4 * v + 3] = x4.w;
      }
    }
    __syncthreads();
#pragma unroll
    for (int c8 = 0; c8 < 8; ++c8) {
      uint32_t wb[4], we[4];
#pragma unroll
      for (int v = 0; v < 4; ++v) {
        const int j0 = 64 * hf + 8 * c8 + 2 * v;
        const float b0 = bs[j0], b1 = bs[j0 + 1];
        const float a0 = t[8 * c8 + 2 * v] * b0, a1 = t[8 * c8 + 2 * v + 1] * b1;
        wb[v] = pack_bf16x2(a0, a1);
        we[v] = pack_bf16x2(a0 * es[j0], a1 * es[j0 + 1]);
      }
      const uint32_t o = swz16(i, 8 * hf + c8);
      *reinterpret_cast<uint4*>(s + kPL + o) = make_uint4(wb[0], wb[1], wb[2], wb[3]);
      *reinterpret_cast<uint4*>(s + kPT + o) = make_uint4(we[0], we[1], we[2], we[3]);
    }
  }
  fence_proxy_async_shared();
  tc_fence_before();
  __syncthreads();
  // U^T = V^T Tb^T -> 0 (lanes = d_v), Cl = Aqk Tb -> 128, W = Tbe K -> 256
  if (tid == 0) {
    tc_fence_after();
    mma_128(tmem + 0, sV, true, sL, false, 0);
    if (!kB) mma_128(tmem + 128, sA, false, sL, true, 0);
    mma_128(tmem + 256, sT, false, sK, true, 0);
    umma_commit(bars + 1);
  }
  wait_bar(bars + 1, (pb + 1) & 1, p.err);
  __syncwarp();
  tc_fence_after();
  // W (bf16, into Tbe's space: the B operand of Aqk W and the stored W);
  // Cm = Cl . lambda-mask (bf16, into Tb's space); U^T staged in K's space
  {
    // the lambda of level bitlen(i ^ j) without indexing lam8 at run time
    // (which puts it in local memory): a 32-column block off the row's own
    // has one level, 6 or 7; inside the row's own block, column jj has level
    // bitlen((i ^ jj) & 31), picked by a tree of selects on the row's bits
    // (tk[m]: the columns whose low k + 1 bits are m)
    float t1[2], t2[4], t3[8], t4[16];
#pragma unroll
    for (int m = 0; m < 2; ++m) t1[m] = ((i & 1) != (m & 1)) ? lam8[1] : lam8[0];
#pragma unroll
    for (int m = 0; m < 4; ++m) t2[m] = ((i & 2) != (m & 2)) ? lam8[2] : t1[m & 1];
#pragma unroll
    for (int m = 0; m < 8; ++m) t3[m] = ((i & 4) != (m & 4)) ? lam8[3] : t2[m & 3];
#pragma unroll
    for (int m = 0; m < 16; ++m) t4[m] = ((i & 8) != (m & 8)) ? lam8[4] : t3[m & 7];
#pragma unroll
    for (int c32 = 0; c32 < 2; ++c32) {
      const int j0 = 64 * hf + 32 * c32;
      float w[32], cl[32], u[32];
      tmem_ld32(tl + 256 + j0, w);
      if (!kB) tmem_ld32(tl + 128 + j0, cl);
      tmem_ld32(tl + 0 + j0, u);
      tmem_ld_wait();
      const bool own = ((i ^ j0) >> 5) == 0;                // the row's own 32-column block
      const float lblk = ((i ^ j0) & 64) ? lam8[7] : lam8[6];  // another block: level 6 or 7
#pragma unroll
      for (int jj = 0; jj < 32; ++jj) {
        const int j = j0 + jj;
        const float lv = own ? (((i & 16) != (jj & 16)) ? lam8[5] : t4[jj & 15]) : lblk;
        cl[jj] = (!kB && j <= i) ? cl[jj] * lv : 0.f;
      }
#pragma unroll
      for (int c8 = 0; c8 < 4; ++c8) {
        const uint32_t o = swz16(i, (j0 >> 3) + c8);
        *reinterpret_cast<uint4*>(s + kPT + o) =
            make_uint4(pack_bf16x2(w[8 * c8], w[8 * c8 + 1]), pack_bf16x2(w[8 * c8 + 2], w[8 * c8 + 3]),
                       pack_bf16x2(w[8 * c8 + 4], w[8 * c8 + 5]), pack_bf16x2(w[8 * c8 + 6], w[8 * c8 + 7]));
        *reinterpret_cast<uint4*>(s + kPL + o) =
            make_uint4(pack_bf16x2(cl[8 * c8], cl[8 * c8 + 1]), pack_bf16x2(cl[8 * c8 + 2], cl[8 * c8 + 3]),
                       pack_bf16x2(cl[8 * c8 + 4], cl[8 * c8 + 5]), pack_bf16x2(cl[8 * c8 + 6], cl[8 * c8 + 7]));
      }
      // U^T: this thread's lane is d_v = i, its columns tokens j0 ..
#pragma unroll
      for (int c8 = 0; c8 < 4; ++c8)
        *reinterpret_cast<uint4*>(s + kPK + swz16(i, (j0 >> 3) + c8)) =
            make_uint4(pack_bf16x2(u[8 * c8], u[8 * c8 + 1]), pack_bf16x2(u[8 * c8 + 2], u[8 * c8 + 3]),
                       pack_bf16x2(u[8 * c8 + 4], u[8 * c8 + 5]), pack_bf16x2(u[8 * c8 + 6], u[8 * c8 + 7]));
    }
  }
  fence_proxy_async_shared();
  tc_fence_before();
  __syncthreads();
  // Q'' = Aqk W -> 0, intra = Cm V -> 128; store U^T and W
  if (tid == 0) {
    tc_fence_after();
    if (!kB) {
      mma_128(tmem + 0, sA, false, sT, true, 0);
      mma_128(tmem + 128, sL, false, sV, true, 0);
      umma_commit(bars + 1);
    }
    const int urow = (bh * p.Nc + c) * kD;
    tma_store_2d(&tut, s + kPK, 0, urow);
    tma_store_2d(&tut, s + kPK + kHalf, 64, urow);
    tma_store_2d(&tw, s + kPT, 0, row0);
    tma_store_2d(&tw, s + kPT + kHalf, 64, row0);
    bulk_commit();
  }
  if (kB) continue;  // reading B: U^T and W are all it needs
  wait_bar(bars + 1, (pb + 2) & 1, p.err);
  __syncwarp();
  tc_fence_after();
  // Q' = diag(e) Q - Aqk W (into Aqk's space), intra (into Cm's space)
  {
    const float ei = es[i];
#pragma unroll
    for (int c32 = 0; c32 < 2; ++c32) {
      const int j0 = 64 * hf + 32 * c32;
      float qq[32], oi[32];
      tmem_ld32(tl + 0 + j0, qq);
      tmem_ld32(tl + 128 + j0, oi);
      tmem_ld_wait();
#pragma unroll
      for (int c8 = 0; c8 < 4; ++c8) {
        const uint32_t o = swz16(i, (j0 >> 3) + c8);
        const uint4 qv = *reinterpret_cast<const uint4*>(s + kPQ + o);
        const uint32_t* qw = reinterpret_cast<const uint32_t*>(&qv);
        uint32_t wq[4], wo[4];
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          const float2 f = unpack_bf16x2(qw[v]);
          wq[v] = pack_bf16x2(ei * f.x - qq[8 * c8 + 2 * v], ei * f.y - qq[8 * c8 + 2 * v + 1]);
          wo[v] = pack_bf16x2(oi[8 * c8 + 2 * v], oi[8 * c8 + 2 * v + 1]);
        }
        *reinterpret_cast<uint4*>(s + kPA + o) = make_uint4(wq[0], wq[1], wq[2], wq[3]);
        *reinterpret_cast<uint4*>(s + kPL + o) = make_uint4(wo[0], wo[1], wo[2], wo[3]);
      }
    }
  }
  fence_proxy_async_shared();
  tc_fence_before();
  __syncthreads();
  if (tid == 0) {
    tma_store_2d(&tqp, s + kPA, 0, row0);
    tma_store_2d(&tqp, s + kPA + kHalf, 64, row0);
    tma_store_2d(&toi, s + kPL, 0, row0);
    tma_store_2d(&toi, s + kPL + kHalf, 64, row0);
    bulk_commit();
  }
  }  // items
  if (tid == 0) bulk_wait0();
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ------------------------------------------------------------------ kernel 2
constexpr uint32_t kSW = 0;                      // W of the chunk
constexpr uint32_t kSQ = kSW + kTileB;           // Q' of the chunk
constexpr uint32_t kSK = kSQ + kTileB;           // K (then Kt) x 2
constexpr uint32_t kSU = kSK + 2 * kTileB;       // U^T slice x 2
constexpr uint32_t kSX = kSU + 2 * kSliceB;      // X (then -Y) operands, four heights at a time
constexpr uint32_t kSTab = kSX + 4 * kSliceB;    // quadrant totals [4]
constexpr uint32_t kSBars = kSTab + 16;
constexpr uint32_t kScanSmem = kSBars + 8 * 8;
constexpr int kScanThreads = 128;
static_assert(kScanSmem <= 232448, "shared memory budget of one CTA");

enum ScanBar : int { SB_WQ = 0, SB_K0, SB_K1, SB_U0, SB_U1, SB_MMA, kScanBars };

struct ScanParams {
  const float* log_alpha;
  const float* lam;
  const __nv_bfloat16* oi;  // intra outputs [BH*T, 128]
  __nv_bfloat16* o;
  int T, L, Nc, nh;
  unsigned* err;
};

__global__ void __launch_bounds__(kScanThreads, 1)
    gdn_tc_scan_kernel(const __grid_constant__ CUtensorMap tw, const __grid_constant__ CUtensorMap tqp,
                       const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tu32,
                       ScanParams p) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  if (smem_u32(smem_raw) & 1023u) {
    if (threadIdx.x == 0) atomicOr(p.err, kErrDeviceArg);
    return;
  }
  unsigned char* s = smem_raw;
  const int tid = threadIdx.x, q = tid >> 5, lane = tid & 31;
  const int sl = blockIdx.x;  // d_v slice: rows 32 sl .. 32 sl + 31
  const int bh = blockIdx.y;
  float* qtot = reinterpret_cast<float*>(s + kSTab);
  uint64_t* bars = reinterpret_cast<uint64_t*>(s + kSBars);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(s + kSBars + kScanBars * 8);
  const uint32_t sW = smem_u32(s + kSW), sQ = smem_u32(s + kSQ);

  auto load_wq = [&](int c) {
    const int r = bh * p.T + c * kC;
    mbar_arrive_expect_tx(bars + SB_WQ, 2 * kTileB);
    tma_load_2d(s + kSW, &tw, bars + SB_WQ, 0, r);
    tma_load_2d(s + kSW + kHalf, &tw, bars + SB_WQ, 64, r);
    tma_load_2d(s + kSQ, &tqp, bars + SB_WQ, 0, r);
    tma_load_2d(s + kSQ + kHalf, &tqp, bars + SB_WQ, 64, r);
  };
  auto load_ku = [&](int c) {
    const int b = c & 1;
    const int r = bh * p.T + c * kC;
    unsigned char* kd = s + kSK + b * kTileB;
    mbar_arrive_expect_tx(bars + SB_K0 + b, kTileB);
    tma_load_2d(kd, &tk, bars + SB_K0 + b, 0, r);
    tma_load_2d(kd + kHalf, &tk, bars + SB_K0 + b, 64, r);
    unsigned char* ud = s + kSU + b * kSliceB;
    const int ur = (bh * p.Nc + c) * kD + kSlice * sl;
    mbar_arrive_expect_tx(bars + SB_U0 + b, kSliceB);
    tma_load_2d(ud, &tu32, bars + SB_U0 + b, 0, ur);
    tma_load_2d(ud + kHalf32, &tu32, bars + SB_U0 + b, 64, ur);
  };

  if (tid == 0) {
    for (int b = 0; b < kScanBars; ++b) mbar_init(bars + b, 1);
    fence_mbar_init();
    load_wq(0);
    load_ku(0);
    if (p.Nc > 1) load_ku(1);
  }
  __syncwarp();
  if (q == 0) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tl = tmem + ((uint32_t)(32 * q) << 16);
  constexpr uint32_t idY = idesc_bf16(128, kSlice, false, false);  // W (K) x X (K, N = 32)
  constexpr uint32_t idX = idesc_bf16(128, kSlice, true, false);   // Kt^T (MN) x -Y / U^T (K, N = 32)
  uint32_t nmma = 0;  // products committed (and waited for) so far

  auto commit_wait = [&]() {
    if (tid == 0) umma_commit(bars + SB_MMA);
    wait_bar(bars + SB_MMA, nmma & 1, p.err);
    ++nmma;
    __syncwarp();
    tc_fence_after();
  };

  // this token's log_alpha, intra output (bf16) and lambdas of the live
  // heights, loaded one chunk ahead
  float la_n;
  uint4 oiv_n[4];
  float lamh_n[kMaxHeights];
  auto fetch = [&](int c1) {
    const size_t r = (size_t)bh * p.T + (size_t)c1 * kC + tid;
    la_n = p.log_alpha[r];
    const uint4* oip = reinterpret_cast<const uint4*>(p.oi + r * kD + kSlice * sl);
#pragma unroll
    for (int v = 0; v < 4; ++v) oiv_n[v] = oip[v];
#pragma unroll
    for (int h = 0; h < kMaxHeights; ++h) lamh_n[h] = ((c1 >> h) & 1) ? p.lam[r * p.L + 8 + h] : 0.f;
  };
  fetch(0);

  for (int c = 0; c < p.Nc; ++c) {
    const int b = c & 1;
    const int row0 = bh * p.T + c * kC;
    const size_t rowt = (size_t)row0 + tid;  // this thread's token
    float x = la_n;
    uint4 oiv[4];
    float lamh[kMaxHeights];
#pragma unroll
    for (int v = 0; v < 4; ++v) oiv[v] = oiv_n[v];
#pragma unroll
    for (int h = 0; h < kMaxHeights; ++h) lamh[h] = lamh_n[h];
    if (c + 1 < p.Nc) fetch(c + 1);
    // cumulative log decay of the chunk
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) qtot[q] = x;
    __syncthreads();
    float off = 0.f;
    for (int qq = 0; qq < q; ++qq) off += qtot[qq];
    const float g_t = x + off;
    const float g_end = qtot[0] + qtot[1] + qtot[2] + qtot[3];
    const float gam = ex2(g_end * kLog2e);
    const float dec = ex2((g_end - g_t) * kLog2e);
    __syncthreads();  // qtot is rewritten by the next chunk

    // Kt = diag(exp(g_end - g)) K in place (row = this token)
    wait_bar(bars + SB_K0 + b, (c >> 1) & 1, p.err);
    unsigned char* kt = s + kSK + b * kTileB;
#pragma unroll
    for (int c8 = 0; c8 < 16; ++c8) {
      uint4 v = *reinterpret_cast<const uint4*>(kt + swz16(tid, c8));
      uint32_t* w = reinterpret_cast<uint32_t*>(&v);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 f = unpack_bf16x2(w[e]);
        w[e] = pack_bf16x2(f.x * dec, f.y * dec);
      }
      *reinterpret_cast<uint4*>(kt + swz16(tid, c8)) = v;
    }
    fence_proxy_async_shared();

    float oacc[kSlice];
#pragma unroll
    for (int r = 0; r < kSlice; ++r) oacc[r] = 0.f;
    const uint32_t sKt = smem_u32(kt);

    // live heights in groups of four
    wait_bar(bars + SB_WQ, c & 1, p.err);
    int hs = 0;
    bool wq_reloaded = false;
    while (true) {
      uint32_t grp = 0;  // the group's heights, 8 bits each (a packed word, not an array indexed at run time)
      int ng = 0;
      for (int h = hs; h < p.nh && ng < 4; ++h)
        if ((c >> h) & 1) {
          grp |= (uint32_t)h << (8 * ng++);
          hs = h + 1;
        }
      if (ng == 0) break;
      // (a) X_h as bf16 operand [32 rows d_v][128 d_k]; gamma X_h back into TMEM
      for (int g = 0; g < ng; ++g) {
        float xv[32];
        tmem_ld32(tl + 32 * ((grp >> (8 * g)) & 255u), xv);
        tmem_ld_wait();
        unsigned char* xb = s + kSX + g * kSliceB;
#pragma unroll
        for (int r = 0; r < kSlice; ++r)
          *reinterpret_cast<__nv_bfloat16*>(xb + swz_off(r, tid, kSlice)) = __float2bfloat16_rn(xv[r]);
        uint32_t wv[32];
#pragma unroll
        for (int r = 0; r < 32; ++r) wv[r] = __float_as_uint(gam * xv[r]);
        tmem_st32(tl + 32 * ((grp >> (8 * g)) & 255u), wv);
      }
      tmem_st_wait();
      fence_proxy_async_shared();
      tc_fence_before();
      __syncthreads();
      if (tid == 0) {
        tc_fence_after();
        for (int g = 0; g < ng; ++g) {
          const uint32_t xb = smem_u32(s + kSX + g * kSliceB);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            umma_bf16(tmem + 256 + 64 * g, desc_k(sW, kk), desc_k32(xb, kk), idY, kk > 0);
            umma_bf16(tmem + 256 + 64 * g + 32, desc_k(sQ, kk), desc_k32(xb, kk), idY, kk > 0);
          }
        }
      }
      commit_wait();
      // (b) -Y as bf16 operand [32 rows d_v][128 tokens]; lambda-weighted Pq into the output
      for (int g = 0; g < ng; ++g) {
        float yv[32], pv[32];
        tmem_ld32(tl + 256 + 64 * g, yv);
        tmem_ld32(tl + 256 + 64 * g + 32, pv);
        tmem_ld_wait();
        unsigned char* yb = s + kSX + g * kSliceB;
#pragma unroll
        for (int r = 0; r < kSlice; ++r)
          *reinterpret_cast<__nv_bfloat16*>(yb + swz_off(r, tid, kSlice)) = __float2bfloat16_rn(-yv[r]);
        float lw = 0.f;
#pragma unroll
        for (int h = 0; h < kMaxHeights; ++h)
          if (h == (int)((grp >> (8 * g)) & 255u)) lw = lamh[h];
#pragma unroll
        for (int r = 0; r < kSlice; ++r) oacc[r] = fmaf(lw, pv[r], oacc[r]);
      }
      fence_proxy_async_shared();
      tc_fence_before();
      __syncthreads();
      if (tid == 0) {
        tc_fence_after();
        const bool last = hs >= p.nh || (c >> hs) == 0;
        if (last && c + 1 < p.Nc) {  // the products have read W and Q': the next chunk's load
          load_wq(c + 1);
        }
        for (int g = 0; g < ng; ++g) {
          const uint32_t yb = smem_u32(s + kSX + g * kSliceB);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) umma_bf16(tmem + 32 * ((grp >> (8 * g)) & 255u), desc_mn(sKt, kk), desc_k32(yb, kk), idX, 1);
        }
      }
      if (hs >= p.nh || (c >> hs) == 0) wq_reloaded = true;
      commit_wait();
    }
    if (!wq_reloaded) {  // no live height: W and Q' of this chunk were not used
      __syncthreads();
      if (tid == 0 && c + 1 < p.Nc) load_wq(c + 1);
    }

    // output rows of this chunk, d_v slice
    {
      uint4 ov[4];
#pragma unroll
      for (int v = 0; v < 4; ++v) {
        const uint32_t* iw = reinterpret_cast<const uint32_t*>(&oiv[v]);
        uint32_t* ow = reinterpret_cast<uint32_t*>(&ov[v]);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 f = unpack_bf16x2(iw[e]);
          ow[e] = pack_bf16x2(f.x + oacc[8 * v + 2 * e], f.y + oacc[8 * v + 2 * e + 1]);
        }
      }
      uint4* op = reinterpret_cast<uint4*>(p.o + rowt * kD + kSlice * sl);
#pragma unroll
      for (int v = 0; v < 4; ++v) op[v] = ov[v];
    }

    // carry into height cto(c): the transported heights below it plus S_c = U^T Kt
    int t = 0;
    while ((c >> t) & 1) ++t;
    if (t < p.nh && c + 1 < p.Nc) {
      if (t > 0) {
        float sum[32];
        tmem_ld32(tl + 0, sum);
        tmem_ld_wait();
        for (int h = 1; h < t; ++h) {
          float xv[32];
          tmem_ld32(tl + 32 * h, xv);
          tmem_ld_wait();
#pragma unroll
          for (int r = 0; r < 32; ++r) sum[r] += xv[r];
        }
        uint32_t wv[32];
#pragma unroll
        for (int r = 0; r < 32; ++r) wv[r] = __float_as_uint(sum[r]);
        tmem_st32(tl + 32 * t, wv);
        tmem_st_wait();
      }
      tc_fence_before();
      __syncthreads();
      wait_bar(bars + SB_U0 + b, (c >> 1) & 1, p.err);
      if (tid == 0) {
        tc_fence_after();
        const uint32_t ub = smem_u32(s + kSU + b * kSliceB);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          umma_bf16(tmem + 32 * t, desc_mn(sKt, kk), desc_k32(ub, kk), idX, (t > 0 || kk > 0) ? 1u : 0u);
      }
      commit_wait();
    } else {
      // the U^T slice of this chunk is not needed; its copy has to land before reuse
      wait_bar(bars + SB_U0 + b, (c >> 1) & 1, p.err);
      __syncthreads();
    }
    // K and U^T buffers of this chunk are free: the chunk after next
    if (tid == 0 && c + 2 < p.Nc) load_ku(c + 2);
  }
  tc_fence_before();
  __syncthreads();
  if (q == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ------------------------------------------------------------------ kernel 2, reading B
// Reading B (log-linear Mamba-2 on the delta rule's pseudo-values) needs one
// gated-delta state and no levels: per chunk, with X the state at the chunk
// start (X = 0 for the first chunk),
//   U_c = U - W X^T            (the pseudo-values, written in bf16)
//   X^T <- gamma X^T + Kt^T U_c^T
// with U, W from the preparation above and Kt = diag(exp(g_end - g)) K.  The
// layout is the level scan's: one CTA per (32 d_v rows, head), X^T in TMEM
// columns 0..31, Y^T = W X^T in columns 256..287, U_c built in place of the
// chunk's U^T slice (thread = token) and used there as the update's operand.
__global__ void __launch_bounds__(kScanThreads, 1)
    gdn_tc_scan_b_kernel(const __grid_constant__ CUtensorMap tw, const __grid_constant__ CUtensorMap tk,
                         const __grid_constant__ CUtensorMap tu32, const float* __restrict__ log_alpha,
                         __nv_bfloat16* __restrict__ uc_out, int T, int Nc, unsigned* err) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  if (smem_u32(smem_raw) & 1023u) {
    if (threadIdx.x == 0) atomicOr(err, kErrDeviceArg);
    return;
  }
  unsigned char* s = smem_raw;
  const int tid = threadIdx.x, q = tid >> 5, lane = tid & 31;
  const int sl = blockIdx.x;  // d_v slice: rows 32 sl .. 32 sl + 31
  const int bh = blockIdx.y;
  float* qtot = reinterpret_cast<float*>(s + kSTab);
  uint64_t* bars = reinterpret_cast<uint64_t*>(s + kSBars);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(s + kSBars + kScanBars * 8);
  const uint32_t sW = smem_u32(s + kSW);

  auto load_w = [&](int c) {
    const int r = bh * T + c * kC;
    mbar_arrive_expect_tx(bars + SB_WQ, kTileB);
    tma_load_2d(s + kSW, &tw, bars + SB_WQ, 0, r);
    tma_load_2d(s + kSW + kHalf, &tw, bars + SB_WQ, 64, r);
  };
  auto load_ku = [&](int c) {
    const int b = c & 1;
    const int r = bh * T + c * kC;
    unsigned char* kd = s + kSK + b * kTileB;
    mbar_arrive_expect_tx(bars + SB_K0 + b, kTileB);
    tma_load_2d(kd, &tk, bars + SB_K0 + b, 0, r);
    tma_load_2d(kd + kHalf, &tk, bars + SB_K0 + b, 64, r);
    unsigned char* ud = s + kSU + b * kSliceB;
    const int ur = (bh * Nc + c) * kD + kSlice * sl;
    mbar_arrive_expect_tx(bars + SB_U0 + b, kSliceB);
    tma_load_2d(ud, &tu32, bars + SB_U0 + b, 0, ur);
    tma_load_2d(ud + kHalf32, &tu32, bars + SB_U0 + b, 64, ur);
  };

  if (tid == 0) {
    for (int b = 0; b < kScanBars; ++b) mbar_init(bars + b, 1);
    fence_mbar_init();
    if (Nc > 1) load_w(1);  // the first chunk reads no W (its state is zero)
    load_ku(0);
    if (Nc > 1) load_ku(1);
  }
  __syncwarp();
  if (q == 0) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tl = tmem + ((uint32_t)(32 * q) << 16);
  constexpr uint32_t idY = idesc_bf16(128, kSlice, false, false);  // W (K) x X (K, N = 32)
  constexpr uint32_t idX = idesc_bf16(128, kSlice, true, false);   // Kt^T (MN) x U_c (K, N = 32)
  uint32_t nmma = 0;
  auto commit_wait = [&]() {
    if (tid == 0) umma_commit(bars + SB_MMA);
    wait_bar(bars + SB_MMA, nmma & 1, err);
    ++nmma;
    __syncwarp();
    tc_fence_after();
  };

  float la_n = log_alpha[(size_t)bh * T + tid];
  uint32_t nw = 0;  // W loads waited for
  for (int c = 0; c < Nc; ++c) {
    const int b = c & 1;
    const size_t rowt = (size_t)bh * T + (size_t)c * kC + tid;  // this thread's token
    float x = la_n;
    if (c + 1 < Nc) la_n = log_alpha[rowt + kC];
    // cumulative log decay of the chunk
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) qtot[q] = x;
    __syncthreads();
    float off = 0.f;
    for (int qq = 0; qq < q; ++qq) off += qtot[qq];
    const float g_t = x + off;
    const float g_end = qtot[0] + qtot[1] + qtot[2] + qtot[3];
    const float gam = ex2(g_end * kLog2e);
    const float dec = ex2((g_end - g_t) * kLog2e);
    __syncthreads();  // qtot is rewritten by the next chunk

    // Kt = diag(exp(g_end - g)) K in place (row = this token)
    wait_bar(bars + SB_K0 + b, (c >> 1) & 1, err);
    unsigned char* kt = s + kSK + b * kTileB;
#pragma unroll
    for (int c8 = 0; c8 < 16; ++c8) {
      uint4 v = *reinterpret_cast<const uint4*>(kt + swz16(tid, c8));
      uint32_t* w = reinterpret_cast<uint32_t*>(&v);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 f = unpack_bf16x2(w[e]);
        w[e] = pack_bf16x2(f.x * dec, f.y * dec);
      }
      *reinterpret_cast<uint4*>(kt + swz16(tid, c8)) = v;
    }
    const uint32_t sKt = smem_u32(kt);

    float yv[kSlice];
#pragma unroll
    for (int r = 0; r < kSlice; ++r) yv[r] = 0.f;
    if (c > 0) {
      // X as bf16 operand [32 rows d_v][128 d_k]; gamma X back into TMEM; Y^T = W X^T
      float xv[32];
      tmem_ld32(tl, xv);
      tmem_ld_wait();
      unsigned char* xb = s + kSX;
#pragma unroll
      for (int r = 0; r < kSlice; ++r)
        *reinterpret_cast<__nv_bfloat16*>(xb + swz_off(r, tid, kSlice)) = __float2bfloat16_rn(xv[r]);
      uint32_t wv[32];
#pragma unroll
      for (int r = 0; r < 32; ++r) wv[r] = __float_as_uint(gam * xv[r]);
      tmem_st32(tl, wv);
      tmem_st_wait();
      wait_bar(bars + SB_WQ, nw & 1, err);
      ++nw;
      fence_proxy_async_shared();
      tc_fence_before();
      __syncthreads();
      if (tid == 0) {
        tc_fence_after();
        const uint32_t xbs = smem_u32(xb);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) umma_bf16(tmem + 256, desc_k(sW, kk), desc_k32(xbs, kk), idY, kk > 0);
      }
      commit_wait();
      if (tid == 0 && c + 1 < Nc) load_w(c + 1);  // the Y product has read W
      tmem_ld32(tl + 256, yv);
      tmem_ld_wait();
    } else {
      fence_proxy_async_shared();  // (the Kt writes, before the update product reads them)
    }
    // U_c = U - Y (row = this token, 32 d_v): in place of the U^T slice, and out
    wait_bar(bars + SB_U0 + b, (c >> 1) & 1, err);
    unsigned char* ub = s + kSU + b * kSliceB;
    uint32_t pk[kSlice / 2];
#pragma unroll
    for (int r = 0; r < kSlice; r += 2) {
      __nv_bfloat16* e0 = reinterpret_cast<__nv_bfloat16*>(ub + swz_off(r, tid, kSlice));
      __nv_bfloat16* e1 = reinterpret_cast<__nv_bfloat16*>(ub + swz_off(r + 1, tid, kSlice));
      const __nv_bfloat16 u0 = __float2bfloat16_rn(__bfloat162float(*e0) - yv[r]);
      const __nv_bfloat16 u1 = __float2bfloat16_rn(__bfloat162float(*e1) - yv[r + 1]);
      *e0 = u0;
      *e1 = u1;
      pk[r / 2] = (uint32_t)__bfloat16_as_ushort(u0) | ((uint32_t)__bfloat16_as_ushort(u1) << 16);
    }
    {
      uint4* op = reinterpret_cast<uint4*>(uc_out + rowt * kD + kSlice * sl);
#pragma unroll
      for (int v = 0; v < 4; ++v) op[v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
    }
    if (c + 1 < Nc) {
      // X^T <- gamma X^T + Kt^T U_c^T (the first chunk: Kt^T U^T)
      fence_proxy_async_shared();
      tc_fence_before();
      __syncthreads();
      if (tid == 0) {
        tc_fence_after();
        const uint32_t ubs = smem_u32(ub);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          umma_bf16(tmem, desc_mn(sKt, kk), desc_k32(ubs, kk), idX, (c > 0 || kk > 0) ? 1u : 0u);
      }
      commit_wait();
    } else {
      __syncthreads();
    }
    // K and U^T buffers of this chunk are free: the chunk after next
    if (tid == 0 && c + 2 < Nc) load_ku(c + 2);
  }
  tc_fence_before();
  __syncthreads();
  if (q == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ------------------------------------------------------------------ host side
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::atomic<bool> tried{false};
  if (!fn && !tried.exchange(true)) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult qr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &qr) ==
            cudaSuccess &&
        qr == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  return fn;
}

// 2-D bf16 tensor map over [rows, 128] with [box_rows x 64] boxes, 128-byte swizzle.
bool make_map(CUtensorMap* m, const void* base, uint64_t rows, uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)kD, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)kD * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// CTAs of the persistent preparation: one per SM (its shared memory allows
// no second), at most one per item.
cudaError_t prep_blocks(int items, int* grid) {
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  *grid = std::max(1, std::min(items, sms));
  return e;
}

int heights_of(int Nc) {
  int h = 0;
  while ((1 << h) < Nc) ++h;  // bit_length(Nc - 1)
  return h;
}

struct TcPlan {
  int Nc, nh;
  size_t off_W, off_Qp, off_Ut, off_Oi, total;
};

TcPlan tc_plan(const ll_shape& s) {
  TcPlan p{};
  p.Nc = s.T / kC;
  p.nh = heights_of(p.Nc);
  const size_t rows = (size_t)s.B * s.H * s.T;
  size_t off = 0;
  p.off_W = off;  off = align_up(off + rows * kD * 2, 1024);
  p.off_Qp = off; off = align_up(off + rows * kD * 2, 1024);
  p.off_Ut = off; off = align_up(off + rows * kD * 2, 1024);
  p.off_Oi = off; off = align_up(off + rows * kD * 2, 1024);
  p.total = off;
  return p;
}

}  // namespace

// Reading B on the tensor cores: the preparation, the single-state scan into
// the pseudo-values (bf16, after the preparation's buffers), then the
// log-linear Mamba-2 forward on them (its workspace after that).
static size_t b_uc_bytes(const ll_shape& s) { return align_up((size_t)s.B * s.H * s.T * kD * 2, 1024); }

bool gdn_tc_supported(const ll_shape& s) {
  return s.io == LL_BF16 && s.dk == kD && s.dv == kD && s.T % kC == 0 && s.T / kC <= (1 << kMaxHeights) &&
         (long long)s.B * s.H * s.T <= (1ll << 31) - 1;
}

size_t gdn_tc_workspace(const ll_shape& s) { return tc_plan(s).total; }

ll_status gdn_tc_launch(const FwdArgs& a) {
  const ll_shape& s = a.s;
  const TcPlan plan = tc_plan(s);
  if (a.ws_bytes < plan.total) return LL_ERR_WORKSPACE;
  unsigned char* ws = static_cast<unsigned char*>(a.ws);
  const int BH = s.B * s.H;
  const uint64_t rows = (uint64_t)BH * s.T;
  CUtensorMap tq, tk, tv, tw, tqp, tut, toi, tu32;
  if (!make_map(&tq, a.q, rows, kC) || !make_map(&tk, a.k, rows, kC) || !make_map(&tv, a.v, rows, kC) ||
      !make_map(&tw, ws + plan.off_W, rows, kC) || !make_map(&tqp, ws + plan.off_Qp, rows, kC) ||
      !make_map(&tut, ws + plan.off_Ut, rows, kC) || !make_map(&toi, ws + plan.off_Oi, rows, kC) ||
      !make_map(&tu32, ws + plan.off_Ut, rows, kSlice))
    return LL_ERR_CUDA;

  PrepParams pp{a.log_alpha, a.beta, a.lam, s.T, s.L, plan.Nc, a.err, static_cast<const __nv_bfloat16*>(a.q),
                static_cast<const __nv_bfloat16*>(a.k), static_cast<const __nv_bfloat16*>(a.v), BH};
  LL_CUDA_OK(cudaFuncSetAttribute(gdn_tc_prep_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)kPrepSmem));
  int prep_grid = 0;
  LL_CUDA_OK(prep_blocks(plan.Nc * BH, &prep_grid));
  gdn_tc_prep_kernel<false><<<prep_grid, kPrepThreads, kPrepSmem, a.stream>>>(tq, tk, tv, tw, tqp, tut, toi, pp);
  LL_CUDA_OK(cudaGetLastError());

  ScanParams sp{a.log_alpha, a.lam, reinterpret_cast<const __nv_bfloat16*>(ws + plan.off_Oi),
                static_cast<__nv_bfloat16*>(a.o), s.T, s.L, plan.Nc, plan.nh, a.err};
  LL_CUDA_OK(cudaFuncSetAttribute(gdn_tc_scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kScanSmem));
  gdn_tc_scan_kernel<<<dim3(kD / kSlice, BH), kScanThreads, kScanSmem, a.stream>>>(tw, tqp, tk, tu32, sp);
  LL_CUDA_OK(cudaGetLastError());
  return LL_OK;
}

size_t gdn_tc_b_workspace(const ll_shape& s) {
  return tc_plan(s).total + b_uc_bytes(s) + (fwd_tc_supported(s) ? fwd_tc_workspace(s) : 0);
}

ll_status gdn_tc_b_launch(const FwdArgs& a) {
  const ll_shape& s = a.s;
  if (!fwd_tc_supported(s)) return LL_ERR_UNSUPPORTED;
  const TcPlan plan = tc_plan(s);
  if (a.ws_bytes < gdn_tc_b_workspace(s)) return LL_ERR_WORKSPACE;
  unsigned char* ws = static_cast<unsigned char*>(a.ws);
  const int BH = s.B * s.H;
  const uint64_t rows = (uint64_t)BH * s.T;
  __nv_bfloat16* uc = reinterpret_cast<__nv_bfloat16*>(ws + plan.total);
  CUtensorMap tq, tk, tv, tw, tqp, tut, toi, tu32;
  if (!make_map(&tq, a.q, rows, kC) || !make_map(&tk, a.k, rows, kC) || !make_map(&tv, a.v, rows, kC) ||
      !make_map(&tw, ws + plan.off_W, rows, kC) || !make_map(&tqp, ws + plan.off_Qp, rows, kC) ||
      !make_map(&tut, ws + plan.off_Ut, rows, kC) || !make_map(&toi, ws + plan.off_Oi, rows, kC) ||
      !make_map(&tu32, ws + plan.off_Ut, rows, kSlice))
    return LL_ERR_CUDA;
  PrepParams pp{a.log_alpha, a.beta, a.lam, s.T, s.L, plan.Nc, a.err, static_cast<const __nv_bfloat16*>(a.q),
                static_cast<const __nv_bfloat16*>(a.k), static_cast<const __nv_bfloat16*>(a.v), BH};
  LL_CUDA_OK(cudaFuncSetAttribute(gdn_tc_prep_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)kPrepSmem));
  int prep_grid = 0;
  LL_CUDA_OK(prep_blocks(plan.Nc * BH, &prep_grid));
  gdn_tc_prep_kernel<true><<<prep_grid, kPrepThreads, kPrepSmem, a.stream>>>(tq, tk, tv, tw, tqp, tut, toi, pp);
  LL_CUDA_OK(cudaGetLastError());
  LL_CUDA_OK(cudaFuncSetAttribute(gdn_tc_scan_b_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kScanSmem));
  gdn_tc_scan_b_kernel<<<dim3(kD / kSlice, BH), kScanThreads, kScanSmem, a.stream>>>(tw, tk, tu32, a.log_alpha, uc,
                                                                                      s.T, plan.Nc, a.err);
  LL_CUDA_OK(cudaGetLastError());
  FwdArgs f = a;
  f.v = uc;
  f.beta = nullptr;
  f.state_out = nullptr;
  f.scale_out = nullptr;
  f.ws = ws + plan.total + b_uc_bytes(s);
  f.ws_bytes = fwd_tc_workspace(s);
  return fwd_tc_launch(f);
}

}  // namespace llattn
