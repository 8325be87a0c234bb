// Backward of the log-linear Mamba-2 forward on the tensor cores (bf16 io,
// d_k = d_v = 128): the chunk-wise algorithm of the CUDA-core backward with
// 128-token tiles and every product a tcgen05.mma (bf16 operands staged in
// 128-byte-swizzled shared memory, float32 accumulators in TMEM).
//
// Gradient of O = (Q K^T . M) V ("Log-Linear Attention" study note §3-4
// parallel form, §3-5 mask composition), per tile c of 128 tokens:
//   intra : A = Q K^T and G = dO V^T (TMEM); per row i the epilogue forms
//           P = A . M and dA = G . M (bf16 tiles) and the levels 0..7 of
//           dlam_i = sum over keys of level l of G A Gamma; then
//           dq = dA K, dk = dA^T Q, dv = P^T dO and the chunk state
//           S_c = (exp(cs_end - cs) V)^T K.  The in-tile part of v_j . dv_j
//           (for dc_j) is the column sum of P . G, taken in float32 from the
//           accumulators rather than from the bf16-rounded P: dc_j is a
//           difference of two terms of the size of do . o, so their rounding
//           would not cancel.
//   query : for every set bit h of c (node e, level 8 + h, decay D from the
//           end of e to the start of c; w_i = exp(cs_i + D), lw_i = lam_i w_i):
//           g = dO F_e (dlam_i = w_i g_i . q_i), dq += diag(lw) dO F_e = lw g
//           (from the float32 g, into a TMEM accumulator) and
//           R_e += (diag(lw) dO)^T Q, the key-side node of e (staged in shared
//           memory and added into R_e by tensor reductions; a first-level node
//           has this one query tile, which stores it).
//   key   : E_c = the R nodes of the blocks that hold c's keys, decayed to the
//           end of c; dv += diag(wdec) K E^T, dk += diag(wdec) V E, and
//           dc_j = sum_l lam_j[l] dlam_j[l] - v_j . dv_j (the in-tile part of
//           v_j . dv_j from the intra kernel).
// The Fenwick nodes F_e (with a bf16 tile copy of each, which the query
// kernel fetches by one bulk copy) and the suffix sums of dc are the
// CUDA-core kernels'.
//
// Thread t owns TMEM lane t mod 128 (row t mod 128 of every accumulator).
// The intra and query kernels are persistent, one CTA of 256 threads per SM
// over the (tile, head) items (the two threads of a row taking one half of its
// columns each); the key kernel runs one CTA of 128 threads per item, two per
// SM.  Full input tiles arrive by TMA (the ragged last tile of a head is
// staged by the threads, its missing rows as zeros).  The phases of a tile run
// in sequence: stage the operands, one thread issues the MMAs and commits them
// to an mbarrier, every thread waits (bounded: after 4 s the error word is set
// and the kernel finishes without the results), then the row-wise epilogue,
// whose tiles leave by tensor stores (or reductions) of swizzled staged boxes
// (row-wise bulk copies for a ragged tile).
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>

#include "bwd.cuh"
#include "sm100.cuh"

namespace llattn {

namespace {

using namespace sm100;

constexpr int kT = 128;                        // tokens per tile
constexpr int kD = 128;
constexpr int kThreads = 128;
constexpr uint32_t kHalf = kT * 64 * 2;        // a [128 x 64] bf16 swizzled block
constexpr uint32_t kTileB = 2 * kHalf;         // a [128 x 128] bf16 tile: 32 KB
constexpr uint64_t kTimeoutNs = 4000000000ull;
constexpr int kLc = 7;                         // log2 of the tile

// Element-wise float32 add of a contiguous shared-memory range into global
// memory by the bulk-copy unit (16-byte aligned addresses, size a multiple of
// 16); completion is tracked by the issuing thread's bulk groups.
__device__ __forceinline__ void bulk_reduce_add_f32(void* dst, const void* src, uint32_t bytes) {
  asm volatile("cp.reduce.async.bulk.global.shared::cta.bulk_group.add.f32 [%0], [%1], %2;" ::"l"(dst),
               "r"(smem_u32(src)), "r"(bytes)
               : "memory");
}

// Element-wise float32 add of one [128 x 32] box (128-byte swizzle) from shared
// memory into a [rows, 128] float32 tensor at column x, row y, by the TMA;
// tracked by the issuing thread's bulk groups.
__device__ __forceinline__ void tma_reduce_add_box(const CUtensorMap* map, const void* src, int x, int y) {
  asm volatile("cp.reduce.async.bulk.tensor.2d.global.shared::cta.add.tile.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(smem_u32(src)), "r"(x), "r"(y)
               : "memory");
}

// Bulk copy of a contiguous shared-memory range to global memory (16-byte
// aligned addresses, size a multiple of 16), tracked by the thread's bulk groups.
__device__ __forceinline__ void bulk_store(void* dst, const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(smem_u32(src)),
               "r"(bytes)
               : "memory");
}

constexpr int kRowP = kD + 4;  // float pitch of rows staged for bulk copies (conflict-free row writes)
// one [128 x 32] float32 box (128-byte swizzle) of a staged float32 tile: 16 KB
constexpr uint32_t kRBox = kT * 32 * 4;
static_assert(4 * kRBox <= kT * kRowP * 4, "a swizzled float32 tile fits the row staging's space");

// byte offset of the 16-byte chunk c8 (elements 8 c8 .. 8 c8 + 7) of row r of a tile
__device__ __forceinline__ uint32_t swz(int r, int c8) {
  return (uint32_t)(c8 >> 3) * kHalf + (uint32_t)r * 128u + ((uint32_t)((c8 & 7) ^ (r & 7)) << 4);
}
// K-major operand (K along the tile's columns), k-step kk of 16
__device__ __forceinline__ uint64_t desc_k(uint32_t tile, int kk) {
  return sw128_desc(tile + (kk >> 2) * kHalf + (kk & 3) * 32, 16, 1024);
}
// MN-major operand (K along the tile's rows), k-step kk of 16 rows
__device__ __forceinline__ uint64_t desc_mn(uint32_t tile, int kk) { return sw128_desc(tile + kk * 2048, kHalf, 1024); }

// D (+)= A B over K = 128
__device__ __forceinline__ void mma128(uint32_t d, uint32_t a, bool a_mn, uint32_t b, bool b_mn, bool acc) {
  const uint32_t id = idesc_bf16(128, 128, a_mn, b_mn);
#pragma unroll
  for (int kk = 0; kk < 8; ++kk)
    umma_bf16(d, a_mn ? desc_mn(a, kk) : desc_k(a, kk), b_mn ? desc_mn(b, kk) : desc_k(b, kk), id,
              (acc || kk > 0) ? 1u : 0u);
}

// Bounded wait of every thread for the phase with parity `par`; false after a timeout.
__device__ __forceinline__ bool wait_phase(uint64_t* bar, uint32_t par, unsigned* err, int* abort_s) {
  if (mbar_try_wait(bar, par)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, par)) {
    if (*(volatile int*)abort_s) return false;
    if (globaltimer_ns() - t0 > kTimeoutNs) {
      if (atomicExch(abort_s, 1) == 0) raise_error(err, kErrTimeout);
      return false;
    }
  }
  return true;
}

// a [128][128] bf16 tile of rows [0, nv) from global (rows of 256 B) into a swizzled tile; rows >= nv are 0
// (all 16 loads of a thread are issued before its stores: the staging is latency-bound)
__device__ __forceinline__ void stage_bf16(unsigned char* tile, const __nv_bfloat16* src, int nv, int tid) {
  uint4 v[16];
#pragma unroll
  for (int u = 0; u < 16; ++u) {
    const int x = tid + u * kThreads, r = x >> 4, c8 = x & 15;
    v[u] = r < nv ? *reinterpret_cast<const uint4*>(src + (size_t)r * kD + 8 * c8) : make_uint4(0u, 0u, 0u, 0u);
  }
#pragma unroll
  for (int u = 0; u < 16; ++u) {
    const int x = tid + u * kThreads, r = x >> 4, c8 = x & 15;
    *reinterpret_cast<uint4*>(tile + swz(r, c8)) = v[u];
  }
}

// sum_m coef[m] * src_m (float32 [128][128] matrices) as a bf16 swizzled tile
// (eight chunks of a thread at a time, their loads issued together)
__device__ __forceinline__ void stage_f32_sum(unsigned char* tile, const float* const* src, const float* coef, int n,
                                              int tid) {
#pragma unroll 1
  for (int pass = 0; pass < 2; ++pass) {
    float a[8][8];
#pragma unroll
    for (int q = 0; q < 8; ++q)
#pragma unroll
      for (int t = 0; t < 8; ++t) a[q][t] = 0.f;
    // node m's part of the pass, loaded one node ahead of its use (two
    // register buffers, the nodes taken in pairs)
    auto load = [&](float4 (&u)[8][2], int m) {
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const int x = tid + (8 * pass + q) * kThreads, r = x >> 4, c8 = x & 15;
        u[q][0] = *reinterpret_cast<const float4*>(src[m] + r * kD + 8 * c8);
        u[q][1] = *reinterpret_cast<const float4*>(src[m] + r * kD + 8 * c8 + 4);
      }
    };
    auto add = [&](const float4 (&u)[8][2], float cf) {
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        a[q][0] = fmaf(cf, u[q][0].x, a[q][0]); a[q][1] = fmaf(cf, u[q][0].y, a[q][1]);
        a[q][2] = fmaf(cf, u[q][0].z, a[q][2]); a[q][3] = fmaf(cf, u[q][0].w, a[q][3]);
        a[q][4] = fmaf(cf, u[q][1].x, a[q][4]); a[q][5] = fmaf(cf, u[q][1].y, a[q][5]);
        a[q][6] = fmaf(cf, u[q][1].z, a[q][6]); a[q][7] = fmaf(cf, u[q][1].w, a[q][7]);
      }
    };
    float4 ua[8][2], ub[8][2];
    load(ua, 0);
#pragma unroll 1
    for (int m = 0; m < n; m += 2) {
      if (m + 1 < n) load(ub, m + 1);
      add(ua, coef[m]);
      if (m + 2 < n) load(ua, m + 2);
      if (m + 1 < n) add(ub, coef[m + 1]);
    }
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const int x = tid + (8 * pass + q) * kThreads, r = x >> 4, c8 = x & 15;
      *reinterpret_cast<uint4*>(tile + swz(r, c8)) =
          make_uint4(pack_bf16x2(a[q][0], a[q][1]), pack_bf16x2(a[q][2], a[q][3]), pack_bf16x2(a[q][4], a[q][5]),
                     pack_bf16x2(a[q][6], a[q][7]));
    }
  }
}

// row r of a swizzled tile, 8 elements of chunk c8, as floats
// 8 bf16 of a 16-byte word as floats
__device__ __forceinline__ void unpack8(const uint4& u, float* x) {
  const float2 a = unpack_bf16x2(u.x), b = unpack_bf16x2(u.y), c = unpack_bf16x2(u.z), d = unpack_bf16x2(u.w);
  x[0] = a.x; x[1] = a.y; x[2] = b.x; x[3] = b.y; x[4] = c.x; x[5] = c.y; x[6] = d.x; x[7] = d.y;
}

__device__ __forceinline__ void row_chunk(const unsigned char* tile, int r, int c8, float* x) {
  const uint4 u = *reinterpret_cast<const uint4*>(tile + swz(r, c8));
  const float2 a = unpack_bf16x2(u.x), b = unpack_bf16x2(u.y), c = unpack_bf16x2(u.z), d = unpack_bf16x2(u.w);
  x[0] = a.x; x[1] = a.y; x[2] = b.x; x[3] = b.y; x[4] = c.x; x[5] = c.y; x[6] = d.x; x[7] = d.y;
}

// this thread's log_alpha of the tile (threads 0..127: rows; 0 past the tile's nv rows and for the other threads)
__device__ __forceinline__ double tile_log_alpha(const float* log_alpha, size_t row0, int nv) {
  const int t = threadIdx.x;
  return (t < kT && t < nv) ? (double)log_alpha[row0 + t] : 0.0;
}

// cs[i] = x_0 + .. + x_i for the values x of tile_log_alpha, float64; every
// thread takes part (a scan over each warp, then the warps' totals); the
// caller synchronises before reading cs
__device__ __forceinline__ void tile_scan(double* cs, double x) {
  __shared__ double wsum[8];  // the warps of the tile's rows (threads past 128 only synchronise)
  const int t = threadIdx.x, lane = t & 31, w = t >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const double y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31 && w < 8) wsum[w] = x;
  __syncthreads();
  if (t < kT) {
    for (int ww = 0; ww < w; ++ww) x += wsum[ww];
    cs[t] = x;
  }
}

// cs[i] = the sum of log_alpha over rows 0..i of the tile (rows >= nv add 0)
__device__ __forceinline__ void tile_cumsum(double* cs, const float* log_alpha, size_t row0, int nv) {
  tile_scan(cs, tile_log_alpha(log_alpha, row0, nv));
}

// L2 prefetch of the 16-byte-aligned interior of [ptr, ptr + bytes) (a bulk
// prefetch needs a 16-byte-aligned start and size, which rows of log_alpha and
// lam do not have when T is not a multiple of 4)
__device__ __forceinline__ void prefetch_l2_inside(const void* ptr, uint32_t bytes) {
  const uintptr_t a = reinterpret_cast<uintptr_t>(ptr);
  const uintptr_t lo = (a + 15) & ~(uintptr_t)15, hi = (a + bytes) & ~(uintptr_t)15;
  if (hi > lo) bulk_prefetch_l2(reinterpret_cast<const void*>(lo), (uint32_t)(hi - lo));
}

// The full tile of rows row0 .. row0+127 of a [rows, 128] bf16 tensor by two
// TMA boxes of [128 x 64] (128-byte swizzle: the layout of swz), completion
// counted on `bar`.
__device__ __forceinline__ void tma_tile(unsigned char* dst, const CUtensorMap* map, uint64_t* bar, size_t row0) {
  tma_load_2d(dst, map, bar, 0, (int)row0);
  tma_load_2d(dst + kHalf, map, bar, 64, (int)row0);
}

// Common prologue: the mbarrier and the TMEM allocation (warp 0).
template <uint32_t kCols>
__device__ __forceinline__ uint32_t setup_tmem(uint64_t* bar, uint32_t* slot) {
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(slot, kCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  return *slot;
}

template <uint32_t kCols>
__device__ __forceinline__ void release_tmem(uint32_t tmem) {
  tc_fence_before();
  __syncthreads();
  if ((threadIdx.x >> 5) == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kCols);
  }
}

// Hand the staged tiles to the tensor cores and the TMEM columns back to them.
__device__ __forceinline__ void to_async() {
  fence_proxy_async_shared();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
}

// this thread's TMEM lane (row threadIdx.x mod 128: warp w reads lanes 32 (w mod 4) ..) at column col
__device__ __forceinline__ uint32_t lane_addr(uint32_t tmem, int col) {
  return tmem + ((uint32_t)(((threadIdx.x >> 5) & 3) * 32) << 16) + (uint32_t)col;
}

// ------------------------------------------------------------------ intra
constexpr uint32_t kIntraQ = 0, kIntraK = kTileB, kIntraV = 2 * kTileB, kIntraG = 3 * kTileB, kIntraP = 4 * kTileB,
                   kIntraA = 5 * kTileB, kIntraEnd = 6 * kTileB;
constexpr int kIntraThreads = 256;
constexpr uint64_t kIntraStaggerNs = 8000;  // the start delay of the CTAs with one item fewer (measured: 3-12 us)  // two threads per row: columns 0..63 and 64..127
constexpr size_t intra_smem() {
  return 1024 + kIntraEnd + kT * 8 + kT * 4 + 4 * kT * 4 + kT * 4 + kT * 8 * 4 + kT * 4 + 64;
}

// v[idx] for a runtime idx < n (n a power of two), by a tree of selects on
// the bits of idx (the values stay in registers)
template <int n>
__device__ __forceinline__ float pick(const float* v, int idx) {
  float r[n / 2];
#pragma unroll
  for (int m = 0; m < n / 2; ++m) r[m] = (idx & 1) ? v[2 * m + 1] : v[2 * m];
  if constexpr (n == 2) {
    return r[0];
  } else {
    return pick<n / 2>(r, idx >> 1);
  }
}

// 2^x by the hardware approximation (relative error ~2^-22, subnormal
// results flushed to 0): for the in-tile decays, whose products end in bf16
// operands or float32 sums of many terms
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Reduce-scatter over a warp: lane l receives the sum over the 32 lanes of v[l].
__device__ __forceinline__ float warp_column_sums(float (&v)[32]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int half = 16; half >= 1; half >>= 1) {
    const bool up = lane & half;
#pragma unroll
    for (int u = 0; u < half; ++u) {
      const float send = up ? v[u] : v[u + half];
      const float keep = up ? v[u + half] : v[u];
      v[u] = keep + __shfl_xor_sync(0xffffffffu, send, half);
    }
  }
  return v[0];
}

__global__ void __launch_bounds__(kIntraThreads, 1) bwd_tc_intra_kernel(
    const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
    const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tg, int use_tma,
    const __grid_constant__ CUtensorMap tdq, const __grid_constant__ CUtensorMap tdk,
    const __grid_constant__ CUtensorMap tdv, const __grid_constant__ CUtensorMap tS, int use_omap,
    const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k, const __nv_bfloat16* __restrict__ v,
    const __nv_bfloat16* __restrict__ dout, const float* __restrict__ log_alpha, const float* __restrict__ lam,
    __nv_bfloat16* __restrict__ dqp, __nv_bfloat16* __restrict__ dkp, __nv_bfloat16* __restrict__ dvp,
    float* __restrict__ dlam,
    float* __restrict__ S, double* __restrict__ tot, float* __restrict__ dc, int T, int L, int N, int BH,
    unsigned* __restrict__ qctr, unsigned* err) {
  extern __shared__ unsigned char sm_raw[];
  unsigned char* base = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(sm_raw) + 1023) & ~uintptr_t(1023));
  double* cs = reinterpret_cast<double*>(base + kIntraEnd);
  float* wdec = reinterpret_cast<float*>(cs + kT);
  float* colpart = wdec + kT;  // [4 warps][128 columns] of sum_i P_ij G_ij
  float* c2 = colpart + 4 * kT;  // cs x log2(e), float: the in-tile decays are exp2(c2_i - c2_j)
  float* dlhalf = c2 + kT;       // [128][8] the in-tile dlam of the columns 64..127
  float* colf = dlhalf + kT * 8;  // exp2(c2_e - c2_j), e = the end of j's 32-column block
  uint64_t* bar = reinterpret_cast<uint64_t*>(colf + kT);
  uint64_t* inbar = bar + 1;  // the TMA loads of the input tiles
  uint32_t* slot = reinterpret_cast<uint32_t*>(bar + 2);
  int* abort_s = reinterpret_cast<int*>(slot + 1);
  const int tid = threadIdx.x;
  if (tid == 0) {
    *abort_s = 0;
    mbar_init(inbar, 1);  // made visible by the fence in setup_tmem
    if (blockIdx.x == 0) *qctr = 0;  // the query kernel's item counter (that kernel runs after this one)
  }
  const uint32_t tmem = setup_tmem<512>(bar, slot);
  // persistent: tile item w = (tile w mod N, head w / N), one after another;
  // each item's inputs are staged in L2 while the previous one is computed
  // The items' memory phases (inputs in, outputs out) are bursts that run at
  // the HBM rate when every SM is in them at once.  The CTAs with one item
  // fewer than the rest start about two thirds of an item later, so that their
  // bursts fall in the others' compute phases; they end no later for it.
  {
    const int items = N * BH, rem = items % (int)gridDim.x;
    if (rem != 0 && items >= 2 * (int)gridDim.x && (int)blockIdx.x >= rem) {
      const uint64_t t0 = globaltimer_ns();
      while (globaltimer_ns() - t0 < kIntraStaggerNs) __nanosleep(256);
    }
  }
  uint32_t n_in = 0;  // the items whose inputs came by TMA so far (one phase of inbar each)
  for (int w = blockIdx.x; w < N * BH; w += gridDim.x) {
  const int c = w % N;
  const size_t bh = (size_t)(w / N);
  const size_t row0 = bh * T + (size_t)c * kT;
  const int nv = min(kT, T - c * kT);
  const bool tma = use_tma && nv == kT;  // a partial tile: its missing rows are zeros, staged by the threads
  bool ok = true;
  if (tid == 0) {
    // this item's input tiles (the previous item's outputs have been read
    // out of these buffers), then the next item's rows staged in L2
    if (tma) {
      mbar_arrive_expect_tx(inbar, 4 * kTileB);
      tma_tile(base + kIntraQ, &tq, inbar, row0);
      tma_tile(base + kIntraK, &tk, inbar, row0);
      tma_tile(base + kIntraV, &tv, inbar, row0);
      tma_tile(base + kIntraG, &tg, inbar, row0);
    }
    const int wn = w + (int)gridDim.x;
    if (wn < N * BH) {
      const size_t rn = (size_t)(wn / N) * T + (size_t)(wn % N) * kT;
      const int nn = min(kT, T - (wn % N) * kT);
      const uint32_t bytes = (uint32_t)(nn * kD * 2);
      bulk_prefetch_l2(q + rn * kD, bytes);
      bulk_prefetch_l2(k + rn * kD, bytes);
      bulk_prefetch_l2(v + rn * kD, bytes);
      bulk_prefetch_l2(dout + rn * kD, bytes);
      prefetch_l2_inside(log_alpha + rn, (uint32_t)(nn * 4));
      prefetch_l2_inside(lam + rn * L, (uint32_t)(nn * L * 4));
    }
  }
  tile_cumsum(cs, log_alpha, row0, nv);  // while the tiles land
  if (tid == kT - 1) tot[bh * N + c] = cs[kT - 1];
  if (tma) {
    ok = wait_phase(inbar, n_in & 1, err, abort_s);
    ++n_in;
  } else if (tid < kT) {
    stage_bf16(base + kIntraQ, q + row0 * kD, nv, tid);
    stage_bf16(base + kIntraK, k + row0 * kD, nv, tid);
    stage_bf16(base + kIntraV, v + row0 * kD, nv, tid);
    stage_bf16(base + kIntraG, dout + row0 * kD, nv, tid);
  }
  to_async();
  const uint32_t sQ = smem_u32(base + kIntraQ), sK = smem_u32(base + kIntraK), sV = smem_u32(base + kIntraV),
                 sG = smem_u32(base + kIntraG), sP = smem_u32(base + kIntraP), sA = smem_u32(base + kIntraA);
  if (tid == 0 && ok) {
    mma128(tmem + 0, sQ, false, sK, false, false);    // A = Q K^T
    mma128(tmem + 128, sG, false, sV, false, false);  // G = dO V^T
    umma_commit(bar);
  }
  // row i = tid mod 128, columns 64 hf .. 64 hf + 63 of it
  const int i = tid & (kT - 1), hf = tid >> 7;
  if (tid < kT) {
    c2[tid] = (float)cs[tid] * 1.4426950408889634f;
    wdec[tid] = expf((float)(cs[kT - 1] - cs[tid]));
    colf[tid] = ex2((float)(cs[(tid | 31)] - cs[tid]) * 1.4426950408889634f);
  }
  float lm[8];  // the row's in-tile lambdas, loaded while the products run
#pragma unroll
  for (int l = 0; l < 8; ++l) lm[l] = (i < nv && l < L) ? lam[(row0 + i) * L + l] : 0.f;
  __syncthreads();
  ok = ok && wait_phase(bar, 0, err, abort_s);
  tc_fence_after();
  {
    // row i: P, dA (bf16) and the in-tile levels of dlam.
    // Warp wi holds rows 32 wi .. 32 wi + 31: the 32-column blocks above its
    // diagonal block are masked, those below it hold one level (5 + bitlen(wi ^ cb)).
    const int wi = (tid >> 5) & 3, lane = tid & 31;
    const bool row_ok = i < nv;
    float dl[8];
#pragma unroll
    for (int l = 0; l < 8; ++l) dl[l] = 0.f;
    const float ci = c2[i];
#pragma unroll 1
    for (int cb = 2 * hf; cb < 2 * hf + 2; ++cb) {
      float p[32], da[32];
      if (cb > wi) {
#pragma unroll
        for (int u = 0; u < 32; ++u) p[u] = da[u] = 0.f;
        colpart[wi * kT + 32 * cb + lane] = 0.f;
      } else {
        float a[32], g[32];
        tmem_ld32(lane_addr(tmem, 32 * cb), a);
        tmem_ld32(lane_addr(tmem, 128 + 32 * cb), g);
        tmem_ld_wait();
        if (cb < wi) {
          const int lvc = 5 + bitlen((unsigned)(wi ^ cb));
          float lmv = lm[6];
          if (lvc == 7) lmv = lm[7];
          // all keys of the block lie before the row: exp2(c_i - c_j) = exp2(c_i -
          // c_e) exp2(c_e - c_j), e = the block's end, both factors <= 1, the
          // second from the per-tile column table
          const float rf = row_ok ? ex2(ci - c2[32 * cb + 31]) : 0.f;
          const float rl = rf * lmv;
          float cfv[32];  // the block's column factors, eight 16-byte loads
#pragma unroll
          for (int u4 = 0; u4 < 8; ++u4) {
            const float4 f = reinterpret_cast<const float4*>(colf + 32 * cb)[u4];
            cfv[4 * u4] = f.x; cfv[4 * u4 + 1] = f.y; cfv[4 * u4 + 2] = f.z; cfv[4 * u4 + 3] = f.w;
          }
          float acc = 0.f;
#pragma unroll
          for (int u = 0; u < 32; ++u) {
            const float cf = cfv[u];
            const float w = rl * cf;
            p[u] = a[u] * w;
            da[u] = g[u] * w;
            acc = fmaf(g[u] * a[u], cf, acc);
          }
          acc *= rf;
          if (lvc == 7) dl[7] += acc;
          else dl[6] += acc;
        } else {
          // the diagonal block, keys j <= i: branch-free over the columns, so
          // that the 32 columns' loads and exponentials overlap instead of
          // running one after another (a masked column's exp2 is selected away,
          // whatever its value).  Column u's level is bitlen(lane ^ u): its
          // lambda by a tree of selects on the lane's bits, tk[m] holding the
          // lambda for the columns whose low k + 1 bits are m
          float t1[2], t2[4], t3[8], t4[16];
#pragma unroll
          for (int m = 0; m < 2; ++m) t1[m] = ((lane & 1) != (m & 1)) ? lm[1] : lm[0];
#pragma unroll
          for (int m = 0; m < 4; ++m) t2[m] = ((lane & 2) != (m & 2)) ? lm[2] : t1[m & 1];
#pragma unroll
          for (int m = 0; m < 8; ++m) t3[m] = ((lane & 4) != (m & 4)) ? lm[3] : t2[m & 3];
#pragma unroll
          for (int m = 0; m < 16; ++m) t4[m] = ((lane & 8) != (m & 8)) ? lm[4] : t3[m & 7];
          float cjv[32];  // the block's column cumsums, eight 16-byte loads
#pragma unroll
          for (int u4 = 0; u4 < 8; ++u4) {
            const float4 f = reinterpret_cast<const float4*>(c2 + 32 * cb)[u4];
            cjv[4 * u4] = f.x; cjv[4 * u4 + 1] = f.y; cjv[4 * u4 + 2] = f.z; cjv[4 * u4 + 3] = f.w;
          }
          float xx[32];
#pragma unroll
          for (int u = 0; u < 32; ++u) {
            const int j = 32 * cb + u;
            const bool on = j <= i && row_ok;
            const float exm = on ? ex2(ci - cjv[u]) : 0.f;
            const float lmv = ((lane & 16) != (u & 16)) ? lm[5] : t4[u & 15];
            const float w = exm * lmv;
            p[u] = a[u] * w;
            da[u] = g[u] * w;
            xx[u] = g[u] * a[u] * exm;
          }
          // row i's keys of level l >= 1 are the aligned block of 2^(l-1)
          // columns beside the row's own block of that size (level 0: its own
          // column; the masked columns hold 0): sums over aligned blocks, the
          // row's picked by the bits of its lane
          float b1[16], b2[8], b3[4], b4[2];
#pragma unroll
          for (int m = 0; m < 16; ++m) b1[m] = xx[2 * m] + xx[2 * m + 1];
#pragma unroll
          for (int m = 0; m < 8; ++m) b2[m] = b1[2 * m] + b1[2 * m + 1];
#pragma unroll
          for (int m = 0; m < 4; ++m) b3[m] = b2[2 * m] + b2[2 * m + 1];
#pragma unroll
          for (int m = 0; m < 2; ++m) b4[m] = b3[2 * m] + b3[2 * m + 1];
          dl[0] += pick<32>(xx, lane);
          dl[1] += pick<32>(xx, lane ^ 1);
          dl[2] += pick<16>(b1, (lane >> 1) ^ 1);
          dl[3] += pick<8>(b2, (lane >> 2) ^ 1);
          dl[4] += pick<4>(b3, (lane >> 3) ^ 1);
          dl[5] += pick<2>(b4, (lane >> 4) ^ 1);
        }
        // v_j . dv_j inside the tile is the column sum of P . G, kept in float32
        float pg[32];
#pragma unroll
        for (int u = 0; u < 32; ++u) pg[u] = p[u] * g[u];
        colpart[wi * kT + 32 * cb + lane] = warp_column_sums(pg);
      }
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        const int c8 = 4 * cb + w;
        *reinterpret_cast<uint4*>(base + kIntraP + swz(i, c8)) =
            make_uint4(pack_bf16x2(p[8 * w], p[8 * w + 1]), pack_bf16x2(p[8 * w + 2], p[8 * w + 3]),
                       pack_bf16x2(p[8 * w + 4], p[8 * w + 5]), pack_bf16x2(p[8 * w + 6], p[8 * w + 7]));
        *reinterpret_cast<uint4*>(base + kIntraA + swz(i, c8)) =
            make_uint4(pack_bf16x2(da[8 * w], da[8 * w + 1]), pack_bf16x2(da[8 * w + 2], da[8 * w + 3]),
                       pack_bf16x2(da[8 * w + 4], da[8 * w + 5]), pack_bf16x2(da[8 * w + 6], da[8 * w + 7]));
      }
    }
    // V rows scaled by wdec (the G product that read V has completed) by the
    // warps with time to spare in this phase: the two with no block at or
    // below the diagonal (rows 0..63, columns 64..127) scale rows 0..95, the
    // two that hold only a diagonal block rows 96..127 after it
    auto scale_v = [&](int j, int c0, int nc) {  // nc = 8 or 16 chunks, eight loads issued together
      const float s = wdec[j];
#pragma unroll 1
      for (int cc = c0; cc < c0 + nc; cc += 8) {
        uint4 raw[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) raw[k] = *reinterpret_cast<const uint4*>(base + kIntraV + swz(j, cc + k));
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          float x[8];
          unpack8(raw[k], x);
          *reinterpret_cast<uint4*>(base + kIntraV + swz(j, cc + k)) =
              make_uint4(pack_bf16x2(s * x[0], s * x[1]), pack_bf16x2(s * x[2], s * x[3]),
                         pack_bf16x2(s * x[4], s * x[5]), pack_bf16x2(s * x[6], s * x[7]));
        }
      }
    };
    if (hf == 1 && wi < 2) {  // threads t = 0..63: row t, and half of row 64 + t / 2
      const int t = tid - 128;
      scale_v(t, 0, 16);
      scale_v(64 + (t >> 1), 8 * (t & 1), 8);
    } else if ((hf == 0 && wi == 0) || (hf == 1 && wi == 2)) {  // threads t = 0..63: half of row 96 + t / 2
      const int t = hf == 0 ? tid : tid - 160;
      scale_v(96 + (t >> 1), 8 * (t & 1), 8);
    }
    if (hf == 1)
#pragma unroll
      for (int l = 0; l < 8; ++l) dlhalf[i * 8 + l] = dl[l];
    __syncthreads();  // the column sums and the second half's levels of every row
    if (hf == 0)  // the row's in-tile levels of dlam, written out while the products run
#pragma unroll
      for (int l = 0; l < 8; ++l) dlhalf[i * 8 + l] += dl[l];
  }
  tmem_ld_wait();
  to_async();
  if (tid == 0 && ok) {
    mma128(tmem + 0, sA, false, sK, true, false);    // dq = dA K
    mma128(tmem + 128, sA, true, sQ, true, false);   // dk = dA^T Q
    mma128(tmem + 256, sP, true, sG, true, false);   // dv = P^T dO
    mma128(tmem + 384, sV, true, sK, true, false);   // S_c = (wdec V)^T K
    umma_commit(bar);
  }
  // while the products run: the in-tile levels of dlam (levels 0..7 of a
  // row are contiguous: a warp's store covers four rows) and the in-tile
  // part of -v_j . dv_j (the key side adds the rest of dc_j)
#pragma unroll
  for (int e = tid; e < kT * 8; e += kIntraThreads) {
    const int r = e >> 3, l = e & 7;
    if (r < nv && l < L) dlam[(row0 + r) * L + l] = dlhalf[e];
  }
  if (tid < nv)
    dc[row0 + tid] = -(colpart[tid] + colpart[kT + tid] + colpart[2 * kT + tid] + colpart[3 * kT + tid]);
  ok = ok && wait_phase(bar, 1, err, abort_s);
  tc_fence_after();
  if (use_omap && nv == kT) {
    // Every operand tile is free now: each output is staged in shared memory
    // (two alternating buffers over the tiles) in the layout of its TMA boxes
    // and written by thread 0's tensor stores: the in-tile parts of dq, dk, dv
    // as bf16 tiles (two [128 x 64] boxes; the later kernels add the
    // inter-tile parts in float32), the chunk state S_c as float32 (four
    // [128 x 32] boxes).  Before each barrier thread 0 waits until its earlier
    // stores have read their buffer, which the staging after the barrier reuses.
    const int r = i;  // this thread's half row: columns 64 hf .. 64 hf + 63
    // the two column blocks of an output are loaded from TMEM together, and
    // the next output's first block is in flight across the barrier
    float xs[2][32];
    tmem_ld32(lane_addr(tmem, 32 * (2 * hf)), xs[0]);  // warp-collective: every lane loads
#pragma unroll 1
    for (int o = 0; o < 4; ++o) {
      unsigned char* buf = base + (o & 1) * (kT * kRowP * 4);
      tmem_ld32(lane_addr(tmem, 128 * o + 32 * (2 * hf + 1)), xs[1]);
      tmem_ld_wait();
#pragma unroll
      for (int hb = 0; hb < 2; ++hb) {
        const int cb = 2 * hf + hb;
        const float* x = xs[hb];
        if (o == 3) {
          unsigned char* box = buf + cb * kRBox + r * 128;
#pragma unroll
          for (int ch = 0; ch < 8; ++ch)
            *reinterpret_cast<float4*>(box + ((ch ^ (r & 7)) << 4)) =
                make_float4(x[4 * ch], x[4 * ch + 1], x[4 * ch + 2], x[4 * ch + 3]);
        } else {
#pragma unroll
          for (int w = 0; w < 4; ++w)
            *reinterpret_cast<uint4*>(buf + swz(r, 4 * cb + w)) =
                make_uint4(pack_bf16x2(x[8 * w], x[8 * w + 1]), pack_bf16x2(x[8 * w + 2], x[8 * w + 3]),
                           pack_bf16x2(x[8 * w + 4], x[8 * w + 5]), pack_bf16x2(x[8 * w + 6], x[8 * w + 7]));
        }
      }
      if (o < 3) tmem_ld32(lane_addr(tmem, 128 * (o + 1) + 32 * (2 * hf)), xs[0]);
      fence_proxy_async_shared();
      if (tid == 0) bulk_wait_read0();
      __syncthreads();
      if (tid == 0 && ok) {
        if (o == 3) {
          const int y = (int)((bh * N + c) * kD);
#pragma unroll
          for (int cb = 0; cb < 4; ++cb) tma_store_2d(&tS, buf + cb * kRBox, 32 * cb, y);
        } else {
          const CUtensorMap* m = o == 0 ? &tdq : o == 1 ? &tdk : &tdv;
          tma_store_2d(m, buf, 0, (int)row0);
          tma_store_2d(m, buf + kHalf, 64, (int)row0);
        }
        bulk_commit();
      }
    }
    if (tid == 0) bulk_wait_read0();  // the writes complete with the grid
  } else
  {
    // Every operand tile is free now: each output row is staged in shared
    // memory (two alternating buffers of padded rows over the tiles) and
    // written by one bulk copy: the in-tile parts of dq, dk, dv as bf16 rows
    // (256 B; the later kernels add the inter-tile parts in float32), the
    // chunk state S_c as float32 rows (512 B).
    const int r = i;  // this thread's half row: columns 64 hf .. 64 hf + 63
    const size_t poff = (row0 + r) * kD + 64 * hf;  // this half row in dq, dk, dv
    float* srow = S + (bh * N + c) * (size_t)(kD * kD) + (size_t)r * kD + 64 * hf;
#pragma unroll 1
    for (int o = 0; o < 4; ++o) {
      const bool keep = o == 3 || r < nv;  // S has every row; the gradients only the present ones
      unsigned char* buf = base + (o & 1) * (kT * kRowP * 4);
      float* rowp = reinterpret_cast<float*>(buf) + r * kRowP;                    // float32 rows, 528 B apart
      __nv_bfloat16* rowb = reinterpret_cast<__nv_bfloat16*>(buf) + r * (kD + 8);  // bf16 rows, 272 B apart
      if (o >= 2) bulk_wait_read0();  // the copy of output o - 2 has read this buffer
#pragma unroll 1
      for (int cb = 2 * hf; cb < 2 * hf + 2; ++cb) {
        float x[32];
        tmem_ld32(lane_addr(tmem, 128 * o + 32 * cb), x);  // warp-collective: every lane loads
        tmem_ld_wait();
        if (o == 3) {
#pragma unroll
          for (int u = 0; u < 32; u += 4)
            *reinterpret_cast<float4*>(rowp + 32 * cb + u) = make_float4(x[u], x[u + 1], x[u + 2], x[u + 3]);
        } else {
#pragma unroll
          for (int u = 0; u < 32; u += 8)
            *reinterpret_cast<uint4*>(rowb + 32 * cb + u) =
                make_uint4(pack_bf16x2(x[u], x[u + 1]), pack_bf16x2(x[u + 2], x[u + 3]),
                           pack_bf16x2(x[u + 4], x[u + 5]), pack_bf16x2(x[u + 6], x[u + 7]));
        }
      }
      if (keep && ok) {
        fence_proxy_async_shared();
        if (o == 3) bulk_store(srow, rowp + 64 * hf, 64 * 4);
        else bulk_store((o == 0 ? dqp : o == 1 ? dkp : dvp) + poff, rowb + 64 * hf, 64 * 2);
        bulk_commit();
      }
    }
    bulk_wait_read0();  // the copies have read their rows; the writes complete with the grid
  }
  __syncthreads();  // every staged row has been read before the next item's tiles land
  }  // items
  release_tmem<512>(tmem);
}

// ------------------------------------------------------------------ query side
constexpr uint32_t kQryQ = 0, kQryG = kTileB, kQryL = 2 * kTileB, kQryF = 3 * kTileB, kQryR = 4 * kTileB;
constexpr uint32_t kQryEnd = kQryR + kT * kRowP * 4;
constexpr int kQryThreads = 256;  // two threads per row: columns 0..63 and 64..127
constexpr int kQryLamL = 32;  // lam rows of up to this many levels staged in shared memory
// + cs, the second halves' dlam dots, an item's log_alpha and lam rows, five
// mbarriers, TMEM slot, flags, next item
constexpr size_t query_smem() { return 1024 + kQryEnd + kT * 8 + kT * 4 + kT * 4 + kT * kQryLamL * 4 + 64; }

// Persistent over the (tile, head) items, one CTA per SM.  Item j is tile
// c = N - 1 - j / BH of head j mod BH: the items of all heads' last tiles
// first, the light ones of the first tiles (few set bits of c) at the end.
// CTA b takes items b and b + gridDim.x, then claims items 2 gridDim.x + k
// from the counter *qctr (zero at the launch), each when it starts the item
// two before: the item after the current one is always known, so that its
// first node tile, its input tiles and its rows of log_alpha and lam stream
// in, and its cumsum is taken, while the current one finishes.

__global__ void __launch_bounds__(kQryThreads, 1) bwd_tc_query_kernel(
    const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tg, int use_tma,
    const __grid_constant__ CUtensorMap tr, int use_rmap,
    const __grid_constant__ CUtensorMap tdi, const __grid_constant__ CUtensorMap tdo, int use_dmap,
    const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ dout, const float* __restrict__ log_alpha,
    const float* __restrict__ lam, const __nv_bfloat16* __restrict__ Ft, const double* __restrict__ G,
    const __nv_bfloat16* __restrict__ dqp, __nv_bfloat16* __restrict__ dq, float* __restrict__ dlam,
    float* __restrict__ R,
    int T, int L, int N, int BH, unsigned* __restrict__ qctr, unsigned* err) {
  extern __shared__ unsigned char sm_raw[];
  unsigned char* base = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(sm_raw) + 1023) & ~uintptr_t(1023));
  double* cs = reinterpret_cast<double*>(base + kQryEnd);
  float* qpart = reinterpret_cast<float*>(cs + kT);  // [128] the dlam dot of the columns 64..127
  float* la_s = qpart + kT;    // [128] an item's log_alpha
  float* lam_s = la_s + kT;    // [128][L] an item's lam rows (L <= kQryLamL)
  uint64_t* bar = reinterpret_cast<uint64_t*>(lam_s + kT * kQryLamL);
  uint64_t* ldbar = bar + 1;  // the bulk load of a node tile
  uint64_t* inbar = bar + 2;  // the TMA loads of the input tiles
  uint64_t* obar = bar + 3;   // the TMA load of the in-tile dq tile
  uint64_t* sbar = bar + 4;   // the bulk loads of an item's log_alpha and lam rows
  uint32_t* slot = reinterpret_cast<uint32_t*>(bar + 5);
  int* abort_s = reinterpret_cast<int*>(slot + 1);
  int* next_s = abort_s + 1;  // [2] the item after the current one (or items: none), by the parity of the item count
  int* stop_s = next_s + 2;   // an abort seen at an item's end
  const int tid = threadIdx.x;
  const int items = N * BH;
  const size_t mat = (size_t)kD * kD;
  auto tile_of = [&](int j) { return N - 1 - j / BH; };
  auto head_of = [&](int j) { return (size_t)(j % BH); };
  auto full_tile = [&](int j) { return use_tma && T - tile_of(j) * kT >= kT; };  // its inputs by TMA
  // its log_alpha and lam rows by bulk copies (16-byte aligned: T a multiple of 4)
  auto rows_smem = [&](int j) { return T - tile_of(j) * kT >= kT && (T & 3) == 0 && L <= kQryLamL; };
  auto next_bit = [](int c, int h) {  // the set bit of c above h, or -1
    for (++h; (c >> h) != 0; ++h)
      if ((c >> h) & 1) return h;
    return -1;
  };
  // thread 0: node tile e(c, h) of head bh into the node buffer; one load per
  // level, each issued once the products of the level before have read the buffer
  auto load_node = [&](int c, size_t bh, int h) {
    const int e = ((c >> (h + 1)) << (h + 1)) + (1 << h) - 1;
    mbar_arrive_expect_tx(ldbar, kTileB);
    bulk_load(base + kQryF, Ft + (bh * N + e) * mat, kTileB, ldbar);
  };
  // thread 0: item j's Q and dO tiles (full tiles only)
  auto load_inputs = [&](int j) {
    const size_t r = head_of(j) * T + (size_t)tile_of(j) * kT;
    mbar_arrive_expect_tx(inbar, 2 * kTileB);
    tma_tile(base + kQryQ, &tq, inbar, r);
    tma_tile(base + kQryG, &tg, inbar, r);
  };
  // thread 0: item j's rows that the threads read from global into L2: of
  // log_alpha and lam where they are not copied to shared memory, of the
  // in-tile dq where it is not loaded by TMA
  auto stage_l2 = [&](int j) {
    const int cn = tile_of(j);
    const size_t r = head_of(j) * T + (size_t)cn * kT;
    const int nn = min(kT, T - cn * kT);
    if (!rows_smem(j)) {
      prefetch_l2_inside(log_alpha + r, (uint32_t)(nn * 4));
      prefetch_l2_inside(lam + r * L, (uint32_t)(nn * L * 4));
    }
    if (!(use_dmap && full_tile(j))) bulk_prefetch_l2(dqp + r * kD, (uint32_t)(nn * kD * 2));
  };
  // thread 0: item j's rows of log_alpha and lam into shared memory (after
  // the last reads of the previous ones)
  auto load_rows = [&](int j) {
    const size_t r = head_of(j) * T + (size_t)tile_of(j) * kT;
    mbar_arrive_expect_tx(sbar, (uint32_t)(kT * 4 + kT * L * 4));
    bulk_load(la_s, log_alpha + r, (uint32_t)(kT * 4), sbar);
    bulk_load(lam_s, lam + r * L, (uint32_t)(kT * L * 4), sbar);
  };
  // thread 0: the in-tile dq tile of rows r.. into the operand buffer, free
  // once the item's last products have read it
  auto load_dqp = [&](size_t r) {
    mbar_arrive_expect_tx(obar, kTileB);
    tma_tile(base + kQryL, &tdi, obar, r);
  };
  int j = blockIdx.x;
  int jn = j + (int)gridDim.x < items ? j + (int)gridDim.x : items;  // thread 0: the item after j
  unsigned jraw = 0;  // thread 0: the claim made during the current item (read at its end)
  if (tid == 0) {
    *abort_s = 0;
    mbar_init(ldbar, 1);
    mbar_init(inbar, 1);
    mbar_init(obar, 1);
    mbar_init(sbar, 1);
    fence_mbar_init();  // the copies below arrive on them
    // the first item's first node tile and input tiles go out before the
    // TMEM allocation and the cumsum, which run while they land
    if (tile_of(j) > 0) load_node(tile_of(j), head_of(j), next_bit(tile_of(j), -1));
    if (full_tile(j)) load_inputs(j);
    if (rows_smem(j)) load_rows(j);
  }
  const uint32_t tmem = setup_tmem<512>(bar, slot);
  const uint32_t sQ = smem_u32(base + kQryQ), sG = smem_u32(base + kQryG), sL = smem_u32(base + kQryL),
                 sF = smem_u32(base + kQryF);
  const int i = tid & (kT - 1), hf = tid >> 7;  // row i, columns 64 hf .. 64 hf + 63
  // the levels (node loads, product commits), the TMA input, dq and row loads so far
  uint32_t nlev = 0, nin = 0, nout = 0, nrow = 0;
  bool pend = false;  // a level's tensor reductions may still read the staged boxes
  // item jj's cumsum (its rows of log_alpha from shared memory where they
  // were copied there): every thread, after the last reads of cs
  auto cumsum_of = [&](int jj) -> bool {
    bool okr = true;
    double x;
    if (rows_smem(jj)) {
      okr = wait_phase(sbar, nrow & 1, err, abort_s);
      ++nrow;
      x = tid < kT ? (double)la_s[tid] : 0.0;
    } else {
      x = tile_log_alpha(log_alpha, head_of(jj) * T + (size_t)tile_of(jj) * kT, min(kT, T - tile_of(jj) * kT));
    }
    tile_scan(cs, x);
    return okr;
  };
  bool okc = cumsum_of(j);
  for (uint32_t it = 0;; ++it) {
  const int c = tile_of(j);
  const size_t bh = head_of(j);
  const size_t row0 = bh * T + (size_t)c * kT;
  const int nv = min(kT, T - c * kT);
  const bool tma = full_tile(j);
  const bool dtma = use_dmap && tma;  // dq in and out by TMA through the operand buffer
  const bool rsm = rows_smem(j);  // lam from shared memory
  if (tid == 0) {
    next_s[it & 1] = jn;  // read after the barrier below
    // the item after jn (a claim past the end, also when jn is none, takes
    // nothing: the claims are handed out in order)
    jraw = atomicAdd(qctr, 1u);
  }
  bool ok = okc;
  if (tma) {
    ok = wait_phase(inbar, nin & 1, err, abort_s);
    ++nin;
  } else if (tid < kT) {
    stage_bf16(base + kQryQ, q + row0 * kD, nv, tid);
    stage_bf16(base + kQryG, dout + row0 * kD, nv, tid);
    fence_proxy_async_shared();  // a later item's tiles land in these buffers by TMA
  }
  if (tid == 0) bulk_wait_read0();  // the previous item's dq store has read the operand buffer
  __syncthreads();
  const int jx = next_s[it & 1];  // the next item, known to every thread
  double D = 0.0;
  bool first = true;
  for (int h = 0; (c >> h) != 0; ++h) {
    if (!((c >> h) & 1)) continue;
    const int e = ((c >> (h + 1)) << (h + 1)) + (1 << h) - 1;
    const int lv = kLc + 1 + h;
    const int hn = next_bit(c, h);  // the item's next level, or -1
    const double g_e = G[bh * N + e];  // added to D at the level's end
    const float w = i < nv ? expf((float)(cs[i] + D)) : 0.f;
    const float lw = i < nv ? w * (rsm ? lam_s[i * L + lv] : lam[(row0 + i) * L + lv]) : 0.f;
    // dO rows scaled by lw (this thread's half row): its eight 16-byte chunks
    // loaded together, then scaled and stored
    {
      uint4 raw[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) raw[k] = *reinterpret_cast<const uint4*>(base + kQryG + swz(i, 8 * hf + k));
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        float x[8];
        unpack8(raw[k], x);
        *reinterpret_cast<uint4*>(base + kQryL + swz(i, 8 * hf + k)) =
            make_uint4(pack_bf16x2(lw * x[0], lw * x[1]), pack_bf16x2(lw * x[2], lw * x[3]),
                       pack_bf16x2(lw * x[4], lw * x[5]), pack_bf16x2(lw * x[6], lw * x[7]));
      }
    }
    ok = ok && wait_phase(ldbar, nlev & 1, err, abort_s);
    to_async();
    if (tid == 0 && ok) {
      mma128(tmem + 0, sG, false, sF, true, false);    // g = dO F_e
      mma128(tmem + 256, sL, true, sQ, true, false);   // R_e part = (diag(lw) dO)^T Q
      umma_commit(bar);
    }
    const bool first_lv = first;
    first = false;
    ok = ok && wait_phase(bar, nlev & 1, err, abort_s);
    ++nlev;
    tc_fence_after();
    if (tid == 0 && ok) {  // the products have read the node buffer: this item's next node, or the next item's first
      if (hn >= 0) {
        load_node(c, bh, hn);
      } else {
        if (jn < items && tile_of(jn) > 0) load_node(tile_of(jn), head_of(jn), next_bit(tile_of(jn), -1));
        if (dtma) load_dqp(row0);  // the last products have read the operand buffer too
      }
    }
    float part = 0.f;
    {
      // both column blocks of g from TMEM together
      float gs[2][32];
      tmem_ld32(lane_addr(tmem, 32 * (2 * hf)), gs[0]);
      tmem_ld32(lane_addr(tmem, 32 * (2 * hf + 1)), gs[1]);
      tmem_ld_wait();
#pragma unroll
      for (int hb = 0; hb < 2; ++hb) {
        const int cb = 2 * hf + hb;
#pragma unroll
        for (int w4 = 0; w4 < 4; ++w4) {
          float x[8];
          row_chunk(base + kQryQ, i, 4 * cb + w4, x);
#pragma unroll
          for (int u = 0; u < 8; ++u) part = fmaf(gs[hb][8 * w4 + u], x[u], part);
        }
      }
      // dq += diag(lw) dO F_e = lw g: the node part of dq accumulates in TMEM
      // columns 128.. from the float32 g (no product of its own)
      if (first_lv) {
#pragma unroll
        for (int hb = 0; hb < 2; ++hb) {
          uint32_t wv[32];
#pragma unroll
          for (int u = 0; u < 32; ++u) wv[u] = __float_as_uint(lw * gs[hb][u]);
          tmem_st32(lane_addr(tmem, 128 + 32 * (2 * hf + hb)), wv);
        }
      } else {  // both column blocks of the running dq loaded together
        float prev[2][32];
        tmem_ld32(lane_addr(tmem, 128 + 32 * (2 * hf)), prev[0]);
        tmem_ld32(lane_addr(tmem, 128 + 32 * (2 * hf + 1)), prev[1]);
        tmem_ld_wait();
#pragma unroll
        for (int hb = 0; hb < 2; ++hb) {
          uint32_t wv[32];
#pragma unroll
          for (int u = 0; u < 32; ++u) wv[u] = __float_as_uint(fmaf(lw, gs[hb][u], prev[hb][u]));
          tmem_st32(lane_addr(tmem, 128 + 32 * (2 * hf + hb)), wv);
        }
      }
      tmem_st_wait();
      if (hf == 1) qpart[i] = part;
      if (use_rmap) {
        // this tile's part of R_e staged as four [128 x 32] float32 boxes
        // (128-byte swizzle), row e' = i; thread 0 adds them into R_e by four
        // tensor reductions after the level's barrier and goes on: the
        // reductions read the boxes while the next level stages its operand
        // and runs its products, and are waited for only here, before the
        // boxes are rewritten
        float xs[2][32];  // both column blocks of the R part from TMEM together
        tmem_ld32(lane_addr(tmem, 256 + 32 * (2 * hf)), xs[0]);
        tmem_ld32(lane_addr(tmem, 256 + 32 * (2 * hf + 1)), xs[1]);
        tmem_ld_wait();
        if (pend) {
          if (tid == 0) bulk_wait_read0();
          __syncthreads();
        }
#pragma unroll
        for (int hb = 0; hb < 2; ++hb) {
          const int cb = 2 * hf + hb;
          const float* x = xs[hb];
          unsigned char* box = base + kQryR + cb * kRBox + i * 128;
#pragma unroll
          for (int ch = 0; ch < 8; ++ch)
            *reinterpret_cast<float4*>(box + ((ch ^ (i & 7)) << 4)) =
                make_float4(x[4 * ch], x[4 * ch + 1], x[4 * ch + 2], x[4 * ch + 3]);
        }
        fence_proxy_async_shared();
      } else {
        // row e' = i of this tile's part of R_e: staged in shared memory, then
        // added into R_e by the bulk-copy unit (a 256-byte reduction per half row)
        float* rrow = reinterpret_cast<float*>(base + kQryR) + i * kRowP;
        bulk_wait_read0();  // the previous level's reduction has read this row
#pragma unroll 1
        for (int cb = 2 * hf; cb < 2 * hf + 2; ++cb) {
          float x[32];
          tmem_ld32(lane_addr(tmem, 256 + 32 * cb), x);
          tmem_ld_wait();
#pragma unroll
          for (int u = 0; u < 32; u += 4)
            *reinterpret_cast<float4*>(rrow + 32 * cb + u) = make_float4(x[u], x[u + 1], x[u + 2], x[u + 3]);
        }
        if (ok) {
          fence_proxy_async_shared();
          float* rdst = R + (bh * N + e) * mat + (size_t)i * kD + 64 * hf;
          if (h == 0)  // the node's only query tile: stored (its memory is not cleared)
            bulk_store(rdst, rrow + 64 * hf, 64 * 4);
          else
            bulk_reduce_add_f32(rdst, rrow + 64 * hf, 64 * 4);
          bulk_commit();
        }
      }
    }
    D += g_e;
    tc_fence_before();
    __syncthreads();  // the next level rewrites the staged tiles and the TMEM columns
    if (hn < 0 && tid == 0 && ok && jn < items) {
      // the item's last level: Q and dO have had their last readers, and the
      // next item's tiles go out ahead of this level's reductions
      if (full_tile(jn)) load_inputs(jn);
      if (rows_smem(jn)) load_rows(jn);  // this level has read the item's lam rows
      stage_l2(jn);
    }
    if (use_rmap && tid == 0 && ok) {
      const int y = (int)((bh * N + e) * kD);
#pragma unroll
      for (int cb = 0; cb < 4; ++cb) {
        if (h == 0)  // the node's only query tile: stored (its memory is not cleared)
          tma_store_2d(&tr, base + kQryR + cb * kRBox, 32 * cb, y);
        else
          tma_reduce_add_box(&tr, base + kQryR + cb * kRBox, 32 * cb, y);
      }
      bulk_commit();
    }
    pend = use_rmap;
    if (hf == 0 && i < nv) dlam[(row0 + i) * L + lv] = w * (part + qpart[i]);
  }
  // an item with no level: the buffers are free for its dq tile and the
  // next item's node and input tiles
  if (tid == 0 && ok && c == 0) {
    if (dtma) load_dqp(row0);
    if (jn < items) {
      if (tile_of(jn) > 0) load_node(tile_of(jn), head_of(jn), next_bit(tile_of(jn), -1));
      if (full_tile(jn)) load_inputs(jn);
      if (rows_smem(jn)) load_rows(jn);
      stage_l2(jn);
    }
  }
  // the levels above 7 that hold no key of this tile's queries
  if (hf == 0 && i < nv)
    for (int l = kLc + 1; l < L; ++l) {
      const int hh = l - kLc - 1;
      if (!(hh < 31 && ((c >> hh) & 1))) dlam[(row0 + i) * L + l] = 0.f;
    }
  {
    const __nv_bfloat16* src = dqp + (row0 + i) * kD;
    __nv_bfloat16* dst = dq + (row0 + i) * kD;
    float xs[2][32];
    if (!first) {  // uniform over the CTA: the warp-collective loads run in every lane
      tmem_ld32(lane_addr(tmem, 128 + 32 * (2 * hf)), xs[0]);
      tmem_ld32(lane_addr(tmem, 128 + 32 * (2 * hf + 1)), xs[1]);
      tmem_ld_wait();
    } else {
#pragma unroll
      for (int u = 0; u < 32; ++u) xs[0][u] = xs[1][u] = 0.f;
    }
    if (dtma) {
      // dq = the in-tile part + the node part, in place in the operand
      // buffer, then out by two tensor stores
      ok = ok && wait_phase(obar, nout & 1, err, abort_s);
      ++nout;
#pragma unroll
      for (int hb = 0; hb < 2; ++hb) {
#pragma unroll
        for (int w4 = 0; w4 < 4; ++w4) {
          const int c8 = 4 * (2 * hf + hb) + w4;
          float a[8];
          row_chunk(base + kQryL, i, c8, a);
          const float* x = xs[hb] + 8 * w4;
          *reinterpret_cast<uint4*>(base + kQryL + swz(i, c8)) =
              make_uint4(pack_bf16x2(a[0] + x[0], a[1] + x[1]), pack_bf16x2(a[2] + x[2], a[3] + x[3]),
                         pack_bf16x2(a[4] + x[4], a[5] + x[5]), pack_bf16x2(a[6] + x[6], a[7] + x[7]));
        }
      }
      fence_proxy_async_shared();
      __syncthreads();
      if (tid == 0 && ok) {
        tma_store_2d(&tdo, base + kQryL, 0, (int)row0);
        tma_store_2d(&tdo, base + kQryL + kHalf, 64, (int)row0);
        bulk_commit();
      }
    } else
#pragma unroll
    for (int hb = 0; hb < 2; ++hb) {
      const int cb = 2 * hf + hb;
      const float* x = xs[hb];
      if (i < nv)
#pragma unroll
      for (int u = 0; u < 32; u += 8) {
        float a[8];
        unpack8(*reinterpret_cast<const uint4*>(src + 32 * cb + u), a);
        *reinterpret_cast<uint4*>(dst + 32 * cb + u) =
            make_uint4(pack_bf16x2(a[0] + x[u], a[1] + x[u + 1]), pack_bf16x2(a[2] + x[u + 2], a[3] + x[u + 3]),
                       pack_bf16x2(a[4] + x[u + 4], a[5] + x[u + 5]), pack_bf16x2(a[6] + x[u + 6], a[7] + x[u + 7]));
      }
    }
  }
  if (jx < items) okc = cumsum_of(jx);  // this item's levels have read cs
  // an abort, published by thread 0 once every thread is past this item (no
  // wait of it can raise the flag after the first barrier); the barriers also
  // order this item's TMEM reads before the next one's products
  tc_fence_before();
  __syncthreads();
  if (tid == 0) {
    *stop_s = *(volatile int*)abort_s;
    const int cand = 2 * (int)gridDim.x + (int)jraw;
    jn = cand < items ? cand : items;
  }
  __syncthreads();
  if (jx >= items || *stop_s) break;
  j = jx;
  }
  bulk_wait_read0();  // this thread's reductions into R (its rows, or thread 0's boxes) have read their sources
  release_tmem<512>(tmem);
}

// ------------------------------------------------------------------ key side
constexpr uint32_t kKeyK = 0, kKeyV = kTileB, kKeyE = 2 * kTileB, kKeyEnd = 3 * kTileB;
constexpr size_t key_smem() { return 1024 + kKeyEnd + kT * 8 + kT * 4 + kT * 4 + 32 * 12 + 64; }

__global__ void __launch_bounds__(kThreads, 1) bwd_tc_key_kernel(
    const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tv, int use_tma,
    const __grid_constant__ CUtensorMap tkpi, const __grid_constant__ CUtensorMap tvpi,
    const __grid_constant__ CUtensorMap tko, const __grid_constant__ CUtensorMap tvo, int use_kmap,
    const __nv_bfloat16* __restrict__ k, const __nv_bfloat16* __restrict__ v, const float* __restrict__ log_alpha,
    const float* __restrict__ lam, const float* __restrict__ dlam, const float* __restrict__ R,
    const double* __restrict__ cum, const __nv_bfloat16* __restrict__ dkp, const __nv_bfloat16* __restrict__ dvp,
    __nv_bfloat16* __restrict__ dk, __nv_bfloat16* __restrict__ dv, float* __restrict__ dc,
    int T, int L, unsigned* err) {
  extern __shared__ unsigned char sm_raw[];
  unsigned char* base = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(sm_raw) + 1023) & ~uintptr_t(1023));
  double* cs = reinterpret_cast<double*>(base + kKeyEnd);
  float* wdec = reinterpret_cast<float*>(cs + kT);
  float* coef = wdec + 2 * kT;                                   // [32]
  const float** srcs = reinterpret_cast<const float**>(coef + 32);  // [32]
  int* n_s = reinterpret_cast<int*>(srcs + 32);
  uint64_t* bar = reinterpret_cast<uint64_t*>(n_s + 2);
  uint64_t* inbar = bar + 1;  // the TMA loads of the input tiles
  uint64_t* obar = bar + 2;   // the TMA loads of the in-tile dk and dv tiles
  uint32_t* slot = reinterpret_cast<uint32_t*>(bar + 3);
  int* abort_s = reinterpret_cast<int*>(slot + 1);
  const int c = blockIdx.x, N = gridDim.x;
  const size_t bh = blockIdx.y;
  const int tid = threadIdx.x;
  const size_t row0 = bh * T + (size_t)c * kT;
  const int nv = min(kT, T - c * kT);
  const size_t mat = (size_t)kD * kD;
  const bool tma = use_tma && nv == kT;
  const bool otma = use_kmap && tma;  // dk and dv in and out by TMA through the K and E buffers
  if (tid == 0) {
    *abort_s = 0;
    mbar_init(inbar, 1);
    mbar_init(obar, 1);
    fence_mbar_init();  // the copies below arrive on them
    if (tma) {  // the input tiles go out first; the node list, cumsum and TMEM allocation run while they land
      mbar_arrive_expect_tx(inbar, 2 * kTileB);
      tma_tile(base + kKeyK, &tk, inbar, row0);
      tma_tile(base + kKeyV, &tv, inbar, row0);
    }
  }
  // this row's log_alpha and its lam, dlam of levels 0..15 go out first: their
  // latency runs under the node list's loads
  const double la = tile_log_alpha(log_alpha, row0, nv);
  float lam16[16], dlam16[16];
  {
    const float* lr = lam + (row0 + tid) * L;
    const float* dr = dlam + (row0 + tid) * L;
#pragma unroll
    for (int u = 0; u < 16; ++u) {
      lam16[u] = tid < nv && u < L ? lr[u] : 0.f;
      dlam16[u] = tid < nv && u < L ? dr[u] : 0.f;
    }
  }
  if (tid < 32) {  // lane h: the node of level h whose block holds the keys of c, if it has queries after it
    const int h = tid;
    const int e = h < 31 ? ((c >> (h + 1)) << (h + 1)) + (1 << h) - 1 : 0;
    const bool has = h < 31 && !((c >> h) & 1) && e + 1 < N;
    float cf = 0.f;
    if (has) cf = expf((float)(cum[bh * N + e] - cum[bh * N + c]));  // the decay from the end of c to the end of e
    const unsigned m = __ballot_sync(0xffffffffu, has);
    if (has) {
      const int at = __popc(m & ((1u << h) - 1u));  // in order of level
      srcs[at] = R + (bh * N + e) * mat;
      coef[at] = cf;
    }
    if (h == 0) *n_s = __popc(m);
  }
  tile_scan(cs, la);
  const uint32_t tmem = setup_tmem<256>(bar, slot);
  const int n = *n_s;
  float lamdot = 0.f;  // sum_l lam_j[l] dlam_j[l] of this row, in order of l
#pragma unroll
  for (int u = 0; u < 16; ++u) lamdot = fmaf(lam16[u], dlam16[u], lamdot);
  if (tid < nv) {
    const float* lr = lam + (row0 + tid) * L;
    const float* dr = dlam + (row0 + tid) * L;
    for (int l0 = 16; l0 < L; l0 += 16) {
      float a[16], d[16];
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        a[u] = l0 + u < L ? lr[l0 + u] : 0.f;
        d[u] = l0 + u < L ? dr[l0 + u] : 0.f;
      }
#pragma unroll
      for (int u = 0; u < 16; ++u) lamdot = fmaf(a[u], d[u], lamdot);
    }
  }
  wdec[tid] = expf((float)(cs[kT - 1] - cs[tid]));
  if (!tma) {
    stage_bf16(base + kKeyK, k + row0 * kD, nv, tid);
    stage_bf16(base + kKeyV, v + row0 * kD, nv, tid);
  }
  if (n > 0) stage_f32_sum(base + kKeyE, srcs, coef, n, tid);  // overlaps the TMA loads
  if (tma) wait_phase(inbar, 0, err, abort_s);
  to_async();
  if (n > 0) {
    const uint32_t sK = smem_u32(base + kKeyK), sV = smem_u32(base + kKeyV), sE = smem_u32(base + kKeyE);
    if (tid == 0) {
      mma128(tmem + 0, sK, false, sE, false, false);   // (E k_j) over rows j
      mma128(tmem + 128, sV, false, sE, true, false);  // (E^T v_j) over rows j
      umma_commit(bar);
    }
    wait_phase(bar, 0, err, abort_s);  // after a timeout the error word is set; the results are not used
    tc_fence_after();
  }
  // the products have read K and E (or there were none): the in-tile dv and
  // dk tiles load into them while the node parts come out of TMEM
  if (otma && tid == 0) {
    mbar_arrive_expect_tx(obar, 2 * kTileB);
    tma_tile(base + kKeyE, &tvpi, obar, row0);
    tma_tile(base + kKeyK, &tkpi, obar, row0);
  }
  const int j = tid;
  const float wj = wdec[j];
  float vdv = 0.f;
  if (otma) {
    bool okd = true, waited = false;
#pragma unroll 1
    for (int o = 0; o < 2; ++o) {  // 0: dv (in the E buffer), 1: dk (in the K buffer)
      unsigned char* tile = base + (o == 0 ? kKeyE : kKeyK);
      // each column block's TMEM load is in flight while the block before is added
      float xs[2][32];
      if (n > 0) tmem_ld32(lane_addr(tmem, 128 * o), xs[0]);
#pragma unroll
      for (int cb = 0; cb < 4; ++cb) {
        float* x = xs[cb & 1];
        if (n > 0) {
          tmem_ld_wait();
          if (cb < 3) tmem_ld32(lane_addr(tmem, 128 * o + 32 * (cb + 1)), xs[(cb + 1) & 1]);
        } else {
#pragma unroll
          for (int u = 0; u < 32; ++u) x[u] = 0.f;
        }
        if (o == 0) {  // the part of v_j . dv_j from the later tiles
#pragma unroll
          for (int w4 = 0; w4 < 4; ++w4) {
            float vv[8];
            row_chunk(base + kKeyV, j, 4 * cb + w4, vv);
#pragma unroll
            for (int t = 0; t < 8; ++t) vdv = fmaf(vv[t], wj * x[8 * w4 + t], vdv);
          }
        }
        if (!waited) {
          okd = wait_phase(obar, 0, err, abort_s);
          waited = true;
        }
#pragma unroll
        for (int w4 = 0; w4 < 4; ++w4) {
          const int c8 = 4 * cb + w4;
          float y[8];
          row_chunk(tile, j, c8, y);
#pragma unroll
          for (int t = 0; t < 8; ++t) y[t] = fmaf(wj, x[8 * w4 + t], y[t]);
          *reinterpret_cast<uint4*>(tile + swz(j, c8)) =
              make_uint4(pack_bf16x2(y[0], y[1]), pack_bf16x2(y[2], y[3]), pack_bf16x2(y[4], y[5]),
                         pack_bf16x2(y[6], y[7]));
        }
      }
    }
    fence_proxy_async_shared();
    __syncthreads();
    if (tid == 0 && okd) {
      tma_store_2d(&tvo, base + kKeyE, 0, (int)row0);
      tma_store_2d(&tvo, base + kKeyE + kHalf, 64, (int)row0);
      tma_store_2d(&tko, base + kKeyK, 0, (int)row0);
      tma_store_2d(&tko, base + kKeyK + kHalf, 64, (int)row0);
      bulk_commit();
      bulk_wait_read0();  // the tiles are read before the CTA's shared memory goes
    }
  } else
#pragma unroll 1
  for (int o = 0; o < 2; ++o) {  // 0: dv, 1: dk
    const __nv_bfloat16* src = (o == 0 ? dvp : dkp) + (row0 + j) * kD;
    __nv_bfloat16* dst = (o == 0 ? dv : dk) + (row0 + j) * kD;
#pragma unroll 1
    for (int cb = 0; cb < 4; ++cb) {
      float x[32];
      if (n > 0) {
        tmem_ld32(lane_addr(tmem, 128 * o + 32 * cb), x);
        tmem_ld_wait();
      } else {
#pragma unroll
        for (int u = 0; u < 32; ++u) x[u] = 0.f;
      }
      if (j < nv) {
#pragma unroll
        for (int u = 0; u < 32; u += 8) {
          float y[8];
          unpack8(*reinterpret_cast<const uint4*>(src + 32 * cb + u), y);
#pragma unroll
          for (int t = 0; t < 8; ++t) y[t] = fmaf(wj, x[u + t], y[t]);
          if (o == 0) {  // the part of v_j . dv_j from the later tiles
            float vv[8];
            row_chunk(base + kKeyV, j, (32 * cb + u) >> 3, vv);
#pragma unroll
            for (int t = 0; t < 8; ++t) vdv = fmaf(vv[t], wj * x[u + t], vdv);
          }
          *reinterpret_cast<uint4*>(dst + 32 * cb + u) =
              make_uint4(pack_bf16x2(y[0], y[1]), pack_bf16x2(y[2], y[3]), pack_bf16x2(y[4], y[5]),
                         pack_bf16x2(y[6], y[7]));
        }
      }
    }
  }
  if (j < nv) dc[row0 + j] = lamdot + dc[row0 + j] - vdv;  // dc held the in-tile part, -sum_i P_ij G_ij
  release_tmem<256>(tmem);
}

}  // namespace

PFN_cuTensorMapEncodeTiled_v12000 map_encoder() {
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

// [rows, 128] bf16 with [128 x 64] boxes and the 128-byte swizzle: two boxes make a tile
bool tile_map(CUtensorMap* m, const void* base, uint64_t rows) {
  auto fn = map_encoder();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)kD, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)kD * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)kT};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// [rows, 128] float32 with [128 x 32] boxes and the 128-byte swizzle (the key-side nodes)
bool f32_box_map(CUtensorMap* m, const void* base, uint64_t rows) {
  auto fn = map_encoder();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)kD, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)kD * 4};
  cuuint32_t box[2] = {32, (cuuint32_t)kT};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool bwd_tc_supported(const ll_shape& s) { return s.io == LL_BF16 && s.dk == 128 && s.dv == 128; }

ll_status bwd_tc_launch(const BwdArgs& a, const BwdTcBuffers& b) {
  const ll_shape& s = a.s;
  const int N = (s.T + kT - 1) / kT;
  const int BH = s.B * s.H;
  const dim3 grid(N, BH);
  // The key-side nodes of the levels above the first (odd e) accumulate from
  // 0, the tensor reductions of several query tiles; a first-level node (even
  // e) has one query tile, which stores it.  With N even the odd nodes
  // alternate with the even ones through R, and one pitched memset clears
  // them; otherwise R is cleared whole.  The query kernel's item counter, the
  // word after R, is cleared by the intra kernel.
  unsigned* qctr = reinterpret_cast<unsigned*>(b.R + (size_t)BH * N * kD * kD);
  const size_t node_bytes = (size_t)kD * kD * sizeof(float);
  if (N % 2 == 0)
    LL_CUDA_OK(cudaMemset2DAsync(b.R + (size_t)kD * kD, 2 * node_bytes, 0, node_bytes, (size_t)BH * N / 2, a.stream));
  else
    LL_CUDA_OK(cudaMemsetAsync(b.R, 0, (size_t)BH * N * node_bytes, a.stream));
  const auto* q = static_cast<const __nv_bfloat16*>(a.q);
  const auto* k = static_cast<const __nv_bfloat16*>(a.k);
  const auto* v = static_cast<const __nv_bfloat16*>(a.v);
  const auto* dout = static_cast<const __nv_bfloat16*>(a.dout);
  // the input tiles by TMA where the row coordinate fits the copy's 32-bit
  // operand; otherwise (and if the maps cannot be made) the threads stage them
  const uint64_t rows = (uint64_t)BH * s.T;
  CUtensorMap tq, tk, tv, tg;
  const int use_tma = rows <= 0x7fffffffull && tile_map(&tq, q, rows) && tile_map(&tk, k, rows) &&
                      tile_map(&tv, v, rows) && tile_map(&tg, dout, rows);
  LL_CUDA_OK(cudaFuncSetAttribute(bwd_tc_intra_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)intra_smem()));
  int sms = 0, dev = 0;
  LL_CUDA_OK(cudaGetDevice(&dev));
  LL_CUDA_OK(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
  const int items = N * BH;
  const int pgrid = std::max(1, std::min(items, sms));  // the persistent kernels: one CTA per SM
  // the intra kernel's outputs by tensor stores where the maps can be made
  CUtensorMap tdq, tdk, tdv, tS;
  const uint64_t srows = (uint64_t)BH * N * kD;
  const int use_omap = use_tma && srows <= 0x7fffffffull && tile_map(&tdq, b.dqp, rows) &&
                       tile_map(&tdk, b.dkp, rows) && tile_map(&tdv, b.dvp, rows) && f32_box_map(&tS, b.S, srows);
  bwd_tc_intra_kernel<<<pgrid, kIntraThreads, intra_smem(), a.stream>>>(
      tq, tk, tv, tg, use_tma, tdq, tdk, tdv, tS, use_omap, q, k, v, dout, a.log_alpha, a.lam, b.dqp, b.dkp, b.dvp, a.dlam, b.S, b.tot, b.dc, s.T,
      s.L, N, BH, qctr, b.err);
  LL_CUDA_OK(cudaGetLastError());
  // the query kernel reads the nodes' bf16 tiles only: no float32 copy where the Fenwick kernel can skip it
  const ll_status fs = simt_fenwick_launch(b.S, b.F, b.tot, b.G, N, kD * kD, BH, a.stream, b.Ft, b.cum, false);
  if (fs != LL_OK) return fs;
  // the key-side nodes' rows by tensor reductions where their row coordinate fits
  const uint64_t rrows = (uint64_t)BH * N * kD;
  CUtensorMap tr;
  const int use_rmap = rrows <= 0x7fffffffull && f32_box_map(&tr, b.R, rrows);
  LL_CUDA_OK(cudaFuncSetAttribute(bwd_tc_query_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)query_smem()));
  // dq's two parts in and out by TMA where the maps can be made
  CUtensorMap tdi, tdo;
  const int use_dmap = use_tma && tile_map(&tdi, b.dqp, rows) && tile_map(&tdo, a.dq, rows);
  bwd_tc_query_kernel<<<pgrid, kQryThreads, query_smem(), a.stream>>>(
      tq, tg, use_tma, tr, use_rmap, tdi, tdo, use_dmap, q, dout, a.log_alpha, a.lam, b.Ft, b.G, b.dqp, static_cast<__nv_bfloat16*>(a.dq),
      a.dlam, b.R, s.T, s.L, N, BH, qctr, b.err);
  LL_CUDA_OK(cudaGetLastError());
  LL_CUDA_OK(cudaFuncSetAttribute(bwd_tc_key_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)key_smem()));
  // dk's and dv's two parts in and out by TMA where the maps can be made
  CUtensorMap tkpi, tvpi, tko, tvo;
  const int use_kmap = use_tma && tile_map(&tkpi, b.dkp, rows) && tile_map(&tvpi, b.dvp, rows) &&
                       tile_map(&tko, a.dk, rows) && tile_map(&tvo, a.dv, rows);
  bwd_tc_key_kernel<<<grid, kThreads, key_smem(), a.stream>>>(
      tk, tv, use_tma, tkpi, tvpi, tko, tvo, use_kmap, k, v, a.log_alpha, a.lam, a.dlam, b.R, b.cum, b.dkp, b.dvp, static_cast<__nv_bfloat16*>(a.dk),
      static_cast<__nv_bfloat16*>(a.dv), b.dc, s.T, s.L, b.err);
  LL_CUDA_OK(cudaGetLastError());
  return LL_OK;
}

}  // namespace llattn
