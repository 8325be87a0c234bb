// Log-linear Mamba-2 forward on the 5th-generation tensor cores (tcgen05,
// TMEM accumulators, TMA-staged bf16 operands), one persistent kernel.
//
// The sequence of each head is cut into 128-token tiles (the MMA M).  Tile j
// of head bh does, with cs = inclusive cumsum of log_alpha inside the tile:
//   state   S_j = sum_s exp(cs_127 - cs_s) v_s k_s^T           (Vt^T K, 128x128x128)
//   Fenwick F_j = S_j + sum_{m < cto(j)} exp(dec_m) F_{j-2^m}   (cto = trailing ones)
//           published to global memory (bf16) with its log-decay total G_j
//   intra   P = (Q K^T) . exp(cs_t - cs_s) . lam_t[bitlen(t^s)] (s <= t), O = P V
//   inter   for each set bit h of j: D_h = Q F_e^T with
//           e = (j with bits 0..h cleared) + 2^h - 1, and
//           O += lam_t[8 + h] exp(cs_t + sum of G over the lower set bits) D_h
// ("Log-Linear Attention" study note §3-4/§3-5; chunk-wise scan of the
// gist.science (zh) summary §2.3; the per-level contractions are summed in
// one accumulator per tile, the pages' "level fusion".)
//
// Roles (320 threads, one CTA per SM, persistent; tiles u = blockIdx.x +
// i * gridDim.x, interleaved across heads: u = j * (B*H) + bh, so that the
// tiles running at the same time are few positions of many heads and the
// chains of node dependencies inside one round of tiles stay short):
//   warp 0      TMA producer: K, V, Q tiles, log_alpha + lambda rows, F nodes
//               (after their publication flags are seen)
//   warp 1      TMEM owner and MMA issuer (one thread)
//   warps 2..9  epilogue: thread (quadrant q = warp % 4, half hf) owns row
//               32q + lane and columns [64 hf, 64 hf + 64) of every 128x128
//               accumulator
//   warp 10     publisher: makes each written node visible at gpu scope and
//               raises its flag, off the epilogue's path
// Cross-CTA dependencies only point to tiles of lower index, every CTA walks
// its tiles in increasing order, and the cooperative launch makes all CTAs
// co-resident, so the waits always make progress.  Every wait is bounded;
// a wait that expires records LL_ERR_TIMEOUT and the kernel runs on to its
// end without the missing data.
#include <cudaTypedefs.h>

#include <atomic>

#include "common.cuh"
#include "sm100.cuh"

namespace llattn {

namespace {

using namespace sm100;

constexpr int kTile = 128;
constexpr int kD = 128;
constexpr int kLmax = 24;
constexpr int kThreads = 352;
constexpr int kPubWarp = 10;
constexpr int kEpi = 256;
constexpr uint32_t kHalf = kTile * 64 * 2;  // one [128 x 64] bf16 swizzled block: 16 KB
constexpr uint32_t kTileBytes = 2 * kHalf;  // 32 KB
constexpr float kLog2e = 1.4426950408889634f;
constexpr uint64_t kTimeoutNs = 4000000000ull;

// TMEM columns of the four 128-column fp32 accumulators
constexpr uint32_t kTmState = 0, kTmS = 128, kTmO = 256, kTmLvl = 384;

// shared-memory layout (offsets from a 1024-aligned base)
constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffK = kOffQ + kTileBytes;
constexpr uint32_t kOffV = kOffK + kTileBytes;
constexpr uint32_t kOffX = kOffV + kTileBytes;  // decayed V, then P
constexpr uint32_t kOffF0 = kOffX + kTileBytes;
constexpr uint32_t kOffF1 = kOffF0 + kTileBytes;
constexpr uint32_t kAuxBytes = kTile * 4 + kTile * kLmax * 4;  // log_alpha row + lambda rows
constexpr uint32_t kOffAux0 = kOffF1 + kTileBytes;
constexpr uint32_t kOffAux1 = kOffAux0 + kAuxBytes;
constexpr uint32_t kOffCs = kOffAux1 + kAuxBytes;      // float[128] cumsum x log2(e)
constexpr uint32_t kOffCol = kOffCs + kTile * 4;       // float[128] exp(cs_e - cs_s), e = end of s's 32-group
constexpr uint32_t kOffMisc = kOffCol + kTile * 4;     // quadrant totals, tmem base, abort flag
constexpr uint32_t kOffBars = kOffMisc + 64;             // mbarriers

// mbarriers (all with arrival count 1: one producer arrive + TMA bytes, one
// tcgen05.commit, or one elected epilogue thread)
enum Bar : int {
  B_KV_FULL, B_Q_FULL, B_AUX_FULL0, B_AUX_FULL1, B_F_FULL0, B_F_FULL1, B_F_FREE0, B_F_FREE1, B_KV_FREE,
  B_Q_FREE, B_AUX_FREE0, B_AUX_FREE1, B_VT_READY, B_STATE_DONE, B_STATE_FREE, B_S_DONE, B_S_FREE, B_P_READY,
  B_LVL_DONE, B_LVL_FREE, B_O_DONE, B_O_FREE, B_FINAL, B_FJ_WRITTEN, kNumBars
};
constexpr uint32_t kSmemBytes = kOffBars + kNumBars * 8 + 1024;  // + slack to align the base to 1024
static_assert(kSmemBytes <= 232448, "shared memory budget of one CTA");

struct TcParams {
  const float* log_alpha;
  const float* lam;
  const __nv_bfloat16* q;
  const __nv_bfloat16* k;
  const __nv_bfloat16* v;
  __nv_bfloat16* o;
  __nv_bfloat16* F;  // [BH * Nt, 128, 128] Fenwick nodes
  float* G;          // [BH * Nt] log-decay totals of the nodes
  uint64_t* flags;   // [BH * Nt] publication tokens
  uint64_t* abort_word;
  uint64_t token;
  int BH, T, Nt, L;
  unsigned* err;
};

struct Ctx {
  unsigned char* base;
  uint64_t* bars;
  volatile int* abort_s;
  const TcParams* p;
};

__device__ __forceinline__ void note_abort(const Ctx& c) {
  if (!*c.abort_s) {
    *c.abort_s = 1;
    atomicOr(c.p->err, kErrTimeout);
    *reinterpret_cast<volatile uint64_t*>(c.p->abort_word) = c.p->token;
  }
}

// Bounded wait for the completion of the phase with parity `par` of barrier `b`.
__device__ __forceinline__ void wait_bar(const Ctx& c, int b, uint32_t par) {
  uint64_t* bar = c.bars + b;
  if (mbar_try_wait(bar, par)) return;
  if (*c.abort_s) return;
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, par)) {
    if (*c.abort_s) return;
    if (globaltimer_ns() - t0 > kTimeoutNs) {
      note_abort(c);
      return;
    }
  }
}

// The same for a whole warp: every lane leaves together (converged), so the
// warp-collective tcgen05 loads and named barriers that follow see a full warp.
__device__ __forceinline__ void wait_bar_w(const Ctx& c, int b, uint32_t par) {
  uint64_t* bar = c.bars + b;
  bool ok = mbar_try_wait(bar, par);
  if (__all_sync(0xffffffffu, ok)) return;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    ok = ok || mbar_try_wait(bar, par);
    if (__all_sync(0xffffffffu, ok)) return;
    if (__any_sync(0xffffffffu, *c.abort_s != 0)) return;
    const bool late = globaltimer_ns() - t0 > kTimeoutNs;
    if (__any_sync(0xffffffffu, late)) {
      if ((threadIdx.x & 31) == 0) note_abort(c);
      __syncwarp();
      return;
    }
  }
}

// Final drain at exit: bounded, ignores the abort flag.
__device__ __forceinline__ void drain_bar(const Ctx& c, int b, uint32_t par) {
  uint64_t* bar = c.bars + b;
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, par))
    if (globaltimer_ns() - t0 > kTimeoutNs / 8) return;
}

// Bounded wait until node `idx` of this call is published.
__device__ __forceinline__ void wait_flag(const Ctx& c, size_t idx) {
  const uint64_t* f = c.p->flags + idx;
  if (ld_acquire_u64(f) == c.p->token) return;
  if (*c.abort_s) return;
  const uint64_t t0 = globaltimer_ns();
  unsigned ns = 32;
  while (ld_acquire_u64(f) != c.p->token) {
    __nanosleep(ns);
    if (ns < 128) ns <<= 1;
    if (*c.abort_s) return;
    if (*reinterpret_cast<volatile uint64_t*>(c.p->abort_word) == c.p->token) {
      *c.abort_s = 1;
      return;
    }
    if (globaltimer_ns() - t0 > kTimeoutNs) {
      note_abort(c);
      return;
    }
  }
}

// Warp-uniform version of wait_flag (all lanes wait for the same node).
__device__ __forceinline__ void wait_flag_w(const Ctx& c, size_t idx) {
  if ((threadIdx.x & 31) == 0) wait_flag(c, idx);
  __syncwarp();
  // every lane acquires the flag itself, so its own later loads are ordered after it
  (void)ld_acquire_u64(c.p->flags + idx);
}

// 2^x with the hardware approximation (relative error ~2^-22, flushes
// subnormals): ample for factors that end in bf16 operands.
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ int node_of_level(int j, int h) { return ((j >> (h + 1)) << (h + 1)) + (1 << h) - 1; }

// K-major operand (rows of 128 B, K split in two 64-column blocks), k-step kk of 16.
__device__ __forceinline__ uint64_t desc_k(uint32_t tile, int kk) {
  return sw128_desc(tile + (kk >> 2) * kHalf + (kk & 3) * 32, 16, 1024);
}
// MN-major operand (rows = K, 64-element M/N blocks 16 KB apart), k-step kk of 16 rows.
__device__ __forceinline__ uint64_t desc_mn(uint32_t tile, int kk) { return sw128_desc(tile + kk * 2048, kHalf, 1024); }

// ------------------------------------------------------------------ producer
__device__ void producer(const Ctx& c, const CUtensorMap* tq, const CUtensorMap* tk, const CUtensorMap* tv,
                         const CUtensorMap* tf) {
  const TcParams& p = *c.p;
  const int total = p.BH * p.Nt;
  uint32_t it = 0, fcnt = 0;
  unsigned char* s = c.base;
  for (int u = blockIdx.x; u < total; u += gridDim.x, ++it) {
    const int bh = u % p.BH, j = u / p.BH;
    const int row0 = bh * p.T + j * kTile;
    // stage the next tile's inputs in L2 while this one is processed
    const int un = u + gridDim.x;
    if (un < total) {
      const size_t rn = (size_t)(un % p.BH) * p.T + (size_t)(un / p.BH) * kTile;
      bulk_prefetch_l2(p.q + rn * kD, kTileBytes);
      bulk_prefetch_l2(p.k + rn * kD, kTileBytes);
      bulk_prefetch_l2(p.v + rn * kD, kTileBytes);
      bulk_prefetch_l2(p.log_alpha + rn, kTile * 4);
      bulk_prefetch_l2(p.lam + rn * p.L, (uint32_t)(kTile * p.L * 4));
    }
    // K, V
    if (it > 0) wait_bar(c, B_KV_FREE, (it - 1) & 1);
    mbar_arrive_expect_tx(c.bars + B_KV_FULL, 2 * kTileBytes);
    tma_load_2d(s + kOffK, tk, c.bars + B_KV_FULL, 0, row0);
    tma_load_2d(s + kOffK + kHalf, tk, c.bars + B_KV_FULL, 64, row0);
    tma_load_2d(s + kOffV, tv, c.bars + B_KV_FULL, 0, row0);
    tma_load_2d(s + kOffV + kHalf, tv, c.bars + B_KV_FULL, 64, row0);
    // log_alpha + lambda rows
    const int slot = it & 1;
    if (it >= 2) wait_bar(c, B_AUX_FREE0 + slot, ((it - 2) >> 1) & 1);
    unsigned char* aux = s + (slot ? kOffAux1 : kOffAux0);
    const uint32_t lam_bytes = (uint32_t)(kTile * p.L * 4);
    mbar_arrive_expect_tx(c.bars + B_AUX_FULL0 + slot, kTile * 4 + lam_bytes);
    bulk_load(aux, p.log_alpha + (size_t)row0, kTile * 4, c.bars + B_AUX_FULL0 + slot);
    bulk_load(aux + kTile * 4, p.lam + (size_t)row0 * p.L, lam_bytes, c.bars + B_AUX_FULL0 + slot);
    // Q
    if (it > 0) wait_bar(c, B_Q_FREE, (it - 1) & 1);
    mbar_arrive_expect_tx(c.bars + B_Q_FULL, kTileBytes);
    tma_load_2d(s + kOffQ, tq, c.bars + B_Q_FULL, 0, row0);
    tma_load_2d(s + kOffQ + kHalf, tq, c.bars + B_Q_FULL, 64, row0);
    // Fenwick nodes of the inter-tile levels, lowest level first
    for (int h = 0; (j >> h) != 0; ++h) {
      if (!((j >> h) & 1)) continue;
      const int e = node_of_level(j, h);
      const size_t node = (size_t)bh * p.Nt + e;
      wait_flag(c, node);
      fence_proxy_async_global();
      const int fs = fcnt & 1;
      if (fcnt >= 2) wait_bar(c, B_F_FREE0 + fs, ((fcnt - 2) >> 1) & 1);
      unsigned char* fdst = s + (fs ? kOffF1 : kOffF0);
      mbar_arrive_expect_tx(c.bars + B_F_FULL0 + fs, kTileBytes);
      tma_load_2d(fdst, tf, c.bars + B_F_FULL0 + fs, 0, (int)(node * kD));
      tma_load_2d(fdst + kHalf, tf, c.bars + B_F_FULL0 + fs, 64, (int)(node * kD));
      ++fcnt;
    }
  }
  // drain: every load armed above has landed before the CTA may exit
  if (it > 0) {
    drain_bar(c, B_KV_FULL, (it - 1) & 1);
    drain_bar(c, B_Q_FULL, (it - 1) & 1);
    const uint32_t last = it - 1;
    drain_bar(c, B_AUX_FULL0 + (last & 1), (last >> 1) & 1);
    if (it >= 2) drain_bar(c, B_AUX_FULL0 + ((last - 1) & 1), ((last - 1) >> 1) & 1);
  }
  if (fcnt > 0) drain_bar(c, B_F_FULL0 + ((fcnt - 1) & 1), ((fcnt - 1) >> 1) & 1);
  if (fcnt > 1) drain_bar(c, B_F_FULL0 + ((fcnt - 2) & 1), ((fcnt - 2) >> 1) & 1);
}

// ------------------------------------------------------------------ MMA issuer
__device__ void mma_issuer(const Ctx& c, uint32_t tmem) {
  const TcParams& p = *c.p;
  const int total = p.BH * p.Nt;
  const uint32_t sQ = smem_u32(c.base + kOffQ), sK = smem_u32(c.base + kOffK), sV = smem_u32(c.base + kOffV),
                 sX = smem_u32(c.base + kOffX), sF0 = smem_u32(c.base + kOffF0), sF1 = smem_u32(c.base + kOffF1);
  constexpr uint32_t id_state = idesc_bf16(128, 128, true, true);   // Vt^T (MN) x K (MN)
  constexpr uint32_t id_qk = idesc_bf16(128, 128, false, false);    // Q (K) x K|F (K)
  constexpr uint32_t id_pv = idesc_bf16(128, 128, false, true);     // P (K) x V (MN)
  uint32_t it = 0, fcnt = 0, lcnt = 0;

  auto issue_level = [&]() {
    const int fs = fcnt & 1;
    wait_bar(c, B_F_FULL0 + fs, (fcnt >> 1) & 1);
    if (lcnt > 0) wait_bar(c, B_LVL_FREE, (lcnt - 1) & 1);
    tc_fence_after();
    const uint32_t sF = fs ? sF1 : sF0;
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) umma_bf16(tmem + kTmLvl, desc_k(sQ, kk), desc_k(sF, kk), id_qk, kk > 0);
    umma_commit(c.bars + B_LVL_DONE);
    umma_commit(c.bars + B_F_FREE0 + fs);
    ++fcnt;
    ++lcnt;
  };

  for (int u = blockIdx.x; u < total; u += gridDim.x, ++it) {
    const int j = u / p.BH;
    // chunk state: D[dv][dk] = sum_s Vt[s][dv] K[s][dk]
    wait_bar(c, B_KV_FULL, it & 1);
    wait_bar(c, B_VT_READY, it & 1);
    if (it > 0) wait_bar(c, B_STATE_FREE, (it - 1) & 1);
    tc_fence_after();
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) umma_bf16(tmem + kTmState, desc_mn(sX, kk), desc_mn(sK, kk), id_state, kk > 0);
    umma_commit(c.bars + B_STATE_DONE);
    // scores: D[t][s] = Q[t] . K[s]
    wait_bar(c, B_Q_FULL, it & 1);
    if (it > 0) wait_bar(c, B_S_FREE, (it - 1) & 1);
    tc_fence_after();
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) umma_bf16(tmem + kTmS, desc_k(sQ, kk), desc_k(sK, kk), id_qk, kk > 0);
    umma_commit(c.bars + B_S_DONE);
    const int nlev = __popc(j);
    // intra output (issued before the levels, which may wait for other tiles' nodes): D[t][dv] = sum_s P[t][s] V[s][dv]
    wait_bar(c, B_P_READY, it & 1);
    if (it > 0) wait_bar(c, B_O_FREE, (it - 1) & 1);
    tc_fence_after();
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) umma_bf16(tmem + kTmO, desc_k(sX, kk), desc_mn(sV, kk), id_pv, kk > 0);
    umma_commit(c.bars + B_O_DONE);
    umma_commit(c.bars + B_KV_FREE);
    for (int l = 0; l < nlev; ++l) issue_level();
    umma_commit(c.bars + B_Q_FREE);
  }
  umma_commit(c.bars + B_FINAL);
  drain_bar(c, B_FINAL, 0);
}

// ------------------------------------------------------------------ epilogue

__device__ void epilogue(const Ctx& c, uint32_t tmem, int warp, int lane) {
  const TcParams& p = *c.p;
  const int total = p.BH * p.Nt;
  const int q = warp & 3;
  const int hf = (warp - 2) >> 2;
  const int row = 32 * q + lane;
  const bool leader = (warp == 2 && lane == 0);
  const uint32_t tl = tmem + ((uint32_t)(32 * q) << 16);  // this warp's lane quadrant
  unsigned char* s = c.base;
  float* cs_s = reinterpret_cast<float*>(s + kOffCs);
  float* col_s = reinterpret_cast<float*>(s + kOffCol);
  float* qtot = reinterpret_cast<float*>(s + kOffMisc);
  uint32_t it = 0, lcnt = 0;

  for (int u = blockIdx.x; u < total; u += gridDim.x, ++it) {
    const int bh = u % p.BH, j = u / p.BH;
    const int slot = it & 1;
    const float* la_s = reinterpret_cast<const float*>(s + (slot ? kOffAux1 : kOffAux0));
    const float* lam_s = la_s + kTile;
    wait_bar_w(c, B_AUX_FULL0 + slot, (it >> 1) & 1);

    // inclusive cumsum of log_alpha over the tile
    float x = la_s[row];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (hf == 0 && lane == 31) qtot[q] = x;
    __syncwarp();
    named_bar_sync(1, kEpi);
    float off = 0.f;
    for (int qq = 0; qq < q; ++qq) off += qtot[qq];
    const float cs_t = x + off;
    const float cs2_t = cs_t * kLog2e;                                   // base-2 log decay
    const float cs2_grp_end = __shfl_sync(0xffffffffu, cs2_t, 31);      // end of this 32-group
    if (hf == 0) {
      cs_s[row] = cs2_t;
      col_s[row] = ex2(cs2_grp_end - cs2_t);
    }
    __syncwarp();
    named_bar_sync(1, kEpi);
    const float cs2_end = cs_s[kTile - 1];
    const float cs_end = cs2_end * 0.69314718055994531f;  // natural log decay of the whole tile

    // decayed V for the chunk state: X[s] = exp(cs_end - cs_s) V[s]
    wait_bar_w(c, B_KV_FULL, it & 1);
    {
      const float dec = ex2(cs2_end - cs2_t);
      const uint32_t off_row = hf * kHalf + row * 128;
      const uint4* src = reinterpret_cast<const uint4*>(s + kOffV + off_row);
      uint4* dst = reinterpret_cast<uint4*>(s + kOffX + off_row);
#pragma unroll
      for (int c8 = 0; c8 < 8; ++c8) {
        const int cc = c8 ^ (row & 7);  // lanes of a warp spread over the banks
        uint4 v = src[cc];
        uint32_t* w = reinterpret_cast<uint32_t*>(&v);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float2 f = unpack_bf16x2(w[i]);
          w[i] = pack_bf16x2(f.x * dec, f.y * dec);
        }
        dst[cc] = v;
      }
    }
    fence_proxy_async_shared();
    __syncwarp();
    named_bar_sync(1, kEpi);
    if (leader) mbar_arrive(c.bars + B_VT_READY);

    // chunk state -> Fenwick node F_j, published for later tiles
    wait_bar_w(c, B_STATE_DONE, it & 1);
    __syncwarp();
    tc_fence_after();
    float acc[64];
    tmem_ld32(tl + kTmState + 64 * hf, acc);
    tmem_ld32(tl + kTmState + 64 * hf + 32, acc + 32);
    tmem_ld_wait();
    tc_fence_before();
    __syncwarp();
    named_bar_sync(1, kEpi);
    if (leader) mbar_arrive(c.bars + B_STATE_FREE);
    {
      const size_t node_j = (size_t)bh * p.Nt + j;
      float dec = cs_end;  // log decay from the end of node j - 2^m to the end of tile j
      for (int m = 0; (j >> m) & 1; ++m) {
        const size_t node = node_j - ((size_t)1 << m);
        wait_flag_w(c, node);
        const uint4* src = reinterpret_cast<const uint4*>(p.F + (node * kD + row) * kD + 64 * hf);
        const float sc = exp2f(dec * kLog2e);
#pragma unroll
        for (int c8 = 0; c8 < 8; ++c8) {
          const uint4 v = src[c8];
          const uint32_t* w = reinterpret_cast<const uint32_t*>(&v);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float2 f = unpack_bf16x2(w[i]);
            acc[c8 * 8 + 2 * i] = fmaf(sc, f.x, acc[c8 * 8 + 2 * i]);
            acc[c8 * 8 + 2 * i + 1] = fmaf(sc, f.y, acc[c8 * 8 + 2 * i + 1]);
          }
        }
        dec += p.G[node];
      }
      uint4* dst = reinterpret_cast<uint4*>(p.F + (node_j * kD + row) * kD + 64 * hf);
#pragma unroll
      for (int c8 = 0; c8 < 8; ++c8) {
        uint4 v;
        uint32_t* w = reinterpret_cast<uint32_t*>(&v);
#pragma unroll
        for (int i = 0; i < 4; ++i) w[i] = pack_bf16x2(acc[c8 * 8 + 2 * i], acc[c8 * 8 + 2 * i + 1]);
        dst[c8] = v;
      }
      if (leader) p.G[node_j] = dec;
      __syncwarp();
      named_bar_sync(1, kEpi);  // every row of F_j is written (CTA scope)
      if (leader) mbar_arrive(c.bars + B_FJ_WRITTEN);  // the publisher warp makes it visible
    }

    // masked scores -> P (bf16, K-major swizzled) in X.  Thread row t, column
    // groups g of 32:  g < q (all s < t): the level is constant over the group
    // and exp(cs_t - cs_s) = exp(cs_t - cs_e) exp(cs_e - cs_s), e = 32 g + 31,
    // the second factor from the per-tile table;  g == q: per element;
    // g > q: zero.
    const float* lam_row = lam_s + row * p.L;
    wait_bar_w(c, B_S_DONE, it & 1);
    __syncwarp();
    tc_fence_after();
#pragma unroll
    for (int c32 = 0; c32 < 2; ++c32) {
      const int g = 2 * hf + c32;
      const int s0 = 32 * g;
      float v[32];
      if (g < q) {
        tmem_ld32(tl + kTmS + s0, v);
        const float rf = lam_row[32 - __clz(row ^ s0)] * ex2(cs2_t - cs_s[s0 + 31]);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] *= rf * col_s[s0 + i];
      } else if (g == q) {
        tmem_ld32(tl + kTmS + s0, v);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const float e = ex2(cs2_t - cs_s[s0 + i]) * lam_row[32 - __clz(lane ^ i)];
          v[i] = (i <= lane) ? v[i] * e : 0.f;
        }
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = 0.f;
      }
      unsigned char* xrow = s + kOffX + hf * kHalf + row * 128;
#pragma unroll
      for (int u4 = 0; u4 < 4; ++u4) {
        const int c8 = 4 * c32 + u4;
        uint4 w;
        w.x = pack_bf16x2(v[8 * u4 + 0], v[8 * u4 + 1]);
        w.y = pack_bf16x2(v[8 * u4 + 2], v[8 * u4 + 3]);
        w.z = pack_bf16x2(v[8 * u4 + 4], v[8 * u4 + 5]);
        w.w = pack_bf16x2(v[8 * u4 + 6], v[8 * u4 + 7]);
        *reinterpret_cast<uint4*>(xrow + ((c8 ^ (row & 7)) << 4)) = w;
      }
    }
    tc_fence_before();
    fence_proxy_async_shared();
    __syncwarp();
    named_bar_sync(1, kEpi);
    if (leader) {
      mbar_arrive(c.bars + B_S_FREE);
      mbar_arrive(c.bars + B_P_READY);
    }

    // inter-tile levels, accumulated in registers with their per-row weights
    float oacc[64];
#pragma unroll
    for (int i = 0; i < 64; ++i) oacc[i] = 0.f;
    float D = 0.f;
    for (int h = 0; (j >> h) != 0; ++h) {
      if (!((j >> h) & 1)) continue;
      const size_t node = (size_t)bh * p.Nt + node_of_level(j, h);
      const float w = lam_s[row * p.L + 8 + h] * exp2f((cs_t + D) * kLog2e);
      wait_bar_w(c, B_LVL_DONE, lcnt & 1);
      __syncwarp();
      tc_fence_after();
#pragma unroll
      for (int c32 = 0; c32 < 2; ++c32) {
        float v[32];
        tmem_ld32(tl + kTmLvl + 64 * hf + 32 * c32, v);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 32; ++i) oacc[32 * c32 + i] = fmaf(w, v[i], oacc[32 * c32 + i]);
      }
      tc_fence_before();
      __syncwarp();
    named_bar_sync(1, kEpi);
      if (leader) mbar_arrive(c.bars + B_LVL_FREE);
      ++lcnt;
      wait_flag_w(c, node);
      D += p.G[node];
    }

    // output = intra + inter, bf16
    wait_bar_w(c, B_O_DONE, it & 1);
    __syncwarp();
    tc_fence_after();
    {
      __nv_bfloat16* orow = p.o + ((size_t)bh * p.T + (size_t)j * kTile + row) * kD + 64 * hf;
#pragma unroll
      for (int c32 = 0; c32 < 2; ++c32) {
        float v[32];
        tmem_ld32(tl + kTmO + 64 * hf + 32 * c32, v);
        tmem_ld_wait();
#pragma unroll
        for (int u4 = 0; u4 < 4; ++u4) {
          uint4 w;
          const float* a = oacc + 32 * c32 + 8 * u4;
          const float* b = v + 8 * u4;
          w.x = pack_bf16x2(a[0] + b[0], a[1] + b[1]);
          w.y = pack_bf16x2(a[2] + b[2], a[3] + b[3]);
          w.z = pack_bf16x2(a[4] + b[4], a[5] + b[5]);
          w.w = pack_bf16x2(a[6] + b[6], a[7] + b[7]);
          reinterpret_cast<uint4*>(orow)[4 * c32 + u4] = w;
        }
      }
    }
    tc_fence_before();
    __syncwarp();
    named_bar_sync(1, kEpi);
    if (leader) {
      mbar_arrive(c.bars + B_O_FREE);
      mbar_arrive(c.bars + B_AUX_FREE0 + slot);
    }
  }
}

// ------------------------------------------------------------------ publisher (warp 10)
// Makes each tile's node visible at gpu scope and raises its flag, so the
// epilogue never stalls on the fence.
__device__ void publisher(const Ctx& c) {
  const TcParams& p = *c.p;
  const int total = p.BH * p.Nt;
  uint32_t it = 0;
  for (int u = blockIdx.x; u < total; u += gridDim.x, ++it) {
    const size_t node_j = (size_t)(u % p.BH) * p.Nt + u / p.BH;
    wait_bar(c, B_FJ_WRITTEN, it & 1);
    __threadfence();
    st_release_u64(p.flags + node_j, p.token);
  }
}

__global__ void __launch_bounds__(kThreads, 1)
    fwd_tc_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                  const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tf, TcParams p) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* base =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + kOffBars);
  volatile int* abort_s = reinterpret_cast<volatile int*>(base + kOffMisc + 16);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base + kOffMisc + 32);
  Ctx c{base, bars, abort_s, &p};

  if (threadIdx.x == 0) {
    *abort_s = 0;
    for (int b = 0; b < kNumBars; ++b) mbar_init(bars + b, 1);
    fence_mbar_init();
    prefetch_tmap(&tq);
    prefetch_tmap(&tk);
    prefetch_tmap(&tv);
    prefetch_tmap(&tf);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) producer(c, &tq, &tk, &tv, &tf);
  } else if (warp == 1) {
    if (lane == 0) mma_issuer(c, tmem);
  } else if (warp == kPubWarp) {
    if (lane == 0) publisher(c);
  } else {
    epilogue(c, tmem, warp, lane);
  }
  __syncwarp();

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// Level states of position T read from the Fenwick nodes (float32, decayed to T-1).
__global__ void __launch_bounds__(256) tc_export_kernel(const __nv_bfloat16* __restrict__ F,
                                                        const float* __restrict__ G, float* __restrict__ state_out,
                                                        float* __restrict__ scale_out, int Nt, int Ls) {
  const size_t bh = blockIdx.y;
  const int idx = blockIdx.x * 256 + threadIdx.x;  // < 128 * 128
  constexpr int mat = kD * kD;
  float D = 0.f;
  for (int slot = 0; slot < Ls; ++slot) {
    const int h = slot + 1 - 8;  // level slot+1 = 8 + h
    float val = 0.f, sc = 0.f;
    if (h >= 0 && h < 31 && ((Nt >> h) & 1)) {
      const size_t e = bh * Nt + node_of_level(Nt, h);
      val = exp2f(D * kLog2e) * __bfloat162float(F[e * mat + idx]);
      sc = 1.f;
      D += G[e];
    }
    state_out[(bh * Ls + slot) * (size_t)mat + idx] = val;
    if (blockIdx.x == 0 && threadIdx.x == 0) scale_out[bh * Ls + slot] = sc;
  }
}

// ------------------------------------------------------------------ host side
struct TcPlan {
  int Nt;
  size_t off_F, off_G, off_flags, total;
};

TcPlan tc_plan(const ll_shape& s) {
  TcPlan p{};
  p.Nt = s.T / kTile;
  const size_t nodes = (size_t)s.B * s.H * p.Nt;
  size_t off = 0;
  p.off_F = off;     off = align_up(off + nodes * kD * kD * 2, 1024);
  p.off_G = off;     off = align_up(off + nodes * 4, 256);
  p.off_flags = off; off = align_up(off + (nodes + 1) * 8, 256);
  p.total = off;
  return p;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::atomic<bool> tried{false};
  if (!fn && !tried.exchange(true)) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  return fn;
}

// 2-D bf16 tensor map over [rows, 128] with [128 x 64] boxes, 128-byte swizzle.
bool make_map(CUtensorMap* m, const void* base, uint64_t rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)kD, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)kD * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)kTile};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

uint64_t next_token() {
  static std::atomic<uint64_t> counter{0x5eed};
  uint64_t x = counter.fetch_add(1) + 0x9E3779B97F4A7C15ull;
  x = (x ^ (x >> 30)) * 0xBF58476D1CE4E5B9ull;
  x = (x ^ (x >> 27)) * 0x94D049BB133111EBull;
  x ^= x >> 31;
  return x | 1ull;
}

}  // namespace

bool fwd_tc_supported(const ll_shape& s) {
  return s.io == LL_BF16 && s.dk == kD && s.dv == kD && s.T % kTile == 0 && s.L <= kLmax &&
         (long long)s.B * s.H * s.T <= (1ll << 31) - 1;
}

size_t fwd_tc_workspace(const ll_shape& s) { return tc_plan(s).total; }

int fwd_tc_launches(const ll_shape& s) { return s.Ls > 0 ? 2 : 1; }

ll_status fwd_tc_launch(const FwdArgs& a) {
  const ll_shape& s = a.s;
  const TcPlan plan = tc_plan(s);
  if (a.ws_bytes < plan.total) return LL_ERR_WORKSPACE;
  unsigned char* ws = static_cast<unsigned char*>(a.ws);
  const int BH = s.B * s.H;
  const uint64_t rows = (uint64_t)BH * s.T;
  const uint64_t node_rows = (uint64_t)BH * plan.Nt * kD;
  CUtensorMap tq, tk, tv, tf;
  if (!make_map(&tq, a.q, rows) || !make_map(&tk, a.k, rows) || !make_map(&tv, a.v, rows) ||
      !make_map(&tf, ws + plan.off_F, node_rows))
    return LL_ERR_CUDA;

  TcParams p;
  p.log_alpha = a.log_alpha;
  p.lam = a.lam;
  p.q = static_cast<const __nv_bfloat16*>(a.q);
  p.k = static_cast<const __nv_bfloat16*>(a.k);
  p.v = static_cast<const __nv_bfloat16*>(a.v);
  p.o = static_cast<__nv_bfloat16*>(a.o);
  p.F = reinterpret_cast<__nv_bfloat16*>(ws + plan.off_F);
  p.G = reinterpret_cast<float*>(ws + plan.off_G);
  p.flags = reinterpret_cast<uint64_t*>(ws + plan.off_flags);
  p.abort_word = p.flags + (size_t)BH * plan.Nt;
  p.token = next_token();
  p.BH = BH;
  p.T = s.T;
  p.Nt = plan.Nt;
  p.L = s.L;
  p.err = a.err;

  int dev = 0, sms = 0, per_sm = 0;
  LL_CUDA_OK(cudaGetDevice(&dev));
  LL_CUDA_OK(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
  LL_CUDA_OK(cudaFuncSetAttribute(fwd_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes));
  LL_CUDA_OK(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fwd_tc_kernel, kThreads, kSmemBytes));
  if (per_sm < 1) return LL_ERR_CUDA;
  const long long tiles = (long long)BH * plan.Nt;
  const int grid = (int)std::min<long long>(tiles, (long long)sms * per_sm);

  void* args[] = {&tq, &tk, &tv, &tf, &p};
  LL_CUDA_OK(cudaLaunchCooperativeKernel((const void*)fwd_tc_kernel, dim3(grid), dim3(kThreads), args, kSmemBytes,
                                         a.stream));
  if (a.state_out) {
    tc_export_kernel<<<dim3(kD * kD / 256, BH), 256, 0, a.stream>>>(p.F, p.G, a.state_out, a.scale_out, plan.Nt,
                                                                   s.Ls);
    LL_CUDA_OK(cudaGetLastError());
  }
  return LL_OK;
}

}  // namespace llattn
