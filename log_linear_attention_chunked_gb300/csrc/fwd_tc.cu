// Log-linear Mamba-2 forward on the 5th-generation tensor cores (tcgen05,
// TMEM accumulators, TMA-staged bf16 operands), one persistent kernel.
//
// The sequence of each head is cut into 128-token tiles (the MMA M).  Tile j
// of head bh does, with cs = inclusive cumsum of log_alpha inside the tile:
//   intra   P = (Q K^T) . exp(cs_t - cs_s) . lam_t[bitlen(t^s)] (s <= t), O = P V
//   state   S_j = sum_s v_s exp(cs_127 - cs_s) k_s^T           (V^T Kdec, 128x128x128)
//   Fenwick F_j = S_j + sum_{m < cto(j)} exp(dec_m) F_{j-2^m}   (cto = trailing ones)
//           published to global memory (bf16) with its log-decay total G_j
//   inter   for each set bit h of j, with e = (j with bits 0..h cleared) +
//           2^h - 1:  O += Q'_h F_e^T,  Q'_h[t] = lam_t[8 + h] exp(cs_t + sum
//           of G over the lower set bits) Q[t]  (the row weights go on Q, so
//           the tensor cores accumulate every level onto the output)
// ("Log-Linear Attention" study note §3-4/§3-5; chunk-wise scan of the
// gist.science (zh) summary §2.3; the per-level contractions are summed in
// one accumulator per tile, the pages' "level fusion".)
// A prefill continuation (tiles at absolute index c0t + j, c0t a multiple of
// the smallest power of two >= the segment's tile count) walks the bits of
// c0t + j: the bits of c0t are further levels whose nodes are the prefix
// buckets of the decode states, written as bf16 nodes before this kernel.
//
// Roles (512 threads in four warpgroups, one CTA per SM, persistent; tiles
// u = blockIdx.x + i * gridDim.x, interleaved across heads: u = j * (B*H) +
// bh, so that the tiles running at the same time are few positions of many
// heads and the chains of node dependencies inside one wave stay short):
//   warp 0      K, V, Q loads (TMA) and the L2 prefetch of the next tile; Q
//               has one buffer, loaded for the tile's scores and again for
//               its inter-tile levels one step later (an L2 hit)
//   warp 1      TMEM owner and MMA issuer (one thread)
//   warp 2      output stores (TMA) from the staging buffer
//   warp 3      the level nodes of the previous tile (two-slot ring), once
//               their publication words are seen, and their log decays
//   warps 4-11  epilogue: thread (quadrant q = warp % 4, half hf) owns row
//               32q + lane of the score / output accumulators
//   warps 12-15 node warps, one per TMEM lane quadrant: the tile's chunk
//               state from its own TMEM accumulator, the merge of the
//               Fenwick children F_{j-2^m} (each waited for and loaded by
//               TMA), the node's store and its gpu-scope publication
// Step i of the epilogue: the front half of tile i (cumsum, K decayed in
// place once the scores have read it, masked scores P back into TMEM), then
// the back half of tile i-1 (level-weighted Q for each level product, the
// output read out and staged).  The MMA issues per step: scores(i), the
// chunk state(i) into the node warps' accumulator (once they have released
// it), the levels of tile i-1 onto its output, then PV(i) into the output
// accumulator once tile i-1's output has been read.  The node warps publish
// each node as soon as its children are published, independently of the
// epilogue, so a node never waits behind a back half.
// With one decay per level (log_alpha [T, L], column l the decay of level l)
// the same roles run with per-level factors: a key's log decay splits into a
// key part K(s, l) and a query part Q(t, l) of the same level (the steps it
// spends on the levels below l, and those on l from the start of t's block;
// see the CUDA-core kernels of the per-level forward).  The epilogue builds
// them per row from quadrant-local scans of the in-tile levels 1..7 (the
// mask, the K decay exp(K(s, 8)) of the chunk state), and keeps the in-tile
// running sums of the inter-tile levels for the back half; the decays across
// tiles (the level producer's, and the node warps' child decays) come from a
// table of per-level running sums over the tiles written by a small kernel
// before this one.
// Cross-CTA dependencies only point to tiles of lower index, every role
// walks its tiles in increasing order, and the cooperative launch makes all
// CTAs co-resident, so the waits always make progress.  Every wait is
// bounded; a wait that expires records LL_ERR_TIMEOUT and the kernel runs on
// to its end without the missing data.
#include <cudaTypedefs.h>
#include <cuda_fp16.h>

#include <atomic>

#include "level_decay.cuh"
#include "sm100.cuh"

namespace llattn {

namespace {

using namespace sm100;

constexpr int kTile = 128;
constexpr int kD = 128;
constexpr int kLmax = 24;
constexpr int kThreads = 512;
constexpr int kEpiWarp0 = 4;    // warps 4..11
constexpr int kNodeWarp0 = 12;  // warps 12..15
constexpr int kEpi = 256;
constexpr int kNodeThreads = 128;
constexpr uint32_t kHalf = kTile * 64 * 2;  // one [128 x 64] bf16 swizzled block: 16 KB
constexpr uint32_t kTileBytes = 2 * kHalf;  // 32 KB
constexpr float kLog2e = 1.4426950408889634f;
constexpr uint64_t kTimeoutNs = 4000000000ull;  // default limit of a bounded wait

// TMEM columns: the output accumulator (PV, then + the inter-tile levels);
// the scores (then P, bf16, in their first 64 columns); two 64-column buffers
// of level-weighted Q (bf16), the A operand of the level products; the node
// warps' accumulator (the chunk state, then + the merged children).
constexpr uint32_t kTmR = 0, kTmS = 128, kTmQP = 256, kTmM = 384;

// shared memory (offsets from the dynamic base, which must be 1024-aligned)
constexpr uint32_t kOffQ = 0;                      // Q: for the scores, then again for the levels
constexpr uint32_t kOffK = kOffQ + kTileBytes;     // K, decayed in place for the chunk state
constexpr uint32_t kOffV = kOffK + kTileBytes;
constexpr uint32_t kOffF0 = kOffV + kTileBytes;    // level-node ring
constexpr uint32_t kOffF1 = kOffF0 + kTileBytes;
constexpr uint32_t kOffC = kOffF1 + kTileBytes;    // node warps: merge children, then the node
constexpr uint32_t kOffX = kOffC + kTileBytes;     // output staging
constexpr uint32_t kOffCs = kOffX + kTileBytes;    // float[128] cumsum x log2(e); per-level mode:
                                                   // float[4][16] quadrant totals of levels 1..16
constexpr uint32_t kOffCol = kOffCs + kTile * 4;   // float[128] exp(cs_e - cs_s), e = end of s's 32-group
constexpr uint32_t kOffLam = kOffCol + kTile * 4;  // half[6][128] lambda levels 0..5 / the row's max;
                                                   // per-level mode: half[6][128] exp(K(s, l)), l = 1..6
// levels of log_alpha the per-level mode reads per row: 1..7 in the tile,
// 8..15 across tiles (so T <= 32768 on this path)
constexpr int kLdLv = 15;
// misc: epilogue quadrant totals [0,16), abort flag 16, tmem base 32, node-warp totals [48,64)
constexpr uint32_t kOffMisc = kOffLam + 6 * kTile * 2;
// level producer -> epilogue: the level log decays of the previous tile
// (float[2][16], by step parity) at 0 and the step-tagged count of levels
// whose decay is ready (u32[2]) at 160; node leader -> node warps: the
// child's log-decay total at 176
constexpr uint32_t kOffNode = kOffMisc + 64;
constexpr uint32_t kOffBars = kOffNode + 192;  // mbarriers

// mbarriers (all with arrival count 1: one producer arrive + TMA bytes, one
// tcgen05.commit, or one elected thread)
enum Bar : int {
  B_K_FULL, B_V_FULL, B_QS_FULL, B_QB_FULL, B_Q_FREE, B_K_FREE, B_V_FREE, B_F_FULL0, B_F_FULL1, B_F_FREE0,
  B_F_FREE1, B_S_DONE, B_KDEC, B_P_READY, B_QP_FULL0, B_QP_FULL1, B_QP_FREE0, B_QP_FREE1, B_O_READY, B_R_FREE,
  B_STATE_DONE, B_M_FREE, B_C_FULL, B_X_STAGED, B_X_FREE, B_LVLD_FREE, B_FINAL, kNumBars
};
constexpr uint32_t kSmemBytes = kOffBars + kNumBars * 8;
static_assert(kSmemBytes <= 232448, "shared memory budget of one CTA");

struct TcParams {
  const float* log_alpha;
  const float* lam;
  const __nv_bfloat16* q;
  const __nv_bfloat16* k;
  const __nv_bfloat16* v;
  __nv_bfloat16* F;  // [BH * Nt, 128, 128] Fenwick nodes
  float* G;          // [BH * Nt] log-decay totals of the nodes
  // [BH * Nt] publication words: this call's token in the high half, the
  // node's log-decay total in the low half, so one atomic load gives both
  uint64_t* flags;
  uint64_t* abort_word;
  uint32_t token;    // per call, never 0
  int BH, T, Nt, L;  // T: rows between the (b, h) slices of the inputs
  // prefill continuation: absolute index of the first tile (a multiple of the
  // smallest power of two >= Nt, so its set bits lie above every tile's own);
  // its levels read the prefix nodes at F[BH * Nt + bh * kPreSlots + h]
  int c0t;
  unsigned* err;
  uint64_t timeout_ns;  // limit of every bounded wait
  long long withhold;   // node whose publication is withheld (expiry test), or -1
  // head size of q, k, v and o (64 or 128): with 64 the operand tiles are
  // filled to 128 columns with zeros by the TMA (its out-of-range fill), every
  // product runs as at 128, and only the first 64 output columns are stored
  int d;
};

// Per-level mode: running sums over the tiles of each inter-tile level's log
// decays, cumL[(bh * Lx + h) * Nt + j] = sum over tiles 0..j of level 8 + h,
// Lx = max(L - 8, 1); the table follows the publication words (and the abort
// word) in the workspace.
__device__ __forceinline__ int ld_levels(const TcParams& p) { return p.L > 9 ? p.L - 8 : 1; }
__device__ __forceinline__ const double* ld_table(const TcParams& p) {
  return reinterpret_cast<const double*>(p.flags + (size_t)p.BH * p.Nt + 1);
}

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
    *reinterpret_cast<volatile uint64_t*>(c.p->abort_word) = ((uint64_t)c.p->token << 32) | 0xffffffffu;
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
    if (globaltimer_ns() - t0 > c.p->timeout_ns) {
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
    const bool late = globaltimer_ns() - t0 > c.p->timeout_ns;
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

__device__ __forceinline__ bool flag_ok(const Ctx& c, uint64_t w) { return (uint32_t)(w >> 32) == c.p->token; }
__device__ __forceinline__ float flag_g(uint64_t w) { return __uint_as_float((uint32_t)w); }
__device__ __forceinline__ bool aborted_elsewhere(const Ctx& c) {
  return flag_ok(c, *reinterpret_cast<volatile uint64_t*>(c.p->abort_word));
}

// Bounded wait until entry `idx` of the word array `flags` carries this
// call's token (acquire); returns the word.
__device__ __forceinline__ uint64_t wait_flag(const Ctx& c, const uint64_t* flags, size_t idx) {
  const uint64_t* f = flags + idx;
  uint64_t w = ld_acquire_u64(f);
  if (flag_ok(c, w) || *c.abort_s) return w;
  const uint64_t t0 = globaltimer_ns();
  unsigned ns = 32;
  while (!flag_ok(c, w = ld_acquire_u64(f))) {
    __nanosleep(ns);
    if (ns < 128) ns <<= 1;
    if (*c.abort_s) return w;
    if (aborted_elsewhere(c)) {
      *c.abort_s = 1;
      return w;
    }
    if (globaltimer_ns() - t0 > c.p->timeout_ns) {
      note_abort(c);
      return w;
    }
  }
  return w;
}

// 2^x with the hardware approximation (relative error ~2^-22, flushes
// subnormals): ample for factors that end in bf16 operands.
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ int node_of_level(int j, int h) { return ((j >> (h + 1)) << (h + 1)) + (1 << h) - 1; }

// prefix nodes (continuation) per head: one per tile height
constexpr int kPreSlots = 16;

// The roles are instantiated for kCont = false (the forward from position 0,
// no prefix levels) and kCont = true (a continuation), and with kLD (one
// decay per level; from position 0 only).
template <bool kCont> __device__ __forceinline__ int start_tile(const TcParams& p) { return kCont ? p.c0t : 0; }

// Per-level mode: the log decay of level 8 + h over tiles [a, b) of head bh.
__device__ __forceinline__ float ld_span(const TcParams& p, int bh, int h, int a, int b) {
  if (b <= a) return 0.f;
  const double* cl = ld_table(p) + ((size_t)bh * ld_levels(p) + h) * p.Nt;
  return (float)(__ldg(cl + b - 1) - (a > 0 ? __ldg(cl + a - 1) : 0.0));
}

// Number of tiles CTA blockIdx.x processes (blockIdx.x < total).
__device__ __forceinline__ int tiles_of_cta(int total) { return (total - 1 - (int)blockIdx.x) / (int)gridDim.x + 1; }

// K-major operand (rows of 128 B, K split in two 64-column blocks), k-step kk of 16.
__device__ __forceinline__ uint64_t desc_k(uint32_t tile, int kk) {
  return sw128_desc(tile + (kk >> 2) * kHalf + (kk & 3) * 32, 16, 1024);
}
// MN-major operand (rows = K, 64-element M/N blocks 16 KB apart), k-step kk of 16 rows.
__device__ __forceinline__ uint64_t desc_mn(uint32_t tile, int kk) { return sw128_desc(tile + kk * 2048, kHalf, 1024); }

// L2 prefetch of the 16-byte-aligned interior of [ptr, ptr + bytes): a bulk
// prefetch needs a 16-byte-aligned start and size, which the rows of
// log_alpha and lam do not have when the row stride between heads is not a
// multiple of the tile
__device__ __forceinline__ void prefetch_l2_inside(const void* ptr, uint32_t bytes) {
  const uintptr_t a = reinterpret_cast<uintptr_t>(ptr);
  const uintptr_t lo = (a + 15) & ~(uintptr_t)15, hi = (a + bytes) & ~(uintptr_t)15;
  if (hi > lo) bulk_prefetch_l2(reinterpret_cast<const void*>(lo), (uint32_t)(hi - lo));
}

// ------------------------------------------------------------------ producers (warps 0 and 3)
// Warp 0 streams K, Q and V of every tile, and Q once more for the tile's
// levels one step later: per step, K(i), Q(i) (the scores' copy), V(i), then
// Q(i-1) again (the levels' copy) -- the one Q buffer alternates between the
// two uses, each load waiting for the previous use to release it.
template <bool kLD>
__device__ void producer_kvq(const Ctx& c, const CUtensorMap* tq, const CUtensorMap* tk, const CUtensorMap* tv) {
  const TcParams& p = *c.p;
  const int n = tiles_of_cta(p.BH * p.Nt);
  uint32_t kc = 0, vc = 0, qs = 0, qb = 0, ql = 0;
  unsigned char* s = c.base;
  auto load_q = [&](int row0, int bar) {
    if (ql > 0) wait_bar(c, B_Q_FREE, (ql - 1) & 1);
    if (*c.abort_s) return false;
    mbar_arrive_expect_tx(c.bars + bar, kTileBytes);
    tma_load_2d(s + kOffQ, tq, c.bars + bar, 0, row0);
    tma_load_2d(s + kOffQ + kHalf, tq, c.bars + bar, 64, row0);
    ++ql;
    return true;
  };
  int row_prev = 0;
  for (int it = 0; it <= n && !*c.abort_s; ++it) {
    const int u = blockIdx.x + it * gridDim.x;
    const int row0 = it < n ? (u % p.BH) * p.T + (u / p.BH) * kTile : 0;
    if (it < n) {
      // stage the next tile's inputs in L2 while this one is processed
      if (it + 1 < n) {
        const int un = u + gridDim.x;
        const size_t rn = (size_t)(un % p.BH) * p.T + (size_t)(un / p.BH) * kTile;
        const uint32_t tb = (uint32_t)(kTile * p.d * 2);  // one tile of q, k or v
        bulk_prefetch_l2(p.q + rn * p.d, tb);
        bulk_prefetch_l2(p.k + rn * p.d, tb);
        bulk_prefetch_l2(p.v + rn * p.d, tb);
        const int la_row = kLD ? p.L : 1;  // floats of log_alpha per token
        prefetch_l2_inside(p.log_alpha + rn * la_row, (uint32_t)(kTile * la_row * 4));
        prefetch_l2_inside(p.lam + rn * p.L, (uint32_t)(kTile * p.L * 4));
      }
      if (it > 0) wait_bar(c, B_K_FREE, (it - 1) & 1);  // the previous state product has read K
      if (*c.abort_s) break;
      mbar_arrive_expect_tx(c.bars + B_K_FULL, kTileBytes);
      tma_load_2d(s + kOffK, tk, c.bars + B_K_FULL, 0, row0);
      tma_load_2d(s + kOffK + kHalf, tk, c.bars + B_K_FULL, 64, row0);
      ++kc;
      // Q before V: the scores need it first, and V waits for the previous PV
      if (!load_q(row0, B_QS_FULL)) break;
      ++qs;
      if (it > 0) wait_bar(c, B_V_FREE, (it - 1) & 1);  // PV and the state product have read V
      if (*c.abort_s) break;
      mbar_arrive_expect_tx(c.bars + B_V_FULL, kTileBytes);
      tma_load_2d(s + kOffV, tv, c.bars + B_V_FULL, 0, row0);
      tma_load_2d(s + kOffV + kHalf, tv, c.bars + B_V_FULL, 64, row0);
      ++vc;
    }
    if (it >= 1) {
      if (!load_q(row_prev, B_QB_FULL)) break;
      ++qb;
    }
    row_prev = row0;
  }
  // drain: every copy armed above has landed before the CTA may exit
  if (kc > 0) drain_bar(c, B_K_FULL, (kc - 1) & 1);
  if (vc > 0) drain_bar(c, B_V_FULL, (vc - 1) & 1);
  if (qs > 0) drain_bar(c, B_QS_FULL, (qs - 1) & 1);
  if (qb > 0) drain_bar(c, B_QB_FULL, (qb - 1) & 1);
}

// Warp 3 runs the F ring (two 32 KB slots) of the level nodes for
// the MMA.  Per step i it acquires the Fenwick nodes of tile i-1's levels in
// order, hands each level's log decay to the epilogue (a step-tagged count
// released in shared memory, so the epilogue starts on level 0 before later
// nodes are published) and loads the node.  Once a wait has expired nothing
// new is armed.
template <bool kCont, bool kLD>
__device__ void producer_levels(const Ctx& c, const CUtensorMap* tf) {
  const TcParams& p = *c.p;
  const int n = tiles_of_cta(p.BH * p.Nt);
  unsigned char* s = c.base;
  float* dl = reinterpret_cast<float*>(s + kOffNode);               // [2][16]
  uint32_t* nlr = reinterpret_cast<uint32_t*>(s + kOffNode + 160);  // [2]
  uint32_t fcnt = 0;
  for (int it = 1; it <= n && !*c.abort_s; ++it) {
    const int up = blockIdx.x + (it - 1) * gridDim.x;
    const int bhp = up % p.BH, jp = up / p.BH;
    // the back half two steps ago is done (so is every earlier one, among
    // them the reader of this parity's decays); every back half waits for
    // this step's tag, so that barrier never runs two phases ahead
    if (it >= 2) wait_bar(c, B_LVLD_FREE, (it - 2) & 1);
    st_release_cta_u32(nlr + (it & 1), (uint32_t)it << 8);
    float D = 0.f;
    uint32_t l = 0;
    const int ja = jp | start_tile<kCont>(p);  // absolute tile index: the segment's bits, then the start tile's
    for (int h = 0; (ja >> h) != 0 && !*c.abort_s; ++h) {
      if (!((ja >> h) & 1)) continue;
      // a prefix level (continuation) holds the prefix bucket, decayed to the
      // segment start and written before this kernel: no word to wait for,
      // and every later prefix level shares the same decay D
      const bool pre = kCont && !((jp >> h) & 1);
      const size_t node = pre ? (size_t)p.BH * p.Nt + (size_t)bhp * kPreSlots + h
                              : (size_t)bhp * p.Nt + node_of_level(jp, h);
      // the decay from the end of the node's block to the start of the tile:
      // the node totals of the lower set bits, or (per-level mode) level
      // 8 + h's own decays over those tiles (read before the node's wait)
      const float dlv = kLD ? ld_span(p, bhp, h, jp & ~((1 << h) - 1), jp) : 0.f;
      float g = 0.f;
      if (!pre) {
        const uint64_t w = wait_flag(c, p.flags, node);
        fence_proxy_async_global();
        g = flag_g(w);
      }
      dl[16 * (it & 1) + l] = kLD ? dlv : D;
      D += g;
      st_release_cta_u32(nlr + (it & 1), ((uint32_t)it << 8) | ++l);
      const int fs = fcnt & 1;
      if (fcnt >= 2) wait_bar(c, B_F_FREE0 + fs, ((fcnt - 2) >> 1) & 1);
      if (*c.abort_s) break;
      unsigned char* dst = s + (fs ? kOffF1 : kOffF0);
      mbar_arrive_expect_tx(c.bars + B_F_FULL0 + fs, kTileBytes);
      tma_load_2d(dst, tf, c.bars + B_F_FULL0 + fs, 0, (int)(node * kD));
      tma_load_2d(dst + kHalf, tf, c.bars + B_F_FULL0 + fs, 64, (int)(node * kD));
      ++fcnt;
    }
  }
  if (fcnt > 0) drain_bar(c, B_F_FULL0 + ((fcnt - 1) & 1), ((fcnt - 1) >> 1) & 1);
  if (fcnt > 1) drain_bar(c, B_F_FULL0 + ((fcnt - 2) & 1), ((fcnt - 2) >> 1) & 1);
}

// ------------------------------------------------------------------ MMA issuer
template <bool kCont>
__device__ void mma_issuer(const Ctx& c, uint32_t tmem) {
  const TcParams& p = *c.p;
  const int n = tiles_of_cta(p.BH * p.Nt);
  const uint32_t sQ = smem_u32(c.base + kOffQ), sK = smem_u32(c.base + kOffK), sV = smem_u32(c.base + kOffV),
                 sF0 = smem_u32(c.base + kOffF0), sF1 = smem_u32(c.base + kOffF1);
  constexpr uint32_t id_state = idesc_bf16(128, 128, true, true);  // V^T (MN) x Kdec (MN)
  constexpr uint32_t id_qk = idesc_bf16(128, 128, false, false);   // Q (K) x K (K); Q' (TMEM) x F (K)
  constexpr uint32_t id_pv = idesc_bf16(128, 128, false, true);    // P (TMEM) x V (MN)
  uint32_t fcnt = 0, qpc = 0;

  // one inter-tile level of the previous tile, accumulated onto its output:
  // D[t][dv] += Q'[t] . F[dv], Q' = the level-weighted Q from the epilogue (TMEM)
  auto issue_level = [&](auto&& wait) {
    const int b = qpc & 1;
    const int fs = fcnt & 1;
    wait(B_F_FULL0 + fs, (fcnt >> 1) & 1);
    wait(B_QP_FULL0 + b, (qpc >> 1) & 1);
    tc_fence_after();
    const uint32_t sF = fs ? sF1 : sF0;
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) umma_bf16_ta(tmem + kTmR, tmem + kTmQP + 64 * b + kk * 8, desc_k(sF, kk), id_qk, 1);
    umma_commit(c.bars + B_QP_FREE0 + b);
    umma_commit(c.bars + B_F_FREE0 + fs);
    ++fcnt;
    ++qpc;
  };
  // chunk state: D[dv][dk] = sum_s V[s][dv] Kdec[s][dk], into the node warps' accumulator
  auto issue_state = [&]() {
    tc_fence_after();
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) umma_bf16(tmem + kTmM, desc_mn(sV, kk), desc_mn(sK, kk), id_state, kk > 0);
    umma_commit(c.bars + B_STATE_DONE);
    umma_commit(c.bars + B_K_FREE);
  };

  // a deferred state product goes out as soon as M and V are ready, checked
  // while this thread waits for anything else
  bool state_pending = false;
  uint32_t m_par = 0;  // parity of the M release the pending state needs
  int pend_it = 0;
  auto try_state = [&]() {
    if (state_pending && mbar_test_wait(c.bars + B_M_FREE, m_par) && mbar_test_wait(c.bars + B_V_FULL, pend_it & 1)) {
      issue_state();
      state_pending = false;
    }
  };
  auto wait_mma = [&](int b, uint32_t par) {
    if (mbar_try_wait(c.bars + b, par)) return;
    if (*c.abort_s) return;
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(c.bars + b, par)) {
      try_state();
      if (*c.abort_s) return;
      if (globaltimer_ns() - t0 > p.timeout_ns) {
        note_abort(c);
        return;
      }
    }
  };

  int jp = 0;
  for (int it = 0; it <= n; ++it) {
    const int u = blockIdx.x + it * gridDim.x;
    const int j = it < n ? u / p.BH : 0;
    const int nlev_p = it >= 1 ? __popc(jp | start_tile<kCont>(p)) : 0;
    if (it < n) {
      // scores: D[t][s] = Q[t] . K[s]
      wait_bar(c, B_K_FULL, it & 1);
      wait_bar(c, B_QS_FULL, it & 1);
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) umma_bf16(tmem + kTmS, desc_k(sQ, kk), desc_k(sK, kk), id_qk, kk > 0);
      umma_commit(c.bars + B_S_DONE);
      umma_commit(c.bars + B_Q_FREE);
      // the state as soon as K is decayed and V has landed, unless the node
      // warps still hold the previous tile's node (then after this step's
      // other products)
      wait_bar(c, B_KDEC, it & 1);
      if ((it == 0 || mbar_test_wait(c.bars + B_M_FREE, (it - 1) & 1)) && mbar_test_wait(c.bars + B_V_FULL, it & 1)) {
        issue_state();
      } else {
        state_pending = true;
        m_par = (it - 1) & 1;
        pend_it = it;
        if (it == 0) m_par = 1;  // no previous node: M is free (phase parity 1 reads as complete)
      }
    }
    if (it >= 1) {
      for (int l = 0; l < nlev_p; ++l) issue_level(wait_mma);
      umma_commit(c.bars + B_O_READY);  // PV of the previous tile + its levels
    }
    if (it < n) {
      // intra output: D[t][dv] = sum_s P[t][s] V[s][dv], P from TMEM, once the
      // previous tile's output has been read out of the accumulator
      wait_mma(B_V_FULL, it & 1);
      wait_mma(B_P_READY, it & 1);
      if (it >= 1) wait_mma(B_R_FREE, (it - 1) & 1);
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) umma_bf16_ta(tmem + kTmR, tmem + kTmS + kk * 8, desc_mn(sV, kk), id_pv, kk > 0);
      if (state_pending) {
        wait_bar(c, B_M_FREE, m_par);
        issue_state();
        state_pending = false;
      }
      umma_commit(c.bars + B_V_FREE);  // PV and the state product have read V
    }
    jp = j;
  }
  umma_commit(c.bars + B_FINAL);
  drain_bar(c, B_FINAL, 0);
}

// ------------------------------------------------------------------ epilogue (warps 4..11)
template <bool kCont, bool kLD>
__device__ void epilogue(const Ctx& c, uint32_t tmem, int warp, int lane) {
  const TcParams& p = *c.p;
  const int total = p.BH * p.Nt;
  const int n = tiles_of_cta(total);
  const int q = warp & 3;
  const int hf = (warp - kEpiWarp0) >> 2;
  const int row = 32 * q + lane;
  const bool leader = (warp == kEpiWarp0 && lane == 0);
  const uint32_t tl = tmem + ((uint32_t)(32 * q) << 16);  // this warp's lane quadrant
  unsigned char* s = c.base;
  float* cs_s = reinterpret_cast<float*>(s + kOffCs);
  float* col_s = reinterpret_cast<float*>(s + kOffCol);
  __half* lamh = reinterpret_cast<__half*>(s + kOffLam);
  float* qtot = reinterpret_cast<float*>(s + kOffMisc);
  uint32_t qpc = 0;  // level-weighted Q tiles written (two TMEM buffers)
  uint32_t xs = 0;   // outputs staged

  // this row's log_alpha (per-level mode: levels 1..kLdLv) and intra-level
  // lambdas, read one tile ahead
  float la_n = 0.f, lam_n[8], lal_n[kLD ? kLdLv : 1];
  auto fetch = [&](int u) {
    const size_t r = (size_t)(u % p.BH) * p.T + (size_t)(u / p.BH) * kTile + row;
    if constexpr (kLD) {
      const float* ar = p.log_alpha + r * p.L;
#pragma unroll
      for (int m = 0; m < kLdLv; ++m) lal_n[m] = m + 1 < p.L ? __ldg(ar + m + 1) : 0.f;
    } else {
      la_n = __ldg(p.log_alpha + r);
    }
    const float* lr = p.lam + r * p.L;
#pragma unroll
    for (int l = 0; l < 8; ++l) lam_n[l] = __ldg(lr + l);
  };
  fetch(blockIdx.x);
  __half* kfh = reinterpret_cast<__half*>(s + kOffLam);  // per-level mode: exp(K(s, l)), l = 1..6
  float* qtl = reinterpret_cast<float*>(s + kOffCs);     // per-level mode: quadrant totals [4][16]

  // The front half's prologue of the CTA's k-th tile: the values of a row
  // that depend on the tile's inputs alone (its cumsum or, per level, the key
  // and query parts of its decays, and the level weights) and the per-tile
  // tables in shared memory.  It runs one tile ahead -- in the previous back
  // half, once that half has handed its first level over -- so that a front half
  // starts at its scores; the tables are free by then (the front half before
  // has read them before its last barrier).  The per-level mode runs it at
  // the start of the front half instead: held across a back half, its
  // per-row state would not fit the epilogue's registers.
  float n_cs_t = 0.f, n_cs2_t = 0.f, n_cs2_diag = 0.f, n_cs2_end = 0.f, n_lam6 = 0.f, n_lam7 = 0.f;
  float n_kdec2 = 0.f, n_rf6 = 0.f, n_rf7 = 0.f, n_gf0 = 0.f, n_rowq[kLD ? 6 : 1], n_csI[kLD ? 8 : 1];
  auto prologue = [&](int k) {
    const float la = la_n;
    float lam[8], lal[kLD ? kLdLv : 1];
#pragma unroll
    for (int l = 0; l < 8; ++l) lam[l] = lam_n[l];
    if constexpr (kLD) {
#pragma unroll
      for (int m = 0; m < kLdLv; ++m) lal[m] = lal_n[m];
    }
    if (k + 1 < n) fetch(blockIdx.x + (k + 1) * gridDim.x);

    // per-level mode: the key and query parts of the log decays of this row
    float kdec2 = 0.f, rf6 = 0.f, rf7 = 0.f, gf0 = 0.f, rowq[kLD ? 6 : 1];
    float cs_t = 0.f, cs2_t = 0.f, cs2_diag = 0.f, cs2_end = 0.f;
    float csI[kLD ? 8 : 1];
#pragma unroll
    for (int h = 0; h < (kLD ? 8 : 1); ++h) csI[h] = 0.f;
    if constexpr (kLD) {
      // quadrant-local running sums of levels 1..kLdLv (levels l = m + 1)
      float cp[kLdLv];
#pragma unroll
      for (int m = 0; m < kLdLv; ++m) {
        float x = lal[m];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const float y = __shfl_up_sync(0xffffffffu, x, o);
          if (lane >= o) x += y;
        }
        cp[m] = x;
      }
      if (hf == 0 && lane == 31) {
#pragma unroll
        for (int m = 0; m < kLdLv; ++m) qtl[q * 16 + m] = cp[m];
      }
      __syncwarp();
      named_bar_sync(1, kEpi);
      // Q(t, l): level l's decays from the start of t's block of 2^(l-1)
      // rows through t; inside the quadrant for l <= 6, the quadrant pair for l = 7
      float qf[6];
      qf[0] = 0.f;
#pragma unroll
      for (int l = 1; l <= 5; ++l) {
        const int src = ((lane >> (l - 1)) << (l - 1)) - 1;
        const float pv = __shfl_sync(0xffffffffu, cp[l - 1], src < 0 ? 0 : src);
        qf[l] = cp[l - 1] - (src < 0 ? 0.f : pv);
      }
      const float qf6 = cp[5];
      const float qf7 = cp[6] + ((q & 1) ? qtl[(q - 1) * 16 + 6] : 0.f);
      // K(t, l): the decays of the sibling blocks above t at the levels
      // below l (bit m-1 of t clear: the next 2^(m-1) rows, at level m)
      float kf[9], K = 0.f;
      kf[1] = 0.f;
#pragma unroll
      for (int m = 1; m <= 5; ++m) {
        const int ss = ((lane >> m) << m) + (1 << (m - 1)), se = ss + (1 << (m - 1)) - 1;
        const float a1 = __shfl_sync(0xffffffffu, cp[m - 1], se & 31);
        const float a0 = __shfl_sync(0xffffffffu, cp[m - 1], (ss - 1) & 31);
        if (!((lane >> (m - 1)) & 1)) K += a1 - a0;
        kf[m + 1] = K;
      }
      if (!(q & 1)) K += qtl[(q + 1) * 16 + 5];
      kf[7] = K;
      if (q < 2) K += qtl[2 * 16 + 6] + qtl[3 * 16 + 6];
      kf[8] = K;
      kdec2 = kf[8] * kLog2e;
      rowq[0] = lam[0];
#pragma unroll
      for (int l = 1; l <= 5; ++l) rowq[l] = lam[l] * ex2(qf[l] * kLog2e);
      rf6 = lam[6] * ex2(qf6 * kLog2e);
      rf7 = lam[7] * ex2(qf7 * kLog2e);
      gf0 = ex2(qtl[16 + 5] * kLog2e);  // keys of group 0 pass group 1 at level 6 on their way to level 7
#pragma unroll
      for (int h = 0; h < 8; ++h) {
        float off = 0.f;
        for (int qq = 0; qq < q; ++qq) off += qtl[qq * 16 + 7 + h];
        csI[h] = cp[7 + h] + off;
      }
      if (hf == 0) {
#pragma unroll
        for (int l = 1; l <= 6; ++l) kfh[(l - 1) * kTile + row] = __float2half_rn(ex2(kf[l] * kLog2e));
      }
      __syncwarp();
      named_bar_sync(1, kEpi);
    } else {
      // inclusive cumsum of log_alpha over the tile
      float x = la;
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
      cs_t = x + off;
      cs2_t = cs_t * kLog2e;                               // base-2 log decay
      const float cs2_grp_end = __shfl_sync(0xffffffffu, cs2_t, 31);  // end of this 32-group
      if (hf == 0) {
        cs_s[row] = cs2_t;
        col_s[row] = ex2(cs2_grp_end - cs2_t);
      }
      // lambda of levels 0..5 (the diagonal group), relative to the row's
      // largest, as half; the largest rides in the exponent
      float lmax = 0.f;
#pragma unroll
      for (int l = 0; l < 6; ++l) lmax = fmaxf(lmax, lam[l]);
      cs2_diag = cs2_t + (lmax > 0.f ? __log2f(lmax) : -INFINITY);
      if (hf == 0) {
        const float inv = lmax > 0.f ? 1.f / lmax : 0.f;
#pragma unroll
        for (int l = 0; l < 6; ++l) lamh[l * kTile + row] = __float2half_rn(lam[l] * inv);
      }
      __syncwarp();
      named_bar_sync(1, kEpi);
      cs2_end = cs_s[kTile - 1];
    }
    n_cs_t = cs_t;
    n_cs2_t = cs2_t;
    n_cs2_diag = cs2_diag;
    n_cs2_end = cs2_end;
    n_lam6 = lam[6];
    n_lam7 = lam[7];
    n_kdec2 = kdec2;
    n_rf6 = rf6;
    n_rf7 = rf7;
    n_gf0 = gf0;
#pragma unroll
    for (int l = 0; l < (kLD ? 6 : 1); ++l) n_rowq[l] = kLD ? rowq[l] : 0.f;
#pragma unroll
    for (int h = 0; h < (kLD ? 8 : 1); ++h) n_csI[h] = csI[h];
  };
  if (!kLD) prologue(0);

  float cs_prev = 0.f, lam_c = 0.f;
  float csI_prev[kLD ? 8 : 1];  // per-level mode: in-tile running sums of levels 8..15 (previous tile)
#pragma unroll
  for (int h = 0; h < (kLD ? 8 : 1); ++h) csI_prev[h] = 0.f;
  int jp = 0, bhp = 0;
  for (int it = 0; it <= n; ++it) {
    const int u = blockIdx.x + it * gridDim.x;
    int bh = 0, j = 0;
    float cs_t = 0.f;
    float csI[kLD ? 8 : 1];
#pragma unroll
    for (int h = 0; h < (kLD ? 8 : 1); ++h) csI[h] = 0.f;
    if (it < n) {
      // ================= front half of tile it
      bh = u % p.BH;
      j = u / p.BH;
      const int jap = jp | start_tile<kCont>(p);  // the previous tile's absolute index bits
      if (it >= 1 && jap != 0)  // the previous tile's first level lambda, ahead of its back half
        lam_c = __ldg(p.lam + ((size_t)bhp * p.T + (size_t)jp * kTile + row) * p.L + 8 + (__ffs(jap) - 1));
      // this tile's values from its prologue (run one tile ahead; in the
      // per-level mode, whose prologue holds more per-row state, here)
      if (kLD) prologue(it);
      cs_t = n_cs_t;
      const float cs2_t = n_cs2_t, cs2_diag = n_cs2_diag, cs2_end = n_cs2_end, lam6 = n_lam6, lam7 = n_lam7;
      const float kdec2 = n_kdec2, rf6 = n_rf6, rf7 = n_rf7, gf0 = n_gf0;
      float rowq[kLD ? 6 : 1];
#pragma unroll
      for (int l = 0; l < (kLD ? 6 : 1); ++l) rowq[l] = n_rowq[l];
#pragma unroll
      for (int h = 0; h < (kLD ? 8 : 1); ++h) csI[h] = n_csI[h];

      // scores ready: K has been read by them, so it is decayed in place for
      // the chunk state, K[s] <- exp(cs_end - cs_s) K[s]
      wait_bar_w(c, B_S_DONE, it & 1);
      __syncwarp();
      tc_fence_after();
      {
        const float dec = kLD ? ex2(kdec2) : ex2(cs2_end - cs2_t);
        uint4* kr = reinterpret_cast<uint4*>(s + kOffK + hf * kHalf + row * 128);
#pragma unroll
        for (int c8 = 0; c8 < 8; ++c8) {
          const int cc = c8 ^ (row & 7);  // lanes of a warp spread over the banks
          uint4 v = kr[cc];
          uint32_t* w = reinterpret_cast<uint32_t*>(&v);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float2 f = unpack_bf16x2(w[i]);
            w[i] = pack_bf16x2(f.x * dec, f.y * dec);
          }
          kr[cc] = v;
        }
      }
      fence_proxy_async_shared();
      __syncwarp();
      named_bar_sync(1, kEpi);
      if (leader) mbar_arrive(c.bars + B_KDEC);

      // masked scores -> P (bf16) back into the scores' TMEM columns.  This
      // thread takes columns 32 g + 16 hf + [0, 16) of each 32-group g, so
      // both warps of a quadrant share its diagonal group.  g < q (all s < t):
      // the level (6 or 7) is constant over the group and exp(cs_t - cs_s) =
      // exp(cs_t - cs_e) exp(cs_e - cs_s), e = 32 g + 31, the second factor
      // from the per-tile table;  g == q: per element, levels 0..5 from the
      // half table;  g > q: zero.
      uint32_t pw[2][8];
#pragma unroll
      for (int g = 0; g < 4; ++g) {
        const int s0 = 32 * g + 16 * hf;
        float v[16];
        if (g < q) {
          tmem_ld16(tl + kTmS + s0, v);
          float rf, cf[16];
          if constexpr (kLD) {
            // level 6 (q ^ g == 1): Q(t, 6) K(s, 6); level 7: Q(t, 7) K(s, 7),
            // K(s, 7) = K(s, 6) + group 1's level-6 decay for keys of group 0
            rf = (q ^ g) == 1 ? rf6 : rf7 * (g == 0 ? gf0 : 1.f);
            const uint4* kp = reinterpret_cast<const uint4*>(kfh + 5 * kTile + s0);
#pragma unroll
            for (int i8 = 0; i8 < 2; ++i8) {
              const uint4 f = kp[i8];
              const __half2* h2 = reinterpret_cast<const __half2*>(&f);
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const float2 f2 = __half22float2(h2[e]);
                cf[8 * i8 + 2 * e] = f2.x;
                cf[8 * i8 + 2 * e + 1] = f2.y;
              }
            }
          } else {
            const float lg = (q ^ g) == 1 ? lam6 : lam7;  // level 5 + bitlen(q ^ g)
            rf = lg * ex2(cs2_t - cs_s[32 * g + 31]);
            const float4* cp = reinterpret_cast<const float4*>(col_s + s0);
#pragma unroll
            for (int i4 = 0; i4 < 4; ++i4) {
              const float4 f = cp[i4];
              cf[4 * i4] = f.x; cf[4 * i4 + 1] = f.y; cf[4 * i4 + 2] = f.z; cf[4 * i4 + 3] = f.w;
            }
          }
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 16; ++i) v[i] *= rf * cf[i];
        } else if (g == q) {
          tmem_ld16(tl + kTmS + s0, v);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int x = 16 * hf + i;  // column inside the diagonal group
            const int lv = 32 - __clz(lane ^ x);
            float e;
            if constexpr (kLD) {
              // lam_t[l] Q(t, l) (a select over this row's six) times K(s, l) from the table
              float rq = rowq[0];
#pragma unroll
              for (int l = 1; l <= 5; ++l) rq = lv == l ? rowq[l] : rq;
              e = lv == 0 ? rq : rq * __half2float(kfh[(lv > 0 ? lv - 1 : 0) * kTile + 32 * q + x]);
            } else {
              e = ex2(cs2_diag - cs_s[s0 + i]) * __half2float(lamh[lv * kTile + row]);
            }
            v[i] = (x <= lane) ? v[i] * e : 0.f;
          }
        } else {
#pragma unroll
          for (int i = 0; i < 16; ++i) v[i] = 0.f;
        }
        uint32_t w[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) w[i] = pack_bf16x2(v[2 * i], v[2 * i + 1]);
        if (g < 2) {
#pragma unroll
          for (int i = 0; i < 8; ++i) pw[g][i] = w[i];
        } else {
          tmem_st8(tl + kTmS + 16 * g + 8 * hf, w);
        }
        if (g == 1) {
          // P (64 columns) overwrites the scores of groups 0 and 1, which the
          // quadrant's other warp reads too: both have read them before either writes
          tc_fence_before();
          named_bar_sync(2 + q, 64);
          tc_fence_after();
          tmem_st8(tl + kTmS + 8 * hf, pw[0]);
          tmem_st8(tl + kTmS + 16 + 8 * hf, pw[1]);
        }
      }
      tmem_st_wait();
      tc_fence_before();  // orders the score reads and the P writes before the PV product
      __syncwarp();
      named_bar_sync(1, kEpi);
      if (leader) mbar_arrive(c.bars + B_P_READY);
      if (!kLD && it == 0 && n > 1) prologue(1);  // (no back half in this step)
    }

    if (it >= 1) {
      // ================= back half of tile it-1: inter-tile levels + output
      const size_t rp = (size_t)bhp * p.T + (size_t)jp * kTile + row;
      // (the CTA's last tile has no front half after it to load this in)
      const int jap = jp | start_tile<kCont>(p);
      if (it == n && jap != 0) lam_c = __ldg(p.lam + rp * p.L + 8 + (__ffs(jap) - 1));
      // log decays of the levels, handed over one by one by the level producer
      // under a step-tagged count; bounded wait until it covers `cnt` levels
      const uint32_t* nlr = reinterpret_cast<const uint32_t*>(s + kOffNode + 160) + (it & 1);
      const volatile float* dl = reinterpret_cast<const volatile float*>(s + kOffNode) + 16 * (it & 1);
      auto wait_levels = [&](uint32_t cnt) {
        const uint32_t want = ((uint32_t)it << 8) | cnt;
        if (ld_acquire_cta_u32(nlr) >= want || *c.abort_s) return;
        const uint64_t t0 = globaltimer_ns();
        while (ld_acquire_cta_u32(nlr) < want) {
          if (*c.abort_s) return;
          if (globaltimer_ns() - t0 > p.timeout_ns) {
            note_abort(c);
            return;
          }
        }
      };
      wait_levels(0);  // the level producer has reached this step
      // this thread's half row of the previous tile's Q (bf16, its second load);
      // once every thread has it the buffer goes to the next tile's scores
      wait_bar_w(c, B_QB_FULL, (it - 1) & 1);
      uint4 qv[8];
      {
        const unsigned char* qrow = s + kOffQ + hf * kHalf + row * 128;
#pragma unroll
        for (int c8 = 0; c8 < 8; ++c8) qv[c8] = *reinterpret_cast<const uint4*>(qrow + ((c8 ^ (row & 7)) << 4));
      }
      __syncwarp();
      named_bar_sync(1, kEpi);
      if (leader) mbar_arrive(c.bars + B_Q_FREE);
      // inter-tile levels: Q'_l = lam_t[8 + h] exp(cs_t + D_l) Q_t goes to TMEM
      // as the A operand of a product the MMA accumulates onto the output
      int l = 0;
      for (int rem = jap; rem != 0; ++l) {
        const int hcur = __ffs(rem) - 1;  // level 8 + hcur
        rem &= rem - 1;
        const float lam_h = lam_c;
        // the next level's lambda loads while this level is written
        if (rem != 0) lam_c = __ldg(p.lam + rp * p.L + 8 + (__ffs(rem) - 1));
        wait_levels((uint32_t)(l + 1));
        float csl = cs_prev;
        if constexpr (kLD) {  // the level's own running sum in the tile
          csl = csI_prev[0];
#pragma unroll
          for (int h = 1; h < 8; ++h) csl = hcur == h ? csI_prev[h] : csl;
        }
        const float w = lam_h * ex2((csl + dl[l]) * kLog2e);
        uint32_t wq[32];
#pragma unroll
        for (int c8 = 0; c8 < 8; ++c8) {
          const uint32_t* q4 = reinterpret_cast<const uint32_t*>(&qv[c8]);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float2 f = unpack_bf16x2(q4[i]);
            wq[4 * c8 + i] = pack_bf16x2(w * f.x, w * f.y);
          }
        }
        const int b = qpc & 1;
        if (qpc >= 2) wait_bar_w(c, B_QP_FREE0 + b, ((qpc - 2) >> 1) & 1);  // its previous product is done
        __syncwarp();
        tc_fence_after();
        tmem_st32(tl + kTmQP + 64 * b + 32 * hf, wq);
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        named_bar_sync(1, kEpi);
        if (leader) mbar_arrive(c.bars + B_QP_FULL0 + b);
        ++qpc;
        // the next tile's prologue once the first level product can start
        if (!kLD && l == 0 && it + 1 < n) prologue(it + 1);
      }

      // (the next tile's prologue when this tile has no level to hand over)
      if (!kLD && it + 1 < n && jap == 0) prologue(it + 1);

      // output = PV + levels, accumulated in TMEM; bf16, staged for the store warp
      if (xs > 0) wait_bar_w(c, B_X_FREE, (xs - 1) & 1);
      wait_bar_w(c, B_O_READY, (it - 1) & 1);
      __syncwarp();
      tc_fence_after();
      {
        unsigned char* xrow = s + kOffX + hf * kHalf + row * 128;
#pragma unroll
        for (int c32 = 0; c32 < 2; ++c32) {
          float v[32];
          tmem_ld32(tl + kTmR + 64 * hf + 32 * c32, v);
          tmem_ld_wait();
#pragma unroll
          for (int c4 = 0; c4 < 4; ++c4) {
            const int c8 = 4 * c32 + c4;
            *reinterpret_cast<uint4*>(xrow + ((c8 ^ (row & 7)) << 4)) =
                make_uint4(pack_bf16x2(v[8 * c4], v[8 * c4 + 1]), pack_bf16x2(v[8 * c4 + 2], v[8 * c4 + 3]),
                           pack_bf16x2(v[8 * c4 + 4], v[8 * c4 + 5]), pack_bf16x2(v[8 * c4 + 6], v[8 * c4 + 7]));
          }
        }
      }
      fence_proxy_async_shared();
      tc_fence_before();  // the accumulator is free once every thread is past this point
      __syncwarp();
      named_bar_sync(1, kEpi);
      if (leader) {
        mbar_arrive(c.bars + B_R_FREE);
        mbar_arrive(c.bars + B_LVLD_FREE);
        mbar_arrive(c.bars + B_X_STAGED);
      }
      ++xs;
    }

    cs_prev = cs_t;
    if constexpr (kLD) {
#pragma unroll
      for (int h = 0; h < 8; ++h) csI_prev[h] = csI[h];
    }
    jp = j;
    bhp = bh;
  }
}

// ------------------------------------------------------------------ store warp (warp 2)
// Stores each staged output with the TMA and hands the staging buffer back
// once the copy has read it.
__device__ void store_warp(const Ctx& c, const CUtensorMap* to) {
  const TcParams& p = *c.p;
  const int n = tiles_of_cta(p.BH * p.Nt);
  const unsigned char* x = c.base + kOffX;
  for (int it = 1; it <= n; ++it) {
    const int up = blockIdx.x + (it - 1) * gridDim.x;
    wait_bar(c, B_X_STAGED, (it - 1) & 1);
    fence_proxy_async_shared();
    const int row0 = (up % p.BH) * p.T + (up / p.BH) * kTile;
    tma_store_2d(to, x, 0, row0);
    if (p.d > 64) tma_store_2d(to, x + kHalf, 64, row0);  // (d = 64: the zero half is not stored)
    bulk_commit();
    bulk_wait_read0();
    mbar_arrive(c.bars + B_X_FREE);
  }
  bulk_wait0();
}

// ------------------------------------------------------------------ node warps (warps 12..15)
// Per tile j, in order: the chunk state S_j is in the accumulator M once the
// state product is done.  For odd j the Fenwick children F_{j-2^m}, m <
// cto(j), are added in float32: each is waited for (its publication word),
// loaded by TMA into the C buffer and added row by row into M with its decay
// exp(dec_m), dec_m = the log decay from the end of the child's block to the
// end of tile j.  Then F_j leaves M as bf16 through C (TMA store), M goes
// back to the MMA, and once the store is complete F_j is published with its
// log-decay total G_j.  Thread t = 32 (warp % 4) + lane owns TMEM lane t: row
// d_v = t of the node.
template <bool kLD>
__device__ void node_warps(const Ctx& c, uint32_t tmem, int warp, int lane, const CUtensorMap* tf) {
  const TcParams& p = *c.p;
  const int n = tiles_of_cta(p.BH * p.Nt);
  const int q = warp & 3;
  const int t = 32 * q + lane;
  const bool leader = (warp == kNodeWarp0 && lane == 0);
  const uint32_t tm = tmem + ((uint32_t)(32 * q) << 16) + kTmM;
  unsigned char* s = c.base;
  float* nq = reinterpret_cast<float*>(s + kOffMisc + 48);        // [4] quadrant sums
  volatile float* gch = reinterpret_cast<volatile float*>(s + kOffNode + 176);  // child's log-decay total
  unsigned char* cb = s + kOffC;
  uint32_t cf = 0;     // child loads waited for
  uint32_t armed = 0;  // child loads armed (the leader)
  for (int it = 0; it < n; ++it) {
    const int u = blockIdx.x + it * gridDim.x;
    const int bh = u % p.BH, j = u / p.BH;
    const size_t node_j = (size_t)bh * p.Nt + j;
    // the tile's log-decay total (also the barrier after which the previous
    // node's store has completed and C is free)
    float x = kLD ? 0.f : __ldg(p.log_alpha + (size_t)bh * p.T + (size_t)j * kTile + t);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    if (lane == 0) nq[q] = x;
    __syncwarp();
    named_bar_sync(6, kNodeThreads);
    const float cs_end = (nq[0] + nq[1]) + (nq[2] + nq[3]);
    float D = cs_end;  // log decay from the end of the next child's block to the end of tile j
    wait_bar_w(c, B_STATE_DONE, it & 1);
    __syncwarp();
    tc_fence_after();
    const int cto = __ffs(~j) - 1;  // trailing ones of j
    for (int m = 0; m < cto; ++m) {
      const size_t child = node_j - ((size_t)1 << m);
      // per-level mode: the child's keys sit at level 8 + m over tiles (j - 2^m, j]
      // (read before the child's wait)
      const float dm = kLD ? ld_span(p, bh, m, j - (1 << m) + 1, j + 1) : 0.f;
      if (leader) {
        const uint64_t w = wait_flag(c, p.flags, child);
        fence_proxy_async_global();
        *gch = flag_g(w);
        if (!*c.abort_s) {
          mbar_arrive_expect_tx(c.bars + B_C_FULL, kTileBytes);
          tma_load_2d(cb, tf, c.bars + B_C_FULL, 0, (int)(child * kD));
          tma_load_2d(cb + kHalf, tf, c.bars + B_C_FULL, 64, (int)(child * kD));
          ++armed;
        }
      }
      wait_bar_w(c, B_C_FULL, cf & 1);
      ++cf;
      __syncwarp();
      const float g = *gch;
      const float sc = ex2((kLD ? dm : D) * kLog2e);
      // row t of the child, 16-byte chunk c8 of its 128-byte-swizzled tile
#pragma unroll
      for (int c32 = 0; c32 < 4; ++c32) {
        float a[32];
        tmem_ld32(tm + 32 * c32, a);
        uint4 ch[4];
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          const int c8 = 4 * c32 + v;
          ch[v] = *reinterpret_cast<const uint4*>(cb + (c8 >> 3) * kHalf + t * 128 + (((c8 & 7) ^ (t & 7)) << 4));
        }
        tmem_ld_wait();
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          const uint32_t* w = reinterpret_cast<const uint32_t*>(&ch[v]);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 f = unpack_bf16x2(w[e]);
            a[8 * v + 2 * e] = fmaf(sc, f.x, a[8 * v + 2 * e]);
            a[8 * v + 2 * e + 1] = fmaf(sc, f.y, a[8 * v + 2 * e + 1]);
          }
        }
        tmem_st32(tm + 32 * c32, reinterpret_cast<const uint32_t*>(a));
      }
      tmem_st_wait();
      __syncwarp();
      named_bar_sync(6, kNodeThreads);  // every row of the child is read: C is free
      D += g;
    }
    const float G = kLD ? 0.f : D;  // cs_end plus the children's totals (unused per level)
    // F_j as bf16 into C (row t), then M is free and the node is stored
#pragma unroll
    for (int c32 = 0; c32 < 4; ++c32) {
      float a[32];
      tmem_ld32(tm + 32 * c32, a);
      tmem_ld_wait();
#pragma unroll
      for (int v = 0; v < 4; ++v) {
        const int c8 = 4 * c32 + v;
        *reinterpret_cast<uint4*>(cb + (c8 >> 3) * kHalf + t * 128 + (((c8 & 7) ^ (t & 7)) << 4)) =
            make_uint4(pack_bf16x2(a[8 * v], a[8 * v + 1]), pack_bf16x2(a[8 * v + 2], a[8 * v + 3]),
                       pack_bf16x2(a[8 * v + 4], a[8 * v + 5]), pack_bf16x2(a[8 * v + 6], a[8 * v + 7]));
      }
    }
    fence_proxy_async_shared();
    tc_fence_before();
    __syncwarp();
    named_bar_sync(6, kNodeThreads);
    if (leader) {
      mbar_arrive(c.bars + B_M_FREE);
      p.G[node_j] = G;
      tma_store_2d(tf, cb, 0, (int)(node_j * kD));
      tma_store_2d(tf, cb + kHalf, 64, (int)(node_j * kD));
      bulk_commit();
      bulk_wait0();  // complete, before C is reused and before the node is published
      fence_proxy_async_global();
      if ((long long)node_j != p.withhold)  // (expiry test: a node nothing will publish)
        st_release_u64(p.flags + node_j, ((uint64_t)p.token << 32) | __float_as_uint(G));
    }
  }
  if (leader && armed > 0) drain_bar(c, B_C_FULL, (armed - 1) & 1);  // (a copy armed before an abort)
}

template <bool kCont, bool kLD>
__global__ void __launch_bounds__(kThreads, 1)
    fwd_tc_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                  const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tf,
                  const __grid_constant__ CUtensorMap to, TcParams p) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  // the 128-byte swizzle of the operand tiles assumes a 1024-aligned base;
  // the budget leaves no room to realign, so refuse (all threads) otherwise
  if (smem_u32(smem_raw) & 1023u) {
    if (threadIdx.x == 0) atomicOr(p.err, kErrDeviceArg);
    return;
  }
  unsigned char* base = smem_raw;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + kOffBars);
  volatile int* abort_s = reinterpret_cast<volatile int*>(base + kOffMisc + 16);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base + kOffMisc + 32);
  Ctx c{base, bars, abort_s, &p};

  if (threadIdx.x == 0) {
    *abort_s = 0;
    // the level producer's step-tagged counts (and the decays they cover)
    // start below every tag: shared memory keeps an earlier launch's values,
    // which a back half would otherwise take for this launch's
    uint32_t* nlr = reinterpret_cast<uint32_t*>(base + kOffNode + 160);
    float* dl = reinterpret_cast<float*>(base + kOffNode);
    nlr[0] = nlr[1] = 0;
    for (int i = 0; i < 32; ++i) dl[i] = 0.f;
    for (int b = 0; b < kNumBars; ++b) mbar_init(bars + b, 1);
    fence_mbar_init();
    prefetch_tmap(&tq);
    prefetch_tmap(&tk);
    prefetch_tmap(&tv);
    prefetch_tmap(&tf);
    prefetch_tmap(&to);
  }
  __syncwarp();
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // registers by warpgroup: the single-thread roles give theirs to the
  // epilogue (88 + 2 x 160 + 104 = 512 per four threads: the 128 of the launch)
  const int wg = warp >> 2;
  if (wg == 0) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 88;\n" ::: "memory");
    if (lane == 0) {
      if (warp == 0) producer_kvq<kLD>(c, &tq, &tk, &tv);
      else if (warp == 1) mma_issuer<kCont>(c, tmem);
      else if (warp == 2) store_warp(c, &to);
      else producer_levels<kCont, kLD>(c, &tf);
    }
  } else if (wg == 3) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 104;\n" ::: "memory");
    node_warps<kLD>(c, tmem, warp, lane, &tf);
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 160;\n" ::: "memory");
    epilogue<kCont, kLD>(c, tmem, warp, lane);
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
// Continuation: the prefix states of position t0 (true state = scale * S,
// decayed to t0 - 1) as bf16 nodes, one per tile height h (level 8 + h).
// With d = 64 the states are [64][64] and the nodes [128][128] with zeros
// outside the first 64 rows and columns.
__global__ void __launch_bounds__(256) tc_prefix_nodes_kernel(const float* __restrict__ state_in,
                                                              const float* __restrict__ scale_in,
                                                              __nv_bfloat16* __restrict__ F, int BH, int Nt, int Ls,
                                                              long long t0, int d) {
  const size_t bh = blockIdx.y;
  const int idx = blockIdx.x * 256 + threadIdx.x;  // < 128 * 128
  const int r = idx >> 7, cc = idx & 127;
  constexpr int mat = kD * kD;
  for (int slot = 7; slot < Ls; ++slot) {  // levels 8 .. Ls (t0 is a multiple of the tile: no lower ones)
    if (!((t0 >> slot) & 1)) continue;
    const int h = slot + 1 - 8;              // tile height: bit h of t0 / 128
    const size_t node = (size_t)BH * Nt + bh * kPreSlots + h;
    const float x = (r < d && cc < d) ? scale_in[bh * Ls + slot] * state_in[(bh * Ls + slot) * (size_t)d * d + r * d + cc]
                                      : 0.f;
    F[node * mat + idx] = __float2bfloat16_rn(x);
  }
}

__global__ void __launch_bounds__(256) tc_export_kernel(const __nv_bfloat16* __restrict__ F,
                                                        const float* __restrict__ G, float* __restrict__ state_out,
                                                        float* __restrict__ scale_out, int Nt, int Ls, int d) {
  const size_t bh = blockIdx.y;
  const int idx = blockIdx.x * 256 + threadIdx.x;  // < 128 * 128
  const int r = idx >> 7, cc = idx & 127;
  const bool in = r < d && cc < d;  // (d = 64: the nodes' first 64 rows and columns)
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
    if (in) state_out[(bh * Ls + slot) * (size_t)d * d + r * d + cc] = val;
    if (blockIdx.x == 0 && threadIdx.x == 0) scale_out[bh * Ls + slot] = sc;
  }
}

// Continuation: the decode states of t1 = t0 + T in one pass (no separate
// export of the segment, no separate sum of its log decays).  With b =
// bitlen(t1 xor t0) and P the smallest power of two >= T, the prefix bucket of
// level l goes to level max(l, b), decayed over the whole segment (whose log
// decay is the sum of the node totals of the tiles' Fenwick prefix); the
// segment's own bucket of level l (the node of tile height l - 8, decayed
// from the end of its block to T - 1) keeps its level if T < P and goes to b
// if T = P.  Thread 0 lists, per output slot, the buckets that land on it and
// their factors; every thread then sums its element of those.
__global__ void __launch_bounds__(256) tc_cont_export_kernel(const __nv_bfloat16* __restrict__ F,
                                                             const float* __restrict__ G,
                                                             const float* __restrict__ state_in,
                                                             const float* __restrict__ scale_in,
                                                             float* __restrict__ state_out,
                                                             float* __restrict__ scale_out, int Nt, int T, int Ls,
                                                             long long t0, int d) {
  constexpr int kMaxSrc = 2 * 64;
  __shared__ int off[64 + 1];
  __shared__ long long srcs[kMaxSrc];  // >= 0: the row offset of a prefix state; < 0: -(node + 1)
  __shared__ float fac[kMaxSrc];
  const size_t bh = blockIdx.y;
  const int idx = blockIdx.x * 256 + threadIdx.x;  // < 128 * 128
  const int r = idx >> 7, cc = idx & 127;
  constexpr int mat = kD * kD;
  const long long t1 = t0 + T;
  if (threadIdx.x == 0) {
    const int b = 64 - __clzll(t1 ^ t0);                         // bitlen(t1 xor t0)
    const long long P = 1ll << (64 - __clzll((long long)T - 1));  // smallest power of two >= T
    // the segment's buckets: node of height h decayed by the node totals of the lower set bits
    float segD[32];
    float D = 0.f;
    for (int h = 0; h < 31; ++h) {
      segD[h] = D;
      if ((Nt >> h) & 1) D += G[bh * Nt + node_of_level(Nt, h)];
    }
    const float dec = exp2f(D * kLog2e);  // the whole segment's decay
    int n = 0;
    for (int o = 0; o < Ls; ++o) {
      off[o] = n;
      if (!((t1 >> o) & 1)) continue;
      for (int sl = 0; sl < Ls && n < kMaxSrc; ++sl) {
        if (((t0 >> sl) & 1) && (sl + 1 > b ? sl + 1 : b) == o + 1) {
          srcs[n] = (long long)(bh * Ls + sl) * d * d;
          fac[n++] = scale_in[bh * Ls + sl] * dec;
        }
        const int h = sl + 1 - 8;
        if (h >= 0 && h < 31 && ((Nt >> h) & 1) && ((long long)T < P ? sl + 1 : b) == o + 1 && n < kMaxSrc) {
          srcs[n] = -(long long)(bh * Nt + node_of_level(Nt, h)) - 1;
          fac[n++] = exp2f(segD[h] * kLog2e);
        }
      }
    }
    off[Ls] = n;
  }
  __syncthreads();
  if (r >= d || cc >= d) return;
  for (int o = 0; o < Ls; ++o) {
    float acc = 0.f;
    for (int e = off[o]; e < off[o + 1]; ++e) {
      const long long sv = srcs[e];
      const float x = sv >= 0 ? state_in[sv + r * d + cc] : __bfloat162float(F[(size_t)(-sv - 1) * mat + idx]);
      acc = fmaf(fac[e], x, acc);
    }
    state_out[(bh * Ls + o) * (size_t)d * d + r * d + cc] = acc;
  }
  if (blockIdx.x == 0 && threadIdx.x == 0)
    for (int o = 0; o < Ls; ++o) scale_out[bh * Ls + o] = ((t1 >> o) & 1) ? 1.f : 0.f;
}

// Per-level mode, first step: the log-decay totals of every tile at the
// inter-tile levels 8..L-1, one CTA per (tile, head), thread = row;
// tot[(bh * Nt + j) * Lx + h] (float).
__global__ void __launch_bounds__(kTile) tc_ld_tile_totals_kernel(const float* __restrict__ la,
                                                                  float* __restrict__ tot, int T, int Nt, int L,
                                                                  int Lx) {
  __shared__ float part[kTile / 32][8];
  const int j = blockIdx.x;
  const size_t bh = blockIdx.y;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const float* r = la + ((size_t)bh * T + (size_t)j * kTile + threadIdx.x) * L;
#pragma unroll
  for (int h = 0; h < 8; ++h) {
    float x = 8 + h < L ? __ldg(r + 8 + h) : 0.f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    if (lane == 0) part[warp][h] = x;
  }
  __syncthreads();
  if (threadIdx.x < Lx && threadIdx.x < 8) {
    const int h = threadIdx.x;
    tot[((size_t)bh * Nt + j) * Lx + h] = (part[0][h] + part[1][h]) + (part[2][h] + part[3][h]);
  }
}

// Second step: their running sums over the tiles, float64, one single-warp
// CTA per (level, head) (float64 arithmetic is scarce on this GPU: spread it
// over the SMs): cumL[(bh * Lx + h) * Nt + j] = sum of tot over tiles 0..j.
__global__ void __launch_bounds__(32) tc_ld_tile_scan_kernel(const float* __restrict__ tot,
                                                             double* __restrict__ cumL, int Nt, int Lx) {
  const int h = blockIdx.x;
  const size_t bh = blockIdx.y;
  const int lane = threadIdx.x;
  double carry = 0.0;
  for (int base = 0; base < Nt; base += 32) {
    const int i = base + lane;
    double y = i < Nt ? (double)tot[((size_t)bh * Nt + i) * Lx + h] : 0.0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const double z = __shfl_up_sync(0xffffffffu, y, o);
      if (lane >= o) y += z;
    }
    y += carry;
    if (i < Nt) cumL[(bh * Lx + h) * Nt + i] = y;
    carry = __shfl_sync(0xffffffffu, y, 31);
  }
}

// Per-level mode: the level states of position T, each node decayed at its
// own level over the tiles after its block.
__global__ void __launch_bounds__(256) tc_ld_export_kernel(const __nv_bfloat16* __restrict__ F,
                                                           const double* __restrict__ cumL,
                                                           float* __restrict__ state_out,
                                                           float* __restrict__ scale_out, int Nt, int Ls, int Lx,
                                                           int d) {
  const size_t bh = blockIdx.y;
  const int idx = blockIdx.x * 256 + threadIdx.x;  // < 128 * 128
  const int r = idx >> 7, cc = idx & 127;
  constexpr int mat = kD * kD;
  for (int slot = 0; slot < Ls; ++slot) {
    const int h = slot + 1 - 8;  // level slot+1 = 8 + h
    float val = 0.f, sc = 0.f;
    if (h >= 0 && h < 31 && ((Nt >> h) & 1)) {
      const size_t e = bh * Nt + node_of_level(Nt, h);
      const int cb = Nt & ~((1 << h) - 1);  // the node's keys are at level 8 + h from tile cb on
      double D = 0.0;
      if (cb < Nt && h < Lx) {
        const double* cl = cumL + (bh * Lx + h) * (size_t)Nt;
        D = cl[Nt - 1] - (cb > 0 ? cl[cb - 1] : 0.0);
      }
      val = exp2f((float)D * kLog2e) * __bfloat162float(F[e * mat + idx]);
      sc = 1.f;
    }
    if (r < d && cc < d) state_out[(bh * Ls + slot) * (size_t)d * d + r * d + cc] = val;
    if (blockIdx.x == 0 && threadIdx.x == 0) scale_out[bh * Ls + slot] = sc;
  }
}

// ------------------------------------------------------------------ host side
struct TcPlan {
  int Nt, Lx;
  size_t off_F, off_G, off_flags, off_tot, off_cum, total;
};

// F holds the tiles' nodes, then kPreSlots prefix nodes per head (used by a
// continuation only, always reserved so one layout serves both); the
// per-level mode adds its table of running sums
TcPlan tc_plan(const ll_shape& s, bool ld = false) {
  TcPlan p{};
  p.Nt = s.T / kTile;
  p.Lx = std::max(s.L - 8, 1);
  const size_t BH = (size_t)s.B * s.H;
  const size_t nodes = BH * p.Nt;
  size_t off = 0;
  p.off_F = off;      off = align_up(off + (nodes + BH * kPreSlots) * kD * kD * 2, 1024);
  p.off_G = off;      off = align_up(off + nodes * 4, 256);
  p.off_flags = off;  off += (nodes + 1) * 8;
  p.off_cum = off;  // directly after the words: the kernel finds it there
  if (ld) off += BH * p.Lx * p.Nt * sizeof(double);
  off = align_up(off, 256);
  p.off_tot = off;
  if (ld) off = align_up(off + BH * p.Lx * p.Nt * sizeof(float), 256);
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

// 2-D bf16 tensor map over [rows, cols] with [128 x 64] boxes, 128-byte
// swizzle; with cols = 64 a box at column 64 lies wholly outside and loads
// as zeros.
bool make_map(CUtensorMap* m, const void* base, uint64_t rows, int cols = kD) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)kTile};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Per-call token of the publication words: a process-wide counter, so two
// calls on one workspace never share it (0 is skipped).
uint32_t next_token() {
  static std::atomic<uint32_t> counter{0x5eed};
  uint32_t t = counter.fetch_add(1);
  if (t == 0) t = counter.fetch_add(1);
  return t;
}

}  // namespace

// bf16 with d = 128, or d = 64 run as 128 with zero-filled tiles
static bool tc_head_ok(const ll_shape& s) { return s.dk == s.dv && (s.dk == kD || s.dk == 64); }

bool fwd_tc_supported(const ll_shape& s) {
  return s.io == LL_BF16 && tc_head_ok(s) && s.T % kTile == 0 && s.L <= kLmax &&
         (long long)s.B * s.H * (s.T + kPreSlots * kTile) <= (1ll << 31) - 1;
}

// A continuation at t0 (already checked: t0 a multiple of the smallest power
// of two >= T) on this path: every prefix level must have a node slot and
// every tile at most 16 levels, which L <= kLmax gives.
bool fwd_tc_cont_supported(const ll_shape& s, long long t0) {
  return fwd_tc_supported(s) && t0 / kTile < (1ll << 30) && s.Ls <= 7 + kPreSlots;
}

size_t fwd_tc_cont_workspace(const ll_shape& s) { return tc_plan(s).total; }

size_t fwd_tc_workspace(const ll_shape& s) { return tc_plan(s).total; }

int fwd_tc_launches(const ll_shape& s) { return s.Ls > 0 ? 2 : 1; }  // (a continuation: 3 with its prefix nodes)

bool fwd_tc_level_decay_supported(const ll_shape& s) {
  return s.io == LL_BF16 && tc_head_ok(s) && s.T % kTile == 0 && s.L <= kLdLv + 1 &&
         (long long)s.B * s.H * (s.T + kPreSlots * kTile) <= (1ll << 31) - 1;
}

size_t fwd_tc_level_decay_workspace(const ll_shape& s) { return tc_plan(s, true).total; }

int fwd_tc_level_decay_launches(const ll_shape& s) { return s.Ls > 0 ? 4 : 3; }

static ll_status tc_launch(const FwdArgs& a, bool ld) {
  const ll_shape& s = a.s;
  const TcPlan plan = tc_plan(s, ld);
  if (ld && a.state_in) return LL_ERR_INVALID_ARG;
  if (a.ws_bytes < plan.total) return LL_ERR_WORKSPACE;
  unsigned char* ws = static_cast<unsigned char*>(a.ws);
  const int BH = s.B * s.H;
  const int stride = a.rows_per_head ? a.rows_per_head : s.T;  // rows between (b, h) slices
  if (stride < s.T || (a.state_in && stride != s.T) || (long long)BH * stride > (1ll << 31) - 1)
    return LL_ERR_INVALID_ARG;
  const uint64_t rows = (uint64_t)BH * stride;
  const uint64_t node_rows = ((uint64_t)BH * plan.Nt + (uint64_t)BH * kPreSlots) * kD;
  CUtensorMap tq, tk, tv, tf, to;
  const int d = s.dk;
  if (!make_map(&tq, a.q, rows, d) || !make_map(&tk, a.k, rows, d) || !make_map(&tv, a.v, rows, d) ||
      !make_map(&tf, ws + plan.off_F, node_rows) || !make_map(&to, a.o, rows, d))
    return LL_ERR_CUDA;

  TcParams p;
  p.log_alpha = a.log_alpha;
  p.lam = a.lam;
  p.q = static_cast<const __nv_bfloat16*>(a.q);
  p.k = static_cast<const __nv_bfloat16*>(a.k);
  p.v = static_cast<const __nv_bfloat16*>(a.v);
  p.F = reinterpret_cast<__nv_bfloat16*>(ws + plan.off_F);
  p.G = reinterpret_cast<float*>(ws + plan.off_G);
  p.flags = reinterpret_cast<uint64_t*>(ws + plan.off_flags);
  p.abort_word = p.flags + (size_t)BH * plan.Nt;
  p.token = next_token();
  p.BH = BH;
  p.T = stride;
  p.Nt = plan.Nt;
  p.L = s.L;
  p.err = a.err;
  p.c0t = a.state_in ? (int)(a.t0 / kTile) : 0;
  p.timeout_ns = a.timeout_ns ? a.timeout_ns : kTimeoutNs;
  p.withhold = a.withhold_node;
  p.d = s.dk;
  if (ld) {
    float* tot = reinterpret_cast<float*>(ws + plan.off_tot);
    tc_ld_tile_totals_kernel<<<dim3(plan.Nt, BH), kTile, 0, a.stream>>>(a.log_alpha, tot, stride, plan.Nt, s.L,
                                                                        plan.Lx);
    LL_CUDA_OK(cudaGetLastError());
    tc_ld_tile_scan_kernel<<<dim3(plan.Lx, BH), 32, 0, a.stream>>>(tot, reinterpret_cast<double*>(ws + plan.off_cum),
                                                                   plan.Nt, plan.Lx);
    LL_CUDA_OK(cudaGetLastError());
  }
  if (a.state_in) {
    tc_prefix_nodes_kernel<<<dim3(kD * kD / 256, BH), 256, 0, a.stream>>>(a.state_in, a.scale_in, p.F, BH, plan.Nt,
                                                                         s.Ls, a.t0, d);
    LL_CUDA_OK(cudaGetLastError());
  }

  int dev = 0, sms = 0, per_sm = 0;
  LL_CUDA_OK(cudaGetDevice(&dev));
  LL_CUDA_OK(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
  const void* kern = ld ? (const void*)fwd_tc_kernel<false, true>
                        : a.state_in ? (const void*)fwd_tc_kernel<true, false> : (const void*)fwd_tc_kernel<false, false>;
  LL_CUDA_OK(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes));
  LL_CUDA_OK(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, kSmemBytes));
  if (per_sm < 1) return LL_ERR_CUDA;
  const long long tiles = (long long)BH * plan.Nt;
  const int grid = (int)std::min<long long>(tiles, (long long)sms * per_sm);

  void* args[] = {&tq, &tk, &tv, &tf, &to, &p};
  LL_CUDA_OK(cudaLaunchCooperativeKernel(kern, dim3(grid), dim3(kThreads), args, kSmemBytes,
                                         a.stream));
  if (a.state_out && a.state_in) {
    tc_cont_export_kernel<<<dim3(kD * kD / 256, BH), 256, 0, a.stream>>>(
        p.F, p.G, a.state_in, a.scale_in, a.state_out, a.scale_out, plan.Nt, s.T, s.Ls, a.t0, d);
    LL_CUDA_OK(cudaGetLastError());
    return LL_OK;
  }
  if (a.state_out && ld) {
    tc_ld_export_kernel<<<dim3(kD * kD / 256, BH), 256, 0, a.stream>>>(
        p.F, reinterpret_cast<const double*>(ws + plan.off_cum), a.state_out, a.scale_out, plan.Nt, s.Ls, plan.Lx, d);
    LL_CUDA_OK(cudaGetLastError());
  } else if (a.state_out) {
    tc_export_kernel<<<dim3(kD * kD / 256, BH), 256, 0, a.stream>>>(p.F, p.G, a.state_out, a.scale_out, plan.Nt,
                                                                   s.Ls, d);
    LL_CUDA_OK(cudaGetLastError());
  }
  return LL_OK;
}

ll_status fwd_tc_launch(const FwdArgs& a) { return tc_launch(a, false); }

ll_status fwd_tc_level_decay_launch(const FwdArgs& a) { return tc_launch(a, true); }

}  // namespace llattn
