// C ABI entry points of libllattn: argument checks, path selection, launch.
//
// Every check here runs on the host before anything is launched, so an
// invalid call never touches device memory.
#include <algorithm>
#include <mutex>

#include "bwd.cuh"
#include "level_decay.cuh"

namespace llattn {

__device__ unsigned g_err_word = 0;

static constexpr int kMaxDevices = 64;

unsigned* err_word() {
  static std::mutex mu;
  static unsigned* addr[kMaxDevices] = {nullptr};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_err_word) != cudaSuccess) return nullptr;
    addr[dev] = static_cast<unsigned*>(p);
  }
  return addr[dev];
}

static bool head_dim_ok(int d) { return is_pow2_in(d, 16, 128); }

// Shape checks shared by the forward entry points.
static ll_status check_shape(const ll_shape* s) {
  if (!s) return LL_ERR_INVALID_ARG;
  if (s->B < 1 || s->H < 1 || s->T < 1) return LL_ERR_INVALID_ARG;
  if (s->io != LL_F32 && s->io != LL_BF16) return LL_ERR_INVALID_ARG;
  if (!is_pow2_in(s->chunk, 16, 128)) return LL_ERR_INVALID_ARG;
  if (s->L < levels_needed(s->T) || s->L > 64) return LL_ERR_INVALID_ARG;
  if (s->Ls < 0 || s->Ls > 62) return LL_ERR_INVALID_ARG;
  if (!head_dim_ok(s->dk) || !head_dim_ok(s->dv)) return LL_ERR_UNSUPPORTED;
  // element counts must stay addressable with 64-bit offsets and 32-bit T
  return LL_OK;
}


// ---------------------------------------------------------------- compositions
// Rows [r0, r0 + n) of every (b, h) slice of a [BH, T, *] tensor with
// `row_bytes` per row, copied into a contiguous [BH, n, *] buffer (or back).
static ll_status copy_rows(void* dst, const void* src, int BH, int T, int r0, int n, size_t row_bytes, bool to_stage,
                           cudaStream_t st) {
  const size_t width = (size_t)n * row_bytes;
  if (width == 0) return LL_OK;
  if (to_stage)
    LL_CUDA_OK(cudaMemcpy2DAsync(dst, width, static_cast<const char*>(src) + (size_t)r0 * row_bytes,
                                 (size_t)T * row_bytes, width, BH, cudaMemcpyDeviceToDevice, st));
  else
    LL_CUDA_OK(cudaMemcpy2DAsync(static_cast<char*>(dst) + (size_t)r0 * row_bytes, (size_t)T * row_bytes, src, width,
                                 width, BH, cudaMemcpyDeviceToDevice, st));
  return LL_OK;
}

// Contiguous copies of n tokens of every input and of the output.
struct Stage {
  size_t off_q, off_k, off_v, off_o, off_la, off_lam, total;
};
static Stage stage_plan(const ll_shape& s, int n) {
  Stage g{};
  const size_t BH = (size_t)s.B * s.H, esz = s.io == LL_F32 ? 4 : 2;
  size_t off = 0;
  g.off_q = off;   off = align_up(off + BH * n * s.dk * esz, 256);
  g.off_k = off;   off = align_up(off + BH * n * s.dk * esz, 256);
  g.off_v = off;   off = align_up(off + BH * n * s.dv * esz, 256);
  g.off_o = off;   off = align_up(off + BH * n * s.dv * esz, 256);
  g.off_la = off;  off = align_up(off + BH * n * 4, 256);
  g.off_lam = off; off = align_up(off + BH * n * (size_t)s.L * 4, 256);
  g.total = off;
  return g;
}

static int bitlen_ll(long long x) {
  int b = 0;
  while (x) { ++b; x >>= 1; }
  return b;
}

// Decode-state buffers of Ls slots per (b, h).
static size_t states_bytes(const ll_shape& s, int Ls) {
  return align_up((size_t)s.B * s.H * Ls * s.dv * s.dk * 4, 256) + align_up((size_t)s.B * s.H * Ls * 4, 256);
}

// One segment of new tokens at position pos, rows [r0, r0 + n) of the caller's
// tensors, run on staged contiguous copies as a single-block continuation.
struct Segment {
  const ll_shape* s;
  const void *q, *k, *v;
  const float *la, *lam;
  void* o;
  int T;  // tokens per (b, h) slice of the caller's tensors
};
static ll_status run_piece(const Segment& g, unsigned char* stage_ws, const Stage& stg, int r0, int n, long long pos,
                           const float* st_in, const float* sc_in, float* st_out, float* sc_out, int Ls,
                           void* cont_ws, size_t cont_bytes, cudaStream_t stream, unsigned* err) {
  const ll_shape& s = *g.s;
  const int BH = s.B * s.H;
  const size_t esz = s.io == LL_F32 ? 4 : 2;
  ll_shape ps = s;
  ps.T = n;
  ps.Ls = Ls;
  unsigned char* w = stage_ws;
  ll_status st;
  if ((st = copy_rows(w + stg.off_q, g.q, BH, g.T, r0, n, s.dk * esz, true, stream)) != LL_OK) return st;
  if ((st = copy_rows(w + stg.off_k, g.k, BH, g.T, r0, n, s.dk * esz, true, stream)) != LL_OK) return st;
  if ((st = copy_rows(w + stg.off_v, g.v, BH, g.T, r0, n, s.dv * esz, true, stream)) != LL_OK) return st;
  if ((st = copy_rows(w + stg.off_la, g.la, BH, g.T, r0, n, 4, true, stream)) != LL_OK) return st;
  if ((st = copy_rows(w + stg.off_lam, g.lam, BH, g.T, r0, n, (size_t)s.L * 4, true, stream)) != LL_OK) return st;
  FwdArgs a{ps, w + stg.off_q, w + stg.off_k, w + stg.off_v, reinterpret_cast<const float*>(w + stg.off_la),
            reinterpret_cast<const float*>(w + stg.off_lam), nullptr, w + stg.off_o, st_out, sc_out, cont_ws,
            cont_bytes, stream, err};
  a.t0 = pos;
  a.state_in = st_in;
  a.scale_in = sc_in;
  st = (pos > 0 && fwd_tc_cont_supported(ps, pos)) || (pos == 0 && fwd_tc_supported(ps)) ? fwd_tc_launch(a)
                                                                                           : fwd_simt_launch(a);
  if (st != LL_OK) return st;
  return copy_rows(g.o, w + stg.off_o, BH, g.T, r0, n, s.dv * esz, false, stream);
}

static size_t piece_workspace(const ll_shape& s, int n, long long pos, int Ls) {
  ll_shape ps = s;
  ps.T = n;
  ps.Ls = Ls;
  if (pos == 0) return fwd_tc_supported(ps) ? fwd_tc_workspace(ps) : fwd_simt_workspace(ps);
  return fwd_tc_cont_supported(ps, pos) ? fwd_tc_cont_workspace(ps) : fwd_simt_cont_workspace(ps);
}

// The aligned pieces of the segment [t0, t0 + T): each piece either is the
// whole remainder, when its start is a multiple of the smallest power of two
// >= the remainder, or the largest power of two that both fits and divides
// its start; either way a single-block continuation.
static int next_piece(long long pos, long long rem) {
  long long P = 1;
  while (P < rem) P <<= 1;
  if (pos % P == 0) return (int)rem;
  long long sz = pos & -pos;  // lowest set bit of pos
  while (sz > rem) sz >>= 1;
  return (int)sz;
}

// Ragged T on the tensor-core path: the whole 128-token tiles in place, their
// decode states at T_full, then the last T % 128 tokens as a continuation.
static bool ragged_tc(const ll_shape& s) {
  if (s.io != LL_BF16 || s.T <= 128 || s.T % 128 == 0) return false;
  ll_shape f = s;
  f.T = s.T - s.T % 128;
  return fwd_tc_supported(f);
}
struct RaggedPlan {
  ll_shape full;
  int Tf, n, Lsm;
  Stage stg;
  size_t off_tc, tc_bytes, off_st, off_stage, off_tail, tail_bytes, total;
};
static RaggedPlan ragged_plan(const ll_shape& s) {
  RaggedPlan r{};
  r.n = s.T % 128;
  r.Tf = s.T - r.n;
  r.Lsm = std::max(s.Ls, bitlen_ll(s.T));
  r.full = s;
  r.full.T = r.Tf;
  r.full.Ls = r.Lsm;
  r.stg = stage_plan(s, r.n);
  size_t off = 0;
  r.off_tc = off;    r.tc_bytes = fwd_tc_workspace(r.full); off = align_up(off + r.tc_bytes, 256);
  r.off_st = off;    off += states_bytes(s, r.Lsm);
  r.off_stage = off; off = align_up(off + r.stg.total, 256);
  r.off_tail = off;  r.tail_bytes = piece_workspace(s, r.n, r.Tf, r.Lsm); off = align_up(off + r.tail_bytes, 256);
  r.total = off;
  return r;
}

// A continuation whose start is not a multiple of the smallest power of two
// >= T: its aligned pieces in turn, the decode states passed from one to the
// next through two buffers.
struct PiecesPlan {
  int maxn, npieces;
  Stage stg;
  size_t off_st0, off_st1, off_stage, off_cont, cont_bytes, total;
};
static PiecesPlan pieces_plan(const ll_shape& s, long long t0) {
  PiecesPlan p{};
  size_t cont = 0;
  for (long long pos = t0, end = t0 + s.T; pos < end;) {
    const int n = next_piece(pos, end - pos);
    p.maxn = std::max(p.maxn, n);
    cont = std::max(cont, piece_workspace(s, n, pos, s.Ls));
    ++p.npieces;
    pos += n;
  }
  p.stg = stage_plan(s, p.maxn);
  size_t off = 0;
  p.off_st0 = off;   off += states_bytes(s, s.Ls);
  p.off_st1 = off;   off += states_bytes(s, s.Ls);
  p.off_stage = off; off = align_up(off + p.stg.total, 256);
  p.off_cont = off;  p.cont_bytes = cont; off = align_up(off + cont, 256);
  p.total = off;
  return p;
}

}  // namespace llattn

using namespace llattn;

extern "C" {

int ll_version(void) { return 100; }

const char* ll_status_str(ll_status s) {
  switch (s) {
    case LL_OK: return "ok";
    case LL_ERR_INVALID_ARG: return "invalid argument";
    case LL_ERR_UNSUPPORTED: return "unsupported shape or dtype";
    case LL_ERR_CUDA: return "CUDA error";
    case LL_ERR_TIMEOUT: return "device-side wait timed out";
    case LL_ERR_WORKSPACE: return "workspace missing or too small";
    case LL_ERR_DEVICE: return "device-side argument check failed";
  }
  return "unknown status";
}

ll_status ll_last_device_error(void* stream) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  unsigned* ew = err_word();
  if (!ew) return LL_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return LL_ERR_CUDA;
  unsigned h = 0;
  if (cudaMemcpyFromSymbolAsync(&h, g_err_word, sizeof(h), 0, cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return LL_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return LL_ERR_CUDA;
  if (h) {
    unsigned zero = 0;
    if (cudaMemcpyToSymbolAsync(g_err_word, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice, st) != cudaSuccess)
      return LL_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return LL_ERR_CUDA;
  }
  if (h & kErrTimeout) return LL_ERR_TIMEOUT;
  if (h & kErrDeviceArg) return LL_ERR_DEVICE;
  return LL_OK;
}

size_t ll_attn_fwd_workspace_size(const ll_shape* s) {
  if (check_shape(s) != LL_OK) return 0;
  if (fwd_tc_supported(*s)) return fwd_tc_workspace(*s);
  if (ragged_tc(*s)) return ragged_plan(*s).total;
  return fwd_simt_workspace(*s);
}

int ll_attn_fwd_launches(const ll_shape* s) {
  if (check_shape(s) != LL_OK) return 0;
  if (fwd_tc_supported(*s)) return fwd_tc_launches(*s);
  if (ragged_tc(*s)) {  // the whole tiles with their export, then the tail as a continuation
    const RaggedPlan r = ragged_plan(*s);
    ll_shape t = *s;
    t.T = r.n;
    t.Ls = r.Lsm;
    return fwd_tc_launches(r.full) + (s->Ls > 0 ? fwd_simt_launches(t) + 2 : fwd_simt_launches(ll_shape{t.B, t.H, t.T, t.dk, t.dv, t.L, t.chunk, 0, t.io}));
  }
  return fwd_simt_launches(*s);
}

ll_status ll_attn_fwd(const ll_shape* s, const void* q, const void* k, const void* v, const float* log_alpha,
                      const float* lam, void* o, float* state_out, float* scale_out, void* workspace,
                      size_t ws_bytes, void* stream) {
  ll_status st = check_shape(s);
  if (st != LL_OK) return st;
  if (!q || !k || !v || !log_alpha || !lam || !o) return LL_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(log_alpha) || !aligned16(lam) ||
      !aligned16(o))
    return LL_ERR_INVALID_ARG;
  if ((state_out == nullptr) != (scale_out == nullptr)) return LL_ERR_INVALID_ARG;
  if (state_out) {
    if (s->Ls < 1 || !aligned16(state_out) || !aligned16(scale_out)) return LL_ERR_INVALID_ARG;
    int need = 0;
    for (unsigned x = (unsigned)s->T; x; x >>= 1) ++need;  // bit_length(T)
    if (s->Ls < need) return LL_ERR_INVALID_ARG;
  }
  const bool tc = fwd_tc_supported(*s);
  const bool ragged = !tc && ragged_tc(*s);
  const size_t need_ws = tc ? fwd_tc_workspace(*s) : ragged ? ragged_plan(*s).total : fwd_simt_workspace(*s);
  if (!workspace || ws_bytes < need_ws) return LL_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return LL_ERR_WORKSPACE;
  FwdArgs a{*s, q, k, v, log_alpha, lam, nullptr, o, state_out, scale_out, workspace, ws_bytes,
            static_cast<cudaStream_t>(stream), err_word()};
  if (!a.err) return LL_ERR_CUDA;
  if (ragged) {
    // the whole tiles on the tensor cores (row stride T) with their decode
    // states at T_full, then the last T % 128 tokens continued from them
    const RaggedPlan r = ragged_plan(*s);
    unsigned char* w = static_cast<unsigned char*>(workspace);
    float* mst = reinterpret_cast<float*>(w + r.off_st);
    float* msc = reinterpret_cast<float*>(w + r.off_st + align_up((size_t)s->B * s->H * r.Lsm * s->dv * s->dk * 4, 256));
    FwdArgs f{r.full, q, k, v, log_alpha, lam, nullptr, o, mst, msc, w + r.off_tc, r.tc_bytes, a.stream, a.err};
    f.rows_per_head = s->T;
    ll_status st = fwd_tc_launch(f);
    if (st != LL_OK) return st;
    const Segment g{s, q, k, v, log_alpha, lam, o, s->T};
    return run_piece(g, w + r.off_stage, r.stg, r.Tf, r.n, r.Tf, mst, msc, state_out, scale_out, r.Lsm,
                     w + r.off_tail, r.tail_bytes, a.stream, a.err);
  }
  return tc ? fwd_tc_launch(a) : fwd_simt_launch(a);
}

// Shape conditions of a prefill continuation at position t0 (beyond check_shape).
static ll_status check_cont(const ll_shape* s, long long t0) {
  ll_status st = check_shape(s);
  if (st != LL_OK) return st;
  if (t0 < 0 || t0 > (1ll << 61)) return LL_ERR_INVALID_ARG;
  const long long T = s->T, t1 = t0 + T;
  int bl = 0;
  for (long long x = t1; x; x >>= 1) ++bl;
  if (s->Ls < 1 || s->Ls < bl) return LL_ERR_INVALID_ARG;  // the levels of t1 need slots
  int need = 1;
  for (long long x = t1 - 1; x; x >>= 1) ++need;
  if (s->L < need) return LL_ERR_INVALID_ARG;  // the segment's keys reach levels up to bitlen(t1 - 1)
  return LL_OK;
}

// The segment sits in one aligned block of positions (t0 a multiple of the
// smallest power of two >= T): a single continuation; otherwise its aligned pieces.
static bool cont_aligned(const ll_shape* s, long long t0) {
  long long P = 1;
  while (P < s->T) P <<= 1;
  return t0 % P == 0;
}

size_t ll_attn_fwd_cont_workspace_size(const ll_shape* s, long long t0) {
  if (check_cont(s, t0) != LL_OK) return 0;
  if (!cont_aligned(s, t0)) return pieces_plan(*s, t0).total;
  return fwd_tc_cont_supported(*s, t0) ? fwd_tc_cont_workspace(*s) : fwd_simt_cont_workspace(*s);
}

ll_status ll_attn_fwd_cont(const ll_shape* s, long long t0, const float* state_in, const float* scale_in,
                           const void* q, const void* k, const void* v, const float* log_alpha, const float* lam,
                           void* o, float* state_out, float* scale_out, void* workspace, size_t ws_bytes,
                           void* stream) {
  ll_status st = check_cont(s, t0);
  if (st != LL_OK) return st;
  if (!state_in || !scale_in || !q || !k || !v || !log_alpha || !lam || !o) return LL_ERR_INVALID_ARG;
  if ((state_out == nullptr) != (scale_out == nullptr)) return LL_ERR_INVALID_ARG;
  if (!aligned16(state_in) || !aligned16(scale_in) || !aligned16(q) || !aligned16(k) || !aligned16(v) ||
      !aligned16(log_alpha) || !aligned16(lam) || !aligned16(o) || (state_out && !aligned16(state_out)) ||
      (scale_out && !aligned16(scale_out)))
    return LL_ERR_INVALID_ARG;
  if (state_out) {  // the new states are written while the old ones are read
    const size_t n = (size_t)s->B * s->H * s->Ls * s->dv * s->dk * sizeof(float);
    const size_t ns = (size_t)s->B * s->H * s->Ls * sizeof(float);
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(state_in), a1 = reinterpret_cast<uintptr_t>(state_out);
    const uintptr_t c0 = reinterpret_cast<uintptr_t>(scale_in), c1 = reinterpret_cast<uintptr_t>(scale_out);
    if (a0 < a1 + n && a1 < a0 + n) return LL_ERR_INVALID_ARG;
    if (c0 < c1 + ns && c1 < c0 + ns) return LL_ERR_INVALID_ARG;
  }
  const size_t need_ws = ll_attn_fwd_cont_workspace_size(s, t0);
  if (!workspace || ws_bytes < need_ws) return LL_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return LL_ERR_WORKSPACE;
  FwdArgs a{*s, q, k, v, log_alpha, lam, nullptr, o, state_out, scale_out, workspace, ws_bytes,
            static_cast<cudaStream_t>(stream), err_word()};
  if (!a.err) return LL_ERR_CUDA;
  if (!cont_aligned(s, t0)) {
    // aligned pieces in turn, each continued from the previous one's states
    const PiecesPlan pp = pieces_plan(*s, t0);
    unsigned char* w = static_cast<unsigned char*>(workspace);
    const size_t sbytes = align_up((size_t)s->B * s->H * s->Ls * s->dv * s->dk * 4, 256);
    float* stb[2] = {reinterpret_cast<float*>(w + pp.off_st0), reinterpret_cast<float*>(w + pp.off_st1)};
    float* scb[2] = {reinterpret_cast<float*>(w + pp.off_st0 + sbytes), reinterpret_cast<float*>(w + pp.off_st1 + sbytes)};
    const Segment g{s, q, k, v, log_alpha, lam, o, s->T};
    const float* sin = state_in;
    const float* scin = scale_in;
    int i = 0;
    for (long long pos = t0, end = t0 + s->T; pos < end; ++i) {
      const int n = next_piece(pos, end - pos);
      const bool last = pos + n == end;
      float* so = last ? state_out : stb[i & 1];
      float* sco = last ? scale_out : scb[i & 1];
      const ll_status st = run_piece(g, w + pp.off_stage, pp.stg, (int)(pos - t0), n, pos, sin, scin, so, sco, s->Ls,
                                     w + pp.off_cont, pp.cont_bytes, a.stream, a.err);
      if (st != LL_OK) return st;
      sin = so;
      scin = sco;
      pos += n;
    }
    return LL_OK;
  }
  const bool tc = fwd_tc_cont_supported(*s, t0);
  a.t0 = t0;
  a.state_in = state_in;
  a.scale_in = scale_in;
  return tc ? fwd_tc_launch(a) : fwd_simt_launch(a);
}

ll_status ll_attn_decode_step(int B, int H, int dk, int dv, int Ls, ll_dtype io, const int64_t* t, const void* q,
                              const void* k, const void* v, const float* log_alpha, const float* lam,
                              float* states, float* scales, void* o, void* stream) {
  if (B < 1 || H < 1 || Ls < 1 || Ls > 62) return LL_ERR_INVALID_ARG;
  if (io != LL_F32 && io != LL_BF16) return LL_ERR_INVALID_ARG;
  if (!head_dim_ok(dk) || !head_dim_ok(dv)) return LL_ERR_UNSUPPORTED;
  if (!t || !q || !k || !v || !log_alpha || !lam || !states || !scales || !o) return LL_ERR_INVALID_ARG;
  if (!aligned16(t) || !aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(log_alpha) ||
      !aligned16(lam) || !aligned16(states) || !aligned16(scales) || !aligned16(o))
    return LL_ERR_INVALID_ARG;
  unsigned* ew = err_word();
  if (!ew) return LL_ERR_CUDA;
  return decode_launch(B, H, dk, dv, Ls, io, t, q, k, v, log_alpha, lam, states, scales, o,
                       static_cast<cudaStream_t>(stream), ew);
}

size_t ll_attn_fwd_level_decay_workspace_size(const ll_shape* s) {
  if (check_shape(s) != LL_OK) return 0;
  if (fwd_tc_level_decay_supported(*s)) return fwd_tc_level_decay_workspace(*s);
  return fwd_level_decay_workspace(*s);
}

int ll_attn_fwd_level_decay_launches(const ll_shape* s) {
  if (check_shape(s) != LL_OK) return 0;
  if (fwd_tc_level_decay_supported(*s)) return fwd_tc_level_decay_launches(*s);
  if (fwd_level_decay_workspace(*s) == 0) return 0;
  return fwd_level_decay_launches(*s);
}

ll_status ll_attn_fwd_level_decay(const ll_shape* s, const void* q, const void* k, const void* v,
                                  const float* log_alpha, const float* lam, void* o, float* state_out,
                                  float* scale_out, void* workspace, size_t ws_bytes, void* stream) {
  ll_status st = check_shape(s);
  if (st != LL_OK) return st;
  if (!q || !k || !v || !log_alpha || !lam || !o) return LL_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(log_alpha) || !aligned16(lam) ||
      !aligned16(o))
    return LL_ERR_INVALID_ARG;
  if ((state_out == nullptr) != (scale_out == nullptr)) return LL_ERR_INVALID_ARG;
  if (state_out) {
    if (s->Ls < 1 || !aligned16(state_out) || !aligned16(scale_out)) return LL_ERR_INVALID_ARG;
    int need = 0;
    for (unsigned x = (unsigned)s->T; x; x >>= 1) ++need;  // bit_length(T)
    if (s->Ls < need) return LL_ERR_INVALID_ARG;
  }
  const bool tc = fwd_tc_level_decay_supported(*s);
  const size_t need_ws = tc ? fwd_tc_level_decay_workspace(*s) : fwd_level_decay_workspace(*s);
  if (need_ws == 0) return LL_ERR_UNSUPPORTED;
  if (!workspace || ws_bytes < need_ws) return LL_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return LL_ERR_WORKSPACE;
  FwdArgs a{*s, q, k, v, log_alpha, lam, nullptr, o, state_out, scale_out, workspace, ws_bytes,
            static_cast<cudaStream_t>(stream), err_word()};
  if (!a.err) return LL_ERR_CUDA;
  return tc ? fwd_tc_level_decay_launch(a) : fwd_level_decay_launch(a);
}

ll_status ll_attn_decode_step_level_decay(int B, int H, int dk, int dv, int Ls, ll_dtype io, const int64_t* t,
                                          const void* q, const void* k, const void* v, const float* log_alpha,
                                          const float* lam, float* states, float* scales, void* o, void* stream) {
  if (B < 1 || H < 1 || Ls < 1 || Ls > 62) return LL_ERR_INVALID_ARG;
  if (io != LL_F32 && io != LL_BF16) return LL_ERR_INVALID_ARG;
  if (!head_dim_ok(dk) || !head_dim_ok(dv)) return LL_ERR_UNSUPPORTED;
  if (!t || !q || !k || !v || !log_alpha || !lam || !states || !scales || !o) return LL_ERR_INVALID_ARG;
  if (!aligned16(t) || !aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(log_alpha) ||
      !aligned16(lam) || !aligned16(states) || !aligned16(scales) || !aligned16(o))
    return LL_ERR_INVALID_ARG;
  unsigned* ew = err_word();
  if (!ew) return LL_ERR_CUDA;
  return decode_level_decay_launch(B, H, dk, dv, Ls, io, t, q, k, v, log_alpha, lam, states, scales, o,
                                   static_cast<cudaStream_t>(stream), ew);
}

size_t ll_attn_bwd_workspace_size(const ll_shape* s) {
  if (check_shape(s) != LL_OK || s->Ls != 0) return 0;
  return bwd_simt_workspace(*s);
}

int ll_attn_bwd_launches(const ll_shape* s) {
  if (check_shape(s) != LL_OK || s->Ls != 0) return 0;
  return bwd_simt_launches(*s);
}

ll_status ll_attn_bwd(const ll_shape* s, const void* q, const void* k, const void* v, const float* log_alpha,
                      const float* lam, const void* dout, void* dq, void* dk, void* dv, float* dlog_alpha,
                      float* dlam, void* workspace, size_t ws_bytes, void* stream) {
  ll_status st = check_shape(s);
  if (st != LL_OK) return st;
  if (s->Ls != 0) return LL_ERR_INVALID_ARG;
  const void* in[6] = {q, k, v, log_alpha, lam, dout};
  const void* out[5] = {dq, dk, dv, dlog_alpha, dlam};
  for (const void* p : in)
    if (!p || !aligned16(p)) return LL_ERR_INVALID_ARG;
  for (const void* p : out)
    if (!p || !aligned16(p)) return LL_ERR_INVALID_ARG;
  // the gradients are written while the inputs are still read: no output may
  // overlap an input or another output
  const size_t es = s->io == LL_F32 ? 4 : 2;
  const size_t rows = (size_t)s->B * s->H * s->T;
  const size_t in_bytes[6] = {rows * s->dk * es, rows * s->dk * es, rows * s->dv * es, rows * 4, rows * s->L * 4,
                              rows * s->dv * es};
  const size_t out_bytes[5] = {rows * s->dk * es, rows * s->dk * es, rows * s->dv * es, rows * 4, rows * s->L * 4};
  auto overlap = [](const void* a, size_t na, const void* b, size_t nb) {
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + nb && y < x + na;
  };
  for (int i = 0; i < 5; ++i) {
    for (int j = 0; j < 6; ++j)
      if (overlap(out[i], out_bytes[i], in[j], in_bytes[j])) return LL_ERR_INVALID_ARG;
    for (int j = i + 1; j < 5; ++j)
      if (overlap(out[i], out_bytes[i], out[j], out_bytes[j])) return LL_ERR_INVALID_ARG;
  }
  const size_t need_ws = bwd_simt_workspace(*s);
  if (!workspace || ws_bytes < need_ws) return LL_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return LL_ERR_WORKSPACE;
  BwdArgs a{*s, q, k, v, dout, log_alpha, lam, dq, dk, dv, dlog_alpha, dlam, workspace, ws_bytes,
            static_cast<cudaStream_t>(stream), err_word()};
  if (!a.err) return LL_ERR_CUDA;
  return bwd_simt_launch(a);
}

size_t ll_gdn_fwd_b_workspace_size(const ll_shape* s) {
  if (check_shape(s) != LL_OK || s->Ls != 0 || s->T % s->chunk != 0) return 0;
  return gdn_b_workspace(*s);
}

ll_status ll_gdn_fwd_b(const ll_shape* s, const void* q, const void* k, const void* v, const float* log_alpha,
                       const float* beta, const float* lam, void* o, void* workspace, size_t ws_bytes,
                       void* stream) {
  ll_status st = check_shape(s);
  if (st != LL_OK) return st;
  if (s->T % s->chunk != 0) return LL_ERR_INVALID_ARG;  // whole chunks only
  if (s->Ls != 0) return LL_ERR_INVALID_ARG;
  if (!q || !k || !v || !log_alpha || !beta || !lam || !o) return LL_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(log_alpha) || !aligned16(beta) ||
      !aligned16(lam) || !aligned16(o))
    return LL_ERR_INVALID_ARG;
  const size_t need_ws = gdn_b_workspace(*s);
  if (need_ws == 0) return LL_ERR_UNSUPPORTED;
  if (!workspace || ws_bytes < need_ws) return LL_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return LL_ERR_WORKSPACE;
  FwdArgs a{*s, q, k, v, log_alpha, lam, beta, o, nullptr, nullptr, workspace, ws_bytes,
            static_cast<cudaStream_t>(stream), err_word()};
  if (!a.err) return LL_ERR_CUDA;
  return gdn_b_launch(a);
}

ll_status ll_gdn_decode_step(int B, int H, int dk, int dv, int Ls, ll_dtype io, const int64_t* t, const void* q,
                             const void* k, const void* v, const float* log_alpha, const float* beta,
                             const float* lam, float* states, void* o, void* stream) {
  if (B < 1 || H < 1 || Ls < 1 || Ls > 62) return LL_ERR_INVALID_ARG;
  if (io != LL_F32 && io != LL_BF16) return LL_ERR_INVALID_ARG;
  if (!head_dim_ok(dk) || !head_dim_ok(dv)) return LL_ERR_UNSUPPORTED;
  if (!t || !q || !k || !v || !log_alpha || !beta || !lam || !states || !o) return LL_ERR_INVALID_ARG;
  if (!aligned16(t) || !aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(log_alpha) ||
      !aligned16(beta) || !aligned16(lam) || !aligned16(states) || !aligned16(o))
    return LL_ERR_INVALID_ARG;
  unsigned* ew = err_word();
  if (!ew) return LL_ERR_CUDA;
  return gdn_decode_launch(B, H, dk, dv, Ls, io, t, q, k, v, log_alpha, beta, lam, states, o,
                           static_cast<cudaStream_t>(stream), ew);
}

size_t ll_gdn_fwd_workspace_size(const ll_shape* s) {
  if (check_shape(s) != LL_OK || s->Ls != 0 || s->T % s->chunk != 0) return 0;
  return gdn_workspace(*s);
}

ll_status ll_gdn_fwd(const ll_shape* s, const void* q, const void* k, const void* v, const float* log_alpha,
                     const float* beta, const float* lam, void* o, void* workspace, size_t ws_bytes,
                     void* stream) {
  ll_status st = check_shape(s);
  if (st != LL_OK) return st;
  if (s->T % s->chunk != 0) return LL_ERR_INVALID_ARG;  // whole chunks only
  if (s->Ls != 0) return LL_ERR_INVALID_ARG;
  if (!q || !k || !v || !log_alpha || !beta || !lam || !o) return LL_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(log_alpha) || !aligned16(beta) ||
      !aligned16(lam) || !aligned16(o))
    return LL_ERR_INVALID_ARG;
  const size_t need_ws = gdn_workspace(*s);
  if (need_ws == 0) return LL_ERR_UNSUPPORTED;
  if (!workspace || ws_bytes < need_ws) return LL_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return LL_ERR_WORKSPACE;
  FwdArgs a{*s, q, k, v, log_alpha, lam, beta, o, nullptr, nullptr, workspace, ws_bytes,
            static_cast<cudaStream_t>(stream), err_word()};
  if (!a.err) return LL_ERR_CUDA;
  return gdn_launch(a);
}

}  // extern "C"
