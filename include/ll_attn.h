/*
 * ll_attn.h -- C ABI of libllattn.so: GB300 (sm_103a) log-linear attention.
 *
 * Operations (sources are the pages' titles and sections):
 *   ll_attn_fwd          causal log-linear Mamba-2 forward
 *                          o_t = sum_{s<=t} (q_t . k_s) Gamma(t,s) lam_t[l(t,s)] v_s,
 *                        i.e. O = (Q K^T . M^S . M^H) V.  "Log-Linear Attention"
 *                        study note (dimensionstp.github.io) §3-4 "Parallel form"
 *                        and §3-5 (M = M^S . M^H, Log-Linear Mamba-2); computed
 *                        chunk-wise in O(T log T) as in §3-1 / the chunk-scan of
 *                        the gist.science (zh) summary §2.3.
 *   ll_attn_fwd_cont     the forward of a segment of new tokens after a prefix held
 *                        as decode states (prefill continuation), §3-4/§3-6.
 *   ll_attn_decode_step  one token of Fenwick-state decoding: study note §3-3
 *                        "Recurrent form" (o_t = sum_l lam_t^(l) q_t^T S_t^(l))
 *                        and §3-6 "Memory-efficient decoding"; carry/merge as in
 *                        the drawer analogy of the gist.science (zh) summary.
 *   ll_attn_bwd          backward of ll_attn_fwd: the gradients of q, k, v,
 *                        log_alpha and lam for an upstream gradient of o.  The
 *                        pages name the backward, and in it the lambda-term
 *                        gradient, as the hard part of an implementation
 *                        (study note §4-5 "Implementation notes" and §6
 *                        "Limitations"; gist.science (zh) summary §5) without
 *                        printing it: it is the exact gradient of §3-4's O.
 *   ll_gdn_fwd           Log-Linear Gated DeltaNet forward, study note §3-5 and
 *                        gist.science (de) Technische Zusammenfassung §2; the
 *                        gated delta rule itself is not on the pages (reading A:
 *                        O = (C_GDN . M^H) V, every level state follows the full
 *                        gated-delta transition).
 *   ll_gdn_fwd_b         the same forward under reading B (log-linear Mamba-2 on the
 *                        delta-rule pseudo-values), study note §3-5.
 *   ll_gdn_decode_step   one token of Log-Linear Gated DeltaNet decoding over the
 *                        Fenwick level states (reading A), study note §3-5/§3-6.
 *   ll_attn_fwd_level_decay, ll_attn_decode_step_level_decay
 *                        the forward and the decode step with one decay per level
 *                        (study note §7 "Follow-up design" names a learned memory
 *                        decay per level; the reading implemented is stated at
 *                        their declarations).
 *
 * Definitions used throughout:
 *   level l(t,s) = 0 if s == t, else floor(log2(t xor s)) + 1   (0 <= s <= t);
 *   Gamma(t,s)   = prod_{r=s+1..t} alpha_r, passed as log_alpha (float32);
 *   a Fenwick level l >= 1 of query t is non-empty iff bit l-1 of t is set.
 *
 * Conventions for every entry point:
 *   - All tensor pointers are DEVICE pointers owned by the caller; the library
 *     never allocates, frees or keeps them.  Layouts are contiguous, row-major,
 *     head-major; every pointer must be 16-byte aligned.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy default
 *     stream).  Argument errors are detected on the host before anything is
 *     launched and return LL_ERR_INVALID_ARG / LL_ERR_UNSUPPORTED /
 *     LL_ERR_WORKSPACE without touching device memory.  A launch failure
 *     returns LL_ERR_CUDA.
 *   - Conditions only the device can see (a decode position that does not fit
 *     the stored levels; a bounded device-side wait that expired) set a
 *     device error word; ll_last_device_error() synchronises the stream and
 *     reports (and clears) it.  No kernel traps or spins unboundedly.
 *   - Output values are unspecified after an error.
 *   - Only one call may use a given workspace at a time.
 */
#ifndef LL_ATTN_H
#define LL_ATTN_H

#include <stddef.h>
#include <stdint.h>

/* Symbols of the C ABI are the only ones the shared library exports. */
#if defined(__GNUC__)
#define LL_API __attribute__((visibility("default")))
#else
#define LL_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  LL_OK = 0,
  LL_ERR_INVALID_ARG = 1, /* null pointer, bad size, misaligned pointer     */
  LL_ERR_UNSUPPORTED = 2, /* valid but not implemented (e.g. head dim 96)   */
  LL_ERR_CUDA = 3,        /* a CUDA runtime call or launch failed            */
  LL_ERR_TIMEOUT = 4,     /* a bounded device-side wait expired             */
  LL_ERR_WORKSPACE = 5,   /* workspace pointer null or too small            */
  LL_ERR_DEVICE = 6       /* device-side argument check failed (e.g. decode
                             position beyond the stored levels)             */
} ll_status;

typedef enum { LL_F32 = 0, LL_BF16 = 1 } ll_dtype;

/* Problem shape of a forward call.
 *   B, H      batch rows and heads (>= 1)
 *   T         sequence length (>= 1); the Gated DeltaNet entry points need a
 *             multiple of `chunk`, the Mamba-2 forward takes any T (with bf16
 *             and d = 128 or 64 the whole 128-token tiles run on the tensor cores
 *             and the last T % 128 tokens as a continuation from their decode
 *             states, on the CUDA cores)
 *   dk, dv    key / value head dims, each in {16, 32, 64, 128}
 *   L         number of lambda levels per token, >= levels touched by T
 *             (1 if T == 1, else bit_length(T-1) + 1)
 *   chunk     chunk length of the chunked algorithm, in {16, 32, 64, 128}; the
 *             result does not depend on it (up to rounding).  The bf16
 *             tensor-core path of ll_attn_fwd tiles by 128 tokens whatever
 *             `chunk` is (it needs T % 128 == 0 and dk == dv in {64, 128}; d = 64
 *             runs as 128 with the operand tiles' upper halves zero).
 *   Ls        number of stored decode levels of state_out (levels 1..Ls);
 *             0 = no state export
 *   io        dtype of q, k, v and o (LL_F32 or LL_BF16); log_alpha, lam,
 *             beta are always float32; accumulation is float32.           */
typedef struct {
  int B, H, T, dk, dv, L, chunk, Ls;
  ll_dtype io;
} ll_shape;

/* Library version (major*10000 + minor*100 + patch). */
LL_API int ll_version(void);

/* Human-readable name of a status code (static string). */
LL_API const char* ll_status_str(ll_status s);

/* Synchronise `stream`, then read and clear the device error word.
 * Returns LL_OK, LL_ERR_TIMEOUT or LL_ERR_DEVICE (or LL_ERR_CUDA if the
 * synchronisation itself failed). */
LL_API ll_status ll_last_device_error(void* stream);

/* Bytes of workspace ll_attn_fwd needs for `shape` (0 on invalid shape). */
LL_API size_t ll_attn_fwd_workspace_size(const ll_shape* shape);

/* Number of kernel launches one ll_attn_fwd call with `shape` makes
 * (0 on an invalid shape); useful when capturing calls in CUDA graphs. */
LL_API int ll_attn_fwd_launches(const ll_shape* shape);

/* Log-linear Mamba-2 forward.
 *   q          [B,H,T,dk]  io dtype
 *   k          [B,H,T,dk]  io dtype
 *   v          [B,H,T,dv]  io dtype
 *   log_alpha  [B,H,T]     float32, log of the per-step decay alpha_t (<= 0
 *                          for a decay; larger values are computed as given
 *                          and may overflow)
 *   lam        [B,H,T,L]   float32, lam[t][l] weights level l of query t
 *   o          [B,H,T,dv]  io dtype, written
 *   state_out  [B,H,Ls,dv,dk] float32 or NULL: the Fenwick level states of
 *              position T (slot i = level i+1; bucket of level l is non-empty
 *              iff bit l-1 of T is set; each decayed to token T-1), ready for
 *              ll_attn_decode_step at t = T.  Empty levels are written as 0.
 *   scale_out  [B,H,Ls]    float32 or NULL (required iff state_out): lazy
 *              decay scale of each slot, written as 1 (non-empty) or 0 (empty).
 *   workspace  device scratch of >= ll_attn_fwd_workspace_size(shape) bytes,
 *              256-byte aligned, caller-owned, contents need not be cleared.
 * Requires Ls >= bit_length(T) when state_out is given. */
LL_API ll_status ll_attn_fwd(const ll_shape* shape, const void* q, const void* k, const void* v,
                      const float* log_alpha, const float* lam, void* o, float* state_out,
                      float* scale_out, void* workspace, size_t ws_bytes, void* stream);

/* One decode step of log-linear Mamba-2 for every (b, h).
 *   B, H, dk, dv  as above (dk, dv in {16, 32, 64, 128}); Ls stored levels
 *   io            dtype of q, k, v, o
 *   t      [B]          int64, position of this token in each batch row
 *   q, k   [B,H,dk]     io dtype;   v [B,H,dv] io dtype
 *   log_alpha [B,H]     float32
 *   lam    [B,H,Ls+1]   float32, lam[0] weights the token itself (level 0)
 *   states [B,H,Ls,dv,dk] float32, in/out.  Slot i holds level i+1 as
 *          S_stored with true state = scale * S_stored; on entry the
 *          non-empty slots are the set bits of t (levels of query t), decayed
 *          to t-1.  On exit they describe position t+1.
 *   scales [B,H,Ls]     float32, in/out, the lazy per-slot scales.
 *   o      [B,H,dv]     io dtype, written.
 * Per (b,h) the step reads the non-empty states once and writes one merged
 * state (level ctz(t+1)+1).  A position with t+1 >= 2^Ls or t < 0 sets the
 * device error word (LL_ERR_DEVICE) and leaves that row untouched. */
LL_API ll_status ll_attn_decode_step(int B, int H, int dk, int dv, int Ls, ll_dtype io, const int64_t* t,
                              const void* q, const void* k, const void* v, const float* log_alpha,
                              const float* lam, float* states, float* scales, void* o, void* stream);

/* Bytes of workspace ll_attn_fwd_cont needs (0 when the shape or t0 is
 * invalid for a continuation). */
LL_API size_t ll_attn_fwd_cont_workspace_size(const ll_shape* shape, long long t0);

/* Prefill continuation: ll_attn_fwd for the tokens at positions t0 .. t0+T-1
 * of a sequence whose first t0 tokens are carried by their decode states
 * (study note §3-6: the O(log T) level states; the chunk-wise form of §3-4 /
 * the gist.science (zh) summary §2.3 for the new tokens).
 *   shape      as ll_attn_fwd for the T new tokens; shape->Ls >= bit_length(t0+T)
 *              slots; shape->L >= bit_length(t0+T-1)+1 (lam indexes absolute levels)
 *   t0         position of the first new token (>= 0).  When t0 is a
 *              multiple of the smallest power of two >= T (the new tokens sit
 *              in one aligned block of positions, as fixed-size power-of-two
 *              segments do) the segment runs as one continuation; otherwise it
 *              runs as its aligned pieces in turn (each the largest power of
 *              two that divides its start and fits, or the whole remainder once
 *              that is aligned), each piece on contiguous copies of its rows
 *              and continued from the previous piece's decode states, so the
 *              workspace then also holds those copies and two state buffers
 *   state_in   [B,H,Ls,dv,dk] float32, scale_in [B,H,Ls]: the decode states of
 *              position t0 (as ll_attn_fwd exports them or ll_attn_decode_step
 *              leaves them; true state = scale * S, decayed to t0-1)
 *   q, k, v, log_alpha, lam, o: the new tokens, layouts of ll_attn_fwd
 *   state_out, scale_out: nullable (both or neither); the decode states of
 *              position t0+T; must not overlap state_in / scale_in
 *   workspace  >= ll_attn_fwd_cont_workspace_size(shape, t0) bytes, 256-aligned
 * o_t = sum over all keys s <= t (prefix included) of
 *       (q_t . k_s) Gamma(t,s) lam_t[l(t,s)] v_s.
 * bf16 io with d = 128 or 64 and T a multiple of 128 runs on the tensor-core
 * path (the prefix levels become extra level products of every tile), every
 * other shape on the CUDA-core path. */
LL_API ll_status ll_attn_fwd_cont(const ll_shape* shape, long long t0, const float* state_in,
                                  const float* scale_in, const void* q, const void* k, const void* v,
                                  const float* log_alpha, const float* lam, void* o, float* state_out,
                                  float* scale_out, void* workspace, size_t ws_bytes, void* stream);

/* ---- one decay per level ----
 * "Log-Linear Attention" study note §7 "Follow-up design" lists a learned
 * memory decay per level and defines nothing more.  The reading implemented:
 * the memory of level l decays at its own rate alpha_t^(l), so at every step
 * r a key decays at the rate of the level it occupies then,
 *   o_t = sum_{s<=t} lam_t[l(t,s)] prod_{r in (s,t]} alpha_r^(l(r,s)) (q_t.k_s) v_s,
 * which is the recurrent form of §3-3 with one decay per level state (the
 * carry-merge unchanged).  With every column of log_alpha equal it is
 * ll_attn_fwd. */

/* Bytes of workspace ll_attn_fwd_level_decay needs (0 on an invalid shape, or
 * when T needs more than 4096 chunks of the effective chunk length). */
LL_API size_t ll_attn_fwd_level_decay_workspace_size(const ll_shape* shape);

/* Kernel launches of one ll_attn_fwd_level_decay call (0 when unsupported). */
LL_API int ll_attn_fwd_level_decay_launches(const ll_shape* shape);

/* The forward with one decay per level.  Arguments as ll_attn_fwd, except
 *   log_alpha  [B,H,T,L]  float32: log_alpha[t][l] is the log decay of level
 *              l at step t (column 0 is never read: a key is at level 0 only
 *              at its own step, which applies no decay).
 * state_out / scale_out: the level states of position T as in ll_attn_fwd
 * (each bucket decayed to token T-1 under this rule), ready for
 * ll_attn_decode_step_level_decay at t = T.
 * bf16 io with d = 128 or 64, T a multiple of 128 and L <= 16 runs on the
 * tensor cores (the forward's persistent kernel in a per-level mode, after
 * two small kernels that tabulate each level's decay over the tiles); every
 * other shape on the CUDA cores (float32 FMA, float64 running sums of the log
 * decays), LL_ERR_UNSUPPORTED there beyond 4096 chunks. */
LL_API ll_status ll_attn_fwd_level_decay(const ll_shape* shape, const void* q, const void* k, const void* v,
                                         const float* log_alpha, const float* lam, void* o, float* state_out,
                                         float* scale_out, void* workspace, size_t ws_bytes, void* stream);

/* One decode step with one decay per level.  Arguments as
 * ll_attn_decode_step, except log_alpha [B,H,Ls+1] float32 (entry l for level
 * l; entry 0 is never read): the lazy scale of slot i is multiplied by
 * alpha_t^(i+1). */
LL_API ll_status ll_attn_decode_step_level_decay(int B, int H, int dk, int dv, int Ls, ll_dtype io,
                                                 const int64_t* t, const void* q, const void* k, const void* v,
                                                 const float* log_alpha, const float* lam, float* states,
                                                 float* scales, void* o, void* stream);

/* Bytes of workspace ll_attn_bwd needs for `shape` (0 on an invalid shape or
 * shape->Ls != 0). */
LL_API size_t ll_attn_bwd_workspace_size(const ll_shape* shape);

/* Number of kernel launches one ll_attn_bwd call makes (0 on an invalid shape).
 * The bf16 d = 128 path also clears its key-side level nodes in the workspace
 * with one cudaMemsetAsync on `stream`, which this count leaves out. */
LL_API int ll_attn_bwd_launches(const ll_shape* shape);

/* Backward of ll_attn_fwd.  For f = sum(o . dout) with o = ll_attn_fwd(q, k,
 * v, log_alpha, lam), writes the exact gradients
 *   dq = (dP . M) K,  dk = (dP . M)^T Q,  dv = (QK^T . M)^T dout,
 *   dlam[t][l]     = sum over keys s of level l of query t of
 *                    (dout_t . v_s)(q_t . k_s) Gamma(t,s),
 *   dlog_alpha[r]  = sum over t >= r of dc_t, where dc_t is the derivative of
 *                    f by the cumulative log-decay c_t (Gamma(t,s) = exp(c_t - c_s)),
 * with M = M^S . M^H and dP = dout V^T on the causal triangle.
 *   shape      as ll_attn_fwd; shape->Ls must be 0 (no state gradients)
 *   q, k, v, log_alpha, lam   the forward's inputs, layouts of ll_attn_fwd
 *   dout       [B,H,T,dv]  io dtype, upstream gradient of o
 *   dq, dk     [B,H,T,dk]  io dtype, written
 *   dv         [B,H,T,dv]  io dtype, written
 *   dlog_alpha [B,H,T]     float32, written (dlog_alpha[0] of every row is 0
 *                          up to rounding: no decay acts before the first token)
 *   dlam       [B,H,T,L]   float32, written (levels no key reaches are 0)
 *   workspace  >= ll_attn_bwd_workspace_size(shape) bytes, 256-byte aligned
 * No output may overlap an input or another output (LL_ERR_INVALID_ARG).
 * Any T is accepted (a partial last chunk is handled).  bf16 io with
 * dk = dv = 128 runs on the tensor cores over 128-token tiles whatever
 * `chunk` is (bf16 operands for the masked scores, their gradient, the
 * Fenwick nodes and the scaled dout; float32 accumulation); every other
 * shape runs in float32 on the CUDA cores.  Cumulative decays and the
 * suffix sums of dlog_alpha are float64.  The order of the float32
 * additions into the key-side level nodes is not fixed, so results can
 * differ in the last bits between calls.  A bounded device-side wait that
 * expires sets the device error word (LL_ERR_TIMEOUT from
 * ll_last_device_error); the gradients are then unspecified. */
LL_API ll_status ll_attn_bwd(const ll_shape* shape, const void* q, const void* k, const void* v,
                             const float* log_alpha, const float* lam, const void* dout, void* dq, void* dk,
                             void* dv, float* dlog_alpha, float* dlam, void* workspace, size_t ws_bytes,
                             void* stream);

/* Size in bytes of the fixed device scratch of ll_attn_fwd_noalloc. */
#define LL_NOALLOC_SCRATCH_BYTES (32u << 20)

/* ll_attn_fwd for callers that cannot allocate device memory.  The paper has
 * no counterpart of this entry point; it exists for callers that can neither
 * pass a workspace nor allocate one -- a host application that reserves all
 * device memory for its own pool at start-up and forbids later cudaMalloc,
 * a plugin of such a runtime with no allocator to hand down, or a loop where
 * a cudaMalloc (which may synchronise the device) is not acceptable.
 *   Arguments, layouts and results are those of ll_attn_fwd without
 *   `workspace`/`ws_bytes`.  The scratch is a fixed array of
 *   LL_NOALLOC_SCRATCH_BYTES inside the library's device image, held on every
 *   GPU that loads the library until the process exits.  The call allocates
 *   and frees nothing.
 *   Returns LL_ERR_WORKSPACE when ll_attn_fwd_workspace_size(shape) exceeds
 *   LL_NOALLOC_SCRATCH_BYTES (the shape is too large for the fixed scratch),
 *   and LL_ERR_INVALID_ARG for an invalid shape.
 *   All calls on a device share the one scratch array, which keeps the last
 *   call's contents (the forward needs none of it cleared): calls whose
 *   execution overlaps on the GPU (other streams, other host threads) race.
 *   The first call on each device (with that device current) looks up the
 *   array's device address; make that first call before any stream capture.
 *   The address is kept for the life of the process: after cudaDeviceReset
 *   (or anything else that destroys and re-creates the device's primary
 *   context) the array may move, so this entry point must not be used on
 *   that device again. */
LL_API ll_status ll_attn_fwd_noalloc(const ll_shape* shape, const void* q, const void* k, const void* v,
                                     const float* log_alpha, const float* lam, void* o, float* state_out,
                                     float* scale_out, void* stream);

/* One decode step of log-linear Gated DeltaNet (reading A) for every (b, h):
 * study note §3-5 (the Gated DeltaNet variant) and §3-6 (decoding with
 * O(log T) level states); the gated delta rule itself is the standard one
 * (the pages print no delta-rule equations).
 *   B, H, dk, dv, Ls, io, t, q, k, v, log_alpha, lam, o: as
 *          ll_attn_decode_step (lam[0] weights the token itself)
 *   beta   [B,H]        float32, delta-rule write strength
 *   states [B,H,Ls,dv,dk] float32, in/out, TRUE states (no lazy scale: the
 *          transition is not a scalar).  Slot i holds level i+1; on entry the
 *          non-empty slots are the set bits of t, each after the transition of
 *          token t-1; on exit they are the set bits of t+1.
 * Per (b,h): every non-empty level S <- alpha S (I - beta k k^T); the token
 * is level 0, beta v k^T; o = lam_0 beta (k.q) v + sum_l lam_l S^(l) q with
 * the transitioned states; level 0 and slots 0..j-1 (j = ctz(t+1)) merge by
 * addition into slot j.  Every non-empty state is read and written once.
 * Keys are expected to be L2-normalised (not checked).  A position with
 * t+1 >= 2^Ls or t < 0 sets the device error word (LL_ERR_DEVICE) and leaves
 * that row untouched. */
LL_API ll_status ll_gdn_decode_step(int B, int H, int dk, int dv, int Ls, ll_dtype io, const int64_t* t,
                                    const void* q, const void* k, const void* v, const float* log_alpha,
                                    const float* beta, const float* lam, float* states, void* o, void* stream);

/* Bytes of workspace ll_gdn_fwd needs for `shape` (0 on invalid shape). */
LL_API size_t ll_gdn_fwd_workspace_size(const ll_shape* shape);

/* Log-Linear Gated DeltaNet forward (reading A), same layouts as
 * ll_attn_fwd plus
 *   beta  [B,H,T] float32, delta-rule write strength.
 * shape->Ls must be 0 (no state export).  Keys are expected to be
 * L2-normalised (as in Gated DeltaNet); this is not checked. */
LL_API ll_status ll_gdn_fwd(const ll_shape* shape, const void* q, const void* k, const void* v,
                     const float* log_alpha, const float* beta, const float* lam, void* o,
                     void* workspace, size_t ws_bytes, void* stream);

/* Bytes of workspace ll_gdn_fwd_b needs for `shape` (0 when the shape is
 * invalid or not supported by reading B: it needs dk = dv = 128 and
 * chunk >= 64). */
LL_API size_t ll_gdn_fwd_b_workspace_size(const ll_shape* shape);

/* Log-Linear Gated DeltaNet forward, reading B: log-linear Mamba-2 applied
 * to the delta rule's pseudo-values,
 *   O = (Q K^T . M^S . M^H) U,  U = (I + diag(beta) SL(K K^T . M^S))^{-1} diag(beta) V,
 * i.e. u_t = beta_t (v_t - alpha_t S_{t-1} k_t) with S the single
 * gated-delta state.  The pages combine Gated DeltaNet with the hierarchical
 * mask (study note §3-5; gist.science (de) Technische Zusammenfassung §2)
 * without fixing where the mask acts; ll_gdn_fwd is reading A, this entry
 * point the other plain reading.  Arguments, layouts, errors: as ll_gdn_fwd.
 * Computed as a chunk-wise pass for U (float32) followed by ll_attn_fwd on
 * (q, k, U) in the io dtype, so U is rounded to bf16 for bf16 io.
 * Returns LL_ERR_UNSUPPORTED unless dk = dv = 128 and chunk >= 64. */
LL_API ll_status ll_gdn_fwd_b(const ll_shape* shape, const void* q, const void* k, const void* v,
                              const float* log_alpha, const float* beta, const float* lam, void* o,
                              void* workspace, size_t ws_bytes, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* LL_ATTN_H */
