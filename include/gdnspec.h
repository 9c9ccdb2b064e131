/*
 * gdnspec: target-side verify and commit of one GatedDeltaNet (GDN)
 * linear-attention layer for MTP speculative decoding, on NVIDIA GB300
 * (sm_103a).  C ABI; every buffer belongs to the caller.
 *
 * The operation.  A verify step scores, per request, the k+1 rows
 * [pending, d1..dk] in one pass [FreeToken #844 "MTP drafts for Qwen3.5
 * family + Flash-Next", Design; FreeToken #828 "Speculative decoding: MTP and
 * DFlash", Design: every request extends by the same k+1 rows].  Each row
 * runs one GDN decode step:
 *   window_t[c] = last W entries of [conv_state[c][0..W-2], x_0[c] .. x_t[c]]
 *   y_t[c]      = SiLU(sum_j conv_w[c][j] * window_t[c][j])   (tap W-1 = newest)
 *   q, k        = per q/k head  y / sqrt(sum y^2 + l2_eps),  v = v block of y
 *   per value head h, with q/k head h / (H_v / H_qk):
 *     S_t = exp(g_t) S_{t-1} + beta_t (v - exp(g_t) S_{t-1} k) k^T
 *     o_t = scale * S_t q
 * The GDN state is only read during the verify; the commit then makes each
 * request's slot hold the state after its accepted rows [FreeToken #828,
 * Design], with the conv window left where the accepted rows put it
 * [FreeToken #844, Flash-Next target verify].  accept_len = a counts accepted
 * drafts; the commit covers rows 0..a (a+1 tokens, the pages' "accept
 * length", FreeToken #844, End-to-end).  The verify may also snapshot every
 * row's state so the commit is a copy [LightLLM #1330 "Qwen3.5 / Qwen3.5-MoE
 * MTP speculative decoding", Summary: widened verify state, snapshot/restore];
 * or verify and commit run in one pass [lmdeploy #5006 "speculative decoding
 * for TurboMind", Verification path: verify-and-commit kernel mode].
 *
 * Layouts (row-major, C = 2*H_qk*d_k + H_v*d_v, channels [q heads|k heads|v heads]):
 *   x           [B][R][C]             in_dtype   pre-conv rows; row t < n_rows[b] valid
 *   g, beta     [B][R][H_v]           fp32       log-decay (exp(g) is the decay), write strength;
 *                                                with GDN_FLAG_RAW_GATING the raw projections
 *                                                a and b they are formed from (below)
 *   A_log       [H_v]                 fp32       GDN_FLAG_RAW_GATING only
 *   conv_w      [C][W]                in_dtype   depthwise taps, tap W-1 multiplies the newest row
 *   conv_state  [pool_slots][C][W-1]  in_dtype   committed window, oldest column first
 *   ssm_state   [pool_slots][H_v][d_v][d_k] fp32 committed state S (d_v x d_k per head)
 *   slot_ids, n_rows, accept_len [B]  int32      request -> slot; valid rows (0 = inactive);
 *                                                accepted drafts, 0..n_rows-1
 *   o           [B][R][H_v][d_v]      fp32       verify output; only rows t < n_rows[b] of
 *                                                active requests are written
 *   scratch_S   [B][R][H_v][d_v][d_k] fp32       snapshot mode: state after row t
 *   scratch_cs  [B][R][C][W-1]        in_dtype   snapshot mode: conv window after row t
 *   work        gdn_work_bytes(args) bytes       the call's own scratch: per row the
 *                                                normalised q and k of every q/k head, v,
 *                                                decay and write strength, and the rows'
 *                                                Gram tables; contents on entry do not matter
 *   status      [1]                   int32      device word; error bits are OR-ed in, never cleared
 *
 * Supported: W = 4; d_k in {16, 32, 64, 128}; d_v a multiple of 16 (d_k = 16)
 * or of 32 (d_k >= 32); H_v a multiple of H_qk; 1 <= R <= 16.
 *
 * Ownership, synchronisation.  All pointers are device pointers owned by the
 * caller; the library keeps none after a call returns, allocates nothing,
 * and never synchronises the stream.  Calls are asynchronous on `stream`
 * (a cudaStream_t; NULL = the legacy default stream).  Active requests must
 * use distinct slots (otherwise their results are undefined; the library's
 * debug/test build checks this and sets GDN_STATUS_DUPLICATE_SLOT, the
 * regular build spends nothing on it); two calls that touch the same slots or the same work
 * buffer must not run concurrently.  Each call is two kernel launches (a
 * prologue and the rows) chained with programmatic dependent launch; the
 * prologue waits for whatever ran before it on the stream.  The rows kernel
 * lets the next kernel on the stream launch early, as each of its CTAs starts
 * its last item: a following kernel launched with programmatic stream
 * serialization must wait (griddepcontrol.wait, cudaGridDependencySynchronize)
 * before it reads this call's outputs, as any such dependent must; kernels
 * launched without that attribute start after this call has finished.  In
 * replay mode the verify and the commit must see the same x, g, beta, conv_w
 * and slot contents.
 *
 * Errors.  Host return codes: GDN_OK, or GDN_ERR_* for arguments the host
 * can check (null pointers, shapes, alignment; nothing is launched) and for a
 * failed launch.  Values only the device sees are not trapped: a request whose
 * slot is outside [0, pool_slots) or whose n_rows is outside [0, R] is skipped
 * entirely (nothing written for it) and sets GDN_STATUS_BAD_SLOT /
 * GDN_STATUS_BAD_NROWS in *status; an accept_len outside [0, n_rows-1]
 * skips that request's commit (its o is still written) and sets
 * GDN_STATUS_BAD_ACCEPT.  A kernel never spins without bound: if one of its
 * staging copies does not land within a bounded wait, the blocks that depend
 * on it write nothing and GDN_STATUS_TIMEOUT is set.  status may be NULL (no
 * bits recorded).
 */
#ifndef GDNSPEC_H
#define GDNSPEC_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define GDN_API __attribute__((visibility("default")))


enum {
  GDN_OK = 0,
  GDN_ERR_INVALID_ARG = 1, /* null pointer, negative or inconsistent size  */
  GDN_ERR_UNSUPPORTED = 2, /* W, d_k, d_v, R or dtype outside the set above */
  GDN_ERR_MISALIGNED = 3,  /* a pointer below its required alignment        */
  GDN_ERR_LAUNCH = 4,      /* the CUDA launch failed                        */
  GDN_ERR_TOO_LARGE = 5    /* the call needs more scratch than the fixed
                              array of gdn_verify_commit_static holds       */
};

enum {
  GDN_STATUS_BAD_SLOT = 1,   /* slot outside [0, pool_slots): request skipped         */
  GDN_STATUS_BAD_NROWS = 2,  /* n_rows outside [0, R]: request skipped                */
  GDN_STATUS_BAD_ACCEPT = 4, /* accept_len outside [0, n_rows-1]: commit skipped      */
  GDN_STATUS_TIMEOUT = 8,    /* a staging copy did not complete within the kernel's
                                bounded wait: that block wrote nothing                */
  GDN_STATUS_DUPLICATE_SLOT = 16 /* debug/test builds only: two active requests name
                                the same slot (their results are undefined)           */
};
enum { GDN_DTYPE_BF16 = 0, GDN_DTYPE_F32 = 1 };
/* flags: GDN_FLAG_RAW_GATING - g and beta hold a layer's raw gating
 * projections a and b, and the prologue forms, per row and value head h,
 *   g = -exp(A_log[h]) * softplus(a),   beta = sigmoid(b)
 * (the standard gating of a Qwen3.5-style GDN layer; the pages feed the
 * recurrence these per-head scalars without printing how they are formed). */
/* GDN_FLAG_STATE_STABLE - a promise by the caller that no kernel that may
 * still be running on `stream` when this call is made writes this call's
 * ssm_state or conv_state slots, slot_ids or n_rows (for gdn_verify_deferred:
 * nor prev->n_rows).  With it the call starts fetching its state slices while
 * the kernels ahead of it on the stream are still draining, instead of after
 * they have finished: in a model, while the projection that writes x, g and
 * beta still runs; in a stack of layers, while the previous layer's call
 * finishes.  Everything else the call reads (x, g, beta, conv_w, A_log,
 * accept_len, the previous call's carry) is still read only after the kernels
 * ahead of it have finished, so accept_len may come from gdn_greedy_accept
 * launched just before.  Without the promise (flag clear) nothing is read
 * before those kernels finish.  The results are the same bits either way.
 * Two calls in a row on the same slots (the same layer's consecutive decode
 * steps with nothing in between) must not set it on the second call. */
enum { GDN_FLAG_RAW_GATING = 1, GDN_FLAG_STATE_STABLE = 2 };
enum { GDN_REPLAY = 0, GDN_SNAPSHOT = 1 };

typedef struct gdn_args {
  int32_t B;          /* requests (0 = nothing to do)                          */
  int32_t R;          /* rows per request in x/g/beta/o (k_max + 1)            */
  int32_t H_qk;       /* q/k heads                                             */
  int32_t H_v;        /* value heads                                           */
  int32_t d_k;        /* q/k head dim = state columns                          */
  int32_t d_v;        /* v head dim = state rows                               */
  int32_t W;          /* conv width, must be 4                                 */
  int32_t pool_slots; /* slots in conv_state / ssm_state                       */
  int32_t in_dtype;   /* GDN_DTYPE_* of x, conv_w, conv_state, scratch_cs      */
  float scale;        /* o = scale * S q (usually d_k^-1/2), finite            */
  float l2_eps;       /* >= 0, added to sum y^2 before the square root         */
  int32_t flags;      /* 0, or GDN_FLAG_RAW_GATING | GDN_FLAG_STATE_STABLE     */
  const void* x;      /* 16-byte aligned: x, conv_w, conv_state, ssm_state, o,  */
  const float* g;     /* scratch_S, scratch_cs; 4-byte: g, beta, int32 arrays   */
  const float* beta;
  const void* conv_w;
  void* conv_state;
  float* ssm_state;
  const int32_t* slot_ids;
  const int32_t* n_rows;
  const int32_t* accept_len; /* commit and fused calls only                    */
  float* o;                  /* verify and fused calls only                    */
  float* scratch_S;          /* snapshot mode only                             */
  void* scratch_cs;          /* snapshot mode only                             */
  void* work;                /* verify, replay commit and fused calls          */
  int32_t* status;           /* may be NULL                                    */
  const float* A_log;        /* GDN_FLAG_RAW_GATING only (4-byte aligned)      */
  void* carry;               /* gdn_verify_deferred only: this call's carry out
                                (gdn_carry_bytes bytes, 16-byte aligned)       */
} gdn_args;

/* Verify: for every active request, run rows 0..n_rows-1 from its slot's
 * committed state and write o.  Never writes conv_state or ssm_state.
 * mode GDN_SNAPSHOT also writes, per row t, the state and conv window a
 * commit at accept_len = t would leave into scratch_S / scratch_cs[b][t]
 * (the widened verify state).  Needs: x, g, beta, conv_w, conv_state,
 * ssm_state, slot_ids, n_rows, work, o (+ scratch_S, scratch_cs in snapshot
 * mode). */
GDN_API int gdn_verify(const gdn_args* args, int mode, void* stream);

/* Commit: make slot slot_ids[b] hold the state and conv window after rows
 * 0..accept_len[b] of request b.  mode GDN_REPLAY reruns those rows from the
 * committed state (same arithmetic as the verify, so the result equals a
 * fused call bit for bit) and needs the verify's inputs plus accept_len;
 * mode GDN_SNAPSHOT copies row accept_len[b] of a snapshot verify's
 * scratch and needs slot_ids, n_rows, accept_len, scratch_S, scratch_cs. */
GDN_API int gdn_commit(const gdn_args* args, int mode, void* stream);

/* Verify and commit in one pass over the state: writes o for every valid
 * row and, at row accept_len[b], the slot.  Each state byte is read once and
 * written once.  Needs everything gdn_verify needs plus accept_len. */
GDN_API int gdn_verify_commit(const gdn_args* args, void* stream);

/* Fused verify + commit that allocates nothing and takes no work buffer
 * (args->work is ignored and may be NULL).  For callers that cannot hand the
 * library device memory of their own: code that runs while a CUDA graph is
 * being captured (cudaMalloc is not a capturable operation), engines that
 * size every device buffer once at start-up and forbid allocation on the
 * decode path, and C hosts with no device allocator.  The call's scratch
 * lives instead in one file-scope device array of GDN_STATIC_WORK_BYTES,
 * which every GPU that loads this library holds until the process exits.
 * The first call on a device looks up that array's device address (with the
 * device current); make that first call before any stream capture starts.
 * Calls whose scratch (gdn_work_bytes) exceeds the array return
 * GDN_ERR_TOO_LARGE without launching.  All calls on a device share the one
 * array, so calls that overlap on the GPU (different streams, or different
 * host threads without ordering) race on it; the array's contents carry over
 * from call to call and nothing in it needs to start at zero.  Results equal
 * gdn_verify_commit's.  The pages have no counterpart: this entry point is a
 * property of this library's interface, not of the method. */
#define GDN_STATIC_WORK_BYTES ((size_t)32 << 20)
GDN_API int gdn_verify_commit_static(const gdn_args* args, void* stream);

/* Bytes of `work` a verify, replay commit or fused call with these shapes
 * needs: 4 * (B * R * (2 * H_qk * d_k + H_v * d_v + 4 * H_v) + B * H_qk * G2), with
 * G2 = 2 * R * R rounded up to a multiple of 4.  Reads only the
 * size fields of args; 0 if they are invalid or unsupported. */
GDN_API size_t gdn_work_bytes(const gdn_args* args);

/* Static description of a return code (never NULL). */
GDN_API const char* gdn_strerror(int code);

/* ---- deferred commit ------------------------------------------------------
 * Step s's verify also commits step s-1, so each step makes one pass over the
 * state: the slot keeps the state from before step s-1 until step s's call,
 * which first commits the previous call's rows 0..accept_len (their accept
 * count carried over from step s-1 [LightLLM #1330, Summary: the accept-count
 * carry; lmdeploy #5006, Verification path: verify-and-commit mode and draft
 * carry]) and then runs the current rows from there, writing their o.  The
 * pages carry the count to the next step without printing where the state
 * commit happens; folding it into the next verify is this library's form of it.
 *
 * The commit needs no replay: each deferred call leaves, in its carry buffer
 * (cur->carry, gdn_carry_bytes(cur) bytes, contents private to the library),
 * what committing any prefix of its rows takes: per row, the rank-one update
 * of every state row (u_t in S_t = exp(g_t) S_{t-1} + u_t k_t^T), k_t and the
 * decay.  The next call reads that carry as prev->carry and forms
 * S_a = (prod alpha) S + sum_{t<=a} (u_t prod_{j>t} alpha_j) k_t^T.
 *
 * prev describes the pending rows, with prev->R rows per request:
 *   x           [B][R][C]     in_dtype  the previous call's pre-conv rows (16-byte
 *                                       aligned); rows 0..accept_len advance the conv window
 *   n_rows      [B]           int32     its valid rows; 0 = nothing pending for request b
 *   accept_len  [B]           int32     its accepted drafts, 0..n_rows-1 when n_rows > 0
 *   carry                               the previous deferred call's cur->carry, unchanged
 * prev->carry and cur->carry must not overlap, nor prev->x and cur->x: a step
 * reads the previous step's carry and rows while it writes its own, so both
 * are double-buffered across steps (overlapping ranges return
 * GDN_ERR_INVALID_ARG before anything is launched).
 * prev may be NULL (nothing pending for any request: the first step).  The
 * result equals gdn_commit (replay) of the previous step followed by
 * gdn_verify of the current one.  prev->R <= 16, like every R.  Only the
 * last three of the pending rows 0..accept_len are read from prev->x (the
 * conv window they leave).  A pending accept_len outside [0, n_rows-1]
 * or an n_rows outside [0, R] skips the request and sets the matching status
 * bit.  Carry rows of a request that a call skipped (a status bit) are
 * undefined; cur->accept_len is not read.  Needs cur's verify inputs (x, g,
 * beta, conv_w, conv_state, ssm_state, slot_ids, n_rows, o), a work buffer of
 * gdn_work_bytes(cur) bytes and cur->carry. */
typedef struct gdn_prev_rows {
  int32_t R;                 /* rows per request of the previous call, >= 1 */
  const void* x;
  const int32_t* n_rows;
  const int32_t* accept_len;
  const void* carry;
} gdn_prev_rows;
GDN_API int gdn_verify_deferred(const gdn_args* cur, const gdn_prev_rows* prev, void* stream);

/* Bytes of carry a deferred call with these shapes writes:
 * 4 * (B * R * (H_v * d_v + H_qk * d_k) + B * H_v * R4), R4 = R rounded up to
 * a multiple of 4.  0 if the shapes are invalid or unsupported. */
GDN_API size_t gdn_carry_bytes(const gdn_args* args);

/* ---- greedy acceptance of drafts on the device --------------------------
 * The commit's accept_len decided on the device, so it feeds gdn_commit /
 * gdn_verify_commit with no device-to-host copy [LightLLM #1330, Summary:
 * the accept length stays on the device; FreeToken #828, Design: the
 * target's choices decide how many drafts are kept].
 *
 * For every request b with 0 < n_rows[b] <= R and every verify row
 * t < n_rows[b]:  target[b][t] = the index of the largest logits[b][t][:]
 * (the lowest index among equal largest values; NaN entries never win, and a
 * row whose entries are all NaN gives 0).
 * Then accept_len[b] = the largest a <= n_rows[b]-1 with drafts[b][i] ==
 * target[b][i] for all i < a: draft i+1 is the token at verify row i+1 and
 * is kept when the target chose it at row i.  target[b][a] is the target's
 * token after the accepted drafts.
 *
 *   logits      [B][R][V]  in_dtype (bf16 or fp32), 16-byte aligned, V % 8 == 0
 *   drafts      [B][R-1]   int32, draft i+1 of request b at [b][i] (may be NULL when R == 1)
 *   n_rows      [B]        int32, valid rows (0 = inactive)
 *   target      [B][R]     int32 out; rows t >= n_rows[b] are not written
 *   accept_len  [B]        int32 out; 0 for inactive requests and for a bad n_rows
 *   status      [1]        int32, may be NULL; GDN_STATUS_BAD_NROWS for n_rows outside [0, R]
 *
 * Two kernels on `stream` (a cluster of 8 CTAs per verify row, then one
 * thread per request), chained by programmatic dependent launch; the first
 * waits for the kernel before it on the stream, and the second lets the next
 * kernel launch early (a following kernel launched with programmatic stream
 * serialization must wait before it reads target or accept_len, as the
 * calls of this library do).  Allocates nothing and does not synchronise.  Returns GDN_ERR_INVALID_ARG,
 * GDN_ERR_UNSUPPORTED (V % 8 != 0, B or R > 65535, dtype),
 * GDN_ERR_MISALIGNED or GDN_ERR_LAUNCH before launching anything. */
typedef struct gdn_accept_args {
  int32_t B, R, V;
  int32_t in_dtype; /* GDN_DTYPE_BF16 or GDN_DTYPE_F32 */
  const void* logits;
  const int32_t* drafts;
  const int32_t* n_rows;
  int32_t* target;
  int32_t* accept_len;
  int32_t* status;
} gdn_accept_args;
GDN_API int gdn_greedy_accept(const gdn_accept_args* args, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* GDNSPEC_H */
