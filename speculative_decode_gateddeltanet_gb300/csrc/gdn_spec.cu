// GatedDeltaNet speculative verify / commit kernels for sm_103a.
//
// Every call is two kernels on the caller's stream, chained by programmatic
// dependent launch so the second one's state loads overlap the first:
//
// prep_kernel (one block per (request, q/k head) and per 256 VV value
//   channels): the width-4 causal conv + SiLU of every row over [committed
//   window | verify rows], then the per-head L2 norm of q and k.  Writes
//   scale*q^, k^, v, the decay and write strength per row, and the rows'
//   Gram tables k^.k^ and k^.(scale q^) into the caller's work buffer.  Each
//   conv channel has exactly one reader in the call, so that thread also
//   writes the channel's committed window (commit modes) or its per-row
//   windows (snapshot mode).  The conv reads only the committed window and
//   the verify rows, staging [history | verify inputs] per channel [FreeToken
//   #844 "MTP drafts for Qwen3.5 family + Flash-Next", Design / Flash-Next
//   target verify].  Before its dependency wait it only issues L2 hints for
//   its own inputs and reads the request's slot as a guess for its window.
//
// rows_kernel (persistent; item = (request, value head, slice of DVS state
//   rows), DVS = 32, 16 at d_k = 16, or 64 in the four-warp geometry chosen
//   for long requests): the slice of the fp32 state S (DVS x d_k, d_k contiguous) arrives
//   by one bulk async copy, issued for the first item before the kernel waits
//   on the prologue, and moves to registers; the item's q, k, v and tables
//   are staged from the work buffer by bulk async copies.  It runs the gated
//   delta rule S_t = alpha S + beta (v - alpha S k) k^T, o_t = scale S_t q
//   with S resident in registers, in the chunked form described at the kernel
//   (all dot products of a chunk of rows on the chunk's starting state, a
//   scalar recurrence per state row, one state update).  Lanes own 4-float
//   column chunks of 2 or 4 rows; a row's dot products are reduced over its
//   8 (d_k >= 32) or 4 (d_k = 16) lanes with a butterfly that leaves each lane
//   holding one row's sums.  Arithmetic is fp32 with packed f32x2 FMA/MUL.
//
// The arithmetic of a row does not depend on the mode, so a fused call, a
// verify followed by a replay commit and a snapshot verify followed by a
// snapshot commit give the same bits.
//
// Modes: verify (o only; the state is only read [FreeToken #828
// "Speculative decoding: MTP and DFlash", Design]), verify with per-row
// snapshots (the widened verify state of [LightLLM #1330 "Qwen3.5 /
// Qwen3.5-MoE MTP speculative decoding", Summary]), replay commit (rows
// 0..a rerun from the slot, then written once), fused verify + commit (the
// slot is written at row a from the registers: one read and one write of the
// state per request, the verify-and-commit kernel mode of [lmdeploy #5006
// "speculative decoding for TurboMind", Verification path]), and deferred
// (the previous call's accepted rows committed from its carry, then this
// call's rows verified; the accept-count carry of [LightLLM #1330, Summary]).
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <cmath>
#include <mutex>

#include "gdnspec.h"

namespace gdnspec {

constexpr int kW = 4;             // conv width the kernels are built for
constexpr int kWS = kW - 1;       // conv-state columns
constexpr int kMaxR = 16;         // rows per request (k <= 15)
constexpr int kPrepThreads = 256; // channels per prologue block (>= 2 * max d_k)
// value channels per prologue thread, loaded as one chunk per row: four when
// a request has at most 4 rows, else two (four would cost more resident
// blocks in registers than the wider loads gain)
template <int RMAX>
__host__ __device__ constexpr int vec_v() { return RMAX <= 4 ? 4 : 2; }
constexpr unsigned kFull = 0xffffffffu;

// kDeferred: the previous call's accepted rows are committed from its carry
// (per row: the state rows' update vectors, k^ and the decay), then the
// current rows are verified from that state (o, and their own carry).
enum Mode : int { kFused = 0, kVerify = 1, kVerifySnap = 2, kCommitReplay = 3, kDeferred = 4 };

// Division of 0 <= n < 2^31 by a divisor d >= 1 fixed for the launch, as
// floor(n m / 2^k) with k = 31 + ceil(log2 d) and m = ceil(2^k / d).  With
// m d = 2^k + e (0 <= e < d) and n = q d + r, n m / 2^k = q + (r + n e / 2^k) / d,
// and n e < 2^31 2^ceil(log2 d) = 2^k makes the fraction below 1.  The product
// is below 2^64 (m < 2^33), so one wide multiply and a shift replace the
// integer division's reciprocal sequence.
struct FastDiv {
  unsigned long long m;
  int k;
};
inline FastDiv make_fastdiv(int d) {
  int c = 0;
  while ((1LL << c) < d) ++c;
  const int k = 31 + c;
  const unsigned long long two_k = 1ULL << k;
  return FastDiv{two_k / (unsigned long long)d + (two_k % (unsigned long long)d != 0), k};
}
__device__ __forceinline__ int fdiv(int n, const FastDiv& f) {
  return (int)(((unsigned long long)(unsigned)n * f.m) >> f.k);
}

struct Params {
  int B, R, H_qk, H_v, d_k, d_v, P, G, slices;
  // item it = ((b H_v) + h) slices + sl: divisions by H_v slices, slices and G
  FastDiv div_hs, div_sl, div_g;
  long long C;
  float scale, eps;
  const void* x;
  const float* g;
  const float* beta;
  const void* conv_w;
  void* conv_state;
  float* S;
  const int* slot_ids;
  const int* n_rows;
  const int* accept_len;
  float* o;
  float* snapS;
  void* snapCs;
  int dvs;     // state rows per rows-kernel item
  float* wqk;  // work: [B][H_qk][R][2 d_k]         scale*q^ | k^
  float* wv;   // work: [B][H_v d_v / dvs][R][dvs]  v
  float* wsc;  // work: [B][H_v][R][4]              exp(g), beta, 0, 0
  float* wgh;  // work: [B][H_qk][gram_floats(R)]   [R][R][2]: k^_s . k^_t, k^_s . (scale q^_t)
  int* status;
  const float* A_log;  // GDN_FLAG_RAW_GATING: g and beta hold the raw projections a and b
  int raw_gating;
  // GDN_FLAG_STATE_STABLE: nothing still running on the stream writes this call's
  // slots, slot_ids or n_rows, so the rows kernel may fetch state slices before
  // the kernels ahead of it have finished
  int early;
  // Deferred commit.  Request b's block of conv rows is the previous call's
  // rows 0..acc_prev[b] (when n_prev[b] > 0; they only advance the window)
  // then its current rows.  The state rows run the current rows only, after
  // committing the previous rows from the previous call's carry.
  const void* xp;       // [B][Rp][C] the previous call's x
  const int* n_prev;    // [B] its valid rows, 0 = nothing pending (NULL: none pending)
  const int* acc_prev;  // [B] its accepted drafts
  const float* pcu;     // carry in:  [B][H_v d_v / dvs][Rp][dvs]  u, the state rows' update vectors
  const float* pck;     //            [B][H_qk][Rp][d_k]           k^
  const float* pca;     //            [B][H_v][Rp4]                exp(g)
  float* cu;            // carry out: the same for this call's rows (R, R4)
  float* ck;
  float* ca;
  int Rp;               // rows per request of the previous call (0: none)
};

__host__ __device__ constexpr int round4(int r) { return (r + 3) & ~3; }

// Lane geometry of the rows kernel for a d_k-column state.  WIDE (d_k = 128
// only): four warps and 64 state rows per item instead of two warps and 32,
// so an item's fixed costs (its waits, its copies, the producers' request
// bookkeeping, the staged q/k rows and tables) are shared by twice the rows.
template <int DK, bool WIDE = false>
struct Geo {
  static_assert(!WIDE || DK == 128, "the wide geometry is for d_k = 128");
  static constexpr int LPR = DK >= 32 ? 8 : 4;   // lanes per state row
  static constexpr int NC4 = DK / (4 * LPR);     // 4-column chunks per lane per row
  static constexpr int RG = 32 / LPR;            // row groups per warp
  static constexpr int M = DK >= 64 ? 4 : 2;     // rows per lane
  static constexpr int ROWS_W = RG * M;          // rows per warp
  static constexpr int NW = DK == 16 ? 1 : (WIDE || M == 2 ? 4 : 2);  // warps per CTA
  static constexpr int DVS = NW * ROWS_W;        // state rows per CTA (32; 16 at d_k = 16; 64 wide)
  static constexpr int NT = NW * 32;
  // resident CTAs per SM the registers must allow
  static constexpr int MIN_CTAS = NT == 64 ? 8 : (NT == 128 ? (WIDE ? 4 : 5) : 16);
};

__host__ __device__ constexpr int ilog2(int v) { return v <= 1 ? 0 : 1 + ilog2(v / 2); }
// Floats of one (request, q/k head) Gram table [R][R][2], padded to 16 bytes so
// every table starts and ends on a bulk-copy boundary.
__host__ __device__ constexpr int gram_floats(int R) { return (2 * R * R + 3) & ~3; }

// ---- packed fp32 pairs (f32x2) ----
typedef unsigned long long f2;
__device__ __forceinline__ f2 pack2(float lo, float hi) {
  f2 r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ float sum2(f2 v) {
  float lo, hi;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
  return __fadd_rn(lo, hi);
}
__device__ __forceinline__ f2 fma2(f2 a, f2 b, f2 c) {
  f2 d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ f2 mul2(f2 a, f2 b) {
  f2 d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

template <typename T>
__device__ __forceinline__ float tof(T v);
template <>
__device__ __forceinline__ float tof<float>(float v) { return v; }
template <>
__device__ __forceinline__ float tof<__nv_bfloat16>(__nv_bfloat16 v) { return __bfloat162float(v); }

// SiLU with the fast exponential and division (a few ulp; the conv output feeds
// a normalisation and a dot product, far below the path's tolerance).
// N consecutive elements of T as one aligned load or store
template <typename T, int N>
struct ChunkOf {
  using type = T;
};
template <>
struct ChunkOf<float, 4> {
  using type = float4;
};
template <>
struct ChunkOf<__nv_bfloat16, 4> {
  using type = uint2;
};
template <>
struct ChunkOf<float, 2> {
  using type = float2;
};
template <>
struct ChunkOf<__nv_bfloat16, 2> {
  using type = uint32_t;
};
__device__ __forceinline__ float silu(float z) { return __fdividef(z, __fadd_rn(1.0f, __expf(-z))); }

__device__ __forceinline__ void flag(int* status, int bit) {
  if (status) atomicOr(status, bit);
}

// ---- programmatic dependent launch ----
// wait: the grid this one depends on has completed and its writes are visible.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// trigger: the grid launched after this one may start once every CTA of this
// grid has triggered or exited.
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// A relaxed GPU-scope load: well defined even while another grid may be
// writing the word, so its value can only serve as a guess that is checked
// against a plain load after the dependency wait.
__device__ __forceinline__ int ld_relaxed(const int* ptr) {
  int v;
  asm volatile("ld.relaxed.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(ptr) : "memory");
  return v;
}

// ---- bulk async copies (TMA, 1-D) into shared memory, tracked by an mbarrier ----
__device__ __forceinline__ uint32_t smem_addr(const void* ptr) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(ptr));
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
               : "memory");
}
// Orders this CTA's earlier generic-proxy shared-memory accesses before later
// bulk async copies (the async proxy) into the same memory.
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}
// Asks L2 to fetch [src, src + bytes) ahead of use; a hint that moves no data
// into the CTA and orders nothing.  src and bytes are multiples of 16.
__device__ __forceinline__ void prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}
// How long a staging wait may last before the kernel gives up on it (ns of
// %globaltimer).  A copy lands in microseconds; the limit only has to catch a
// barrier whose bytes will never all arrive.
#ifndef GDN_WAIT_LIMIT_NS
#define GDN_WAIT_LIMIT_NS 500000000ull
#endif
__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
// Waits for phase `parity` of the barrier; gives up and returns false once
// GDN_WAIT_LIMIT_NS have passed (the clock is read every 256 polls; 2^24 polls
// end the wait whatever the clock says).
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  uint64_t t0 = 0;
  for (uint32_t i = 1; i < (1u << 24); ++i) {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    if (done) return true;
    if ((i & 255) == 0) {
      const uint64_t now = global_ns();
      if (t0 == 0)
        t0 = now;
      else if (now - t0 > GDN_WAIT_LIMIT_NS)
        return false;
    }
  }
  return false;
}

#ifdef GDN_TEST_HOOKS
// Test builds only: the rows-kernel item whose state copy the producer
// declares on its barrier but never issues, so that item's wait runs out with
// no copy in flight (-1: none).  Set by gdn_test_drop_state_copy.
__device__ int g_test_drop_item = -1;
// Test builds only: prologue blocks whose slot read before the wait differed
// from the request's slot (so they loaded the window again).
__device__ unsigned int g_test_guess_misses = 0;
__device__ __forceinline__ void count_guess_miss() {
  if (threadIdx.x == 0) atomicAdd(&g_test_guess_misses, 1u);
}
// Test builds only: a kernel ahead of a call that lets the call's grids
// launch at once and only then, after delay_ns of %globaltimer (at most 2^22
// polls), copies src[0..n) to dst: it rewrites the call's request data after
// releasing it, as a producer of slot_ids may.
__global__ void test_late_write_kernel(int* dst, const int* src, int n, unsigned long long delay_ns) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  unsigned long long t0, t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
  for (int i = 0; i < (1 << 22); ++i) {
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    if (t - t0 >= delay_ns) break;
  }
  for (int i = threadIdx.x; i < n; i += blockDim.x) dst[i] = src[i];
}
#else
__device__ __forceinline__ void count_guess_miss() {}
#endif

// Validity of a request as every kernel reads it, from its n_rows n, slot and
// accept length a.  Returns the number of rows to run (0 = nothing to do for
// this request); crow receives the commit row (-1: none) and `report` a status
// bit for a bad request (the caller decides who records it).
template <bool kCommits, bool kReplay>
__device__ __forceinline__ int request_rows_of(const Params& p, int n, int slot, int a, int& crow, int& report) {
  report = 0;
  crow = -1;
  if (n == 0) return 0;
  if (slot < 0 || slot >= p.P) {
    report = GDN_STATUS_BAD_SLOT;
    return 0;
  }
  if (n < 0 || n > p.R) {
    report = GDN_STATUS_BAD_NROWS;
    return 0;
  }
  if (kCommits) {
    if (a >= 0 && a < n) {
      crow = a;
    } else {
      report = GDN_STATUS_BAD_ACCEPT;
      if (kReplay) return 0;
    }
  }
  return kReplay ? a + 1 : n;
}
// Deferred commit: from the current n_rows n, the slot and the previous
// call's n_prev np and accepted drafts ap.  The block of conv rows is ap + 1
// previous rows (off, 0 when nothing is pending) and then the n current rows;
// the slot is committed after previous row ap.  A bad ap skips the request.
__device__ __forceinline__ int deferred_rows_of(const Params& p, int n, int slot, int np, int ap, int& off,
                                                int& crow, int& report) {
  report = 0;
  crow = -1;
  off = 0;
  if (n == 0 && np == 0) return 0;
  if (slot < 0 || slot >= p.P) {
    report = GDN_STATUS_BAD_SLOT;
    return 0;
  }
  if (n < 0 || n > p.R || np < 0 || np > p.Rp) {
    report = GDN_STATUS_BAD_NROWS;
    return 0;
  }
  if (np > 0) {
    if (ap < 0 || ap >= np) {
      report = GDN_STATUS_BAD_ACCEPT;
      return 0;
    }
    off = ap + 1;
    crow = ap;
  }
  return off + n;
}
// Request b's block of rows as every kernel of a call in mode MODE reads it:
// rows to run; slot; crow = commit row (-1 none); off = leading rows that
// are the previous call's (deferred mode; else 0); report = status bit.
template <int MODE>
__device__ __forceinline__ int request_block(const Params& p, int b, int& slot, int& crow, int& off, int& report) {
  slot = p.slot_ids[b];
  off = 0;
  if constexpr (MODE == kDeferred) {
    const int np = p.n_prev ? p.n_prev[b] : 0;
    const int ap = p.n_prev ? p.acc_prev[b] : -1;
    return deferred_rows_of(p, p.n_rows[b], slot, np, ap, off, crow, report);
  } else {
    constexpr bool kCommits = MODE == kFused || MODE == kCommitReplay;
    const int a = kCommits ? p.accept_len[b] : -1;
    return request_rows_of<kCommits, MODE == kCommitReplay>(p, p.n_rows[b], slot, a, crow, report);
  }
}

// ------------------------------------------------------------ prologue
// grid (H_qk + ceil(H_v d_v / (256 VV)), B): block x < H_qk holds the 2 d_k q
// and k channels of q/k head x (one per thread), the other blocks 256 VV v
// channels each (VV consecutive channels per thread).  Work layout:
//   wqk [B][H_qk][R][2 d_k]   scale*q^ | k^       (one contiguous run per (b, q/k head))
//   wv  [B][H_v d_v/DVS][R][DVS]  v               (one run per (b, head, row slice))
//   wsc [B][H_v][R][4]        exp(g), beta, k^.(scale q^), 0   (one run per (b, head))
template <typename T, int MODE, int RMAX>
__global__ void __launch_bounds__(kPrepThreads) prep_kernel(const Params p) {
  constexpr bool kCommits = MODE == kFused || MODE == kCommitReplay || MODE == kDeferred;
  constexpr bool kSnap = MODE == kVerifySnap;
  // Requests of at most 4 rows: the block's loads are issued right after the
  // wait, together with the request data, so they do not wait for a second
  // round trip: every row of x and gating the buffers hold, the taps and the
  // conv window of the request's slot as read before the wait (a guess, since
  // the kernels ahead may still be writing slot_ids; a block whose request
  // turns out to use another slot loads that slot's window again).  Longer
  // requests read the request first and load only its rows: measured, the
  // early loads' registers cost more blocks in flight than the round trip.
  constexpr bool kGuess = RMAX <= 4;
  const int slot_seen = ld_relaxed(p.slot_ids + blockIdx.y);
  // L2 hints for this block's own inputs (its channels of the current rows of
  // x, the slot's conv window and the taps), issued while the call waits for
  // the work before it so the loads after the wait find them in L2.  A hint
  // returns no data, so it may run before the wait: a slot id read early
  // warms at worst the wrong slot, never memory outside the buffers.
  {
    const int b = blockIdx.y;
    const bool qk = blockIdx.x < p.H_qk;
    const int nrng = qk ? 2 : 1;
    const long long vb = (long long)(blockIdx.x - p.H_qk) * kPrepThreads * vec_v<RMAX>();
    const long long c0 = qk ? (long long)blockIdx.x * p.d_k : 2LL * p.H_qk * p.d_k + vb;
    const long long c1 = qk ? (long long)(p.H_qk + blockIdx.x) * p.d_k : c0;
    const long long nch = qk ? p.d_k : min((long long)kPrepThreads * vec_v<RMAX>(), (long long)p.H_v * p.d_v - vb);
    const int nreq = nrng * (p.R + 2);  // per channel range: the rows of x, the window, the taps
    if (threadIdx.x < nreq) {
      const int r = threadIdx.x % nrng, j = threadIdx.x / nrng;
      const long long ch = r == 0 ? c0 : c1;
      const char* src = nullptr;
      size_t bytes = 0;
      if (j < p.R) {
        src = static_cast<const char*>(p.x) + (((size_t)b * p.R + j) * p.C + ch) * sizeof(T);
        bytes = nch * sizeof(T);
      } else if (j == p.R) {
        if (slot_seen >= 0 && slot_seen < p.P) {
          src = static_cast<const char*>(p.conv_state) + ((size_t)slot_seen * p.C + ch) * kWS * sizeof(T);
          bytes = nch * kWS * sizeof(T);
        }
      } else {
        src = static_cast<const char*>(p.conv_w) + ch * kW * sizeof(T);
        bytes = nch * kW * sizeof(T);
      }
      if (src != nullptr && bytes > 0 && ((reinterpret_cast<uintptr_t>(src) | bytes) & 15) == 0)
        prefetch_l2(src, (uint32_t)bytes);
    }
  }
  // The rows kernel may start loading its state once every block has passed
  // here: with the caller's promise that nothing still running writes the
  // state, before this block's wait; else after it.
  if (p.early) pdl_trigger();
  pdl_wait();  // whatever ran before on the stream is complete and visible
  if (!p.early) pdl_trigger();
#ifdef GDN_TEST_HOOKS
  // Debug/test builds: active requests must name distinct slots.  Block x = 0
  // of each request compares its slot with every other active request's.
  if (blockIdx.x == 0) {
    auto active_req = [&](int j) {
      const int nj = p.n_rows[j];
      return (nj > 0 && nj <= p.R) || (MODE == kDeferred && p.n_prev != nullptr && p.n_prev[j] > 0);
    };
    const int b0 = blockIdx.y, s0 = p.slot_ids[b0];
    bool dup = false;
    if (s0 >= 0 && s0 < p.P && active_req(b0))
      for (int j = threadIdx.x; j < p.B; j += blockDim.x)
        if (j != b0 && p.slot_ids[j] == s0 && active_req(j)) dup = true;
    if (__syncthreads_or(dup) && threadIdx.x == 0) flag(p.status, GDN_STATUS_DUPLICATE_SLOT);
  }
#endif
  __shared__ float sy[RMAX][kPrepThreads];  // q/k blocks: conv outputs, [row][q | k]

  const int b = blockIdx.y;
  const bool guess_ok = slot_seen >= 0 && slot_seen < p.P;
  // The request's block of rows (the rows kernel records bad requests).
  // Block rows t < off are the previous call's (deferred mode): they only
  // advance the conv window.  The current rows t >= off are outputs r = t - off.
  int slot, a, off, report;
  auto request = [&]() { return request_block<MODE>(p, b, slot, a, off, report); };
  int t_end = 0;
  if constexpr (!kGuess) {  // longer requests: read first, then only their rows loaded
    t_end = request();
    if (t_end == 0) return;
  }
  // gating of current row r for value head h
  auto load_gate = [&](int r, int h, float& gv, float& bv) {
    const size_t i = ((size_t)b * p.R + r) * p.H_v + h;
    gv = __ldg(p.g + i);
    bv = __ldg(p.beta + i);
  };

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int DK = p.d_k;
  const bool qk_block = blockIdx.x < p.H_qk;
  const int hq = blockIdx.x;

  if (!qk_block) {
    // value channels: VV consecutive channels per thread, loaded and stored
    // as one chunk per row; conv + SiLU only (no norm), written as v rows
    constexpr int VV = vec_v<RMAX>();
    using Chunk = typename ChunkOf<T, VV>::type;
    const int v0 = ((blockIdx.x - p.H_qk) * kPrepThreads + tid) * VV;
    if (v0 >= p.H_v * p.d_v) return;
    const long long cv = 2LL * p.H_qk * DK + v0;
    const Chunk* wg = reinterpret_cast<const Chunk*>(static_cast<const T*>(p.conv_w) + cv * kW);
    auto window = [&](int sl) {
      return reinterpret_cast<Chunk*>(static_cast<T*>(p.conv_state) + ((size_t)sl * p.C + cv) * kWS);
    };
    // every load first, so they are all in flight together
    Chunk xr[RMAX], xq[kWS], wc[kW], rc[kWS];
    auto load_x = [&](int t) {
      xr[t] = *reinterpret_cast<const Chunk*>(static_cast<const T*>(p.x) + ((size_t)b * p.R + t) * p.C + cv);
    };
    if constexpr (kGuess) {  // every row the buffer holds, the taps, the guessed window; then the request
#pragma unroll
      for (int t = 0; t < RMAX; ++t)
        if (t < p.R) load_x(t);
#pragma unroll
      for (int i = 0; i < kW; ++i) wc[i] = wg[i];
      if (guess_ok) {
        const Chunk* g0 = window(slot_seen);
#pragma unroll
        for (int i = 0; i < kWS; ++i) rc[i] = g0[i];
      }
      t_end = request();
      if (t_end == 0) return;
      if (slot != slot_seen) {  // the guess missed: the request's own window
        count_guess_miss();
        const Chunk* w0 = window(slot);
#pragma unroll
        for (int i = 0; i < kWS; ++i) rc[i] = w0[i];
      }
    } else {  // the request's rows, the taps, its window
#pragma unroll
      for (int t = 0; t < RMAX; ++t)
        if (t < t_end - off) load_x(t);
#pragma unroll
      for (int i = 0; i < kW; ++i) wc[i] = wg[i];
      const Chunk* w0 = window(slot);
#pragma unroll
      for (int i = 0; i < kWS; ++i) rc[i] = w0[i];
    }
    const bool commit = a >= 0;
    const int n = t_end - off;
    Chunk* cs = window(slot);
    // (deferred) the last kWS of the previous call's rows 0..off-1
    if (MODE == kDeferred) {
#pragma unroll
      for (int i = 0; i < kWS; ++i) {
        const int t = off - kWS + i;
        if (t >= 0)
          xq[i] = *reinterpret_cast<const Chunk*>(static_cast<const T*>(p.xp) + ((size_t)b * p.Rp + t) * p.C + cv);
      }
    }
    const T* we = reinterpret_cast<const T*>(wc);  // [channel][tap]
    T* re = reinterpret_cast<T*>(rc);               // [channel][window column], oldest first
    float w[VV][kW];
#pragma unroll
    for (int j = 0; j < VV; ++j)
#pragma unroll
      for (int i = 0; i < kW; ++i) w[j][i] = tof(we[j * kW + i]);
    if (MODE == kDeferred) {  // the window after the previous call's rows: the one the slot commits
#pragma unroll
      for (int i = 0; i < kWS; ++i) {
        if (off - kWS + i >= 0) {
          const T* xe = reinterpret_cast<const T*>(&xq[i]);
#pragma unroll
          for (int j = 0; j < VV; ++j) {
            T* r = re + j * kWS;
            r[0] = r[1];
            r[1] = r[2];
            r[2] = xe[j];
          }
        }
      }
    }
    Chunk cc[kWS];  // window after row a (deferred: after the previous rows)
#pragma unroll
    for (int i = 0; i < kWS; ++i) cc[i] = rc[i];
    float* vdst = p.wv + (((size_t)b * p.H_v * p.slices + v0 / p.dvs) * p.R) * p.dvs + (v0 % p.dvs);
#pragma unroll
    for (int t = 0; t < RMAX; ++t) {
      if (t < n) {
        const T* xe = reinterpret_cast<const T*>(&xr[t]);
        float y[VV];
#pragma unroll
        for (int j = 0; j < VV; ++j) {
          T* r = re + j * kWS;
          float z = __fmul_rn(w[j][0], tof(r[0]));
          z = __fmaf_rn(w[j][1], tof(r[1]), z);
          z = __fmaf_rn(w[j][2], tof(r[2]), z);
          z = __fmaf_rn(w[j][3], tof(xe[j]), z);
          y[j] = silu(z);
          r[0] = r[1];
          r[1] = r[2];
          r[2] = xe[j];
        }
        float* vd = vdst + (size_t)t * p.dvs;
        if constexpr (VV == 4)
          *reinterpret_cast<float4*>(vd) = make_float4(y[0], y[1], y[2], y[3]);
        else if constexpr (VV == 2)
          *reinterpret_cast<float2*>(vd) = make_float2(y[0], y[1]);
        else
          vd[0] = y[0];
        if (kSnap) {
          Chunk* sc = reinterpret_cast<Chunk*>(static_cast<T*>(p.snapCs) + (((size_t)b * p.R + t) * p.C + cv) * kWS);
#pragma unroll
          for (int i = 0; i < kWS; ++i) sc[i] = rc[i];
        }
        if (kCommits && MODE != kDeferred && t == a) {
#pragma unroll
          for (int i = 0; i < kWS; ++i) cc[i] = rc[i];
        }
      }
    }
    if (kCommits && commit) {  // this thread was these channels' only reader in the call
#pragma unroll
      for (int i = 0; i < kWS; ++i) cs[i] = cc[i];
    }
    return;
  }

  // q/k blocks: one channel per thread, q channels of head hq then its k channels
  const bool active = tid < 2 * DK;
  const long long ch =
      tid < DK ? (long long)hq * DK + tid : (long long)p.H_qk * DK + (long long)hq * DK + (tid - DK);

  // gating of the value heads that read this q/k head, (head, row) pair
  // i = (h - hq G) gr + t: loaded now, written at the end for the request's
  // rows.  gr = R when the loads come before the request is read, else n.
  float g_i = 0.f, beta_i = 0.f;
  // channel ch: every load first, so they are all in flight together (the
  // window oldest first, as stored)
  T xr[RMAX], q0, q1, q2, q3, r0, r1, r2;
  auto load_x = [&](int t) { xr[t] = static_cast<const T*>(p.x)[((size_t)b * p.R + t) * p.C + ch]; };
  auto load_taps = [&]() {
    const T* wg = static_cast<const T*>(p.conv_w) + ch * kW;
    q0 = wg[0];
    q1 = wg[1];
    q2 = wg[2];
    q3 = wg[3];
  };
  auto load_window = [&](int sl) {
    const T* w0 = static_cast<const T*>(p.conv_state) + ((size_t)sl * p.C + ch) * kWS;
    r0 = w0[0];
    r1 = w0[1];
    r2 = w0[2];
  };
  if constexpr (kGuess) {  // every row the buffers hold, the taps, the guessed window; then the request
    if (tid < p.G * p.R) load_gate(tid % p.R, hq * p.G + tid / p.R, g_i, beta_i);
    if (active) {
#pragma unroll
      for (int t = 0; t < RMAX; ++t)
        if (t < p.R) load_x(t);
      load_taps();
      if (guess_ok) load_window(slot_seen);
    }
    t_end = request();
    if (t_end == 0) return;
    if (slot != slot_seen) {  // the guess missed: the request's own window
      count_guess_miss();
      if (active) load_window(slot);
    }
  } else {  // the request's rows, the taps, its window
    const int n0 = t_end - off;
    if (tid < p.G * n0) load_gate(tid % n0, hq * p.G + tid / n0, g_i, beta_i);
    if (active) {
#pragma unroll
      for (int t = 0; t < RMAX; ++t)
        if (t < n0) load_x(t);
      load_taps();
      load_window(slot);
    }
  }
  const bool commit = a >= 0;
  const int n = t_end - off;
  const int gr = kGuess ? p.R : n;
  if (active) {
    T* cs = static_cast<T*>(p.conv_state) + ((size_t)slot * p.C + ch) * kWS;
    // (deferred) the last kWS of the previous call's rows 0..off-1
    T xq[kWS];
    if (MODE == kDeferred) {
#pragma unroll
      for (int i = 0; i < kWS; ++i) {
        const int t = off - kWS + i;
        if (t >= 0) xq[i] = static_cast<const T*>(p.xp)[((size_t)b * p.Rp + t) * p.C + ch];
      }
    }
    const float w0 = tof(q0), w1 = tof(q1), w2 = tof(q2), w3 = tof(q3);
    if (MODE == kDeferred) {  // the window after the previous call's rows: the one the slot commits
#pragma unroll
      for (int i = 0; i < kWS; ++i) {
        if (off - kWS + i >= 0) {
          r0 = r1;
          r1 = r2;
          r2 = xq[i];
        }
      }
    }
    T c0 = r0, c1 = r1, c2 = r2;  // window after row a (deferred: after the previous rows)
#pragma unroll
    for (int t = 0; t < RMAX; ++t) {
      if (t < n) {
        const T r3 = xr[t];
        float z = __fmul_rn(w0, tof(r0));
        z = __fmaf_rn(w1, tof(r1), z);
        z = __fmaf_rn(w2, tof(r2), z);
        z = __fmaf_rn(w3, tof(r3), z);
        sy[t][tid] = silu(z);
        r0 = r1;
        r1 = r2;
        r2 = r3;
        if (kSnap) {
          T* sc = static_cast<T*>(p.snapCs) + (((size_t)b * p.R + t) * p.C + ch) * kWS;
          sc[0] = r0;
          sc[1] = r1;
          sc[2] = r2;
        }
        if (kCommits && MODE != kDeferred && t == a) {
          c0 = r0;
          c1 = r1;
          c2 = r2;
        }
      }
    }
    if (kCommits && commit) {  // this thread was the channel's only reader in the call
      cs[0] = c0;
      cs[1] = c1;
      cs[2] = c2;
    }
  }
  if (n == 0) return;  // only the previous call's rows: the window was all there was to do
  __syncthreads();
  // Raw dot products of the rows' conv outputs, packed in n-row order: entries
  // e < n are q_t.q_t, then pairs (s, t) at n + 2 (s n + t) + {0: k_s.k_t,
  // 1: k_s.q_t}.  They give the L2 norms (diagonals) and, scaled, the Gram
  // tables.
  const int nd = n + 2 * n * n;
  __shared__ float sdot[RMAX + 2 * RMAX * RMAX];
  if constexpr (RMAX <= 4) {
    // few rows: thread c < d_k forms all products of its channel, summed by a
    // warp butterfly and then over the warps' partials in order
    constexpr int ND = RMAX + 2 * RMAX * RMAX;
    __shared__ float spart[kPrepThreads / 32][ND];
    float prod[ND];
#pragma unroll
    for (int e = 0; e < ND; ++e) prod[e] = 0.f;
    if (tid < DK) {
      float qv[RMAX], kv[RMAX];
#pragma unroll
      for (int t = 0; t < RMAX; ++t) {
        qv[t] = t < n ? sy[t][tid] : 0.f;
        kv[t] = t < n ? sy[t][DK + tid] : 0.f;
      }
#pragma unroll
      for (int t = 0; t < RMAX; ++t) prod[t] = __fmul_rn(qv[t], qv[t]);
#pragma unroll
      for (int s0 = 0; s0 < RMAX; ++s0)
#pragma unroll
        for (int t0 = 0; t0 < RMAX; ++t0) {
          prod[RMAX + 2 * (s0 * RMAX + t0)] = __fmul_rn(kv[s0], kv[t0]);
          prod[RMAX + 2 * (s0 * RMAX + t0) + 1] = __fmul_rn(kv[s0], qv[t0]);
        }
    }
    if (warp * 32 < DK) {
      // entries 0..31: reduce-scatter over the warp (each step a lane keeps
      // half of its values and adds the partner's copy of that half), so lane
      // e ends with entry e's sum; the rest: a plain butterfly
      static_assert(ND >= 32, "the reduce-scatter takes the first 32 entries");
#pragma unroll
      for (int off = 16, half = 16; off >= 1; off >>= 1, half >>= 1) {
        const bool up = (lane & off) != 0;
#pragma unroll
        for (int i = 0; i < half; ++i) {
          const float send = up ? prod[i] : prod[i + half];
          const float keep = up ? prod[i + half] : prod[i];
          prod[i] = __fadd_rn(keep, __shfl_xor_sync(kFull, send, off));
        }
      }
      spart[warp][lane] = prod[0];
#pragma unroll
      for (int e = 32; e < ND; ++e) {
        float v = prod[e];
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) v = __fadd_rn(v, __shfl_xor_sync(kFull, v, off));
        if (lane == 0) spart[warp][e] = v;
      }
    }
    __syncthreads();
    if (tid < nd) {
      int src;
      if (tid < n) {
        src = tid;
      } else {
        const int e2 = tid - n, s0 = (e2 >> 1) / n, t0 = (e2 >> 1) % n;
        src = RMAX + 2 * (s0 * RMAX + t0) + (e2 & 1);
      }
      float acc = 0.f;
      for (int w = 0; w * 32 < DK; ++w) acc = __fadd_rn(acc, spart[w][src]);
      sdot[tid] = acc;
    }
  } else {
    // many rows: one warp per entry
    for (int e = warp; e < nd; e += kPrepThreads / 32) {
      const float* x0;
      const float* x1;
      if (e < n) {
        x0 = x1 = &sy[e][0];
      } else {
        const int e2 = e - n, which = e2 & 1, s0 = (e2 >> 1) / n, t0 = (e2 >> 1) % n;
        x0 = &sy[s0][DK];
        x1 = which ? &sy[t0][0] : &sy[t0][DK];
      }
      float acc = 0.f;
      for (int j = lane; j < DK; j += 32) acc = __fmaf_rn(x0[j], x1[j], acc);
#pragma unroll
      for (int off = 16; off >= 1; off >>= 1) acc = __fadd_rn(acc, __shfl_xor_sync(kFull, acc, off));
      if (lane == 0) sdot[e] = acc;
    }
  }
  __syncthreads();
  auto fq = [&](int t) { return __fmul_rn(p.scale, rsqrtf(__fadd_rn(sdot[t], p.eps))); };
  auto fk = [&](int t) { return rsqrtf(__fadd_rn(sdot[n + 2 * (t * n + t)], p.eps)); };
  if (active) {  // publish scale*q^ | k^ (and, deferred, k^ into the carry)
    float* dst = p.wqk + ((size_t)b * p.H_qk + hq) * p.R * 2 * DK + tid;
    float* kc = MODE == kDeferred && tid >= DK ? p.ck + ((size_t)b * p.H_qk + hq) * p.R * DK + (tid - DK) : nullptr;
    for (int t = 0; t < n; ++t) {
      const float v = __fmul_rn(sy[t][tid], tid < DK ? fq(t) : fk(t));
      dst[(size_t)t * 2 * DK] = v;
      if (kc != nullptr) kc[(size_t)t * DK] = v;
    }
  }
  // Gram tables [R][R][2]: k^_s . k^_t and k^_s . (scale q^_t); rows past n are zero
  float* gh = p.wgh + ((size_t)b * p.H_qk + hq) * gram_floats(p.R);
  for (int i = tid; i < 2 * p.R * p.R; i += kPrepThreads) {
    const int which = i & 1, s0 = (i >> 1) / p.R, t0 = (i >> 1) % p.R;
    float val = 0.f;
    if (s0 < n && t0 < n)
      val = __fmul_rn(__fmul_rn(sdot[n + 2 * (s0 * n + t0) + which], fk(s0)), which ? fq(t0) : fk(t0));
    gh[i] = val;
  }
  // per-row decay and write strength of the value heads that read this q/k head
  for (int i = tid; i < p.G * gr; i += kPrepThreads) {
    const int h = hq * p.G + i / gr, t = i % gr;
    if (t >= n) continue;
    if (i >= kPrepThreads) load_gate(t, h, g_i, beta_i);  // more (head, row) pairs than threads: load now
    float gg = g_i, bb = beta_i;
    if (p.raw_gating) {  // g = -exp(A_log) softplus(a), beta = sigmoid(b), overflow-free forms
      gg = -expf(__ldg(p.A_log + h)) * (fmaxf(g_i, 0.f) + log1pf(expf(-fabsf(g_i))));
      bb = 1.f / (1.f + expf(-beta_i));
    }
    const float decay = expf(gg);
    *reinterpret_cast<float4*>(p.wsc + (((size_t)b * p.H_v + h) * p.R + t) * 4) = make_float4(decay, bb, 0.f, 0.f);
    if (MODE == kDeferred) p.ca[((size_t)b * p.H_v + h) * round4(p.R) + t] = decay;
  }
}

// ------------------------------------------------------------ the rows
// Persistent: CTA j runs items j, j + gridDim.x, ...; item = (request b,
// value head h, row slice sl), numbered ((b H_v) + h) slices + sl.  The state
// slice has one shared-memory buffer: as soon as an item's slice is in
// registers, the next item's slice (one bulk copy) is requested, so it is in
// flight while the item computes.  The item's q/k rows, v rows, per-row
// scalars and Gram tables are small and double-buffered, or single-buffered
// when that lets a quarter more CTAs be resident (long requests).  In
// deferred mode an item first commits the previous call's rows from its
// carry (one rank-(a+1) update of the registers, stored to the slot).
//
// The rows of an item run in chunks of up to CH rows.  With C_t the product of
// the decays of the chunk's rows up to t and z_s^(t) = (C_t / C_s) u_s, the
// recurrence unrolls over the chunk to
//   r_t = C_t (S0 k_t) + sum_{s<t} z_s^(t-1) alpha_t (k_s . k_t)      u_t = beta_t (v_t - r_t)
//   o_t = C_t (S0 q~_t) + sum_{s<=t} z_s^(t) (k_s . q~_t)
//   S_t = C_t S0 + sum_{s<=t} z_s^(t) k_s^T
// so every dot product of the chunk is taken on the chunk's starting state S0
// in one pass, each state row then runs a short scalar recurrence, and the
// state is written once (at the commit row, or advanced to the chunk's end).
template <int DK, bool WIDE = false>
struct Stage {
  static constexpr int DVS = Geo<DK, WIDE>::DVS;
  __host__ __device__ static int rows_floats(int R) { return R * 2 * DK + R * DVS + R * 4 + gram_floats(R); }
  // deferred mode: a previous call's carry rows, [Rp][DVS] u | [Rp][DK] k^ | [Rp4] exp(g)
  __host__ __device__ static int carry_floats(int Rp) { return Rp * DVS + Rp * DK + round4(Rp); }
  __host__ __device__ static size_t bytes(int R, int Rp, int stages) {
    return sizeof(float) * ((size_t)DVS * DK + stages * (size_t)(rows_floats(R) + carry_floats(Rp)));
  }
};

// Sums, over the LPR lanes of a row group, each lane's partial dot products of
// its M rows with NV vectors (v[m][x]), and leaves the lane holding the NV
// finished sums of one row: row_of_lane<LPR, M>(lane).  Partners are taken at
// offsets LPR/2, LPR/4, .., 1 in that order, the same for every value.
template <int LPR, int M, int NV>
__device__ __forceinline__ void reduce_rows(float (&v)[M][NV], float (&out)[NV], int lane) {
  constexpr int LM = ilog2(M);
  static_assert((1 << LM) == M && M <= LPR, "M must be a power of two <= LPR");
#pragma unroll
  for (int l = 0; l < LM; ++l) {
    const int off = LPR >> (l + 1);
    const int half = M >> (l + 1);
    const bool up = (lane & off) != 0;
#pragma unroll
    for (int i = 0; i < half; ++i)
#pragma unroll
      for (int x = 0; x < NV; ++x) {
        const float send = up ? v[i][x] : v[i + half][x];
        const float keep = up ? v[i + half][x] : v[i][x];
        v[i][x] = __fadd_rn(keep, __shfl_xor_sync(kFull, send, off));
      }
  }
#pragma unroll
  for (int off = LPR >> (LM + 1); off >= 1; off >>= 1)
#pragma unroll
    for (int x = 0; x < NV; ++x) v[0][x] = __fadd_rn(v[0][x], __shfl_xor_sync(kFull, v[0][x], off));
#pragma unroll
  for (int x = 0; x < NV; ++x) out[x] = v[0][x];
}
template <int LPR, int M>
__device__ __forceinline__ int row_of_lane(int lane) {
  int m = 0;
#pragma unroll
  for (int l = 0; l < ilog2(M); ++l)
    if (lane & (LPR >> (l + 1))) m += M >> (l + 1);
  return m;
}
// offset within the row group of a lane that holds row m's sums
template <int LPR, int M>
__device__ __forceinline__ int lane_of_row(int m) {
  int off = 0;
#pragma unroll
  for (int l = 0; l < ilog2(M); ++l)
    if ((m / (M >> (l + 1))) & 1) off |= LPR >> (l + 1);
  return off;
}

// STAGES: buffers for an item's staged rows, 2 (the next item's rows land
// while this one computes) or 1 (they land once this item is done with them).
template <int DK, int MODE, int STAGES, bool WIDE>
__global__ void __launch_bounds__(Geo<DK, WIDE>::NT, Geo<DK, WIDE>::MIN_CTAS) rows_kernel(const Params p) {
  constexpr bool one_stage = STAGES == 1;
  using Gm = Geo<DK, WIDE>;
  constexpr int LPR = Gm::LPR, NC4 = Gm::NC4, RG = Gm::RG, M = Gm::M;
  constexpr int DVS = Gm::DVS, ROWS_W = Gm::ROWS_W;
  constexpr int NP = 2 * NC4;  // column pairs per lane per row
  constexpr int CH = 4;        // rows per chunk
  constexpr int kDup = (LPR >> ilog2(M)) - 1;  // low lane bits that repeat a row's sums
  constexpr bool kWantO = MODE != kCommitReplay;
  constexpr bool kCommits = MODE == kFused || MODE == kCommitReplay || MODE == kDeferred;
  constexpr bool kSnap = MODE == kVerifySnap;
  constexpr uint32_t kSBytes = DVS * DK * sizeof(float);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n_items = p.B * p.H_v * p.slices;
  const int R = p.R;
  const int Rp = MODE == kDeferred ? p.Rp : 0;
  // The CTA's item after item `it` (-1: none): CTA j runs items j, j + G, j + 2G, ...
  auto next_item = [&](int it) -> int { return it + (int)gridDim.x < n_items ? it + (int)gridDim.x : -1; };
  const int rfl = Stage<DK, WIDE>::rows_floats(R) + Stage<DK, WIDE>::carry_floats(Rp);
  extern __shared__ __align__(16) float smem[];
  float* const stS = smem;  // [DVS][DK] state slice of the next item
  auto stQK = [&](int s) { return smem + DVS * DK + (size_t)s * rfl; };  // [R][2 DK]  scale*q^ | k^
  auto stV = [&](int s) { return stQK(s) + R * 2 * DK; };               // [R][DVS]   v
  auto stSC = [&](int s) { return stV(s) + R * DVS; };                  // [R][4]     exp(g), beta
  auto stGH = [&](int s) { return stSC(s) + R * 4; };                   // [R][R][2]  k.k, k.q~ (padded)
  auto stCU = [&](int s) { return stGH(s) + gram_floats(R); };          // [Rp][DVS]  previous rows' u
  auto stCK = [&](int s) { return stCU(s) + Rp * DVS; };                // [Rp][DK]   previous rows' k^
  auto stCA = [&](int s) { return stCK(s) + Rp * DK; };                 // [Rp4]      previous rows' exp(g)
  __shared__ __align__(8) uint64_t barS, barQ[2];
  __shared__ int sMeta[2][4];  // per item parity: slot, rows to run, commit row (-1 none), previous rows to commit

  // ---- producer side (thread 0) ----
  // An item's request data is loaded one item ahead of its use and evaluated
  // only when its copies are issued, so the producer's warp never waits on
  // those loads while the item before it computes.
  struct Req {
    int n, slot, a, np;  // np: the previous call's rows (deferred mode), a then its accepted drafts
  };
  auto load_req = [&](int it) {
    const int b = fdiv(it, p.div_hs);
    Req q;
    q.n = p.n_rows[b];
    q.slot = p.slot_ids[b];
    if (MODE == kDeferred) {
      q.np = p.n_prev ? p.n_prev[b] : 0;
      q.a = p.n_prev ? p.acc_prev[b] : -1;
    } else {
      q.np = 0;
      q.a = kCommits ? p.accept_len[b] : -1;
    }
    return q;
  };
  // item it's request data -> its row of sMeta; reports a bad request once per request
  auto meta = [&](int it, const Req& q, int* m) {
    const int hs = it - fdiv(it, p.div_hs) * p.H_v * p.slices;
    int report, crow, off = 0;
    m[0] = q.slot;
    if (MODE == kDeferred) {  // rows = the current rows only; off previous rows are committed first
      const int t_end = deferred_rows_of(p, q.n, q.slot, q.np, q.a, off, crow, report);
      m[1] = t_end - off;
    } else
      m[1] = request_rows_of<kCommits, MODE == kCommitReplay>(p, q.n, q.slot, q.a, crow, report);
    m[2] = crow;
    m[3] = off;
    if (report && hs == 0) flag(p.status, report);
  };
  auto issue_state = [&](int it, int slot, int rows) {
    if (rows == 0) {
      mbar_arrive(&barS);
      return;
    }
    const int b = fdiv(it, p.div_hs);
    const int hs = it - b * p.H_v * p.slices;  // h * slices + sl
    mbar_expect_tx(&barS, kSBytes);
#ifdef GDN_TEST_HOOKS
    if (it == g_test_drop_item) return;  // declared, never issued: the item's wait runs out
#endif
    bulk_load(stS, p.S + ((size_t)slot * p.H_v * p.slices + hs) * DVS * DK, kSBytes, &barS);
  };
  // rows: current rows to stage; prev: previous rows whose carry is staged (deferred mode)
  auto issue_rows = [&](int s, int it, int rows, int prev) {
    const uint32_t rb = rows > 0 ? (rows * (2 * DK + DVS + 4) + gram_floats(R)) * sizeof(float) : 0;
    const uint32_t cb = prev > 0 ? (prev * (DVS + DK) + round4(prev)) * sizeof(float) : 0;
    if (rb + cb == 0) {
      mbar_arrive(&barQ[s]);
      return;
    }
    const int b = fdiv(it, p.div_hs);
    const int hs = it - b * p.H_v * p.slices;
    const int h = fdiv(hs, p.div_sl);
    const int hq = fdiv(h, p.div_g);
    mbar_expect_tx(&barQ[s], rb + cb);
    if (rows > 0) {
      bulk_load(stQK(s), p.wqk + ((size_t)b * p.H_qk + hq) * R * 2 * DK, rows * 2 * DK * sizeof(float), &barQ[s]);
      bulk_load(stV(s), p.wv + ((size_t)b * p.H_v * p.slices + hs) * R * DVS, rows * DVS * sizeof(float), &barQ[s]);
      bulk_load(stSC(s), p.wsc + ((size_t)b * p.H_v + h) * R * 4, rows * 4 * sizeof(float), &barQ[s]);
      bulk_load(stGH(s), p.wgh + ((size_t)b * p.H_qk + hq) * gram_floats(R), gram_floats(R) * sizeof(float),
                &barQ[s]);
    }
    if (MODE == kDeferred && prev > 0) {
      bulk_load(stCU(s), p.pcu + ((size_t)b * p.H_v * p.slices + hs) * Rp * DVS, prev * DVS * sizeof(float),
                &barQ[s]);
      bulk_load(stCK(s), p.pck + ((size_t)b * p.H_qk + hq) * Rp * DK, prev * DK * sizeof(float), &barQ[s]);
      bulk_load(stCA(s), p.pca + ((size_t)b * p.H_v + h) * round4(Rp), round4(prev) * sizeof(float), &barQ[s]);
    }
  };

  // Two producer threads, one per warp, so each warp issues part of the next
  // item's copies: thread 0 the state slice, thread 32 (thread 0 when the CTA
  // has one warp) the q/k/v rows and tables.  Both keep the next item's
  // request data.
  constexpr int kRowsProducer = Gm::NT > 32 ? 32 : 0;
  const bool producer = tid == 0 || tid == kRowsProducer;
  Req qn{0, 0, -1, 0};  // producer: request data of the item after the current one
  const int it0 = (int)blockIdx.x < n_items ? (int)blockIdx.x : -1;
  const int it1st = it0 >= 0 ? next_item(it0) : -1;
  if (!p.early && tid == kRowsProducer && it1st >= 0) qn = load_req(it1st);
  if (tid == 0) {
    mbar_init(&barS, 1);
    mbar_init(&barQ[0], 1);
    mbar_init(&barQ[1], 1);
    if (it0 >= 0) {
      if (p.early) {
        // Only the slot and the row count are read before the wait (the
        // caller promised nothing in flight writes them or the state); the
        // slice is fetched whenever the request could need it, and what the
        // item does with it is decided after the wait.
        const int b = fdiv(it0, p.div_hs);
        const int slot = p.slot_ids[b], n = p.n_rows[b];
        const bool need = slot >= 0 && slot < p.P && n >= 0 && n <= p.R && (n > 0 || MODE == kDeferred);
        issue_state(it0, slot, need ? 1 : 0);
      } else {
        const Req q0 = load_req(it0);
        if (it1st >= 0) qn = load_req(it1st);  // both in flight
        meta(it0, q0, sMeta[0]);
        issue_state(it0, sMeta[0][0], sMeta[0][1] + sMeta[0][3]);  // before the prologue has finished
      }
    }
  }
  __syncthreads();  // the barriers are initialised before anyone waits on them
  pdl_wait();       // the prologue's q, k, v and tables are complete and visible
  if (p.early) {    // the rest of the request data, now that the kernels before have finished
    if (tid == 0 && it0 >= 0) meta(it0, load_req(it0), sMeta[0]);
    if (producer && it1st >= 0) qn = load_req(it1st);
    __syncthreads();
  }
  if (tid == kRowsProducer && it0 >= 0) issue_rows(0, it0, sMeta[0][1], sMeta[0][3]);

  const int c = lane & (LPR - 1);
  const int rg = lane / LPR;
  const int wrow = warp * ROWS_W + rg;  // slice-local row of m = 0; row m adds m * RG
  const int gbase = lane & ~(LPR - 1);
  const int rl = wrow + row_of_lane<LPR, M>(lane) * RG;  // the row whose sums this lane holds
  const bool writer = (lane & kDup) == 0;
  const size_t o_tstride = (size_t)p.H_v * p.d_v;

  // With one rows stage an item's rows are copied once the item before it
  // has finished reading the buffer.
  int pend_it = -1, pend_rows = 0, pend_prev = 0;  // rows producer: copy deferred to the item's end

  for (int k = 0, it = it0; it >= 0; ++k, it = next_item(it)) {
    const int mi = k & 1;                                  // sMeta slot
    const int s = one_stage ? 0 : mi;                      // rows stage
    const uint32_t qpar = one_stage ? k & 1 : (k >> 1) & 1;  // phase of barQ[s] for this item
    // the arrive that completes each phase releases the producer's sMeta write
    const bool late = !(mbar_wait(&barS, k & 1) && mbar_wait(&barQ[s], qpar));
    if (__syncthreads_or(late)) {
      // Nothing of this item or later ones is written.  The copies in flight
      // are this item's (its successor's are issued only after this wait):
      // a second bounded wait lets a slow one land before the CTA leaves.
      // The limit is far beyond a copy's microseconds, so only a barrier
      // whose declared bytes were never issued still reads incomplete here,
      // and such a barrier has no copy in flight.
      if (tid == 0) flag(p.status, GDN_STATUS_TIMEOUT);
      mbar_wait(&barS, k & 1);
      mbar_wait(&barQ[s], qpar);
      return;
    }
    const int slot = sMeta[mi][0], rows = sMeta[mi][1];
    const int prev = MODE == kDeferred ? sMeta[mi][3] : 0;  // previous call's rows to commit first
    const int a = MODE == kDeferred ? -1 : sMeta[mi][2];    // commit row among this call's rows
    const bool busy = rows > 0 || prev > 0;

    f2 S[M][NP];  // column pairs of the lane's 4-column chunks
    if (busy) {
#pragma unroll
      for (int m = 0; m < M; ++m)
#pragma unroll
        for (int j = 0; j < NC4; ++j) {
          const ulonglong2 v = *reinterpret_cast<const ulonglong2*>(stS + (wrow + m * RG) * DK + 4 * (c + LPR * j));
          S[m][2 * j] = v.x;
          S[m][2 * j + 1] = v.y;
        }
    }
    __syncthreads();  // the state buffer is free: request the next item
    // On its last item the CTA lets the next call's prologue launch, so that
    // prologue's blocks take the SMs as CTAs leave and warm their inputs.
    const int it1 = next_item(it);
    if (it1 < 0) pdl_trigger();
    if (producer) {
      if (it1 >= 0) {
        fence_proxy_async();  // the reads above happen before the bulk copies overwrite the buffers
        int m[4];
        meta(it1, qn, m);  // loaded an item ago
        if (tid == 0) {
#pragma unroll
          for (int j = 0; j < 4; ++j) sMeta[mi ^ 1][j] = m[j];
          issue_state(it1, m[0], m[1] + m[3]);
        }
        if (tid == kRowsProducer) {
          if (!one_stage) {
            issue_rows(s ^ 1, it1, m[1], m[3]);
          } else if (!busy) {
            issue_rows(0, it1, m[1], m[3]);  // this item does not use the buffer
          } else {
            pend_it = it1;
            pend_rows = m[1];
            pend_prev = m[3];
          }
        }
        const int it2 = next_item(it1);
        if (it2 >= 0) qn = load_req(it2);  // in flight while this item computes
      }
    }
    if (!busy) continue;

    const int b = fdiv(it, p.div_hs);
    const int hs = it - b * p.H_v * p.slices;
    const int h = fdiv(hs, p.div_sl), sl = hs - h * p.slices;
    const float* sQK = stQK(s);
    const float* sV = stV(s);
    const float* sSC = stSC(s);
    const float* sGH = stGH(s);
    float* Sg = p.S + ((size_t)slot * p.H_v * p.slices + hs) * DVS * DK;
    float* og = nullptr;
    if (kWantO) og = p.o + ((size_t)b * p.R * p.H_v + h) * p.d_v + (size_t)sl * DVS + rl;

    // lane's column pairs of the d_k-vector at rp
    auto load_row = [&](const float* rp, f2 (&vv)[NP]) {
      const ulonglong2* vp = reinterpret_cast<const ulonglong2*>(rp);
#pragma unroll
      for (int j = 0; j < NC4; ++j) {
        const ulonglong2 v = vp[c + LPR * j];
        vv[2 * j] = v.x;
        vv[2 * j + 1] = v.y;
      }
    };
    // row vector t of the item's rows: q at part 0, k at part DK
    auto load_vec = [&](int t, int part, f2 (&vv)[NP]) { load_row(sQK + t * 2 * DK + part, vv); };
    // dst[m] = cc * S[m] + sum_{x<nt} w_x(row m) k_x, k_x the d_k-vector at kb + x ks, in that order;
    // in place when dst is S
    auto combine = [&](const float* kb, int ks, int nt, float cc, const float (&w)[CH], bool in_place,
                       float* out) {
      // coefficient x of row m lives in the lane holding row m's sums
      auto wm = [&](int m, int x) { return __shfl_sync(kFull, w[x], gbase | lane_of_row<LPR, M>(m)); };
      const f2 cc2 = pack2(cc, cc);
      if (in_place) {
#pragma unroll
        for (int m = 0; m < M; ++m)
#pragma unroll
          for (int j = 0; j < NP; ++j) S[m][j] = mul2(cc2, S[m][j]);
#pragma unroll
        for (int x = 0; x < CH; ++x) {
          if (x < nt) {
            f2 kv[NP];
            load_row(kb + x * ks, kv);
#pragma unroll
            for (int m = 0; m < M; ++m) {
              const float wx = wm(m, x);
              const f2 w2 = pack2(wx, wx);
#pragma unroll
              for (int j = 0; j < NP; ++j) S[m][j] = fma2(w2, kv[j], S[m][j]);
            }
          }
        }
      } else {
#pragma unroll
        for (int m = 0; m < M; ++m) {
          f2 acc[NP];
#pragma unroll
          for (int j = 0; j < NP; ++j) acc[j] = mul2(cc2, S[m][j]);
#pragma unroll
          for (int x = 0; x < CH; ++x) {
            if (x < nt) {
              f2 kv[NP];
              load_row(kb + x * ks, kv);
              const float wx = wm(m, x);
              const f2 w2 = pack2(wx, wx);
#pragma unroll
              for (int j = 0; j < NP; ++j) acc[j] = fma2(w2, kv[j], acc[j]);
            }
          }
#pragma unroll
          for (int j = 0; j < NC4; ++j)
            *reinterpret_cast<ulonglong2*>(out + (size_t)(wrow + m * RG) * DK + 4 * (c + LPR * j)) =
                make_ulonglong2(acc[2 * j], acc[2 * j + 1]);
        }
      }
    };
    auto store_state = [&](float* out) {
#pragma unroll
      for (int m = 0; m < M; ++m)
#pragma unroll
        for (int j = 0; j < NC4; ++j)
          *reinterpret_cast<ulonglong2*>(out + (size_t)(wrow + m * RG) * DK + 4 * (c + LPR * j)) =
              make_ulonglong2(S[m][2 * j], S[m][2 * j + 1]);
    };

    // ---- deferred: commit the previous call's rows 0..prev-1 from its carry ----
    //   S <- C S + sum_{s<prev} (u_s prod_{s<j<prev} alpha_j) k_s^T,  C = prod_{j<prev} alpha_j
    if (MODE == kDeferred && prev > 0) {
      const float* sCU = stCU(s);
      const float* sCK = stCK(s);
      const float* sCA = stCA(s);
      float ctot = 1.f;
      for (int j = 0; j < prev; ++j) ctot = __fmul_rn(ctot, sCA[j]);
      for (int s0 = 0; s0 < prev; s0 += CH) {
        float w[CH];
#pragma unroll
        for (int x = 0; x < CH; ++x) {
          const int sx = s0 + x;
          float d = 0.f;
          if (sx < prev) {
            d = sCU[sx * DVS + rl];
            for (int j = sx + 1; j < prev; ++j) d = __fmul_rn(d, sCA[j]);
          }
          w[x] = d;
        }
        combine(sCK + s0 * DK, DK, prev - s0 < CH ? prev - s0 : CH, s0 == 0 ? ctot : 1.f, w, true, nullptr);
      }
      store_state(Sg);
    }

    for (int c0 = 0; c0 < rows; c0 += CH) {
      const int nc = rows - c0 < CH ? rows - c0 : CH;
      const bool last = c0 + CH >= rows;
      // ---- every dot product of the chunk on its starting state ----
      float pk[CH], pq[CH];
      {
        float part[M][CH];
#pragma unroll
        for (int x = 0; x < CH; ++x) {
          if (x < nc) {
            f2 kv[NP];
            load_vec(c0 + x, DK, kv);
#pragma unroll
            for (int m = 0; m < M; ++m) {
              f2 acc = fma2(S[m][0], kv[0], pack2(0.f, 0.f));
#pragma unroll
              for (int j = 1; j < NP; ++j) acc = fma2(S[m][j], kv[j], acc);
              part[m][x] = sum2(acc);
            }
          } else {
#pragma unroll
            for (int m = 0; m < M; ++m) part[m][x] = 0.f;
          }
        }
        reduce_rows<LPR, M, CH>(part, pk, lane);
      }
      if constexpr (kWantO) {
        float part[M][CH];
#pragma unroll
        for (int x = 0; x < CH; ++x) {
          if (x < nc) {
            f2 qv[NP];
            load_vec(c0 + x, 0, qv);
#pragma unroll
            for (int m = 0; m < M; ++m) {
              f2 acc = fma2(S[m][0], qv[0], pack2(0.f, 0.f));
#pragma unroll
              for (int j = 1; j < NP; ++j) acc = fma2(S[m][j], qv[j], acc);
              part[m][x] = sum2(acc);
            }
          } else {
#pragma unroll
            for (int m = 0; m < M; ++m) part[m][x] = 0.f;
          }
        }
        reduce_rows<LPR, M, CH>(part, pq, lane);
      }
      // ---- the lane's row: scalar recurrence over the chunk ----
      float z[CH], zc[CH];  // z[s] = decayed u_s; zc = z at the commit row
      float cdec = 1.f, ccom = 1.f;
      int ncom = 0;  // terms of the commit combination (0: commit row not in this chunk)
#pragma unroll
      for (int x = 0; x < CH; ++x) z[x] = zc[x] = 0.f;
#pragma unroll
      for (int t = 0; t < CH; ++t) {
        if (t < nc) {
          const float2 ab = *reinterpret_cast<const float2*>(sSC + 4 * (c0 + t));  // exp(g), beta
          cdec = __fmul_rn(cdec, ab.x);
          float r = __fmul_rn(cdec, pk[t]);
#pragma unroll
          for (int x = 0; x < CH; ++x)
            if (x < t) {
              z[x] = __fmul_rn(z[x], ab.x);
              r = __fmaf_rn(z[x], sGH[((c0 + x) * R + (c0 + t)) * 2], r);
            }
          z[t] = __fmul_rn(ab.y, __fsub_rn(sV[(c0 + t) * DVS + rl], r));
          if (MODE == kDeferred && writer)  // the row's update vector, for the next call's commit
            p.cu[(((size_t)b * p.H_v * p.slices + hs) * R + c0 + t) * DVS + rl] = z[t];
          if constexpr (kWantO) {
            float oo = __fmul_rn(cdec, pq[t]);
#pragma unroll
            for (int x = 0; x < CH; ++x)
              if (x <= t) oo = __fmaf_rn(z[x], sGH[((c0 + x) * R + (c0 + t)) * 2 + 1], oo);
            if (writer) og[(size_t)(c0 + t) * o_tstride] = oo;
          }
          if (kCommits && c0 + t == a) {
#pragma unroll
            for (int x = 0; x < CH; ++x) zc[x] = x <= t ? z[x] : 0.f;
            ccom = cdec;
            ncom = t + 1;
          }
          if (kSnap)
            combine(sQK + c0 * 2 * DK + DK, 2 * DK, t + 1, cdec, z, false,
                    p.snapS + (((size_t)b * R + c0 + t) * p.H_v * p.slices + hs) * DVS * DK);
        }
      }
      // ---- commit: S_a = C_a S0 + sum_{s<=a} z_s k_s^T ----
      if (kCommits && ncom > 0) {
        if (last) {
          combine(sQK + c0 * 2 * DK + DK, 2 * DK, ncom, ccom, zc, true, nullptr);
          store_state(Sg);
        } else {
          combine(sQK + c0 * 2 * DK + DK, 2 * DK, ncom, ccom, zc, false, Sg);
        }
      }
      // ---- advance the state to the chunk's end when rows follow ----
      if (!last) combine(sQK + c0 * 2 * DK + DK, 2 * DK, nc, cdec, z, true, nullptr);
    }
    if (one_stage) {
      __syncthreads();  // every warp is done with the rows buffer: the next item's rows may land
      if (tid == kRowsProducer && pend_it >= 0) {
        fence_proxy_async();
        issue_rows(0, pend_it, pend_rows, pend_prev);
        pend_it = -1;
      }
    }
  }
  pdl_trigger();  // CTAs that had no item
}

// Snapshot commit: slot <- scratch row accept_len[b] (state and conv window).
template <typename T>
__global__ void __launch_bounds__(256) snapshot_commit_kernel(const Params p) {
  pdl_wait();  // the snapshot verify before it is complete and visible
  const int b = blockIdx.y;
  int slot, a, off, report;  // a: the commit row
  const int t_end = request_block<kCommitReplay>(p, b, slot, a, off, report);
  if (report && blockIdx.x == 0 && threadIdx.x == 0) flag(p.status, report);
  if (t_end == 0) return;
  const size_t slot_elems = (size_t)p.H_v * p.d_v * p.d_k;
  const float4* src = reinterpret_cast<const float4*>(p.snapS + ((size_t)b * p.R + a) * slot_elems);
  float4* dst = reinterpret_cast<float4*>(p.S + (size_t)slot * slot_elems);
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  const size_t i0 = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  for (size_t i = i0; i < slot_elems / 4; i += stride) dst[i] = src[i];
  const size_t cs_bytes = (size_t)p.C * kWS * sizeof(T);  // a multiple of 16: C % 16 == 0
  const uint4* csrc = reinterpret_cast<const uint4*>(static_cast<const T*>(p.snapCs) +
                                                     ((size_t)b * p.R + a) * p.C * kWS);
  uint4* cdst = reinterpret_cast<uint4*>(static_cast<T*>(p.conv_state) + (size_t)slot * p.C * kWS);
  for (size_t i = i0; i < cs_bytes / 16; i += stride) cdst[i] = csrc[i];
}

// ------------------------------------------------------------------ host
template <typename Kernel>
int launch(Kernel kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t st, const Params& p) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kernel, p) != cudaSuccess) return GDN_ERR_LAUNCH;
  return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_LAUNCH;
}

// Both kernels ask for the same (largest) shared-memory carveout: an SM whose
// carveout differs from a waiting kernel's cannot take that kernel's CTAs until
// it drains, which would keep the rows kernel from starting while the
// prologue still runs.
template <typename Kernel>
int prefer_max_shared(Kernel kernel) {
  return cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                              (int)cudaSharedmemCarveoutMaxShared) == cudaSuccess
             ? GDN_OK
             : GDN_ERR_LAUNCH;
}

// Once per kernel instantiation and device (bit dev of done): the max-shared
// carveout and a dynamic shared-memory cap large enough for every shape, so
// no later call lowers what a concurrent launch relies on.  Racing first
// calls set the same values.
template <typename Kernel>
int setup_kernel(Kernel kernel, size_t max_smem, std::atomic<unsigned long long>& done, int dev) {
  if (dev < 0 || dev >= 64) return GDN_ERR_UNSUPPORTED;
  const unsigned long long bit = 1ull << dev;
  if (done.load(std::memory_order_acquire) & bit) return GDN_OK;
  if (prefer_max_shared(kernel) != GDN_OK) return GDN_ERR_LAUNCH;
  if (max_smem > 48 * 1024 &&
      cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)max_smem) != cudaSuccess)
    return GDN_ERR_LAUNCH;
  done.fetch_or(bit, std::memory_order_acq_rel);
  return GDN_OK;
}

// Persistent grid of the rows kernel: as many CTAs as fit at once (at most one
// per item).
template <int DK, int MODE, bool WIDE>
int launch_rows(const Params& p, cudaStream_t st) {
  using Gm = Geo<DK, WIDE>;
  const int Rp = MODE == kDeferred ? p.Rp : 0;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return GDN_ERR_LAUNCH;
  static std::atomic<unsigned long long> set1{0}, set2{0};
  const int max_rp = MODE == kDeferred ? kMaxR : 0;
  int rc = setup_kernel(rows_kernel<DK, MODE, 1, WIDE>, Stage<DK, WIDE>::bytes(kMaxR, max_rp, 1), set1, dev);
  if (rc == GDN_OK) rc = setup_kernel(rows_kernel<DK, MODE, 2, WIDE>, Stage<DK, WIDE>::bytes(kMaxR, max_rp, 2), set2, dev);
  if (rc != GDN_OK) return rc;
  // Double-buffered rows staging unless one buffer lets at least a quarter
  // more CTAs be resident (long requests): measured, one more CTA per SM
  // does not pay for the exposed copy of each item's rows, three more do.
  struct Choice {
    int dev = -1, R = -1, Rp = -1;
    int stages = 2;
    size_t smem = 0;
    int ctas = 0;  // resident CTAs on the device for this shape
  };
  static std::mutex mu;
  static Choice last;  // per instantiation: the last shape's choice
  Choice c;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (last.dev != dev || last.R != p.R || last.Rp != Rp) {
      const size_t smem2 = Stage<DK, WIDE>::bytes(p.R, Rp, 2), smem1 = Stage<DK, WIDE>::bytes(p.R, Rp, 1);
      int per2 = 0, per1 = 0, sms = 0;
      if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per2, rows_kernel<DK, MODE, 2, WIDE>, Gm::NT, smem2) !=
              cudaSuccess ||
          cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per1, rows_kernel<DK, MODE, 1, WIDE>, Gm::NT, smem1) !=
              cudaSuccess ||
          cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || per1 < 1)
        return GDN_ERR_LAUNCH;
      last.dev = dev;
      last.R = p.R;
      last.Rp = Rp;
      last.stages = 4 * per1 >= 5 * per2 ? 1 : 2;
      last.smem = last.stages == 2 ? smem2 : smem1;
      last.ctas = (last.stages == 2 ? per2 : per1) * sms;
    }
    c = last;
  }
  const long long items = (long long)p.B * p.H_v * p.slices;
  const long long grid = items < c.ctas ? items : c.ctas;
  return c.stages == 2 ? launch(rows_kernel<DK, MODE, 2, WIDE>, dim3((unsigned)grid), dim3(Gm::NT), c.smem, st, p)
                       : launch(rows_kernel<DK, MODE, 1, WIDE>, dim3((unsigned)grid), dim3(Gm::NT), c.smem, st, p);
}

template <int MODE>
int dispatch_rows(const Params& p, cudaStream_t st) {
  switch (p.d_k) {
    case 16:
      return launch_rows<16, MODE, false>(p, st);
    case 32:
      return launch_rows<32, MODE, false>(p, st);
    case 64:
      return launch_rows<64, MODE, false>(p, st);
    default:
      if constexpr (MODE != kDeferred)
        if (p.dvs == Geo<128, true>::DVS) return launch_rows<128, MODE, true>(p, st);
      return launch_rows<128, MODE, false>(p, st);
  }
}

template <typename T, int MODE, int RMAX>
int launch_prep_r(const Params& p, cudaStream_t st) {
  constexpr int VV = vec_v<RMAX>();
  const int v_blocks = (p.H_v * p.d_v + kPrepThreads * VV - 1) / (kPrepThreads * VV);
  const dim3 grid(p.H_qk + v_blocks, p.B), block(kPrepThreads);
  static std::atomic<unsigned long long> set{0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return GDN_ERR_LAUNCH;
  const int rc = setup_kernel(prep_kernel<T, MODE, RMAX>, 0, set, dev);
  if (rc != GDN_OK) return rc;
  return launch(prep_kernel<T, MODE, RMAX>, grid, block, 0, st, p);
}

template <typename T, int MODE>
int launch_prep(const Params& p, cudaStream_t st) {
  if (p.R <= 4) return launch_prep_r<T, MODE, 4>(p, st);
  if (p.R <= 8) return launch_prep_r<T, MODE, 8>(p, st);
  return launch_prep_r<T, MODE, kMaxR>(p, st);
}

template <int MODE>
int run_mode(const Params& p, int in_dtype, cudaStream_t st) {
  const int rc = in_dtype == GDN_DTYPE_BF16 ? launch_prep<__nv_bfloat16, MODE>(p, st)
                                            : launch_prep<float, MODE>(p, st);
  if (rc != GDN_OK) return rc;
  return dispatch_rows<MODE>(p, st);
}

inline bool aligned(const void* ptr, size_t a) { return (reinterpret_cast<uintptr_t>(ptr) % a) == 0; }
// [a, a + na) and [b, b + nb) share a byte (empty ranges share none)
inline bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return na > 0 && nb > 0 && x < y + nb && y < x + na;
}

inline int rows_per_cta(int d_k) { return d_k >= 32 ? Geo<32>::DVS : Geo<16>::DVS; }

#ifdef GDN_TEST_HOOKS
// Test builds only: the rows per item later calls are forced to (0: chosen by
// shape; 64: the wide geometry wherever it applies; any other positive value:
// the two-warp one) and the rows per item the last call chose.
std::atomic<int> g_test_item_rows{0}, g_test_last_item_rows{0};
#endif

// Resident CTAs of the two-warp d_k = 128 rows kernel on the current device
// (8 per SM), read once per device; 0 when it cannot be read.
int narrow_slots() {
  static std::atomic<int> cached[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  int v = cached[dev].load(std::memory_order_relaxed);
  if (v > 0) return v;
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  v = Geo<128>::MIN_CTAS * sms;
  cached[dev].store(v, std::memory_order_relaxed);
  return v;
}

// State rows per rows-kernel item.  The wide geometry (64 rows, four warps)
// when d_k = 128, requests have more than 4 rows and its items still
// outnumber the two-warp kernel's resident CTAs: measured on the ragged
// B = 256 batch (up to 9 rows) 2.59 M against 2.03 M rows/s, while at 4 rows
// it is even with the two-warp form and at B = 1 it leaves CTAs idle.  Never
// for deferred calls, whose carry layout (by slice) must not change between
// calls of different row counts.
int rows_per_item(const gdn_args* a, bool wide_ok) {
  constexpr int kWide = Geo<128, true>::DVS;
  const bool can_wide = wide_ok && a->d_k == 128 && a->d_v % kWide == 0;
  int rows = rows_per_cta(a->d_k);
  if (can_wide && a->R > 4) {
    const long long items = (long long)a->B * a->H_v * (a->d_v / kWide);
    const int slots = narrow_slots();
    if (slots > 0 && items >= slots) rows = kWide;
  }
#ifdef GDN_TEST_HOOKS
  const int forced = g_test_item_rows.load(std::memory_order_relaxed);
  if (forced == kWide && can_wide)
    rows = kWide;
  else if (forced > 0 && forced != kWide)
    rows = rows_per_cta(a->d_k);
  g_test_last_item_rows.store(rows, std::memory_order_relaxed);
#endif
  return rows;
}

enum Need : unsigned {
  kNeedRows = 1u,  // x, g, beta, conv_w, work
  kNeedO = 2u,
  kNeedAccept = 4u,
  kNeedScratch = 8u
};

int check_shape(const gdn_args* a) {
  if (!a) return GDN_ERR_INVALID_ARG;
  if (a->B < 0 || a->R < 1 || a->H_qk < 1 || a->H_v < 1 || a->d_k < 1 || a->d_v < 1 || a->W < 1 ||
      a->pool_slots < 1)
    return GDN_ERR_INVALID_ARG;
  if ((a->flags & ~(GDN_FLAG_RAW_GATING | GDN_FLAG_STATE_STABLE)) != 0) return GDN_ERR_INVALID_ARG;
  if (a->in_dtype != GDN_DTYPE_BF16 && a->in_dtype != GDN_DTYPE_F32) return GDN_ERR_UNSUPPORTED;
  if (a->W != kW || a->R > kMaxR) return GDN_ERR_UNSUPPORTED;
  if (a->d_k != 16 && a->d_k != 32 && a->d_k != 64 && a->d_k != 128) return GDN_ERR_UNSUPPORTED;
  if (a->d_v % rows_per_cta(a->d_k) != 0) return GDN_ERR_UNSUPPORTED;
  if (a->H_v % a->H_qk != 0) return GDN_ERR_UNSUPPORTED;
  if (a->B > 65535) return GDN_ERR_UNSUPPORTED;
  if ((long long)a->H_v * a->d_v > 0x7fffffffLL) return GDN_ERR_UNSUPPORTED;
  return GDN_OK;
}

// Work buffer: wqk [B][H_qk][R][2 d_k], wv [B][H_v d_v / dvs][R][dvs],
// wsc [B][H_v][R][4], wgh [B][H_qk][gram_floats(R)].  Every region and every
// run a rows-kernel item copies is a multiple of 16 bytes.
size_t work_floats(const gdn_args* a, size_t* off_v, size_t* off_sc, size_t* off_gh) {
  const size_t rows = (size_t)a->B * a->R;
  const size_t qk = rows * a->H_qk * 2 * a->d_k;
  const size_t v = rows * a->H_v * a->d_v;
  const size_t sc = rows * a->H_v * 4;
  if (off_v) *off_v = qk;
  if (off_sc) *off_sc = qk + v;
  if (off_gh) *off_gh = qk + v + sc;
  return qk + v + sc + (size_t)a->B * a->H_qk * gram_floats(a->R);
}

int validate(const gdn_args* a, unsigned need, Params* out, bool wide_ok = false) {
  int rc = check_shape(a);
  if (rc != GDN_OK) return rc;
  if (!std::isfinite(a->scale) || !std::isfinite(a->l2_eps) || a->l2_eps < 0.f) return GDN_ERR_INVALID_ARG;

  if (!a->conv_state || !a->ssm_state || !a->slot_ids || !a->n_rows) return GDN_ERR_INVALID_ARG;
  if (!aligned(a->conv_state, 16) || !aligned(a->ssm_state, 16) || !aligned(a->slot_ids, 4) ||
      !aligned(a->n_rows, 4))
    return GDN_ERR_MISALIGNED;
  if (need & kNeedRows) {
    if (!a->x || !a->g || !a->beta || !a->conv_w || !a->work) return GDN_ERR_INVALID_ARG;
    if ((a->flags & GDN_FLAG_RAW_GATING) && !a->A_log) return GDN_ERR_INVALID_ARG;
    if ((a->flags & GDN_FLAG_RAW_GATING) && !aligned(a->A_log, 4)) return GDN_ERR_MISALIGNED;
    if (!aligned(a->x, 16) || !aligned(a->conv_w, 16) || !aligned(a->g, 4) || !aligned(a->beta, 4) ||
        !aligned(a->work, 16))
      return GDN_ERR_MISALIGNED;
  }
  if (need & kNeedO) {
    if (!a->o) return GDN_ERR_INVALID_ARG;
    if (!aligned(a->o, 16)) return GDN_ERR_MISALIGNED;
  }
  if (need & kNeedAccept) {
    if (!a->accept_len) return GDN_ERR_INVALID_ARG;
    if (!aligned(a->accept_len, 4)) return GDN_ERR_MISALIGNED;
  }
  if (need & kNeedScratch) {
    if (!a->scratch_S || !a->scratch_cs) return GDN_ERR_INVALID_ARG;
    if (!aligned(a->scratch_S, 16) || !aligned(a->scratch_cs, 16)) return GDN_ERR_MISALIGNED;
  }
  if (a->status && !aligned(a->status, 4)) return GDN_ERR_MISALIGNED;

  Params& p = *out;
  p.B = a->B;
  p.R = a->R;
  p.H_qk = a->H_qk;
  p.H_v = a->H_v;
  p.d_k = a->d_k;
  p.d_v = a->d_v;
  p.P = a->pool_slots;
  p.G = a->H_v / a->H_qk;
  p.dvs = rows_per_item(a, wide_ok);
  p.slices = a->d_v / p.dvs;
  p.div_hs = make_fastdiv(p.H_v * p.slices);
  p.div_sl = make_fastdiv(p.slices);
  p.div_g = make_fastdiv(p.G);
  p.C = 2LL * a->H_qk * a->d_k + (long long)a->H_v * a->d_v;
  p.scale = a->scale;
  p.eps = a->l2_eps;
  p.x = a->x;
  p.g = a->g;
  p.beta = a->beta;
  p.conv_w = a->conv_w;
  p.conv_state = a->conv_state;
  p.S = a->ssm_state;
  p.slot_ids = a->slot_ids;
  p.n_rows = a->n_rows;
  p.accept_len = a->accept_len;
  p.o = a->o;
  p.snapS = a->scratch_S;
  p.snapCs = a->scratch_cs;
  size_t off_v = 0, off_sc = 0, off_gh = 0;
  work_floats(a, &off_v, &off_sc, &off_gh);
  p.wqk = static_cast<float*>(a->work);
  p.wv = p.wqk ? p.wqk + off_v : nullptr;
  p.wsc = p.wqk ? p.wqk + off_sc : nullptr;
  p.wgh = p.wqk ? p.wqk + off_gh : nullptr;
  p.status = a->status;
  p.raw_gating = (a->flags & GDN_FLAG_RAW_GATING) != 0;
  p.early = (a->flags & GDN_FLAG_STATE_STABLE) != 0;
  p.A_log = p.raw_gating ? a->A_log : nullptr;
  p.xp = nullptr;
  p.n_prev = p.acc_prev = nullptr;
  p.pcu = p.pck = p.pca = nullptr;
  p.cu = p.ck = p.ca = nullptr;
  p.Rp = 0;
  return GDN_OK;
}

// Carry of a deferred call with R rows per request:
//   u [B][H_v d_v / dvs][R][dvs], k^ [B][H_qk][R][d_k], exp(g) [B][H_v][R4]
// (R4 = R rounded up to 4).  Every region starts on 16 bytes.
size_t carry_floats(const gdn_args* a, int R, size_t* off_k, size_t* off_a) {
  const size_t u = (size_t)a->B * R * a->H_v * a->d_v;
  const size_t k = (size_t)a->B * R * a->H_qk * a->d_k;
  if (off_k) *off_k = u;
  if (off_a) *off_a = u + k;
  return u + k + (size_t)a->B * a->H_v * round4(R);
}

int run_rows(const gdn_args* args, unsigned need, int mode, void* stream) {
  Params p;
  const int rc = validate(args, need, &p, true);
  if (rc != GDN_OK || p.B == 0) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  switch (mode) {
    case kFused:
      return run_mode<kFused>(p, args->in_dtype, st);
    case kVerify:
      return run_mode<kVerify>(p, args->in_dtype, st);
    case kVerifySnap:
      return run_mode<kVerifySnap>(p, args->in_dtype, st);
    default:
      return run_mode<kCommitReplay>(p, args->in_dtype, st);
  }
}

int run_deferred(const gdn_args* cur, const gdn_prev_rows* prev, void* stream) {
  int rc = check_shape(cur);
  if (rc != GDN_OK) return rc;
  if (prev != nullptr) {
    if (prev->R < 1) return GDN_ERR_INVALID_ARG;
    if (prev->R > kMaxR) return GDN_ERR_UNSUPPORTED;
  }
  Params p;
  rc = validate(cur, kNeedRows | kNeedO, &p);
  if (rc != GDN_OK) return rc;
  if (!cur->carry) return GDN_ERR_INVALID_ARG;
  if (!aligned(cur->carry, 16)) return GDN_ERR_MISALIGNED;
  size_t ok = 0, oa = 0;
  carry_floats(cur, cur->R, &ok, &oa);
  p.cu = static_cast<float*>(cur->carry);
  p.ck = p.cu + ok;
  p.ca = p.cu + oa;
  if (prev != nullptr) {
    if (!prev->x || !prev->n_rows || !prev->accept_len || !prev->carry) return GDN_ERR_INVALID_ARG;
    if (!aligned(prev->x, 16) || !aligned(prev->n_rows, 4) || !aligned(prev->accept_len, 4) ||
        !aligned(prev->carry, 16))
      return GDN_ERR_MISALIGNED;
    // The previous call's carry and rows must survive until this call has
    // read them, while it writes its own: the two carries, and the two x
    // blocks, are different buffers (double-buffered across steps).
    const size_t esz = cur->in_dtype == GDN_DTYPE_BF16 ? 2 : 4;
    const size_t xrow = (size_t)cur->B * (size_t)p.C * esz;
    if (overlaps(cur->carry, sizeof(float) * carry_floats(cur, cur->R, nullptr, nullptr), prev->carry,
                 sizeof(float) * carry_floats(cur, prev->R, nullptr, nullptr)) ||
        overlaps(cur->x, xrow * cur->R, prev->x, xrow * prev->R))
      return GDN_ERR_INVALID_ARG;
    carry_floats(cur, prev->R, &ok, &oa);
    p.pcu = static_cast<const float*>(prev->carry);
    p.pck = p.pcu + ok;
    p.pca = p.pcu + oa;
    p.xp = prev->x;
    p.n_prev = prev->n_rows;
    p.acc_prev = prev->accept_len;
    p.Rp = prev->R;
  }
  if (p.B == 0) return GDN_OK;
  return run_mode<kDeferred>(p, cur->in_dtype, static_cast<cudaStream_t>(stream));
}

}  // namespace gdnspec

using namespace gdnspec;

extern "C" {

GDN_API size_t gdn_work_bytes(const gdn_args* args) {
  if (check_shape(args) != GDN_OK) return 0;
  return sizeof(float) * work_floats(args, nullptr, nullptr, nullptr);
}

GDN_API int gdn_verify(const gdn_args* args, int mode, void* stream) {
  if (mode != GDN_REPLAY && mode != GDN_SNAPSHOT) return GDN_ERR_INVALID_ARG;
  const bool snap = mode == GDN_SNAPSHOT;
  return run_rows(args, kNeedRows | kNeedO | (snap ? kNeedScratch : 0u), snap ? kVerifySnap : kVerify, stream);
}

GDN_API int gdn_commit(const gdn_args* args, int mode, void* stream) {
  if (mode == GDN_REPLAY) return run_rows(args, kNeedRows | kNeedAccept, kCommitReplay, stream);
  if (mode != GDN_SNAPSHOT) return GDN_ERR_INVALID_ARG;
  Params p;
  const int rc = validate(args, kNeedAccept | kNeedScratch, &p);
  if (rc != GDN_OK || p.B == 0) return rc;
  const size_t per_req4 = (size_t)p.H_v * p.d_v * p.d_k / 4;
  int gx = (int)((per_req4 + 2047) / 2048);
  gx = gx < 1 ? 1 : (gx > 256 ? 256 : gx);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  return args->in_dtype == GDN_DTYPE_BF16
             ? launch(snapshot_commit_kernel<__nv_bfloat16>, dim3(gx, p.B), dim3(256), 0, st, p)
             : launch(snapshot_commit_kernel<float>, dim3(gx, p.B), dim3(256), 0, st, p);
}

GDN_API int gdn_verify_commit(const gdn_args* args, void* stream) {
  return run_rows(args, kNeedRows | kNeedO | kNeedAccept, kFused, stream);
}

GDN_API size_t gdn_carry_bytes(const gdn_args* args) {
  if (check_shape(args) != GDN_OK) return 0;
  return sizeof(float) * carry_floats(args, args->R, nullptr, nullptr);
}

GDN_API int gdn_verify_deferred(const gdn_args* cur, const gdn_prev_rows* prev, void* stream) {
  return run_deferred(cur, prev, stream);
}

#ifdef GDN_TEST_HOOKS
// Test builds only: make the state copy of rows-kernel item `item` of later
// calls be declared but never issued (-1 restores normal copies).
GDN_API int gdn_test_drop_state_copy(int item) {
  return cudaMemcpyToSymbol(g_test_drop_item, &item, sizeof(int)) == cudaSuccess ? GDN_OK : GDN_ERR_LAUNCH;
}
// Test builds only: force the rows per rows-kernel item of later calls (0:
// chosen by shape; 32: the two-warp geometry; 64: the wide geometry where it
// applies) and read the rows per item of the last call.
GDN_API int gdn_test_force_item_rows(int rows) {
  if (rows != 0 && rows != 32 && rows != 64) return GDN_ERR_INVALID_ARG;
  g_test_item_rows.store(rows, std::memory_order_relaxed);
  return GDN_OK;
}
GDN_API int gdn_test_last_item_rows() { return g_test_last_item_rows.load(std::memory_order_relaxed); }
// Test builds only: launch the late writer on `stream` (see
// test_late_write_kernel); read, and with reset != 0 clear, the prologue's
// count of missed slot guesses.
GDN_API int gdn_test_late_write(int* dst, const int* src, int n, unsigned long long delay_ns, void* stream) {
  if (!dst || !src || n < 0) return GDN_ERR_INVALID_ARG;
  test_late_write_kernel<<<1, 128, 0, static_cast<cudaStream_t>(stream)>>>(dst, src, n, delay_ns);
  return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_LAUNCH;
}
GDN_API long long gdn_test_guess_misses(int reset) {
  unsigned int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_test_guess_misses, sizeof v) != cudaSuccess) return -1;
  if (reset) {
    const unsigned int z = 0;
    if (cudaMemcpyToSymbol(g_test_guess_misses, &z, sizeof z) != cudaSuccess) return -1;
  }
  return v;
}
#endif

GDN_API const char* gdn_strerror(int code) {
  switch (code) {
    case GDN_OK:
      return "ok";
    case GDN_ERR_INVALID_ARG:
      return "invalid argument (null pointer, negative or inconsistent size, bad mode or flags)";
    case GDN_ERR_UNSUPPORTED:
      return "unsupported shape or dtype (W must be 4, d_k in {16,32,64,128}, d_v a multiple of the "
             "rows per block, H_v a multiple of H_qk, R <= 16, B <= 65535)";
    case GDN_ERR_MISALIGNED:
      return "misaligned pointer (x, conv_w, conv_state, ssm_state, work, scratch and o need 16 bytes; "
             "the int32 and g/beta arrays 4)";
    case GDN_ERR_LAUNCH:
      return "CUDA kernel launch failed";
    case GDN_ERR_TOO_LARGE:
      return "the call's scratch exceeds GDN_STATIC_WORK_BYTES (use gdn_verify_commit with a work buffer)";
    default:
      return "unknown gdnspec error code";
  }
}

}  // extern "C"

// ----------------------------------------------------------------------------
// Fused verify + commit without a caller-provided work buffer: the scratch is
// a file-scope device array.  Host code must not use the array's name as a
// device address (on the host it names a stand-in object); its device address
// is looked up once per device with cudaGetSymbolAddress while that device is
// current, cached, and passed to the kernels like any work buffer.

namespace gdnspec {
static __device__ __align__(256) unsigned char g_static_work[GDN_STATIC_WORK_BYTES];
constexpr int kMaxDevices = 64;
std::atomic<void*> g_static_work_addr[kMaxDevices];  // per device, set by its first call
}  // namespace gdnspec

extern "C" GDN_API int gdn_verify_commit_static(const gdn_args* args, void* stream) {
  const int rc = check_shape(args);
  if (rc != GDN_OK) return rc;
  if (sizeof(float) * work_floats(args, nullptr, nullptr, nullptr) > GDN_STATIC_WORK_BYTES) return GDN_ERR_TOO_LARGE;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return GDN_ERR_LAUNCH;
  if (dev < 0 || dev >= kMaxDevices) return GDN_ERR_UNSUPPORTED;
  void* work = g_static_work_addr[dev].load(std::memory_order_acquire);
  if (work == nullptr) {
    if (cudaGetSymbolAddress(&work, g_static_work) != cudaSuccess || work == nullptr) return GDN_ERR_LAUNCH;
    g_static_work_addr[dev].store(work, std::memory_order_release);
  }
  gdn_args a = *args;
  a.work = work;
  return gdn_verify_commit(&a, stream);
}
