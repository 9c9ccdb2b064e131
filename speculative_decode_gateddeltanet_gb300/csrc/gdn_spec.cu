// GatedDeltaNet speculative verify / commit kernels for sm_103a.
//
// Every call is two kernels on the caller's stream, chained by programmatic
// dependent launch so the second one's state loads overlap the first:
//
// prep_kernel (one thread per channel): the width-4 causal conv + SiLU of
//   every row over [committed window | verify rows], then the per-head L2
//   norm of q and k.  Writes scale*q^, k^, v, the decay and write strength
//   per row, and the rows' Gram tables k^.k^ and k^.(scale q^) into the
//   caller's work buffer.  Each conv channel has exactly one reader in
//   the call, so that thread also writes the channel's committed window
//   (commit modes) or its per-row windows (snapshot mode).  The conv reads
//   only the committed window and the verify rows, staging [history | verify
//   inputs] per channel [FreeToken #844 "MTP drafts for Qwen3.5 family +
//   Flash-Next", Design / Flash-Next target verify].
//
// rows_kernel (one CTA per (request, value head, slice of DVS state rows)):
//   loads its slice of the fp32 state S (DVS x d_k, d_k contiguous) with
//   128-bit loads into registers before waiting on the prologue, stages the
//   rows' q, k, v and tables from the work buffer with bulk async copies, and
//   runs the gated delta rule S_t = alpha S + beta (v - alpha S k) k^T,
//   o_t = scale S_t q with S resident in registers, in the chunked form
//   described at the kernel (all dot products of a chunk of rows on the
//   chunk's starting state, a scalar recurrence per state row, one state
//   update).  Lanes own 4-float column chunks of 2 or 4 rows; a row's dot
//   products are reduced over its 8 (d_k >= 32) or 4 (d_k = 16) lanes with a
//   butterfly that leaves each lane holding one row's sums.  Arithmetic is
//   fp32 with packed f32x2 FMA/MUL.
//
// The arithmetic of a row does not depend on the mode, so a fused call, a
// verify followed by a replay commit and a snapshot verify followed by a
// snapshot commit give the same bits.
//
// Modes: verify (o only; the state is only read [FreeToken #828
// "Speculative decoding: MTP and DFlash", Design]), verify with per-row
// snapshots (the widened verify state of [LightLLM #1330 "Qwen3.5 /
// Qwen3.5-MoE MTP speculative decoding", Summary]), replay commit (rows
// 0..a rerun from the slot, then written once), and fused verify + commit
// (the slot is written at row a from the registers: one read and one write
// of the state per request, the verify-and-commit kernel mode of [lmdeploy
// #5006 "speculative decoding for TurboMind", Verification path]).
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <cmath>

#include "gdnspec.h"

namespace gdnspec {

constexpr int kW = 4;             // conv width the kernels are built for
constexpr int kWS = kW - 1;       // conv-state columns
constexpr int kMaxR = 16;         // rows per request (k <= 15)
constexpr unsigned kFull = 0xffffffffu;

enum Mode : int { kFused = 0, kVerify = 1, kVerifySnap = 2, kCommitReplay = 3 };

struct Params {
  int B, R, H_qk, H_v, d_k, d_v, P, G;
  int nw;      // warps per CTA
  int dvs;     // state rows per item: nw * ROWS_W
  int slices;  // items per value head: d_v / dvs
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
  int cs;        // CTAs per cluster
  int qs;        // q (and k) channels of a q/k head that one CTA convolves: d_k / cs
  int ipc;       // state items per CTA per group: G * slices / cs
  int n_groups;  // B * H_qk
  int* status;
};

// Lane geometry of the state rows for a d_k-column state.  A warp holds
// ROWS_W rows; a CTA has nw (1..8, chosen per call) warps, so an item is a
// slice of DVS = nw * ROWS_W state rows.
template <int DK>
struct Geo {
  static constexpr int LPR = DK >= 32 ? 8 : 4;   // lanes per state row
  static constexpr int NC4 = DK / (4 * LPR);     // 4-column chunks per lane per row
  static constexpr int RG = 32 / LPR;            // row groups per warp
  static constexpr int M = DK >= 64 ? 4 : 2;     // rows per lane
  static constexpr int ROWS_W = RG * M;          // rows per warp
};
constexpr int kMaxWarps = 8;
constexpr int kMaxThreads = 32 * kMaxWarps;

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
// Waits for phase `parity` of the barrier; gives up after a bounded number of
// polls (each poll may itself suspend briefly) and returns false.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  constexpr int kMaxPolls = 1 << 22;
  for (int i = 0; i < kMaxPolls; ++i) {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    if (done) return true;
  }
  return false;
}

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

// ------------------------------------------------------------ the kernel
// Persistent clusters.  A "group" is one (request b, q/k head hq): the q and k
// rows of head hq and the G value heads h = hq G .. hq G + G - 1 that read
// them.  Its state is G * slices items of DVS state rows; CTA `rank` of a
// cluster of CS CTAs owns items rank*IPC .. rank*IPC + IPC - 1 (consecutive
// slices, so its v channels are one contiguous run).  Cluster c runs groups
// c, c + clusters, c + 2 clusters, ...
//
// Per group, each CTA first runs the conv + SiLU of its share of QS = d_k / CS
// q channels and the same share of k channels, and of the v channels of its
// items; it is the only reader of those channels' conv windows in the call, so
// it also writes the committed window (or the per-row windows).  It forms the
// partial dot products of its share that the L2 norms and the Gram tables need
// (q_t.q_t, k_s.k_t, k_s.q_t over QS channels).  After a cluster barrier each
// CTA sums the CS partials in rank order (every CTA ends with the same bits),
// forms the normalisation factors and the Gram tables k^_s.k^_t and
// k^_s.(scale q^_t), and copies every share's rows, scaled, out of its peers'
// shared memory into its own [R][scale q^ | k^] table.
//
// Inputs are staged by bulk async copies two groups ahead; each item's state
// slice is one bulk copy into a single buffer, requested as soon as the
// previous item's slice is in registers.
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

// Shared-memory layout of the kernel, in floats from the dynamic base (every
// region starts on 16 bytes), then two input stages of stage_bytes() each.
template <int DK>
struct Layout {
  int R, qs, ipc, es, DVS;
  __host__ __device__ int nd4() const { return (R + 2 * R * R + 3) & ~3; }
  __host__ __device__ int qk() const { return DVS * DK; }                 // [R][2 DK]       scale*q^ | k^
  __host__ __device__ int v() const { return qk() + R * 2 * DK; }         // [IPC][R][DVS]   v
  __host__ __device__ int gh() const { return v() + ipc * R * DVS; }      // [R][R][2]       k^.k^, k^.(scale q^)
  __host__ __device__ int ab() const { return gh() + gram_floats(R); }    // [2][IPC][R][2]  exp(g), beta
  __host__ __device__ int y() const { return ab() + 4 * ipc * R; }        // [R][2 QS]       conv output of the share
  __host__ __device__ int pd() const { return y() + R * 2 * qs; }         // [nd]            partial dot products
  __host__ __device__ int dot() const { return pd() + nd4(); }            // [nd]            summed dot products
  __host__ __device__ int stage() const { return dot() + nd4(); }
  // bytes within one input stage
  __host__ __device__ int st_w() const { return R * 2 * qs * es; }            // after [R][2 QS] x (q | k share)
  __host__ __device__ int st_cs() const { return st_w() + 2 * qs * kW * es; }  // after [2 QS][4] taps
  __host__ __device__ int st_xv() const { return st_cs() + 2 * qs * kWS * es; }  // after [2 QS][3] windows
  __host__ __device__ int st_wv() const { return st_xv() + R * ipc * DVS * es; }  // after [R][IPC DVS] v x
  __host__ __device__ int st_csv() const { return st_wv() + ipc * DVS * kW * es; }
  __host__ __device__ int stage_bytes() const { return st_csv() + ipc * DVS * kWS * es; }
  __host__ __device__ size_t bytes() const { return sizeof(float) * (size_t)stage() + 2 * (size_t)stage_bytes(); }
};

// ---- thread-block cluster ----
__device__ __forceinline__ int cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return (int)r;
}
__device__ __forceinline__ int cluster_index() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return (int)r;
}
__device__ __forceinline__ int cluster_total() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
  return (int)r;
}
// Arrive publishing this thread's earlier shared-memory writes to the cluster.
// The fence is restricted to shared memory, so global stores still in flight
// (committed state, o, windows) are not waited for, as a plain release would.
__device__ __forceinline__ void cluster_arrive_shared() {
  asm volatile(
      "fence.release.sync_restrict::shared::cta.cluster;\n\t"
      "barrier.cluster.arrive.relaxed.aligned;" ::
          : "memory");
}
// Arrive with no ordering: the thread's reads of its peers have completed.
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
// Wait for every thread of the cluster to arrive; acquires what they published.
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }
// the address of the same shared-memory location in CTA `rank` of the cluster
__device__ __forceinline__ uint32_t peer(const void* ptr, int rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_addr(ptr)), "r"(rank));
  return r;
}
__device__ __forceinline__ float ld_peer(uint32_t addr) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr));
  return v;
}
__device__ __forceinline__ float4 ld_peer4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr));
  return v;
}
// ---- asynchronous copies global -> shared (4 or 16 bytes), completed per thread by group ----
__device__ __forceinline__ void cp_async4(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_addr(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// all but the newest `N` committed groups of this thread have landed
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

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

template <int DK, typename T, int MODE>
__global__ void __launch_bounds__(kMaxThreads, 2) verify_kernel(const Params p) {
  using Gm = Geo<DK>;
  constexpr int LPR = Gm::LPR, NC4 = Gm::NC4, RG = Gm::RG, M = Gm::M;
  constexpr int ROWS_W = Gm::ROWS_W;
  const int NT = blockDim.x, DVS = p.dvs;
  constexpr int NP = 2 * NC4;  // column pairs per lane per row
  constexpr int CH = 4;        // rows per chunk
  constexpr int kDup = (LPR >> ilog2(M)) - 1;  // low lane bits that repeat a row's sums
  constexpr bool kWantO = MODE != kCommitReplay;
  constexpr bool kCommits = MODE == kFused || MODE == kCommitReplay;
  constexpr bool kReplay = MODE == kCommitReplay;
  constexpr bool kSnap = MODE == kVerifySnap;
  const uint32_t kSBytes = DVS * DK * sizeof(float);
  constexpr int ES = sizeof(T);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int R = p.R, qs = p.qs, ipc = p.ipc, cs = p.cs;
  const int nqk = 2 * qs, nv = ipc * DVS;
  const Layout<DK> L{R, qs, ipc, ES, DVS};
  extern __shared__ __align__(16) float smem[];
  float* const stS = smem;  // [DVS][DK] state slice of the next item
  float* const sQK = smem + L.qk();
  float* const sVall = smem + L.v();
  float* const sGH = smem + L.gh();
  float* const sABall = smem + L.ab();
  float* const sY = smem + L.y();
  float* const sPD = smem + L.pd();
  float* const sDot = smem + L.dot();
  unsigned char* const stage0 = reinterpret_cast<unsigned char*>(smem + L.stage());
  auto stage = [&](int s) { return stage0 + s * L.stage_bytes(); };
  __shared__ __align__(8) uint64_t barS;
  __shared__ int sMeta[3][3];  // group k's at [k % 3]: slot, rows to run, commit row (-1 none)
  __shared__ int sReq[3];      // request data of group k + 2, loaded by thread 0 at group k's start
  __shared__ int sIssued, sCons;  // state copies requested; consumed when a wait gave up

  // cluster coordinates are re-read where they are used rather than kept live
  // through the row recurrence
  const int K = cluster_index() < p.n_groups ? (p.n_groups - 1 - cluster_index()) / cluster_total() + 1 : 0;

  auto load_req = [&](int gi) {  // thread 0
    const int b = gi / p.H_qk;
    sReq[0] = p.n_rows[b];
    sReq[1] = p.slot_ids[b];
    sReq[2] = kCommits ? p.accept_len[b] : 0;
  };
  // thread 0: request data (n, slot, a) -> sMeta[k % 3]; reports a bad request once
  auto eval_req = [&](int k, int n, int slot, int a) {
    const int gi = cluster_index() + k * cluster_total();
    int* m = sMeta[k % 3];
    int report = 0;
    m[0] = slot;
    m[1] = request_rows_of<kCommits, kReplay>(p, n, slot, a, m[2], report);
    if (report && gi % p.H_qk == 0 && cluster_rank() == 0) flag(p.status, report);
  };
  // first channels of this CTA's q share, k share and v channels in group gi
  auto share = [&](int gi, long long& chq, long long& chk, long long& chv) {
    const int hq = gi % p.H_qk, rank = cluster_rank();
    chq = (long long)hq * DK + (long long)rank * qs;
    chk = (long long)p.H_qk * DK + chq;
    chv = 2LL * p.H_qk * DK + (long long)hq * p.G * p.d_v + (long long)rank * nv;
  };
  // a run of 16-byte chunks, chunk c issued by thread (base + c) % NT (NT a power of two)
  auto copy_run = [&](unsigned char* dst, const T* src, int bytes, int& base) {
    const int n = bytes >> 4;
    for (int c = (tid - base) & (NT - 1); c < n; c += NT)
      cp_async16(dst + 16 * c, reinterpret_cast<const unsigned char*>(src) + 16 * c);
    base += n;
  };
  // x rows and taps of group k into stage k & 1 (no request data needed: every row of x exists)
  auto issue_x = [&](int k) {
    const int gi = cluster_index() + k * cluster_total(), b = gi / p.H_qk;
    long long chq, chk, chv;
    share(gi, chq, chk, chv);
    const int bq = qs * ES, bv = nv * ES;
    const T* X = static_cast<const T*>(p.x) + (size_t)b * R * p.C;
    const T* Wt = static_cast<const T*>(p.conv_w);
    unsigned char* st = stage(k & 1);
    int base = 0;
    for (int t = 0; t < R; ++t) {
      copy_run(st + t * 2 * bq, X + t * p.C + chq, bq, base);
      copy_run(st + t * 2 * bq + bq, X + t * p.C + chk, bq, base);
      copy_run(st + L.st_xv() + t * bv, X + t * p.C + chv, bv, base);
    }
    copy_run(st + L.st_w(), Wt + chq * kW, kW * bq, base);
    copy_run(st + L.st_w() + kW * bq, Wt + chk * kW, kW * bq, base);
    copy_run(st + L.st_wv(), Wt + chv * kW, kW * bv, base);
  };
  // committed conv windows of group k (after its request data: none for a request that runs no rows)
  auto issue_cs = [&](int k) {
    const int* m = sMeta[k % 3];
    if (m[1] == 0) return;
    long long chq, chk, chv;
    share(cluster_index() + k * cluster_total(), chq, chk, chv);
    const int bq = qs * ES, bv = nv * ES;
    const T* csr = static_cast<const T*>(p.conv_state) + (size_t)m[0] * p.C * kWS;
    unsigned char* st = stage(k & 1);
    int base = 0;
    copy_run(st + L.st_cs(), csr + chq * kWS, kWS * bq, base);
    copy_run(st + L.st_cs() + kWS * bq, csr + chk * kWS, kWS * bq, base);
    copy_run(st + L.st_csv(), csr + chv * kWS, kWS * bv, base);
  };
  // thread 0: item i of group k's state slice into the state buffer (one bulk copy)
  auto issue_state = [&](int k, int i) {
    const int* m = sMeta[k % 3];
    ++sIssued;
    if (m[1] == 0) {
      mbar_arrive(&barS);
      return;
    }
    const int gi = cluster_index() + k * cluster_total();
    const int hs = (gi % p.H_qk) * p.G * p.slices + cluster_rank() * ipc + i;  // h * slices + sl
    mbar_expect_tx(&barS, kSBytes);
    bulk_load(stS, p.S + ((size_t)m[0] * p.H_v * p.slices + hs) * DVS * DK, kSBytes, &barS);
  };
  // decay and write strength rows of the CTA's items in group k, into buffer k & 1; commits
  auto issue_ab = [&](int k) {
    if (k < K) {
      const int gi = cluster_index() + k * cluster_total(), rank = cluster_rank();
      const int b = gi / p.H_qk, hq = gi - b * p.H_qk;
      float* dst = sABall + (k & 1) * 2 * ipc * R;
      for (int j = tid; j < 2 * ipc * R; j += NT) {
        const int which = j & 1, t = (j >> 1) % R, i = (j >> 1) / R;
        const int h = hq * p.G + (rank * ipc + i) / p.slices;
        cp_async4(dst + j, (which ? p.beta : p.g) + ((size_t)b * R + t) * p.H_v + h);
      }
    }
    cp_async_commit();
  };

  // Copies in flight per thread, as commit groups: {x 0, ab 0}, {x 1}, {cs 0, cs 1},
  // then per group k: {ab k+1} at its start and {x k+2, cs k+2} after its prologue.
  // At group k's start that leaves group k's inputs behind at most 1 (k = 0) or
  // 2 newer groups.
  if (tid == 0) {
    sIssued = 0;
    mbar_init(&barS, 1);
  }
  pdl_wait();     // whatever ran before on the stream is complete and visible
  pdl_trigger();  // the next call may launch; it waits for this grid before reading
  // Start-up: the first two groups' request data (both loads in flight at
  // once), their x rows and taps meanwhile, then their windows, and only
  // then the first state slice, so the small loads are not queued behind it.
  int q0[3] = {0, 0, 0}, q1[3] = {0, 0, 0};
  if (tid == 0) {
    const int cid = cluster_index(), ncl = cluster_total();
    if (K > 0) {
      const int b = cid / p.H_qk;
      q0[0] = p.n_rows[b];
      q0[1] = p.slot_ids[b];
      q0[2] = kCommits ? p.accept_len[b] : 0;
    }
    if (K > 1) {
      const int b = (cid + ncl) / p.H_qk;
      q1[0] = p.n_rows[b];
      q1[1] = p.slot_ids[b];
      q1[2] = kCommits ? p.accept_len[b] : 0;
    }
  }
  if (K > 0) issue_x(0);
  issue_ab(0);
  if (K > 1) issue_x(1);
  cp_async_commit();
  if (tid == 0) {
    if (K > 0) eval_req(0, q0[0], q0[1], q0[2]);
    if (K > 1) eval_req(1, q1[0], q1[1], q1[2]);
  }
  __syncthreads();  // the barrier is initialised and the first groups' request data published
  if (K > 0) issue_cs(0);
  if (K > 1) issue_cs(1);
  cp_async_commit();
  if (tid == 0 && K > 0) issue_state(0, 0);

  const int c = lane & (LPR - 1);
  const int rg = lane / LPR;
  const int wrow = warp * ROWS_W + rg;  // slice-local row of m = 0; row m adds m * RG
  const int gbase = lane & ~(LPR - 1);
  const int rl = wrow + row_of_lane<LPR, M>(lane) * RG;  // the row whose sums this lane holds
  const bool writer = (lane & kDup) == 0;
  const size_t o_tstride = (size_t)p.H_v * p.d_v;

  // A wait that gives up sets `broken`: the CTA records how many state copies it
  // consumed, stops computing and requesting state, but keeps taking part in
  // the cluster's barriers.
  bool broken = false;
  for (int k = 0; k < K; ++k) {
    const int s = k & 1;
    const int gi = cluster_index() + k * cluster_total();
    const int b = gi / p.H_qk, hq = gi - b * p.H_qk;
    if (tid == 0 && k + 2 < K) load_req(gi + 2 * cluster_total());  // in flight during the prologue
    __syncthreads();  // the previous group's items are done with the tables, sV and sAB
    issue_ab(k + 1);
    if (k == 0)
      cp_async_wait<1>();  // this thread's copies of group k have landed
    else
      cp_async_wait<2>();
    if (k > 0) cluster_wait();  // every peer has finished reading this CTA's sY and sPD
    __syncthreads();            // every thread's copies of group k are visible
    const int slot = sMeta[k % 3][0], rows = sMeta[k % 3][1], crow = sMeta[k % 3][2];

    // ---- conv + SiLU of the CTA's channels; committed or per-row windows ----
    if (rows > 0) {
      const unsigned char* st = stage(s);
      const T* sx = reinterpret_cast<const T*>(st);
      const T* sw = reinterpret_cast<const T*>(st + L.st_w());
      const T* scw = reinterpret_cast<const T*>(st + L.st_cs());
      const T* sxv = reinterpret_cast<const T*>(st + L.st_xv());
      const T* swv = reinterpret_cast<const T*>(st + L.st_wv());
      const T* scv = reinterpret_cast<const T*>(st + L.st_csv());
      for (int j = tid; j < nqk + nv; j += NT) {
        const bool isv = j >= nqk;
        const int jj = isv ? j - nqk : j;
        const T* wp = (isv ? swv : sw) + jj * kW;
        const T* cw = (isv ? scv : scw) + jj * kWS;
        const T* xp = (isv ? sxv : sx) + jj;
        const int xs = isv ? nv : nqk;
        const int rank = cluster_rank();
        const long long ch = isv ? 2LL * p.H_qk * DK + (long long)hq * p.G * p.d_v + (long long)rank * nv + jj
                                 : (jj < qs ? (long long)hq * DK + (long long)rank * qs + jj
                                            : (long long)(p.H_qk + hq) * DK + (long long)rank * qs + (jj - qs));
        const float w0 = tof(wp[0]), w1 = tof(wp[1]), w2 = tof(wp[2]), w3 = tof(wp[3]);
        T r0 = cw[0], r1 = cw[1], r2 = cw[2];  // window, oldest first, kept as stored
        T c0 = r0, c1 = r1, c2 = r2;           // window after the commit row
        float* yd = isv ? sVall + (jj / DVS) * R * DVS + (jj % DVS) : sY + jj;
        const int ys = isv ? DVS : nqk;
        for (int t = 0; t < rows; ++t) {
          const T r3 = xp[t * xs];
          float z = __fmul_rn(w0, tof(r0));
          z = __fmaf_rn(w1, tof(r1), z);
          z = __fmaf_rn(w2, tof(r2), z);
          z = __fmaf_rn(w3, tof(r3), z);
          yd[t * ys] = silu(z);
          r0 = r1;
          r1 = r2;
          r2 = r3;
          if (kSnap) {
            T* sc = static_cast<T*>(p.snapCs) + (((size_t)b * R + t) * p.C + ch) * kWS;
            sc[0] = r0;
            sc[1] = r1;
            sc[2] = r2;
          }
          if (kCommits && t == crow) {
            c0 = r0;
            c1 = r1;
            c2 = r2;
          }
        }
        if (kCommits && crow >= 0 && !broken) {  // this thread is the channel's only reader in the call
          T* cs = static_cast<T*>(p.conv_state) + ((size_t)slot * p.C + ch) * kWS;
          cs[0] = c0;
          cs[1] = c1;
          cs[2] = c2;
        }
      }
    }
    __syncthreads();
    // ---- partial dot products of the share, packed in n-row order: entries
    // e < n are q_t.q_t, then pairs (s, t) at n + 2 (s n + t) + {0: k_s.k_t,
    // 1: k_s.q_t}; and exp(g) of the decay rows ----
    const int n = rows, nd = n + 2 * n * n;
    if (rows > 0) {
      // each entry over 4 adjacent lanes (quarters of the share, joined by two
      // shuffles in a fixed order); the trip count is the same for every lane
      const int nq = qs >> 2, quarter = tid & 3;
      for (int e0 = 0; e0 < nd; e0 += NT >> 2) {
        const int e = e0 + (tid >> 2);
        float acc = 0.f;
        if (e < nd) {
          const float* x0;
          const float* x1;
          if (e < n) {
            x0 = x1 = sY + e * nqk;
          } else {
            const int e2 = e - n, which = e2 & 1, s0 = (e2 >> 1) / n, t0 = (e2 >> 1) % n;
            x0 = sY + s0 * nqk + qs;
            x1 = sY + t0 * nqk + (which ? 0 : qs);
          }
          x0 += quarter * nq;
          x1 += quarter * nq;
          for (int j = 0; j < nq; ++j) acc = __fmaf_rn(x0[j], x1[j], acc);
        }
        acc = __fadd_rn(acc, __shfl_xor_sync(kFull, acc, 1));
        acc = __fadd_rn(acc, __shfl_xor_sync(kFull, acc, 2));
        if (e < nd && quarter == 0) sPD[e] = acc;
      }
      float* ab = sABall + s * 2 * ipc * R;
      for (int j = tid; j < ipc * R; j += NT) ab[2 * j] = expf(ab[2 * j]);
    }
    cluster_arrive_shared();  // the partials and the conv output of every CTA are published
    cluster_wait();
    if (rows > 0) {
      for (int e = tid; e < nd; e += NT) {
        float v[8];  // every peer's partial in flight at once, then summed in rank order
#pragma unroll
        for (int r = 0; r < 8; ++r) v[r] = r < cs ? ld_peer(peer(sPD + e, r)) : 0.f;
        float acc = 0.f;
#pragma unroll
        for (int r = 0; r < 8; ++r)
          if (r < cs) acc = __fadd_rn(acc, v[r]);
        sDot[e] = acc;
      }
    }
    __syncthreads();
    if (rows > 0) {
      auto fq = [&](int t) { return __fmul_rn(p.scale, rsqrtf(__fadd_rn(sDot[t], p.eps))); };
      auto fk = [&](int t) { return rsqrtf(__fadd_rn(sDot[n + 2 * (t * n + t)], p.eps)); };
      // Gram tables [R][R][2]: k^_s . k^_t and k^_s . (scale q^_t); rows past n are zero
      for (int i = tid; i < 2 * R * R; i += NT) {
        const int which = i & 1, s0 = (i >> 1) / R, t0 = (i >> 1) % R;
        float val = 0.f;
        if (s0 < n && t0 < n)
          val = __fmul_rn(__fmul_rn(sDot[n + 2 * (s0 * n + t0) + which], fk(s0)), which ? fq(t0) : fk(t0));
        sGH[i] = val;
      }
      // every share's rows, scaled: scale*q^ | k^
      constexpr int kChunks = 2 * DK / 4;
      constexpr int kBatch = 4;  // remote loads in flight per thread
      for (int j0 = tid; j0 < n * kChunks; j0 += kBatch * NT) {
        float4 v[kBatch];
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
          const int j = j0 + u * NT;
          if (j < n * kChunks) {
            const int t = j / kChunks, cc = (j - t * kChunks) * 4;
            const bool isk = cc >= DK;
            const int cq = isk ? cc - DK : cc;
            const int r = cq / qs, off = cq - r * qs + (isk ? qs : 0);
            v[u] = ld_peer4(peer(sY + t * nqk + off, r));
          }
        }
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
          const int j = j0 + u * NT;
          if (j < n * kChunks) {
            const int t = j / kChunks, cc = (j - t * kChunks) * 4;
            const float f = cc >= DK ? fk(t) : fq(t);
            *reinterpret_cast<float4*>(sQK + t * 2 * DK + cc) =
                make_float4(__fmul_rn(v[u].x, f), __fmul_rn(v[u].y, f), __fmul_rn(v[u].z, f), __fmul_rn(v[u].w, f));
          }
        }
      }
    }
    cluster_arrive_relaxed();  // this CTA has read what it needs from its peers; waited on at the next group
    if (tid == 0 && k + 2 < K) eval_req(k + 2, sReq[0], sReq[1], sReq[2]);
    __syncthreads();  // tables complete; stage s consumed; group k + 2's request data published
    if (k + 2 < K) {
      issue_x(k + 2);
      issue_cs(k + 2);
    }
    cp_async_commit();

    // ---- the CTA's items ----
    for (int i = 0; i < ipc; ++i) {
      if (!broken && __syncthreads_or(!mbar_wait(&barS, (k * ipc + i) & 1))) {
        broken = true;
        if (tid == 0) {
          flag(p.status, GDN_STATUS_TIMEOUT);
          sCons = k * ipc + i;
        }
      }
      const bool run = rows > 0 && !broken;
      f2 S[M][NP];  // column pairs of the lane's 4-column chunks
      if (run) {
#pragma unroll
        for (int m = 0; m < M; ++m)
#pragma unroll
          for (int j = 0; j < NC4; ++j) {
            const ulonglong2 v = *reinterpret_cast<const ulonglong2*>(stS + (wrow + m * RG) * DK + 4 * (c + LPR * j));
            S[m][2 * j] = v.x;
            S[m][2 * j + 1] = v.y;
          }
      }
      __syncthreads();  // the state buffer is free: request the next item's slice
      if (tid == 0 && !broken) {
        if (i + 1 < ipc) {
          fence_proxy_async();
          issue_state(k, i + 1);
        } else if (k + 1 < K) {
          fence_proxy_async();
          issue_state(k + 1, 0);
        }
      }
      if (!run) continue;

      const int item = cluster_rank() * ipc + i;
      const int h = hq * p.G + item / p.slices, sl = item % p.slices;
      const int hs = h * p.slices + sl;
      const float* sV = sVall + i * R * DVS;
      const float* sAB = sABall + (s * ipc + i) * 2 * R;
      float* Sg = p.S + ((size_t)slot * p.H_v * p.slices + hs) * DVS * DK;
      float* og = nullptr;
      if (kWantO) og = p.o + ((size_t)b * R * p.H_v + h) * p.d_v + (size_t)sl * DVS + rl;

      // lane's column pairs of row vector t (q at offset 0, k at offset DK)
      auto load_vec = [&](int t, int off, f2 (&vv)[NP]) {
        const ulonglong2* vp = reinterpret_cast<const ulonglong2*>(sQK + t * 2 * DK + off);
#pragma unroll
        for (int j = 0; j < NC4; ++j) {
          const ulonglong2 v = vp[c + LPR * j];
          vv[2 * j] = v.x;
          vv[2 * j + 1] = v.y;
        }
      };
      // dst[m] = cc * S[m] + sum_{s<nt} w_s(row m) k_{c0+s}, in that order; in place when dst is S
      auto combine = [&](int c0, int nt, float cc, const float (&w)[CH], bool in_place, float* out) {
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
              load_vec(c0 + x, DK, kv);
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
                load_vec(c0 + x, DK, kv);
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
            const float2 ab = *reinterpret_cast<const float2*>(sAB + 2 * (c0 + t));  // exp(g), beta
            cdec = __fmul_rn(cdec, ab.x);
            float r = __fmul_rn(cdec, pk[t]);
#pragma unroll
            for (int x = 0; x < CH; ++x)
              if (x < t) {
                z[x] = __fmul_rn(z[x], ab.x);
                r = __fmaf_rn(z[x], sGH[((c0 + x) * R + (c0 + t)) * 2], r);
              }
            z[t] = __fmul_rn(ab.y, __fsub_rn(sV[(c0 + t) * DVS + rl], r));
            if constexpr (kWantO) {
              float oo = __fmul_rn(cdec, pq[t]);
#pragma unroll
              for (int x = 0; x < CH; ++x)
                if (x <= t) oo = __fmaf_rn(z[x], sGH[((c0 + x) * R + (c0 + t)) * 2 + 1], oo);
              if (writer) og[(size_t)(c0 + t) * o_tstride] = oo;
            }
            if (kCommits && c0 + t == crow) {
#pragma unroll
              for (int x = 0; x < CH; ++x) zc[x] = x <= t ? z[x] : 0.f;
              ccom = cdec;
              ncom = t + 1;
            }
            if (kSnap)
              combine(c0, t + 1, cdec, z, false,
                      p.snapS + (((size_t)b * R + c0 + t) * p.H_v * p.slices + hs) * DVS * DK);
          }
        }
        // ---- commit: S_a = C_a S0 + sum_{s<=a} z_s k_s^T ----
        if (kCommits && ncom > 0) {
          if (last) {
            combine(c0, ncom, ccom, zc, true, nullptr);
            store_state(Sg);
          } else {
            combine(c0, ncom, ccom, zc, false, Sg);
          }
        }
        // ---- advance the state to the chunk's end when rows follow ----
        if (!last) combine(c0, nc, cdec, z, true, nullptr);
      }
    }
  }
  if (K > 0) cluster_wait();  // no peer reads this CTA's shared memory after it exits
  cp_async_wait<0>();
  if (broken && tid == 0)  // let a state copy still in flight land before leaving (bounded)
    for (int ph = sCons; ph < sIssued; ++ph) mbar_wait(&barS, ph & 1);
}

// Snapshot commit: slot <- scratch row accept_len[b] (state and conv window).
template <typename T>
__global__ void __launch_bounds__(256) snapshot_commit_kernel(const Params p) {
  pdl_wait();  // the snapshot verify before it is complete and visible
  const int b = blockIdx.y;
  const int slot = p.slot_ids[b], n = p.n_rows[b];
  int a = p.accept_len[b], report;
  const int t_end = request_rows_of<true, true>(p, n, slot, a, a, report);
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

// The kernel asks for the largest shared-memory carveout, so the next call's
// CTAs (launched early by programmatic dependent launch) find SMs configured
// alike and can become resident while this call's CTAs drain.
template <typename Kernel>
int prefer_max_shared(Kernel kernel) {
  return cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                              (int)cudaSharedmemCarveoutMaxShared) == cudaSuccess
             ? GDN_OK
             : GDN_ERR_LAUNCH;
}

// Persistent grid: as many clusters as fit at once (at most one per group).
template <int DK, typename T, int MODE>
int launch_verify(const Params& p, cudaStream_t st) {
  auto kernel = verify_kernel<DK, T, MODE>;
  const size_t smem = Layout<DK>{p.R, p.qs, p.ipc, (int)sizeof(T), p.dvs}.bytes();
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.cs);
  cfg.blockDim = dim3(32 * p.nw);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = p.cs;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  struct Cache {
    int dev = -1;
    size_t smem = 0;
    int cs = 0, nw = 0;
    int clusters = 0;  // resident clusters on the device for this shape
  };
  static Cache cache;  // per instantiation
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return GDN_ERR_LAUNCH;
  if (cache.dev != dev || cache.smem != smem || cache.cs != p.cs || cache.nw != p.nw) {
    if (prefer_max_shared(kernel) != GDN_OK) return GDN_ERR_LAUNCH;
    if (smem > 48 * 1024 &&
        cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
      return GDN_ERR_LAUNCH;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) != cudaSuccess || n < 1) return GDN_ERR_LAUNCH;
    cache.dev = dev;
    cache.smem = smem;
    cache.cs = p.cs;
    cache.nw = p.nw;
    cache.clusters = n;
  }
  const int ncl = p.n_groups < cache.clusters ? p.n_groups : cache.clusters;
  cfg.gridDim = dim3(ncl * p.cs);
  if (cudaLaunchKernelEx(&cfg, kernel, p) != cudaSuccess) return GDN_ERR_LAUNCH;
  return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_LAUNCH;
}

template <typename T, int MODE>
int dispatch(const Params& p, cudaStream_t st) {
  switch (p.d_k) {
    case 16:
      return launch_verify<16, T, MODE>(p, st);
    case 32:
      return launch_verify<32, T, MODE>(p, st);
    case 64:
      return launch_verify<64, T, MODE>(p, st);
    default:
      return launch_verify<128, T, MODE>(p, st);
  }
}

template <int MODE>
int run_mode(const Params& p, int in_dtype, cudaStream_t st) {
  return in_dtype == GDN_DTYPE_BF16 ? dispatch<__nv_bfloat16, MODE>(p, st) : dispatch<float, MODE>(p, st);
}

inline bool aligned(const void* ptr, size_t a) { return (reinterpret_cast<uintptr_t>(ptr) % a) == 0; }

// d_v must be a multiple of this (two warps of state rows at the smallest d_k)
inline int d_v_unit(int d_k) { return d_k >= 32 ? 32 : 16; }
inline int rows_per_warp(int d_k) {
  return d_k >= 64 ? Geo<64>::ROWS_W : (d_k == 32 ? Geo<32>::ROWS_W : Geo<16>::ROWS_W);
}

// Cluster shape of a call: CS CTAs per (request, q/k head) group, each taking
// QS = d_k / CS q (and k) channels and IPC = G * slices / CS state items.  CS
// is the largest power of two <= 8 that divides the group's items and keeps
// every share's copies whole 16-byte runs.
inline int cluster_size(int d_k, int items, int es) {
  for (int cs = 8; cs > 1; cs >>= 1)
    if (items % cs == 0 && (d_k / cs) * es % 16 == 0) return cs;
  return 1;
}

// Dynamic shared memory of one CTA (0 if d_k is not built).
inline size_t layout_bytes(int d_k, int R, int qs, int ipc, int es, int dvs) {
  switch (d_k) {
    case 16:
      return Layout<16>{R, qs, ipc, es, dvs}.bytes();
    case 32:
      return Layout<32>{R, qs, ipc, es, dvs}.bytes();
    case 64:
      return Layout<64>{R, qs, ipc, es, dvs}.bytes();
    case 128:
      return Layout<128>{R, qs, ipc, es, dvs}.bytes();
    default:
      return 0;
  }
}
constexpr size_t kMaxSmem = 227 * 1024;  // opt-in shared memory per block on sm_103

struct Plan {
  int nw, dvs, slices, cs, qs, ipc;
};
// Item and cluster shape of a call.  Warps per CTA: the most (8, 4, 2, 1) whose
// slice of state rows divides d_v and whose CTA fits in shared memory while
// the call still has at least one item per SM; a call with fewer items than
// SMs takes the fewest warps (the most, smallest items).  False if no shape fits.
inline bool plan_call(const gdn_args* a, int sms, Plan* out) {
  const int es = a->in_dtype == GDN_DTYPE_BF16 ? 2 : 4;
  const int G = a->H_v / a->H_qk, rw = rows_per_warp(a->d_k);
  bool have_best = false, have_any = false;
  Plan best{}, last{};
  for (int nw = kMaxWarps; nw >= 1; nw >>= 1) {
    Plan q;
    q.nw = nw;
    q.dvs = nw * rw;
    if (a->d_v % q.dvs != 0) continue;
    q.slices = a->d_v / q.dvs;
    q.cs = cluster_size(a->d_k, G * q.slices, es);
    q.qs = a->d_k / q.cs;
    q.ipc = G * q.slices / q.cs;
    const size_t smem = layout_bytes(a->d_k, a->R, q.qs, q.ipc, es, q.dvs);
    if (smem == 0 || smem > kMaxSmem) continue;
    last = q;
    have_any = true;
    if (!have_best && (long long)a->B * a->H_v * q.slices >= sms) {
      best = q;
      have_best = true;
    }
  }
  if (!have_any) return false;
  *out = have_best ? best : last;
  return true;
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
  if (a->flags != 0) return GDN_ERR_INVALID_ARG;
  if (a->in_dtype != GDN_DTYPE_BF16 && a->in_dtype != GDN_DTYPE_F32) return GDN_ERR_UNSUPPORTED;
  if (a->W != kW || a->R > kMaxR) return GDN_ERR_UNSUPPORTED;
  if (a->d_k != 16 && a->d_k != 32 && a->d_k != 64 && a->d_k != 128) return GDN_ERR_UNSUPPORTED;
  if (a->d_v % d_v_unit(a->d_k) != 0) return GDN_ERR_UNSUPPORTED;
  if (a->H_v % a->H_qk != 0) return GDN_ERR_UNSUPPORTED;
  if (a->B > 65535) return GDN_ERR_UNSUPPORTED;
  if ((long long)a->H_v * a->d_v > 0x7fffffffLL) return GDN_ERR_UNSUPPORTED;
  Plan plan;
  if (!plan_call(a, 1, &plan)) return GDN_ERR_UNSUPPORTED;
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

int validate(const gdn_args* a, unsigned need, Params* out) {
  int rc = check_shape(a);
  if (rc != GDN_OK) return rc;
  if (!std::isfinite(a->scale) || !std::isfinite(a->l2_eps) || a->l2_eps < 0.f) return GDN_ERR_INVALID_ARG;

  if (!a->conv_state || !a->ssm_state || !a->slot_ids || !a->n_rows) return GDN_ERR_INVALID_ARG;
  if (!aligned(a->conv_state, 16) || !aligned(a->ssm_state, 16) || !aligned(a->slot_ids, 4) ||
      !aligned(a->n_rows, 4))
    return GDN_ERR_MISALIGNED;
  if (need & kNeedRows) {
    if (!a->x || !a->g || !a->beta || !a->conv_w || !a->work) return GDN_ERR_INVALID_ARG;
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
  p.n_groups = a->B * a->H_qk;
  p.status = a->status;
  return GDN_OK;
}

// SMs of the current device (cached per device; 0 on error).
int sm_count() {
  static std::atomic<int> cached[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  int n = cached[dev].load(std::memory_order_relaxed);
  if (n == 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    cached[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

int run_rows(const gdn_args* args, unsigned need, int mode, void* stream) {
  Params p;
  const int rc = validate(args, need, &p);
  if (rc != GDN_OK || p.B == 0) return rc;
  const int sms = sm_count();
  Plan plan;
  if (sms == 0) return GDN_ERR_LAUNCH;
  if (!plan_call(args, sms, &plan)) return GDN_ERR_UNSUPPORTED;
  p.nw = plan.nw;
  p.dvs = plan.dvs;
  p.slices = plan.slices;
  p.cs = plan.cs;
  p.qs = plan.qs;
  p.ipc = plan.ipc;
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
