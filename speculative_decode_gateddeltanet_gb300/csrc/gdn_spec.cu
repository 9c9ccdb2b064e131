// GatedDeltaNet speculative verify / commit kernels for sm_103a.
//
// Work split.  One CTA owns one (request b, value head h, slice of DVS state
// rows).  Its slice of the fp32 state S (DVS x d_k, d_k contiguous) is loaded
// once with 128-bit loads into registers and stays there across all k+1
// rows.  The CTAs that share a q/k head (G value heads x slices) form
// thread-block clusters of up to 8: each convolves only its share of the q
// and k channels, and the shares and the partial sums of the L2 norms are
// read back from the peers' shared memory, so the q/k conv is done once per
// cluster instead of once per CTA.  A CTA's conv inputs (x rows, committed
// window, taps of its channels) arrive in one batch of bulk async copies.
// The conv spec-update reads only the committed window and the verify rows,
// staging [history | verify inputs] per channel [FreeToken #844 "MTP drafts
// for Qwen3.5 family + Flash-Next", Design / Flash-Next target verify].
//
// Per row t each warp runs (alpha = exp(g_t), fp32, packed f32x2 arithmetic):
//   r = S k, p = S q~           (q~ = scale * q)       dot products on the old S
//   u = beta (v - alpha r)
//   o = alpha p + u (k . q~)    = scale * S_t q
//   S <- alpha S + u k^T
// which is the gated delta rule S_t = alpha S + beta (v - alpha S k) k^T,
// o_t = scale S_t q.  Lanes own 4-float column chunks of two rows; a row's
// dot products are reduced over its 8 (d_k >= 32) or 4 (d_k = 16) lanes
// with a reduce-scatter butterfly, so each lane ends up with one finished
// sum.  The arithmetic of a row does not depend on the mode, on how many rows
// the call has or on which rows follow, so a fused call, a verify followed by
// a replay commit, and a chain of one-row calls give the same bits.
//
// Modes: verify (o only; the state is only read [FreeToken #828
// "Speculative decoding: MTP and DFlash", Design]), verify with per-row
// snapshots (the widened verify state of [LightLLM #1330 "Qwen3.5 /
// Qwen3.5-MoE MTP speculative decoding", Summary]), replay commit (rows
// 0..a rerun from the slot, then written once), and fused verify + commit
// (the slot is written at row a from the registers: one read and one write
// of the state per request, the verify-and-commit kernel mode of [lmdeploy
// #5006 "speculative decoding for TurboMind", Verification path]).
//
// Conv-state ownership.  Each q/k channel share is read by one CTA per
// cluster.  When one cluster covers the whole q/k head that CTA is the only
// reader and commits the share's window itself; otherwise the last of the
// readers to arrive (an atomic count per (request, q/k head, share), reset
// by that CTA) writes it.  No CTA waits on another except at its cluster's
// hardware barriers.  v channels have a single reader.
#include <cooperative_groups.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <cmath>

#include "gdnspec.h"

namespace cg = cooperative_groups;

namespace gdnspec {

constexpr int kW = 4;        // conv width the kernels are built for
constexpr int kWS = kW - 1;  // conv-state columns
constexpr int kMaxR = 16;    // rows per request (k <= 15)
constexpr int kMaxCluster = GDN_COUNTERS_PER_QK_HEAD;
constexpr unsigned kFull = 0xffffffffu;

enum Mode : int { kFused = 0, kVerify = 1, kVerifySnap = 2, kCommitReplay = 3 };

struct Params {
  int B, R, H_qk, H_v, d_k, d_v, P, G, slices;
  int cs;               // CTAs per cluster (share the q/k conv of one q/k head)
  int clusters_per_qk;  // clusters per (request, q/k head) = readers of each share
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
  int* counters;
  int* status;
};

// Lane geometry for a d_k-column state.
template <int DK>
struct Geo {
  static constexpr int LPR = DK >= 32 ? 8 : 4;   // lanes per state row
  static constexpr int NC4 = DK / (4 * LPR);     // 4-column chunks per lane per row
  static constexpr int RG = 32 / LPR;            // row groups per warp
  static constexpr int M = 2;                    // rows per lane
  static constexpr int ROWS_W = RG * M;          // rows per warp
  static constexpr int NW = DK >= 32 ? 4 : 1;    // warps per CTA
  static constexpr int DVS = NW * ROWS_W;        // state rows per CTA
  static constexpr int NT = NW * 32;
  static constexpr int MIN_CTAS = DK >= 32 ? 5 : 16;  // resident CTAs per SM the registers must allow
};

__host__ __device__ constexpr int ilog2(int v) { return v <= 1 ? 0 : 1 + ilog2(v / 2); }

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

__device__ __forceinline__ float silu(float z) { return __fdiv_rn(z, __fadd_rn(1.0f, expf(-z))); }

// Sum each of a lane's V values over the LPR lanes of its row group.  The
// first log2(V) butterfly levels halve the values a lane carries (it keeps
// one half and trades the other), the remaining levels are all-reduce steps.
// On return the lane holds the finished sum of value `idx`.  The summation
// tree of a value (partners at LPR/2, LPR/4, .., 1) is the same for every V.
template <int LPR, int V>
__device__ __forceinline__ float reduce_scatter(float (&v)[V], int lane, int& idx) {
  constexpr int kHalvings = ilog2(V);
  static_assert((1 << kHalvings) == V && V <= LPR, "V must be a power of two <= LPR");
  idx = 0;
#pragma unroll
  for (int l = 0; l < kHalvings; ++l) {
    const int off = LPR >> (l + 1);
    const int half = V >> (l + 1);
    const bool up = (lane & off) != 0;
#pragma unroll
    for (int i = 0; i < half; ++i) {
      const float send = up ? v[i] : v[i + half];
      const float keep = up ? v[i + half] : v[i];
      v[i] = __fadd_rn(keep, __shfl_xor_sync(kFull, send, off));
    }
    if (up) idx += half;
  }
#pragma unroll
  for (int off = LPR >> (kHalvings + 1); off >= 1; off >>= 1)
    v[0] = __fadd_rn(v[0], __shfl_xor_sync(kFull, v[0], off));
  return v[0];
}

// Offset, within a row group, of a lane that holds value `idx` after
// reduce_scatter<LPR, V>.
template <int LPR, int V>
__device__ __forceinline__ int value_lane(int idx) {
  int off = 0;
#pragma unroll
  for (int l = 0; (V >> (l + 1)) >= 1; ++l)
    if ((idx / (V >> (l + 1))) & 1) off |= LPR >> (l + 1);
  return off;
}

__device__ __forceinline__ void flag(int* status, int bit) {
  if (status) atomicOr(status, bit);
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
// Cluster barrier halves: every thread of every CTA of the cluster arrives;
// wait returns once all have arrived (a hardware barrier; the CTAs of a
// cluster are always resident together).
__device__ __forceinline__ void cluster_arrive() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }

// Shared-memory plan of one CTA.  QS = d_k / cluster size q (and k) channels
// are convolved here, NL = 2 QS + DVS channels in all.
//   xs  [R][NL] T      staged x rows: q share | k share | v slice
//   css [NL][3] T      staged committed window of the same channels
//   ws  [NL][4] T      staged conv taps
//   yq, yk [R][QS] f32 raw conv outputs of the shares (read by the peers)
//   part [R][4] f32    partial sums y_q^2, y_k^2, y_q.y_k over the share (read by the peers)
//   sQ, sK [R][DK] f32 scale * q^, k^;   sV [R][DVS] f32 v slice
//   sA, sBt, sKQ, sFq, sFk [kMaxR]  exp(g), beta, k^ . (scale q^), norm factors
template <int DK>
struct Plan {
  static constexpr int DVS = Geo<DK>::DVS;
  __host__ __device__ static int NL(int qs) { return 2 * qs + DVS; }
  __host__ __device__ static size_t staged(int R, int qs, int es) {
    return (size_t)(R * NL(qs) + NL(qs) * kWS + NL(qs) * kW) * es;
  }
  __host__ __device__ static size_t total(int R, int qs, int es) {
    return staged(R, qs, es) +
           sizeof(float) * ((size_t)2 * R * qs + 4 * (size_t)R + (size_t)2 * R * DK + (size_t)R * DVS + 5 * kMaxR);
  }
};

template <int DK, typename T, int MODE>
__global__ void __launch_bounds__(Geo<DK>::NT, Geo<DK>::MIN_CTAS) rows_kernel(const Params p) {
  using Gm = Geo<DK>;
  constexpr int LPR = Gm::LPR, NC4 = Gm::NC4, RG = Gm::RG, M = Gm::M, NW = Gm::NW;
  constexpr int DVS = Gm::DVS, NT = Gm::NT, ROWS_W = Gm::ROWS_W;
  constexpr int ES = sizeof(T);
  constexpr bool kWantO = MODE != kCommitReplay;
  constexpr bool kCommits = MODE == kFused || MODE == kCommitReplay;
  constexpr bool kSnap = MODE == kVerifySnap;
  constexpr int V = kWantO ? 2 * M : M;
  constexpr int kDupMask = (LPR >> ilog2(V)) - 1;  // lanes that repeat a finished sum

  cg::cluster_group cluster = cg::this_cluster();
  const int b = blockIdx.y;
  const int h = blockIdx.x / p.slices;
  const int sl = blockIdx.x - h * p.slices;
  const int hq = h / p.G;
  const int crank = (int)cluster.block_rank();  // == blockIdx.x % p.cs
  const int QS = DK / p.cs;                     // q (and k) channels convolved here
  const int NL = 2 * QS + DVS;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const bool reporter = h == 0 && sl == 0 && tid == 0;

  // ---- request validity (uniform over the cluster: it shares b) ----
  const int n = p.n_rows[b];
  if (n == 0) return;
  const int slot = p.slot_ids[b];
  if (slot < 0 || slot >= p.P) {
    if (reporter) flag(p.status, GDN_STATUS_BAD_SLOT);
    return;
  }
  if (n < 0 || n > p.R) {
    if (reporter) flag(p.status, GDN_STATUS_BAD_NROWS);
    return;
  }
  int a = -1;
  bool commit = false;
  if (kCommits) {
    a = p.accept_len[b];
    commit = a >= 0 && a < n;
    if (!commit) {
      if (reporter) flag(p.status, GDN_STATUS_BAD_ACCEPT);
      if (MODE == kCommitReplay) return;
    }
  }
  const int t_end = MODE == kCommitReplay ? a + 1 : n;

  // ---- state slice -> registers (issued first so it overlaps the staging) ----
  const int c = lane & (LPR - 1);
  const int rg = lane / LPR;
  const int wrow = warp * ROWS_W + rg;  // slice-local row of m = 0; row m adds m * RG
  const size_t head_elems = (size_t)p.d_v * DK;
  float* Sg = p.S + ((size_t)slot * p.H_v + h) * head_elems + (size_t)sl * DVS * DK;
  f2 S[M][2 * NC4];  // column pairs of the lane's 4-column chunks
#pragma unroll
  for (int m = 0; m < M; ++m)
#pragma unroll
    for (int j = 0; j < NC4; ++j) {
      const ulonglong2 v =
          *reinterpret_cast<const ulonglong2*>(Sg + (size_t)(wrow + m * RG) * DK + 4 * (c + LPR * j));
      S[m][2 * j] = v.x;
      S[m][2 * j + 1] = v.y;
    }

  // ---- shared memory ----
  extern __shared__ __align__(16) unsigned char smem[];
  T* xs = reinterpret_cast<T*>(smem);
  T* css = xs + (size_t)p.R * NL;
  T* ws = css + NL * kWS;
  float* yq = reinterpret_cast<float*>(ws + NL * kW);
  float* yk = yq + p.R * QS;
  float* part = yk + p.R * QS;
  float* sQ = part + 4 * p.R;
  float* sK = sQ + p.R * DK;
  float* sV = sK + p.R * DK;
  float* sA = sV + p.R * DVS;
  float* sBt = sA + kMaxR;
  float* sKQ = sBt + kMaxR;
  float* sFq = sKQ + kMaxR;
  float* sFk = sFq + kMaxR;
  __shared__ __align__(8) uint64_t bar;
  __shared__ int sOk;     // this CTA's staging completed (read by the peers)
  __shared__ int sAllOk;  // every CTA of the cluster staged its inputs
  __shared__ int sLast;

  // first channel of each staged block: q share, k share, v slice
  const long long ch_q = (long long)hq * DK + (long long)crank * QS;
  const long long ch_k = (long long)p.H_qk * DK + ch_q;
  const long long ch_v = 2LL * p.H_qk * DK + (long long)h * p.d_v + (long long)sl * DVS;
  const T* xg = static_cast<const T*>(p.x) + (size_t)b * p.R * p.C;
  const T* wg = static_cast<const T*>(p.conv_w);
  T* csg = static_cast<T*>(p.conv_state) + (size_t)slot * p.C * kWS;

  // ---- stage the rows, the committed window and the taps: one batch of bulk copies ----
  if (tid == 0) mbar_init(&bar, 1);
  __syncthreads();
  if (warp == 0) {
    if (lane == 0) mbar_expect_tx(&bar, (uint32_t)((t_end * NL + NL * kWS + NL * kW) * ES));
    __syncwarp();
    for (int i = lane; i < 3 * t_end + 6; i += 32) {
      const int blk = i < 3 * t_end ? i % 3 : (i - 3 * t_end) % 3;
      const long long base = blk == 0 ? ch_q : (blk == 1 ? ch_k : ch_v);
      const int off = blk * QS;  // block offset within this CTA's channel list
      const int len = blk == 2 ? DVS : QS;
      if (i < 3 * t_end) {
        const int t = i / 3;
        bulk_load(xs + t * NL + off, xg + (size_t)t * p.C + base, len * ES, &bar);
      } else if (i < 3 * t_end + 3) {
        bulk_load(css + off * kWS, csg + base * kWS, len * kWS * ES, &bar);
      } else {
        bulk_load(ws + off * kW, wg + base * kW, len * kW * ES, &bar);
      }
    }
  }
  float g_t = 0.f, beta_t = 0.f;  // gating of row `tid`, loaded while the copies fly
  if (tid < t_end) {
    const size_t gi = ((size_t)b * p.R + tid) * p.H_v + h;
    g_t = __ldg(p.g + gi);
    beta_t = __ldg(p.beta + gi);
  }
  const bool late = !mbar_wait(&bar, 0);
  const bool ok = !__syncthreads_or(late);
  if (!ok) mbar_wait(&bar, 0);  // bounded: let copies still in flight land before going on

  // entry `idx` of channel ci's staged sequence [window | rows]
  auto seq_at = [&](int ci, int idx) -> T { return idx < kWS ? css[ci * kWS + idx] : xs[(idx - kWS) * NL + ci]; };

  // Each share has one reader per cluster; with one cluster per q/k head that
  // reader commits it, otherwise the share's last reader does (below).
  const bool direct_qk = p.clusters_per_qk == 1;
  const bool snap_qk = (blockIdx.x % (p.G * p.slices)) < p.cs;  // first cluster of the q/k head

  // ---- conv spec-update + SiLU of this CTA's channels over [history | rows] ----
  if (ok) {
    for (int ci = tid; ci < NL; ci += NT) {
      const bool is_v = ci >= 2 * QS;
      const long long ch = ci < QS ? ch_q + ci : (is_v ? ch_v + (ci - 2 * QS) : ch_k + (ci - QS));
      float* dst = ci < QS ? yq + ci : (is_v ? sV + (ci - 2 * QS) : yk + (ci - QS));
      const int dstride = is_v ? DVS : QS;
      const float w0 = tof(ws[ci * kW + 0]), w1 = tof(ws[ci * kW + 1]);
      const float w2 = tof(ws[ci * kW + 2]), w3 = tof(ws[ci * kW + 3]);
      float s0 = tof(css[ci * kWS + 0]), s1 = tof(css[ci * kWS + 1]), s2 = tof(css[ci * kWS + 2]);
      for (int t = 0; t < t_end; ++t) {
        const float s3 = tof(xs[t * NL + ci]);
        float z = __fmul_rn(w0, s0);
        z = __fmaf_rn(w1, s1, z);
        z = __fmaf_rn(w2, s2, z);
        z = __fmaf_rn(w3, s3, z);
        dst[t * dstride] = silu(z);
        s0 = s1;
        s1 = s2;
        s2 = s3;
        if (kSnap && (is_v || snap_qk)) {
          T* sc = static_cast<T*>(p.snapCs) + (((size_t)b * p.R + t) * p.C + ch) * kWS;
#pragma unroll
          for (int j = 0; j < kWS; ++j) sc[j] = seq_at(ci, t + 1 + j);  // window after row t, as stored
        }
      }
      if (kCommits && commit && (is_v || direct_qk)) {  // this CTA is the channel's only reader
#pragma unroll
        for (int j = 0; j < kWS; ++j) csg[ch * kWS + j] = seq_at(ci, a + 1 + j);
      }
    }
    if (tid < t_end) {
      sA[tid] = expf(g_t);
      sBt[tid] = beta_t;
    }
  }
  __syncthreads();
  // partial L2 sums of the share, one warp per row
  if (ok) {
    for (int t = warp; t < t_end; t += NW) {
      float sq = 0.f, sk = 0.f, qk = 0.f;
      for (int e = lane; e < QS; e += 32) {
        const float qv = yq[t * QS + e], kv = yk[t * QS + e];
        sq = __fmaf_rn(qv, qv, sq);
        sk = __fmaf_rn(kv, kv, sk);
        qk = __fmaf_rn(qv, kv, qk);
      }
#pragma unroll
      for (int off = 16; off >= 1; off >>= 1) {
        sq = __fadd_rn(sq, __shfl_xor_sync(kFull, sq, off));
        sk = __fadd_rn(sk, __shfl_xor_sync(kFull, sk, off));
        qk = __fadd_rn(qk, __shfl_xor_sync(kFull, qk, off));
      }
      if (lane == 0) {
        part[4 * t + 0] = sq;
        part[4 * t + 1] = sk;
        part[4 * t + 2] = qk;
      }
    }
  }
  if (tid == 0) sOk = ok;
  __syncthreads();
  cluster_arrive();  // #1: shares, partial sums and staging flags are visible cluster-wide
  cluster_wait();

  // ---- gather q^, k^ of the whole q/k head from the cluster ----
  if (tid == 0) {
    int all = 1;
    for (int r = 0; r < p.cs; ++r) all &= *cluster.map_shared_rank(&sOk, r);
    sAllOk = all;
    if (!all) flag(p.status, GDN_STATUS_TIMEOUT);
  }
  __syncthreads();
  const bool run = sAllOk != 0;
  if (run) {
    // per-row factors: every CTA adds the partial sums in rank order -> identical bits
    if (tid < t_end) {
      float sq = 0.f, sk = 0.f, qk = 0.f;
      for (int r = 0; r < p.cs; ++r) {
        const float* pr = cluster.map_shared_rank(part, r) + 4 * tid;
        sq = __fadd_rn(sq, pr[0]);
        sk = __fadd_rn(sk, pr[1]);
        qk = __fadd_rn(qk, pr[2]);
      }
      const float fq = __fmul_rn(p.scale, rsqrtf(__fadd_rn(sq, p.eps)));
      const float fk = rsqrtf(__fadd_rn(sk, p.eps));
      sFq[tid] = fq;
      sFk[tid] = fk;
      sKQ[tid] = __fmul_rn(__fmul_rn(qk, fq), fk);
    }
    __syncthreads();
    const int per_row4 = DK / 4;
    for (int i = tid; i < 2 * t_end * per_row4; i += NT) {
      const int which = i / (t_end * per_row4);
      const int rem = i - which * t_end * per_row4;
      const int t = rem / per_row4;
      const int j = (rem - t * per_row4) * 4;
      const int r = j / QS, jj = j - r * QS;
      const float4 v = *reinterpret_cast<const float4*>(cluster.map_shared_rank(which ? yk : yq, r) + t * QS + jj);
      const float f = which ? sFk[t] : sFq[t];
      *reinterpret_cast<float4*>((which ? sK : sQ) + t * DK + j) =
          make_float4(__fmul_rn(v.x, f), __fmul_rn(v.y, f), __fmul_rn(v.z, f), __fmul_rn(v.w, f));
    }
  }
  __syncthreads();
  cluster_arrive();  // #2: done reading the peers (waited for before exit)

  // ---- arrival of this share's reader (result used after the rows) ----
  int* cnt = p.counters + ((size_t)b * p.H_qk + hq) * kMaxCluster + crank;
  int prev = -1;
  if (kCommits && commit && run && !direct_qk && tid == 0) {
    __threadfence();
    prev = atomicAdd(cnt, 1);
  }

  // ---- the rows ----
  if (run) {
    float* og = nullptr;
    if (kWantO) og = p.o + ((size_t)b * p.R * p.H_v + h) * p.d_v + (size_t)sl * DVS;
    const size_t o_tstride = (size_t)p.H_v * p.d_v;
    const int gbase = lane & ~(LPR - 1);
    for (int t = 0; t < t_end; ++t) {
      const float alpha = sA[t], bt = sBt[t];
      const f2 alpha2 = pack2(alpha, alpha);
      const ulonglong2* k4 = reinterpret_cast<const ulonglong2*>(sK + t * DK);
      f2 kv[2 * NC4];
#pragma unroll
      for (int j = 0; j < NC4; ++j) {
        const ulonglong2 v = k4[c + LPR * j];
        kv[2 * j] = v.x;
        kv[2 * j + 1] = v.y;
      }
      float part_v[V];
#pragma unroll
      for (int m = 0; m < M; ++m) {
        f2 acc = fma2(S[m][0], kv[0], pack2(0.f, 0.f));
#pragma unroll
        for (int j = 1; j < 2 * NC4; ++j) acc = fma2(S[m][j], kv[j], acc);
        part_v[m] = sum2(acc);
      }
      if constexpr (kWantO) {
        const ulonglong2* q4 = reinterpret_cast<const ulonglong2*>(sQ + t * DK);
        f2 qv[2 * NC4];
#pragma unroll
        for (int j = 0; j < NC4; ++j) {
          const ulonglong2 v = q4[c + LPR * j];
          qv[2 * j] = v.x;
          qv[2 * j + 1] = v.y;
        }
#pragma unroll
        for (int m = 0; m < M; ++m) {
          f2 acc = fma2(S[m][0], qv[0], pack2(0.f, 0.f));
#pragma unroll
          for (int j = 1; j < 2 * NC4; ++j) acc = fma2(S[m][j], qv[j], acc);
          part_v[(M + m) % V] = sum2(acc);
        }
      }
      int idx;
      const float red = reduce_scatter<LPR, V>(part_v, lane, idx);
      const int mrow = idx % M;
      const int rloc = wrow + mrow * RG;
      // u is meaningful on the lanes holding an S k sum (idx < M)
      const float u = __fmul_rn(bt, __fsub_rn(sV[t * DVS + rloc], __fmul_rn(alpha, red)));
      if constexpr (kWantO) {
        const float up = __shfl_xor_sync(kFull, u, LPR / 2);  // u of the same row
        if (idx >= M && (c & kDupMask) == 0)
          og[(size_t)t * o_tstride + rloc] = __fmaf_rn(up, sKQ[t], __fmul_rn(alpha, red));
      }
#pragma unroll
      for (int m = 0; m < M; ++m) {
        const float um = __shfl_sync(kFull, u, gbase | value_lane<LPR, V>(m));
        const f2 u2 = pack2(um, um);
#pragma unroll
        for (int j = 0; j < 2 * NC4; ++j) S[m][j] = fma2(u2, kv[j], mul2(alpha2, S[m][j]));
      }

      if (kCommits && commit && t == a) {
#pragma unroll
        for (int m = 0; m < M; ++m)
#pragma unroll
          for (int j = 0; j < NC4; ++j)
            *reinterpret_cast<ulonglong2*>(Sg + (size_t)(wrow + m * RG) * DK + 4 * (c + LPR * j)) =
                make_ulonglong2(S[m][2 * j], S[m][2 * j + 1]);
      }
      if (kSnap) {
        float* Ss = p.snapS + (((size_t)b * p.R + t) * p.H_v + h) * head_elems + (size_t)sl * DVS * DK;
#pragma unroll
        for (int m = 0; m < M; ++m)
#pragma unroll
          for (int j = 0; j < NC4; ++j)
            *reinterpret_cast<ulonglong2*>(Ss + (size_t)(wrow + m * RG) * DK + 4 * (c + LPR * j)) =
                make_ulonglong2(S[m][2 * j], S[m][2 * j + 1]);
      }
    }
  }

  // ---- committed q/k share windows when several clusters read them ----
  if (kCommits && commit && run && !direct_qk) {
    if (tid == 0) {
      const bool last = prev == p.clusters_per_qk - 1;
      if (last) atomicExch(cnt, 0);
      sLast = last;
    }
    __syncthreads();
    if (sLast) {
      for (int ci = tid; ci < 2 * QS; ci += NT) {
        const long long ch = ci < QS ? ch_q + ci : ch_k + (ci - QS);
#pragma unroll
        for (int j = 0; j < kWS; ++j) csg[ch * kWS + j] = seq_at(ci, a + 1 + j);
      }
    }
  }
  cluster_wait();  // #2: peers have finished reading this CTA's shared memory
}

// Snapshot commit: slot <- scratch row accept_len[b] (state and conv window).
template <typename T>
__global__ void __launch_bounds__(256) snapshot_commit_kernel(const Params p) {
  const int b = blockIdx.y;
  const bool reporter = blockIdx.x == 0 && threadIdx.x == 0;
  const int n = p.n_rows[b];
  if (n == 0) return;
  const int slot = p.slot_ids[b];
  if (slot < 0 || slot >= p.P) {
    if (reporter) flag(p.status, GDN_STATUS_BAD_SLOT);
    return;
  }
  if (n < 0 || n > p.R) {
    if (reporter) flag(p.status, GDN_STATUS_BAD_NROWS);
    return;
  }
  const int a = p.accept_len[b];
  if (a < 0 || a >= n) {
    if (reporter) flag(p.status, GDN_STATUS_BAD_ACCEPT);
    return;
  }
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

template <int DK, typename T, int MODE>
int launch_mode(const Params& p, cudaStream_t st) {
  using Gm = Geo<DK>;
  const size_t smem = Plan<DK>::total(p.R, DK / p.cs, sizeof(T));
  if (smem > 48 * 1024) {
    static int attr_set_on = -1;  // device on which the opt-in was last made
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return GDN_ERR_LAUNCH;
    if (attr_set_on != dev) {
      if (cudaFuncSetAttribute(rows_kernel<DK, T, MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)smem > 100 * 1024 ? (int)smem : 100 * 1024) != cudaSuccess)
        return GDN_ERR_LAUNCH;
      attr_set_on = dev;
    }
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.H_v * p.slices, p.B);
  cfg.blockDim = dim3(Gm::NT);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = p.cs;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, rows_kernel<DK, T, MODE>, p) != cudaSuccess) return GDN_ERR_LAUNCH;
  return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_LAUNCH;
}

template <int DK, typename T>
int launch_rows(const Params& p, int mode, cudaStream_t st) {
  switch (mode) {
    case kFused:
      return launch_mode<DK, T, kFused>(p, st);
    case kVerify:
      return launch_mode<DK, T, kVerify>(p, st);
    case kVerifySnap:
      return launch_mode<DK, T, kVerifySnap>(p, st);
    default:
      return launch_mode<DK, T, kCommitReplay>(p, st);
  }
}

template <typename T>
int dispatch_rows(const Params& p, int mode, cudaStream_t st) {
  switch (p.d_k) {
    case 16:
      return launch_rows<16, T>(p, mode, st);
    case 32:
      return launch_rows<32, T>(p, mode, st);
    case 64:
      return launch_rows<64, T>(p, mode, st);
    default:
      return launch_rows<128, T>(p, mode, st);
  }
}

// ------------------------------------------------------------------ host
inline bool aligned(const void* ptr, size_t a) { return (reinterpret_cast<uintptr_t>(ptr) % a) == 0; }

inline int rows_per_cta(int d_k) { return d_k >= 32 ? Geo<32>::DVS : Geo<16>::DVS; }

// CTAs per cluster: the largest power of two <= 8 that divides the CTAs of one
// q/k head and keeps each CTA's q/k channel share a multiple of 16 bytes.
inline int cluster_size(int group, int d_k, int es) {
  int cs = kMaxCluster;
  while (cs > 1 && (group % cs != 0 || ((d_k / cs) * es) % 16 != 0)) cs >>= 1;
  return cs;
}

enum Need : unsigned {
  kNeedRows = 1u,  // x, g, beta, conv_w
  kNeedO = 2u,
  kNeedAccept = 4u,
  kNeedScratch = 8u,
  kNeedCounters = 16u
};

int validate(const gdn_args* a, unsigned need, Params* out) {
  if (!a) return GDN_ERR_INVALID_ARG;
  if (a->B < 0 || a->R < 1 || a->H_qk < 1 || a->H_v < 1 || a->d_k < 1 || a->d_v < 1 || a->W < 1 ||
      a->pool_slots < 1)
    return GDN_ERR_INVALID_ARG;
  if (a->flags != 0) return GDN_ERR_INVALID_ARG;
  if (a->in_dtype != GDN_DTYPE_BF16 && a->in_dtype != GDN_DTYPE_F32) return GDN_ERR_UNSUPPORTED;
  if (a->W != kW || a->R > kMaxR) return GDN_ERR_UNSUPPORTED;
  if (a->d_k != 16 && a->d_k != 32 && a->d_k != 64 && a->d_k != 128) return GDN_ERR_UNSUPPORTED;
  if (a->d_v % rows_per_cta(a->d_k) != 0) return GDN_ERR_UNSUPPORTED;
  if (a->H_v % a->H_qk != 0) return GDN_ERR_UNSUPPORTED;
  if (a->B > 65535) return GDN_ERR_UNSUPPORTED;
  if ((long long)a->H_v * (a->d_v / rows_per_cta(a->d_k)) > 0x7fffffffLL) return GDN_ERR_UNSUPPORTED;
  if (!std::isfinite(a->scale) || !std::isfinite(a->l2_eps) || a->l2_eps < 0.f) return GDN_ERR_INVALID_ARG;

  if (!a->conv_state || !a->ssm_state || !a->slot_ids || !a->n_rows) return GDN_ERR_INVALID_ARG;
  if (!aligned(a->conv_state, 16) || !aligned(a->ssm_state, 16) || !aligned(a->slot_ids, 4) ||
      !aligned(a->n_rows, 4))
    return GDN_ERR_MISALIGNED;
  if (need & kNeedRows) {
    if (!a->x || !a->g || !a->beta || !a->conv_w) return GDN_ERR_INVALID_ARG;
    if (!aligned(a->x, 16) || !aligned(a->conv_w, 16) || !aligned(a->g, 4) || !aligned(a->beta, 4))
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
  if (need & kNeedCounters) {
    if (!a->counters) return GDN_ERR_INVALID_ARG;
    if (!aligned(a->counters, 4)) return GDN_ERR_MISALIGNED;
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
  p.slices = a->d_v / rows_per_cta(a->d_k);
  p.cs = cluster_size(p.G * p.slices, a->d_k, a->in_dtype == GDN_DTYPE_BF16 ? 2 : 4);
  p.clusters_per_qk = p.G * p.slices / p.cs;
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
  p.counters = a->counters;
  p.status = a->status;
  return GDN_OK;
}

int run_rows(const gdn_args* args, unsigned need, int mode, void* stream) {
  Params p;
  const int rc = validate(args, need, &p);
  if (rc != GDN_OK || p.B == 0) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  return args->in_dtype == GDN_DTYPE_BF16 ? dispatch_rows<__nv_bfloat16>(p, mode, st)
                                          : dispatch_rows<float>(p, mode, st);
}

}  // namespace gdnspec

using namespace gdnspec;

extern "C" {

GDN_API int gdn_verify(const gdn_args* args, int mode, void* stream) {
  if (mode != GDN_REPLAY && mode != GDN_SNAPSHOT) return GDN_ERR_INVALID_ARG;
  const bool snap = mode == GDN_SNAPSHOT;
  return run_rows(args, kNeedRows | kNeedO | (snap ? kNeedScratch : 0u), snap ? kVerifySnap : kVerify, stream);
}

GDN_API int gdn_commit(const gdn_args* args, int mode, void* stream) {
  if (mode == GDN_REPLAY) return run_rows(args, kNeedRows | kNeedAccept | kNeedCounters, kCommitReplay, stream);
  if (mode != GDN_SNAPSHOT) return GDN_ERR_INVALID_ARG;
  Params p;
  const int rc = validate(args, kNeedAccept | kNeedScratch, &p);
  if (rc != GDN_OK || p.B == 0) return rc;
  const size_t per_req4 = (size_t)p.H_v * p.d_v * p.d_k / 4;
  int gx = (int)((per_req4 + 2047) / 2048);
  gx = gx < 1 ? 1 : (gx > 256 ? 256 : gx);
  const dim3 grid(gx, p.B);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (args->in_dtype == GDN_DTYPE_BF16)
    snapshot_commit_kernel<__nv_bfloat16><<<grid, 256, 0, st>>>(p);
  else
    snapshot_commit_kernel<float><<<grid, 256, 0, st>>>(p);
  return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_LAUNCH;
}

GDN_API int gdn_verify_commit(const gdn_args* args, void* stream) {
  return run_rows(args, kNeedRows | kNeedO | kNeedAccept | kNeedCounters, kFused, stream);
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
      return "misaligned pointer (x, conv_w, conv_state, ssm_state, scratch and o need 16 bytes; the "
             "int32 and g/beta arrays 4)";
    case GDN_ERR_LAUNCH:
      return "CUDA kernel launch failed";
    default:
      return "unknown gdnspec error code";
  }
}

}  // extern "C"
