// GatedDeltaNet speculative verify / commit kernels for sm_103a.
//
// One CTA owns one (request b, value head h, slice of DVS state rows).  Its
// slice of the fp32 state S (DVS x d_k, d_k contiguous) is loaded once with
// 128-bit loads into registers and stays there across all k+1 rows; the CTA
// also runs the width-4 causal conv + SiLU and the per-head L2 norm for the q,
// k channels of its q/k head and the v channels of its rows (the conv
// spec-update reads only the committed window and the verify rows, staging
// [history | verify inputs] per channel [FreeToken #844 "MTP drafts for
// Qwen3.5 family + Flash-Next", Design / Flash-Next target verify]).
//
// Per row t the warp-level step is (alpha = exp(g_t), all fp32):
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
// Conv-state ownership.  The q and k channels of a q/k head are read by all
// G * slices CTAs of that head.  In the commit modes the last of them to
// finish reading (an atomic arrival count per (request, q/k head), reset by
// that CTA) writes the committed window; nobody waits.  v channels have a
// single reader, which writes them itself.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <cmath>

#include "gdnspec.h"

namespace gdnspec {

constexpr int kW = 4;        // conv width the kernels are built for
constexpr int kWS = kW - 1;  // conv-state columns
constexpr int kMaxR = 16;    // rows per request (k <= 15)
constexpr unsigned kFull = 0xffffffffu;

enum Mode : int { kFused = 0, kVerify = 1, kVerifySnap = 2, kCommitReplay = 3 };

struct Params {
  int B, R, H_qk, H_v, d_k, d_v, P, G, slices;
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
  static constexpr int NC4 = DK / (4 * LPR);     // float4 column chunks per lane
  static constexpr int RG = 32 / LPR;            // row groups per warp
  static constexpr int M = 2;                    // rows per lane
  static constexpr int ROWS_W = RG * M;          // rows per warp
  static constexpr int NW = DK >= 32 ? 4 : 1;    // warps per CTA
  static constexpr int DVS = NW * ROWS_W;        // state rows per CTA
  static constexpr int NT = NW * 32;
};

__host__ __device__ constexpr int ilog2(int v) { return v <= 1 ? 0 : 1 + ilog2(v / 2); }

template <typename T>
__device__ __forceinline__ float ld_ro(const T* p);
template <>
__device__ __forceinline__ float ld_ro<float>(const float* p) { return __ldg(p); }
template <>
__device__ __forceinline__ float ld_ro<__nv_bfloat16>(const __nv_bfloat16* p) {
  return __bfloat162float(__ldg(p));
}
template <typename T>
__device__ __forceinline__ float ld_rw(const T* p);
template <>
__device__ __forceinline__ float ld_rw<float>(const float* p) { return *p; }
template <>
__device__ __forceinline__ float ld_rw<__nv_bfloat16>(const __nv_bfloat16* p) {
  return __bfloat162float(*p);
}
template <typename T>
__device__ __forceinline__ void st(T* p, float v);
template <>
__device__ __forceinline__ void st<float>(float* p, float v) { *p = v; }
template <>
__device__ __forceinline__ void st<__nv_bfloat16>(__nv_bfloat16* p, float v) {
  *p = __float2bfloat16_rn(v);  // exact: v came from a bf16
}

__device__ __forceinline__ float silu(float z) {
  return __fdiv_rn(z, __fadd_rn(1.0f, expf(-z)));
}

__device__ __forceinline__ float dot4(const float4 s, const float4 k, float acc) {
  acc = __fmaf_rn(s.x, k.x, acc);
  acc = __fmaf_rn(s.y, k.y, acc);
  acc = __fmaf_rn(s.z, k.z, acc);
  return __fmaf_rn(s.w, k.w, acc);
}

__device__ __forceinline__ float4 decay_add(const float4 s, float alpha, float u, const float4 k) {
  return make_float4(__fmaf_rn(u, k.x, __fmul_rn(alpha, s.x)), __fmaf_rn(u, k.y, __fmul_rn(alpha, s.y)),
                     __fmaf_rn(u, k.z, __fmul_rn(alpha, s.z)), __fmaf_rn(u, k.w, __fmul_rn(alpha, s.w)));
}

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

template <int DK, typename T, int MODE>
__global__ void __launch_bounds__(Geo<DK>::NT) rows_kernel(const Params p) {
  using Gm = Geo<DK>;
  constexpr int LPR = Gm::LPR, NC4 = Gm::NC4, RG = Gm::RG, M = Gm::M, NW = Gm::NW;
  constexpr int DVS = Gm::DVS, NT = Gm::NT, ROWS_W = Gm::ROWS_W;
  constexpr bool kWantO = MODE != kCommitReplay;
  constexpr bool kCommits = MODE == kFused || MODE == kCommitReplay;
  constexpr bool kSnap = MODE == kVerifySnap;
  constexpr int V = kWantO ? 2 * M : M;
  constexpr int kDupMask = (LPR >> ilog2(V)) - 1;  // lanes that repeat a finished sum

  const int b = blockIdx.y;
  const int h = blockIdx.x / p.slices;
  const int sl = blockIdx.x - h * p.slices;
  const int hq = h / p.G;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const bool reporter = h == 0 && sl == 0 && tid == 0;

  // ---- request validity (uniform over the CTA) ----
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

  // ---- state slice -> registers (issued first so it overlaps the prologue) ----
  const int c = lane & (LPR - 1);
  const int rg = lane / LPR;
  const int wrow = warp * ROWS_W + rg;  // slice-local row of m = 0; row m adds m * RG
  const size_t head_elems = (size_t)p.d_v * DK;
  float* Sg = p.S + ((size_t)slot * p.H_v + h) * head_elems + (size_t)sl * DVS * DK;
  float4 S[M][NC4];
#pragma unroll
  for (int m = 0; m < M; ++m)
#pragma unroll
    for (int j = 0; j < NC4; ++j)
      S[m][j] = *reinterpret_cast<const float4*>(Sg + (size_t)(wrow + m * RG) * DK + 4 * (c + LPR * j));

  // ---- shared memory ----
  extern __shared__ float4 smem4[];
  float* sQ = reinterpret_cast<float*>(smem4);  // [R][DK]  scale * q^
  float* sK = sQ + p.R * DK;                    // [R][DK]  k^
  float* sV = sK + p.R * DK;                    // [R][DVS] v of this slice
  float* sA = sV + p.R * DVS;                   // [kMaxR]  exp(g)
  float* sBt = sA + kMaxR;                      // [kMaxR]  beta
  float* sKQ = sBt + kMaxR;                     // [kMaxR]  k^ . (scale q^)
  float* sNew = sKQ + kMaxR;                    // [2*DK][kWS] committed q/k windows
  __shared__ int sLast;

  // ---- conv spec-update + SiLU over [history | rows] ----
  const T* xb = static_cast<const T*>(p.x) + (size_t)b * p.R * p.C;
  const T* cw = static_cast<const T*>(p.conv_w);
  T* cs = static_cast<T*>(p.conv_state) + (size_t)slot * p.C * kWS;
  const bool qk_snap_owner = (h % p.G) == 0 && sl == 0;
  constexpr int NCH = 2 * DK + DVS;
  for (int ci = tid; ci < NCH; ci += NT) {
    long long ch;
    float* dst;
    int dstride;
    if (ci < DK) {
      ch = (long long)hq * DK + ci;
      dst = sQ + ci;
      dstride = DK;
    } else if (ci < 2 * DK) {
      ch = (long long)p.H_qk * DK + (long long)hq * DK + (ci - DK);
      dst = sK + (ci - DK);
      dstride = DK;
    } else {
      ch = 2LL * p.H_qk * DK + (long long)h * p.d_v + (long long)sl * DVS + (ci - 2 * DK);
      dst = sV + (ci - 2 * DK);
      dstride = DVS;
    }
    const float w0 = ld_ro(cw + ch * kW + 0), w1 = ld_ro(cw + ch * kW + 1);
    const float w2 = ld_ro(cw + ch * kW + 2), w3 = ld_ro(cw + ch * kW + 3);
    float s0 = ld_rw(cs + ch * kWS + 0), s1 = ld_rw(cs + ch * kWS + 1), s2 = ld_rw(cs + ch * kWS + 2);
    float n0 = 0.f, n1 = 0.f, n2 = 0.f;
    for (int t = 0; t < t_end; ++t) {
      const float s3 = ld_ro(xb + (size_t)t * p.C + ch);
      float z = __fmul_rn(w0, s0);
      z = __fmaf_rn(w1, s1, z);
      z = __fmaf_rn(w2, s2, z);
      z = __fmaf_rn(w3, s3, z);
      dst[t * dstride] = silu(z);
      s0 = s1;
      s1 = s2;
      s2 = s3;  // window after row t
      if (kSnap && (ci >= 2 * DK || qk_snap_owner)) {
        T* sc = static_cast<T*>(p.snapCs) + (((size_t)b * p.R + t) * p.C + ch) * kWS;
        st(sc + 0, s0);
        st(sc + 1, s1);
        st(sc + 2, s2);
      }
      if (kCommits && t == a) {
        n0 = s0;
        n1 = s1;
        n2 = s2;
      }
    }
    if (kCommits && commit) {
      if (ci >= 2 * DK) {  // v channel: this thread was its only reader
        st(cs + ch * kWS + 0, n0);
        st(cs + ch * kWS + 1, n1);
        st(cs + ch * kWS + 2, n2);
      } else {
        sNew[ci * kWS + 0] = n0;
        sNew[ci * kWS + 1] = n1;
        sNew[ci * kWS + 2] = n2;
      }
    }
  }
  if (tid < t_end) {
    const size_t gi = ((size_t)b * p.R + tid) * p.H_v + h;
    sA[tid] = expf(__ldg(p.g + gi));
    sBt[tid] = __ldg(p.beta + gi);
  }
  __syncthreads();

  // ---- per-head L2 norm of q and k (scale folded into q), k.q per row ----
  for (int t = warp; t < t_end; t += NW) {
    float sq = 0.f, sk = 0.f, qk = 0.f;
    for (int e = lane; e < DK; e += 32) {
      const float qv = sQ[t * DK + e], kv = sK[t * DK + e];
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
    const float fq = __fmul_rn(p.scale, rsqrtf(__fadd_rn(sq, p.eps)));
    const float fk = rsqrtf(__fadd_rn(sk, p.eps));
    for (int e = lane; e < DK; e += 32) {
      sQ[t * DK + e] = __fmul_rn(sQ[t * DK + e], fq);
      sK[t * DK + e] = __fmul_rn(sK[t * DK + e], fk);
    }
    if (lane == 0) sKQ[t] = __fmul_rn(__fmul_rn(qk, fq), fk);
  }
  __syncthreads();

  // ---- committed q/k windows: written by the group's last reader ----
  if (kCommits && commit) {
    if (tid == 0) {
      __threadfence();
      int* cnt = p.counters + (size_t)b * p.H_qk + hq;
      const int prev = atomicAdd(cnt, 1);
      const bool last = prev == p.G * p.slices - 1;
      if (last) atomicExch(cnt, 0);
      sLast = last;
    }
    __syncthreads();
    if (sLast) {
      for (int ci = tid; ci < 2 * DK; ci += NT) {
        const long long ch =
            ci < DK ? (long long)hq * DK + ci : (long long)p.H_qk * DK + (long long)hq * DK + (ci - DK);
        st(cs + ch * kWS + 0, sNew[ci * kWS + 0]);
        st(cs + ch * kWS + 1, sNew[ci * kWS + 1]);
        st(cs + ch * kWS + 2, sNew[ci * kWS + 2]);
      }
    }
  }

  // ---- the rows ----
  float* og = nullptr;
  if (kWantO) og = p.o + ((size_t)b * p.R * p.H_v + h) * p.d_v + (size_t)sl * DVS;
  const size_t o_tstride = (size_t)p.H_v * p.d_v;
  const int gbase = lane & ~(LPR - 1);
  for (int t = 0; t < t_end; ++t) {
    const float alpha = sA[t], bt = sBt[t];
    const float4* k4 = reinterpret_cast<const float4*>(sK + t * DK);
    float4 kv[NC4];
#pragma unroll
    for (int j = 0; j < NC4; ++j) kv[j] = k4[c + LPR * j];
    float part[V];
#pragma unroll
    for (int m = 0; m < M; ++m) {
      float acc = 0.f;
#pragma unroll
      for (int j = 0; j < NC4; ++j) acc = dot4(S[m][j], kv[j], acc);
      part[m] = acc;
    }
    if constexpr (kWantO) {
      const float4* q4 = reinterpret_cast<const float4*>(sQ + t * DK);
#pragma unroll
      for (int m = 0; m < M; ++m) {
        float acc = 0.f;
#pragma unroll
        for (int j = 0; j < NC4; ++j) acc = dot4(S[m][j], q4[c + LPR * j], acc);
        part[(M + m) % V] = acc;
      }
    }
    int idx;
    const float red = reduce_scatter<LPR, V>(part, lane, idx);
    const int mrow = idx % M;
    const int rloc = wrow + mrow * RG;
    // u is meaningful on the lanes holding an S k sum (idx < M)
    const float u = __fmul_rn(bt, __fsub_rn(sV[t * DVS + rloc], __fmul_rn(alpha, red)));
    if constexpr (kWantO) {
      const float up = __shfl_xor_sync(kFull, u, LPR / 2);  // u of the same row
      if (idx >= M && (c & kDupMask) == 0)
        og[(size_t)t * o_tstride + rloc] = __fmaf_rn(up, sKQ[t], __fmul_rn(alpha, red));
    }
    float um[M];
#pragma unroll
    for (int m = 0; m < M; ++m) um[m] = __shfl_sync(kFull, u, gbase | value_lane<LPR, V>(m));
#pragma unroll
    for (int m = 0; m < M; ++m)
#pragma unroll
      for (int j = 0; j < NC4; ++j) S[m][j] = decay_add(S[m][j], alpha, um[m], kv[j]);

    if (kCommits && commit && t == a) {
#pragma unroll
      for (int m = 0; m < M; ++m)
#pragma unroll
        for (int j = 0; j < NC4; ++j)
          *reinterpret_cast<float4*>(Sg + (size_t)(wrow + m * RG) * DK + 4 * (c + LPR * j)) = S[m][j];
    }
    if (kSnap) {
      float* Ss = p.snapS + (((size_t)b * p.R + t) * p.H_v + h) * head_elems + (size_t)sl * DVS * DK;
#pragma unroll
      for (int m = 0; m < M; ++m)
#pragma unroll
        for (int j = 0; j < NC4; ++j)
          *reinterpret_cast<float4*>(Ss + (size_t)(wrow + m * RG) * DK + 4 * (c + LPR * j)) = S[m][j];
    }
  }
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

template <int DK, typename T>
int launch_rows(const Params& p, int mode, cudaStream_t st) {
  using Gm = Geo<DK>;
  const dim3 grid(p.H_v * p.slices, p.B), block(Gm::NT);
  const size_t smem = sizeof(float) * ((size_t)2 * p.R * DK + (size_t)p.R * Gm::DVS + 3 * kMaxR + 2 * DK * kWS);
  switch (mode) {
    case kFused:
      rows_kernel<DK, T, kFused><<<grid, block, smem, st>>>(p);
      break;
    case kVerify:
      rows_kernel<DK, T, kVerify><<<grid, block, smem, st>>>(p);
      break;
    case kVerifySnap:
      rows_kernel<DK, T, kVerifySnap><<<grid, block, smem, st>>>(p);
      break;
    default:
      rows_kernel<DK, T, kCommitReplay><<<grid, block, smem, st>>>(p);
      break;
  }
  return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_LAUNCH;
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

enum Need : unsigned {
  kNeedRows = 1u,      // x, g, beta, conv_w, conv_state, ssm_state
  kNeedO = 2u,
  kNeedAccept = 4u,
  kNeedScratch = 8u,
  kNeedCounters = 16u,
  kNeedSlots = 32u     // conv_state, ssm_state, slot_ids, n_rows
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

  const size_t es = a->in_dtype == GDN_DTYPE_BF16 ? 2 : 4;  // element size of x, conv_w
  need |= kNeedSlots;
  if (need & kNeedSlots) {
    if (!a->conv_state || !a->ssm_state || !a->slot_ids || !a->n_rows) return GDN_ERR_INVALID_ARG;
    if (!aligned(a->conv_state, 16) || !aligned(a->ssm_state, 16) || !aligned(a->slot_ids, 4) ||
        !aligned(a->n_rows, 4))
      return GDN_ERR_MISALIGNED;
  }
  if (need & kNeedRows) {
    if (!a->x || !a->g || !a->beta || !a->conv_w) return GDN_ERR_INVALID_ARG;
    if (!aligned(a->x, es) || !aligned(a->conv_w, es) || !aligned(a->g, 4) || !aligned(a->beta, 4))
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
      return "misaligned pointer (state, scratch and o need 16 bytes; others their element size)";
    case GDN_ERR_LAUNCH:
      return "CUDA kernel launch failed";
    default:
      return "unknown gdnspec error code";
  }
}

}  // extern "C"
