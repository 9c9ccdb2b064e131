// Greedy acceptance of MTP drafts on the device, feeding the commit without a
// device-to-host copy of accept_len [LightLLM #1330 "Qwen3.5 / Qwen3.5-MoE MTP
// speculative decoding", Summary: accept length kept on the device; FreeToken
// #828 "Speculative decoding: MTP and DFlash", Design: the target's choices
// decide how many drafts are kept].
//
// argmax_kernel: one thread-block cluster of kCluster CTAs per (request b,
//   verify row t < n_rows[b]).  CTA r of the cluster scans its slice of the
//   vocabulary with 16-byte loads, keeping the largest logit and, among equal
//   largest values, the lowest token index; the block reduces its threads'
//   pairs through shared memory; rank 0 combines the kCluster pairs read from
//   its peers' shared memory and writes target[b][t].  HBM bound: the logits
//   are read once.
// accept_kernel: per request, the number of leading drafts equal to the
//   target's choice at the row before them.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "gdnspec.h"

namespace gdnaccept {

constexpr int kThreads = 512;
constexpr int kCluster = 8;
constexpr unsigned kFull = 0xffffffffu;

struct Params {
  int B, R, V;
  const void* logits;
  const int32_t* drafts;
  const int32_t* n_rows;
  int32_t* target;
  int32_t* accept_len;
  int32_t* status;
};

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// (value, index) of the larger value; equal values keep the lower index
__device__ __forceinline__ void better(float& v, int& i, float v2, int i2) {
  if (v2 > v || (v2 == v && i2 < i)) {
    v = v2;
    i = i2;
  }
}

__device__ __forceinline__ float lo_bf16(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float hi_bf16(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t peer_addr(const void* p, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;"
               : "=r"(r)
               : "r"((uint32_t)__cvta_generic_to_shared(p)), "r"(rank));
  return r;
}

template <typename T>
__global__ void __launch_bounds__(kThreads) argmax_kernel(const Params p) {
  pdl_wait();     // the logits of the kernel before are complete and visible
  pdl_trigger();  // the acceptance kernel may launch; it waits for this grid before reading
  __shared__ float sv[kThreads / 32];
  __shared__ int si[kThreads / 32];
  __shared__ float cv;
  __shared__ int ci;
  const int t = blockIdx.y, b = blockIdx.z;
  const int n = p.n_rows[b];
  if (n <= 0 || n > p.R || t >= n) return;  // the whole cluster leaves together
  const int rank = (int)cluster_rank();
  // this CTA's slice of the row, in whole 16-byte chunks
  constexpr int kPer = 16 / sizeof(T);  // elements per chunk
  const int chunks = p.V / kPer;
  const int per_cta = (chunks + kCluster - 1) / kCluster;
  const int c0 = rank * per_cta, c1 = min(chunks, c0 + per_cta);
  const uint4* row = reinterpret_cast<const uint4*>(static_cast<const T*>(p.logits) +
                                                    ((size_t)b * p.R + t) * p.V);
  float best = -INFINITY;
  int bi = 0x7fffffff;
  constexpr int kUnroll = 5;  // a 151936-token bf16 row slice in one batch of loads per thread
  for (int c = c0 + threadIdx.x; c < c1; c += kUnroll * kThreads) {
    uint4 w[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u)
      if (c + u * kThreads < c1) w[u] = __ldcs(row + c + u * kThreads);  // streamed: read once
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int cc = c + u * kThreads;
      if (cc < c1) {
        const int e0 = cc * kPer;
        const uint32_t ws[4] = {w[u].x, w[u].y, w[u].z, w[u].w};
        if constexpr (sizeof(T) == 2) {
#pragma unroll
          for (int j = 0; j < 4; ++j) {  // element order: low half first
            better(best, bi, lo_bf16(ws[j]), e0 + 2 * j);
            better(best, bi, hi_bf16(ws[j]), e0 + 2 * j + 1);
          }
        } else {
#pragma unroll
          for (int j = 0; j < 4; ++j) better(best, bi, __uint_as_float(ws[j]), e0 + j);
        }
      }
    }
  }
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) {
    const float v2 = __shfl_xor_sync(kFull, best, off);
    const int i2 = __shfl_xor_sync(kFull, bi, off);
    better(best, bi, v2, i2);
  }
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) {
    sv[warp] = best;
    si[warp] = bi;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < kThreads / 32; ++w) better(best, bi, sv[w], si[w]);
    cv = best;
    ci = bi;
  }
  cluster_sync();  // every CTA's pair is in its shared memory
  if (rank == 0 && threadIdx.x == 0) {
    float v = cv;
    int i = ci;
    for (uint32_t r = 1; r < kCluster; ++r) {
      float v2;
      int i2;
      asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v2) : "r"(peer_addr(&cv, r)) : "memory");
      asm volatile("ld.shared::cluster.s32 %0, [%1];" : "=r"(i2) : "r"(peer_addr(&ci, r)) : "memory");
      better(v, i, v2, i2);
    }
    // no entry ever won: every logit of the row is NaN, and the row's token is 0
    p.target[(size_t)b * p.R + t] = i == 0x7fffffff ? 0 : i;
  }
  cluster_sync();  // no CTA leaves while rank 0 reads its shared memory
}

// accept_len[b] = largest a <= n_rows[b] - 1 with drafts[b][i] == target[b][i]
// for every i < a: draft i + 1 sits at verify row i + 1 and is the token the
// target chose at row i.  Inactive requests (n_rows 0) get 0; a bad n_rows
// gets 0 and a status bit.
__global__ void __launch_bounds__(256) accept_kernel(const Params p) {
  pdl_wait();     // the target tokens are complete and visible
  pdl_trigger();  // the next kernel may launch; it waits for this grid before reading accept_len
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= p.B) return;
  const int n = p.n_rows[b];
  int a = 0;
  if (n < 0 || n > p.R) {
    if (p.status) atomicOr(p.status, GDN_STATUS_BAD_NROWS);
  } else {
    const int32_t* d = p.drafts + (size_t)b * (p.R - 1);
    const int32_t* tg = p.target + (size_t)b * p.R;
    while (a < n - 1 && d[a] == tg[a]) ++a;
  }
  p.accept_len[b] = a;
}

template <typename Kernel>
int launch(Kernel kernel, dim3 grid, dim3 block, int cluster, cudaStream_t st, const Params& p) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  int na = 0;
  attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[na++].val.programmaticStreamSerializationAllowed = 1;
  if (cluster > 1) {
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = cluster;
    attr[na].val.clusterDim.y = 1;
    attr[na++].val.clusterDim.z = 1;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  if (cudaLaunchKernelEx(&cfg, kernel, p) != cudaSuccess) return GDN_ERR_LAUNCH;
  return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_LAUNCH;
}

int check(const gdn_accept_args* a) {
  if (!a) return GDN_ERR_INVALID_ARG;
  if (a->B < 0 || a->R < 1 || a->V < 1) return GDN_ERR_INVALID_ARG;
  if (a->in_dtype != GDN_DTYPE_BF16 && a->in_dtype != GDN_DTYPE_F32) return GDN_ERR_UNSUPPORTED;
  if (a->V % 8 != 0 || a->B > 65535 || a->R > 65535) return GDN_ERR_UNSUPPORTED;
  if (a->B == 0) return GDN_OK;
  if (!a->logits || !a->n_rows || !a->target || !a->accept_len || (a->R > 1 && !a->drafts))
    return GDN_ERR_INVALID_ARG;
  auto al = [](const void* ptr, uintptr_t n) { return (reinterpret_cast<uintptr_t>(ptr) % n) == 0; };
  if (!al(a->logits, 16) || !al(a->n_rows, 4) || !al(a->target, 4) || !al(a->accept_len, 4) ||
      (a->drafts && !al(a->drafts, 4)) || (a->status && !al(a->status, 4)))
    return GDN_ERR_MISALIGNED;
  return GDN_OK;
}

}  // namespace gdnaccept

using namespace gdnaccept;

extern "C" GDN_API int gdn_greedy_accept(const gdn_accept_args* args, void* stream) {
  const int rc = check(args);
  if (rc != GDN_OK || args->B == 0) return rc;
  Params p{args->B, args->R, args->V, args->logits, args->drafts, args->n_rows,
           args->target, args->accept_len, args->status};
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const dim3 grid(kCluster, p.R, p.B);
  const int r = args->in_dtype == GDN_DTYPE_BF16
                    ? launch(argmax_kernel<__nv_bfloat16>, grid, dim3(kThreads), kCluster, st, p)
                    : launch(argmax_kernel<float>, grid, dim3(kThreads), kCluster, st, p);
  if (r != GDN_OK) return r;
  return launch(accept_kernel, dim3((p.B + 255) / 256), dim3(256), 1, st, p);
}
