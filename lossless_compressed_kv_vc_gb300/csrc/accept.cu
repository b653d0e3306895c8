// Greedy accept: "VeriCache: Turning Lossy KV Cache into Lossless LLM Inference", "Core
// algorithm" step 3 — accept drafts up to the first mismatch with the full-cache prediction, plus
// one bonus token when all of them match.
//
// Two launches: one CTA per logits row finds the row's argmax (first maximal index) with 16-byte
// loads and writes it into the request's output slot; then one warp per request finds the first
// mismatch with a ballot, pads the output with -1 and writes the accepted count. Slots i <= n
// already hold the right token: a_i == draft_i for i < n, and a_n is the correction or the bonus.
#include "vc_internal.cuh"

#include <limits.h>
#include <math.h>

namespace vc {

__device__ __forceinline__ void better(float& bv, int& bi, float v, int i) {
  if (v > bv || (v == bv && i < bi)) {
    bv = v;
    bi = i;
  }
}

// L[b] from the device, held to [0, L_max] so that no row or draft outside request b's is read.
__device__ __forceinline__ int clamp_L(int Lb, int L_max) { return Lb < 0 ? 0 : (Lb > L_max ? L_max : Lb); }

constexpr int kAcceptThreads = 512;

__global__ void __launch_bounds__(kAcceptThreads) accept_argmax_kernel(AcceptArgs a) {
  pdl_launch_dependents();
  pdl_wait();
  const int row = blockIdx.x;
  const int rows = a.L_max + 1;
  const int b = row / rows, i = row % rows;
  if (i > clamp_L(__ldg(a.L + b), a.L_max)) return;
  const float* x = a.logits + (size_t)row * a.V;
  const int V = a.V;
  float bv = -INFINITY;
  int bi = INT_MAX;
  // scalar head up to 16-byte alignment, vector body, scalar tail
  int pre = (int)(((16 - ((uintptr_t)x & 15)) & 15) >> 2);
  if (pre > V) pre = V;
  if ((int)threadIdx.x < pre) better(bv, bi, __ldg(x + threadIdx.x), threadIdx.x);
  const int nv = (V - pre) >> 2;
  const float4* xv = reinterpret_cast<const float4*>(x + pre);
  int j = threadIdx.x;
#pragma unroll 1
  for (; j + 3 * kAcceptThreads < nv; j += 4 * kAcceptThreads) {
    float4 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) v[u] = __ldg(xv + j + u * kAcceptThreads);
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int base = pre + 4 * (j + u * kAcceptThreads);
      better(bv, bi, v[u].x, base);
      better(bv, bi, v[u].y, base + 1);
      better(bv, bi, v[u].z, base + 2);
      better(bv, bi, v[u].w, base + 3);
    }
  }
  for (; j < nv; j += kAcceptThreads) {
    const float4 v = __ldg(xv + j);
    const int base = pre + 4 * j;
    better(bv, bi, v.x, base);
    better(bv, bi, v.y, base + 1);
    better(bv, bi, v.z, base + 2);
    better(bv, bi, v.w, base + 3);
  }
  const int tail0 = pre + 4 * nv;
  if (tail0 + (int)threadIdx.x < V) better(bv, bi, __ldg(x + tail0 + threadIdx.x), tail0 + threadIdx.x);
  // warp then block reduction
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
    const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
    better(bv, bi, ov, oi);
  }
  __shared__ float sv[kAcceptThreads / 32];
  __shared__ int si[kAcceptThreads / 32];
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) {
    sv[w] = bv;
    si[w] = bi;
  }
  __syncthreads();
  if (w == 0) {
    bv = lane < kAcceptThreads / 32 ? sv[lane] : -INFINITY;
    bi = lane < kAcceptThreads / 32 ? si[lane] : INT_MAX;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
      better(bv, bi, ov, oi);
    }
    if (lane == 0) a.out_tokens[(size_t)b * rows + i] = bi;
  }
}

__global__ void accept_finalize_kernel(AcceptArgs a) {
  pdl_launch_dependents();
  pdl_wait();
  const int b = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (b >= a.B) return;
  const int rows = a.L_max + 1;
  const int Lb = clamp_L(__ldg(a.L + b), a.L_max);
  int32_t* out = a.out_tokens + (size_t)b * rows;
  const int32_t* x = a.draft + (size_t)b * a.L_max;
  int n = Lb;
  for (int i0 = 0; i0 < Lb; i0 += 32) {
    const int i = i0 + lane;
    const bool mis = i < Lb && out[i] != x[i];
    const unsigned ball = __ballot_sync(0xffffffffu, mis);
    if (ball) {
      n = i0 + __ffs(ball) - 1;
      break;
    }
  }
  __syncwarp();
  for (int i = lane; i < rows; i += 32)
    if (i > n) out[i] = -1;
  if (lane == 0) a.n_acc[b] = n + 1;
}

cudaError_t launch_accept(const AcceptArgs& a, cudaStream_t s) {
  cudaError_t e = launch_pdl(accept_argmax_kernel, dim3(a.B * (a.L_max + 1)), dim3(kAcceptThreads), 0, s, a);
  if (e != cudaSuccess) return e;
  return launch_pdl(accept_finalize_kernel, dim3((a.B + 3) / 4), dim3(128), 0, s, a);
}

}  // namespace vc
