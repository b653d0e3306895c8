// Compression behind one interface: "VeriCache: Turning Lossy KV Cache into Lossless LLM
// Inference", "Architecture support" — the framework plugs token-drop (SnapKV, KVzip) and
// quantising (KIVI) compressors in without touching scheduling or verification.
//
// Token drop: one CTA per request selects the keep-set with a 4-pass MSB radix select over the
// order-preserving uint32 image of the fp32 importance (-0 folded onto +0), then writes the kept
// indices in ascending order with block-wide ballot scans (ties at the threshold go to the lower
// indices), then appends the recent window. An optional second launch gathers the kept rows.
// Quantisation: key groups (32 tokens of one channel) one thread per channel; value groups
// (32 channels of one token) one lane per 4 channels with shuffle min/max; every float decision
// uses IEEE round-to-nearest (division, rint half-to-even, fp32->fp16), as the format defines.
#include "vc_internal.cuh"

#include <math.h>

namespace vc {

__device__ __forceinline__ uint32_t order_key(float f) {
  uint32_t u = __float_as_uint(f);
  if (u == 0x80000000u) u = 0u;  // -0 == +0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

constexpr int kKeepThreads = 1024;

// Exclusive block scan of one flag per thread; returns the prefix, writes the block total.
__device__ __forceinline__ int block_scan_flag(bool f, int* warp_tot, int& total) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const unsigned ball = __ballot_sync(0xffffffffu, f);
  const int in_warp = __popc(ball & ((1u << lane) - 1u));
  if (lane == 0) warp_tot[w] = __popc(ball);
  __syncthreads();
  if (w == 0) {
    int v = warp_tot[lane];
    int incl = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int o = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += o;
    }
    warp_tot[32 + lane] = incl - v;
    if (lane == 31) warp_tot[64] = incl;
  }
  __syncthreads();
  const int r = warp_tot[32 + w] + in_warp;
  total = warp_tot[64];
  __syncthreads();
  return r;
}

__global__ void __launch_bounds__(kKeepThreads) keepset_kernel(const __grid_constant__ KeepParams p) {
  pdl_launch_dependents();
  pdl_wait();
  const KeepReq& r = p.req[blockIdx.x];
  const int n = r.ctx, tid = threadIdx.x;
  if (r.keep >= n) {
    for (int j = tid; j < n; j += kKeepThreads) r.idx[j] = j;
    return;
  }
  const int n_cand = n - r.recent;
  const int need = r.keep - r.recent;
  __shared__ uint32_t hist[256];
  __shared__ uint32_t s_prefix, s_mask, s_rem;
  __shared__ int scan_buf[65];
  if (tid == 0) {
    s_prefix = 0;
    s_mask = 0;
    s_rem = (uint32_t)need;
  }
  __syncthreads();
  if (need > 0) {
#pragma unroll 1
    for (int pass = 0; pass < 4; ++pass) {
      const int shift = 24 - 8 * pass;
      for (int i = tid; i < 256; i += kKeepThreads) hist[i] = 0;
      __syncthreads();
      const uint32_t prefix = s_prefix, mask = s_mask;
#pragma unroll 1
      for (int base = 0; base < n_cand; base += kKeepThreads) {  // whole warps iterate together
        const int i = base + tid;
        const uint32_t u = i < n_cand ? order_key(__ldg(r.imp + i)) : 0u;
        const bool in = i < n_cand && (u & mask) == prefix;
        const uint32_t dg = (u >> shift) & 255u;
        // aggregate equal digits of a warp into one shared atomic
        const unsigned act = __ballot_sync(0xffffffffu, in);
        if (in) {
          const unsigned peers = __match_any_sync(act, dg);
          if ((threadIdx.x & 31) == (__ffs(peers) - 1)) atomicAdd(&hist[dg], (uint32_t)__popc(peers));
        }
      }
      __syncthreads();
      if (tid == 0) {
        uint32_t rem = s_rem, cum = 0;
        int sel = 0;
        for (int dg = 255; dg >= 0; --dg) {
          if (cum + hist[dg] >= rem) {
            sel = dg;
            break;
          }
          cum += hist[dg];
        }
        s_rem = rem - cum;
        s_prefix = prefix | ((uint32_t)sel << shift);
        s_mask = mask | (255u << shift);
      }
      __syncthreads();
    }
  }
  const uint32_t T = s_prefix;
  const int need_eq = need > 0 ? (int)s_rem : 0;
  int running = 0, eq_seen = 0;
#pragma unroll 1
  for (int base = 0; base < n_cand && running < need; base += kKeepThreads) {
    const int i = base + tid;
    const uint32_t u = i < n_cand ? order_key(__ldg(r.imp + i)) : 0u;
    const bool gt = i < n_cand && need > 0 && u > T;
    const bool eq = i < n_cand && need > 0 && u == T;
    int tot_eq;
    const int eq_rank = block_scan_flag(eq, scan_buf, tot_eq);
    const bool sel = gt || (eq && eq_seen + eq_rank < need_eq);
    int tot_sel;
    const int pos = block_scan_flag(sel, scan_buf, tot_sel);
    if (sel) r.idx[running + pos] = i;
    running += tot_sel;
    eq_seen += tot_eq;
  }
  for (int j = tid; j < r.recent; j += kKeepThreads) r.idx[need + j] = n_cand + j;
}

// Gather kept rows into a compact copy: dst[h][j] = src[h][idx[j]] (one warp per row pair).
__global__ void __launch_bounds__(256) gather_rows_kernel(const __grid_constant__ KeepParams p) {
  pdl_launch_dependents();
  pdl_wait();
  const KeepReq& r = p.req[blockIdx.z];
  if (!r.compact) return;
  const int keep = min(r.keep, r.ctx);
  const int j = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int h = blockIdx.y, lane = threadIdx.x & 31;
  if (j >= keep) return;
  const int t = r.idx[j];
  if (t < 0 || (int64_t)t >= r.src_cap) {
    if (lane == 0) set_status(p.dev_status, VC_DEV_BOUNDS);
    return;
  }
  const int v16 = p.d * 2 / 16;
  const uint4* ks = reinterpret_cast<const uint4*>(r.k_src + ((size_t)h * r.src_cap + t) * p.d);
  const uint4* vs = reinterpret_cast<const uint4*>(r.v_src + ((size_t)h * r.src_cap + t) * p.d);
  uint4* kd = reinterpret_cast<uint4*>(r.k_dst + ((size_t)h * r.dst_cap + j) * p.d);
  uint4* vd = reinterpret_cast<uint4*>(r.v_dst + ((size_t)h * r.dst_cap + j) * p.d);
  for (int e = lane; e < 2 * v16; e += 32) {
    if (e < v16)
      kd[e] = __ldg(ks + e);
    else
      vd[e - v16] = __ldg(vs + e - v16);
  }
}

cudaError_t launch_keepset(const KeepParams& p, int max_keep, cudaStream_t s) {
  cudaError_t e = launch_pdl(keepset_kernel, dim3(p.B), dim3(kKeepThreads), 0, s, p);
  if (e != cudaSuccess) return e;
  bool any = false;
  for (int b = 0; b < p.B; ++b) any |= p.req[b].compact != 0;
  if (any && max_keep > 0) e = launch_pdl(gather_rows_kernel, dim3((max_keep + 7) / 8, p.Hkv, p.B), dim3(256), 0, s, p);
  return e;
}

// ---------------------------------------------------------------------------------------------
template <int BITS>
__device__ __forceinline__ void quant_params(float mn, float mx, __half& s16, __half& z16, float& sf, float& zf,
                                             int32_t* st) {
  constexpr float QMAX = (float)((1 << BITS) - 1);
  s16 = __float2half_rn(__fdiv_rn(__fsub_rn(mx, mn), QMAX));
  z16 = __float2half_rn(mn);
  sf = __half2float(s16);
  zf = __half2float(z16);
  if (!isfinite(sf) || !isfinite(zf)) set_status(st, VC_DEV_RANGE);
}

template <int BITS>
__device__ __forceinline__ uint32_t quant_code(float x, float sf, float zf) {
  constexpr float QMAX = (float)((1 << BITS) - 1);
  if (sf == 0.f) return 0u;
  float t = rintf(__fdiv_rn(__fsub_rn(x, zf), sf));
  t = fminf(fmaxf(t, 0.f), QMAX);
  return (uint32_t)t;
}

// keys: grid (ng_max, Hkv, B), block D: thread c quantises channel c over the group's 32 tokens.
template <int D, int BITS>
__global__ void __launch_bounds__(D) quant_keys_kernel(const __grid_constant__ QuantParams p) {
  const QuantReq& r = p.req[blockIdx.z];
  const int g = blockIdx.x, h = blockIdx.y, c = threadIdx.x;
  if (g >= r.ng) return;
  const bf16* src = r.k + ((size_t)h * r.cap + 32 * g) * D + c;
  float x[32];
  float mn = INFINITY, mx = -INFINITY;
#pragma unroll
  for (int t = 0; t < 32; ++t) {
    x[t] = __bfloat162float(src[(size_t)t * D]);
    mn = fminf(mn, x[t]);
    mx = fmaxf(mx, x[t]);
  }
  __half s16, z16;
  float sf, zf;
  quant_params<BITS>(mn, mx, s16, z16, sf, zf, p.dev_status);
  const size_t gi = ((size_t)h * r.ng + g) * D + c;
  r.ks[gi] = s16;
  r.kz[gi] = z16;
  // 32 codes packed little-endian along tokens: 8 bytes (2-bit) or 16 bytes (4-bit)
  uint32_t w[BITS];
#pragma unroll
  for (int k = 0; k < BITS; ++k) w[k] = 0u;
#pragma unroll
  for (int t = 0; t < 32; ++t) {
    const uint32_t q = quant_code<BITS>(x[t], sf, zf);
    const int bit = BITS * t;
    w[bit / 32] |= q << (bit % 32);
  }
  uint8_t* dst = r.kc + gi * (4 * BITS);
  if (BITS == 2) {
    *reinterpret_cast<uint2*>(dst) = make_uint2(w[0], w[1 % BITS]);
  } else {
    *reinterpret_cast<uint4*>(dst) = make_uint4(w[0], w[1 % BITS], w[2 % BITS], w[3 % BITS]);
  }
}

// values: grid (ceil(Tq/8), Hkv, B), block 256: warp per token, lane per D/32 channels.
template <int D, int BITS>
__global__ void __launch_bounds__(256) quant_values_kernel(const __grid_constant__ QuantParams p) {
  const QuantReq& r = p.req[blockIdx.z];
  const int h = blockIdx.y, lane = threadIdx.x & 31;
  const int t = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int Tq = 32 * r.ng;
  if (t >= Tq) return;
  constexpr int CPL = D / 32;
  constexpr int LPG = 32 / CPL;  // lanes per 32-channel group
  const int c0 = CPL * lane;
  const bf16* src = r.v + ((size_t)h * r.cap + t) * D + c0;
  float x[CPL];
  float mn = INFINITY, mx = -INFINITY;
#pragma unroll
  for (int e = 0; e < CPL; ++e) {
    x[e] = __bfloat162float(src[e]);
    mn = fminf(mn, x[e]);
    mx = fmaxf(mx, x[e]);
  }
#pragma unroll
  for (int off = 1; off < LPG; off <<= 1) {
    mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, off));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
  }
  __half s16, z16;
  float sf, zf;
  quant_params<BITS>(mn, mx, s16, z16, sf, zf, p.dev_status);
  uint32_t bitsw = 0;
#pragma unroll
  for (int e = 0; e < CPL; ++e) bitsw |= quant_code<BITS>(x[e], sf, zf) << (BITS * e);
  const size_t row = (size_t)h * Tq + t;
  if ((lane % LPG) == 0) {
    r.vs[row * (D / 32) + c0 / 32] = s16;
    r.vz[row * (D / 32) + c0 / 32] = z16;
  }
  uint8_t* dst = r.vc + row * (D * BITS / 8);
  constexpr int LBITS = CPL * BITS;  // 4, 8 or 16 bits per lane
  if (LBITS == 4) {
    const uint32_t nb = __shfl_down_sync(0xffffffffu, bitsw, 1);
    if ((lane & 1) == 0) dst[lane >> 1] = (uint8_t)(bitsw | (nb << 4));
  } else if (LBITS == 8) {
    dst[lane] = (uint8_t)bitsw;
  } else {
    reinterpret_cast<uint16_t*>(dst)[lane] = (uint16_t)bitsw;
  }
}

// residual: rows [Tq, ctx) of K and V -> window rows [0, n_res); grid (ceil(max_res/8), Hkv, B).
__global__ void __launch_bounds__(256) copy_residual_kernel(const __grid_constant__ QuantParams p) {
  const QuantReq& r = p.req[blockIdx.z];
  const int h = blockIdx.y, lane = threadIdx.x & 31;
  const int j = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (j >= r.n_res) return;
  const int t = 32 * r.ng + j;
  const int v16 = p.d * 2 / 16;
  const uint4* ks = reinterpret_cast<const uint4*>(r.k + ((size_t)h * r.cap + t) * p.d);
  const uint4* vs = reinterpret_cast<const uint4*>(r.v + ((size_t)h * r.cap + t) * p.d);
  uint4* kd = reinterpret_cast<uint4*>(r.k_win + ((size_t)h * r.win_cap + j) * p.d);
  uint4* vd = reinterpret_cast<uint4*>(r.v_win + ((size_t)h * r.win_cap + j) * p.d);
  for (int e = lane; e < 2 * v16; e += 32) {
    if (e < v16)
      kd[e] = __ldg(ks + e);
    else
      vd[e - v16] = __ldg(vs + e - v16);
  }
}

template <int D, int BITS>
static cudaError_t launch_quant_t(const QuantParams& p, int max_ng, int max_tq, int max_res, cudaStream_t s) {
  if (max_ng > 0) {
    quant_keys_kernel<D, BITS><<<dim3(max_ng, p.Hkv, p.B), D, 0, s>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    quant_values_kernel<D, BITS><<<dim3((max_tq + 7) / 8, p.Hkv, p.B), 256, 0, s>>>(p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  if (max_res > 0) copy_residual_kernel<<<dim3((max_res + 7) / 8, p.Hkv, p.B), 256, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_quant(const QuantParams& p, int max_ng, int max_tq, cudaStream_t s) {
  int max_res = 0;
  for (int b = 0; b < p.B; ++b) max_res = max_res > p.req[b].n_res ? max_res : p.req[b].n_res;
  if (p.d == 128) return p.bits == 2 ? launch_quant_t<128, 2>(p, max_ng, max_tq, max_res, s)
                                     : launch_quant_t<128, 4>(p, max_ng, max_tq, max_res, s);
  if (p.d == 64) return p.bits == 2 ? launch_quant_t<64, 2>(p, max_ng, max_tq, max_res, s)
                                    : launch_quant_t<64, 4>(p, max_ng, max_tq, max_res, s);
  return cudaErrorInvalidValue;
}

}  // namespace vc
