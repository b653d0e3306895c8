// Compression behind one interface: "VeriCache: Turning Lossy KV Cache into Lossless LLM
// Inference", "Architecture support" — the framework plugs token-drop (SnapKV, KVzip) and
// quantising (KIVI) compressors in without touching scheduling or verification.
//
// Token drop: one 8-CTA thread-block cluster per request selects the keep-set with a 4-pass MSB
// radix select over the order-preserving uint32 image of the fp32 importance (-0 folded onto +0),
// summing the CTAs' histograms through distributed shared memory, then writes the kept indices in
// ascending order (each CTA its slice, offset by the lower-ranked CTAs' counts; ties at the
// threshold go to the lower indices), then appends the recent window. An optional second launch
// gathers the kept rows.
// Quantisation: key groups (32 tokens of one channel) one thread per channel; value groups
// (32 channels of one token) one thread per group (the post-accept append: one lane per D/32
// channels with shuffle min/max); every code equals the format's definition with IEEE
// round-to-nearest (division, rint half-to-even, fp32->fp16), by a fast rounding whose result is
// proven equal away from half-integers and the exact division near them.
#include "vc_internal.cuh"

#include <math.h>

namespace vc {

__device__ __forceinline__ uint32_t order_key(float f) {
  uint32_t u = __float_as_uint(f);
  if (u == 0x80000000u) u = 0u;  // -0 == +0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

constexpr int kKeepCL = 8;                 // CTAs per request: one thread-block cluster
constexpr int kKeepThreads = 512;
constexpr int kKeepWarps = kKeepThreads / 32;
constexpr int kKeepCacheKeys = 48 * 1024;  // keys of a CTA's slice that fit in shared memory (192 KB)

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// Every thread of every CTA of the cluster arrives; shared-memory writes before it are visible to
// the cluster's reads after it.
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// A word of CTA `rank`'s shared memory at the address of `p` in this CTA's.
__device__ __forceinline__ uint32_t ld_cluster_u32(const void* p, uint32_t rank) {
  uint32_t a, v;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"(smem_u32(p)), "r"(rank));
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(a) : "memory");
  return v;
}

// One cluster of kKeepCL CTAs per request; CTA `rank` owns candidates [rank*n/CL, (rank+1)*n/CL).
// The radix passes sum the CTAs' 256-bin histograms through distributed shared memory after a
// cluster barrier (every CTA then takes the same digit), and the compaction offsets a CTA's slice
// by the kept counts of the lower-ranked CTAs.
__global__ void __cluster_dims__(kKeepCL, 1, 1) __launch_bounds__(kKeepThreads)
    keepset_kernel(const __grid_constant__ KeepParams p, int cache_keys) {
  pdl_launch_dependents();
  pdl_wait();
  const int b = blockIdx.x / kKeepCL;
  const uint32_t rank = cluster_rank();
  const KeepReq& r = p.req[b];
  const int n = r.ctx, tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;
  if (r.keep >= n) {  // keep everything (uniform over the cluster: no shared state is touched)
    const int j0 = (int)((int64_t)rank * n / kKeepCL), j1 = (int)((int64_t)(rank + 1) * n / kKeepCL);
    for (int j = j0 + tid; j < j1; j += kKeepThreads) r.idx[j] = j;
    return;
  }
  const int n_cand = n - r.recent;
  const int need = r.keep - r.recent;
  const int s0 = (int)((int64_t)rank * n_cand / kKeepCL), s1 = (int)((int64_t)(rank + 1) * n_cand / kKeepCL);
  const int ns = s1 - s0;  // this CTA's candidates
  extern __shared__ uint32_t kcache[];
  __shared__ uint32_t hist[2][256];  // this CTA's histogram, double-buffered by pass
  __shared__ uint32_t tot[256];      // the cluster's histogram
  __shared__ uint32_t s_prefix, s_mask, s_rem;
  __shared__ int s_cnt[2][kKeepWarps];
  __shared__ int s_cta[2];           // this CTA's candidates above T and equal to T
  const bool cached = ns <= cache_keys;
  if (cached) {
#pragma unroll 4
    for (int i = tid; i < ns; i += kKeepThreads) kcache[i] = order_key(__ldg(r.imp + s0 + i));
  }
  if (tid == 0) {
    s_prefix = 0;
    s_mask = 0;
    s_rem = (uint32_t)need;
  }
  __syncthreads();
  auto key = [&](int i) -> uint32_t { return cached ? kcache[i] : order_key(__ldg(r.imp + s0 + i)); };
  // 1. radix select, most significant byte first, over the whole request: the key T of the
  //    need-th largest candidate and how many candidates equal to T are kept (s_rem at the end)
  if (need > 0) {
#pragma unroll 1
    for (int pass = 0; pass < 4; ++pass) {
      const int shift = 24 - 8 * pass;
      uint32_t* h = hist[pass & 1];  // last read by the cluster before the previous cluster barrier
      if (tid < 256) h[tid] = 0;
      __syncthreads();
      const uint32_t prefix = s_prefix, mask = s_mask;
#pragma unroll 4
      for (int base = 0; base < ns; base += kKeepThreads) {  // whole warps iterate together
        const int i = base + tid;
        const uint32_t u = i < ns ? key(i) : 0u;
        const bool in = i < ns && (u & mask) == prefix;
        const uint32_t dg = (u >> shift) & 255u;
        // aggregate equal digits of a warp into one shared atomic
        const unsigned act = __ballot_sync(0xffffffffu, in);
        if (in) {
          const unsigned peers = __match_any_sync(act, dg);
          if (lane == (__ffs(peers) - 1)) atomicAdd(&h[dg], (uint32_t)__popc(peers));
        }
      }
      __syncthreads();
      cluster_sync();  // every CTA's histogram of this pass is complete
      if (tid < 256) {
        uint32_t t = 0;
#pragma unroll
        for (int q = 0; q < kKeepCL; ++q) t += ld_cluster_u32(&h[tid], (uint32_t)q);
        tot[tid] = t;
      }
      __syncthreads();
      if (warp == 0) {
        // lane l owns digits 8l..8l+7; counts of larger digits come from the lanes above
        uint32_t c[8], own = 0;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          c[k] = tot[8 * lane + k];
          own += c[k];
        }
        uint32_t above = own;  // inclusive suffix sum over lanes >= l
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
          const uint32_t o = __shfl_down_sync(0xffffffffu, above, off);
          if (lane + off < 32) above += o;
        }
        uint32_t cum = above - own;  // candidates with a larger digit than this lane's range
        const uint32_t rem = s_rem;
        __syncwarp();  // every lane has read s_rem before the selected lane overwrites it
#pragma unroll
        for (int k = 7; k >= 0; --k) {
          if (cum < rem && cum + c[k] >= rem) {  // exactly one (lane, k) satisfies this
            s_rem = rem - cum;
            s_prefix = prefix | ((uint32_t)(8 * lane + k) << shift);
            s_mask = mask | (255u << shift);
          }
          cum += c[k];
        }
      }
      __syncthreads();
    }
  }
  // 2. ascending compaction over contiguous per-warp segments, 32 elements per ballot: an element's
  //    slot is the number of larger keys before it plus min(equal keys before it, need_eq), where
  //    "before" spans the lower-ranked CTAs' slices too
  if (need > 0) {
    const uint32_t T = s_prefix;
    const int need_eq = (int)s_rem;
    const int segw = ((ns + 31) / 32 + kKeepWarps - 1) / kKeepWarps * 32;
    const int w0 = min(ns, warp * segw), w1 = min(ns, w0 + segw);
    const unsigned lt = (1u << lane) - 1u;
    int gt = 0, eq = 0;
#pragma unroll 4
    for (int base = w0; base < w1; base += 32) {
      const int i = base + lane;
      const uint32_t u = i < w1 ? key(i) : 0u;
      gt += __popc(__ballot_sync(0xffffffffu, i < w1 && u > T));
      eq += __popc(__ballot_sync(0xffffffffu, i < w1 && u == T));
    }
    if (lane == 0) {
      s_cnt[0][warp] = gt;
      s_cnt[1][warp] = eq;
    }
    __syncthreads();
    if (tid == 0) {
      int g = 0, e = 0;
      for (int w = 0; w < kKeepWarps; ++w) {
        g += s_cnt[0][w];
        e += s_cnt[1][w];
      }
      s_cta[0] = g;
      s_cta[1] = e;
    }
    __syncthreads();
    cluster_sync();  // every CTA's counts are complete
    int gt_before = 0, eq_before = 0;
    for (uint32_t q = 0; q < rank; ++q) {
      gt_before += (int)ld_cluster_u32(&s_cta[0], q);
      eq_before += (int)ld_cluster_u32(&s_cta[1], q);
    }
    for (int w = 0; w < warp; ++w) {
      gt_before += s_cnt[0][w];
      eq_before += s_cnt[1][w];
    }
    int out = gt_before + min(eq_before, need_eq), eq_run = eq_before;
#pragma unroll 2
    for (int base = w0; base < w1; base += 32) {
      const int i = base + lane;
      const bool valid = i < w1;
      const uint32_t u = valid ? key(i) : 0u;
      const unsigned bgt = __ballot_sync(0xffffffffu, valid && u > T);
      const unsigned beq = __ballot_sync(0xffffffffu, valid && u == T);
      const bool take_eq = valid && u == T && eq_run + __popc(beq & lt) < need_eq;
      const unsigned bsel = bgt | __ballot_sync(0xffffffffu, take_eq);
      if ((bsel >> lane) & 1u) r.idx[out + __popc(bsel & lt)] = s0 + i;
      out += __popc(bsel);
      eq_run += __popc(beq);
    }
  }
  {
    const int j0 = (int)((int64_t)rank * r.recent / kKeepCL), j1 = (int)((int64_t)(rank + 1) * r.recent / kKeepCL);
    for (int j = j0 + tid; j < j1; j += kKeepThreads) r.idx[need + j] = n_cand + j;
  }
  cluster_sync();  // no CTA leaves while another may still read its shared memory
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
  int max_slice = 0;
  for (int b = 0; b < p.B; ++b) {
    const int nc = p.req[b].ctx - p.req[b].recent;
    const int sl = (nc + kKeepCL - 1) / kKeepCL;
    if (sl > max_slice) max_slice = sl;
  }
  const int cache_keys = max_slice < kKeepCacheKeys ? max_slice : kKeepCacheKeys;
  static std::atomic<uint64_t> attr{0};
  {
    cudaError_t e = raise_smem_limit(keepset_kernel, kKeepCacheKeys * (int)sizeof(uint32_t), attr);
    if (e != cudaSuccess) return e;
  }
  cudaError_t e = launch_pdl(keepset_kernel, dim3(p.B * kKeepCL), dim3(kKeepThreads),
                             (size_t)(cache_keys > 0 ? cache_keys : 1) * sizeof(uint32_t), s, p, cache_keys);
  if (e != cudaSuccess) return e;
  bool any = false;
  for (int b = 0; b < p.B; ++b) any |= p.req[b].compact != 0;
  if (any && max_keep > 0) e = launch_pdl(gather_rows_kernel, dim3((max_keep + 7) / 8, p.Hkv, p.B), dim3(256), 0, s, p);
  return e;
}

// ---------------------------------------------------------------------------------------------
// rs = the correctly rounded reciprocal of sf (0 when sf is 0), for quant_code.
template <int BITS>
__device__ __forceinline__ void quant_params(float mn, float mx, __half& s16, __half& z16, float& sf, float& zf,
                                             float& rs, int32_t* st) {
  constexpr float QMAX = (float)((1 << BITS) - 1);
  s16 = __float2half_rn(__fdiv_rn(__fsub_rn(mx, mn), QMAX));
  z16 = __float2half_rn(mn);
  sf = __half2float(s16);
  zf = __half2float(z16);
  rs = sf != 0.f ? __frcp_rn(sf) : 0.f;
  if (!isfinite(sf) || !isfinite(zf)) set_status(st, VC_DEV_RANGE);
}

// code = clamp(rint(fl((x - z) / s)), 0, 2^BITS - 1) with fl the IEEE float32 quotient, computed as
// y = fl(a * rs): rs is within 2^-24 of 1/s (relative) and the product adds one rounding, so
// |y - a/s| <= 2^-23 |y| (+ tiny), below 3e-6 wherever the clamp does not decide (|y| <= 17). When
// y is at least 1e-4 away from every half-integer, y, a/s and fl(a/s) lie strictly between the
// same two half-integers and round to the same integer; otherwise (rarely) the quotient itself is
// taken.
template <int BITS>
__device__ __forceinline__ uint32_t quant_code(float x, float sf, float zf, float rs) {
  constexpr float QMAX = (float)((1 << BITS) - 1);
  if (sf == 0.f) return 0u;
  const float a = __fsub_rn(x, zf);
  const float y = __fmul_rn(a, rs);
  float t = rintf(y);
  if (fabsf(y) <= QMAX + 2.f && fabsf(y - t) > 0.5f - 1e-4f) t = rintf(__fdiv_rn(a, sf));
  t = fminf(fmaxf(t, 0.f), QMAX);
  return (uint32_t)t;
}

// quant_code for two values that share a scale and zero, by packed f32x2 arithmetic: with
// a = x - z, u = fl(a rs + 1.5 * 2^23) holds rint of the exact product a rs (half to even) in its bit
// pattern (kMagicBits + rint for |a rs| < 2^22, and ordered like a rs outside), so an integer clamp
// of the pattern gives the clamped code; d = fl(a rs - rint) is the product's distance from it.
// Where the clamp does not decide (|a rs| <= 2^b + 1), a rs is within 2^-23 (2^b + 1) < 2.1e-6 of
// fl(a / s), so a product at least 1e-5 from every half-integer rounds like the quotient; a pair
// with either value nearer (or not a number) is recomputed by quant_code.
constexpr float kMagic = 12582912.f;
constexpr int32_t kMagicBits = 0x4B400000;
constexpr float kTieGuard = 0.5f - 1e-5f;
__device__ __forceinline__ unsigned long long f32x2_pack(float lo, float hi) {
  return (unsigned long long)__float_as_uint(lo) | ((unsigned long long)__float_as_uint(hi) << 32);
}
template <int BITS>
__device__ __forceinline__ void quant_code2(float x0, float x1, float sf, float zf, float rs, uint32_t& c0,
                                            uint32_t& c1) {
  constexpr int32_t QMAX = (1 << BITS) - 1;
  const unsigned long long m2 = f32x2_pack(kMagic, kMagic), rs2 = f32x2_pack(rs, rs);
  unsigned long long a2, u2, tn2, d2;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(a2) : "l"(f32x2_pack(x0, x1)), "l"(f32x2_pack(-zf, -zf)));
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(u2) : "l"(a2), "l"(rs2), "l"(m2));
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(tn2) : "l"(m2), "l"(u2));
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d2) : "l"(a2), "l"(rs2), "l"(tn2));
  if (!(fabsf(__uint_as_float((uint32_t)d2)) <= kTieGuard) || !(fabsf(__uint_as_float((uint32_t)(d2 >> 32))) <= kTieGuard)) {
    c0 = quant_code<BITS>(x0, sf, zf, rs);
    c1 = quant_code<BITS>(x1, sf, zf, rs);
    return;
  }
  c0 = (uint32_t)(min(max((int32_t)(uint32_t)u2, kMagicBits), kMagicBits + QMAX) - kMagicBits);
  c1 = (uint32_t)(min(max((int32_t)(uint32_t)(u2 >> 32), kMagicBits), kMagicBits + QMAX) - kMagicBits);
}

// A group's minimum and maximum from 16 bf16x2 words by pairwise trees (min and max select exactly,
// so the order does not change the result): the two lanes of the results hold the minimum (maximum)
// over the words' low and high halves.
__device__ __forceinline__ void minmax_tree16(const uint32_t (&w)[16], __nv_bfloat162& mn, __nv_bfloat162& mx) {
  __nv_bfloat162 lo[8], hi[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const __nv_bfloat162 x = *reinterpret_cast<const __nv_bfloat162*>(&w[2 * k]);
    const __nv_bfloat162 y = *reinterpret_cast<const __nv_bfloat162*>(&w[2 * k + 1]);
    lo[k] = __hmin2(x, y);
    hi[k] = __hmax2(x, y);
  }
#pragma unroll
  for (int st = 4; st >= 1; st >>= 1)
#pragma unroll
    for (int k = 0; k < st; ++k) {
      lo[k] = __hmin2(lo[k], lo[k + st]);
      hi[k] = __hmax2(hi[k], hi[k + st]);
    }
  mn = lo[0];
  mx = hi[0];
}

// A 32-token block's codes in shared memory, one byte per (token or channel row, column); rows are
// padded by 4 bytes so that eight consecutive rows fall on eight different banks.
template <int D>
using CodeTile = uint8_t[32][D + 4];

// Storage of one 32-token block's codes: 32-bit words w[half][j][lane] (4-bit) or w[half][p][lane]
// (2-bit, p covers steps j = 2p and 2p + 1). Word (half, j, lane), a = lane / 4, b = lane % 4, holds
// four (low, high) code pairs i = 0..3; pair i puts its low code at bit BITS*i' and its high code at
// bit 16 + BITS*i', with i' = i (4-bit) or i + 4 * (j - 2p) (2-bit). The pairs, as (token, channel):
//   keys:   t0 = 16 half + a, c0 = 16 j + 2 b:
//           (t0, c0|c0+1), (t0+8, c0|c0+1), (t0, c0+8|c0+9), (t0+8, c0+8|c0+9)
//   values: r0 = 16 j + a, k0 = 16 half + 2 b:
//           (k0|k0+1, r0), (k0|k0+1, r0+8), (k0+8|k0+9, r0), (k0+8|k0+9, r0+8)
// so a lane's word is exactly the four 16-bit A-fragment registers of an m16n8k16 MMA over that
// 16 x 16 tile (keys: M = tokens, K = channels; values: M = channels, K = tokens).
template <int D, int BITS, bool KEYS>
__device__ __forceinline__ uint32_t block_word(const uint8_t (*codes)[D + 4], int widx) {
  constexpr int STEPS = BITS == 4 ? D / 16 : D / 32;  // words per (half, lane) row
  const int lane = widx & 31;
  const int step = (widx >> 5) % STEPS;
  const int half = (widx >> 5) / STEPS;
  const int a = lane >> 2, b = lane & 3;
  uint32_t w = 0;
#pragma unroll
  for (int f = 0; f < (BITS == 4 ? 4 : 8); ++f) {
    const int j = BITS == 4 ? step : 2 * step + (f >> 2);
    const int i = f & 3;
    const int sh = BITS * f;
    uint32_t lo, hi;
    if (KEYS) {
      const int t = 16 * half + a + ((i & 1) ? 8 : 0);
      const int c = 16 * j + 2 * b + ((i & 2) ? 8 : 0);
      lo = codes[t][c];
      hi = codes[t][c + 1];
    } else {
      const int r = 16 * j + a + ((i & 1) ? 8 : 0);
      const int k = 16 * half + 2 * b + ((i & 2) ? 8 : 0);
      lo = codes[k][r];
      hi = codes[k + 1][r];
    }
    w |= (lo << sh) | (hi << (16 + sh));
  }
  return w;
}

// keys: grid (ng_max, Hkv, B), block D. The block's 32 x D keys (contiguous rows) are staged with
// 16-byte loads; thread c then quantises channel c over the 32 tokens.
template <int D, int BITS>
__global__ void __launch_bounds__(D) quant_keys_kernel(const __grid_constant__ QuantParams p) {
  const QuantReq& r = p.req[blockIdx.z];
  const int g = blockIdx.x, h = blockIdx.y, c = threadIdx.x;
  if (g >= r.ng) return;
  __shared__ __align__(16) bf16 tile[32 * D];
  __shared__ CodeTile<D> codes;
  const uint4* src = reinterpret_cast<const uint4*>(r.k + ((size_t)h * r.cap + 32 * g) * D);
#pragma unroll
  for (int e = c; e < 32 * D / 8; e += D) reinterpret_cast<uint4*>(tile)[e] = __ldg(src + e);
  __syncthreads();
  float x[32];
  float mn = INFINITY, mx = -INFINITY;
#pragma unroll
  for (int t = 0; t < 32; ++t) {
    x[t] = __bfloat162float(tile[t * D + c]);
    mn = fminf(mn, x[t]);
    mx = fmaxf(mx, x[t]);
  }
  __half s16, z16;
  float sf, zf, rs;
  quant_params<BITS>(mn, mx, s16, z16, sf, zf, rs, p.dev_status);
  const size_t gi = ((size_t)h * r.ng_cap + g) * D + c;
  r.ks[gi] = s16;
  r.kz[gi] = z16;
#pragma unroll
  for (int t = 0; t < 32; t += 2) {
    uint32_t c0, c1;
    quant_code2<BITS>(x[t], x[t + 1], sf, zf, rs, c0, c1);
    codes[t][c] = (uint8_t)c0;
    codes[t + 1][c] = (uint8_t)c1;
  }
  __syncthreads();
  uint32_t* dst = reinterpret_cast<uint32_t*>(r.kc + ((size_t)h * r.ng_cap + g) * (4 * D * BITS));
  for (int wi = c; wi < D * BITS; wi += D) dst[wi] = block_word<D, BITS, true>(codes, wi);
}

// values: grid (ng_max, Hkv, B), block D: thread i quantises token i / (D/32) of the block over
// its 32-channel group i % (D/32), reading the group's 64 contiguous bytes with four 16-byte loads
// (a warp covers 2 KB of consecutive rows); the codes meet in shared memory for the word packing.
template <int D, int BITS>
__global__ void __launch_bounds__(D, 12) quant_values_kernel(const __grid_constant__ QuantParams p) {
  const QuantReq& r = p.req[blockIdx.z];
  const int g = blockIdx.x, h = blockIdx.y;
  if (g >= r.ng) return;
  __shared__ CodeTile<D> codes;
  constexpr int NG = D / 32;  // channel groups per token
  const int tt = threadIdx.x / NG, cg = threadIdx.x % NG;
  const int t = 32 * g + tt;
  const uint4* src = reinterpret_cast<const uint4*>(r.v + ((size_t)h * r.cap + t) * D + 32 * cg);
  // the group's 32 values stay bf16, paired (channels 2e, 2e + 1) in 16 registers
  uint32_t xw[16];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const uint4 u = __ldg(src + k);
    xw[4 * k] = u.x;
    xw[4 * k + 1] = u.y;
    xw[4 * k + 2] = u.z;
    xw[4 * k + 3] = u.w;
  }
  __nv_bfloat162 mn2, mx2;
  minmax_tree16(xw, mn2, mx2);
  const float mn = fminf(__low2float(mn2), __high2float(mn2));
  const float mx = fmaxf(__low2float(mx2), __high2float(mx2));
  __half s16, z16;
  float sf, zf, rs;
  quant_params<BITS>(mn, mx, s16, z16, sf, zf, rs, p.dev_status);
  const size_t row = (size_t)h * (32 * r.ng_cap) + t;
  r.vs[row * NG + cg] = s16;
  r.vz[row * NG + cg] = z16;
#pragma unroll
  for (int e = 0; e < 16; ++e) {
    uint32_t c0, c1;
    quant_code2<BITS>(__uint_as_float(xw[e] << 16), __uint_as_float(xw[e] & 0xFFFF0000u), sf, zf, rs, c0, c1);
    codes[tt][32 * cg + 2 * e] = (uint8_t)c0;
    codes[tt][32 * cg + 2 * e + 1] = (uint8_t)c1;
  }
  __syncthreads();
  uint32_t* dst = reinterpret_cast<uint32_t*>(r.vc + ((size_t)h * r.ng_cap + g) * (4 * D * BITS));
  for (int wi = threadIdx.x; wi < D * BITS; wi += D) dst[wi] = block_word<D, BITS, false>(codes, wi);
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
    quant_values_kernel<D, BITS><<<dim3(max_ng, p.Hkv, p.B), D, 0, s>>>(p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  if (max_res > 0) copy_residual_kernel<<<dim3((max_res + 7) / 8, p.Hkv, p.B), 256, 0, s>>>(p);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------------------------
// Append after accept: grid (Hkv, B), block 256, dynamic shared memory for the extended residual.
// Every request: KV_full rows ctx .. ctx+n-1 <- the new rows. VC_QUANT requests: the residual
// (window rows [0, n_res)) followed by the new rows is staged in shared memory; its first
// 32 * (ng_new - ng) rows become blocks ng .. ng_new-1 by the same arithmetic and word order as
// quant_keys_kernel / quant_values_kernel, and the rest is written back as the new window. One CTA
// owns a (request, head), so the window is rewritten from its staged copy without hazards.
constexpr int kAppendThreads = 256;

template <int D, int BITS>
__global__ void __launch_bounds__(kAppendThreads) append_kernel(const __grid_constant__ AppendParams p) {
  pdl_launch_dependents();
  pdl_wait();
  const AppendReq& r = p.req[blockIdx.y];
  const int h = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n = r.n_rows;
  if (n <= 0) return;
  constexpr int V16 = D * 2 / 16;  // 16-byte pieces of a bf16 row
  for (int e = tid; e < n * 2 * V16; e += kAppendThreads) {
    const int i = e / (2 * V16), q = e % (2 * V16);
    const bool isv = q >= V16;
    const uint4* src = reinterpret_cast<const uint4*>((isv ? r.v_rows : r.k_rows) + ((size_t)i * p.Hkv + h) * D);
    uint4* dst = reinterpret_cast<uint4*>((isv ? r.v_full : r.k_full) + ((size_t)h * r.cap + r.ctx + i) * D);
    dst[q % V16] = __ldg(src + q % V16);
  }
  if (!r.quant) return;
  extern __shared__ uint4 ext_raw[];
  const int n_res = r.ctx - VC_GROUP * r.ng, n_ext = n_res + n;
  bf16* ek = reinterpret_cast<bf16*>(ext_raw);  // [n_ext][D] keys, then [n_ext][D] values
  bf16* ev = ek + (size_t)n_ext * D;
  for (int e = tid; e < n_ext * 2 * V16; e += kAppendThreads) {
    const int j = e / (2 * V16), q = e % (2 * V16);
    const bool isv = q >= V16;
    const bf16* row = j < n_res ? (isv ? r.v_win : r.k_win) + ((size_t)h * r.win_cap + j) * D
                                : (isv ? r.v_rows : r.k_rows) + ((size_t)(j - n_res) * p.Hkv + h) * D;
    reinterpret_cast<uint4*>((isv ? ev : ek) + (size_t)j * D)[q % V16] = reinterpret_cast<const uint4*>(row)[q % V16];
  }
  __syncthreads();
  __shared__ CodeTile<D> codes;
  constexpr int CPL = D / 32;    // channels per lane (values)
  constexpr int LPG = 32 / CPL;  // lanes per 32-channel group
  for (int gi = 0; gi < r.ng_new - r.ng; ++gi) {
    const int g = r.ng + gi;
    const bf16* kb = ek + (size_t)(VC_GROUP * gi) * D;
    const bf16* vb = ev + (size_t)(VC_GROUP * gi) * D;
    // keys: thread c quantises channel c over the block's 32 tokens
    if (tid < D) {
      const int c = tid;
      float x[32];
      float mn = INFINITY, mx = -INFINITY;
#pragma unroll
      for (int t = 0; t < 32; ++t) {
        x[t] = __bfloat162float(kb[(size_t)t * D + c]);
        mn = fminf(mn, x[t]);
        mx = fmaxf(mx, x[t]);
      }
      __half s16, z16;
      float sf, zf, rs;
      quant_params<BITS>(mn, mx, s16, z16, sf, zf, rs, p.dev_status);
      const size_t gidx = ((size_t)h * r.ng_cap + g) * D + c;
      r.ks[gidx] = s16;
      r.kz[gidx] = z16;
#pragma unroll
      for (int t = 0; t < 32; ++t) codes[t][c] = (uint8_t)quant_code<BITS>(x[t], sf, zf, rs);
    }
    __syncthreads();
    uint32_t* kdst = reinterpret_cast<uint32_t*>(r.kc + ((size_t)h * r.ng_cap + g) * (4 * D * BITS));
    for (int wi = tid; wi < D * BITS; wi += kAppendThreads) kdst[wi] = block_word<D, BITS, true>(codes, wi);
    __syncthreads();
    // values: warp w quantises tokens w, w+8, w+16, w+24; lane l channels CPL*l .. CPL*l+CPL-1
    const int c0 = CPL * lane;
    for (int tt = warp; tt < 32; tt += kAppendThreads / 32) {
      float x[CPL];
      float mn = INFINITY, mx = -INFINITY;
#pragma unroll
      for (int e = 0; e < CPL; ++e) {
        x[e] = __bfloat162float(vb[(size_t)tt * D + c0 + e]);
        mn = fminf(mn, x[e]);
        mx = fmaxf(mx, x[e]);
      }
#pragma unroll
      for (int off = 1; off < LPG; off <<= 1) {
        mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, off));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
      }
      __half s16, z16;
      float sf, zf, rs;
      quant_params<BITS>(mn, mx, s16, z16, sf, zf, rs, p.dev_status);
      const size_t row = (size_t)h * (VC_GROUP * (size_t)r.ng_cap) + VC_GROUP * g + tt;
      if ((lane % LPG) == 0) {
        r.vs[row * (D / 32) + c0 / 32] = s16;
        r.vz[row * (D / 32) + c0 / 32] = z16;
      }
#pragma unroll
      for (int e = 0; e < CPL; ++e) codes[tt][c0 + e] = (uint8_t)quant_code<BITS>(x[e], sf, zf, rs);
    }
    __syncthreads();
    uint32_t* vdst = reinterpret_cast<uint32_t*>(r.vc + ((size_t)h * r.ng_cap + g) * (4 * D * BITS));
    for (int wi = tid; wi < D * BITS; wi += kAppendThreads) vdst[wi] = block_word<D, BITS, false>(codes, wi);
    __syncthreads();
  }
  // the new residual: staged rows [32 * (ng_new - ng), n_ext) -> window rows [0, ...)
  const int sh = VC_GROUP * (r.ng_new - r.ng);
  for (int e = tid; e < (n_ext - sh) * 2 * V16; e += kAppendThreads) {
    const int j = e / (2 * V16), q = e % (2 * V16);
    const bool isv = q >= V16;
    uint4* dst = reinterpret_cast<uint4*>((isv ? r.v_win : r.k_win) + ((size_t)h * r.win_cap + j) * D);
    dst[q % V16] = reinterpret_cast<const uint4*>((isv ? ev : ek) + (size_t)(sh + j) * D)[q % V16];
  }
}

template <int D, int BITS>
static cudaError_t launch_append_t(const AppendParams& p, int max_ext_rows, cudaStream_t s) {
  const size_t smem = (size_t)(max_ext_rows > 0 ? max_ext_rows : 1) * 2 * D * sizeof(bf16);
  static std::atomic<uint64_t> attr{0};
  {
    cudaError_t e = raise_smem_limit(append_kernel<D, BITS>, VC_APPEND_MAX_ROWS * 2 * D * (int)sizeof(bf16), attr);
    if (e != cudaSuccess) return e;
  }
  return launch_pdl(append_kernel<D, BITS>, dim3(p.Hkv, p.B), dim3(kAppendThreads), smem, s, p);
}

cudaError_t launch_append(const AppendParams& p, int max_ext_rows, cudaStream_t s) {
  const int bits = p.bits == 4 ? 4 : 2;  // token-drop-only calls take the 2-bit instance (no blocks)
  if (p.d == 128) return bits == 2 ? launch_append_t<128, 2>(p, max_ext_rows, s) : launch_append_t<128, 4>(p, max_ext_rows, s);
  if (p.d == 64) return bits == 2 ? launch_append_t<64, 2>(p, max_ext_rows, s) : launch_append_t<64, 4>(p, max_ext_rows, s);
  return cudaErrorInvalidValue;
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
