// Draft decode attention over the compressed cache KV_comp.
//
// "VeriCache: Turning Lossy KV Cache into Lossless LLM Inference", "Core algorithm" step 1
// (drafting with KV_comp) and "Cross-resource staggering (P1)" (drafting is bound by HBM
// bandwidth: it streams the compressed cache).
//
// Design (one launch per draft step, plus a small split-combine launch):
//   grid  = (sum over requests of its KV splits, Hkv), 128 threads (4 warps).
//   A CTA owns one (request, KV head, split). The G = Hq/Hkv query heads of the KV head are the
//   M rows of m16n8k16 tensor-core MMAs (rows >= G are zero), so each KV row read from HBM
//   serves all G heads. KV rows reach shared memory through 1-D bulk copies on the TMA engine
//   (one copy per kept row: the gather by index costs no extra instruction per byte), each warp
//   running its own ring of stages on mbarriers. Quantised groups arrive as raw codes and are
//   dequantised in registers into a bf16 tile just before the MMAs. Each warp keeps an online
//   softmax (fp32, exp2 domain); warps merge in shared memory and a split writes either the final
//   bf16 row or an (o, lse) partial that the combine kernel merges.
//   The step's own K/V row (k_new, v_new) is read straight from its input and also stored into
//   window row n_win by the first split (fused append).
#include "vc_internal.cuh"

#include <math.h>

namespace vc {

template <int D, int KIND>  // KIND 0: bf16 rows (token drop); 2 or 4: quantised, bits
struct DraftCfg {
  static constexpr int NW = 4;
  static constexpr int ROWB = D * 2;                     // bytes of one bf16 row
  static constexpr int RS = ROWB + 16;                   // padded smem row stride (conflict-free ldmatrix)
  static constexpr int TILE = 16 * RS;                   // 16 bf16 rows
  static constexpr int QRAW = (KIND == 0) ? 0 : 8 * D * (KIND + 1);  // raw bytes of one 32-token group
  static constexpr int STAGE = (2 * TILE > QRAW) ? 2 * TILE : QRAW;
  static constexpr int NST = (KIND == 0) ? 3 : 2;
  static constexpr int DQ = (KIND == 0) ? 0 : 2 * TILE;  // dequantised K+V tile (quant only)
  static constexpr int PER_WARP = NST * STAGE + DQ;
  static constexpr int BAR_OFF = NW * PER_WARP;
  static constexpr int SMEM = BAR_OFF + NW * NST * 8;
  static constexpr int CHUNK_MAIN = (KIND == 0) ? 16 : 32;
  static constexpr int NT = D / 8;                       // output n-tiles
  static constexpr int KS = D / 16;                      // k-steps over the head dim
  // raw layout of a quantised group inside a stage
  static constexpr int OFF_KC = 0;
  static constexpr int OFF_KS = OFF_KC + D * 4 * (KIND == 0 ? 2 : KIND);
  static constexpr int OFF_KZ = OFF_KS + 2 * D;
  static constexpr int OFF_VC = OFF_KZ + 2 * D;
  static constexpr int OFF_VS = OFF_VC + 4 * D * (KIND == 0 ? 2 : KIND);
  static constexpr int OFF_VZ = OFF_VS + 2 * D;
  static_assert(NW * PER_WARP <= 112 * 1024, "two CTAs per SM");
};

// Scores for one 16-token tile, online-softmax update and P*V accumulation.
template <int D>
__device__ __forceinline__ void tile_attend(const uint8_t* kt, const uint8_t* vt, int cnt, int RS, float scale_log2,
                                            const uint32_t (&qa)[D / 16][4], float (&o)[D / 8][4], float& m0,
                                            float& m1, float& l0, float& l1, int lane) {
  float s[2][4];
#pragma unroll
  for (int nt = 0; nt < 2; ++nt)
#pragma unroll
    for (int e = 0; e < 4; ++e) s[nt][e] = 0.f;
#pragma unroll
  for (int ks = 0; ks < D / 16; ks += 2) {
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      const uint8_t* a = kt + (nt * 8 + (lane & 7)) * RS + (16 * ks + 8 * (lane >> 3)) * 2;
      uint32_t b0, b1, b2, b3;
      ldsm_x4(b0, b1, b2, b3, a);
      mma_bf16_16816(s[nt], qa[ks], b0, b1);
      mma_bf16_16816(s[nt], qa[ks + 1], b2, b3);
    }
  }
  const int tq = 2 * (lane & 3);
  float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
  for (int nt = 0; nt < 2; ++nt)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const bool ok = (nt * 8 + tq + e) < cnt;
      s[nt][e] = ok ? s[nt][e] * scale_log2 : -INFINITY;
      s[nt][e + 2] = ok ? s[nt][e + 2] * scale_log2 : -INFINITY;
      mx0 = fmaxf(mx0, s[nt][e]);
      mx1 = fmaxf(mx1, s[nt][e + 2]);
    }
  mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
  mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
  mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
  mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
  const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
  const float mu0 = (mn0 == -INFINITY) ? 0.f : mn0;
  const float mu1 = (mn1 == -INFINITY) ? 0.f : mn1;
  const float c0 = exp2f(m0 - mu0), c1 = exp2f(m1 - mu1);
  m0 = mn0;
  m1 = mn1;
  float p[2][4];
  float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
  for (int nt = 0; nt < 2; ++nt) {
    p[nt][0] = exp2f(s[nt][0] - mu0);
    p[nt][1] = exp2f(s[nt][1] - mu0);
    p[nt][2] = exp2f(s[nt][2] - mu1);
    p[nt][3] = exp2f(s[nt][3] - mu1);
    ps0 += p[nt][0] + p[nt][1];
    ps1 += p[nt][2] + p[nt][3];
  }
  l0 = l0 * c0 + ps0;
  l1 = l1 * c1 + ps1;
#pragma unroll
  for (int nt = 0; nt < D / 8; ++nt) {
    o[nt][0] *= c0;
    o[nt][1] *= c0;
    o[nt][2] *= c1;
    o[nt][3] *= c1;
  }
  uint32_t pa[4];
  pa[0] = pack_bf16x2(p[0][0], p[0][1]);
  pa[1] = pack_bf16x2(p[0][2], p[0][3]);
  pa[2] = pack_bf16x2(p[1][0], p[1][1]);
  pa[3] = pack_bf16x2(p[1][2], p[1][3]);
#pragma unroll
  for (int nd = 0; nd < D / 16; ++nd) {
    const uint8_t* a = vt + ((lane & 7) + 8 * ((lane >> 3) & 1)) * RS + (16 * nd + 8 * (lane >> 4)) * 2;
    uint32_t b0, b1, b2, b3;
    ldsm_x4_t(b0, b1, b2, b3, a);
    mma_bf16_16816(o[2 * nd], pa, b0, b1);
    mma_bf16_16816(o[2 * nd + 1], pa, b2, b3);
  }
}

// Dequantise tokens [16*half, 16*half+16) of a raw 32-token group into bf16 K and V tiles.
template <int D, int BITS>
__device__ __forceinline__ void dequant_half(const uint8_t* raw, uint8_t* kt, uint8_t* vt, int half, int lane) {
  using C = DraftCfg<D, BITS>;
  constexpr int CPL = D / 32;  // channels per lane
  constexpr uint32_t MASK = (1u << BITS) - 1u;
  const int c0 = CPL * lane;
  // keys: per channel, the 32 tokens' codes are one run of 4*BITS bytes
  const __half* ks = reinterpret_cast<const __half*>(raw + C::OFF_KS);
  const __half* kz = reinterpret_cast<const __half*>(raw + C::OFF_KZ);
  float sk[CPL], zk[CPL];
  uint64_t wk[CPL];
#pragma unroll
  for (int e = 0; e < CPL; ++e) {
    const int c = c0 + e;
    sk[e] = __half2float(ks[c]);
    zk[e] = __half2float(kz[c]);
    if (BITS == 2) {
      wk[e] = *reinterpret_cast<const uint32_t*>(raw + C::OFF_KC + c * 8 + 4 * half);
    } else {
      wk[e] = *reinterpret_cast<const uint64_t*>(raw + C::OFF_KC + c * 16 + 8 * half);
    }
  }
#pragma unroll
  for (int t = 0; t < 16; ++t) {
    float x[CPL];
#pragma unroll
    for (int e = 0; e < CPL; ++e) x[e] = fmaf((float)((uint32_t)(wk[e] >> (BITS * t)) & MASK), sk[e], zk[e]);
    uint8_t* dst = kt + t * C::RS + c0 * 2;
    if (CPL == 4) {
      uint2 v;
      v.x = pack_bf16x2(x[0], x[1]);
      v.y = pack_bf16x2(x[CPL > 2 ? 2 : 0], x[CPL > 3 ? 3 : 0]);
      *reinterpret_cast<uint2*>(dst) = v;
    } else {
      *reinterpret_cast<uint32_t*>(dst) = pack_bf16x2(x[0], x[CPL > 1 ? 1 : 0]);
    }
  }
  // values: per token, the D channels' codes are one run of D*BITS/8 bytes
  const __half* vs = reinterpret_cast<const __half*>(raw + C::OFF_VS);
  const __half* vz = reinterpret_cast<const __half*>(raw + C::OFF_VZ);
  const int grp = c0 / 32;
  const int bit0 = c0 * BITS;
#pragma unroll 4
  for (int tt = 0; tt < 16; ++tt) {
    const int t = 16 * half + tt;
    const uint32_t w =
        *reinterpret_cast<const uint32_t*>(raw + C::OFF_VC + t * (D * BITS / 8) + (bit0 / 32) * 4) >> (bit0 % 32);
    const float s = __half2float(vs[t * (D / 32) + grp]);
    const float z = __half2float(vz[t * (D / 32) + grp]);
    float x[CPL];
#pragma unroll
    for (int e = 0; e < CPL; ++e) x[e] = fmaf((float)((w >> (BITS * e)) & MASK), s, z);
    uint8_t* dst = vt + tt * C::RS + c0 * 2;
    if (CPL == 4) {
      uint2 v;
      v.x = pack_bf16x2(x[0], x[1]);
      v.y = pack_bf16x2(x[CPL > 2 ? 2 : 0], x[CPL > 3 ? 3 : 0]);
      *reinterpret_cast<uint2*>(dst) = v;
    } else {
      *reinterpret_cast<uint32_t*>(dst) = pack_bf16x2(x[0], x[CPL > 1 ? 1 : 0]);
    }
  }
}

template <int D, int KIND>
__global__ void __launch_bounds__(128, 2) draft_attn_kernel(const __grid_constant__ DraftParams p) {
  using C = DraftCfg<D, KIND>;
  extern __shared__ __align__(128) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int hk = blockIdx.y;
  int b = 0;
#pragma unroll 1
  for (int i = 1; i < p.B; ++i)
    if (p.req[i].split_begin <= (int)blockIdx.x) b = i;
  const DraftReqDev& r = p.req[b];
  const int split = (int)blockIdx.x - r.split_begin;
  const int G = p.G;

  uint8_t* wb = smem + warp * C::PER_WARP;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::BAR_OFF) + warp * C::NST;

  // fused append of this step's K/V row into the window (first split only)
  if (split == 0 && warp == 0) {
    constexpr int V16 = C::ROWB / 16;
    const int l = lane & 15;
    if (l < V16) {
      const uint4* src = reinterpret_cast<const uint4*>((lane < 16 ? r.k_new : r.v_new) + (size_t)hk * D);
      bf16* dst_row = (lane < 16 ? r.k_win : r.v_win) + ((size_t)hk * r.win_cap + r.n_win) * D;
      reinterpret_cast<uint4*>(dst_row)[l] = src[l];
    }
  }

  // zero the warp's buffers so rows never written hold finite values (masked with p = 0)
  for (int i = lane; i < C::PER_WARP / 16; i += 32) reinterpret_cast<uint4*>(wb)[i] = make_uint4(0, 0, 0, 0);
  if (lane == 0) {
    for (int s = 0; s < C::NST; ++s) mbar_init(&bars[s], 1);
    fence_mbar_init();
  }
  fence_proxy_async_smem();
  __syncwarp();

  // query fragments: rows = heads of this KV head (zero beyond G), columns = head dim
  uint32_t qa[C::KS][4];
  {
    const int g0 = lane >> 2, g1 = g0 + 8;
    const int cq = 2 * (lane & 3);
    const bf16* qb = r.q + (size_t)hk * G * D;
#pragma unroll
    for (int ks = 0; ks < C::KS; ++ks) {
      const int c = 16 * ks + cq;
      qa[ks][0] = g0 < G ? *reinterpret_cast<const uint32_t*>(qb + g0 * D + c) : 0u;
      qa[ks][1] = g1 < G ? *reinterpret_cast<const uint32_t*>(qb + g1 * D + c) : 0u;
      qa[ks][2] = g0 < G ? *reinterpret_cast<const uint32_t*>(qb + g0 * D + c + 8) : 0u;
      qa[ks][3] = g1 < G ? *reinterpret_cast<const uint32_t*>(qb + g1 * D + c + 8) : 0u;
    }
  }

  // chunk list of this split: main chunks, then (last split) window chunks of 16 rows
  const int m_begin = split * r.main_per_split;
  const int m_end = min(r.n_main, m_begin + r.main_per_split);
  const int n_mc = m_end > m_begin ? (m_end - m_begin + C::CHUNK_MAIN - 1) / C::CHUNK_MAIN : 0;
  const bool last = split == r.n_splits - 1;
  const int n_w = last ? r.n_win + 1 : 0;
  const int n_wc = (n_w + 15) / 16;
  const int n_chunks = n_mc + n_wc;
  const int my_n = n_chunks > warp ? (n_chunks - warp + C::NW - 1) / C::NW : 0;

  auto issue = [&](int i, int st) {
    const int c = warp + C::NW * i;
    uint8_t* sb = wb + st * C::STAGE;
    if (KIND != 0 && c < n_mc) {
      // one quantised 32-token group: six contiguous runs
      const int g = (m_begin / 32) + c;
      const int Tq = 32 * r.ng;
      constexpr int KCB = D * 4 * (KIND == 0 ? 2 : KIND);
      if (lane == 0) mbar_arrive_expect_tx(&bars[st], C::QRAW);
      __syncwarp();
      if (lane == 0) bulk_g2s(sb + C::OFF_KC, r.kc + ((size_t)hk * r.ng + g) * KCB, KCB, &bars[st]);
      if (lane == 1) bulk_g2s(sb + C::OFF_KS, r.ks + ((size_t)hk * r.ng + g) * D, 2 * D, &bars[st]);
      if (lane == 2) bulk_g2s(sb + C::OFF_KZ, r.kz + ((size_t)hk * r.ng + g) * D, 2 * D, &bars[st]);
      if (lane == 3) bulk_g2s(sb + C::OFF_VC, r.vc + ((size_t)hk * Tq + 32 * g) * (D * (KIND == 0 ? 2 : KIND) / 8),
                              KCB, &bars[st]);
      if (lane == 4) bulk_g2s(sb + C::OFF_VS, r.vs + ((size_t)hk * Tq + 32 * g) * (D / 32), 2 * D, &bars[st]);
      if (lane == 5) bulk_g2s(sb + C::OFF_VZ, r.vz + ((size_t)hk * Tq + 32 * g) * (D / 32), 2 * D, &bars[st]);
      return;
    }
    // 16 bf16 rows: lanes 0-15 copy K rows, lanes 16-31 the matching V rows
    const int row = lane & 15;
    const bool isv = lane >= 16;
    const bf16* src = nullptr;
    if (c < n_mc) {
      const int j = m_begin + c * 16 + row;
      if (j < m_end) {
        int t = r.compact ? j : __ldg(r.idx + j);
        if (t >= 0 && (int64_t)t < r.rows_cap) {
          src = (isv ? r.v_rows : r.k_rows) + ((size_t)hk * r.rows_cap + t) * D;
        } else {
          set_status(p.dev_status, VC_DEV_BOUNDS);
        }
      }
    } else {
      const int j = (c - n_mc) * 16 + row;
      if (j < r.n_win) {
        src = (isv ? r.v_win : r.k_win) + ((size_t)hk * r.win_cap + j) * D;
      } else if (j == r.n_win) {
        src = (isv ? r.v_new : r.k_new) + (size_t)hk * D;
      }
    }
    const unsigned ball = __ballot_sync(0xffffffffu, src != nullptr);
    if (lane == 0) mbar_arrive_expect_tx(&bars[st], __popc(ball) * C::ROWB);
    __syncwarp();
    if (src) bulk_g2s(sb + (isv ? C::TILE : 0) + row * C::RS, src, C::ROWB, &bars[st]);
  };

  float o[C::NT][4];
#pragma unroll
  for (int nt = 0; nt < C::NT; ++nt)
#pragma unroll
    for (int e = 0; e < 4; ++e) o[nt][e] = 0.f;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;

  const int pre = my_n < C::NST ? my_n : C::NST;
  for (int i = 0; i < pre; ++i) issue(i, i);
  bool ok = true;
#pragma unroll 1
  for (int i = 0; i < my_n; ++i) {
    const int st = i % C::NST;
    if (!mbar_wait_bounded(&bars[st], (i / C::NST) & 1, p.dev_status)) {
      // drain what is still in flight (bounded) and stop
      for (int j = i + 1; j < my_n && j < i + C::NST; ++j)
        mbar_wait_bounded(&bars[j % C::NST], (j / C::NST) & 1, p.dev_status);
      ok = false;
      break;
    }
    const int c = warp + C::NW * i;
    uint8_t* sb = wb + st * C::STAGE;
    if (KIND != 0 && c < n_mc) {
      uint8_t* kt = wb + C::NST * C::STAGE;
      uint8_t* vt = kt + C::TILE;
#pragma unroll 1
      for (int half = 0; half < 2; ++half) {
        dequant_half<D, (KIND == 0 ? 2 : KIND)>(sb, kt, vt, half, lane);
        __syncwarp();
        tile_attend<D>(kt, vt, 16, C::RS, p.scale_log2, qa, o, m0, m1, l0, l1, lane);
        __syncwarp();
      }
    } else {
      const int cnt = (c < n_mc) ? min(16, m_end - (m_begin + c * 16)) : min(16, n_w - (c - n_mc) * 16);
      tile_attend<D>(sb, sb + C::TILE, cnt, C::RS, p.scale_log2, qa, o, m0, m1, l0, l1, lane);
    }
    __syncwarp();
    if (i + C::NST < my_n) {
      fence_proxy_async_smem();
      issue(i + C::NST, st);
    }
  }
  (void)ok;

  // per-warp results -> shared memory (reusing the warp's stage area), then merge across warps
  l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
  l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
  __syncthreads();  // every warp is done with its stages
  float* mo = reinterpret_cast<float*>(wb);  // [16][D] o, then m[16], l[16]
  float* mm = mo + 16 * D;
  float* ml = mm + 16;
  {
    const int g0 = lane >> 2, g1 = g0 + 8;
    const int cq = 2 * (lane & 3);
#pragma unroll
    for (int nt = 0; nt < C::NT; ++nt) {
      mo[g0 * D + nt * 8 + cq] = o[nt][0];
      mo[g0 * D + nt * 8 + cq + 1] = o[nt][1];
      mo[g1 * D + nt * 8 + cq] = o[nt][2];
      mo[g1 * D + nt * 8 + cq + 1] = o[nt][3];
    }
    if ((lane & 3) == 0) {
      mm[g0] = m0;
      ml[g0] = l0;
      mm[g1] = m1;
      ml[g1] = l1;
    }
  }
  __syncthreads();
  const bool single = r.n_splits == 1;
  for (int e = threadIdx.x; e < G * D; e += blockDim.x) {
    const int g = e / D, c = e % D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < C::NW; ++w) M = fmaxf(M, reinterpret_cast<float*>(smem + w * C::PER_WARP)[16 * D + g]);
    const float Mu = (M == -INFINITY) ? 0.f : M;
    float Ls = 0.f, Os = 0.f;
#pragma unroll
    for (int w = 0; w < C::NW; ++w) {
      const float* base = reinterpret_cast<float*>(smem + w * C::PER_WARP);
      const float wt = exp2f(base[16 * D + g] - Mu);
      Ls += wt * base[16 * D + 16 + g];
      Os += wt * base[g * D + c];
    }
    const float val = Ls > 0.f ? Os / Ls : 0.f;
    const int h = hk * G + g;
    if (single) {
      r.o[(size_t)h * D + c] = __float2bfloat16_rn(val);
    } else {
      const size_t slot = ((size_t)b * p.Hq + h) * p.S_max + split;
      p.ws_o[slot * D + c] = val;
      if (c == 0) p.ws_lse[slot] = Ls > 0.f ? Mu + log2f(Ls) : -INFINITY;
    }
  }
}

// Merge the per-split partials (o_s, lse_s) of one (request, head): o = sum_s 2^(lse_s - LSE) o_s.
template <int D>
__global__ void __launch_bounds__(D) draft_combine_kernel(const __grid_constant__ DraftParams p) {
  const int b = blockIdx.x, h = blockIdx.y, c = threadIdx.x;
  const DraftReqDev& r = p.req[b];
  if (r.n_splits == 1) return;
  const size_t base = ((size_t)b * p.Hq + h) * p.S_max;
  float M = -INFINITY;
  for (int s = 0; s < r.n_splits; ++s) M = fmaxf(M, p.ws_lse[base + s]);
  const float Mu = (M == -INFINITY) ? 0.f : M;
  float acc = 0.f, L = 0.f;
  for (int s = 0; s < r.n_splits; ++s) {
    const float w = exp2f(p.ws_lse[base + s] - Mu);
    L += w;
    acc += w * p.ws_o[(base + s) * D + c];
  }
  r.o[(size_t)h * D + c] = __float2bfloat16_rn(L > 0.f ? acc / L : 0.f);
}

template <int D, int KIND>
static cudaError_t launch_draft_t(const DraftParams& p, int total_ctas, cudaStream_t s) {
  using C = DraftCfg<D, KIND>;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(draft_attn_kernel<D, KIND>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::SMEM);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  draft_attn_kernel<D, KIND><<<dim3(total_ctas, p.Hkv), 128, C::SMEM, s>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  draft_combine_kernel<D><<<dim3(p.B, p.Hq), D, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_draft(const DraftParams& p, int d, int kind, int total_ctas, cudaStream_t s) {
  if (d == 128) {
    if (kind == 0) return launch_draft_t<128, 0>(p, total_ctas, s);
    if (kind == 2) return launch_draft_t<128, 2>(p, total_ctas, s);
    if (kind == 4) return launch_draft_t<128, 4>(p, total_ctas, s);
  } else if (d == 64) {
    if (kind == 0) return launch_draft_t<64, 0>(p, total_ctas, s);
    if (kind == 2) return launch_draft_t<64, 2>(p, total_ctas, s);
    if (kind == 4) return launch_draft_t<64, 4>(p, total_ctas, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace vc
