// Draft decode attention over the compressed cache KV_comp.
//
// "VeriCache: Turning Lossy KV Cache into Lossless LLM Inference", "Core algorithm" step 1
// (drafting with KV_comp) and "Cross-resource staggering (P1)" (drafting is bound by HBM
// bandwidth: it streams the compressed cache).
//
// Work decomposition (one launch per draft step):
//   For one KV head, each request's rows form a list of chunks: its KV_comp rows (16 kept bf16
//   rows, or one 32-token quantised group, per chunk) followed by its bf16 window rows (16 per
//   chunk; the last window row is this step's own K/V). The host gives each request a whole number
//   of warps in proportion to its chunks (one wave of 4-warp CTAs, one grid row per KV head), and
//   a request's chunks are cut into equal contiguous ranges over its warps, so no warp holds two
//   requests. A warp owns its range outright: its own ring of shared-memory stages and its own
//   online softmax; its (o, lse) partial stays in its drained ring. At the end each CTA merges,
//   per request it holds, its warps' partials into the output (the request lies in this CTA) or
//   into a CTA partial; the CTA that arrives last among the request's CTAs (a per-request arrival
//   counter) merges those, in CTA order, so a step needs no second launch.

// Tensor cores: scores are S^T = K Q^T and the output O^T += V^T P^T on m16n8k16 MMAs with the
// 16 tokens (or 16 channels) of a tile as M and the query heads of the KV head as N (8 per MMA,
// zero-padded), so a KV byte serves all G heads and a 16-token tile costs d/8 MMAs. P^T, produced
// in the accumulator layout, becomes the next B operand through an in-register 8x8 transpose
// (movmatrix). A head's running maximum moves only when a tile exceeds it by more than 2^8, so
// O^T is rescaled rarely; exponentials use the SFU's ex2.approx.
//
// Loads: kept bf16 rows arrive by TMA tile::gather4 (four rows by index per load, whole 128-byte
// lines, 128-byte swizzle; indices prefetched one stage ahead); quantised groups arrive as six
// contiguous 1-D bulk copies and enter the MMAs in their stored form; bf16 window rows arrive by
// 16-byte cp.async into the same swizzled tile layout.
// The warp holding a request's first chunk also stores the step's K/V row into window row n_win
// (fused append); that row is read from its input, so no other warp depends on the store.
#include "vc_internal.cuh"
#include "draft_common.cuh"

#include <math.h>

namespace vc {

// KIND 0: bf16 rows (token drop); 2 or 4: quantised, bits. A 2-stage ring per warp (measured better
// than 3 stages with fewer CTAs: more warps in flight beat deeper rings). Token drop: three 4-warp
// CTAs per SM, a stage holds a 16-row K and V tile. Quantised: a stage holds one chunk of quantised
// groups (6 KB at d 128), and a window chunk -- only at the end of a warp's range -- takes the
// whole ring (WIN_SPANS: it is issued once nothing else is in flight), so four CTAs (16 warps) fit
// per SM: the quantised steps are bound by instruction latency, and more warps hide more of it.
template <int D, int KIND>
struct DraftCfg {
  static constexpr int NW = 4;
  static constexpr int ROWB = D * 2;                     // bytes of one bf16 row
  static constexpr int HALVES = D / 64;                  // 128-byte column blocks of a row
  static constexpr int BLK = 16 * 128;                   // one column block of a 16-row tile
  static constexpr int TILE = HALVES * BLK;              // 16 bf16 rows (swizzled column blocks)
  static constexpr int BITS = (KIND == 0) ? 2 : KIND;
  static constexpr int QRAW = (KIND == 0) ? 0 : 8 * D * (BITS + 1);  // raw bytes of one 32-token group
  static constexpr int GPC = (KIND == 2) ? 2 : 1;       // quantised groups per chunk (two 2-bit groups fit a stage)
  static constexpr int STAGE = (KIND == 0 ? 2 * TILE : GPC * QRAW + 1023) / 1024 * 1024;
  static constexpr int NST = 2;
  static constexpr bool WIN_SPANS = STAGE < 2 * TILE;   // a window tile needs more than one stage
  static constexpr int CTAS_PER_SM = (KIND == 0) ? 3 : 4;
  static constexpr int PER_WARP = NST * STAGE;
  static constexpr int BAR_OFF = NW * PER_WARP;
  static constexpr int SMEM = BAR_OFF + NW * NST * 8 + 1024;  // + slack to put the stages on 1024 B
  static constexpr int G4_OPS = 2 * HALVES * 4;          // gather4 loads that fill a 16-row K+V stage
  static constexpr int CHUNK_MAIN = (KIND == 0) ? 16 : 32 * GPC;
  static constexpr int MT = D / 16;                      // 16-wide tiles over the head dim
  // raw layout of a quantised group inside a stage
  static constexpr int KCB = D * 4 * BITS;               // key codes of one group
  static constexpr int OFF_KC = 0;
  static constexpr int OFF_KS = OFF_KC + KCB;
  static constexpr int OFF_KZ = OFF_KS + 2 * D;
  static constexpr int OFF_VC = OFF_KZ + 2 * D;
  static constexpr int OFF_VS = OFF_VC + KCB;
  static constexpr int OFF_VZ = OFF_VS + 2 * D;
  static_assert(SMEM + 1024 <= 228 * 1024 / CTAS_PER_SM, "CTAs per SM");
  static_assert(GPC * QRAW <= STAGE && QRAW % 16 == 0, "quantised groups of a chunk in one stage");
  static_assert(NST * STAGE >= 2 * TILE, "a window tile fits the ring");
  static_assert(PER_WARP >= 16 * (D + 1) * 4, "a warp's partial fits its drained ring");
};

// Tensor maps are an argument of the token-drop kernels only.
struct DraftNoMaps {
  int32_t unused;
};
template <int KIND>
struct DraftMapsOf {
  using T = DraftNoMaps;
};
template <>
struct DraftMapsOf<0> {
  using T = DraftMaps;
};

// Byte offset of 16-byte chunk cc (8 channels) of row r in a 16-row bf16 tile: column blocks of
// 16 x 128 bytes, the chunk index XOR (r mod 8) inside a block. This is the TMA 128-byte swizzle on
// a 1024-byte aligned block, and it keeps the eight rows an ldmatrix reads on distinct banks.
__device__ __forceinline__ int sw_off(int r, int cc) { return (cc >> 3) * 2048 + r * 128 + (((cc & 7) ^ (r & 7)) << 4); }

// 2^x for a pair of fp16 arguments, as an fp16 pair (one SFU instruction).
__device__ __forceinline__ uint32_t ex2_f16x2(uint32_t x) {
  uint32_t y;
  asm("ex2.approx.f16x2 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

// d = A B with a zero accumulator (m16n8k16, fp16 operands, fp32 result).
__device__ __forceinline__ void mma_f16_16816_c0(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%10,%10,%10,%10};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(0.f));
}

__device__ __forceinline__ uint32_t movmatrix_t(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

// One 16-token tile: scores, online softmax (per query head, exp2 domain) and P V accumulation.
// qb: Q^T B fragments [head block][k-step][2]; o: O^T accumulators [head block][channel tile][4];
// m, l: running max and (lane-partial) sum for this lane's two heads of each head block.
// PLO: the weights enter P V as two bf16 parts (p = hi + lo, each MMA'd against V), which keeps
// their 16 significant bits instead of 8. The quantised kernels take it for their window tiles:
// a request with only a few hundred bf16 rows (a short context, all residual) and peaked weights
// otherwise carries the weights' bf16 rounding almost undamped into its output.
template <int D, int NHB, bool PLO = false>
__device__ __forceinline__ void tile_attend(const uint8_t* kt, const uint8_t* vt, int cnt, float scale_log2,
                                            const uint32_t (&qb)[NHB][D / 16][2], float (&o)[NHB][D / 16][4],
                                            float (&m)[NHB][2], float (&l)[NHB][2], int lane) {
  float s[NHB][4];
#pragma unroll
  for (int hb = 0; hb < NHB; ++hb)
#pragma unroll
    for (int e = 0; e < 4; ++e) s[hb][e] = 0.f;
#pragma unroll
  for (int ks = 0; ks < D / 16; ++ks) {
    const uint8_t* a_ptr = kt + sw_off((lane & 7) + 8 * ((lane >> 3) & 1), 2 * ks + (lane >> 4));
    uint32_t a[4];
    ldsm_x4(a[0], a[1], a[2], a[3], a_ptr);
#pragma unroll
    for (int hb = 0; hb < NHB; ++hb) mma_bf16_16816(s[hb], a, qb[hb][ks][0], qb[hb][ks][1]);
  }
  // rows of the accumulator are tokens lane/4 and lane/4 + 8; columns heads 2(lane%4) + {0,1}.
  // The running maximum m (exp2 domain, per head) moves only when a tile's maximum exceeds it by
  // more than 8, so weights stay below 2^8 and O is rescaled rarely (never lowering the result's
  // precision: the final division by l uses the same m).
  const bool ok0 = (lane >> 2) < cnt, ok1 = (lane >> 2) + 8 < cnt;
  float p[NHB][2][2];  // [head block][head e][token row 0/1]
  // each lane tests its own scores; the reduction over the tile's lanes runs only when the
  // running maximum moves (the tile's maximum exceeds it by 2^8 exactly when some lane's does)
  float tmax[NHB][2];
  bool need = false;
#pragma unroll
  for (int hb = 0; hb < NHB; ++hb)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const float mx = fmaxf(ok0 ? s[hb][e] : -INFINITY, ok1 ? s[hb][e + 2] : -INFINITY);
      tmax[hb][e] = mx * scale_log2;  // the scale is positive: it keeps the order
      need |= tmax[hb][e] > m[hb][e] + 8.f;
    }
  if (__any_sync(0xffffffffu, need)) {
#pragma unroll
    for (int hb = 0; hb < NHB; ++hb) {
      float corr[2];
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        float mx = tmax[hb][e];
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
        const float mn = fmaxf(m[hb][e], mx);
        corr[e] = ex2_approx(m[hb][e] - mn);  // 0 when m was -inf (nothing accumulated yet)
        l[hb][e] *= corr[e];
        m[hb][e] = mn;
      }
#pragma unroll
      for (int mt = 0; mt < D / 16; ++mt) {
        o[hb][mt][0] *= corr[0];
        o[hb][mt][1] *= corr[1];
        o[hb][mt][2] *= corr[0];
        o[hb][mt][3] *= corr[1];
      }
    }
  }
#pragma unroll
  for (int hb = 0; hb < NHB; ++hb)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const float mu = m[hb][e] == -INFINITY ? 0.f : m[hb][e];
      p[hb][e][0] = ok0 ? ex2_approx(fmaf(s[hb][e], scale_log2, -mu)) : 0.f;
      p[hb][e][1] = ok1 ? ex2_approx(fmaf(s[hb][e + 2], scale_log2, -mu)) : 0.f;
      l[hb][e] += p[hb][e][0] + p[hb][e][1];
    }
  // P^T as the B operand (k = token, n = head): transpose the two 8x8 bf16 blocks of the accumulator
  uint32_t pb[NHB][2], pl[NHB][2];
#pragma unroll
  for (int hb = 0; hb < NHB; ++hb) {
    const uint32_t h0 = pack_bf16x2(p[hb][0][0], p[hb][1][0]), h1 = pack_bf16x2(p[hb][0][1], p[hb][1][1]);
    pb[hb][0] = movmatrix_t(h0);  // tokens 0-7
    pb[hb][1] = movmatrix_t(h1);  // tokens 8-15
    if constexpr (PLO) {
      // the remainders p - bf16(p) (exact in fp32), rounded to bf16 in turn
      const float2 f0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&h0));
      const float2 f1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&h1));
      pl[hb][0] = movmatrix_t(pack_bf16x2(p[hb][0][0] - f0.x, p[hb][1][0] - f0.y));
      pl[hb][1] = movmatrix_t(pack_bf16x2(p[hb][0][1] - f1.x, p[hb][1][1] - f1.y));
    }
  }
#pragma unroll
  for (int mt = 0; mt < D / 16; ++mt) {
    const uint8_t* a_ptr = vt + sw_off((lane & 7) + 8 * (lane >> 4), 2 * mt + ((lane >> 3) & 1));
    uint32_t a[4];
    ldsm_x4_t(a[0], a[1], a[2], a[3], a_ptr);
#pragma unroll
    for (int hb = 0; hb < NHB; ++hb) {
      mma_bf16_16816(o[hb][mt], a, pb[hb][0], pb[hb][1]);
      if constexpr (PLO) mma_bf16_16816(o[hb][mt], a, pl[hb][0], pl[hb][1]);
    }
  }
}

// One quantised 32-token block, read in its stored form (see the block layout in compress.cu): each
// lane's 32-bit word is its A fragment for an m16n8k16 MMA, turned into exact fp16 operands by one
// AND per register (code_frag_sub: the code keeps its bit position P, the exponent field stays zero,
// so the register holds code x 2^(P-24)); the tensor cores take the codes with no dequantised tile
// between, and the powers of two are folded into the other operand or the result.
// qn holds the query as fp16 scaled by 2^-E (|qn| < 1, E per warp), scale_q = log2(e)/sqrt(d) * 2^E.
//   keys (scale s_c, zero z_c per channel):
//     S^T[t][h] = sum_c code (s_c qn_hc) + sum_c z_c qn_hc
//     -> B operand fp16(s o qn) per block (B <= s: no overflow), the accumulator read back times
//        2^24 over the row's power of two; the per-head term z . qn is an MMA (z broadcast over
//        tokens) against qn, once per block for both 16-token halves;
//   values (scale s_t, zero z_t per token and 32-channel group g), P <= 1 (the running maximum moves
//   at every new maximum inside quantised blocks), codes as exact fp16 subnormals (code_frag_sub):
//     O^T[c][h] += sum_t code (s_t p_th) + sum_t z_t p_th
//     -> A = the code times a power of two per register, B operand fp16(s o p) per channel group;
//        the zero terms are one MMA per 16 tokens into zacc (rows = channel groups, B = the raw
//        weights), in the softmax frame of O, added when a run of quantised groups ends (fold_zs).
template <int D, int BITS, int NHB>
__device__ __forceinline__ void qblock_attend(const uint8_t* raw, float scale_q,
                                              const uint32_t (&qn)[NHB][D / 16][2], float (&o)[NHB][D / 16][4],
                                              float (&m)[NHB][2], float (&l)[NHB][2], float (&zacc)[NHB][4],
                                              int lane) {
  using C = DraftCfg<D, BITS>;
  constexpr int MT = D / 16;
  constexpr int STEPS = BITS == 4 ? D / 16 : D / 32;  // words per (half, lane)
  constexpr bool RS_MMA = BITS == 2;                   // row sums from the zero-term MMA (see below)
  const uint32_t* kw = reinterpret_cast<const uint32_t*>(raw + C::OFF_KC);
  const uint32_t* vw = reinterpret_cast<const uint32_t*>(raw + C::OFF_VC);
  const __half* ksc = reinterpret_cast<const __half*>(raw + C::OFF_KS);
  const __half* kze = reinterpret_cast<const __half*>(raw + C::OFF_KZ);
  const __half* vsc = reinterpret_cast<const __half*>(raw + C::OFF_VS);
  const __half* vze = reinterpret_cast<const __half*>(raw + C::OFF_VZ);
  const int b4 = lane & 3, a8 = lane >> 2;
  // block setup: the scaled query fragments qs = s o qn and the zero term z . qn of each head. The
  // key codes enter as exact fp16 subnormals (code_frag_sub): 2 bits put channels 8-15 of a k-step
  // 16x higher, which the query absorbs (its channels 8-15 arrive divided by 16), and token rows
  // 8-15 4x higher (2 bits) or 16x (4 bits), which the score scale of those rows absorbs. For 2
  // bits the zero term's A fragment keeps channels 0-7 in rows 0-7 and channels 8-15 in rows 8-15,
  // so the two sums come out separately and the second takes back its factor 16.
  uint32_t qs[NHB][MT][2];
  float cz[NHB][4];
#pragma unroll
  for (int hb = 0; hb < NHB; ++hb)
#pragma unroll
    for (int e = 0; e < 4; ++e) cz[hb][e] = 0.f;
  // The lane's key scales and zeros, channels 16 ks + 2 (lane % 4) + {0, 1} and the same + 8, by
  // ldmatrix: one x4 load covers two k-steps (its four matrices: k-step 2t channels 0-7, 8-15,
  // k-step 2t + 1 channels 0-7, 8-15), every row address of a matrix naming the same 16 bytes, so
  // that each lane receives the pair at 2 (lane % 4) of them.
  const int kchunk = 32 * (lane >> 4) + 16 * ((lane >> 3) & 1);
#pragma unroll
  for (int t = 0; t < MT / 2; ++t) {
    uint32_t sv[2][2], zv[2][2];
    ldsm_x4(sv[0][0], sv[0][1], sv[1][0], sv[1][1], reinterpret_cast<const uint8_t*>(ksc) + 64 * t + kchunk);
    ldsm_x4(zv[0][0], zv[0][1], zv[1][0], zv[1][1], reinterpret_cast<const uint8_t*>(kze) + 64 * t + kchunk);
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int ks = 2 * t + j;
      uint32_t az[4];
      az[0] = zv[j][0];
      az[1] = BITS == 2 ? 0u : zv[j][0];
      az[2] = BITS == 2 ? 0u : zv[j][1];
      az[3] = zv[j][1];
#pragma unroll
      for (int hb = 0; hb < NHB; ++hb) {
        qs[hb][ks][0] = hmul2_u32(qn[hb][ks][0], *reinterpret_cast<const __half2*>(&sv[j][0]));
        qs[hb][ks][1] = hmul2_u32(qn[hb][ks][1], *reinterpret_cast<const __half2*>(&sv[j][1]));
        mma_f16_16816(cz[hb], az, qn[hb][ks][0], qn[hb][ks][1]);
      }
    }
  }
  // scaled scores T = S scale_q = acc (2^24 scale_q / R) + z . qn scale_q, R = 1 for token rows 0-7
  // and 4 (2 bits) or 16 (4 bits) for rows 8-15; cbq: the last term for the lane's two heads
  const float kl = scale_q * 16777216.f, kh = kl * (BITS == 2 ? 0.25f : 0.0625f);
  const uint64_t kl2 = f2_pack(kl, kl), kh2 = f2_pack(kh, kh), sq2 = f2_pack(scale_q, scale_q);
  uint64_t cbq[NHB];
#pragma unroll
  for (int hb = 0; hb < NHB; ++hb) {
    uint64_t cb = f2_pack(cz[hb][0], cz[hb][1]);
    if constexpr (BITS == 2) cb = f2_fma(f2_pack(cz[hb][2], cz[hb][3]), f2_pack(16.f, 16.f), cb);
    cbq[hb] = f2_fma(cb, sq2, 0ull);
  }
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    // even and odd k-steps in separate accumulators (two chains of MT / 2), added afterwards
    float s[NHB][4], s2[NHB][4];
#pragma unroll
    for (int hb = 0; hb < NHB; ++hb)
#pragma unroll
      for (int e = 0; e < 4; ++e) s[hb][e] = s2[hb][e] = 0.f;
#pragma unroll
    for (int ks = 0; ks < MT; ++ks) {
      uint32_t a[4];
      code_frag_sub<BITS>(kw[(half * STEPS + (BITS == 4 ? ks : ks >> 1)) * 32 + lane], ks, a);
#pragma unroll
      for (int hb = 0; hb < NHB; ++hb) mma_f16_16816((ks & 1) ? s2[hb] : s[hb], a, qs[hb][ks][0], qs[hb][ks][1]);
    }
    // s becomes the scaled scores of token rows lane/4 (s[0], s[1]) and lane/4 + 8 (s[2], s[3])
#pragma unroll
    for (int hb = 0; hb < NHB; ++hb) {
      f2_unpack(f2_fma(f2_add(f2_pack(s[hb][0], s[hb][1]), f2_pack(s2[hb][0], s2[hb][1])), kl2, cbq[hb]), s[hb][0],
                s[hb][1]);
      f2_unpack(f2_fma(f2_add(f2_pack(s[hb][2], s[hb][3]), f2_pack(s2[hb][2], s2[hb][3])), kh2, cbq[hb]), s[hb][2],
                s[hb][3]);
    }
    // online softmax over the 16 tokens (rows lane/4 and lane/4 + 8; all valid); inside quantised
    // blocks the running maximum follows every new maximum, so the weights stay <= 1 (fp16 B)
    // The tile maximum decides only whether the running maximum moves, and it moves exactly when
    // some lane's own scores exceed it, so each lane tests its own and the reduction over the
    // tile's lanes runs only then (rarely, once a range has seen its first few blocks).
    float tmax[NHB][2];
    bool need = false;
#pragma unroll
    for (int hb = 0; hb < NHB; ++hb)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        tmax[hb][e] = fmaxf(s[hb][e], s[hb][e + 2]);
        need |= tmax[hb][e] > m[hb][e];
      }
    if (__any_sync(0xffffffffu, need)) {
#pragma unroll
      for (int hb = 0; hb < NHB; ++hb) {
        float corr[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          float mx = tmax[hb][e];
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
          const float mn = fmaxf(m[hb][e], mx);
          corr[e] = ex2_approx(m[hb][e] - mn);
          l[hb][e] *= corr[e];
          m[hb][e] = mn;
        }
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          o[hb][mt][0] *= corr[0];
          o[hb][mt][1] *= corr[1];
          o[hb][mt][2] *= corr[0];
          o[hb][mt][3] *= corr[1];
        }
        zacc[hb][0] *= corr[0];
        zacc[hb][1] *= corr[1];
      }
    }
    // fp16 weights of tokens t0, t1 for this lane's two heads. RS_MMA (2 bits): one fp16-pair
    // exponential each (arguments <= 0: the running maximum covers the block), their row sums out
    // of the zero-term MMA below, from the same fp16 weights. Otherwise fp32 exponentials, the row
    // sums in fp32, then rounded (4 bits: the kernel runs at its register limit, and the fp16 form
    // spilled there and measured slower).
    uint32_t pt0[NHB], pt1[NHB];
#pragma unroll
    for (int hb = 0; hb < NHB; ++hb) {
      const uint64_t nm = f2_pack(-m[hb][0], -m[hb][1]);
      float a0, a1, b0, b1;
      f2_unpack(f2_add(f2_pack(s[hb][0], s[hb][1]), nm), a0, a1);
      f2_unpack(f2_add(f2_pack(s[hb][2], s[hb][3]), nm), b0, b1);
      if constexpr (RS_MMA) {
        pt0[hb] = ex2_f16x2(pack_half2(a0, a1));
        pt1[hb] = ex2_f16x2(pack_half2(b0, b1));
      } else {
        const uint64_t pp0 = f2_pack(ex2_approx(a0), ex2_approx(a1));  // token t0, the lane's two heads
        const uint64_t pp1 = f2_pack(ex2_approx(b0), ex2_approx(b1));  // token t1
        f2_unpack(f2_add(f2_pack(l[hb][0], l[hb][1]), f2_add(pp0, pp1)), l[hb][0], l[hb][1]);
        float x0, x1, y0, y1;
        f2_unpack(pp0, x0, x1);
        f2_unpack(pp1, y0, y1);
        pt0[hb] = pack_half2(x0, x1);
        pt1[hb] = pack_half2(y0, y1);
      }
    }
    constexpr uint32_t k16b = 0x2C002C00u;  // fp16 1/16, both halves
    const __half2 k16 = *reinterpret_cast<const __half2*>(&k16b);
    // The weights as B fragments of the value MMAs, transposed once: the lane holds tokens u0, u0 + 1
    // (pr0) and u0 + 8, u0 + 9 (pr1) of the half for head a8. Each channel group g then scales them
    // by its own per-token value scales, which pair up over the same tokens. For 2 bits the codes of
    // token rows 8-15 sit 16x higher (code_frag_sub), so those weights enter times 1/16 (exact: a
    // power of two on weights <= 1).
    constexpr int NG = D / 32;           // channel groups, one value scale and zero per token each
    const int u0 = 16 * half + 2 * b4;  // the lane's first token of this half in the B layout
    uint32_t pr0[NHB], pr1[NHB], pq1[NHB];
#pragma unroll
    for (int hb = 0; hb < NHB; ++hb) {
      pr0[hb] = movmatrix_t(pt0[hb]);
      pr1[hb] = movmatrix_t(pt1[hb]);
      pq1[hb] = BITS == 2 ? hmul2_u32(pr1[hb], k16) : pr1[hb];
    }
    // the value scales of the lane's four tokens, all NG groups of each: token-major, NG / 2 fp16
    // pairs per token
    uint32_t sv[4][NG / 2];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const __half* row = vsc + (u0 + (j & 1) + 8 * (j >> 1)) * NG;  // 2 NG bytes per token
      if constexpr (NG == 4) {
        const uint2 w2 = *reinterpret_cast<const uint2*>(row);
        sv[j][0] = w2.x;
        sv[j][NG / 2 - 1] = w2.y;
      } else {
#pragma unroll
        for (int k = 0; k < NG / 2; ++k) sv[j][k] = reinterpret_cast<const uint32_t*>(row)[k];
      }
    }
    // Value zero terms sum_t z_tg p_th (and with RS_MMA the row sums sum_t p_th) as one more MMA
    // per half: the A fragment's row g < NG holds the zeros of group g over the half's tokens, rows
    // NG..7 hold ones with RS_MMA (without, they repeat a valid group and are never read; rows 8-15
    // repeat rows 0-7), B the raw transposed weights. Row g of zacc, in the lanes with a8 = g,
    // accumulates group g's term for the lane's two heads; with RS_MMA row NG the row sums. Each half's MMA
    // starts from zero and its sum is added to zacc in fp32: the zero terms of a long range are
    // large against an output in which they cancel with the code terms (by about 400x for
    // N(0,1) values at 64K tokens), and the tensor cores' accumulation, truncating, would carry
    // a bias of that size into the output if zacc were the MMA's accumulator.
    {
      const uint16_t* z16 = reinterpret_cast<const uint16_t*>(vze);
      const int gz = a8 & (NG - 1);
      const bool zrow = a8 < NG;
      uint32_t az[4];
      constexpr uint32_t ones = 0x3C003C00u;  // fp16 1, both halves
      if constexpr (RS_MMA) {
        az[0] = az[1] = zrow ? (uint32_t)z16[u0 * NG + gz] | ((uint32_t)z16[(u0 + 1) * NG + gz] << 16) : ones;
        az[2] = az[3] = zrow ? (uint32_t)z16[(u0 + 8) * NG + gz] | ((uint32_t)z16[(u0 + 9) * NG + gz] << 16) : ones;
      } else {
        az[0] = az[1] = (uint32_t)z16[u0 * NG + gz] | ((uint32_t)z16[(u0 + 1) * NG + gz] << 16);
        az[2] = az[3] = (uint32_t)z16[(u0 + 8) * NG + gz] | ((uint32_t)z16[(u0 + 9) * NG + gz] << 16);
      }
#pragma unroll
      for (int hb = 0; hb < NHB; ++hb) {
        float zd[4];
        mma_f16_16816_c0(zd, az, pr0[hb], pr1[hb]);
        zacc[hb][0] += zd[0];
        zacc[hb][1] += zd[1];
      }
    }
#pragma unroll
    for (int g = 0; g < NG; ++g) {
      // (scale of token u0, scale of token u0 + 1) of group g, and the same for u0 + 8, u0 + 9
      const uint32_t sel = (g & 1) ? 0x7632u : 0x5410u;
      const uint32_t s01 = __byte_perm(sv[0][g >> 1], sv[1][g >> 1], sel);
      const uint32_t s89 = __byte_perm(sv[2][g >> 1], sv[3][g >> 1], sel);
      uint32_t pb[NHB][2];
#pragma unroll
      for (int hb = 0; hb < NHB; ++hb) {
        pb[hb][0] = hmul2_u32(pr0[hb], *reinterpret_cast<const __half2*>(&s01));
        pb[hb][1] = hmul2_u32(pq1[hb], *reinterpret_cast<const __half2*>(&s89));
      }
#pragma unroll
      for (int mm = 0; mm < 2; ++mm) {
        const int mt = 2 * g + mm;
        uint32_t a[4];
        code_frag_sub<BITS>(vw[(half * STEPS + (BITS == 4 ? mt : mt >> 1)) * 32 + lane], mt, a);
#pragma unroll
        for (int hb = 0; hb < NHB; ++hb) mma_f16_16816(o[hb][mt], a, pb[hb][0], pb[hb][1]);
      }
    }
  }
}

// End of a run of quantised groups: take O out of the value codes' power-of-two domain (channel
// row g of each 16-channel tile at 2^-24, row g + 8 at 2^-22 (2 bits) or 2^-20 (4 bits), see
// code_frag_sub; exact), add the value zero terms (group g's, for the lane's two heads, from the
// lane of row g in zacc) and clear them.
template <int D, int BITS, int NHB>
__device__ __forceinline__ void fold_zs(float (&o)[NHB][D / 16][4], float (&zacc)[NHB][4], float (&l)[NHB][2],
                                        int lane) {
  constexpr float R0 = 16777216.f;                         // 2^24
  constexpr float R1 = BITS == 2 ? 4194304.f : 1048576.f;  // 2^22 / 2^20
#pragma unroll
  for (int hb = 0; hb < NHB; ++hb)
#pragma unroll
    for (int mt = 0; mt < D / 16; ++mt) {
      o[hb][mt][0] *= R0;
      o[hb][mt][1] *= R0;
      o[hb][mt][2] *= R1;
      o[hb][mt][3] *= R1;
    }
#pragma unroll
  for (int hb = 0; hb < NHB; ++hb) {
#pragma unroll
    for (int g = 0; g < D / 32; ++g)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const float z = __shfl_sync(0xffffffffu, zacc[hb][e], 4 * g + (lane & 3));
        o[hb][2 * g][e] += z;
        o[hb][2 * g][e + 2] += z;
        o[hb][2 * g + 1][e] += z;
        o[hb][2 * g + 1][e + 2] += z;
      }
    // 2 bits: the row sums (row D / 32 of zacc) into the lane-partial sums, once per head (lanes
    // 0-3)
    if constexpr (BITS == 2) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const float ls = __shfl_sync(0xffffffffu, zacc[hb][e], 4 * (D / 32) + (lane & 3));
        if (lane < 4) l[hb][e] += ls;
      }
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) zacc[hb][e] = 0.f;
  }
}

// Edge w of T chunks cut into W equal ranges: w * T / W. The host bounds T * (W + 1) below 2^32,
// so this stays 32-bit (a 64-bit division is a long software routine).
__device__ __forceinline__ uint32_t range_edge(uint32_t w, uint32_t T, uint32_t W) { return w * T / W; }



__device__ __forceinline__ void fence_acq_rel_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }

// Count this CTA's partial of request b (KV head hk) as arrived; true for the CTA that arrives last
// of the n CTAs holding the request, which then merges. atomicInc wraps the word back to zero on
// the last arrival, so a counter is zero between calls: the workspace starts zeroed and every CTA
// arrives exactly once per split request, also when a wait of its own gave up. One thread.
__device__ __forceinline__ bool cta_arrive(const DraftParams& p, int hk, int b, int n) {
  const uint32_t old = atomicInc(p.ws_ctr + (size_t)hk * VC_MAX_BATCH + b, (uint32_t)(n - 1));
  return old == (uint32_t)(n - 1);
}

// Merge the partials of one CTA for query head h, each given by its o row base (head 0) and lse
// base, in warp order (a null slot holds none); they live in this CTA's shared memory or were
// written by this CTA's warps to the workspace, so plain loads see them after the CTA barrier.
// Output as in merge_head.
template <int D, int NW>
__device__ __forceinline__ void merge_local(const float* const (&po)[NW], const float* const (&pl)[NW], int G,
                                            int h, int lane, bf16* out, float* out_o, float* out_lse) {
  constexpr int CPL = D / 32;
  float lse[NW], v[NW][CPL];
  float M = -INFINITY;
#pragma unroll
  for (int k = 0; k < NW; ++k) {
    lse[k] = -INFINITY;
#pragma unroll
    for (int c = 0; c < CPL; ++c) v[k][c] = 0.f;
    if (po[k]) {
      lse[k] = pl[k][h];
      const float* row = po[k] + (size_t)h * D + CPL * lane;
#pragma unroll
      for (int c = 0; c < CPL; ++c) v[k][c] = row[c];
      M = fmaxf(M, lse[k]);
    }
  }
  if (M == -INFINITY) M = 0.f;
  float L = 0.f, acc[CPL];
#pragma unroll
  for (int c = 0; c < CPL; ++c) acc[c] = 0.f;
#pragma unroll
  for (int k = 0; k < NW; ++k) {
    const float w = exp2f(lse[k] - M);
    L += w;
#pragma unroll
    for (int c = 0; c < CPL; ++c) acc[c] += w * v[k][c];
  }
  const float inv = L > 0.f ? 1.f / L : 0.f;
  if (out) {
    bf16* dst = out + CPL * lane;
    if constexpr (CPL == 4) {
      uint2 o2;
      o2.x = pack_bf16x2(acc[0] * inv, acc[1 % CPL] * inv);
      o2.y = pack_bf16x2(acc[2 % CPL] * inv, acc[3 % CPL] * inv);
      *reinterpret_cast<uint2*>(dst) = o2;
    } else {
      *reinterpret_cast<uint32_t*>(dst) = pack_bf16x2(acc[0] * inv, acc[1 % CPL] * inv);
    }
  } else {
#pragma unroll
    for (int c = 0; c < CPL; ++c) out_o[CPL * lane + c] = acc[c] * inv;
    if (lane == 0) *out_lse = L > 0.f ? M + log2f(L) : -INFINITY;
  }
}

// More than 8 query heads per KV head (NHB = 2) doubles the accumulators: two CTAs per SM.
template <int D, int KIND, int NHB>
__global__ void __launch_bounds__(128, NHB == 1 ? DraftCfg<D, KIND>::CTAS_PER_SM : 2)
    draft_attn_kernel(const __grid_constant__ DraftParams p, const __grid_constant__ typename DraftMapsOf<KIND>::T maps) {
  using C = DraftCfg<D, KIND>;
  constexpr bool BF16_ROWS = KIND == 0;  // kept rows by TMA gather4; otherwise quantised groups by bulk copies
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);  // swizzled stages need 1024 B
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int hk = blockIdx.y;
  const int G = p.G;

  // Each stage completes on its mbarrier: TMA loads (kept rows, quantised groups) by their bytes,
  // window rows (cp.async) by a plain arrive once issued, after which the lanes' cp.async groups
  // are waited for as well. Every stage also commits one cp.async group (possibly empty), so
  // "all but NST-1 groups done" always means "this stage's copies done".
  uint8_t* wb = smem + warp * C::PER_WARP;
  const uint64_t stream_pol = l2_evict_first_policy();  // KV_comp is read once per step
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::BAR_OFF) + warp * C::NST;
  if (lane == 0) {
    for (int s = 0; s < C::NST; ++s) mbar_init(&bars[s], 1);
    fence_mbar_init();
  }
  __shared__ int32_t s_cb[VC_MAX_BATCH + 1];  // first chunk of each request; s_cb[B] = total chunks
  __shared__ int32_t s_wb[VC_MAX_BATCH + 1];  // first warp (of a head) of each request; s_wb[B] = warps
  __shared__ bf16* s_o[VC_MAX_BATCH];         // output rows of each request
  __shared__ int32_t s_wreq[C::NW];           // each warp's request (-1: none)
  __shared__ int32_t s_has[C::NW];            // the warp left a partial in its stage ring
  if (threadIdx.x < p.B) {
    s_cb[threadIdx.x] = p.req[threadIdx.x].chunk_begin;
    s_wb[threadIdx.x] = p.req[threadIdx.x].warp_begin;
    s_o[threadIdx.x] = p.req[threadIdx.x].o;
  }
  if (threadIdx.x == 0) {
    s_cb[p.B] = (int32_t)p.total_chunks;
    s_wb[p.B] = p.n_warp_head;
  }
  __syncthreads();
  // This warp's request rb (warps [s_wb[rb], s_wb[rb+1]) of the head hold it) and its range: the
  // request's chunks cut evenly over its warps (32-bit: the host bounds the products). Warps past
  // the last request's (the tail of the last CTA) hold nothing.
  const int wgl = (int)blockIdx.x * C::NW + warp;
  int rb = 0;
  while (rb + 1 < p.B && s_wb[rb + 1] <= wgl) ++rb;
  const bool in_part = wgl < s_wb[p.B];
  const uint32_t nb = (uint32_t)(s_cb[rb + 1] - s_cb[rb]), kw = (uint32_t)(s_wb[rb + 1] - s_wb[rb]);
  const uint32_t wr = (uint32_t)(wgl - s_wb[rb]);
  const int64_t p0 = s_cb[rb] + (in_part ? (int64_t)range_edge(wr, nb, kw) : 0);
  const int64_t p1 = s_cb[rb] + (in_part ? (int64_t)range_edge(wr + 1, nb, kw) : 0);
  const int n = (int)(p1 - p0);  // may be 0: the warp still takes part in the CTA's merge
  if (lane == 0) s_wreq[warp] = in_part ? rb : -1;
  // Quantised groups: lane k < 6 streams one of a group's six contiguous runs (key codes, key
  // scales, key zeros, value codes, value scales, value zeros); group g's run starts at this
  // head's base plus g times a fixed stride, so the addresses are set up once per warp.
  // With C::GPC = 2 (2-bit), lanes 6-11 stream the chunk's second group into the stage's second half.
  const uint8_t* q_src = nullptr;
  uint32_t q_stride = 0, q_dst = 0;
  int q_grp = 0;
  int q_ng = 0;  // the request's quantised groups
  if (!BF16_ROWS && in_part) q_ng = p.req[rb].n_main / VC_GROUP;
  if (!BF16_ROWS && in_part && lane < 6 * C::GPC) {
    const DraftReqDev& r = p.req[rb];
    const size_t gcap = (size_t)hk * r.ng_cap;  // this head's first group (groups can be appended)
    constexpr uint32_t SC = 2 * D;               // bytes of a group's scales (or zeros), keys or values
    q_grp = lane / 6;
    switch (lane % 6) {
      case 0: q_src = r.kc + gcap * C::KCB, q_stride = C::KCB, q_dst = C::OFF_KC; break;
      case 1: q_src = reinterpret_cast<const uint8_t*>(r.ks) + gcap * SC, q_stride = SC, q_dst = C::OFF_KS; break;
      case 2: q_src = reinterpret_cast<const uint8_t*>(r.kz) + gcap * SC, q_stride = SC, q_dst = C::OFF_KZ; break;
      case 3: q_src = r.vc + gcap * C::KCB, q_stride = C::KCB, q_dst = C::OFF_VC; break;
      case 4: q_src = reinterpret_cast<const uint8_t*>(r.vs) + gcap * SC, q_stride = SC, q_dst = C::OFF_VS; break;
      default: q_src = reinterpret_cast<const uint8_t*>(r.vz) + gcap * SC, q_stride = SC, q_dst = C::OFF_VZ; break;
    }
    q_dst += q_grp * C::QRAW;
  }
  pdl_launch_dependents();
  // Ordering against the previous kernel in the stream (programmatic dependent launch): queries,
  // kept rows and indices are never written by a draft step, verify or accept, so with p.early the
  // warp streams them at once and waits only before it reads window rows (the previous step
  // appended one), stores this step's row, or writes outputs and partials (the previous step's
  // merges may still be reading the workspace).
  bool waited = !p.early;
  if (waited) pdl_wait();
  auto ensure_wait = [&]() {
    if (!waited) {
      pdl_wait();
      waited = true;
    }
  };

  // chunk i of this warp -> (request, chunk within request); a warp holds one request only
  int cur_row = 0, cur_issue = 0, cur_proc = 0;
  auto locate = [&](int i, int& b, int& lc, int& /*cursor*/) {
    b = rb;
    lc = (int)(p0 + i - s_cb[rb]);
  };
  // the row a lane copies for chunk i (its lane & 15 row), or -1 for a padding row: a token index
  // for kept rows (a negative one from the caller becomes INT_MAX, so the bounds check flags it),
  // a window row number for window chunks; loaded one stage ahead of its copy
  auto row_of = [&](int i) -> int {
    int b, lc;
    locate(i, b, lc, cur_row);
    const DraftReqDev& r = p.req[b];
    const int row = lane & 15;
    if (lc < r.n_mc) {
      if (!BF16_ROWS) return 0;
      const int j = lc * 16 + row;
      if (j >= r.n_main) return -1;
      if (r.compact) return j;
      const int t = __ldg(r.idx + j);
      return t < 0 ? INT_MAX : t;
    }
    const int j = (lc - r.n_mc) * 16 + row;
    return j <= r.n_win ? j : -1;
  };

  auto issue = [&](int i, int st, int t) {
    int b, lc;
    locate(i, b, lc, cur_issue);
    const DraftReqDev& r = p.req[b];
    uint8_t* sb = wb + st * C::STAGE;
    if (lc < r.n_mc) {
      if constexpr (!BF16_ROWS) {
        // the chunk's quantised groups (C::GPC, fewer at an odd end): six contiguous runs each, one
        // per lane (set up above)
        const int g0 = C::GPC * lc;
        const int ngc = q_ng - g0 < C::GPC ? q_ng - g0 : C::GPC;
        if (lane == 0) mbar_arrive_expect_tx(&bars[st], C::QRAW * ngc);
        __syncwarp();
        if (lane < 6 * ngc)
          bulk_g2s_hint(sb + q_dst, q_src + (size_t)(g0 + q_grp) * q_stride, q_stride, &bars[st], stream_pol);
      } else {
        // 16 kept rows by TMA gather4: lane l < G4_OPS loads rows 4(l%4)..4(l%4)+3 of one 64-channel
        // block of K or V. A row past the kept count repeats the chunk's first row, a kept row
        // whose probability the softmax sets to zero.
        int coord = -1;
        if (t >= 0) {
          if ((int64_t)t < r.rows_cap)
            coord = (int)((int64_t)hk * r.rows_cap + t);
          else
            set_status(p.dev_status, VC_DEV_BOUNDS);
        }
        const int first = __shfl_sync(0xffffffffu, coord, 0);
        if (coord < 0) coord = first < 0 ? 0 : first;
        const int g4 = lane & 3;
        const int c0 = __shfl_sync(0xffffffffu, coord, 4 * g4);
        const int c1 = __shfl_sync(0xffffffffu, coord, 4 * g4 + 1);
        const int c2 = __shfl_sync(0xffffffffu, coord, 4 * g4 + 2);
        const int c3 = __shfl_sync(0xffffffffu, coord, 4 * g4 + 3);
        if (lane == 0) mbar_arrive_expect_tx(&bars[st], 2 * C::TILE);
        __syncwarp();
        if (lane < C::G4_OPS) {
          const int h = (lane >> 2) % C::HALVES, isv = (lane >> 2) / C::HALVES;
          tma_gather4(sb + isv * C::TILE + h * C::BLK + g4 * 512, &maps.kv[b][isv], 64 * h, c0, c1, c2, c3,
                      &bars[st], stream_pol);
        }
      }
      // cp.async groups count stages only where window tiles fit a stage; with WIN_SPANS a window
      // chunk is issued alone and waited for with everything (the quantised kernels)
      if constexpr (!C::WIN_SPANS) cp_async_commit();
      return;
    }
    ensure_wait();  // window rows: the previous step appended one
    if constexpr (C::WIN_SPANS) sb = wb;  // a window tile takes the whole ring (issued when it is empty)
    // 16 bf16 rows: lane & 15 names the row; lanes 0-15 own its K row, lanes 16-31 its V row
    const bool isv = lane >= 16;
    const bf16* src = nullptr;
    if (t >= 0)
      src = t < r.n_win ? (isv ? r.v_win : r.k_win) + ((size_t)hk * r.win_cap + t) * D
                        : (isv ? r.v_new : r.k_new) + (size_t)hk * D;
    // instruction k copies rows RPI*k .. RPI*k+RPI-1 of the 32 (K rows, then V rows): lane l moves
    // 16-byte piece l % PPR of its row into the swizzled tile; rows without a source are zero-filled
    constexpr int PPR = C::ROWB / 16;  // pieces per row: 16 (d=128) or 8 (d=64)
    constexpr int RPI = 32 / PPR;      // rows per instruction
    const unsigned long long sp = reinterpret_cast<unsigned long long>(src);
    const int piece = lane % PPR;
#pragma unroll
    for (int k = 0; k < 32 / RPI; ++k) {
      const int R = RPI * k + lane / PPR;
      const unsigned long long rs = __shfl_sync(0xffffffffu, sp, R);
      uint8_t* dst = sb + (R >= 16 ? C::TILE : 0) + sw_off(R & 15, piece);
      const uint8_t* srow = reinterpret_cast<const uint8_t*>(rs);
      cp_async16(dst, srow ? srow + piece * 16 : reinterpret_cast<const uint8_t*>(r.k_new), srow ? 16u : 0u);
    }
    cp_async_commit();
    if (lane == 0) mbar_arrive(&bars[st]);
  };

  float o[NHB][C::MT][4];
  float m[NHB][2], l[NHB][2];
  float zacc[NHB][4];  // value zero terms of quantised blocks not yet folded into o (row g: group g)
  uint32_t qb[NHB][C::MT][2];
  int cur_b = -1;
  bool zs_live = false;

  auto reset = [&]() {
#pragma unroll
    for (int hb = 0; hb < NHB; ++hb) {
#pragma unroll
      for (int mt = 0; mt < C::MT; ++mt)
#pragma unroll
        for (int e = 0; e < 4; ++e) o[hb][mt][e] = 0.f;
      m[hb][0] = m[hb][1] = -INFINITY;
      l[hb][0] = l[hb][1] = 0.f;
#pragma unroll
      for (int e = 0; e < 4; ++e) zacc[hb][e] = 0.f;
    }
  };
  // Q^T B fragments: k = channel 16ks + 2(lane%4) (+8), n = head 8hb + lane/4 (zero beyond G)
  auto load_q = [&](int b) {
    const bf16* qbase = p.req[b].q + (size_t)hk * G * D;
#pragma unroll
    for (int hb = 0; hb < NHB; ++hb) {
      const int h = 8 * hb + (lane >> 2);
#pragma unroll
      for (int ks = 0; ks < C::MT; ++ks) {
        const int c = 16 * ks + 2 * (lane & 3);
        qb[hb][ks][0] = h < G ? __ldg(reinterpret_cast<const unsigned int*>(qbase + h * D + c)) : 0u;
        qb[hb][ks][1] = h < G ? __ldg(reinterpret_cast<const unsigned int*>(qbase + h * D + c + 8)) : 0u;
      }
    }
  };
  // For quantised blocks the same registers hold the query as fp16 scaled by 2^-E, E the exponent
  // of the warp's largest |q| (so |qn| < 1 and the scaled query s o qn stays below the key scale);
  // the softmax then uses scale_q = scale_log2 * 2^E. Window tiles reload the bf16 query.
  float scale_q = p.scale_log2;
  bool q_f16 = false;
  auto load_qn = [&](int b) {
    load_q(b);
    float mx = 0.f;
#pragma unroll
    for (int hb = 0; hb < NHB; ++hb)
#pragma unroll
      for (int ks = 0; ks < C::MT; ++ks)
#pragma unroll
        for (int r2 = 0; r2 < 2; ++r2) {
          const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&qb[hb][ks][r2]));
          mx = fmaxf(mx, fmaxf(fabsf(f.x), fabsf(f.y)));
        }
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    int E = 0;
    if (mx > 0.f) frexpf(mx, &E);  // mx = f 2^E with f in [0.5, 1)
    const float inv = ldexpf(1.f, -E);
#pragma unroll
    for (int hb = 0; hb < NHB; ++hb)
#pragma unroll
      for (int ks = 0; ks < C::MT; ++ks)
#pragma unroll
        for (int r2 = 0; r2 < 2; ++r2) {
          // 2 bits: channels 8-15 of each k-step divided by 16 as well (their key codes sit 16x
          // higher in the subnormal operands, see qblock_attend)
          const float sc = (C::BITS == 2 && r2 == 1) ? inv * 0.0625f : inv;
          const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&qb[hb][ks][r2]));
          qb[hb][ks][r2] = pack_half2(f.x * sc, f.y * sc);
        }
    scale_q = ldexpf(p.scale_log2, E);
    q_f16 = true;
  };
  // end of the warp's range: its (o, lse) partial, normalised, into its drained stage ring as
  // [G][D] o then [G] lse. The lane holds O^T[channel 16mt + lane/4 (+8)][head 8hb + 2(lane%4) + e].
  auto finish = [&]() {
#pragma unroll
    for (int hb = 0; hb < NHB; ++hb)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        float lt = l[hb][e];
        lt += __shfl_xor_sync(0xffffffffu, lt, 4);
        lt += __shfl_xor_sync(0xffffffffu, lt, 8);
        lt += __shfl_xor_sync(0xffffffffu, lt, 16);
        const int h = 8 * hb + 2 * (lane & 3) + e;
        if (h >= G) continue;
        const float inv = lt > 0.f ? 1.f / lt : 0.f;
        float* dst = reinterpret_cast<float*>(wb) + h * D;
#pragma unroll
        for (int mt = 0; mt < C::MT; ++mt) {
          const int c = 16 * mt + (lane >> 2);
          dst[c] = o[hb][mt][e] * inv;
          dst[c + 8] = o[hb][mt][e + 2] * inv;
        }
        if ((lane >> 2) == 0) reinterpret_cast<float*>(wb)[G * D + h] = lt > 0.f ? m[hb][e] + log2f(lt) : -INFINITY;
      }
  };

  bool aborted = false;
  // Chunks are issued in order, NST ahead; chunk k completes on bars[k % NST]. When a window tile
  // spans the ring (WIN_SPANS), the warp's window chunks (they follow all its KV_comp chunks) are
  // issued one at a time, each once the chunk before it has been read.
  int iw = n;  // the warp's first window chunk
  if constexpr (C::WIN_SPANS) {
    const int64_t first_win = (int64_t)s_cb[rb] + p.req[rb].n_mc - p0;
    iw = first_win < 0 ? 0 : (first_win < n ? (int)first_win : n);
  }
  int issued = 0;
  while (issued < n && issued < C::NST && (issued < iw || issued == 0)) {
    issue(issued, issued, row_of(issued));
    ++issued;
  }
  for (int k = issued; k < C::NST; ++k) cp_async_commit();  // one group per stage in flight
#pragma unroll 1
  for (int i = 0; i < n; ++i) {
    const int st = i % C::NST;
    const bool win_span = C::WIN_SPANS && i >= iw;
    const int t_next = (!C::WIN_SPANS && i + C::NST < n) ? row_of(i + C::NST) : -1;  // prefetch: used after this chunk
    int b, lc;
    locate(i, b, lc, cur_proc);
    if (b != cur_b) {
      if (!BF16_ROWS && zs_live) {
        fold_zs<D, C::BITS, NHB>(o, zacc, l, lane);
        zs_live = false;
      }
      reset();
      if (!BF16_ROWS && lc < p.req[b].n_mc)
        load_qn(b);
      else
        load_q(b);
      cur_b = b;
      if (lc == 0) {
        // fused append of the step's K/V row (the warp holding the request's first chunk)
        ensure_wait();
        const DraftReqDev& r = p.req[b];
        constexpr int V16 = C::ROWB / 16;
        const int l16 = lane & 15;
        if (l16 < V16) {
          const uint4* src = reinterpret_cast<const uint4*>((lane < 16 ? r.k_new : r.v_new) + (size_t)hk * D);
          bf16* dst_row = (lane < 16 ? r.k_win : r.v_win) + ((size_t)hk * r.win_cap + r.n_win) * D;
          reinterpret_cast<uint4*>(dst_row)[l16] = __ldg(src + l16);
        }
      }
    }
    if (win_span)
      cp_async_wait<0>();            // nothing else is in flight: all this lane's copies
    else if constexpr (!C::WIN_SPANS)
      cp_async_wait<C::NST - 1>();   // this lane's copies of chunk i have landed
    __syncwarp();                    // ... and every other lane's
    if (!mbar_wait_bounded(&bars[st], (i / C::NST) & 1, p.dev_status, p.spin_limit)) {
      // give up on this range, but not on the copies already issued into the ring (this chunk's
      // and the ones after it): wait for them with the full bound so that no copy is still
      // writing shared memory when the CTA exits
      for (int j = i; j < issued; ++j) mbar_wait_bounded(&bars[j % C::NST], (j / C::NST) & 1, p.dev_status);
      aborted = true;
      break;
    }
    const DraftReqDev& r = p.req[b];
    uint8_t* sb = win_span ? wb : wb + st * C::STAGE;
    if (!BF16_ROWS && lc < r.n_mc) {
      qblock_attend<D, C::BITS, NHB>(sb, scale_q, qb, o, m, l, zacc, lane);
      if (C::GPC == 2 && C::GPC * lc + 1 < q_ng)
        qblock_attend<D, C::BITS, NHB>(sb + C::QRAW, scale_q, qb, o, m, l, zacc, lane);
      zs_live = true;
    } else {
      if (!BF16_ROWS && zs_live) {
        fold_zs<D, C::BITS, NHB>(o, zacc, l, lane);
        zs_live = false;
      }
      if (!BF16_ROWS && q_f16) {
        load_q(b);
        q_f16 = false;
      }
      const int cnt = (lc < r.n_mc) ? min(16, r.n_main - lc * 16) : min(16, r.n_win + 1 - (lc - r.n_mc) * 16);
      tile_attend<D, NHB, !BF16_ROWS>(sb, sb + C::TILE, cnt, p.scale_log2, qb, o, m, l, lane);
    }
    __syncwarp();
    // next issue: a KV_comp chunk into the stage just read (NST ahead), or -- spanning the ring --
    // a window chunk once this was the last chunk in flight
    const bool go = C::WIN_SPANS ? (issued < n && (issued < iw ? issued == i + C::NST : issued == i + 1))
                                 : (i + C::NST < n);
    if (go) {
      fence_proxy_async_smem();  // this warp's reads of the stage come before the TMA overwrites it
      // (with WIN_SPANS the row is needed for window chunks only: a quantised chunk ignores it)
      issue(issued, issued % C::NST, C::WIN_SPANS ? (issued >= iw ? row_of(issued) : 0) : t_next);
      ++issued;
    } else if constexpr (!C::WIN_SPANS) {
      cp_async_commit();  // empty group: the wait above always leaves NST-1 groups pending
    }
  }
  cp_async_wait<0>();
  const bool has = !aborted && cur_b >= 0;
  if (has) {
    if (!BF16_ROWS && zs_live) fold_zs<D, C::BITS, NHB>(o, zacc, l, lane);
    finish();  // the stage ring is drained: the partial stays in shared memory
  }
  if (lane == 0) s_has[warp] = has ? 1 : 0;

  // Merge, per request held by this CTA (by the partition, so every CTA arrives once for each of
  // its requests even when a wait of its own gave up): the CTA's warps' partials of the request
  // (one query head per warp) go into the output when the request lies in this CTA alone, else
  // into the CTA's partial slot (CTA + request); the CTA that arrives last among the request's
  // CTAs then merges their partials, in CTA order, into the output.
  ensure_wait();  // the workspace and outputs are written below
  __syncthreads();
  __shared__ int s_last;
  const int cx = blockIdx.x, NC = p.n_cta_head;
  int bA = VC_MAX_BATCH, bB = -1;
#pragma unroll
  for (int k = 0; k < C::NW; ++k) {
    if (s_wreq[k] >= 0 && s_wreq[k] < bA) bA = s_wreq[k];
    if (s_wreq[k] > bB) bB = s_wreq[k];
  }
#pragma unroll 1
  for (int b = bA; b <= bB; ++b) {
    const int c0 = s_wb[b] / C::NW, c1 = (s_wb[b + 1] - 1) / C::NW;  // CTAs holding b
    const bool one_cta = c0 == c1;
    const float* po[C::NW];
    const float* pl[C::NW];
#pragma unroll
    for (int k = 0; k < C::NW; ++k) {
      po[k] = (s_wreq[k] == b && s_has[k]) ? reinterpret_cast<const float*>(smem + k * C::PER_WARP) : nullptr;
      pl[k] = po[k] ? po[k] + G * D : nullptr;
    }
    bf16* orow = s_o[b] + (size_t)hk * G * D;
    const int64_t cslot = (int64_t)hk * (NC + p.B) + cx + b;
    for (int h = warp; h < G; h += C::NW)
      merge_local<D, C::NW>(po, pl, G, h, lane, one_cta ? orow + (size_t)h * D : nullptr,
                            p.ws_o + (cslot * G + h) * D, p.ws_lse + cslot * G + h);
    if (one_cta) continue;
    // The barrier orders every thread's CTA-partial stores before thread 0's release fence and
    // arrival; the last arriver's acquire fence and the second barrier order the other CTAs'
    // partials before this CTA reads them.
    __syncthreads();
    if (threadIdx.x == 0) {
      fence_acq_rel_gpu();
      const bool last = cta_arrive(p, hk, b, c1 - c0 + 1);
      if (last) fence_acq_rel_gpu();
      s_last = last ? 1 : 0;
    }
    __syncthreads();
    if (s_last) {
      for (int h = warp; h < G; h += C::NW)
        merge_head<D>(p.ws_o, p.ws_lse, (int64_t)hk * (NC + p.B) + b + c0, c1 - c0 + 1, G, h, lane,
                      orow + (size_t)h * D, nullptr, nullptr);
    }
  }
}

template <int D, int KIND, int NHB>
static cudaError_t launch_draft_t(const DraftParams& p, const DraftMaps* maps, int ctas_per_head, cudaStream_t s) {
  using C = DraftCfg<D, KIND>;
  static std::atomic<uint64_t> attr{0};
  {
    cudaError_t e = raise_smem_limit(draft_attn_kernel<D, KIND, NHB>, C::SMEM, attr);
    if (e != cudaSuccess) return e;
  }
  cudaError_t e;
  if constexpr (KIND == 0) {
    e = launch_pdl(draft_attn_kernel<D, KIND, NHB>, dim3(ctas_per_head, p.Hkv), dim3(128), C::SMEM, s, p, *maps);
  } else {
    e = launch_pdl(draft_attn_kernel<D, KIND, NHB>, dim3(ctas_per_head, p.Hkv), dim3(128), C::SMEM, s, p,
                   DraftNoMaps{0});
  }
  return e;
}

template <int D, int KIND>
static cudaError_t launch_draft_g(const DraftParams& p, const DraftMaps* maps, int ctas_per_head, cudaStream_t s) {
  return p.G <= 8 ? launch_draft_t<D, KIND, 1>(p, maps, ctas_per_head, s)
                  : launch_draft_t<D, KIND, 2>(p, maps, ctas_per_head, s);
}

int draft_ctas_per_sm(int G, int kind) {
  if (G > 8) return 2;
  return kind == 0 ? DraftCfg<128, 0>::CTAS_PER_SM : DraftCfg<128, 2>::CTAS_PER_SM;
}

cudaError_t launch_draft(const DraftParams& p, const DraftMaps* maps, int d, int kind, int ctas_per_head,
                         cudaStream_t s) {
  if (kind == 0 && !maps) return cudaErrorInvalidValue;
  if (d == 128) {
    if (kind == 0) return launch_draft_g<128, 0>(p, maps, ctas_per_head, s);
    if (kind == 2) return launch_draft_g<128, 2>(p, maps, ctas_per_head, s);
    if (kind == 4) return launch_draft_g<128, 4>(p, maps, ctas_per_head, s);
  } else if (d == 64) {
    if (kind == 0) return launch_draft_g<64, 0>(p, maps, ctas_per_head, s);
    if (kind == 2) return launch_draft_g<64, 2>(p, maps, ctas_per_head, s);
    if (kind == 4) return launch_draft_g<64, 4>(p, maps, ctas_per_head, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace vc
