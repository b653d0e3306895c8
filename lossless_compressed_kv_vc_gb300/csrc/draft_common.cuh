// Shared by the two draft kernels: quantised KV_comp blocks in their stored form (the LOP3 turn of
// stored codes into exact fp16 MMA operands; the layout is described in compress.cu) and the merge
// of per-CTA (o, lse) partials.
#pragma once

#include "vc_internal.cuh"

namespace vc {

// Two stored codes of a block word as one fp16x2 operand, by a single LOP3: the code at bit position
// P of each 16-bit half (P + BITS <= 8) lands in the mantissa of 2^(10-P), giving the exact value
// 2^(10-P) + code (code_centred_f16x2 takes the offset and the centre off again).
template <int BITS, int P>
__device__ __forceinline__ uint32_t code_f16x2(uint32_t w) {
  constexpr uint32_t m = ((1u << BITS) - 1u) << P;
  constexpr uint32_t e = (25u - P) << 10;  // fp16 exponent field of 2^(10-P)
  return (w & (m | (m << 16))) | (e | (e << 16));
}

// The value side's A fragment as exact, centred fp16 codes: code - C0 with C0 = (2^BITS - 1) / 2, so
// the products with the B operand (scale o weight) have zero mean and the fp32 accumulator only ever
// holds sums of the output's own size. (Leaving the codes offset by 2^(10-P) and removing the offset
// with a second MMA adds and then subtracts 2^(10-P) * sum(scale o weight) in the accumulator; at
// 65K tokens the truncation of those transients reached 0.5% of the output.) The word is shifted so
// that each code sits at an odd bit position P' (P' + BITS <= 9): 2^(10-P') + C0 is then exact in
// fp16 (a half-integer needs an ulp <= 0.5, i.e. 2^(10-P') <= 512), and one HSUB2 per register
// leaves code - C0 exactly.
// fp16 bits of 2^E + C0 (C0 = (2^BITS - 1) / 2), both halves of the pair, as a compile-time
// immediate: exponent field E + 15, fraction field C0 * 2^(10-E) (an integer when the value is
// exact in fp16, which the assertion checks).
template <int BITS, int E>
__host__ __device__ constexpr uint32_t centre_f16x2() {
  constexpr uint32_t c0x2 = (1u << BITS) - 1u;           // 2 C0 (an integer)
  constexpr uint32_t frac = (c0x2 << 10) >> (E + 1);    // C0 * 2^(10-E)
  static_assert(((c0x2 << 10) % (1u << (E + 1))) == 0, "2^E + C0 exact in fp16");
  constexpr uint32_t h = ((uint32_t)(E + 15) << 10) | frac;
  return h | (h << 16);
}

template <int BITS, int P>
__device__ __forceinline__ uint32_t code_centred_f16x2(uint32_t w) {
  constexpr uint32_t cb = centre_f16x2<BITS, 10 - P>();
  const uint32_t x = code_f16x2<BITS, P>(w);
  const __half2 r = __hsub2(*reinterpret_cast<const __half2*>(&x), *reinterpret_cast<const __half2*>(&cb));
  return *reinterpret_cast<const uint32_t*>(&r);
}

template <int BITS>
__device__ __forceinline__ void code_frag_centred(uint32_t w, int ks, uint32_t (&a)[4]) {
  if constexpr (BITS == 2) {
    const uint32_t x = (ks & 1) ? (w >> 7) : (w << 1);  // codes of pair i at bits 2i + 1 of each half
    a[0] = code_centred_f16x2<2, 1>(x);
    a[1] = code_centred_f16x2<2, 3>(x);
    a[2] = code_centred_f16x2<2, 5>(x);
    a[3] = code_centred_f16x2<2, 7>(x);
  } else {
    const uint32_t x0 = w << 1, x1 = w >> 7;  // codes at bits 1 and 5 of each half
    a[0] = code_centred_f16x2<4, 1>(x0);
    a[1] = code_centred_f16x2<4, 5>(x0);
    a[2] = code_centred_f16x2<4, 1>(x1);
    a[3] = code_centred_f16x2<4, 5>(x1);
  }
}

// The four A-fragment registers of k-step ks held by block word w (see the block layout in
// compress.cu: 2-bit words carry two k-steps, the odd one in bits 8-15 of each half; 4-bit words
// one, registers 2 and 3 in bits 8-15) as exact fp16 subnormals: each code keeps its bit position P
// inside its 16-bit half and the exponent field stays zero, so the register holds code x 2^(P-24)
// exactly, with no offset to remove (one shift per word, one AND per register). The positions:
// 2-bit registers 0-3 at P = 0, 2, 4, 6, 4-bit registers 0 and 2 at P = 0, 1 and 3 at P = 4.
// Registers 0 and 1 hold MMA columns (k) 0-7 of the k-step, 2 and 3 columns 8-15; registers 0 and
// 2 rows 0-7, 1 and 3 rows 8-15. Relative to register 0, rows 8-15 therefore sit 4x higher (2 bits)
// or 16x (4 bits) and columns 8-15 16x higher (2 bits) or equal (4 bits). Keys (rows = tokens,
// columns = channels) take the column factor into the query and the row factor into the score
// scale; values (rows = channels, columns = tokens) take the column factor into the weights of
// tokens 8-15 and leave channel row g at 2^-24 and row g + 8 at 2^-22 (2 bits) or 2^-20 (4 bits),
// which fold_zs takes back.
template <int BITS>
__device__ __forceinline__ void code_frag_sub(uint32_t w, int ks, uint32_t (&a)[4]) {
  if constexpr (BITS == 2) {
    const uint32_t x = (ks & 1) ? (w >> 8) : w;
    a[0] = x & 0x00030003u;
    a[1] = x & 0x000C000Cu;
    a[2] = x & 0x00300030u;
    a[3] = x & 0x00C000C0u;
  } else {
    const uint32_t x = w >> 8;
    a[0] = w & 0x000F000Fu;
    a[1] = w & 0x00F000F0u;
    a[2] = x & 0x000F000Fu;
    a[3] = x & 0x00F000F0u;
  }
}

__device__ __forceinline__ uint32_t hmul2_u32(uint32_t x, __half2 y) {
  const __half2 r = __hmul2(*reinterpret_cast<const __half2*>(&x), y);
  return *reinterpret_cast<const uint32_t*>(&r);
}

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
  const __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// Merge n partials of one query head h (consecutive slots s0 .. s0 + n - 1 of po / pl, in slot
// order): o = sum_k 2^(lse_k - M) o_k / sum_k 2^(lse_k - M), lse = M + log2(sum_k 2^(lse_k - M)),
// M the largest lse (log2 domain). One warp; a lane owns D/32 channels. Partials are taken eight
// at a time with a running maximum (the earlier sum is rescaled when it grows), and each batch's
// lse values and rows are all loaded before any is used, so a batch costs one trip to L2. Writes
// the bf16 output row `out` if given, else the merged partial (out_o, out_lse). The partials come
// from other warps of this launch, so they are read through L2.
template <int D>
__device__ __forceinline__ void merge_head(const float* po, const float* pl, int64_t s0, int n, int G, int h, int lane,
                                           bf16* out, float* out_o, float* out_lse) {
  constexpr int CPL = D / 32;
  constexpr int NB = 8;
  float M = -INFINITY, L = 0.f, acc[CPL];
#pragma unroll
  for (int c = 0; c < CPL; ++c) acc[c] = 0.f;
#pragma unroll 1
  for (int j0 = 0; j0 < n; j0 += NB) {
    float lse[NB], v[NB][CPL];
#pragma unroll
    for (int jj = 0; jj < NB; ++jj) {
      lse[jj] = -INFINITY;
#pragma unroll
      for (int c = 0; c < CPL; ++c) v[jj][c] = 0.f;
      if (j0 + jj < n) {
        const int64_t slot = s0 + j0 + jj;
        lse[jj] = __ldcg(pl + slot * G + h);
        const float* row = po + (slot * G + h) * D + CPL * lane;
        if constexpr (CPL == 4) {
          const float4 t = __ldcg(reinterpret_cast<const float4*>(row));
          v[jj][0] = t.x;
          v[jj][1 % CPL] = t.y;
          v[jj][2 % CPL] = t.z;
          v[jj][3 % CPL] = t.w;
        } else {
          const float2 t = __ldcg(reinterpret_cast<const float2*>(row));
          v[jj][0] = t.x;
          v[jj][1 % CPL] = t.y;
        }
      }
    }
    float mb = M;
#pragma unroll
    for (int jj = 0; jj < NB; ++jj) mb = fmaxf(mb, lse[jj]);
    if (mb == -INFINITY) continue;  // nothing to add yet (empty partials)
    const float f = exp2f(M - mb);  // 0 on the first batch (M = -inf)
    L *= f;
#pragma unroll
    for (int c = 0; c < CPL; ++c) acc[c] *= f;
#pragma unroll
    for (int jj = 0; jj < NB; ++jj) {
      const float w = exp2f(lse[jj] - mb);  // 0 for padding and empty partials
      L += w;
#pragma unroll
      for (int c = 0; c < CPL; ++c) acc[c] += w * v[jj][c];
    }
    M = mb;
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

}  // namespace vc
