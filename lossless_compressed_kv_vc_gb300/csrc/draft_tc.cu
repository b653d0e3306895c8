// Draft decode attention over quantised KV_comp on the 5th-generation tensor cores (tcgen05).
//
// "VeriCache: Turning Lossy KV Cache into Lossless LLM Inference", "Core algorithm" step 1
// (drafting reads the compressed cache KV_comp), "Architecture support" (KIVI-style groupwise
// asymmetric 2/4-bit quantisation), "Cross-resource staggering (P1)" (drafting is bound by HBM
// bandwidth: it streams KV_comp once per draft step).
//
// Same call, inputs and result as the mma.sync kernel of draft.cu, for d = 128 with up to 8 query
// heads per KV head, reading the same stored blocks; chosen with VC_DRAFT_TC=1 (the mma.sync kernel
// stays the default: with at most 8 heads both products have N = 32, and an M = 128 tcgen05 MMA
// costs the same ~46 cycles for any N <= 64, so a 128-token block's 17 MMAs take ~775 cycles of
// the tensor pipe -- about the whole budget of a block at the HBM rate -- while the roles below
// each hold one block at a time; measured about 3x slower).
//
// Work: a KV head's requests are cut into units -- quantised blocks of four 32-token groups (128
// tokens), then window blocks of up to 128 bf16 rows (the residual and the drafted rows, the last
// being this step's own row) -- and the units of a grid row (one KV head) are split over its CTAs
// by a cost weight (a window block streams about WW quantised blocks' bytes). A CTA holds one SM
// (its TMEM and most of its shared memory) and runs its units in order through a warp-specialised
// pipeline; the units of one request in one CTA form a segment, whose (o, lse) partial goes to the
// output (the request lies in this CTA alone) or to a CTA partial merged by the last CTA to arrive.
//
// Per unit, with G <= 8 query heads padded to 8 and the block's four groups g stacked in the MMA's
// N = 32 columns (n = 8g + h):
//   K warps (one per TMEM lane quarter = group g of the block): the group's key codes, centred
//     (code - C0, exact fp16), go straight from the stored word to TMEM as the A operand of
//     S = A_K B_QK^T (lane = token, M = 128); the B rows 8g..8g+7 are the query scaled by the
//     group's key scales (fp16(qn o s_g), written with stmatrix), and a ninth k-step against two
//     ones columns of A adds the group's zero term sum_c qn_c (z_c + C0 s_c) (an mma.sync dot
//     product, stored as an fp16 hi/lo pair). A token reads only its own group's 8 columns.
//   V warps (one per lane quarter = 32-channel group of the value scales): the value codes,
//     centred, go to TMEM as the A operand of O = A_V B_PV^T (lane = channel, K = token).
//   softmax warps (one per quarter = group g): S from TMEM in the accumulator fragment order, the
//     block maximum across the four warps (a named barrier), weights p <= 1 (the running maximum
//     follows every new maximum; O, in TMEM, is rescaled when it moves), and B_PV rows
//     8cg + h = fp16(p s_{t,cg}) (the value scale of token t and channel group cg), written
//     transposed with stmatrix; the value zero term sum_t p (z + C0 s) accumulates in registers.
//     A channel reads only its own group's 8 columns of O.
//   MMA warp: one thread issues S(j) = 9 MMAs, then O += P V of unit j - 1 = 8 MMAs (M 128, N 32).
//   producer warp: one bulk copy per stored array per block (codes, scales, zeros of four groups),
//     window rows by 16-byte cp.async into a 128-byte-swizzled tile (bf16; loaded with ldmatrix
//     into the same A fragment order, the MMAs then in bf16).
// Every wait is bounded; a wait that gives up records VC_DEV_TIMEOUT and stops the CTA's pipeline
// (the others see a shared flag), which still waits for its copies and MMAs before it frees TMEM.
#include "tc05.cuh"
#include "draft_common.cuh"

#include <math.h>

namespace vc {

template <int BITS>
struct QtCfg {
  static constexpr int D = 128;
  static constexpr int NQ = 8;              // query heads per KV head (padded)
  static constexpr int N = 4 * NQ;          // MMA columns: four stacked groups
  static constexpr int KCB = D * 4 * BITS;  // codes of one 32-token group (keys or values), bytes
  static constexpr int SCB = 2 * D;         // key scales (or zeros) of one group
  static constexpr int VSB = 32 * (D / 32) * 2;  // value scales (or zeros) of one group
  static constexpr int STEPS = BITS == 4 ? D / 16 : D / 32;  // code words per (half, lane)
  // stage of one quantised block (four groups), one region per stored array
  static constexpr int OFF_KC = 0;
  static constexpr int OFF_KS = OFF_KC + 4 * KCB;
  static constexpr int OFF_KZ = OFF_KS + 4 * SCB;
  static constexpr int OFF_VC = OFF_KZ + 4 * SCB;
  static constexpr int OFF_VS = OFF_VC + 4 * KCB;
  static constexpr int OFF_VZ = OFF_VS + 4 * VSB;
  static constexpr int GROUP_BYTES = 2 * KCB + 2 * SCB + 2 * VSB;
  static constexpr int STAGE = (OFF_VZ + 4 * VSB + 1023) / 1024 * 1024;
  static constexpr int NST = BITS == 2 ? 6 : 4;
  // window tile: 128 rows of K then of V, bf16, 64-channel column blocks, 128-byte swizzle
  static constexpr int WBLK = 128 * 128;
  static constexpr int WBUF = 4 * WBLK;
  static constexpr int WW = BITS == 2 ? 6 : 3;  // cost of a window block in quantised blocks
  // B operands (K-major, 128-byte swizzle, 64-element column blocks of N rows)
  static constexpr int KB = N * 128;  // one column block
  static constexpr int BQK = 3 * KB;  // channels 0-63, 64-127, and the zero-term extension
  static constexpr int BPV = 2 * KB;  // tokens 0-63, 64-127
  static constexpr int OFF_RING = 0;
  static constexpr int OFF_WIN = OFF_RING + NST * STAGE;
  static constexpr int OFF_BQK = OFF_WIN + WBUF;
  static constexpr int OFF_BPV = OFF_BQK + 2 * BQK;
  static constexpr int OFF_MISC = OFF_BPV + 2 * BPV;
  static constexpr int MISC = 4096;
  static constexpr int SMEM = OFF_MISC + MISC + 1024;  // + slack to align the base to 1024 B
  // TMEM columns
  static constexpr uint32_t T_AK = 0;     // two buffers of 72 (64 + the extension k-step)
  static constexpr uint32_t T_AV = 160;   // two buffers of 64
  static constexpr uint32_t T_S = 288;    // two buffers of 32
  static constexpr uint32_t T_O = 352;    // 32
  static constexpr uint32_t T_COLS = 512;
  static_assert(SMEM <= 227 * 1024, "one CTA per SM");
  static_assert(STAGE % 1024 == 0 && GROUP_BYTES % 16 == 0, "stages");
};

constexpr int kTcThreads = 14 * 32;
constexpr uint32_t kIdescF16 = tc05::idesc_f16(128, 32, false);
constexpr uint32_t kIdescBF16 = tc05::idesc_bf16(128, 32, false);

// Byte offset of element (row n, column k) of a K-major B operand (16-bit elements) in 64-column
// blocks of `rows` rows with the 128-byte swizzle; k a multiple of 8 for a 16-byte chunk.
__device__ __forceinline__ uint32_t b_off(int n, int k, int rows) {
  return (uint32_t)((k >> 6) * rows * 128 + n * 128 + ((((k & 63) >> 3) ^ (n & 7)) << 4) + ((k & 7) << 1));
}
// Byte offset of 16-byte chunk cc (8 channels) of window row r.
__device__ __forceinline__ uint32_t w_off(int r, int cc) {
  return (uint32_t)((cc >> 3) * (128 * 128) + r * 128 + (((cc & 7) ^ (r & 7)) << 4));
}

__device__ __forceinline__ void bar_named(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}
__device__ __forceinline__ void cp_async_mbar_arrive(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// The first unit of a request (cost start ucb: nqb quantised blocks of cost 1, then nwb window
// blocks of cost ww) whose cost start is at least X.
__device__ __forceinline__ int first_unit_at(int64_t X, int64_t ucb, int nqb, int nwb, int ww) {
  const int64_t x = X - ucb;
  if (x <= 0) return 0;
  if (x <= nqb) return (int)x;
  const int64_t w = (x - nqb + ww - 1) / ww;
  return nqb + (int)(w < nwb ? w : nwb);
}

// Bounded wait that also gives up as soon as another role of the CTA has given up.
__device__ __forceinline__ bool tc_wait(uint64_t* bar, uint32_t parity, const DraftParams& p, volatile int* abort) {
  for (uint32_t it = 0; it < p.spin_limit; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 255u) == 255u && *abort) return false;
  }
  set_status(p.dev_status, VC_DEV_TIMEOUT);
  *abort = 1;
  return false;
}
// The same for a whole warp: every lane waits (each gets the phase's ordering), and the warp
// proceeds only if all of them saw it complete, so the lanes never part.
__device__ __forceinline__ bool tc_wait_warp(uint64_t* bar, uint32_t parity, const DraftParams& p, volatile int* abort) {
  return __all_sync(0xffffffffu, tc_wait(bar, parity, p, abort));
}

template <int BITS>
__global__ void __launch_bounds__(kTcThreads, 1)
    draft_tc_kernel(const __grid_constant__ DraftParams p) {
  using C = QtCfg<BITS>;
  constexpr int D = C::D;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int quarter = warp & 3;
  const int hk = blockIdx.y, cta = blockIdx.x;
  const int G = p.G;

  uint8_t* misc = smem + C::OFF_MISC;
  uint64_t* full = reinterpret_cast<uint64_t*>(misc);  // [NST]
  uint64_t* empty = full + C::NST;                     // [NST]
  uint64_t* wfull = empty + C::NST;
  uint64_t* wempty = wfull + 1;
  uint64_t* ak_full = wempty + 1;  // [2]
  uint64_t* ak_empty = ak_full + 2;
  uint64_t* av_full = ak_empty + 2;
  uint64_t* av_empty = av_full + 2;
  uint64_t* s_full = av_empty + 2;
  uint64_t* s_empty = s_full + 2;
  uint64_t* p_full = s_empty + 2;
  uint64_t* p_empty = p_full + 2;
  uint64_t* o_free = p_empty + 2;
  uint64_t* drain = o_free + 1;
  float* red = reinterpret_cast<float*>(misc + 512);    // [2][4][8] block maxima
  float* lred = red + 64;                               // [4][8] row sums
  float* zred = lred + 32;                              // [4][4][8] value zero terms
  uint32_t* tslot = reinterpret_cast<uint32_t*>(zred + 128);
  volatile int* abort = reinterpret_cast<volatile int*>(tslot + 1);

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::NST; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 12);
    }
    mbar_init(wfull, 32);
    mbar_init(wempty, 8);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&ak_full[i], 4);
      mbar_init(&ak_empty[i], 1);
      mbar_init(&av_full[i], 4);
      mbar_init(&av_empty[i], 1);
      mbar_init(&s_full[i], 1);
      mbar_init(&s_empty[i], 4);
      mbar_init(&p_full[i], 4);
      mbar_init(&p_empty[i], 1);
    }
    mbar_init(o_free, 4);
    mbar_init(drain, 1);
    *abort = 0;
    fence_mbar_init();
  }
  if (warp == 0) tc05::alloc(tslot, C::T_COLS);
  if (((smem_u32(smem) & 1023u) != 0) && threadIdx.x == 0) set_status(p.dev_status, VC_DEV_INTERNAL);
  tc05::fence_before();
  __syncthreads();
  tc05::fence_after();
  const uint32_t tmem = *tslot;
  pdl_launch_dependents();
  bool waited = !p.early;
  if (waited) pdl_wait();

  // this CTA's cost range and the requests it touches
  const int64_t Tot = p.tc_total, P = p.n_cta_head;
  const int64_t X0 = (cta * Tot + P - 1) / P, X1 = ((cta + 1) * Tot + P - 1) / P;
  int b_lo = p.B, b_hi = -1;
  for (int b = 0; b < p.B; ++b)
    if (p.req[b].tc_c0 <= cta && cta <= p.req[b].tc_c1) {
      b_lo = b_lo < b ? b_lo : b;
      b_hi = b;
    }
  auto units_of = [&](int b, int& u0, int& u1) {
    const DraftReqDev& r = p.req[b];
    u0 = first_unit_at(X0, r.tc_ucb, r.tc_nqb, r.tc_nwb, C::WW);
    u1 = first_unit_at(X1, r.tc_ucb, r.tc_nqb, r.tc_nwb, C::WW);
  };
  const uint8_t* ring = smem + C::OFF_RING;
  uint8_t* wtile = smem + C::OFF_WIN;
  const uint32_t bqk0 = smem_u32(smem + C::OFF_BQK), bpv0 = smem_u32(smem + C::OFF_BPV);

  // ============================ producer ============================
  if (warp == 0) {
    const uint64_t pol = l2_evict_first_policy();
    int qi = 0, wi = 0;
    bool ok = true;
    for (int b = b_lo; b <= b_hi && ok; ++b) {
      const DraftReqDev& r = p.req[b];
      int u0, u1;
      units_of(b, u0, u1);
      if (u0 == 0 && u1 > 0) {
        // fused append: the step's K/V row into window row n_win (read from its input by this step)
        if (!waited) {
          pdl_wait();
          waited = true;
        }
        constexpr int V16 = D * 2 / 16;
        const int l16 = lane & 15;
        if (l16 < V16) {
          const uint4* src = reinterpret_cast<const uint4*>((lane < 16 ? r.k_new : r.v_new) + (size_t)hk * D);
          bf16* dst = (lane < 16 ? r.k_win : r.v_win) + ((size_t)hk * r.win_cap + r.n_win) * D;
          reinterpret_cast<uint4*>(dst)[l16] = __ldg(src + l16);
        }
      }
      for (int u = u0; u < u1 && ok; ++u) {
        if (u < r.tc_nqb) {
          const int st = qi % C::NST;
          if (qi >= C::NST && !tc_wait_warp(&empty[st], ((qi / C::NST) - 1) & 1, p, abort)) {
            ok = false;
            break;
          }
          const int g0 = 4 * u, ngb = r.ng - g0 < 4 ? r.ng - g0 : 4;
          if (lane == 0) mbar_arrive_expect_tx(&full[st], (uint32_t)(ngb * C::GROUP_BYTES));
          __syncwarp();
          if (lane < 6) {
            const size_t gi = (size_t)hk * r.ng_cap + g0;
            const uint8_t* src;
            uint32_t per, off;
            switch (lane) {
              case 0: src = r.kc + gi * C::KCB, per = C::KCB, off = C::OFF_KC; break;
              case 1: src = reinterpret_cast<const uint8_t*>(r.ks) + gi * C::SCB, per = C::SCB, off = C::OFF_KS; break;
              case 2: src = reinterpret_cast<const uint8_t*>(r.kz) + gi * C::SCB, per = C::SCB, off = C::OFF_KZ; break;
              case 3: src = r.vc + gi * C::KCB, per = C::KCB, off = C::OFF_VC; break;
              case 4: src = reinterpret_cast<const uint8_t*>(r.vs) + gi * C::VSB, per = C::VSB, off = C::OFF_VS; break;
              default: src = reinterpret_cast<const uint8_t*>(r.vz) + gi * C::VSB, per = C::VSB, off = C::OFF_VZ; break;
            }
            bulk_g2s_hint(const_cast<uint8_t*>(ring) + st * C::STAGE + off, src, per * ngb, &full[st], pol);
          }
          ++qi;
        } else {
          if (wi >= 1 && !tc_wait_warp(wempty, (wi - 1) & 1, p, abort)) {
            ok = false;
            break;
          }
          if (!waited) {
            pdl_wait();  // window rows: the previous step appended one
            waited = true;
          }
          const int row0 = 128 * (u - r.tc_nqb);
          // 2 x 128 rows x 16 pieces: lane l moves pieces l, l + 32, ...; rows past the window
          // (and past its own row n_win) are zero-filled
          for (int k = lane; k < 2 * 128 * 16; k += 32) {
            const int isv = k >> 11, rr = (k >> 4) & 127, piece = k & 15;
            const int R = row0 + rr;
            const bf16* src = nullptr;
            if (R < r.n_win)
              src = (isv ? r.v_win : r.k_win) + ((size_t)hk * r.win_cap + R) * D;
            else if (R == r.n_win)
              src = (isv ? r.v_new : r.k_new) + (size_t)hk * D;
            uint8_t* dst = wtile + isv * 2 * C::WBLK + w_off(rr, piece);
            cp_async16(dst, src ? reinterpret_cast<const uint8_t*>(src) + piece * 16 : reinterpret_cast<const uint8_t*>(r.k_new),
                       src ? 16u : 0u);
          }
          cp_async_mbar_arrive(wfull);
          ++wi;
        }
      }
    }
    if (!ok) {
      // stop: wait (bounded) for the copies already issued, so none lands after the CTA exits
      for (int k = qi > C::NST ? qi - C::NST : 0; k < qi; ++k) mbar_wait_bounded(&full[k % C::NST], (k / C::NST) & 1, p.dev_status);
    }
    cp_async_wait<0>();
  }

  // ============================ MMA issue ============================
  else if (warp == 1) {
    if (lane == 0) {
      int j = 0, seg = 0, last_first = 0, prev_seg = -1;
      bool ok = true, prev_bf = false;
      // PV of unit jj (of segment sg, its first unit when first)
      auto issue_pv = [&](int jj, int sg, bool first, bool bf) -> bool {
        const int pb = jj & 1;
        if (!tc_wait(&av_full[pb], (jj >> 1) & 1, p, abort)) return false;
        if (!tc_wait(&p_full[pb], (jj >> 1) & 1, p, abort)) return false;
        if (first && sg > 0 && !tc_wait(o_free, (sg - 1) & 1, p, abort)) return false;
        tc05::fence_after();
        const uint32_t id = bf ? kIdescBF16 : kIdescF16;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint64_t bd = tc05::sdesc_sw128(bpv0 + pb * C::BPV + (kk >> 2) * C::KB + (kk & 3) * 32, 16, 1024);
          tc05::mma_ts(tmem + C::T_O, tmem + C::T_AV + pb * 64 + 8 * kk, bd, id, (first && kk == 0) ? 0u : 1u);
        }
        tc05::commit(&p_empty[pb]);
        tc05::commit(&av_empty[pb]);
        return true;
      };
      for (int b = b_lo; b <= b_hi && ok; ++b) {
        const DraftReqDev& r = p.req[b];
        int u0, u1;
        units_of(b, u0, u1);
        if (u1 <= u0) continue;
        for (int u = u0; u < u1; ++u, ++j) {
          const int buf = j & 1;
          const bool bf = u >= r.tc_nqb;
          if (!tc_wait(&ak_full[buf], (j >> 1) & 1, p, abort)) { ok = false; break; }
          if (j >= 2 && !tc_wait(&s_empty[buf], ((j - 2) >> 1) & 1, p, abort)) { ok = false; break; }
          tc05::fence_after();
          const uint32_t id = bf ? kIdescBF16 : kIdescF16;
#pragma unroll
          for (int kk = 0; kk < 9; ++kk) {
            const uint64_t bd = tc05::sdesc_sw128(bqk0 + buf * C::BQK + (kk >> 2) * C::KB + (kk & 3) * 32, 16, 1024);
            tc05::mma_ts(tmem + C::T_S + buf * 32, tmem + C::T_AK + buf * 80 + 8 * kk, bd, id, kk > 0 ? 1u : 0u);
          }
          tc05::commit(&s_full[buf]);
          tc05::commit(&ak_empty[buf]);
          if (j >= 1 && !issue_pv(j - 1, prev_seg, last_first == j - 1, prev_bf)) { ok = false; break; }
          if (u == u0) last_first = j;
          prev_seg = seg;
          prev_bf = bf;
        }
        ++seg;
      }
      if (ok && j >= 1) issue_pv(j - 1, prev_seg, last_first == j - 1, prev_bf);
      // every MMA issued has completed before TMEM is freed
      tc05::commit(drain);
      mbar_wait_bounded(drain, 0, p.dev_status);
    }
    __syncwarp();
  }

  // ============================ K warps ============================
  else if (warp < 6) {
    const int g = quarter;  // the block's group this warp stages
    const int h = lane >> 2, q4 = lane & 3;
    // the two ones columns of the zero-term k-step (elements 128, 129), zero elsewhere; never rewritten
    {
      uint32_t one[8] = {0x3C003C00u, 0, 0, 0, 0, 0, 0, 0};
      for (int buf = 0; buf < 2; ++buf) tc05::st8(tmem + ((uint32_t)(32 * quarter) << 16) + C::T_AK + buf * 80 + 64, one);
      tc05::wait_st();
      // the B side of that k-step: elements 130..143 of every row stay zero (128, 129 are written
      // per unit), so stale shared memory never meets the zero columns of A
      for (int i = threadIdx.x - 64; i < 2 * (C::KB / 16); i += 128)
        *reinterpret_cast<uint4*>(smem + C::OFF_BQK + (i / (C::KB / 16)) * C::BQK + 2 * C::KB + (i % (C::KB / 16)) * 16) =
            make_uint4(0u, 0u, 0u, 0u);
    }
    int j = 0, qi = 0, wi = 0;
    bool ok = true;
    for (int b = b_lo; b <= b_hi && ok; ++b) {
      const DraftReqDev& r = p.req[b];
      int u0, u1;
      units_of(b, u0, u1);
      if (u1 <= u0) continue;
      // the query of this lane's head and channels 16ks + 2q4 (+1), 16ks + 8 + 2q4 (+1): bf16 pairs,
      // and as fp16 scaled by 2^-E (E from the KV head's largest |q|, so |qn| < 1)
      uint32_t qb[8][2], qn[8][2];
      float mx = 0.f;
      const bf16* qbase = r.q + ((size_t)hk * G + h) * D;
#pragma unroll
      for (int ks = 0; ks < 8; ++ks)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int c = 16 * ks + 8 * e + 2 * q4;
          qb[ks][e] = h < G ? __ldg(reinterpret_cast<const unsigned int*>(qbase + c)) : 0u;
          const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&qb[ks][e]));
          mx = fmaxf(mx, fmaxf(fabsf(f.x), fabsf(f.y)));
        }
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
      int E = 0;
      if (mx > 0.f) frexpf(mx, &E);
      const float inv = ldexpf(1.f, -E);
#pragma unroll
      for (int ks = 0; ks < 8; ++ks)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&qb[ks][e]));
          qn[ks][e] = pack_half2(f.x * inv, f.y * inv);
        }
      for (int u = u0; u < u1; ++u, ++j) {
        const int buf = j & 1;
        const bool quant = u < r.tc_nqb;
        if (j >= 2 && !tc_wait_warp(&ak_empty[buf], ((j - 2) >> 1) & 1, p, abort)) { ok = false; break; }
        const uint32_t bq = bqk0 + buf * C::BQK;
        const uint32_t ta = tmem + ((uint32_t)(32 * quarter) << 16) + C::T_AK + buf * 80;
        // B rows 8g + (lane & 7), channel blocks: the thread's stmatrix row address for tile i = lane / 8
        const int srow = 8 * g + (lane & 7), si = lane >> 3;
        if (quant) {
          if (!tc_wait_warp(&full[qi % C::NST], (qi / C::NST) & 1, p, abort)) { ok = false; break; }
          const uint8_t* st = ring + (qi % C::NST) * C::STAGE;
          const uint32_t* kw = reinterpret_cast<const uint32_t*>(st + C::OFF_KC + g * C::KCB);
          // A: the group's codes, both 16-token halves
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            uint32_t a[32];
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
              uint32_t f[4];
              code_frag_centred<BITS>(kw[(half * C::STEPS + (BITS == 4 ? ks : ks >> 1)) * 32 + lane], ks, f);
              a[4 * ks] = f[0];
              a[4 * ks + 1] = f[1];
              a[4 * ks + 2] = f[2];
              a[4 * ks + 3] = f[3];
            }
            tc05::st16x128_x16(ta + ((uint32_t)(16 * half) << 16), a);
          }
          // B: qn o s_g (rows 8g + h) and the zero term sum_c qn_c (z_c + C0 s_c) as an MMA dot product
          const __half* ksc = reinterpret_cast<const __half*>(st + C::OFF_KS + g * C::SCB);
          const __half* kzc = reinterpret_cast<const __half*>(st + C::OFF_KZ + g * C::SCB);
          constexpr uint32_t c0b = BITS == 2 ? 0x3E003E00u : 0x47804780u;  // fp16 1.5 / 7.5, both halves
          const __half2 c0h = *reinterpret_cast<const __half2*>(&c0b);
          uint32_t qs[8][2];
          float zq[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int ks = 0; ks < 8; ++ks) {
            uint32_t az[4];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const int c = 16 * ks + 8 * e + 2 * q4;
              const __half2 s2 = *reinterpret_cast<const __half2*>(ksc + c);
              const __half2 z2 = __hfma2(c0h, s2, *reinterpret_cast<const __half2*>(kzc + c));
              qs[ks][e] = hmul2_u32(qn[ks][e], s2);
              az[2 * e] = az[2 * e + 1] = *reinterpret_cast<const uint32_t*>(&z2);
            }
            mma_f16_16816(zq, az, qn[ks][0], qn[ks][1]);
          }
#pragma unroll
          for (int k4 = 0; k4 < 4; ++k4)
            tc05::stsm_x4(bq + b_off(srow, 8 * (4 * k4 + si), C::N), qs[2 * k4][0], qs[2 * k4][1], qs[2 * k4 + 1][0],
                          qs[2 * k4 + 1][1]);
          if (lane < 4) {
            // zq[0], zq[1]: heads 2 lane, 2 lane + 1 (every row of the accumulator holds the same sum)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const float z = zq[e];
              const __half hi = __float2half_rn(z);
              const __half lo = __float2half_rn(z - __half2float(hi));
              const __half2 hl = __halves2half2(hi, lo);
              const int n = 8 * g + 2 * lane + e;
              *reinterpret_cast<__half2*>(smem + (bq - smem_u32(smem)) + b_off(n, 128, C::N)) = hl;
            }
          }
        } else {
          if (!tc_wait_warp(wfull, wi & 1, p, abort)) { ok = false; break; }
          // A: window K rows 32g .. 32g + 31 (bf16), m16n8k16 fragments by ldmatrix
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            uint32_t a[32];
            const int r0 = 32 * g + 16 * half;
#pragma unroll
            for (int ks = 0; ks < 8; ++ks)
              ldsm_x4(a[4 * ks], a[4 * ks + 1], a[4 * ks + 2], a[4 * ks + 3],
                      wtile + w_off(r0 + (lane & 7) + 8 * ((lane >> 3) & 1), 2 * ks + (lane >> 4)));
            tc05::st16x128_x16(ta + ((uint32_t)(16 * half) << 16), a);
          }
          // B: the bf16 query in rows 8g + h, no zero term
#pragma unroll
          for (int k4 = 0; k4 < 4; ++k4)
            tc05::stsm_x4(bq + b_off(srow, 8 * (4 * k4 + si), C::N), qb[2 * k4][0], qb[2 * k4][1], qb[2 * k4 + 1][0],
                          qb[2 * k4 + 1][1]);
          if (lane < 4) {
#pragma unroll
            for (int e = 0; e < 2; ++e)
              *reinterpret_cast<uint32_t*>(smem + (bq - smem_u32(smem)) + b_off(8 * g + 2 * lane + e, 128, C::N)) = 0u;
          }
        }
        tc05::wait_st();
        tc05::fence_before();
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&ak_full[buf]);
          mbar_arrive(quant ? &empty[qi % C::NST] : wempty);
        }
        if (quant) ++qi; else ++wi;
      }
    }
  }

  // ============================ V warps ============================
  else if (warp < 10) {
    const int vq = quarter;  // channels 32 vq .. 32 vq + 31 (channel tiles 2 vq, 2 vq + 1)
    int j = 0, qi = 0, wi = 0;
    bool ok = true;
    for (int b = b_lo; b <= b_hi && ok; ++b) {
      const DraftReqDev& r = p.req[b];
      int u0, u1;
      units_of(b, u0, u1);
      for (int u = u0; u < u1; ++u, ++j) {
        const int buf = j & 1;
        const bool quant = u < r.tc_nqb;
        if (j >= 2 && !tc_wait_warp(&av_empty[buf], ((j - 2) >> 1) & 1, p, abort)) { ok = false; break; }
        const uint32_t ta = tmem + ((uint32_t)(32 * vq) << 16) + C::T_AV + buf * 64;
        if (quant) {
          if (!tc_wait_warp(&full[qi % C::NST], (qi / C::NST) & 1, p, abort)) { ok = false; break; }
          const uint8_t* st = ring + (qi % C::NST) * C::STAGE;
#pragma unroll
          for (int mm = 0; mm < 2; ++mm) {
            const int mt = 2 * vq + mm;
            uint32_t a[32];
#pragma unroll
            for (int g = 0; g < 4; ++g) {
              const uint32_t* vw = reinterpret_cast<const uint32_t*>(st + C::OFF_VC + g * C::KCB);
#pragma unroll
              for (int half = 0; half < 2; ++half) {
                uint32_t f[4];
                code_frag_centred<BITS>(vw[(half * C::STEPS + (BITS == 4 ? mt : mt >> 1)) * 32 + lane], mt, f);
                const int k = 2 * g + half;
                a[4 * k] = f[0];
                a[4 * k + 1] = f[1];
                a[4 * k + 2] = f[2];
                a[4 * k + 3] = f[3];
              }
            }
            tc05::st16x128_x16(ta + ((uint32_t)(16 * mm) << 16), a);
          }
        } else {
          if (!tc_wait_warp(wfull, wi & 1, p, abort)) { ok = false; break; }
          const uint8_t* vt = wtile + 2 * C::WBLK;
#pragma unroll
          for (int mm = 0; mm < 2; ++mm) {
            const int mt = 2 * vq + mm;
            uint32_t a[32];
#pragma unroll
            for (int k = 0; k < 8; ++k)
              ldsm_x4_t(a[4 * k], a[4 * k + 1], a[4 * k + 2], a[4 * k + 3],
                        vt + w_off(16 * k + (lane & 7) + 8 * (lane >> 4), 2 * mt + ((lane >> 3) & 1)));
            tc05::st16x128_x16(ta + ((uint32_t)(16 * mm) << 16), a);
          }
        }
        tc05::wait_st();
        tc05::fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&av_full[buf]);
          mbar_arrive(quant ? &empty[qi % C::NST] : wempty);
        }
        if (quant) ++qi; else ++wi;
      }
    }
  }

  // ============================ softmax warps ============================
  else {
    const int g = quarter;  // tokens 32g .. 32g + 31 of a block; O rows (channels) of group g
    const int q4 = lane & 3, a8 = lane >> 2;
    int* flg = reinterpret_cast<int*>(zred + 128 + 8);  // [2][4] per-warp failure flags, by barrier parity
    int nbar = 0;  // named barriers passed (their parity picks the flag and maximum buffers)
    // A named barrier of the four softmax warps that also tells each whether any of them failed a
    // wait since the last one: they then all stop together (no warp is left at a barrier).
    auto sync_flags = [&](bool bad) -> bool {
      int* f = flg + (nbar & 1) * 4;
      if (lane == 0) f[g] = bad ? 1 : 0;
      bar_named(1, 128);
      const bool any = (f[0] | f[1] | f[2] | f[3]) != 0;
      ++nbar;
      return any;
    };
    int j = 0, qi = 0;
    bool stop = false;
    for (int b = b_lo; b <= b_hi && !stop; ++b) {
      const DraftReqDev& r = p.req[b];
      int u0, u1;
      units_of(b, u0, u1);
      const bool one_cta = r.tc_c0 == r.tc_c1;
      const int NC = p.n_cta_head;
      const int64_t cslot = (int64_t)hk * (NC + p.B) + cta + b;
      const int c = 32 * g + lane;  // this thread's channel in epilogues
      if (u1 <= u0) {
        // a CTA inside the request's span that holds none of its units: an empty partial
        if (!waited) {
          pdl_wait();
          waited = true;
        }
        if (!one_cta)
          for (int hh = 0; hh < G && hh < 8; ++hh) {
            p.ws_o[(cslot * G + hh) * D + c] = 0.f;
            if (c == 0) p.ws_lse[cslot * G + hh] = -INFINITY;
          }
        continue;
      }
      // the query's exponent E (as the K warps compute it) for the quantised blocks' scale
      float mxq = 0.f;
      {
        const bf16* qbase = r.q + ((size_t)hk * G + a8) * D;
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int cc = 16 * ks + 8 * e + 2 * q4;
            const uint32_t w = a8 < G ? __ldg(reinterpret_cast<const unsigned int*>(qbase + cc)) : 0u;
            const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w));
            mxq = fmaxf(mxq, fmaxf(fabsf(f.x), fabsf(f.y)));
          }
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) mxq = fmaxf(mxq, __shfl_xor_sync(0xffffffffu, mxq, off));
      }
      int E = 0;
      if (mxq > 0.f) frexpf(mxq, &E);
      const float scale_q = ldexpf(p.scale_log2, E);
      float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f}, zs[4][2] = {};
      for (int u = u0; u < u1; ++u, ++j) {
        const int buf = j & 1;
        const bool quant = u < r.tc_nqb;
        bool bad = false;
        // token validity: a whole group of a quantised block, or window rows up to n_win
        bool val[4];
        if (quant) {
          const bool gv = 4 * u + g < r.ng;
#pragma unroll
          for (int t = 0; t < 4; ++t) val[t] = gv;
        } else {
          const int row0 = 128 * (u - r.tc_nqb) + 32 * g + a8;
#pragma unroll
          for (int t = 0; t < 4; ++t) val[t] = row0 + 8 * t <= r.n_win;
        }
        float x[4][2];
        if (tc_wait_warp(&s_full[buf], (j >> 1) & 1, p, abort)) {
          tc05::fence_after();
          uint32_t sr[8];
          uint32_t t4[4];
          const uint32_t ts = tmem + ((uint32_t)(32 * g) << 16) + C::T_S + buf * 32 + 8 * g;
          tc05::ld16x256_x1(ts, t4);
          sr[0] = t4[0], sr[1] = t4[1], sr[2] = t4[2], sr[3] = t4[3];
          tc05::ld16x256_x1(ts + (16u << 16), t4);
          sr[4] = t4[0], sr[5] = t4[1], sr[6] = t4[2], sr[7] = t4[3];
          tc05::wait_ld();
          tc05::fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&s_empty[buf]);
          // x[t][e]: token t in {a8, a8 + 8, 16 + a8, 24 + a8} of the group, head 2 q4 + e
          const float sc = quant ? scale_q : p.scale_log2;
#pragma unroll
          for (int t = 0; t < 4; ++t)
#pragma unroll
            for (int e = 0; e < 2; ++e) x[t][e] = val[t] ? __uint_as_float(sr[2 * t + e]) * sc : -INFINITY;
        } else {
          bad = true;
#pragma unroll
          for (int t = 0; t < 4; ++t) x[t][0] = x[t][1] = -INFINITY;
        }
        // block maximum per head over the four warps' tokens
        float bm[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          float v = fmaxf(fmaxf(x[0][e], x[1][e]), fmaxf(x[2][e], x[3][e]));
          v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 4));
          v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 8));
          v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 16));
          bm[e] = v;
        }
        float* rb = red + (nbar & 1) * 32;
        if (lane < 4) {
          rb[g * 8 + 2 * lane] = bm[0];
          rb[g * 8 + 2 * lane + 1] = bm[1];
        }
        if (sync_flags(bad)) {
          stop = true;
          break;
        }
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int hh = 2 * q4 + e;
          bm[e] = fmaxf(fmaxf(rb[hh], rb[8 + hh]), fmaxf(rb[16 + hh], rb[24 + hh]));
        }
        float corr[2] = {1.f, 1.f};
        bool need = false;
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const float mn = fmaxf(m[e], bm[e]);
          if (mn > m[e]) {
            need = true;
            corr[e] = ex2_approx(m[e] - mn);  // 0 while nothing is accumulated (m = -inf)
            m[e] = mn;
          }
        }
        need = __any_sync(0xffffffffu, need);
        if (need) {
          l[0] *= corr[0];
          l[1] *= corr[1];
#pragma unroll
          for (int cg = 0; cg < 4; ++cg) {
            zs[cg][0] *= corr[0];
            zs[cg][1] *= corr[1];
          }
          if (u > u0) {
            // O holds this segment's earlier units: wait for unit j - 1's PV, then rescale the
            // columns of every head (O rows are this warp's channels, 32 columns n = 8 cg + h)
            if (tc_wait_warp(&p_empty[(j - 1) & 1], ((j - 1) >> 1) & 1, p, abort)) {
              tc05::fence_after();
              float c8[8];
#pragma unroll
              for (int hh = 0; hh < 8; ++hh) c8[hh] = __shfl_sync(0xffffffffu, corr[hh & 1], hh >> 1);
              const uint32_t to = tmem + ((uint32_t)(32 * g) << 16) + C::T_O;
#pragma unroll
              for (int cg = 0; cg < 4; ++cg) {
                uint32_t o8[8];
                tc05::ld8(to + 8 * cg, o8);
                tc05::wait_ld();
#pragma unroll
                for (int hh = 0; hh < 8; ++hh) o8[hh] = __float_as_uint(__uint_as_float(o8[hh]) * c8[hh]);
                tc05::st8(to + 8 * cg, o8);
              }
              tc05::wait_st();
              tc05::fence_before();
            } else {
              bad = true;
            }
          }
        }
        float pw[4][2];
#pragma unroll
        for (int t = 0; t < 4; ++t)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const float mu = m[e] == -INFINITY ? 0.f : m[e];
            pw[t][e] = val[t] ? ex2_approx(x[t][e] - mu) : 0.f;
          }
#pragma unroll
        for (int e = 0; e < 2; ++e) l[e] += (pw[0][e] + pw[1][e]) + (pw[2][e] + pw[3][e]);
        // B_PV of this unit: its buffer's previous PV (unit j - 2) must have completed
        if (!bad && j >= 2 && !tc_wait_warp(&p_empty[buf], ((j - 2) >> 1) & 1, p, abort)) bad = true;
        const uint32_t bp = bpv0 + buf * C::BPV;
        // stmatrix.trans: tile i = tokens 8i .. 8i + 7 of the group; memory row n = 8 cg + (lane & 7)
        const uint32_t saddr = bp + b_off(lane & 7, 32 * g + 8 * (lane >> 3), C::N);
        if (quant) {
          if (!bad && !tc_wait_warp(&full[qi % C::NST], (qi / C::NST) & 1, p, abort)) bad = true;
          if (!bad) {
            const uint8_t* st = ring + (qi % C::NST) * C::STAGE;
            const __half* vsc = reinterpret_cast<const __half*>(st + C::OFF_VS + g * C::VSB);
            const __half* vze = reinterpret_cast<const __half*>(st + C::OFF_VZ + g * C::VSB);
            constexpr float C0 = BITS == 2 ? 1.5f : 7.5f;
            uint32_t pp[4];
#pragma unroll
            for (int t = 0; t < 4; ++t) pp[t] = pack_half2(pw[t][0], pw[t][1]);
            __half sv[4][4], zv[4][4];
#pragma unroll
            for (int t = 0; t < 4; ++t) {
              const int tok = a8 + 8 * t;
              const uint2 s4 = *reinterpret_cast<const uint2*>(vsc + tok * 4);
              const uint2 z4 = *reinterpret_cast<const uint2*>(vze + tok * 4);
              const __half2 s01 = *reinterpret_cast<const __half2*>(&s4.x), s23 = *reinterpret_cast<const __half2*>(&s4.y);
              const __half2 z01 = *reinterpret_cast<const __half2*>(&z4.x), z23 = *reinterpret_cast<const __half2*>(&z4.y);
              sv[t][0] = __low2half(s01), sv[t][1] = __high2half(s01), sv[t][2] = __low2half(s23), sv[t][3] = __high2half(s23);
              zv[t][0] = __low2half(z01), zv[t][1] = __high2half(z01), zv[t][2] = __low2half(z23), zv[t][3] = __high2half(z23);
            }
#pragma unroll
            for (int cg = 0; cg < 4; ++cg) {
              uint32_t rr[4];
#pragma unroll
              for (int t = 0; t < 4; ++t) {
                rr[t] = val[t] ? hmul2_u32(pp[t], __half2half2(sv[t][cg])) : 0u;
                // value zero term with the centring: z + C0 s (fp32), weighted by p
                const float zc = val[t] ? fmaf(C0, __half2float(sv[t][cg]), __half2float(zv[t][cg])) : 0.f;
                zs[cg][0] = fmaf(pw[t][0], zc, zs[cg][0]);
                zs[cg][1] = fmaf(pw[t][1], zc, zs[cg][1]);
              }
              tc05::stsm_x4_t(saddr + 8 * cg * 128, rr[0], rr[1], rr[2], rr[3]);
            }
          }
        } else if (!bad) {
          uint32_t pp[4];
#pragma unroll
          for (int t = 0; t < 4; ++t) pp[t] = pack_bf16x2(pw[t][0], pw[t][1]);
#pragma unroll
          for (int cg = 0; cg < 4; ++cg) tc05::stsm_x4_t(saddr + 8 * cg * 128, pp[0], pp[1], pp[2], pp[3]);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0 && !bad) {
          mbar_arrive(&p_full[buf]);
          if (quant) mbar_arrive(&empty[qi % C::NST]);
        }
        if (quant) ++qi;
        if (u + 1 < u1) continue;  // a failure here reaches the others at the next unit's barrier
        // ---- end of the segment: this CTA's partial of request b ----
        uint32_t o8[8];
        if (!bad && tc_wait_warp(&p_empty[buf], (j >> 1) & 1, p, abort)) {
          tc05::fence_after();
          tc05::ld8(tmem + ((uint32_t)(32 * g) << 16) + C::T_O + 8 * g, o8);
          tc05::wait_ld();
          tc05::fence_before();
        } else {
          bad = true;
        }
        // row sums and value zero terms: over this warp's tokens, then over the four warps
        float lw[2], zw[4][2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          float v = l[e];
          v += __shfl_xor_sync(0xffffffffu, v, 4);
          v += __shfl_xor_sync(0xffffffffu, v, 8);
          v += __shfl_xor_sync(0xffffffffu, v, 16);
          lw[e] = v;
#pragma unroll
          for (int cg = 0; cg < 4; ++cg) {
            float z = zs[cg][e];
            z += __shfl_xor_sync(0xffffffffu, z, 4);
            z += __shfl_xor_sync(0xffffffffu, z, 8);
            z += __shfl_xor_sync(0xffffffffu, z, 16);
            zw[cg][e] = z;
          }
        }
        if (lane < 4) {
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            lred[g * 8 + 2 * lane + e] = lw[e];
#pragma unroll
            for (int cg = 0; cg < 4; ++cg) zred[(g * 4 + cg) * 8 + 2 * lane + e] = zw[cg][e];
          }
        }
        if (sync_flags(bad)) {
          stop = true;
          break;
        }
        if (!waited) {
          pdl_wait();  // outputs and partials: the previous step's merges may still read the workspace
          waited = true;
        }
#pragma unroll
        for (int hh = 0; hh < 8; ++hh) {
          if (hh >= G) break;
          const float L = lred[hh] + lred[8 + hh] + lred[16 + hh] + lred[24 + hh];
          const float Z = zred[(0 * 4 + g) * 8 + hh] + zred[(1 * 4 + g) * 8 + hh] + zred[(2 * 4 + g) * 8 + hh] +
                          zred[(3 * 4 + g) * 8 + hh];
          const float mh = __shfl_sync(0xffffffffu, m[hh & 1], hh >> 1);
          const float inv = L > 0.f ? 1.f / L : 0.f;
          const float ov = (__uint_as_float(o8[hh]) + Z) * inv;
          if (one_cta) {
            r.o[((size_t)hk * G + hh) * D + c] = __float2bfloat16(ov);
          } else {
            p.ws_o[(cslot * G + hh) * D + c] = ov;
            if (c == 0) p.ws_lse[cslot * G + hh] = L > 0.f ? mh + log2f(L) : -INFINITY;
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(o_free);
        // lred/zred are written again only in a later segment's epilogue, after at least one
        // block-maximum barrier that every warp reaches after reading them here
      }
    }
    if (*abort) {
      // a wait gave up somewhere in the CTA: every request it touches gets finite (zero) results
      if (!waited) {
        pdl_wait();
        waited = true;
      }
      for (int b = b_lo; b <= b_hi; ++b) {
        const DraftReqDev& r = p.req[b];
        const int c = 32 * g + lane;
        const int64_t cslot = (int64_t)hk * (p.n_cta_head + p.B) + cta + b;
        for (int hh = 0; hh < G && hh < 8; ++hh) {
          if (r.tc_c0 == r.tc_c1) {
            r.o[((size_t)hk * G + hh) * D + c] = __float2bfloat16(0.f);
          } else {
            p.ws_o[(cslot * G + hh) * D + c] = 0.f;
            if (c == 0) p.ws_lse[cslot * G + hh] = -INFINITY;
          }
        }
      }
    }
  }

  // ============================ merge of split requests ============================
  tc05::fence_before();
  __syncthreads();
  if (!waited) {
    pdl_wait();
    waited = true;
  }
  __shared__ int s_last;
  const int NC = p.n_cta_head;
  for (int b = b_lo; b <= b_hi; ++b) {
    const DraftReqDev& r = p.req[b];
    if (r.tc_c0 == r.tc_c1) continue;
    // every thread's partial stores come before thread 0's release fence and arrival; the last
    // arriver's acquire fence and the barrier after it order the other CTAs' partials before it reads
    __syncthreads();
    if (threadIdx.x == 0) {
      asm volatile("fence.acq_rel.gpu;" ::: "memory");
      const uint32_t n = (uint32_t)(r.tc_c1 - r.tc_c0 + 1);
      const uint32_t old = atomicInc(p.ws_ctr + (size_t)hk * VC_MAX_BATCH + b, n - 1);
      const bool last = old == n - 1;
      if (last) asm volatile("fence.acq_rel.gpu;" ::: "memory");
      s_last = last ? 1 : 0;
    }
    __syncthreads();
    if (s_last) {
      for (int hh = warp; hh < G; hh += kTcThreads / 32)
        merge_head<D>(p.ws_o, p.ws_lse, (int64_t)hk * (NC + p.B) + b + r.tc_c0, r.tc_c1 - r.tc_c0 + 1, G, hh, lane,
                      r.o + ((size_t)hk * G + hh) * D, nullptr, nullptr);
    }
  }
  __syncthreads();
  tc05::fence_after();
  if (warp == 0) tc05::dealloc(tmem, C::T_COLS);
}

// ---------------------------------------------------------------------------------------------
// Host: the unit plan (per request, the same for every KV head) and the launch.
int draft_tc_ctas_per_head(int Hkv, int sm_count) {
  const int n = sm_count / Hkv;
  return n > 1 ? n : 1;
}

template <int BITS>
static cudaError_t launch_tc_t(DraftParams p, int sm_count, cudaStream_t s) {
  using C = QtCfg<BITS>;
  static std::atomic<uint64_t> attr{0};
  cudaError_t e = raise_smem_limit(draft_tc_kernel<BITS>, C::SMEM, attr);
  if (e != cudaSuccess) return e;
  int64_t tot = 0;
  for (int b = 0; b < p.B; ++b) {
    DraftReqDev& r = p.req[b];
    r.tc_nqb = (r.ng + 3) / 4;
    r.tc_nwb = (r.n_win + 1 + 127) / 128;
    r.tc_ucb = tot;
    tot += r.tc_nqb + (int64_t)C::WW * r.tc_nwb;
  }
  const int P = draft_tc_ctas_per_head(p.Hkv, sm_count);
  for (int b = 0; b < p.B; ++b) {
    DraftReqDev& r = p.req[b];
    const int64_t xl = r.tc_ucb + r.tc_nqb + (int64_t)C::WW * r.tc_nwb - (r.tc_nwb > 0 ? C::WW : 1);
    r.tc_c0 = (int32_t)(r.tc_ucb * P / tot);
    r.tc_c1 = (int32_t)(xl * P / tot);
  }
  p.tc_total = tot;
  p.n_cta_head = P;
  p.ws_lse = p.ws_o + (size_t)p.Hkv * (P + p.B) * p.G * C::D;
  return launch_pdl(draft_tc_kernel<BITS>, dim3(P, p.Hkv), dim3(kTcThreads), C::SMEM, s, p);
}

cudaError_t launch_draft_tc(const DraftParams& p, int kind, int sm_count, cudaStream_t s) {
  if (kind == 2) return launch_tc_t<2>(p, sm_count, s);
  if (kind == 4) return launch_tc_t<4>(p, sm_count, s);
  return cudaErrorInvalidValue;
}

}  // namespace vc
