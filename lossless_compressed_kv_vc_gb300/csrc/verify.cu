// Verification attention on tcgen05 tensor cores with TMEM accumulators.
//
// "VeriCache: Turning Lossy KV Cache into Lossless LLM Inference", "Core algorithm" step 2: one
// forward pass over the full cache KV_full checks all drafted tokens in parallel; "Cross-resource
// staggering (P1)": verification is bound by the host link and by compute.
//
// Work decomposition. The n_rows drafted tokens of a request times the G = Hq/Hkv query heads of
// one KV head form up to 128 query rows per tile (row r -> token r / G, head r % G), so
// S = Q K^T and O += P V are dense 128 x 64 x d and 128 x d x 64 contractions. A "unit" is one
// (request, KV head, 128-row tile); its KV tiles are the ceil(ctx/64) tiles of KV_full followed by
// the ceil(n_rows/64) tiles of the drafted rows (causal mask: row of token i sees draft rows <= i).
// All units' tiles form one sequence that is cut into equal contiguous ranges, one per CTA (two
// CTAs per SM), so every CTA streams the same number of KV bytes; a CTA whose range covers a whole
// unit writes the bf16 output, otherwise it writes an (o, lse) partial into slot cta + unit, and a
// small combine kernel merges the partials of split units.
//
// Per CTA (192 threads, three roles that meet on mbarriers):
//   warps 0-3 (softmax): thread r owns TMEM lane r = query row r; it loads its Q row into the unit's
//     Q tile, then per KV tile loads its S row (tcgen05.ld), masks, takes the online softmax in fp32
//     (exp2 domain, ex2.approx; O is rescaled in TMEM only when the row maximum grows by more than
//     2^8) and writes its P row (bf16) into shared memory in the swizzled K-major layout;
//   warp 4 (MMA issue): S of tile g = Q K_g^T into TMEM buffer g & 1 (columns [0,64) or [64,128)),
//     then O += P_{g-1} V_{g-1} (columns [128, 128 + d)), so the next tile's QK^T runs while the
//     softmax warps work on the current one;
//   warp 5 (TMA): K and V tiles (64 tokens, 128-byte swizzle) into 2-stage rings, K a tile ahead of
//     V; a stage is reloaded once the MMA that read it has completed (tcgen05.commit).
#include "tc05.cuh"

#include <cuda.h>
#include <cudaTypedefs.h>
#include <math.h>
#include <stdlib.h>
#include <string.h>

namespace vc {

constexpr int VM = 128;  // query rows per tile
constexpr int VBN = 64;  // KV tokens per tile

// The largest of a row's VBN scores (three-input maxima: 64 -> 22 -> 8 -> 3 -> 1).
__device__ __forceinline__ float row_max(const float (&x)[VBN]) {
  static_assert(VBN == 64, "the tree is laid out for 64 scores");
  float a[22], b[8];
#pragma unroll
  for (int e = 0; e < 21; ++e) a[e] = max3f(x[3 * e], x[3 * e + 1], x[3 * e + 2]);
  a[21] = x[63];
#pragma unroll
  for (int e = 0; e < 7; ++e) b[e] = max3f(a[3 * e], a[3 * e + 1], a[3 * e + 2]);
  b[7] = a[21];
  return max3f(max3f(b[0], b[1], b[2]), max3f(b[3], b[4], b[5]), fmaxf(b[6], b[7]));
}

// P = 2^(x scale - mu) of a row's VBN scores, stored in bf16 as row r of a P tile in the 128-byte
// swizzled K-major layout (prow = the tile + 128 r; 16-byte chunk c at position c ^ (r & 7)).
// Returns the row's sum of the fp32 values.
__device__ __forceinline__ float row_exp_to_p(const float (&x)[VBN], float scale, float mu, uint8_t* prow, int r) {
  const uint64_t sc = f2_pack(scale, scale), nm = f2_pack(-mu, -mu);
  uint64_t acc[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
  for (int ch = 0; ch < 8; ++ch) {
    uint32_t w[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      float a0, a1;
      f2_unpack(f2_fma(f2_pack(x[ch * 8 + 2 * e], x[ch * 8 + 2 * e + 1]), sc, nm), a0, a1);
      const float p0 = ex2_approx(a0), p1 = ex2_approx(a1);
      acc[e] = f2_add(acc[e], f2_pack(p0, p1));
      w[e] = pack_bf16x2(p0, p1);
    }
    *reinterpret_cast<uint4*>(prow + ((ch ^ (r & 7)) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
  }
  float u0, u1;
  f2_unpack(f2_add(f2_add(acc[0], acc[1]), f2_add(acc[2], acc[3])), u0, u1);
  return u0 + u1;
}

struct VerifyReqDev {
  const bf16* q;
  bf16* o;
  int32_t ctx, n_rows, mtiles, n_full, tiles;
  int32_t unit_begin;   // first (KV head, row tile) unit of the request
  int32_t ug_begin;     // row-tile mode: first (KV head) unit of the request
  int64_t tile_begin;
  // row-statistics / column-sum modes (the importance votes): lse [Hkv][mtiles * 128] (written by
  // the statistics pass, read by the votes pass) and votes [Hkv * mtiles][ctx + n_rows]
  float* lse;
  float* votes;
};

// Kernel modes: attention (verification), the rows' log-sum-exp only, and the column sums of the
// normalised weights (sum over the tile's rows of 2^(s - lse) for every key). VMODE_ROWS (opt-in,
// VC_VERIFY_ROWS=1) is attention with every 128-row tile of a (request, KV head) in one CTA: a
// unit is the KV head, each K/V tile is loaded once and serves all its row tiles (up to VROWS), one
// O accumulator per row tile in TMEM. By default a KV head with more than 128 rows (L x G > 128) is
// one unit per row tile and streams its K and V once per row tile.
// VMODE_PAIR (the default for a KV head of exactly two row tiles): both row tiles of the head in one
// CTA with a softmax warpgroup each (warps 0-3 and 6-9), each with its own Q and P tiles, S double
// buffer and O accumulator; a K/V tile is loaded once and serves both, and the two warpgroups keep
// the softmax throughput of two one-tile CTAs.
// VMODE_TRIO (opt-in, VC_VERIFY_TRIO=1, for a KV head of exactly three row tiles): all three in
// one CTA, reading each K/V tile once. Three O accumulators take 384 TMEM columns, which leaves one 64-column S
// buffer for each of two softmax warpgroups: warpgroup 0 holds row tiles 0 and 2, warpgroup 1 row
// tile 1. A warpgroup's S buffer is freed as soon as its softmax has read it into registers, so the
// next S is computed while that softmax works; P alternates between two shared-memory tiles.
constexpr int VMODE_ATTN = 0, VMODE_STATS = 1, VMODE_VOTES = 2, VMODE_ROWS = 3, VMODE_PAIR = 4, VMODE_TRIO = 5;
constexpr int VROWS = 3;  // row tiles a row-tile-mode CTA holds (3 x 128 O columns + S fill TMEM)

struct VerifyParams {
  CUtensorMap tm[VC_MAX_BATCH][4];  // K full, V full, K new, V new
  VerifyReqDev req[VC_MAX_BATCH];
  int32_t B, Hq, Hkv, G, n_cta, n_units;
  int32_t h0;  // first KV head of the call's head range (units cover heads h0 .. h0 + nh - 1)
  int32_t rows;  // 0: a unit per row tile; 1 row-tile, 2 pair, 3 trio mode: a unit per (request, KV head)
  int64_t total_tiles;
  float scale_log2;
  float* ws_o;    // [slots][128][d]
  float* ws_lse;  // [slots][128]
  int32_t* dev_status;
};

// NQ: Q tiles a CTA holds; MWG: 0 one softmax warpgroup, 1 pair mode, 2 trio mode.
template <int D, int NQ = 1, int MWG = 0>
struct VCfg {
  static constexpr bool PAIR = MWG == 1, TRIO = MWG == 2;
  static constexpr int KB = D / 64;                // 64-channel (128-byte) blocks
  static constexpr int Q_BYTES = KB * VM * 128;    // Q tile, K-major SW128 (NQ of them)
  static constexpr int P_BYTES = VM * 128;         // P tile (64 tokens), K-major SW128
  static constexpr int KV_BYTES = KB * VBN * 128;  // one K (or V) tile
  static constexpr int OFF_P = NQ * Q_BYTES;       // P tile (pair mode: one per warpgroup; trio: two)
  static constexpr int OFF_K = OFF_P + (TRIO ? 4 : PAIR ? 2 : 1) * P_BYTES;  // K stages [2]
  static constexpr int OFF_V = OFF_K + 2 * KV_BYTES;  // V stages [2]
  static constexpr int OFF_BAR = OFF_V + 2 * KV_BYTES;
  static constexpr int SMEM = OFF_BAR + 256;
  static_assert(SMEM <= 227 * 1024, "one CTA's shared memory");
  static constexpr int SCOL = 64;                  // S double buffer: TMEM columns [0,64) and [64,128)
  static constexpr int OCOL = 128;                 // O: TMEM columns [128, 128 + D) (row tile m: + m D)
  static constexpr uint32_t TCOLS = NQ == 1 ? 256 : 512;
  static_assert(OCOL + NQ * D <= (int)TCOLS, "O accumulators fit the TMEM allocation");
  static constexpr int THREADS = MWG ? 352 : 192;  // warps 0-3 softmax, 4 MMA issue, 5 TMA loads (pair, trio: 6-9 softmax, 10 MMA issue)
  // pair mode: warpgroup m's S double buffer at TMEM columns [m 128, m 128 + 128), its O at 256 + m D
  static constexpr int PSCOL = 128;
  static constexpr int POCOL = 256;
  static_assert(!PAIR || (POCOL + 2 * D <= (int)TCOLS && NQ == 2), "pair mode fits TMEM");
  // trio mode: warpgroup w's S buffer at TMEM columns [64 w, 64 w + 64), row tile m's O at 128 + m D
  static_assert(!TRIO || (OCOL + 3 * D <= (int)TCOLS && NQ == 3), "trio mode fits TMEM");
  // votes mode, over the (unused) V stages: a second P tile, then the all-ones A operand of the
  // column-sum MMA. Its 128 rows are alike, so the operand's descriptor steps 16 bytes from one
  // 8-row group to the next and every row it reads lies in the first 1,264 bytes of the tile
  static constexpr int OFF_P1_VOTES = OFF_V;
  static constexpr int OFF_ONES_VOTES = OFF_V + P_BYTES;
  static constexpr int ONES_BYTES = 2048;
  static constexpr int OFF_BAR_VOTES =
      OFF_ONES_VOTES + ONES_BYTES > OFF_BAR ? OFF_ONES_VOTES + ONES_BYTES : OFF_BAR;
  static constexpr int SMEM_VOTES = OFF_BAR_VOTES + 256;
};

template <int D, int MODE>
using VCfgOf = VCfg<D, MODE == VMODE_ROWS ? VROWS : MODE == VMODE_TRIO ? 3 : MODE == VMODE_PAIR ? 2 : 1,
                    MODE == VMODE_TRIO ? 2 : MODE == VMODE_PAIR ? 1 : 0>;

__device__ __forceinline__ int find_req(const VerifyParams& p, int64_t tile) {
  int b = 0;
#pragma unroll 1
  for (int i = 1; i < p.B; ++i)
    if (p.req[i].tile_begin <= tile) b = i;
  return b;
}

// Bounded mbarrier wait that also gives up when another role of the CTA has aborted.
__device__ __forceinline__ bool vwait(uint64_t* bar, uint32_t parity, int32_t* st, volatile int* abort) {
  for (uint32_t it = 0; it < kSpinLimit; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 31u) == 31u && *abort) return false;
  }
  set_status(st, VC_DEV_TIMEOUT);
  *abort = 1;
  return false;
}

// One piece of the CTA's tile range: tiles [j0, j1) of unit ul of request b.
struct VPiece {
  int b, ul, j0, j1;
};

__device__ __forceinline__ VPiece verify_piece(const VerifyParams& p, int64_t pos, int64_t end) {
  VPiece q;
  q.b = find_req(p, pos);
  const VerifyReqDev& R = p.req[q.b];
  const int64_t rel = pos - R.tile_begin;
  q.ul = (int)(rel / R.tiles);
  q.j0 = (int)(rel % R.tiles);
  const int64_t left = end - pos;
  q.j1 = left < (int64_t)(R.tiles - q.j0) ? q.j0 + (int)left : R.tiles;
  return q;
}

template <int D, int MODE>
__global__ void __launch_bounds__((MODE == VMODE_PAIR || MODE == VMODE_TRIO) ? 352 : 192,
                                  (MODE == VMODE_ROWS || MODE == VMODE_PAIR || MODE == VMODE_TRIO) ? 1 : 2)
    verify_attn_kernel(const __grid_constant__ VerifyParams p) {
  using C = VCfgOf<D, MODE>;
  constexpr bool KV_HEAD_UNITS = MODE == VMODE_ROWS || MODE == VMODE_PAIR || MODE == VMODE_TRIO;
  // K stages: the statistics mode loads no V, so its K ring also takes the V stages (four K tiles
  // in flight per CTA instead of two)
  constexpr int KST = MODE == VMODE_STATS ? 4 : 2;
  extern __shared__ __align__(1024) uint8_t smem[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (smem_u32(smem) & 1023u) {  // the swizzled layouts need 1024-byte aligned tiles
    pdl_launch_dependents();
    pdl_wait();
    if (tid == 0) set_status(p.dev_status, VC_DEV_INTERNAL);
    return;
  }
  uint8_t* sQ = smem;
  uint8_t* sP = smem + C::OFF_P;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + (MODE == VMODE_VOTES ? C::OFF_BAR_VOTES : C::OFF_BAR));
  uint64_t* kfull = bars + 0;   // [2] K tile landed (TMA bytes)
  uint64_t* vfull = bars + 2;   // [2] V tile landed
  uint64_t* kempty = bars + 4;  // [2] the S MMA that read a K stage is done
  uint64_t* vempty = bars + 6;  // [2] the P V MMA that read a V stage is done
  uint64_t* sfull = bars + 8;   // [2] S tile g in TMEM buffer g & 1
  uint64_t* pfull = bars + 10;  // P tile in shared memory (4 softmax warps)
  uint64_t* ofull = bars + 11;  // O += P V done
  uint64_t* qfull = bars + 12;  // the unit's Q tile in shared memory (4 softmax warps)
  uint64_t* xbar = bars + 13;   // drain on the error path
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + 14);
  volatile int* s_abort = reinterpret_cast<volatile int*>(bars + 15);
  // pair mode, warpgroup 1: its S buffers' fills, P tile, P V done, Q tile (warpgroup 0 uses the above)
  uint64_t* sfull1 = bars + 16;  // [2]
  uint64_t* pfull1 = bars + 18;
  uint64_t* ofull1 = bars + 19;
  uint64_t* qfull1 = bars + 20;
  uint64_t* xbar1 = bars + 21;  // warpgroup 1's MMA issuer's drain
  // trio mode, warpgroup w's block at bars + 16 + 8 w (in place of the pair block): S filled, S read
  // into registers (4 softmax warps), P tile b written [2] (4 warps), P V of P tile b done [2], the
  // unit's Q tiles written (4 warps), its MMA issuer's drain
  auto trio_bars = [&](int w) { return bars + 16 + 8 * w; };
  // the K ring's barriers: kfull / kempty, or in the statistics mode four of each in the block the
  // pair and trio modes use
  uint64_t* kf = MODE == VMODE_STATS ? bars + 16 : kfull;
  uint64_t* ke = MODE == VMODE_STATS ? bars + 20 : kempty;
  // votes mode: P tile b written (4 softmax warps) and its column sums done, b = tile & 1
  uint64_t* pfv = bars + 16;  // [2]
  uint64_t* ofv = bars + 18;  // [2]

  if (warp == 0) tc05::alloc(tslot, C::TCOLS);
  if (tid == 0) {
    for (int i = 0; i < 10; ++i) mbar_init(&bars[i], 1);
    // statistics mode: the (unused) V barriers become per-S-buffer releases by the 4 softmax warps.
    // A single release barrier could complete two phases (two tiles read) before the MMA warp
    // waits for the first, and the parity wait would then miss it; per buffer, a phase can only
    // complete after the MMA warp has waited for the previous one (it issues that buffer's next S).
    if (MODE == VMODE_VOTES) {
      for (int i = 0; i < 2; ++i) {
        mbar_init(&pfv[i], 4);
        mbar_init(&ofv[i], 1);
      }
    }
    if (MODE == VMODE_STATS) {
      mbar_init(&vfull[0], 4);
      mbar_init(&vfull[1], 4);
      for (int i = 0; i < KST; ++i) {
        mbar_init(&kf[i], 1);
        mbar_init(&ke[i], 1);
      }
    }
    mbar_init(pfull, 4);
    mbar_init(ofull, 1);
    mbar_init(qfull, 4);
    mbar_init(xbar, 1);
    if (MODE == VMODE_PAIR || MODE == VMODE_TRIO) {
      // a K (V) stage is free once both warpgroups' issuers have committed their S (P V) of it
      for (int i = 0; i < 2; ++i) {
        mbar_init(&kempty[i], 2);
        mbar_init(&vempty[i], 2);
      }
    }
    if (MODE == VMODE_TRIO) {
      for (int w = 0; w < 2; ++w) {
        uint64_t* tb = trio_bars(w);
        const uint32_t cnt[8] = {1, 4, 4, 4, 1, 1, 4, 1};
        for (int i = 0; i < 8; ++i) mbar_init(&tb[i], cnt[i]);
      }
    }
    if (MODE == VMODE_PAIR) {
      mbar_init(xbar1, 1);
      mbar_init(&sfull1[0], 1);
      mbar_init(&sfull1[1], 1);
      mbar_init(pfull1, 4);
      mbar_init(ofull1, 1);
      mbar_init(qfull1, 4);
    }
    fence_mbar_init();
    *s_abort = 0;
  }
  if constexpr (MODE == VMODE_VOTES) {
    for (int e = tid; e < C::ONES_BYTES / 16; e += C::THREADS)
      reinterpret_cast<uint4*>(smem + C::OFF_ONES_VOTES)[e] =
          make_uint4(0x3C003C00u, 0x3C003C00u, 0x3C003C00u, 0x3C003C00u);
    fence_proxy_async_smem();  // the tensor cores read it
  }
  tc05::fence_before();
  __syncthreads();
  tc05::fence_after();
  pdl_launch_dependents();
  pdl_wait();
  const uint32_t tmem = *tslot;

  const int64_t T = p.total_tiles, N = p.n_cta, c = blockIdx.x;
  const int64_t beg = c * T / N, end = (c + 1) * T / N;

  // pair mode: the MMA chain of warpgroup m's row tile over the CTA's units, issued by one thread
  // (warp 4 for warpgroup 0, warp 10 for warpgroup 1): S of tile g before P V of tile g - 1, as in
  // the one-tile mode; both issuers commit every K and V stage's release (two arrivals each), the
  // second also for tiles of a one-tile head, where it has no MMA of its own
  auto pair_issue = [&](int m) -> bool {
    constexpr uint32_t IDESC_S = tc05::idesc_bf16(VM, VBN, false);
    constexpr uint32_t IDESC_O = tc05::idesc_bf16(VM, D, true);
    const uint32_t aQ = smem_u32(sQ) + m * C::Q_BYTES, aP = smem_u32(sP) + m * C::P_BYTES,
                   aK = smem_u32(smem + C::OFF_K), aV = smem_u32(smem + C::OFF_V);
    uint64_t* sf = m ? sfull1 : sfull;
    uint64_t* pf = m ? pfull1 : pfull;
    uint64_t* of = m ? ofull1 : ofull;
    uint64_t* qf = m ? qfull1 : qfull;
    uint32_t g = 0, t = 0, pw = 0, uq = 0;
    bool ok = true;
    auto pv = [&](uint32_t gp, bool acc, bool mine) -> bool {
      if (!vwait(&vfull[gp & 1], (gp >> 1) & 1, p.dev_status, s_abort)) return false;
      if (mine) {
        if (!vwait(pf, pw & 1, p.dev_status, s_abort)) return false;
        tc05::fence_after();
        const uint32_t vaddr = aV + (gp & 1) * C::KV_BYTES;
#pragma unroll
        for (int kk = 0; kk < VBN / 16; ++kk) {
          const uint64_t da = tc05::sdesc_sw128(aP + kk * 32, 16, 1024);
          const uint64_t db = tc05::sdesc_sw128(vaddr + kk * 2048, VBN * 128, 1024);
          tc05::mma_bf16(tmem + C::POCOL + m * D, da, db, IDESC_O, (acc || kk > 0) ? 1u : 0u);
        }
        tc05::commit(of);
        ++pw;
      }
      tc05::commit(&vempty[gp & 1]);
      return true;
    };
    for (int64_t pos = beg; pos < end && ok;) {
      const VPiece q = verify_piece(p, pos, end);
      const int nt = q.j1 - q.j0;
      const bool mine = m < p.req[q.b].mtiles;
      if (mine) {
        ok = vwait(qf, uq & 1, p.dev_status, s_abort);
        ++uq;
      }
      for (int jj = 0; jj < nt && ok; ++jj) {
        const uint32_t gc = g + jj;
        if (!vwait(&kfull[gc & 1], (gc >> 1) & 1, p.dev_status, s_abort)) {
          ok = false;
          break;
        }
        if (mine) {
          tc05::fence_after();
          const uint32_t kaddr = aK + (gc & 1) * C::KV_BYTES;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint64_t da = tc05::sdesc_sw128(aQ + (kk >> 2) * (VM * 128) + (kk & 3) * 32, 16, 1024);
            const uint64_t db = tc05::sdesc_sw128(kaddr + (kk >> 2) * (VBN * 128) + (kk & 3) * 32, 16, 1024);
            tc05::mma_bf16(tmem + m * C::PSCOL + (t & 1) * C::SCOL, da, db, IDESC_S, kk > 0);
          }
          tc05::commit(&sf[t & 1]);
          ++t;
        }
        tc05::commit(&kempty[gc & 1]);
        if (jj > 0) ok = pv(gc - 1, jj > 1, mine);
      }
      if (ok) ok = pv(g + nt - 1, nt > 1, mine);
      g += nt;
      pos += nt;
    }
    return ok;
  };

  // trio mode: the MMA chain of warpgroup w (warp 4 for w = 0, warp 10 for w = 1) over the CTA's
  // units. Its steps are (KV tile, row tile) pairs in order, its row tiles being w and w + 2 of the
  // three. Step k's S goes into the warpgroup's one S buffer once the softmax has read step
  // k - 1's out of it (early in that step), and S runs one KV tile ahead of P V: the P V of a
  // step follows the S of the same row tile on the next KV tile (for warpgroup 0, two steps
  // later). So warpgroup 0's next S never queues behind a P V that waits for the P of the step
  // just finished, and the softmax of step k, which rewrites the P tile of step k - 2, finds that
  // P V issued; a lag of one KV tile, not more, keeps each V stage in use for about one KV tile.
  // A unit's pending P V are issued before the next unit's Q is awaited. Both issuers commit each
  // K stage's release after their last S on it and each V stage's after their last P V on it.
  auto trio_issue = [&](int w) -> bool {
    constexpr uint32_t IDESC_S = tc05::idesc_bf16(VM, VBN, false);
    constexpr uint32_t IDESC_O = tc05::idesc_bf16(VM, D, true);
    uint64_t* tb = trio_bars(w);
    uint64_t *sf = tb, *sr = tb + 1, *pf = tb + 2, *of = tb + 4, *qf = tb + 6;
    const int ntw = w == 0 ? 2 : 1;
    const uint32_t aQ = smem_u32(sQ), aP = smem_u32(sP) + 2 * w * C::P_BYTES, aK = smem_u32(smem + C::OFF_K),
                   aV = smem_u32(smem + C::OFF_V), tS = tmem + w * VBN;
    uint32_t g = 0, k = 0, uq = 0;
    bool ok = true;
    // a step whose P V is still to be issued: row tile m, KV tile (V stage) gp; acc: not the unit's
    // first KV tile; last: this warpgroup's last row tile on that V tile
    struct Pend {
      uint32_t s, gp;
      int m;
      bool acc, last;
    };
    auto pv = [&](const Pend& e) -> bool {
      if (!vwait(&vfull[e.gp & 1], (e.gp >> 1) & 1, p.dev_status, s_abort)) return false;
      if (!vwait(&pf[e.s & 1], (e.s >> 1) & 1, p.dev_status, s_abort)) return false;
      tc05::fence_after();
      const uint32_t pbuf = aP + (e.s & 1) * C::P_BYTES, vaddr = aV + (e.gp & 1) * C::KV_BYTES;
#pragma unroll
      for (int kk = 0; kk < VBN / 16; ++kk) {
        const uint64_t da = tc05::sdesc_sw128(pbuf + kk * 32, 16, 1024);
        const uint64_t db = tc05::sdesc_sw128(vaddr + kk * 2048, VBN * 128, 1024);
        tc05::mma_bf16(tmem + C::OCOL + e.m * D, da, db, IDESC_O, (e.acc || kk > 0) ? 1u : 0u);
      }
      tc05::commit(&of[e.s & 1]);
      if (e.last) tc05::commit(&vempty[e.gp & 1]);
      return true;
    };
    for (int64_t pos = beg; pos < end && ok;) {
      const VPiece q = verify_piece(p, pos, end);
      const int nt = q.j1 - q.j0;
      ok = vwait(qf, uq & 1, p.dev_status, s_abort);
      ++uq;
      Pend pa{}, pb{};  // pending P V, oldest first
      int np = 0;
      for (int jj = 0; jj < nt && ok; ++jj) {
        const uint32_t gc = g + jj;
        if (!vwait(&kfull[gc & 1], (gc >> 1) & 1, p.dev_status, s_abort)) {
          ok = false;
          break;
        }
        for (int i = 0; i < ntw && ok; ++i) {
          const int m = w + 2 * i;
          // the softmax has read step k - 1's S out of the buffer
          if (k >= 1 && !vwait(sr, (k - 1) & 1, p.dev_status, s_abort)) {
            ok = false;
            break;
          }
          tc05::fence_after();
          const uint32_t kaddr = aK + (gc & 1) * C::KV_BYTES;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint64_t da =
                tc05::sdesc_sw128(aQ + m * C::Q_BYTES + (kk >> 2) * (VM * 128) + (kk & 3) * 32, 16, 1024);
            const uint64_t db = tc05::sdesc_sw128(kaddr + (kk >> 2) * (VBN * 128) + (kk & 3) * 32, 16, 1024);
            tc05::mma_bf16(tS, da, db, IDESC_S, kk > 0);
          }
          tc05::commit(sf);
          if (i == ntw - 1) tc05::commit(&kempty[gc & 1]);
          if (np == ntw) {
            ok = pv(pa);
            pa = pb;
            --np;
          }
          (np == 0 ? pa : pb) = Pend{k, gc, m, jj > 0, i == ntw - 1};
          ++np;
          ++k;
        }
      }
      if (np >= 1 && ok) ok = pv(pa);
      if (np == 2 && ok) ok = pv(pb);
      g += nt;
      pos += nt;
    }
    return ok;
  };

  if (warp == 5) {
    // ---- TMA producer: K of tile g, then V of tile g - 1 (K runs a tile ahead of V) ----------
    if (lane == 0) {
      uint32_t g = 0, gk = 0, gv = 0;  // tiles issued (K, V)
      int pv_b = 0, pv_hk = 0, pv_j = 0;
      bool pv_pending = false;
      auto load = [&](bool isv, uint32_t gi, int b, int hk, int j) -> bool {
        const uint32_t nst = isv ? 2 : KST;
        const int st = gi % nst;
        if (gi >= nst && !vwait(isv ? &vempty[st] : &ke[st], ((gi - nst) / nst) & 1, p.dev_status, s_abort))
          return false;
        const VerifyReqDev& R = p.req[b];
        uint64_t* bar = isv ? &vfull[st] : &kf[st];
        uint8_t* dst = smem + (isv ? C::OFF_V : C::OFF_K) + st * C::KV_BYTES;
        const bool isnew = j >= R.n_full;
        const int tok = isnew ? (j - R.n_full) * VBN : j * VBN;
        const void* map = &p.tm[b][(isnew ? 2 : 0) + (isv ? 1 : 0)];
        mbar_arrive_expect_tx(bar, C::KV_BYTES);
#pragma unroll
        for (int kb = 0; kb < C::KB; ++kb) tc05::tma_load_3d(dst + kb * (VBN * 128), map, kb * 64, tok, hk, bar);
        return true;
      };
      bool ok = true;
      for (int64_t pos = beg; pos < end && ok;) {
        const VPiece q = verify_piece(p, pos, end);
        const int hk = p.h0 + (KV_HEAD_UNITS ? q.ul : q.ul / p.req[q.b].mtiles);
        for (int j = q.j0; j < q.j1 && ok; ++j, ++g) {
          ok = load(false, gk, q.b, hk, j);
          if (ok) ++gk;
          if ((MODE == VMODE_ATTN || KV_HEAD_UNITS) && ok && pv_pending) {
            ok = load(true, gv, pv_b, pv_hk, pv_j);
            if (ok) ++gv;
          }
          pv_b = q.b, pv_hk = hk, pv_j = j, pv_pending = true;
        }
        pos += q.j1 - q.j0;
      }
      if ((MODE == VMODE_ATTN || KV_HEAD_UNITS) && ok && pv_pending &&
          load(true, gv, pv_b, pv_hk, pv_j))
        ++gv;
      if (*s_abort) {
        // drain (bounded): the loads of the last tiles of each kind (a ring's worth) may still be landing
        for (uint32_t gi = (gk > (uint32_t)KST ? gk - KST : 0); gi < gk; ++gi)
          mbar_wait_bounded(&kf[gi % KST], (gi / KST) & 1, p.dev_status);
        for (uint32_t gi = (gv > 2 ? gv - 2 : 0); gi < gv; ++gi) mbar_wait_bounded(&vfull[gi & 1], (gi >> 1) & 1, p.dev_status);
      }
    }
  } else if (warp == 4) {
    // ---- MMA issue: S of tile g (into TMEM buffer g & 1) before P V of tile g - 1 -------------
    if (lane == 0) {
      constexpr uint32_t IDESC_S = tc05::idesc_bf16(VM, VBN, false);
      constexpr uint32_t IDESC_O = tc05::idesc_bf16(VM, D, true);
      const uint32_t aQ = smem_u32(sQ), aP = smem_u32(sP), aK = smem_u32(smem + C::OFF_K),
                     aV = smem_u32(smem + C::OFF_V);
      uint32_t g = 0, u = 0;
      bool ok = true;
      auto issue_pv = [&](uint32_t gp, bool acc) -> bool {
        if constexpr (MODE == VMODE_STATS) {
          // tile gp's S has been read: its TMEM buffer may take tile gp + 2
          return vwait(&vfull[gp & 1], (gp >> 1) & 1, p.dev_status, s_abort);
        }
        if constexpr (MODE == VMODE_VOTES) {
          // column sums of P tile gp & 1 (fp16, [128 rows = K][64 keys = N], MN-major) by an
          // all-ones A, into TMEM buffer gp & 1
          if (!vwait(&pfv[gp & 1], (gp >> 1) & 1, p.dev_status, s_abort)) return false;
          constexpr uint32_t IDESC_C = tc05::idesc_f16(VM, VBN, true);
          const uint32_t aOnes = smem_u32(smem + C::OFF_ONES_VOTES);
          const uint32_t aPb = (gp & 1) ? smem_u32(smem + C::OFF_P1_VOTES) : aP;
          tc05::fence_after();
#pragma unroll
          for (int kk = 0; kk < VM / 16; ++kk) {
            const uint64_t da = tc05::sdesc_sw128(aOnes + (kk & 3) * 32, 16, 16);
            const uint64_t db = tc05::sdesc_sw128(aPb + kk * 2048, VM * 128, 1024);
            tc05::mma_bf16(tmem + C::OCOL + (gp & 1) * VBN, da, db, IDESC_C, kk > 0 ? 1u : 0u);
          }
          tc05::commit(&ofv[gp & 1]);
          return true;
        }
        if (!vwait(pfull, gp & 1, p.dev_status, s_abort)) return false;
        if (!vwait(&vfull[gp & 1], (gp >> 1) & 1, p.dev_status, s_abort)) return false;
        tc05::fence_after();
        const uint32_t vaddr = aV + (gp & 1) * C::KV_BYTES;
#pragma unroll
        for (int kk = 0; kk < VBN / 16; ++kk) {
          const uint64_t da = tc05::sdesc_sw128(aP + kk * 32, 16, 1024);
          const uint64_t db = tc05::sdesc_sw128(vaddr + kk * 2048, VBN * 128, 1024);
          tc05::mma_bf16(tmem + C::OCOL, da, db, IDESC_O, (acc || kk > 0) ? 1u : 0u);
        }
        tc05::commit(ofull);
        tc05::commit(&vempty[gp & 1]);
        return true;
      };
      // row-tile mode: steps are (KV tile, row tile) pairs, S of step v before P V of step v - 1;
      // a K stage is released after its last row tile's S, a V stage after its last row tile's P V
      uint32_t vg = 0;  // steps issued
      auto issue_pv_rows = [&](uint32_t vp, uint32_t gp, int m, bool first_v, bool last_v, bool acc) -> bool {
        if (!vwait(pfull, vp & 1, p.dev_status, s_abort)) return false;
        if (first_v && !vwait(&vfull[gp & 1], (gp >> 1) & 1, p.dev_status, s_abort)) return false;
        tc05::fence_after();
        const uint32_t vaddr = aV + (gp & 1) * C::KV_BYTES;
#pragma unroll
        for (int kk = 0; kk < VBN / 16; ++kk) {
          const uint64_t da = tc05::sdesc_sw128(aP + kk * 32, 16, 1024);
          const uint64_t db = tc05::sdesc_sw128(vaddr + kk * 2048, VBN * 128, 1024);
          tc05::mma_bf16(tmem + C::OCOL + m * D, da, db, IDESC_O, (acc || kk > 0) ? 1u : 0u);
        }
        tc05::commit(ofull);
        if (last_v) tc05::commit(&vempty[gp & 1]);
        return true;
      };
      for (int64_t pos = beg; pos < end && ok && MODE == VMODE_ROWS;) {
        const VPiece q = verify_piece(p, pos, end);
        const int nt = q.j1 - q.j0, mt = p.req[q.b].mtiles;
        ok = vwait(qfull, u & 1, p.dev_status, s_abort);
        ++u;
        bool pend = false, pv_first = false, pv_last = false, pv_acc = false;
        uint32_t pv_v = 0, pv_g = 0;
        int pv_m = 0;
        for (int jj = 0; jj < nt && ok; ++jj) {
          const uint32_t gc = g + jj;
          if (!vwait(&kfull[gc & 1], (gc >> 1) & 1, p.dev_status, s_abort)) {
            ok = false;
            break;
          }
          tc05::fence_after();
          const uint32_t kaddr = aK + (gc & 1) * C::KV_BYTES;
          for (int m = 0; m < mt && ok; ++m) {
            const uint32_t vc = vg++;
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint64_t da =
                  tc05::sdesc_sw128(aQ + m * C::Q_BYTES + (kk >> 2) * (VM * 128) + (kk & 3) * 32, 16, 1024);
              const uint64_t db = tc05::sdesc_sw128(kaddr + (kk >> 2) * (VBN * 128) + (kk & 3) * 32, 16, 1024);
              tc05::mma_bf16(tmem + (vc & 1) * C::SCOL, da, db, IDESC_S, kk > 0);
            }
            tc05::commit(&sfull[vc & 1]);
            if (m == mt - 1) tc05::commit(&kempty[gc & 1]);
            if (pend) ok = issue_pv_rows(pv_v, pv_g, pv_m, pv_first, pv_last, pv_acc);
            pend = true;
            pv_v = vc, pv_g = gc, pv_m = m, pv_first = m == 0, pv_last = m == mt - 1, pv_acc = jj > 0;
          }
        }
        if (ok && pend) ok = issue_pv_rows(pv_v, pv_g, pv_m, pv_first, pv_last, pv_acc);
        g += nt;
        pos += nt;
      }
      // pair mode: this thread issues the MMAs of warpgroup 0 (warp 4) -- warpgroup 1 has its own
      // issuer (warp 10, below) -- so the two row tiles' chains run independently; each commits its
      // S and P V to the shared K and V stage releases (two arrivals each)
      if constexpr (MODE == VMODE_PAIR) ok = pair_issue(0);
      if constexpr (MODE == VMODE_TRIO) ok = trio_issue(0);
      for (int64_t pos = beg; pos < end && ok && !KV_HEAD_UNITS;) {
        const VPiece q = verify_piece(p, pos, end);
        const int nt = q.j1 - q.j0;
        ok = vwait(qfull, u & 1, p.dev_status, s_abort);
        ++u;
        for (int jj = 0; jj < nt && ok; ++jj) {
          const uint32_t gc = g + jj;
          if (!vwait(&kf[gc % KST], (gc / KST) & 1, p.dev_status, s_abort)) {
            ok = false;
            break;
          }
          tc05::fence_after();
          const uint32_t kaddr = aK + (gc % KST) * C::KV_BYTES;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint64_t da = tc05::sdesc_sw128(aQ + (kk >> 2) * (VM * 128) + (kk & 3) * 32, 16, 1024);
            const uint64_t db = tc05::sdesc_sw128(kaddr + (kk >> 2) * (VBN * 128) + (kk & 3) * 32, 16, 1024);
            tc05::mma_bf16(tmem + (gc & 1) * C::SCOL, da, db, IDESC_S, kk > 0);
          }
          tc05::commit(&sfull[gc & 1]);
          tc05::commit(&ke[gc % KST]);
          if (jj > 0) ok = issue_pv(gc - 1, jj > 1);
        }
        if (ok) ok = issue_pv(g + nt - 1, nt > 1);
        g += nt;
        pos += nt;
      }
      // every MMA issued so far has completed before TMEM is released (bounded, even after an abort)
      tc05::commit(xbar);
      mbar_wait_bounded(xbar, 0, p.dev_status);
    }
  } else if (MODE == VMODE_PAIR && warp == 10) {
    // ---- pair mode: warpgroup 1's MMA issue; its MMAs complete before TMEM is released ----------
    if (lane == 0) {
      pair_issue(1);
      tc05::commit(xbar1);
      mbar_wait_bounded(xbar1, 0, p.dev_status);
    }
  } else if (MODE == VMODE_TRIO && warp == 10) {
    // ---- trio mode: warpgroup 1's MMA issue -------------------------------------------------------
    if (lane == 0) {
      trio_issue(1);
      tc05::commit(&trio_bars(1)[7]);
      mbar_wait_bounded(&trio_bars(1)[7], 0, p.dev_status);
    }
  } else {
    // ---- softmax warps: thread tid owns TMEM lane tid = query row tid of the tile ---------------
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    uint32_t g = 0;
    bool ok = true;
    if constexpr (MODE == VMODE_PAIR) {
      // warpgroup wg (warps 0-3: 0, warps 6-9: 1) owns row tile wg of each unit; thread rt =
      // (warp % 4) * 32 + lane owns row rt of that tile, which is its TMEM lane
      const int wg = warp >= 6 ? 1 : 0;
      const int rt = (warp & 3) * 32 + lane;
      const uint32_t lo = (uint32_t)((warp & 3) * 32) << 16;
      uint64_t* sf = wg ? sfull1 : sfull;
      uint64_t* pf = wg ? pfull1 : pfull;
      uint64_t* of = wg ? ofull1 : ofull;
      uint64_t* qf = wg ? qfull1 : qfull;
      uint8_t* sQw = sQ + wg * C::Q_BYTES;
      uint8_t* sPw = sP + wg * C::P_BYTES;
      const uint32_t t_s0 = tmem + lo + wg * C::PSCOL, t_o0 = tmem + lo + C::POCOL + wg * D;
      uint32_t t = 0, sp = 0;  // this warpgroup's S tiles read and P tiles written
      for (int64_t pos = beg; pos < end && ok;) {
        const VPiece q = verify_piece(p, pos, end);
        const VerifyReqDev& R = p.req[q.b];
        const int nt = q.j1 - q.j0;
        pos += nt;
        if (wg >= R.mtiles) continue;  // a head of one row tile: warpgroup 1 holds nothing of it
        const int hk = p.h0 + q.ul;
        const int ug_global = R.ug_begin + q.ul;
        const int Rw = wg * VM + rt, qi = Rw / p.G, qg = Rw % p.G;
        const bool row_ok = qi < R.n_rows;
        // this thread's query row into the warpgroup's swizzled Q tile; its previous unit's MMAs are
        // complete (that unit's epilogue waited for its last P V, which follows all its S)
        {
          const uint4* src = reinterpret_cast<const uint4*>(R.q + ((size_t)qi * p.Hq + hk * p.G + qg) * D);
#pragma unroll
          for (int kb = 0; kb < C::KB; ++kb)
#pragma unroll
            for (int ch = 0; ch < 8; ++ch) {
              const uint4 v = row_ok ? __ldg(src + kb * 8 + ch) : make_uint4(0, 0, 0, 0);
              *reinterpret_cast<uint4*>(sQw + kb * (VM * 128) + rt * 128 + ((ch ^ (rt & 7)) << 4)) = v;
            }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(qf);
        float m_run = -INFINITY, l_run = 0.f;
        for (int jj = 0; jj < nt; ++jj) {
          const int j = q.j0 + jj;
          if (!vwait(&sf[t & 1], (t >> 1) & 1, p.dev_status, s_abort)) {
            ok = false;
            break;
          }
          tc05::fence_after();
          float x[VBN];
          {
            uint32_t r0[32], r1[32];
            const uint32_t t_s = t_s0 + (t & 1) * C::SCOL;
            tc05::ld32(t_s, r0);
            tc05::ld32(t_s + 32, r1);
            tc05::wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) {
              x[e] = __uint_as_float(r0[e]);
              x[32 + e] = __uint_as_float(r1[e]);
            }
          }
          ++t;
          {
            const int last = j < R.n_full ? R.ctx - j * VBN - 1 : qi - (j - R.n_full) * VBN;  // last visible key
            if (last < VBN - 1) {
#pragma unroll
              for (int e = 0; e < VBN; ++e)
                if (e > last) x[e] = -INFINITY;
            }
          }
          const float mx = row_max(x) * p.scale_log2;
          const float m_new = fmaxf(m_run, mx);
          const bool need = jj > 0 && m_new > m_run + 8.f;
          if (jj > 0) {
            // this warpgroup's P V of the previous tile: O is stable and its P tile is free
            if (!vwait(of, (sp - 1) & 1, p.dev_status, s_abort)) {
              ok = false;
              break;
            }
            tc05::fence_after();
          }
          if (jj == 0) {
            m_run = m_new;
          } else {
            float f = 1.f;
            if (need) {
              f = ex2_approx(m_run - m_new);
              l_run *= f;
              m_run = m_new;
            }
            if (__any_sync(0xffffffffu, need)) {
#pragma unroll 1
              for (int cb = 0; cb < D / 32; ++cb) {
                uint32_t r[32];
                tc05::ld32(t_o0 + cb * 32, r);
                tc05::wait_ld();
#pragma unroll
                for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * f);
                tc05::st32(t_o0 + cb * 32, r);
              }
              tc05::wait_st();
            }
          }
          const float mu = (m_run == -INFINITY) ? 0.f : m_run;
          l_run += row_exp_to_p(x, p.scale_log2, mu, sPw + rt * 128, rt);
          fence_proxy_async_smem();
          tc05::fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(pf);
          ++sp;
        }
        if (!ok) break;
        // output: wait for this warpgroup's last P V of the unit
        if (!vwait(of, (sp - 1) & 1, p.dev_status, s_abort)) {
          ok = false;
          break;
        }
        tc05::fence_after();
        const bool whole = (q.j0 == 0 && q.j1 == R.tiles);
        const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
        const size_t slot = (size_t)(c + ug_global) * VROWS + wg;
#pragma unroll 1
        for (int cb = 0; cb < D / 32; ++cb) {
          uint32_t r[32];
          tc05::ld32(t_o0 + cb * 32, r);  // warp-collective: every lane loads
          tc05::wait_ld();
          if (!row_ok) continue;
          if (whole) {
            uint4* dst = reinterpret_cast<uint4*>(R.o + ((size_t)qi * p.Hq + hk * p.G + qg) * D + cb * 32);
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              uint32_t w[4];
#pragma unroll
              for (int e = 0; e < 4; ++e)
                w[e] = pack_bf16x2(__uint_as_float(r[8 * v + 2 * e]) * inv, __uint_as_float(r[8 * v + 2 * e + 1]) * inv);
              dst[v] = make_uint4(w[0], w[1], w[2], w[3]);
            }
          } else {
            float4* dst = reinterpret_cast<float4*>(p.ws_o + (slot * VM + rt) * D + cb * 32);
#pragma unroll
            for (int v = 0; v < 8; ++v)
              dst[v] = make_float4(__uint_as_float(r[4 * v]) * inv, __uint_as_float(r[4 * v + 1]) * inv,
                                   __uint_as_float(r[4 * v + 2]) * inv, __uint_as_float(r[4 * v + 3]) * inv);
          }
        }
        if (row_ok && !whole) p.ws_lse[slot * VM + rt] = l_run > 0.f ? m_run + log2f(l_run) : -INFINITY;
        tc05::fence_before();
      }
    }
    if constexpr (MODE == VMODE_TRIO) {
      // warpgroup w (warps 0-3: 0, warps 6-9: 1) owns row tiles w and w + 2 of each unit (warpgroup
      // 1: tile 1 only); thread rt = (warp % 4) * 32 + lane owns row rt of each, its TMEM lane
      const int w = warp >= 6 ? 1 : 0, ntw = w == 0 ? 2 : 1;
      const int rt = (warp & 3) * 32 + lane;
      const uint32_t lo = (uint32_t)((warp & 3) * 32) << 16;
      uint64_t* tb = trio_bars(w);
      uint64_t *sf = tb, *sr = tb + 1, *pf = tb + 2, *of = tb + 4, *qf = tb + 6;
      uint8_t* sPw = sP + 2 * w * C::P_BYTES;
      const uint32_t t_s = tmem + lo + w * VBN;
      uint32_t t = 0;  // this warpgroup's steps over the CTA's units
      // P V of step k done (P tile k & 1). Every step t >= 2 waits for k = t - 2 before it rewrites
      // that tile, so a wait for k finds the P V of k - 2 observed, and the P V of k + 2 cannot
      // have been issued (it needs this warpgroup's P of k + 2): the parity wait is exact
      auto pv_done = [&](uint32_t k) { return vwait(&of[k & 1], (k >> 1) & 1, p.dev_status, s_abort); };
      for (int64_t pos = beg; pos < end && ok;) {
        const VPiece q = verify_piece(p, pos, end);
        const VerifyReqDev& R = p.req[q.b];
        const int nt = q.j1 - q.j0;
        pos += nt;
        const int hk = p.h0 + q.ul;
        const int ug_global = R.ug_begin + q.ul;
        // this thread's query rows into the warpgroup's Q tiles (the previous unit's MMAs are
        // complete: its outputs waited for its last P V, which follow all its S)
        for (int i = 0; i < ntw; ++i) {
          const int m = w + 2 * i;
          const int Rw = m * VM + rt, qi = Rw / p.G, qg = Rw % p.G;
          const bool row_ok = qi < R.n_rows;
          const uint4* src = reinterpret_cast<const uint4*>(R.q + ((size_t)qi * p.Hq + hk * p.G + qg) * D);
          uint8_t* dQ = sQ + m * C::Q_BYTES;
#pragma unroll
          for (int kb = 0; kb < C::KB; ++kb)
#pragma unroll
            for (int ch = 0; ch < 8; ++ch) {
              const uint4 v = row_ok ? __ldg(src + kb * 8 + ch) : make_uint4(0, 0, 0, 0);
              *reinterpret_cast<uint4*>(dQ + kb * (VM * 128) + rt * 128 + ((ch ^ (rt & 7)) << 4)) = v;
            }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(qf);
        float m_run0 = -INFINITY, l_run0 = 0.f, m_run1 = -INFINITY, l_run1 = 0.f;
        for (int jj = 0; jj < nt && ok; ++jj) {
          const int j = q.j0 + jj;
          for (int i = 0; i < ntw; ++i) {
            const int m = w + 2 * i;
            const int qi = (m * VM + rt) / p.G;
            if (!vwait(sf, t & 1, p.dev_status, s_abort)) {
              ok = false;
              break;
            }
            tc05::fence_after();
            float x[VBN];
            {
              uint32_t r0[32], r1[32];
              tc05::ld32(t_s, r0);
              tc05::ld32(t_s + 32, r1);
              tc05::wait_ld();
              tc05::fence_before();  // the buffer may take the next step's S
              __syncwarp();
              if (lane == 0) mbar_arrive(sr);
#pragma unroll
              for (int e = 0; e < 32; ++e) {
                x[e] = __uint_as_float(r0[e]);
                x[32 + e] = __uint_as_float(r1[e]);
              }
            }
            {
              const int last = j < R.n_full ? R.ctx - j * VBN - 1 : qi - (j - R.n_full) * VBN;  // last visible key
              if (last < VBN - 1) {
#pragma unroll
                for (int e = 0; e < VBN; ++e)
                  if (e > last) x[e] = -INFINITY;
              }
            }
            const float mx = row_max(x) * p.scale_log2;
            // P tile t & 1 was read by the P V of step t - 2 (for warpgroup 0, also the last P V into
            // this row tile's O)
            if (t >= 2 && !pv_done(t - 2)) {
              ok = false;
              break;
            }
            float mr = i ? m_run1 : m_run0, lr = i ? l_run1 : l_run0;
            const float m_new = fmaxf(mr, mx);
            const bool need = jj > 0 && m_new > mr + 8.f;
            if (jj == 0) {
              mr = m_new;
            } else if (__any_sync(0xffffffffu, need)) {
              // O is rescaled once its last P V has completed: warpgroup 1's is the previous step's,
              // warpgroup 0's was waited for above
              if (ntw == 1 && !pv_done(t - 1)) {
                ok = false;
                break;
              }
              tc05::fence_after();
              float f = 1.f;
              if (need) {
                f = ex2_approx(mr - m_new);
                lr *= f;
                mr = m_new;
              }
              const uint32_t t_o = tmem + lo + C::OCOL + m * D;
#pragma unroll 1
              for (int cb = 0; cb < D / 32; ++cb) {
                uint32_t r[32];
                tc05::ld32(t_o + cb * 32, r);
                tc05::wait_ld();
#pragma unroll
                for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * f);
                tc05::st32(t_o + cb * 32, r);
              }
              tc05::wait_st();
            }
            const float mu = (mr == -INFINITY) ? 0.f : mr;
            lr += row_exp_to_p(x, p.scale_log2, mu, sPw + (t & 1) * C::P_BYTES + rt * 128, rt);
            if (i) {
              m_run1 = mr;
              l_run1 = lr;
            } else {
              m_run0 = mr;
              l_run0 = lr;
            }
            fence_proxy_async_smem();
            tc05::fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&pf[t & 1]);
            ++t;
          }
        }
        if (!ok) break;
        // outputs: each row tile's last P V of the unit (steps t - ntw .. t - 1)
        const bool whole = (q.j0 == 0 && q.j1 == R.tiles);
        for (int i = 0; i < ntw && ok; ++i) {
          const int m = w + 2 * i;
          if (!pv_done(t - ntw + i)) {
            ok = false;
            break;
          }
          tc05::fence_after();
          const int Rw = m * VM + rt, qi = Rw / p.G, qg = Rw % p.G;
          const bool row_ok = qi < R.n_rows;
          const float lr = i ? l_run1 : l_run0, mr = i ? m_run1 : m_run0;
          const float inv = lr > 0.f ? 1.f / lr : 0.f;
          const size_t slot = (size_t)(c + ug_global) * VROWS + m;
          const uint32_t t_o = tmem + lo + C::OCOL + m * D;
#pragma unroll 1
          for (int cb = 0; cb < D / 32; ++cb) {
            uint32_t r[32];
            tc05::ld32(t_o + cb * 32, r);  // warp-collective: every lane loads
            tc05::wait_ld();
            if (!row_ok) continue;
            if (whole) {
              uint4* dst = reinterpret_cast<uint4*>(R.o + ((size_t)qi * p.Hq + hk * p.G + qg) * D + cb * 32);
#pragma unroll
              for (int v = 0; v < 4; ++v) {
                uint32_t wv[4];
#pragma unroll
                for (int e = 0; e < 4; ++e)
                  wv[e] = pack_bf16x2(__uint_as_float(r[8 * v + 2 * e]) * inv, __uint_as_float(r[8 * v + 2 * e + 1]) * inv);
                dst[v] = make_uint4(wv[0], wv[1], wv[2], wv[3]);
              }
            } else {
              float4* dst = reinterpret_cast<float4*>(p.ws_o + (slot * VM + rt) * D + cb * 32);
#pragma unroll
              for (int v = 0; v < 8; ++v)
                dst[v] = make_float4(__uint_as_float(r[4 * v]) * inv, __uint_as_float(r[4 * v + 1]) * inv,
                                     __uint_as_float(r[4 * v + 2]) * inv, __uint_as_float(r[4 * v + 3]) * inv);
            }
          }
          if (row_ok && !whole) p.ws_lse[slot * VM + rt] = lr > 0.f ? mr + log2f(lr) : -INFINITY;
        }
        tc05::fence_before();
      }
    }
    // row-tile mode: thread tid owns row tid of every row tile of the unit; steps (KV tile, row
    // tile) in the MMA warp's order, one running maximum and sum per row tile
    uint32_t vg = 0;  // steps consumed
    for (int64_t pos = beg; pos < end && ok && MODE == VMODE_ROWS;) {
      const VPiece q = verify_piece(p, pos, end);
      const VerifyReqDev& R = p.req[q.b];
      const int nt = q.j1 - q.j0, mt = R.mtiles;
      const int hk = p.h0 + q.ul;
      const int ug_global = R.ug_begin + q.ul;
      // this thread's query row of each row tile into its swizzled Q tile (the previous unit's MMAs
      // are complete: its epilogue waited for the last P V, which follows every S of the unit)
      for (int m = 0; m < mt; ++m) {
        const int Rw = m * VM + tid, qi = Rw / p.G, qg = Rw % p.G;
        const bool row_ok = qi < R.n_rows;
        const uint4* src = reinterpret_cast<const uint4*>(R.q + ((size_t)qi * p.Hq + hk * p.G + qg) * D);
        uint8_t* dQ = sQ + m * C::Q_BYTES;
#pragma unroll
        for (int kb = 0; kb < C::KB; ++kb)
#pragma unroll
          for (int ch = 0; ch < 8; ++ch) {
            const uint4 v = row_ok ? __ldg(src + kb * 8 + ch) : make_uint4(0, 0, 0, 0);
            *reinterpret_cast<uint4*>(dQ + kb * (VM * 128) + tid * 128 + ((ch ^ (tid & 7)) << 4)) = v;
          }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(qfull);
      float mr[VROWS], lr[VROWS];
#pragma unroll
      for (int m = 0; m < VROWS; ++m) mr[m] = -INFINITY, lr[m] = 0.f;
      const uint32_t v0 = vg;
      for (int jj = 0; jj < nt && ok; ++jj) {
        const int j = q.j0 + jj;
        for (int m = 0; m < mt && ok; ++m) {
          const uint32_t vc = vg++;
          const int qi = (m * VM + tid) / p.G;
          if (!vwait(&sfull[vc & 1], (vc >> 1) & 1, p.dev_status, s_abort)) {
            ok = false;
            break;
          }
          tc05::fence_after();
          float x[VBN];
          {
            uint32_t r0[32], r1[32];
            const uint32_t t_s = tmem + lane_off + (vc & 1) * C::SCOL;
            tc05::ld32(t_s, r0);
            tc05::ld32(t_s + 32, r1);
            tc05::wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) {
              x[e] = __uint_as_float(r0[e]);
              x[32 + e] = __uint_as_float(r1[e]);
            }
          }
          {
            const int last = j < R.n_full ? R.ctx - j * VBN - 1 : qi - (j - R.n_full) * VBN;  // last visible key
            if (last < VBN - 1) {
#pragma unroll
              for (int e = 0; e < VBN; ++e)
                if (e > last) x[e] = -INFINITY;
            }
          }
          const float mx = row_max(x) * p.scale_log2;
          float m_run = m == 0 ? mr[0] : (m == 1 ? mr[1] : mr[2]);
          float l_run = m == 0 ? lr[0] : (m == 1 ? lr[1] : lr[2]);
          const float m_new = fmaxf(m_run, mx);
          const bool need = jj > 0 && m_new > m_run + 8.f;
          if (vc > v0) {
            // P V of the previous step: the P buffer is free and this row tile's O is stable
            if (!vwait(ofull, (vc - 1) & 1, p.dev_status, s_abort)) {
              ok = false;
              break;
            }
            tc05::fence_after();
          }
          if (jj == 0) {
            m_run = m_new;
          } else {
            float f = 1.f;
            if (need) {
              f = ex2_approx(m_run - m_new);
              l_run *= f;
              m_run = m_new;
            }
            if (__any_sync(0xffffffffu, need)) {
#pragma unroll 1
              for (int cb = 0; cb < D / 32; ++cb) {
                uint32_t r[32];
                const uint32_t t_o = tmem + lane_off + C::OCOL + m * D + cb * 32;
                tc05::ld32(t_o, r);
                tc05::wait_ld();
#pragma unroll
                for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * f);
                tc05::st32(t_o, r);
              }
              tc05::wait_st();
            }
          }
          const float mu = (m_run == -INFINITY) ? 0.f : m_run;
          l_run += row_exp_to_p(x, p.scale_log2, mu, sP + tid * 128, tid);
          if (m == 0) {
            mr[0] = m_run, lr[0] = l_run;
          } else if (m == 1) {
            mr[1] = m_run, lr[1] = l_run;
          } else {
            mr[2] = m_run, lr[2] = l_run;
          }
          fence_proxy_async_smem();
          tc05::fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(pfull);
        }
      }
      if (!ok) break;
      // outputs: wait for the unit's last P V, then each row tile's O
      if (!vwait(ofull, (vg - 1) & 1, p.dev_status, s_abort)) {
        ok = false;
        break;
      }
      tc05::fence_after();
      g += nt;
      const bool whole = (q.j0 == 0 && q.j1 == R.tiles);
#pragma unroll 1
      for (int m = 0; m < mt; ++m) {
        const int Rw = m * VM + tid, qi = Rw / p.G, qg = Rw % p.G;
        const bool row_ok = qi < R.n_rows;
        const float l_run = m == 0 ? lr[0] : (m == 1 ? lr[1] : lr[2]);
        const float m_run = m == 0 ? mr[0] : (m == 1 ? mr[1] : mr[2]);
        const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
        const size_t slot = (size_t)(c + ug_global) * VROWS + m;
#pragma unroll 1
        for (int cb = 0; cb < D / 32; ++cb) {
          uint32_t r[32];
          tc05::ld32(tmem + lane_off + C::OCOL + m * D + cb * 32, r);  // warp-collective: every lane loads
          tc05::wait_ld();
          if (!row_ok) continue;
          if (whole) {
            uint4* dst = reinterpret_cast<uint4*>(R.o + ((size_t)qi * p.Hq + hk * p.G + qg) * D + cb * 32);
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              uint32_t w[4];
#pragma unroll
              for (int e = 0; e < 4; ++e)
                w[e] = pack_bf16x2(__uint_as_float(r[8 * v + 2 * e]) * inv, __uint_as_float(r[8 * v + 2 * e + 1]) * inv);
              dst[v] = make_uint4(w[0], w[1], w[2], w[3]);
            }
          } else {
            float4* dst = reinterpret_cast<float4*>(p.ws_o + (slot * VM + tid) * D + cb * 32);
#pragma unroll
            for (int v = 0; v < 8; ++v)
              dst[v] = make_float4(__uint_as_float(r[4 * v]) * inv, __uint_as_float(r[4 * v + 1]) * inv,
                                   __uint_as_float(r[4 * v + 2]) * inv, __uint_as_float(r[4 * v + 3]) * inv);
          }
        }
        if (row_ok && !whole) p.ws_lse[slot * VM + tid] = l_run > 0.f ? m_run + log2f(l_run) : -INFINITY;
      }
      tc05::fence_before();
      pos += nt;
    }
    for (int64_t pos = beg; pos < end && ok && !KV_HEAD_UNITS;) {
      const VPiece q = verify_piece(p, pos, end);
      const VerifyReqDev& R = p.req[q.b];
      const int nt = q.j1 - q.j0;
      const int hk = p.h0 + q.ul / R.mtiles, mt = q.ul % R.mtiles;
      const int u_global = R.unit_begin + q.ul;
      const int Rw = mt * VM + tid;
      const int qi = Rw / p.G, qg = Rw % p.G;
      const bool row_ok = qi < R.n_rows;
      // this thread's query row into the swizzled Q tile; the previous unit's MMAs are complete
      // (its epilogue waited for the last P V, which follows every S of the unit)
      {
        const uint4* src = reinterpret_cast<const uint4*>(R.q + ((size_t)qi * p.Hq + hk * p.G + qg) * D);
#pragma unroll
        for (int kb = 0; kb < C::KB; ++kb)
#pragma unroll
          for (int ch = 0; ch < 8; ++ch) {
            const uint4 v = row_ok ? __ldg(src + kb * 8 + ch) : make_uint4(0, 0, 0, 0);
            *reinterpret_cast<uint4*>(sQ + kb * (VM * 128) + tid * 128 + ((ch ^ (tid & 7)) << 4)) = v;
          }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(qfull);

      if constexpr (MODE == VMODE_ATTN) {
      float m_run = -INFINITY, l_run = 0.f;
      for (int jj = 0; jj < nt; ++jj) {
        const int j = q.j0 + jj;
        const uint32_t gc = g + jj;
        if (!vwait(&sfull[gc & 1], (gc >> 1) & 1, p.dev_status, s_abort)) {
          ok = false;
          break;
        }
        tc05::fence_after();
        float x[VBN];
        {
          uint32_t r0[32], r1[32];
          const uint32_t t_s = tmem + lane_off + (gc & 1) * C::SCOL;
          tc05::ld32(t_s, r0);
          tc05::ld32(t_s + 32, r1);
          tc05::wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            x[e] = __uint_as_float(r0[e]);
            x[32 + e] = __uint_as_float(r1[e]);
          }
        }
        // mask invisible keys (only a ragged last KV_full tile or a drafted-rows tile has any),
        // then the row max by a tree; the scale is folded into the exponent below
        {
          const int last = j < R.n_full ? R.ctx - j * VBN - 1 : qi - (j - R.n_full) * VBN;  // last visible key
          if (last < VBN - 1) {
#pragma unroll
            for (int e = 0; e < VBN; ++e)
              if (e > last) x[e] = -INFINITY;
          }
        }
        const float mx = row_max(x) * p.scale_log2;  // the scale is positive: it keeps the order
        const float m_new = fmaxf(m_run, mx);
        // rescale O only when the running max grew by more than 2^8; TMEM loads/stores are
        // warp-collective, so the warp rescales together (factor 1 for rows that need none)
        const bool need = jj > 0 && m_new > m_run + 8.f;
        if (jj > 0) {
          // P V of the previous tile: O is stable and the P buffer is free after it
          if (!vwait(ofull, (gc - 1) & 1, p.dev_status, s_abort)) {
            ok = false;
            break;
          }
          tc05::fence_after();
        }
        if (jj == 0) {
          m_run = m_new;
        } else {
          float f = 1.f;
          if (need) {
            f = ex2_approx(m_run - m_new);
            l_run *= f;
            m_run = m_new;
          }
          if (__any_sync(0xffffffffu, need)) {
#pragma unroll 1
            for (int cb = 0; cb < D / 32; ++cb) {
              uint32_t r[32];
              const uint32_t t_o = tmem + lane_off + C::OCOL + cb * 32;
              tc05::ld32(t_o, r);
              tc05::wait_ld();
#pragma unroll
              for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * f);
              tc05::st32(t_o, r);
            }
            tc05::wait_st();
          }
        }
        const float mu = (m_run == -INFINITY) ? 0.f : m_run;
        l_run += row_exp_to_p(x, p.scale_log2, mu, sP + tid * 128, tid);
        fence_proxy_async_smem();
        tc05::fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(pfull);
      }
      if (!ok) break;
      // output: wait for the unit's last P V
      if (!vwait(ofull, (g + nt - 1) & 1, p.dev_status, s_abort)) {
        ok = false;
        break;
      }
      tc05::fence_after();
      g += nt;
      const bool whole = (q.j0 == 0 && q.j1 == R.tiles);
      const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
      const size_t slot = (size_t)(c + u_global);
#pragma unroll 1
      for (int cb = 0; cb < D / 32; ++cb) {
        uint32_t r[32];
        tc05::ld32(tmem + lane_off + C::OCOL + cb * 32, r);  // warp-collective: every lane loads
        tc05::wait_ld();
        if (!row_ok) continue;
        if (whole) {
          uint4* dst = reinterpret_cast<uint4*>(R.o + ((size_t)qi * p.Hq + hk * p.G + qg) * D + cb * 32);
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e)
              w[e] = pack_bf16x2(__uint_as_float(r[8 * v + 2 * e]) * inv, __uint_as_float(r[8 * v + 2 * e + 1]) * inv);
            dst[v] = make_uint4(w[0], w[1], w[2], w[3]);
          }
        } else {
          float4* dst = reinterpret_cast<float4*>(p.ws_o + (slot * VM + tid) * D + cb * 32);
#pragma unroll
          for (int v = 0; v < 8; ++v)
            dst[v] = make_float4(__uint_as_float(r[4 * v]) * inv, __uint_as_float(r[4 * v + 1]) * inv,
                                 __uint_as_float(r[4 * v + 2]) * inv, __uint_as_float(r[4 * v + 3]) * inv);
        }
      }
      if (row_ok && !whole) p.ws_lse[slot * VM + tid] = l_run > 0.f ? m_run + log2f(l_run) : -INFINITY;
      } else if constexpr (MODE == VMODE_STATS) {
        // the row's maximum and sum of 2^(s scale - max) over the piece's tiles, exactly tracked
        float m_run = -INFINITY, l_run = 0.f;
        for (int jj = 0; jj < nt; ++jj) {
          const int j = q.j0 + jj;
          const uint32_t gc = g + jj;
          if (!vwait(&sfull[gc & 1], (gc >> 1) & 1, p.dev_status, s_abort)) {
            ok = false;
            break;
          }
          tc05::fence_after();
          float x[VBN];
          {
            uint32_t r0[32], r1[32];
            const uint32_t t_s = tmem + lane_off + (gc & 1) * C::SCOL;
            tc05::ld32(t_s, r0);
            tc05::ld32(t_s + 32, r1);
            tc05::wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) {
              x[e] = __uint_as_float(r0[e]) * p.scale_log2;
              x[32 + e] = __uint_as_float(r1[e]) * p.scale_log2;
            }
          }
          tc05::fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&vfull[gc & 1]);  // this warp is done with the S buffer
          const int last = j < R.n_full ? R.ctx - j * VBN - 1 : qi - (j - R.n_full) * VBN;
          if (last < VBN - 1) {
#pragma unroll
            for (int e = 0; e < VBN; ++e)
              if (e > last) x[e] = -INFINITY;
          }
          // tree reductions: a linear chain of 64 dependent max (or add) steps per tile would leave
          // the two softmax warps per scheduler waiting on their own latency
          const float mx = row_max(x);
          const float m_new = fmaxf(m_run, mx);
          if (m_new != -INFINITY) {
            const uint64_t nm = f2_pack(-m_new, -m_new);
            uint64_t acc[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
            for (int e = 0; e < VBN / 2; ++e) {
              float a0, a1;
              f2_unpack(f2_add(f2_pack(x[2 * e], x[2 * e + 1]), nm), a0, a1);
              acc[e & 3] = f2_add(acc[e & 3], f2_pack(ex2_approx(a0), ex2_approx(a1)));
            }
            float s0, s1;
            f2_unpack(f2_add(f2_add(acc[0], acc[1]), f2_add(acc[2], acc[3])), s0, s1);
            const float sum = s0 + s1;
            l_run = l_run * ex2_approx(m_run - m_new) + sum;
            m_run = m_new;
          }
        }
        if (!ok) break;
        g += nt;
        const bool whole = (q.j0 == 0 && q.j1 == R.tiles);
        const float lse = l_run > 0.f ? m_run + log2f(l_run) : -INFINITY;
        if (row_ok) {
          if (whole)
            R.lse[((size_t)hk * R.mtiles + mt) * VM + tid] = lse;
          else
            p.ws_lse[(size_t)(c + u_global) * VM + tid] = lse;
        }
      } else if constexpr (MODE == VMODE_VOTES) {
        // votes: P = 2^(s scale - lse) (0 for padding rows and invisible keys) in fp16 for the
        // column-sum MMA, alternating between two P tiles. Every row of a tile's sums is the same;
        // warp w stores keys 16 w .. 16 w + 15 of them, two tiles after the tile's P (when the
        // next P into that buffer needs its sums done anyway), the unit's last two at its end
        const float lse = row_ok ? R.lse[((size_t)hk * R.mtiles + mt) * VM + tid] : 0.f;
        float* vdst = R.votes + ((size_t)hk * R.mtiles + mt) * (size_t)(R.ctx + R.n_rows);
        auto sums_done = [&](uint32_t gp) { return vwait(&ofv[gp & 1], (gp >> 1) & 1, p.dev_status, s_abort); };
        auto store_votes = [&](uint32_t gp, int jp) {
          uint32_t r0[8], r1[8];
          const uint32_t t_c = tmem + lane_off + C::OCOL + (gp & 1) * VBN + 16 * warp;
          tc05::ld8(t_c, r0);
          tc05::ld8(t_c + 8, r1);
          tc05::wait_ld();
          float v = 0.f;
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            if (e == lane) v = __uint_as_float(r0[e]);
            if (e + 8 == lane) v = __uint_as_float(r1[e]);
          }
          const int j = q.j0 + jp;
          const int key0 = j < R.n_full ? j * VBN : R.ctx + (j - R.n_full) * VBN;
          const int nv = j < R.n_full ? min(VBN, R.ctx - j * VBN) : min(VBN, R.n_rows - (j - R.n_full) * VBN);
          const int k = 16 * warp + lane;
          if (lane < 16 && k < nv) vdst[key0 + k] = v;
        };
        for (int jj = 0; jj < nt; ++jj) {
          const int j = q.j0 + jj;
          const uint32_t gc = g + jj;
          if (!vwait(&sfull[gc & 1], (gc >> 1) & 1, p.dev_status, s_abort)) {
            ok = false;
            break;
          }
          tc05::fence_after();
          float x[VBN];
          {
            uint32_t r0[32], r1[32];
            const uint32_t t_s = tmem + lane_off + (gc & 1) * C::SCOL;
            tc05::ld32(t_s, r0);
            tc05::ld32(t_s + 32, r1);
            tc05::wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) {
              x[e] = __uint_as_float(r0[e]);
              x[32 + e] = __uint_as_float(r1[e]);
            }
          }
          const int last = !row_ok ? -1 : j < R.n_full ? R.ctx - j * VBN - 1 : qi - (j - R.n_full) * VBN;
          if (gc >= 2) {
            // P tile gc & 1 and TMEM sums buffer gc & 1 were last used by tile gc - 2: its column
            // sums are done (a wait that is exact: tile gc - 4's were observed two tiles ago, and
            // tile gc's cannot start before this tile's P); a tile of this unit has its votes stored
            if (!sums_done(gc - 2)) {
              ok = false;
              break;
            }
            tc05::fence_after();
            if (jj >= 2) store_votes(gc - 2, jj - 2);
          }
          uint8_t* pb = (gc & 1) ? smem + C::OFF_P1_VOTES : sP;
          if (last >= VBN - 1) {
            // every key of the tile visible (all but a unit's last tiles): packed f32x2 FMAs, no masks
            const uint64_t sc2 = f2_pack(p.scale_log2, p.scale_log2), nl2 = f2_pack(-lse, -lse);
#pragma unroll
            for (int ch = 0; ch < 8; ++ch) {
              uint32_t w[4];
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const int k0 = ch * 8 + 2 * e;
                float a0, a1;
                f2_unpack(f2_fma(f2_pack(x[k0], x[k0 + 1]), sc2, nl2), a0, a1);
                const __half2 h = __floats2half2_rn(ex2_approx(a0), ex2_approx(a1));
                w[e] = *reinterpret_cast<const uint32_t*>(&h);
              }
              *reinterpret_cast<uint4*>(pb + tid * 128 + ((ch ^ (tid & 7)) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
            }
          } else {
#pragma unroll
            for (int ch = 0; ch < 8; ++ch) {
              uint32_t w[4];
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const int k0 = ch * 8 + 2 * e;
                const float p0 = k0 <= last ? ex2_approx(fmaf(x[k0], p.scale_log2, -lse)) : 0.f;
                const float p1 = k0 + 1 <= last ? ex2_approx(fmaf(x[k0 + 1], p.scale_log2, -lse)) : 0.f;
                const __half2 h = __floats2half2_rn(p0, p1);
                w[e] = *reinterpret_cast<const uint32_t*>(&h);
              }
              *reinterpret_cast<uint4*>(pb + tid * 128 + ((ch ^ (tid & 7)) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
            }
          }
          fence_proxy_async_smem();
          tc05::fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&pfv[gc & 1]);
        }
        if (!ok) break;
        // the unit's last two tiles: their sums, then their votes
        for (int jp = nt > 2 ? nt - 2 : 0; jp < nt && ok; ++jp) {
          if (!sums_done(g + jp)) {
            ok = false;
            break;
          }
          tc05::fence_after();
          store_votes(g + jp, jp);
        }
        if (!ok) break;
        g += nt;
      }
      tc05::fence_before();
      pos += nt;
    }
  }

  tc05::fence_before();
  __syncthreads();
  tc05::fence_after();
  if (warp == 0) tc05::dealloc(tmem, C::TCOLS);
}

// Merge the partials of units split across CTAs: o = sum_k 2^(lse_k - LSE) o_k / L.
// grid (units, 128 / 8): a CTA takes 8 query rows of a unit, a thread one row's 4 channels (d=128) or
// 2 channels (d=64), so partial reads are spread across threads.
template <int D>
__global__ void __launch_bounds__(256) verify_combine_kernel(const __grid_constant__ VerifyParams p) {
  constexpr int TPR = 32;          // threads per row
  constexpr int CPT = D / TPR;     // channels per thread (4 or 2)
  const int u = blockIdx.x;
  pdl_launch_dependents();
  pdl_wait();
  int b = 0;
#pragma unroll 1
  for (int i = 1; i < p.B; ++i)
    if (p.req[i].unit_begin <= u) b = i;
  const VerifyReqDev& R = p.req[b];
  const int ul = u - R.unit_begin;
  // the unit's tiles in the call's tile sequence: per (KV head, row tile), or in row-tile mode per
  // KV head (its row tiles share the tiles); a CTA c that held part of it left its partial in slot
  // c + unit (row-tile mode: (c + KV-head unit) * VROWS + row tile)
  const int hl = ul / R.mtiles, mt = ul % R.mtiles;
  const int64_t U0 = R.tile_begin + (int64_t)(p.rows ? hl : ul) * R.tiles, U1 = U0 + R.tiles;
  const int64_t T = p.total_tiles, N = p.n_cta;
  const int64_t c0 = ((U0 + 1) * N - 1) / T, c1 = (U1 * N - 1) / T;
  if (c0 == c1) return;
  const int r = blockIdx.y * 8 + (threadIdx.x / TPR), cc = (threadIdx.x % TPR) * CPT;
  const int hk = p.h0 + hl;
  const int Rw = mt * VM + r, qi = Rw / p.G, qg = Rw % p.G;
  if (qi >= R.n_rows) return;
  auto slot_of = [&](int64_t c) -> int64_t { return p.rows ? (c + R.ug_begin + hl) * VROWS + mt : c + u; };
  float M = -INFINITY;
  for (int64_t c = c0; c <= c1; ++c) M = fmaxf(M, p.ws_lse[slot_of(c) * VM + r]);
  const float Mu = M == -INFINITY ? 0.f : M;
  float L = 0.f, acc[CPT];
#pragma unroll
  for (int e = 0; e < CPT; ++e) acc[e] = 0.f;
#pragma unroll 4
  for (int64_t c = c0; c <= c1; ++c) {
    const int64_t sl = slot_of(c);
    const float w = exp2f(p.ws_lse[sl * VM + r] - Mu);
    const float* src = p.ws_o + (sl * VM + r) * D + cc;
    L += w;
    if (CPT == 4) {
      const float4 v = *reinterpret_cast<const float4*>(src);
      acc[0] += w * v.x;
      acc[1 % CPT] += w * v.y;
      acc[2 % CPT] += w * v.z;
      acc[3 % CPT] += w * v.w;
    } else {
      const float2 v = *reinterpret_cast<const float2*>(src);
      acc[0] += w * v.x;
      acc[1 % CPT] += w * v.y;
    }
  }
  const float inv = L > 0.f ? 1.f / L : 0.f;
  bf16* dst = R.o + ((size_t)qi * p.Hq + hk * p.G + qg) * D + cc;
  if (CPT == 4) {
    uint2 o;
    o.x = pack_bf16x2(acc[0] * inv, acc[1 % CPT] * inv);
    o.y = pack_bf16x2(acc[2 % CPT] * inv, acc[3 % CPT] * inv);
    *reinterpret_cast<uint2*>(dst) = o;
  } else {
    *reinterpret_cast<uint32_t*>(dst) = pack_bf16x2(acc[0] * inv, acc[1 % CPT] * inv);
  }
}

// ------------------------------------------------------------------------------------------------
static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(tmap_encoder());
}

// bf16 [Hkv][cap][d] rows 0..rows-1 as a 3-D tensor (d, rows, Hkv); box 64 x 64 x 1, 128-byte swizzle.
static bool make_map(CUtensorMap* m, const void* base, int d, int rows, int cap, int Hkv) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)rows, (cuuint64_t)Hkv};
  cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)cap * d * 2};
  cuuint32_t box[3] = {64, (cuuint32_t)VBN, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

static int sm_count_v() {
  static int n = 0;
  if (n == 0) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      n = 152;
  }
  return n;
}

static int64_t verify_ctas(int64_t T, int per_sm = 2) {
  const char* e = getenv("VC_VERIFY_CTAS");
  int64_t n = e ? atoll(e) : per_sm * (int64_t)sm_count_v();
  if (n < 1) n = 1;
  return n < T ? n : T;
}

size_t verify_workspace_size(const vc_shape* s, int32_t max_rows) {
  if (max_rows < 1) return 0;
  const int G = s->Hq / s->Hkv;
  const int64_t mtiles = ((int64_t)max_rows * G + VM - 1) / VM;
  const int64_t units = (int64_t)s->B * s->Hkv * mtiles;
  // CTAs of a launch: two per SM (one in row-tile mode), or VC_VERIFY_CTAS when set
  const char* ev = getenv("VC_VERIFY_CTAS");
  const int64_t ctas = ev && atoll(ev) > 2 * (int64_t)sm_count_v() ? atoll(ev) : 2 * (int64_t)sm_count_v();
  int64_t slots = units + ctas + 8;
  // row-tile mode: VROWS slots per (CTA + KV-head unit)
  const int64_t rslots = ((int64_t)s->B * s->Hkv + ctas + 8) * VROWS;
  if (rslots > slots) slots = rslots;
  return (size_t)slots * VM * (s->d + 1) * sizeof(float) + 256;
}

template <int D, int MODE>
static cudaError_t launch_modes_t(const VerifyParams& p, cudaStream_t s) {
  using C = VCfgOf<D, MODE>;
  constexpr int SMEM = MODE == VMODE_VOTES ? C::SMEM_VOTES : C::SMEM;
  static std::atomic<uint64_t> attr{0};
  {
    cudaError_t e = raise_smem_limit(verify_attn_kernel<D, MODE>, SMEM, attr);
    if (e != cudaSuccess) return e;
  }
  return launch_pdl(verify_attn_kernel<D, MODE>, dim3(p.n_cta), dim3(C::THREADS), SMEM, s, p);
}

template <int D>
static cudaError_t launch_verify_t(const VerifyParams& p, cudaStream_t s) {
  cudaError_t e = p.rows == 3   ? launch_modes_t<D, VMODE_TRIO>(p, s)
                  : p.rows == 2 ? launch_modes_t<D, VMODE_PAIR>(p, s)
                  : p.rows == 1 ? launch_modes_t<D, VMODE_ROWS>(p, s)
                                : launch_modes_t<D, VMODE_ATTN>(p, s);
  if (e != cudaSuccess) return e;
  return launch_pdl(verify_combine_kernel<D>, dim3(p.n_units, VM / 8), dim3(256), 0, s, p);
}

// Row log-sum-exp of units split across CTAs (statistics mode): LSE = log2 sum_k 2^lse_k over the
// unit's CTA slots; grid (units), a thread per row. Whole units were written by the kernel.
__global__ void __launch_bounds__(VM) stats_combine_kernel(const __grid_constant__ VerifyParams p) {
  const int u = blockIdx.x, r = threadIdx.x;
  pdl_launch_dependents();
  pdl_wait();
  int b = 0;
#pragma unroll 1
  for (int i = 1; i < p.B; ++i)
    if (p.req[i].unit_begin <= u) b = i;
  const VerifyReqDev& R = p.req[b];
  const int ul = u - R.unit_begin;
  const int64_t U0 = R.tile_begin + (int64_t)ul * R.tiles, U1 = U0 + R.tiles;
  const int64_t T = p.total_tiles, N = p.n_cta;
  const int64_t c0 = ((U0 + 1) * N - 1) / T, c1 = (U1 * N - 1) / T;
  if (c0 == c1) return;
  const int hk = p.h0 + ul / R.mtiles, mt = ul % R.mtiles;
  if (mt * VM + r >= R.n_rows * p.G) return;
  float M = -INFINITY;
  for (int64_t c = c0; c <= c1; ++c) M = fmaxf(M, p.ws_lse[(c + u) * VM + r]);
  float L = 0.f;
  if (M != -INFINITY)
    for (int64_t c = c0; c <= c1; ++c) L += exp2f(p.ws_lse[(c + u) * VM + r] - M);
  R.lse[((size_t)hk * R.mtiles + mt) * VM + r] = L > 0.f ? M + log2f(L) : -INFINITY;
}

static bool a16(const void* p) { return p && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int obs_mtiles(int W, int G) { return (W * G + VM - 1) / VM; }

size_t obs_slot_floats(int B, int Hkv, int mtiles) {
  return ((size_t)B * Hkv * mtiles + 2 * (size_t)sm_count_v() + 8) * VM;
}

// The observation window's two passes on the tensor cores: for request b, the W window queries
// q_obs attend to keys 0 .. ctx-W-1 of KV_full (the "full" part) and, causally, to the window's own
// W keys (the "new" part: KV_full rows ctx-W .. ctx-1, row stride cap); the statistics pass writes
// each window row's log-sum-exp, the votes pass each 128-row tile's column sums per key.
cudaError_t launch_obs_passes(const ObsArgs& a, cudaStream_t s) {
  const int d = a.d, G = a.Hq / a.Hkv;
  VerifyParams p;
  memset(&p, 0, sizeof(p));
  p.B = a.B;
  p.Hq = a.Hq;
  p.Hkv = a.Hkv;
  p.G = G;
  p.h0 = 0;
  p.scale_log2 = (float)(1.4426950408889634 / sqrt((double)d));
  p.dev_status = a.dev_status;
  int64_t tiles = 0;
  int32_t units = 0;
  const int mtiles = obs_mtiles(a.W, G);
  for (int b = 0; b < a.B; ++b) {
    const ObsReq& q = a.req[b];
    const int full = q.ctx - a.W;
    const bf16* knew = q.k + (size_t)full * d;
    if (!make_map(&p.tm[b][0], q.k, d, full > 0 ? full : 1, q.cap, a.Hkv) ||
        !make_map(&p.tm[b][2], knew, d, a.W, q.cap, a.Hkv))
      return cudaErrorInvalidValue;
    p.tm[b][1] = p.tm[b][0];
    p.tm[b][3] = p.tm[b][2];
    VerifyReqDev& R = p.req[b];
    R.q = q.q;
    R.o = nullptr;
    R.ctx = full;
    R.n_rows = a.W;
    R.mtiles = mtiles;
    R.n_full = (full + VBN - 1) / VBN;
    R.tiles = R.n_full + (a.W + VBN - 1) / VBN;
    R.unit_begin = units;
    R.tile_begin = tiles;
    R.lse = q.lse;
    R.votes = q.votes;
    units += a.Hkv * mtiles;
    tiles += (int64_t)a.Hkv * mtiles * R.tiles;
  }
  p.total_tiles = tiles;
  p.n_cta = (int32_t)verify_ctas(tiles);
  p.n_units = units;
  if (((size_t)p.n_cta + units) * VM > a.ws_lse_floats) return cudaErrorInvalidValue;
  p.ws_o = nullptr;
  p.ws_lse = a.ws_lse;
  cudaError_t e = d == 128 ? launch_modes_t<128, VMODE_STATS>(p, s) : launch_modes_t<64, VMODE_STATS>(p, s);
  if (e != cudaSuccess) return e;
  e = launch_pdl(stats_combine_kernel, dim3(p.n_units), dim3(VM), 0, s, p);
  if (e != cudaSuccess) return e;
  return d == 128 ? launch_modes_t<128, VMODE_VOTES>(p, s) : launch_modes_t<64, VMODE_VOTES>(p, s);
}

// One launch (verification kernel, then the combine of split units) over the requests sel[0..n):
// rows 0 = one unit per (request, KV head, row tile); 1 = row-tile mode (every row tile of a head in
// one CTA, one softmax warpgroup); 2 = pair mode (both row tiles of a two-tile head in one CTA, a
// softmax warpgroup each); 3 = trio mode (the three row tiles of a three-tile head in one CTA, two
// softmax warpgroups).
static cudaError_t verify_launch(const vc_shape* shape, const vc_verify_req* req, const int* sel, int n, int rows,
                                 int h0, int h1, void* ws, size_t ws_bytes, int32_t* dev_status, cudaStream_t stream,
                                 vc_status* st) {
  const int d = shape->d, G = shape->Hq / shape->Hkv;
  VerifyParams p;  // about 18 KB: the tensor maps travel as kernel parameters
  memset(&p, 0, sizeof(p));
  p.B = n;
  p.Hq = shape->Hq;
  p.Hkv = shape->Hkv;
  p.G = G;
  p.h0 = h0;
  const int nh = h1 - h0;
  p.scale_log2 = (float)(1.4426950408889634 / sqrt((double)d));
  p.dev_status = dev_status;
  p.rows = rows;
  int64_t tiles = 0;
  int32_t units = 0, ugs = 0, max_rows = 0;
  for (int b = 0; b < n; ++b) {
    const vc_verify_req& r = req[sel[b]];
    const vc_kv_full& f = r.full;
    if (!a16(f.k) || !a16(f.v) || !a16(r.q) || !a16(r.o) || !a16(r.k_new) || !a16(r.v_new) || f.ctx < 1 ||
        f.cap < f.ctx || r.n_rows < 1 || r.new_cap < r.n_rows) {
      *st = VC_ERR_INVALID;
      return cudaSuccess;
    }
    if (!make_map(&p.tm[b][0], f.k, d, f.ctx, f.cap, shape->Hkv) ||
        !make_map(&p.tm[b][1], f.v, d, f.ctx, f.cap, shape->Hkv) ||
        !make_map(&p.tm[b][2], r.k_new, d, r.n_rows, r.new_cap, shape->Hkv) ||
        !make_map(&p.tm[b][3], r.v_new, d, r.n_rows, r.new_cap, shape->Hkv)) {
      *st = VC_ERR_CUDA;
      return cudaSuccess;
    }
    VerifyReqDev& R = p.req[b];
    R.q = static_cast<const bf16*>(r.q);
    R.o = static_cast<bf16*>(r.o);
    R.ctx = f.ctx;
    R.n_rows = r.n_rows;
    R.mtiles = (r.n_rows * G + VM - 1) / VM;
    R.n_full = (f.ctx + VBN - 1) / VBN;
    R.tiles = R.n_full + (r.n_rows + VBN - 1) / VBN;
    R.unit_begin = units;
    R.ug_begin = ugs;
    R.tile_begin = tiles;
    units += nh * R.mtiles;
    ugs += nh;
    tiles += (int64_t)nh * (p.rows ? 1 : R.mtiles) * R.tiles;
    if (r.n_rows > max_rows) max_rows = r.n_rows;
  }
  p.total_tiles = tiles;
  p.n_cta = (int32_t)verify_ctas(tiles, p.rows ? 1 : 2);
  p.n_units = units;
  const size_t slots = p.rows ? ((size_t)p.n_cta + ugs) * VROWS : (size_t)p.n_cta + units;
  const size_t need = slots * VM * (d + 1) * sizeof(float);
  if (!ws || ws_bytes < need || !a16(ws)) {
    *st = VC_ERR_WORKSPACE;
    return cudaSuccess;
  }
  p.ws_o = static_cast<float*>(ws);
  p.ws_lse = p.ws_o + slots * VM * d;
  return d == 128 ? launch_verify_t<128>(p, stream) : launch_verify_t<64>(p, stream);
}

// How the requests of a call are verified, by their KV heads' 128-row tiles (L x G rows):
//   one tile: one unit per (request, KV head) at two CTAs per SM;
//   exactly two: pair mode (VC_VERIFY_PAIR=0 turns it off): each K/V tile read once for both
//     tiles, with a softmax warpgroup per tile;
//   three or more: one unit per row tile (each reads KV_full again); with VC_VERIFY_TRIO=1 a head
//     of exactly three goes to trio mode (read once, two softmax warpgroups; slower at present:
//     its first warpgroup holds two of the three tiles);
//   with VC_VERIFY_ROWS=1, every request of the call in row-tile mode when none has more than
//     VROWS tiles (read once; one softmax warpgroup per CTA, so slower).
// Requests of different kinds go to separate launches (each a kernel and its merge), one after the
// other on the stream, in the order of sel[] below; every request is checked first.
struct VerifyPlan {
  int sel[3][VC_MAX_BATCH];  // requests of the one-unit-per-tile, pair-mode and trio-mode launches
  int n[3];
  bool rows_all;             // one row-tile-mode launch over every request (listed in sel[0])
};

static vc_status plan_verify(const vc_shape* shape, const vc_verify_req* req, VerifyPlan* pl) {
  if (!shape || shape->B < 1 || shape->B > VC_MAX_BATCH || shape->Hkv < 1 || shape->Hq < shape->Hkv ||
      shape->Hq % shape->Hkv != 0 || !req)
    return VC_ERR_INVALID;
  if (shape->d != 64 && shape->d != 128) return VC_ERR_UNSUPPORTED;
  const int G = shape->Hq / shape->Hkv;
  int max_mt = 1;
  for (int b = 0; b < shape->B; ++b) {
    const vc_verify_req& r = req[b];
    const vc_kv_full& f = r.full;
    if (!a16(f.k) || !a16(f.v) || !a16(r.q) || !a16(r.o) || !a16(r.k_new) || !a16(r.v_new) || f.ctx < 1 ||
        f.cap < f.ctx || r.n_rows < 1 || r.new_cap < r.n_rows)
      return VC_ERR_INVALID;
    const int mtb = (r.n_rows * G + VM - 1) / VM;
    if (mtb > max_mt) max_mt = mtb;
  }
  pl->n[0] = pl->n[1] = pl->n[2] = 0;
  const char* er = getenv("VC_VERIFY_ROWS");
  pl->rows_all = max_mt >= 2 && max_mt <= VROWS && er && atoi(er) == 1;
  const char* ep = getenv("VC_VERIFY_PAIR");
  const char* et = getenv("VC_VERIFY_TRIO");
  const bool pair = !(ep && atoi(ep) == 0), trio = et && atoi(et) == 1;
  for (int b = 0; b < shape->B; ++b) {
    const int mtb = (req[b].n_rows * G + VM - 1) / VM;
    const int k = pl->rows_all ? 0 : (pair && mtb == 2) ? 1 : (trio && mtb == 3) ? 2 : 0;
    pl->sel[k][pl->n[k]++] = b;
  }
  return VC_OK;
}

cudaError_t launch_verify(const vc_shape* shape, const vc_verify_req* req, int h0, int h1, void* ws,
                          size_t ws_bytes, int32_t* dev_status, cudaStream_t stream, vc_status* st) {
  *st = VC_OK;
  if (!shape || h0 < 0 || h1 <= h0 || h1 > shape->Hkv) {
    *st = VC_ERR_INVALID;
    return cudaSuccess;
  }
  VerifyPlan pl;
  *st = plan_verify(shape, req, &pl);
  if (*st != VC_OK) return cudaSuccess;
  if (pl.rows_all) return verify_launch(shape, req, pl.sel[0], pl.n[0], 1, h0, h1, ws, ws_bytes, dev_status, stream, st);
  constexpr int kRows[3] = {0, 2, 3};  // verify_launch's layout of each list
  for (int k = 0; k < 3; ++k) {
    if (pl.n[k] == 0) continue;
    const cudaError_t e = verify_launch(shape, req, pl.sel[k], pl.n[k], kRows[k], h0, h1, ws, ws_bytes, dev_status,
                                        stream, st);
    if (e != cudaSuccess || *st != VC_OK) return e;
  }
  return cudaSuccess;
}

int32_t verify_launch_count(const vc_shape* shape, const vc_verify_req* req) {
  VerifyPlan pl;
  if (plan_verify(shape, req, &pl) != VC_OK) return -1;
  if (pl.rows_all) return 2;
  return 2 * ((pl.n[0] > 0) + (pl.n[1] > 0) + (pl.n[2] > 0));
}

}  // namespace vc
