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
// Per CTA (128 threads; thread r owns TMEM lane r = query row r):
//   thread 0 issues TMA loads of K/V tiles (64 tokens, 128-byte swizzle, 2 stages) and the MMAs;
//   S lands in TMEM columns [0,64), O accumulates in TMEM columns [OCOL, OCOL+d).
//   Every thread loads its S row (tcgen05.ld), applies scale, mask and online softmax in fp32
//   (exp2 domain; O is rescaled in TMEM only when the running max grows by more than 8), writes
//   its P row (bf16) into shared memory in the swizzled K-major layout, and the next MMA reads it.
#include "tc05.cuh"

#include <cuda.h>
#include <cudaTypedefs.h>
#include <math.h>
#include <stdlib.h>
#include <string.h>

namespace vc {

constexpr int VM = 128;  // query rows per tile
constexpr int VBN = 64;  // KV tokens per tile

struct VerifyReqDev {
  const bf16* q;
  bf16* o;
  int32_t ctx, n_rows, mtiles, n_full, tiles;
  int32_t unit_begin;
  int64_t tile_begin;
};

struct VerifyParams {
  CUtensorMap tm[VC_MAX_BATCH][4];  // K full, V full, K new, V new
  VerifyReqDev req[VC_MAX_BATCH];
  int32_t B, Hq, Hkv, G, n_cta, n_units;
  int64_t total_tiles;
  float scale_log2;
  float* ws_o;    // [slots][128][d]
  float* ws_lse;  // [slots][128]
  int32_t* dev_status;
};

template <int D>
struct VCfg {
  static constexpr int KB = D / 64;              // 64-channel (128-byte) blocks
  static constexpr int Q_BYTES = KB * VM * 128;  // Q tile, K-major SW128
  static constexpr int P_BYTES = VM * 128;       // P tile (64 tokens), K-major SW128
  static constexpr int KV_BYTES = KB * VBN * 128;  // one K (or V) tile
  static constexpr int STAGE = 2 * KV_BYTES;
  static constexpr int OFF_P = Q_BYTES;
  static constexpr int OFF_ST = OFF_P + P_BYTES;
  static constexpr int OFF_BAR = OFF_ST + 2 * STAGE;
  static constexpr int SMEM = OFF_BAR + 64;
  static constexpr int OCOL = D == 128 ? 128 : 64;
  static constexpr uint32_t TCOLS = D == 128 ? 256 : 128;
};

__device__ __forceinline__ int find_req(const VerifyParams& p, int64_t tile) {
  int b = 0;
#pragma unroll 1
  for (int i = 1; i < p.B; ++i)
    if (p.req[i].tile_begin <= tile) b = i;
  return b;
}

template <int D>
__global__ void __launch_bounds__(128, 2) verify_attn_kernel(const __grid_constant__ VerifyParams p) {
  using C = VCfg<D>;
  extern __shared__ __align__(1024) uint8_t smem[];
  const int tid = threadIdx.x, warp = tid >> 5;
  if (smem_u32(smem) & 1023u) {  // the swizzled layouts need 1024-byte aligned tiles
    pdl_launch_dependents();
    pdl_wait();
    if (tid == 0) set_status(p.dev_status, VC_DEV_INTERNAL);
    return;
  }
  uint8_t* sQ = smem;
  uint8_t* sP = smem + C::OFF_P;
  uint8_t* sST = smem + C::OFF_ST;
  uint64_t* kfull = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);  // [2] K tile landed
  uint64_t* vfull = kfull + 2;                                          // [2] V tile landed
  uint64_t* sbar = kfull + 4;                                           // S = Q K^T done
  uint64_t* obar = kfull + 5;                                           // O += P V done
  uint64_t* xbar = kfull + 6;                                           // drain on the error path
  uint32_t* tslot = reinterpret_cast<uint32_t*>(kfull + 7);
  volatile int& s_abort = *reinterpret_cast<volatile int*>(reinterpret_cast<uint8_t*>(kfull + 7) + 4);

  if (warp == 0) tc05::alloc(tslot, C::TCOLS);
  if (tid == 0) {
    for (int i = 0; i < 4; ++i) mbar_init(&kfull[i], 1);  // kfull[0..1], vfull[0..1]
    mbar_init(sbar, 1);
    mbar_init(obar, 1);
    mbar_init(xbar, 1);
    fence_mbar_init();
    s_abort = 0;
  }
  tc05::fence_before();
  __syncthreads();
  tc05::fence_after();
  pdl_launch_dependents();
  pdl_wait();
  const uint32_t tmem = *tslot;
  const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
  const uint32_t t_s = tmem + lane_off;
  const uint32_t t_o = tmem + lane_off + C::OCOL;

  constexpr uint32_t IDESC_S = tc05::idesc_bf16(VM, VBN, false);
  constexpr uint32_t IDESC_O = tc05::idesc_bf16(VM, D, true);
  const uint32_t aQ = smem_u32(sQ), aP = smem_u32(sP), aST = smem_u32(sST);

  const int64_t T = p.total_tiles, N = p.n_cta, c = blockIdx.x;
  int64_t pos = c * T / N;
  const int64_t end = (c + 1) * T / N;
  uint32_t g_tile = 0;  // global tile counter (stage = g & 1, phase = (g >> 1) & 1)
  uint32_t gk_issued = 0, gv_issued = 0;  // K / V tiles whose loads thread 0 has issued (error drain)
  uint32_t s_cnt = 0, o_cnt = 0;
  bool failed = false;

#pragma unroll 1
  while (pos < end && !failed) {
    const int b = find_req(p, pos);
    const VerifyReqDev& R = p.req[b];
    const int64_t rel = pos - R.tile_begin;
    const int ul = (int)(rel / R.tiles);
    const int j0 = (int)(rel % R.tiles);
    const int64_t left = end - pos;
    const int j1 = left < (int64_t)(R.tiles - j0) ? j0 + (int)left : R.tiles;
    const int nt = j1 - j0;
    const int hk = ul / R.mtiles, mt = ul % R.mtiles;
    const int u_global = R.unit_begin + ul;
    const CUtensorMap* tm = p.tm[b];

    // this thread's query row
    const int Rw = mt * VM + tid;
    const int qi = Rw / p.G, qg = Rw % p.G;
    const bool row_ok = qi < R.n_rows;
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
    tc05::fence_before();
    __syncthreads();

    // K and V of a tile have their own barriers: a K stage is reloaded as soon as the S MMA that
    // read it is done (start of the next-but-one iteration's wait), a V stage once its P V is done,
    // so each load has about two tile periods to land.
    auto issue_kv = [&](int j, uint32_t g, bool isv) {
      const int st = g & 1;
      uint8_t* dst = sST + st * C::STAGE + (isv ? C::KV_BYTES : 0);
      uint64_t* bar = isv ? &vfull[st] : &kfull[st];
      mbar_arrive_expect_tx(bar, C::KV_BYTES);
      (isv ? gv_issued : gk_issued) = g + 1;
      const bool isnew = j >= R.n_full;
      const int tok = isnew ? (j - R.n_full) * VBN : j * VBN;
      const void* map = &tm[(isnew ? 2 : 0) + (isv ? 1 : 0)];
#pragma unroll
      for (int kb = 0; kb < C::KB; ++kb) tc05::tma_load_3d(dst + kb * (VBN * 128), map, kb * 64, tok, hk, bar);
    };
    auto issue_s = [&](uint32_t g) -> bool {
      const int st = g & 1;
      if (!mbar_wait_bounded(&kfull[st], (g >> 1) & 1, p.dev_status)) return false;
      tc05::fence_after();
      const uint32_t kaddr = aST + st * C::STAGE;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint64_t da = tc05::sdesc_sw128(aQ + (kk >> 2) * (VM * 128) + (kk & 3) * 32, 16, 1024);
        const uint64_t db = tc05::sdesc_sw128(kaddr + (kk >> 2) * (VBN * 128) + (kk & 3) * 32, 16, 1024);
        tc05::mma_bf16(tmem, da, db, IDESC_S, kk > 0);
      }
      tc05::commit(sbar);
      return true;
    };

    if (tid == 0) {
      tc05::fence_after();
      issue_kv(j0, g_tile, false);
      issue_kv(j0, g_tile, true);
      if (nt > 1) {
        issue_kv(j0 + 1, g_tile + 1, false);
        issue_kv(j0 + 1, g_tile + 1, true);
      }
      if (!issue_s(g_tile)) s_abort = 1;
    }

    float m_run = -INFINITY, l_run = 0.f;
#pragma unroll 1
    for (int jj = 0; jj < nt; ++jj) {
      const int j = j0 + jj;
      const uint32_t g = g_tile + jj;
      bool ok = mbar_wait_bounded(sbar, s_cnt & 1, p.dev_status);
      s_cnt++;
      tc05::fence_after();
      if (tid == 0 && ok && jj + 2 < nt) issue_kv(j + 2, g + 2, false);  // S_g has read K stage g & 1
      float x[VBN];
      {
        uint32_t r0[32], r1[32];
        tc05::ld32(t_s, r0);
        tc05::ld32(t_s + 32, r1);
        tc05::wait_ld();
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          x[e] = __uint_as_float(r0[e]);
          x[32 + e] = __uint_as_float(r1[e]);
        }
      }
      // mask invisible keys (only a ragged last KV_full tile or a drafted-rows tile has any), then
      // the row max by a tree; the scale is folded into the exponent below
      {
        const int last = j < R.n_full ? R.ctx - j * VBN - 1 : qi - (j - R.n_full) * VBN;  // last visible key
        if (last < VBN - 1) {
#pragma unroll
          for (int e = 0; e < VBN; ++e)
            if (e > last) x[e] = -INFINITY;
        }
      }
      float mx;
      {
        float t[VBN / 2];
#pragma unroll
        for (int e = 0; e < VBN / 2; ++e) t[e] = fmaxf(x[2 * e], x[2 * e + 1]);
#pragma unroll
        for (int w = VBN / 4; w >= 1; w >>= 1)
#pragma unroll
          for (int e = 0; e < w; ++e) t[e] = fmaxf(t[e], t[e + w]);
        mx = t[0] * p.scale_log2;  // the scale is positive: it keeps the order
      }
      if (jj > 0) {
        ok = mbar_wait_bounded(obar, o_cnt & 1, p.dev_status) && ok;  // P V of the previous tile done
        o_cnt++;
        tc05::fence_after();
        if (tid == 0 && ok && jj + 1 < nt) issue_kv(j + 1, g + 1, true);  // it has read V stage (g - 1) & 1
      }
      const float m_new = fmaxf(m_run, mx);
      if (jj == 0) {
        m_run = m_new;
      } else {
        // rescale O only when the running max grew by more than 2^8; TMEM loads/stores are
        // warp-collective, so the warp rescales together (factor 1 for rows that need none)
        const bool need = m_new > m_run + 8.f;
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
            tc05::ld32(t_o + cb * 32, r);
            tc05::wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * f);
            tc05::st32(t_o + cb * 32, r);
          }
          tc05::wait_st();
        }
      }
      const float mu = (m_run == -INFINITY) ? 0.f : m_run;
      float ls[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int ch = 0; ch < 8; ++ch) {
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float p0 = ex2_approx(fmaf(x[ch * 8 + 2 * e], p.scale_log2, -mu));
          const float p1 = ex2_approx(fmaf(x[ch * 8 + 2 * e + 1], p.scale_log2, -mu));
          ls[e] += p0 + p1;
          w[e] = pack_bf16x2(p0, p1);
        }
        *reinterpret_cast<uint4*>(sP + tid * 128 + ((ch ^ (tid & 7)) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
      }
      l_run += (ls[0] + ls[1]) + (ls[2] + ls[3]);
      if (!ok) s_abort = 1;
      fence_proxy_async_smem();
      tc05::fence_before();
      __syncthreads();
      if (s_abort) {
        failed = true;
        break;
      }
      if (tid == 0) {
        tc05::fence_after();
        if (!mbar_wait_bounded(&vfull[g & 1], (g >> 1) & 1, p.dev_status)) {
          s_abort = 1;
        } else {
          const uint32_t vaddr = aST + (g & 1) * C::STAGE + C::KV_BYTES;
#pragma unroll
          for (int kk = 0; kk < VBN / 16; ++kk) {
            const uint64_t da = tc05::sdesc_sw128(aP + kk * 32, 16, 1024);
            const uint64_t db = tc05::sdesc_sw128(vaddr + kk * 2048, VBN * 128, 1024);
            tc05::mma_bf16(tmem + C::OCOL, da, db, IDESC_O, (jj > 0 || kk > 0) ? 1u : 0u);
          }
        }
        tc05::commit(obar);
        if (jj + 1 < nt && !issue_s(g + 1)) s_abort = 1;
      }
    }
    if (failed) break;
    g_tile += nt;
    // output: wait for the last P V
    bool ok = mbar_wait_bounded(obar, o_cnt & 1, p.dev_status);
    o_cnt++;
    tc05::fence_after();
    const bool whole = (j0 == 0 && j1 == R.tiles);
    const bool store = ok && row_ok;
    {
      const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
      const size_t slot = (size_t)(c + u_global);
#pragma unroll 1
      for (int cb = 0; cb < D / 32; ++cb) {
        uint32_t r[32];
        tc05::ld32(t_o + cb * 32, r);  // warp-collective: every lane loads, valid rows store
        tc05::wait_ld();
        if (!store) continue;
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
      if (store && !whole) p.ws_lse[slot * VM + tid] = l_run > 0.f ? m_run + log2f(l_run) : -INFINITY;
    }
    if (!ok) s_abort = 1;
    tc05::fence_before();
    __syncthreads();
    if (s_abort) failed = true;
    pos += nt;
  }

  if (failed && tid == 0) {
    // drain: every MMA issued so far, then (bounded) any TMA still landing
    tc05::commit(xbar);
    mbar_wait_bounded(xbar, 0, p.dev_status);
    for (uint32_t g = (gk_issued > 2 ? gk_issued - 2 : 0); g < gk_issued; ++g)
      mbar_wait_bounded(&kfull[g & 1], (g >> 1) & 1, p.dev_status);
    for (uint32_t g = (gv_issued > 2 ? gv_issued - 2 : 0); g < gv_issued; ++g)
      mbar_wait_bounded(&vfull[g & 1], (g >> 1) & 1, p.dev_status);
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
  const int64_t U0 = R.tile_begin + (int64_t)ul * R.tiles, U1 = U0 + R.tiles;
  const int64_t T = p.total_tiles, N = p.n_cta;
  const int64_t c0 = ((U0 + 1) * N - 1) / T, c1 = (U1 * N - 1) / T;
  if (c0 == c1) return;
  const int r = blockIdx.y * 8 + (threadIdx.x / TPR), cc = (threadIdx.x % TPR) * CPT;
  const int hk = ul / R.mtiles, mt = ul % R.mtiles;
  const int Rw = mt * VM + r, qi = Rw / p.G, qg = Rw % p.G;
  if (qi >= R.n_rows) return;
  float M = -INFINITY;
  for (int64_t c = c0; c <= c1; ++c) M = fmaxf(M, p.ws_lse[(c + u) * VM + r]);
  const float Mu = M == -INFINITY ? 0.f : M;
  float L = 0.f, acc[CPT];
#pragma unroll
  for (int e = 0; e < CPT; ++e) acc[e] = 0.f;
#pragma unroll 4
  for (int64_t c = c0; c <= c1; ++c) {
    const float w = exp2f(p.ws_lse[(c + u) * VM + r] - Mu);
    const float* src = p.ws_o + ((c + u) * VM + r) * D + cc;
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

static int64_t verify_ctas(int64_t T) {
  const char* e = getenv("VC_VERIFY_CTAS");
  int64_t n = e ? atoll(e) : 2 * (int64_t)sm_count_v();
  if (n < 1) n = 1;
  return n < T ? n : T;
}

size_t verify_workspace_size(const vc_shape* s, int32_t max_rows) {
  if (max_rows < 1) return 0;
  const int G = s->Hq / s->Hkv;
  const int64_t mtiles = ((int64_t)max_rows * G + VM - 1) / VM;
  const int64_t units = (int64_t)s->B * s->Hkv * mtiles;
  const int64_t slots = units + 2 * (int64_t)sm_count_v() + 8;
  return (size_t)slots * VM * (s->d + 1) * sizeof(float) + 256;
}

template <int D>
static cudaError_t launch_verify_t(const VerifyParams& p, cudaStream_t s) {
  using C = VCfg<D>;
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(verify_attn_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  cudaError_t e = launch_pdl(verify_attn_kernel<D>, dim3(p.n_cta), dim3(128), C::SMEM, s, p);
  if (e != cudaSuccess) return e;
  return launch_pdl(verify_combine_kernel<D>, dim3(p.n_units, VM / 8), dim3(256), 0, s, p);
}

static bool a16(const void* p) { return p && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

cudaError_t launch_verify(const vc_shape* shape, const vc_verify_req* req, void* ws, size_t ws_bytes,
                          int32_t* dev_status, cudaStream_t stream, vc_status* st) {
  *st = VC_OK;
  if (!shape || shape->B < 1 || shape->B > VC_MAX_BATCH || shape->Hkv < 1 || shape->Hq < shape->Hkv ||
      shape->Hq % shape->Hkv != 0 || !req) {
    *st = VC_ERR_INVALID;
    return cudaSuccess;
  }
  if (shape->d != 64 && shape->d != 128) {
    *st = VC_ERR_UNSUPPORTED;
    return cudaSuccess;
  }
  const int d = shape->d, G = shape->Hq / shape->Hkv;
  VerifyParams p;  // about 18 KB: the tensor maps travel as kernel parameters
  memset(&p, 0, sizeof(p));
  p.B = shape->B;
  p.Hq = shape->Hq;
  p.Hkv = shape->Hkv;
  p.G = G;
  p.scale_log2 = (float)(1.4426950408889634 / sqrt((double)d));
  p.dev_status = dev_status;
  int64_t tiles = 0;
  int32_t units = 0, max_rows = 0;
  for (int b = 0; b < shape->B; ++b) {
    const vc_verify_req& r = req[b];
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
    R.tile_begin = tiles;
    units += shape->Hkv * R.mtiles;
    tiles += (int64_t)shape->Hkv * R.mtiles * R.tiles;
    if (r.n_rows > max_rows) max_rows = r.n_rows;
  }
  p.total_tiles = tiles;
  p.n_cta = (int32_t)verify_ctas(tiles);
  p.n_units = units;
  const size_t slots = (size_t)p.n_cta + units;
  const size_t need = slots * VM * (d + 1) * sizeof(float);
  if (!ws || ws_bytes < need || !a16(ws)) {
    *st = VC_ERR_WORKSPACE;
    return cudaSuccess;
  }
  p.ws_o = static_cast<float*>(ws);
  p.ws_lse = p.ws_o + slots * VM * d;
  return d == 128 ? launch_verify_t<128>(p, stream) : launch_verify_t<64>(p, stream);
}

}  // namespace vc
