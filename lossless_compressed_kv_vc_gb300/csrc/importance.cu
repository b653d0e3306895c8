// SnapKV-style token importance for the token-drop compressor ("VeriCache: Turning Lossy KV Cache
// into Lossless LLM Inference", "Architecture support": SnapKV is named among the token-drop
// compressors behind the single compressor interface; the pages do not define its scoring).
//
// For each request, the queries of its last W context tokens (the observation window) attend to
// the keys of KV_full, causally (window query i sits at position ctx - W + i). A key's vote is the
// sum of its softmax weights over the W window queries and all Hq query heads; the importance is
// the votes smoothed by a 1-D pooling of odd width k (max, or average with zero padding).
//
// Kernels (all requests and KV heads in every launch):
//   imp_stats_kernel  pass 1, grid (key chunks, Hkv, B): per window row, the running maximum and
//                     sum of 2^(s log2e / sqrt(d)) over the chunk's keys;
//   imp_lse_kernel    grid (Hkv, B): the rows' log-sum-exp over all chunks;
//   imp_votes_kernel  pass 2, same grid as pass 1: sum over the rows of 2^(s' - lse) per key, one
//                     partial per KV head;
//   imp_pool_kernel   grid (token blocks, B): the sum over KV heads, then the pooling.
// Tensor cores: mma.sync m16n8k16 with the 64 keys of a tile as M (A operand, from shared memory
// by ldmatrix) and 8 window rows as N (B operand, the rows' queries held in registers); each warp
// owns 32 of the W * G rows of a KV head. A key's sum over rows is then a sum over the N columns
// (in-lane, then over the 4 lanes of a quad) and across warps through shared memory.
#include "vc_internal.cuh"

namespace vc {

namespace {

constexpr int IT_KEYS = 64;                  // keys per tile
constexpr int IT_TPC = 16;                   // tiles per CTA chunk
constexpr int IT_CHUNK = IT_KEYS * IT_TPC;   // keys per chunk
constexpr int IT_POOL_BLOCK = 256;           // tokens per pooling CTA
constexpr int IT_MAX_HALF = 32;              // largest pooling half-width

struct ImpReqDev {
  const bf16* k;      // [Hkv][cap][d]
  const bf16* q;      // [W][Hq][d]
  float* imp;         // [ctx]
  int32_t ctx, cap, n_chunks;
  int64_t vote_off;   // this request's votes in the workspace: [Hkv][ctx] floats
};

struct ImpParams {
  ImpReqDev req[VC_MAX_BATCH];
  int32_t B, Hq, Hkv, G, W, R;  // R = W * G window rows per KV head
  int32_t max_chunks, pool_half, pool_avg, pool_k;
  float scale_log2;
  float2* ws_ml;   // [B][Hkv][max_chunks][R]: (max, sum) per chunk and row, exp2 domain
  float* ws_lse;   // [B][Hkv][R]
  float* ws_vote;  // per request [Hkv][ctx]
  int32_t* dev_status;
};

// Byte offset of 16-byte piece cc of key row r in a 64-key tile: 64-channel halves of
// [64 rows][128 B], pieces XOR-swizzled by the row so that the 8 rows an ldmatrix reads use
// distinct banks.
__device__ __forceinline__ int it_off(int r, int cc) {
  return (cc >> 3) * (IT_KEYS * 128) + r * 128 + (((cc & 7) ^ (r & 7)) << 4);
}

template <int D, int NW>
__device__ __forceinline__ void it_load_tile(uint8_t* dst, const ImpReqDev& r, int j, int tb) {
  const bf16* kbase = r.k + (size_t)j * r.cap * D;
  for (int e = threadIdx.x; e < IT_KEYS * (D / 8); e += NW * 32) {
    const int row = e / (D / 8), cc = e % (D / 8);
    const int tok = tb + row;
    const bool ok = tok < r.ctx;
    cp_async16(dst + it_off(row, cc), kbase + (size_t)(ok ? tok : 0) * D + cc * 8, ok ? 16u : 0u);
  }
  cp_async_commit();
}

// The warp's 32 window rows as B fragments: row 8 nt + lane/4 (within the warp's rows), channels
// 16 ks + 2 (lane % 4) (+1) and +8.
template <int D>
__device__ __forceinline__ void it_load_q(uint32_t (&qb)[4][D / 16][2], const ImpParams& p, const ImpReqDev& r,
                                          int j, int warp, int lane) {
#pragma unroll
  for (int nt = 0; nt < 4; ++nt) {
    const int row = 32 * warp + 8 * nt + (lane >> 2);
    const int i = row / p.G, gq = row % p.G;
    const bf16* qr = r.q + ((size_t)i * p.Hq + (size_t)j * p.G + gq) * D;
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
      qb[nt][ks][0] = *reinterpret_cast<const uint32_t*>(qr + 16 * ks + 2 * (lane & 3));
      qb[nt][ks][1] = *reinterpret_cast<const uint32_t*>(qr + 16 * ks + 8 + 2 * (lane & 3));
    }
  }
}

// S^T for keys 16 mt .. 16 mt + 15 of the tile and the warp's 32 rows: s[nt][c] with c = 0, 1 the
// key 16 mt + lane/4 and rows 8 nt + 2 (lane % 4) + c, c = 2, 3 the key + 8.
template <int D>
__device__ __forceinline__ void it_scores(float (&s)[4][4], const uint8_t* kt, const uint32_t (&qb)[4][D / 16][2],
                                          int mt, int lane) {
#pragma unroll
  for (int nt = 0; nt < 4; ++nt)
#pragma unroll
    for (int c = 0; c < 4; ++c) s[nt][c] = 0.f;
  const int arow = 16 * mt + (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
  for (int ks = 0; ks < D / 16; ++ks) {
    uint32_t a[4];
    ldsm_x4(a[0], a[1], a[2], a[3], kt + it_off(arow, 2 * ks + (lane >> 4)));
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) mma_bf16_16816(s[nt], a, qb[nt][ks][0], qb[nt][ks][1]);
  }
}

// Three 4-warp CTAs per SM (the register cap that allows is met without spills): the MMAs are
// issue-bound, so the extra warps matter more than registers.
template <int D, int NW>
__global__ void __launch_bounds__(NW * 32, NW <= 4 ? 12 / NW : 1) imp_stats_kernel(const __grid_constant__ ImpParams p) {
  pdl_launch_dependents();
  pdl_wait();
  const int chunk = blockIdx.x, j = blockIdx.y, b = blockIdx.z;
  const ImpReqDev& r = p.req[b];
  if (chunk >= r.n_chunks) return;
  __shared__ __align__(1024) uint8_t kt[2][IT_KEYS * D * 2];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t4 = lane & 3;
  const int t_begin = chunk * IT_CHUNK;
  const int t_end = min(r.ctx, t_begin + IT_CHUNK);
  const int ntiles = (t_end - t_begin + IT_KEYS - 1) / IT_KEYS;
  const int win0 = r.ctx - p.W;  // position of window query 0
  uint32_t qb[4][D / 16][2];
  it_load_q<D>(qb, p, r, j, warp, lane);
  float m[8], l[8];
  int pos[8];
#pragma unroll
  for (int rr = 0; rr < 8; ++rr) {
    m[rr] = -INFINITY;
    l[rr] = 0.f;
    pos[rr] = win0 + (32 * warp + 8 * (rr >> 1) + 2 * t4 + (rr & 1)) / p.G;
  }
  it_load_tile<D, NW>(kt[0], r, j, t_begin);
  for (int tile = 0; tile < ntiles; ++tile) {
    if (tile + 1 < ntiles)
      it_load_tile<D, NW>(kt[(tile + 1) & 1], r, j, t_begin + (tile + 1) * IT_KEYS);
    else
      cp_async_commit();
    cp_async_wait<1>();
    __syncthreads();
    const int tb = t_begin + tile * IT_KEYS;
    const bool all_visible = tb + IT_KEYS - 1 <= win0;
    float s[4][4][4];
#pragma unroll
    for (int mt = 0; mt < 4; ++mt) it_scores<D>(s[mt], kt[tile & 1], qb, mt, lane);
#pragma unroll
    for (int rr = 0; rr < 8; ++rr) {
      const int nt = rr >> 1, e = rr & 1;
      float v[8];
      float mx = -INFINITY;
#pragma unroll
      for (int mt = 0; mt < 4; ++mt)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int key = tb + 16 * mt + g + 8 * h;
          float x = s[mt][nt][e + 2 * h] * p.scale_log2;
          if (!all_visible && key > pos[rr]) x = -INFINITY;
          v[2 * mt + h] = x;
          mx = fmaxf(mx, x);
        }
      const float mn = fmaxf(m[rr], mx);
      if (mn == -INFINITY) continue;  // no visible key for this row yet
      float sum = 0.f;
#pragma unroll
      for (int c = 0; c < 8; ++c) sum += ex2_approx(v[c] - mn);
      l[rr] = l[rr] * ex2_approx(m[rr] - mn) + sum;
      m[rr] = mn;
    }
    __syncthreads();  // every warp is done with this buffer before it is refilled
  }
  // combine the 8 lanes that hold the same rows (same lane % 4)
#pragma unroll
  for (int rr = 0; rr < 8; ++rr) {
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      const float mo = __shfl_xor_sync(0xffffffffu, m[rr], off);
      const float lo = __shfl_xor_sync(0xffffffffu, l[rr], off);
      const float mn = fmaxf(m[rr], mo);
      if (mn != -INFINITY) {
        l[rr] = l[rr] * ex2_approx(m[rr] - mn) + lo * ex2_approx(mo - mn);
        m[rr] = mn;
      }
    }
  }
  if (g == 0) {
    float2* dst = p.ws_ml + (((size_t)b * p.Hkv + j) * p.max_chunks + chunk) * p.R + 32 * warp;
#pragma unroll
    for (int rr = 0; rr < 8; ++rr) dst[8 * (rr >> 1) + 2 * t4 + (rr & 1)] = make_float2(m[rr], l[rr]);
  }
}

// log-sum-exp (base 2) of every window row over all chunks; thread = row.
__global__ void __launch_bounds__(256) imp_lse_kernel(const __grid_constant__ ImpParams p) {
  pdl_launch_dependents();
  pdl_wait();
  const int j = blockIdx.x, b = blockIdx.y, row = threadIdx.x;
  if (row >= p.R) return;
  const ImpReqDev& r = p.req[b];
  const float2* src = p.ws_ml + ((size_t)b * p.Hkv + j) * p.max_chunks * p.R + row;
  float M = -INFINITY;
  for (int c = 0; c < r.n_chunks; ++c) M = fmaxf(M, src[(size_t)c * p.R].x);
  float L = 0.f;
  for (int c = 0; c < r.n_chunks; ++c) {
    const float2 ml = src[(size_t)c * p.R];
    if (ml.x != -INFINITY) L += ml.y * ex2_approx(ml.x - M);
  }
  p.ws_lse[((size_t)b * p.Hkv + j) * p.R + row] = M + log2f(L);
}

template <int D, int NW>
__global__ void __launch_bounds__(NW * 32) imp_votes_kernel(const __grid_constant__ ImpParams p) {
  pdl_launch_dependents();
  pdl_wait();
  const int chunk = blockIdx.x, j = blockIdx.y, b = blockIdx.z;
  const ImpReqDev& r = p.req[b];
  if (chunk >= r.n_chunks) return;
  __shared__ __align__(1024) uint8_t kt[2][IT_KEYS * D * 2];
  __shared__ float vs[NW][IT_KEYS];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t4 = lane & 3;
  const int t_begin = chunk * IT_CHUNK;
  const int t_end = min(r.ctx, t_begin + IT_CHUNK);
  const int ntiles = (t_end - t_begin + IT_KEYS - 1) / IT_KEYS;
  const int win0 = r.ctx - p.W;
  uint32_t qb[4][D / 16][2];
  it_load_q<D>(qb, p, r, j, warp, lane);
  float lse[8];
  int pos[8];
  const float* lsrc = p.ws_lse + ((size_t)b * p.Hkv + j) * p.R + 32 * warp;
#pragma unroll
  for (int rr = 0; rr < 8; ++rr) {
    const int row = 8 * (rr >> 1) + 2 * t4 + (rr & 1);
    lse[rr] = lsrc[row];
    pos[rr] = win0 + (32 * warp + row) / p.G;
  }
  float* vote = p.ws_vote + r.vote_off + (size_t)j * r.ctx;
  it_load_tile<D, NW>(kt[0], r, j, t_begin);
  for (int tile = 0; tile < ntiles; ++tile) {
    if (tile + 1 < ntiles)
      it_load_tile<D, NW>(kt[(tile + 1) & 1], r, j, t_begin + (tile + 1) * IT_KEYS);
    else
      cp_async_commit();
    cp_async_wait<1>();
    __syncthreads();
    const int tb = t_begin + tile * IT_KEYS;
    const bool all_visible = tb + IT_KEYS - 1 <= win0;
#pragma unroll
    for (int mt = 0; mt < 4; ++mt) {
      float s[4][4];
      it_scores<D>(s, kt[tile & 1], qb, mt, lane);
      const int k0 = tb + 16 * mt + g, k1 = k0 + 8;
      float v0 = 0.f, v1 = 0.f;
#pragma unroll
      for (int rr = 0; rr < 8; ++rr) {
        const int nt = rr >> 1, e = rr & 1;
        const float p0 = ex2_approx(fmaf(s[nt][e], p.scale_log2, -lse[rr]));
        const float p1 = ex2_approx(fmaf(s[nt][e + 2], p.scale_log2, -lse[rr]));
        v0 += (all_visible || k0 <= pos[rr]) ? p0 : 0.f;
        v1 += (all_visible || k1 <= pos[rr]) ? p1 : 0.f;
      }
      v0 += __shfl_xor_sync(0xffffffffu, v0, 1);
      v0 += __shfl_xor_sync(0xffffffffu, v0, 2);
      v1 += __shfl_xor_sync(0xffffffffu, v1, 1);
      v1 += __shfl_xor_sync(0xffffffffu, v1, 2);
      if (t4 == 0) {
        vs[warp][16 * mt + g] = v0;
        vs[warp][16 * mt + g + 8] = v1;
      }
    }
    __syncthreads();
    for (int kk = threadIdx.x; kk < IT_KEYS; kk += NW * 32) {  // one warp covers the 64 keys in two steps
      float sum = 0.f;
#pragma unroll
      for (int w = 0; w < NW; ++w) sum += vs[w][kk];
      const int key = tb + kk;
      if (key < r.ctx) vote[key] = sum;
    }
    __syncthreads();  // vs and this K buffer are reused
  }
}

// importance[t] = pool over |u - t| <= half of sum_j vote_j[u]: max over the in-range tokens, or
// the in-range sum divided by the kernel width (zero padding).
__global__ void __launch_bounds__(IT_POOL_BLOCK) imp_pool_kernel(const __grid_constant__ ImpParams p) {
  pdl_launch_dependents();
  pdl_wait();
  const int b = blockIdx.y;
  const ImpReqDev& r = p.req[b];
  const int t0 = blockIdx.x * IT_POOL_BLOCK;
  if (t0 >= r.ctx) return;
  __shared__ float sm[IT_POOL_BLOCK + 2 * IT_MAX_HALF];
  const int half = p.pool_half;
  const float pad = p.pool_avg ? 0.f : -INFINITY;
  const float* vote = p.ws_vote + r.vote_off;
  for (int e = threadIdx.x; e < IT_POOL_BLOCK + 2 * half; e += IT_POOL_BLOCK) {
    const int t = t0 - half + e;
    float v = pad;
    if (t >= 0 && t < r.ctx) {
      v = 0.f;
      for (int j = 0; j < p.Hkv; ++j) v += vote[(size_t)j * r.ctx + t];
    }
    sm[e] = v;
  }
  __syncthreads();
  const int t = t0 + threadIdx.x;
  if (t >= r.ctx) return;
  float acc = p.pool_avg ? 0.f : -INFINITY;
  for (int u = 0; u <= 2 * half; ++u) acc = p.pool_avg ? acc + sm[threadIdx.x + u] : fmaxf(acc, sm[threadIdx.x + u]);
  r.imp[t] = p.pool_avg ? acc / (float)p.pool_k : acc;
}

template <int D, int NW>
cudaError_t launch_passes(const ImpParams& p, int max_ctx, cudaStream_t s) {
  const dim3 grid(p.max_chunks, p.Hkv, p.B);
  cudaError_t e = launch_pdl(imp_stats_kernel<D, NW>, grid, dim3(NW * 32), 0, s, p);
  if (e != cudaSuccess) return e;
  e = launch_pdl(imp_lse_kernel, dim3(p.Hkv, p.B), dim3(256), 0, s, p);
  if (e != cudaSuccess) return e;
  e = launch_pdl(imp_votes_kernel<D, NW>, grid, dim3(NW * 32), 0, s, p);
  if (e != cudaSuccess) return e;
  return launch_pdl(imp_pool_kernel, dim3((max_ctx + IT_POOL_BLOCK - 1) / IT_POOL_BLOCK, p.B), dim3(IT_POOL_BLOCK), 0,
                    s, p);
}

template <int D>
cudaError_t launch_d(const ImpParams& p, int max_ctx, cudaStream_t s) {
  switch (p.R / 32) {
    case 1: return launch_passes<D, 1>(p, max_ctx, s);
    case 2: return launch_passes<D, 2>(p, max_ctx, s);
    case 4: return launch_passes<D, 4>(p, max_ctx, s);
    case 8: return launch_passes<D, 8>(p, max_ctx, s);
    default: return cudaErrorInvalidValue;
  }
}

bool a16(const void* q) { return q && (reinterpret_cast<uintptr_t>(q) & 15u) == 0; }

// Workspace layout for B requests of at most max_ctx tokens (floats, 256-byte aligned parts).
struct ImpWs {
  size_t ml, lse, vote, total;
};
ImpWs imp_ws(int B, int Hkv, int R, int max_chunks, int64_t vote_floats) {
  auto up = [](size_t x) { return (x + 255) & ~size_t(255); };
  ImpWs w;
  w.ml = 0;
  w.lse = up((size_t)B * Hkv * max_chunks * R * sizeof(float2));
  w.vote = w.lse + up((size_t)B * Hkv * R * sizeof(float));
  w.total = w.vote + up((size_t)vote_floats * sizeof(float));
  return w;
}

}  // namespace

}  // namespace vc

using namespace vc;

extern "C" size_t vc_importance_workspace_size(const vc_shape* shape, int32_t window, int32_t max_ctx) {
  if (!shape || shape->B < 1 || shape->B > VC_MAX_BATCH || shape->Hkv < 1 || shape->Hq % shape->Hkv != 0 ||
      window < 1 || max_ctx < window)
    return 0;
  const int R = window * (shape->Hq / shape->Hkv);
  const int max_chunks = (max_ctx + IT_CHUNK - 1) / IT_CHUNK;
  return imp_ws(shape->B, shape->Hkv, R, max_chunks, (int64_t)shape->B * shape->Hkv * max_ctx).total + 256;
}

extern "C" vc_status vc_snapkv_importance(const vc_shape* shape, const vc_importance_req* req, int32_t window,
                                          int32_t pool_kernel, int32_t pool_kind, void* ws, size_t ws_bytes,
                                          int32_t* dev_status, cudaStream_t stream) {
  if (!shape || !req || shape->B < 1 || shape->B > VC_MAX_BATCH || shape->Hkv < 1 || shape->Hq < shape->Hkv ||
      shape->Hq % shape->Hkv != 0 || window < 1 || pool_kernel < 1 || (pool_kernel & 1) == 0 ||
      (pool_kind != VC_POOL_MAX && pool_kind != VC_POOL_AVG))
    return VC_ERR_INVALID;
  const int d = shape->d, G = shape->Hq / shape->Hkv, R = window * G;
  if ((d != 64 && d != 128) || R % 32 != 0 || R > 256 || pool_kernel / 2 > IT_MAX_HALF) return VC_ERR_UNSUPPORTED;
  ImpParams p;
  memset(&p, 0, sizeof(p));
  p.B = shape->B;
  p.Hq = shape->Hq;
  p.Hkv = shape->Hkv;
  p.G = G;
  p.W = window;
  p.R = R;
  p.pool_half = pool_kernel / 2;
  p.pool_k = pool_kernel;
  p.pool_avg = pool_kind == VC_POOL_AVG;
  p.scale_log2 = (float)(1.4426950408889634 / sqrt((double)d));
  p.dev_status = dev_status;
  int max_ctx = 0, max_chunks = 0;
  int64_t vote_floats = 0;
  for (int b = 0; b < shape->B; ++b) {
    const vc_importance_req& q = req[b];
    if (!a16(q.full.k) || !a16(q.q_obs) || !q.importance || (reinterpret_cast<uintptr_t>(q.importance) & 3u) ||
        q.full.ctx < window || q.full.cap < q.full.ctx)
      return VC_ERR_INVALID;
    ImpReqDev& r = p.req[b];
    r.k = static_cast<const bf16*>(q.full.k);
    r.q = static_cast<const bf16*>(q.q_obs);
    r.imp = q.importance;
    r.ctx = q.full.ctx;
    r.cap = q.full.cap;
    r.n_chunks = (q.full.ctx + IT_CHUNK - 1) / IT_CHUNK;
    r.vote_off = vote_floats;
    vote_floats += (int64_t)shape->Hkv * q.full.ctx;
    if (q.full.ctx > max_ctx) max_ctx = q.full.ctx;
    if (r.n_chunks > max_chunks) max_chunks = r.n_chunks;
  }
  if (max_chunks > 65535) return VC_ERR_UNSUPPORTED;
  p.max_chunks = max_chunks;
  const ImpWs lay = imp_ws(shape->B, shape->Hkv, R, max_chunks, vote_floats);
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u) || ws_bytes < lay.total) return VC_ERR_WORKSPACE;
  uint8_t* base = static_cast<uint8_t*>(ws);
  p.ws_ml = reinterpret_cast<float2*>(base + lay.ml);
  p.ws_lse = reinterpret_cast<float*>(base + lay.lse);
  p.ws_vote = reinterpret_cast<float*>(base + lay.vote);
  const cudaError_t e = d == 128 ? launch_d<128>(p, max_ctx, stream) : launch_d<64>(p, max_ctx, stream);
  return e == cudaSuccess ? VC_OK : VC_ERR_CUDA;
}
