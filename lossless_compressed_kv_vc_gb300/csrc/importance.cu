// SnapKV-style token importance for the token-drop compressor ("VeriCache: Turning Lossy KV Cache
// into Lossless LLM Inference", "Architecture support": SnapKV is named among the token-drop
// compressors behind the single compressor interface; the pages do not define its scoring).
//
// For each request, the queries of its last W context tokens (the observation window) attend to
// the keys of KV_full, causally (window query i sits at position ctx - W + i). A key's vote is the
// sum of its softmax weights over the W window queries and all Hq query heads; the importance is
// the votes smoothed by a 1-D pooling of odd width k (max, or average with zero padding).
//
// The two passes over the keys run on the tcgen05 tensor cores in the verification kernel's
// row-statistics and column-sum modes (launch_obs_passes in verify.cu): the W x G window rows of a
// KV head are the M = 128 rows of its tiles, exactly like drafted tokens in verification (the
// window's own keys are the causal "new" part). Pass 1 gives every row's log-sum-exp; pass 2 sums
// 2^(s - lse) over each tile's rows for every key with an all-ones MMA, one partial per (KV head,
// row tile). imp_pool_kernel adds the partials and pools.
#include "vc_internal.cuh"

namespace vc {

namespace {

constexpr int IT_POOL_BLOCK = 256;           // tokens per pooling CTA
constexpr int IT_MAX_HALF = 32;              // largest pooling half-width

struct ImpReqDev {
  float* imp;         // [ctx]
  const float* votes; // [n_part][ctx]
  int32_t ctx;
};

struct ImpParams {
  ImpReqDev req[VC_MAX_BATCH];
  int32_t B, n_part, pool_half, pool_avg, pool_k;
};

// importance[t] = pool over |u - t| <= half of sum_j vote_j[u] (j over the KV-head x row-tile
// partials): max over the in-range tokens, or the in-range sum divided by the width (zero padding).
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
  const float* vote = r.votes;
  for (int e = threadIdx.x; e < IT_POOL_BLOCK + 2 * half; e += IT_POOL_BLOCK) {
    const int t = t0 - half + e;
    float v = pad;
    if (t >= 0 && t < r.ctx) {
      v = 0.f;
      for (int j = 0; j < p.n_part; ++j) v += vote[(size_t)j * r.ctx + t];
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

bool a16(const void* q) { return q && (reinterpret_cast<uintptr_t>(q) & 15u) == 0; }

// Workspace parts (256-byte aligned): split-unit row statistics, the rows' lse, the votes.
struct ImpWs {
  size_t slots, lse, vote, total;
};
ImpWs imp_ws(int B, int Hkv, int mtiles, int64_t vote_floats) {
  auto up = [](size_t x) { return (x + 255) & ~size_t(255); };
  ImpWs w;
  w.slots = 0;
  w.lse = up(obs_slot_floats(B, Hkv, mtiles) * sizeof(float));
  w.vote = w.lse + up((size_t)B * Hkv * mtiles * 128 * sizeof(float));
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
  const int mtiles = obs_mtiles(window, shape->Hq / shape->Hkv);
  return imp_ws(shape->B, shape->Hkv, mtiles, (int64_t)shape->B * shape->Hkv * mtiles * max_ctx).total + 256;
}

extern "C" vc_status vc_snapkv_importance(const vc_shape* shape, const vc_importance_req* req, int32_t window,
                                          int32_t pool_kernel, int32_t pool_kind, void* ws, size_t ws_bytes,
                                          int32_t* dev_status, cudaStream_t stream) {
  if (!shape || !req || shape->B < 1 || shape->B > VC_MAX_BATCH || shape->Hkv < 1 || shape->Hq < shape->Hkv ||
      shape->Hq % shape->Hkv != 0 || window < 1 || pool_kernel < 1 || (pool_kernel & 1) == 0 ||
      (pool_kind != VC_POOL_MAX && pool_kind != VC_POOL_AVG))
    return VC_ERR_INVALID;
  const int d = shape->d, G = shape->Hq / shape->Hkv;
  if ((d != 64 && d != 128) || pool_kernel / 2 > IT_MAX_HALF) return VC_ERR_UNSUPPORTED;
  const int mtiles = obs_mtiles(window, G);
  ObsArgs oa;
  memset(&oa, 0, sizeof(oa));
  oa.B = shape->B;
  oa.Hq = shape->Hq;
  oa.Hkv = shape->Hkv;
  oa.d = d;
  oa.W = window;
  oa.dev_status = dev_status;
  ImpParams p;
  memset(&p, 0, sizeof(p));
  p.B = shape->B;
  p.n_part = shape->Hkv * mtiles;
  p.pool_half = pool_kernel / 2;
  p.pool_k = pool_kernel;
  p.pool_avg = pool_kind == VC_POOL_AVG;
  int max_ctx = 0;
  int64_t vote_floats = 0;
  for (int b = 0; b < shape->B; ++b) {
    const vc_importance_req& q = req[b];
    if (!a16(q.full.k) || !a16(q.q_obs) || !q.importance || (reinterpret_cast<uintptr_t>(q.importance) & 3u) ||
        q.full.ctx < window || q.full.cap < q.full.ctx)
      return VC_ERR_INVALID;
    vote_floats += (int64_t)p.n_part * q.full.ctx;
    if (q.full.ctx > max_ctx) max_ctx = q.full.ctx;
  }
  const ImpWs lay = imp_ws(shape->B, shape->Hkv, mtiles, vote_floats);
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u) || ws_bytes < lay.total) return VC_ERR_WORKSPACE;
  uint8_t* base = static_cast<uint8_t*>(ws);
  oa.ws_lse = reinterpret_cast<float*>(base + lay.slots);
  oa.ws_lse_floats = obs_slot_floats(shape->B, shape->Hkv, mtiles);
  float* lse = reinterpret_cast<float*>(base + lay.lse);
  float* votes = reinterpret_cast<float*>(base + lay.vote);
  int64_t off = 0;
  for (int b = 0; b < shape->B; ++b) {
    const vc_importance_req& q = req[b];
    ObsReq& o = oa.req[b];
    o.k = static_cast<const bf16*>(q.full.k);
    o.q = static_cast<const bf16*>(q.q_obs);
    o.ctx = q.full.ctx;
    o.cap = q.full.cap;
    o.lse = lse + (size_t)b * shape->Hkv * mtiles * 128;
    o.votes = votes + off;
    p.req[b].imp = q.importance;
    p.req[b].votes = votes + off;
    p.req[b].ctx = q.full.ctx;
    off += (int64_t)p.n_part * q.full.ctx;
  }
  cudaError_t e = launch_obs_passes(oa, stream);
  if (e == cudaSuccess)
    e = launch_pdl(imp_pool_kernel, dim3((max_ctx + IT_POOL_BLOCK - 1) / IT_POOL_BLOCK, shape->B), dim3(IT_POOL_BLOCK),
                   0, stream, p);
  return e == cudaSuccess ? VC_OK : VC_ERR_CUDA;
}
