// C-ABI entry points of libvc: argument validation, split planning and kernel launches.
// Validation failures return a status and launch nothing; nothing here allocates or synchronises.
#include "vc_internal.cuh"

#include <math.h>
#include <stdlib.h>
#include <string.h>

#include <mutex>
#include <unordered_map>

namespace vc {
cudaError_t launch_verify(const vc_shape* shape, const vc_verify_req* req, int h0, int h1, void* ws,
                          size_t ws_bytes, int32_t* dev_status, cudaStream_t stream, vc_status* st);
size_t verify_workspace_size(const vc_shape* shape, int32_t max_rows);
int32_t verify_launch_count(const vc_shape* shape, const vc_verify_req* req);
}  // namespace vc

using namespace vc;

static bool aligned16(const void* p) { return p && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

static bool shape_ok(const vc_shape* s) {
  return s && s->B >= 1 && s->B <= VC_MAX_BATCH && s->Hkv >= 1 && s->Hq >= s->Hkv && s->Hq % s->Hkv == 0 &&
         (s->d == 64 || s->d == 128);
}

static int env_int(const char* name, int dflt) {
  const char* v = getenv(name);
  return v ? atoi(v) : dflt;
}

static int sm_count() {
  static int n = 0;
  if (n == 0) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      n = 152;
  }
  return n;
}

namespace vc {
int draft_ctas_per_sm(int G, int kind);
}

// CTAs per KV head of a draft launch: one wave of CTAs over all heads.
static int draft_ctas_per_head_max(int Hkv, int G, int kind) {
  const int n = vc::draft_ctas_per_sm(G, kind) * sm_count() / Hkv;
  return n > 1 ? n : 1;
}

// The largest wave of any draft launch (G <= 8 gives the most CTAs per SM), for the workspace bound.
static int draft_ctas_per_head_bound(int Hkv) {
  int n = 1;
  for (int kind : {0, 2, 4}) {
    const int k = draft_ctas_per_head_max(Hkv, 1, kind);
    n = k > n ? k : n;
  }
  return n;
}

// Arrival counters at the start of the draft workspace: one 32-bit word per (KV head, request slot),
// in a block of fixed size for up to VC_DRAFT_MAX_KV_HEADS heads. The block does not depend on the
// call's shape, so the counters of every head sit at the same bytes for every call: a workspace
// zero-filled once keeps zero counters whatever shapes later calls have (a shape-dependent block
// would let a call with more KV heads read an earlier call's partials as counters).
static_assert(VC_DRAFT_COUNTER_BYTES % 256 == 0, "partials start 256-byte aligned");
static size_t draft_counter_bytes() { return VC_DRAFT_COUNTER_BYTES; }

// Last library operation launched on each stream. A draft step may start streaming before the
// kernel ahead of it in the stream finishes unless that kernel writes KV_comp (a compress or an
// append after accept: the only writers of kept rows, indices and quantised blocks among the
// library's kernels, all of which trigger their dependents early).
enum { kOpNone = 0, kOpCompress = 1, kOpDraft = 2, kOpVerify = 3, kOpAccept = 4 };
static std::mutex g_op_mu;
static std::unordered_map<cudaStream_t, int> g_last_op;

static int last_op(cudaStream_t s) {
  std::lock_guard<std::mutex> lock(g_op_mu);
  auto it = g_last_op.find(s);
  return it == g_last_op.end() ? kOpNone : it->second;
}

static void set_last_op(cudaStream_t s, int op) {
  std::lock_guard<std::mutex> lock(g_op_mu);
  g_last_op[s] = op;
}

extern "C" {

int32_t vc_version(void) { return 100; }

const char* vc_status_string(vc_status s) {
  switch (s) {
    case VC_OK: return "ok";
    case VC_ERR_INVALID: return "invalid argument";
    case VC_ERR_UNSUPPORTED: return "unsupported configuration";
    case VC_ERR_CUDA: return "CUDA error";
    case VC_ERR_NOT_PINNED: return "host buffer is not page-locked";
    case VC_ERR_WORKSPACE: return "workspace too small";
  }
  return "unknown status";
}

size_t vc_workspace_size(int32_t call, const vc_shape* shape, int32_t max_rows) {
  if (!shape_ok(shape)) return 0;
  if (call == VC_CALL_DRAFT) {
    // CTA partials: slots (CTA + request) per head, CTAs per head at most one wave plus B
    const size_t G = shape->Hq / shape->Hkv;
    const size_t slots = (size_t)shape->Hkv * (draft_ctas_per_head_bound(shape->Hkv) + 2 * shape->B);
    return draft_counter_bytes() + slots * G * (shape->d + 1) * sizeof(float) + 256;
  }
  if (call == VC_CALL_VERIFY) return verify_workspace_size(shape, max_rows);
  return 0;
}

// ---------------------------------------------------------------------------------------------
// The quantised layout rule every call shares: whole 32-token blocks while at least residual_min
// trailing tokens stay bf16.
static int quant_blocks(int ctx, int residual_min) { return ctx > residual_min ? (ctx - residual_min) / VC_GROUP : 0; }

vc_status vc_comp_bytes(const vc_shape* shape, int32_t mode, int32_t bits, int32_t ctx, int32_t max_ctx,
                        int32_t keep, int32_t residual_min, int32_t max_drafts, vc_comp_sizes* out) {
  if (!out || !shape || shape->Hkv < 1 || (shape->d != 64 && shape->d != 128)) return VC_ERR_INVALID;
  if (ctx < 1 || max_ctx < ctx || keep < 0 || residual_min < 0 || max_drafts < 0) return VC_ERR_INVALID;
  if (mode != VC_TOKEN_DROP && mode != VC_QUANT) return VC_ERR_INVALID;
  memset(out, 0, sizeof(*out));
  const size_t Hkv = shape->Hkv, d = shape->d;
  int res_max = 0;
  if (mode == VC_QUANT) {
    if (bits != 2 && bits != 4) return VC_ERR_UNSUPPORTED;
    out->ng = quant_blocks(ctx, residual_min);
    out->n_res = ctx - VC_GROUP * out->ng;
    const int cap = quant_blocks(max_ctx, residual_min);
    out->ng_cap = cap > 1 ? cap : 1;
    // the residual of a context c > residual_min is residual_min .. residual_min + 31 rows
    const int grown = max_ctx < residual_min + VC_GROUP - 1 ? max_ctx : residual_min + VC_GROUP - 1;
    res_max = max_ctx > ctx && grown > out->n_res ? grown : out->n_res;
    out->codes_bytes = Hkv * out->ng_cap * (VC_GROUP * d * bits / 8);
    out->kscale_bytes = Hkv * out->ng_cap * d * 2;
    out->vscale_bytes = Hkv * (size_t)VC_GROUP * out->ng_cap * (d / VC_GROUP) * 2;
  } else {
    out->keep = keep < ctx ? keep : ctx;
    out->idx_bytes = (size_t)(out->keep > 1 ? out->keep : 1) * 4;
    out->rows_bytes = Hkv * out->keep * d * 2;
  }
  out->win_cap = res_max + max_drafts + 1;
  out->win_bytes = Hkv * out->win_cap * d * 2;
  return VC_OK;
}

// ---------------------------------------------------------------------------------------------
vc_status vc_compress_kv(const vc_shape* shape, const vc_kv_full* full, const float* const* importance,
                         const int32_t* recent, int32_t residual_min, vc_kv_comp* comp, int32_t* dev_status,
                         cudaStream_t stream) {
  if (!shape_ok(shape) || !full || !comp) return VC_ERR_INVALID;
  const int B = shape->B, d = shape->d;
  const int mode = comp[0].mode;
  for (int b = 0; b < B; ++b) {
    const vc_kv_full& f = full[b];
    if (comp[b].mode != mode) return VC_ERR_UNSUPPORTED;
    if (!aligned16(f.k) || !aligned16(f.v) || f.ctx < 1 || f.cap < f.ctx) return VC_ERR_INVALID;
  }
  if (mode == VC_TOKEN_DROP) {
    if (!importance || !recent) return VC_ERR_INVALID;
    KeepParams kp;
    memset(&kp, 0, sizeof(kp));
    kp.B = B;
    kp.Hkv = shape->Hkv;
    kp.d = d;
    kp.dev_status = dev_status;
    int max_keep = 0;
    for (int b = 0; b < B; ++b) {
      vc_kv_comp& c = comp[b];
      const vc_kv_full& f = full[b];
      if (!importance[b] || (reinterpret_cast<uintptr_t>(importance[b]) & 3u) || !c.idx) return VC_ERR_INVALID;
      if (recent[b] < 0 || c.keep < recent[b] || c.keep < 1) return VC_ERR_INVALID;
      const int keep = c.keep < f.ctx ? c.keep : f.ctx;
      if (c.compact) {
        if (!aligned16(c.k_rows) || !aligned16(c.v_rows) || c.rows_cap < keep) return VC_ERR_INVALID;
      }
      KeepReq& r = kp.req[b];
      r.imp = importance[b];
      r.idx = c.idx;
      r.ctx = f.ctx;
      r.keep = c.keep;
      r.recent = recent[b] < f.ctx ? recent[b] : f.ctx;
      r.k_src = static_cast<const bf16*>(f.k);
      r.v_src = static_cast<const bf16*>(f.v);
      r.src_cap = f.cap;
      r.k_dst = static_cast<bf16*>(c.k_rows);
      r.v_dst = static_cast<bf16*>(c.v_rows);
      r.dst_cap = c.rows_cap;
      r.compact = c.compact;
      if (keep > max_keep) max_keep = keep;
    }
    if (launch_keepset(kp, max_keep, stream) != cudaSuccess) return VC_ERR_CUDA;
    set_last_op(stream, kOpCompress);
    for (int b = 0; b < B; ++b) {
      if (comp[b].keep > full[b].ctx) comp[b].keep = full[b].ctx;
      comp[b].n_win = 0;
      if (!comp[b].compact) {
        comp[b].k_rows = const_cast<void*>(full[b].k);
        comp[b].v_rows = const_cast<void*>(full[b].v);
        comp[b].rows_cap = full[b].cap;
      }
    }
    return VC_OK;
  }
  if (mode != VC_QUANT) return VC_ERR_INVALID;
  if (residual_min < 0) return VC_ERR_INVALID;
  const int bits = comp[0].bits;
  if (bits != 2 && bits != 4) return VC_ERR_UNSUPPORTED;
  QuantParams qp;
  memset(&qp, 0, sizeof(qp));
  qp.B = B;
  qp.Hkv = shape->Hkv;
  qp.d = d;
  qp.bits = bits;
  qp.dev_status = dev_status;
  int max_ng = 0;
  for (int b = 0; b < B; ++b) {
    vc_kv_comp& c = comp[b];
    const vc_kv_full& f = full[b];
    if (c.bits != bits) return VC_ERR_UNSUPPORTED;
    const int ng = quant_blocks(f.ctx, residual_min);
    const int n_res = f.ctx - VC_GROUP * ng;
    if (ng > c.ng_cap) return VC_ERR_INVALID;  // the buffers hold ng_cap blocks per head
    if (ng > 0 && (!aligned16(c.kc) || !aligned16(c.ks) || !aligned16(c.kz) || !aligned16(c.vc) ||
                   !aligned16(c.vs) || !aligned16(c.vz)))
      return VC_ERR_INVALID;
    if (!aligned16(c.k_win) || !aligned16(c.v_win) || c.win_cap < n_res + 1) return VC_ERR_INVALID;
    QuantReq& r = qp.req[b];
    r.k = static_cast<const bf16*>(f.k);
    r.v = static_cast<const bf16*>(f.v);
    r.cap = f.cap;
    r.ctx = f.ctx;
    r.ng = ng;
    r.ng_cap = c.ng_cap;
    r.n_res = n_res;
    r.kc = c.kc;
    r.ks = reinterpret_cast<__half*>(c.ks);
    r.kz = reinterpret_cast<__half*>(c.kz);
    r.vc = c.vc;
    r.vs = reinterpret_cast<__half*>(c.vs);
    r.vz = reinterpret_cast<__half*>(c.vz);
    r.k_win = static_cast<bf16*>(c.k_win);
    r.v_win = static_cast<bf16*>(c.v_win);
    r.win_cap = c.win_cap;
    if (ng > max_ng) max_ng = ng;
  }
  if (launch_quant(qp, max_ng, VC_GROUP * max_ng, stream) != cudaSuccess) return VC_ERR_CUDA;
  set_last_op(stream, kOpCompress);
  for (int b = 0; b < B; ++b) {
    comp[b].ng = qp.req[b].ng;
    comp[b].n_win = qp.req[b].n_res;
  }
  return VC_OK;
}

// ---------------------------------------------------------------------------------------------
vc_status vc_append_kv(const vc_shape* shape, vc_kv_full* full, vc_kv_comp* comp, const vc_append_req* req,
                       int32_t residual_min, int32_t* dev_status, cudaStream_t stream) {
  if (!shape_ok(shape) || !full || !comp || !req || residual_min < 0) return VC_ERR_INVALID;
  const int B = shape->B, d = shape->d;
  AppendParams ap;
  memset(&ap, 0, sizeof(ap));
  ap.B = B;
  ap.Hkv = shape->Hkv;
  ap.d = d;
  ap.bits = 0;
  ap.dev_status = dev_status;
  int max_ext = 0, ng_new[VC_MAX_BATCH], n_win_new[VC_MAX_BATCH];
  bool any = false;
  for (int b = 0; b < B; ++b) {
    const vc_append_req& q = req[b];
    const vc_kv_full& f = full[b];
    const vc_kv_comp& c = comp[b];
    if (q.n_rows < 0) return VC_ERR_INVALID;
    if (q.n_rows > 0 && (!aligned16(q.k_rows) || !aligned16(q.v_rows))) return VC_ERR_INVALID;
    if (!aligned16(f.k) || !aligned16(f.v) || f.ctx < 1 || (int64_t)f.ctx + q.n_rows > f.cap) return VC_ERR_INVALID;
    AppendReq& r = ap.req[b];
    r.k_rows = static_cast<const bf16*>(q.k_rows);
    r.v_rows = static_cast<const bf16*>(q.v_rows);
    r.n_rows = q.n_rows;
    r.k_full = static_cast<bf16*>(const_cast<void*>(f.k));
    r.v_full = static_cast<bf16*>(const_cast<void*>(f.v));
    r.cap = f.cap;
    r.ctx = f.ctx;
    r.quant = c.mode == VC_QUANT;
    ng_new[b] = c.ng;
    n_win_new[b] = c.n_win;
    if (r.quant) {
      if (c.bits != 2 && c.bits != 4) return VC_ERR_UNSUPPORTED;
      if (ap.bits == 0) ap.bits = c.bits;
      if (c.bits != ap.bits) return VC_ERR_UNSUPPORTED;
      const int ctx2 = f.ctx + q.n_rows;
      const int ng2 = quant_blocks(ctx2, residual_min);
      const int n_res = f.ctx - VC_GROUP * c.ng, n_ext = n_res + q.n_rows;
      if (c.ng < 0 || ng2 < c.ng || ng2 > c.ng_cap || n_res < 0 || n_res > c.win_cap) return VC_ERR_INVALID;
      if (n_ext > VC_APPEND_MAX_ROWS) return VC_ERR_UNSUPPORTED;
      if (n_ext - VC_GROUP * (ng2 - c.ng) > c.win_cap) return VC_ERR_INVALID;
      if (ng2 > 0 && (!aligned16(c.kc) || !aligned16(c.ks) || !aligned16(c.kz) || !aligned16(c.vc) ||
                      !aligned16(c.vs) || !aligned16(c.vz)))
        return VC_ERR_INVALID;
      if (!aligned16(c.k_win) || !aligned16(c.v_win)) return VC_ERR_INVALID;
      r.ng = c.ng;
      r.ng_new = ng2;
      r.ng_cap = c.ng_cap;
      r.kc = c.kc;
      r.ks = reinterpret_cast<__half*>(c.ks);
      r.kz = reinterpret_cast<__half*>(c.kz);
      r.vc = c.vc;
      r.vs = reinterpret_cast<__half*>(c.vs);
      r.vz = reinterpret_cast<__half*>(c.vz);
      r.k_win = static_cast<bf16*>(c.k_win);
      r.v_win = static_cast<bf16*>(c.v_win);
      r.win_cap = c.win_cap;
      if (q.n_rows > 0 && n_ext > max_ext) max_ext = n_ext;
      ng_new[b] = ng2;
      n_win_new[b] = n_ext - VC_GROUP * (ng2 - c.ng);
    }
    any |= q.n_rows > 0;
  }
  if (!any) return VC_OK;
  if (launch_append(ap, max_ext, stream) != cudaSuccess) return VC_ERR_CUDA;
  // it rewrites KV_comp and KV_full: a draft step after it must not start before it finishes
  set_last_op(stream, kOpCompress);
  for (int b = 0; b < B; ++b) {
    full[b].ctx += req[b].n_rows;
    comp[b].ng = ng_new[b];
    comp[b].n_win = n_win_new[b];
  }
  return VC_OK;
}

// ---------------------------------------------------------------------------------------------
vc_status vc_draft_attn(const vc_shape* shape, const vc_draft_req* req, void* ws, size_t ws_bytes,
                        int32_t* dev_status, cudaStream_t stream) {
  if (!shape_ok(shape) || !req) return VC_ERR_INVALID;
  const int B = shape->B, d = shape->d, Hkv = shape->Hkv, G = shape->Hq / shape->Hkv;
  if (G > 16 || Hkv > VC_DRAFT_MAX_KV_HEADS) return VC_ERR_UNSUPPORTED;
  const int mode = req[0].comp.mode;
  const int bits = req[0].comp.bits;
  if (mode != VC_TOKEN_DROP && mode != VC_QUANT) return VC_ERR_INVALID;
  if (mode == VC_QUANT && bits != 2 && bits != 4) return VC_ERR_UNSUPPORTED;
  // main chunk: 16 kept rows, one 4-bit group, or two 2-bit groups (the draft kernel's layout)
  const int chunk = mode == VC_QUANT ? (bits == 2 ? 64 : 32) : 16;

  DraftParams p;
  memset(&p, 0, sizeof(p));
  p.B = B;
  p.Hq = shape->Hq;
  p.Hkv = Hkv;
  p.G = G;
  p.scale_log2 = (float)(1.4426950408889634 / sqrt((double)d));
  p.dev_status = dev_status;
  // VC_SPIN_LIMIT (tries; default kSpinLimit): how long a warp waits for a stage's data before it
  // records VC_DEV_TIMEOUT and leaves its range (a short limit makes the wait run out on purpose,
  // with every copy still completing; used to test the timeout path)
  const int spin = env_int("VC_SPIN_LIMIT", -1);
  p.spin_limit = spin >= 0 ? (uint32_t)spin : kSpinLimit;

  int64_t total = 0;
  for (int b = 0; b < B; ++b) {
    const vc_draft_req& q = req[b];
    const vc_kv_comp& c = q.comp;
    if (c.mode != mode || (mode == VC_QUANT && c.bits != bits)) return VC_ERR_UNSUPPORTED;
    if (!aligned16(q.q) || !aligned16(q.k_new) || !aligned16(q.v_new) || !aligned16(q.o)) return VC_ERR_INVALID;
    if (!aligned16(c.k_win) || !aligned16(c.v_win) || c.n_win < 0 || c.n_win >= c.win_cap) return VC_ERR_INVALID;
    int n_main = 0;
    if (mode == VC_TOKEN_DROP) {
      if (c.keep < 0 || (c.keep > 0 && (!aligned16(c.k_rows) || !aligned16(c.v_rows) || c.rows_cap < 1)))
        return VC_ERR_INVALID;
      if (c.keep > 0 && !c.compact && !c.idx) return VC_ERR_INVALID;
      if (c.compact && c.keep > c.rows_cap) return VC_ERR_INVALID;
      n_main = c.keep;
    } else {
      if (c.ng < 0 || c.ng > c.ng_cap) return VC_ERR_INVALID;
      if (c.ng > 0 && (!aligned16(c.kc) || !aligned16(c.ks) || !aligned16(c.kz) || !aligned16(c.vc) ||
                       !aligned16(c.vs) || !aligned16(c.vz)))
        return VC_ERR_INVALID;
      n_main = VC_GROUP * c.ng;
    }
    DraftReqDev& r = p.req[b];
    r.q = static_cast<const bf16*>(q.q);
    r.k_new = static_cast<const bf16*>(q.k_new);
    r.v_new = static_cast<const bf16*>(q.v_new);
    r.o = static_cast<bf16*>(q.o);
    r.idx = c.idx;
    r.k_rows = static_cast<const bf16*>(c.k_rows);
    r.v_rows = static_cast<const bf16*>(c.v_rows);
    r.rows_cap = c.rows_cap;
    r.n_main = n_main;
    r.compact = c.compact;
    r.kc = c.kc;
    r.ks = reinterpret_cast<const __half*>(c.ks);
    r.kz = reinterpret_cast<const __half*>(c.kz);
    r.vc = c.vc;
    r.vs = reinterpret_cast<const __half*>(c.vs);
    r.vz = reinterpret_cast<const __half*>(c.vz);
    r.ng = c.ng;
    r.ng_cap = c.ng_cap;
    r.k_win = static_cast<bf16*>(c.k_win);
    r.v_win = static_cast<bf16*>(c.v_win);
    r.win_cap = c.win_cap;
    r.n_win = c.n_win;
    r.n_mc = (n_main + chunk - 1) / chunk;
    r.n_chunks = r.n_mc + (c.n_win + 1 + 15) / 16;
    r.chunk_begin = (int32_t)total;
    total += r.n_chunks;
  }
  // token drop: tensor maps of the kept K and V rows (2-D over the Hkv * rows_cap rows of each)
  static thread_local DraftMaps maps;
  if (mode == VC_TOKEN_DROP) {
    for (int b = 0; b < B; ++b) {
      const vc_kv_comp& c = req[b].comp;
      if (c.keep <= 0) continue;
      const int64_t rows = (int64_t)Hkv * c.rows_cap;
      if (rows >= (int64_t(1) << 31)) return VC_ERR_UNSUPPORTED;
      if (!rows_tmap(&maps.kv[b][0], c.k_rows, d, rows) || !rows_tmap(&maps.kv[b][1], c.v_rows, d, rows))
        return VC_ERR_CUDA;
    }
  }
  // Warps per KV head: one wave of CTAs over the heads (and on average at least ~4 chunks per
  // warp). Each request gets a whole number of warps in proportion to its chunks, so no warp holds
  // two requests; warps left over go, a whole tier at a time, to the requests with the largest
  // chunks-per-warp load, and only while that lowers it.
  const int kind = mode == VC_TOKEN_DROP ? 0 : bits;
  int P = draft_ctas_per_head_max(Hkv, G, kind);
  const int env = env_int("VC_DRAFT_CTAS", 0);
  if (env > 0 && env / Hkv < P) P = env / Hkv > 1 ? env / Hkv : 1;
  const int64_t by_work = (total + 4 * kDraftWarps - 1) / (4 * kDraftWarps);
  if (by_work < P) P = (int)(by_work > 1 ? by_work : 1);
  const int Wmax = P * kDraftWarps;
  int kw[VC_MAX_BATCH];
  int used = 0;
  for (int b = 0; b < B; ++b) {
    const int64_t share = Wmax > B ? (int64_t)p.req[b].n_chunks * Wmax / total : 1;
    kw[b] = share > 1 ? (int)share : 1;
    used += kw[b];
  }
  for (int left = Wmax - used; left > 0;) {
    int bm = 0;  // the largest load n_b / k_b, compared exactly by cross products
    for (int b = 1; b < B; ++b)
      if ((int64_t)p.req[b].n_chunks * kw[bm] > (int64_t)p.req[bm].n_chunks * kw[b]) bm = b;
    int tier = 0;
    for (int b = 0; b < B; ++b)
      tier += (int64_t)p.req[b].n_chunks * kw[bm] == (int64_t)p.req[bm].n_chunks * kw[b];
    if (tier > left) break;
    for (int b = 0; b < B; ++b)
      if ((int64_t)p.req[b].n_chunks * kw[bm] == (int64_t)p.req[bm].n_chunks * kw[b]) ++kw[b];
    left -= tier;
  }
  int n_warp = 0;
  for (int b = 0; b < B; ++b) {
    // a warp's range edge is w * n_b / k_b with w <= k_b, computed in 32 bits
    if ((uint64_t)p.req[b].n_chunks * (uint64_t)(kw[b] + 1) >= (uint64_t(1) << 32)) return VC_ERR_UNSUPPORTED;
    p.req[b].warp_begin = n_warp;
    n_warp += kw[b];
  }
  const int n_cta = (n_warp + kDraftWarps - 1) / kDraftWarps;
  p.n_warp_head = n_warp;
  p.n_cta_head = n_cta;
  p.total_chunks = total;
  const size_t need = vc_workspace_size(VC_CALL_DRAFT, shape, 0);
  if (!ws || ws_bytes < need || !aligned16(ws)) return VC_ERR_WORKSPACE;
  p.ws_ctr = static_cast<uint32_t*>(ws);
  p.ws_o = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + draft_counter_bytes());
  p.ws_lse = p.ws_o + (size_t)Hkv * (n_cta + B) * G * d;
  p.early = last_op(stream) != kOpCompress;
  // VC_DRAFT_TC=1: quantised caches at d = 128 with up to 8 query heads per KV head on the tcgen05
  // kernel (draft_tc.cu). Same results; measured about 3x slower than the mma.sync kernel, whose
  // independent warps hide latency that the tcgen05 pipeline serialises, so it is not the default.
  const bool tc = kind != 0 && d == 128 && G <= 8 && env_int("VC_DRAFT_TC", 0) != 0;
  if (tc) {
    if (launch_draft_tc(p, kind, sm_count(), stream) != cudaSuccess) return VC_ERR_CUDA;
  } else if (launch_draft(p, &maps, d, kind, n_cta, stream) != cudaSuccess) {
    return VC_ERR_CUDA;
  }
  set_last_op(stream, kOpDraft);
  return VC_OK;
}

// ---------------------------------------------------------------------------------------------
vc_status vc_verify_attn_heads(const vc_shape* shape, const vc_verify_req* req, int32_t kv_head_begin,
                               int32_t kv_head_end, void* ws, size_t ws_bytes, int32_t* dev_status,
                               cudaStream_t stream) {
  vc_status st = VC_OK;
  cudaError_t e = launch_verify(shape, req, kv_head_begin, kv_head_end, ws, ws_bytes, dev_status, stream, &st);
  if (st != VC_OK) return st;
  if (e != cudaSuccess) return VC_ERR_CUDA;
  set_last_op(stream, kOpVerify);
  return VC_OK;
}

vc_status vc_verify_attn(const vc_shape* shape, const vc_verify_req* req, void* ws, size_t ws_bytes,
                         int32_t* dev_status, cudaStream_t stream) {
  if (!shape) return VC_ERR_INVALID;
  return vc_verify_attn_heads(shape, req, 0, shape->Hkv, ws, ws_bytes, dev_status, stream);
}

int32_t vc_verify_launches(const vc_shape* shape, const vc_verify_req* req) {
  return verify_launch_count(shape, req);
}

// ---------------------------------------------------------------------------------------------
vc_status vc_accept(int32_t B, int32_t L_max, int32_t V, const float* logits, const int32_t* draft,
                    const int32_t* L, int32_t* out_tokens, int32_t* n_acc, cudaStream_t stream) {
  if (B < 1 || L_max < 0 || V < 1 || !logits || !L || !out_tokens || !n_acc) return VC_ERR_INVALID;
  if (L_max > 0 && !draft) return VC_ERR_INVALID;
  if ((reinterpret_cast<uintptr_t>(logits) & 3u) || (reinterpret_cast<uintptr_t>(out_tokens) & 3u)) return VC_ERR_INVALID;
  AcceptArgs a{logits, draft, L, out_tokens, n_acc, B, L_max, V};
  if (launch_accept(a, stream) != cudaSuccess) return VC_ERR_CUDA;
  set_last_op(stream, kOpAccept);
  return VC_OK;
}

// ---------------------------------------------------------------------------------------------
vc_status vc_stage_full_kv(const void* host_src, void* dev_dst, size_t bytes, size_t chunk_bytes,
                           cudaStream_t copy_stream, cudaEvent_t done) {
  if (!host_src || !dev_dst) return VC_ERR_INVALID;
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, host_src) != cudaSuccess) {
    cudaGetLastError();
    return VC_ERR_NOT_PINNED;
  }
  if (at.type != cudaMemoryTypeHost) return VC_ERR_NOT_PINNED;
  cudaPointerAttributes dt;
  if (cudaPointerGetAttributes(&dt, dev_dst) != cudaSuccess) {
    cudaGetLastError();
    return VC_ERR_INVALID;
  }
  if (dt.type != cudaMemoryTypeDevice) return VC_ERR_INVALID;
  if (chunk_bytes == 0 || chunk_bytes > bytes) chunk_bytes = bytes;
  const char* s = static_cast<const char*>(host_src);
  char* dptr = static_cast<char*>(dev_dst);
  // VC_FAIL_STAGE_CHUNK=k (test hook, host side): chunk k's copy is treated as a failed
  // cudaMemcpyAsync; nothing after it is issued and `done` is not recorded
  const int fail_at = env_int("VC_FAIL_STAGE_CHUNK", -1);
  int chunk = 0;
  for (size_t off = 0; off < bytes; off += chunk_bytes, ++chunk) {
    const size_t n = bytes - off < chunk_bytes ? bytes - off : chunk_bytes;
    if (chunk == fail_at || cudaMemcpyAsync(dptr + off, s + off, n, cudaMemcpyHostToDevice, copy_stream) != cudaSuccess)
      return VC_ERR_CUDA;
  }
  if (done && cudaEventRecord(done, copy_stream) != cudaSuccess) return VC_ERR_CUDA;
  return VC_OK;
}

}  // extern "C"
