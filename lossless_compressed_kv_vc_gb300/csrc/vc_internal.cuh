// Internal declarations shared by the kernels and the C-ABI layer of libvc (sm_103a only).
#pragma once

#include <atomic>
#include <cuda.h>  // CUtensorMap (the encoder itself is fetched from the driver at run time)
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include <utility>

#include "../../include/vc.h"

#if defined(__CUDA_ARCH__) && (__CUDA_ARCH__ < 1000)
#error "libvc is written for sm_103a (Blackwell); compile with -gencode arch=compute_103a,code=sm_103a"
#endif

namespace vc {

typedef __nv_bfloat16 bf16;

// Bound on every spin-wait in a kernel: a wait that exceeds it records VC_DEV_TIMEOUT and returns.
constexpr uint32_t kSpinLimit = 1u << 22;

__device__ __forceinline__ void set_status(int32_t* st, int32_t code) {
  if (st) atomicCAS(st, 0, code);
}

// ---- shared-memory addressing, mbarrier and bulk-copy (TMA engine) wrappers -------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait: returns false (after recording VC_DEV_TIMEOUT) if the phase does not complete
// within `limit` tries.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, int32_t* st,
                                                  uint32_t limit = kSpinLimit) {
  for (uint32_t it = 0; it < limit; ++it)
    if (mbar_try_wait(bar, parity)) return true;
  set_status(st, VC_DEV_TIMEOUT);
  return false;
}

// 1-D bulk copy global -> shared through the TMA engine, completing on an mbarrier.
__device__ __forceinline__ void bulk_g2s(void* dst_smem, const void* src_gmem, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst_smem)),
      "l"(src_gmem), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// L2 policy for data a kernel reads once while streaming far more than the L2 holds: evict it
// first, so that small data written and read back within the launch (split partials) stays.
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// Four whole rows of a 2-D tensor map (box 64 elements x 1 row) gathered by row coordinate into
// four consecutive 128-byte rows of shared memory starting at dst, in the map's swizzle; c0 is the
// first element of the 64-element column block (a multiple of 64 here, so the 16-byte rule holds).
// `pol` is an L2 cache policy (l2_evict_first_policy).
__device__ __forceinline__ void tma_gather4(void* dst, const void* tmap, int c0, int r0, int r1, int r2, int r3,
                                            uint64_t* bar, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cta.global.tile::gather4.mbarrier::complete_tx::bytes.L2::cache_hint [%0], "
      "[%1, {%2, %3, %4, %5, %6}], [%7], %8;" ::"r"(smem_u32(dst)),
      "l"(tmap), "r"(c0), "r"(r0), "r"(r1), "r"(r2), "r"(r3), "r"(smem_u32(bar)), "l"(pol)
      : "memory");
}

// 1-D bulk copy global -> shared with an L2 cache policy, completing on an mbarrier.
__device__ __forceinline__ void bulk_g2s_hint(void* dst_smem, const void* src_gmem, uint32_t bytes, uint64_t* bar,
                                              uint64_t pol) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          smem_u32(dst_smem)),
      "l"(src_gmem), "r"(bytes), "r"(smem_u32(bar)), "l"(pol)
      : "memory");
}

// 16-byte asynchronous global -> shared copy (L2 only); src_bytes = 0 fills the 16 bytes with zeros.
__device__ __forceinline__ void cp_async16(void* dst_smem, const void* src_gmem, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst_smem)), "l"(src_gmem),
               "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// ---- warp-level tensor-core helpers (mma.sync m16n8k16) -----------------------------------------
__device__ __forceinline__ void ldsm_x4(uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3, const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(smem_u32(p)));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3, const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(smem_u32(p)));
}

__device__ __forceinline__ void mma_bf16_16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void mma_f16_16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// 2^x with the SFU's approximate exp2 (relative error about 2^-22); subnormal results flush to
// zero, which is harmless for softmax weights (arguments are <= 0).
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Packed f32x2 arithmetic (two independent fp32 lanes per instruction, each rounded as its scalar
// form) and a three-input maximum, for the softmax and accumulator updates of the attention kernels.
__device__ __forceinline__ uint64_t f2_pack(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t v, float& a, float& b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ float max3f(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// ---- launch helpers ---------------------------------------------------------------------------------
// Raise a kernel's dynamic shared-memory limit on the current device, once per device (the
// attribute belongs to the device's context, so a process driving several GPUs sets it on each).
template <typename Kernel>
inline cudaError_t raise_smem_limit(Kernel kernel, int bytes, std::atomic<uint64_t>& devices_done) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = dev < 64 ? (uint64_t(1) << dev) : 0;
  if (bit && (devices_done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && bit) devices_done.fetch_or(bit, std::memory_order_acq_rel);
  return e;
}

// ---- programmatic dependent launch ----------------------------------------------------------------
// Every kernel of the round is launched with programmatic stream serialisation: it lets the next
// kernel in the stream start launching once all of its CTAs are running, and waits for the
// previous kernel's results (grid completion and memory flush) before touching any global data.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" :::); }

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                              Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// ---- per-request kernel descriptors (travel by value in kernel params) -------------------------
struct DraftReqDev {
  const bf16* q;
  const bf16* k_new;
  const bf16* v_new;
  bf16* o;
  // main rows
  const int32_t* idx;
  const bf16* k_rows;
  const bf16* v_rows;
  int64_t rows_cap;
  int32_t n_main;      // kept rows (drop) or 32*ng (quant)
  int32_t compact;
  const uint8_t* kc;
  const __half* ks;
  const __half* kz;
  const uint8_t* vc;
  const __half* vs;
  const __half* vz;
  int32_t ng;
  int32_t ng_cap;       // head stride of the quantised buffers, in blocks
  // window
  bf16* k_win;
  bf16* v_win;
  int64_t win_cap;
  int32_t n_win;
  // chunk plan: n_mc chunks of KV_comp rows, then ceil((n_win + 1) / 16) window chunks
  int32_t chunk_begin;  // first chunk of this request in the per-head concatenation
  int32_t n_mc;
  int32_t n_chunks;
  int32_t warp_begin;   // first warp (of a head's grid row) holding it; it holds them up to the next request's
  // unit plan of the tcgen05 quantised kernel (draft_tc.cu): tc_nqb blocks of four groups (cost 1
  // each), then tc_nwb window blocks of 128 rows (cost WW each), from cost tc_ucb of the head's
  // concatenation; CTAs tc_c0 .. tc_c1 of the grid row hold its units
  int64_t tc_ucb;
  int32_t tc_nqb, tc_nwb, tc_c0, tc_c1;
};

// The observation-window passes of the SnapKV-style importance, run by the verification kernel's
// row-statistics and column-sum modes (verify.cu).
struct ObsReq {
  const bf16* k;   // KV_full keys [Hkv][cap][d]
  const bf16* q;   // window queries [W][Hq][d]
  int32_t ctx, cap;
  float* lse;      // [Hkv][mtiles * 128] window rows' log-sum-exp (exp2 domain)
  float* votes;    // [Hkv * mtiles][ctx] per-tile column sums
};
struct ObsArgs {
  ObsReq req[VC_MAX_BATCH];
  int32_t B, Hq, Hkv, d, W;
  float* ws_lse;   // split-unit partials
  size_t ws_lse_floats;
  int32_t* dev_status;
};
int obs_mtiles(int W, int G);
size_t obs_slot_floats(int B, int Hkv, int mtiles);
cudaError_t launch_obs_passes(const ObsArgs& a, cudaStream_t s);

struct DraftParams {
  DraftReqDev req[VC_MAX_BATCH];
  int32_t B, Hq, Hkv, G;
  float scale_log2;      // log2(e) / sqrt(d)
  float* ws_o;           // [Hkv][n_cta_head + B][G][d] per-CTA partials (slot = CTA + request)
  float* ws_lse;         // [Hkv][n_cta_head + B][G]  (log2 domain)
  uint32_t* ws_ctr;      // [Hkv][VC_MAX_BATCH] CTA-partial arrival counts (zero between calls)
  int32_t n_cta_head;    // CTAs per KV head (grid.x)
  int32_t n_warp_head;   // warps per KV head that hold work (the last CTA may hold fewer)
  int64_t total_chunks;  // chunks per KV head over all requests
  int32_t* dev_status;
  // tries of a warp's wait for a stage's data before it gives up (VC_DEV_TIMEOUT); its drain of the
  // copies still in flight then waits with the full kSpinLimit
  uint32_t spin_limit;
  // 1: the kernel may stream queries, kept rows and indices before the previous kernel in the
  // stream has finished (set when that kernel is not a compress); it waits for it before reading
  // window rows, storing the step's row and writing any output.
  int32_t early;
  int64_t tc_total;      // tcgen05 quantised kernel: unit cost per KV head over all requests
};

// Tensor maps of the kept K and V rows of each request (token drop): 2-D (d, Hkv * rows_cap) over
// the bf16 rows, box 64 x 1, 128-byte swizzle. A separate kernel argument: the kernels for
// quantised caches take none.
struct DraftMaps {
  CUtensorMap kv[VC_MAX_BATCH][2];
};

constexpr int kDraftWarps = 4;

// launchers (return cudaError_t of the launch); maps is read for token drop only
cudaError_t launch_draft(const DraftParams& p, const DraftMaps* maps, int d, int mode_kind, int ctas_per_head,
                         cudaStream_t s);
// quantised caches at d = 128 with at most 8 query heads per KV head on the tcgen05 kernel: one CTA
// per SM, draft_tc_ctas_per_head(Hkv) per KV head; fills in its own unit plan and CTA partial slots
cudaError_t launch_draft_tc(const DraftParams& p, int kind, int sm_count, cudaStream_t s);
int draft_tc_ctas_per_head(int Hkv, int sm_count);

// ---- host: TMA tensor maps --------------------------------------------------------------------------
// cuTensorMapEncodeTiled from the driver (fetched once through the runtime), or nullptr.
void* tmap_encoder();
// 2-D map over `rows` bf16 rows of d elements (row pitch d * 2 bytes): box 64 x 1, 128-byte swizzle,
// for tile::gather4. Maps are cached per (base, rows, d). False if the encoder is unavailable or
// rejects the layout.
bool rows_tmap(CUtensorMap* out, const void* base, int d, int64_t rows);

struct AcceptArgs {
  const float* logits;
  const int32_t* draft;
  const int32_t* L;
  int32_t* out_tokens;
  int32_t* n_acc;
  int32_t B, L_max, V;
};
cudaError_t launch_accept(const AcceptArgs& a, cudaStream_t s);

struct KeepReq {
  const float* imp;
  int32_t* idx;
  int32_t ctx, keep, recent;
  // compaction (optional)
  const bf16* k_src;
  const bf16* v_src;
  int64_t src_cap;
  bf16* k_dst;
  bf16* v_dst;
  int64_t dst_cap;
  int32_t compact;
};
struct KeepParams {
  KeepReq req[VC_MAX_BATCH];
  int32_t B, Hkv, d;
  int32_t* dev_status;
};
cudaError_t launch_keepset(const KeepParams& p, int max_keep, cudaStream_t s);

struct QuantReq {
  const bf16* k;
  const bf16* v;
  int64_t cap;
  int32_t ctx, ng, n_res;
  int32_t ng_cap;  // head stride of the quantised buffers, in blocks
  uint8_t* kc;
  __half* ks;
  __half* kz;
  uint8_t* vc;
  __half* vs;
  __half* vz;
  bf16* k_win;
  bf16* v_win;
  int64_t win_cap;
};
struct QuantParams {
  QuantReq req[VC_MAX_BATCH];
  int32_t B, Hkv, d, bits;
  int32_t* dev_status;
};
cudaError_t launch_quant(const QuantParams& p, int max_ng, int max_tq, cudaStream_t s);

// Append accepted drafted rows to KV_full and, for quantised caches, quantise the blocks that
// became whole and rewrite the residual window (one CTA per request and KV head).
struct AppendReq {
  const bf16* k_rows;  // [n_rows][Hkv][d]
  const bf16* v_rows;
  int32_t n_rows;
  bf16* k_full;        // [Hkv][cap][d]
  bf16* v_full;
  int64_t cap;
  int32_t ctx;         // before the append
  int32_t quant;       // 1: VC_QUANT request
  int32_t ng, ng_new;  // quantised blocks before / after
  int32_t ng_cap;
  uint8_t* kc;
  __half* ks;
  __half* kz;
  uint8_t* vc;
  __half* vs;
  __half* vz;
  bf16* k_win;
  bf16* v_win;
  int64_t win_cap;
};
struct AppendParams {
  AppendReq req[VC_MAX_BATCH];
  int32_t B, Hkv, d, bits;
  int32_t* dev_status;
};
cudaError_t launch_append(const AppendParams& p, int max_ext_rows, cudaStream_t s);

}  // namespace vc
