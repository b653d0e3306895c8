/*
 * vc.h — C ABI of the VeriCache draft-then-verify hot path on one GB300 (sm_103a).
 *
 * The loop this library runs is the one stated in "VeriCache: Turning Lossy KV Cache into
 * Lossless LLM Inference", section "Core algorithm":
 *   1. draft: the target model decodes candidate tokens x with the compressed cache KV_comp;
 *   2. verify: one forward pass over the full cache KV_full checks all drafts in parallel;
 *   3. accept: tokens are accepted up to the first mismatch, plus one "bonus" token when every
 *      draft matches; the next round restarts from the last accepted token.
 * Section "Architecture support" adds the long-context scenario (KV_comp in GPU HBM, KV_full in
 * CPU memory, loaded over the host link for each verification) and a single compressor
 * interface for token-drop and quantising compressors. Section "Cross-resource staggering (P1)"
 * overlaps the host-link copy of some requests with the drafting of others.
 *
 * One attention layer is covered: compress (vc_compress_kv), draft attention (vc_draft_attn),
 * verify attention (vc_verify_attn, vc_verify_attn_heads), greedy accept (vc_accept), full-KV
 * staging (vc_stage_full_kv) and the post-accept cache update (vc_append_kv). Every compute step
 * runs in this library's CUDA kernels.
 *
 * Conventions for every call
 *   - The caller owns every buffer. The library never allocates device or host memory and never
 *     synchronises a stream. Device pointers must be 16-byte aligned.
 *   - bf16 tensors are stored as raw 16-bit words (`void*`); fp16 scales/zeros as uint16_t.
 *   - Host-side validation returns a status and launches nothing when it fails.
 *   - `dev_status` (may be NULL) is a device int32 the kernels set to a VC_DEV_* code when they
 *     detect a problem they can survive (an index outside its buffer is skipped, a bounded wait
 *     gives up); the first code written wins. The caller reads it when convenient.
 *   - Calls are asynchronous on `stream`; a call returns before its kernels finish.
 *   - At most VC_MAX_BATCH requests per call (per-request descriptors travel as kernel params).
 *   - Head dim d is 64 or 128; Hq is a multiple of Hkv; query head h reads KV head h / (Hq/Hkv).
 *   - Every wait inside a kernel is bounded; one that gives up records VC_DEV_TIMEOUT, waits (with
 *     the full bound) for the copies it has already issued, and returns. The environment variable
 *     VC_SPIN_LIMIT (read by each vc_draft_attn call) sets how many tries a draft warp's wait for its
 *     next stage of data makes before it gives up (default 4194304; 0 gives up at once): a short
 *     limit makes that wait run out without any fault, which is how its error path is tested.
 *   - Kernel choices read from the environment by each call, with the same results either way:
 *     VC_DRAFT_TC=1 runs vc_draft_attn for quantised caches at d = 128 with at most 8 query heads
 *     per KV head on the tcgen05 draft kernel (the mma.sync kernel is the default and faster);
 *     a (request, KV head) whose drafts fill two 128-row tiles (129 to 256 rows) is verified by one
 *     CTA that reads its KV_full once for both tiles, and VC_VERIFY_PAIR=0 gives each of those
 *     tiles a unit of its own instead; a head of one tile, or of three or more, has a unit per
 *     tile, each of which reads KV_full; VC_VERIFY_TRIO=1 verifies a head of exactly three tiles
 *     in one CTA with two softmax warpgroups, reading KV_full once (slower at present);
 *     VC_VERIFY_ROWS=1 verifies every tile of every head in one CTA per head with one softmax
 *     warpgroup, reading KV_full once (slower still).
 */
#ifndef VC_H_
#define VC_H_

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime.h>

#ifdef __cplusplus
extern "C" {
#endif

#define VC_MAX_BATCH 32
#define VC_GROUP 32            /* quantisation group size (tokens per key group, channels per value group) */

typedef enum vc_status {
  VC_OK = 0,
  VC_ERR_INVALID = 1,      /* null pointer, bad size, misaligned buffer, inconsistent descriptor */
  VC_ERR_UNSUPPORTED = 2,  /* well-formed but outside what the kernels implement (d, bits, G) */
  VC_ERR_CUDA = 3,         /* a CUDA runtime call or launch failed */
  VC_ERR_NOT_PINNED = 4,   /* a host source for staging is not page-locked */
  VC_ERR_WORKSPACE = 5     /* workspace smaller than vc_workspace_size() */
} vc_status;

/* Codes the kernels write into *dev_status. */
#define VC_DEV_OK 0
#define VC_DEV_BOUNDS 1        /* a gather index fell outside its buffer; the row was skipped */
#define VC_DEV_TIMEOUT 2       /* a bounded wait on a copy gave up; outputs of that block are invalid */
#define VC_DEV_RANGE 3         /* a quantisation scale or zero is not finite in fp16 */
#define VC_DEV_INTERNAL 4      /* a kernel precondition failed (shared-memory alignment); outputs invalid */

typedef enum vc_mode { VC_TOKEN_DROP = 0, VC_QUANT = 1 } vc_mode;
typedef enum vc_call { VC_CALL_DRAFT = 0, VC_CALL_VERIFY = 1 } vc_call;

typedef struct vc_shape {
  int32_t B;     /* requests in this call, 1..VC_MAX_BATCH */
  int32_t Hq;    /* query heads */
  int32_t Hkv;   /* KV heads */
  int32_t d;     /* head dim: 64 or 128 */
} vc_shape;

/* One request's full-precision cache KV_full, resident in device memory (HBM, or a staging
 * buffer filled by vc_stage_full_kv). Rows 0..ctx-1 are valid. */
typedef struct vc_kv_full {
  const void* k;     /* bf16 [Hkv][cap][d], head h row t at (h*cap + t)*d */
  const void* v;     /* bf16 [Hkv][cap][d] */
  int32_t ctx;       /* tokens held */
  int32_t cap;       /* rows per head, cap >= ctx */
} vc_kv_full;

/* One request's compressed cache KV_comp (device memory). Two families share it:
 *
 * VC_TOKEN_DROP: a keep-set of `keep` token indices `idx` (ascending). With compact == 0 the
 *   kept rows are read in place at k_rows[h][idx[j]] (k_rows is normally the full cache); with
 *   compact == 1 vc_compress_kv gathers them into k_rows[h][j], j < keep, and the draft reads them
 *   contiguously (needed when KV_full leaves HBM).
 * VC_QUANT: groupwise asymmetric `bits`-bit codes for the first Tq = 32*ng tokens, in blocks of 32
 *   tokens (keys: one scale/zero per (block, channel); values: per (token, 32-channel group)),
 *   in buffers sized for ng_cap >= ng blocks (the head stride, so blocks can be appended):
 *   kc  uint8 [Hkv][ng_cap][32*d*bits/8]   key codes of each block, in block word order (below)
 *   ks,kz fp16 [Hkv][ng_cap][d]            key scale and zero per (block, channel)
 *   vc  uint8 [Hkv][ng_cap][32*d*bits/8]   value codes of each block, in block word order
 *   vs,vz fp16 [Hkv][32*ng_cap][d/32]      value scale and zero per (token, 32-channel group)
 *   Dequantised value: code * scale + zero.
 *   Block word order: little-endian 32-bit words w[half][j][lane] (4-bit; half = 16-token half,
 *   j = 16-channel step, lane = 0..31) or w[half][p][lane] (2-bit, p covers j = 2p, 2p+1). With
 *   a = lane/4, b = lane%4, word (half, j, lane) holds pairs i = 0..3 of (token, channel):
 *     keys   (t0 = 16 half + a, c0 = 16 j + 2b): (t0, c0|c0+1), (t0+8, c0|c0+1),
 *                                              (t0, c0+8|c0+9), (t0+8, c0+8|c0+9)
 *     values (r0 = 16 j + a, k0 = 16 half + 2b): (k0|k0+1, r0), (k0|k0+1, r0+8),
 *                                              (k0+8|k0+9, r0), (k0+8|k0+9, r0+8)
 *   pair i' (i' = i, or i + 4(j - 2p) at 2-bit) has its first code at bit bits*i' and its second
 *   at bit 16 + bits*i': each lane's word is its tensor-core operand fragment for that tile.
 *
 * Both families end with a bf16 window k_win/v_win [Hkv][win_cap][d]: for VC_QUANT it starts
 * with the n_res trailing tokens kept in bf16 (the residual), then — for both — the drafted
 * tokens' own K/V, one row per draft step. `n_win` counts the rows present before a draft step;
 * the caller increases it by one after each vc_draft_attn. */
typedef struct vc_kv_comp {
  int32_t mode;        /* vc_mode */
  int32_t bits;        /* VC_QUANT: 2 or 4 */
  /* VC_TOKEN_DROP */
  int32_t keep;        /* kept rows */
  int32_t compact;     /* 0: rows in place at idx; 1: rows gathered contiguously */
  int32_t* idx;        /* int32 [keep] ascending token indices (written by vc_compress_kv) */
  void* k_rows;        /* bf16 [Hkv][rows_cap][d] */
  void* v_rows;
  int32_t rows_cap;    /* rows per head of k_rows/v_rows (indices must be < rows_cap) */
  /* VC_QUANT */
  int32_t ng;          /* quantised 32-token groups (set by vc_compress_kv) */
  uint8_t* kc;
  uint16_t* ks;
  uint16_t* kz;
  uint8_t* vc;
  uint16_t* vs;
  uint16_t* vz;
  /* bf16 window (both) */
  void* k_win;         /* bf16 [Hkv][win_cap][d] */
  void* v_win;
  int32_t win_cap;
  int32_t n_win;       /* rows present before this draft step (set to n_res / 0 by vc_compress_kv) */
  int32_t ng_cap;      /* VC_QUANT: blocks the quantised buffers hold per head (>= ng) */
} vc_kv_comp;

/* ------------------------------------------------------------------------------------------ */
/* vc_comp_bytes — the buffers one request's KV_comp needs, by the rules vc_compress_kv,
 * vc_draft_attn and vc_append_kv follow ("Architecture support": one compressor interface), so a
 * caller sizes them without restating those rules.
 *
 * VC_QUANT: ng = max(0, (ctx - residual_min) / 32) blocks are quantised and n_res = ctx - 32 ng
 * rows stay bf16; ng_cap = the blocks of a context grown to max_ctx (at least 1), the head stride of
 * kc/ks/kz/vc/vs/vz. VC_TOKEN_DROP: keep = min(keep, ctx) kept rows (idx; k_rows/v_rows when
 * compact). Both: win_cap = the largest residual over contexts ctx .. max_ctx (0 for token drop)
 * plus max_drafts + 1 window rows. Byte counts are for one buffer each (k and v alike).
 * Errors: VC_ERR_INVALID (null pointers, a bad shape, ctx < 1, max_ctx < ctx, negative keep,
 * residual_min or max_drafts); VC_ERR_UNSUPPORTED (bits not 2 or 4 for VC_QUANT). Host only. */
typedef struct vc_comp_sizes {
  int32_t ng;            /* VC_QUANT: quantised 32-token blocks at ctx tokens */
  int32_t n_res;         /* VC_QUANT: bf16 residual rows at ctx tokens (window rows 0..n_res-1) */
  int32_t ng_cap;        /* VC_QUANT: blocks to allocate per head (>= ng, >= 1) */
  int32_t win_cap;       /* window rows to allocate per head */
  int32_t keep;          /* VC_TOKEN_DROP: kept rows */
  int32_t pad_;
  size_t idx_bytes;      /* VC_TOKEN_DROP: int32 [keep] (at least 4) */
  size_t rows_bytes;     /* VC_TOKEN_DROP, compact: each of k_rows, v_rows, bf16 [Hkv][keep][d] */
  size_t codes_bytes;    /* VC_QUANT: each of kc, vc, uint8 [Hkv][ng_cap][32*d*bits/8] */
  size_t kscale_bytes;   /* VC_QUANT: each of ks, kz, fp16 [Hkv][ng_cap][d] */
  size_t vscale_bytes;   /* VC_QUANT: each of vs, vz, fp16 [Hkv][32*ng_cap][d/32] */
  size_t win_bytes;      /* each of k_win, v_win, bf16 [Hkv][win_cap][d] */
} vc_comp_sizes;

vc_status vc_comp_bytes(const vc_shape* shape, int32_t mode, int32_t bits, int32_t ctx, int32_t max_ctx,
                        int32_t keep, int32_t residual_min, int32_t max_drafts, vc_comp_sizes* out);

/* ------------------------------------------------------------------------------------------ */
/* vc_compress_kv — build KV_comp from KV_full ("Architecture support": one compressor interface
 * for token drop and quantisation).
 *
 * Per request b (all requests of a call use one mode):
 *   VC_TOKEN_DROP: idx = the `recent` last tokens plus the keep-recent tokens of [0, ctx-recent)
 *     with the largest importance (fp32 order, -0 == +0, ties to the lower index), ascending.
 *     keep >= ctx keeps every token. With compact == 1 the kept rows are gathered into k_rows.
 *     Sets n_win = 0.
 *   VC_QUANT: ng = max(0, (ctx - residual_min) / 32) groups are quantised (fp32 min/max, scale =
 *     fp16(fp32(max-min)/(2^bits-1)), zero = fp16(min), code = clamp(rint((x - zero)/scale))
 *     with IEEE round-to-nearest-even, code 0 when scale == 0); the n_res = ctx - 32*ng
 *     trailing tokens are copied to window rows 0..n_res-1. Sets ng and n_win = n_res.
 * importance: host array of B device pointers to fp32 [ctx] (token drop; NULL for quant).
 * recent: host int32 [B] (token drop; NULL for quant). residual_min: trailing bf16 tokens (128).
 * comp: host array of B descriptors; mode, bits/keep/compact and the buffers are inputs, ng and
 *   n_win are written. Requirements: 0 <= recent <= keep; window capacity >= n_res (+ drafts).
 */
vc_status vc_compress_kv(const vc_shape* shape, const vc_kv_full* full, const float* const* importance,
                         const int32_t* recent, int32_t residual_min, vc_kv_comp* comp,
                         int32_t* dev_status, cudaStream_t stream);

/* ------------------------------------------------------------------------------------------ */
/* vc_append_kv — after accept, grow the caches by the accepted drafted tokens ("Core algorithm":
 * the loop restarts from the last accepted token, so the tokens before it are now context).
 *
 * For each request b the first n_rows rows of k_rows/v_rows (the drafted tokens' K/V, in draft
 * order; n_rows = n_acc - 1, the accepted drafts without the bonus/correction token, whose K/V the
 * next forward pass produces) become KV_full rows ctx .. ctx+n_rows-1 and full[b].ctx grows by
 * n_rows. VC_QUANT requests also grow KV_comp: with ctx' = ctx + n_rows, ng' = max(0, (ctx' -
 * residual_min) / 32) blocks are kept quantised; the ng' - ng blocks that became whole are
 * quantised from the residual and the new rows exactly as vc_compress_kv would (same rule, same
 * words), and the window restarts with the n_res' = ctx' - 32*ng' trailing tokens; comp[b].ng and
 * comp[b].n_win are updated. The state equals vc_compress_kv of the grown KV_full. VC_TOKEN_DROP
 * requests keep their keep-set until the next vc_compress_kv.
 * Requirements: ctx + n_rows <= full[b].cap; VC_QUANT: ng' <= ng_cap, the residual plus n_rows
 * at most VC_APPEND_MAX_ROWS rows. Returns VC_ERR_INVALID / VC_ERR_UNSUPPORTED before launching
 * anything when a requirement fails. */
#define VC_APPEND_MAX_ROWS 256

typedef struct vc_append_req {
  const void* k_rows;  /* bf16 [>= n_rows][Hkv][d]: the accepted drafts' keys (as the verification
                          pass computed them), in draft order; not inside this request's window */
  const void* v_rows;  /* bf16 [>= n_rows][Hkv][d] */
  int32_t n_rows;      /* rows to append (>= 0) */
} vc_append_req;

vc_status vc_append_kv(const vc_shape* shape, vc_kv_full* full, vc_kv_comp* comp, const vc_append_req* req,
                       int32_t residual_min, int32_t* dev_status, cudaStream_t stream);

/* ------------------------------------------------------------------------------------------ */
/* vc_draft_attn — one draft decode step for B requests ("Core algorithm", step 1: drafting with
 * KV_comp; "Cross-resource staggering (P1)": drafting is bound by HBM bandwidth).
 *
 * For each request and query head h: o = softmax(q K^T / sqrt(d)) V over the rows of KV_comp
 * (kept rows, or dequantised groups) followed by window rows 0..n_win, where window row n_win is
 * (k_new, v_new). The call also stores k_new/v_new into window row n_win (needs n_win < win_cap).
 * Accumulation is fp32; the output is rounded to bf16.
 * ws: a workspace of at least vc_workspace_size(VC_CALL_DRAFT, shape, 0) bytes whose first
 * VC_DRAFT_COUNTER_BYTES were zero-filled once (see vc_workspace_size). Hkv <= VC_DRAFT_MAX_KV_HEADS
 * and Hq/Hkv <= 16 (VC_ERR_UNSUPPORTED otherwise).
 */
#define VC_DRAFT_MAX_KV_HEADS 256                                   /* Hkv limit of a draft call */
#define VC_DRAFT_COUNTER_BYTES ((size_t)VC_DRAFT_MAX_KV_HEADS * VC_MAX_BATCH * 4)  /* 32 KiB */

typedef struct vc_draft_req {
  const void* q;       /* bf16 [Hq][d]: query of the token drafted at this step */
  const void* k_new;   /* bf16 [Hkv][d]: its key */
  const void* v_new;   /* bf16 [Hkv][d]: its value */
  void* o;             /* bf16 [Hq][d] output */
  vc_kv_comp comp;     /* the request's compressed cache */
} vc_draft_req;

vc_status vc_draft_attn(const vc_shape* shape, const vc_draft_req* req, void* ws, size_t ws_bytes,
                        int32_t* dev_status, cudaStream_t stream);

/* ------------------------------------------------------------------------------------------ */
/* vc_draft_attn_noalloc — vc_draft_attn without a caller workspace. The paper has no counterpart:
 * this is a library convenience for callers that cannot allocate device memory, for example a
 * plugin whose host application owns every device allocation and gives it no allocator, or a
 * serving loop that must not call cudaMalloc/cudaFree (those can synchronise the whole device).
 *
 * Same arguments and results as vc_draft_attn, minus ws/ws_bytes. The partials live in a fixed
 * array of VC_DRAFT_NOALLOC_SCRATCH_BYTES compiled into the library; every GPU that loads the
 * library holds it until the process exits. The first call made with a given device current looks
 * up the array's device address (cudaGetSymbolAddress), zero-fills the array on `stream` and
 * caches the address: make that first call before any stream capture. The call allocates nothing.
 * Returns VC_ERR_WORKSPACE when the call needs more scratch than the array holds
 * (vc_workspace_size(VC_CALL_DRAFT, shape, 0) > the limit). All calls share the array, which keeps
 * the last call's contents: its arrival counters (the first VC_DRAFT_COUNTER_BYTES, at the same
 * place for every shape) start at zero and every call leaves them at zero, and the partials after
 * them are written before they are read, so calls of different shapes may follow one another.
 * Calls that overlap on the GPU race on the array, so issue them on one stream or order them with
 * events. */
#define VC_DRAFT_NOALLOC_SCRATCH_BYTES ((size_t)32 << 20)

vc_status vc_draft_attn_noalloc(const vc_shape* shape, const vc_draft_req* req, int32_t* dev_status,
                                cudaStream_t stream);

/* ------------------------------------------------------------------------------------------ */
/* vc_verify_attn — verification attention, all drafts of a request in one pass ("Core
 * algorithm", step 2: one forward pass over KV_full).
 *
 * Query row i of a request (0 <= i < n_rows, position ctx+i) and head h attend to KV_full rows
 * 0..ctx-1 and to the drafted tokens' rows 0..i (causal among the drafts), scale 1/sqrt(d).
 * Runs the rows of one KV head (n_rows * Hq/Hkv of them) as dense tensor-core tiles.
 */
typedef struct vc_verify_req {
  vc_kv_full full;     /* KV_full in device memory */
  const void* q;       /* bf16 [n_rows][Hq][d] */
  const void* k_new;   /* bf16 [Hkv][new_cap][d], rows 0..n_rows-1: the drafted tokens' keys */
  const void* v_new;
  int32_t new_cap;     /* rows per head of k_new/v_new */
  int32_t n_rows;      /* drafted tokens to verify, >= 1 */
  void* o;             /* bf16 [n_rows][Hq][d] output */
} vc_verify_req;

vc_status vc_verify_attn(const vc_shape* shape, const vc_verify_req* req, void* ws, size_t ws_bytes,
                         int32_t* dev_status, cudaStream_t stream);

/* vc_verify_attn_heads — vc_verify_attn restricted to the query heads of KV heads
 * kv_head_begin .. kv_head_end-1 (0 <= begin < end <= Hkv); outputs of the other heads are not
 * written, and only those KV heads' rows of KV_full, k_new and v_new are read.
 *
 * For chunk-pipelined staging ("Cross-resource staggering (P1)": the host-link copy of KV_full
 * overlaps work on the GPU; here the copy also overlaps the verification itself): KV_full is
 * [Hkv][cap][d], so one KV head's K (and V) rows are one contiguous range. A caller copies KV_full
 * a head range at a time, records an event per range, and verifies each range as soon as its
 * event completes; only the last range's verification remains after the copy ends.
 * Same arguments, workspace (vc_workspace_size(VC_CALL_VERIFY, ...) covers every range) and
 * errors as vc_verify_attn; a bad head range returns VC_ERR_INVALID before launching anything.
 * Calls issued in order on one stream may share one workspace. */
vc_status vc_verify_attn_heads(const vc_shape* shape, const vc_verify_req* req, int32_t kv_head_begin,
                               int32_t kv_head_end, void* ws, size_t ws_bytes, int32_t* dev_status,
                               cudaStream_t stream);

/* vc_verify_launches — how many kernels one vc_verify_attn call (and each vc_verify_attn_heads
 * call) launches for these requests: two (the verification kernel and the merge of heads split
 * across CTAs) per kind of launch the requests need, by their KV heads' 128-row tiles (one tile,
 * two, three in trio mode) and the environment switches described at the top of this file, as
 * they are set when this is called. Host only: reads shape and each request's n_rows, new_cap and
 * pointers' alignment, no device memory. Returns -1 for arguments vc_verify_attn would refuse. */
int32_t vc_verify_launches(const vc_shape* shape, const vc_verify_req* req);

/* ------------------------------------------------------------------------------------------ */
/* vc_accept — greedy acceptance ("Core algorithm", step 3).
 *
 * logits: fp32 [B][L_max+1][V]; row i of request b is the full-cache prediction after its i-th
 *   verified input (row 0 follows the last accepted token, row i follows draft i-1).
 * draft: int32 [B][L_max]; L: device int32 [B], 0 <= L[b] <= L_max (a value outside that range is
 * clamped to it on the device, so no row outside request b's is read).
 * a_i = argmax of row i (first maximal index; logits must be finite); n = first i < L[b] with
 * a_i != draft[i], else L[b]. Writes out_tokens[b] = draft[0..n-1], a_n, then -1 up to L_max+1
 * entries, and n_acc[b] = n + 1 (1..L[b]+1).
 */
vc_status vc_accept(int32_t B, int32_t L_max, int32_t V, const float* logits, const int32_t* draft,
                    const int32_t* L, int32_t* out_tokens, int32_t* n_acc, cudaStream_t stream);

/* ------------------------------------------------------------------------------------------ */
/* vc_stage_full_kv — copy a request's KV_full from page-locked host memory into device memory
 * ("Architecture support", long-context decoding: KV_full lives in CPU memory and is loaded over
 * the host link for verification; "Cross-resource staggering (P1)": the copy overlaps other
 * requests' drafting).
 *
 * Issues cudaMemcpyAsync host-to-device copies of `chunk_bytes` (0 = one copy) on copy_stream and
 * records `done` (may be NULL) on it after the last chunk; the caller makes the verifying stream
 * wait on `done`. host_src must be page-locked (VC_ERR_NOT_PINNED otherwise). A copy that cannot be
 * issued returns VC_ERR_CUDA: the chunks before it are in flight, none after it is issued and `done`
 * is not recorded. Test hook: with the environment variable VC_FAIL_STAGE_CHUNK=k the call treats
 * chunk k (0-based) as such a failed copy.
 */
vc_status vc_stage_full_kv(const void* host_src, void* dev_dst, size_t bytes, size_t chunk_bytes,
                           cudaStream_t copy_stream, cudaEvent_t done);

/* ------------------------------------------------------------------------------------------ */
/* vc_snapkv_importance — token importance for the keep-set of a token-drop request, SnapKV style
 * ("Architecture support": SnapKV is one of the token-drop compressors behind the compressor
 * interface; the pages name it without defining its scoring, so this is a plain reading of it).
 *
 * The last `window` = W context tokens form the observation window; their queries q_obs attend,
 * causally, to the keys of KV_full (window query i sits at position ctx - W + i and sees keys
 * 0 .. ctx - W + i), scale 1/sqrt(d), GQA as in the other calls. The vote of key t is the sum of
 * its softmax weights over the W queries and all Hq query heads; importance[t] pools the votes over
 * |u - t| <= pool_kernel / 2: VC_POOL_MAX takes the largest in-range vote, VC_POOL_AVG the sum of
 * the in-range votes divided by pool_kernel (zero padding). pool_kernel = 1 leaves the votes as
 * they are. The result feeds vc_compress_kv's importance (any scale: only the order matters).
 * Arithmetic: bf16 products accumulated in fp32 on the tensor cores, softmax in fp32 (exp2 domain),
 * each key's sum over 128 window rows of the fp16-rounded weights (<= 1) on the tensor cores.
 *
 * Requirements: d = 64 or 128; any W >= 1 (the W * Hq/Hkv window rows of a KV head are processed
 * in 128-row tiles); pool_kernel odd, 1..65; W <= ctx <= cap for every request; k, q_obs 16-byte
 * aligned, importance 4-byte aligned. The workspace (256-byte aligned) holds the window rows'
 * log-sum-exp (and per-CTA partials of it) and one vote partial per (KV head, row tile):
 * vc_importance_workspace_size(shape, W, max_ctx) bytes cover requests of up to max_ctx tokens.
 * Returns VC_ERR_INVALID / VC_ERR_UNSUPPORTED / VC_ERR_WORKSPACE before launching anything. */
#define VC_POOL_MAX 0
#define VC_POOL_AVG 1

typedef struct vc_importance_req {
  vc_kv_full full;        /* keys read: K rows 0..ctx-1 of every KV head (V is not read) */
  const void* q_obs;      /* bf16 [W][Hq][d]: queries of context tokens ctx-W .. ctx-1 */
  float* importance;      /* fp32 [ctx] output */
} vc_importance_req;

vc_status vc_snapkv_importance(const vc_shape* shape, const vc_importance_req* req, int32_t window,
                               int32_t pool_kernel, int32_t pool_kind, void* ws, size_t ws_bytes,
                               int32_t* dev_status, cudaStream_t stream);

size_t vc_importance_workspace_size(const vc_shape* shape, int32_t window, int32_t max_ctx);

/* ------------------------------------------------------------------------------------------ */
/* vc_plan_stagger — choose the two alternating groups of cross-resource staggering ("Cross-resource
 * staggering (P1)": while some requests draft, bound by HBM bandwidth, the KV_full of others moves
 * over the host link and is verified; the pages fix no rule for choosing who does which).
 *
 * The schedule: a compute stream repeats [draft A, verify B, draft B, verify A] and a copy stream
 * repeats [copy B, copy A]; verify X waits for copy X (of the same period), and copy X waits for
 * the previous verification of X (its staging slot is free again). With per-request costs d (draft
 * phase), v (verification and accept) and s (copy; 0 for a request whose KV_full stays in HBM) and
 * D_X, S_X, V_X their sums over group X (D, S, V over all requests), the steady-state period is
 * the maximum cycle mean of that dependency graph (max-plus algebra):
 *     T(A) = max(D + V, S, S_A + V_A, S_B + V_B, (S + V + D_A) / 2, (S + V + D_B) / 2).
 * T(A) = T(B). The call returns, in group[r] (0 = A, 1 = B), a split of minimum T with request 0
 * in A and, when n >= 2, both groups non-empty; among equal T (compared exactly, as 2T) the one
 * with the smallest longer phase, max(D_A + V_B, D_B + V_A) (balanced phases: a lopsided split
 * that the model ties with a balanced one measured slower), then the smallest sum of
 * group[r] * 2^(r-1) over r >= 1. period_ns (may be NULL) receives T rounded
 * up to a whole ns. Exact: all 2^(n-1) - 1 such splits are enumerated in Gray-code order, O(1)
 * each (about 8 M at n = VC_STAGGER_MAX).
 * Errors: VC_ERR_INVALID (null pointers, n < 1, a negative cost or one above 2^40 ns);
 * VC_ERR_UNSUPPORTED (n > VC_STAGGER_MAX). Host only, no GPU work. */
#define VC_STAGGER_MAX 24

typedef struct vc_stagger_cost {
  int64_t draft_ns;   /* GPU time of the request's draft phase */
  int64_t verify_ns;  /* GPU time of its verification and acceptance */
  int64_t stage_ns;   /* host-link time of copying its KV_full (0 when KV_full stays in HBM) */
} vc_stagger_cost;

vc_status vc_plan_stagger(const vc_stagger_cost* cost, int32_t n, int32_t* group, int64_t* period_ns);

/* T of a given split (group[r] in {0, 1}) under the same model; same errors, any n >= 1. */
vc_status vc_stagger_period(const vc_stagger_cost* cost, int32_t n, const int32_t* group, int64_t* period_ns);

/* vc_plan_stagger_local — a split for batches beyond the exact planner's reach (any n up to
 * VC_STAGGER_LOCAL_MAX), under the same model, arguments and output convention (request 0 in A,
 * both groups non-empty when n >= 2, period_ns may be NULL). Local search, no optimality
 * guarantee: three seeds (first half / second half, alternating, and a greedy pass by decreasing
 * d + s + v that adds each request where the split-dependent part of 2T over the partial sums is
 * lower) are each improved by first-improvement descent over single moves and swaps of one request
 * of each group, compared exactly as (2T, longer phase) as above; the best result (ties: the
 * earlier seed) is returned. The
 * returned split is one that no single move and no swap improves, unless a descent reached its
 * limit of 64 n + 1024 improving steps. O(n^2) per improving step; deterministic.
 * Errors: VC_ERR_INVALID (as vc_plan_stagger); VC_ERR_UNSUPPORTED (n > VC_STAGGER_LOCAL_MAX).
 * Host only, no GPU work. */
#define VC_STAGGER_LOCAL_MAX 4096
vc_status vc_plan_stagger_local(const vc_stagger_cost* cost, int32_t n, int32_t* group, int64_t* period_ns);

/* ------------------------------------------------------------------------------------------ */
/* Workspace bytes vc_draft_attn (call = VC_CALL_DRAFT) or vc_verify_attn (VC_CALL_VERIFY) needs
 * for `shape`; max_rows = the largest n_rows of a verify call (ignored for draft). The workspace
 * holds per-split partial outputs. The draft workspace also starts with a block of
 * VC_DRAFT_COUNTER_BYTES of per-(KV head, request) arrival counters, the same bytes for every
 * shape (room for VC_DRAFT_MAX_KV_HEADS heads): zero-fill at least that block once before the
 * first call; every call returns the counters to zero, so one workspace can serve calls of any
 * shape it is large enough for. The verify workspace needs no initialisation. Calls that overlap
 * on the GPU must not share a workspace. */
size_t vc_workspace_size(int32_t call, const vc_shape* shape, int32_t max_rows);

const char* vc_status_string(vc_status s);

/* Library version, major*10000 + minor*100 + patch. */
int32_t vc_version(void);

#ifdef __cplusplus
}
#endif
#endif /* VC_H_ */
