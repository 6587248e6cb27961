/*
 * pkv_attn.h -- C ABI of a GB300 (sm_103a) library for batched attention over a paged KV cache.
 *
 * The calls follow the plan-once-per-batch / run-per-layer contract the pages describe:
 *   - "vLLM 源码完全拆解（六）：Attention Backend", section «plan() 与 run() 分别做什么»: plan()
 *     consumes the batch's variable-length structure once; run() receives only this layer's Q and
 *     the KV cache view and reuses the plan.
 *   - "FlashInfer and the attention-backend abstraction", section «What plan() actually computes»:
 *     the plan takes shape and policy only (no data tensors), picks the kernel specialisation,
 *     assigns work tiles to CTAs and sizes the split-K temporaries inside a caller-owned workspace.
 *   - "手写 mini-sglang 阶段四 · GPU 注意力后端", section «FlashInfer：plan 与 run»: plan() computes
 *     the work partition on the CPU and copies it to the GPU asynchronously; the pinned staging
 *     buffer it reuses must not be rewritten before the previous copy has finished.
 *
 * Conventions shared by every call:
 *   - Pointers named "host" are CPU memory; every other data pointer is device memory on the
 *     current CUDA device.  The library allocates NO device memory: every device buffer
 *     (caches, Q, O, LSE, the plan workspace) belongs to the caller.
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default stream).  All device
 *     work of a call is enqueued on that stream; no call synchronises the device except
 *     pkv_attn_plan (which waits for ITS OWN previous host-to-device copy, see below) and
 *     pkv_device_error.
 *   - Every call returns a pkv_status.  On a non-OK status nothing was enqueued, and
 *     pkv_last_error() returns a message (thread-local) naming the violated condition.  Nothing
 *     ever falls back silently to another implementation ("vLLM 源码完全拆解（六）：Attention
 *     Backend", section «自动选择与手工指定语义不同»: an explicit choice that cannot be honoured
 *     fails loudly).
 *   - Element counts and strides are in ELEMENTS, not bytes.
 */
#ifndef PKV_ATTN_H_
#define PKV_ATTN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---------------------------------------------------------------------------------------------- */
/* status codes and element types                                                                 */
/* ---------------------------------------------------------------------------------------------- */
typedef enum {
  PKV_OK = 0,
  PKV_EINVAL = -1,        /* an argument violates the documented contract                     */
  PKV_EUNSUPPORTED = -2,  /* a valid request this build does not implement (never a fallback) */
  PKV_EWORKSPACE = -3,    /* the workspace is too small (or missing) for this plan            */
  PKV_ECUDA = -4,         /* a CUDA runtime/driver call or kernel launch failed               */
  PKV_EDEVICE = -5        /* a kernel recorded an error in the device error word              */
} pkv_status;

typedef enum {
  PKV_BF16 = 0,     /* bfloat16                                                            */
  PKV_FP8_E4M3 = 1  /* OCP FP8 E4M3 ("fn"): code bytes; real value = decode(code) * scale     */
} pkv_dtype;

typedef enum {
  PKV_MODE_DECODE = 0,  /* one new token per request (qo_indptr[i+1] - qo_indptr[i] in {0, 1}) */
  PKV_MODE_PREFILL = 1, /* any number of new tokens per request (prefill / prefix-cached extend) */
  PKV_MODE_MIXED = 2,   /* both in one batch: requests with one new token are planned for the
                         * decode kernel, requests with more for the prefill kernel, and the two
                         * runs write their rows of one output (the decode / prefill-extend split
                         * of "vLLM 源码完全拆解（六）：Attention Backend", sections «为什么先把 Decode
                         * 移到前面» and «FlashInfer Builder 的结果»).  Requests may come in any order: every
                         * CTA carries its own token row, so no decode-first reordering is needed. */
  PKV_MODE_RAGGED = 3,  /* prefill / extend over CONTIGUOUS K/V tensors instead of the paged pool
                         * (the ragged form of "SGLang 源码完全拆解(八)：Attention Backend", section
                         * «extend 的两种形态»): kv_indptr holds TOKEN offsets into k / v, kv_indices,
                         * last_page_len and page_size are ignored; run with pkv_attn_ragged_run. */
  PKV_MODE_PAGED_RAGGED = 4 /* prefill / extend in one pass over TWO sources: kv_indptr, kv_indices and
                         * last_page_len describe only each request's CACHED PREFIX in the paged
                         * pool (no pages = no prefix), and the n_i new tokens' K/V are rows
                         * qo_indptr[i].. of contiguous k_new / v_new tensors (the "ragged" segment).
                         * Key j < prefix_i comes from the pool, key prefix_i + t from new row t, and
                         * one online softmax covers both: the result of the paged + ragged + merge form
                         * of "SGLang 源码完全拆解(八)：Attention Backend", section «extend 的两种形态»,
                         * without the separate passes or the merge.  Run with pkv_attn_paged_ragged_run. */
} pkv_mode;

/* Device error codes a kernel may record (read with pkv_device_error). */
enum {
  PKV_DEVERR_NONE = 0,
  PKV_DEVERR_SLOT_RANGE = 1,   /* kv_store: slot_mapping entry >= num_pages * page_size           */
  PKV_DEVERR_PAGE_RANGE = 2,   /* attention: a page id outside [0, num_pages)                     */
  PKV_DEVERR_TIMEOUT = 3       /* a bounded wait inside a kernel ran out; the kernel returned     */
};

/* ---------------------------------------------------------------------------------------------- */
/* one layer's KV pool                                                                            */
/* ---------------------------------------------------------------------------------------------- */
/*
 * Layout: K and V are separate pools, each logically [num_pages, page_size, num_kv_heads, head_dim]
 * ("NHD"), with the innermost (head_dim) dimension contiguous and arbitrary strides for the other
 * three ("vLLM 源码完全拆解（六）：Attention Backend", section «KV Cache 视图必须匹配 Kernel ABI»: the
 * backend adapts strides and never copies the KV; "手写 mini-sglang 阶段四 · GPU 注意力后端": k_cache /
 * v_cache of shape [pages, page_size, H, D]).  Element (p, t, h, d) of K is at
 *   k + p * stride_page + t * stride_token + h * stride_head + d.
 * Token slot s lives at page s / page_size, offset s % page_size.
 * Requirements: k and v 16-byte aligned; stride_page, stride_token, stride_head multiples of
 * 16 / element_size; head_dim in {64, 128}.  The prefill path further requires the slots to form
 * one uniform row space (stride_page == page_size * stride_token) and head_dim == 128.
 * FP8 pools hold E4M3 codes; k_scale / v_scale (> 0, finite) define real = code * scale on both the
 * write and the read side ("SGLang 源码完全拆解(八)：Attention Backend", section «层与后端的边界»).
 */
typedef struct pkv_cache {
  void* k;
  void* v;
  int64_t num_pages;
  int32_t page_size;
  int32_t num_kv_heads;
  int32_t head_dim;
  int32_t dtype; /* pkv_dtype */
  int64_t stride_page;
  int64_t stride_token;
  int64_t stride_head;
  float k_scale; /* FP8 only */
  float v_scale; /* FP8 only */
} pkv_cache;

/* ---------------------------------------------------------------------------------------------- */
/* the KV write                                                                                   */
/* ---------------------------------------------------------------------------------------------- */
/*
 * pkv_kv_store: write this step's K/V rows into the pool through slot_mapping, BEFORE attention
 * reads the cache on the same stream ("vLLM 源码完全拆解（六）：Attention Backend", sections
 * «Runner 先构造公共事实» (slot = physical_page * page_size + offset_in_page) and «为什么 KV 写入在
 * Attention 之前»; "手写 mini-sglang 阶段四 · GPU 注意力后端": store_kv(k, v, out_loc, layer)).
 *
 *   k, v          device, bf16, [num_tokens, cache->num_kv_heads, cache->head_dim], contiguous.
 *   slot_mapping  device, int64, [num_tokens].  A negative entry marks a padding token: nothing is
 *                 written for it.  An entry >= num_pages * page_size is skipped and recorded as
 *                 PKV_DEVERR_SLOT_RANGE in the device error word.
 *   cache         host pointer to the pool description (read during the call only).
 * BF16 pools receive a bit-exact copy.  FP8 pools receive code = E4M3_RNE_satfinite(float(x) *
 * inv_scale) with inv_scale = 1.0f / scale computed once in float32 on the host.
 * Two tokens mapped to the same slot in one call race; the caller must not do that.
 * num_tokens == 0 is a no-op.
 */
int pkv_kv_store(const void* k, const void* v, const int64_t* slot_mapping, int64_t num_tokens,
                 const pkv_cache* cache, void* stream);

/* ---------------------------------------------------------------------------------------------- */
/* the plan                                                                                       */
/* ---------------------------------------------------------------------------------------------- */
/*
 * The batch is described by the CSR page table of "SGLang 源码完全拆解(八)：Attention Backend",
 * section «统一元数据的编译», and "vLLM 源码完全拆解（六）：Attention Backend", section «从二维 Block
 * Table 到 CSR 页表»:
 *   qo_indptr      host int32 [batch_size + 1]: new-token row ranges in Q / O; qo_indptr[0] == 0,
 *                  non-decreasing.  n_i = qo_indptr[i+1] - qo_indptr[i].
 *   kv_indptr      host int32 [batch_size + 1]: page ranges in kv_indices; kv_indptr[0] == 0,
 *                  non-decreasing.
 *   kv_indices     host int32 [kv_indptr[batch_size]]: physical page ids, each request's pages in
 *                  logical order; every id >= 0 (checked against the pool size at run time).
 *   last_page_len  host int32 [batch_size]: valid tokens on each request's last page, in
 *                  [1, page_size] (a full last page is page_size, never 0); ignored for a request
 *                  with no pages.
 * The KV length of request i is L_i = (pages_i - 1) * page_size + last_page_len[i] (0 without
 * pages) and INCLUDES this step's new tokens (already written by pkv_kv_store).  New token t of
 * request i sits at absolute position P = L_i - n_i + t and attends to keys j <= P (causal,
 * bottom-right aligned: "手写 mini-sglang 阶段四 · GPU 注意力后端", section «在 CPU 上验证»), and with
 * window_left = w >= 0 only to keys j >= P - w ("SGLang 源码完全拆解(八)：Attention Backend",
 * section «mask 从哪里来»).  Query head h reads KV head h / (num_qo_heads / num_kv_heads).
 * Checked: L_i >= n_i; L_i == 0 only if n_i == 0 (invariants 3-6 of "vLLM 源码完全拆解（六）：
 * Attention Backend", section «九条必须成立的不变量»); with causal == 0 only kv_indptr's order.
 * PKV_MODE_RAGGED: kv_indptr[i] .. kv_indptr[i+1]-1 are the rows of the contiguous k / v tensors
 * that request i owns (L_i = kv_indptr[i+1] - kv_indptr[i]); no page table is involved.
 */
typedef struct pkv_plan_args {
  int32_t batch_size;
  const int32_t* qo_indptr;
  const int32_t* kv_indptr;
  const int32_t* kv_indices;
  const int32_t* last_page_len;
  int32_t num_qo_heads;  /* multiple of num_kv_heads                                         */
  int32_t num_kv_heads;
  int32_t head_dim;      /* 64 or 128 (decode); 128 (prefill)                                */
  int32_t page_size;     /* >= 1                                                             */
  int32_t mode;          /* pkv_mode                                                         */
  int32_t causal;        /* 1: bottom-right-aligned causal mask (every mode).  0: every query */
                         /* of request i sees all L_i keys (PKV_MODE_PREFILL / _RAGGED only; */
                         /* window_left must be -1; L_i < n_i is allowed and L_i == 0 gives  */
                         /* the empty state o = 0, lse = -inf) -- the cached-prefix segment  */
                         /* of the paged + merge extend, attended with causal=False          */
  int32_t window_left;   /* -1: no window; w >= 0 keeps keys P - w .. P                       */
  float sm_scale;        /* <= 0 selects 1 / sqrt(head_dim)                                  */
  int32_t q_dtype;       /* PKV_BF16                                                         */
  int32_t kv_dtype;      /* PKV_BF16 or PKV_FP8_E4M3 (FP8 KV: decode mode only)               */
  int32_t max_splits;    /* split-KV chunks per (request, KV head): 0 = planner's choice,    */
                         /* 1 = never split, k > 1 = at most k.  Prefill items are split only */
                         /* when there are fewer of them than SMs (at most 64 chunks each)    */
  int32_t num_sms;       /* SMs to plan for; 0 = query the current device                    */
} pkv_plan_args;

typedef struct pkv_plan pkv_plan; /* opaque; owns host memory (including pinned staging) only */

/* Create an empty plan object.  It owns a pinned host staging buffer that grows on demand and is
 * reused by every pkv_attn_plan call on this object. */
int pkv_plan_create(pkv_plan** out);

/* Destroy a plan: waits for its last host-to-device copy, then frees its host memory.  The
 * caller's workspace is untouched.  NULL is a no-op. */
void pkv_plan_destroy(pkv_plan* plan);

/* Exact workspace bytes pkv_attn_plan needs for these arguments (validates them first). */
int pkv_plan_workspace_size(const pkv_plan_args* args, size_t* bytes);

/*
 * pkv_attn_plan: validate the batch, copy its host arrays, build the CTA work list (split-KV
 * chunks for decode, query tiles for prefill, longest first), lay out the workspace and enqueue ONE
 * copy of the metadata from the plan's pinned staging buffer into `workspace` on `stream`: a small
 * copy kernel that reads the staging buffer through its device mapping (a DMA copy where the device
 * cannot map host memory).  Before rewriting the staging buffer it waits for this plan object's
 * previous copy.
 * The host arrays may be reused by the caller as soon as the call returns.
 *   workspace       device, 256-byte aligned, >= pkv_plan_workspace_size() bytes; it must stay
 *                   allocated and unmodified until the last run that uses this plan has finished.
 *                   workspace == NULL builds a HOST-ONLY plan (for inspection: pkv_plan_info,
 *                   pkv_plan_work_items); running it returns PKV_EINVAL.
 * A re-plan invalidates the previous plan held by the same object.
 */
int pkv_attn_plan(pkv_plan* plan, const pkv_plan_args* args, void* workspace, size_t workspace_bytes,
                  void* stream);

/* ---------------------------------------------------------------------------------------------- */
/* the runs (once per layer)                                                                      */
/* ---------------------------------------------------------------------------------------------- */
/*
 * pkv_attn_decode_run / pkv_attn_prefill_run: attention for every new token of the planned batch,
 * reading K/V through the plan's page table from `cache`.
 *   q    device, bf16, [total_tokens, num_qo_heads, head_dim], contiguous (total_tokens =
 *        qo_indptr[batch_size] of the plan).
 *   o    device, bf16, same shape as q: o[row, h, :] = sum_j softmax_j(scale * q.k_j) v_j.
 *   lse  device float32 [total_tokens, num_qo_heads] or NULL: natural-log log-sum-exp of the scaled
 *        scores of each row (the statistic "SGLang 源码完全拆解(八)：Attention Backend", section
 *        «extend 的两种形态», merges states with).
 * The cache geometry (heads, head_dim, dtype) must match the plan, and the plan's largest page id
 * must be < cache->num_pages (checked on the host, O(1)).  decode_run needs a PKV_MODE_DECODE or
 * PKV_MODE_MIXED plan, prefill_run a PKV_MODE_PREFILL or PKV_MODE_MIXED plan; on a mixed plan each
 * writes only its own rows (decode_run the rows of one-token requests, prefill_run the others), and
 * both must run for o to be complete (in either order; they touch disjoint rows).  A run with no
 * rows of its kind launches nothing.  Rows of requests with n_i == 0 do not exist; no other row of
 * o is left unwritten.  The runs allocate nothing, read no host data of the batch and never
 * synchronise; several runs (e.g. one per layer) may share one plan as long as the workspace is not
 * used by two runs at the same time.
 */
int pkv_attn_decode_run(const pkv_plan* plan, const void* q, const pkv_cache* cache, void* o, float* lse,
                        void* stream);
int pkv_attn_prefill_run(const pkv_plan* plan, const void* q, const pkv_cache* cache, void* o, float* lse,
                         void* stream);

/*
 * pkv_attn_prefill_run_merge: pkv_attn_prefill_run whose result is merged into a state the caller
 * already holds in (o, lse) -- the merge of "SGLang 源码完全拆解(八)：Attention Backend", section
 * «extend 的两种形态», done in the epilogue instead of a separate pkv_merge_state call: a prefix-cached
 * extend is pkv_attn_ragged_run over the new tokens (causal) into (o, lse), then this call over the
 * cached prefix (a PKV_MODE_PREFILL plan with causal = 0).
 *   o     device bf16 [total_tokens, num_qo_heads, 128]: on entry the held normalised outputs, on exit
 *         the merged ones (weights e^(s - m) / sum, m the larger of the two lse).
 *   lse   device float32 [total_tokens, num_qo_heads], required: on entry the held natural-log lse
 *         (-inf = empty state), on exit the merged lse.
 * Rows whose segment for this pass has no key keep their held state.  A PKV_MODE_PREFILL plan only.
 */
int pkv_attn_prefill_run_merge(const pkv_plan* plan, const void* q, const pkv_cache* cache, void* o, float* lse,
                               void* stream);

/*
 * pkv_attn_ragged_run: attention of a PKV_MODE_RAGGED plan, K/V read from contiguous tensors (the
 * ragged wrapper's forward of "SGLang 源码完全拆解(八)：Attention Backend", section «extend 的两种
 * 形态»: the new tokens' K/V straight from this step's k / v, not through the page table).
 *   q     device bf16 [total_tokens, num_qo_heads, 128], contiguous.
 *   k, v  device bf16 [kv_indptr[batch_size], num_kv_heads, 128], contiguous, 16-byte aligned.
 *   o, lse as for pkv_attn_prefill_run (o bf16; lse natural log, NULL allowed).
 * Same kernel, visibility rule and errors as pkv_attn_prefill_run.
 */
int pkv_attn_ragged_run(const pkv_plan* plan, const void* q, const void* k, const void* v, void* o, float* lse,
                        void* stream);

/*
 * pkv_merge_state: merge two attention states of the same rows ("SGLang 源码完全拆解(八)：Attention
 * Backend", section «extend 的两种形态»: o = (o_a e^(s_a - m) + o_b e^(s_b - m)) / (e^(s_a - m) +
 * e^(s_b - m)), m = max(s_a, s_b); the merged log-sum-exp is m + ln(e^(s_a - m) + e^(s_b - m));
 * "vLLM 源码完全拆解（六）：Attention Backend", section «Cascade Attention 把共享前缀只算一次»: the
 * shared-prefix and suffix outputs are combined by their LSE weights, never added).
 *   o_a, o_b, o   device bf16 [num_states, head_dim] (a state = one (token row, query head) pair;
 *                 [tokens, heads, head_dim] contiguous is the same thing), 16-byte aligned.
 *   lse_a, lse_b  device float32 [num_states], natural log (as the runs export it).  A state with
 *                 lse = -inf is empty and contributes nothing; two empty states give o = 0,
 *                 lse = -inf.
 *   lse           device float32 [num_states] or NULL.
 * o may alias o_a or o_b and lse may alias lse_a or lse_b (in-place merge).  head_dim 64 or 128.
 * Arithmetic in float32, output rounded to bf16 once.
 */
/*
 * pkv_attn_paged_ragged_run: run a PKV_MODE_PAGED_RAGGED plan (a5 over two K/V sources).
 *   q      device bf16 [total_tokens, Hq, D], row-contiguous.
 *   cache  the paged pool holding every request's cached prefix (the plan's page table).
 *   k_new, v_new  device bf16 [total_tokens, Hkv, D], row-contiguous, 16-byte aligned: row r is the K /
 *          V of new token r (the same rows as q); they need not be in the pool (the KV write of this
 *          step may come before or after this call, on the caller's stream order).
 *   o, lse as pkv_attn_prefill_run.
 * Token t of request i sits at position P = prefix_i + t and sees keys 0..P (causal, optional window)
 * or every key (causal == 0).
 */
int pkv_attn_paged_ragged_run(const pkv_plan* plan, const void* q, const pkv_cache* cache, const void* k_new,
                              const void* v_new, void* o, float* lse, void* stream);

/*
 * pkv_cascade_run: attention of a batch whose requests share a prefix, with the shared part computed
 * once ("vLLM 源码完全拆解（六）：Attention Backend", section «Cascade Attention 把共享前缀只算一次»: each
 * query's attention is split into the shared prefix and its request's own suffix, and the two results
 * are combined by their log-sum-exp weights).
 *   shared  a non-causal (causal == 0) PKV_MODE_PREFILL plan over the shared prefix's pages whose
 *           query rows are every row of the batch (normally one "request": qo_indptr = {0, T});
 *   suffix  a plan over each request's own pages after the shared prefix (holding its new tokens):
 *           PKV_MODE_DECODE, PKV_MODE_PREFILL or PKV_MODE_MIXED, with the same head counts, head_dim and
 *           total_tokens T as `shared`;
 *   q, cache  as pkv_attn_prefill_run (one pool holds both levels' pages);
 *   o, lse  device bf16 [T, Hq, D] and fp32 [T, Hq] (lse is required: the merge needs it).
 * The suffix plan's runs write (o, lse), then the shared pass runs with its state merged into them
 * in its epilogue (pkv_attn_prefill_run_merge): two launches, three with a decode/prefill-mixed suffix
 * or a split shared pass, and no scratch.  Errors as the runs it makes; nothing is enqueued when the
 * plans do not match.
 */
int pkv_cascade_run(const pkv_plan* shared, const pkv_plan* suffix, const void* q, const pkv_cache* cache, void* o,
                    float* lse, void* stream);

int pkv_merge_state(const void* o_a, const float* lse_a, const void* o_b, const float* lse_b, void* o, float* lse,
                    int64_t num_states, int32_t head_dim, void* stream);

/*
 * pkv_attn_decode_run_noalloc: pkv_attn_decode_run for callers that cannot allocate device memory.
 * (The pages have no counterpart: this entry point is an addition of this library.)
 *
 * Who needs it: code that is not allowed to call cudaMalloc -- a host framework whose memory pool
 * forbids raw allocations (an allocation made behind the pool's back breaks its accounting and its
 * out-of-memory handling), or an embedded runtime that receives a fixed device-memory budget up
 * front -- and therefore cannot provide the plan workspace.  This call needs no workspace: the plan's metadata (work list, per-request facts,
 * page list) and the split-KV partial outputs live in one statically sized device array inside the
 * library (32 MiB per device that loads the library, held until the process exits).  The caller
 * still passes Q, the cache and the outputs, exactly as for pkv_attn_decode_run.
 *
 *   plan   a PKV_MODE_DECODE plan; a host-only plan (pkv_attn_plan with workspace == NULL) is
 *          enough, and its workspace, if any, is not used.  Its pkv_plan_info().workspace_bytes
 *          must not exceed 32 MiB, otherwise PKV_EWORKSPACE is returned and nothing runs.
 * Same kernels and outputs as pkv_attn_decode_run, and the same checks of the cache against the
 * plan (geometry, page range, 16-byte alignment, positive strides, FP8 scales).  The call itself
 * allocates no device or pinned memory: it copies the plan's metadata from the plan's (pageable)
 * host arrays into the static array on `stream`, then launches the kernels.
 * Every call shares the one array per device and it keeps the last call's contents; calls whose
 * work may overlap on the GPU (other streams, other threads) race on it and must be serialised by
 * the caller.  The first call on a device looks up the array's device address; make that first
 * call before any stream capture begins.
 */
int pkv_attn_decode_run_noalloc(const pkv_plan* plan, const void* q, const pkv_cache* cache, void* o, float* lse,
                                void* stream);

/* ---------------------------------------------------------------------------------------------- */
/* errors and inspection                                                                          */
/* ---------------------------------------------------------------------------------------------- */
/* Message of the last non-OK status returned on this thread ("" if none). */
const char* pkv_last_error(void);

/* Synchronise `stream`, read the device error word of the current device into *code (a
 * PKV_DEVERR_* value; the first error recorded wins) and clear it when reset != 0.  Returns
 * PKV_EDEVICE when *code != 0. */
int pkv_device_error(int32_t* code, int32_t reset, void* stream);

/*
 * pkv_set_wait_limit: the bound on each wait inside the prefill kernel (a K/V tile, a score block,
 * the probabilities of the softmax warps), in SM clock cycles, for every prefill, ragged and
 * merging run launched after the call by any thread of the process; clock_cycles <= 0 restores the
 * default of 4e9 (about 2 s).  The pages ask that failures be loud, never silent ("vLLM 源码完全拆解
 * （六）：Attention Backend", section «自动选择与手工指定语义不同»): a wait that runs out makes its CTA
 * record PKV_DEVERR_TIMEOUT in the device error word, wait (with a fixed bound of 5e8 cycles) for the
 * copies and MMAs it already issued, free its tensor memory and exit without writing its rows; the
 * error is read with pkv_device_error.  The decode kernel has no such waits.
 * Returns PKV_EINVAL when clock_cycles exceeds 2^41.
 */
int pkv_set_wait_limit(int64_t clock_cycles);

/*
 * pkv_test_hold_wait: a testing aid for the timeout path above.  While `on` is nonzero, every prefill
 * CTA launched afterwards first waits on a barrier that nothing arrives at; the wait runs out after
 * the current wait limit and the CTA takes the timeout path (PKV_DEVERR_TIMEOUT, no output rows).
 * Nothing faults or hangs: the held wait is bounded like every other.  No counterpart on the pages.
 */
int pkv_test_hold_wait(int32_t on);

typedef struct pkv_plan_info {
  int32_t mode;
  int32_t batch_size;
  int64_t total_tokens;   /* qo_indptr[batch_size]                                       */
  int64_t num_work;       /* CTAs of the main kernel                                      */
  int64_t num_merge;      /* (request, KV head, head group) units that need a split merge */
  int64_t num_partials;   /* partial (o, lse) slots in the workspace                      */
  int64_t kv_chunk;       /* split-KV chunk length in tokens (decode)                      */
  int64_t workspace_bytes;
  int64_t max_page_id;    /* -1 if the batch has no pages                                  */
  int64_t kv_tokens;      /* sum over requests of the keys the plan reads (per KV head)     */
  int64_t num_decode_work;    /* CTAs of the decode kernel (the first num_decode_work items)  */
  int64_t num_decodes;        /* requests planned for the decode kernel                      */
  int64_t num_decode_tokens;  /* their token rows                                            */
  int64_t num_prefills;       /* requests planned for the prefill kernel                     */
  int64_t num_prefill_tokens; /* their token rows                                            */
  int64_t num_prefill_partials; /* prefill split-KV partial states (256 rows each)            */
} pkv_plan_info;

int pkv_plan_info_get(const pkv_plan* plan, pkv_plan_info* info);

/* Copy the plan's work list to host memory: 8 int32 per CTA, in launch order:
 *   {request, kv_head, head_group, kv_begin, kv_end, q_row, out_slot, q_rows}
 * (out_slot = partial slot or -1 when the CTA writes the final output; decode and prefill items
 * number their partial slots separately).  A prefill item with a partial slot reads exactly
 * [kv_begin, kv_end), a whole number of 128-key tiles except at the end of the item's range; the
 * prefill run merges the pieces of each item with a second kernel.  A decode CTA with
 * out_slot = -1 reads all of [kv_begin, kv_end); the CTAs with consecutive partial slots of one
 * (request, kv_head, head_group) share the same [kv_begin, kv_end) and divide its 32-key groups
 * among themselves at run time (each warp starts on its own group, then takes the next unclaimed
 * one from a counter in the workspace).  `capacity` is in int32. */
int pkv_plan_work_items(const pkv_plan* plan, int32_t* out, int64_t capacity);

/* ---------------------------------------------------------------------------------------------- */
/* host helpers for building the plan inputs (no GPU needed)                                       */
/* ---------------------------------------------------------------------------------------------- */
/*
 * 2-D block table -> CSR page table ("vLLM 源码完全拆解（六）：Attention Backend", section «从二维 Block
 * Table 到 CSR 页表»; "FlashInfer and the attention-backend abstraction", section «What plan()
 * actually computes»: a running sum of page counts, a gather of each row's valid prefix, a modulo).
 *   block_table    host int32 [batch_size, max_pages] row-major (entries past a row's valid pages
 *                  are ignored).
 *   seq_lens       host int32 [batch_size], >= 0, ceil(seq_len / page_size) <= max_pages.
 *   kv_indptr      host int32 [batch_size + 1] (out); kv_indices host int32 [capacity] (out);
 *   last_page_len  host int32 [batch_size] (out; 0 for a request of length 0).
 */
int pkv_block_table_to_csr(const int32_t* block_table, int32_t batch_size, int32_t max_pages,
                           const int32_t* seq_lens, int32_t page_size, int32_t* kv_indptr,
                           int32_t* kv_indices, int64_t capacity, int32_t* last_page_len);

/*
 * Token-granular table -> page table: page_table[i, k] = token_table[i, k * page_size] / page_size
 * for k < ceil(max(seq_lens) / page_size) ("手写 mini-sglang 阶段四 · GPU 注意力后端", section
 * «FlashAttention：页号表»).  token_table host int32 [batch_size, table_width]; page_table host
 * int32 [batch_size, ceil(max_len / page_size)] (out).
 */
int pkv_token_table_to_page_table(const int32_t* token_table, int32_t batch_size, int32_t table_width,
                                  const int32_t* seq_lens, int32_t page_size, int32_t* page_table,
                                  int64_t capacity);

#ifdef __cplusplus
} /* extern "C" */
#endif

#endif /* PKV_ATTN_H_ */
