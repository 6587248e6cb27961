// C ABI and host planner for batched attention over a paged KV cache (GB300, sm_103a).
//
// The planner follows the plan/run split of "FlashInfer and the attention-backend abstraction",
// section «What plan() actually computes» (shape and policy in, CTA work assignment and split-K
// temporaries out) and "手写 mini-sglang 阶段四 · GPU 注意力后端", section «FlashInfer：plan 与 run»
// (work partition computed on the CPU, copied to the GPU asynchronously through a reused pinned
// buffer that is only rewritten after the previous copy has completed).
//
// Load balancing follows the idea of "SGLang 源码完全拆解(八)：Attention Backend", section «其他后端的
// 元数据» (split long sequences into more KV chunks, spread ragged work evenly over CTAs using the
// lengths): every (request, KV head, head group) is cut into chunks of one common length chosen
// from the total work and the SM count, and the CTAs are launched longest first.

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <climits>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <string>
#include <vector>

#include "pkv_internal.h"

using pkv::MergeItem;
using pkv::ReqInfo;
using pkv::WorkItem;

namespace {

thread_local std::string g_err;

int fail(int code, const std::string& msg) {
  g_err = msg;
  return code;
}

#define PKV_CUDA(expr, what)                                                        \
  do {                                                                              \
    cudaError_t _e = (expr);                                                        \
    if (_e != cudaSuccess) return fail(PKV_ECUDA, std::string(what) + ": " + cudaGetErrorString(_e)); \
  } while (0)

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

constexpr int kDecodeWaves = 1;          // chunk = total work / (SMs * CTAs/SM * waves)
constexpr int kDecodeMinChunk = 256;     // never split below this many keys
constexpr int kDecodeChunkAlign = 64;    // 4 warps x 16 keys
constexpr int kPrefillRows = 128;        // query rows (tokens x heads of one KV head) per Q tile
constexpr int kPrefillTiles = 2;         // Q tiles per CTA (they share every K/V tile)
constexpr int kPrefillKeyTile = 128;     // keys per K/V tile of the prefill kernel
constexpr int kPrefillMinChunk = 256;    // never split a prefill key range below this many keys
constexpr int kPrefillMaxSplits = 64;    // chunks per prefill item at most (the chunk grows instead)
constexpr bool kDecodeSplitMajor = true;   // the CTAs of a split unit spread over the launch order
constexpr bool kPrefillGroupOrder = true;  // prefill CTAs grouped by (request, KV head) for L2 reuse
constexpr int kPrefillTailNum = 10, kPrefillTailDen = 100;  // share of the work ordered longest first at the end

constexpr int64_t kDefaultWaitLimit = 4000000000LL;  // clock cycles per in-kernel wait (about 2 s)
std::atomic<int64_t> g_wait_limit{kDefaultWaitLimit};
std::atomic<int32_t> g_hold_wait{0};

}  // namespace

int pkv::set_last_error(int code, const char* msg) { return fail(code, msg ? msg : ""); }


namespace {

int query_num_sms(int32_t requested, int32_t* out) {
  if (requested > 0) {
    *out = requested;
    return PKV_OK;
  }
  static int cached[64] = {0};  // SM count per device (a plan per batch asks for it every time)
  int dev = 0, n = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess && dev >= 0 && dev < 64 && cached[dev] > 0) {
    *out = cached[dev];
    return PKV_OK;
  }
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess || n <= 0) {
    cudaGetLastError();
    return fail(PKV_EINVAL, "num_sms == 0 needs a visible CUDA device; pass num_sms > 0 for a host-only plan");
  }
  if (dev >= 0 && dev < 64) cached[dev] = n;
  *out = n;
  return PKV_OK;
}

// Keys one CTA of the item is expected to read: its range, shared by num_splits CTAs.
inline int32_t item_share(const WorkItem& x) {
  return (x.kv_end - x.kv_begin + x.num_splits - 1) / x.num_splits;
}

// Order the work list longest first (stable counting sort on the per-CTA share, bucketed: the order
// is exact up to 1/B of the longest share, B = the number of items clamped to [64, 4096]).
void order_longest_first(std::vector<WorkItem>& all, size_t begin, size_t end) {
  const size_t n = end - begin;
  if (n < 2) return;
  WorkItem* w = all.data() + begin;
  // one key per item (a division each; consecutive items of one split unit share theirs)
  thread_local std::vector<int32_t> key;
  key.resize(n);
  int32_t maxlen = 0;
  for (size_t i = 0; i < n; ++i) {
    const bool same = i > 0 && w[i].kv_begin == w[i - 1].kv_begin && w[i].kv_end == w[i - 1].kv_end &&
                      w[i].num_splits == w[i - 1].num_splits;
    key[i] = same ? key[i - 1] : item_share(w[i]);
    maxlen = std::max(maxlen, key[i]);
  }
  // about one bucket per item (at least 64, at most 4096): the prefix sum over the buckets then
  // costs no more than the passes over the items
  const int32_t max_buckets = (int32_t)std::min<size_t>(4096, std::max<size_t>(64, n));
  int shift = 0;
  while ((maxlen >> shift) >= max_buckets) ++shift;
  const int nb = (maxlen >> shift) + 1;
  thread_local std::vector<uint32_t> count;
  thread_local std::vector<WorkItem> tmp;
  count.assign(nb + 1, 0u);
  tmp.resize(n);
  uint32_t* c = count.data();
  const int32_t* k = key.data();
  for (size_t i = 0; i < n; ++i) ++c[nb - (k[i] >> shift)];
  for (int d = 0; d < nb; ++d) c[d + 1] += c[d];
  WorkItem* dst = tmp.data();
  for (size_t i = 0; i < n; ++i) dst[c[nb - 1 - (k[i] >> shift)]++] = w[i];
  std::memcpy(w, dst, n * sizeof(WorkItem));
}

// Split-major order of the decode items, applied before the longest-first order (which is stable):
// split 0 of every unit, then split 1 of every unit, and so on, so the CTAs of one split unit are
// spread over the whole launch order instead of sitting next to each other.  The block scheduler
// fills the SMs' resident slots in launch order, and measured per-CTA timelines show the CTAs
// launched into an SM's last slots streaming more slowly than its first ones; a unit launched as
// one contiguous block lands on the same slot of every SM and, with the run-time claims balancing
// only within a unit, units launched late finished ~3.5 us after units launched early.  Spread
// over all slots, every unit streams at the same aggregate rate and all of them end together.
void order_split_major(std::vector<WorkItem>& all, size_t begin, size_t end) {
  const size_t n = end - begin;
  if (n < 2) return;
  WorkItem* w = all.data() + begin;
  int32_t max_split = 0;
  for (size_t i = 0; i < n; ++i) max_split = std::max(max_split, w[i].split);
  if (max_split == 0) return;
  thread_local std::vector<uint32_t> count;
  thread_local std::vector<WorkItem> tmp;
  count.assign((size_t)max_split + 2, 0u);
  tmp.resize(n);
  for (size_t i = 0; i < n; ++i) ++count[(size_t)w[i].split + 1];
  for (int32_t s = 0; s <= max_split; ++s) count[(size_t)s + 1] += count[(size_t)s];
  for (size_t i = 0; i < n; ++i) tmp[count[(size_t)w[i].split]++] = w[i];
  std::memcpy(w, tmp.data(), n * sizeof(WorkItem));
}

// Group-major order of the prefill items on top of the longest-first order: the (request, KV head)
// groups by total work, largest first, and inside a group its items still longest first (a stable
// counting sort on the group's rank).  The CTAs resident at any moment then come from a few groups,
// so the K/V rows they gather stay in L2 between the query tiles that read them.
void order_by_group(std::vector<WorkItem>& all, size_t begin, size_t end, int32_t num_kv_heads) {
  const size_t n = end - begin;
  if (n < 2) return;
  WorkItem* w = all.data() + begin;
  int32_t max_req = 0;
  for (size_t i = 0; i < n; ++i) max_req = std::max(max_req, w[i].req);
  const size_t ng = (size_t)(max_req + 1) * (size_t)num_kv_heads;
  thread_local std::vector<int64_t> total;
  thread_local std::vector<int32_t> rank, order;
  total.assign(ng, 0);
  for (size_t i = 0; i < n; ++i) total[(size_t)w[i].req * num_kv_heads + w[i].kv_head] += item_share(w[i]);
  order.resize(ng);
  for (size_t g = 0; g < ng; ++g) order[g] = (int32_t)g;
  std::stable_sort(order.begin(), order.end(), [&](int32_t a, int32_t b) { return total[a] > total[b]; });
  rank.resize(ng);
  for (size_t r = 0; r < ng; ++r) rank[order[r]] = (int32_t)r;
  thread_local std::vector<uint32_t> count;
  thread_local std::vector<WorkItem> tmp;
  count.assign(ng + 1, 0u);
  tmp.resize(n);
  for (size_t i = 0; i < n; ++i) ++count[rank[(size_t)w[i].req * num_kv_heads + w[i].kv_head] + 1];
  for (size_t g = 0; g < ng; ++g) count[g + 1] += count[g];
  for (size_t i = 0; i < n; ++i) tmp[count[rank[(size_t)w[i].req * num_kv_heads + w[i].kv_head]]++] = w[i];
  std::memcpy(w, tmp.data(), n * sizeof(WorkItem));
  // the last part of the work goes longest first again, so that no long item starts near the end
  int64_t all_work = 0;
  for (size_t g = 0; g < ng; ++g) all_work += total[g];
  int64_t acc = 0;
  size_t cut = n;
  for (size_t i = 0; i < n; ++i) {
    acc += item_share(w[i]);
    if (acc * kPrefillTailDen > all_work * (kPrefillTailDen - kPrefillTailNum)) {
      cut = i + 1;
      break;
    }
  }
  if (kPrefillTailNum > 0) order_longest_first(all, begin + cut, end);
}

// Validate the arguments and build the work list into P (no device work).
int build_plan(const pkv_plan_args* a, pkv_plan* P) {
  if (!a) return fail(PKV_EINVAL, "args is NULL");
  const int32_t B = a->batch_size;
  if (B < 0) return fail(PKV_EINVAL, "batch_size < 0");
  if (a->mode != PKV_MODE_DECODE && a->mode != PKV_MODE_PREFILL && a->mode != PKV_MODE_MIXED &&
      a->mode != PKV_MODE_RAGGED && a->mode != PKV_MODE_PAGED_RAGGED)
    return fail(PKV_EINVAL, "unknown mode");
  const bool ragged = a->mode == PKV_MODE_RAGGED;  // K/V rows of contiguous tensors, no page table
  const bool two_src = a->mode == PKV_MODE_PAGED_RAGGED;  // pages = prefix, new rows contiguous
  if (B > 0 && (!a->qo_indptr || !a->kv_indptr || (!ragged && !a->last_page_len)))
    return fail(PKV_EINVAL, ragged ? "qo_indptr and kv_indptr must be non-NULL"
                                   : "qo_indptr, kv_indptr and last_page_len must be non-NULL");
  if (a->num_qo_heads <= 0 || a->num_kv_heads <= 0) return fail(PKV_EINVAL, "head counts must be positive");
  if (a->num_qo_heads % a->num_kv_heads)
    return fail(PKV_EINVAL, "num_qo_heads must be a multiple of num_kv_heads");
  if (a->head_dim != 64 && a->head_dim != 128) return fail(PKV_EUNSUPPORTED, "head_dim must be 64 or 128");
  if (!ragged && a->page_size < 1) return fail(PKV_EINVAL, "page_size must be >= 1");
  if (a->causal != 0 && a->causal != 1) return fail(PKV_EINVAL, "causal must be 0 or 1");
  if (a->window_left < -1) return fail(PKV_EINVAL, "window_left must be -1 or >= 0");
  const bool causal = a->causal == 1;
  if (!causal && a->mode != PKV_MODE_PREFILL && !ragged && !two_src)
    return fail(PKV_EINVAL, "causal == 0 needs a PKV_MODE_PREFILL, PKV_MODE_RAGGED or PKV_MODE_PAGED_RAGGED plan");
  if (!causal && a->window_left >= 0) return fail(PKV_EINVAL, "a sliding window needs causal == 1");
  if (!(std::isfinite(a->sm_scale))) return fail(PKV_EINVAL, "sm_scale is not finite");
  if (a->q_dtype != PKV_BF16) return fail(PKV_EUNSUPPORTED, "q_dtype must be PKV_BF16");
  if (a->kv_dtype != PKV_BF16 && a->kv_dtype != PKV_FP8_E4M3) return fail(PKV_EINVAL, "unknown kv_dtype");
  if (a->kv_dtype == PKV_FP8_E4M3 && a->head_dim != 128)
    return fail(PKV_EUNSUPPORTED, "FP8 KV needs head_dim 128");
  if (a->max_splits < 0) return fail(PKV_EINVAL, "max_splits < 0");
  const int32_t G = a->num_qo_heads / a->num_kv_heads;
  // requests with more than one new token go to the prefill kernel (all of them in prefill mode)
  bool any_extend = a->mode == PKV_MODE_PREFILL || ragged || two_src;
  if (a->mode == PKV_MODE_MIXED)
    for (int32_t i = 0; i < B && !any_extend; ++i) any_extend = a->qo_indptr[i + 1] - a->qo_indptr[i] > 1;
  if (any_extend) {
    const char* why = nullptr;
    if (!pkv::prefill_supported(&why)) return fail(PKV_EUNSUPPORTED, why ? why : "prefill kernel unavailable");
    if (a->head_dim != 128) return fail(PKV_EUNSUPPORTED, "prefill / extend rows need head_dim 128");
    if (a->kv_dtype != PKV_BF16) return fail(PKV_EUNSUPPORTED, "prefill / extend rows need a bf16 KV cache");
    if (G > kPrefillRows || kPrefillRows % G) return fail(PKV_EUNSUPPORTED, "prefill needs 128 % (Hq/Hkv) == 0");
  }

  if (B > 0) {
    if (a->qo_indptr[0] != 0) return fail(PKV_EINVAL, "qo_indptr[0] must be 0");
    if (a->kv_indptr[0] != 0) return fail(PKV_EINVAL, "kv_indptr[0] must be 0");
  }
  // paged: kv_indptr counts pages of kv_indices; ragged: it counts rows of the k / v tensors
  int64_t nnz = B > 0 ? a->kv_indptr[B] : 0;
  if (!ragged && nnz > 0 && !a->kv_indices) return fail(PKV_EINVAL, "kv_indices is NULL");

  P->req.assign(B, ReqInfo{});
  P->max_page_id = -1;
  int64_t total_tokens = B > 0 ? a->qo_indptr[B] : 0;
  for (int32_t i = 0; i < B; ++i) {
    const int64_t n = (int64_t)a->qo_indptr[i + 1] - a->qo_indptr[i];
    const int64_t np = (int64_t)a->kv_indptr[i + 1] - a->kv_indptr[i];
    if (n < 0) return fail(PKV_EINVAL, "qo_indptr must be non-decreasing (request " + std::to_string(i) + ")");
    if (np < 0) return fail(PKV_EINVAL, "kv_indptr must be non-decreasing (request " + std::to_string(i) + ")");
    int64_t L = 0;
    if (ragged) {
      L = np;
    } else if (np > 0) {
      const int32_t last = a->last_page_len[i];
      if (last < 1 || last > a->page_size)
        return fail(PKV_EINVAL, "last_page_len must be in [1, page_size] (request " + std::to_string(i) + ")");
      L = (np - 1) * (int64_t)a->page_size + last;
    }
    if (two_src) L += n;  // the pages hold the prefix; the new tokens follow it
    if (L > INT32_MAX) return fail(PKV_EUNSUPPORTED, "KV length exceeds 2^31-1");
    if (causal && L < n)
      return fail(PKV_EINVAL, "kv_len < q_len (request " + std::to_string(i) + "): seq_len - query_len must be the cached context");
    if (a->mode == PKV_MODE_DECODE && n > 1)
      return fail(PKV_EINVAL, "decode mode allows at most one new token per request (request " + std::to_string(i) + ")");
    P->req[i] = ReqInfo{a->kv_indptr[i], (int32_t)L, a->qo_indptr[i], (int32_t)n};
  }
  P->indices.resize(ragged ? 0 : nnz);
  if (ragged) {
    P->max_page_id = nnz - 1;  // the largest K/V row the plan reads
  } else {
    // copy the page list, then find its range with eight independent min / max chains
    const int32_t* ix = a->kv_indices;
    if (nnz) std::memcpy(P->indices.data(), ix, (size_t)nnz * sizeof(int32_t));
    int32_t mn[8], mx[8];
    for (int u = 0; u < 8; ++u) {
      mn[u] = INT32_MAX;
      mx[u] = -1;
    }
    int64_t k = 0;
    for (; k + 8 <= nnz; k += 8) {
      for (int u = 0; u < 8; ++u) {
        const int32_t v = ix[k + u];
        mn[u] = v < mn[u] ? v : mn[u];
        mx[u] = v > mx[u] ? v : mx[u];
      }
    }
    for (; k < nnz; ++k) {
      mn[0] = std::min(mn[0], ix[k]);
      mx[0] = std::max(mx[0], ix[k]);
    }
    int32_t lo = mn[0], hi = mx[0];
    for (int u = 1; u < 8; ++u) {
      lo = std::min(lo, mn[u]);
      hi = std::max(hi, mx[u]);
    }
    if (nnz && lo < 0) return fail(PKV_EINVAL, "kv_indices entries must be >= 0");
    P->max_page_id = nnz ? hi : -1;
  }

  int32_t sms = 0;
  int st = query_num_sms(a->num_sms, &sms);
  if (st != PKV_OK) return st;

  P->mode = a->mode;
  P->batch = B;
  P->Hq = a->num_qo_heads;
  P->Hkv = a->num_kv_heads;
  P->D = a->head_dim;
  P->ps = ragged ? 1 : a->page_size;
  P->causal = causal;
  P->ragged = ragged;
  P->paged_ragged = two_src;
  P->window_left = a->window_left;
  P->kv_dtype = a->kv_dtype;
  P->q_dtype = a->q_dtype;
  P->sm_scale = a->sm_scale > 0.f ? a->sm_scale : 1.0f / std::sqrt((float)a->head_dim);
  P->total_tokens = total_tokens;
  P->work.clear();
  P->merge.clear();
  P->num_partials = 0;
  P->kv_tokens = 0;
  P->kv_chunk = 0;
  P->num_decode_work = 0;
  P->num_decode_merge = 0;
  P->num_prefill_partials = 0;
  P->num_decodes = P->num_decode_tokens = P->num_prefills = P->num_prefill_tokens = 0;

  // decode rows: every request in decode mode, the one-token requests in mixed mode
  const bool plan_decode = a->mode == PKV_MODE_DECODE || a->mode == PKV_MODE_MIXED;
  const bool plan_prefill = a->mode == PKV_MODE_PREFILL || a->mode == PKV_MODE_MIXED || ragged || two_src;
  if (plan_decode) {
    const int32_t groups = (G + pkv::kDecodeRows - 1) / pkv::kDecodeRows;
    struct Unit { int32_t req, lo, hi; };
    std::vector<Unit> units;
    units.reserve(B);
    int64_t total = 0;
    for (int32_t i = 0; i < B; ++i) {
      if (P->req[i].q_len != 1) continue;
      ++P->num_decodes;
      ++P->num_decode_tokens;
      const int32_t L = P->req[i].kv_len;
      const int32_t pos = L - 1;
      const int32_t lo = a->window_left >= 0 ? std::max(0, pos - a->window_left) : 0;
      units.push_back({i, lo, L});
      total += (int64_t)(L - lo);
    }
    P->kv_tokens = total;
    const int64_t work_total = total * a->num_kv_heads * groups;
    int64_t chunk;
    if (a->max_splits == 1) {
      chunk = INT32_MAX;
    } else {
      const int64_t target = (int64_t)sms * pkv::decode_ctas_per_sm(a->kv_dtype, a->head_dim, G) * kDecodeWaves;
      chunk = (work_total + target - 1) / std::max<int64_t>(1, target);
      chunk = std::max<int64_t>(chunk, kDecodeMinChunk);
      chunk = align_up(chunk, kDecodeChunkAlign);
    }
    // A unit is split only when it is clearly longer than the chunk: every split costs a partial
    // write and a merge, and units up to 1.25 chunks still balance under longest-first launch.
    auto splits_for = [&](int64_t len, int64_t c) -> int64_t {
      int64_t ns = len <= c + c / 4 ? 1 : (len + c - 1) / c;
      if (a->max_splits > 1) ns = std::min<int64_t>(ns, a->max_splits);
      const int64_t piece = align_up((len + ns - 1) / ns, 16);
      return (len + piece - 1) / piece;
    };
    if (a->max_splits != 1) {
      // Wave fit: CTAs longer than half a chunk cannot share a slot, so when there are more of them
      // than resident slots (many equally long requests) a second wave would run a few of them
      // alone.  Grow the chunk in 1/16 steps until they fit one wave.
      const int64_t slots = (int64_t)sms * pkv::decode_ctas_per_sm(a->kv_dtype, a->head_dim, G) * kDecodeWaves;
      auto long_items = [&](int64_t c) -> int64_t {
        int64_t n = 0;
        for (const Unit& u : units) {
          const int64_t len = u.hi - u.lo, ns = splits_for(len, c);
          if (2 * ((len + ns - 1) / ns) > c) n += ns;
        }
        return n * a->num_kv_heads * groups;
      };
      int64_t c = chunk;
      for (int it = 0; it < 16 && long_items(c) > slots; ++it) c = align_up(c + c / 16, kDecodeChunkAlign);
      if (long_items(c) <= slots) chunk = c;
    }
    P->kv_chunk = chunk;
    auto num_splits = [&](int64_t len) -> int64_t { return splits_for(len, chunk); };
    int64_t items = 0, merges = 0;
    for (const Unit& u : units) {
      const int64_t ns = num_splits(u.hi - u.lo);
      items += ns;
      merges += ns > 1;
    }
    const int64_t per_unit = (int64_t)a->num_kv_heads * groups;
    P->work.resize((size_t)(items * per_unit));
    P->merge.resize((size_t)(merges * per_unit));
    WorkItem* wi = P->work.data();
    MergeItem* mi = P->merge.data();
    int64_t slot = 0;
    // The ns CTAs of a split unit all draw from the unit's whole key range: each warp starts on a
    // 64-key group of its own and then claims further groups from a per-unit counter at run time,
    // so CTAs on faster SMs read more and all of them finish together.
    for (const Unit& u : units) {
      const int64_t ns = num_splits(u.hi - u.lo);
      const int32_t q_row = P->req[u.req].q_begin;
      for (int32_t h = 0; h < a->num_kv_heads; ++h) {
        for (int32_t g = 0; g < groups; ++g) {
          const int32_t unit = ns > 1 ? (int32_t)(mi - P->merge.data()) : -1;
          for (int64_t s = 0; s < ns; ++s) {
            WorkItem& w = *wi++;
            w.req = u.req;
            w.kv_head = h;
            w.head_group = g;
            w.kv_begin = u.lo;
            w.kv_end = u.hi;
            w.q_row = q_row;
            w.out_slot = ns > 1 ? (int32_t)(slot + s) : -1;
            w.q_rows = 1;
            w.page_base = P->req[u.req].page_base;
            w.split = (int32_t)s;
            w.num_splits = (int32_t)ns;
            w.unit = unit;
          }
          if (ns > 1) {
            MergeItem& m = *mi++;
            m = MergeItem{};
            m.q_row = q_row;
            m.kv_head = h;
            m.head_group = g;
            m.first_slot = (int32_t)slot;
            m.num_splits = (int32_t)ns;
            slot += ns;
          }
        }
      }
    }
    P->num_partials = slot;
  }
  P->num_decode_work = (int64_t)P->work.size();
  P->num_decode_merge = (int64_t)P->merge.size();
  if (plan_prefill) {
    const int32_t tok_per_tile = kPrefillTiles * (kPrefillRows / G);  // tokens per CTA
    for (int32_t i = 0; i < B; ++i) {
      const ReqInfo& r = P->req[i];
      if (r.q_len == 0 || (a->mode == PKV_MODE_MIXED && r.q_len == 1)) continue;
      ++P->num_prefills;
      P->num_prefill_tokens += r.q_len;
      for (int32_t t0 = 0; t0 < r.q_len; t0 += tok_per_tile) {
        const int32_t rows = std::min(tok_per_tile, r.q_len - t0);
        // causal: keys up to the last row's position (bottom-right aligned); otherwise all L keys
        const int32_t pos0 = r.kv_len - r.q_len + t0;
        const int32_t last_pos = causal ? pos0 + rows - 1 : r.kv_len - 1;
        const int32_t lo = a->window_left >= 0 ? std::max(0, pos0 - a->window_left) : 0;
        P->kv_tokens += (int64_t)(last_pos + 1 - lo);
        for (int32_t h = 0; h < a->num_kv_heads; ++h) {
          WorkItem w;
          w.req = i;
          w.kv_head = h;
          w.head_group = 0;
          w.kv_begin = lo;
          w.kv_end = last_pos + 1;
          w.q_row = r.q_begin + t0;
          w.out_slot = -1;
          w.q_rows = rows;
          w.page_base = r.page_base;
          w.split = 0;
          w.num_splits = 1;
          w.unit = -1;
          P->work.push_back(w);
        }
      }
    }
    // Split-KV for prefill items: when they cannot fill one wave (one CTA per SM) -- a few long
    // requests, or a shared prefix attended by all of a batch's queries -- cut the long key ranges
    // into chunks of whole key tiles.  Each piece writes a normalised fp32 partial state and its
    // log2-sum-exp; a merge kernel combines the pieces of an item (the split-KV merge of
    // "SGLang 源码完全拆解(八)：Attention Backend", section «extend 的两种形态», per row).
    const size_t first = (size_t)P->num_decode_work;
    const int64_t n_items = (int64_t)(P->work.size() - first);
    if (a->max_splits != 1 && n_items > 0 && n_items < sms) {
      int64_t total = 0;
      for (size_t k = first; k < P->work.size(); ++k) total += P->work[k].kv_end - P->work[k].kv_begin;
      const int64_t cap = a->max_splits > 1 ? std::min(a->max_splits, kPrefillMaxSplits) : kPrefillMaxSplits;
      auto splits_of = [&](int64_t len, int64_t c) -> int64_t {
        const int64_t ns = len <= c + c / 4 ? 1 : (len + c - 1) / c;
        return std::min(ns, cap);
      };
      // smallest chunk (whole key tiles, at least kPrefillMinChunk) whose pieces fit one wave: the
      // pieces of equally long items finish together, and a second, mostly idle wave costs as much
      // as the first
      int64_t chunk = std::max<int64_t>(align_up((total + sms - 1) / sms, kPrefillKeyTile), kPrefillMinChunk);
      auto pieces = [&](int64_t c) -> int64_t {
        int64_t n = 0;
        for (size_t k = first; k < P->work.size(); ++k) n += splits_of(P->work[k].kv_end - P->work[k].kv_begin, c);
        return n;
      };
      for (int it = 0; it < 64 && pieces(chunk) > sms; ++it) chunk = align_up(chunk + chunk / 16, kPrefillKeyTile);
      std::vector<WorkItem> items(P->work.begin() + first, P->work.end());
      P->work.resize(first);
      int64_t pslot = 0;
      for (const WorkItem& it : items) {
        const int64_t len = it.kv_end - it.kv_begin;
        int64_t ns = splits_of(len, chunk);
        if (ns <= 1) {
          P->work.push_back(it);
          continue;
        }
        const int64_t piece = align_up((len + ns - 1) / ns, kPrefillKeyTile);
        ns = (len + piece - 1) / piece;
        MergeItem m{};
        m.q_row = it.q_row;
        m.kv_head = it.kv_head;
        m.head_group = 0;
        m.first_slot = (int32_t)pslot;
        m.num_splits = (int32_t)ns;
        m.q_rows = it.q_rows;
        const int32_t unit = (int32_t)P->merge.size();
        P->merge.push_back(m);
        for (int64_t sp = 0; sp < ns; ++sp) {
          WorkItem w = it;
          w.kv_begin = (int32_t)(it.kv_begin + sp * piece);
          w.kv_end = (int32_t)std::min<int64_t>(it.kv_end, it.kv_begin + (sp + 1) * piece);
          w.out_slot = (int32_t)(pslot + sp);
          w.split = (int32_t)sp;
          w.num_splits = (int32_t)ns;
          w.unit = unit;
          P->work.push_back(w);
        }
        pslot += ns;
      }
      P->num_prefill_partials = pslot;
    }
  }
  // longest first: the block scheduler hands out CTAs roughly in launch order
  if (kDecodeSplitMajor) order_split_major(P->work, 0, (size_t)P->num_decode_work);
  order_longest_first(P->work, 0, (size_t)P->num_decode_work);
  order_longest_first(P->work, (size_t)P->num_decode_work, P->work.size());
  if (kPrefillGroupOrder) order_by_group(P->work, (size_t)P->num_decode_work, P->work.size(), a->num_kv_heads);
  if ((int64_t)P->work.size() > INT32_MAX) return fail(PKV_EUNSUPPORTED, "too many CTAs");

  // workspace layout: [work][merge][req][kv_indices] | [partial lse][partial o]
  size_t off = 0;
  P->off_work = off;
  off = align_up(off + P->work.size() * sizeof(WorkItem), 256);
  P->off_merge = off;
  off = align_up(off + P->merge.size() * sizeof(MergeItem), 256);
  P->off_req = off;
  off = align_up(off + P->req.size() * sizeof(ReqInfo), 256);
  P->off_idx = off;
  off = align_up(off + P->indices.size() * sizeof(int32_t), 256);
  P->off_count = off;  // [unit_count | claim lines], zero-filled by the metadata copy; zero again after each run
  off = align_up(off + P->merge.size() * sizeof(int32_t), 256);
  P->off_claim = off;
  off = align_up(off + P->merge.size() * pkv::kClaimStride * sizeof(int32_t), 256);
  P->meta_bytes = off;
  P->off_plse = off;
  off = align_up(off + (size_t)P->num_partials * pkv::kDecodeRows * sizeof(float), 256);
  P->off_po = off;
  off = align_up(off + (size_t)P->num_partials * pkv::kDecodeRows * P->D * sizeof(float), 256);
  P->off_pplse = off;
  off = align_up(off + (size_t)P->num_prefill_partials * pkv::kPrefillItemRows * sizeof(float), 256);
  P->off_ppo = off;
  off = align_up(off + (size_t)P->num_prefill_partials * pkv::kPrefillPartialFloats * sizeof(float), 256);
  P->need_bytes = std::max<size_t>(off, 256);
  P->valid = true;
  return PKV_OK;
}

}  // namespace

int pkv::check_cache(const pkv_plan* P, const pkv_cache* c) {
  if (!c) return fail(PKV_EINVAL, "cache is NULL");
  if (!c->k || !c->v) return fail(PKV_EINVAL, "cache k/v pointers are NULL");
  if (c->num_kv_heads != P->Hkv || c->head_dim != P->D || c->page_size != P->ps || c->dtype != P->kv_dtype)
    return fail(PKV_EINVAL, "cache geometry (kv heads, head_dim, page_size, dtype) does not match the plan");
  if (c->num_pages <= P->max_page_id)
    return fail(PKV_EINVAL, "the plan references page " + std::to_string(P->max_page_id) + " but the pool has " +
                                std::to_string(c->num_pages) + " pages");
  const int64_t esz = c->dtype == PKV_FP8_E4M3 ? 1 : 2;
  const int64_t vec = 16 / esz;
  if (((uintptr_t)c->k | (uintptr_t)c->v) & 15) return fail(PKV_EINVAL, "cache k/v must be 16-byte aligned");
  if (c->stride_page % vec || c->stride_token % vec || c->stride_head % vec)
    return fail(PKV_EINVAL, "cache strides must be multiples of 16 bytes");
  if (c->stride_page <= 0 || c->stride_token <= 0 || c->stride_head <= 0)
    return fail(PKV_EINVAL, "cache strides must be positive");
  if (c->dtype == PKV_FP8_E4M3) {
    if (!(c->k_scale > 0.f) || !(c->v_scale > 0.f) || !std::isfinite(c->k_scale) || !std::isfinite(c->v_scale))
      return fail(PKV_EINVAL, "FP8 cache scales must be finite and > 0");
  }
  return PKV_OK;
}

namespace {

// Kernel parameters for the work items [first, first + count) of the plan.
pkv::RunParams make_params(const pkv_plan* P, const void* q, const pkv_cache* c, void* o, float* lse, int64_t first,
                           int64_t count) {
  pkv::RunParams p{};
  char* ws = (char*)P->ws;
  p.work = (const WorkItem*)(ws + P->off_work) + first;
  p.merge = (const MergeItem*)(ws + P->off_merge);
  p.req = (const ReqInfo*)(ws + P->off_req);
  p.kv_indices = (const int32_t*)(ws + P->off_idx);
  p.part_lse = (float*)(ws + P->off_plse);
  p.part_o = (float*)(ws + P->off_po);
  p.ppart_lse = (float*)(ws + P->off_pplse);
  p.ppart_o = (float*)(ws + P->off_ppo);
  p.unit_count = (int32_t*)(ws + P->off_count);
  p.claim = (int32_t*)(ws + P->off_claim);
  p.q = q;
  p.o = o;
  p.lse = lse;
  const int64_t esz = c->dtype == PKV_FP8_E4M3 ? 1 : 2;
  p.k_pool = (const char*)c->k;
  p.v_pool = (const char*)c->v;
  p.stride_page_b = c->stride_page * esz;
  p.stride_token_b = c->stride_token * esz;
  p.stride_head_b = c->stride_head * esz;
  p.num_pages = c->num_pages;
  p.page_size = P->ps;
  p.num_qo_heads = P->Hq;
  p.num_kv_heads = P->Hkv;
  p.group = P->Hq / P->Hkv;
  p.head_dim = P->D;
  p.window_left = P->window_left;
  p.noncausal = P->causal ? 0 : 1;
  p.ragged_kv = P->ragged ? 1 : 0;
  p.ext_k = p.ext_v = nullptr;
  p.ext_row_b = 0;
  p.wait_limit_k = (int32_t)((g_wait_limit.load(std::memory_order_relaxed) + 1023) >> 10);
  p.hold_wait = g_hold_wait.load(std::memory_order_relaxed);
  const float log2e = 1.4426950408889634f;
  p.scale_log2 = P->sm_scale * log2e * (c->dtype == PKV_FP8_E4M3 ? c->k_scale : 1.0f);
  p.out_scale = c->dtype == PKV_FP8_E4M3 ? c->v_scale : 1.0f;
  p.num_work = count;
  p.num_merge = (int64_t)P->merge.size();
  return p;
}

int check_run(const pkv_plan* P, int mode, const void* q, const pkv_cache* c, void* o) {
  if (!P || !P->valid) return fail(PKV_EINVAL, "plan is NULL or has not been planned");
  if (!P->ws) return fail(PKV_EINVAL, "the plan is host-only (planned without a workspace)");
  if (mode == PKV_MODE_RAGGED || mode == PKV_MODE_PAGED_RAGGED ? P->mode != mode
                                                             : (P->mode != mode && P->mode != PKV_MODE_MIXED))
    return fail(PKV_EINVAL, mode == PKV_MODE_DECODE    ? "decode_run needs a PKV_MODE_DECODE or PKV_MODE_MIXED plan"
                            : mode == PKV_MODE_RAGGED ? "ragged_run needs a PKV_MODE_RAGGED plan"
                            : mode == PKV_MODE_PAGED_RAGGED ? "paged_ragged_run needs a PKV_MODE_PAGED_RAGGED plan"
                                                      : "prefill_run needs a PKV_MODE_PREFILL or PKV_MODE_MIXED plan");
  int st = pkv::check_cache(P, c);
  if (st != PKV_OK) return st;
  if (P->total_tokens > 0 && (!q || !o)) return fail(PKV_EINVAL, "q and o must be non-NULL");
  if (((uintptr_t)q | (uintptr_t)o) & 15) return fail(PKV_EINVAL, "q and o must be 16-byte aligned");
  int dev = -1;
  PKV_CUDA(cudaGetDevice(&dev), "cudaGetDevice");
  if (dev != P->device) return fail(PKV_EINVAL, "the current device is not the device the plan was made on");
  return PKV_OK;
}

// ---- TMA tensor maps (driver entry point fetched at run time; no link against libcuda) ----
PFN_cuTensorMapEncodeTiled_v12000 get_encode_tiled() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = (PFN_cuTensorMapEncodeTiled_v12000)p;
    else
      cudaGetLastError();
  }
  return fn;
}

}  // namespace

// ================================================================================================
// C ABI
// ================================================================================================
extern "C" {

const char* pkv_last_error(void) { return g_err.c_str(); }

int pkv_plan_create(pkv_plan** out) {
  if (!out) return fail(PKV_EINVAL, "out is NULL");
  *out = new pkv_plan();
  return PKV_OK;
}

void pkv_plan_destroy(pkv_plan* plan) {
  if (!plan) return;
  if (plan->copy_done) {
    cudaEventSynchronize(plan->copy_done);
    cudaEventDestroy(plan->copy_done);
  }
  if (plan->pinned) cudaFreeHost(plan->pinned);
  cudaGetLastError();
  delete plan;
}

int pkv_plan_workspace_size(const pkv_plan_args* args, size_t* bytes) {
  if (!bytes) return fail(PKV_EINVAL, "bytes is NULL");
  pkv_plan tmp;
  int st = build_plan(args, &tmp);
  if (st != PKV_OK) return st;
  *bytes = tmp.need_bytes;
  return PKV_OK;
}

int pkv_attn_plan(pkv_plan* plan, const pkv_plan_args* args, void* workspace, size_t workspace_bytes, void* stream) {
  if (!plan) return fail(PKV_EINVAL, "plan is NULL");
  plan->valid = false;
  // the pinned staging buffer may still be the source of the previous plan's copy
  if (plan->copy_pending && plan->copy_done) {
    PKV_CUDA(cudaEventSynchronize(plan->copy_done), "waiting for the previous plan copy");
    plan->copy_pending = false;
  }
  int st = build_plan(args, plan);
  if (st != PKV_OK) {
    plan->valid = false;
    return st;
  }
  plan->ws = nullptr;
  plan->ws_bytes = 0;
  if (!workspace) return PKV_OK;  // host-only plan
  plan->valid = false;
  if ((uintptr_t)workspace & 255) return fail(PKV_EINVAL, "workspace must be 256-byte aligned");
  if (workspace_bytes < plan->need_bytes)
    return fail(PKV_EWORKSPACE, "workspace has " + std::to_string(workspace_bytes) + " bytes, the plan needs " +
                                    std::to_string(plan->need_bytes));
  int dev = -1;
  PKV_CUDA(cudaGetDevice(&dev), "cudaGetDevice");
  if (plan->pinned && plan->device != dev) {
    // staging and event belong to another device: start over
    if (plan->copy_done) cudaEventDestroy(plan->copy_done);
    cudaFreeHost(plan->pinned);
    plan->pinned = nullptr;
    plan->pinned_dev = nullptr;
    plan->pinned_bytes = 0;
    plan->copy_done = nullptr;
  }
  plan->device = dev;
  if (plan->pinned_bytes < plan->meta_bytes) {
    if (plan->pinned) cudaFreeHost(plan->pinned);
    plan->pinned = nullptr;
    plan->pinned_dev = nullptr;
    size_t want = std::max<size_t>(plan->meta_bytes, 64 << 10);
    want = std::max<size_t>(want, plan->pinned_bytes * 2);
    // mapped, so that a kernel can read it directly (the metadata copy below); where the device
    // cannot map host memory, plain pinned memory and a DMA copy
    int can_map = 0;
    if (cudaDeviceGetAttribute(&can_map, cudaDevAttrCanMapHostMemory, dev) != cudaSuccess) can_map = 0;
    if (!can_map || cudaHostAlloc(&plan->pinned, want, cudaHostAllocMapped) != cudaSuccess) {
      plan->pinned = nullptr;
      cudaGetLastError();
      PKV_CUDA(cudaHostAlloc(&plan->pinned, want, cudaHostAllocDefault), "cudaHostAlloc (plan staging)");
    } else {
      void* d = nullptr;
      if (cudaHostGetDevicePointer(&d, plan->pinned, 0) == cudaSuccess) plan->pinned_dev = d;
      cudaGetLastError();  // a failed mapping query only selects the DMA copy
    }
    plan->pinned_bytes = want;
  }
  if (!plan->copy_done) PKV_CUDA(cudaEventCreateWithFlags(&plan->copy_done, cudaEventDisableTiming), "cudaEventCreate");
  char* h = (char*)plan->pinned;
  // the segments below are rewritten in full; only the split counters must start at zero (the
  // alignment gaps between segments are never read)
  std::memset(h + plan->off_count, 0, plan->meta_bytes - plan->off_count);
  std::memcpy(h + plan->off_work, plan->work.data(), plan->work.size() * sizeof(WorkItem));
  std::memcpy(h + plan->off_merge, plan->merge.data(), plan->merge.size() * sizeof(MergeItem));
  std::memcpy(h + plan->off_req, plan->req.data(), plan->req.size() * sizeof(ReqInfo));
  std::memcpy(h + plan->off_idx, plan->indices.data(), plan->indices.size() * sizeof(int32_t));
  cudaStream_t s = (cudaStream_t)stream;
  // a small kernel reading the mapped staging buffer: a DMA copy of this size spends most of its
  // time in fixed start-up latency on the stream
  if (plan->pinned_dev)
    PKV_CUDA(pkv::launch_meta_copy(workspace, plan->pinned_dev, plan->meta_bytes, s), "plan metadata copy");
  else
    PKV_CUDA(cudaMemcpyAsync(workspace, h, plan->meta_bytes, cudaMemcpyHostToDevice, s), "plan metadata copy");
  PKV_CUDA(cudaEventRecord(plan->copy_done, s), "cudaEventRecord");
  plan->copy_pending = true;
  plan->ws = workspace;
  plan->ws_bytes = workspace_bytes;
  plan->valid = true;
  return PKV_OK;
}

int pkv_kv_store(const void* k, const void* v, const int64_t* slot_mapping, int64_t num_tokens, const pkv_cache* cache,
                 void* stream) {
  if (num_tokens < 0) return fail(PKV_EINVAL, "num_tokens < 0");
  if (!cache) return fail(PKV_EINVAL, "cache is NULL");
  if (num_tokens == 0) return PKV_OK;
  if (!k || !v || !slot_mapping || !cache->k || !cache->v) return fail(PKV_EINVAL, "NULL pointer argument");
  if (cache->head_dim != 64 && cache->head_dim != 128) return fail(PKV_EUNSUPPORTED, "head_dim must be 64 or 128");
  if (cache->dtype != PKV_BF16 && cache->dtype != PKV_FP8_E4M3) return fail(PKV_EINVAL, "unknown cache dtype");
  if (cache->num_kv_heads <= 0 || cache->page_size < 1 || cache->num_pages < 0)
    return fail(PKV_EINVAL, "bad cache geometry");
  const int64_t esz = cache->dtype == PKV_FP8_E4M3 ? 1 : 2;
  const int64_t vec = cache->dtype == PKV_FP8_E4M3 ? 8 : 16;  // bytes each thread stores
  if (((uintptr_t)k | (uintptr_t)v) & 15) return fail(PKV_EINVAL, "k and v must be 16-byte aligned");
  if (((uintptr_t)cache->k | (uintptr_t)cache->v) & (vec - 1)) return fail(PKV_EINVAL, "cache k/v misaligned");
  if ((cache->stride_page * esz) % vec || (cache->stride_token * esz) % vec || (cache->stride_head * esz) % vec)
    return fail(PKV_EINVAL, "cache strides must be multiples of 16 bytes (bf16) or 8 bytes (fp8)");
  float inv_k = 1.f, inv_v = 1.f;
  if (cache->dtype == PKV_FP8_E4M3) {
    if (!(cache->k_scale > 0.f) || !(cache->v_scale > 0.f) || !std::isfinite(cache->k_scale) ||
        !std::isfinite(cache->v_scale))
      return fail(PKV_EINVAL, "FP8 cache scales must be finite and > 0");
    inv_k = 1.0f / cache->k_scale;
    inv_v = 1.0f / cache->v_scale;
  }
  PKV_CUDA(pkv::launch_kv_store(k, v, slot_mapping, num_tokens, *cache, inv_k, inv_v, (cudaStream_t)stream),
           "kv_store launch");
  return PKV_OK;
}

int pkv_attn_decode_run(const pkv_plan* plan, const void* q, const pkv_cache* cache, void* o, float* lse,
                        void* stream) {
  int st = check_run(plan, PKV_MODE_DECODE, q, cache, o);
  if (st != PKV_OK) return st;
  if (plan->num_decode_work == 0) return PKV_OK;
  pkv::RunParams p = make_params(plan, q, cache, o, lse, 0, plan->num_decode_work);
  PKV_CUDA(pkv::launch_decode(p, cache->dtype, (cudaStream_t)stream), "decode launch");
  return PKV_OK;
}

}  // extern "C"

namespace {
// The prefill kernel over the plan's prefill items; `cache` is the pool (paged) or a one-token-page
// view of the contiguous K/V tensors (ragged).
int run_prefill(const pkv_plan* plan, int mode, const void* q, const pkv_cache* cache, void* o, float* lse,
                void* stream, bool merge = false, const void* k_new = nullptr, const void* v_new = nullptr) {
  int st = check_run(plan, mode, q, cache, o);
  if (st != PKV_OK) return st;
  if (merge && !lse) return fail(PKV_EINVAL, "a merging run needs the held state's lse");
  if (merge && plan->mode != PKV_MODE_PREFILL) return fail(PKV_EINVAL, "a merging run needs a PKV_MODE_PREFILL plan");
  const int64_t first = plan->num_decode_work, count = (int64_t)plan->work.size() - first;
  if (count == 0) return PKV_OK;
  if (cache->stride_page != (int64_t)cache->page_size * cache->stride_token)
    return fail(PKV_EUNSUPPORTED, "prefill needs stride_page == page_size * stride_token (uniform slot rows)");
  if (cache->stride_head != cache->head_dim)
    return fail(PKV_EUNSUPPORTED, "prefill needs the heads of a token contiguous (stride_head == head_dim)");
  auto encode = get_encode_tiled();
  if (!encode) return fail(PKV_ECUDA, "cuTensorMapEncodeTiled is unavailable");
  alignas(64) CUtensorMap tq;
  // Q: 3-D (head_dim, num_qo_heads, tokens), box (64, group, 128 / group), 128-byte swizzle
  {
    const int G = plan->Hq / plan->Hkv;
    cuuint64_t dims[3] = {(cuuint64_t)plan->D, (cuuint64_t)plan->Hq, (cuuint64_t)plan->total_tokens};
    cuuint64_t strides[2] = {(cuuint64_t)plan->D * 2, (cuuint64_t)plan->Hq * plan->D * 2};
    cuuint32_t box[3] = {64, (cuuint32_t)G, (cuuint32_t)(128 / G)};
    cuuint32_t es[3] = {1, 1, 1};
    CUresult r = encode(&tq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(q), dims, strides, box, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(PKV_ECUDA, "cuTensorMapEncodeTiled(Q) failed: " + std::to_string((int)r));
  }
  // the slot rows the kernel computes are 32-bit
  if (cache->num_pages * (int64_t)cache->page_size > INT32_MAX)
    return fail(PKV_EUNSUPPORTED, "prefill needs num_pages * page_size < 2^31");
  // O: the same 3-D view and box as Q (full output tiles go out by TMA stores of the box they came in)
  alignas(64) CUtensorMap to;
  {
    const int G = plan->Hq / plan->Hkv;
    cuuint64_t dims[3] = {(cuuint64_t)plan->D, (cuuint64_t)plan->Hq, (cuuint64_t)plan->total_tokens};
    cuuint64_t strides[2] = {(cuuint64_t)plan->D * 2, (cuuint64_t)plan->Hq * plan->D * 2};
    cuuint32_t box[3] = {64, (cuuint32_t)G, (cuuint32_t)(128 / G)};
    cuuint32_t es[3] = {1, 1, 1};
    CUresult r = encode(&to, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, o, dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(PKV_ECUDA, "cuTensorMapEncodeTiled(O) failed: " + std::to_string((int)r));
  }
  pkv::RunParams p = make_params(plan, q, cache, o, lse, first, count);
  p.merge_into = merge ? 1 : 0;
  if (plan->paged_ragged) {
    p.ext_k = static_cast<const char*>(k_new);
    p.ext_v = static_cast<const char*>(v_new);
    p.ext_row_b = (int64_t)plan->Hkv * plan->D * 2;
  }
  PKV_CUDA(pkv::launch_prefill(p, &tq, &to, plan->total_tokens, (cudaStream_t)stream), "prefill launch");
  const int64_t nm = (int64_t)plan->merge.size() - plan->num_decode_merge;
  if (nm > 0)
    PKV_CUDA(pkv::launch_prefill_merge(p, plan->num_decode_merge, nm, (cudaStream_t)stream), "prefill merge launch");
  return PKV_OK;
}
}  // namespace

extern "C" {

int pkv_attn_prefill_run(const pkv_plan* plan, const void* q, const pkv_cache* cache, void* o, float* lse,
                         void* stream) {
  return run_prefill(plan, PKV_MODE_PREFILL, q, cache, o, lse, stream);
}

int pkv_attn_prefill_run_merge(const pkv_plan* plan, const void* q, const pkv_cache* cache, void* o, float* lse,
                               void* stream) {
  return run_prefill(plan, PKV_MODE_PREFILL, q, cache, o, lse, stream, true);
}

int pkv_attn_ragged_run(const pkv_plan* plan, const void* q, const void* k, const void* v, void* o, float* lse,
                        void* stream) {
  if (!plan || !plan->valid) return fail(PKV_EINVAL, "plan is NULL or has not been planned");
  if (plan->mode != PKV_MODE_RAGGED) return fail(PKV_EINVAL, "ragged_run needs a PKV_MODE_RAGGED plan");
  if (plan->work.empty()) return PKV_OK;  // no request has a new token
  if (plan->max_page_id >= 0 && (!k || !v)) return fail(PKV_EINVAL, "k and v must be non-NULL");
  // [rows, Hkv, D] contiguous tensors seen as a pool of one-token pages
  pkv_cache view{};
  view.k = const_cast<void*>(k ? k : q);
  view.v = const_cast<void*>(v ? v : q);
  view.num_pages = plan->max_page_id + 1;
  view.page_size = 1;
  view.num_kv_heads = plan->Hkv;
  view.head_dim = plan->D;
  view.dtype = PKV_BF16;
  view.stride_page = view.stride_token = (int64_t)plan->Hkv * plan->D;
  view.stride_head = plan->D;
  view.k_scale = view.v_scale = 1.f;
  if (view.num_pages == 0) view.num_pages = 1;  // no rows read; keeps the tensor maps well formed
  return run_prefill(plan, PKV_MODE_RAGGED, q, &view, o, lse, stream);
}

int pkv_attn_paged_ragged_run(const pkv_plan* plan, const void* q, const pkv_cache* cache, const void* k_new,
                              const void* v_new, void* o, float* lse, void* stream) {
  if (!plan || !plan->valid) return fail(PKV_EINVAL, "plan is NULL or has not been planned");
  if (plan->mode != PKV_MODE_PAGED_RAGGED)
    return fail(PKV_EINVAL, "paged_ragged_run needs a PKV_MODE_PAGED_RAGGED plan");
  if (plan->total_tokens > 0 && (!k_new || !v_new)) return fail(PKV_EINVAL, "k_new and v_new must be non-NULL");
  if (((uintptr_t)k_new | (uintptr_t)v_new) & 15) return fail(PKV_EINVAL, "k_new and v_new must be 16-byte aligned");
  return run_prefill(plan, PKV_MODE_PAGED_RAGGED, q, cache, o, lse, stream, false, k_new, v_new);
}

int pkv_cascade_run(const pkv_plan* shared, const pkv_plan* suffix, const void* q, const pkv_cache* cache, void* o,
                    float* lse, void* stream) {
  if (!shared || !suffix || !shared->valid || !suffix->valid)
    return fail(PKV_EINVAL, "both plans must be planned");
  if (shared->mode != PKV_MODE_PREFILL || shared->causal)
    return fail(PKV_EINVAL, "the shared plan must be a non-causal PKV_MODE_PREFILL plan");
  if (suffix->mode != PKV_MODE_DECODE && suffix->mode != PKV_MODE_PREFILL && suffix->mode != PKV_MODE_MIXED)
    return fail(PKV_EINVAL, "the suffix plan must be a PKV_MODE_DECODE, PREFILL or MIXED plan");
  if (shared->Hq != suffix->Hq || shared->Hkv != suffix->Hkv || shared->D != suffix->D ||
      shared->total_tokens != suffix->total_tokens)
    return fail(PKV_EINVAL, "the shared and suffix plans must have the same heads, head_dim and query rows");
  if (shared->total_tokens > 0 && !lse) return fail(PKV_EINVAL, "lse is required (the levels merge by it)");
  // every check of both runs before anything is enqueued
  int st = check_run(suffix, suffix->mode == PKV_MODE_DECODE ? PKV_MODE_DECODE : PKV_MODE_PREFILL, q, cache, o);
  if (st == PKV_OK) st = check_run(shared, PKV_MODE_PREFILL, q, cache, o);
  if (st != PKV_OK) return st;
  if (suffix->num_decode_work > 0) {
    st = pkv_attn_decode_run(suffix, q, cache, o, lse, stream);
    if (st != PKV_OK) return st;
  }
  if ((int64_t)suffix->work.size() > suffix->num_decode_work) {
    st = run_prefill(suffix, PKV_MODE_PREFILL, q, cache, o, lse, stream);
    if (st != PKV_OK) return st;
  }
  return run_prefill(shared, PKV_MODE_PREFILL, q, cache, o, lse, stream, true);
}

int pkv_merge_state(const void* o_a, const float* lse_a, const void* o_b, const float* lse_b, void* o, float* lse,
                    int64_t num_states, int32_t head_dim, void* stream) {
  if (num_states < 0) return fail(PKV_EINVAL, "num_states < 0");
  if (head_dim != 64 && head_dim != 128) return fail(PKV_EUNSUPPORTED, "head_dim must be 64 or 128");
  if (num_states == 0) return PKV_OK;
  if (!o_a || !lse_a || !o_b || !lse_b || !o) return fail(PKV_EINVAL, "NULL pointer argument");
  if (((uintptr_t)o_a | (uintptr_t)o_b | (uintptr_t)o) & 15) return fail(PKV_EINVAL, "o_a, o_b and o must be 16-byte aligned");
  PKV_CUDA(pkv::launch_merge_state(o_a, lse_a, o_b, lse_b, o, lse, num_states, head_dim, (cudaStream_t)stream),
           "merge launch");
  return PKV_OK;
}

int pkv_set_wait_limit(int64_t clock_cycles) {
  if (clock_cycles > ((int64_t)INT32_MAX << 10)) return fail(PKV_EINVAL, "clock_cycles is too large");
  g_wait_limit.store(clock_cycles <= 0 ? kDefaultWaitLimit : clock_cycles, std::memory_order_relaxed);
  return PKV_OK;
}

int pkv_test_hold_wait(int32_t on) {
  g_hold_wait.store(on ? 1 : 0, std::memory_order_relaxed);
  return PKV_OK;
}

int pkv_device_error(int32_t* code, int32_t reset, void* stream) {
  if (!code) return fail(PKV_EINVAL, "code is NULL");
  PKV_CUDA(pkv::read_device_error(code, reset, (cudaStream_t)stream), "reading the device error word");
  if (*code != 0) return fail(PKV_EDEVICE, "device error word = " + std::to_string(*code));
  return PKV_OK;
}

int pkv_plan_info_get(const pkv_plan* plan, pkv_plan_info* info) {
  if (!plan || !info) return fail(PKV_EINVAL, "NULL argument");
  if (!plan->valid) return fail(PKV_EINVAL, "plan has not been planned");
  info->mode = plan->mode;
  info->batch_size = plan->batch;
  info->total_tokens = plan->total_tokens;
  info->num_work = (int64_t)plan->work.size();
  info->num_merge = (int64_t)plan->merge.size();
  info->num_partials = plan->num_partials;
  info->kv_chunk = plan->kv_chunk;
  info->workspace_bytes = (int64_t)plan->need_bytes;
  info->max_page_id = plan->max_page_id;
  info->kv_tokens = plan->kv_tokens;
  info->num_decode_work = plan->num_decode_work;
  info->num_decodes = plan->num_decodes;
  info->num_decode_tokens = plan->num_decode_tokens;
  info->num_prefills = plan->num_prefills;
  info->num_prefill_tokens = plan->num_prefill_tokens;
  info->num_prefill_partials = plan->num_prefill_partials;
  return PKV_OK;
}

int pkv_plan_work_items(const pkv_plan* plan, int32_t* out, int64_t capacity) {
  if (!plan || !out) return fail(PKV_EINVAL, "NULL argument");
  if (!plan->valid) return fail(PKV_EINVAL, "plan has not been planned");
  const int64_t need = (int64_t)plan->work.size() * pkv::kWorkItemPublicFields;
  if (capacity < need) return fail(PKV_EINVAL, "capacity too small: need " + std::to_string(need));
  for (size_t i = 0; i < plan->work.size(); ++i)
    std::memcpy(out + i * pkv::kWorkItemPublicFields, &plan->work[i], pkv::kWorkItemPublicFields * sizeof(int32_t));
  return PKV_OK;
}

int pkv_block_table_to_csr(const int32_t* block_table, int32_t batch_size, int32_t max_pages, const int32_t* seq_lens,
                           int32_t page_size, int32_t* kv_indptr, int32_t* kv_indices, int64_t capacity,
                           int32_t* last_page_len) {
  if (batch_size < 0 || max_pages < 0 || page_size < 1) return fail(PKV_EINVAL, "bad sizes");
  if (batch_size > 0 && (!block_table || !seq_lens || !kv_indptr || !last_page_len))
    return fail(PKV_EINVAL, "NULL argument");
  if (!kv_indptr) return fail(PKV_EINVAL, "kv_indptr is NULL");
  kv_indptr[0] = 0;
  int64_t at = 0;
  for (int32_t i = 0; i < batch_size; ++i) {
    const int64_t L = seq_lens[i];
    if (L < 0) return fail(PKV_EINVAL, "seq_lens must be >= 0");
    const int64_t np = (L + page_size - 1) / page_size;  // pages of this request
    if (np > max_pages) return fail(PKV_EINVAL, "a row needs more pages than the block table is wide");
    if (at + np > capacity) return fail(PKV_EINVAL, "kv_indices capacity too small");
    if (at + np > INT32_MAX) return fail(PKV_EINVAL, "too many pages");
    for (int64_t p = 0; p < np; ++p) kv_indices[at + p] = block_table[(int64_t)i * max_pages + p];
    at += np;
    kv_indptr[i + 1] = (int32_t)at;
    last_page_len[i] = np ? (int32_t)(L - (np - 1) * page_size) : 0;  // a full last page is page_size
  }
  return PKV_OK;
}

int pkv_token_table_to_page_table(const int32_t* token_table, int32_t batch_size, int32_t table_width,
                                  const int32_t* seq_lens, int32_t page_size, int32_t* page_table, int64_t capacity) {
  if (batch_size < 0 || table_width < 0 || page_size < 1) return fail(PKV_EINVAL, "bad sizes");
  if (batch_size == 0) return PKV_OK;
  if (!token_table || !seq_lens || !page_table) return fail(PKV_EINVAL, "NULL argument");
  int64_t max_len = 0;
  for (int32_t i = 0; i < batch_size; ++i) max_len = std::max<int64_t>(max_len, seq_lens[i]);
  if (max_len > table_width) return fail(PKV_EINVAL, "seq_len exceeds the token table width");
  const int64_t cols = (max_len + page_size - 1) / page_size;
  if (capacity < cols * batch_size) return fail(PKV_EINVAL, "page_table capacity too small");
  for (int32_t i = 0; i < batch_size; ++i)
    for (int64_t c = 0; c < cols; ++c)
      page_table[i * cols + c] = token_table[(int64_t)i * table_width + c * page_size] / page_size;
  return PKV_OK;
}

}  // extern "C"
