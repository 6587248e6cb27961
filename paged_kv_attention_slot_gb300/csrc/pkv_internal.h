// Internal declarations shared by the host planner / C ABI (api.cpp) and the CUDA kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <vector>

#include "pkv_attn.h"

namespace pkv {

// One CTA of a run kernel.  The first 8 fields are the public pkv_plan_work_items() rows.
struct WorkItem {
  int32_t req;         // request index
  int32_t kv_head;     // KV head
  int32_t head_group;  // group of up to 16 query heads of this KV head (decode); 0 (prefill)
  int32_t kv_begin;    // first key (logical position) of the range this CTA draws from
  int32_t kv_end;      // one past the last key of that range
  int32_t q_row;       // first token row of Q / O
  int32_t out_slot;    // decode: partial slot, or -1 = write the final output
  int32_t q_rows;      // tokens of this request in this CTA's tile (decode: 1)
  int32_t page_base;   // first kv_indices entry of the request
  int32_t split;       // decode: index of this CTA among the CTAs sharing [kv_begin, kv_end)
  int32_t num_splits;  // decode: CTAs sharing the range (1 = this CTA reads all of it)
  int32_t unit;        // decode: merge item of the shared range, or -1
};
static_assert(sizeof(WorkItem) == 48, "WorkItem is 48 bytes");
constexpr int kWorkItemPublicFields = 8;

// One (request, KV head, head group) whose split-KV partials must be merged.  Decode units come
// first in the plan's list; a prefill unit (a two-tile query item cut into key chunks) follows them.
struct MergeItem {
  int32_t q_row;
  int32_t kv_head;
  int32_t head_group;
  int32_t first_slot;
  int32_t num_splits;
  int32_t q_rows;  // prefill: tokens of the item (decode: 1)
  int32_t pad1, pad2;
};
static_assert(sizeof(MergeItem) == 32, "MergeItem is 32 bytes");

// Per-request facts the kernels need: page list start, KV length, first token row, token count.
struct ReqInfo {
  int32_t page_base;
  int32_t kv_len;
  int32_t q_begin;
  int32_t q_len;
};
static_assert(sizeof(ReqInfo) == 16, "ReqInfo is 16 bytes");

// Each split unit's claim counter sits on its own 128-byte line: every warp of the unit's CTAs
// updates it once per key group, and counters sharing a line would serialise in one L2 slice.
constexpr int kClaimStride = 32;

// Max query rows one decode CTA handles per KV head (one m16 MMA tile).
constexpr int kDecodeRows = 16;

// Query rows of one prefill CTA (two 128-row tiles) and the layout of one prefill partial slot:
// lse [256] (log2 units), then O as [32 four-column groups][256 rows] float4 (coalesced per group).
constexpr int kPrefillItemRows = 256;
constexpr int kPrefillPartialFloats = kPrefillItemRows * 128;

// Everything a run kernel reads, passed by value.
struct RunParams {
  const WorkItem* work;
  const MergeItem* merge;
  const ReqInfo* req;
  const int32_t* kv_indices;
  float* part_o;    // [num_partials, 16, head_dim]
  float* part_lse;  // [num_partials, 16] (log2 units)
  float* ppart_o;    // prefill: [prefill partials, 32, 256, 4] normalised fp32 O
  float* ppart_lse;  // prefill: [prefill partials, 256] log2-sum-exp (-inf = no visible key)
  int32_t* unit_count;       // [num_merge]: partials written so far (0 between runs)
  int32_t* claim;            // [num_merge * kClaimStride]: groups claimed beyond the static ones (0 between runs)
  const void* q;
  void* o;
  float* lse;  // nullable
  const char* k_pool;
  const char* v_pool;
  int64_t stride_page_b;   // bytes
  int64_t stride_token_b;  // bytes
  int64_t stride_head_b;   // bytes
  int64_t num_pages;
  int32_t page_size;
  int32_t num_qo_heads;
  int32_t num_kv_heads;
  int32_t group;       // num_qo_heads / num_kv_heads
  int32_t head_dim;
  int32_t window_left;
  int32_t noncausal;   // prefill: 1 = every query sees all of its request's keys (0 = causal)
  int32_t ragged_kv;   // prefill: 1 = key j of request i is row page_base + j of the pools (no page table)
  int32_t merge_into;  // prefill: 1 = merge this pass's state into the state held in (o, lse) (LSE weights)
  const char* ext_k;   // prefill over two sources: contiguous new-token K rows [tokens, Hkv, D] (else null)
  const char* ext_v;
  int64_t ext_row_b;   // bytes between consecutive new-token rows
  int32_t wait_limit_k;  // prefill: bound on each in-kernel wait, in units of 1024 SM clock cycles
  int32_t hold_wait;     // prefill: 1 = the MMA thread first waits on a barrier nothing arrives at (the
                         // wait runs out and the CTA takes its timeout path; a test of that path)
  float scale_log2;    // sm_scale * log2(e) (* k_scale for FP8 KV)
  float out_scale;     // 1, or v_scale for FP8 KV
  int64_t num_work;
  int64_t num_merge;
};

// launchers (return cudaError_t of the launch)
cudaError_t launch_kv_store(const void* k, const void* v, const int64_t* slots, int64_t T, const pkv_cache& c,
                            float inv_k, float inv_v, cudaStream_t s);
cudaError_t launch_decode(const RunParams& p, int kv_dtype, cudaStream_t s);
int decode_ctas_per_sm(int kv_dtype, int head_dim, int group);  // resident decode CTAs per SM
cudaError_t launch_prefill(const RunParams& p, const void* tmap_q, const void* tmap_o, int64_t total_tokens,
                           cudaStream_t s);
int prefill_supported(const char** why);
cudaError_t launch_prefill_merge(const RunParams& p, int64_t first_merge, int64_t count, cudaStream_t s);
// copy of plan metadata from a mapped pinned host buffer (device alias src_mapped) to the workspace
cudaError_t launch_meta_copy(void* dst, const void* src_mapped, size_t bytes, cudaStream_t s);
cudaError_t launch_merge_state(const void* o_a, const float* lse_a, const void* o_b, const float* lse_b, void* o,
                               float* lse, int64_t num_states, int head_dim, cudaStream_t s);

cudaError_t read_device_error(int32_t* code, int reset, cudaStream_t s);

// record `msg` as this thread's pkv_last_error() text and return `code`
int set_last_error(int code, const char* msg);

// The run-time checks of a KV cache against a plan (geometry, page range, alignment, positive
// strides, FP8 scales); PKV_OK or an error status with its message set.
int check_cache(const pkv_plan* P, const pkv_cache* c);

}  // namespace pkv

// Host-side plan object behind the opaque pkv_plan handle.
struct pkv_plan {
  bool valid = false;
  int32_t mode = 0, batch = 0, Hq = 0, Hkv = 0, D = 0, ps = 0, window_left = -1, kv_dtype = 0, q_dtype = 0;
  bool causal = true;   // false: every query sees all keys of its request (prefill / ragged plans)
  bool ragged = false;  // PKV_MODE_RAGGED: request i reads rows kv_indptr[i].. of contiguous K/V; max_page_id = last row
  bool paged_ragged = false;  // PKV_MODE_PAGED_RAGGED: pages hold the prefix, the new rows come from k_new / v_new
  float sm_scale = 0.f;
  int64_t total_tokens = 0, max_page_id = -1, kv_tokens = 0, kv_chunk = 0, num_partials = 0;
  int64_t num_decode_work = 0;  // the decode kernel's items come first in `work`, the prefill kernel's after
  int64_t num_decode_merge = 0;  // decode merge units first in `merge`, prefill units after
  int64_t num_prefill_partials = 0;
  int64_t num_decodes = 0, num_decode_tokens = 0, num_prefills = 0, num_prefill_tokens = 0;
  std::vector<pkv::WorkItem> work;
  std::vector<pkv::MergeItem> merge;
  std::vector<pkv::ReqInfo> req;
  std::vector<int32_t> indices;
  size_t off_work = 0, off_merge = 0, off_req = 0, off_idx = 0, off_count = 0, off_claim = 0, off_plse = 0, off_po = 0;
  size_t off_pplse = 0, off_ppo = 0;  // prefill partials
  size_t meta_bytes = 0, need_bytes = 0;
  void* ws = nullptr;
  size_t ws_bytes = 0;
  void* pinned = nullptr;
  void* pinned_dev = nullptr;  // device alias of the staging buffer (null: copied by DMA instead)
  size_t pinned_bytes = 0;
  cudaEvent_t copy_done = nullptr;
  bool copy_pending = false;
  int device = -1;
};

