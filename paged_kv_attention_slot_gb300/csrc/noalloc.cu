// Decode for callers that cannot allocate device memory.
//
// Some hosts of this library cannot call cudaMalloc at all: code running inside another
// framework's memory pool that forbids raw allocations (an allocation behind the pool's back
// breaks its accounting or its out-of-memory handling), or embedded runtimes that are handed a
// fixed budget of device memory up front and must not grow past it.  For them,
// pkv_attn_decode_run_noalloc keeps everything the decode needs besides its inputs and outputs --
// the plan's work list, the per-request facts, the page list and the split-KV partial outputs -- in
// one file-scope __device__ array of kNoAllocScratchBytes, and runs the same decode kernel (with
// its split-KV merge) as pkv_attn_decode_run on it.
//
// The array exists once per device that loads the library and stays allocated until the process
// exits.  Every call shares it and it keeps the last call's contents; nothing in it has to start at
// zero except the per-unit split counters, which every call clears before its kernels run (every
// partial slot a call reads was written earlier in the same call).  Two calls whose
// work overlaps on the GPU (different streams, or different host threads without ordering) race
// on the array.  The first call on a device looks up the array's device address; that first call
// should be made before any stream capture begins.  Each call copies the plan's metadata from the
// plan's host arrays with ordinary (pageable) host-to-device copies.

#include <cuda_runtime.h>

#include <atomic>
#include <cstring>
#include <string>

#include "pkv_internal.h"

namespace pkv {

constexpr size_t kNoAllocScratchBytes = 32u << 20;  // 32 MiB

// The scratch itself.  In host code this name is only a stand-in for the symbol: its device
// address comes from cudaGetSymbolAddress below, never from taking the address here.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

namespace {

constexpr int kMaxDevices = 64;
// Device address of the scratch array per device, filled by the first call on that device.  Two
// host threads making that first call at once both look it up and store the same value.
std::atomic<void*> g_scratch_addr[kMaxDevices];

int noalloc_fail(int code, const std::string& msg) { return pkv::set_last_error(code, msg.c_str()); }

// Device address of the scratch array on the current device (looked up once per device).
cudaError_t scratch_address(void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  void* ptr = g_scratch_addr[dev].load(std::memory_order_acquire);
  if (!ptr) {
    e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev].store(ptr, std::memory_order_release);
  }
  *out = ptr;
  return cudaSuccess;
}

}  // namespace

}  // namespace pkv

extern "C" int pkv_attn_decode_run_noalloc(const pkv_plan* plan, const void* q, const pkv_cache* cache, void* o,
                                           float* lse, void* stream) {
  using namespace pkv;
  if (!plan || !plan->valid) return noalloc_fail(PKV_EINVAL, "plan is NULL or has not been planned");
  if (plan->mode != PKV_MODE_DECODE) return noalloc_fail(PKV_EINVAL, "needs a PKV_MODE_DECODE plan");
  if (plan->need_bytes > kNoAllocScratchBytes)
    return noalloc_fail(PKV_EWORKSPACE, "the plan needs " + std::to_string(plan->need_bytes) +
                                            " bytes of scratch; the no-allocation path has " +
                                            std::to_string(kNoAllocScratchBytes));
  // the same cache checks as every other run entry point (geometry against the plan, page range,
  // alignment, positive strides, FP8 scales)
  const int st = check_cache(plan, cache);
  if (st != PKV_OK) return st;
  const int64_t esz = cache->dtype == PKV_FP8_E4M3 ? 1 : 2;
  if (plan->total_tokens > 0 && (!q || !o)) return noalloc_fail(PKV_EINVAL, "q and o must be non-NULL");
  if (((uintptr_t)q | (uintptr_t)o) & 15) return noalloc_fail(PKV_EINVAL, "q and o must be 16-byte aligned");
  if (plan->work.empty()) return PKV_OK;

  void* ws = nullptr;
  cudaError_t e = scratch_address(&ws);
  if (e != cudaSuccess) return noalloc_fail(PKV_ECUDA, std::string("scratch lookup: ") + cudaGetErrorString(e));
  cudaStream_t s = (cudaStream_t)stream;
  char* base = static_cast<char*>(ws);
  // the plan's metadata, straight from its host arrays (stream-ordered before the kernels)
  struct Seg { size_t off; const void* src; size_t bytes; };
  const Seg segs[4] = {
      {plan->off_work, plan->work.data(), plan->work.size() * sizeof(WorkItem)},
      {plan->off_merge, plan->merge.data(), plan->merge.size() * sizeof(MergeItem)},
      {plan->off_req, plan->req.data(), plan->req.size() * sizeof(ReqInfo)},
      {plan->off_idx, plan->indices.data(), plan->indices.size() * sizeof(int32_t)},
  };
  for (const Seg& g : segs) {
    if (!g.bytes) continue;
    e = cudaMemcpyAsync(base + g.off, g.src, g.bytes, cudaMemcpyHostToDevice, s);
    if (e != cudaSuccess) return noalloc_fail(PKV_ECUDA, std::string("metadata copy: ") + cudaGetErrorString(e));
  }
  if (!plan->merge.empty()) {
    e = cudaMemsetAsync(base + plan->off_count, 0, plan->off_plse - plan->off_count, s);
    if (e != cudaSuccess) return noalloc_fail(PKV_ECUDA, std::string("counter reset: ") + cudaGetErrorString(e));
  }

  RunParams p{};
  p.work = reinterpret_cast<const WorkItem*>(base + plan->off_work);
  p.merge = reinterpret_cast<const MergeItem*>(base + plan->off_merge);
  p.req = reinterpret_cast<const ReqInfo*>(base + plan->off_req);
  p.kv_indices = reinterpret_cast<const int32_t*>(base + plan->off_idx);
  p.part_lse = reinterpret_cast<float*>(base + plan->off_plse);
  p.part_o = reinterpret_cast<float*>(base + plan->off_po);
  p.unit_count = reinterpret_cast<int32_t*>(base + plan->off_count);
  p.claim = reinterpret_cast<int32_t*>(base + plan->off_claim);
  p.q = q;
  p.o = o;
  p.lse = lse;
  p.k_pool = static_cast<const char*>(cache->k);
  p.v_pool = static_cast<const char*>(cache->v);
  p.stride_page_b = cache->stride_page * esz;
  p.stride_token_b = cache->stride_token * esz;
  p.stride_head_b = cache->stride_head * esz;
  p.num_pages = cache->num_pages;
  p.page_size = plan->ps;
  p.num_qo_heads = plan->Hq;
  p.num_kv_heads = plan->Hkv;
  p.group = plan->Hq / plan->Hkv;
  p.head_dim = plan->D;
  p.window_left = plan->window_left;
  p.scale_log2 = plan->sm_scale * 1.4426950408889634f * (cache->dtype == PKV_FP8_E4M3 ? cache->k_scale : 1.0f);
  p.out_scale = cache->dtype == PKV_FP8_E4M3 ? cache->v_scale : 1.0f;
  p.num_work = (int64_t)plan->work.size();
  p.num_merge = (int64_t)plan->merge.size();
  e = launch_decode(p, cache->dtype, s);
  if (e != cudaSuccess) return noalloc_fail(PKV_ECUDA, std::string("decode launch: ") + cudaGetErrorString(e));
  return PKV_OK;
}
