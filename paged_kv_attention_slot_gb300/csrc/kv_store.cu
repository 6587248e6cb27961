// The KV write: scatter this step's K/V rows into the paged pool through slot_mapping.
//
// "vLLM 源码完全拆解（六）：Attention Backend", sections «Runner 先构造公共事实» (slot =
// physical_page * page_size + offset_in_page) and «为什么 KV 写入在 Attention 之前» (the write runs
// before attention on the same stream so a query sees its own step's keys); "SGLang 源码完全拆解(八)：
// Attention Backend", section «层与后端的边界» (FP8 caches quantise on write with the same scale the
// read side uses).
//
// One thread moves one 16-byte chunk of one (token, head) row: for D = 128 bf16 a row is 16
// chunks, so a warp writes two full rows and every global access is a full 16-byte vector.  The
// kernel is a pure memory op; it is launched with enough CTAs to cover every chunk once.

#include "pkv_internal.h"
#include "ptx.cuh"

namespace pkv {

__device__ int32_t g_device_error;  // first error recorded by any kernel of this library

int32_t* device_error_ptr() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return nullptr;
  static int32_t* cache[64] = {nullptr};
  if (dev < 0 || dev >= 64) return nullptr;
  if (!cache[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) {
      cudaGetLastError();
      return nullptr;
    }
    cache[dev] = static_cast<int32_t*>(p);
  }
  return cache[dev];
}

cudaError_t read_device_error(int32_t* code, int reset, cudaStream_t s) {
  int32_t* p = device_error_ptr();
  if (!p) return cudaErrorInvalidDevice;
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return e;
  e = cudaMemcpy(code, p, sizeof(int32_t), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return e;
  if (reset) e = cudaMemset(p, 0, sizeof(int32_t));
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  return e;
}

struct StoreParams {
  const uint8_t* k;
  const uint8_t* v;
  const int64_t* slots;
  uint8_t* k_pool;
  uint8_t* v_pool;
  int64_t T;
  int64_t total_slots;
  int64_t sp_b, st_b, sh_b;  // strides in bytes
  int32_t page_size;
  int32_t heads;
  int32_t chunks;  // 16-byte source chunks per (token, head) row
  float inv_k, inv_v;
  int32_t* err;
};

template <bool FP8>
__global__ void __launch_bounds__(256) kv_store_kernel(const StoreParams p) {
  pdl_wait();
  pdl_launch_dependents();  // the attention run that follows may be scheduled now (it waits for us)
  const int64_t n = p.T * p.heads * p.chunks;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t row = i / p.chunks;  // token * heads + head
    const int c = (int)(i - row * p.chunks);
    const int64_t tok = row / p.heads;
    const int h = (int)(row - tok * p.heads);
    const int64_t slot = __ldg(p.slots + tok);
    if (slot < 0) continue;  // padding token
    if (slot >= p.total_slots) {
      record_error(p.err, PKV_DEVERR_SLOT_RANGE);
      continue;
    }
    const int64_t page = slot / p.page_size;
    const int64_t off = slot - page * p.page_size;
    const int64_t src = row * (int64_t)p.chunks * 16 + c * 16;
    const uint4 kx = __ldg(reinterpret_cast<const uint4*>(p.k + src));
    const uint4 vx = __ldg(reinterpret_cast<const uint4*>(p.v + src));
    if constexpr (!FP8) {
      const int64_t dst = page * p.sp_b + off * p.st_b + h * p.sh_b + c * 16;
      *reinterpret_cast<uint4*>(p.k_pool + dst) = kx;
      *reinterpret_cast<uint4*>(p.v_pool + dst) = vx;
    } else {
      // 8 bf16 -> 8 E4M3 codes: code = E4M3_RNE_satfinite(float(x) * inv_scale), product in fp32
      const int64_t dst = page * p.sp_b + off * p.st_b + h * p.sh_b + c * 8;
      auto quant = [](const uint4 x, float inv) {
        const uint32_t w[4] = {x.x, x.y, x.z, x.w};
        uint32_t b[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float lo = __uint_as_float(w[j] << 16) * inv;
          const float hi = __uint_as_float(w[j] & 0xffff0000u) * inv;
          b[j] = f32x2_to_e4m3x2(lo, hi);
        }
        return make_uint2(b[0] | (b[1] << 16), b[2] | (b[3] << 16));
      };
      *reinterpret_cast<uint2*>(p.k_pool + dst) = quant(kx, p.inv_k);
      *reinterpret_cast<uint2*>(p.v_pool + dst) = quant(vx, p.inv_v);
    }
  }
}

cudaError_t launch_kv_store(const void* k, const void* v, const int64_t* slots, int64_t T, const pkv_cache& c,
                            float inv_k, float inv_v, cudaStream_t s) {
  const bool fp8 = c.dtype == PKV_FP8_E4M3;
  const int64_t esz = fp8 ? 1 : 2;
  StoreParams p;
  p.k = static_cast<const uint8_t*>(k);
  p.v = static_cast<const uint8_t*>(v);
  p.slots = slots;
  p.k_pool = static_cast<uint8_t*>(c.k);
  p.v_pool = static_cast<uint8_t*>(c.v);
  p.T = T;
  p.total_slots = c.num_pages * (int64_t)c.page_size;
  p.sp_b = c.stride_page * esz;
  p.st_b = c.stride_token * esz;
  p.sh_b = c.stride_head * esz;
  p.page_size = c.page_size;
  p.heads = c.num_kv_heads;
  p.chunks = c.head_dim * 2 / 16;
  p.inv_k = inv_k;
  p.inv_v = inv_v;
  p.err = device_error_ptr();
  if (!p.err) return cudaErrorInvalidDevice;
  const int64_t n = T * p.heads * p.chunks;
  int64_t blocks = (n + 255) / 256;
  if (blocks > 152 * 16) blocks = 152 * 16;
  return fp8 ? launch_pdl(kv_store_kernel<true>, dim3((unsigned)blocks), dim3(256), 0, s, p)
             : launch_pdl(kv_store_kernel<false>, dim3((unsigned)blocks), dim3(256), 0, s, p);
}

}  // namespace pkv
