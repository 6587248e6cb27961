// Merge of two attention states by their log-sum-exp.
//
// "SGLang 源码完全拆解(八)：Attention Backend", section «extend 的两种形态»: an extend over a cached
// prefix may be computed as two passes -- the new tokens' queries over the new tokens' own K/V
// (causal) and over the cached prefix (every key visible) -- and the two normalised outputs are
// combined with the weights e^(s_a - m), e^(s_b - m), m = max(s_a, s_b), where s is each pass's
// natural-log log-sum-exp.  "vLLM 源码完全拆解（六）：Attention Backend", section «Cascade Attention
// 把共享前缀只算一次» combines a shared-prefix pass with per-request suffix passes the same way.
//
// The op is a pure stream over HBM: per state it reads two bf16 rows and two floats and writes one
// bf16 row (and a float).  Layout: 16 lanes per 128-wide state (8 per 64-wide state), one 16-byte
// vector each, so a warp moves two (four) whole rows per instruction, coalesced.  The grid is a
// multiple of the SM count and strides over the states.

#include <cuda_bf16.h>
#include <math.h>

#include "pkv_internal.h"
#include "ptx.cuh"

namespace pkv {

namespace {

constexpr int kMergeThreads = 256;

__device__ __forceinline__ void unpack8(const uint4& u, float* f) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}

template <int LANES>  // lanes per state: head_dim / 8
__global__ void __launch_bounds__(kMergeThreads) merge_state_kernel(const uint4* o_a, const float* lse_a,
                                                                     const uint4* o_b, const float* lse_b, uint4* o,
                                                                     float* lse, int64_t num_states) {
  // plain loads throughout: o may alias o_a or o_b, and lse may alias lse_a or lse_b
  constexpr int per_warp = 32 / LANES;
  const int lane = threadIdx.x & 31, sub = lane % LANES;
  const int64_t warps = (int64_t)gridDim.x * (kMergeThreads / 32);
  for (int64_t w0 = ((int64_t)blockIdx.x * (kMergeThreads / 32) + (threadIdx.x >> 5)) * per_warp; w0 < num_states;
       w0 += warps * per_warp) {  // warp-uniform loop
    const int64_t st = w0 + lane / LANES;
    const bool valid = st < num_states;
    const int64_t at = st * LANES + sub;
    float sa = -INFINITY, sb = -INFINITY;
    uint4 ua = make_uint4(0u, 0u, 0u, 0u), ub = ua;
    if (valid) {
      sa = lse_a[st];
      sb = lse_b[st];
      ua = o_a[at];
      ub = o_b[at];
    }
    const float m = fmaxf(sa, sb);
    float wa = 0.f, wb = 0.f, s = -INFINITY;
    if (m != -INFINITY) {  // at least one state is non-empty
      wa = expf(sa - m);
      wb = expf(sb - m);
      s = m + logf(wa + wb);
      const float inv = 1.f / (wa + wb);
      wa *= inv;
      wb *= inv;
    }
    float fa[8], fb[8];
    unpack8(ua, fa);
    unpack8(ub, fb);
    uint4 r;
    r.x = pack_bf16(fa[0] * wa + fb[0] * wb, fa[1] * wa + fb[1] * wb);
    r.y = pack_bf16(fa[2] * wa + fb[2] * wb, fa[3] * wa + fb[3] * wb);
    r.z = pack_bf16(fa[4] * wa + fb[4] * wb, fa[5] * wa + fb[5] * wb);
    r.w = pack_bf16(fa[6] * wa + fb[6] * wb, fa[7] * wa + fb[7] * wb);
    __syncwarp();  // every lane has read its state's LSEs before one lane overwrites them in place
    if (valid) {
      o[at] = r;
      if (lse && sub == 0) lse[st] = s;
    }
  }
}

}  // namespace

cudaError_t launch_merge_state(const void* o_a, const float* lse_a, const void* o_b, const float* lse_b, void* o,
                               float* lse, int64_t num_states, int head_dim, cudaStream_t s) {
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const int lanes = head_dim / 8;
  const int64_t per_block = kMergeThreads / lanes;  // states per block per iteration
  const int64_t need = (num_states + per_block - 1) / per_block;
  const int64_t grid = std::min<int64_t>(need, (int64_t)sms * 8);  // 8 resident 256-thread blocks per SM
  if (head_dim == 128)
    merge_state_kernel<16><<<(unsigned)grid, kMergeThreads, 0, s>>>(
        (const uint4*)o_a, lse_a, (const uint4*)o_b, lse_b, (uint4*)o, lse, num_states);
  else
    merge_state_kernel<8><<<(unsigned)grid, kMergeThreads, 0, s>>>(
        (const uint4*)o_a, lse_a, (const uint4*)o_b, lse_b, (uint4*)o, lse, num_states);
  return cudaGetLastError();
}

// Copy of a plan's metadata from its pinned staging buffer, read directly through the buffer's
// device mapping (on GB300 the Grace memory is reachable over NVLink-C2C): a few CTAs with four
// 16-byte loads in flight per thread finish well before a DMA copy of the same ~100 KB has
// paid its fixed start-up latency.  bytes is a multiple of 16; both pointers are 16-byte aligned.
constexpr int kMetaThreads = 256, kMetaUnroll = 4;
__global__ void __launch_bounds__(kMetaThreads) meta_copy_kernel(uint4* dst, const uint4* src, int64_t n16) {
  pdl_launch_dependents();
  const int64_t base = (int64_t)blockIdx.x * (kMetaThreads * kMetaUnroll) + threadIdx.x;
  uint4 v[kMetaUnroll];
  // the staging buffer is written by the host before the launch, by no kernel: read it at once
#pragma unroll
  for (int u = 0; u < kMetaUnroll; ++u) {
    const int64_t i = base + u * kMetaThreads;
    if (i < n16) v[u] = src[i];
  }
  pdl_wait();  // an earlier kernel (a run of the previous plan) may still read the workspace
#pragma unroll
  for (int u = 0; u < kMetaUnroll; ++u) {
    const int64_t i = base + u * kMetaThreads;
    if (i < n16) dst[i] = v[u];
  }
}

cudaError_t launch_meta_copy(void* dst, const void* src_mapped, size_t bytes, cudaStream_t s) {
  const int64_t n16 = (int64_t)(bytes / 16);
  if (n16 == 0) return cudaSuccess;
  const int64_t per_cta = kMetaThreads * kMetaUnroll;
  return launch_pdl(meta_copy_kernel, dim3((unsigned)((n16 + per_cta - 1) / per_cta)), dim3(kMetaThreads), 0, s,
                    static_cast<uint4*>(dst), static_cast<const uint4*>(src_mapped), n16);
}

}  // namespace pkv
