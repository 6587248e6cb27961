// Batched paged decode (one new token per request) with the split-KV merge fused in.
//
// What it computes: for request i, KV head h and every query head of h's group, the softmax over
// the visible keys of the scaled scores q.k_j, applied to v_j, with K/V read through the CSR page
// table ("SGLang 源码完全拆解(八)：Attention Backend", sections «统一元数据的编译» and «其他后端的元数据»
// (split-KV: partial outputs and log-sum-exps per KV chunk, merged by a reduction); "手写 mini-sglang
// 阶段四 · GPU 注意力后端", section «FlashInfer：plan 与 run»: with a GQA group >= 4, decode is a chain of
// small matrix products and tensor cores pay).
//
// GB300 design.  Decode is HBM-bound (about G flops per byte of KV), so the kernel is built around
// streaming the pages at full bandwidth:
//  * one CTA = 4 warps = one work item (request, KV head, head group of <= 16 query heads, KV chunk);
//    the planner cuts long sequences into equal chunks and launches CTAs longest first;
//  * every warp runs its own cp.async ring (16 keys per stage, K and V rows gathered page by page
//    through kv_indices, 16-byte vectors, XOR-swizzled so ldmatrix reads are conflict-free) and takes
//    every 4th 16-key tile of the chunk, so no CTA-wide barrier sits in the main loop;
//  * the query heads of one KV head are packed into the M dimension of an m16n8k16 tensor-core MMA,
//    so each K/V row is read from HBM exactly once per KV head; S = Q K^T and O += P V both run on
//    the tensor cores with fp32 accumulation, and the online softmax lives in the MMA fragments
//    (warp shuffles across the 4 lanes of a row);
//  * FP8 (E4M3) pages are widened to f16 in registers (exact), the K scale is folded into the score
//    scale and the V scale into the output; for FP8 the head-dim order inside each 16-element block
//    is permuted identically for Q and K (a sum does not depend on order) so that one ldmatrix feeds
//    two code bytes per register half directly;
//  * the 4 warps merge their softmax states through shared memory at the end; a CTA either writes
//    the final bf16 output (no split) or a normalised fp32 partial plus its log2-sum-exp; the last
//    CTA of a split unit to finish (an atomic count per unit, reset after use, no waiting) merges
//    the unit: m = max lse_s, o = sum_s 2^(lse_s - m) o_s / sum_s 2^(lse_s - m).

#include <cuda_bf16.h>
#include <math.h>

#include "pkv_internal.h"
#include "ptx.cuh"

namespace pkv {

int32_t* device_error_ptr();

template <int D, bool FP8>
struct DecodeCfg {
  static constexpr int ROWB = FP8 ? D : 2 * D;  // bytes per key row of one head
  static constexpr int CH = ROWB / 16;          // 16-byte chunks per row
  static constexpr int KEYS = 16;               // keys per warp tile
  static constexpr int TILE_B = KEYS * ROWB;    // bytes of one K (or V) tile
  static constexpr int STAGES = (2 * TILE_B <= 4096) ? 6 : 3;
  static constexpr int WARPS = 4;
  static constexpr int WARP_SMEM = STAGES * 2 * TILE_B;
  static constexpr int PIPE_SMEM = WARPS * WARP_SMEM;
  static constexpr int MERGE_SMEM = (WARPS * kDecodeRows * D + 2 * WARPS * kDecodeRows + WARPS * kDecodeRows) * 4;
  static constexpr int SMEM = PIPE_SMEM > MERGE_SMEM ? PIPE_SMEM : MERGE_SMEM;
  static constexpr int NB = D / 8;   // 8-column n-blocks of O
  static constexpr int KS = D / 16;  // k-steps of Q K^T
  static_assert(CH >= 8, "rows must span at least 8 chunks for the XOR swizzle");
};

// Column (head-dim index) of accumulator element j (0..3) of O n-block nb for lane quad t.
template <bool FP8>
__device__ __forceinline__ int o_col(int nb, int j, int t) {
  if constexpr (!FP8) {
    return nb * 8 + 2 * t + (j & 1);
  } else {
    // n-block nb = 2 * chunk + parity covers head dims 16 * chunk + 2 n + parity
    return (nb >> 1) * 16 + 4 * t + 2 * (j & 1) + (nb & 1);
  }
}

template <int D, bool FP8>
__global__ void __launch_bounds__(128, 2) decode_kernel(const RunParams p, int32_t* err) {
  using C = DecodeCfg<D, FP8>;
  extern __shared__ __align__(128) uint8_t smem[];

  const WorkItem w = p.work[blockIdx.x];
  const ReqInfo ri = p.req[w.req];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int g = lane >> 2;
  const int t = lane & 3;
  const int qh0 = w.kv_head * p.group + w.head_group * kDecodeRows;
  const int rows = min(kDecodeRows, p.group - w.head_group * kDecodeRows);

  // ---- Q fragments (A operand, rows = query heads of this group, zero beyond `rows`) ----
  uint32_t qa[C::KS][4];
  {
    const uint16_t* qb = static_cast<const uint16_t*>(p.q) + ((int64_t)w.q_row * p.num_qo_heads + qh0) * D;
    const uint16_t* r0 = qb + (int64_t)g * D;
    const uint16_t* r1 = qb + (int64_t)(g + 8) * D;
    const bool v0 = g < rows, v1 = g + 8 < rows;
#pragma unroll
    for (int ks = 0; ks < C::KS; ++ks) {
      if constexpr (!FP8) {
        const int c0 = ks * 16 + 2 * t;
        qa[ks][0] = v0 ? *reinterpret_cast<const uint32_t*>(r0 + c0) : 0u;
        qa[ks][1] = v1 ? *reinterpret_cast<const uint32_t*>(r1 + c0) : 0u;
        qa[ks][2] = v0 ? *reinterpret_cast<const uint32_t*>(r0 + c0 + 8) : 0u;
        qa[ks][3] = v1 ? *reinterpret_cast<const uint32_t*>(r1 + c0 + 8) : 0u;
      } else {
        // permuted order: logical k {2t, 2t+1} <- dims 16ks+4t+{0,1}; {2t+8, 2t+9} <- 16ks+4t+{2,3}
        const int c0 = ks * 16 + 4 * t;
        uint2 x0 = v0 ? *reinterpret_cast<const uint2*>(r0 + c0) : make_uint2(0, 0);
        uint2 x1 = v1 ? *reinterpret_cast<const uint2*>(r1 + c0) : make_uint2(0, 0);
        auto cv = [](uint32_t two_bf16) {
          return pack_f16(__uint_as_float(two_bf16 << 16), __uint_as_float(two_bf16 & 0xffff0000u));
        };
        qa[ks][0] = cv(x0.x);
        qa[ks][1] = cv(x1.x);
        qa[ks][2] = cv(x0.y);
        qa[ks][3] = cv(x1.y);
      }
    }
  }

  // ---- per-warp cp.async ring ----
  uint8_t* wsm = smem + warp * C::WARP_SMEM;
  const uint32_t wsm_u = smem_u32(wsm);
  const int n_keys = w.kv_end - w.kv_begin;
  const int n_tiles = (n_keys + C::KEYS - 1) / C::KEYS;
  const int my_tiles = n_tiles > warp ? (n_tiles - warp + C::WARPS - 1) / C::WARPS : 0;
  const int lr = lane & 15;  // row whose page this lane resolves
  const int64_t head_off = (int64_t)w.kv_head * p.stride_head_b;

  // Lane lr (0..15) resolves the page of row lr of a tile; then every warp-wide cp.async covers
  // 32 / CH whole rows with consecutive lanes on consecutive 16-byte chunks (fully coalesced).
  constexpr int RPI = 32 / C::CH;  // rows per warp instruction
  const int lc = lane % C::CH;
  const int lsub = lane / C::CH;
  // The page id of the row this lane resolves is fetched one tile ahead (this warp's next tile is
  // 4 tiles = 64 keys further), so the index load never stalls the issue of the copies.
  auto fetch_page = [&](int key) -> int {
    return key < w.kv_end ? __ldg(p.kv_indices + ri.page_base + key / p.page_size) : 0;
  };
  int next_page = fetch_page(w.kv_begin + warp * C::KEYS + lr);
  auto load_tile = [&](int i, int stage) {
    const int key = w.kv_begin + (warp + i * C::WARPS) * C::KEYS + lr;
    const int page = next_page;
    next_page = fetch_page(key + C::WARPS * C::KEYS);
    int64_t roff = -1;
    if (key < w.kv_end) {
      const int lp = key / p.page_size;
      const int off = key - lp * p.page_size;
      if ((unsigned long long)(unsigned)page >= (unsigned long long)p.num_pages)
        record_error(err, PKV_DEVERR_PAGE_RANGE);
      else
        roff = (int64_t)page * p.stride_page_b + (int64_t)off * p.stride_token_b + head_off;
    }
    const uint32_t dk = wsm_u + stage * 2 * C::TILE_B;
    const uint32_t dv = dk + C::TILE_B;
#pragma unroll
    for (int j = 0; j < C::KEYS / RPI; ++j) {
      const int row = j * RPI + lsub;
      const int64_t o = __shfl_sync(0xffffffffu, roff, row);
      const uint32_t sw = row * C::ROWB + ((lc ^ (row & 7)) << 4);
      const bool ok = o >= 0;
      cp_async16(dk + sw, ok ? p.k_pool + o + lc * 16 : p.k_pool, ok ? 16u : 0u);
      cp_async16(dv + sw, ok ? p.v_pool + o + lc * 16 : p.v_pool, ok ? 16u : 0u);
    }
  };

  float m0 = -INFINITY, m1 = -INFINITY;  // running max (log2 units) of rows g and g + 8
  float l0 = 0.f, l1 = 0.f;              // running sums (this lane's columns only)
  float o[C::NB][4];
#pragma unroll
  for (int nb = 0; nb < C::NB; ++nb) o[nb][0] = o[nb][1] = o[nb][2] = o[nb][3] = 0.f;

#pragma unroll
  for (int s = 0; s < C::STAGES - 1; ++s) {
    if (s < my_tiles) load_tile(s, s);
    cp_async_commit();
  }

  // ldmatrix lane roles
  const int mi = lane >> 3, rr = lane & 7;
  const int k_key = FP8 ? (((mi & 1) << 3) + rr) : (((mi >> 1) << 3) + rr);
  const int v_key = ((mi & 1) << 3) + rr;

  for (int i = 0; i < my_tiles; ++i) {
    cp_async_wait<C::STAGES - 2>();
    __syncwarp();
    const int stage = i % C::STAGES;
    const uint32_t kb = wsm_u + stage * 2 * C::TILE_B;
    const uint32_t vb = kb + C::TILE_B;
    const int key0 = w.kv_begin + (warp + i * C::WARPS) * C::KEYS;

    // ---- S = Q K^T for 16 keys (two n-blocks of 8) ----
    float s[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    if constexpr (!FP8) {
#pragma unroll
      for (int ks = 0; ks < C::KS; ++ks) {
        uint32_t b[4];
        const int chunk = 2 * ks + (mi & 1);
        ldsm_x4(b, kb + k_key * C::ROWB + ((chunk ^ (k_key & 7)) << 4));
        mma_bf16(s[0], qa[ks], b[0], b[1]);
        mma_bf16(s[1], qa[ks], b[2], b[3]);
      }
    } else {
#pragma unroll
      for (int c = 0; c < C::KS; c += 2) {
        uint32_t b[4];
        const int chunk = c + (mi >> 1);
        ldsm_x4(b, kb + k_key * C::ROWB + ((chunk ^ (k_key & 7)) << 4));
        // b[0]: keys 0-7 / chunk c, b[1]: keys 8-15 / chunk c, b[2], b[3]: chunk c + 1
        mma_f16(s[0], qa[c], e4m3x2_to_f16x2(b[0] & 0xffffu), e4m3x2_to_f16x2(b[0] >> 16));
        mma_f16(s[1], qa[c], e4m3x2_to_f16x2(b[1] & 0xffffu), e4m3x2_to_f16x2(b[1] >> 16));
        mma_f16(s[0], qa[c + 1], e4m3x2_to_f16x2(b[2] & 0xffffu), e4m3x2_to_f16x2(b[2] >> 16));
        mma_f16(s[1], qa[c + 1], e4m3x2_to_f16x2(b[3] & 0xffffu), e4m3x2_to_f16x2(b[3] >> 16));
      }
    }

    // ---- online softmax (log2 domain) ----
    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
    for (int nb = 0; nb < 2; ++nb) {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int key = key0 + nb * 8 + 2 * t + (j & 1);
        s[nb][j] = key < w.kv_end ? s[nb][j] * p.scale_log2 : -INFINITY;
      }
      mx0 = fmaxf(mx0, fmaxf(s[nb][0], s[nb][1]));
      mx1 = fmaxf(mx1, fmaxf(s[nb][2], s[nb][3]));
    }
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
    const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
    const float c0 = ex2(m0 - mn0), c1 = ex2(m1 - mn1);
    m0 = mn0;
    m1 = mn1;
    float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
    for (int nb = 0; nb < 2; ++nb) {
      s[nb][0] = ex2(s[nb][0] - mn0);
      s[nb][1] = ex2(s[nb][1] - mn0);
      s[nb][2] = ex2(s[nb][2] - mn1);
      s[nb][3] = ex2(s[nb][3] - mn1);
      ps0 += s[nb][0] + s[nb][1];
      ps1 += s[nb][2] + s[nb][3];
    }
    l0 = l0 * c0 + ps0;
    l1 = l1 * c1 + ps1;
#pragma unroll
    for (int nb = 0; nb < C::NB; ++nb) {
      o[nb][0] *= c0;
      o[nb][1] *= c0;
      o[nb][2] *= c1;
      o[nb][3] *= c1;
    }

    // ---- O += P V ----
    uint32_t pa[4];
    if constexpr (!FP8) {
      pa[0] = pack_bf16(s[0][0], s[0][1]);
      pa[1] = pack_bf16(s[0][2], s[0][3]);
      pa[2] = pack_bf16(s[1][0], s[1][1]);
      pa[3] = pack_bf16(s[1][2], s[1][3]);
#pragma unroll
      for (int dn = 0; dn < D / 16; ++dn) {
        uint32_t b[4];
        const int chunk = 2 * dn + (mi >> 1);
        ldsm_x4_t(b, vb + v_key * C::ROWB + ((chunk ^ (v_key & 7)) << 4));
        mma_bf16(o[2 * dn], pa, b[0], b[1]);
        mma_bf16(o[2 * dn + 1], pa, b[2], b[3]);
      }
    } else {
      pa[0] = pack_f16(s[0][0], s[0][1]);
      pa[1] = pack_f16(s[0][2], s[0][3]);
      pa[2] = pack_f16(s[1][0], s[1][1]);
      pa[3] = pack_f16(s[1][2], s[1][3]);
#pragma unroll
      for (int c = 0; c < D / 16; c += 2) {
        uint32_t b[4];
        const int chunk = c + (mi >> 1);
        ldsm_x4_t(b, vb + v_key * C::ROWB + ((chunk ^ (v_key & 7)) << 4));
        // b[0]: keys 0-7 x chunk c, b[1]: keys 8-15 x chunk c, b[2]/b[3]: chunk c + 1.  Each register
        // holds, for byte pair column g: (key 2t: d, d+1), (key 2t+1: d, d+1) with d = 16 chunk + 2g.
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          const uint32_t lo = b[2 * q], hi = b[2 * q + 1];
          const uint32_t e0 = e4m3x2_to_f16x2(__byte_perm(lo, 0, 0x0020));
          const uint32_t e1 = e4m3x2_to_f16x2(__byte_perm(hi, 0, 0x0020));
          const uint32_t d0 = e4m3x2_to_f16x2(__byte_perm(lo, 0, 0x0031));
          const uint32_t d1 = e4m3x2_to_f16x2(__byte_perm(hi, 0, 0x0031));
          mma_f16(o[2 * (c + q)], pa, e0, e1);
          mma_f16(o[2 * (c + q) + 1], pa, d0, d1);
        }
      }
    }
    __syncwarp();
    const int nx = i + C::STAGES - 1;
    if (nx < my_tiles) load_tile(nx, nx % C::STAGES);
    cp_async_commit();
  }
  cp_async_wait<0>();

  // full row sums across the 4 lanes of each row
  l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
  l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 2);

  // ---- merge the 4 warps' states through shared memory ----
  __syncthreads();
  float* so = reinterpret_cast<float*>(smem);                 // [4][16][D]
  float* sm = so + C::WARPS * kDecodeRows * D;                // [4][16]
  float* sl = sm + C::WARPS * kDecodeRows;                    // [4][16]
  float* sf = sl + C::WARPS * kDecodeRows;                    // [4][16] weights
  if (t == 0) {
    sm[warp * kDecodeRows + g] = m0;
    sm[warp * kDecodeRows + g + 8] = m1;
    sl[warp * kDecodeRows + g] = l0;
    sl[warp * kDecodeRows + g + 8] = l1;
  }
#pragma unroll
  for (int nb = 0; nb < C::NB; ++nb) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int r = g + ((j >> 1) << 3);
      so[(warp * kDecodeRows + r) * D + o_col<FP8>(nb, j, t)] = o[nb][j];
    }
  }
  __syncthreads();
  __shared__ float s_lse2[kDecodeRows];
  if (threadIdx.x < kDecodeRows) {
    const int r = threadIdx.x;
    float M = -INFINITY;
#pragma unroll
    for (int k = 0; k < C::WARPS; ++k) M = fmaxf(M, sm[k * kDecodeRows + r]);
    float W = 0.f;
    float e[C::WARPS];
#pragma unroll
    for (int k = 0; k < C::WARPS; ++k) {
      e[k] = ex2(sm[k * kDecodeRows + r] - M);
      W += e[k] * sl[k * kDecodeRows + r];
    }
    const float inv = W > 0.f ? 1.f / W : 0.f;
#pragma unroll
    for (int k = 0; k < C::WARPS; ++k) sf[k * kDecodeRows + r] = e[k] * inv;
    s_lse2[r] = M + __log2f(W);
  }
  __syncthreads();
  if (w.out_slot < 0) {
    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.o) + ((int64_t)w.q_row * p.num_qo_heads + qh0) * D;
    for (int idx = threadIdx.x; idx < rows * D; idx += blockDim.x) {
      const int r = idx / D, d = idx - r * D;
      float acc = 0.f;
#pragma unroll
      for (int k = 0; k < C::WARPS; ++k) acc += sf[k * kDecodeRows + r] * so[(k * kDecodeRows + r) * D + d];
      out[idx] = __float2bfloat16_rn(acc * p.out_scale);
    }
    if (p.lse && threadIdx.x < rows)
      p.lse[(int64_t)w.q_row * p.num_qo_heads + qh0 + threadIdx.x] = s_lse2[threadIdx.x] * 0.69314718055994531f;
  } else {
    float* po = p.part_o + (int64_t)w.out_slot * kDecodeRows * D;
    for (int idx = threadIdx.x; idx < rows * D; idx += blockDim.x) {
      const int r = idx / D, d = idx - r * D;
      float acc = 0.f;
#pragma unroll
      for (int k = 0; k < C::WARPS; ++k) acc += sf[k * kDecodeRows + r] * so[(k * kDecodeRows + r) * D + d];
      po[idx] = acc;
    }
    if (threadIdx.x < rows) p.part_lse[(int64_t)w.out_slot * kDecodeRows + threadIdx.x] = s_lse2[threadIdx.x];
    // The last chunk of a (request, KV head, group) to finish merges all of its partials:
    // m = max lse_s, o = sum_s 2^(lse_s - m) o_s / sum_s 2^(lse_s - m).  No CTA waits for another.
    __shared__ int s_last;
    __threadfence();
    __syncthreads();
    const int unit = p.slot_unit[w.out_slot];
    const MergeItem m = p.merge[unit];
    if (threadIdx.x == 0) {
      const int done = atomicAdd(p.unit_count + unit, 1);
      s_last = done == m.num_splits - 1;
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    __shared__ float sM[kDecodeRows], sInv[kDecodeRows];
    const float* lse = p.part_lse + (int64_t)m.first_slot * kDecodeRows;
    if (threadIdx.x < rows) {
      const int r = threadIdx.x;
      float M = -INFINITY;
      for (int s = 0; s < m.num_splits; ++s) M = fmaxf(M, __ldcg(lse + s * kDecodeRows + r));
      float W = 0.f;
      for (int s = 0; s < m.num_splits; ++s) W += ex2(__ldcg(lse + s * kDecodeRows + r) - M);
      sM[r] = M;
      sInv[r] = 1.f / W;
      if (p.lse) p.lse[(int64_t)m.q_row * p.num_qo_heads + qh0 + r] = (M + __log2f(W)) * 0.69314718055994531f;
    }
    __syncthreads();
    const float* pm = p.part_o + (int64_t)m.first_slot * kDecodeRows * D;
    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.o) + ((int64_t)m.q_row * p.num_qo_heads + qh0) * D;
    for (int idx = threadIdx.x; idx < rows * D; idx += blockDim.x) {
      const int r = idx / D;
      const float M = sM[r];
      float acc = 0.f;
      for (int s = 0; s < m.num_splits; ++s)
        acc += ex2(__ldcg(lse + s * kDecodeRows + r) - M) * __ldcg(pm + (int64_t)s * kDecodeRows * D + idx);
      out[idx] = __float2bfloat16_rn(acc * sInv[r] * p.out_scale);
    }
    if (threadIdx.x == 0) p.unit_count[unit] = 0;  // ready for the next run of this plan
  }
}

template <int D, bool FP8>
static cudaError_t launch_decode_t(const RunParams& p, cudaStream_t s) {
  using C = DecodeCfg<D, FP8>;
  static bool attr_set[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(decode_kernel<D, FP8>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  int32_t* err = device_error_ptr();
  if (!err) return cudaErrorInvalidDevice;
  decode_kernel<D, FP8><<<(unsigned)p.num_work, 128, C::SMEM, s>>>(p, err);
  return cudaGetLastError();
}

cudaError_t launch_decode(const RunParams& p, int kv_dtype, cudaStream_t s) {
  if (kv_dtype == PKV_FP8_E4M3) {
    if (p.head_dim == 128) return launch_decode_t<128, true>(p, s);
    return cudaErrorInvalidValue;
  }
  if (p.head_dim == 128) return launch_decode_t<128, false>(p, s);
  if (p.head_dim == 64) return launch_decode_t<64, false>(p, s);
  return cudaErrorInvalidValue;
}

}  // namespace pkv
