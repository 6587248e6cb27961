// Causal prefill / prefix-cached extend over a paged KV cache on 5th-generation tensor cores.
//
// What it computes: new token t of request i sits at position P = L_i - n_i + t and attends to keys
// 0..P of the request (bottom-right-aligned causal mask, optional window keeping keys >= P - w),
// gathered through the request's page list; query head h reads KV head h / G.  The new tokens' own
// K/V were written into the pool beforehand, so one paged pass covers prefix + new tokens
// ("vLLM 源码完全拆解（六）：Attention Backend", sections «为什么 KV 写入在 Attention 之前» and «FlashAttention
// Builder 的结果»: multi-token queries apply the causal mask inside their own request only;
// "手写 mini-sglang 阶段四 · GPU 注意力后端", section «在 CPU 上验证»: queries are the last n positions).
//
// GB300 design (one CTA = 128 query rows x one KV head; rows are (token, head) pairs of the KV
// head's query-head group, so every K/V tile feeds all G heads):
//  * warps 9-12 (producers): the Q tile by one 3-D TMA box; K (warps 9-10) and V (warps 11-12) tiles of
//    128 keys gathered row by row through the page table with 16-byte cp.async, 16 lanes per
//    256-byte row (fully coalesced), written straight into the 128-byte-swizzled K-major layout
//    the tensor core reads, double-buffered; each producer thread waits for its own copies, fences
//    them into the async proxy and arrives on the stage's mbarrier.  (TMA tile::gather4 moves only
//    512 bytes per instruction; issued one lane at a time it was the bottleneck for token-granular
//    pools, which is why the rows go through cp.async instead);
//  * warp 8 (MMA): one elected thread issues tcgen05.mma (M=128, N=128, K=16, bf16 in, fp32 out):
//    S_j = Q K_j^T into one of two TMEM score buffers, and O += P_{j-1} V_{j-1} into a TMEM output
//    accumulator, software-pipelined so S_j runs while the softmax works on tile j-1;
//  * warps 0-7 (softmax): warp w owns query rows 32 (w % 4) .. +31 (= its TMEM lanes) and key
//    columns 64 (w / 4) .. +63 of every tile: one tcgen05.ld of its 64 scores, causal/window mask on
//    diagonal tiles only, row maximum shared with the partner warp of the other column half through
//    shared memory and a 2-arrival mbarrier (bounded wait), online softmax in base 2 with the score scale
//    folded into one FFMA before ex2, and a lazy rescale (the reference maximum only moves when a
//    row's maximum grows by more than 2^8, exact because numerator and denominator share the
//    reference); P written as bf16 into a swizzled shared tile for the next MMA, O rescaled in TMEM
//    only when needed, then the final O / l and log-sum-exp.
// Every wait is bounded: on timeout the CTA records PKV_DEVERR_TIMEOUT, waits (bounded) for its
// own copies and MMAs, frees its TMEM and exits.

#include <cuda.h>
#include <cuda_bf16.h>
#include <math.h>

#include "pkv_internal.h"
#include "ptx.cuh"
#include "tc.cuh"

namespace pkv {

int32_t* device_error_ptr();

namespace pf {
constexpr int ROWS = 128;               // query rows per CTA
constexpr int KT = 128;                 // keys per K/V tile
constexpr int D = 128;                  // head dim
constexpr int HALF_B = ROWS * 128;      // one 64-column half of a 128-row bf16 tile (16 KB)
constexpr int TILE_B = 2 * HALF_B;      // 32 KB
constexpr int STAGES = 2;
constexpr int OFF_Q = 0;
constexpr int OFF_K = OFF_Q + TILE_B;
constexpr int OFF_V = OFF_K + STAGES * TILE_B;
constexpr int OFF_P = OFF_V + STAGES * TILE_B;
constexpr int OFF_BAR = OFF_P + TILE_B;
constexpr int NUM_BARS = 32;
constexpr int OFF_TMEM = OFF_BAR + NUM_BARS * 8;
constexpr int OFF_ABORT = OFF_TMEM + 8;
constexpr int OFF_XCH = OFF_ABORT + 8;               // row-max exchange [2 tiles][2 halves][128] + sums
constexpr int SMEM_USED = OFF_XCH + (2 * 2 * 128 + 2 * 128) * 4;
constexpr int SMEM_ALLOC = SMEM_USED + 1024;  // room to align the base to 1024 bytes
enum {
  B_Q = 0, B_KF = 1, B_VF = 3, B_KE = 5, B_VE = 7, B_SF = 9, B_SE = 11, B_PF = 13, B_OD = 14, B_FIN = 15,
  B_XM = 16,  // [4 row quarters][2 tile parities]: the two column-half warps exchanged their maxima
  B_XL = 24   // [4 row quarters]: the two column-half warps exchanged their final row sums
};
constexpr uint32_t TMEM_COLS = 512;     // S0 [0,128), S1 [128,256), O [256,384)
constexpr uint32_t TMEM_O = 256;
constexpr int THREADS = 416;  // 8 softmax warps, 1 MMA warp, 2 K-producer warps, 2 V-producer warps
constexpr int SOFTMAX_WARPS = 8;
constexpr int MMA_WARP = 8;
constexpr int PRODUCER_WARP0 = 9;
constexpr int PRODUCER_THREADS = 64;  // per operand (K or V)
constexpr long long WAIT_LIMIT = 4000000000LL;  // clock cycles (about 2 s)
constexpr float RESCALE_THRESHOLD = 8.0f;      // log2 units
}  // namespace pf

__global__ void __launch_bounds__(pf::THREADS, 1)
    prefill_kernel(const RunParams p, const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                   const __grid_constant__ CUtensorMap tv, int32_t* err) {
  using namespace pf;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u = smem_u32(smem_raw);
  const uint32_t base = (raw_u + 1023u) & ~1023u;
  uint8_t* sbase = smem_raw + (base - raw_u);
  const uint32_t sQ = base + OFF_Q, sK = base + OFF_K, sV = base + OFF_V, sP = base + OFF_P;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sbase + OFF_ABORT);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sbase + OFF_TMEM);
#define BAR(i) (base + OFF_BAR + 8u * (uint32_t)(i))

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const WorkItem w = p.work[blockIdx.x];
  const ReqInfo ri = p.req[w.req];
  const int G = p.group;
  const int nkt = (w.kv_end - w.kv_begin + KT - 1) / KT;

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    tc::mbar_init(BAR(B_Q), 1);
    for (int s = 0; s < STAGES; ++s) {
      tc::mbar_init(BAR(B_KF + s), PRODUCER_THREADS);
      tc::mbar_init(BAR(B_VF + s), PRODUCER_THREADS);
      tc::mbar_init(BAR(B_KE + s), 1);
      tc::mbar_init(BAR(B_VE + s), 1);
      tc::mbar_init(BAR(B_SF + s), 1);
      tc::mbar_init(BAR(B_SE + s), SOFTMAX_WARPS);
    }
    tc::mbar_init(BAR(B_PF), SOFTMAX_WARPS);
    tc::mbar_init(BAR(B_OD), 1);
    tc::mbar_init(BAR(B_FIN), 1);
    for (int i = 0; i < 8; ++i) tc::mbar_init(BAR(B_XM + i), 2);
    for (int i = 0; i < 4; ++i) tc::mbar_init(BAR(B_XL + i), 2);
    tc::mbar_fence_init();
  }
  if (warp == MMA_WARP) {
    tc::tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  if (warp >= PRODUCER_WARP0) {
    // ------------------------------------------------------------------ producers (cp.async)
    const bool is_k = warp < PRODUCER_WARP0 + 2;
    const int pw = (warp - PRODUCER_WARP0) & 1;  // which 64-row half of the tile this warp fills
    const char* pool = is_k ? p.k_pool : p.v_pool;
    const uint32_t s_base = is_k ? sK : sV;
    const uint32_t full0 = is_k ? BAR(B_KF) : BAR(B_VF);
    const uint32_t empty0 = is_k ? BAR(B_KE) : BAR(B_VE);
    if (warp == PRODUCER_WARP0 && lane == 0) {
      tc::tma_prefetch_desc(&tq);
      tc::mbar_arrive_expect_tx(BAR(B_Q), TILE_B);
      tc::tma_load_3d(sQ, &tq, BAR(B_Q), 0, w.kv_head * G, w.q_row);
      tc::tma_load_3d(sQ + HALF_B, &tq, BAR(B_Q), 64, w.kv_head * G, w.q_row);
    }
    const int64_t head_off = (int64_t)w.kv_head * p.stride_head_b;
    const int c = lane & 15;  // 16-byte chunk of the 256-byte row
    const int half = c >> 3, cc = c & 7;
    auto slot_of = [&](int key) -> int {
      if (key >= w.kv_end) return -1;
      const int lp = key / p.page_size;
      const int page = __ldg(p.kv_indices + ri.page_base + lp);
      if ((unsigned long long)(unsigned)page >= (unsigned long long)p.num_pages) {
        record_error(err, PKV_DEVERR_PAGE_RANGE);
        return -1;
      }
      return page * p.page_size + (key - lp * p.page_size);
    };
    bool ok = true;
    int pending = 0;  // tiles issued whose arrival is still owed
    // slot rows of the next tile are loaded one iteration ahead so their latency overlaps the copies
    int next_a = slot_of(w.kv_begin + pw * 64 + lane);
    int next_b = slot_of(w.kv_begin + pw * 64 + 32 + lane);
    for (int j = 0; j < nkt && ok; ++j) {
      const int st = j & 1;
      const int slot_a = next_a, slot_b = next_b;
      if (j + 1 < nkt) {
        const int key1 = w.kv_begin + (j + 1) * KT + pw * 64;
        next_a = slot_of(key1 + lane);
        next_b = slot_of(key1 + 32 + lane);
      }
      ok = __all_sync(0xffffffffu, tc::mbar_wait(empty0 + 8 * st, ((j >> 1) & 1) ^ 1, abort_flag, WAIT_LIMIT));
      if (!ok) break;
      const uint32_t dst0 = s_base + st * TILE_B + half * HALF_B;
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const int rr = 2 * i + (lane >> 4);  // row within this warp's 64
        const int slot = __shfl_sync(0xffffffffu, i < 16 ? slot_a : slot_b, rr & 31);
        const int row = pw * 64 + rr;
        const uint32_t dst = dst0 + row * 128 + ((cc ^ (row & 7)) << 4);
        const char* src = pool + (slot >= 0 ? (int64_t)slot * p.stride_token_b + head_off + c * 16 : 0);
        cp_async16(dst, src, slot >= 0 ? 16u : 0u);
      }
      cp_async_commit();
      ++pending;
      if (j > 0) {
        // this thread's copies of tile j-1 have landed: publish them to the tensor core
        cp_async_wait<1>();
        tc::fence_proxy_async_smem();
        tc::mbar_arrive(full0 + 8 * ((j - 1) & 1));
        --pending;
      }
    }
    cp_async_wait<0>();
    if (pending > 0 && ok) {
      tc::fence_proxy_async_smem();
      tc::mbar_arrive(full0 + 8 * ((nkt - 1) & 1));
    }
    if (!ok) {
      *abort_flag = 1;
      if (lane == 0) record_error(err, PKV_DEVERR_TIMEOUT);
    }
  } else if (warp == MMA_WARP) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_qk = tc::idesc_bf16_f32(ROWS, KT, false);
      constexpr uint32_t idesc_pv = tc::idesc_bf16_f32(ROWS, D, true);
      bool ok = tc::mbar_wait(BAR(B_Q), 0, abort_flag, WAIT_LIMIT);
      tc::fence_after_sync();
      // Issue S_j = Q K_j^T as soon as K_j has landed and its score buffer is free, and
      // O += P_j V_j as soon as P_j and V_j are ready (in tile order each), polling both so
      // neither waits behind the other's inputs.
      int js = 0, jp = 0;  // next S tile, next PV tile
      long long t0 = clock64();
      while (ok && jp < nkt) {
        bool progressed = false;
        if (js < nkt && js <= jp + 1) {
          const int st = js & 1;
          const uint32_t ph = (js >> 1) & 1;
          if (tc::mbar_try_wait(BAR(B_KF + st), ph) && tc::mbar_try_wait(BAR(B_SE + st), ph ^ 1)) {
            tc::fence_proxy_async_smem();
            tc::fence_after_sync();
            const uint32_t d = tmem + (uint32_t)st * KT;
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks) {
              const uint32_t off = (ks >> 2) * HALF_B + (ks & 3) * 32;
              const uint64_t a = tc::smem_desc_sw128(sQ + off, 16, 1024);
              const uint64_t b = tc::smem_desc_sw128(sK + st * TILE_B + off, 16, 1024);
              tc::mma_bf16_ss(d, a, b, idesc_qk, ks > 0 ? 1u : 0u);
            }
            tc::commit(BAR(B_SF + st));
            tc::commit(BAR(B_KE + st));
            ++js;
            progressed = true;
          }
        }
        if (jp < js) {
          const int st = jp & 1;
          const uint32_t ph = (jp >> 1) & 1;
          if (tc::mbar_try_wait(BAR(B_PF), jp & 1) && tc::mbar_try_wait(BAR(B_VF + st), ph)) {
            tc::fence_proxy_async_smem();
            tc::fence_after_sync();
#pragma unroll
            for (int kk = 0; kk < KT / 16; ++kk) {
              const uint64_t a = tc::smem_desc_sw128(sP + (kk >> 2) * HALF_B + (kk & 3) * 32, 16, 1024);
              const uint64_t b = tc::smem_desc_sw128(sV + st * TILE_B + kk * 2048, HALF_B, 1024);
              tc::mma_bf16_ss(tmem + TMEM_O, a, b, idesc_pv, (jp > 0 || kk > 0) ? 1u : 0u);
            }
            tc::commit(BAR(B_OD));
            tc::commit(BAR(B_VE + st));
            ++jp;
            progressed = true;
          }
        }
        if (progressed) {
          t0 = clock64();
        } else if (*abort_flag || clock64() - t0 > WAIT_LIMIT) {
          ok = false;
        }
      }
      if (!ok) {
        *abort_flag = 1;
        record_error(err, PKV_DEVERR_TIMEOUT);
        // every MMA issued so far must be complete before the TMEM is freed
        tc::commit(BAR(B_FIN));
        volatile int never = 0;
        tc::mbar_wait(BAR(B_FIN), 0, &never, WAIT_LIMIT / 8);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------------ softmax (warps 0-7)
    const int quarter = warp & 3;
    const int ch = warp >> 2;                 // key-column half of every tile
    const int r = quarter * 32 + lane;        // query row == TMEM lane
    const int t = r / G;
    const int g = r - t * G;
    const bool row_valid = t < w.q_rows;
    const int pos0 = ri.kv_len - ri.q_len + (w.q_row - ri.q_begin);  // position of the tile's first token
    const int P = pos0 + min(t, w.q_rows - 1);
    const int lo = p.window_left >= 0 ? max(0, P - p.window_left) : 0;
    const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
    const uint32_t col_half = (uint32_t)ch * 64;
    const float sc = p.scale_log2;
    float* xch = reinterpret_cast<float*>(sbase + OFF_XCH);  // [2][2][128] maxima, then [2][128] sums
    float m_used = -INFINITY;
    float l = 0.f;  // this half's share of the row sum
    bool ok = true;
    for (int j = 0; j < nkt; ++j) {
      const int sb = j & 1;
      ok = __all_sync(0xffffffffu, tc::mbar_wait(BAR(B_SF + sb), (j >> 1) & 1, abort_flag, WAIT_LIMIT));
      if (!ok) break;
      tc::fence_after_sync();
      uint32_t v[64];
      tc::tmem_ld64(tmem + lane_base + (uint32_t)sb * KT + col_half, v);
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(BAR(B_SE + sb));

      // raw-score maximum over the visible columns of this half (the scale is positive)
      const int k0 = w.kv_begin + j * KT + ch * 64;
      const int hi_c = P - k0, lo_c = lo - k0;  // visible columns: lo_c <= c <= hi_c
      const bool full = __all_sync(0xffffffffu, hi_c >= 63 && lo_c <= 0);
      float ma[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
      if (full) {
#pragma unroll
        for (int c = 0; c < 64; ++c) ma[c & 3] = fmaxf(ma[c & 3], __uint_as_float(v[c]));
      } else {
#pragma unroll
        for (int c = 0; c < 64; ++c) {
          if (c > hi_c || c < lo_c) v[c] = __float_as_uint(-INFINITY);
          ma[c & 3] = fmaxf(ma[c & 3], __uint_as_float(v[c]));
        }
      }
      float mx = fmaxf(fmaxf(ma[0], ma[1]), fmaxf(ma[2], ma[3])) * sc;
      // share the maximum with the partner warp holding the other 64 columns of the same rows
      xch[(sb * 2 + ch) * 128 + r] = mx;
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(BAR(B_XM + quarter * 2 + sb));
      ok = __all_sync(0xffffffffu,
                      tc::mbar_wait(BAR(B_XM + quarter * 2 + sb), (j >> 1) & 1, abort_flag, WAIT_LIMIT));
      if (!ok) break;
      mx = fmaxf(mx, xch[(sb * 2 + (ch ^ 1)) * 128 + r]);
      float corr = 1.f;
      bool rescale = false;
      if (mx > m_used + RESCALE_THRESHOLD) {
        corr = ex2(m_used - mx);  // 0 on the first visible tile
        m_used = mx;
        l *= corr;
        rescale = true;
      }
      const float nref = m_used == -INFINITY ? 0.f : -m_used;
      float sa[4] = {0.f, 0.f, 0.f, 0.f};
      uint32_t pk[32];
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        const float p0 = ex2(fmaf(__uint_as_float(v[2 * c]), sc, nref));
        const float p1 = ex2(fmaf(__uint_as_float(v[2 * c + 1]), sc, nref));
        sa[c & 3] += p0 + p1;
        pk[c] = pack_bf16(p0, p1);
      }
      l += (sa[0] + sa[1]) + (sa[2] + sa[3]);

      // PV of the previous tile must be complete: O is stable and the P buffer is free
      if (j > 0) {
        ok = __all_sync(0xffffffffu, tc::mbar_wait(BAR(B_OD), (j - 1) & 1, abort_flag, WAIT_LIMIT));
        if (!ok) break;
        tc::fence_after_sync();
        if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll
          for (int c4 = 0; c4 < 2; ++c4) {
            uint32_t o[32];
            const uint32_t ta = tmem + lane_base + TMEM_O + col_half + c4 * 32;
            tc::tmem_ld32(ta, o);
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * corr);
            tc::tmem_st32(ta, o);
          }
        }
      }
      // this half of the P row -> swizzled K-major bf16 tile
#pragma unroll
      for (int c8 = 0; c8 < 8; ++c8) {
        const uint32_t addr = sP + ch * HALF_B + r * 128 + ((c8 ^ (r & 7)) << 4);
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};\n" ::"r"(addr), "r"(pk[4 * c8]),
                     "r"(pk[4 * c8 + 1]), "r"(pk[4 * c8 + 2]), "r"(pk[4 * c8 + 3])
                     : "memory");
      }
      tc::fence_proxy_async_smem();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(BAR(B_PF));
    }
    if (ok) ok = __all_sync(0xffffffffu, tc::mbar_wait(BAR(B_OD), (nkt - 1) & 1, abort_flag, WAIT_LIMIT));
    if (ok) {
      // full row sum from the two halves
      float* xl = xch + 2 * 2 * 128;
      xl[ch * 128 + r] = l;
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(BAR(B_XL + quarter));
      ok = __all_sync(0xffffffffu, tc::mbar_wait(BAR(B_XL + quarter), 0, abort_flag, WAIT_LIMIT));
    }
    if (ok) {
      const float lt = l + xch[2 * 2 * 128 + (ch ^ 1) * 128 + r];
      tc::fence_after_sync();
      const float inv = lt > 0.f ? 1.f / lt : 0.f;
      const int head = w.kv_head * G + g;
      const int64_t row = (int64_t)(w.q_row + t);
      uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.o) + (row * p.num_qo_heads + head) * D +
                                            ch * 64);
      uint32_t o[64];
      tc::tmem_ld64(tmem + lane_base + TMEM_O + col_half, o);
      if (row_valid) {
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          uint4 u;
          u.x = pack_bf16(__uint_as_float(o[8 * q + 0]) * inv, __uint_as_float(o[8 * q + 1]) * inv);
          u.y = pack_bf16(__uint_as_float(o[8 * q + 2]) * inv, __uint_as_float(o[8 * q + 3]) * inv);
          u.z = pack_bf16(__uint_as_float(o[8 * q + 4]) * inv, __uint_as_float(o[8 * q + 5]) * inv);
          u.w = pack_bf16(__uint_as_float(o[8 * q + 6]) * inv, __uint_as_float(o[8 * q + 7]) * inv);
          dst[q] = u;
        }
        if (ch == 0 && p.lse) p.lse[row * p.num_qo_heads + head] = (m_used + __log2f(lt)) * 0.69314718055994531f;
      }
    } else {
      *abort_flag = 1;
      if (lane == 0) record_error(err, PKV_DEVERR_TIMEOUT);
    }
  }

  tc::fence_before_sync();
  __syncthreads();
  if (warp == MMA_WARP) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, TMEM_COLS);
  }
#undef BAR
}

int prefill_supported(const char** why) {
  if (why) *why = nullptr;
  return 1;
}

cudaError_t launch_prefill(const RunParams& p, const void* tmap_q, const void* tmap_k, const void* tmap_v, int64_t,
                           cudaStream_t s) {
  static bool attr_set[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, pf::SMEM_ALLOC);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  int32_t* err = device_error_ptr();
  if (!err) return cudaErrorInvalidDevice;
  prefill_kernel<<<(unsigned)p.num_work, pf::THREADS, pf::SMEM_ALLOC, s>>>(
      p, *static_cast<const CUtensorMap*>(tmap_q), *static_cast<const CUtensorMap*>(tmap_k),
      *static_cast<const CUtensorMap*>(tmap_v), err);
  return cudaGetLastError();
}

}  // namespace pkv
