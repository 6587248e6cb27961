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
// streaming the pages at full bandwidth while keeping the per-key work short:
//  * one CTA = 4 warps = one work item (request, KV head, group of <= 16 query heads) with a key
//    range; a range short enough for one CTA is read by it alone (each warp takes every 4th 16-key
//    tile), a long one is shared by several CTAs whose warps claim 32-key groups of it from a
//    per-range counter at run time, so the CTAs of a range finish together;
//  * every warp runs its own cp.async ring (16 keys per stage, K and V rows gathered page by page
//    through kv_indices, 16-byte vectors, XOR-swizzled so ldmatrix reads are conflict-free), so no
//    CTA-wide barrier sits in the main loop;
//  * the products run on m16n8k16 tensor-core MMAs with the KEYS in M and the (<= 8 per n-block)
//    query heads of one KV head in N: S^T = K Q^T, then O^T += V^T P^T.  Each K/V row is read once
//    per KV head, a 16-key tile costs 8 MMAs per product (not 16 with heads in M), and the output
//    accumulator is 32 registers per 8 heads.  P^T goes from the accumulator layout of the first MMA
//    to the operand layout of the second with one movmatrix.trans per 8x8 block;
//  * the online softmax runs per head column: a max over the 16 keys of the tile (3 shuffles), base-2
//    exponentials with the scale folded in, running sums kept per lane and reduced at the end;
//  * FP8 (E4M3) pages are widened to f16 in registers (exact); the K scale is folded into the score
//    scale and the V scale into the output; the head-dim order inside each 16-element block is
//    permuted identically for Q and K (a dot product does not depend on order) so one ldmatrix feeds
//    two code bytes per register half, and V's byte pairs are split into even/odd head-dim rows;
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

// The K/V rows are read once per launch: they are copied with an evict-first L2 policy, so the
// stream (hundreds of MB through a 129 MB L2) does not push out the lines that are read again -- the
// work list, the page table, the split partials and whatever the surrounding layers keep there.
__device__ __forceinline__ uint64_t l2_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;\n" : "=l"(pol));
  return pol;
}
// cp.async of 16 bytes (src_bytes < 16 zero-fills the rest) under an L2 cache policy.
__device__ __forceinline__ void cp_async16_pol(uint32_t dst, const void* src, uint32_t src_bytes, uint64_t pol) {
  asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2, %3;\n" ::"r"(dst), "l"(src),
               "r"(src_bytes), "l"(pol)
               : "memory");
}

template <int D, bool FP8, int NB>
struct DecodeCfg {
  static constexpr int ROWB = FP8 ? D : 2 * D;  // bytes per key row of one head
  static constexpr int CH = ROWB / 16;          // 16-byte chunks per row
  static constexpr int KEYS = 16;               // keys per warp tile
  static constexpr int TILE_B = KEYS * ROWB;    // bytes of one K (or V) tile
  static constexpr int HEADS = 8 * NB;          // query heads per CTA (n dimension)
  static constexpr int STAGES = 3;
  static constexpr int WARPS = 4;
  // resident CTAs per SM: the 8-KB-per-stage bf16/D128 variant fits 2 (shared memory), the 4-KB
  // variants fit 4 when the accumulators are for 8 heads (registers)
  static constexpr int CTAS = (2 * TILE_B > 4096 || NB > 1) ? 2 : 4;
  static constexpr int WARP_SMEM = STAGES * 2 * TILE_B;
  static constexpr int PIPE_SMEM = WARPS * WARP_SMEM;
  static constexpr int MERGE_SMEM = (WARPS * HEADS * D + 3 * WARPS * HEADS) * 4;
  static constexpr int SMEM = PIPE_SMEM > MERGE_SMEM ? PIPE_SMEM : MERGE_SMEM;
  static constexpr int MB = D / 16;  // 16-row m-blocks of O^T
  static constexpr int KS = D / 16;  // k-steps of S^T
  static_assert(CH >= 8, "rows must span at least 8 chunks for the XOR swizzle");
  static_assert(SMEM * CTAS <= 232448, "shared memory per SM");
};

// Head-dim index of accumulator element j (0..3) of O^T m-block mb, lane row g.
template <bool FP8>
__device__ __forceinline__ int o_dim(int mb, int j, int g) {
  if constexpr (!FP8) {
    return mb * 16 + g + 8 * (j >> 1);
  } else {
    // m-block mb = 2 q + parity: rows g -> dims 32 q + 2 g + parity, rows g + 8 -> 32 q + 16 + 2 g + parity
    return (mb >> 1) * 32 + 16 * (j >> 1) + 2 * g + (mb & 1);
  }
}

// acc[k] += sum over the ns partials of weight(partial, row of column k) * partial[column k], for
// the NC float4 columns col[k] < n4 of this thread, U partial reads per column in flight.
template <int NC, int U, int HEADS, int NA>
__device__ __forceinline__ void merge_accumulate(float4 (&acc)[NA], const int (&col)[NA], const int (&crow)[NA], int n4,
                                                 const float4* base, int ns, const float* wgt, int slot4) {
  int sp = 0;
  for (; sp + U <= ns; sp += U) {
    float4 x[U][NC];
#pragma unroll
    for (int u = 0; u < U; ++u)
#pragma unroll
      for (int k = 0; k < NC; ++k)
        x[u][k] = col[k] < n4 ? __ldcg(base + (int64_t)(sp + u) * slot4 + col[k]) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int u = 0; u < U; ++u)
#pragma unroll
      for (int k = 0; k < NC; ++k) {
        const float wv = wgt[(sp + u) * HEADS + (col[k] < n4 ? crow[k] : 0)];
        acc[k].x += wv * x[u][k].x;
        acc[k].y += wv * x[u][k].y;
        acc[k].z += wv * x[u][k].z;
        acc[k].w += wv * x[u][k].w;
      }
  }
  for (; sp < ns; ++sp) {
#pragma unroll
    for (int k = 0; k < NC; ++k) {
      if (col[k] < n4) {
        const float4 x = __ldcg(base + (int64_t)sp * slot4 + col[k]);
        const float wv = wgt[sp * HEADS + crow[k]];
        acc[k].x += wv * x.x;
        acc[k].y += wv * x.y;
        acc[k].z += wv * x.z;
        acc[k].w += wv * x.w;
      }
    }
  }
}

template <int D, bool FP8, int NB>
__global__ void __launch_bounds__(128, DecodeCfg<D, FP8, NB>::CTAS) decode_kernel(const RunParams p, int32_t* err) {
  using C = DecodeCfg<D, FP8, NB>;
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ int s_stage_key[C::WARPS][C::STAGES];

  pdl_wait();  // the plan's metadata copy and the KV write before this run must be complete
  const WorkItem w = p.work[blockIdx.x];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int g = lane >> 2;
  const int t = lane & 3;
  const int qh0 = w.kv_head * p.group + w.head_group * kDecodeRows;
  const int rows = min(C::HEADS, p.group - w.head_group * kDecodeRows);

  // ---- Q^T fragments (B operand: k = head dim, n = query head g of each n-block) ----
  uint32_t qb[C::KS][NB][2];
#pragma unroll
  for (int nb = 0; nb < NB; ++nb) {
    const int head = nb * 8 + g;
    const bool valid = head < rows;
    const uint16_t* qr = static_cast<const uint16_t*>(p.q) + ((int64_t)w.q_row * p.num_qo_heads + qh0 + head) * D;
#pragma unroll
    for (int ks = 0; ks < C::KS; ++ks) {
      if constexpr (!FP8) {
        qb[ks][nb][0] = valid ? *reinterpret_cast<const uint32_t*>(qr + ks * 16 + 2 * t) : 0u;
        qb[ks][nb][1] = valid ? *reinterpret_cast<const uint32_t*>(qr + ks * 16 + 8 + 2 * t) : 0u;
      } else {
        // permuted order: logical k {2t, 2t+1} <- dims 16ks+4t+{0,1}; {2t+8, 2t+9} <- 16ks+4t+{2,3}
        // (raw bf16 pairs here; widened to f16 below)
        const uint2 x = valid ? *reinterpret_cast<const uint2*>(qr + ks * 16 + 4 * t) : make_uint2(0, 0);
        qb[ks][nb][0] = x.x;
        qb[ks][nb][1] = x.y;
      }
    }
  }
  // ---- per-warp cp.async ring ----
  uint8_t* wsm = smem + warp * C::WARP_SMEM;
  const uint32_t wsm_u = smem_u32(wsm);
  const int lr = lane & 15;  // row whose page this lane resolves
  const int64_t head_off = (int64_t)w.kv_head * p.stride_head_b;
  const uint64_t kv_policy = l2_evict_first();

  // Lane lr (0..15) resolves the page of row lr of a tile; then every warp-wide cp.async covers
  // 32 / CH whole rows with consecutive lanes on consecutive 16-byte chunks (fully coalesced).
  constexpr int RPI = 32 / C::CH;  // rows per warp instruction
  const int lc = lane % C::CH;
  const int lsub = lane / C::CH;
  const int ps = p.page_size;
  const int ps_shift = (ps & (ps - 1)) == 0 ? __ffs(ps) - 1 : -1;  // page sizes are usually powers of 2
  auto page_of = [&](int key) -> int { return ps_shift >= 0 ? key >> ps_shift : key / ps; };
  const int64_t row_step = (int64_t)RPI * p.stride_token_b;  // bytes between the rows of consecutive instructions

  // ---- the warp's tile sequence ----
  // Alone on its range (num_splits == 1) a warp takes every 4th 16-key tile.  When num_splits CTAs
  // share the range, it is cut into 32-key groups: warp w of split s starts on group 4 s + w and
  // then claims group 4 num_splits + atomicAdd(claim, 1), and so on, until the groups run out (so
  // the warps of all the CTAs end within about one group of each other).  The claim for the next
  // group is sent when the warp starts loading a group, 2 tiles before it is needed.  A key >=
  // kv_end ends the sequence.
  constexpr int GROUP_KEYS = 2 * C::KEYS;
  const bool shared_range = w.num_splits > 1;
  const int claim_base = w.num_splits * C::WARPS;
  int pending = 0;  // lane 0: value returned by the outstanding claim
  if (shared_range && lane == 0) pending = atomicAdd(p.claim + w.unit * kClaimStride, 1);
  auto next_key = [&](int k) -> int {  // first key of the tile after the one starting at k (k < kv_end)
    if (!shared_range) return k + C::WARPS * C::KEYS;
    if (((k - w.kv_begin) & (GROUP_KEYS - 1)) != GROUP_KEYS - C::KEYS) return k + C::KEYS;
    const int grp = claim_base + __shfl_sync(0xffffffffu, pending, 0);
    const int nk = grp < (w.kv_end - w.kv_begin + GROUP_KEYS - 1) / GROUP_KEYS ? w.kv_begin + grp * GROUP_KEYS : w.kv_end;
    if (nk < w.kv_end && lane == 0) pending = atomicAdd(p.claim + w.unit * kClaimStride, 1);
    return nk;
  };
  int lkey = w.kv_begin + (shared_range ? (w.split * C::WARPS + warp) * GROUP_KEYS : warp * C::KEYS);
  lkey = min(lkey, w.kv_end);
  int nkey = lkey < w.kv_end ? next_key(lkey) : w.kv_end;
  int* key_of_stage = s_stage_key[warp];  // first key of the tile in each ring stage (kv_end: none)

  // The page id of the row this lane resolves is fetched one tile ahead, so the index load never
  // stalls the issue of the copies.
  auto fetch_page = [&](int key) -> int {
    return key < w.kv_end ? __ldg(p.kv_indices + w.page_base + page_of(key)) : 0;
  };
  int next_page = fetch_page(lkey + lr);
  // Load the tile starting at lkey into `stage` and advance the sequence.
  auto load_tile = [&](int stage) {
    const int key0 = lkey;
    const int key = key0 + lr;
    const int page = next_page;
    next_page = fetch_page(nkey + lr);
    lkey = nkey;
    nkey = nkey < w.kv_end ? next_key(nkey) : w.kv_end;
    const uint32_t dk = wsm_u + stage * 2 * C::TILE_B;
    const uint32_t dv = dk + C::TILE_B;
    // Common case: all 16 keys present and on one page (page size >= 16, chunk starts aligned), so
    // every lane has the same page id and the row addresses follow from one base and a stride.
    const bool one_page = key0 + C::KEYS <= w.kv_end && page_of(key0) == page_of(key0 + C::KEYS - 1) &&
                          (unsigned long long)(unsigned)page < (unsigned long long)p.num_pages;
    if (__all_sync(0xffffffffu, one_page)) {
      const int off0 = key0 - page_of(key0) * ps;
      const int64_t base = (int64_t)page * p.stride_page_b + (int64_t)(off0 + lsub) * p.stride_token_b + head_off + lc * 16;
      const char* ks = p.k_pool + base;
      const char* vs = p.v_pool + base;
#pragma unroll
      for (int j = 0; j < C::KEYS / RPI; ++j) {
        const int row = j * RPI + lsub;
        const uint32_t sw = row * C::ROWB + ((lc ^ (row & 7)) << 4);
        cp_async16_pol(dk + sw, ks + j * row_step, 16u, kv_policy);
        cp_async16_pol(dv + sw, vs + j * row_step, 16u, kv_policy);
      }
      return;
    }
    int64_t roff = -1;
    if (key < w.kv_end) {
      const int off = key - page_of(key) * ps;
      if ((unsigned long long)(unsigned)page >= (unsigned long long)p.num_pages)
        record_error(err, PKV_DEVERR_PAGE_RANGE);
      else
        roff = (int64_t)page * p.stride_page_b + (int64_t)off * p.stride_token_b + head_off;
    }
#pragma unroll
    for (int j = 0; j < C::KEYS / RPI; ++j) {
      const int row = j * RPI + lsub;
      const int64_t o = __shfl_sync(0xffffffffu, roff, row);
      const uint32_t sw = row * C::ROWB + ((lc ^ (row & 7)) << 4);
      const bool ok = o >= 0;
      cp_async16_pol(dk + sw, ok ? p.k_pool + o + lc * 16 : p.k_pool, ok ? 16u : 0u, kv_policy);
      cp_async16_pol(dv + sw, ok ? p.v_pool + o + lc * 16 : p.v_pool, ok ? 16u : 0u, kv_policy);
    }
  };

  float m[NB][2], l[NB][2];  // per head column 2t, 2t+1: reference max (log2 units) and this lane's sum
  float o[C::MB][NB][4];     // O^T: rows = head dims, columns = heads
#pragma unroll
  for (int nb = 0; nb < NB; ++nb) {
    m[nb][0] = m[nb][1] = -INFINITY;
    l[nb][0] = l[nb][1] = 0.f;
#pragma unroll
    for (int mb = 0; mb < C::MB; ++mb) o[mb][nb][0] = o[mb][nb][1] = o[mb][nb][2] = o[mb][nb][3] = 0.f;
  }

#pragma unroll
  for (int s = 0; s < C::STAGES - 1; ++s) {
    if (lane == 0) key_of_stage[s] = lkey;
    if (lkey < w.kv_end) load_tile(s);
    cp_async_commit();
  }

  // (Done here, after the first tiles' copies are issued, so the Q loads overlap them.)
  // FP8 KV runs the products in f16, whose largest finite value is 65504: a larger |q| would become
  // inf.  The CTA's Q rows are scaled by 2^-e, with e the smallest power that brings max |q| below
  // 2^15, and the score scale is multiplied by 2^e.  The scaling is exact (a bf16 value inside the f16
  // normal range is an f16 value), and e = 0 whenever max |q| < 2^15.
  float sc = p.scale_log2;
  if constexpr (FP8) {
    uint32_t amax = 0;  // largest |q| as bf16 magnitude bits (monotonic in the value)
#pragma unroll
    for (int ks = 0; ks < C::KS; ++ks)
#pragma unroll
      for (int nb = 0; nb < NB; ++nb)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const uint32_t r = qb[ks][nb][h];
          amax = max(amax, max(r & 0x7fffu, (r >> 16) & 0x7fffu));
        }
    amax = __reduce_max_sync(0xffffffffu, amax);  // every warp holds the CTA's whole Q
    const int e = max(0, (int)(amax >> 7) - 127 - 14);  // bf16 exponent field -> floor(log2 max |q|)
    const float down = __uint_as_float((uint32_t)(127 - e) << 23);  // 2^-e (e <= 114: a normal float)
    sc *= __uint_as_float((uint32_t)(127 + e) << 23);              // 2^e
#pragma unroll
    for (int ks = 0; ks < C::KS; ++ks)
#pragma unroll
      for (int nb = 0; nb < NB; ++nb)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const uint32_t r = qb[ks][nb][h];
          qb[ks][nb][h] = pack_f16(__uint_as_float(r << 16) * down, __uint_as_float(r & 0xffff0000u) * down);
        }
  }

  // ldmatrix lane roles: K as the A operand (rows = keys), V^T as the A operand (.trans, rows = dims)
  const int mi = lane >> 3, rr = lane & 7;
  const int k_key = ((mi & 1) << 3) + rr;  // matrices: (keys 0-7, c), (keys 8-15, c), (keys 0-7, c+1), (8-15, c+1)
  const int v_key = ((mi >> 1) << 3) + rr; // matrices: (keys 0-7, c), (keys 0-7, c+1), (keys 8-15, c), (8-15, c+1)

  int stage = 0, fill = C::STAGES - 1;  // ring slot of the tile computed now and of the one loaded now
  while (true) {
    cp_async_wait<C::STAGES - 2>();
    __syncwarp();
    const int key0 = key_of_stage[stage];
    if (key0 >= w.kv_end) break;
    // refill the stage the previous tile used before computing this one, so STAGES-1 tiles stay
    // in flight during the compute
    if (lane == 0) key_of_stage[fill] = lkey;
    if (lkey < w.kv_end) load_tile(fill);
    cp_async_commit();
    fill = fill + 1 == C::STAGES ? 0 : fill + 1;
    const uint32_t kb = wsm_u + stage * 2 * C::TILE_B;
    const uint32_t vb = kb + C::TILE_B;
    stage = stage + 1 == C::STAGES ? 0 : stage + 1;

    // ---- S^T = K Q^T for 16 keys ----
    float s[NB][4];
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) s[nb][0] = s[nb][1] = s[nb][2] = s[nb][3] = 0.f;
    if constexpr (!FP8) {
#pragma unroll
      for (int ks = 0; ks < C::KS; ++ks) {
        uint32_t a[4];
        const int chunk = 2 * ks + (mi >> 1);
        ldsm_x4(a, kb + k_key * C::ROWB + ((chunk ^ (k_key & 7)) << 4));
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) mma_bf16(s[nb], a, qb[ks][nb][0], qb[ks][nb][1]);
      }
    } else {
#pragma unroll
      for (int c = 0; c < C::KS; c += 2) {
        uint32_t r[4];
        const int chunk = c + (mi >> 1);
        ldsm_x4(r, kb + k_key * C::ROWB + ((chunk ^ (k_key & 7)) << 4));
        // r[0]: keys 0-7 / chunk c, r[1]: keys 8-15 / chunk c, r[2], r[3]: chunk c + 1; the low
        // code pair of each register feeds k-step c + h's first half, the high pair its second
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t a[4];
          e4m3x4_to_f16x2x2(r[2 * h], a[0], a[2]);
          e4m3x4_to_f16x2x2(r[2 * h + 1], a[1], a[3]);
#pragma unroll
          for (int nb = 0; nb < NB; ++nb) mma_f16(s[nb], a, qb[c + h][nb][0], qb[c + h][nb][1]);
        }
      }
    }

    // ---- online softmax per head column (log2 domain) ----
    // The reference max m moves only when a column's tile max exceeds it by more than 2^8 (one
    // warp-wide decision), so most tiles skip the O rescale; probabilities stay below 2^8.
    const bool full = key0 + C::KEYS <= w.kv_end;
    uint32_t pb[NB][2];
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
      float x0 = s[nb][0] * sc;  // key g,     head 2t
      float x1 = s[nb][1] * sc;  // key g,     head 2t+1
      float x2 = s[nb][2] * sc;  // key g + 8, head 2t
      float x3 = s[nb][3] * sc;  // key g + 8, head 2t+1
      if (!full) {
        const bool lo_ok = key0 + g < w.kv_end, hi_ok = key0 + g + 8 < w.kv_end;
        x0 = lo_ok ? x0 : -INFINITY;
        x1 = lo_ok ? x1 : -INFINITY;
        x2 = hi_ok ? x2 : -INFINITY;
        x3 = hi_ok ? x3 : -INFINITY;
      }
      float mx0 = fmaxf(x0, x2), mx1 = fmaxf(x1, x3);
#pragma unroll
      for (int sh = 4; sh < 32; sh <<= 1) {
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, sh));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, sh));
      }
      // every tile holds at least one visible key, so the tile maxima are finite
      if (__any_sync(0xffffffffu, mx0 > m[nb][0] + 8.f || mx1 > m[nb][1] + 8.f)) {
        const float mn0 = fmaxf(m[nb][0], mx0), mn1 = fmaxf(m[nb][1], mx1);
        const float c0 = ex2(m[nb][0] - mn0), c1 = ex2(m[nb][1] - mn1);
        m[nb][0] = mn0;
        m[nb][1] = mn1;
        l[nb][0] *= c0;
        l[nb][1] *= c1;
#pragma unroll
        for (int mb = 0; mb < C::MB; ++mb) {
          o[mb][nb][0] *= c0;
          o[mb][nb][1] *= c1;
          o[mb][nb][2] *= c0;
          o[mb][nb][3] *= c1;
        }
      }
      x0 = ex2(x0 - m[nb][0]);
      x1 = ex2(x1 - m[nb][1]);
      x2 = ex2(x2 - m[nb][0]);
      x3 = ex2(x3 - m[nb][1]);
      l[nb][0] += x0 + x2;
      l[nb][1] += x1 + x3;
      // P^T in accumulator layout (row = key, column pair = heads) -> B operand (k = keys, n = head)
      if constexpr (!FP8) {
        pb[nb][0] = movmatrix_trans(pack_bf16(x0, x1));
        pb[nb][1] = movmatrix_trans(pack_bf16(x2, x3));
      } else {
        pb[nb][0] = movmatrix_trans(pack_f16(x0, x1));
        pb[nb][1] = movmatrix_trans(pack_f16(x2, x3));
      }
    }

    // ---- O^T += V^T P^T ----
    if constexpr (!FP8) {
#pragma unroll
      for (int mb = 0; mb < C::MB; ++mb) {
        uint32_t a[4];
        const int chunk = 2 * mb + (mi & 1);
        ldsm_x4_t(a, vb + v_key * C::ROWB + ((chunk ^ (v_key & 7)) << 4));
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) mma_bf16(o[mb][nb], a, pb[nb][0], pb[nb][1]);
      }
    } else {
#pragma unroll
      for (int c = 0; c < D / 16; c += 2) {
        uint32_t r[4];
        const int chunk = c + (mi & 1);
        ldsm_x4_t(r, vb + v_key * C::ROWB + ((chunk ^ (v_key & 7)) << 4));
        // r[0]: keys 0-7 x chunk c, r[1]: keys 0-7 x chunk c+1, r[2]: keys 8-15 x chunk c,
        // r[3]: keys 8-15 x chunk c+1.  Each register holds, for byte-pair column g:
        // (key 2t: d, d+1), (key 2t+1: d, d+1) with d = 16 chunk + 2g; bytes 0/2 are the even dim,
        // bytes 1/3 the odd one.  One byte permute puts the even pair in the low half and the odd
        // pair in the high half.
        uint32_t ev[4], od[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) e4m3x4_to_f16x2x2(__byte_perm(r[k], 0, 0x3120u), ev[k], od[k]);
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) {
          mma_f16(o[c][nb], ev, pb[nb][0], pb[nb][1]);
          mma_f16(o[c + 1][nb], od, pb[nb][0], pb[nb][1]);
        }
      }
    }
    __syncwarp();
  }
  cp_async_wait<0>();

  // full per-head sums across the 8 key rows g of the warp
#pragma unroll
  for (int nb = 0; nb < NB; ++nb) {
#pragma unroll
    for (int sh = 4; sh < 32; sh <<= 1) {
      l[nb][0] += __shfl_xor_sync(0xffffffffu, l[nb][0], sh);
      l[nb][1] += __shfl_xor_sync(0xffffffffu, l[nb][1], sh);
    }
  }

  // ---- merge the 4 warps' states through shared memory ----
  __syncthreads();
  float* so = reinterpret_cast<float*>(smem);   // [4][HEADS][D]
  float* sm = so + C::WARPS * C::HEADS * D;     // [4][HEADS]
  float* sl = sm + C::WARPS * C::HEADS;         // [4][HEADS]
  float* sf = sl + C::WARPS * C::HEADS;         // [4][HEADS] weights
  if (g == 0) {
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
      sm[warp * C::HEADS + nb * 8 + 2 * t] = m[nb][0];
      sm[warp * C::HEADS + nb * 8 + 2 * t + 1] = m[nb][1];
      sl[warp * C::HEADS + nb * 8 + 2 * t] = l[nb][0];
      sl[warp * C::HEADS + nb * 8 + 2 * t + 1] = l[nb][1];
    }
  }
#pragma unroll
  for (int mb = 0; mb < C::MB; ++mb) {
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int head = nb * 8 + 2 * t + (j & 1);
        if (head < rows) so[(warp * C::HEADS + head) * D + o_dim<FP8>(mb, j, g)] = o[mb][nb][j];
      }
    }
  }
  __syncthreads();
  __shared__ float s_lse2[C::HEADS];
  if (threadIdx.x < C::HEADS) {
    const int r = threadIdx.x;
    float M = -INFINITY;
#pragma unroll
    for (int k = 0; k < C::WARPS; ++k) M = fmaxf(M, sm[k * C::HEADS + r]);
    float W = 0.f;
    float e[C::WARPS];
#pragma unroll
    for (int k = 0; k < C::WARPS; ++k) {
      e[k] = ex2(sm[k * C::HEADS + r] - M);  // a warp without tiles has m = -inf: weight 0
      W += e[k] * sl[k * C::HEADS + r];
    }
    const float inv = W > 0.f ? 1.f / W : 0.f;
#pragma unroll
    for (int k = 0; k < C::WARPS; ++k) sf[k * C::HEADS + r] = e[k] * inv;
    s_lse2[r] = M + __log2f(W);
  }
  __syncthreads();
  if (w.out_slot < 0) {
    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.o) + ((int64_t)w.q_row * p.num_qo_heads + qh0) * D;
    for (int idx = threadIdx.x; idx < rows * D; idx += blockDim.x) {
      const int r = idx / D, d = idx - r * D;
      float acc = 0.f;
#pragma unroll
      for (int k = 0; k < C::WARPS; ++k) acc += sf[k * C::HEADS + r] * so[(k * C::HEADS + r) * D + d];
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
      for (int k = 0; k < C::WARPS; ++k) acc += sf[k * C::HEADS + r] * so[(k * C::HEADS + r) * D + d];
      po[idx] = acc;
    }
    if (threadIdx.x < rows) p.part_lse[(int64_t)w.out_slot * kDecodeRows + threadIdx.x] = s_lse2[threadIdx.x];
    // The last chunk of a (request, KV head, group) to finish merges all of its partials:
    // m = max lse_s, o = sum_s 2^(lse_s - m) o_s / sum_s 2^(lse_s - m).  No CTA waits for another.
    __shared__ int s_last;
    __threadfence();
    __syncthreads();
    const int unit = w.unit;
    const MergeItem mi_ = p.merge[unit];
    if (threadIdx.x == 0) {
      const int done = atomicAdd(p.unit_count + unit, 1);
      s_last = done == mi_.num_splits - 1;
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    if (rows * D <= 4 * 128) {
      // One float4 column per thread (up to 4 rows of 128 dims): an online merge.  Each thread loads
      // the log2-sum-exp of its row and its column of U partials at once (as many as its registers
      // hold: 20 with 4 resident CTAs, 32 with 2) and folds them in under a running maximum, so 38
      // partials cost two dependent L2 round trips and no shared-memory staging.
      constexpr int U = C::CTAS >= 4 ? 20 : 32;
      const int ns = mi_.num_splits;
      const int n4 = rows * D / 4;
      const int col = threadIdx.x;
      const bool active = col < n4;
      const int crow = active ? col * 4 / D : 0;
      const float* lse_g = p.part_lse + (int64_t)mi_.first_slot * kDecodeRows + crow;
      const float4* pm = reinterpret_cast<const float4*>(p.part_o + (int64_t)mi_.first_slot * kDecodeRows * D) + col;
      constexpr int SLOT4 = kDecodeRows * D / 4;
      float la[U];
      float4 oa[U];
      auto fetch = [&](float (&l)[U], float4 (&o)[U], int s0) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const bool in = active && s0 + u < ns;
          l[u] = in ? __ldcg(lse_g + (int64_t)(s0 + u) * kDecodeRows) : -INFINITY;
          o[u] = in ? __ldcg(pm + (int64_t)(s0 + u) * SLOT4) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
      };
      float m = -INFINITY, W = 0.f;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      auto fold = [&](const float (&l)[U], const float4 (&o)[U]) {
        float mb = m;
#pragma unroll
        for (int u = 0; u < U; ++u) mb = fmaxf(mb, l[u]);
        if (mb == -INFINITY) return;  // a partial without keys has lse -inf and weight 0
        const float c = ex2(m - mb);  // 0 while nothing has been seen
        W *= c;
        acc.x *= c;
        acc.y *= c;
        acc.z *= c;
        acc.w *= c;
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const float wv = ex2(l[u] - mb);
          W += wv;
          acc.x = fmaf(wv, o[u].x, acc.x);
          acc.y = fmaf(wv, o[u].y, acc.y);
          acc.z = fmaf(wv, o[u].z, acc.z);
          acc.w = fmaf(wv, o[u].w, acc.w);
        }
        m = mb;
      };
      for (int s0 = 0; s0 < ns; s0 += U) {
        fetch(la, oa, s0);
        fold(la, oa);
      }
      __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.o) + ((int64_t)mi_.q_row * p.num_qo_heads + qh0) * D;
      if (active) {
        const float f = W > 0.f ? p.out_scale / W : 0.f;
        __nv_bfloat162* o2 = reinterpret_cast<__nv_bfloat162*>(out + col * 4);
        o2[0] = __floats2bfloat162_rn(acc.x * f, acc.y * f);
        o2[1] = __floats2bfloat162_rn(acc.z * f, acc.w * f);
        if (p.lse && (col * 4) % D == 0)  // the row's first column writes its log-sum-exp
          p.lse[(int64_t)mi_.q_row * p.num_qo_heads + qh0 + crow] = (m + __log2f(W)) * 0.69314718055994531f;
      }
      if (threadIdx.x == 0) {  // ready for the next run of this plan
        p.unit_count[unit] = 0;
        atomicExch(p.claim + unit * kClaimStride, 0);
      }
      return;
    }
    // Online merge over chunks of splits: the chunk's log2-sum-exps are staged in shared memory by
    // all threads and turned into per-row weights 2^(lse_s - M) once, one warp per row (lanes over
    // the splits, shuffle reductions); each thread owns float4 columns of the output and keeps 8-16
    // partial reads per column in flight.  With one column per thread and one chunk (the usual
    // case) the first 8-16 partials are read before the weights are known, so that round trip
    // overlaps the staging of the log2-sum-exps.
    constexpr int V4 = C::HEADS * D / 4;            // float4s of the (at most HEADS) output rows
    constexpr int PER_T = (V4 + 127) / 128;         // float4s per thread
    constexpr int SLOT4 = kDecodeRows * D / 4;      // float4s between consecutive partials
    const int n4 = rows * D / 4;
    const int cap = C::SMEM / (4 * C::HEADS) - 2;   // splits per chunk that fit the shared scratch
    float* wgt = reinterpret_cast<float*>(smem);    // [cap][HEADS] lse, then weights
    __shared__ float sM[C::HEADS], sScale[C::HEADS], sW[C::HEADS];
    if (threadIdx.x < C::HEADS) {
      sM[threadIdx.x] = -INFINITY;
      sW[threadIdx.x] = 0.f;
    }
    float4 acc[PER_T];
    int col[PER_T], crow[PER_T];
#pragma unroll
    for (int k = 0; k < PER_T; ++k) {
      acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
      col[k] = threadIdx.x + k * 128;
      crow[k] = col[k] * 4 / D;
    }
    const float* lse_g = p.part_lse + (int64_t)mi_.first_slot * kDecodeRows;
    const float4* pm = reinterpret_cast<const float4*>(p.part_o + (int64_t)mi_.first_slot * kDecodeRows * D);
    constexpr int PRE = C::CTAS >= 4 ? 8 : 16;  // registers: 4 resident CTAs leave ~128 per thread
    const int npre = (n4 <= 128 && mi_.num_splits <= cap) ? min(PRE, mi_.num_splits) : 0;
    float4 pre[PRE];
#pragma unroll
    for (int u = 0; u < PRE; ++u)
      pre[u] = (u < npre && col[0] < n4) ? __ldcg(pm + (int64_t)u * SLOT4 + col[0]) : make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s0 = 0; s0 < mi_.num_splits; s0 += cap) {
      const int ns = min(cap, mi_.num_splits - s0);
      __syncthreads();
      for (int e = threadIdx.x; e < ns * C::HEADS; e += blockDim.x) {
        const int sp = e / C::HEADS, r = e - sp * C::HEADS;
        wgt[e] = r < rows ? __ldcg(lse_g + (int64_t)(s0 + sp) * kDecodeRows + r) : -INFINITY;
      }
      __syncthreads();
      for (int r = warp; r < rows; r += C::WARPS) {
        float m = -INFINITY;
        for (int sp = lane; sp < ns; sp += 32) m = fmaxf(m, wgt[sp * C::HEADS + r]);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        const float m_prev = sM[r];
        const float Mc = fmaxf(m_prev, m);
        const bool none = Mc == -INFINITY;              // no key seen yet: keep every weight 0
        const float sc = none ? 1.f : ex2(m_prev - Mc);  // 0 on the first chunk
        float W = 0.f;
        for (int sp = lane; sp < ns; sp += 32) {
          const float e = none ? 0.f : ex2(wgt[sp * C::HEADS + r] - Mc);
          wgt[sp * C::HEADS + r] = e;
          W += e;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) W += __shfl_xor_sync(0xffffffffu, W, o);
        __syncwarp();  // every lane has read sM[r] before lane 0 rewrites it
        if (lane == 0) {
          sW[r] = sW[r] * sc + W;
          sM[r] = Mc;
          sScale[r] = sc;
        }
      }
      __syncthreads();
#pragma unroll
      for (int k = 0; k < PER_T; ++k) {
        if (col[k] < n4) {
          const float sc = sScale[crow[k]];
          acc[k].x *= sc;
          acc[k].y *= sc;
          acc[k].z *= sc;
          acc[k].w *= sc;
        }
      }
      const float4* base = pm + (int64_t)s0 * SLOT4;
      if (npre > 0) {  // one chunk: the first npre partials are already in registers
        if (col[0] < n4) {
#pragma unroll
          for (int u = 0; u < PRE; ++u) {
            const float wv = u < npre ? wgt[u * C::HEADS + crow[0]] : 0.f;
            acc[0].x += wv * pre[u].x;
            acc[0].y += wv * pre[u].y;
            acc[0].z += wv * pre[u].z;
            acc[0].w += wv * pre[u].w;
          }
        }
        merge_accumulate<1, 16, C::HEADS>(acc, col, crow, n4, base + (int64_t)npre * SLOT4, ns - npre,
                                          wgt + npre * C::HEADS, SLOT4);
      } else if (n4 <= 128)  // one column per thread (up to 4 rows of 128 dims): 16 reads in flight
        merge_accumulate<1, 16, C::HEADS>(acc, col, crow, n4, base, ns, wgt, SLOT4);
      else
        merge_accumulate<PER_T, 8, C::HEADS>(acc, col, crow, n4, base, ns, wgt, SLOT4);
    }
    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.o) + ((int64_t)mi_.q_row * p.num_qo_heads + qh0) * D;
#pragma unroll
    for (int k = 0; k < PER_T; ++k) {
      if (col[k] < n4) {
        const float W = sW[crow[k]];
        const float f = W > 0.f ? p.out_scale / W : 0.f;
        __nv_bfloat162* o2 = reinterpret_cast<__nv_bfloat162*>(out + col[k] * 4);
        o2[0] = __floats2bfloat162_rn(acc[k].x * f, acc[k].y * f);
        o2[1] = __floats2bfloat162_rn(acc[k].z * f, acc[k].w * f);
      }
    }
    if (p.lse && threadIdx.x < rows)
      p.lse[(int64_t)mi_.q_row * p.num_qo_heads + qh0 + threadIdx.x] =
          (sM[threadIdx.x] + __log2f(sW[threadIdx.x])) * 0.69314718055994531f;
    if (threadIdx.x == 0) {  // ready for the next run of this plan
      p.unit_count[unit] = 0;
      atomicExch(p.claim + unit * kClaimStride, 0);
    }
  }
}

template <int D, bool FP8, int NB>
static cudaError_t launch_decode_t(const RunParams& p, cudaStream_t s) {
  using C = DecodeCfg<D, FP8, NB>;
  static bool attr_set[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr_set[dev]) {
    cudaError_t e =
        cudaFuncSetAttribute(decode_kernel<D, FP8, NB>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  int32_t* err = device_error_ptr();
  if (!err) return cudaErrorInvalidDevice;
  return launch_pdl(decode_kernel<D, FP8, NB>, dim3((unsigned)p.num_work), dim3(128), (size_t)C::SMEM, s, p, err);
}

int decode_ctas_per_sm(int kv_dtype, int head_dim, int group) {
  const bool nb2 = group > 8;
  if (kv_dtype == PKV_FP8_E4M3) return nb2 ? DecodeCfg<128, true, 2>::CTAS : DecodeCfg<128, true, 1>::CTAS;
  if (head_dim == 64) return nb2 ? DecodeCfg<64, false, 2>::CTAS : DecodeCfg<64, false, 1>::CTAS;
  return nb2 ? DecodeCfg<128, false, 2>::CTAS : DecodeCfg<128, false, 1>::CTAS;
}

cudaError_t launch_decode(const RunParams& p, int kv_dtype, cudaStream_t s) {
  const bool nb2 = p.group > 8;
  if (kv_dtype == PKV_FP8_E4M3) {
    if (p.head_dim != 128) return cudaErrorInvalidValue;
    return nb2 ? launch_decode_t<128, true, 2>(p, s) : launch_decode_t<128, true, 1>(p, s);
  }
  if (p.head_dim == 128) return nb2 ? launch_decode_t<128, false, 2>(p, s) : launch_decode_t<128, false, 1>(p, s);
  if (p.head_dim == 64) return nb2 ? launch_decode_t<64, false, 2>(p, s) : launch_decode_t<64, false, 1>(p, s);
  return cudaErrorInvalidValue;
}

}  // namespace pkv
