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
// GB300 design.  One CTA = two 128-row query tiles (A and B: consecutive tokens of one request, rows
// = (token, head) pairs of one KV head's query-head group) sharing every K/V tile, so each gathered
// K/V byte feeds twice the tensor-core work of a single tile:
//  * warps 8-11 and 13-15 (producers): Q_A and Q_B by 3-D TMA boxes (128-byte swizzle, warp 8); K
//    (warps 9-11) and V (warps 13-15) tiles of 128 keys gathered row by row through the page table with
//    16-byte cp.async, 16 lanes per 256-byte row, straight into the 128-byte-swizzled layout the
//    tensor core reads; two stages.  Each lane resolves the global addresses of two of its warp's
//    rows of the next tile while the stage is still in use, so the unrolled copy loop spends one
//    shuffle, a bit test and an add per cp.async: the producers share the schedulers with the softmax
//    warps, and their instruction count sets the pace of the gather.  Each producer thread's arrival
//    on the stage's mbarrier is posted by the hardware when its copies land
//    (cp.async.mbarrier.arrive.noinc), so a tile is announced as soon as it is in shared memory; the
//    MMA thread fences it into the async proxy after its wait.  (TMA tile::gather4 moves 512 bytes
//    per instruction and measured slower here for token-granular pools.)
//  * warp 12 (MMA): one thread issues tcgen05.mma (kind::f16, M=128, N=128, K=16, bf16 in, fp32
//    accumulate in TMEM) in the order S_A(0) S_B(0) | PV_A(j) S_A(j+1) PV_B(j) S_B(j+1) | ..., so the
//    tensor core works on one tile while the other tile's softmax runs.  P lives in TMEM on top of
//    its own scores and is the A operand of the PV MMA (V is an MN-major shared-memory operand, no
//    transpose).  MMAs of one thread execute in issue order, so S_X(j+1) overwriting P_X(j) is safe
//    once PV_X(j) was issued, and "S_X(j) complete" implies "PV_X(j-1) complete".
//  * warps 0-3 / 4-7 (softmax of tile A / B): thread r owns row r (TMEM lane r).  All 128 scores of
//    the row come into registers with four TMEM loads and one wait; then the row maximum,
//    p = 2^(s * scale * log2 e - m) with packed FFMA + ex2, bf16 pairs packed in place and stored
//    over the scores in two 32-column TMEM stores.  Each half is signalled on its own barrier, so
//    the PV MMAs over keys 0-63 start while keys 64-127 are still being exponentiated.  Causal /
//    window masking only on tiles that need it.  The row maximum moves lazily (only when it grows
//    by more than 2^8; exact because numerator and denominator share it), and O is rescaled in TMEM
//    only then, before the first half is signalled.  Epilogue: O / l to bf16 rows and the LSE, or an
//    fp32 partial of a split item; a tile whose rows all belong to the item is staged in its Q
//    buffer in the swizzled layout of the Q box and leaves by two TMA stores.
// Registers are rebalanced with setmaxnreg: the two softmax warpgroups take 184 per thread, the
// producer and MMA warpgroups keep 72.  Every wait is bounded: on timeout the CTA records PKV_DEVERR_TIMEOUT, waits (bounded) for its own
// copies and MMAs, frees its TMEM and exits.

#include <cuda.h>
#include <cuda_bf16.h>
#include <math.h>

#include "pkv_internal.h"
#include "ptx.cuh"
#include "tc.cuh"

namespace pkv {

int32_t* device_error_ptr();

namespace pf {
constexpr int ROWS = 128;               // query rows per Q tile
constexpr int KT = 128;                 // keys per K/V tile
constexpr int D = 128;                  // head dim
constexpr int HALF_B = ROWS * 128;      // one 64-column half of a 128-row bf16 tile (16 KB)
constexpr int TILE_B = 2 * HALF_B;      // 32 KB
constexpr int STAGES = 2;
constexpr int OFF_QA = 0;
constexpr int OFF_QB = OFF_QA + TILE_B;
constexpr int OFF_K = OFF_QB + TILE_B;
constexpr int OFF_V = OFF_K + STAGES * TILE_B;
constexpr int OFF_BAR = OFF_V + STAGES * TILE_B;
constexpr int NUM_BARS = 21;
constexpr int OFF_TMEM = OFF_BAR + NUM_BARS * 8;
constexpr int OFF_ABORT = OFF_TMEM + 8;
constexpr int SMEM_USED = OFF_ABORT + 8;
constexpr int SMEM_ALLOC = SMEM_USED + 1024;  // room to align the base to 1024 bytes
enum {
  B_Q = 0, B_KF = 1, B_VF = 3, B_KE = 5, B_VE = 7,
  B_SF = 9,   // [2]: S_X(j) complete (and with it PV_X(j-1))
  B_PF = 11,  // [2]: all of P_X(j) stored in TMEM by the 4 softmax warps of tile X
  B_OD = 13,  // [2]: the last PV_X complete
  B_FIN = 15,
  B_PH = 16,  // [2]: the first half (keys 0-63) of P_X(j) stored by the 4 softmax warps of tile X
  B_HOLD = 18,  // nothing arrives here: the held wait of a timeout-path test
  B_OS = 19     // [2]: tile X's output rows staged in its Q buffer by its 4 softmax warps
};
constexpr uint32_t TMEM_COLS = 512;  // S_A/P_A [0,128), S_B/P_B [128,256), O_A [256,384), O_B [384,512)
constexpr uint32_t TMEM_O = 256;
constexpr int THREADS = 512;          // 4 warpgroups: softmax A, softmax B, producers, MMA + producers
constexpr int PRODUCER_WARP0 = 8;     // warp 8 loads Q; warps 9-11 and 13-15 gather K and V
constexpr int MMA_WARP = 12;
// Producer roles: K by warps 9-11 and V by warps 13-15 (K is needed first, by S); warp 8 only loads
// Q.  Warp w runs on scheduler w % 4, so each of schedulers 1-3 carries one K and one V warp (21-22
// row pairs of each a tile) and scheduler 0 is left to the MMA thread, whose issue rate it sets.
constexpr int K_WARPS = 3, V_WARPS = 3;
// launched at 65536 / 512 = 128 registers per thread, then rebalanced per warpgroup:
// 2 x 128 x SOFTMAX_REGS + 2 x 128 x OTHER_REGS = 47104 + 18432 = 65536 <= 65536
constexpr uint32_t SOFTMAX_REGS = 184;
constexpr uint32_t OTHER_REGS = 72;
constexpr int K_PRODUCER_THREADS = 32 * K_WARPS;
constexpr int V_PRODUCER_THREADS = 32 * V_WARPS;
// The waits of the pipeline give up after the run's limit (RunParams::wait_limit_k x 1024 clock
// cycles, about 2 s by default); the waits of the timeout path itself, for copies and MMAs already
// in flight, use DRAIN_LIMIT whatever the run's limit.
constexpr long long DRAIN_LIMIT = 500000000LL;  // clock cycles (about 0.25 s)
constexpr float RESCALE_THRESHOLD = 8.0f;      // log2 units
}  // namespace pf

// Merge of a held state (natural-log lse `s_prev`) with this pass's (`s_this`, updated in place to the
// merged lse): the normalised weights e^(s - m) / (e^(s_prev - m) + e^(s_this - m)), m = max; two
// empty states (-inf) give weights 0 and lse -inf.
__device__ __forceinline__ void merge_weights(float s_prev, float& s_this, float& w_prev, float& w_this) {
  const float m = fmaxf(s_prev, s_this);
  if (m == -INFINITY) {
    w_prev = w_this = 0.f;
    return;
  }
  const float a = expf(s_prev - m), b = expf(s_this - m), sum = a + b;
  w_prev = a / sum;
  w_this = b / sum;
  s_this = m + logf(sum);
}
// f[e] += w * (bf16 element e of v), for the 8 elements of a 16-byte vector
__device__ __forceinline__ void add_scaled_bf16x8(const uint4& v, float w, float (&f)[8]) {
  const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = fmaf(w, __uint_as_float(u[i] << 16), f[2 * i]);
    f[2 * i + 1] = fmaf(w, __uint_as_float(u[i] & 0xffff0000u), f[2 * i + 1]);
  }
}

// One warp's share of a K or V tile: NW warps share the tile's 64 row pairs, this one (pw) copies
// pairs pw, pw + NW, ...; in each cp.async lanes 0-15 copy the 16 chunks of the pair's first row and
// lanes 16-31 those of its second, into the 128-byte-swizzled K-major layout (64-column halves).
// Lane l holds the global addresses of the warp's rows l (ra) and 32 + l (rb).  Fully unrolled: the
// destination of pair i is a per-lane base plus a constant, because the swizzle of row 2 (pw + NW i) +
// hi repeats with period 4 in i.
template <int NW>
__device__ __forceinline__ void issue_rows(uint32_t dst0, int pw, int pairs, uint64_t ra, uint64_t rb, int c,
                                           int hi) {
  constexpr int MAXP = (pf::KT / 2 + NW - 1) / NW;
  const int cc = c & 7;
  uint32_t base[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int r = 2 * (pw + NW * k) + hi;
    base[k] = dst0 + r * 128 + ((cc ^ (r & 7)) << 4);
  }
#pragma unroll
  for (int i = 0; i < MAXP; ++i) {
    if (i == MAXP - 1 && i >= pairs) break;  // only the last pair can be missing (V warps)
    const uint64_t src = __shfl_sync(0xffffffffu, i < 16 ? ra : rb, (2 * i + hi) & 31);
    const uint32_t dst = base[i & 3] + (uint32_t)((i >> 2) * 8 * NW * 128);
    cp_async16(dst, reinterpret_cast<const char*>(src) + c * 16, 16u);
  }
}

__global__ void __launch_bounds__(pf::THREADS, 1)
    prefill_kernel(const RunParams p, const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap to,
                   int32_t* err) {
  using namespace pf;
  pdl_wait();  // the plan's metadata copy and the KV write before this run must be complete
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u = smem_u32(smem_raw);
  const uint32_t base = (raw_u + 1023u) & ~1023u;
  uint8_t* sbase = smem_raw + (base - raw_u);
  const uint32_t sQ = base + OFF_QA, sK = base + OFF_K, sV = base + OFF_V;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sbase + OFF_ABORT);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sbase + OFF_TMEM);
#define BAR(i) (base + OFF_BAR + 8u * (uint32_t)(i))

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const WorkItem w = p.work[blockIdx.x];
  const ReqInfo ri = p.req[w.req];
  const int G = p.group;
  const int T = ROWS / G;              // tokens per Q tile
  const bool two = w.q_rows > T;       // does tile B hold any token?
  const int nkt = (w.kv_end - w.kv_begin + KT - 1) / KT;
  const long long wait_limit = (long long)p.wait_limit_k << 10;

  if (nkt == 0) {
    // a non-causal segment without keys: the empty state (o = 0, lse = -inf) for every row.
    // Thread i writes half (i & 1) of row i / 2 of the two tiles.
    const int r = threadIdx.x >> 1, half = threadIdx.x & 1;
    const int x = r >> 7, rr = r & (ROWS - 1);
    const int t = x * T + rr / G, g = rr % G;
    if (t < w.q_rows && !p.merge_into) {  // merging an empty state leaves the held state unchanged
      const int64_t row = (int64_t)(w.q_row + t);
      const int head = w.kv_head * G + g;
      uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.o) + (row * p.num_qo_heads + head) * D +
                                            half * (D / 2));
#pragma unroll
      for (int i = 0; i < D / 16; ++i) dst[i] = make_uint4(0u, 0u, 0u, 0u);
      if (half == 0 && p.lse) p.lse[row * p.num_qo_heads + head] = -INFINITY;
    }
    return;
  }

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    tc::mbar_init(BAR(B_Q), 1);
    for (int s = 0; s < STAGES; ++s) {
      tc::mbar_init(BAR(B_KF + s), K_PRODUCER_THREADS);
      tc::mbar_init(BAR(B_VF + s), V_PRODUCER_THREADS);
      tc::mbar_init(BAR(B_KE + s), 1);
      tc::mbar_init(BAR(B_VE + s), 1);
    }
    for (int x = 0; x < 2; ++x) {
      tc::mbar_init(BAR(B_SF + x), 1);
      tc::mbar_init(BAR(B_PF + x), 4);
      tc::mbar_init(BAR(B_PH + x), 4);
      tc::mbar_init(BAR(B_OD + x), 1);
      tc::mbar_init(BAR(B_OS + x), 4);
    }
    tc::mbar_init(BAR(B_FIN), 1);
    tc::mbar_init(BAR(B_HOLD), 1);
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

  if (warp >= PRODUCER_WARP0 && warp != MMA_WARP) {
    // ------------------------------------------------------------------ producers (cp.async)
    tc::reg_dealloc<OTHER_REGS>();
    // role: operand and index among that operand's warps; warp k of n copies the row pairs
    // q = k, k + n, k + 2n, ... (rows 2q and 2q + 1, 16 lanes per 256-byte row)
    const bool is_k = warp < MMA_WARP;  // K: warps 9-11, V: warps 13-15 (warp 8 loads Q only)
    const int pw = is_k ? warp - PRODUCER_WARP0 - 1 : warp - MMA_WARP - 1;
    const int nw = is_k ? K_WARPS : V_WARPS;
    const int pairs = (KT / 2 - pw + nw - 1) / nw;  // row pairs of this warp per tile
    auto row_of = [&](int idx) -> int { return 2 * (pw + nw * (idx >> 1)) + (idx & 1); };  // idx-th row
    const char* pool = is_k ? p.k_pool : p.v_pool;
    const uint32_t s_base = is_k ? sK : sV;
    const uint32_t full0 = is_k ? BAR(B_KF) : BAR(B_VF);
    const uint32_t empty0 = is_k ? BAR(B_KE) : BAR(B_VE);
    if (warp == PRODUCER_WARP0 && lane == 0) {
      tc::tma_prefetch_desc(&tq);
      tc::mbar_arrive_expect_tx(BAR(B_Q), two ? 2 * TILE_B : TILE_B);
      tc::tma_load_3d(sQ, &tq, BAR(B_Q), 0, w.kv_head * G, w.q_row);
      tc::tma_load_3d(sQ + HALF_B, &tq, BAR(B_Q), 64, w.kv_head * G, w.q_row);
      if (two) {
        tc::tma_load_3d(sQ + TILE_B, &tq, BAR(B_Q), 0, w.kv_head * G, w.q_row + T);
        tc::tma_load_3d(sQ + TILE_B + HALF_B, &tq, BAR(B_Q), 64, w.kv_head * G, w.q_row + T);
      }
    }
    const int64_t head_off = (int64_t)w.kv_head * p.stride_head_b;
    const char* ext_base = is_k ? p.ext_k : p.ext_v;
    const int64_t ext_head_off = (int64_t)w.kv_head * D * 2;
    const int prefix = ri.kv_len - ri.q_len;  // keys before the request's first new token
    const int ps = p.page_size;
    const int ps_shift = (ps & (ps - 1)) == 0 ? __ffs(ps) - 1 : -1;
    // Global address of the row holding `key` of this warp's operand, or null (no such key: the
    // copy zero-fills).  Two-source plans take the keys from the prefix on from the contiguous
    // new-token rows; ragged plans read row page_base + key; paged plans go through the page table.
    auto row_addr = [&](int key) -> const char* {
      if (key >= w.kv_end) return nullptr;
      if (ext_base && key >= prefix) return ext_base + (int64_t)(ri.q_begin + key - prefix) * p.ext_row_b + ext_head_off;
      int64_t slot;
      if (p.ragged_kv) {  // contiguous K/V: key j of the request is row page_base + j
        slot = (int64_t)ri.page_base + key;
        if (slot >= p.num_pages) {
          record_error(err, PKV_DEVERR_PAGE_RANGE);
          return nullptr;
        }
      } else {
        const int lp = ps_shift >= 0 ? key >> ps_shift : key / ps;
        const int page = __ldg(p.kv_indices + ri.page_base + lp);
        if ((unsigned long long)(unsigned)page >= (unsigned long long)p.num_pages) {
          record_error(err, PKV_DEVERR_PAGE_RANGE);
          return nullptr;
        }
        slot = (int64_t)page * ps + (key - lp * ps);
      }
      return pool + slot * p.stride_token_b + head_off;
    };
    // Lane l resolves the addresses of this warp's rows l and 32 + l of a tile one tile ahead (the
    // page-table loads overlap the wait for the stage).  A row past the item's last key copies the
    // row of its first key instead of zeros: its score is masked to -inf and its probability is 0,
    // and a real row's values are finite, so it adds nothing (the split chunks of an item are whole
    // tiles, so only the item's end, where the mask applies, has such rows).
    const bool gathers = warp != PRODUCER_WARP0;
    const int nrows = 2 * pairs;
    const char* first_row = gathers ? row_addr(w.kv_begin) : nullptr;
    if (!first_row) first_row = pool;  // a page outside the pool (recorded): any readable row
    struct Rows {
      uint64_t a, b;
    };
    auto resolve = [&](int tile) -> Rows {
      const int k0 = w.kv_begin + tile * KT;
      const char* ra = lane < nrows ? row_addr(k0 + row_of(lane)) : nullptr;
      const char* rb = 32 + lane < nrows ? row_addr(k0 + row_of(32 + lane)) : nullptr;
      return Rows{(uint64_t)(ra ? ra : first_row), (uint64_t)(rb ? rb : first_row)};
    };
    const int c = lane & 15, hi = lane >> 4;  // 16-byte chunk of the 256-byte row; first or second row of a pair
    bool ok = true;
    Rows next = gathers ? resolve(0) : Rows{0, 0};
    for (int j = 0; j < nkt && ok && gathers; ++j) {
      const int st = j & 1;
      const Rows cur = next;
      if (j + 1 < nkt) next = resolve(j + 1);
      ok = __all_sync(0xffffffffu, tc::mbar_wait(empty0 + 8 * st, ((j >> 1) & 1) ^ 1, abort_flag, wait_limit));
      if (!ok) break;
      const uint32_t dst0 = s_base + st * TILE_B + (c >> 3) * HALF_B;
      if (is_k)
        issue_rows<K_WARPS>(dst0, pw, pairs, cur.a, cur.b, c, hi);
      else
        issue_rows<V_WARPS>(dst0, pw, pairs, cur.a, cur.b, c, hi);
      // the stage's barrier receives this thread's arrival when its copies have landed; the MMA
      // thread fences them into the async proxy after its wait
      cp_async_arrive_noinc(full0 + 8 * st);
    }
    cp_async_wait_all();
    if (!ok) {
      *abort_flag = 1;
      if (lane == 0) record_error(err, PKV_DEVERR_TIMEOUT);
    }
    // the Q tiles must have landed before the CTA exits, also when the MMA thread gave up before
    // waiting for them (returns at once otherwise)
    if (warp == PRODUCER_WARP0 && lane == 0) {
      volatile int never = 0;
      tc::mbar_wait(BAR(B_Q), 0, &never, DRAIN_LIMIT);
    }
  } else if (warp == MMA_WARP) {
    // ------------------------------------------------------------------ MMA issuer
    tc::reg_dealloc<OTHER_REGS>();
    if (warp == MMA_WARP && lane == 0) {
      constexpr uint32_t idesc_qk = tc::idesc_bf16_f32(ROWS, KT, false);
      constexpr uint32_t idesc_pv = tc::idesc_bf16_f32(ROWS, D, true);
      // Shared-memory descriptors: one per operand buffer (Q tile, K stage, V stage); a k-step's
      // descriptor is its buffer's plus the step's byte offset / 16 in the start-address field (exact:
      // every operand address is below 256 KB, so the 14-bit field never carries).  The add is opaque
      // to the compiler, so it stays next to its MMA as one 64-bit add per operand; measured 3.7 %
      // faster on the prefix-extend workload than descriptors formed by the compiler from each address.
      const uint64_t dq0 = tc::smem_desc_sw128(sQ, 16, 1024), dq1 = tc::smem_desc_sw128(sQ + TILE_B, 16, 1024);
      const uint64_t dk0 = tc::smem_desc_sw128(sK, 16, 1024), dk1 = tc::smem_desc_sw128(sK + TILE_B, 16, 1024);
      const uint64_t dv0 = tc::smem_desc_sw128(sV, HALF_B, 1024), dv1 = tc::smem_desc_sw128(sV + TILE_B, HALF_B, 1024);
      auto step = [](uint64_t d, uint32_t off) -> uint64_t {
        uint64_t r;
        asm volatile("add.s64 %0, %1, %2;\n" : "=l"(r) : "l"(d), "l"((uint64_t)(off >> 4)));
        return r;
      };
      auto issue_s = [&](int x, int st) {  // S_x = Q_x K_st^T into TMEM columns [128 x, 128 x + 128)
        const uint32_t d = tmem + (uint32_t)x * 128;
        const uint64_t qa = x ? dq1 : dq0, kb = st ? dk1 : dk0;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint32_t off = (ks >> 2) * HALF_B + (ks & 3) * 32;
          tc::mma_bf16_ss(d, step(qa, off), step(kb, off), idesc_qk, ks > 0 ? 1u : 0u);
        }
        tc::commit(BAR(B_SF + x));
      };
      // O_x += P_x V_st over key steps [k0, k1) of the tile, P_x from TMEM
      auto issue_pv = [&](int x, int st, bool first, int k0 = 0, int k1 = KT / 16) {
        const uint32_t a0 = tmem + (uint32_t)x * 128;
        const uint32_t d = tmem + TMEM_O + (uint32_t)x * 128;
        const uint64_t vb = st ? dv1 : dv0;
#pragma unroll
        for (int kk = k0; kk < k1; ++kk)
          tc::mma_bf16_ts(d, a0 + kk * 8, step(vb, kk * 2048), idesc_pv, (!first || kk > 0) ? 1u : 0u);
      };
      auto wait = [&](uint32_t bar, uint32_t parity) {
        return tc::mbar_wait(bar, parity, abort_flag, wait_limit);
      };
      // a test of the timeout path holds the thread on a barrier nothing arrives at
      bool ok = !p.hold_wait || wait(BAR(B_HOLD), 0);
      ok = ok && wait(BAR(B_Q), 0) && wait(BAR(B_KF), 0);
      if (ok) {
        tc::fence_proxy_async_smem();
        tc::fence_after_sync();
        issue_s(0, 0);
        if (two) issue_s(1, 0);
        tc::commit(BAR(B_KE));
      }
      for (int j = 0; j < nkt && ok; ++j) {
        const int st = j & 1, st1 = (j + 1) & 1;
        const uint32_t ph = (j >> 1) & 1, ph1 = ((j + 1) >> 1) & 1;
        const bool more = j + 1 < nkt;
        ok = wait(BAR(B_PH + 0), j & 1) && wait(BAR(B_VF + st), ph);
        if (!ok) break;
        tc::fence_proxy_async_smem();
        tc::fence_after_sync();
        issue_pv(0, st, j == 0, 0, KT / 32);
        ok = wait(BAR(B_PF + 0), j & 1);
        if (!ok) break;
        tc::fence_after_sync();
        issue_pv(0, st, j == 0, KT / 32, KT / 16);
        if (more) {
          ok = wait(BAR(B_KF + st1), ph1);
          if (!ok) break;
          tc::fence_proxy_async_smem();
          tc::fence_after_sync();
          issue_s(0, st1);
        }
        if (two) {
          ok = wait(BAR(B_PH + 1), j & 1);
          if (!ok) break;
          tc::fence_after_sync();
          issue_pv(1, st, j == 0, 0, KT / 32);
          ok = wait(BAR(B_PF + 1), j & 1);
          if (!ok) break;
          tc::fence_after_sync();
          issue_pv(1, st, j == 0, KT / 32, KT / 16);
          if (more) issue_s(1, st1);
        }
        tc::commit(BAR(B_VE + st));
        if (more) tc::commit(BAR(B_KE + st1));
      }
      if (ok) {
        tc::commit(BAR(B_OD + 0));
        tc::commit(BAR(B_OD + 1));
      } else {
        *abort_flag = 1;
        record_error(err, PKV_DEVERR_TIMEOUT);
        // every MMA issued so far must be complete before the TMEM is freed
        tc::commit(BAR(B_FIN));
        volatile int never = 0;
        tc::mbar_wait(BAR(B_FIN), 0, &never, DRAIN_LIMIT);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------------ softmax (tile A: warps 0-3, B: 4-7)
    tc::reg_alloc<SOFTMAX_REGS>();
    if (warp < 4 || two) {
    const int x = warp >> 2;  // which Q tile
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;  // row of the tile == TMEM lane
    const int t = x * T + r / G;        // token of the item
    const int g = r - (r / G) * G;
    const bool row_valid = t < w.q_rows;
    const int pos0 = ri.kv_len - ri.q_len + (w.q_row - ri.q_begin);  // position of the item's first token
    // the row's last visible key: its own position (causal) or the request's last key
    const int P = p.noncausal ? ri.kv_len - 1 : pos0 + min(t, w.q_rows - 1);
    const int lo = p.window_left >= 0 ? max(0, P - p.window_left) : 0;
    const uint32_t tS = tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)x * 128;
    const uint32_t tO = tS + TMEM_O;
    const float sc = p.scale_log2;
    float m_used = -INFINITY;
    float l = 0.f;
    bool ok = true;
    for (int j = 0; j < nkt; ++j) {
      ok = __all_sync(0xffffffffu, tc::mbar_wait(BAR(B_SF + x), j & 1, abort_flag, wait_limit));
      if (!ok) break;
      tc::fence_after_sync();
      const int k0 = w.kv_begin + j * KT;
      const int hi_c = P - k0, lo_c = lo - k0;  // visible columns: lo_c <= c <= hi_c
      const bool full = __all_sync(0xffffffffu, hi_c >= KT - 1 && lo_c <= 0);
      // all 128 scores of the row in registers: four TMEM loads in flight, one wait
      uint32_t v[KT];
      tc::tmem_ld128(tS, v);
      if (!full) {
#pragma unroll
        for (int c = 0; c < KT; ++c)
          if (!(c <= hi_c && c >= lo_c)) v[c] = __float_as_uint(-INFINITY);
      }
      // row maximum of the raw scores (the scale is positive)
      float ma[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
      for (int c = 0; c < KT; c += 2)  // three-input max: half the instructions
        ma[(c >> 1) & 3] = fmax3(ma[(c >> 1) & 3], __uint_as_float(v[c]), __uint_as_float(v[c + 1]));
      const float mx = fmaxf(fmaxf(ma[0], ma[1]), fmaxf(ma[2], ma[3])) * sc;
      float corr = 1.f;
      bool rescale = false;
      if (mx > m_used + RESCALE_THRESHOLD) {
        corr = ex2(m_used - mx);  // 0 on the first visible tile
        m_used = mx;
        l *= corr;
        rescale = true;
      }
      // P = 2^(s * sc - m) as bf16 pairs, packed in place and stored over the scores in two halves:
      // PV on keys 0-63 starts while keys 64-127 are still being exponentiated
      const float nref = m_used == -INFINITY ? 0.f : -m_used;
      // packed fp32x2 FFMA / FADD: one instruction per column pair (the MUFU ex2 stays per column)
      const uint64_t sc2 = f2pack(sc, sc), nref2 = f2pack(nref, nref);
      uint64_t sum2[2] = {0ull, 0ull};
#pragma unroll
      for (int h = 0; h < 2; ++h) {
#pragma unroll
        for (int c = h * (KT / 4); c < (h + 1) * (KT / 4); ++c) {
          const uint64_t x2 = ffma2(f2pack(__uint_as_float(v[2 * c]), __uint_as_float(v[2 * c + 1])), sc2, nref2);
          float x0, x1;
          f2unpack(x2, x0, x1);
          const float p0 = ex2(x0), p1 = ex2(x1);
          sum2[c & 1] = fadd2(sum2[c & 1], f2pack(p0, p1));
          v[c] = pack_bf16(p0, p1);
        }
        tc::tmem_st32(tS + h * 32, *reinterpret_cast<const uint32_t(*)[32]>(v + h * 32));
        // O_X is stable here (S_X(j) completing implies PV_X(j-1) completed), and PV_X(j) cannot
        // start before the first half of P_X(j) is signalled: rescale O_X now if the maximum moved
        if (h == 0 && j > 0 && __any_sync(0xffffffffu, rescale)) {
#pragma unroll
          for (int c4 = 0; c4 < D / 32; ++c4) {
            uint32_t o[32];
            tc::tmem_ld32(tO + c4 * 32, o);
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * corr);
            tc::tmem_st32(tO + c4 * 32, o);
          }
        }
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(BAR(h == 0 ? B_PH + x : B_PF + x));
      }
      float sa[4];
      f2unpack(sum2[0], sa[0], sa[1]);
      f2unpack(sum2[1], sa[2], sa[3]);
      l += (sa[0] + sa[1]) + (sa[2] + sa[3]);
    }
    if (ok) ok = __all_sync(0xffffffffu, tc::mbar_wait(BAR(B_OD + x), 0, abort_flag, wait_limit));
    if (ok && w.out_slot >= 0) {
      // one key chunk of a split item: normalised fp32 partial + log2-sum-exp, merged afterwards.
      // O goes out as [32 four-column groups][256 rows] float4, so each store is coalesced.
      tc::fence_after_sync();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      const int prow = x * ROWS + r;
      float4* dst = reinterpret_cast<float4*>(p.ppart_o + (int64_t)w.out_slot * kPrefillPartialFloats) + prow;
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        uint32_t o[32];
        tc::tmem_ld32(tO + h * 32, o);
        if (row_valid) {
#pragma unroll
          for (int q = 0; q < 8; ++q)
            dst[(h * 8 + q) * kPrefillItemRows] =
                make_float4(__uint_as_float(o[4 * q]) * inv, __uint_as_float(o[4 * q + 1]) * inv,
                            __uint_as_float(o[4 * q + 2]) * inv, __uint_as_float(o[4 * q + 3]) * inv);
        }
      }
      if (row_valid)
        p.ppart_lse[(int64_t)w.out_slot * kPrefillItemRows + prow] = l > 0.f ? m_used + __log2f(l) : -INFINITY;
    } else if (ok) {
      tc::fence_after_sync();
      const int head = w.kv_head * G + g;
      const int64_t row = (int64_t)(w.q_row + t);
      // this pass's state (o = O / l, natural-log lse); merged into the state already held by
      // (o, lse) when the run merges (weights e^(s - m) / sum over the two states)
      float lse_out = l > 0.f ? (m_used + __log2f(l)) * 0.69314718055994531f : -INFINITY;
      float w_prev = 0.f, w_this = 1.f;
      if (p.merge_into && row_valid) merge_weights(p.lse[row * p.num_qo_heads + head], lse_out, w_prev, w_this);
      const float inv = (l > 0.f ? 1.f / l : 0.f) * w_this;
      if (!p.merge_into && (x + 1) * T <= w.q_rows) {
        // Every row of the tile is a token of this item: the rows go out as the Q tile came in -- into
        // the Q tile's shared memory (free: every MMA that read it is complete), in the 128-byte
        // swizzled layout of the same 3-D box, then one TMA store per 64-column half.  (A partial
        // tile's box would also cover the next request's rows, so those take the per-thread stores.)
        const uint32_t srow = sQ + (uint32_t)x * TILE_B + (uint32_t)r * 128;
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          uint32_t o[32];
          tc::tmem_ld32(tO + h * 32, o);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint32_t u[4];
#pragma unroll
            for (int e = 0; e < 4; ++e)
              u[e] = pack_bf16(__uint_as_float(o[8 * q + 2 * e]) * inv, __uint_as_float(o[8 * q + 2 * e + 1]) * inv);
            const int c = (h & 1) * 4 + q;  // 16-byte chunk within the 64-column half h / 2
            tc::st_shared_v4(srow + (h >> 1) * HALF_B + ((c ^ (r & 7)) << 4), u[0], u[1], u[2], u[3]);
          }
        }
        // each warp's rows into the async proxy, then one arrival per warp; thread 0 of the tile waits
        // (bounded) for all four and stores the box
        tc::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(BAR(B_OS + x));
        if (r == 0) {
          if (tc::mbar_wait(BAR(B_OS + x), 0, abort_flag, wait_limit)) {
            const int c1 = w.kv_head * G, c2 = w.q_row + x * T;
            tc::tma_store_3d(&to, sQ + x * TILE_B, 0, c1, c2);
            tc::tma_store_3d(&to, sQ + x * TILE_B + HALF_B, 64, c1, c2);
            tc::bulk_commit_group();
            tc::bulk_wait_group_read0();  // the shared memory must stay put until the stores have read it
          } else {
            *abort_flag = 1;
            record_error(err, PKV_DEVERR_TIMEOUT);
          }
        }
      } else {
        uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.o) + (row * p.num_qo_heads + head) * D);
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          uint32_t o[32];
          tc::tmem_ld32(tO + h * 32, o);
          if (row_valid) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              float f[8];
#pragma unroll
              for (int e = 0; e < 8; ++e) f[e] = __uint_as_float(o[8 * q + e]) * inv;
              if (p.merge_into) {
                const uint4 prev = dst[h * 4 + q];
                add_scaled_bf16x8(prev, w_prev, f);
              }
              uint4 u;
              u.x = pack_bf16(f[0], f[1]);
              u.y = pack_bf16(f[2], f[3]);
              u.z = pack_bf16(f[4], f[5]);
              u.w = pack_bf16(f[6], f[7]);
              dst[h * 4 + q] = u;
            }
          }
        }
      }
      if (row_valid && p.lse) p.lse[row * p.num_qo_heads + head] = lse_out;
    } else {
      *abort_flag = 1;
      if (lane == 0) record_error(err, PKV_DEVERR_TIMEOUT);
    }
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

// Merge of the key chunks of split prefill items.  Grid (items, slices): CTA (u, y) merges the
// four-column groups [32 y / slices, 32 (y + 1) / slices) of item u, G4 at a time; thread r = row r
// of the item's two tiles (the prefill kernel's (token, head) order).  m = max_s lse_s, w_s =
// 2^(lse_s - m) / sum_s 2^(lse_s - m), o = sum_s w_s o_s; a row whose chunks saw no key gets o = 0 and
// lse = -inf.  Few items (a shared prefix, a few long requests) take one group per CTA so that the
// grid still covers the SMs.  In a merging run (the result merged into the state held in (o, lse)) every
// slice reads a row's held lse and the last slice of the item to finish (a per-item counter) rewrites
// it, so no slice can read a merged lse.
template <int G4>
__global__ void __launch_bounds__(kPrefillItemRows) prefill_merge_kernel(const RunParams p, int64_t first_merge) {
  const MergeItem m = p.merge[first_merge + blockIdx.x];
  const int r = threadIdx.x;
  const int G = p.group;
  const int T = pf::ROWS / G;
  const int x = r / pf::ROWS, rr = r % pf::ROWS;
  const int t = x * T + rr / G, g = rr % G;
  const bool valid = t < m.q_rows;  // rows past the item's tokens do nothing (no early exit: barriers below)
  const int64_t row = (int64_t)(m.q_row + t);
  const int head = m.kv_head * G + g;
  float lse_out = -INFINITY;
  if (valid) {
    const float* lse_s = p.ppart_lse + (int64_t)m.first_slot * kPrefillItemRows + r;
    float mx = -INFINITY;
    for (int sp = 0; sp < m.num_splits; ++sp) mx = fmaxf(mx, lse_s[(int64_t)sp * kPrefillItemRows]);
    float sum = 0.f;
    if (mx != -INFINITY)
      for (int sp = 0; sp < m.num_splits; ++sp) sum += ex2(lse_s[(int64_t)sp * kPrefillItemRows] - mx);
    // the merged state of the pieces; merged in turn into the held (o, lse) when the run merges
    lse_out = sum > 0.f ? (mx + __log2f(sum)) * 0.69314718055994531f : -INFINITY;
    float w_prev = 0.f, w_this = 1.f;
    if (p.merge_into) merge_weights(p.lse[row * p.num_qo_heads + head], lse_out, w_prev, w_this);
    const float inv = (sum > 0.f ? 1.f / sum : 0.f) * w_this;
    const int per_cta = 32 / gridDim.y;  // four-column groups of this CTA
    uint2* dst = reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(p.o) + (row * p.num_qo_heads + head) * pf::D);
    for (int g0 = blockIdx.y * per_cta; g0 < (blockIdx.y + 1) * per_cta; g0 += G4) {
      float4 acc[G4];
#pragma unroll
      for (int c = 0; c < G4; ++c) acc[c] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (mx != -INFINITY) {
        for (int sp = 0; sp < m.num_splits; ++sp) {
          const float wgt = ex2(lse_s[(int64_t)sp * kPrefillItemRows] - mx);
          const float4* src = reinterpret_cast<const float4*>(p.ppart_o + (int64_t)(m.first_slot + sp) *
                                                                              kPrefillPartialFloats) +
                              g0 * kPrefillItemRows + r;
#pragma unroll
          for (int c = 0; c < G4; ++c) {
            const float4 v = src[c * kPrefillItemRows];
            acc[c].x = fmaf(wgt, v.x, acc[c].x);
            acc[c].y = fmaf(wgt, v.y, acc[c].y);
            acc[c].z = fmaf(wgt, v.z, acc[c].z);
            acc[c].w = fmaf(wgt, v.w, acc[c].w);
          }
        }
      }
#pragma unroll
      for (int c = 0; c < G4; ++c) {
        float f[4] = {acc[c].x * inv, acc[c].y * inv, acc[c].z * inv, acc[c].w * inv};
        if (p.merge_into) {
          const uint2 prev = dst[g0 + c];
          f[0] = fmaf(w_prev, __uint_as_float(prev.x << 16), f[0]);
          f[1] = fmaf(w_prev, __uint_as_float(prev.x & 0xffff0000u), f[1]);
          f[2] = fmaf(w_prev, __uint_as_float(prev.y << 16), f[2]);
          f[3] = fmaf(w_prev, __uint_as_float(prev.y & 0xffff0000u), f[3]);
        }
        dst[g0 + c] = make_uint2(pack_bf16(f[0], f[1]), pack_bf16(f[2], f[3]));
      }
    }
  }
  if (!p.lse) return;
  if (!p.merge_into) {
    if (valid && blockIdx.y == 0) p.lse[row * p.num_qo_heads + head] = lse_out;
    return;
  }
  // merging run: every slice has read the held lse of its rows before the last slice of the item to
  // finish rewrites them; its counter is zero before the run and again after it
  __shared__ int s_last;
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    s_last = atomicAdd(p.unit_count + first_merge + blockIdx.x, 1) == (int)gridDim.y - 1;
  }
  __syncthreads();
  if (!s_last) return;
  if (valid) p.lse[row * p.num_qo_heads + head] = lse_out;
  if (threadIdx.x == 0) p.unit_count[first_merge + blockIdx.x] = 0;
}

cudaError_t launch_prefill_merge(const RunParams& p, int64_t first_merge, int64_t count, cudaStream_t s) {
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  if (count * 8 >= 2 * (int64_t)sms)
    prefill_merge_kernel<4><<<dim3((unsigned)count, 8), kPrefillItemRows, 0, s>>>(p, first_merge);
  else
    prefill_merge_kernel<1><<<dim3((unsigned)count, 32), kPrefillItemRows, 0, s>>>(p, first_merge);
  return cudaGetLastError();
}

int prefill_supported(const char** why) {
  if (why) *why = nullptr;
  return 1;
}

cudaError_t launch_prefill(const RunParams& p, const void* tmap_q, const void* tmap_o, int64_t, cudaStream_t s) {
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
  return launch_pdl(prefill_kernel, dim3((unsigned)p.num_work), dim3(pf::THREADS), (size_t)pf::SMEM_ALLOC, s, p,
                    *static_cast<const CUtensorMap*>(tmap_q), *static_cast<const CUtensorMap*>(tmap_o), err);
}

}  // namespace pkv
