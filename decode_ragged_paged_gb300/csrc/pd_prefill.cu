// pd_prefill.cu -- causal (or full) prefill attention over an HND paged KV
// cache on the 5th-generation tensor cores (tcgen05, accumulators in TMEM).
//
// Perplexity, "Disaggregated prefill and decode" (2025), section "Prefill vs
// Decode performance": prefill requests bring many tokens (large qo_len) and
// are compute bound, their attention being GEMM-shaped along the query axis.
// Query rows of a request are the last qo_len positions of its kv_len cached
// tokens, so row i may attend keys j <= kv_len - qo_len + i.
//
// One persistent CTA per SM walks a list of (request, 128-row q tile, query
// head) items sorted heaviest first, in serpentine order (round k forward over
// the grid, round k + 1 backward). Warp roles:
//   warp 0    TMA producer of Q tiles (a ring of two or three) and K tiles (a
//             ring of three or two), each tile one 128-byte-swizzled box per
//             page and 64-column half; boxes past the request's pages are
//             fetched out of range and arrive as zeros;
//   warp 6    TMA producer of V tiles (2-slot ring), same boxes;
//   warp 1    allocates 512 TMEM columns and issues S = Q K^T (tcgen05.mma)
//             into one of two S buffers;
//   warp 7    issues O += P V into the item's O buffer (two, alternating
//             between items) with P read from tensor memory (two issuing
//             warps: one thread's tcgen05.mma issue rate and commits limited a
//             single issuer);
//   warps 2-5 one query row per thread: one-pass online softmax on S read from
//             TMEM, P written back over S as bf16 pairs (for items whose rows
//             see few keys, also their rounding remainders, which enter P V
//             too), O rescaled in TMEM
//             only when the running max grows by more than 2^8; an item's
//             epilogue (O / l, log-sum-exp) runs after the next item's first
//             tile, a full bf16 O tile staged in the item's Q buffer and
//             stored by TMA, other tiles stored row by row.
// Every wait is bounded; on a timeout the CTA records PD_DEV_TIMEOUT, drains
// and frees its TMEM.
#include <atomic>
#include <math.h>
#include <string.h>

#include "pd_common.cuh"
#include "pd_internal.h"
#include "pd_tc.cuh"

namespace pd {

namespace {

constexpr int kBM = 128;          // query rows per tile
constexpr int kBN = 128;          // keys per tile
constexpr int kD = 128;           // head_dim
constexpr int kThreadsPf = 256;   // 8 warps: Q/K loads, S MMA, 4 softmax, V loads, P V MMA
constexpr int kWarpV = 6;         // the warp that loads V tiles
constexpr int kWarpPV = 7;        // the warp that issues O += P V
constexpr uint32_t kTileBytes = kBM * kD * 2;  // one bf16 128 x 128 tile
constexpr uint32_t kHalf = kTileBytes / 2;     // one 64-column half: 128 rows x 128 B
constexpr uint32_t kTmemCols = 512;
constexpr int kSB = 2;                         // S / P buffers in TMEM (128 columns each)
// two O accumulators after them, alternating between consecutive items
__device__ __forceinline__ uint32_t col_s(int b) { return (uint32_t)b * 128; }
__device__ __forceinline__ uint32_t col_o(int b) { return (uint32_t)(kSB + b) * 128; }
static_assert((kSB + 2) * 128 <= 512, "TMEM columns");
constexpr float kRescaleThreshold = 8.0f;      // log2 units
constexpr float kSpecSumLimit = 256.0f;        // 2^kRescaleThreshold
constexpr int kBuckets = 1024;

// Shared memory (offsets from a 1024-byte aligned base): QB Q buffers, then a
// ring of KS K slots and one of 7 - QB - KS V slots, seven 32 KiB tiles in all.
// Two shapes are built: QB 3 / KS 2 for calls made mostly of long query blocks
// (a Q tile is fetched an item ahead; full bf16 O tiles are staged in their Q
// buffer and written by TMA), QB 2 / KS 3 for decode-like calls (K runs a tile
// further ahead; O rows are stored directly, so a Q buffer is free once its
// item's last S product is done).
constexpr uint32_t kOffQ = 0;
constexpr int kRingTiles = 7;
constexpr uint32_t kOffBar = kRingTiles * kTileBytes;
constexpr size_t kPrefillSmem = kRingTiles * kTileBytes + 256 + 1024;

// Every ring slot has its own full and empty barriers: a slot freed by the
// phases of a barrier that serves other buffers could see its waiter fall two
// phases behind, where a parity wait no longer tells them apart.
template <int QB, int KS, int VS>
struct BarsT {
  uint64_t q_full[QB], q_empty[QB], k_full[KS], k_empty[KS], v_full[VS], v_empty[VS];
  uint64_t s_full[kSB], p_full[kSB], pv_done[kSB], drain, o_sync;
  uint32_t tmem_slot;
  int abort;
};
static_assert(sizeof(BarsT<3, 2, 2>) <= 256 && sizeof(BarsT<2, 3, 2>) <= 256, "barrier block");

// An item is (request, q tile of p.tile_rows query rows, group of p.tile_heads
// query heads sharing KV head g). Tile row m holds query row q0 + m / tile_heads
// of head h + m % tile_heads (with tile_heads = 1: one head, 128 rows).
struct PItem {
  int r, qt, h, g, q0, rows, qo_len, kv, n_kv, pbase, need;
};

// Items whose first query row sees fewer keys than this take P to P V in two
// bf16 parts. Rounding P to bf16 (8 significant bits) moves a row's output by
// up to a few 1e-3 when a few keys carry the weight, as in the first rows of
// a causal prefill; over more keys the independent rounding errors of the
// weights average out.
constexpr int kSplitBelowKeys = 128;
__device__ __forceinline__ bool split_item(int causal, int tile_rows, int qt, int qo_len, int kv) {
  const int first_keys = causal ? min(kv, kv - qo_len + qt * tile_rows + 1) : kv;
  return first_keys < kSplitBelowKeys;
}

__device__ __forceinline__ int kv_tiles(int qt, int qo_len, int kv, int causal, int tile_rows) {
  if (kv <= 0) return 0;
  int last_key = kv - 1;
  if (causal) {
    const int last_row = min(qt * tile_rows + tile_rows - 1, qo_len - 1);
    last_key = min(last_key, kv - qo_len + last_row);
  }
  return last_key < 0 ? 0 : last_key / kBN + 1;
}

__device__ __forceinline__ PItem prefill_item(const PrefillParams& p, int it) {
  PItem I;
  const int rq = it / p.item_heads;
  I.h = (it - rq * p.item_heads) * p.tile_heads;  // first query head of the tile
  const int2 v = p.rq_list[rq];
  I.r = v.x;
  I.qt = v.y;
  I.g = I.h / p.group;
  // no qo_indptr: one query row per request, row r (a decode batch)
  const int a = p.qo_indptr != nullptr ? p.qo_indptr[I.r] : I.r;
  I.qo_len = p.qo_indptr != nullptr ? p.qo_indptr[I.r + 1] - a : 1;
  I.q0 = a + I.qt * p.tile_rows;
  I.rows = min(p.tile_rows, I.qo_len - I.qt * p.tile_rows);  // valid query rows
  I.kv = p.kv_len[I.r];
  I.n_kv = kv_tiles(I.qt, I.qo_len, I.kv, p.causal, p.tile_rows);
  I.pbase = p.page_indptr[I.r];
  I.need = (I.kv + p.page_size - 1) / p.page_size;
  return I;
}

// With staging on, a full bf16 O tile is staged in its item's Q buffer and
// stored by TMA, which then frees that buffer; other tiles are stored row by
// row, and their Q buffer is free as soon as the item's last S product has
// completed.
template <bool STAGE>
__device__ __forceinline__ bool o_staged(const PrefillParams& p, const PItem& I) {
  return STAGE && p.o_dtype == PD_BF16 && I.rows == p.tile_rows;
}

// Item a CTA takes in round k: rounds alternate direction over the grid, so on
// a list sorted heaviest first every CTA's total stays near the mean.
__device__ __forceinline__ int round_item(uint32_t k) {
  const int g = (int)gridDim.x, b = (int)blockIdx.x;
  return (int)k * g + ((k & 1u) ? g - 1 - b : b);
}

// The item after the current one is read while the current one is worked on,
// so the dependent loads of its description leave the critical path.
__device__ __forceinline__ PItem prefill_item_or_empty(const PrefillParams& p, int it, int n_items) {
  if (it < n_items) return prefill_item(p, it);
  PItem I{};
  return I;
}

__device__ __forceinline__ bool request_ok(const PrefillParams& p, int r) {
  const int a = p.qo_indptr != nullptr ? p.qo_indptr[r] : r;
  const int b = p.qo_indptr != nullptr ? p.qo_indptr[r + 1] : r + 1;
  const int n = p.kv_len[r];
  int code = 0;
  if (a < 0 || b < a || b > p.total_qo) code = PD_DEV_BAD_INDPTR;
  else if (n < 0 || n > p.max_kv_len || b - a > p.max_qo_len || (p.causal && b - a > n)) code = PD_DEV_BAD_LENGTH;
  else {
    const int pa = p.page_indptr[r], pb = p.page_indptr[r + 1];
    if (pa < 0 || pb < pa) code = PD_DEV_BAD_INDPTR;
    else if ((long long)(pb - pa) * p.page_size < n) code = PD_DEV_BAD_PAGE_TABLE;
  }
  if (code) report(p.status, code);
  return code == 0;
}

// An item's page ids are read 32 at a time: lane l of a producer warp holds
// the id of page 32 w + l of the request's list (window w; unused past its
// last page). The read is issued a window (or, for an item's first window, an
// item) before the ids are needed, so its latency stays off the loads.
__device__ __forceinline__ int window_pid(const PrefillParams& p, int pbase, int need, int w, int lane) {
  const int pidx = w * 32 + lane;
  return pidx < need ? __ldg(p.page_indices + pbase + pidx) : 0;
}

// Window holding the first page of 128-token tile j (a tile's pages never
// straddle two windows: a tile spans 128 / page_size pages, a power of two
// up to 16, or one page).
__device__ __forceinline__ int tile_window(const PrefillParams& p, int j) { return (j * kBN / p.page_size) >> 5; }

// Boxes of one 128-token K or V tile: per 64-column half, one box per page (or
// one box of 128 slots when a page holds at least 128 tokens). Lane l < boxes
// takes its box's page id from the window and its slot offset; pages past the
// request's end (and bad ids) map to num_pages, which the TMA unit fetches as
// zeros.
struct TileBox {
  int pid, soff;
};

__device__ __forceinline__ TileBox tile_box(const PrefillParams& p, int need, int j, int win_pid, int lane) {
  const int pb = p.page_size < kBN ? p.page_size : kBN;  // slots per box
  const int nb = kBN / pb;                                // boxes per half
  const int tok = j * kBN + (lane < nb ? lane : 0) * pb;
  const int pidx = tok / p.page_size;
  TileBox t{__shfl_sync(0xffffffffu, win_pid, pidx & 31), tok % p.page_size};
  if (pidx >= need) {
    t.pid = p.num_pages;
  } else if (t.pid < 0 || t.pid >= p.num_pages) {
    if (lane < nb) report(p.status, PD_DEV_BAD_PAGE_TABLE);
    t.pid = p.num_pages;
  }
  return t;
}

__device__ __forceinline__ void load_kv_tile(const PrefillParams& p, const TileBox& t, const CUtensorMap* map,
                                             int g, uint8_t* dst, uint64_t* bar, int lane) {
  const int pb = p.page_size < kBN ? p.page_size : kBN;
  const int nb = kBN / pb;
  if (lane == 0) mbar_arrive_expect_tx(bar, kTileBytes);
  __syncwarp();
  if (lane < nb) {
    // the NHD map orders its coordinates (dim, head, slot, page), HND (dim, slot, head, page)
    const int c1 = p.nhd ? g : t.soff, c2 = p.nhd ? t.soff : g;
    tma_load_4d(dst + lane * pb * 128, map, 0, c1, c2, t.pid, bar);
    tma_load_4d(dst + kHalf + lane * pb * 128, map, 64, c1, c2, t.pid, bar);
  }
}

// bf16 pair of two accumulator words (fp32 bits) times a factor, with one
// packed multiply.
__device__ __forceinline__ uint32_t scale_pack(const uint32_t* v, float2 f2) {
  const float2 q = fmul2(make_float2(__uint_as_float(v[0]), __uint_as_float(v[1])), f2);
  return pack_bf16x2(q.x, q.y);
}

// Split items: the rounding remainders bf16(p - bf16(p)) of one row's weights
// P = 2^(s * scale - m), written to TMEM columns 64 .. 127 of its S buffer
// (keys 32c .. 32c + 31 in columns 64 + 16c .. 64 + 16c + 15) before the bf16
// pairs of P overwrite columns 0 .. 63. S is read back from TMEM 32 columns at
// a time, highest first, so no chunk is overwritten before it is read; keys at
// or past ncol (masked) get weight 0, as in the pairs. P V adds
// the product of these remainders to that of the pairs, so it sees p to about
// 16 bits.
__device__ __forceinline__ void write_p_remainders(uint32_t s_addr, float2 sc2, float2 nm2, int ncol) {
#pragma unroll 1
  for (int c = kBN / 32 - 1; c >= 0; --c) {
    uint32_t v[32], w[16];
    tmem_ld32(s_addr + 32 * c, v);
    tmem_wait_ld();
#pragma unroll
    for (int e = 0; e < 32; ++e) v[e] = 32 * c + e < ncol ? v[e] : 0xff800000u;  // masked keys: weight 0
#pragma unroll
    for (int e = 0; e < 32; e += 2) {
      const float2 x = ffma2(make_float2(__uint_as_float(v[e]), __uint_as_float(v[e + 1])), sc2, nm2);
      const float2 pe = make_float2(fast_exp2(x.x), fast_exp2(x.y));
      const uint32_t hi = pack_bf16x2(pe.x, pe.y);
      const float2 r = ffma2(make_float2(bf16_lo(hi), bf16_hi(hi)), make_float2(-1.f, -1.f), pe);  // exact
      w[e / 2] = pack_bf16x2(r.x, r.y);
    }
    tmem_st16(s_addr + kBN / 2 + 16 * c, w);
  }
}

}  // namespace

// ------------------------------------------------------------------- plan
// One CTA: validate, then order the (request, q tile) pairs by decreasing
// number of KV tiles (counting sort) so that the heaviest items start first.
static_assert(kBuckets == 1024, "the plan kernel scans one bucket per thread of its 1024");
__global__ void __launch_bounds__(1024) prefill_plan_kernel(const PrefillParams p) {
  __shared__ int hist[kBuckets];
  __shared__ int cursor[kBuckets];
  pdl_launch_dependents();
  const int tid = threadIdx.x;
  for (int b = tid; b < kBuckets; b += blockDim.x) hist[b] = 0;
  __syncthreads();
  for (int r = tid; r < p.batch; r += blockDim.x) {
    if (!request_ok(p, r)) continue;
    const int qo = p.qo_indptr != nullptr ? p.qo_indptr[r + 1] - p.qo_indptr[r] : 1, n = p.kv_len[r];
    for (int qt = 0; qt * p.tile_rows < qo; ++qt)
      atomicAdd(&hist[min(kv_tiles(qt, qo, n, p.causal, p.tile_rows), kBuckets - 1)], 1);
  }
  __syncthreads();
  {
    // exclusive scan over the buckets in decreasing order, one bucket per thread
    __shared__ int warp_tot[32];
    const int lane = tid & 31, warp = tid >> 5;
    const int b = kBuckets - 1 - tid;
    const int c = hist[b];
    int x = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) warp_tot[warp] = x;
    __syncthreads();
    if (warp == 0) {
      int w = warp_tot[lane];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, w, o);
        if (lane >= o) w += y;
      }
      warp_tot[lane] = w;  // inclusive
    }
    __syncthreads();
    cursor[b] = (warp > 0 ? warp_tot[warp - 1] : 0) + x - c;
    if (tid == 0) p.hdr[0] = min(warp_tot[31], p.max_rq) * p.item_heads;
  }
  __syncthreads();
  for (int r = tid; r < p.batch; r += blockDim.x) {
    if (!request_ok(p, r)) continue;
    const int qo = p.qo_indptr != nullptr ? p.qo_indptr[r + 1] - p.qo_indptr[r] : 1, n = p.kv_len[r];
    for (int qt = 0; qt * p.tile_rows < qo; ++qt) {
      const int pos = atomicAdd(&cursor[min(kv_tiles(qt, qo, n, p.causal, p.tile_rows), kBuckets - 1)], 1);
      if (pos < p.max_rq) p.rq_list[pos] = make_int2(r, qt);
    }
  }
}

// ----------------------------------------------------------------- kernel
template <int QB, int KS, bool STAGE>
__global__ void __launch_bounds__(kThreadsPf, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                   const PrefillParams p) {
  constexpr int kQB = QB, kKSlots = KS, kVSlots = kRingTiles - QB - KS;
  static_assert(kQB >= 2 && kKSlots >= 2 && kVSlots >= 2, "ring depths");
  constexpr uint32_t kOffK = kQB * kTileBytes;
  constexpr uint32_t kOffV = (kQB + kKSlots) * kTileBytes;
  using Bars = BarsT<kQB, kKSlots, kVSlots>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = base + kOffQ;
  uint8_t* sK = base + kOffK;
  uint8_t* sV = base + kOffV;
  Bars* bars = reinterpret_cast<Bars*>(base + kOffBar);
  volatile int* abort = &bars->abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kQB; ++i) {
      mbar_init(&bars->q_full[i], 1);
      // the item's last S product, or the read of the O tile staged in it
      mbar_init(&bars->q_empty[i], 1);
    }
    for (int i = 0; i < kKSlots; ++i) {
      mbar_init(&bars->k_full[i], 1);
      mbar_init(&bars->k_empty[i], 1);
    }
    for (int i = 0; i < kVSlots; ++i) {
      mbar_init(&bars->v_full[i], 1);
      mbar_init(&bars->v_empty[i], 1);
    }
    for (int i = 0; i < kSB; ++i) {
      mbar_init(&bars->s_full[i], 1);
      mbar_init(&bars->p_full[i], 4);
      mbar_init(&bars->pv_done[i], 1);
    }
    mbar_init(&bars->drain, 2);  // one commit from each MMA-issuing warp
    mbar_init(&bars->o_sync, 4);
    bars->abort = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_map(&tm_q);
    tma_prefetch_map(&tm_k);
    tma_prefetch_map(&tm_v);
  }
  if (warp == 1) {
    tmem_alloc(&bars->tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_slot;
  pdl_wait_primary();  // the plan kernel's item list
  const int n_items = p.hdr[0];

  if (warp == 0 || warp == kWarpV) {
    // ------------------------------------------------------------- producers
    // Warp 0 loads the Q tile of each item and its K tiles, warp kWarpV its V
    // tiles: a warp keeps only a few TMA copies in flight, so two issuing warps
    // double the rate at which a tile's page boxes are requested.
    const bool is_v = warp == kWarpV;
    uint32_t it_ctr = 0, kv_ctr = 0;
    PItem nxt = prefill_item_or_empty(p, round_item(0), n_items);
    int pid_first = window_pid(p, nxt.pbase, nxt.need, 0, lane);  // first page-id window of the next item
    for (int it = round_item(0); it < n_items; ++it_ctr, it = round_item(it_ctr)) {
      const PItem I = nxt;
      nxt = prefill_item_or_empty(p, round_item(it_ctr + 1), n_items);
      int pid_win = pid_first, win = 0;
      int pid_ahead = window_pid(p, I.pbase, I.need, 1, lane);
      pid_first = window_pid(p, nxt.pbase, nxt.need, 0, lane);
      if (!is_v) {
        const int qb = it_ctr % kQB;
        if (!warp_mbar_wait(&bars->q_empty[qb], ((it_ctr / kQB) & 1u) ^ 1u, abort, p.status)) break;
        if (lane == 0) {
          mbar_arrive_expect_tx(&bars->q_full[qb], kTileBytes);
          tma_load_3d(sQ + qb * kTileBytes, &tm_q, 0, I.h, I.q0, &bars->q_full[qb]);
          tma_load_3d(sQ + qb * kTileBytes + kHalf, &tm_q, 64, I.h, I.q0, &bars->q_full[qb]);
        }
        __syncwarp();
      }
      bool ok = true;
      const uint32_t depth = is_v ? (uint32_t)kVSlots : (uint32_t)kKSlots;
      for (int j = 0; j < I.n_kv && ok; ++j, ++kv_ctr) {
        const int slot = kv_ctr % depth;
        const int w = tile_window(p, j);
        if (w != win) {  // the window read ahead; read the one after it
          pid_win = pid_ahead;
          win = w;
          pid_ahead = window_pid(p, I.pbase, I.need, w + 1, lane);
        }
        const TileBox box = tile_box(p, I.need, j, pid_win, lane);
        // A K slot is free again once the S product of its previous tile has
        // completed (k_empty); a V slot once the P V product of its previous
        // tile has (v_empty).
        ok = is_v ? warp_mbar_wait(&bars->v_empty[slot], ((kv_ctr / kVSlots) & 1u) ^ 1u, abort, p.status)
                  : warp_mbar_wait(&bars->k_empty[slot], ((kv_ctr / kKSlots) & 1u) ^ 1u, abort, p.status);
        if (ok) {
          if (!is_v)
            load_kv_tile(p, box, &tm_k, I.g, sK + slot * kTileBytes, &bars->k_full[slot], lane);
          else
            load_kv_tile(p, box, &tm_v, I.g, sV + slot * kTileBytes, &bars->v_full[slot], lane);
        }
      }
      if (!ok) break;
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------- S = Q K^T
    // S_j into TMEM buffer j % kSB, as soon as K_j has landed and the buffer's
    // previous tile has gone through P V. The softmax warps overwrite S_j with
    // P_j (bf16), which warp kWarpPV multiplies into O.
    constexpr uint32_t idesc_s = idesc_bf16_f32(kBM, kBN, 0);
    const uint32_t sQa = smem_u32(sQ), sKa = smem_u32(sK);
    uint32_t it_ctr = 0, kv_ctr = 0;
    bool ok = true;
    PItem nxt = prefill_item_or_empty(p, round_item(0), n_items);
    for (int it = round_item(0); it < n_items && ok; ++it_ctr, it = round_item(it_ctr)) {
      const PItem I = nxt;
      nxt = prefill_item_or_empty(p, round_item(it_ctr + 1), n_items);
      const int qb = it_ctr % kQB;
      ok = warp_mbar_wait(&bars->q_full[qb], (it_ctr / kQB) & 1u, abort, p.status);
      if (!ok) break;
      tc_fence_after();
      const uint64_t dq = sw128_desc(sQa + qb * kTileBytes, 16, 1024);
      for (int j = 0; j < I.n_kv; ++j, ++kv_ctr) {
        const int slot = kv_ctr % kKSlots;
        const int sb = kv_ctr % kSB;
        // every tile's phase of pv_done is waited in order (tiles >= kSB)
        ok = warp_mbar_wait(&bars->k_full[slot], (kv_ctr / kKSlots) & 1u, abort, p.status) &&
             (kv_ctr < (uint32_t)kSB ||
              warp_mbar_wait(&bars->pv_done[sb], ((kv_ctr - kSB) / kSB) & 1u, abort, p.status));
        if (!ok) break;
        tc_fence_after();
        if (lane == 0) {
          const uint64_t dk = sw128_desc(sKa + slot * kTileBytes, 16, 1024);
#pragma unroll
          for (int kk = 0; kk < kD / 16; ++kk) {
            const uint32_t off = (kk / 4) * kHalf + (kk % 4) * 32;
            tc_mma_f16(tmem + col_s(sb), desc_advance(dq, off), desc_advance(dk, off), idesc_s, kk > 0);
          }
          tc_commit(&bars->s_full[sb]);
          tc_commit(&bars->k_empty[slot]);
          if (j == I.n_kv - 1 && !o_staged<STAGE>(p, I)) tc_commit(&bars->q_empty[qb]);
        }
        __syncwarp();
      }
      if (!ok) break;
      if (I.n_kv == 0 && !o_staged<STAGE>(p, I) && lane == 0) mbar_arrive(&bars->q_empty[qb]);
      __syncwarp();
    }
    // all MMAs of this thread complete before TMEM is released
    if (lane == 0) {
      tc_commit(&bars->drain);
      const uint64_t t0 = globaltimer_ns();
      while (!mbar_try_wait(&bars->drain, 0) && globaltimer_ns() - t0 < kWaitLimitNs) {
      }
    }
    __syncwarp();
  } else if (warp == kWarpPV) {
    // ---------------------------------------------------------- O += P V
    constexpr uint32_t idesc_pv = idesc_bf16_f32(kBM, kD, 1);
    const uint32_t sVa = smem_u32(sV);
    uint32_t kv_ctr = 0, it_ctr = 0;
    bool ok = true;
    PItem nxt = prefill_item_or_empty(p, round_item(0), n_items);
    for (int it = round_item(0); it < n_items && ok; ++it_ctr, it = round_item(it_ctr)) {
      const PItem I = nxt;
      nxt = prefill_item_or_empty(p, round_item(it_ctr + 1), n_items);
      const uint32_t t_o = tmem + col_o(it_ctr & 1);  // this item's O accumulator
      for (int j = 0; j < I.n_kv; ++j, ++kv_ctr) {
        const int slot = kv_ctr % kVSlots;
        const int sb = kv_ctr % kSB;
        ok = warp_mbar_wait(&bars->p_full[sb], (kv_ctr / kSB) & 1u, abort, p.status) &&
             warp_mbar_wait(&bars->v_full[slot], (kv_ctr / kVSlots) & 1u, abort, p.status);
        if (!ok) break;
        // keys past kv_len in the request's last tile: zero their V rows so that
        // stale values cannot reach O through a zero weight
        const int valid = I.kv - j * kBN;
        if (valid < kBN) {
          const uint32_t vt = sVa + slot * kTileBytes;
          for (int i = lane; i < (kBN - valid) * 16; i += 32) {
            const int rr = valid + i / 16, c16 = i % 16;
            asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};" ::"r"(vt + (c16 / 8) * kHalf + rr * 128 +
                                                                        (c16 % 8) * 16),
                         "r"(0)
                         : "memory");
          }
          fence_proxy_async_smem();
          __syncwarp();
        }
        tc_fence_after();
        if (lane == 0) {
          const uint64_t dv = sw128_desc(sVa + slot * kTileBytes, kHalf, 1024);
          const uint32_t pa = tmem + col_s(sb);
          // P: 64 columns of bf16 pairs; for split items the rounding
          // remainders follow in the buffer's other 64 columns
#pragma unroll
          for (int kk = 0; kk < kBN / 16; ++kk)
            tc_mma_f16_tmem_a(t_o, pa + 8 * kk, desc_advance(dv, kk * 2048), idesc_pv, (j > 0 || kk > 0) ? 1u : 0u);
          if (split_item(p.causal, p.tile_rows, I.qt, I.qo_len, I.kv)) {
#pragma unroll
            for (int kk = 0; kk < kBN / 16; ++kk)
              tc_mma_f16_tmem_a(t_o, pa + kBN / 2 + 8 * kk, desc_advance(dv, kk * 2048), idesc_pv, 1u);
          }
          tc_commit(&bars->pv_done[sb]);  // also frees the S buffer
          tc_commit(&bars->v_empty[slot]);
        }
        __syncwarp();
      }
    }
    if (lane == 0) {
      tc_commit(&bars->drain);
      const uint64_t t0 = globaltimer_ns();
      while (!mbar_try_wait(&bars->drain, 0) && globaltimer_ns() - t0 < kWaitLimitNs) {
      }
    }
    __syncwarp();
  } else if (warp >= 2 && warp < 6) {
    // --------------------------------------------------- softmax / epilogue
    // Item i's epilogue is deferred until item i + 1's first tile has been
    // published: the wait for item i's last P V then overlaps useful work.
    // Items alternate between the two O accumulators.
    const int wq = warp & 3;
    const int row = wq * 32 + lane;  // tile row: query row qrow of head (first head) + qhead
    const int qrow = row / p.tile_heads, qhead = row - qrow * p.tile_heads;
    const uint32_t t_lane = tmem + ((uint32_t)(wq * 32) << 16);
    uint32_t s_ctr = 0, o_phase = 0, it_ctr = 0;
    const bool o_issuer = (warp == 2 && lane == 0);
    int pending_q = -1;  // Q buffer holding an O tile whose TMA store may still read it
    bool ok = true;
    struct Pend {
      int q0, h, rows, n_kv, qb, ob;  // h: the tile's first query head; rows: valid query rows
      bool staged;  // O goes through the Q buffer (which it then releases)
      uint32_t last;  // running index of the item's last tile
      float m, l;
    };
    Pend pend{};
    bool has_pend = false;
    // Once a staged O tile has been read by its TMA store, its Q buffer may be
    // reloaded (the store has long finished when this is called).
    auto release_staged = [&]() {
      if (o_issuer && pending_q >= 0) {
        bulk_wait_read_all();
        mbar_arrive(&bars->q_empty[pending_q]);
        pending_q = -1;
      }
    };
    // O / l and the log-sum-exp of a finished item, once its last P V is done.
    auto epilogue = [&](const Pend& E) -> bool {
      if (E.n_kv > 0) {
        if (!warp_mbar_wait(&bars->pv_done[E.last % kSB], (E.last / kSB) & 1u, abort, p.status)) return false;
        tc_fence_after();
      }
      const float inv_l = E.l > 0.f ? 1.0f / E.l : 0.f;
      const float2 il2 = make_float2(inv_l, inv_l);
      const bool store = qrow < E.rows;
      const int64_t orow = ((int64_t)(E.q0 + qrow) * p.hq + E.h + qhead) * kD;
      const uint32_t o_addr = t_lane + col_o(E.ob);
      uint32_t v[kD];
      if (E.n_kv > 0) {
        tmem_ld32(o_addr + 0, *reinterpret_cast<uint32_t(*)[32]>(v + 0));
        tmem_ld32(o_addr + 32, *reinterpret_cast<uint32_t(*)[32]>(v + 32));
        tmem_ld32(o_addr + 64, *reinterpret_cast<uint32_t(*)[32]>(v + 64));
        tmem_ld32(o_addr + 96, *reinterpret_cast<uint32_t(*)[32]>(v + 96));
        tmem_wait_ld();
      } else {
#pragma unroll
        for (int e = 0; e < kD; ++e) v[e] = 0u;
      }
      const bool staged = E.staged;
      if (staged) {
        // full tile: stage bf16 O (128-byte swizzled like Q) in the item's Q
        // buffer, free now that its last S product has completed, and write it
        // with two TMA stores
        uint8_t* sO = sQ + E.qb * kTileBytes;
        const uint32_t so = smem_u32(sO);
#pragma unroll
        for (int k = 0; k < kD / 8; ++k) {
          const uint32_t a0 = scale_pack(v + 8 * k + 0, il2);
          const uint32_t a1 = scale_pack(v + 8 * k + 2, il2);
          const uint32_t a2 = scale_pack(v + 8 * k + 4, il2);
          const uint32_t a3 = scale_pack(v + 8 * k + 6, il2);
          const uint32_t addr = so + (k / 8) * kHalf + row * 128 + (((k % 8) ^ (row & 7)) * 16);
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a0), "r"(a1), "r"(a2), "r"(a3)
                       : "memory");
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->o_sync);
        if (!warp_mbar_wait(&bars->o_sync, o_phase & 1u, abort, p.status)) return false;
        ++o_phase;
        if (o_issuer) {
          tma_store_3d(&tm_o, 0, E.h, E.q0, sO);
          tma_store_3d(&tm_o, 64, E.h, E.q0, sO + kHalf);
          bulk_commit_group();
          pending_q = E.qb;
        }
      } else if (store) {
        if (p.o_dtype == PD_BF16) {
          uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.o) + orow);
#pragma unroll
          for (int k = 0; k < kD / 8; ++k) {
            uint4 u;
            u.x = scale_pack(v + 8 * k + 0, il2);
            u.y = scale_pack(v + 8 * k + 2, il2);
            u.z = scale_pack(v + 8 * k + 4, il2);
            u.w = scale_pack(v + 8 * k + 6, il2);
            dst[k] = u;
          }
        } else {
          float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.o) + orow);
#pragma unroll
          for (int k = 0; k < kD / 4; ++k)
            dst[k] = make_float4(__uint_as_float(v[4 * k]) * inv_l, __uint_as_float(v[4 * k + 1]) * inv_l,
                                 __uint_as_float(v[4 * k + 2]) * inv_l, __uint_as_float(v[4 * k + 3]) * inv_l);
        }
      }
      if (store && p.lse != nullptr)
        p.lse[(int64_t)(E.q0 + qrow) * p.hq + E.h + qhead] =
            (E.n_kv > 0 && E.l > 0.f) ? (E.m + log2f(E.l)) * kLn2 : -INFINITY;
      tc_fence_before();
      return true;
    };
    PItem nxt = prefill_item_or_empty(p, round_item(0), n_items);
    for (int it = round_item(0); it < n_items && ok; ++it_ctr, it = round_item(it_ctr)) {
      const PItem I = nxt;
      nxt = prefill_item_or_empty(p, round_item(it_ctr + 1), n_items);
      const int qb = it_ctr % kQB, ob = it_ctr & 1;
      const uint32_t o_addr = t_lane + col_o(ob);
      const int lim = I.kv - I.qo_len + I.qt * p.tile_rows + qrow;  // last key this row may see (causal)
      // l: sum of the fp32 weights (normalises O, gives the lse)
      float m = -INFINITY, l = 0.f;
      for (int j = 0; j < I.n_kv; ++j) {
        const int sb = s_ctr % kSB;
        ok = warp_mbar_wait(&bars->s_full[sb], (s_ctr / kSB) & 1u, abort, p.status);
        if (!ok) break;
        tc_fence_after();
        const int k0 = j * kBN;
        int ncol = min(kBN, I.kv - k0);
        if (p.causal) ncol = min(ncol, lim - k0 + 1);
        const uint32_t s_addr = t_lane + col_s(sb);
        // the whole S row in registers: four loads, one wait
        uint32_t v[kBN];
        tmem_ld32(s_addr + 0, *reinterpret_cast<uint32_t(*)[32]>(v + 0));
        tmem_ld32(s_addr + 32, *reinterpret_cast<uint32_t(*)[32]>(v + 32));
        tmem_ld32(s_addr + 64, *reinterpret_cast<uint32_t(*)[32]>(v + 64));
        tmem_ld32(s_addr + 96, *reinterpret_cast<uint32_t(*)[32]>(v + 96));
        tmem_wait_ld();
        // columns past ncol are masked only in tiles where some row of the warp has any
        const bool full_tile = __all_sync(0xffffffffu, ncol >= kBN);
        if (!full_tile) {
          // masked keys score -inf: weight 0 below
#pragma unroll
          for (int e = 0; e < kBN; ++e) v[e] = e < ncol ? v[e] : 0xff800000u;
        }
        // P = 2^(s * scale - m) as bf16 pairs, written over the S columns
        // (masked columns: -inf, weight 0), sums in packed pairs. Once a
        // warp's rows all have a finite running max m, a tile's P is computed
        // with that m at once and accepted if the row's weights sum to at most
        // 2^kRescaleThreshold, which bounds every weight by it; otherwise the
        // tile is redone with its exact row max (then O is rescaled). The
        // check costs one comparison per row where a running maximum of the
        // exponents would cost an instruction per pair of weights, and the
        // softmax warps are bound by the instructions they issue. The first
        // tile of an item, and split items (whose remainder pass reads S from
        // tensor memory, where the pairs are written), take the exact max
        // first.
        const bool split = split_item(p.causal, p.tile_rows, I.qt, I.qo_len, I.kv);
        bool spec = !split && __all_sync(0xffffffffu, m > -INFINITY);
        uint32_t w[kBN / 2];
        float2 ls2[2];
        for (;;) {
          float m_new = m;
          bool rescale = false;
          if (!spec) {
            // row max of the tile (four independent chains)
            float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
            for (int e = 0; e < kBN; e += 2)
              mx[(e / 2) & 3] = fmax3(mx[(e / 2) & 3], __uint_as_float(v[e]), __uint_as_float(v[e + 1]));
            const float mt = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
            if (mt > -INFINITY) {
              const float ms = mt * p.scale_log2;
              if (m == -INFINITY) {
                m_new = ms;
              } else if (ms > m + kRescaleThreshold) {
                m_new = ms;
                rescale = true;
              }
            }
            // tcgen05.ld / st are warp-collective: the whole warp rescales its
            // rows of O when any of them needs it (factor 1 for the others),
            // after the previous P V product has completed. That product's
            // barrier (buffer of tile s_ctr - 1) cannot move past this phase
            // before this tile's P is published, so waiting only when needed
            // keeps the phase count exact.
            if (__any_sync(0xffffffffu, rescale)) {
              const uint32_t prev = s_ctr - 1;
              ok = warp_mbar_wait(&bars->pv_done[prev % kSB], (prev / kSB) & 1u, abort, p.status);
              if (!ok) break;
              tc_fence_after();
              const float alpha = rescale ? exp2f(m - m_new) : 1.0f;
              l *= alpha;
#pragma unroll
              for (int c = 0; c < kD / 32; ++c) {
                uint32_t o[32];
                tmem_ld32(o_addr + c * 32, o);
                tmem_wait_ld();
#pragma unroll
                for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                tmem_st32(o_addr + c * 32, o);
              }
              tmem_wait_st();
            }
            m = m_new;
          }
          const float2 sc2 = make_float2(p.scale_log2, p.scale_log2), nm2 = make_float2(-m, -m);
          if (split) write_p_remainders(s_addr, sc2, nm2, ncol);
          ls2[0] = make_float2(0.f, 0.f);
          ls2[1] = make_float2(0.f, 0.f);
#pragma unroll
          for (int e = 0; e < kBN; e += 2) {
            const float2 x = ffma2(make_float2(__uint_as_float(v[e]), __uint_as_float(v[e + 1])), sc2, nm2);
            const float2 pe = make_float2(fast_exp2(x.x), fast_exp2(x.y));
            w[e / 2] = pack_bf16x2(pe.x, pe.y);
            ls2[(e / 2) & 1] = fadd2(ls2[(e / 2) & 1], pe);
          }
          if (!spec || !__any_sync(0xffffffffu, (ls2[0].x + ls2[0].y) + (ls2[1].x + ls2[1].y) > kSpecSumLimit)) break;
          spec = false;  // a weight may pass 2^8: redo the tile with its exact max
        }
        if (!ok) break;
        l += (ls2[0].x + ls2[0].y) + (ls2[1].x + ls2[1].y);
        tmem_st32(s_addr + 0, *reinterpret_cast<uint32_t(*)[32]>(w + 0));
        tmem_st32(s_addr + 32, *reinterpret_cast<uint32_t(*)[32]>(w + 32));
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->p_full[sb]);
        ++s_ctr;
        if (j == 0 && has_pend) {
          // the previous item's epilogue, now that this item's first P is out
          ok = epilogue(pend);
          has_pend = false;
          if (!ok) break;
        } else {
          release_staged();
        }
      }
      if (!ok) break;
      release_staged();
      const Pend cur{I.q0, I.h, I.rows, I.n_kv, qb, ob, o_staged<STAGE>(p, I), s_ctr - 1, m, l};
      if (I.n_kv == 0) {
        // no tile to overlap with: finish the pending item and this one now
        if (has_pend) {
          ok = epilogue(pend);
          has_pend = false;
          if (!ok) break;
          release_staged();
        }
        ok = epilogue(cur);
        if (!ok) break;
      } else {
        pend = cur;
        has_pend = true;
      }
    }
    if (ok && has_pend) ok = epilogue(pend);
    if (o_issuer) bulk_wait_all();
  }

  // Normally every copy has been consumed here. After an abort, copies may still
  // be in flight: give them a bounded 2 ms to land before shared memory is freed.
  if (*abort && warp == 0 && lane == 0) {
    const uint64_t t0 = globaltimer_ns();
    while (globaltimer_ns() - t0 < 2000000ull) {
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

// ------------------------------------------------------------------- host
// GQA packing on (1) or off (0: one query head per tile, any group).
#ifndef PD_PREFILL_GQA_PACK
#define PD_PREFILL_GQA_PACK 1
#endif
int32_t prefill_tile_heads(int32_t group) {
  return PD_PREFILL_GQA_PACK && group >= 1 && kBM % group == 0 ? group : 1;
}

PrefillLayout prefill_layout(int32_t batch, int32_t total_qo, int32_t max_qo_len, int32_t tile_heads) {
  PrefillLayout L{};
  const int rows = kBM / (tile_heads > 0 ? tile_heads : 1);
  const int64_t by_len = (int64_t)batch * ((max_qo_len + rows - 1) / rows);
  const int64_t by_rows = (int64_t)(total_qo + rows - 1) / rows + batch;
  L.max_rq = (int32_t)(by_len < by_rows ? by_len : by_rows);
  if (L.max_rq < 1) L.max_rq = 1;
  size_t off = 0;
  L.hdr = off;
  off = align_up(off + 64 * sizeof(int32_t), 256);
  L.rq_list = off;
  off = align_up(off + sizeof(int2) * (size_t)L.max_rq, 256);
  L.total = off;
  return L;
}

int prefill_supported(int32_t kv_dtype, int32_t head_dim, int32_t page_size) {
  if (kv_dtype != PD_BF16 || head_dim != kD) return PD_ERR_UNSUPPORTED;
  // page sizes that tile a 128-token block with whole boxes (powers of two >= 8)
  if (page_size < 8 || (page_size & (page_size - 1)) != 0) return PD_ERR_UNSUPPORTED;
  return PD_OK;
}

int launch_prefill(PrefillParams& p, const void* q, const void* k_pool, const void* v_pool, cudaStream_t stream) {
  CUtensorMap tq, tk, tv, to;
  const int pb = p.page_size < kBN ? p.page_size : kBN;
  memset(&to, 0, sizeof(to));
  if (p.o_dtype == PD_BF16 &&
      !make_rows_map(&to, p.o, PD_BF16, p.total_qo, p.hq, kD, 64, p.tile_rows, true, p.tile_heads))
    return PD_ERR_CUDA;
  if (!make_rows_map(&tq, q, PD_BF16, p.total_qo, p.hq, kD, 64, p.tile_rows, true, p.tile_heads) ||
      !make_pool_map(&tk, k_pool, PD_BF16, p.num_pages, p.hkv, p.page_size, kD, 64, pb, true, p.nhd != 0) ||
      !make_pool_map(&tv, v_pool, PD_BF16, p.num_pages, p.hkv, p.page_size, kD, 64, pb, true, p.nhd != 0))
    return PD_ERR_CUDA;
  // Calls whose requests average at least half a tile of query rows run the
  // shape that fetches Q an item ahead and stages O; decode-like calls the
  // deeper K ring and direct O stores.
  const bool long_q = (int64_t)p.total_qo * 2 >= (int64_t)kBM * p.batch;
  auto kernel = long_q ? prefill_kernel<3, 2, true> : prefill_kernel<2, 3, false>;
  // per device and kernel shape: whether the shared-memory attribute is set
  // there (callers may run on several threads)
  static std::atomic<bool> configured[64][2];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PD_ERR_CUDA;
  const bool cached = dev >= 0 && dev < 64 && partition_sms() == 0;
  if (!cached || !configured[dev][long_q].load(std::memory_order_acquire)) {
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kPrefillSmem) != cudaSuccess)
      return PD_ERR_CUDA;
    if (cached) configured[dev][long_q].store(true, std::memory_order_release);
  }
  last_kernel() = "prefill_kernel";
  prefill_plan_kernel<<<1, 1024, 0, stream>>>(p);
  int64_t grid = device_sm_count();
  const int64_t max_items = (int64_t)p.max_rq * p.item_heads;
  if (grid > max_items) grid = max_items;
  if (grid < 1) grid = 1;
  // A programmatic dependent of the plan (CTAs set up while it finishes),
  // except when timed alone through the profiling events.
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kThreadsPf);
  cfg.dynamicSmemBytes = kPrefillSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = profile_events().start != nullptr ? 0 : 1;
  profile_begin(stream);
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, tq, tk, tv, to, p);
  profile_end(stream);
  return e == cudaSuccess && cudaGetLastError() == cudaSuccess ? PD_OK : PD_ERR_CUDA;
}

}  // namespace pd
