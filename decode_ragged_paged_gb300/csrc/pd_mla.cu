// pd_mla.cu -- MLA decode over a paged latent cache on the 5th-generation
// tensor cores (tcgen05, accumulators in TMEM).
//
// Perplexity, "Disaggregated prefill and decode" (2025), section
// "Disaggregated Deployments", "DeepSeek-R1": multi-head latent attention keeps
// one compressed vector per token that every query head reads, so the cache is
// one row per token and is never split by head. With the up-projections folded
// into q and o (MLA's published decode form) a token's row is
// [c^kv (512 values) | k^rope (64 values)]: scores use the whole 576-value row,
// values its first 512 entries.
//
// All query heads (up to 128, zero-padded) form the 128 rows of one tile, so
// the latent row of each token is read once per request. O for 128 rows x 512
// values fills all of TMEM, so each (request, chunk) is run by a pair of CTAs,
// each owning 256 of the value columns (half h: columns [256h, 256h + 256));
// both compute the full 128 x 64 score tile from the same latent tiles, the
// second read of a tile coming from L2.
//
// Shared memory holds Q (144 KiB) for the whole request, so a 64-token tile
// (72 KiB) is not double-buffered whole: it streams through in nine column
// chunks of 64 tokens x 64 values (8 KiB), and this half's value columns are
// read a second time (from L2) into a 16 KiB slot of their own for O += P C_h,
// two column chunks at a time (two products of 128 columns per tile). Each
// MMA of the score product then reads its 4 KiB slice of Q for 64 keys. The
// column-chunk rings take what the value slot leaves: their depth, not the
// tensor pipe, sets the pace (a 32 KiB value slot used once per tile, with
// three ring slots per issuer instead of four, was 7 % slower).
//
// Three launches, each a programmatic dependent of the one before:
//   1. plan    one CTA: validates requests, picks the chunk length from the
//              batch's total tokens (about one chunk per CTA pair), lists the
//              (request, chunk) pairs longest first;
//   2. decode  persistent CTA pairs (one CTA per SM) walk the list in
//              serpentine order. Warp roles:
//                warp 0    TMA producer: the request's Q tile (9 boxes of 64
//                          columns x 128 heads) and each tile's nine column
//                          chunks (128-byte-swizzled boxes, one per page
//                          run), even chunks to one 4-slot ring, odd chunks
//                          to another;
//                warp 8    TMA producer of the value slot (this half's four
//                          column chunks of the tile, two at a time);
//                warps 1, 6  issue S = Q C^T as two partial products, over
//                          the even and the odd column chunks (one thread
//                          issues a tcgen05.mma about every 94 cycles
//                          whatever N, so one issuer would bound the tile);
//                          warp 1 also allocates TMEM;
//                warp 7    issues O += P C_h with P read from TMEM (bf16
//                          pairs and their rounding remainders), over the
//                          value slot's two column chunks at a time;
//                warps 2-5 one head per thread: S = the sum of the two
//                          partials, online softmax (lazy O
//                          rescale), the epilogue (final o and lse, or a fp32
//                          partial for a request split into chunks);
//   3. merge   requests split into chunks (listed by the plan): log-sum-exp
//              merge of the partials, a small grid striding over them.
// Every wait is bounded; on a timeout the CTA records PD_DEV_TIMEOUT, drains
// and frees its TMEM.
#include <atomic>
#include <math.h>

#include "pd_common.cuh"
#include "pd_internal.h"
#include "pd_tc.cuh"

namespace pd {

namespace {

constexpr int kDc = 512;                 // latent (value) width
constexpr int kDr = 64;                  // rope width (scores only)
constexpr int kW = kDc + kDr;            // stored row: 576 values
constexpr int kWC = kW / 64;             // 9 column chunks of 64 values (128 bytes)
constexpr int kRows = 128;               // tile rows: query heads, zero-padded
constexpr int kN = 64;                   // tokens per latent tile
constexpr int kHalfV = kDc / 2;          // value columns per CTA of a pair
constexpr int kVChunks = kHalfV / 64;    // 4 column chunks per half
constexpr int kThreadsMla = 288;         // 9 warps
constexpr int kWarpPV = 7;
constexpr int kWarpV = 8;                // producer of the value slot
// warps issuing the partial score products (one issuer, with one 6-slot ring,
// was measured slower: a thread issues an MMA about every 94 cycles)
constexpr int kSIssuers = 2;
static_assert(kSIssuers == 1 || kSIssuers == 2, "one or two score issuers");
// index of the partial product warp w issues, or -1; partial i takes the
// column chunks c with c % kSIssuers == i
__device__ __forceinline__ int s_issuer(int w) { return w == 1 ? 0 : (w == 6 && kSIssuers > 1) ? 1 : -1; }
constexpr int kRing = 8 / kSIssuers;     // column-chunk ring of each issuer
// tile t's column chunk c travels through ring c % kSIssuers as that ring's
// entry ring_seq(t, c) (with two rings: five chunks per tile in ring 0, four in ring 1)
__device__ __forceinline__ uint32_t ring_seq(uint32_t t, int c) {
  const int r = c % kSIssuers;
  return t * (uint32_t)((kWC - r + kSIssuers - 1) / kSIssuers) + (uint32_t)(c / kSIssuers);
}
constexpr int kSB = 2;                   // S / P buffers in TMEM
constexpr uint32_t kQChunk = kRows * 128;          // 16 KiB: 128 rows x 64 values
constexpr uint32_t kQBytes = kWC * kQChunk;        // 144 KiB
constexpr uint32_t kCChunk = kN * 128;             // 8 KiB: 64 tokens x 64 values
constexpr int kVPass = 2;                          // value-slot fills (and P C_h products) per tile
constexpr int kVSlotChunks = kVChunks / kVPass;    // column chunks per fill
constexpr uint32_t kVBytes = kVSlotChunks * kCChunk;  // 16 KiB
constexpr uint32_t kOffC = kQBytes;
constexpr uint32_t kOffV = kOffC + kSIssuers * kRing * kCChunk;
constexpr uint32_t kOffBar = kOffV + kVBytes;
constexpr size_t kMlaSmem = kOffBar + 256 + 1024;
static_assert(kMlaSmem <= 227 * 1024, "shared memory");
constexpr uint32_t kTmemCols = 512;
// partial score product `part` of S buffer b (P is written over part 0)
__device__ __forceinline__ uint32_t col_s(int b, int part = 0) { return (uint32_t)(b * kSIssuers + part) * kN; }
constexpr uint32_t kColO = 256;                    // O half: columns [256, 512)
static_assert(kSB * kSIssuers * kN <= (int)kColO && kColO + kHalfV <= kTmemCols, "TMEM columns");
static_assert(kCChunk % 1024 == 0 && kOffV % 1024 == 0, "128-byte-swizzled chunks start on 1 KiB");
constexpr float kRescaleThreshold = 8.0f;          // log2 units
constexpr int kBuckets = 1024;
static_assert(kBuckets == 1024, "the plan kernel scans one bucket per thread of its 1024");

struct Bars {
  uint64_t q_full, q_empty, c_full[kSIssuers][kRing], c_empty[kSIssuers][kRing], v_full, v_empty;
  uint64_t s_full[kSB], p_full[kSB], pv_done[kSB], o_free, drain;
  uint32_t tmem_slot;
  int abort;
};
static_assert(sizeof(Bars) <= 256, "barrier block");

// A (request, chunk) pair of the work list and what the kernels need of it.
struct MItem {
  int r, c, first, nch, t0, len, ntiles, pbase, need;
  bool valid;
};

__device__ __forceinline__ MItem mla_item(const MlaParams& p, int idx) {
  MItem I{};
  const int2 rc = p.chunk_list[idx];
  const int4 info = p.req_info[rc.x];
  const int cl = p.hdr[1];
  I.r = rc.x;
  I.c = rc.y;
  I.first = info.x;
  I.nch = info.y;
  I.valid = info.z >= 0;
  const int kv = info.z >= 0 ? info.z : 0;
  I.t0 = I.c * cl;
  I.len = max(0, min(cl, kv - I.t0));
  I.ntiles = (I.len + kN - 1) / kN;
  I.pbase = p.page_indptr[I.r];
  I.need = (kv + p.page_size - 1) / p.page_size;
  return I;
}

__device__ __forceinline__ int pair_item(int k, int pair, int pairs) {
  return k * pairs + ((k & 1) ? pairs - 1 - pair : pair);
}

// P = 2^(s * scale - m) for one head's row of a 64-token tile, written over
// the first partial-score buffer in TMEM; l accumulates the fp32 weights. Each
// 32-column chunk of S is replaced by its own words: per 16 keys, 8 words of
// bf16 pairs, then 8 words of their rounding remainders bf16(p - hi), and
// P C_h adds both products, so it sees p to about 16 bits. MLA's scores, over
// 576-value rows, are peaked: a few keys carry most of the weight at any
// length, and bf16 weights alone (8 significant bits) would move such outputs
// by several 1e-3.
__device__ __forceinline__ void mla_write_p(const uint32_t (&v)[kN], uint32_t s_addr, float2 sc2, float2 nm2,
                                            float& l) {
  float2 ls2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
  for (int c = 0; c < kN / 32; ++c) {
    uint32_t w[32];
#pragma unroll
    for (int e = 0; e < 32; e += 2) {
      const int x0 = 32 * c + e;
      const float2 x = ffma2(make_float2(__uint_as_float(v[x0]), __uint_as_float(v[x0 + 1])), sc2, nm2);
      const float2 pe = make_float2(fast_exp2(x.x), fast_exp2(x.y));
      const int wi = (e / 16) * 16 + (e % 16) / 2;  // word of this pair in the chunk
      w[wi] = pack_bf16x2(pe.x, pe.y);
      const float2 r = ffma2(make_float2(bf16_lo(w[wi]), bf16_hi(w[wi])), make_float2(-1.f, -1.f), pe);  // exact
      w[wi + 8] = pack_bf16x2(r.x, r.y);
      ls2[(e / 2) & 1] = fadd2(ls2[(e / 2) & 1], pe);
    }
    tmem_st32(s_addr + 32 * c, w);
  }
  l += (ls2[0].x + ls2[0].y) + (ls2[1].x + ls2[1].y);
}

}  // namespace

// ------------------------------------------------------------------- plan
__global__ void __launch_bounds__(1024) mla_plan_kernel(const MlaParams p) {
  __shared__ int s_bucket[kBuckets];
  __shared__ int s_warp[32];
  __shared__ long long s_total;
  __shared__ int s_carry;
  __shared__ int s_nsplit;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  pdl_launch_dependents();
  s_bucket[tid] = 0;
  if (tid == 0) {
    s_total = 0;
    s_carry = 0;
    s_nsplit = 0;
  }
  __syncthreads();
  // 1. validate, total tokens of the valid requests
  long long part = 0;
  for (int r = tid; r < p.batch; r += 1024) {
    const int n = p.kv_len[r];
    const int pa = p.page_indptr[r], pb = p.page_indptr[r + 1];
    int code = 0;
    if (pa < 0 || pb < pa) code = PD_DEV_BAD_INDPTR;
    else if (n < 0 || n > p.max_kv_len) code = PD_DEV_BAD_LENGTH;
    else if ((long long)(pb - pa) * p.page_size < n) code = PD_DEV_BAD_PAGE_TABLE;
    if (code) report(p.status, code);
    p.req_info[r] = make_int4(0, 0, code ? -1 : n, 0);
    if (!code) part += n;
  }
  atomicAdd(reinterpret_cast<unsigned long long*>(&s_total), (unsigned long long)part);
  __syncthreads();
  // 2. chunk length: about one chunk per CTA pair, whole 256-token multiples,
  // at least 512; then every request has at most total / cl + 1 chunks, so the
  // list never holds more than batch + pairs entries. A request longer than
  // the chunk is cut and merged afterwards, which writes and reads its fp32
  // partial outputs; two chunks per pair measured slower on the 128-request
  // batch (kernel 0.1925 against 0.1884 ms, call 0.214 against 0.202 ms).
  long long cl = (s_total + p.pairs - 1) / p.pairs;
  cl = ((cl + 255) / 256) * 256;
  if (cl < 512) cl = 512;
  const int chunk_len = (int)min(cl, (long long)1 << 30);
  // 3. chunks per request and their first index (block-wide exclusive scan)
  for (int base = 0; base < p.batch; base += 1024) {
    const int r = base + tid;
    int nch = 0;
    if (r < p.batch) {
      const int n = p.req_info[r].z;
      nch = n > 0 ? (n + chunk_len - 1) / chunk_len : 1;  // an empty request still writes o = 0
    }
    int x = nch;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) s_warp[wid] = x;
    __syncthreads();
    if (wid == 0) {
      int w = s_warp[lane];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, w, o);
        if (lane >= o) w += y;
      }
      s_warp[lane] = w;
    }
    __syncthreads();
    const int excl = s_carry + (wid > 0 ? s_warp[wid - 1] : 0) + x - nch;
    if (r < p.batch) {
      int4 info = p.req_info[r];
      info.x = excl;
      info.y = nch;
      p.req_info[r] = info;
    }
    __syncthreads();
    if (tid == 0) s_carry += s_warp[31];
    __syncthreads();
  }
  const int total = s_carry;
  // 4. the (request, chunk) list, longest chunks first (counting sort on tiles)
  for (int r = tid; r < p.batch; r += 1024) {
    const int4 info = p.req_info[r];
    const int n = info.z > 0 ? info.z : 0;
    for (int c = 0; c < info.y; ++c) {
      const int len = max(0, min(chunk_len, n - c * chunk_len));
      atomicAdd(&s_bucket[min((len + kN - 1) / kN, kBuckets - 1)], 1);
    }
  }
  __syncthreads();
  // descending bucket order: position of bucket b = count of buckets above it
  {
    const int b = kBuckets - 1 - tid;  // thread 0 takes the longest bucket
    const int cnt = s_bucket[b];
    int x = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) s_warp[wid] = x;
    __syncthreads();
    if (wid == 0) {
      int w = s_warp[lane];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, w, o);
        if (lane >= o) w += y;
      }
      s_warp[lane] = w;
    }
    __syncthreads();
    const int start = (wid > 0 ? s_warp[wid - 1] : 0) + x - cnt;
    __syncthreads();
    s_bucket[b] = start;  // becomes the bucket's write cursor
  }
  __syncthreads();
  for (int r = tid; r < p.batch; r += 1024) {
    const int4 info = p.req_info[r];
    const int n = info.z > 0 ? info.z : 0;
    for (int c = 0; c < info.y; ++c) {
      const int len = max(0, min(chunk_len, n - c * chunk_len));
      const int pos = atomicAdd(&s_bucket[min((len + kN - 1) / kN, kBuckets - 1)], 1);
      if (pos < p.max_chunks) p.chunk_list[pos] = make_int2(r, c);
    }
    // the merge kernel's list: requests cut into chunks, in any order
    if (info.y > 1 && info.z >= 0) p.split_list[atomicAdd(&s_nsplit, 1)] = r;
  }
  __syncthreads();
  if (tid == 0) {
    p.hdr[0] = min(total, p.max_chunks);
    p.hdr[1] = chunk_len;
    p.hdr[2] = s_nsplit;
  }
}

// ----------------------------------------------------------------- decode
__global__ void __launch_bounds__(kThreadsMla, 1)
    mla_decode_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_c,
                      const MlaParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem;
  uint8_t* sC = smem + kOffC;
  uint8_t* sV = smem + kOffV;
  Bars* bars = reinterpret_cast<Bars*>(smem + kOffBar);
  volatile int* abort = &bars->abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int pair = blockIdx.x >> 1, half = blockIdx.x & 1, pairs = gridDim.x >> 1;

  if (threadIdx.x == 0) {
    mbar_init(&bars->q_full, 1);
    mbar_init(&bars->q_empty, kSIssuers);
    for (int r = 0; r < kSIssuers; ++r)
      for (int i = 0; i < kRing; ++i) {
        mbar_init(&bars->c_full[r][i], 1);
        mbar_init(&bars->c_empty[r][i], 1);
      }
    mbar_init(&bars->v_full, 1);
    mbar_init(&bars->v_empty, 1);
    for (int i = 0; i < kSB; ++i) {
      mbar_init(&bars->s_full[i], kSIssuers);
      mbar_init(&bars->p_full[i], 4);
      mbar_init(&bars->pv_done[i], 1);
    }
    mbar_init(&bars->o_free, 4);
    mbar_init(&bars->drain, kSIssuers + 1);  // one commit from each MMA-issuing warp
    bars->abort = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_map(&tm_q);
    tma_prefetch_map(&tm_c);
  }
  if (warp == 1) {
    tmem_alloc(&bars->tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_slot;
  pdl_wait_primary();  // the plan kernel's list and chunk length
  pdl_launch_dependents();
  const int n_items = (blockIdx.x < 2 * pairs) ? p.hdr[0] : 0;  // an odd last CTA has no partner
  const int pb = p.page_size < kN ? p.page_size : kN;  // tokens per box
  const int nb = kN / pb;                              // boxes per column chunk

  if (warp == 0 || warp == kWarpV) {
    // ----------------------------------------------------------- producers
    // warp 0: the request's Q tile, then every tile's nine column chunks of
    // 64 tokens x 64 values, in order, through the two issuers' rings (one
    // consumer per ring); warp 8: this half's four value chunks of every
    // tile, two at a time, into the value slot, once the previous product
    // O += P C_h has read it (the second read of those rows comes from L2)
    const bool is_v = warp == kWarpV;
    uint32_t item_ctr = 0, tile_ctr = 0;
    bool ok = true;
    for (int k = 0; ok; ++k, ++item_ctr) {
      const int idx = pair_item(k, pair, pairs);
      if (idx >= n_items) break;
      const MItem I = mla_item(p, idx);
      if (!is_v) {
        // the previous item's S products have all completed before Q is replaced
        ok = warp_mbar_wait(&bars->q_empty, (item_ctr & 1u) ^ 1u, abort, p.status);
        if (!ok) break;
        if (lane == 0) mbar_arrive_expect_tx(&bars->q_full, kQBytes);
        __syncwarp();
        if (lane < kWC) tma_load_3d(sQ + lane * kQChunk, &tm_q, lane * 64, 0, I.r, &bars->q_full);
      }
      for (int j = 0; j < I.ntiles && ok; ++j, ++tile_ctr) {
        // page of box `sub` (lanes below nb), read before any slot wait
        int pid = p.num_pages, soff = 0;
        const int sub = lane % nb;
        {
          const int tok = I.t0 + j * kN + sub * pb;
          const int pidx = tok / p.page_size;
          soff = tok % p.page_size;
          if (pidx < I.need) {
            pid = __ldg(p.page_indices + I.pbase + pidx);
            if (pid < 0 || pid >= p.num_pages) {
              if (lane < nb) report(p.status, PD_DEV_BAD_PAGE_TABLE);
              pid = p.num_pages;  // out of range: the box arrives as zeros
            }
          }
        }
        if (is_v) {
          for (int ps = 0; ps < kVPass && ok; ++ps) {
            const uint32_t vseq = tile_ctr * kVPass + ps;
            ok = warp_mbar_wait(&bars->v_empty, (vseq & 1u) ^ 1u, abort, p.status);
            if (!ok) break;
            if (lane == 0) mbar_arrive_expect_tx(&bars->v_full, kVBytes);
            __syncwarp();
            if (lane < kVSlotChunks * nb) {
              const int ch = lane / nb;
              tma_load_4d(sV + ch * kCChunk + sub * pb * 128, &tm_c, (half * kVChunks + ps * kVSlotChunks + ch) * 64,
                          soff, 0, pid, &bars->v_full);
            }
          }
        } else {
          for (int c = 0; c < kWC && ok; ++c) {
            const int r = c % kSIssuers;
            const uint32_t seq = ring_seq(tile_ctr, c), slot = seq % kRing;
            ok = warp_mbar_wait(&bars->c_empty[r][slot], ((seq / kRing) & 1u) ^ 1u, abort, p.status);
            if (!ok) break;
            if (lane == 0) mbar_arrive_expect_tx(&bars->c_full[r][slot], kCChunk);
            __syncwarp();
            if (lane < nb)
              tma_load_4d(sC + (r * kRing + slot) * kCChunk + sub * pb * 128, &tm_c, c * 64, soff, 0, pid,
                          &bars->c_full[r][slot]);
          }
        }
      }
    }
  } else if (s_issuer(warp) >= 0) {
    // ------------------ partial S = Q C^T over this warp's column chunks
    constexpr uint32_t idesc_s = idesc_bf16_f32(kRows, kN, 0);
    const uint32_t sQa = smem_u32(sQ), sCa = smem_u32(sC);
    const int part = s_issuer(warp);
    uint32_t item_ctr = 0, tile_ctr = 0;
    bool ok = true;
    for (int k = 0; ok; ++k, ++item_ctr) {
      const int idx = pair_item(k, pair, pairs);
      if (idx >= n_items) break;
      const MItem I = mla_item(p, idx);
      ok = warp_mbar_wait(&bars->q_full, item_ctr & 1u, abort, p.status);
      if (!ok) break;
      tc_fence_after();
      const uint64_t dq = sw128_desc(sQa, 16, 1024);
      for (int j = 0; j < I.ntiles && ok; ++j, ++tile_ctr) {
        const int sb = tile_ctr % kSB;
        // S buffer sb is free once the P C product of two tiles back is done
        if (tile_ctr >= (uint32_t)kSB) {
          ok = warp_mbar_wait(&bars->pv_done[sb], ((tile_ctr - kSB) / kSB) & 1u, abort, p.status);
          if (!ok) break;
        }
        for (int c = part; c < kWC; c += kSIssuers) {
          const uint32_t seq = ring_seq(tile_ctr, c), slot = seq % kRing;
          ok = warp_mbar_wait(&bars->c_full[part][slot], (seq / kRing) & 1u, abort, p.status);
          if (!ok) break;
          tc_fence_after();
          if (lane == 0) {
            const uint64_t dc = sw128_desc(sCa + (part * kRing + slot) * kCChunk, 16, 1024);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              tc_mma_f16(tmem + col_s(sb, part), desc_advance(dq, c * kQChunk + kk * 32), desc_advance(dc, kk * 32),
                         idesc_s, (c > part || kk > 0) ? 1u : 0u);
            tc_commit(&bars->c_empty[part][slot]);
          }
          __syncwarp();
        }
        if (!ok) break;
        if (lane == 0) {
          tc_commit(&bars->s_full[sb]);
          if (j == I.ntiles - 1) tc_commit(&bars->q_empty);
        }
        __syncwarp();
      }
      if (!ok) break;
      if (I.ntiles == 0 && lane == 0) mbar_arrive(&bars->q_empty);
      __syncwarp();
    }
    if (lane == 0) {
      tc_commit(&bars->drain);
      const uint64_t t0 = globaltimer_ns();
      while (!mbar_try_wait(&bars->drain, 0) && globaltimer_ns() - t0 < kWaitLimitNs) {
      }
    }
    __syncwarp();
  } else if (warp == kWarpPV) {
    // ---------------------------------------------------------- O += P C_h
    constexpr uint32_t idesc_pv = idesc_bf16_f32(kRows, kVSlotChunks * 64, 1);
    const uint32_t sVa = smem_u32(sV);
    uint32_t item_ctr = 0, tile_ctr = 0;
    bool ok = true;
    for (int k = 0; ok; ++k, ++item_ctr) {
      const int idx = pair_item(k, pair, pairs);
      if (idx >= n_items) break;
      const MItem I = mla_item(p, idx);
      // the previous item's epilogue has read O out of TMEM
      if (item_ctr > 0) {
        ok = warp_mbar_wait(&bars->o_free, (item_ctr - 1) & 1u, abort, p.status);
        if (!ok) break;
      }
      for (int j = 0; j < I.ntiles; ++j, ++tile_ctr) {
        const int sb = tile_ctr % kSB;
        ok = warp_mbar_wait(&bars->p_full[sb], (tile_ctr / kSB) & 1u, abort, p.status);
        if (!ok) break;
        for (int ps = 0; ps < kVPass; ++ps) {
          const uint32_t vseq = tile_ctr * kVPass + ps;
          ok = warp_mbar_wait(&bars->v_full, vseq & 1u, abort, p.status);
          if (!ok) break;
          const int valid = I.len - j * kN;
          if (valid < kN) {
            for (int i = lane; i < (kN - valid) * 8 * kVSlotChunks; i += 32) {
              const int ch = i / ((kN - valid) * 8), rem = i % ((kN - valid) * 8);
              const int rr = valid + rem / 8, c16 = rem % 8;
              asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};" ::"r"(sVa + ch * kCChunk + rr * 128 + c16 * 16),
                           "r"(0)
                           : "memory");
            }
            fence_proxy_async_smem();
            __syncwarp();
          }
          tc_fence_after();
          if (lane == 0) {
            const uint64_t dv = sw128_desc(sVa, kCChunk, 1024);
            const uint32_t pa = tmem + col_s(sb);
            const uint32_t od = tmem + kColO + ps * kVSlotChunks * 64;
#pragma unroll
            for (int kk = 0; kk < kN / 16; ++kk) {
              tc_mma_f16_tmem_a(od, pa + 16 * kk, desc_advance(dv, kk * 2048), idesc_pv, (j > 0 || kk > 0) ? 1u : 0u);
              tc_mma_f16_tmem_a(od, pa + 16 * kk + 8, desc_advance(dv, kk * 2048), idesc_pv, 1u);
            }
            if (ps == kVPass - 1) tc_commit(&bars->pv_done[sb]);
            tc_commit(&bars->v_empty);
          }
          __syncwarp();
        }
        if (!ok) break;
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
    const int wq = warp & 3;
    const int row = wq * 32 + lane;  // query head
    const uint32_t t_lane = tmem + ((uint32_t)(wq * 32) << 16);
    const uint32_t o_addr = t_lane + kColO;
    uint32_t item_ctr = 0, tile_ctr = 0;
    bool ok = true;
    for (int k = 0; ok; ++k, ++item_ctr) {
      const int idx = pair_item(k, pair, pairs);
      if (idx >= n_items) break;
      const MItem I = mla_item(p, idx);
      float m = -INFINITY, l = 0.f;
      for (int j = 0; j < I.ntiles; ++j, ++tile_ctr) {
        const int sb = tile_ctr % kSB;
        ok = warp_mbar_wait(&bars->s_full[sb], (tile_ctr / kSB) & 1u, abort, p.status);
        if (!ok) break;
        tc_fence_after();
        const int ncol = min(kN, I.len - j * kN);
        const uint32_t s_addr = t_lane + col_s(sb);
        // S (with two issuers: the sum of the partial products over the even
        // and the odd column chunks)
        uint32_t v[kN];
        tmem_ld32(s_addr, *reinterpret_cast<uint32_t(*)[32]>(v));
        tmem_ld32(s_addr + 32, *reinterpret_cast<uint32_t(*)[32]>(v + 32));
        if (kSIssuers > 1) {
          uint32_t v1[kN];
          tmem_ld32(t_lane + col_s(sb, 1), *reinterpret_cast<uint32_t(*)[32]>(v1));
          tmem_ld32(t_lane + col_s(sb, 1) + 32, *reinterpret_cast<uint32_t(*)[32]>(v1 + 32));
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < kN; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) + __uint_as_float(v1[e]));
        } else {
          tmem_wait_ld();
        }
        if (ncol < kN) {
#pragma unroll
          for (int e = 0; e < kN; ++e) v[e] = e < ncol ? v[e] : 0xff800000u;  // -inf: weight 0
        }
        float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
        for (int e = 0; e < kN; e += 2)
          mx[(e / 2) & 3] = fmax3(mx[(e / 2) & 3], __uint_as_float(v[e]), __uint_as_float(v[e + 1]));
        const float mt = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
        float m_new = m;
        bool rescale = false;
        if (mt > -INFINITY) {
          const float ms = mt * p.scale_log2;
          if (m == -INFINITY) {
            m_new = ms;
          } else if (ms > m + kRescaleThreshold) {
            m_new = ms;
            rescale = true;
          }
        }
        // warp-collective rescale of this warp's O rows once the previous P C
        // product has completed (its barrier cannot pass this phase before this
        // tile's P is published)
        if (__any_sync(0xffffffffu, rescale)) {
          const uint32_t prev = tile_ctr - 1;
          ok = warp_mbar_wait(&bars->pv_done[prev % kSB], (prev / kSB) & 1u, abort, p.status);
          if (!ok) break;
          tc_fence_after();
          const float alpha = rescale ? exp2f(m - m_new) : 1.0f;
          l *= alpha;
#pragma unroll 1
          for (int c = 0; c < kHalfV / 32; ++c) {
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
        const float2 sc2 = make_float2(p.scale_log2, p.scale_log2), nm2 = make_float2(-m, -m);
        mla_write_p(v, s_addr, sc2, nm2, l);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->p_full[sb]);
      }
      if (!ok) break;
      // epilogue: O / l for this half's 256 columns, once the last P C is done
      if (I.ntiles > 0) {
        const uint32_t last = tile_ctr - 1;
        ok = warp_mbar_wait(&bars->pv_done[last % kSB], (last / kSB) & 1u, abort, p.status);
        if (!ok) break;
        tc_fence_after();
      }
      const bool store = I.valid && row < p.hq;
      const bool final_out = I.nch == 1;
      const float inv_l = l > 0.f ? 1.0f / l : 0.f;
      const float lse2 = (I.ntiles > 0 && l > 0.f) ? m + log2f(l) : -INFINITY;
#pragma unroll 1
      for (int c = 0; c < kHalfV / 32; ++c) {
        uint32_t o[32];
        if (I.ntiles > 0) {
          tmem_ld32(o_addr + c * 32, o);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = 0u;
        }
        if (!store) continue;
        const int col = half * kHalfV + c * 32;
        if (!final_out) {
          float4* dst = reinterpret_cast<float4*>(p.part_o + ((int64_t)(I.first + I.c) * p.hq + row) * kDc + col);
#pragma unroll
          for (int e = 0; e < 8; ++e)
            dst[e] = make_float4(__uint_as_float(o[4 * e]) * inv_l, __uint_as_float(o[4 * e + 1]) * inv_l,
                                 __uint_as_float(o[4 * e + 2]) * inv_l, __uint_as_float(o[4 * e + 3]) * inv_l);
        } else if (p.o_dtype == PD_BF16) {
          uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.o) + ((int64_t)I.r * p.hq + row) * kDc + col);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            uint4 u;
            u.x = pack_bf16x2(__uint_as_float(o[8 * e + 0]) * inv_l, __uint_as_float(o[8 * e + 1]) * inv_l);
            u.y = pack_bf16x2(__uint_as_float(o[8 * e + 2]) * inv_l, __uint_as_float(o[8 * e + 3]) * inv_l);
            u.z = pack_bf16x2(__uint_as_float(o[8 * e + 4]) * inv_l, __uint_as_float(o[8 * e + 5]) * inv_l);
            u.w = pack_bf16x2(__uint_as_float(o[8 * e + 6]) * inv_l, __uint_as_float(o[8 * e + 7]) * inv_l);
            dst[e] = u;
          }
        } else {
          float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.o) + ((int64_t)I.r * p.hq + row) * kDc + col);
#pragma unroll
          for (int e = 0; e < 8; ++e)
            dst[e] = make_float4(__uint_as_float(o[4 * e]) * inv_l, __uint_as_float(o[4 * e + 1]) * inv_l,
                                 __uint_as_float(o[4 * e + 2]) * inv_l, __uint_as_float(o[4 * e + 3]) * inv_l);
        }
      }
      if (store && half == 0) {
        if (!final_out) p.part_lse[(int64_t)(I.first + I.c) * p.hq + row] = lse2;
        else if (p.lse != nullptr) p.lse[(int64_t)I.r * p.hq + row] = lse2 * kLn2;
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->o_free);
    }
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

// ------------------------------------------------------------------ merge
// Requests split into chunks: lse2 = log2 sum_c 2^lse2_c, o = sum_c 2^(lse2_c -
// lse2) o_c. A unit is (request of the plan's split list, pair of heads), a
// thread owns 4 columns; a small grid strides over the units, so that a batch
// with few split requests does not launch a CTA per request and head pair.
__global__ void __launch_bounds__(256) mla_merge_kernel(const MlaParams p) {
  pdl_wait_primary();
  const int hpairs = (p.hq + 1) / 2;
  const int units = p.hdr[2] * hpairs;
  const int col = (threadIdx.x & 127) * 4;
  for (int u = blockIdx.x; u < units; u += gridDim.x) {
    const int r = p.split_list[u / hpairs];
    const int h = (u % hpairs) * 2 + (threadIdx.x >> 7);
    const int4 info = p.req_info[r];
    if (info.y <= 1 || info.z < 0 || h >= p.hq) continue;
    const float* lse_c = p.part_lse + (int64_t)info.x * p.hq + h;
    float mx = -INFINITY;
    for (int c = 0; c < info.y; ++c) mx = fmaxf(mx, lse_c[(int64_t)c * p.hq]);
    float s = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    if (mx > -INFINITY) {
      for (int c = 0; c < info.y; ++c) {
        const float wgt = exp2f(lse_c[(int64_t)c * p.hq] - mx);
        const float4 v = *reinterpret_cast<const float4*>(p.part_o + ((int64_t)(info.x + c) * p.hq + h) * kDc + col);
        s += wgt;
        acc.x += wgt * v.x;
        acc.y += wgt * v.y;
        acc.z += wgt * v.z;
        acc.w += wgt * v.w;
      }
    }
    const float inv = s > 0.f ? 1.0f / s : 0.f;
    const int64_t o_off = ((int64_t)r * p.hq + h) * kDc + col;
    if (p.o_dtype == PD_BF16) {
      uint2 packed;
      packed.x = pack_bf16x2(acc.x * inv, acc.y * inv);
      packed.y = pack_bf16x2(acc.z * inv, acc.w * inv);
      *reinterpret_cast<uint2*>(static_cast<uint16_t*>(p.o) + o_off) = packed;
    } else {
      *reinterpret_cast<float4*>(static_cast<float*>(p.o) + o_off) =
          make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
    }
    if (col == 0 && p.lse != nullptr) p.lse[(int64_t)r * p.hq + h] = s > 0.f ? (mx + log2f(s)) * kLn2 : -INFINITY;
  }
}

// ------------------------------------------------------------------- host
int mla_supported(int32_t d_c, int32_t d_r, int32_t dtype, int32_t hq, int32_t page_size) {
  if (d_c != kDc || d_r != kDr || dtype != PD_BF16) return PD_ERR_UNSUPPORTED;
  if (hq < 1 || hq > kRows) return PD_ERR_UNSUPPORTED;
  // 64-token tiles of whole boxes: at most four boxes per column chunk, eight per value-slot fill
  if (page_size < 16 || page_size > 256 || (page_size & (page_size - 1)) != 0) return PD_ERR_UNSUPPORTED;
  return PD_OK;
}

int mla_pairs() { return device_sm_count() / 2; }

MlaLayout mla_layout(int32_t batch, int32_t hq) {
  MlaLayout L{};
  L.max_chunks = batch + 2 * mla_pairs();
  size_t off = 0;
  L.hdr = off;
  off = align_up(off + 64 * sizeof(int32_t), 256);
  L.req_info = off;
  off = align_up(off + sizeof(int4) * (size_t)batch, 256);
  L.chunk_list = off;
  off = align_up(off + sizeof(int2) * (size_t)L.max_chunks, 256);
  L.split_list = off;
  off = align_up(off + sizeof(int32_t) * (size_t)(batch > 0 ? batch : 1), 256);
  L.part_lse = off;
  off = align_up(off + sizeof(float) * (size_t)L.max_chunks * hq, 256);
  L.part_o = off;
  off = align_up(off + sizeof(float) * (size_t)L.max_chunks * hq * kDc, 256);
  L.total = off;
  return L;
}

int launch_mla(MlaParams& p, const void* q, const void* kv_pool, cudaStream_t stream) {
  CUtensorMap tq, tc;
  const int pb = p.page_size < kN ? p.page_size : kN;
  // q [batch][hq][576]: one box = 64 values of 128 heads (heads past hq read as zeros)
  if (!make_rows_map(&tq, q, PD_BF16, p.batch, p.hq, kW, 64, 1, true, kRows) ||
      !make_pool_map(&tc, kv_pool, PD_BF16, p.num_pages, 1, p.page_size, kW, 64, pb, true))
    return PD_ERR_CUDA;
  // per device: whether the kernel's shared-memory attribute is set there
  // (callers may run on several threads)
  static std::atomic<bool> configured[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PD_ERR_CUDA;
  const bool cached = dev >= 0 && dev < 64;
  if (!cached || !configured[dev].load(std::memory_order_acquire)) {
    if (cudaFuncSetAttribute(mla_decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kMlaSmem) !=
        cudaSuccess)
      return PD_ERR_CUDA;
    if (cached) configured[dev].store(true, std::memory_order_release);
  }
  last_kernel() = "mla_decode_kernel";
  mla_plan_kernel<<<1, 1024, 0, stream>>>(p);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  const bool pdl = profile_events().start == nullptr;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((unsigned)(2 * p.pairs));
  cfg.blockDim = dim3(kThreadsMla);
  cfg.dynamicSmemBytes = kMlaSmem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  profile_begin(stream);
  cudaError_t e = cudaLaunchKernelEx(&cfg, mla_decode_kernel, tq, tc, p);
  profile_end(stream);
  if (e != cudaSuccess) return PD_ERR_CUDA;
  cudaLaunchConfig_t mcfg{};
  // two CTAs per SM, or one per unit if the batch has fewer
  const int64_t merge_units = (int64_t)p.batch * ((p.hq + 1) / 2);
  int64_t merge_grid = 2 * (int64_t)device_sm_count();
  if (merge_grid > merge_units) merge_grid = merge_units;
  if (merge_grid < 1) merge_grid = 1;
  mcfg.gridDim = dim3((unsigned)merge_grid);
  mcfg.blockDim = dim3(256);
  mcfg.stream = stream;
  mcfg.attrs = attr;
  mcfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&mcfg, mla_merge_kernel, p);
  return e == cudaSuccess ? PD_OK : PD_ERR_CUDA;
}

}  // namespace pd
