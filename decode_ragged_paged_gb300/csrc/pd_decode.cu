// pd_decode.cu -- split-KV decode attention over an HND paged KV cache.
//
// Perplexity, "Disaggregated prefill and decode" (2025), section "Prefill vs
// Decode performance": decode requests carry one token (qo_len = 1), attention
// cost grows with kv_len, decode is memory bound, and attention can be
// parallelised over requests and over kv_len (the post's "Split-K" argument,
// applied here to the KV axis). Section "Qwen3-Coder": grouped-query attention,
// so one KV head serves several query heads.
//
// Three launches on the caller's stream, each a programmatic dependent of the
// one before:
//   1. plan    one CTA validates lengths and tables, cuts every request's KV
//              into equal chunks and writes the work list, longest chunks
//              first, into the workspace;
//   2. decode  persistent CTAs; per work item (request, group of query heads
//              sharing one KV head, KV chunk) a producer warp streams the
//              chunk's K then V page slices (contiguous runs in the HND layout)
//              into a shared-memory ring with bulk async copies (TMA engine),
//              and the consumer warps compute the scores, the chunk softmax and
//              the weighted value sum in fp32;
//   3. merge   chunks of one request are combined by their log-sum-exp.
#include <atomic>
#include <math.h>

#include "pd_common.cuh"
#include "pd_internal.h"

namespace pd {

namespace {

// Tuning knobs (compile-time). Measured on GB300 for the 128-request GQA
// decode: a TMA bulk copy stream is limited per issuing warp (a warp keeps only
// a few copies in flight), so bandwidth comes from many small CTAs, each with
// its own producer warp: 2 consumer warps, 32-token stages, a 32 KiB ring and
// 5 CTAs per SM.
#ifndef PD_DECODE_STAGE_TOKENS
#define PD_DECODE_STAGE_TOKENS 32
#endif
#ifndef PD_DECODE_WARPS
#define PD_DECODE_WARPS 2
#endif
#ifndef PD_DECODE_RING_KB
#define PD_DECODE_RING_KB 32
#endif
#ifndef PD_DECODE_MIN_BLOCKS
#define PD_DECODE_MIN_BLOCKS 5
#endif
// Producer lanes: lane j of the producer warp issues the stages whose running
// index is j modulo this count.
#ifndef PD_DECODE_PRODUCER_LANES
#define PD_DECODE_PRODUCER_LANES 1
#endif
constexpr int kTS = PD_DECODE_STAGE_TOKENS;  // tokens per ring stage
constexpr int kTPL = kTS / 4;                 // tokens per lane per stage (4 token groups per warp)
constexpr int kNC = PD_DECODE_WARPS;          // consumer warps
constexpr int kPL = PD_DECODE_PRODUCER_LANES;  // issuing lanes of the producer warp
constexpr int kThreads = (kNC + 1) * 32;
static_assert(kPL >= 1 && kPL <= 32, "producer lanes");
#ifndef PD_DECODE_MAX_CHUNK
#define PD_DECODE_MAX_CHUNK 512
#endif
constexpr int kMaxChunk = PD_DECODE_MAX_CHUNK;  // longest chunk (tokens) a work item covers
constexpr int kRingBytes = PD_DECODE_RING_KB * 1024;
static_assert(kTS % 4 == 0 && kMaxChunk % kTS == 0, "stage size");
constexpr unsigned kFull = 0xffffffffu;

template <int ES, int D>
struct Geo {
  static constexpr int kRowBytes = D * ES;            // one token of one head
  static constexpr int kVecPerRow = kRowBytes / 16;   // 16-byte vectors per row
  static constexpr int kVecPerLane = kVecPerRow / 8;  // lane dg takes vectors dg, dg+8, ...
  static constexpr int kEpv = 16 / ES;                // elements per vector
  static constexpr int kE = kVecPerLane * kEpv;       // elements per lane = D / 8
  static constexpr int kStageBytes = kTS * kRowBytes;
  // as many stages as the ring holds (at most 32), rounded down to a multiple of
  // the consumer warps
  static constexpr int kStagesRaw = kRingBytes / kStageBytes < 32 ? kRingBytes / kStageBytes : 32;
  static constexpr int kStages = kStagesRaw / kNC * kNC;
  static_assert(kVecPerLane >= 1, "row too short");
  // Within a K or V phase stage s belongs to consumer warp s % kNC and uses ring
  // slot (running index) % kStages. With kStages a multiple of kNC every use of
  // a slot inside one phase belongs to the same warp, so a warp never waits on a
  // slot whose previous use (another warp's stage) is still in flight: an
  // mbarrier parity wait cannot tell a phase two steps back from the pending
  // one. Phases and items are separated by all-consumer syncs.
  static_assert(kStages >= kNC && kStages % kNC == 0, "ring stages must be a multiple of the consumer warps");
};

template <int GS, int D>
struct DecodeSmem {
  static constexpr size_t kScores = sizeof(float) * kMaxChunk * GS;
  static constexpr size_t kOpart = sizeof(float) * kNC * GS * D;
  static constexpr size_t kStats = sizeof(float) * 2 * GS;
};

template <int ES, int D, int GS>
constexpr size_t decode_smem_bytes() {
  using G = Geo<ES, D>;
  return (size_t)G::kStages * G::kStageBytes + DecodeSmem<GS, D>::kScores + DecodeSmem<GS, D>::kOpart +
         DecodeSmem<GS, D>::kStats + 8 * (2 * G::kStages + 2) + 16;
}

// element e of lane dg sits at dimension (dg + 8 * (e / Epv)) * Epv + e % Epv
template <int ES, int D>
__device__ __forceinline__ void load_lane_row(const uint8_t* row, int dg, float (&f)[Geo<ES, D>::kE]) {
  using G = Geo<ES, D>;
  const uint4* v = reinterpret_cast<const uint4*>(row);
#pragma unroll
  for (int vi = 0; vi < G::kVecPerLane; ++vi) {
    const uint4 x = v[dg + 8 * vi];
    if constexpr (ES == 2) {
      f[vi * 8 + 0] = bf16_lo(x.x);
      f[vi * 8 + 1] = bf16_hi(x.x);
      f[vi * 8 + 2] = bf16_lo(x.y);
      f[vi * 8 + 3] = bf16_hi(x.y);
      f[vi * 8 + 4] = bf16_lo(x.z);
      f[vi * 8 + 5] = bf16_hi(x.z);
      f[vi * 8 + 6] = bf16_lo(x.w);
      f[vi * 8 + 7] = bf16_hi(x.w);
    } else {
      f[vi * 4 + 0] = __uint_as_float(x.x);
      f[vi * 4 + 1] = __uint_as_float(x.y);
      f[vi * 4 + 2] = __uint_as_float(x.z);
      f[vi * 4 + 3] = __uint_as_float(x.w);
    }
  }
}

template <int ES, int D>
__device__ __forceinline__ int lane_dim(int dg, int e) {
  using G = Geo<ES, D>;
  return (dg + 8 * (e / G::kEpv)) * G::kEpv + e % G::kEpv;
}

// Transposed butterfly reduction over the 8 lanes of a group (lane bits 0..2):
// at each step a lane keeps half of its values and receives the partner's
// partial sums of that half, so N values are reduced with N - 1 shuffles.
// Afterwards lane dg holds the full sums of indices [dg*N/8, (dg+1)*N/8) for
// N >= 8, or of index dg >> (3 - log2 N) for N < 8.
template <int N, int M>
__device__ __forceinline__ void xreduce(float* v, int lane) {
  if constexpr (N > 1) {
    constexpr int H = N / 2;
    const bool up = (lane & M) != 0;
#pragma unroll
    for (int i = 0; i < H; ++i) {
      const float send = up ? v[i] : v[i + H];
      const float keep = up ? v[i + H] : v[i];
      v[i] = keep + __shfl_xor_sync(kFull, send, M);
    }
  } else {
    v[0] += __shfl_xor_sync(kFull, v[0], M);
  }
  if constexpr (M > 1) xreduce<(N > 1 ? N / 2 : 1), M / 2>(v, lane);
}

struct Item {
  int r, h0, g, t_begin, t_end, chunk, q_row, first_chunk, n_chunks;
};

__device__ __forceinline__ Item decode_item(const DecodeParams& p, int it) {
  Item I;
  const int rc = it / p.items_per_chunk;
  const int hs = it - rc * p.items_per_chunk;
  const int2 rcv = p.rc_list[rc];
  const int4 info = p.req_info[rcv.x];
  I.r = rcv.x;
  I.chunk = rcv.y;
  I.h0 = hs * p.heads_per_item;
  I.g = I.h0 / p.group;
  I.first_chunk = info.x;
  I.n_chunks = info.y;
  I.t_begin = rcv.y * info.z;
  I.t_end = min(I.t_begin + info.z, p.kv_len[rcv.x]);
  I.q_row = info.w;
  return I;
}

// Item of CTA b in hand-out round k: rounds alternate direction over the
// grid, so with items sorted longest first each CTA's total stays close to the
// mean.
#ifndef PD_DECODE_SERPENTINE
#define PD_DECODE_SERPENTINE 1
#endif
__device__ __forceinline__ int serpentine_item(int k, int b, int grid) {
  return k * grid + ((PD_DECODE_SERPENTINE && (k & 1)) ? grid - 1 - b : b);
}

__device__ __forceinline__ bool consumer_sync(uint64_t* bar, uint32_t& phase, int lane,
                                              volatile int* abort, int32_t* status) {
  __syncwarp();
  if (lane == 0) mbar_arrive(bar);
  const bool ok = warp_mbar_wait(bar, phase & 1u, abort, status);
  ++phase;
  return ok;
}

}  // namespace

// ------------------------------------------------------------------- plan
// One CTA. Per request: validate, choose the chunk length (equal chunks of at
// most chunk_target tokens, multiples of the stage size), scan the chunk
// counts (each chunk's slot for its partial result) and give requests without
// keys their final o = 0, lse = -inf. Then list the
// (request, chunk) pairs longest first (counting sort on the stage count), so
// that the decode kernel's serpentine hand-out balances the CTAs.
#ifndef PD_DECODE_SORT
#define PD_DECODE_SORT 1
#endif
constexpr int kLenBuckets = kMaxChunk / kTS;  // chunk lengths in stages: 1 .. kLenBuckets

__global__ void __launch_bounds__(1024) decode_plan_kernel(const DecodeParams p) {
  pdl_launch_dependents();
  __shared__ int warp_sums[32];
  __shared__ int carry;
  __shared__ int bucket_cnt[kLenBuckets + 1];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) carry = 0;
  if (tid <= kLenBuckets) bucket_cnt[tid] = 0;
  __syncthreads();
  for (int base = 0; base < p.batch; base += blockDim.x) {
    const int r = base + tid;
    int n_c = 0, clen = 0, row = -1;
    if (r < p.batch) {
      int code = 0;
      const int n = p.kv_len[r];
      if (n < 0 || n > p.max_kv_len) code = PD_DEV_BAD_LENGTH;
      if (p.qo_indptr != nullptr) {
        const int a = p.qo_indptr[r], b = p.qo_indptr[r + 1];
        if (a < 0 || b < a || b > p.total_qo) code = PD_DEV_BAD_INDPTR;
        else if (b - a != 1) code = PD_DEV_NOT_DECODE;
        row = a;
      } else {
        row = r;
        if (r >= p.total_qo) code = PD_DEV_BAD_INDPTR;
      }
      const int pa = p.page_indptr[r], pb = p.page_indptr[r + 1];
      if (code == 0 && (pa < 0 || pb < pa)) code = PD_DEV_BAD_INDPTR;
      if (code == 0 && (long long)(pb - pa) * p.page_size < n) code = PD_DEV_BAD_PAGE_TABLE;
      if (code != 0) {
        report(p.status, code);
        row = -1;
      } else if (n > 0) {
        n_c = (n + p.chunk_target - 1) / p.chunk_target;
        clen = (n + n_c - 1) / n_c;
        clen = (clen + kTS - 1) / kTS * kTS;
        n_c = (n + clen - 1) / clen;
        const int last = n - (n_c - 1) * clen;
        const int full = last == clen ? n_c : n_c - 1;
        if (full > 0) atomicAdd(&bucket_cnt[clen / kTS], full);
        if (last != clen) atomicAdd(&bucket_cnt[(last + kTS - 1) / kTS], 1);
      }
    }
    // block-wide exclusive scan of n_c
    int x = n_c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(kFull, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) warp_sums[warp] = x;
    __syncthreads();
    if (warp == 0) {
      int w = lane < (int)(blockDim.x >> 5) ? warp_sums[lane] : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(kFull, w, o);
        if (lane >= o) w += y;
      }
      warp_sums[lane] = w;  // inclusive
    }
    __syncthreads();
    const int excl = carry + (warp > 0 ? warp_sums[warp - 1] : 0) + x - n_c;
    if (r < p.batch) p.req_info[r] = make_int4(excl, n_c, clen, row);
    __syncthreads();
    if (tid == 0) carry += warp_sums[(blockDim.x >> 5) - 1];
    __syncthreads();
  }
  // bucket starts, longest chunks first (bucket_cnt becomes a cursor)
  if (tid == 0) {
    int pos = 0;
    for (int b = kLenBuckets; b >= 1; --b) {
      const int c = bucket_cnt[b];
      bucket_cnt[b] = pos;
      pos += c;
    }
  }
  __syncthreads();
  for (int r = tid; r < p.batch; r += blockDim.x) {
    const int4 info = p.req_info[r];
    if (info.w < 0) continue;
    if (info.y == 0) {
      // no keys: final output now (the decode kernel never sees this request)
      for (int k = 0; k < p.hq * p.head_dim; ++k) {
        const int64_t off = (int64_t)info.w * p.hq * p.head_dim + k;
        if (p.o_dtype == PD_BF16)
          static_cast<uint16_t*>(p.o)[off] = 0;
        else
          static_cast<float*>(p.o)[off] = 0.f;
      }
      if (p.lse != nullptr)
        for (int h = 0; h < p.hq; ++h) p.lse[(int64_t)info.w * p.hq + h] = -INFINITY;
      continue;
    }
    const int n = p.kv_len[r], clen = info.z, n_c = info.y;
    if (!PD_DECODE_SORT) {
      for (int c = 0; c < n_c; ++c) p.rc_list[info.x + c] = make_int2(r, c);
      continue;
    }
    const int last = n - (n_c - 1) * clen;
    const int full = last == clen ? n_c : n_c - 1;
    if (full > 0) {
      const int q = atomicAdd(&bucket_cnt[clen / kTS], full);
      for (int c = 0; c < full; ++c) p.rc_list[q + c] = make_int2(r, c);
    }
    if (last != clen) p.rc_list[atomicAdd(&bucket_cnt[(last + kTS - 1) / kTS], 1)] = make_int2(r, n_c - 1);
  }
  if (tid == 0) {
    p.hdr[1] = carry;
    p.hdr[0] = carry * p.items_per_chunk;
  }
}

// ----------------------------------------------------------------- decode
template <int ES, int D, int GS>
__global__ void __launch_bounds__(kThreads, PD_DECODE_MIN_BLOCKS) decode_kernel(const DecodeParams p) {
  using G = Geo<ES, D>;
  constexpr int E = G::kE;
  constexpr int NS = G::kStages;
  constexpr int SB = G::kStageBytes;
  constexpr int RB = G::kRowBytes;

  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* ring = smem;
  float* s_scores = reinterpret_cast<float*>(smem + (size_t)NS * SB);   // [kMaxChunk][GS]
  float* s_opart = s_scores + kMaxChunk * GS;                           // [kNC][GS][D]
  float* s_m = s_opart + kNC * GS * D;                                  // [GS]
  float* s_l = s_m + GS;                                                // [GS]
  uint64_t* full = reinterpret_cast<uint64_t*>(s_l + GS + ((GS & 1) ? 0 : 0));
  full = reinterpret_cast<uint64_t*>((reinterpret_cast<uintptr_t>(full) + 7) & ~uintptr_t(7));
  uint64_t* empty = full + NS;
  uint64_t* sync_bar = empty + NS;
  volatile int* abort = reinterpret_cast<volatile int*>(sync_bar + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(sync_bar, kNC);
    *abort = 0;
    fence_barrier_init();
  }
  __syncthreads();
  pdl_wait_primary();  // the plan kernel's list, counters and lengths
  pdl_launch_dependents();

  const int n_items = p.hdr[0];

  if (warp == kNC) {
    // ---------------------------------------------------------- producer
    // Lanes 0..kPL-1 are independent producers: each walks the same item and
    // stage sequence and issues the stages that fall to it (one bulk copy per
    // contiguous page run of the HND layout, per token row of the NHD layout).
    uint32_t ctr = 0;
    if (lane < kPL) {
      const uint64_t policy = make_evict_first();
      const uint8_t* kpool = static_cast<const uint8_t*>(p.k_pool);
      const uint8_t* vpool = static_cast<const uint8_t*>(p.v_pool);
      for (int k = 0;; ++k) {
        const int it = serpentine_item(k, blockIdx.x, gridDim.x);
        if (it >= n_items) break;
        const Item I = decode_item(p, it);
        if (I.q_row < 0) continue;
        const int32_t* pages = p.page_indices + p.page_indptr[I.r];
        for (int kv = 0; kv < 2; ++kv) {
          const uint8_t* pool = kv ? vpool : kpool;
          for (int t0 = I.t_begin; t0 < I.t_end; t0 += kTS, ++ctr) {
            if ((int)(ctr % kPL) != lane) continue;
            const int slot = ctr % NS;
            if (!mbar_wait(&empty[slot], ((ctr / NS) & 1u) ^ 1u, abort, p.status)) goto producer_done;
            const int t1 = min(t0 + kTS, I.t_end);
            mbar_arrive_expect_tx(&full[slot], (uint32_t)((t1 - t0) * RB));
            for (int t = t0; t < t1;) {
              const int slot_in_page = t % p.page_size;
              // HND: the rest of the page's head slice is one run; NHD: one token row
              // (slots of a head are hkv rows apart) unless there is a single head
              const int run = (p.nhd && p.hkv > 1) ? 1 : min(t1 - t, p.page_size - slot_in_page);
              int32_t pid = __ldg(pages + t / p.page_size);
              if (pid < 0 || pid >= p.num_pages) {
                report(p.status, PD_DEV_BAD_PAGE_TABLE);
                pid = 0;
              }
              const int64_t row = p.nhd ? ((int64_t)pid * p.page_size + slot_in_page) * p.hkv + I.g
                                        : ((int64_t)pid * p.hkv + I.g) * p.page_size + slot_in_page;
              const uint8_t* src = pool + row * (int64_t)RB;
              bulk_g2s_hint(ring + (size_t)slot * SB + (size_t)(t - t0) * RB, src, (uint32_t)(run * RB), &full[slot],
                            policy);
              t += run;
            }
          }
        }
      }
    }
  producer_done:
    // On an abort, give this lane's copies still in flight a bounded chance to
    // land before the CTA's shared memory is released.
    if (*abort && lane < kPL) {
      for (uint32_t k = (ctr > (uint32_t)NS ? ctr - NS : 0); k < ctr; ++k) {
        if ((int)(k % kPL) != lane) continue;
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait(&full[k % NS], (k / NS) & 1u) && globaltimer_ns() - t0 < kWaitLimitNs) {
        }
      }
    }
  } else {
    // ---------------------------------------------------------- consumers
    const int cw = warp;
    const int tg = lane >> 3, dg = lane & 7;
    uint32_t ctr = 0, sync_phase = 0;
    for (int k = 0;; ++k) {
      const int it = serpentine_item(k, blockIdx.x, gridDim.x);
      if (it >= n_items) break;
      const Item I = decode_item(p, it);
      if (I.q_row < 0) continue;
      const int n_tok = I.t_end - I.t_begin;
      const int n_st = (n_tok + kTS - 1) / kTS;

      // query rows of the GS heads, pre-scaled so that scores are in log2 units
      float qr[GS][E];
      {
        const uint8_t* qb = static_cast<const uint8_t*>(p.q) + ((int64_t)I.q_row * p.hq + I.h0) * RB;
#pragma unroll
        for (int h = 0; h < GS; ++h) {
          load_lane_row<ES, D>(qb + (size_t)h * RB, dg, qr[h]);
#pragma unroll
          for (int e = 0; e < E; ++e) qr[h][e] *= p.scale_log2;
        }
      }

      // ---- K phase: scores of this warp's stages into s_scores[token][head]
      for (int s = 0; s < n_st; ++s, ++ctr) {
        if ((s % kNC) != cw) continue;
        const int slot = ctr % NS;
        if (!warp_mbar_wait(&full[slot], (ctr / NS) & 1u, abort, p.status)) goto consumer_done;
        const uint8_t* buf = ring + (size_t)slot * SB;
        float acc[kTPL * GS];
#pragma unroll
        for (int i = 0; i < kTPL; ++i) {
          float kf[E];
          load_lane_row<ES, D>(buf + (size_t)(tg + 4 * i) * RB, dg, kf);
#pragma unroll
          for (int h = 0; h < GS; ++h) {
            float2 a = make_float2(0.f, 0.f);
#pragma unroll
            for (int e = 0; e < E; e += 2)
              a = ffma2(make_float2(qr[h][e], qr[h][e + 1]), make_float2(kf[e], kf[e + 1]), a);
            acc[i * GS + h] = a.x + a.y;
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[slot]);
        xreduce<kTPL * GS, 4>(acc, lane);
        constexpr int N = kTPL * GS;
        constexpr int CNT = N >= 8 ? N / 8 : 1;
        constexpr int SHIFT = N >= 8 ? 0 : (N == 4 ? 1 : 2);
        const bool writer = N >= 8 ? true : ((dg & ((1 << SHIFT) - 1)) == 0);
        const int base = N >= 8 ? dg * (N / 8) : (dg >> SHIFT);
        const int valid = min(kTS, n_tok - s * kTS);
        if (writer) {
#pragma unroll
          for (int c = 0; c < CNT; ++c) {
            const int idx = base + c;
            const int i = idx / GS, h = idx % GS;
            const int j = tg + 4 * i;
            if (j < valid) s_scores[(s * kTS + j) * GS + h] = acc[c];
          }
        }
      }
      if (!consumer_sync(sync_bar, sync_phase, lane, abort, p.status)) goto consumer_done;

      // ---- chunk softmax: max, exp2 in place, sum (warp per head)
      for (int h = cw; h < GS; h += kNC) {
        float m = -INFINITY;
        for (int j = lane; j < n_tok; j += 32) m = fmaxf(m, s_scores[j * GS + h]);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, o));
        float l = 0.f;
        for (int j = lane; j < n_tok; j += 32) {
          const float e = exp2f(s_scores[j * GS + h] - m);
          s_scores[j * GS + h] = e;
          l += e;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(kFull, l, o);
        if (lane == 0) {
          s_m[h] = m;
          s_l[h] = l;
        }
      }
      if (!consumer_sync(sync_bar, sync_phase, lane, abort, p.status)) goto consumer_done;

      // ---- V phase: weighted sum of this warp's stages
      float2 oacc[GS][E / 2];
#pragma unroll
      for (int h = 0; h < GS; ++h)
#pragma unroll
        for (int e = 0; e < E / 2; ++e) oacc[h][e] = make_float2(0.f, 0.f);
      for (int s = 0; s < n_st; ++s, ++ctr) {
        if ((s % kNC) != cw) continue;
        const int slot = ctr % NS;
        if (!warp_mbar_wait(&full[slot], (ctr / NS) & 1u, abort, p.status)) goto consumer_done;
        const uint8_t* buf = ring + (size_t)slot * SB;
        const int valid = min(kTS, n_tok - s * kTS);
#pragma unroll
        for (int i = 0; i < kTPL; ++i) {
          const int j = tg + 4 * i;
          if (j < valid) {
            float pw[GS];
#pragma unroll
            for (int h = 0; h < GS; ++h) pw[h] = s_scores[(s * kTS + j) * GS + h];
            float vf[E];
            load_lane_row<ES, D>(buf + (size_t)j * RB, dg, vf);
#pragma unroll
            for (int h = 0; h < GS; ++h)
#pragma unroll
              for (int e = 0; e < E / 2; ++e)
                oacc[h][e] = ffma2(make_float2(pw[h], pw[h]), make_float2(vf[2 * e], vf[2 * e + 1]), oacc[h][e]);
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[slot]);
      }
      // sum the four token groups of the warp, then park the warp's partial
#pragma unroll
      for (int h = 0; h < GS; ++h)
#pragma unroll
        for (int e = 0; e < E / 2; ++e) {
          float2 v = oacc[h][e];
          v.x += __shfl_xor_sync(kFull, v.x, 8);
          v.y += __shfl_xor_sync(kFull, v.y, 8);
          v.x += __shfl_xor_sync(kFull, v.x, 16);
          v.y += __shfl_xor_sync(kFull, v.y, 16);
          oacc[h][e] = v;
        }
      if (tg == 0) {
#pragma unroll
        for (int h = 0; h < GS; ++h)
#pragma unroll
          for (int e = 0; e < E / 2; ++e) {
            s_opart[(cw * GS + h) * D + lane_dim<ES, D>(dg, 2 * e)] = oacc[h][e].x;
            s_opart[(cw * GS + h) * D + lane_dim<ES, D>(dg, 2 * e + 1)] = oacc[h][e].y;
          }
      }
      if (!consumer_sync(sync_bar, sync_phase, lane, abort, p.status)) goto consumer_done;

      // ---- epilogue: final output for single-chunk requests, partials otherwise
      {
        const bool single = I.n_chunks == 1;
        for (int idx = threadIdx.x; idx < GS * D; idx += kNC * 32) {
          const int h = idx / D, d = idx % D;
          float v = 0.f;
#pragma unroll
          for (int w = 0; w < kNC; ++w) v += s_opart[(w * GS + h) * D + d];
          v /= s_l[h];
          const int qh = I.h0 + h;
          if (single) {
            const int64_t off = ((int64_t)I.q_row * p.hq + qh) * D + d;
            if (p.o_dtype == PD_BF16)
              static_cast<uint16_t*>(p.o)[off] = f32_to_bf16_bits(v);
            else
              static_cast<float*>(p.o)[off] = v;
            if (d == 0 && p.lse != nullptr) p.lse[(int64_t)I.q_row * p.hq + qh] = (s_m[h] + log2f(s_l[h])) * kLn2;
          } else {
            const int64_t pc = (int64_t)(I.first_chunk + I.chunk) * p.hq + qh;
            p.part_o[pc * D + d] = v;
            if (d == 0) p.part_lse[pc] = s_m[h] + log2f(s_l[h]);
          }
        }
      }
      if (!consumer_sync(sync_bar, sync_phase, lane, abort, p.status)) goto consumer_done;
    }
  consumer_done:;
  }
}

// ------------------------------------------------------------------ merge
// One warp per (request, query head) of a request split into several chunks:
// combine the chunks' partial outputs by their log-sum-exp. Each lane owns
// D / 32 consecutive dimensions; four chunks' loads are in flight at a time.
template <int D>
__global__ void __launch_bounds__(256) decode_merge_kernel(const DecodeParams p) {
  pdl_wait_primary();  // the decode kernel's partials
  const int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (gw >= p.batch * p.hq) return;
  const int r = gw / p.hq, h = gw % p.hq;
  const int4 info = p.req_info[r];
  if (info.w < 0 || info.y <= 1) return;
  constexpr int PER = D / 32;
  static_assert(PER == 2 || PER == 4, "head_dim 64 or 128");
  const int n = info.y;
  const float* pl = p.part_lse + (int64_t)info.x * p.hq + h;
  float m = -INFINITY;
  for (int c = lane; c < n; c += 32) m = fmaxf(m, __ldcg(pl + (int64_t)c * p.hq));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, o));
  float l = 0.f;
  for (int c = lane; c < n; c += 32) l += exp2f(__ldcg(pl + (int64_t)c * p.hq) - m);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(kFull, l, o);
  const float* po = p.part_o + ((int64_t)info.x * p.hq + h) * D + lane * PER;
  const int64_t cs = (int64_t)p.hq * D;  // chunk stride of part_o
  float acc[PER];
#pragma unroll
  for (int e = 0; e < PER; ++e) acc[e] = 0.f;
  auto load = [&](int c, float (&v)[PER]) {
    if constexpr (PER == 4) {
      const float4 x = __ldcg(reinterpret_cast<const float4*>(po + c * cs));
      v[0] = x.x, v[1] = x.y, v[2] = x.z, v[3] = x.w;
    } else {
      const float2 x = __ldcg(reinterpret_cast<const float2*>(po + c * cs));
      v[0] = x.x, v[1] = x.y;
    }
  };
  int c = 0;
  for (; c + 4 <= n; c += 4) {
    float lw[4], v[4][PER];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      lw[j] = __ldcg(pl + (int64_t)(c + j) * p.hq);
      load(c + j, v[j]);
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float w = exp2f(lw[j] - m);
#pragma unroll
      for (int e = 0; e < PER; ++e) acc[e] = fmaf(w, v[j][e], acc[e]);
    }
  }
  for (; c < n; ++c) {
    float v[PER];
    load(c, v);
    const float w = exp2f(__ldcg(pl + (int64_t)c * p.hq) - m);
#pragma unroll
    for (int e = 0; e < PER; ++e) acc[e] = fmaf(w, v[e], acc[e]);
  }
  const float inv = 1.f / l;
  const int64_t orow = ((int64_t)info.w * p.hq + h) * D + lane * PER;
#pragma unroll
  for (int e = 0; e < PER; ++e) {
    if (p.o_dtype == PD_BF16)
      static_cast<uint16_t*>(p.o)[orow + e] = f32_to_bf16_bits(acc[e] * inv);
    else
      static_cast<float*>(p.o)[orow + e] = acc[e] * inv;
  }
  if (lane == 0 && p.lse != nullptr) p.lse[(int64_t)info.w * p.hq + h] = (m + log2f(l)) * kLn2;
}

// ------------------------------------------------------------------- host
int32_t decode_heads_per_item(int32_t group, int32_t head_dim) {
  for (int gs = 8; gs >= 1; gs >>= 1)
    if (group % gs == 0 && gs * head_dim <= 512) return gs;
  return 1;
}

DecodeLayout decode_layout(int32_t batch, int32_t hq, int32_t head_dim, int32_t max_kv_len,
                           int32_t items_per_chunk, int32_t sm_count) {
  DecodeLayout L{};
  // Chunk target: enough work items to cover every SM several times over,
  // never longer than kMaxChunk, never shorter than four stages.
  const int64_t want_items = (int64_t)8 * 2 * (sm_count > 0 ? sm_count : 148);
  const int64_t kv = max_kv_len > 0 ? max_kv_len : 1;
  int64_t c = ((int64_t)batch * items_per_chunk * kv + want_items - 1) / want_items;
  c = (c + kTS - 1) / kTS * kTS;
  if (c < 4 * kTS) c = 4 * kTS;
  if (c > kMaxChunk) c = kMaxChunk;
  L.chunk_target = (int32_t)c;
  const int64_t per_req = (kv + c - 1) / c;
  L.max_chunks = (int32_t)((int64_t)(batch > 0 ? batch : 1) * per_req);
  size_t off = 0;
  L.hdr = off;
  off = align_up(off + 64 * sizeof(int32_t), 256);
  L.req_info = off;
  off = align_up(off + sizeof(int4) * (size_t)(batch > 0 ? batch : 1), 256);
  L.rc_list = off;
  off = align_up(off + sizeof(int2) * (size_t)L.max_chunks, 256);
  L.part_o = off;
  off = align_up(off + sizeof(float) * (size_t)L.max_chunks * hq * head_dim, 256);
  L.part_lse = off;
  off = align_up(off + sizeof(float) * (size_t)L.max_chunks * hq, 256);
  L.total = off;
  return L;
}

namespace {

// Launch with programmatic stream serialisation when `pdl` is set.
template <typename Kernel>
cudaError_t launch_dependent(Kernel kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t stream, bool pdl,
                             const DecodeParams& p) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, p);
}

template <int ES, int D, int GS>
int run_decode(DecodeParams& p, cudaStream_t stream) {
  constexpr size_t smem = decode_smem_bytes<ES, D, GS>();
  // per device: 1 + resident CTAs per SM once the kernel's shared-memory
  // attribute is set there (0: not yet); callers may run on several threads
  static std::atomic<int> configured[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PD_ERR_CUDA;
  const bool cached = dev >= 0 && dev < 64 && partition_sms() == 0;
  int blocks_per_sm = cached ? configured[dev].load(std::memory_order_acquire) - 1 : 0;
  if (blocks_per_sm < 1) {
    if (cudaFuncSetAttribute(decode_kernel<ES, D, GS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem) != cudaSuccess)
      return PD_ERR_CUDA;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks_per_sm, decode_kernel<ES, D, GS>, kThreads,
                                                      smem) != cudaSuccess)
      return PD_ERR_CUDA;
    if (blocks_per_sm < 1) blocks_per_sm = 1;
    if (cached) configured[dev].store(blocks_per_sm + 1, std::memory_order_release);
  }
  decode_plan_kernel<<<1, 1024, 0, stream>>>(p);
  const int64_t max_items = (int64_t)p.max_chunks * p.items_per_chunk;
  int64_t grid = (int64_t)device_sm_count() * blocks_per_sm;
  if (grid > max_items) grid = max_items;
  if (grid < 1) grid = 1;
  last_kernel() = "decode_kernel";
  // Each kernel is a programmatic dependent of the previous one: its CTAs are
  // placed and set up while the previous kernel drains. When the decode kernel
  // is timed alone (profiling events) it runs without that overlap.
  const bool timed = profile_events().start != nullptr;
  profile_begin(stream);
  if (launch_dependent(decode_kernel<ES, D, GS>, dim3((unsigned)grid), dim3(kThreads), smem, stream, !timed, p) !=
      cudaSuccess)
    return PD_ERR_CUDA;
  profile_end(stream);
  const int warps = p.batch * p.hq;
  if (warps > 0 &&
      launch_dependent(decode_merge_kernel<D>, dim3((unsigned)((warps + 7) / 8)), dim3(256), 0, stream, !timed, p) !=
          cudaSuccess)
    return PD_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? PD_OK : PD_ERR_CUDA;
}

template <int ES, int D>
int run_decode_gs(DecodeParams& p, cudaStream_t stream) {
  switch (p.heads_per_item) {
    case 1: return run_decode<ES, D, 1>(p, stream);
    case 2: return run_decode<ES, D, 2>(p, stream);
    case 4: return run_decode<ES, D, 4>(p, stream);
    case 8:
      if constexpr (D <= 64) return run_decode<ES, D, 8>(p, stream);
      return PD_ERR_UNSUPPORTED;
    default: return PD_ERR_UNSUPPORTED;
  }
}

}  // namespace

int launch_decode(DecodeParams& p, int32_t kv_dtype, cudaStream_t stream) {
  if (kv_dtype == PD_BF16) {
    if (p.head_dim == 128) return run_decode_gs<2, 128>(p, stream);
    if (p.head_dim == 64) return run_decode_gs<2, 64>(p, stream);
  } else if (kv_dtype == PD_F32) {
    if (p.head_dim == 128) return run_decode_gs<4, 128>(p, stream);
    if (p.head_dim == 64) return run_decode_gs<4, 64>(p, stream);
  }
  return PD_ERR_UNSUPPORTED;
}

}  // namespace pd
