// pd_kvcopy.cu -- KV-cache append and the page pack / unpack of the KV handoff.
//
// Perplexity, "Disaggregated prefill and decode" (2025):
//   section "KV Messenger": page copies of a layer start as soon as the model
//   has appended that layer's KV entries to the cache;
//   section "Sharded KV cache transfers" and its figure on NHD/HND layouts: with
//   the HND layout each head's slice of a page is contiguous, so a page slice
//   moves as one run; when prefiller and decoder cut pages differently, pages
//   are split or rebuilt.
//
// All three are pure byte moves, bound by HBM bandwidth. A unit of work of
// pack / unpack is a (page, head) slice, contiguous on both sides for HND pools
// and a run of head_dim rows hkv rows apart on the pool side for NHD pools
// (pack from NHD pools takes a token's rows of all copied heads instead, one
// contiguous run there); one warp copies a unit with 16-byte vector loads,
// several in flight per lane.
#include "pd_common.cuh"
#include "pd_internal.h"

namespace pd {

namespace {

constexpr int kCopyThreads = 256;
constexpr int kUnroll = 8;  // 16-byte vectors in flight per lane

__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ void st_stream(uint4* p, uint4 v) {
  asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}

// One warp copies nvec 16-byte vectors from src to dst.
__device__ __forceinline__ void warp_copy(const uint4* __restrict__ src, uint4* __restrict__ dst, int nvec,
                                          int lane) {
  for (int base = 0; base < nvec; base += 32 * kUnroll) {
    uint4 t[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int i = base + u * 32 + lane;
      if (i < nvec) t[u] = ld_stream(src + i);
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int i = base + u * 32 + lane;
      if (i < nvec) st_stream(dst + i, t[u]);
    }
  }
}

// One warp copies `rows` rows of vpr 16-byte vectors; row i sits src_stride
// vectors after row i-1 on the source side and dst_stride on the destination
// side (a head's slots in an NHD pool are hkv rows apart).
__device__ __forceinline__ void warp_copy_rows(const uint4* __restrict__ src, int64_t src_stride,
                                               uint4* __restrict__ dst, int64_t dst_stride, int rows, int vpr,
                                               int lane) {
  if (src_stride == vpr && dst_stride == vpr) {
    warp_copy(src, dst, rows * vpr, lane);
    return;
  }
  const int nvec = rows * vpr;
  // row of vector i: a shift when vpr is a power of two (every head_dim the
  // benchmarks use), a division otherwise
  const bool pow2 = (vpr & (vpr - 1)) == 0;
  const int lg = __ffs(vpr) - 1;
  for (int base = 0; base < nvec; base += 32 * kUnroll) {
    uint4 t[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int i = base + u * 32 + lane;
      if (i < nvec) {
        const int r = pow2 ? i >> lg : i / vpr, c = i - r * vpr;
        t[u] = ld_stream(src + r * src_stride + c);
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int i = base + u * 32 + lane;
      if (i < nvec) {
        const int r = pow2 ? i >> lg : i / vpr, c = i - r * vpr;
        st_stream(dst + r * dst_stride + c, t[u]);
      }
    }
  }
}

// Vector offset of (page, head, slot) in one layer's pool, and the distance
// between consecutive slots of one head.
__device__ __forceinline__ int64_t pool_vec(const KvCopyParams& p, int64_t page, int h, int slot, int vpr) {
  return (p.nhd ? (page * p.page_size + slot) * p.hkv + h : (page * p.hkv + h) * p.page_size + slot) * vpr;
}
__device__ __forceinline__ int64_t slot_stride_vec(const KvCopyParams& p, int vpr) {
  return p.nhd ? (int64_t)p.hkv * vpr : vpr;
}

// Unit u of a pack / unpack enumerates (request r, layer, K/V, head h of the
// range, page k of the request). Page k carries tokens [k*P, min((k+1)*P,
// kv_len)); packed head h is pool head head_begin + h. For HND pools k is
// fastest, so consecutive warps touch consecutive bytes of the packed buffer;
// for NHD pools (unpack) h is fastest, so consecutive warps cover the rows of
// one page, which are contiguous in the pool.
struct Unit {
  int r, layer, kv, h, k;
};

__device__ __forceinline__ Unit unit_of(int64_t u, int kp, int hkv, int layers, bool head_fastest) {
  Unit x;
  if (head_fastest) {
    x.h = (int)(u % hkv);
    u /= hkv;
    x.k = (int)(u % kp);
    u /= kp;
  } else {
    x.k = (int)(u % kp);
    u /= kp;
    x.h = (int)(u % hkv);
    u /= hkv;
  }
  x.kv = (int)(u % 2);
  u /= 2;
  x.layer = (int)(u % layers);
  x.r = (int)(u / layers);
  return x;
}

}  // namespace

// --------------------------------------------------------------- append
// Each CTA takes blocks of up to kAppendRows consecutive new-token rows. One
// thread per row finds the row's request (binary search over the new-token
// indptr), checks it and looks up its page, all rows at once; then the CTA
// copies the block's K and V rows (every head), row by row, with several
// 16-byte vectors in flight per thread.
constexpr int kAppendRows = 32;

__global__ void __launch_bounds__(kCopyThreads) kv_append_kernel(const KvCopyParams p, int rows_per_cta) {
  __shared__ int s_page[kAppendRows], s_slot[kAppendRows];
  const int vpr = p.head_dim * p.elem_size / 16;  // vectors per (token, head) row
  const int hv = p.hkv * vpr;                     // vectors of one token's K (or V)
  const int per_row = 2 * hv;                     // vectors of K and V of one token
  // pool vector offset of (page, head h, slot) = page * page_vecs + slot * slot_stride + h * head_stride
  const int64_t page_vecs = (int64_t)p.hkv * p.page_size * vpr;
  const int64_t slot_stride = slot_stride_vec(p, vpr);
  const int head_stride = p.nhd ? vpr : p.page_size * vpr;
  const bool pow2 = (vpr & (vpr - 1)) == 0;
  const int lg = __ffs(vpr) - 1;
  for (int r0 = blockIdx.x * rows_per_cta; r0 < p.max_new; r0 += gridDim.x * rows_per_cta) {
    const int nrows = min(rows_per_cta, p.max_new - r0);
    if (threadIdx.x < nrows) {
      const int row = r0 + threadIdx.x;
      // request owning the row: last r with new_indptr[r] <= row
      int lo = 0, hi = p.batch;  // answer in [lo, hi)
      while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (__ldg(p.new_indptr + mid) <= row) lo = mid;
        else hi = mid;
      }
      const int r = lo;
      const int a = __ldg(p.new_indptr + r), b = __ldg(p.new_indptr + r + 1);
      int page = -1, slot = 0;
      if (row >= a && row < b) {  // else: a row past the last request's tokens
        const int n_new = b - a, n = __ldg(p.kv_len + r);
        const int pa = __ldg(p.page_indptr + r), pb = __ldg(p.page_indptr + r + 1);
        const int t = n - n_new + (row - a);
        if (n_new <= n && n <= p.max_kv_len && pa >= 0 && pb >= pa && (int64_t)(pb - pa) * p.page_size >= n) {
          const int pg = __ldg(p.page_indices + pa + t / p.page_size);
          if (pg >= 0 && pg < p.num_pages) {
            page = pg;
            slot = t % p.page_size;
          } else {
            report(p.status, PD_DEV_BAD_PAGE_TABLE);
          }
        } else {
          report(p.status, PD_DEV_BAD_LENGTH);
        }
      }
      s_page[threadIdx.x] = page;
      s_slot[threadIdx.x] = slot;
    }
    __syncthreads();
    // Row by row: the row's (page, slot) base once, then its K and V vectors,
    // several in flight per thread; the head of a vector by a shift when
    // head_dim * elem_size / 16 is a power of two.
    for (int k = 0; k < nrows; ++k) {
      const int page = s_page[k];
      if (page < 0) continue;
      const int64_t base = (int64_t)page * page_vecs + (int64_t)s_slot[k] * slot_stride;
      const int64_t row = (int64_t)(r0 + k) * hv;
      for (int q0 = 0; q0 < per_row; q0 += kCopyThreads * kUnroll) {
        uint4 t[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
          const int q = q0 + u * kCopyThreads + threadIdx.x;
          if (q < per_row) {
            const bool second = q >= hv;
            t[u] = ld_stream(static_cast<const uint4*>(second ? p.src2 : p.src) + row + (q - (second ? hv : 0)));
          }
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
          const int q = q0 + u * kCopyThreads + threadIdx.x;
          if (q < per_row) {
            const bool second = q >= hv;
            const int w = q - (second ? hv : 0);
            const int h = pow2 ? w >> lg : w / vpr, v = w - h * vpr;
            static_cast<uint4*>(second ? p.dst2 : p.dst)[base + (int64_t)h * head_stride + v] = t[u];
          }
        }
      }
    }
    __syncthreads();  // the block's metadata is rewritten next
  }
}

// ----------------------------------------------------------------- pack
// NHD pools: a token's rows of the copied heads are contiguous in the pool, so
// a unit is (request, layer, K/V, token): one contiguous read of those rows,
// each row then written to its head's slab of the packed block. Consecutive
// units are consecutive tokens, so the warps of a CTA read a page's bytes in
// order (per-head units would read it in 256-byte pieces a token apart).
__device__ __forceinline__ void pack_nhd_tokens(const KvCopyParams& p, int lane, int64_t warp0, int64_t nwarps) {
  const int vpr = p.head_dim * p.elem_size / 16;
  const int64_t units = (int64_t)p.batch * p.layer_count * 2 * p.max_kv_len;
  for (int64_t u = warp0; u < units; u += nwarps) {
    const int t = (int)(u % p.max_kv_len);
    int64_t rest = u / p.max_kv_len;
    const int kv = (int)(rest % 2);
    rest /= 2;
    const int layer = p.layer_begin + (int)(rest % p.layer_count);
    const int r = (int)(rest / p.layer_count);
    const int n = __ldg(p.kv_len + r);
    if (t >= n) continue;
    const int pa = __ldg(p.page_indptr + r), pb = __ldg(p.page_indptr + r + 1);
    const int64_t off = __ldg(p.offsets + r);
    const int64_t block = (int64_t)p.num_layers * 2 * p.head_count * n * vpr * 16;
    const bool bad_off = (off & 15) != 0 || off < 0 || off + block > p.buf_bytes;
    if (n > p.max_kv_len || pa < 0 || (int64_t)(pb - pa) * p.page_size < n || bad_off) {
      if (lane == 0) report(p.status, bad_off ? PD_DEV_BAD_OFFSET : PD_DEV_BAD_PAGE_TABLE);
      continue;
    }
    const int32_t page = __ldg(p.page_indices + pa + t / p.page_size);
    if (page < 0 || page >= p.num_pages) {
      if (lane == 0) report(p.status, PD_DEV_BAD_PAGE_TABLE);
      continue;
    }
    const uint8_t* pool = static_cast<const uint8_t*>(kv ? p.src2 : p.src) + (int64_t)layer * p.layer_stride;
    const uint4* src = reinterpret_cast<const uint4*>(pool) + pool_vec(p, page, p.head_begin, t % p.page_size, vpr);
    uint4* dst = reinterpret_cast<uint4*>(static_cast<uint8_t*>(p.dst) + off) +
                 (((int64_t)layer * 2 + kv) * p.head_count * n + t) * vpr;
    warp_copy_rows(src, vpr, dst, (int64_t)n * vpr, p.head_count, vpr, lane);
  }
}

__global__ void __launch_bounds__(kCopyThreads) kv_pack_kernel(const KvCopyParams p) {
  const int lane = threadIdx.x & 31;
  const int64_t warp0 = ((int64_t)blockIdx.x * kCopyThreads + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * kCopyThreads) >> 5;
  if (p.nhd) {
    pack_nhd_tokens(p, lane, warp0, nwarps);
    return;
  }
  const int kp = (p.max_kv_len + p.page_size - 1) / p.page_size;
  const int64_t units = (int64_t)p.batch * p.layer_count * 2 * p.head_count * kp;
  const int vpr = p.head_dim * p.elem_size / 16;
  for (int64_t u = warp0; u < units; u += nwarps) {
    Unit x = unit_of(u, kp, p.head_count, p.layer_count, p.nhd != 0);
    x.layer += p.layer_begin;  // blocks keep all num_layers layers
    const int n = __ldg(p.kv_len + x.r);
    if ((int64_t)x.k * p.page_size >= n) continue;
    const int pa = __ldg(p.page_indptr + x.r), pb = __ldg(p.page_indptr + x.r + 1);
    const int64_t off = __ldg(p.offsets + x.r);
    const int64_t block = (int64_t)p.num_layers * 2 * p.head_count * n * vpr * 16;
    const bool bad_off = (off & 15) != 0 || off < 0 || off + block > p.buf_bytes;
    if (n > p.max_kv_len || pa < 0 || (int64_t)(pb - pa) * p.page_size < n || bad_off) {
      if (lane == 0) report(p.status, bad_off ? PD_DEV_BAD_OFFSET : PD_DEV_BAD_PAGE_TABLE);
      continue;
    }
    const int32_t page = __ldg(p.page_indices + pa + x.k);
    if (page < 0 || page >= p.num_pages) {
      if (lane == 0) report(p.status, PD_DEV_BAD_PAGE_TABLE);
      continue;
    }
    const int rows = min(p.page_size, n - x.k * p.page_size);
    const uint8_t* pool = static_cast<const uint8_t*>(x.kv ? p.src2 : p.src) + (int64_t)x.layer * p.layer_stride;
    const uint4* src = reinterpret_cast<const uint4*>(pool) + pool_vec(p, page, p.head_begin + x.h, 0, vpr);
    uint4* dst = reinterpret_cast<uint4*>(static_cast<uint8_t*>(p.dst) + off) +
                 ((((int64_t)x.layer * 2 + x.kv) * p.head_count + x.h) * n + (int64_t)x.k * p.page_size) * vpr;
    warp_copy_rows(src, slot_stride_vec(p, vpr), dst, vpr, rows, vpr, lane);
  }
}

// --------------------------------------------------------------- unpack
__global__ void __launch_bounds__(kCopyThreads) kv_unpack_kernel(const KvCopyParams p) {
  const int lane = threadIdx.x & 31;
  const int64_t warp0 = ((int64_t)blockIdx.x * kCopyThreads + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * kCopyThreads) >> 5;
  const int kp = (p.max_kv_len + p.page_size - 1) / p.page_size;
  const int64_t units = (int64_t)p.batch * p.num_layers * 2 * p.head_count * kp;
  const int vpr = p.head_dim * p.elem_size / 16;
  for (int64_t u = warp0; u < units; u += nwarps) {
    const Unit x = unit_of(u, kp, p.head_count, p.num_layers, p.nhd != 0);
    const int n = __ldg(p.kv_len + x.r);
    if ((int64_t)x.k * p.page_size >= n) continue;
    const int pa = __ldg(p.page_indptr + x.r), pb = __ldg(p.page_indptr + x.r + 1);
    const int64_t off = __ldg(p.offsets + x.r);
    const int64_t block = (int64_t)p.num_layers * 2 * p.head_count * n * vpr * 16;
    const bool bad_off = (off & 15) != 0 || off < 0 || off + block > p.buf_bytes;
    if (n > p.max_kv_len || pa < 0 || (int64_t)(pb - pa) * p.page_size < n || bad_off) {
      if (lane == 0) report(p.status, bad_off ? PD_DEV_BAD_OFFSET : PD_DEV_BAD_PAGE_TABLE);
      continue;
    }
    const int32_t page = __ldg(p.page_indices + pa + x.k);
    if (page < 0 || page >= p.num_pages) {
      if (lane == 0) report(p.status, PD_DEV_BAD_PAGE_TABLE);
      continue;
    }
    const int rows = min(p.page_size, n - x.k * p.page_size);
    uint8_t* pool = static_cast<uint8_t*>(x.kv ? p.dst2 : p.dst) + (int64_t)x.layer * p.layer_stride;
    uint4* dst = reinterpret_cast<uint4*>(pool) + pool_vec(p, page, p.head_begin + x.h, 0, vpr);
    const uint4* src = reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(p.src) + off) +
                       ((((int64_t)x.layer * 2 + x.kv) * p.head_count + x.h) * n + (int64_t)x.k * p.page_size) * vpr;
    warp_copy_rows(src, vpr, dst, slot_stride_vec(p, vpr), rows, vpr, lane);
  }
}

// ----------------------------------------------------------------- host
namespace {
int copy_grid() { return device_sm_count() * (2048 / kCopyThreads); }
}  // namespace

int launch_kv_append(const KvCopyParams& p, cudaStream_t stream) {
  if (p.max_new <= 0 || p.batch <= 0) return PD_OK;
  // blocks of consecutive rows, about one per CTA slot of the GPU
  const int slots = copy_grid();
  int rows_per_cta = (p.max_new + slots - 1) / slots;
  if (rows_per_cta > kAppendRows) rows_per_cta = kAppendRows;
  const int grid = (p.max_new + rows_per_cta - 1) / rows_per_cta < slots
                       ? (p.max_new + rows_per_cta - 1) / rows_per_cta
                       : slots;
  last_kernel() = "kv_append_kernel";
  profile_begin(stream);
  kv_append_kernel<<<grid, kCopyThreads, 0, stream>>>(p, rows_per_cta);
  profile_end(stream);
  return cudaGetLastError() == cudaSuccess ? PD_OK : PD_ERR_CUDA;
}

int launch_kv_pack(const KvCopyParams& p, cudaStream_t stream) {
  if (p.batch <= 0 || p.max_kv_len <= 0) return PD_OK;
  last_kernel() = "kv_pack_kernel";
  profile_begin(stream);
  kv_pack_kernel<<<copy_grid(), kCopyThreads, 0, stream>>>(p);
  profile_end(stream);
  return cudaGetLastError() == cudaSuccess ? PD_OK : PD_ERR_CUDA;
}

int launch_kv_unpack(const KvCopyParams& p, cudaStream_t stream) {
  if (p.batch <= 0 || p.max_kv_len <= 0) return PD_OK;
  last_kernel() = "kv_unpack_kernel";
  profile_begin(stream);
  kv_unpack_kernel<<<copy_grid(), kCopyThreads, 0, stream>>>(p);
  profile_end(stream);
  return cudaGetLastError() == cudaSuccess ? PD_OK : PD_ERR_CUDA;
}

}  // namespace pd
