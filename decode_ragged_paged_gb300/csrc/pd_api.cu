// pd_api.cu -- the C ABI declared in include/pd.h: host-side argument checks,
// workspace layout and dispatch to the kernel launchers. No entry point
// allocates device memory, synchronises the stream or throws.
#include <math.h>
#include <stdint.h>

#include <atomic>

#include "pd_internal.h"

namespace pd {

int& partition_sms() {
  static thread_local int n = 0;
  return n;
}

int device_sm_count() {
  if (partition_sms() > 0) return partition_sms();
  static std::atomic<int> cache[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (dev >= 0 && dev < 64) {
    int v = cache[dev].load(std::memory_order_relaxed);
    if (v > 0) return v;
  }
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
  if (dev >= 0 && dev < 64) cache[dev].store(n, std::memory_order_relaxed);
  return n;
}

const char*& last_kernel() {
  static thread_local const char* name = "";
  return name;
}

ProfileEvents& profile_events() {
  static thread_local ProfileEvents ev;
  return ev;
}

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int elem_size(int32_t dtype) { return dtype == PD_BF16 ? 2 : dtype == PD_F32 ? 4 : 0; }

// Host-side checks shared by the attention entry points.
int check_attn(const pd_attn_desc* d, const pd_batch* b, bool need_qo_indptr) {
  if (d == nullptr || b == nullptr) return PD_ERR_INVALID_ARG;
  if (d->num_qo_heads <= 0 || d->num_kv_heads <= 0 || d->num_qo_heads % d->num_kv_heads != 0)
    return PD_ERR_INVALID_ARG;
  if (d->page_size <= 0 || d->head_dim <= 0) return PD_ERR_INVALID_ARG;
  if (elem_size(d->kv_dtype) == 0 || elem_size(d->o_dtype) == 0) return PD_ERR_INVALID_ARG;
  if (d->layout != PD_LAYOUT_HND && d->layout != PD_LAYOUT_NHD) return PD_ERR_INVALID_ARG;
  if (d->head_dim != 64 && d->head_dim != 128) return PD_ERR_UNSUPPORTED;
  if (!(d->sm_scale <= 0.f || isfinite(d->sm_scale))) return PD_ERR_INVALID_ARG;
  if (b->batch_size < 0 || b->total_qo < 0 || b->max_qo_len < 0 || b->max_kv_len < 0) return PD_ERR_INVALID_ARG;
  if (b->batch_size > 0) {
    if (b->kv_len == nullptr || b->page_indptr == nullptr || b->page_indices == nullptr) return PD_ERR_INVALID_ARG;
    if (need_qo_indptr && b->qo_indptr == nullptr) return PD_ERR_INVALID_ARG;
    if (b->num_pages <= 0) return PD_ERR_INVALID_ARG;
  }
  return PD_OK;
}

float scale_of(const pd_attn_desc* d) {
  return d->sm_scale > 0.f ? d->sm_scale : 1.0f / sqrtf((float)d->head_dim);
}

// A large GQA decode batch runs faster on the tensor-core kernel with the
// query heads of a group packed into one tile (one item per request and KV
// head reads each KV tile once) than on the split-KV kernel; small batches need
// the split to use the whole GPU, and MHA gains nothing from packing. The
// tensor-core path takes decode batches without qo_indptr (row r = request r).
bool decode_on_tensor_cores(const pd_attn_desc* d, const pd_batch* b) {
  if (b->qo_indptr != nullptr || d->kv_dtype != PD_BF16) return false;
  if (prefill_supported(d->kv_dtype, d->head_dim, d->page_size) != PD_OK) return false;
  if (prefill_tile_heads(d->num_qo_heads / d->num_kv_heads) < 2) return false;
  return (int64_t)b->batch_size * d->num_kv_heads >= 4LL * device_sm_count();
}

size_t decode_tc_workspace(const pd_batch* b, const pd_attn_desc* d) {
  return prefill_layout(b->batch_size, b->total_qo, 1, prefill_tile_heads(d->num_qo_heads / d->num_kv_heads)).total;
}

DecodeLayout decode_layout_for(const pd_attn_desc* d, const pd_batch* b) {
  const int gs = decode_heads_per_item(d->num_qo_heads / d->num_kv_heads, d->head_dim);
  return decode_layout(b->batch_size, d->num_qo_heads, d->head_dim, b->max_kv_len, d->num_qo_heads / gs,
                       device_sm_count());
}

}  // namespace

// pd_attn_mixed_split's workspace: the prefill part's plan, then the decode
// part's plan and partials, each sized for the whole batch. The decode part's
// chunk length depends on the SMs of its partition and on how many requests
// it gets; sized for the shortest chunk the plan ever picks (an SM count so
// large that the length sits at its lower bound), it holds any of them.
MixedSplitLayout mixed_split_layout(const pd_attn_desc* d, const pd_batch* b) {
  MixedSplitLayout L{};
  L.decode = align_up(prefill_layout(b->batch_size, b->total_qo, b->max_qo_len,
                                     prefill_tile_heads(d->num_qo_heads / d->num_kv_heads))
                          .total,
                      256);
  const int gs = decode_heads_per_item(d->num_qo_heads / d->num_kv_heads, d->head_dim);
  L.total = L.decode + decode_layout(b->batch_size, d->num_qo_heads, d->head_dim, b->max_kv_len,
                                     d->num_qo_heads / gs, 1 << 20)
                           .total;
  return L;
}

// Plans and launches the tensor-core kernel; arguments already validated.
int run_prefill(const pd_attn_desc* desc, const pd_batch* batch, int32_t max_qo_len, int32_t causal, const void* q,
                const void* k_pool, const void* v_pool, void* o, float* lse, void* workspace, size_t workspace_bytes,
                int32_t* dev_status, void* stream) {
  const int32_t tile_heads = prefill_tile_heads(desc->num_qo_heads / desc->num_kv_heads);
  const PrefillLayout L = prefill_layout(batch->batch_size, batch->total_qo, max_qo_len, tile_heads);
  if (workspace_bytes < L.total) return PD_ERR_WORKSPACE;
  PrefillParams p{};
  p.batch = batch->batch_size;
  p.hq = desc->num_qo_heads;
  p.hkv = desc->num_kv_heads;
  p.group = p.hq / p.hkv;
  p.page_size = desc->page_size;
  p.num_pages = batch->num_pages;
  p.total_qo = batch->total_qo;
  p.max_qo_len = max_qo_len;
  p.max_kv_len = batch->max_kv_len;
  p.causal = causal ? 1 : 0;
  p.o_dtype = desc->o_dtype;
  p.max_rq = L.max_rq;
  p.tile_heads = tile_heads;
  p.tile_rows = 128 / tile_heads;
  p.item_heads = p.hq / tile_heads;
  p.nhd = desc->layout == PD_LAYOUT_NHD;
  p.scale_log2 = scale_of(desc) * kLog2e;
  p.qo_indptr = batch->qo_indptr;
  p.kv_len = batch->kv_len;
  p.page_indptr = batch->page_indptr;
  p.page_indices = batch->page_indices;
  p.o = o;
  p.lse = lse;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  p.hdr = reinterpret_cast<int32_t*>(ws + L.hdr);
  p.rq_list = reinterpret_cast<int2*>(ws + L.rq_list);
  p.status = dev_status;
  return launch_prefill(p, q, k_pool, v_pool, static_cast<cudaStream_t>(stream));
}

}  // namespace pd

using namespace pd;

extern "C" {

int32_t pd_version(void) { return 100; }

const char* pd_last_kernel(void) { return last_kernel(); }

int pd_profile_events(void* start_event, void* stop_event) {
  if ((start_event == nullptr) != (stop_event == nullptr)) return PD_ERR_INVALID_ARG;
  profile_events().start = static_cast<cudaEvent_t>(start_event);
  profile_events().stop = static_cast<cudaEvent_t>(stop_event);
  return PD_OK;
}

const char* pd_status_string(int32_t code) {
  switch (code) {
    case PD_OK: return "ok";
    case PD_ERR_INVALID_ARG: return "invalid argument";
    case PD_ERR_UNSUPPORTED: return "unsupported configuration";
    case PD_ERR_WORKSPACE: return "workspace too small";
    case PD_ERR_CUDA: return "CUDA error";
    case PD_ERR_TIMEOUT: return "timed out waiting for a layer signal";
    default: return "unknown status";
  }
}

const char* pd_device_status_string(int32_t code) {
  switch (code) {
    case PD_DEV_OK: return "ok";
    case PD_DEV_BAD_INDPTR: return "indptr decreasing or out of range";
    case PD_DEV_BAD_LENGTH: return "length out of range";
    case PD_DEV_BAD_PAGE_TABLE: return "page table too short or page id out of range";
    case PD_DEV_NOT_DECODE: return "decode request with qo_len != 1";
    case PD_DEV_TIMEOUT: return "bounded wait timed out inside a kernel";
    case PD_DEV_BAD_OFFSET: return "pack/unpack block misaligned or outside the packed buffer";
    default: return "unknown device status";
  }
}

size_t pd_attn_workspace_size(const pd_attn_desc* desc, const pd_batch* batch, int32_t kind) {
  if (check_attn(desc, batch, false) != PD_OK) return 0;
  if (kind == PD_KIND_DECODE) {
    const size_t split = decode_layout_for(desc, batch).total;
    if (!decode_on_tensor_cores(desc, batch)) return split;
    const size_t tc = decode_tc_workspace(batch, desc);
    return split > tc ? split : tc;
  }
  if (kind == PD_KIND_PREFILL || kind == PD_KIND_MIXED)
    return prefill_layout(batch->batch_size, batch->total_qo, batch->max_qo_len,
                          prefill_tile_heads(desc->num_qo_heads / desc->num_kv_heads))
        .total;
  if (kind == PD_KIND_MIXED_SPLIT) return pd::mixed_split_layout(desc, batch).total;
  return 0;
}

int pd_attn_decode(const pd_attn_desc* desc, const pd_batch* batch, const void* q, const void* k_pool,
                   const void* v_pool, void* o, float* lse, void* workspace, size_t workspace_bytes,
                   int32_t* dev_status, void* stream) {
  int rc = check_attn(desc, batch, false);
  if (rc != PD_OK) return rc;
  if (batch->batch_size == 0) return PD_OK;
  if (q == nullptr || k_pool == nullptr || v_pool == nullptr || o == nullptr || workspace == nullptr)
    return PD_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_pool) || !aligned16(v_pool) || !aligned16(o) || !aligned16(workspace))
    return PD_ERR_INVALID_ARG;
  if (batch->qo_indptr == nullptr && batch->total_qo < batch->batch_size) return PD_ERR_INVALID_ARG;
  if (decode_on_tensor_cores(desc, batch)) {
    // one query row per request at the last position: the bottom-right causal
    // mask admits every key, so the tile runs unmasked (kv_len 0 gives o = 0)
    return run_prefill(desc, batch, 1, 0, q, k_pool, v_pool, o, lse, workspace, workspace_bytes, dev_status,
                       stream);
  }
  const DecodeLayout L = decode_layout_for(desc, batch);
  if (workspace_bytes < L.total) return PD_ERR_WORKSPACE;

  DecodeParams p{};
  p.batch = batch->batch_size;
  p.hq = desc->num_qo_heads;
  p.hkv = desc->num_kv_heads;
  p.head_dim = desc->head_dim;
  p.page_size = desc->page_size;
  p.group = p.hq / p.hkv;
  p.nhd = desc->layout == PD_LAYOUT_NHD;
  p.heads_per_item = decode_heads_per_item(p.group, p.head_dim);
  p.items_per_chunk = p.hq / p.heads_per_item;
  p.total_qo = batch->total_qo;
  p.max_kv_len = batch->max_kv_len;
  p.num_pages = batch->num_pages;
  p.chunk_target = L.chunk_target;
  p.max_chunks = L.max_chunks;
  p.o_dtype = desc->o_dtype;
  p.scale_log2 = scale_of(desc) * kLog2e;
  p.qo_indptr = batch->qo_indptr;
  p.kv_len = batch->kv_len;
  p.page_indptr = batch->page_indptr;
  p.page_indices = batch->page_indices;
  p.q = q;
  p.k_pool = k_pool;
  p.v_pool = v_pool;
  p.o = o;
  p.lse = lse;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  p.hdr = reinterpret_cast<int32_t*>(ws + L.hdr);
  p.req_info = reinterpret_cast<int4*>(ws + L.req_info);
  p.rc_list = reinterpret_cast<int2*>(ws + L.rc_list);
  p.part_o = reinterpret_cast<float*>(ws + L.part_o);
  p.part_lse = reinterpret_cast<float*>(ws + L.part_lse);
  p.status = dev_status;
  return launch_decode(p, desc->kv_dtype, static_cast<cudaStream_t>(stream));
}

int pd_attn_prefill(const pd_attn_desc* desc, const pd_batch* batch, const void* q, const void* k_pool,
                    const void* v_pool, void* o, float* lse, void* workspace, size_t workspace_bytes,
                    int32_t* dev_status, void* stream) {
  int rc = check_attn(desc, batch, true);
  if (rc != PD_OK) return rc;
  rc = prefill_supported(desc->kv_dtype, desc->head_dim, desc->page_size);
  if (rc != PD_OK) return rc;
  if (batch->batch_size == 0 || batch->total_qo == 0) return PD_OK;
  if (q == nullptr || k_pool == nullptr || v_pool == nullptr || o == nullptr || workspace == nullptr)
    return PD_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_pool) || !aligned16(v_pool) || !aligned16(o) || !aligned16(workspace))
    return PD_ERR_INVALID_ARG;
  return pd::run_prefill(desc, batch, batch->max_qo_len, desc->causal, q, k_pool, v_pool, o, lse, workspace,
                         workspace_bytes, dev_status, stream);
}

int pd_attn_mixed(const pd_attn_desc* desc, const pd_batch* batch, const void* q, const void* k_pool,
                  const void* v_pool, void* o, float* lse, void* workspace, size_t workspace_bytes,
                  int32_t* dev_status, void* stream) {
  // One launch of the persistent tensor-core kernel over the whole batch: each
  // decode request (qo_len = 1) is a one-row query tile in the same
  // heaviest-first work list as the prefill tiles, so prefill and decode work
  // share the grid, the TMA pipeline and the MMA/softmax warps.
  return pd_attn_prefill(desc, batch, q, k_pool, v_pool, o, lse, workspace, workspace_bytes, dev_status, stream);
}

namespace {

int check_mla(const pd_mla_desc* d, const pd_batch* b) {
  if (d == nullptr || b == nullptr) return PD_ERR_INVALID_ARG;
  if (d->num_qo_heads <= 0 || d->kv_lora_rank <= 0 || d->rope_dim < 0 || d->page_size <= 0)
    return PD_ERR_INVALID_ARG;
  if (elem_size(d->kv_dtype) == 0 || elem_size(d->o_dtype) == 0) return PD_ERR_INVALID_ARG;
  if (!(d->sm_scale <= 0.f || isfinite(d->sm_scale))) return PD_ERR_INVALID_ARG;
  if (b->batch_size < 0 || b->max_kv_len < 0) return PD_ERR_INVALID_ARG;
  if (b->batch_size > 0) {
    if (b->kv_len == nullptr || b->page_indptr == nullptr || b->page_indices == nullptr) return PD_ERR_INVALID_ARG;
    if (b->num_pages <= 0) return PD_ERR_INVALID_ARG;
  }
  if (mla_pairs() < 1) return PD_ERR_CUDA;
  return mla_supported(d->kv_lora_rank, d->rope_dim, d->kv_dtype, d->num_qo_heads, d->page_size);
}

}  // namespace

size_t pd_mla_workspace_size(const pd_mla_desc* desc, const pd_batch* batch) {
  if (check_mla(desc, batch) != PD_OK) return 0;
  return mla_layout(batch->batch_size, desc->num_qo_heads).total;
}

int pd_mla_decode(const pd_mla_desc* desc, const pd_batch* batch, const void* q, const void* kv_pool, void* o,
                  float* lse, void* workspace, size_t workspace_bytes, int32_t* dev_status, void* stream) {
  const int rc = check_mla(desc, batch);
  if (rc != PD_OK) return rc;
  if (batch->batch_size == 0) return PD_OK;
  if (q == nullptr || kv_pool == nullptr || o == nullptr || workspace == nullptr) return PD_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(kv_pool) || !aligned16(o) || !aligned16(workspace)) return PD_ERR_INVALID_ARG;
  const MlaLayout L = mla_layout(batch->batch_size, desc->num_qo_heads);
  if (workspace_bytes < L.total) return PD_ERR_WORKSPACE;
  MlaParams p{};
  p.batch = batch->batch_size;
  p.hq = desc->num_qo_heads;
  p.page_size = desc->page_size;
  p.num_pages = batch->num_pages;
  p.max_kv_len = batch->max_kv_len;
  p.o_dtype = desc->o_dtype;
  p.pairs = mla_pairs();
  p.max_chunks = L.max_chunks;
  const float scale =
      desc->sm_scale > 0.f ? desc->sm_scale : 1.0f / sqrtf((float)(desc->kv_lora_rank + desc->rope_dim));
  p.scale_log2 = scale * kLog2e;
  p.kv_len = batch->kv_len;
  p.page_indptr = batch->page_indptr;
  p.page_indices = batch->page_indices;
  p.o = o;
  p.lse = lse;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  p.hdr = reinterpret_cast<int32_t*>(ws + L.hdr);
  p.req_info = reinterpret_cast<int4*>(ws + L.req_info);
  p.chunk_list = reinterpret_cast<int2*>(ws + L.chunk_list);
  p.split_list = reinterpret_cast<int32_t*>(ws + L.split_list);
  p.part_lse = reinterpret_cast<float*>(ws + L.part_lse);
  p.part_o = reinterpret_cast<float*>(ws + L.part_o);
  p.status = dev_status;
  return launch_mla(p, q, kv_pool, static_cast<cudaStream_t>(stream));
}

namespace {

int check_kv(const pd_kv_desc* d, const pd_batch* b) {
  if (d == nullptr || b == nullptr) return PD_ERR_INVALID_ARG;
  const int es = elem_size(d->dtype);
  if (es == 0 || d->num_kv_heads <= 0 || d->head_dim <= 0 || d->page_size <= 0 || d->num_layers <= 0)
    return PD_ERR_INVALID_ARG;
  if (d->layout != PD_LAYOUT_HND && d->layout != PD_LAYOUT_NHD) return PD_ERR_INVALID_ARG;
  if ((d->head_dim * es) % 16 != 0) return PD_ERR_UNSUPPORTED;
  if (d->num_layers > 1 && (d->layer_stride_bytes <= 0 || d->layer_stride_bytes % 16 != 0))
    return PD_ERR_INVALID_ARG;
  if (b->batch_size < 0 || b->max_kv_len < 0 || b->total_qo < 0) return PD_ERR_INVALID_ARG;
  if (b->batch_size > 0) {
    if (b->kv_len == nullptr || b->page_indptr == nullptr || b->page_indices == nullptr) return PD_ERR_INVALID_ARG;
    if (b->num_pages <= 0) return PD_ERR_INVALID_ARG;
  }
  return PD_OK;
}

KvCopyParams kv_params(const pd_kv_desc* d, const pd_batch* b, int32_t* status) {
  KvCopyParams p{};
  p.batch = b->batch_size;
  p.hkv = d->num_kv_heads;
  p.head_dim = d->head_dim;
  p.page_size = d->page_size;
  p.num_layers = d->num_layers;
  p.num_pages = b->num_pages;
  p.elem_size = elem_size(d->dtype);
  p.nhd = d->layout == PD_LAYOUT_NHD;
  p.head_begin = 0;
  p.head_count = d->num_kv_heads;
  p.layer_begin = 0;
  p.layer_count = d->num_layers;
  p.max_kv_len = b->max_kv_len;
  p.max_new = b->total_qo;
  p.layer_stride = d->layer_stride_bytes;
  p.new_indptr = b->qo_indptr;
  p.kv_len = b->kv_len;
  p.page_indptr = b->page_indptr;
  p.page_indices = b->page_indices;
  p.status = status;
  return p;
}

}  // namespace

int pd_kv_append(const pd_kv_desc* desc, const pd_batch* batch, const void* k_new, const void* v_new,
                 void* k_pool, void* v_pool, int32_t* dev_status, void* stream) {
  int rc = check_kv(desc, batch);
  if (rc != PD_OK) return rc;
  if (desc->num_layers != 1) return PD_ERR_INVALID_ARG;
  if (batch->batch_size == 0 || batch->total_qo == 0) return PD_OK;
  if (batch->qo_indptr == nullptr || k_new == nullptr || v_new == nullptr || k_pool == nullptr || v_pool == nullptr)
    return PD_ERR_INVALID_ARG;
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_pool) || !aligned16(v_pool)) return PD_ERR_INVALID_ARG;
  KvCopyParams p = kv_params(desc, batch, dev_status);
  p.src = k_new;
  p.src2 = v_new;
  p.dst = k_pool;
  p.dst2 = v_pool;
  return launch_kv_append(p, static_cast<cudaStream_t>(stream));
}

int pd_kv_pack_heads(const pd_kv_desc* desc, const pd_batch* batch, int32_t head_begin, int32_t head_count,
                     const void* k_pool, const void* v_pool, void* dst, size_t dst_bytes,
                     const int64_t* dst_offsets, int32_t* dev_status, void* stream) {
  int rc = check_kv(desc, batch);
  if (rc != PD_OK) return rc;
  if (head_begin < 0 || head_count < 1 || head_count > desc->num_kv_heads - head_begin) return PD_ERR_INVALID_ARG;
  if (batch->batch_size == 0) return PD_OK;
  if (k_pool == nullptr || v_pool == nullptr || dst == nullptr || dst_offsets == nullptr) return PD_ERR_INVALID_ARG;
  if (!aligned16(k_pool) || !aligned16(v_pool) || !aligned16(dst)) return PD_ERR_INVALID_ARG;
  KvCopyParams p = kv_params(desc, batch, dev_status);
  p.head_begin = head_begin;
  p.head_count = head_count;
  p.src = k_pool;
  p.src2 = v_pool;
  p.dst = dst;
  p.offsets = dst_offsets;
  p.buf_bytes = (int64_t)dst_bytes;
  return launch_kv_pack(p, static_cast<cudaStream_t>(stream));
}

int pd_kv_pack_layers(const pd_kv_desc* desc, const pd_batch* batch, int32_t layer_begin, int32_t layer_count,
                      const void* k_pool, const void* v_pool, void* dst, size_t dst_bytes,
                      const int64_t* dst_offsets, int32_t* dev_status, void* stream) {
  int rc = check_kv(desc, batch);
  if (rc != PD_OK) return rc;
  if (layer_begin < 0 || layer_count < 1 || layer_count > desc->num_layers - layer_begin) return PD_ERR_INVALID_ARG;
  if (batch->batch_size == 0) return PD_OK;
  if (k_pool == nullptr || v_pool == nullptr || dst == nullptr || dst_offsets == nullptr) return PD_ERR_INVALID_ARG;
  if (!aligned16(k_pool) || !aligned16(v_pool) || !aligned16(dst)) return PD_ERR_INVALID_ARG;
  KvCopyParams p = kv_params(desc, batch, dev_status);
  p.layer_begin = layer_begin;
  p.layer_count = layer_count;
  p.src = k_pool;
  p.src2 = v_pool;
  p.dst = dst;
  p.offsets = dst_offsets;
  p.buf_bytes = (int64_t)dst_bytes;
  return launch_kv_pack(p, static_cast<cudaStream_t>(stream));
}

int pd_kv_pack(const pd_kv_desc* desc, const pd_batch* batch, const void* k_pool, const void* v_pool, void* dst,
               size_t dst_bytes, const int64_t* dst_offsets, int32_t* dev_status, void* stream) {
  if (desc == nullptr) return PD_ERR_INVALID_ARG;
  return pd_kv_pack_heads(desc, batch, 0, desc->num_kv_heads, k_pool, v_pool, dst, dst_bytes, dst_offsets,
                          dev_status, stream);
}

int pd_kv_unpack_heads(const pd_kv_desc* desc, const pd_batch* batch, int32_t head_begin, int32_t head_count,
                       const void* src, size_t src_bytes, const int64_t* src_offsets, void* k_pool, void* v_pool,
                       int32_t* dev_status, void* stream) {
  int rc = check_kv(desc, batch);
  if (rc != PD_OK) return rc;
  if (head_begin < 0 || head_count < 1 || head_count > desc->num_kv_heads - head_begin) return PD_ERR_INVALID_ARG;
  if (batch->batch_size == 0) return PD_OK;
  if (k_pool == nullptr || v_pool == nullptr || src == nullptr || src_offsets == nullptr) return PD_ERR_INVALID_ARG;
  if (!aligned16(k_pool) || !aligned16(v_pool) || !aligned16(src)) return PD_ERR_INVALID_ARG;
  KvCopyParams p = kv_params(desc, batch, dev_status);
  p.head_begin = head_begin;
  p.head_count = head_count;
  p.src = src;
  p.dst = k_pool;
  p.dst2 = v_pool;
  p.offsets = src_offsets;
  p.buf_bytes = (int64_t)src_bytes;
  return launch_kv_unpack(p, static_cast<cudaStream_t>(stream));
}

int pd_kv_unpack(const pd_kv_desc* desc, const pd_batch* batch, const void* src, size_t src_bytes,
                 const int64_t* src_offsets, void* k_pool, void* v_pool, int32_t* dev_status, void* stream) {
  if (desc == nullptr) return PD_ERR_INVALID_ARG;
  return pd_kv_unpack_heads(desc, batch, 0, desc->num_kv_heads, src, src_bytes, src_offsets, k_pool, v_pool,
                            dev_status, stream);
}

}  // extern "C"
