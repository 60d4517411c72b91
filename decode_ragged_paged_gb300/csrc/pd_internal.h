// pd_internal.h -- launch parameters and launcher declarations shared between
// the C-ABI layer (pd_api.cu) and the kernel translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/pd.h"

namespace pd {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// ------------------------------------------------------------------ decode
// Workspace of the split-KV decode (all offsets 256-byte aligned):
//   hdr       int32[64]            hdr[0] = work items, hdr[1] = chunks in total
//   req_info  int4[B]              {first chunk, chunks, chunk length, q row or -1 if skipped}
//   rc_list   int2[max_chunks]     (request, chunk index) of every chunk, longest chunks first
//   part_o    float[max_chunks][Hq][D]   normalised partial outputs
//   part_lse  float[max_chunks][Hq]      their log2-sum-exp2 of scaled scores
struct DecodeParams {
  int32_t batch, hq, hkv, head_dim, page_size, group, heads_per_item, items_per_chunk;
  int32_t nhd;  // pools [page][slot][head][dim] instead of [page][head][slot][dim]
  int32_t total_qo, max_kv_len, num_pages, chunk_target, max_chunks;
  int32_t o_dtype;
  float scale_log2;  // softmax scale times log2(e)
  const int32_t* qo_indptr;  // may be null: row r = request r
  const int32_t* kv_len;
  const int32_t* page_indptr;
  const int32_t* page_indices;
  const void* q;
  const void* k_pool;
  const void* v_pool;
  void* o;
  float* lse;
  int32_t* hdr;
  int4* req_info;
  int2* rc_list;
  float* part_o;
  float* part_lse;
  int32_t* status;
};

struct DecodeLayout {
  size_t hdr, req_info, rc_list, part_o, part_lse, total;
  int32_t chunk_target, max_chunks;
};

// Chunk length and workspace layout of a decode over `batch` requests of at
// most max_kv_len tokens; `sm_count` sizes the split.
DecodeLayout decode_layout(int32_t batch, int32_t hq, int32_t head_dim, int32_t max_kv_len,
                           int32_t items_per_chunk, int32_t sm_count);

// Heads of one group processed together by a decode work item.
int32_t decode_heads_per_item(int32_t group, int32_t head_dim);

// Plans and runs a decode. Returns a pd_status.
int launch_decode(DecodeParams& p, int32_t kv_dtype, cudaStream_t stream);

// ----------------------------------------------------------------- prefill
// Workspace of the tensor-core prefill (offsets 256-byte aligned):
//   hdr      int32[64]     hdr[0] = work items (q tiles x query heads)
//   rq_list  int2[max_rq]  (request, q tile) ordered by decreasing KV-tile count
struct PrefillParams {
  int32_t batch, hq, hkv, group, page_size, num_pages, total_qo, max_qo_len, max_kv_len, causal, o_dtype;
  int32_t max_rq;
  // GQA packing: a 128-row tile holds tile_rows query rows x tile_heads query
  // heads of one KV head (tile_heads = the group, or 1); items per q tile =
  // item_heads = hq / tile_heads
  int32_t tile_heads, tile_rows, item_heads;
  int32_t nhd;       // pools [page][slot][head][dim] instead of [page][head][slot][dim]
  float scale_log2;  // softmax scale times log2(e)
  const int32_t* qo_indptr;
  const int32_t* kv_len;
  const int32_t* page_indptr;
  const int32_t* page_indices;
  void* o;
  float* lse;
  int32_t* hdr;
  int2* rq_list;
  int32_t* status;
};

struct PrefillLayout {
  size_t hdr, rq_list, total;
  int32_t max_rq;
};

// Query heads a prefill tile packs for this group size (the group when it
// divides 128, else 1).
int32_t prefill_tile_heads(int32_t group);
PrefillLayout prefill_layout(int32_t batch, int32_t total_qo, int32_t max_qo_len, int32_t tile_heads);

// Workspace of pd_attn_mixed_split: the prefill part at 0, the decode part at
// `decode` (bytes).
struct MixedSplitLayout {
  size_t decode, total;
};
MixedSplitLayout mixed_split_layout(const pd_attn_desc* d, const pd_batch* b);

// Checks what the tensor-core prefill supports; returns a pd_status.
int prefill_supported(int32_t kv_dtype, int32_t head_dim, int32_t page_size);

// Plans and runs a prefill over bf16 q / pools. Returns a pd_status.
int launch_prefill(PrefillParams& p, const void* q, const void* k_pool, const void* v_pool, cudaStream_t stream);

// --------------------------------------------------------------- KV copies
struct KvCopyParams {
  int32_t batch, hkv, head_dim, page_size, num_layers, num_pages, elem_size;
  int32_t head_begin, head_count;    // pack / unpack: pool heads [head_begin, head_begin + head_count)
  int32_t layer_begin, layer_count;  // pack: layers [layer_begin, layer_begin + layer_count) of num_layers
  int32_t max_kv_len, max_new;
  int32_t nhd;                       // pools [page][slot][head][dim] instead of [page][head][slot][dim]
  int64_t layer_stride;
  const int32_t* new_indptr;   // append only
  const int32_t* kv_len;
  const int32_t* page_indptr;
  const int32_t* page_indices;
  const void* src;             // append: k_new; pack: k pool; unpack: packed buffer
  const void* src2;            // append: v_new; pack: v pool
  void* dst;                   // append: k pool; pack: packed buffer; unpack: k pool
  void* dst2;                  // append: v pool; unpack: v pool
  const int64_t* offsets;      // pack: dst offsets; unpack: src offsets
  int64_t buf_bytes;           // size of the packed buffer
  int32_t* status;
};

int launch_kv_append(const KvCopyParams& p, cudaStream_t stream);
int launch_kv_pack(const KvCopyParams& p, cudaStream_t stream);
int launch_kv_unpack(const KvCopyParams& p, cudaStream_t stream);

// -------------------------------------------------------------- MLA decode
// Workspace (offsets 256-byte aligned):
//   hdr        int32[64]   hdr[0] = chunks listed, hdr[1] = chunk length
//   req_info   int4[B]     {first chunk, chunks, kv_len or -1 if invalid, 0}
//   chunk_list int2[max_chunks]  (request, chunk) longest first
//   part_lse   float[max_chunks][Hq]        log2-sum-exp2 of scaled scores
//   part_o     float[max_chunks][Hq][512]   normalised partial outputs
struct MlaParams {
  int32_t batch, hq, page_size, num_pages, max_kv_len, o_dtype, pairs, max_chunks;
  float scale_log2;  // softmax scale times log2(e)
  const int32_t* kv_len;
  const int32_t* page_indptr;
  const int32_t* page_indices;
  void* o;
  float* lse;
  int32_t* hdr;
  int4* req_info;
  int2* chunk_list;
  int32_t* split_list;  // requests cut into several chunks (hdr[2] of them)
  float* part_lse;
  float* part_o;
  int32_t* status;
};

struct MlaLayout {
  size_t hdr, req_info, chunk_list, split_list, part_lse, part_o, total;
  int32_t max_chunks;
};

// What the MLA kernel supports (latent 512 + rope 64, bf16, 1..128 heads,
// page size a power of two in [16, 256]); returns a pd_status.
int mla_supported(int32_t d_c, int32_t d_r, int32_t dtype, int32_t hq, int32_t page_size);
// CTA pairs of the persistent MLA grid (one CTA per SM).
int mla_pairs();
MlaLayout mla_layout(int32_t batch, int32_t hq);
int launch_mla(MlaParams& p, const void* q, const void* kv_pool, cudaStream_t stream);

// ------------------------------------------------------------ tensor maps
bool make_pool_map(CUtensorMap* map, const void* pool, int32_t dtype, int32_t num_pages, int32_t hkv,
                   int32_t page_size, int32_t head_dim, int32_t box_cols, int32_t box_rows, bool swizzle128,
                   bool nhd = false);
bool make_rows_map(CUtensorMap* map, const void* base, int32_t dtype, int32_t total, int32_t hq, int32_t head_dim,
                   int32_t box_cols, int32_t box_rows, bool swizzle128, int32_t box_heads = 1);

// ------------------------------------------------------------------- misc
// SMs of the device, or of the SM partition (green context) the calling thread
// launches into while partition_sms() is set.
int device_sm_count();
// Set (thread-local) while a call launches into an SM partition: grids are
// sized for the partition's SMs, and the kernels' one-time attribute setup,
// which is per context, runs again.
int& partition_sms();

// Events of pd_profile_events() (per host thread); recorded around main kernels.
struct ProfileEvents {
  cudaEvent_t start = nullptr, stop = nullptr;
};
ProfileEvents& profile_events();
// Name of the main kernel the last call of this host thread launched.
const char*& last_kernel();
inline void profile_begin(cudaStream_t s) {
  if (profile_events().start) cudaEventRecord(profile_events().start, s);
}
inline void profile_end(cudaStream_t s) {
  if (profile_events().stop) cudaEventRecord(profile_events().stop, s);
}

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

}  // namespace pd
