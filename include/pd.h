/*
 * pd.h -- C ABI of the paged ragged-attention and KV-handoff library for
 * NVIDIA GB300 (sm_103a).
 *
 * The library implements the single-GPU hot path behind disaggregated
 * prefill/decode serving described in Perplexity, "Disaggregated prefill and
 * decode" (2025):
 *   - attention over a paged KV cache for ragged batches of decode requests
 *     (qo_len = 1, long kv_len), causal prefill requests (large qo_len) and
 *     mixed batches of both (section "Prefill vs Decode performance");
 *   - appending a layer's new K/V entries into their pages, after which that
 *     layer's pages may be shipped (section "KV Messenger");
 *   - packing a finished prefill's pages into a contiguous buffer and unpacking
 *     them into a decoder's pool with a different page size and page table
 *     (section "Sharded KV cache transfers").
 *
 * Conventions shared by every call
 * --------------------------------
 * Memory. Every pointer argument named "device" points to GPU memory owned by
 * the caller; the library allocates nothing per call and keeps no pointer after
 * a call returns. All work is enqueued on `stream` (a cudaStream_t; NULL is the
 * legacy default stream) and runs asynchronously: buffers must stay alive until
 * the stream has passed the call. Descriptor structs are read on the host
 * during the call only.
 *
 * Pool layouts (from the post's figure on NHD and HND KV-cache layouts):
 *   PD_LAYOUT_HND, "head before token" (the default): a pool is
 *     [num_pages][num_kv_heads][page_size][head_dim], row-major, so each head's
 *     slice of a page is one contiguous run of page_size * head_dim elements;
 *   PD_LAYOUT_NHD, "token before head": a pool is
 *     [num_pages][page_size][num_kv_heads][head_dim], row-major, so each token's
 *     heads are one contiguous run and a head's slots are num_kv_heads rows
 *     apart.
 * K and V live in two pools of the same layout that share one page table.
 * Pools must be 16-byte aligned.
 *
 * Page table (CSR): request r owns pages
 * page_indices[page_indptr[r] .. page_indptr[r+1]); logical token t of r sits in
 * page page_indices[page_indptr[r] + t / page_size], slot t % page_size.
 *
 * Ragged rows: q and o are [total_qo][num_qo_heads][head_dim]; the rows of
 * request r are qo_indptr[r] .. qo_indptr[r+1]. kv_len[r] counts all of r's
 * cached tokens including the new ones, so the new rows are the last qo_len
 * positions (bottom-right causal alignment: row i may attend keys
 * j <= kv_len - qo_len + i).
 *
 * Grouped-query attention (section "Qwen3-Coder"): num_kv_heads divides
 * num_qo_heads; query head h reads KV head h / (num_qo_heads / num_kv_heads).
 *
 * Errors. Host-side checks run first; on failure a negative pd_status is
 * returned and nothing is enqueued. Checks of device-resident data (indptr
 * monotonicity, lengths against the host bounds, page ids against num_pages)
 * run on the GPU: a request that fails one is skipped (its outputs are left
 * unspecified) and, when `dev_status` is not NULL, the first failure's
 * pd_device_status code is stored there with an atomic compare-and-swap from 0
 * (the caller zeroes it and reads it back when it wants to know). No call
 * faults the GPU on bad table contents; every wait inside a kernel is bounded
 * and reports PD_DEV_TIMEOUT instead of hanging.
 *
 * Thread safety: calls are stateless apart from per-device launch attributes
 * cached on first use; distinct streams may call concurrently with distinct
 * workspaces.
 */
#ifndef PD_H_
#define PD_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define PD_API __attribute__((visibility("default")))
#else
#define PD_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Return codes of every entry point. */
typedef enum {
  PD_OK = 0,
  PD_ERR_INVALID_ARG = -1, /* null pointer, negative or inconsistent host-side size */
  PD_ERR_UNSUPPORTED = -2, /* valid request the library does not implement */
  PD_ERR_WORKSPACE = -3,   /* workspace smaller than pd_attn_workspace_size() */
  PD_ERR_CUDA = -4,        /* a CUDA runtime call or kernel launch failed */
  PD_ERR_TIMEOUT = -5      /* a host-side wait (the layer messenger) ran out */
} pd_status;

/* Codes stored into *dev_status by the kernels (first failure wins). */
typedef enum {
  PD_DEV_OK = 0,
  PD_DEV_BAD_INDPTR = 1,     /* qo_indptr / page_indptr decreasing or past total_qo */
  PD_DEV_BAD_LENGTH = 2,     /* kv_len < 0, > max_kv_len, qo_len > max_qo_len, or causal qo_len > kv_len */
  PD_DEV_BAD_PAGE_TABLE = 3, /* fewer pages than ceil(kv_len / page_size), or a page id outside [0, num_pages) */
  PD_DEV_NOT_DECODE = 4,     /* pd_attn_decode given a request with qo_len != 1 */
  PD_DEV_TIMEOUT = 5,        /* a bounded wait inside a kernel ran out; the kernel returned early */
  PD_DEV_BAD_OFFSET = 6      /* a pack / unpack block misaligned or outside the packed buffer */
} pd_device_status;

typedef enum { PD_F32 = 0, PD_BF16 = 1 } pd_dtype;

typedef enum { PD_LAYOUT_HND = 0, PD_LAYOUT_NHD = 1 } pd_layout;

typedef enum { PD_KIND_DECODE = 0, PD_KIND_PREFILL = 1, PD_KIND_MIXED = 2, PD_KIND_MIXED_SPLIT = 3 } pd_attn_kind;

/* Shape and numerics of one attention call. */
typedef struct {
  int32_t num_qo_heads; /* Hq */
  int32_t num_kv_heads; /* Hkv; must divide Hq */
  int32_t head_dim;     /* D: 64 or 128 */
  int32_t page_size;    /* P: tokens per page, >= 1 */
  int32_t kv_dtype;     /* pd_dtype of q, k_pool and v_pool */
  int32_t o_dtype;      /* pd_dtype of o */
  int32_t layout;       /* pd_layout of k_pool and v_pool */
  int32_t causal;       /* 1: bottom-right causal mask; 0: every row sees all kv_len keys */
  float sm_scale;       /* softmax scale; <= 0 selects 1/sqrt(head_dim) */
} pd_attn_desc;

/* A ragged batch. Device arrays are int32. */
typedef struct {
  int32_t batch_size;          /* B >= 0 */
  const int32_t *qo_indptr;    /* device [B+1]; NULL in pd_attn_decode means row r = request r */
  const int32_t *kv_len;       /* device [B] */
  const int32_t *page_indptr;  /* device [B+1] */
  const int32_t *page_indices; /* device [page_indptr[B]] */
  int32_t num_pages;           /* pages in each pool (bound for page ids) */
  int32_t total_qo;            /* host: rows of q and o, qo_indptr[B] */
  int32_t max_qo_len;          /* host: bound on every qo_len (sizes grids and workspace) */
  int32_t max_kv_len;          /* host: bound on every kv_len (sizes grids and workspace) */
} pd_batch;

/* Shape of KV pools for append / pack / unpack. */
typedef struct {
  int32_t num_kv_heads;       /* Hkv */
  int32_t head_dim;           /* D; head_dim * element size must be a multiple of 16 bytes */
  int32_t page_size;          /* P >= 1 */
  int32_t dtype;              /* pd_dtype of the pools */
  int32_t layout;             /* pd_layout of the pools */
  int32_t num_layers;         /* L >= 1 (append: the layer count is 1) */
  int64_t layer_stride_bytes; /* bytes from layer l's pool to layer l+1's; same for K and V */
} pd_kv_desc;

/*
 * Bytes of device workspace an attention call of `kind` needs for this
 * descriptor and the batch's host-side sizes (batch_size, total_qo, max_qo_len,
 * max_kv_len). 16-byte alignment required. Returns 0 when the arguments are
 * invalid. The workspace carries the per-call plan and the split-KV partial
 * results; it needs no initialisation and may be reused once a previous call
 * using it has finished on the GPU.
 */
PD_API size_t pd_attn_workspace_size(const pd_attn_desc *desc, const pd_batch *batch, int32_t kind);

/*
 * Decode attention (section "Prefill vs Decode performance": qo_len = 1 per
 * request, attention parallelised over requests and over kv_len).
 *   q        device [B][Hq][D] (kv_dtype)
 *   k_pool   device [num_pages][Hkv][P][D] (kv_dtype), v_pool likewise
 *   o        device [B][Hq][D] (o_dtype): softmax(q K^T * scale) V
 *   lse      device [B][Hq] fp32, natural-log log-sum-exp of the scaled scores;
 *            may be NULL. A request with kv_len = 0 gives o = 0, lse = -inf.
 *   workspace / workspace_bytes: see pd_attn_workspace_size(kind = PD_KIND_DECODE)
 *   dev_status: device int32 or NULL (see "Errors" above)
 * The KV axis is split into chunks processed by separate CTAs; the partial
 * results are merged by log-sum-exp. Supported: kv_dtype f32 or bf16, D 64 or
 * 128, any page size, any group size Hq/Hkv. The causal flag is irrelevant for
 * one row per request. A large grouped-query batch (bf16, D 128, page size a
 * power of two >= 8, group 2..128 dividing 128, no qo_indptr, and at least
 * four (request, KV head) pairs per SM) instead runs on the tensor-core kernel
 * of pd_attn_prefill with the group's query heads packed into one tile, which
 * reads each KV tile once per group without splitting; the workspace size
 * query covers both. Results agree within the stated tolerances either way.
 */
PD_API int pd_attn_decode(const pd_attn_desc *desc, const pd_batch *batch, const void *q,
                   const void *k_pool, const void *v_pool, void *o, float *lse,
                   void *workspace, size_t workspace_bytes, int32_t *dev_status, void *stream);

/*
 * Decode attention without a caller-provided workspace. (The pages have no
 * counterpart for this call; it exists for callers of this library.)
 * For callers that cannot allocate device memory for a workspace: for example
 * a C host program that only receives tensors from a framework owning every
 * device allocation, or a loop where calling cudaMalloc is not allowed.
 * Arguments and results are those of pd_attn_decode minus the workspace; the
 * scratch space is a fixed array of 32 MiB in device memory defined by the
 * library, reserved on every GPU where it is first used until the process
 * exits. A batch whose plan and split-KV partials need more than that returns
 * PD_ERR_WORKSPACE and launches nothing. Batches that take the tensor-core
 * kernel use only a few KiB of the array (a header and the work list); the
 * split-KV kernel keeps its partial results there, which for 128 requests with
 * kv_len up to 4096 and 32 query heads of 128 would take about 17 MiB. All
 * calls on one GPU share the array: calls whose work overlaps on the GPU (e.g.
 * on two streams) race and must be serialised by the caller. The first call on
 * each GPU looks up the array's device address through the CUDA runtime (a
 * one-time step that may load the library's device code) and keeps it for the
 * life of the process; make that first call outside any stream capture, and do
 * not use this call on a device after cudaDeviceReset there (the kept address
 * belonged to the context that the reset destroyed).
 */
PD_API int pd_attn_decode_static(const pd_attn_desc *desc, const pd_batch *batch, const void *q,
                                 const void *k_pool, const void *v_pool, void *o, float *lse,
                                 int32_t *dev_status, void *stream);

/*
 * Prefill attention: any qo_len <= kv_len per request, causal or not (section
 * "Prefill vs Decode performance": prefill requests bring many tokens and are
 * compute bound). Arguments as pd_attn_decode with q, o [total_qo][Hq][D]
 * and lse [total_qo][Hq]. Supported: kv_dtype bf16, D 128; tensor-core tiles
 * of 128 query rows.
 */
PD_API int pd_attn_prefill(const pd_attn_desc *desc, const pd_batch *batch, const void *q,
                    const void *k_pool, const void *v_pool, void *o, float *lse,
                    void *workspace, size_t workspace_bytes, int32_t *dev_status, void *stream);

/*
 * Mixed batch in one launch (section "Prefill vs Decode performance": mixing
 * prefill into decode batches). Prefill requests (qo_len > 1) and decode
 * requests (qo_len = 1) go through one persistent tensor-core kernel: every
 * request's query rows are cut into 128-row tiles (a decode request is a
 * one-row tile) and all tiles form one work list ordered by decreasing KV
 * length, so both kinds of work share the grid and the TMA/MMA pipeline.
 * Arguments, layouts and support as pd_attn_prefill; the workspace is that of
 * pd_attn_workspace_size(kind = PD_KIND_MIXED).
 */
PD_API int pd_attn_mixed(const pd_attn_desc *desc, const pd_batch *batch, const void *q,
                  const void *k_pool, const void *v_pool, void *o, float *lse,
                  void *workspace, size_t workspace_bytes, int32_t *dev_status, void *stream);

/*
 * Mixed batch whose prefill and decode requests the caller has separated, as
 * a serving loop that piggybacks prefill chunks on a decode batch knows them
 * (section "Prefill vs Decode performance"): requests [0, num_prefill) are
 * prefill requests (any qo_len), requests [num_prefill, B) decode requests
 * (qo_len = 1; any other length is reported as PD_DEV_NOT_DECODE). The two
 * parts run at the same time on disjoint sets of SMs (green contexts): the
 * prefill part on the tensor-core kernel over prefill_sms SMs (0: sized from
 * the batch's host-side bounds; rounded to the partition granularity of 8),
 * the decode part on the split-KV kernel over the rest. The call orders both
 * after the work already queued on `stream` and makes `stream` wait for both.
 * Where green contexts cannot be created, one part is empty, or a CUDA tool
 * is injected into the process (profilers and sanitizers, which may not
 * follow launches into green contexts; detected from the variables they set in
 * the environment: CUDA_INJECTION64_PATH or Nsight's injection variables), it
 * runs as pd_attn_mixed on `stream`; pd_last_kernel() then names
 * prefill_kernel.
 * Arguments and layouts as pd_attn_mixed; batch->qo_indptr is required; the
 * workspace is that of pd_attn_workspace_size(kind = PD_KIND_MIXED_SPLIT).
 * Host-side state: one pair of green contexts with a stream and two events
 * each per device and partition size (at most one pair per multiple of 8
 * SMs), created on first use and kept for the life of the process (not valid
 * after cudaDeviceReset); calls on one device are serialised on the host while
 * they enqueue. The parts run on the green contexts' own streams, so the call
 * cannot be recorded by stream capture into a CUDA graph on `stream`.
 */
PD_API int pd_attn_mixed_split(const pd_attn_desc *desc, const pd_batch *batch, int32_t num_prefill,
                               int32_t prefill_sms, const void *q, const void *k_pool, const void *v_pool,
                               void *o, float *lse, void *workspace, size_t workspace_bytes,
                               int32_t *dev_status, void *stream);

/*
 * MLA decode (section "Disaggregated Deployments", "DeepSeek-R1": multi-head
 * latent attention compresses the KV heads of a token into one latent vector
 * that every query head reads, so the cache holds one row per token and is
 * never split by head). With the up-projections folded into q and o (MLA's
 * published decode form), token j's stored row is
 * c_j = [c_j^kv (kv_lora_rank values) | k_j^rope (rope_dim values)] and, for
 * request r and query head h:
 *   s_j = sm_scale * <q[r][h], c_j>                 (all kv_lora_rank + rope_dim values)
 *   o[r][h] = sum_j softmax(s)_j * c_j^kv           (the first kv_lora_rank values)
 *   lse[r][h] = log sum_j exp(s_j)                  (natural log; -inf when kv_len = 0)
 * Layouts (row-major, device, 16-byte aligned):
 *   q        [batch][num_qo_heads][kv_lora_rank + rope_dim]
 *   kv_pool  [num_pages][page_size][kv_lora_rank + rope_dim]   one row per token
 *   o        [batch][num_qo_heads][kv_lora_rank] (o_dtype); lse fp32 [batch][num_qo_heads] or NULL
 * One query row per request (row r = request r; the batch's qo_indptr is
 * ignored); kv_len, page_indptr and page_indices as for attention. Supported:
 * kv_lora_rank 512, rope_dim 64, bf16 q and pool, 1..128 query heads, page_size
 * a power of two in [16, 256]; otherwise PD_ERR_UNSUPPORTED. Invalid requests
 * are skipped and reported through dev_status as for attention.
 */
typedef struct {
  int32_t num_qo_heads; /* Hq: query heads reading the latent row, 1..128 */
  int32_t kv_lora_rank; /* latent (value) width: 512 */
  int32_t rope_dim;     /* rope width, scores only: 64 */
  int32_t page_size;    /* tokens per page */
  int32_t kv_dtype;     /* pd_dtype of q and kv_pool: PD_BF16 */
  int32_t o_dtype;      /* pd_dtype of o */
  float sm_scale;       /* softmax scale; <= 0 selects 1/sqrt(kv_lora_rank + rope_dim) */
} pd_mla_desc;

/* Bytes of device workspace pd_mla_decode needs (0 for an invalid descriptor). */
PD_API size_t pd_mla_workspace_size(const pd_mla_desc *desc, const pd_batch *batch);

PD_API int pd_mla_decode(const pd_mla_desc *desc, const pd_batch *batch, const void *q, const void *kv_pool,
                         void *o, float *lse, void *workspace, size_t workspace_bytes, int32_t *dev_status,
                         void *stream);

/*
 * KV append (section "KV Messenger": page copies of a layer start once the
 * model has appended that layer's KV entries). The batch's qo_indptr counts
 * the new tokens: request r brings n_r = qo_indptr[r+1] - qo_indptr[r] rows of
 * k_new / v_new ([total_qo][Hkv][D], device) that land at logical positions
 * kv_len[r] - n_r .. kv_len[r] - 1 of its pages in k_pool / v_pool (device,
 * written in place). Bit-exact copy. desc->num_layers must be 1.
 */
PD_API int pd_kv_append(const pd_kv_desc *desc, const pd_batch *batch, const void *k_new,
                 const void *v_new, void *k_pool, void *v_pool, int32_t *dev_status,
                 void *stream);

/*
 * KV pack (sections "KV Messenger" and "Sharded KV cache transfers": a
 * finished prefill's pages leave the prefiller). For every request r the
 * kv_len[r] tokens of every layer are gathered into a contiguous block at
 * dst + dst_offsets[r] bytes, laid out [L][2 (K, V)][Hkv][kv_len[r]][D] for
 * either pool layout (so an HND pool can hand off to an NHD pool); with the HND
 * layout each (page, head) slice is one contiguous run on both sides, with NHD
 * the pool side is read one head_dim row per token.
 * Layer l's pools start at k_pool / v_pool + l * layer_stride_bytes (device).
 * dst_offsets: device int64 [B], 16-byte multiples; dst_bytes: size of dst. A
 * request whose block would not fit inside dst is skipped and reported
 * (PD_DEV_BAD_OFFSET). Bit-exact copy. The batch's qo_indptr is ignored.
 */
PD_API int pd_kv_pack(const pd_kv_desc *desc, const pd_batch *batch, const void *k_pool,
                      const void *v_pool, void *dst, size_t dst_bytes, const int64_t *dst_offsets,
                      int32_t *dev_status, void *stream);

/*
 * KV unpack: the inverse of pd_kv_pack into a pool with its own page size and
 * page table (section "Sharded KV cache transfers": pages are split or rebuilt
 * when the two sides differ). Only slots of tokens t < kv_len[r] are written.
 * src_bytes bounds the blocks read from src as dst_bytes does for pd_kv_pack.
 */
PD_API int pd_kv_unpack(const pd_kv_desc *desc, const pd_batch *batch, const void *src,
                        size_t src_bytes, const int64_t *src_offsets, void *k_pool, void *v_pool,
                        int32_t *dev_status, void *stream);

/*
 * Head-range forms of pack and unpack (section "Sharded KV cache transfers":
 * when prefiller and decoder shard the KV heads differently, pages are split or
 * rebuilt by the ratio of the slices). desc->num_kv_heads is the pool's head
 * count; the call moves pool heads [head_begin, head_begin + head_count), and
 * each request's block holds those heads only:
 * [L][2 (K, V)][head_count][kv_len[r]][D]. Example: two prefiller shards with
 * 20 heads each pack their own pools; the decoder unpacks the two blocks into
 * one 40-head pool with head_begin 0 and 20. pd_kv_pack / pd_kv_unpack are the
 * full range. head_begin < 0, head_count < 1 or a range past the pool's heads
 * return PD_ERR_INVALID_ARG. Other arguments, checks and errors as pd_kv_pack /
 * pd_kv_unpack.
 */
PD_API int pd_kv_pack_heads(const pd_kv_desc *desc, const pd_batch *batch, int32_t head_begin,
                            int32_t head_count, const void *k_pool, const void *v_pool, void *dst,
                            size_t dst_bytes, const int64_t *dst_offsets, int32_t *dev_status,
                            void *stream);
PD_API int pd_kv_unpack_heads(const pd_kv_desc *desc, const pd_batch *batch, int32_t head_begin,
                              int32_t head_count, const void *src, size_t src_bytes,
                              const int64_t *src_offsets, void *k_pool, void *v_pool,
                              int32_t *dev_status, void *stream);

/*
 * Layer range of pd_kv_pack (section "KV Messenger": a layer's page copies
 * start as soon as the model has appended that layer's KV entries). Packs
 * layers [layer_begin, layer_begin + layer_count) of every request into the
 * same places of its [L][2][Hkv][kv_len][D] block as the full pack would, with
 * L = desc->num_layers; k_pool / v_pool point at layer 0's pools. A range
 * outside [0, L) returns PD_ERR_INVALID_ARG; otherwise as pd_kv_pack.
 */
PD_API int pd_kv_pack_layers(const pd_kv_desc *desc, const pd_batch *batch, int32_t layer_begin,
                             int32_t layer_count, const void *k_pool, const void *v_pool, void *dst,
                             size_t dst_bytes, const int64_t *dst_offsets, int32_t *dev_status,
                             void *stream);

/*
 * Layer-streamed handoff (section "KV Messenger": a polling thread watches a
 * counter that the GPU advances after each layer; the step stays capturable in
 * a CUDA graph).
 *
 * pd_counter_alloc: one 32-bit word of mapped pinned host memory, set to 0;
 * host_word is its host address, device_word the address kernels write. Freed
 * by pd_counter_free(host_word).
 *
 * pd_layer_signal: enqueues on `stream` a one-thread kernel that stores
 * `value` to device_word with a system-scope release store once every earlier
 * kernel on the stream has completed. A model signals value l + 1 after
 * appending layer l. The call is a kernel launch, so it can be captured.
 *
 * pd_messenger_start_pack: starts a host thread that, for each layer l of
 * desc->num_layers in order, waits until *host_word > l (at most timeout_ms,
 * counted from when it starts waiting for that layer), then enqueues
 * pd_kv_pack_layers(l, 1) with the given arguments on `stream` (the
 * messenger's own stream; the caller's model runs on another). Descriptor
 * structs are copied; buffers must stay alive until the packs have run.
 * Returns PD_OK and the handle in *out, or PD_ERR_INVALID_ARG (null
 * arguments, timeout_ms <= 0) and nothing started.
 *
 * pd_messenger_join: waits for the thread and frees the handle. Returns PD_OK
 * when every layer's pack was enqueued; PD_ERR_TIMEOUT when a layer's signal
 * did not arrive in time; or the error of a failed pd_kv_pack_layers. Layers
 * enqueued before the failure are reported in *layers_sent (may be NULL).
 */
typedef struct pd_messenger pd_messenger;
PD_API int pd_counter_alloc(uint32_t **host_word, uint32_t **device_word);
PD_API int pd_counter_free(uint32_t *host_word);
PD_API int pd_layer_signal(uint32_t *device_word, uint32_t value, void *stream);
PD_API int pd_messenger_start_pack(pd_messenger **out, const uint32_t *host_word, const pd_kv_desc *desc,
                                   const pd_batch *batch, const void *k_pool, const void *v_pool,
                                   void *dst, size_t dst_bytes, const int64_t *dst_offsets,
                                   int32_t *dev_status, void *stream, int32_t timeout_ms);
PD_API int pd_messenger_join(pd_messenger *m, int32_t *layers_sent);

/*
 * Profiling hook (not part of the method): while set, every call of this host
 * thread records `start_event` on its stream just before launching its main
 * kernel (the split-KV decode kernel, the prefill/mixed kernel, the append,
 * pack or unpack kernel) and `stop_event` just after it, so that
 * cudaEventElapsedTime gives that kernel's device time alone. Both are
 * cudaEvent_t handles owned by the caller; pass NULL, NULL to stop. Returns
 * PD_ERR_INVALID_ARG if exactly one of them is NULL.
 */
PD_API int pd_profile_events(void *start_event, void *stop_event);

/*
 * Name of the main kernel the last call of this host thread launched
 * ("decode_kernel", "prefill_kernel", "kv_pack_kernel", ...; "" before any
 * call). Not part of the method: pd_attn_decode runs a large GQA batch on the
 * tensor-core kernel and other batches on the split-KV kernel, and profiling
 * needs to know which. The string is static.
 */
PD_API const char *pd_last_kernel(void);

/* Static description of a pd_status or pd_device_status code (never NULL). */
PD_API const char *pd_status_string(int32_t code);
PD_API const char *pd_device_status_string(int32_t code);

/* Library version, major * 10000 + minor * 100 + patch. */
PD_API int32_t pd_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PD_H_ */
