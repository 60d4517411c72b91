// pd_green.cu -- pd_attn_mixed_split: the prefill and the decode requests of a
// mixed batch run at the same time on disjoint sets of SMs.
//
// Perplexity, "Disaggregated prefill and decode" (2025), section "Prefill vs
// Decode performance": prefill requests are compute bound, decode requests
// bound by the KV bytes they read, and a batch that mixes them pays for both.
// The split-KV decode kernel reaches most of the HBM bandwidth on its own but
// wants the SMs in numbers (several small CTAs per SM), while a prefill request
// of a few thousand rows keeps a handful of SMs busy for as long. So the batch
// runs as its two parts, each on its own kernel, at the same time: green
// contexts (the driver's SM partitions) give the prefill part a small set of
// SMs and the decode part the rest, so neither kernel's CTAs can take the
// other's SMs, whatever order the hardware places them in.
//
// Green-context handling goes through the driver's entry points, looked up
// through the runtime (the library links only against libcudart).
#include <cuda.h>
#include <cudaTypedefs.h>

#include <stdlib.h>

#include <map>
#include <mutex>

#include "pd_internal.h"

namespace pd {

namespace {

struct DriverFns {
  PFN_cuDeviceGet_v2000 device_get = nullptr;
  PFN_cuDeviceGetDevResource_v12040 get_resource = nullptr;
  PFN_cuDevSmResourceSplitByCount_v12040 split = nullptr;
  PFN_cuDevResourceGenerateDesc_v12040 make_desc = nullptr;
  PFN_cuGreenCtxCreate_v12040 green_create = nullptr;
  PFN_cuCtxFromGreenCtx_v12040 to_ctx = nullptr;
  PFN_cuGreenCtxStreamCreate_v12050 stream_create = nullptr;
  PFN_cuCtxPushCurrent_v4000 push = nullptr;
  PFN_cuCtxPopCurrent_v4000 pop = nullptr;
  bool ok = false;
};

template <typename F>
bool entry(const char* name, int version, F* out) {
  void* p = nullptr;
  cudaDriverEntryPointQueryResult q{};
  if (cudaGetDriverEntryPointByVersion(name, &p, version, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess || p == nullptr)
    return false;
  *out = reinterpret_cast<F>(p);
  return true;
}

const DriverFns& driver() {
  static DriverFns f;
  static std::once_flag once;
  std::call_once(once, [] {
    f.ok = entry("cuDeviceGet", 2000, &f.device_get) && entry("cuDeviceGetDevResource", 12040, &f.get_resource) &&
           entry("cuDevSmResourceSplitByCount", 12040, &f.split) &&
           entry("cuDevResourceGenerateDesc", 12040, &f.make_desc) &&
           entry("cuGreenCtxCreate", 12040, &f.green_create) && entry("cuCtxFromGreenCtx", 12040, &f.to_ctx) &&
           entry("cuGreenCtxStreamCreate", 12050, &f.stream_create) &&
           entry("cuCtxPushCurrent", 4000, &f.push) && entry("cuCtxPopCurrent", 4000, &f.pop);
  });
  return f;
}

// Two green contexts on one device: part 0 with `sms[0]` SMs, part 1 with the
// rest; each with a stream and an event, plus an event of the device's
// primary context that orders both after the caller's stream.
struct GreenPair {
  bool ok = false;
  int sms[2] = {0, 0};
  CUcontext ctx[2] = {nullptr, nullptr};
  cudaStream_t stream[2] = {nullptr, nullptr};
  cudaEvent_t done[2] = {nullptr, nullptr};
  cudaEvent_t start = nullptr;
  std::mutex mu;  // one call at a time enqueues through the pair
};

std::mutex g_pairs_mu;
std::map<std::pair<int, int>, GreenPair*> g_pairs;

bool create_pair(int dev, int first_sms, GreenPair* g) {
  const DriverFns& f = driver();
  if (!f.ok) return false;
  CUdevice cu_dev = 0;
  if (f.device_get(&cu_dev, dev) != CUDA_SUCCESS) return false;
  CUdevResource all{};
  if (f.get_resource(cu_dev, &all, CU_DEV_RESOURCE_TYPE_SM) != CUDA_SUCCESS) return false;
  CUdevResource part[1]{}, rest{};
  unsigned int groups = 1;
  if (f.split(part, &groups, &all, &rest, 0, (unsigned int)first_sms) != CUDA_SUCCESS || groups != 1) return false;
  if (part[0].sm.smCount == 0 || rest.sm.smCount == 0) return false;
  if (cudaEventCreateWithFlags(&g->start, cudaEventDisableTiming) != cudaSuccess) return false;
  CUdevResource* res[2] = {&part[0], &rest};
  for (int i = 0; i < 2; ++i) {
    CUdevResourceDesc desc = nullptr;
    CUgreenCtx green = nullptr;
    if (f.make_desc(&desc, res[i], 1) != CUDA_SUCCESS) return false;
    if (f.green_create(&green, desc, cu_dev, CU_GREEN_CTX_DEFAULT_STREAM) != CUDA_SUCCESS) return false;
    if (f.to_ctx(&g->ctx[i], green) != CUDA_SUCCESS) return false;
    CUstream s = nullptr;
    if (f.stream_create(&s, green, CU_STREAM_NON_BLOCKING, 0) != CUDA_SUCCESS) return false;
    g->stream[i] = reinterpret_cast<cudaStream_t>(s);
    if (f.push(g->ctx[i]) != CUDA_SUCCESS) return false;
    const bool ev = cudaEventCreateWithFlags(&g->done[i], cudaEventDisableTiming) == cudaSuccess;
    CUcontext popped = nullptr;
    f.pop(&popped);
    if (!ev) return false;
    g->sms[i] = (int)res[i]->sm.smCount;
  }
  return true;
}

// The pair for this device and prefill partition size, created on first use
// (a failed creation is remembered too); nullptr where green contexts are not
// available.
GreenPair* green_pair(int dev, int first_sms) {
  std::lock_guard<std::mutex> lock(g_pairs_mu);
  auto it = g_pairs.find({dev, first_sms});
  if (it != g_pairs.end()) return it->second->ok ? it->second : nullptr;
  GreenPair* g = new GreenPair;  // kept for the life of the process
  g->ok = create_pair(dev, first_sms, g);
  g_pairs[{dev, first_sms}] = g;
  return g->ok ? g : nullptr;
}

// A CUDA tool injected into the process (a profiler or a sanitizer) may not
// follow launches into green contexts: Nsight Compute stops the application at
// the first of them. Such tools announce themselves in the environment they
// give the process: the CUDA injection path, or Nsight's own injection and
// launch variables.
bool tool_attached() {
  static const bool attached = [] {
    const char* names[] = {"CUDA_INJECTION64_PATH", "NV_NSIGHT_INJECTION_TRANSPORT_TYPE",
                           "NV_COMPUTE_PROFILER_PERFWORKS_DIR", "NV_TPS_LAUNCH_TOKEN"};
    for (const char* n : names)
      if (getenv(n) != nullptr) return true;
    return false;
  }();
  return attached;
}

// SMs for the prefill part when the caller gives none: enough for it to finish
// in about the time the decode part takes, from the host-side bounds. The
// decode part is bound by HBM (about 6 TB/s on the split-KV kernel) and its
// requests are taken to average half of max_kv_len (the bound also covers the
// prefill requests' keys); a 128 x 128 prefill tile costs about 2 us of one SM
// on the tensor-core kernel, the prefill part taken as one causal request of
// all the prefill rows over max_kv_len keys. Rounded up to the partition
// granularity: a prefill part short of SMs holds the whole call back, while a
// few SMs more slow the decode part only a little.
int auto_prefill_sms(const pd_attn_desc* d, const pd_batch* b, int num_prefill) {
  const int64_t n_dec = b->batch_size - num_prefill;
  const int64_t rows = b->total_qo - n_dec > 0 ? b->total_qo - n_dec : 0;
  const int64_t q_tiles = (rows + 127) / 128, kv_tiles = ((int64_t)b->max_kv_len + 127) / 128;
  const int64_t tiles_per_head = d->causal ? (q_tiles < kv_tiles ? q_tiles * (2 * kv_tiles - q_tiles + 1) / 2
                                                                 : kv_tiles * (kv_tiles + 1) / 2)
                                           : q_tiles * kv_tiles;
  const double pf_sm_us = 2.0 * (double)tiles_per_head * d->num_qo_heads;
  const double dec_bytes = (double)n_dec * 0.5 * b->max_kv_len * d->num_kv_heads * d->head_dim * 2.0 *
                           (d->kv_dtype == PD_BF16 ? 2.0 : 4.0);
  const double dec_us = dec_bytes / 6.0e6;
  if (dec_us <= 0.0) return 1 << 20;
  return (int)(pf_sm_us / dec_us + 0.999);
}

}  // namespace
}  // namespace pd

extern "C" int pd_attn_mixed_split(const pd_attn_desc* desc, const pd_batch* batch, int32_t num_prefill,
                                   int32_t prefill_sms, const void* q, const void* k_pool, const void* v_pool,
                                   void* o, float* lse, void* workspace, size_t workspace_bytes,
                                   int32_t* dev_status, void* stream) {
  using namespace pd;
  if (desc == nullptr || batch == nullptr) return PD_ERR_INVALID_ARG;
  if (batch->batch_size < 0 || num_prefill < 0 || num_prefill > batch->batch_size || prefill_sms < 0)
    return PD_ERR_INVALID_ARG;
  if (batch->batch_size > 0 && batch->qo_indptr == nullptr) return PD_ERR_INVALID_ARG;
  if (batch->total_qo < batch->batch_size - num_prefill) return PD_ERR_INVALID_ARG;
  const size_t need = pd_attn_workspace_size(desc, batch, PD_KIND_MIXED_SPLIT);
  if (need == 0) return PD_ERR_INVALID_ARG;
  if (workspace_bytes < need) return PD_ERR_WORKSPACE;
  const int n_dec = batch->batch_size - num_prefill;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // One part only, or no partitions: the one-launch path on the caller's stream.
  if (num_prefill == 0 || n_dec == 0)
    return pd_attn_mixed(desc, batch, q, k_pool, v_pool, o, lse, workspace, workspace_bytes, dev_status, stream);
  const int sms = device_sm_count();
  int first = prefill_sms > 0 ? prefill_sms : auto_prefill_sms(desc, batch, num_prefill);
  first = (first + 7) / 8 * 8;
  if (first < 8) first = 8;
  if (first > sms - 8) first = (sms - 8) / 8 * 8;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PD_ERR_CUDA;
  GreenPair* g = first >= 8 && !tool_attached() ? green_pair(dev, first) : nullptr;
  if (g == nullptr)
    return pd_attn_mixed(desc, batch, q, k_pool, v_pool, o, lse, workspace, workspace_bytes, dev_status, stream);

  // The two sub-batches: the same device arrays from request 0 and from
  // request num_prefill (qo_indptr values are rows of q and o throughout).
  pd_batch bp = *batch, bd = *batch;
  bp.batch_size = num_prefill;
  bd.batch_size = n_dec;
  bd.qo_indptr = batch->qo_indptr + num_prefill;
  bd.kv_len = batch->kv_len + num_prefill;
  bd.page_indptr = batch->page_indptr + num_prefill;
  bd.max_qo_len = 1;
  const MixedSplitLayout L = mixed_split_layout(desc, batch);
  uint8_t* ws = static_cast<uint8_t*>(workspace);

  const DriverFns& f = driver();
  std::lock_guard<std::mutex> lock(g->mu);
  // kernel-only profiling events do not apply to a call on two streams
  const ProfileEvents saved = profile_events();
  profile_events() = ProfileEvents{};
  int rc[2] = {PD_OK, PD_OK};
  bool recorded[2] = {false, false};
  bool cuda_ok = cudaEventRecord(g->start, s) == cudaSuccess;
  for (int i = 0; i < 2 && cuda_ok; ++i) {
    if (f.push(g->ctx[i]) != CUDA_SUCCESS) {
      cuda_ok = false;
      break;
    }
    cuda_ok = cudaStreamWaitEvent(g->stream[i], g->start, 0) == cudaSuccess;
    if (cuda_ok) {
      partition_sms() = g->sms[i];
      rc[i] = i == 0 ? pd_attn_prefill(desc, &bp, q, k_pool, v_pool, o, lse, ws, L.decode, dev_status, g->stream[i])
                     : pd_attn_decode(desc, &bd, q, k_pool, v_pool, o, lse, ws + L.decode, L.total - L.decode,
                                      dev_status, g->stream[i]);
      partition_sms() = 0;
      recorded[i] = cudaEventRecord(g->done[i], g->stream[i]) == cudaSuccess;
      cuda_ok = recorded[i];
    }
    CUcontext popped = nullptr;
    f.pop(&popped);
  }
  profile_events() = saved;
  // the caller's stream waits for every part that was enqueued, also on failure
  for (int i = 0; i < 2; ++i)
    if (recorded[i] && cudaStreamWaitEvent(s, g->done[i], 0) != cudaSuccess) cuda_ok = false;
  last_kernel() = "prefill_kernel+decode_kernel";
  if (!cuda_ok) return PD_ERR_CUDA;
  return rc[0] != PD_OK ? rc[0] : rc[1];
}
