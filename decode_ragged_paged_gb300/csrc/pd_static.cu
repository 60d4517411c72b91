// pd_static.cu -- decode attention for callers that cannot provide a workspace.
//
// Some callers have no way to hand the library scratch memory: a plain C host
// program that only receives tensors from a framework owning every device
// allocation, or a latency-critical loop where calling cudaMalloc (which can
// synchronise the device) is not allowed. pd_attn_decode_static serves them:
// its scratch lives in one fixed-size array in device memory that the library
// itself defines, so the call allocates nothing.
//
// The array is a file-scope __device__ variable, so every GPU on which this
// part of the library is loaded keeps kStaticScratchBytes reserved until the
// process exits. All calls on a device share that one array and it keeps what
// the previous call left there; nothing in it has to start at zero, because
// every word a call reads was written earlier by the same call (the plan, the
// work list and the split partials). Calls whose work overlaps on the GPU (for
// example on two streams) use the same array at the same time and corrupt each
// other's results: serialise them.
#include <mutex>

#include "pd_internal.h"

namespace pd {

namespace {

// Fixed maximum scratch per device. The tensor-core decode path uses a few
// KiB of it (a header and the work list); the split-KV path keeps its partial
// results here, about 17 MiB for 128 requests with kv_len up to 4096 and 32
// query heads of 128.
constexpr size_t kStaticScratchBytes = size_t(32) << 20;

__device__ __align__(256) unsigned char g_decode_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of this device's copy of the array. In host code
// g_decode_scratch names a host-side stand-in, not device memory, so the
// address is looked up through the runtime once per device (with that device
// current) and cached for the life of the process. A cudaDeviceReset destroys
// the context the address belongs to; the header tells callers not to use this
// entry point on a device after resetting it.
int scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PD_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (dev >= 0 && dev < kMaxDevices && g_scratch_ptr[dev] != nullptr) {
    *out = g_scratch_ptr[dev];
    return PD_OK;
  }
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || p == nullptr) return PD_ERR_CUDA;
  if (dev >= 0 && dev < kMaxDevices) g_scratch_ptr[dev] = p;
  *out = p;
  return PD_OK;
}

}  // namespace
}  // namespace pd

extern "C" int pd_attn_decode_static(const pd_attn_desc* desc, const pd_batch* batch, const void* q,
                                     const void* k_pool, const void* v_pool, void* o, float* lse,
                                     int32_t* dev_status, void* stream) {
  void* scratch = nullptr;
  const int rc = pd::scratch_address(&scratch);
  if (rc != PD_OK) return rc;
  // The ordinary decode path with the library's array as its workspace; a batch
  // whose plan and partials need more than the array holds is rejected with
  // PD_ERR_WORKSPACE before anything is launched.
  return pd_attn_decode(desc, batch, q, k_pool, v_pool, o, lse, scratch, pd::kStaticScratchBytes, dev_status,
                        stream);
}
