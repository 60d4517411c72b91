// pd_messenger.cu -- layer-streamed KV handoff: a completion counter written by
// the GPU and a host thread that ships each layer as soon as it is ready.
//
// Perplexity, "Disaggregated prefill and decode" (2025), section "KV Messenger":
// the copies of a layer's pages start as soon as the model has appended that
// layer's KV entries; a polling thread watches a counter that the GPU advances
// after each layer, which keeps the model's step capturable in a CUDA graph.
// Here the counter is a word of mapped pinned host memory written by a
// one-thread kernel with a system-scope release store, and the "copy" of a layer
// is its pack into the per-request blocks (pd_kv_pack_layers) on the
// messenger's own stream.
#include <atomic>
#include <chrono>
#include <thread>

#include "pd_common.cuh"
#include "pd_internal.h"

namespace pd {
namespace {

// Runs once every earlier kernel on the stream has completed (stream order)
// and publishes `value` to the host.
__global__ void layer_signal_kernel(uint32_t* counter, uint32_t value) {
  asm volatile("st.release.sys.global.u32 [%0], %1;" ::"l"(counter), "r"(value) : "memory");
}

}  // namespace
}  // namespace pd

struct pd_messenger {
  std::thread thread;
  std::atomic<int> status{PD_OK};
  std::atomic<int> layers_sent{0};
};

extern "C" {

int pd_counter_alloc(uint32_t** host_word, uint32_t** device_word) {
  if (host_word == nullptr || device_word == nullptr) return PD_ERR_INVALID_ARG;
  *host_word = nullptr;
  *device_word = nullptr;
  void* h = nullptr;
  if (cudaHostAlloc(&h, 64, cudaHostAllocMapped) != cudaSuccess) return PD_ERR_CUDA;
  void* d = nullptr;
  if (cudaHostGetDevicePointer(&d, h, 0) != cudaSuccess) {
    cudaFreeHost(h);
    return PD_ERR_CUDA;
  }
  __atomic_store_n(static_cast<uint32_t*>(h), 0u, __ATOMIC_RELEASE);
  *host_word = static_cast<uint32_t*>(h);
  *device_word = static_cast<uint32_t*>(d);
  return PD_OK;
}

int pd_counter_free(uint32_t* host_word) {
  if (host_word == nullptr) return PD_OK;
  return cudaFreeHost(host_word) == cudaSuccess ? PD_OK : PD_ERR_CUDA;
}

int pd_layer_signal(uint32_t* device_word, uint32_t value, void* stream) {
  if (device_word == nullptr) return PD_ERR_INVALID_ARG;
  pd::layer_signal_kernel<<<1, 1, 0, static_cast<cudaStream_t>(stream)>>>(device_word, value);
  return cudaGetLastError() == cudaSuccess ? PD_OK : PD_ERR_CUDA;
}

int pd_messenger_start_pack(pd_messenger** out, const uint32_t* host_word, const pd_kv_desc* desc,
                            const pd_batch* batch, const void* k_pool, const void* v_pool, void* dst,
                            size_t dst_bytes, const int64_t* dst_offsets, int32_t* dev_status, void* stream,
                            int32_t timeout_ms) {
  if (out == nullptr) return PD_ERR_INVALID_ARG;
  *out = nullptr;
  if (host_word == nullptr || desc == nullptr || batch == nullptr || timeout_ms <= 0 || desc->num_layers < 1)
    return PD_ERR_INVALID_ARG;
  int device = -1;
  if (cudaGetDevice(&device) != cudaSuccess) device = -1;
  pd_messenger* m = new pd_messenger();
  const pd_kv_desc d = *desc;  // the thread keeps its own copies
  const pd_batch b = *batch;
  m->thread = std::thread([=]() {
    if (device >= 0) cudaSetDevice(device);
    using clock = std::chrono::steady_clock;
    for (int layer = 0; layer < d.num_layers; ++layer) {
      // wait until the GPU has passed layer `layer`, at most timeout_ms
      const auto t0 = clock::now();
      while (__atomic_load_n(host_word, __ATOMIC_ACQUIRE) <= (uint32_t)layer) {
        if (clock::now() - t0 > std::chrono::milliseconds(timeout_ms)) {
          m->status.store(PD_ERR_TIMEOUT);
          return;
        }
        std::this_thread::yield();
      }
      const int rc = pd_kv_pack_layers(&d, &b, layer, 1, k_pool, v_pool, dst, dst_bytes, dst_offsets,
                                       dev_status, stream);
      if (rc != PD_OK) {
        m->status.store(rc);
        return;
      }
      m->layers_sent.store(layer + 1);
    }
  });
  *out = m;
  return PD_OK;
}

int pd_messenger_join(pd_messenger* m, int32_t* layers_sent) {
  if (m == nullptr) return PD_ERR_INVALID_ARG;
  if (m->thread.joinable()) m->thread.join();
  const int rc = m->status.load();
  if (layers_sent != nullptr) *layers_sent = m->layers_sent.load();
  delete m;
  return rc;
}

}  // extern "C"
