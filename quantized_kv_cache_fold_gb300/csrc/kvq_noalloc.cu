// Allocation-free variant of kvq_decode_attn_int4.
//
// Some callers cannot allocate device memory when they decode: an engine that reserves all
// GPU memory for its KV pool up front, a host process whose allocator must not be touched
// from the decode thread, or code running where cudaMalloc (or a framework allocator) is
// not allowed. This entry point takes the attention workspace from a fixed scratch array
// that lives in this library's device image instead of from the caller. Every GPU that
// loads the library holds the array (KVQ_NOALLOC_SCRATCH_BYTES) until the process exits.
//
// The array is shared by every call on a device and keeps the last call's contents. The
// workspace needs no zeroing: each call writes every part of it before reading it. Calls
// whose execution overlaps on the GPU (different streams without ordering, or several host
// threads) race on the array; the caller serialises them.
//
// In host code the array's name is only a host-side stand-in for the device symbol, never
// a device address: the device address is looked up once per device with
// cudaGetSymbolAddress (with that device current) and cached. That set-up happens in the
// first call on each device, so make the first call before any stream capture.

#include <cuda_runtime.h>

#include <atomic>
#include <mutex>

#include "kvq.h"

namespace {

static __device__ __align__(256) unsigned char g_kvq_noalloc_scratch[KVQ_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::atomic<void*> g_scratch_addr[kMaxDevices];
std::mutex g_setup_mutex;

// Device address of the scratch array on the current device (nullptr on failure).
void* scratch_address(int dev) {
  void* p = g_scratch_addr[dev].load(std::memory_order_acquire);
  if (p) return p;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  p = g_scratch_addr[dev].load(std::memory_order_relaxed);
  if (p) return p;
  void* addr = nullptr;
  if (cudaGetSymbolAddress(&addr, g_kvq_noalloc_scratch) != cudaSuccess || addr == nullptr) return nullptr;
  g_scratch_addr[dev].store(addr, std::memory_order_release);
  return addr;
}

}  // namespace

extern "C" kvq_status kvq_decode_attn_int4_noalloc(const kvq_int4_cache* cache, const float* Mq, const float* Mk,
                                                   const void* q, kvq_dtype dtype, int B, int S, int num_q_heads,
                                                   const int32_t* ctx_len, const void* k_new, const void* v_new,
                                                   float sm_scale, float eps, float* out, float* q_rot_out,
                                                   int32_t* dev_err, kvq_stream_t stream) {
  if (!cache) return KVQ_ERR_INVALID_ARG;
  const size_t need = kvq_decode_workspace_bytes(B, S, num_q_heads, cache->num_kv_heads);
  if (need == 0) return KVQ_ERR_UNSUPPORTED;
  if (need > (size_t)KVQ_NOALLOC_SCRATCH_BYTES) return KVQ_ERR_SCRATCH_TOO_SMALL;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return KVQ_ERR_CUDA;
  void* ws = scratch_address(dev);
  if (!ws) return KVQ_ERR_CUDA;
  return kvq_decode_attn_int4(cache, Mq, Mk, q, dtype, B, S, num_q_heads, ctx_len, k_new, v_new, sm_scale, eps,
                              out, ws, (size_t)KVQ_NOALLOC_SCRATCH_BYTES, q_rot_out, dev_err, stream);
}
