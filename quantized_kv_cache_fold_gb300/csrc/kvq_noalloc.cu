// Allocation-free variant of kvq_decode_attn_int4.
//
// Some callers cannot allocate device memory when they decode: an engine that reserves all
// GPU memory for its KV pool up front, a host process whose allocator must not be touched
// from the decode thread, or code running where cudaMalloc (or a framework allocator) is
// not allowed. This entry point takes the attention workspace from a fixed scratch array
// that lives in this library's device image instead of from the caller.
//
// When the array is allocated: this file is its own CUDA module. Under lazy module loading
// (CUDA_MODULE_LOADING=LAZY, the default) the module, and with it the array's
// KVQ_NOALLOC_SCRATCH_BYTES of device memory, is loaded on a device by the first call of this
// entry point there (its cudaGetSymbolAddress); under eager loading, when the library's
// modules load. Either way the device holds the array until the process exits (or the device
// is reset). So make the first call on each device before reserving the memory pool the
// engine hands out, and before any stream capture.
//
// The array is shared by every call on a device and keeps the last call's contents. The
// workspace needs no zeroing: each call writes every part of it before reading it. Calls
// whose execution overlaps on the GPU (different streams without ordering, or several host
// threads) race on the array; the caller serialises them.
//
// In host code the array's name is only a host-side stand-in for the device symbol, never
// a device address. The first call on a device, with that device current, looks the device
// address up with cudaGetSymbolAddress under a lock (that set-up loads the module). Every
// later call repeats the lookup, which is cheap once the module is loaded, so a
// cudaDeviceReset between calls (after which the array may sit elsewhere) cannot leave a
// stale address behind.

#include <cuda_runtime.h>

#include <atomic>
#include <mutex>

#include "kvq.h"
#include "kvq_internal.h"

namespace {

static __device__ __align__(256) unsigned char g_kvq_noalloc_scratch[KVQ_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::atomic<bool> g_set_up[kMaxDevices];
std::mutex g_setup_mutex;

// Device address of the scratch array on the current device `dev` (nullptr on failure).
void* scratch_address(int dev) {
  void* addr = nullptr;
  if (!g_set_up[dev].load(std::memory_order_acquire)) {
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (!g_set_up[dev].load(std::memory_order_relaxed)) {
      if (cudaGetSymbolAddress(&addr, g_kvq_noalloc_scratch) != cudaSuccess || addr == nullptr) return nullptr;
      g_set_up[dev].store(true, std::memory_order_release);
      return addr;
    }
  }
  if (cudaGetSymbolAddress(&addr, g_kvq_noalloc_scratch) != cudaSuccess) return nullptr;
  return addr;
}

}  // namespace

extern "C" kvq_status kvq_decode_attn_int4_noalloc(const kvq_int4_cache* cache, const float* Mq, const float* Mk,
                                                   const void* q, kvq_dtype dtype, int B, int S, int num_q_heads,
                                                   const int32_t* ctx_len, const void* k_new, const void* v_new,
                                                   float sm_scale, float eps, float* out, float* q_rot_out,
                                                   int32_t* dev_err, kvq_stream_t stream) {
  // the same argument checks (and status codes) as kvq_decode_attn_int4, before the scratch size
  const kvq_status st = kvq::check_decode_int4_args(cache, Mq, Mk, q, dtype, B, S, num_q_heads, ctx_len, k_new,
                                                    v_new, sm_scale, eps, out, q_rot_out, dev_err);
  if (st != KVQ_OK) return st;
  const size_t need = kvq_decode_workspace_bytes(B, S, num_q_heads, cache->num_kv_heads);
  if (need > (size_t)KVQ_NOALLOC_SCRATCH_BYTES) return KVQ_ERR_SCRATCH_TOO_SMALL;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return KVQ_ERR_CUDA;
  void* ws = scratch_address(dev);
  if (!ws) return KVQ_ERR_CUDA;
  return kvq_decode_attn_int4(cache, Mq, Mk, q, dtype, B, S, num_q_heads, ctx_len, k_new, v_new, sm_scale, eps,
                              out, ws, (size_t)KVQ_NOALLOC_SCRATCH_BYTES, q_rot_out, dev_err, stream);
}
