// Block scoring without caller-provided or library-allocated scratch.
//
// sparse_attn_score needs a workspace for the pooled queries and keys.  Some
// callers cannot provide one at the point where they score a layer: code
// that must never allocate on its hot path (cudaMalloc may synchronise the
// device and its latency is unbounded), hosts whose device memory is owned
// by their own pool allocator and hand plugins only the input and output
// buffers, and callers running with a fixed memory budget set at start-up.
// For them this entry point keeps the pooled vectors in one fixed area of
// device memory that is part of this file's module.  CUDA loads modules
// lazily by default, so a device reserves those kNoAllocScratchBytes at the
// first call on it (at library load when modules load eagerly) and keeps them
// until the process exits; the call itself allocates nothing.
//
// The first call on a device looks the area's address up, with that device
// current, and may load the module: make it before any stream capture.  The
// address is kept for the life of the process, so after cudaDeviceReset (or
// any other teardown of the device's primary context) this entry point must
// not be called again in that process: the module is reloaded elsewhere and
// the kept address would be stale.
//
// The area is shared by every call on a device and keeps whatever the last
// call left in it.  Nothing in it needs to start at zero: each call
// overwrites every pooled vector it reads.  Calls whose execution overlaps on
// the GPU (different streams, or different host threads without ordering)
// race on the area and may produce wrong scores; serialise them.

#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <mutex>

#include "kernels.h"
#include "plan_impl.h"
#include "sparse_attn.h"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;   // 32 MiB
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_score_scratch[kNoAllocScratchBytes];

// Device address of g_score_scratch per device, looked up on first use with
// that device current (the host-side symbol is only a stand-in).
std::atomic<void*> g_scratch_addr[kMaxDevices];
std::mutex g_scratch_mutex;

sa_status scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return SA_ERR_CUDA;
  if (dev >= kMaxDevices) return SA_ERR_UNSUPPORTED;
  void* p = g_scratch_addr[dev].load(std::memory_order_acquire);
  if (!p) {
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    p = g_scratch_addr[dev].load(std::memory_order_relaxed);
    if (!p) {
      if (cudaGetSymbolAddress(&p, g_score_scratch) != cudaSuccess || !p) return SA_ERR_CUDA;
      g_scratch_addr[dev].store(p, std::memory_order_release);
    }
  }
  *out = p;
  return SA_OK;
}

}  // namespace

extern "C" sa_status sparse_attn_score_noalloc(const sa_shape* shp, const void* q, const void* k,
                                               float* scores, sa_stream_t stream) {
  sa_status s = sa_host::check_supported(shp);
  if (s != SA_OK) return s;
  if (!q || !k || !scores) return SA_ERR_INVALID_ARG;
  const uintptr_t mis = reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) |
                        reinterpret_cast<uintptr_t>(scores);
  if (mis & 15u) return SA_ERR_INVALID_ARG;
  if (shp->mode == SA_MODE_DECODE)   // the decode path pools nothing per call
    return sparse_attn_score(shp, q, k, scores, nullptr, 0, stream);
  size_t need = 0;
  s = sparse_attn_score_workspace_size(shp, &need);
  if (s != SA_OK) return s;
  if (need > kNoAllocScratchBytes) return SA_ERR_UNSUPPORTED;
  void* ws = nullptr;
  s = scratch_address(&ws);
  if (s != SA_OK) return s;
  // the same stages as sparse_attn_score, with the area as the workspace
  return sa_k::cuda_status(sa_k::launch_prefill_index(
      q, k, scores, static_cast<float*>(ws), shp->num_q_heads, shp->num_kv_heads,
      int(shp->seq_len / shp->block), shp->block, shp->head_dim,
      reinterpret_cast<cudaStream_t>(stream)));
}
