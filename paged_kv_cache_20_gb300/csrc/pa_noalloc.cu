// pa_noalloc.cu -- split-KV decode that needs no caller-provided workspace.
//
// pa_decode_partial / pa_decode_combine exchange per-partition softmax statistics
// through a workspace that the caller allocates.  Some callers cannot allocate
// device memory at the point where they run attention: a plug-in inside a host
// runtime that owns every device allocation through its own pool and forbids
// raw cudaMalloc; a serving loop with a fixed memory budget that must not
// allocate (or implicitly synchronise the device, as cudaMalloc/cudaFree can)
// once it is running; a real-time path that may not block.  For them this file
// keeps the workspace in a fixed file-scope device array instead.
//
// Costs and rules of the fixed array:
//   * kScratchBytes (8 MiB) of device memory on every GPU that loads the library,
//     held until the process exits;
//   * every call on a device uses the same array, so calls whose kernels can
//     overlap on the GPU (different streams without ordering between them) race
//     and produce wrong results -- order them on one stream or with events;
//   * the array keeps the previous call's contents; nothing in it has to start at
//     zero because the partial pass writes every entry the combine pass reads;
//   * the first call on a device looks up the array's device address
//     (cudaGetSymbolAddress) with that device current; make that first call
//     before any stream capture;
//   * that address is kept for the life of the process, so the library must not
//     outlive a reset of the device's primary context (cudaDeviceReset): after a
//     reset the kept address no longer names the array.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/pagedattn.h"

namespace {

constexpr size_t kScratchBytes = PA_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

// In host code this name is only a host-side stand-in for the device array; its
// device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_split_scratch[kScratchBytes];

std::mutex g_mutex;
void *g_scratch[kMaxDevices] = {};

// Device address of this device's array; looked up once per device.
void *scratch_address() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (g_scratch[dev] == nullptr) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_split_scratch) != cudaSuccess || p == nullptr) return nullptr;
    g_scratch[dev] = p;
  }
  return g_scratch[dev];
}

}  // namespace

extern "C" PA_API pa_status pa_decode_split_noalloc(
    void *out, const void *q, const void *k_cache, const void *v_cache,
    const int32_t *block_tables, const int32_t *context_lens, int num_seqs, int num_q_heads,
    int num_kv_heads, int head_dim, int block_size, float scale, int num_splits,
    int max_blocks_per_seq, int num_blocks, int q_len, pa_dtype dtype, void *stream) {
  const size_t need = pa_decode_workspace_size(num_seqs, num_q_heads, q_len, head_dim, num_splits);
  if (need == 0) return PA_ERR_INVALID_ARG;
  if (need > kScratchBytes) return PA_ERR_INVALID_ARG;  // beyond the fixed array: nothing launched
  void *ws = scratch_address();
  if (ws == nullptr) return PA_ERR_CUDA;
  pa_status st = pa_decode_partial(ws, kScratchBytes, q, k_cache, v_cache, block_tables,
                                   context_lens, num_seqs, num_q_heads, num_kv_heads, head_dim,
                                   block_size, scale, num_splits, max_blocks_per_seq, num_blocks,
                                   q_len, dtype, stream);
  if (st != PA_OK) return st;
  return pa_decode_combine(out, ws, kScratchBytes, num_seqs, num_q_heads, head_dim, q_len,
                           num_splits, dtype, stream);
}
