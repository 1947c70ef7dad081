// pa_decode_inst.cuh -- host launchers templated on the element type; included by
// pa_decode_fp16.cu and pa_decode_bf16.cu, which instantiate one type each.
#pragma once

#include <atomic>

#include "pa_decode.cuh"
#include "pa_launch.h"

namespace pa {

constexpr int kMaxDevices = 64;

// Pipeline shape: warps per CTA, stages per warp.
constexpr int kWarps = 4;
constexpr int kStages = 3;

template <typename T, int D, class Path, bool PARTIAL>
static cudaError_t launch_one(const CUtensorMap &kmap, const CUtensorMap &vmap,
                              const DecodeArgs &a, int units, int row_groups, cudaStream_t st) {
  constexpr int kStageBytes = 2 * kTileTokens * D * 2;
  constexpr int kSmem = kWarps * kStages * kStageBytes + 1024;
  auto kern = paged_decode_kernel<T, D, kWarps, kStages, Path, PARTIAL>;
  // the shared-memory opt-in is a per-device function attribute: set it once per device
  static std::atomic<bool> configured[kMaxDevices];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  if (!configured[dev].load(std::memory_order_acquire)) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e != cudaSuccess) return e;
    configured[dev].store(true, std::memory_order_release);
  }
  kern<<<dim3(units, row_groups), kWarps * 32, kSmem, st>>>(kmap, vmap, a);
  return cudaGetLastError();
}

template <typename T, int D, bool PARTIAL>
static cudaError_t launch_paths(const CUtensorMap &kmap, const CUtensorMap &vmap,
                                const DecodeArgs &a, int units, cudaStream_t st) {
  if (a.rows == 1) return launch_one<T, D, FmaPath<T, D, 4, 1>, PARTIAL>(kmap, vmap, a, units, 1, st);
  if (a.rows == 2) return launch_one<T, D, FmaPath<T, D, 8, 2>, PARTIAL>(kmap, vmap, a, units, 1, st);
  const int groups = (a.rows + 15) / 16;
  return launch_one<T, D, MmaPath<T, D>, PARTIAL>(kmap, vmap, a, units, groups, st);
}

template <typename T>
static cudaError_t launch_decode_t(const CUtensorMap &kmap, const CUtensorMap &vmap,
                                   const DecodeArgs &a, int head_dim, bool partial, int units,
                                   cudaStream_t st) {
  if (head_dim == 128)
    return partial ? launch_paths<T, 128, true>(kmap, vmap, a, units, st)
                   : launch_paths<T, 128, false>(kmap, vmap, a, units, st);
  if (head_dim == 64)
    return partial ? launch_paths<T, 64, true>(kmap, vmap, a, units, st)
                   : launch_paths<T, 64, false>(kmap, vmap, a, units, st);
  return cudaErrorInvalidValue;
}

template <typename T>
static cudaError_t launch_combine_t(const CombineArgs &a, int head_dim, cudaStream_t st) {
  const long long warps = (long long)a.num_seqs * a.rows_per_seq;
  const int blocks = (int)((warps * 32 + 127) / 128);
  if (blocks == 0) return cudaSuccess;
  if (head_dim == 128)
    split_combine_kernel<T, 128><<<blocks, 128, 0, st>>>(a);
  else if (head_dim == 64)
    split_combine_kernel<T, 64><<<blocks, 128, 0, st>>>(a);
  else
    return cudaErrorInvalidValue;
  return cudaGetLastError();
}

}  // namespace pa
