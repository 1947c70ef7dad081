// pa_decode_inst.cuh -- host launchers templated on the element type; included by
// pa_decode_fp16.cu and pa_decode_bf16.cu, which instantiate one type each.
#pragma once

#include <atomic>

#include "pa_decode.cuh"
#include "pa_launch.h"

namespace pa {

constexpr int kMaxDevices = 64;

// Pipeline shape: warps per CTA, stages per warp (measured on GB300).  The single
// pass uses 4 warps of 2 stages, which fits 3 CTAs per SM (12 warps) and helps the
// skewed-length workloads; with few units the single pass uses 3 warps instead
// (launch_few_units).  The split-KV partial pass gets the caller's
// equal-size partitions; with 3 stages (2 CTAs per SM) its CTAs are deeper and
// fewer, which measured faster there.
constexpr int kWarps = 4;
template <bool PARTIAL>
constexpr int stages_for() { return PARTIAL ? 3 : 2; }
// An FP8 stage carries half the bytes, so FP8 keeps 4 stages per warp in flight
// (still 3 CTAs per SM).  On the swapped-operand FP8 path this measured faster than
// 3 stages with 4 CTAs per SM or 2 stages.
template <class Path, bool PARTIAL, bool KV8>
constexpr int stages_of() { return KV8 ? 4 : stages_for<PARTIAL>(); }
constexpr int kMaxCluster = 8;  // portable cluster size limit

// Per device: SM count and resident CTAs per SM of one kernel (cached).
struct DeviceFit {
  std::atomic<int> sms{0};
  std::atomic<int> ctas_per_sm{0};
};

// Resident slots (SMs x CTAs per SM) of one kernel instance on the current device,
// cached per device; the first call also sets the kernel's shared-memory opt-in.
template <int BS, typename T, int D, class Path, bool PARTIAL, bool KV8, int NW>
static cudaError_t resident_slots(long long &slots) {
  constexpr int kStages = stages_of<Path, PARTIAL, KV8>();
  constexpr int kStageBytes = 2 * kTileTokens * D * (KV8 ? 1 : 2);
  constexpr int kSmem = NW * kStages * kStageBytes + 1024;
  auto kern = paged_decode_kernel<T, D, NW, kStages, Path, PARTIAL, KV8, BS>;
  static DeviceFit fit[kMaxDevices];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  DeviceFit &f = fit[dev];
  if (f.ctas_per_sm.load(std::memory_order_acquire) == 0) {
    // the shared-memory opt-in is a per-device function attribute
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e != cudaSuccess) return e;
    int sms = 0, per_sm = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, NW * 32, kSmem);
    if (e != cudaSuccess) return e;
    f.sms.store(sms, std::memory_order_relaxed);
    f.ctas_per_sm.store(per_sm > 0 ? per_sm : 1, std::memory_order_release);
  }
  slots = (long long)f.sms.load(std::memory_order_relaxed) * f.ctas_per_sm.load();
  return cudaSuccess;
}

// Launch one kernel instance with NW warps per CTA.  Single pass: while the units
// would fill fewer than wave_num / wave_den waves of resident CTAs, double the
// cluster size (up to kMaxCluster) so long sequences spread over several SMs.
template <int BS, typename T, int D, class Path, bool PARTIAL, bool KV8 = false, int NW = kWarps>
static cudaError_t launch_one(const CUtensorMap &kmap, const CUtensorMap &vmap,
                              const DecodeArgs &a, int units, int row_groups, cudaStream_t st,
                              int wave_num = 2, int wave_den = 1) {
  constexpr int kStages = stages_of<Path, PARTIAL, KV8>();
  constexpr int kStageBytes = 2 * kTileTokens * D * (KV8 ? 1 : 2);
  constexpr int kSmem = NW * kStages * kStageBytes + 1024;
  auto kern = paged_decode_kernel<T, D, NW, kStages, Path, PARTIAL, KV8, BS>;
  long long slots = 0;
  cudaError_t e = resident_slots<BS, T, D, Path, PARTIAL, KV8, NW>(slots);
  if (e != cudaSuccess) return e;
  // The partial pass already has the caller's partitions (clusters measured slower
  // there: each CTA's fixed cost outweighs the shorter tail).
  int cluster = 1;
  if (!PARTIAL) {
    const long long work = (long long)units * row_groups;
    while (cluster < kMaxCluster && work * cluster * wave_den < wave_num * slots) cluster *= 2;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)units * cluster, (unsigned)row_groups, 1);
  cfg.blockDim = dim3(NW * 32, 1, 1);
  cfg.dynamicSmemBytes = kSmem;
  cfg.stream = st;
  // attribute 0: programmatic dependent launch (the kernel waits on griddepcontrol
  // before reading global memory); attribute 1: the cluster shape, if any
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = cluster;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = cluster > 1 ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, kern, kmap, vmap, a);
}

// Single pass with one row group, head_dim 128.  Measured over batch sizes (MHA,
// GQA and verify shapes, every path, 16-bit and FP8 caches): while the units fit
// in one wave of 3-warp CTAs (4 per SM where registers allow), those beat 4-warp
// CTAs (3 per SM) by 4-23 %, with clusters growing up to 1.5 waves; a CTA's fixed
// start and end-of-unit merge then overlap a fourth CTA's loads.  Above that,
// 4-warp CTAs with the caller's cluster threshold: 1.5 waves on the FP8
// swapped-operand path, 2 elsewhere.
template <int BS, typename T, class Path, bool KV8, int WAVE4_NUM, int WAVE4_DEN>
static cudaError_t launch_few_units(const CUtensorMap &kmap, const CUtensorMap &vmap,
                                    const DecodeArgs &a, int units, cudaStream_t st) {
  long long slots3 = 0;
  const cudaError_t e = resident_slots<BS, T, 128, Path, false, KV8, 3>(slots3);
  if (e != cudaSuccess) return e;
  if (units < slots3) return launch_one<BS, T, 128, Path, false, KV8, 3>(kmap, vmap, a, units, 1, st, 3, 2);
  return launch_one<BS, T, 128, Path, false, KV8>(kmap, vmap, a, units, 1, st, WAVE4_NUM, WAVE4_DEN);
}

template <int BS, typename T, int D, bool PARTIAL>
static cudaError_t launch_paths(const CUtensorMap &kmap, const CUtensorMap &vmap,
                                const DecodeArgs &a, int units, cudaStream_t st) {
  if constexpr (!PARTIAL && D == 128) {
    if (a.rows == 1) return launch_few_units<BS, T, FmaPath<T, D, 4, 1>, false, 2, 1>(kmap, vmap, a, units, st);
    if (a.rows == 2) return launch_few_units<BS, T, FmaPath<T, D, 8, 2>, false, 2, 1>(kmap, vmap, a, units, st);
  }
  if (a.rows == 1) return launch_one<BS, T, D, FmaPath<T, D, 4, 1>, PARTIAL>(kmap, vmap, a, units, 1, st);
  if (a.rows == 2) return launch_one<BS, T, D, FmaPath<T, D, 8, 2>, PARTIAL>(kmap, vmap, a, units, 1, st);
  if (a.rows <= 8) {
    if constexpr (!PARTIAL && D == 128)
      return launch_few_units<BS, T, MmaTPath<T, D>, false, 2, 1>(kmap, vmap, a, units, st);
    return launch_one<BS, T, D, MmaTPath<T, D>, PARTIAL>(kmap, vmap, a, units, 1, st);
  }
  const int groups = (a.rows + 15) / 16;
  if constexpr (!PARTIAL && D == 128)
    if (groups == 1) return launch_few_units<BS, T, MmaPath<T, D>, false, 2, 1>(kmap, vmap, a, units, st);
  return launch_one<BS, T, D, MmaPath<T, D>, PARTIAL>(kmap, vmap, a, units, groups, st);
}

template <int BS, typename T, bool PARTIAL>
static cudaError_t launch_paths8(const CUtensorMap &kmap, const CUtensorMap &vmap,
                                 const DecodeArgs &a, int units, cudaStream_t st) {
  if constexpr (!PARTIAL) {
    if (a.rows == 1) return launch_few_units<BS, T, Fma8Path<T, 1>, true, 2, 1>(kmap, vmap, a, units, st);
    if (a.rows == 2) return launch_few_units<BS, T, Fma8Path<T, 2>, true, 2, 1>(kmap, vmap, a, units, st);
  }
  if (a.rows == 1) return launch_one<BS, T, 128, Fma8Path<T, 1>, PARTIAL, true>(kmap, vmap, a, units, 1, st);
  if (a.rows == 2) return launch_one<BS, T, 128, Fma8Path<T, 2>, PARTIAL, true>(kmap, vmap, a, units, 1, st);
  if (a.rows <= 8) {
    if constexpr (!PARTIAL) return launch_few_units<BS, T, Mma8TPath<T>, true, 3, 2>(kmap, vmap, a, units, st);
    return launch_one<BS, T, 128, Mma8TPath<T>, PARTIAL, true>(kmap, vmap, a, units, 1, st);
  }
  const int groups = (a.rows + 15) / 16;
  if constexpr (!PARTIAL)
    if (groups == 1) return launch_few_units<BS, T, Mma8Path<T>, true, 2, 1>(kmap, vmap, a, units, st);
  return launch_one<BS, T, 128, Mma8Path<T>, PARTIAL, true>(kmap, vmap, a, units, groups, st);
}

// FP8 (e4m3) cache, head_dim 128; T is the type of q and out.
// BS = 16: kernels built for 16-token blocks; BS = 0: kernels that read the block
// size (8 or 32) from the arguments.
template <int BS, typename T>
static cudaError_t launch_decode8_t(const CUtensorMap &kmap, const CUtensorMap &vmap,
                                    const DecodeArgs &a, bool partial, int units, cudaStream_t st) {
  return partial ? launch_paths8<BS, T, true>(kmap, vmap, a, units, st)
                 : launch_paths8<BS, T, false>(kmap, vmap, a, units, st);
}

template <int BS, typename T>
static cudaError_t launch_decode_t(const CUtensorMap &kmap, const CUtensorMap &vmap,
                                   const DecodeArgs &a, int head_dim, bool partial, int units,
                                   cudaStream_t st) {
  if (head_dim == 128)
    return partial ? launch_paths<BS, T, 128, true>(kmap, vmap, a, units, st)
                   : launch_paths<BS, T, 128, false>(kmap, vmap, a, units, st);
  if (head_dim == 64)
    return partial ? launch_paths<BS, T, 64, true>(kmap, vmap, a, units, st)
                   : launch_paths<BS, T, 64, false>(kmap, vmap, a, units, st);
  return cudaErrorInvalidValue;
}

template <typename T>
static cudaError_t launch_combine_t(const CombineArgs &a, int head_dim, cudaStream_t st) {
  const long long rows = (long long)a.num_seqs * a.rows_per_seq;
  if (rows == 0) return cudaSuccess;
  // One dimension per lane (split_combine_spread_kernel) for more than 8 partitions
  // of at most 512 rows.  Measured on GB300: 4 x 32 rows of 16 partitions, 92.5 ->
  // 90.5 us per step; 8 x 32 rows of 8 partitions and 64 x 32 rows of 4 partitions
  // were slower spread.
  if (a.num_splits > 8 && rows <= 512) {
    const int blocks = (int)((rows * (head_dim / 32) * 32 + 127) / 128);
    if (head_dim == 128)
      return launch_dependent(split_combine_spread_kernel<T, 128>, blocks, 128, st, a);
    if (head_dim == 64)
      return launch_dependent(split_combine_spread_kernel<T, 64>, blocks, 128, st, a);
    return cudaErrorInvalidValue;
  }
  const int blocks = (int)((rows * 32 + 127) / 128);
  if (head_dim == 128) return launch_dependent(split_combine_kernel<T, 128>, blocks, 128, st, a);
  if (head_dim == 64) return launch_dependent(split_combine_kernel<T, 64>, blocks, 128, st, a);
  return cudaErrorInvalidValue;
}

}  // namespace pa
