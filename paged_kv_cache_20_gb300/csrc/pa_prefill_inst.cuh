// pa_prefill_inst.cuh -- host launchers of the many-row (chunked-prefill /
// shared-prefix) tensor-core kernel, templated on the element type and on whether
// the cache's blocks are 16 tokens; included by pa_prefill.cu (16-token blocks)
// and pa_prefill_blocks.cu (8 or 32).
#pragma once

#include <algorithm>
#include <atomic>

#include "pa_launch.h"
#include "pa_prefill_tc.cuh"

namespace pa {

namespace {

// K and V ring depths (chunks in flight per CTA); with head_dim 128 the rings fill
// what shared memory remains after Q (227 KiB per CTA at most).  Over an FP8 cache,
// where the codes are widened in place before the MMAs read a stage, 2 K and 3 V
// stages measured the same as 3 and 2 (616.7 against 619.3 us on 16 x 512-token
// chunks).
template <int D> constexpr int kRingK = D == 128 ? 3 : 4;
template <int D> constexpr int kRingV = D == 128 ? 2 : 4;

template <typename T, int D, bool PARTIAL, bool KV8, bool BS16>
cudaError_t launch_prefill_t(const CUtensorMap &kmap, const CUtensorMap &vmap, const CUtensorMap &qmap,
                             const DecodeArgs &a, cudaStream_t st) {
  // the MMA operands are fp16 over an FP8 cache; the layout's sizes match either way
  using TM = typename TcPick<KV8, __half, T>::type;
  constexpr int kSmem = TcLayout<TM, D>::smem_bytes(kRingK<D>, kRingV<D>);
  auto kern = paged_prefill_tc_kernel<T, D, kRingK<D>, kRingV<D>, PARTIAL, KV8, BS16>;
  static std::atomic<unsigned long long> opted{0};  // bit per device: smem opt-in done
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!(opted.load(std::memory_order_acquire) & (1ull << dev))) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e != cudaSuccess) return e;
    if (KV8) {
      // the register split of the FP8 form adds up to exactly the registers a block
      // launched with kTcRegsLaunch8 per thread holds; with fewer, the softmax
      // warpgroups' setmaxnreg.inc could never be granted, so refuse to launch
      cudaFuncAttributes fa;
      e = cudaFuncGetAttributes(&fa, kern);
      if (e != cudaSuccess) return e;
      if (fa.numRegs != kTcRegsLaunch8) return cudaErrorInvalidConfiguration;
    }
    opted.fetch_or(1ull << dev, std::memory_order_acq_rel);
  }
  const long long rows_per_seq = (long long)a.q_len * a.group;
  const long long rows = a.shared_prefix > 0 ? rows_per_seq * a.num_seqs : rows_per_seq;
  const long long nz = a.shared_prefix > 0 ? a.num_splits : (long long)a.num_seqs * a.num_splits;
  const long long units = (rows + kTcRows - 1) / kTcRows * nz * a.num_kv_heads;
  if (units <= 0) return cudaSuccess;
  if (units > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  // persistent CTAs, one per SM (the shared memory and tensor memory of one CTA
  // fill an SM): each walks a list of units
  static std::atomic<int> sm_count[64];
  int sms = sm_count[dev].load(std::memory_order_relaxed);
  if (sms <= 0) {
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    sm_count[dev].store(sms, std::memory_order_relaxed);
  }
  long long cap = std::max(1, sms);
  if (a.max_ctas > 0) cap = std::min<long long>(cap, a.max_ctas);
  const long long gx = std::min<long long>(units, cap);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)gx, 1, 1);
  cfg.blockDim = dim3(KV8 ? kTcThreads8 : kTcThreads, 1, 1);
  cfg.dynamicSmemBytes = kSmem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, kmap, vmap, qmap, a);
}

template <bool BS16, typename T>
cudaError_t dispatch(const CUtensorMap &kmap, const CUtensorMap &vmap, const CUtensorMap &qmap,
                     const DecodeArgs &a, int head_dim, bool partial, bool kv8, cudaStream_t st) {
  if (kv8) {
    if (head_dim != 128) return cudaErrorInvalidValue;
    return partial ? launch_prefill_t<T, 128, true, true, BS16>(kmap, vmap, qmap, a, st)
                   : launch_prefill_t<T, 128, false, true, BS16>(kmap, vmap, qmap, a, st);
  }
  if (head_dim == 128)
    return partial ? launch_prefill_t<T, 128, true, false, BS16>(kmap, vmap, qmap, a, st)
                   : launch_prefill_t<T, 128, false, false, BS16>(kmap, vmap, qmap, a, st);
  if (head_dim == 64)
    return partial ? launch_prefill_t<T, 64, true, false, BS16>(kmap, vmap, qmap, a, st)
                   : launch_prefill_t<T, 64, false, false, BS16>(kmap, vmap, qmap, a, st);
  return cudaErrorInvalidValue;
}

}  // namespace

}  // namespace pa
