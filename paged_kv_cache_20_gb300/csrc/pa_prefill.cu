// pa_prefill.cu -- host launchers of the many-row (chunked-prefill / shared-prefix)
// tensor-core kernel, both element types.
#include <algorithm>
#include <atomic>

#include "pa_launch.h"
#include "pa_prefill_tc.cuh"

namespace pa {

namespace {

constexpr int kRingK8 = 3, kRingV8 = 2;

// K and V ring depths (chunks in flight per CTA); with head_dim 128 the rings fill
// what shared memory remains after Q (227 KiB per CTA at most).  Over an FP8 cache
// a stage is held longer (its codes are widened in place before the MMAs read it).
template <int D, bool KV8> constexpr int kRingK = D == 128 ? (KV8 ? kRingK8 : 3) : 4;
template <int D, bool KV8> constexpr int kRingV = D == 128 ? (KV8 ? kRingV8 : 2) : 4;

template <typename T, int D, bool PARTIAL, bool KV8>
cudaError_t launch_prefill_t(const CUtensorMap &kmap, const CUtensorMap &vmap, const CUtensorMap &qmap,
                             const DecodeArgs &a, cudaStream_t st) {
  // the MMA operands are fp16 over an FP8 cache; the layout's sizes match either way
  using TM = typename TcPick<KV8, __half, T>::type;
  constexpr int kSmem = TcLayout<TM, D>::smem_bytes(kRingK<D, KV8>, kRingV<D, KV8>);
  auto kern = paged_prefill_tc_kernel<T, D, kRingK<D, KV8>, kRingV<D, KV8>, PARTIAL, KV8>;
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

template <typename T>
cudaError_t dispatch(const CUtensorMap &kmap, const CUtensorMap &vmap, const CUtensorMap &qmap,
                     const DecodeArgs &a, int head_dim, bool partial, bool kv8, cudaStream_t st) {
  if (kv8) {
    if (head_dim != 128) return cudaErrorInvalidValue;
    return partial ? launch_prefill_t<T, 128, true, true>(kmap, vmap, qmap, a, st)
                   : launch_prefill_t<T, 128, false, true>(kmap, vmap, qmap, a, st);
  }
  if (head_dim == 128)
    return partial ? launch_prefill_t<T, 128, true, false>(kmap, vmap, qmap, a, st)
                   : launch_prefill_t<T, 128, false, false>(kmap, vmap, qmap, a, st);
  if (head_dim == 64)
    return partial ? launch_prefill_t<T, 64, true, false>(kmap, vmap, qmap, a, st)
                   : launch_prefill_t<T, 64, false, false>(kmap, vmap, qmap, a, st);
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_prefill(const CUtensorMap &kmap, const CUtensorMap &vmap, const CUtensorMap &qmap,
                           const DecodeArgs &args, int head_dim, bool fp16, bool partial,
                           bool kv8, cudaStream_t stream) {
  return fp16 ? dispatch<__half>(kmap, vmap, qmap, args, head_dim, partial, kv8, stream)
              : dispatch<__nv_bfloat16>(kmap, vmap, qmap, args, head_dim, partial, kv8, stream);
}

}  // namespace pa
