// pa_prefill.cu -- host launchers of the many-row (chunked-prefill / shared-prefix)
// tensor-core kernel, both element types.
#include <algorithm>
#include <atomic>

#include "pa_launch.h"
#include "pa_prefill_tc.cuh"

namespace pa {

namespace {

// K and V ring depths (chunks in flight per CTA); with head_dim 128 the rings fill
// what shared memory remains after Q (227 KiB per CTA at most)
template <int D> constexpr int kRingK = D == 128 ? 3 : 4;
template <int D> constexpr int kRingV = D == 128 ? 2 : 4;

template <typename T, int D, bool PARTIAL>
cudaError_t launch_prefill_t(const CUtensorMap &kmap, const CUtensorMap &vmap, const CUtensorMap &qmap,
                             const DecodeArgs &a, cudaStream_t st) {
  constexpr int kSmem = TcLayout<T, D>::smem_bytes(kRingK<D>, kRingV<D>);
  auto kern = paged_prefill_tc_kernel<T, D, kRingK<D>, kRingV<D>, PARTIAL>;
  static std::atomic<unsigned long long> opted{0};  // bit per device: smem opt-in done
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!(opted.load(std::memory_order_acquire) & (1ull << dev))) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e != cudaSuccess) return e;
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
  cfg.blockDim = dim3(kTcThreads, 1, 1);
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
                     const DecodeArgs &a, int head_dim, bool partial, cudaStream_t st) {
  if (head_dim == 128)
    return partial ? launch_prefill_t<T, 128, true>(kmap, vmap, qmap, a, st)
                   : launch_prefill_t<T, 128, false>(kmap, vmap, qmap, a, st);
  if (head_dim == 64)
    return partial ? launch_prefill_t<T, 64, true>(kmap, vmap, qmap, a, st)
                   : launch_prefill_t<T, 64, false>(kmap, vmap, qmap, a, st);
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_prefill(const CUtensorMap &kmap, const CUtensorMap &vmap, const CUtensorMap &qmap,
                           const DecodeArgs &args, int head_dim, bool fp16, bool partial,
                           cudaStream_t stream) {
  return fp16 ? dispatch<__half>(kmap, vmap, qmap, args, head_dim, partial, stream)
              : dispatch<__nv_bfloat16>(kmap, vmap, qmap, args, head_dim, partial, stream);
}

}  // namespace pa
