// pa_prefill.cu -- host launchers of the many-row (chunked-prefill / shared-prefix)
// tensor-core kernel for caches of 16-token blocks, both element types.
#include "pa_prefill_inst.cuh"

namespace pa {

cudaError_t launch_prefill(const CUtensorMap &kmap, const CUtensorMap &vmap, const CUtensorMap &qmap,
                           const DecodeArgs &args, int head_dim, bool fp16, bool partial,
                           bool kv8, cudaStream_t stream) {
  return fp16 ? dispatch<true, __half>(kmap, vmap, qmap, args, head_dim, partial, kv8, stream)
              : dispatch<true, __nv_bfloat16>(kmap, vmap, qmap, args, head_dim, partial, kv8, stream);
}

}  // namespace pa
