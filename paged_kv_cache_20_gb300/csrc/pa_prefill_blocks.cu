// pa_prefill_blocks.cu -- host launchers of the many-row tensor-core kernel for
// caches of 8- or 32-token blocks (the block size read at run time).
#include "pa_prefill_inst.cuh"

namespace pa {

cudaError_t launch_prefill_bx(const CUtensorMap &kmap, const CUtensorMap &vmap,
                              const CUtensorMap &qmap, const DecodeArgs &args, int head_dim,
                              bool fp16, bool partial, bool kv8, cudaStream_t stream) {
  return fp16 ? dispatch<false, __half>(kmap, vmap, qmap, args, head_dim, partial, kv8, stream)
              : dispatch<false, __nv_bfloat16>(kmap, vmap, qmap, args, head_dim, partial, kv8, stream);
}

}  // namespace pa
