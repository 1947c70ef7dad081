// pa_decode_blocks_bf16.cu -- bf16 instantiations of the decode kernels that read
// the cache's block size (8 or 32 tokens) at run time.
#include "pa_decode_inst.cuh"

namespace pa {
cudaError_t launch_decode_bf16_bx(const CUtensorMap &kmap, const CUtensorMap &vmap,
                               const DecodeArgs &args, int head_dim, bool partial, int units,
                               cudaStream_t stream) {
  return launch_decode_t<0, __nv_bfloat16>(kmap, vmap, args, head_dim, partial, units, stream);
}
cudaError_t launch_decode8_bf16_bx(const CUtensorMap &kmap, const CUtensorMap &vmap,
                                const DecodeArgs &args, bool partial, int units,
                                cudaStream_t stream) {
  return launch_decode8_t<0, __nv_bfloat16>(kmap, vmap, args, partial, units, stream);
}
}  // namespace pa
