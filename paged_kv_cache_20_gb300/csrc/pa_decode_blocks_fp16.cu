// pa_decode_blocks_fp16.cu -- fp16 instantiations of the decode kernels that read
// the cache's block size (8 or 32 tokens) at run time.
#include "pa_decode_inst.cuh"

namespace pa {
cudaError_t launch_decode_fp16_bx(const CUtensorMap &kmap, const CUtensorMap &vmap,
                               const DecodeArgs &args, int head_dim, bool partial, int units,
                               cudaStream_t stream) {
  return launch_decode_t<0, __half>(kmap, vmap, args, head_dim, partial, units, stream);
}
cudaError_t launch_decode8_fp16_bx(const CUtensorMap &kmap, const CUtensorMap &vmap,
                                const DecodeArgs &args, bool partial, int units,
                                cudaStream_t stream) {
  return launch_decode8_t<0, __half>(kmap, vmap, args, partial, units, stream);
}
}  // namespace pa
