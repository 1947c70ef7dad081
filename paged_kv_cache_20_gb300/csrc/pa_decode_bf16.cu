// pa_decode_bf16.cu -- bf16 instantiations of the decode and combine kernels
// (16-token blocks; pa_decode_blocks_bf16.cu holds those for 8 and 32).
#include "pa_decode_inst.cuh"

namespace pa {
cudaError_t launch_decode_bf16(const CUtensorMap &kmap, const CUtensorMap &vmap,
                               const DecodeArgs &args, int head_dim, bool partial, int units,
                               cudaStream_t stream) {
  return launch_decode_t<16, __nv_bfloat16>(kmap, vmap, args, head_dim, partial, units, stream);
}
cudaError_t launch_combine_bf16(const CombineArgs &args, int head_dim, cudaStream_t stream) {
  return launch_combine_t<__nv_bfloat16>(args, head_dim, stream);
}
cudaError_t launch_decode8_bf16(const CUtensorMap &kmap, const CUtensorMap &vmap,
                                const DecodeArgs &args, bool partial, int units,
                                cudaStream_t stream) {
  return launch_decode8_t<16, __nv_bfloat16>(kmap, vmap, args, partial, units, stream);
}
}  // namespace pa
