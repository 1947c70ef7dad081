// pa_launch.h -- internal launch entry points shared by the ABI translation unit
// and the per-dtype kernel translation units (host code only).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

namespace pa {

// Launch `kern` as a programmatic dependent of the previous work on `stream`: it
// may be scheduled before that work finishes, and must call griddepcontrol.wait
// before touching global memory (every kernel of this library does).
template <typename... Params, typename... Args>
cudaError_t launch_dependent(void (*kern)(Params...), dim3 grid, unsigned block,
                             cudaStream_t stream, Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(block, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<Args &&>(args)...);
}

struct DecodeArgs;
struct CombineArgs;

// rows_per_unit = (num_q_heads / num_kv_heads) * q_len selects the path;
// grid.x = num_seqs * num_kv_heads * num_splits is set by the caller in `units`.
// These take a cache of 16-token blocks.
cudaError_t launch_decode_fp16(const CUtensorMap &kmap, const CUtensorMap &vmap,
                               const DecodeArgs &args, int head_dim, bool partial, int units,
                               cudaStream_t stream);
cudaError_t launch_decode_bf16(const CUtensorMap &kmap, const CUtensorMap &vmap,
                               const DecodeArgs &args, int head_dim, bool partial, int units,
                               cudaStream_t stream);
// FP8 (e4m3) cache, head_dim 128; the suffix names the type of q and out.
cudaError_t launch_decode8_fp16(const CUtensorMap &kmap, const CUtensorMap &vmap,
                                const DecodeArgs &args, bool partial, int units,
                                cudaStream_t stream);
cudaError_t launch_decode8_bf16(const CUtensorMap &kmap, const CUtensorMap &vmap,
                                const DecodeArgs &args, bool partial, int units,
                                cudaStream_t stream);
// The same for a cache of 8- or 32-token blocks (the block size read at run time).
cudaError_t launch_decode_fp16_bx(const CUtensorMap &kmap, const CUtensorMap &vmap,
                                  const DecodeArgs &args, int head_dim, bool partial, int units,
                                  cudaStream_t stream);
cudaError_t launch_decode_bf16_bx(const CUtensorMap &kmap, const CUtensorMap &vmap,
                                  const DecodeArgs &args, int head_dim, bool partial, int units,
                                  cudaStream_t stream);
cudaError_t launch_decode8_fp16_bx(const CUtensorMap &kmap, const CUtensorMap &vmap,
                                   const DecodeArgs &args, bool partial, int units,
                                   cudaStream_t stream);
cudaError_t launch_decode8_bf16_bx(const CUtensorMap &kmap, const CUtensorMap &vmap,
                                   const DecodeArgs &args, bool partial, int units,
                                   cudaStream_t stream);
// Many query rows per KV head (q_len above the decode kernel's limit, or the
// shared-prefix pass of a cascade when args.shared_prefix > 0): units of 128 query
// rows of one KV head, walked by persistent CTAs (one per SM, at most
// args.max_ctas when that is positive).  kv8: the cache holds e4m3 codes
// (head_dim 128; fp16 names the type of q and out).
cudaError_t launch_prefill(const CUtensorMap &kmap, const CUtensorMap &vmap, const CUtensorMap &qmap,
                           const DecodeArgs &args, int head_dim, bool fp16, bool partial,
                           bool kv8, cudaStream_t stream);
// The same for a cache of 8- or 32-token blocks.
cudaError_t launch_prefill_bx(const CUtensorMap &kmap, const CUtensorMap &vmap,
                              const CUtensorMap &qmap, const DecodeArgs &args, int head_dim,
                              bool fp16, bool partial, bool kv8, cudaStream_t stream);
cudaError_t launch_combine_fp16(const CombineArgs &args, int head_dim, cudaStream_t stream);
cudaError_t launch_combine_bf16(const CombineArgs &args, int head_dim, cudaStream_t stream);

}  // namespace pa
