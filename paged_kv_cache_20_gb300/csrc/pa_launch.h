// pa_launch.h -- internal launch entry points shared by the ABI translation unit
// and the per-dtype kernel translation units (host code only).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

namespace pa {

struct DecodeArgs;
struct CombineArgs;

// rows_per_unit = (num_q_heads / num_kv_heads) * q_len selects the path;
// grid.x = num_seqs * num_kv_heads * num_splits is set by the caller in `units`.
cudaError_t launch_decode_fp16(const CUtensorMap &kmap, const CUtensorMap &vmap,
                               const DecodeArgs &args, int head_dim, bool partial, int units,
                               cudaStream_t stream);
cudaError_t launch_decode_bf16(const CUtensorMap &kmap, const CUtensorMap &vmap,
                               const DecodeArgs &args, int head_dim, bool partial, int units,
                               cudaStream_t stream);
cudaError_t launch_combine_fp16(const CombineArgs &args, int head_dim, cudaStream_t stream);
cudaError_t launch_combine_bf16(const CombineArgs &args, int head_dim, cudaStream_t stream);

}  // namespace pa
