// pa_api.cu -- the C ABI of libpagedattn.so: argument validation, TMA tensor-map
// encoding, launch dispatch, the per-device error word, and the two small
// scatter kernels (slot mapping and KV append).
//
// Slot arithmetic and append follow "LLM 推理优化全景实战：从 PagedAttention 到投机解码"
// §2.3 (write_kv: logical_block = pos // block_size, block_offset = pos % block_size,
// physical block from the request's page table) and "09-inference-optimization.md"
// (LLM-Code-Hot-100), PagedKVCache.append_token (write the new token's K/V into
// its slot of the last page).
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "../../include/pagedattn.h"
#include "pa_decode.cuh"
#include "pa_launch.h"

namespace {

// Block sizes the kernels take: a block of 32 tokens is read as two 16-token tiles,
// a 16-token tile spans two blocks of 8
bool supported_block(int b) { return b == 8 || b == 16 || b == 32; }
constexpr int kMaxDevices = 64;
constexpr int kMaxQLen = 4096;       // query rows per sequence accepted by the ABI
constexpr int kMaxDecodeQLen = 16;   // at most this many go to the decode kernel
// Share of the SMs a cascade's shared-prefix pass runs on (num / den); the rest
// serve the tail pass that overlaps it.  Measured on 128 sequences sharing a
// 1024-token prefix (q_len 4, 32/8 heads): 152, 128, 96, 76, 64, 48 and 38 prefix
// CTAs gave 112.2, 112.4, 103.2, 100.7, 104.4, 110.4 and 117.7 us per step; after
// a shorter decode prologue, 68, 72, 76, 80 and 84 gave 103.4, 101.9, 101.0, 100.4
// and 100.5 us.
constexpr int kCascadePrefixShareNum = 10;
constexpr int kCascadePrefixShareDen = 19;

__device__ unsigned int g_error_word;  // one per device (module global)

// ---- scatter kernels ---------------------------------------------------------------

__global__ void slot_mapping_kernel(int64_t *out, const int32_t *block_tables,
                                    const int32_t *context_lens, int num_seqs,
                                    int max_blocks_per_seq, int block_size, int q_len,
                                    unsigned *err) {
  pa::griddep_wait();  // inputs may come from the previous kernel on the stream
  pa::griddep_launch_dependents();
  const int idx = blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= num_seqs * q_len) return;
  const int i = idx / q_len, u = idx % q_len;
  const int64_t pos = (int64_t)context_lens[i] - q_len + u;
  int64_t slot = -1;
  if (pos >= 0) {
    const int64_t logical_block = pos / block_size;
    if (logical_block < max_blocks_per_seq) {
      const int64_t physical_block = block_tables[(int64_t)i * max_blocks_per_seq + logical_block];
      slot = physical_block * block_size + pos % block_size;
    } else {
      pa::record_error(err, pa::kErrCheck);
    }
  }
  out[idx] = slot;
}

// The appends: one CTA per new token row (its slot worked out once), its threads
// over the (head, 16-byte chunk) pieces of that row, K and V together.
inline unsigned append_threads(int num_kv_heads, int head_dim) {
  const int pieces = num_kv_heads * (head_dim / 8);
  return (unsigned)std::min(1024, (pieces + 31) / 32 * 32);
}

// Row t of k_new / v_new (all heads) into block blk, row off of every head.
template <int D>
__device__ __forceinline__ void append_row(uint16_t *__restrict__ k_cache,
                                           uint16_t *__restrict__ v_cache,
                                           const uint16_t *__restrict__ k_new,
                                           const uint16_t *__restrict__ v_new, int64_t t,
                                           int num_kv_heads, int block_size, int64_t blk, int off) {
  constexpr int kChunks = D / 8;
  for (int hc = threadIdx.x; hc < num_kv_heads * kChunks; hc += blockDim.x) {
    const int h = hc / kChunks, c = hc % kChunks;
    const int64_t dst = ((blk * num_kv_heads + h) * block_size + off) * D + c * 8;
    const int64_t src = (t * num_kv_heads + h) * D + c * 8;
    const uint4 kv = __ldg(reinterpret_cast<const uint4 *>(k_new + src));
    const uint4 vv = __ldg(reinterpret_cast<const uint4 *>(v_new + src));
    *reinterpret_cast<uint4 *>(k_cache + dst) = kv;
    *reinterpret_cast<uint4 *>(v_cache + dst) = vv;
  }
}

// The same into an FP8 cache, quantising: code = e4m3(x / scale[head]).
template <typename T, int D>
__device__ __forceinline__ void append_row_fp8(uint8_t *__restrict__ k_cache,
                                               uint8_t *__restrict__ v_cache,
                                               const uint16_t *__restrict__ k_new,
                                               const uint16_t *__restrict__ v_new, int64_t t,
                                               int num_kv_heads, int block_size, int64_t blk,
                                               int off, const float *k_scale,
                                               const float *v_scale) {
  constexpr int kChunks = D / 8;
  for (int hc = threadIdx.x; hc < num_kv_heads * kChunks; hc += blockDim.x) {
    const int h = hc / kChunks, c = hc % kChunks;
    const int64_t dst = ((blk * num_kv_heads + h) * block_size + off) * D + c * 8;
    const int64_t src = (t * num_kv_heads + h) * D + c * 8;
    const uint4 kv = __ldg(reinterpret_cast<const uint4 *>(k_new + src));
    const uint4 vv = __ldg(reinterpret_cast<const uint4 *>(v_new + src));
    *reinterpret_cast<uint2 *>(k_cache + dst) = pa::quantize8<T>(kv, __ldg(k_scale + h));
    *reinterpret_cast<uint2 *>(v_cache + dst) = pa::quantize8<T>(vv, __ldg(v_scale + h));
  }
}

// Append through a slot mapping: CTA t takes token row t.
template <int D>
__global__ void append_kv_kernel(uint16_t *k_cache, uint16_t *v_cache, const uint16_t *k_new,
                                 const uint16_t *v_new, const int64_t *slot_mapping, int n_tokens,
                                 int num_kv_heads, int block_size, int64_t num_slots, unsigned *err) {
  pa::griddep_wait();  // the slot mapping may come from the previous kernel
  pa::griddep_launch_dependents();
  const int64_t t = blockIdx.x;
  const int64_t slot = slot_mapping[t];
  if (slot < 0) return;
  if (slot >= num_slots) {
    if (threadIdx.x == 0) pa::record_error(err, pa::kErrCheck);
    return;
  }
  const int64_t blk = slot / block_size;
  append_row<D>(k_cache, v_cache, k_new, v_new, t, num_kv_heads, block_size, blk,
                (int)(slot - blk * block_size));
}

// Append of one step's new rows straight from the block tables: token u of
// sequence i sits at position context_lens[i] - q_len + u (the slot of the slot
// mapping kernel, computed in place).  CTA t takes token row t = i * q_len + u.
// Returns the row's block (-1: nothing to write).
__device__ __forceinline__ int64_t step_slot_block(const int32_t *block_tables,
                                                   const int32_t *context_lens, int q_len,
                                                   int block_size, int max_blocks_per_seq,
                                                   int64_t num_slots, unsigned *err, int &off) {
  const int t = blockIdx.x;
  const int i = t / q_len, u = t - i * q_len;
  const int64_t pos = (int64_t)context_lens[i] - q_len + u;
  if (pos < 0) return -1;
  const int64_t lb = pos / block_size;
  if (lb >= max_blocks_per_seq) {
    if (threadIdx.x == 0) pa::record_error(err, pa::kErrCheck);
    return -1;
  }
  const int64_t slot =
      (int64_t)block_tables[(int64_t)i * max_blocks_per_seq + lb] * block_size +
      (pos - lb * block_size);
  if (slot < 0 || slot >= num_slots) {
    if (threadIdx.x == 0) pa::record_error(err, pa::kErrCheck);
    return -1;
  }
  const int64_t blk = slot / block_size;
  off = (int)(slot - blk * block_size);
  return blk;
}

template <int D>
__global__ void append_step_kernel(uint16_t *k_cache, uint16_t *v_cache, const uint16_t *k_new,
                                   const uint16_t *v_new, const int32_t *block_tables,
                                   const int32_t *context_lens, int num_seqs, int q_len,
                                   int num_kv_heads, int block_size, int max_blocks_per_seq,
                                   int64_t num_slots, unsigned *err) {
  pa::griddep_wait();
  pa::griddep_launch_dependents();
  int off = 0;
  const int64_t blk = step_slot_block(block_tables, context_lens, q_len, block_size,
                                      max_blocks_per_seq, num_slots, err, off);
  if (blk < 0) return;
  append_row<D>(k_cache, v_cache, k_new, v_new, blockIdx.x, num_kv_heads, block_size, blk, off);
}

// The same append into an FP8 cache, quantising: code = e4m3(x / scale[head]).
template <typename T, int D>
__global__ void append_step_fp8_kernel(uint8_t *k_cache, uint8_t *v_cache, const uint16_t *k_new,
                                       const uint16_t *v_new, const int32_t *block_tables,
                                       const int32_t *context_lens, int num_seqs, int q_len,
                                       int num_kv_heads, int block_size, int max_blocks_per_seq,
                                       int64_t num_slots, const float *k_scale,
                                       const float *v_scale, unsigned *err) {
  pa::griddep_wait();
  pa::griddep_launch_dependents();
  int off = 0;
  const int64_t blk = step_slot_block(block_tables, context_lens, q_len, block_size,
                                      max_blocks_per_seq, num_slots, err, off);
  if (blk < 0) return;
  append_row_fp8<T, D>(k_cache, v_cache, k_new, v_new, blockIdx.x, num_kv_heads, block_size, blk,
                       off, k_scale, v_scale);
}

// Quantising append into an FP8 cache through a slot mapping: CTA t takes token row t.
template <typename T, int D>
__global__ void append_kv_fp8_kernel(uint8_t *k_cache, uint8_t *v_cache, const uint16_t *k_new,
                                     const uint16_t *v_new, const int64_t *slot_mapping,
                                     int n_tokens, int num_kv_heads, int block_size,
                                     int64_t num_slots, const float *k_scale,
                                     const float *v_scale, unsigned *err) {
  pa::griddep_wait();
  pa::griddep_launch_dependents();
  const int64_t t = blockIdx.x;
  const int64_t slot = slot_mapping[t];
  if (slot < 0) return;
  if (slot >= num_slots) {
    if (threadIdx.x == 0) pa::record_error(err, pa::kErrCheck);
    return;
  }
  const int64_t blk = slot / block_size;
  append_row_fp8<T, D>(k_cache, v_cache, k_new, v_new, t, num_kv_heads, block_size, blk,
                       (int)(slot - blk * block_size), k_scale, v_scale);
}

// Copy-on-write block copy.  Pair i = blockIdx.y (+ gridDim.y steps); each thread
// copies kCopyUnroll 16-byte chunks of the block's K and of its V, blockDim.x
// chunks apart, with all of its loads issued before its stores (eight 16-byte
// loads in flight per thread).
constexpr int kCopyUnroll = 4;
constexpr int kCopyThreads = 256;
__global__ void __launch_bounds__(kCopyThreads)
    copy_blocks_kernel(uint4 *k_cache, uint4 *v_cache, const int32_t *src, const int32_t *dst,
                       int n_pairs, int64_t chunks_per_block, int num_blocks, unsigned *err) {
  pa::griddep_wait();
  pa::griddep_launch_dependents();
  const int64_t c0 = (int64_t)blockIdx.x * (kCopyThreads * kCopyUnroll) + threadIdx.x;
  for (int i = blockIdx.y; i < n_pairs; i += gridDim.y) {
    const int s = __ldg(src + i), d = __ldg(dst + i);
    if (s < 0 || s >= num_blocks || d < 0 || d >= num_blocks) {
      if (blockIdx.x == 0 && threadIdx.x == 0) pa::record_error(err, pa::kErrCheck);
      continue;
    }
    const uint4 *ks = k_cache + (int64_t)s * chunks_per_block;
    const uint4 *vs = v_cache + (int64_t)s * chunks_per_block;
    uint4 *kd = k_cache + (int64_t)d * chunks_per_block;
    uint4 *vd = v_cache + (int64_t)d * chunks_per_block;
    uint4 kv[kCopyUnroll], vv[kCopyUnroll];
#pragma unroll
    for (int u = 0; u < kCopyUnroll; ++u) {
      const int64_t c = c0 + u * kCopyThreads;
      if (c < chunks_per_block) {
        kv[u] = ks[c];
        vv[u] = vs[c];
      }
    }
#pragma unroll
    for (int u = 0; u < kCopyUnroll; ++u) {
      const int64_t c = c0 + u * kCopyThreads;
      if (c < chunks_per_block) {
        kd[c] = kv[u];
        vd[c] = vv[u];
      }
    }
  }
}

// A wait nobody satisfies: an mbarrier expecting one arrival that never comes.
__global__ void wait_timeout_kernel(unsigned *err) {
  __shared__ __align__(8) uint64_t bar;
  const uint32_t b = pa::smem_u32(&bar);
  pa::mbar_init(b, 1);
  pa::fence_mbar_init();
  if (!pa::mbar_wait_bounded(b, 0)) pa::record_error(err, pa::kErrTimeout);
}

// ---- host helpers --------------------------------------------------------------------

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

void load_encode() {
  void *fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                       &q) == cudaSuccess &&
      q == cudaDriverEntryPointSuccess)
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
}

std::mutex g_err_mutex;
unsigned *g_err_ptr[kMaxDevices] = {};

// Device address of this device's error word (looked up once per device).
unsigned *error_word() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_err_mutex);
  if (g_err_ptr[dev] == nullptr) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_error_word) != cudaSuccess) return nullptr;
    g_err_ptr[dev] = static_cast<unsigned *>(p);
  }
  return g_err_ptr[dev];
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool supported_dtype(pa_dtype d) { return d == PA_FP16 || d == PA_BF16; }

// Tensor map over one cache: [num_blocks * num_kv_heads tiles][16 rows][head_dim],
// box = 16 rows x 64 columns, 128-byte swizzle, zero fill outside.
// Tensor map over a cache [num_blocks][num_kv_heads][block_size][head_dim] as
// [head_dim, R, num_blocks * num_kv_heads * block_size / R] with R = min(block_size,
// 16) rows per box: a (block, head) pair of a 32-token block is two consecutive
// 16-row boxes; an 8-token block is one 8-row box.  128-byte rows, 128-byte swizzle.
pa_status make_map(CUtensorMap *map, const void *cache, pa_dtype dtype, int head_dim,
                   int num_blocks, int num_kv_heads, int block_size, bool fp8 = false) {
  std::call_once(g_encode_once, load_encode);
  if (g_encode == nullptr) return PA_ERR_CUDA;
  const int elt = fp8 ? 1 : 2;
  const int rows = block_size < 16 ? block_size : 16;
  cuuint64_t dims[3] = {(cuuint64_t)head_dim, (cuuint64_t)rows,
                        (cuuint64_t)num_blocks * (cuuint64_t)num_kv_heads * (block_size / rows)};
  cuuint64_t strides[2] = {(cuuint64_t)head_dim * elt, (cuuint64_t)rows * head_dim * elt};
  cuuint32_t box[3] = {(cuuint32_t)(128 / elt), (cuuint32_t)rows, 1};  // 128-byte rows
  cuuint32_t elem_strides[3] = {1, 1, 1};
  const CUtensorMapDataType ty = fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                     : (dtype == PA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                         : CU_TENSOR_MAP_DATA_TYPE_FLOAT16);
  CUresult r = g_encode(map, ty, 3, const_cast<void *>(cache), dims, strides, box, elem_strides,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? PA_OK : PA_ERR_CUDA;
}

// Tensor map over q [tokens][num_q_heads][head_dim] as [head_dim, num_q_heads,
// tokens], box = 64 columns x `group` heads x 128/group tokens: the 128 query rows
// (token, head) of one KV head's row block, 128-byte swizzle, zero fill outside.
pa_status make_q_map(CUtensorMap *map, const void *q, pa_dtype dtype, int head_dim,
                     int num_q_heads, int64_t tokens, int group) {
  std::call_once(g_encode_once, load_encode);
  if (g_encode == nullptr) return PA_ERR_CUDA;
  cuuint64_t dims[3] = {(cuuint64_t)head_dim, (cuuint64_t)num_q_heads, (cuuint64_t)tokens};
  cuuint64_t strides[2] = {(cuuint64_t)head_dim * 2, (cuuint64_t)num_q_heads * head_dim * 2};
  cuuint32_t box[3] = {64u, (cuuint32_t)group, (cuuint32_t)(128 / group)};
  cuuint32_t elem_strides[3] = {1, 1, 1};
  CUresult r = g_encode(map, dtype == PA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                        3, const_cast<void *>(q), dims, strides, box, elem_strides,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? PA_OK : PA_ERR_CUDA;
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

struct WsLayout {
  size_t acc_off, m_off, l_off, total;
};

WsLayout ws_layout(int num_seqs, int num_q_heads, int q_len, int head_dim, int num_splits) {
  const size_t rows = (size_t)num_seqs * num_splits * q_len * num_q_heads;
  WsLayout w;
  w.acc_off = 0;
  w.m_off = align256(rows * head_dim * sizeof(float));
  w.l_off = w.m_off + align256(rows * sizeof(float));
  w.total = w.l_off + align256(rows * sizeof(float));
  return w;
}

// Checks shared by pa_decode and pa_decode_partial.
pa_status check_decode(const void *q, const void *k_cache, const void *v_cache,
                       const int32_t *block_tables, const int32_t *context_lens, int num_seqs,
                       int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                       float scale, int max_blocks_per_seq, int num_blocks, int q_len,
                       pa_dtype dtype) {
  if (!q || !k_cache || !v_cache || !block_tables || !context_lens) return PA_ERR_INVALID_ARG;
  if (num_seqs <= 0 || num_q_heads <= 0 || num_kv_heads <= 0 || max_blocks_per_seq <= 0 ||
      num_blocks <= 0 || q_len <= 0 || head_dim <= 0 || block_size <= 0)
    return PA_ERR_INVALID_ARG;
  if (num_q_heads % num_kv_heads != 0) return PA_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return PA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache)) return PA_ERR_INVALID_ARG;
  if (!supported_dtype(dtype)) return PA_ERR_UNSUPPORTED;
  if (head_dim != 64 && head_dim != 128) return PA_ERR_UNSUPPORTED;
  if (!supported_block(block_size)) return PA_ERR_UNSUPPORTED;
  if (q_len > kMaxQLen) return PA_ERR_UNSUPPORTED;
  // 32-bit index limits used by the kernels
  if ((int64_t)num_blocks * num_kv_heads * 2 >= (int64_t)1 << 31) return PA_ERR_INVALID_ARG;
  if ((int64_t)num_seqs * max_blocks_per_seq * 2 >= (int64_t)1 << 31) return PA_ERR_INVALID_ARG;
  if ((int64_t)max_blocks_per_seq * block_size >= (int64_t)1 << 31) return PA_ERR_INVALID_ARG;
  if ((int64_t)num_seqs * q_len * num_q_heads >= (int64_t)1 << 31) return PA_ERR_INVALID_ARG;
  return PA_OK;
}

// Where a launch's partitions go inside a workspace shared with other passes (the
// cascade): the sequence's partitions start at its block first_block, and the
// launch writes workspace partitions [ws_split0, ws_split0 + num_splits) of
// ws_splits.  shared_prefix > 0 selects the shared-prefix pass.
struct Placement {
  int first_block = 0;
  int ws_splits = 0;  // 0: num_splits
  int ws_split0 = 0;
  int shared_prefix = 0;
  int max_ctas = 0;  // prefill kernel: cap on its persistent grid (0: one CTA per SM)
  // single pass: merge partition 0 of this workspace (prior_splits partitions) into
  // the result
  const float *prior_ws = nullptr;
  const WsLayout *prior_lay = nullptr;
  int prior_splits = 0;
};

// CTAs of a cascade's shared-prefix pass: a share of the SMs, so that the tail
// pass, which overlaps it, keeps the rest (a prefill CTA fills its SM).
int cascade_prefix_ctas() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return 0;
  return sms * kCascadePrefixShareNum / kCascadePrefixShareDen;
}

pa_status decode_common(void *out, float *ws, const WsLayout *lay, const void *q,
                        const void *k_cache, const void *v_cache, const int32_t *block_tables,
                        const int32_t *context_lens, int num_seqs, int num_q_heads,
                        int num_kv_heads, int head_dim, int block_size, float scale, int num_splits,
                        int max_blocks_per_seq, int num_blocks, int q_len, pa_dtype dtype,
                        void *stream, const void *k_new = nullptr, const void *v_new = nullptr,
                        const float *k_scale = nullptr, const float *v_scale = nullptr,
                        const Placement &place = Placement()) {
  const int64_t units = (int64_t)num_seqs * num_kv_heads * num_splits;
  if (units >= (int64_t)1 << 31) return PA_ERR_INVALID_ARG;
  const bool fp8 = k_scale != nullptr;
  // many query rows (or the shared-prefix pass): the CTA-shared pipeline kernel,
  // over a 16-bit or an FP8 cache
  if (fp8 && place.shared_prefix > 0) return PA_ERR_UNSUPPORTED;
  const bool prefill = place.shared_prefix > 0 || q_len > kMaxDecodeQLen;
  CUtensorMap kmap, vmap;
  pa_status st = make_map(&kmap, k_cache, dtype, head_dim, num_blocks, num_kv_heads, block_size, fp8);
  if (st != PA_OK) return st;
  st = make_map(&vmap, v_cache, dtype, head_dim, num_blocks, num_kv_heads, block_size, fp8);
  if (st != PA_OK) return st;
  pa::DecodeArgs a;
  a.q = q;
  a.out = out;
  a.ws_acc = ws ? reinterpret_cast<float *>(reinterpret_cast<char *>(ws) + lay->acc_off) : nullptr;
  a.ws_m = ws ? reinterpret_cast<float *>(reinterpret_cast<char *>(ws) + lay->m_off) : nullptr;
  a.ws_l = ws ? reinterpret_cast<float *>(reinterpret_cast<char *>(ws) + lay->l_off) : nullptr;
  a.block_tables = block_tables;
  a.context_lens = context_lens;
  a.err = error_word();
  if (a.err == nullptr) return PA_ERR_CUDA;
  a.num_seqs = num_seqs;
  a.num_q_heads = num_q_heads;
  a.num_kv_heads = num_kv_heads;
  a.q_len = q_len;
  a.group = num_q_heads / num_kv_heads;
  a.rows = a.group * q_len;
  a.max_blocks_per_seq = max_blocks_per_seq;
  a.block_size = block_size;
  a.max_tiles = (int)(((int64_t)max_blocks_per_seq * block_size + pa::kTileTokens - 1) /
                      pa::kTileTokens);
  a.num_blocks = num_blocks;
  a.num_splits = num_splits;
  a.lpt = num_seqs <= pa::kLptMaxSeqs ? 1 : 0;
  a.k_new = static_cast<const uint16_t *>(k_new);
  a.v_new = static_cast<const uint16_t *>(v_new);
  a.k_cache = static_cast<uint16_t *>(const_cast<void *>(k_cache));
  a.v_cache = static_cast<uint16_t *>(const_cast<void *>(v_cache));
  a.k_scale = k_scale;
  a.v_scale = v_scale;
  // (the callers' block counts cover whole 16-token tiles)
  a.first_block = place.first_block * block_size / pa::kTileTokens;
  a.ws_splits = place.ws_splits > 0 ? place.ws_splits : num_splits;
  a.ws_split0 = place.ws_split0;
  a.shared_prefix = place.shared_prefix * block_size / pa::kTileTokens;
  a.max_ctas = place.max_ctas;
  a.q_tma = 0;
  a.s_negate = 0;
  a.prior_splits = place.prior_splits;
  if (place.prior_ws != nullptr) {
    const char *pb = reinterpret_cast<const char *>(place.prior_ws);
    a.prior_acc = reinterpret_cast<const float *>(pb + place.prior_lay->acc_off);
    a.prior_m = reinterpret_cast<const float *>(pb + place.prior_lay->m_off);
    a.prior_l = reinterpret_cast<const float *>(pb + place.prior_lay->l_off);
  } else {
    a.prior_acc = a.prior_m = a.prior_l = nullptr;
  }
  a.scale_log2 = scale * 1.4426950408889634f;  // log2(e)
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const bool partial = ws != nullptr;
  cudaError_t e;
  if (prefill) {
    if (k_new != nullptr) {
      // The rows of a CTA depend on new tokens that other CTAs' rows own, so the
      // append runs as its own launch first (ordered by the stream).
      const unsigned blocks = (unsigned)(num_seqs * q_len);  // one CTA per token row
      const unsigned threads = append_threads(num_kv_heads, head_dim);
      const int64_t num_slots = (int64_t)num_blocks * block_size;
      auto kn = static_cast<const uint16_t *>(k_new);
      auto vn = static_cast<const uint16_t *>(v_new);
      if (fp8) {  // quantising (head_dim 128)
        auto kc8 = static_cast<uint8_t *>(const_cast<void *>(k_cache));
        auto vc8 = static_cast<uint8_t *>(const_cast<void *>(v_cache));
        e = dtype == PA_FP16
                ? pa::launch_dependent(append_step_fp8_kernel<__half, 128>, blocks, threads, s,
                                       kc8, vc8, kn, vn, block_tables, context_lens, num_seqs, q_len,
                                       num_kv_heads, block_size, max_blocks_per_seq, num_slots,
                                       k_scale, v_scale, a.err)
                : pa::launch_dependent(append_step_fp8_kernel<__nv_bfloat16, 128>, blocks,
                                       threads, s, kc8, vc8, kn, vn, block_tables, context_lens, num_seqs,
                                       q_len, num_kv_heads, block_size, max_blocks_per_seq,
                                       num_slots, k_scale, v_scale, a.err);
      } else {
        auto kc = static_cast<uint16_t *>(const_cast<void *>(k_cache));
        auto vc = static_cast<uint16_t *>(const_cast<void *>(v_cache));
        e = head_dim == 128
                ? pa::launch_dependent(append_step_kernel<128>, blocks, threads, s, kc, vc, kn, vn,
                                       block_tables, context_lens, num_seqs, q_len, num_kv_heads,
                                       block_size, max_blocks_per_seq, num_slots, a.err)
                : pa::launch_dependent(append_step_kernel<64>, blocks, threads, s, kc, vc, kn, vn,
                                       block_tables, context_lens, num_seqs, q_len, num_kv_heads,
                                       block_size, max_blocks_per_seq, num_slots, a.err);
      }
      if (e != cudaSuccess) return PA_ERR_CUDA;
      a.k_new = a.v_new = nullptr;
    }
    // The prefill kernel scales scores inside exp2's argument (one multiply-add),
    // which needs a positive scale: a negative one negates Q K^T in the MMA instead,
    // and a zero one (every visible weight equal) becomes one too small to move an
    // exponent of a finite score
    if (a.scale_log2 < 0.f) {
      a.s_negate = 1;
      a.scale_log2 = -a.scale_log2;
    }
    if (a.scale_log2 == 0.f) a.scale_log2 = 1e-30f;
    CUtensorMap qmap;
    // (over an FP8 cache a bf16 q is converted to fp16 by the softmax threads)
    a.q_tma = (128 % a.group == 0 && !(fp8 && dtype == PA_BF16)) ? 1 : 0;
    if (a.q_tma) {
      st = make_q_map(&qmap, q, dtype, head_dim, num_q_heads, (int64_t)num_seqs * q_len, a.group);
      if (st != PA_OK) return st;
    } else {
      qmap = kmap;  // unused
    }
    e = block_size == 16
            ? pa::launch_prefill(kmap, vmap, qmap, a, head_dim, dtype == PA_FP16, partial, fp8, s)
            : pa::launch_prefill_bx(kmap, vmap, qmap, a, head_dim, dtype == PA_FP16, partial, fp8, s);
  } else if (fp8 && block_size == 16)
    e = dtype == PA_FP16 ? pa::launch_decode8_fp16(kmap, vmap, a, partial, (int)units, s)
                         : pa::launch_decode8_bf16(kmap, vmap, a, partial, (int)units, s);
  else if (fp8)
    e = dtype == PA_FP16 ? pa::launch_decode8_fp16_bx(kmap, vmap, a, partial, (int)units, s)
                         : pa::launch_decode8_bf16_bx(kmap, vmap, a, partial, (int)units, s);
  else if (block_size == 16)
    e = dtype == PA_FP16 ? pa::launch_decode_fp16(kmap, vmap, a, head_dim, partial, (int)units, s)
                         : pa::launch_decode_bf16(kmap, vmap, a, head_dim, partial, (int)units, s);
  else
    e = dtype == PA_FP16 ? pa::launch_decode_fp16_bx(kmap, vmap, a, head_dim, partial, (int)units, s)
                         : pa::launch_decode_bf16_bx(kmap, vmap, a, head_dim, partial, (int)units, s);
  return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

}  // namespace

extern "C" {

PA_API const char *pa_status_string(pa_status status) {
  switch (status) {
    case PA_OK: return "PA_OK";
    case PA_ERR_INVALID_ARG: return "PA_ERR_INVALID_ARG";
    case PA_ERR_UNSUPPORTED: return "PA_ERR_UNSUPPORTED";
    case PA_ERR_CUDA: return "PA_ERR_CUDA";
    case PA_ERR_DEVICE_CHECK: return "PA_ERR_DEVICE_CHECK";
    case PA_ERR_DEVICE_TIMEOUT: return "PA_ERR_DEVICE_TIMEOUT";
  }
  return "PA_UNKNOWN_STATUS";
}

PA_API int pa_version(void) { return 100; }

PA_API pa_status pa_slot_mapping(int64_t *slot_mapping, const int32_t *block_tables,
                                 const int32_t *context_lens, int num_seqs,
                                 int max_blocks_per_seq, int block_size, int q_len,
                                 void *stream) {
  if (!slot_mapping || !block_tables || !context_lens) return PA_ERR_INVALID_ARG;
  if (num_seqs <= 0 || max_blocks_per_seq <= 0 || block_size <= 0 || q_len <= 0)
    return PA_ERR_INVALID_ARG;
  if (!supported_block(block_size)) return PA_ERR_UNSUPPORTED;
  if ((int64_t)num_seqs * q_len >= (int64_t)1 << 31 ||
      (int64_t)num_seqs * max_blocks_per_seq >= (int64_t)1 << 31)
    return PA_ERR_INVALID_ARG;
  unsigned *err = error_word();
  if (err == nullptr) return PA_ERR_CUDA;
  const int n = num_seqs * q_len;
  cudaError_t e = pa::launch_dependent(slot_mapping_kernel, (n + 255) / 256, 256,
                                       static_cast<cudaStream_t>(stream), slot_mapping,
                                       block_tables, context_lens, num_seqs, max_blocks_per_seq,
                                       block_size, q_len, err);
  return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

PA_API pa_status pa_append_kv(void *k_cache, void *v_cache, const void *k_new, const void *v_new,
                              const int64_t *slot_mapping, int n_tokens, int num_kv_heads,
                              int head_dim, int block_size, int num_blocks, pa_dtype dtype,
                              void *stream) {
  if (!k_cache || !v_cache || !k_new || !v_new || !slot_mapping) return PA_ERR_INVALID_ARG;
  if (n_tokens < 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 || num_blocks <= 0)
    return PA_ERR_INVALID_ARG;
  if (!aligned16(k_cache) || !aligned16(v_cache) || !aligned16(k_new) || !aligned16(v_new))
    return PA_ERR_INVALID_ARG;
  if (!supported_dtype(dtype)) return PA_ERR_UNSUPPORTED;
  if (head_dim != 64 && head_dim != 128) return PA_ERR_UNSUPPORTED;
  if (!supported_block(block_size)) return PA_ERR_UNSUPPORTED;
  if (n_tokens == 0) return PA_OK;
  unsigned *err = error_word();
  if (err == nullptr) return PA_ERR_CUDA;
  const unsigned blocks = (unsigned)n_tokens;  // one CTA per token row
  const unsigned threads = append_threads(num_kv_heads, head_dim);
  const int64_t num_slots = (int64_t)num_blocks * block_size;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  auto kc = static_cast<uint16_t *>(k_cache);
  auto vc = static_cast<uint16_t *>(v_cache);
  auto kn = static_cast<const uint16_t *>(k_new);
  auto vn = static_cast<const uint16_t *>(v_new);
  cudaError_t e = head_dim == 128
                      ? pa::launch_dependent(append_kv_kernel<128>, blocks, threads, s, kc, vc, kn,
                                             vn, slot_mapping, n_tokens, num_kv_heads, block_size,
                                             num_slots, err)
                      : pa::launch_dependent(append_kv_kernel<64>, blocks, threads, s, kc, vc, kn,
                                             vn, slot_mapping, n_tokens, num_kv_heads, block_size,
                                             num_slots, err);
  return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

PA_API pa_status pa_copy_blocks(void *k_cache, void *v_cache, const int32_t *src_blocks,
                                const int32_t *dst_blocks, int n_pairs, int num_kv_heads,
                                int head_dim, int block_size, int num_blocks, pa_dtype dtype,
                                void *stream) {
  if (!k_cache || !v_cache || !src_blocks || !dst_blocks) return PA_ERR_INVALID_ARG;
  if (n_pairs < 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 || num_blocks <= 0)
    return PA_ERR_INVALID_ARG;
  if (!aligned16(k_cache) || !aligned16(v_cache)) return PA_ERR_INVALID_ARG;
  if (!supported_dtype(dtype)) return PA_ERR_UNSUPPORTED;
  if (head_dim != 64 && head_dim != 128) return PA_ERR_UNSUPPORTED;
  if (!supported_block(block_size)) return PA_ERR_UNSUPPORTED;
  if (n_pairs == 0) return PA_OK;
  unsigned *err = error_word();
  if (err == nullptr) return PA_ERR_CUDA;
  const int64_t chunks = (int64_t)num_kv_heads * block_size * head_dim * 2 / 16;
  // x: the chunks of one block; y: the pairs (further pairs loop)
  const int64_t per_cta = (int64_t)kCopyThreads * kCopyUnroll;
  const dim3 blocks((unsigned)((chunks + per_cta - 1) / per_cta),
                    (unsigned)std::min(n_pairs, 65535), 1);
  cudaError_t e = pa::launch_dependent(copy_blocks_kernel, blocks, kCopyThreads,
                                       static_cast<cudaStream_t>(stream),
                                       static_cast<uint4 *>(k_cache), static_cast<uint4 *>(v_cache),
                                       src_blocks, dst_blocks, n_pairs, chunks, num_blocks, err);
  return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

PA_API pa_status pa_decode(void *out, const void *q, const void *k_cache, const void *v_cache,
                           const int32_t *block_tables, const int32_t *context_lens,
                           int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                           int block_size, float scale, void *stream, int max_blocks_per_seq,
                           int num_blocks, int q_len, pa_dtype dtype) {
  if (!out || !aligned16(out)) return PA_ERR_INVALID_ARG;
  pa_status st = check_decode(q, k_cache, v_cache, block_tables, context_lens, num_seqs,
                              num_q_heads, num_kv_heads, head_dim, block_size, scale,
                              max_blocks_per_seq, num_blocks, q_len, dtype);
  if (st != PA_OK) return st;
  return decode_common(out, nullptr, nullptr, q, k_cache, v_cache, block_tables, context_lens,
                       num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, scale, 1,
                       max_blocks_per_seq, num_blocks, q_len, dtype, stream);
}

PA_API pa_status pa_append_decode(void *out, const void *q, const void *k_new, const void *v_new,
                                  void *k_cache, void *v_cache, const int32_t *block_tables,
                                  const int32_t *context_lens, int num_seqs, int num_q_heads,
                                  int num_kv_heads, int head_dim, int block_size, float scale,
                                  int max_blocks_per_seq, int num_blocks, int q_len,
                                  pa_dtype dtype, int num_splits, void *workspace,
                                  size_t workspace_bytes, void *stream) {
  if (!out || !aligned16(out) || !k_new || !v_new || !aligned16(k_new) || !aligned16(v_new))
    return PA_ERR_INVALID_ARG;
  if (num_splits <= 0) return PA_ERR_INVALID_ARG;
  pa_status st = check_decode(q, k_cache, v_cache, block_tables, context_lens, num_seqs,
                              num_q_heads, num_kv_heads, head_dim, block_size, scale,
                              max_blocks_per_seq, num_blocks, q_len, dtype);
  if (st != PA_OK) return st;
  if (num_splits == 1)
    return decode_common(out, nullptr, nullptr, q, k_cache, v_cache, block_tables, context_lens,
                         num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, scale, 1,
                         max_blocks_per_seq, num_blocks, q_len, dtype, stream, k_new, v_new);
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return PA_ERR_INVALID_ARG;
  const WsLayout lay = ws_layout(num_seqs, num_q_heads, q_len, head_dim, num_splits);
  if (workspace_bytes < lay.total) return PA_ERR_INVALID_ARG;
  st = decode_common(nullptr, static_cast<float *>(workspace), &lay, q, k_cache, v_cache,
                     block_tables, context_lens, num_seqs, num_q_heads, num_kv_heads, head_dim,
                     block_size, scale, num_splits, max_blocks_per_seq, num_blocks, q_len, dtype, stream,
                     k_new, v_new);
  if (st != PA_OK) return st;
  return pa_decode_combine(out, workspace, workspace_bytes, num_seqs, num_q_heads, head_dim,
                           q_len, num_splits, dtype, stream);
}

PA_API pa_status pa_decode_cascade(void *out, const void *q, const void *k_new, const void *v_new,
                                   void *k_cache, void *v_cache, const int32_t *block_tables,
                                   const int32_t *context_lens, int num_seqs, int num_q_heads,
                                   int num_kv_heads, int head_dim, int block_size, float scale,
                                   int max_blocks_per_seq, int num_blocks, int q_len,
                                   pa_dtype dtype, int prefix_blocks, int tail_splits,
                                   void *workspace, size_t workspace_bytes, void *stream) {
  if (!out || !aligned16(out)) return PA_ERR_INVALID_ARG;
  if ((k_new == nullptr) != (v_new == nullptr)) return PA_ERR_INVALID_ARG;
  if (k_new && (!aligned16(k_new) || !aligned16(v_new))) return PA_ERR_INVALID_ARG;
  if (tail_splits <= 0 || prefix_blocks <= 0) return PA_ERR_INVALID_ARG;
  pa_status st = check_decode(q, k_cache, v_cache, block_tables, context_lens, num_seqs,
                              num_q_heads, num_kv_heads, head_dim, block_size, scale,
                              max_blocks_per_seq, num_blocks, q_len, dtype);
  if (st != PA_OK) return st;
  if (prefix_blocks > max_blocks_per_seq) return PA_ERR_INVALID_ARG;
  // the two passes split each row's positions at a 16-token tile boundary
  if ((int64_t)prefix_blocks * block_size % pa::kTileTokens != 0) return PA_ERR_UNSUPPORTED;
  if (tail_splits >= (1 << 20)) return PA_ERR_INVALID_ARG;
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return PA_ERR_INVALID_ARG;
  const int parts = 1 + tail_splits;
  const WsLayout lay = ws_layout(num_seqs, num_q_heads, q_len, head_dim, parts);
  if (workspace_bytes < lay.total) return PA_ERR_INVALID_ARG;
  float *ws = static_cast<float *>(workspace);
  // 1. the shared prefix: every query row of every sequence against the first
  //    prefix_blocks blocks of table row 0 -> workspace partition 0
  Placement head;
  head.ws_splits = parts;
  head.shared_prefix = prefix_blocks;
  head.max_ctas = cascade_prefix_ctas();
  st = decode_common(nullptr, ws, &lay, q, k_cache, v_cache, block_tables, context_lens, num_seqs,
                     num_q_heads, num_kv_heads, head_dim, block_size, scale, 1, max_blocks_per_seq,
                     num_blocks, q_len, dtype, stream, nullptr, nullptr, nullptr, nullptr, head);
  if (st != PA_OK) return st;
  // 2. each sequence's own blocks past the prefix (with this step's append, if
  //    given).  One tail partition and q_len <= 16: a single pass of the decode
  //    kernel that merges partition 0 into its result and writes out.  Otherwise:
  //    partitions 1 .. tail_splits, then the combine.
  Placement tail;
  tail.first_block = prefix_blocks;
  if (tail_splits == 1 && q_len <= kMaxDecodeQLen) {  // (the decode kernel merges)
    tail.prior_ws = ws;
    tail.prior_lay = &lay;
    tail.prior_splits = parts;
    return decode_common(out, nullptr, nullptr, q, k_cache, v_cache, block_tables, context_lens,
                         num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, scale, 1,
                         max_blocks_per_seq, num_blocks, q_len, dtype, stream, k_new, v_new,
                         nullptr, nullptr, tail);
  }
  tail.ws_splits = parts;
  tail.ws_split0 = 1;
  st = decode_common(nullptr, ws, &lay, q, k_cache, v_cache, block_tables, context_lens, num_seqs,
                     num_q_heads, num_kv_heads, head_dim, block_size, scale, tail_splits, max_blocks_per_seq,
                     num_blocks, q_len, dtype, stream, k_new, v_new, nullptr, nullptr, tail);
  if (st != PA_OK) return st;
  // 3. merge the partitions
  return pa_decode_combine(out, workspace, workspace_bytes, num_seqs, num_q_heads, head_dim, q_len,
                           parts, dtype, stream);
}

PA_API pa_status pa_append_kv_fp8(void *k_cache, void *v_cache, const void *k_new,
                                  const void *v_new, const int64_t *slot_mapping, int n_tokens,
                                  int num_kv_heads, int head_dim, int block_size, int num_blocks,
                                  pa_dtype new_dtype, const float *k_scale, const float *v_scale,
                                  void *stream) {
  if (!k_cache || !v_cache || !k_new || !v_new || !slot_mapping || !k_scale || !v_scale)
    return PA_ERR_INVALID_ARG;
  if (n_tokens < 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 || num_blocks <= 0)
    return PA_ERR_INVALID_ARG;
  if (!aligned16(k_cache) || !aligned16(v_cache) || !aligned16(k_new) || !aligned16(v_new))
    return PA_ERR_INVALID_ARG;
  if (!supported_dtype(new_dtype)) return PA_ERR_UNSUPPORTED;
  if (head_dim != 128 || !supported_block(block_size)) return PA_ERR_UNSUPPORTED;
  if (n_tokens == 0) return PA_OK;
  unsigned *err = error_word();
  if (err == nullptr) return PA_ERR_CUDA;
  const unsigned blocks = (unsigned)n_tokens;  // one CTA per token row
  const unsigned threads = append_threads(num_kv_heads, head_dim);
  const int64_t num_slots = (int64_t)num_blocks * block_size;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  auto kc = static_cast<uint8_t *>(k_cache);
  auto vc = static_cast<uint8_t *>(v_cache);
  auto kn = static_cast<const uint16_t *>(k_new);
  auto vn = static_cast<const uint16_t *>(v_new);
  cudaError_t e = new_dtype == PA_FP16
                      ? pa::launch_dependent(append_kv_fp8_kernel<__half, 128>, blocks, threads, s,
                                             kc, vc, kn, vn, slot_mapping, n_tokens, num_kv_heads,
                                             block_size, num_slots, k_scale, v_scale, err)
                      : pa::launch_dependent(append_kv_fp8_kernel<__nv_bfloat16, 128>, blocks,
                                             threads, s, kc, vc, kn, vn, slot_mapping, n_tokens,
                                             num_kv_heads, block_size, num_slots, k_scale, v_scale,
                                             err);
  return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

PA_API pa_status pa_decode_fp8(void *out, const void *q, const void *k_new, const void *v_new,
                               void *k_cache, void *v_cache, const float *k_scale,
                               const float *v_scale, const int32_t *block_tables,
                               const int32_t *context_lens, int num_seqs, int num_q_heads,
                               int num_kv_heads, int head_dim, int block_size, float scale,
                               int max_blocks_per_seq, int num_blocks, int q_len, pa_dtype dtype,
                               int num_splits, void *workspace, size_t workspace_bytes,
                               void *stream) {
  if (!out || !aligned16(out) || !k_scale || !v_scale) return PA_ERR_INVALID_ARG;
  if ((k_new == nullptr) != (v_new == nullptr)) return PA_ERR_INVALID_ARG;
  if (k_new && (!aligned16(k_new) || !aligned16(v_new))) return PA_ERR_INVALID_ARG;
  if (num_splits <= 0) return PA_ERR_INVALID_ARG;
  pa_status st = check_decode(q, k_cache, v_cache, block_tables, context_lens, num_seqs,
                              num_q_heads, num_kv_heads, head_dim, block_size, scale,
                              max_blocks_per_seq, num_blocks, q_len, dtype);
  if (st != PA_OK) return st;
  if (head_dim != 128) return PA_ERR_UNSUPPORTED;
  if (num_splits == 1)
    return decode_common(out, nullptr, nullptr, q, k_cache, v_cache, block_tables, context_lens,
                         num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, scale, 1,
                         max_blocks_per_seq, num_blocks, q_len, dtype, stream, k_new, v_new,
                         k_scale, v_scale);
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return PA_ERR_INVALID_ARG;
  const WsLayout lay = ws_layout(num_seqs, num_q_heads, q_len, head_dim, num_splits);
  if (workspace_bytes < lay.total) return PA_ERR_INVALID_ARG;
  st = decode_common(nullptr, static_cast<float *>(workspace), &lay, q, k_cache, v_cache,
                     block_tables, context_lens, num_seqs, num_q_heads, num_kv_heads, head_dim,
                     block_size, scale, num_splits, max_blocks_per_seq, num_blocks, q_len, dtype, stream,
                     k_new, v_new, k_scale, v_scale);
  if (st != PA_OK) return st;
  return pa_decode_combine(out, workspace, workspace_bytes, num_seqs, num_q_heads, head_dim,
                           q_len, num_splits, dtype, stream);
}

PA_API size_t pa_decode_workspace_size(int num_seqs, int num_q_heads, int q_len, int head_dim,
                                       int num_splits) {
  if (num_seqs <= 0 || num_q_heads <= 0 || q_len <= 0 || head_dim <= 0 || num_splits <= 0)
    return 0;
  return ws_layout(num_seqs, num_q_heads, q_len, head_dim, num_splits).total;
}

PA_API pa_status pa_decode_partial(void *workspace, size_t workspace_bytes, const void *q,
                                   const void *k_cache, const void *v_cache,
                                   const int32_t *block_tables, const int32_t *context_lens,
                                   int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                                   int block_size, float scale, int num_splits,
                                   int max_blocks_per_seq, int num_blocks, int q_len,
                                   pa_dtype dtype, void *stream) {
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return PA_ERR_INVALID_ARG;
  if (num_splits <= 0) return PA_ERR_INVALID_ARG;
  pa_status st = check_decode(q, k_cache, v_cache, block_tables, context_lens, num_seqs,
                              num_q_heads, num_kv_heads, head_dim, block_size, scale,
                              max_blocks_per_seq, num_blocks, q_len, dtype);
  if (st != PA_OK) return st;
  const WsLayout lay = ws_layout(num_seqs, num_q_heads, q_len, head_dim, num_splits);
  if (workspace_bytes < lay.total) return PA_ERR_INVALID_ARG;
  return decode_common(nullptr, static_cast<float *>(workspace), &lay, q, k_cache, v_cache,
                       block_tables, context_lens, num_seqs, num_q_heads, num_kv_heads, head_dim,
                       block_size, scale, num_splits, max_blocks_per_seq, num_blocks, q_len, dtype, stream);
}

PA_API pa_status pa_decode_combine(void *out, const void *workspace, size_t workspace_bytes,
                                   int num_seqs, int num_q_heads, int head_dim, int q_len,
                                   int num_splits, pa_dtype dtype, void *stream) {
  if (!out || !workspace || !aligned16(out) || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return PA_ERR_INVALID_ARG;
  if (num_seqs <= 0 || num_q_heads <= 0 || head_dim <= 0 || q_len <= 0 || num_splits <= 0)
    return PA_ERR_INVALID_ARG;
  if (!supported_dtype(dtype)) return PA_ERR_UNSUPPORTED;
  if (head_dim != 64 && head_dim != 128) return PA_ERR_UNSUPPORTED;
  if (q_len > kMaxQLen) return PA_ERR_UNSUPPORTED;
  if ((int64_t)num_seqs * q_len * num_q_heads >= (int64_t)1 << 31) return PA_ERR_INVALID_ARG;
  const WsLayout lay = ws_layout(num_seqs, num_q_heads, q_len, head_dim, num_splits);
  if (workspace_bytes < lay.total) return PA_ERR_INVALID_ARG;
  const char *base = static_cast<const char *>(workspace);
  pa::CombineArgs a;
  a.out = out;
  a.ws_acc = reinterpret_cast<const float *>(base + lay.acc_off);
  a.ws_m = reinterpret_cast<const float *>(base + lay.m_off);
  a.ws_l = reinterpret_cast<const float *>(base + lay.l_off);
  a.num_seqs = num_seqs;
  a.rows_per_seq = q_len * num_q_heads;
  a.num_splits = num_splits;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = dtype == PA_FP16 ? pa::launch_combine_fp16(a, head_dim, s)
                                   : pa::launch_combine_bf16(a, head_dim, s);
  return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

PA_API pa_status pa_selftest_wait_timeout(void *stream) {
  unsigned *err = error_word();
  if (err == nullptr) return PA_ERR_CUDA;
  wait_timeout_kernel<<<1, 1, 0, static_cast<cudaStream_t>(stream)>>>(err);
  return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

PA_API pa_status pa_device_error(void *stream, int clear) {
  unsigned *err = error_word();
  if (err == nullptr) return PA_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  unsigned host = 0;
  if (cudaMemcpyAsync(&host, err, sizeof(host), cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return PA_ERR_CUDA;
  if (clear && cudaMemsetAsync(err, 0, sizeof(unsigned), s) != cudaSuccess) return PA_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return PA_ERR_CUDA;
  if (host & pa::kErrTimeout) return PA_ERR_DEVICE_TIMEOUT;
  if (host & pa::kErrCheck) return PA_ERR_DEVICE_CHECK;
  return PA_OK;
}

}  // extern "C"
