// pa_decode.cuh -- paged decode attention kernels for sm_103a.
//
// What is computed (pages cited by title):
//   "LLM 推理优化全景实战：从 PagedAttention 到投机解码" §2.4: attention of a query
//   over the K/V rows gathered from the sequence's physical blocks,
//   softmax(q K^T * scale) V;
//   "09-inference-optimization.md" (LLM-Code-Hot-100), PagedKVCache.get_kv: only
//   the used slots of the last page take part; AttentionWithKVCache.forward: the
//   causal offset triu(diagonal = Lk - Lq + 1) when several queries are new;
//   "推理机制动态图解（进阶）" §5: online softmax -- running max m, running sum l,
//   unnormalised output rescaled by 2^(m_old - m_new) when the max grows, O / l at
//   the end, so the score row is never written out;
//   "Scaling Book 入门第 11 章" §11.8 (FlashDecoding): a sequence's KV split over
//   several thread blocks, merged afterwards.
//
// Design (GB300-first, not a port of any earlier kernel):
//   * One CTA = one work unit (sequence, KV head, split partition, row group).
//     All query rows of a GQA group (times the q_len new positions) are served
//     by every K/V tile the CTA reads, so each KV byte leaves HBM once.
//   * Each of the NW warps owns an NSTAGE-deep ring of shared-memory stages.
//     Lane 0 of the warp looks up the physical block id and issues TMA tiled
//     loads (cp.async.bulk.tensor, 128-byte swizzle) of the whole 16-token K and
//     V tiles of its next block into a stage; completion arrives on the stage's
//     mbarrier.  Warps take the unit's blocks round-robin and keep independent
//     online-softmax states, merged once at the end (warp shuffles, then shared
//     memory).  No CTA-wide synchronisation inside the block loop.
//   * A tensor map covers the cache as [num_blocks*num_kv_heads][16][head_dim],
//     so a bad block id turns into an out-of-range TMA coordinate (zero fill),
//     never an out-of-bounds address; the id is also reported in the error word.
//   * Rows per unit 1..2: CUDA-core FMA path.  The K lanes sharing a token each
//     hold head_dim/K dimensions of q in registers; partial dot products are
//     summed with a K-lane butterfly.  Lanes that hold different tokens keep
//     separate softmax states, so no warp-wide reduction is needed per block.
//   * Rows per unit 3..8: warp-level tensor cores (mma.sync m16n8k16, fp32
//     accumulate) with the operands swapped: the 16 tokens of a tile are the M
//     dimension and the rows N = 8, S^T = K q^T and O^T += V^T P^T, P^T's B
//     fragments by movmatrix.trans from S^T's accumulator.
//   * Rows per unit 9..16: S = Q K^T with Q (16 rows, padded) as the A operand from
//     registers and K^T from ldmatrix; P = 2^(S - m) re-packed in registers as the
//     A operand of O += P V, V^T fragments from ldmatrix.trans.
//   * FP8 (e4m3) cache: the same three layouts over fp16 arithmetic, the codes
//     widened in registers (K and V fragments straight from 16-byte shared loads
//     and byte permutes), the per-KV-head scales folded into q and the output.
//   * Few units (at most one wave of 3-warp CTAs): 3-warp CTAs, 4 per SM; units
//     that fill under about two waves are shared by a 2/4/8-CTA cluster that merges
//     through distributed shared memory.
//   * Slots past the context (and NaN-poisoned padding) never reach the
//     arithmetic: scores are replaced by -inf with a select and V rows past the
//     context are zeroed in shared memory before P.V (0 * NaN would be NaN).
#pragma once

#include "pa_device.cuh"

namespace pa {

// Tokens per tile: the kernels walk a sequence in 16-token tiles.  A cache block of
// 16 tokens is one tile, one of 32 tokens two tiles, one of 8 tokens half a tile.
constexpr int kTileTokens = 16;

struct DecodeArgs {
  const void *q;                 // [num_seqs][q_len][num_q_heads][D]
  void *out;                     // [num_seqs][q_len][num_q_heads][D]   (single pass)
  float *ws_acc;                 // split-KV workspace sections (partial pass)
  float *ws_m;
  float *ws_l;
  const int32_t *block_tables;   // [num_seqs][max_blocks_per_seq]
  const int32_t *context_lens;   // [num_seqs]
  unsigned *err;                 // device error word
  int num_seqs, num_q_heads, num_kv_heads, q_len, group, rows;  // rows = group * q_len
  int max_blocks_per_seq, num_blocks, num_splits;
  int block_size;                // tokens per cache block: 8, 16 or 32
  int max_tiles;                 // 16-token tiles a block-table row covers (rounded up)
  int lpt;                       // 1: take sequences longest first (num_seqs <= kLptMaxSeqs)
  float scale_log2;              // scale * log2(e): scores in base-2 units
  // fused append (k_new == nullptr: none).  The CTAs of a unit that read a tile
  // holding one of this step's new tokens -- positions context_len - q_len + u --
  // write the unit's KV head's rows of them into the cache before reading it.
  const uint16_t *k_new;         // [num_seqs * q_len][num_kv_heads][D]
  const uint16_t *v_new;
  uint16_t *k_cache;             // the memory the tensor maps describe
  uint16_t *v_cache;
  // FP8 (e4m3) cache: value = code * scale of its KV head ([num_kv_heads] each)
  const float *k_scale;
  const float *v_scale;
  // Partitioning of each sequence's tiles: tiles before first_block are skipped
  // (a shared prefix handled elsewhere); the partial pass writes partitions
  // ws_split0 .. ws_split0 + num_splits - 1 of a workspace laid out for ws_splits.
  int first_block;
  int ws_splits, ws_split0;
  // Prefill kernel, shared-prefix mode (> 0): the query rows of every sequence
  // attend to the first `shared_prefix` tiles of block-table row 0.
  int shared_prefix;
  // Prefill kernel: most persistent CTAs to launch (0: one per SM).  A cascade's
  // shared-prefix pass leaves the other SMs to the tail pass that overlaps it.
  int max_ctas;
  // Prefill kernel: q rows arrive by TMA through the kernel's q tensor map (the KV
  // group size divides 128); otherwise each thread loads its own row
  int q_tma;
  // Prefill kernel: the score MMA negates Q K^T (scale_log2 then holds |scale| *
  // log2(e)), so that the kernel's base-2 scale is always positive
  int s_negate;
  // Single pass only: a partition of the same rows computed by another pass (the
  // shared prefix of a cascade), merged into the result before it is written.
  // Workspace layout of pa_decode_partial with prior_splits partitions; the prior
  // is partition 0.  prior_m == nullptr: none.
  const float *prior_acc, *prior_m, *prior_l;
  int prior_splits;
};

constexpr int kLptMaxSeqs = 256;

// A table entry that is not read: no block, the tile rows it would hold are
// zero-filled and nothing is reported
constexpr int kNoBlock = -2147483647 - 1;

// The tile range [tb, te) of partition `split` of a walk over tiles [fb, nb): the
// partitions cover whole cache blocks where a block spans whole tiles (16 or 32
// tokens: the split counts blocks), whole tiles where it is smaller (8 tokens).
struct TileRange {
  int tb, te;
};
__device__ __forceinline__ TileRange partition_tiles(int nb, int fb, int num_splits, int split,
                                                     int block_size) {
  const int upb = block_size > kTileTokens ? block_size / kTileTokens : 1;  // tiles per unit
  const int units = (nb - fb + upb - 1) / upb;
  const int per = (units + num_splits - 1) / num_splits * upb;
  TileRange r;
  r.tb = min(nb, fb + split * per);
  r.te = min(nb, r.tb + per);
  return r;
}

// Block-table entries behind tile j of a sequence's walk (row `table`, context
// length L): e0 holds the tile's rows (16-token block j; first block j / 2 of a
// 32-token pair of tiles; 8-token block 2j), e1 the second 8-token block 2j + 1
// while it lies inside the row and holds a position < L (else kNoBlock).
__device__ __forceinline__ void tile_entries(const int32_t *table, int j, int block_size,
                                             int max_blocks, int L, int &e0, int &e1) {
  e1 = kNoBlock;
  if (block_size == 16) {
    e0 = __ldg(table + j);
  } else if (block_size == 32) {
    e0 = __ldg(table + (j >> 1));
  } else {
    e0 = __ldg(table + 2 * j);
    if (2 * j + 1 < max_blocks && j * kTileTokens + 8 < L) e1 = __ldg(table + 2 * j + 1);
  }
}

// TMA box index (z of the cache's tensor map) of block `id` for KV head kvh;
// sub = which 16-row half of a 32-token block.  -1 (outside the map: zero fill)
// for kNoBlock, and for an id outside the pool, which is also reported.
__device__ __forceinline__ int tile_box(int id, int sub, int kvh, int num_kv_heads, int num_blocks,
                                        int block_size, unsigned *err) {
  if (id == kNoBlock) return -1;
  if (id < 0 || id >= num_blocks) {
    record_error(err, kErrCheck);
    return -1;
  }
  const int z = id * num_kv_heads + kvh;
  return block_size == 32 ? 2 * z + sub : z;
}

// Longest-processing-time order: the sequence of rank `rank` when sequences are
// sorted by context length, longest first (ties by index).  Every CTA computes
// the same order from context_lens, so consecutive CTAs start on the longest
// sequences and short ones fill the tail.  All threads of the CTA must call it.
__device__ __forceinline__ int lpt_sequence(const int32_t *lens, int n, int rank, int *s_lens,
                                            int *s_pick) {
  const int n4 = (n + 3) & ~3;
  for (int i = threadIdx.x; i < n4; i += blockDim.x)
    s_lens[i] = i < n ? max(0, __ldg(lens + i)) : -1;  // -1 pads: never longer than a real one
  if (threadIdx.x == 0) *s_pick = rank;
  __syncthreads();
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    const int li = s_lens[i];
    int r = 0;
    for (int j = 0; j < n4; j += 4) {  // broadcast 16-byte reads: 4 lengths per load
      const int4 l4 = *reinterpret_cast<const int4 *>(s_lens + j);
      r += (l4.x > li) | ((l4.x == li) & (j < i));
      r += (l4.y > li) | ((l4.y == li) & (j + 1 < i));
      r += (l4.z > li) | ((l4.z == li) & (j + 2 < i));
      r += (l4.w > li) | ((l4.w == li) & (j + 3 < i));
    }
    if (r == rank) *s_pick = i;
  }
  __syncthreads();
  return *s_pick;
}

// ---------------------------------------------------------------------------------
// Row bookkeeping shared by both paths.  Unit row rho (0 <= rho < rows) is query
// position u = rho / group of query head kvh * group + rho % group.
struct RowInfo {
  int u, h, valid;
};

__device__ __forceinline__ RowInfo row_info(const DecodeArgs &a, int kvh, int rho) {
  RowInfo ri;
  ri.valid = rho < a.rows;
  const int r = ri.valid ? rho : 0;
  ri.u = r / a.group;
  ri.h = kvh * a.group + r % a.group;
  return ri;
}

// ---------------------------------------------------------------------------------
// CUDA-core path: R rows, K lanes per token.
template <typename T, int D, int K, int R>
struct FmaPath {
  static constexpr int RPC = R;                    // rows per CTA
  static constexpr int TPP = 32 / K;               // tokens per pass
  static constexpr int PASSES = kTileTokens / TPP;  // passes per tile
  static constexpr int CH = D / 8 / K;             // 16-byte chunks per lane per token
  // Under the 128-byte swizzle, head_dim 128 with 4 or 8 lanes per token puts
  // two lanes of an 8-lane shared-memory phase on one bank group unless each lane
  // starts its chunk loop at a lane-dependent rotation; the rotation below makes
  // every phase hit 8 distinct groups (checked exhaustively for these shapes).
  static constexpr bool kRotate = (D == 128 && (K == 4 || K == 8));
  static constexpr int kRotShift = (K == 8) ? 2 : 0;
  static_assert(PASSES * TPP == kTileTokens && CH >= 1, "bad lane layout");

  float q[R][CH * 8];
  float acc[R][CH * 8];
  float m[R], l[R];
  int lim[R];
  int part, tip, rot;

  __device__ __forceinline__ int chunk(int jj) const {
    return part * CH + (kRotate ? ((jj + rot) % CH) : jj);
  }


  __device__ __forceinline__ void init(const DecodeArgs &a, int seq, int kvh, int row0, int L,
                                       float sscale) {
    const int lane = threadIdx.x & 31;
    part = lane % K;
    tip = lane / K;
    rot = (lane >> kRotShift) % CH;
    const T *qb = static_cast<const T *>(a.q);
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const RowInfo ri = row_info(a, kvh, row0 + r);
      lim[r] = ri.valid ? (L - a.q_len + ri.u + 1) : 0;
      m[r] = -INFINITY;
      l[r] = 0.f;
      const T *qrow = qb + ((size_t)(seq * a.q_len + ri.u) * a.num_q_heads + ri.h) * D;
#pragma unroll
      for (int jj = 0; jj < CH; ++jj) {
        uint4 v = make_uint4(0, 0, 0, 0);
        if (ri.valid) v = __ldg(reinterpret_cast<const uint4 *>(qrow + chunk(jj) * 8));
        const float2 f0 = Elt<T>::to_f2(v.x), f1 = Elt<T>::to_f2(v.y);
        const float2 f2 = Elt<T>::to_f2(v.z), f3 = Elt<T>::to_f2(v.w);
        const float f[8] = {f0.x, f0.y, f1.x, f1.y, f2.x, f2.y, f3.x, f3.y};
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          q[r][jj * 8 + e] = f[e] * sscale;
          acc[r][jj * 8 + e] = 0.f;
        }
      }
    }
  }

  template <bool MASKED>
  __device__ __forceinline__ void tile(uint32_t kt, uint32_t vt, int tile_idx, float) {
    float s[PASSES][R];
#pragma unroll
    for (int p = 0; p < PASSES; ++p) {
      const int t = p * TPP + tip;
#pragma unroll
      for (int r = 0; r < R; ++r) s[p][r] = 0.f;
#pragma unroll
      for (int jj = 0; jj < CH; ++jj) {
        const uint4 kv = lds128(kt + sw128_offset<kTileTokens>(t, chunk(jj)));
        const float2 f0 = Elt<T>::to_f2(kv.x), f1 = Elt<T>::to_f2(kv.y);
        const float2 f2 = Elt<T>::to_f2(kv.z), f3 = Elt<T>::to_f2(kv.w);
        const float f[8] = {f0.x, f0.y, f1.x, f1.y, f2.x, f2.y, f3.x, f3.y};
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
          for (int e = 0; e < 8; ++e) s[p][r] = fmaf(q[r][jj * 8 + e], f[e], s[p][r]);
      }
    }
    // sum the K partial dot products of each token (bitwise identical on all K lanes)
#pragma unroll
    for (int p = 0; p < PASSES; ++p)
#pragma unroll
      for (int r = 0; r < R; ++r)
#pragma unroll
        for (int o = 1; o < K; o <<= 1) s[p][r] += __shfl_xor_sync(0xffffffffu, s[p][r], o);
    if (MASKED) {
#pragma unroll
      for (int p = 0; p < PASSES; ++p) {
        const int tg = tile_idx * kTileTokens + p * TPP + tip;
#pragma unroll
        for (int r = 0; r < R; ++r)
          if (tg >= lim[r]) s[p][r] = -INFINITY;
      }
    }
    // online softmax, per lane group (tokens p*TPP + tip)
#pragma unroll
    for (int r = 0; r < R; ++r) {
      float mx = s[0][r];
#pragma unroll
      for (int p = 1; p < PASSES; ++p) mx = fmaxf(mx, s[p][r]);
      if (mx > m[r]) {
        const float c = fast_exp2(m[r] - mx);  // m = -inf -> 0
        l[r] *= c;
#pragma unroll
        for (int e = 0; e < CH * 8; ++e) acc[r][e] *= c;
        m[r] = mx;
      }
#pragma unroll
      for (int p = 0; p < PASSES; ++p) {
        float pv;
        if (MASKED)
          pv = (s[p][r] == -INFINITY) ? 0.f : fast_exp2(s[p][r] - m[r]);
        else
          pv = fast_exp2(s[p][r] - m[r]);
        s[p][r] = pv;
        l[r] += pv;
      }
    }
    // P.V
#pragma unroll
    for (int p = 0; p < PASSES; ++p) {
      const int t = p * TPP + tip;
#pragma unroll
      for (int jj = 0; jj < CH; ++jj) {
        const uint4 vv = lds128(vt + sw128_offset<kTileTokens>(t, chunk(jj)));
        const float2 f0 = Elt<T>::to_f2(vv.x), f1 = Elt<T>::to_f2(vv.y);
        const float2 f2 = Elt<T>::to_f2(vv.z), f3 = Elt<T>::to_f2(vv.w);
        const float f[8] = {f0.x, f0.y, f1.x, f1.y, f2.x, f2.y, f3.x, f3.y};
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
          for (int e = 0; e < 8; ++e) acc[r][jj * 8 + e] = fmaf(s[p][r], f[e], acc[r][jj * 8 + e]);
      }
    }
  }

  // Merge the lane groups of this warp, then publish the warp's state:
  // mrg_m/mrg_l [RPC], mrg_acc [RPC][STRIDE] for this warp.
  template <int STRIDE>
  __device__ __forceinline__ void publish(float *mrg_m, float *mrg_l, float *mrg_acc) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int o = K; o < 32; o <<= 1) {
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const float mo = __shfl_xor_sync(0xffffffffu, m[r], o);
        const float lo = __shfl_xor_sync(0xffffffffu, l[r], o);
        const float mn = fmaxf(m[r], mo);
        const float cs = (m[r] == -INFINITY) ? 0.f : fast_exp2(m[r] - mn);
        const float co = (mo == -INFINITY) ? 0.f : fast_exp2(mo - mn);
        l[r] = l[r] * cs + lo * co;
#pragma unroll
        for (int e = 0; e < CH * 8; ++e) {
          const float ao = __shfl_xor_sync(0xffffffffu, acc[r][e], o);
          acc[r][e] = acc[r][e] * cs + ao * co;
        }
        m[r] = mn;
      }
    }
    if (lane < K) {
#pragma unroll
      for (int r = 0; r < R; ++r) {
        if (lane == 0) {
          mrg_m[r] = m[r];
          mrg_l[r] = l[r];
        }
#pragma unroll
        for (int jj = 0; jj < CH; ++jj) {
          float4 *dst = reinterpret_cast<float4 *>(mrg_acc + r * STRIDE + chunk(jj) * 8);
          dst[0] = make_float4(acc[r][jj * 8 + 0], acc[r][jj * 8 + 1], acc[r][jj * 8 + 2],
                               acc[r][jj * 8 + 3]);
          dst[1] = make_float4(acc[r][jj * 8 + 4], acc[r][jj * 8 + 5], acc[r][jj * 8 + 6],
                               acc[r][jj * 8 + 7]);
        }
      }
    }
  }
};

// ---------------------------------------------------------------------------------
// Tensor-core path: up to 16 rows (padded), warp-level mma.sync m16n8k16.
template <typename T, int D>
struct MmaPath {
  static constexpr int RPC = 16;
  static constexpr int KS = D / 16;  // k-steps of S = Q K^T
  static constexpr int NT = D / 8;   // n-tiles (8 dims) of O

  uint32_t qa[KS][4];  // A fragments of Q
  float o[NT][4];      // O: rows (lane/4, lane/4 + 8), dims nt*8 + (lane%4)*2 + {0,1}
  float m[2], l[2];
  float rs[2];         // base-2 score scale of each of this lane's two rows
  int lim[2];


  // Row bookkeeping; returns this lane's two q rows (nullptr for padding rows).
  template <typename TQ>
  __device__ __forceinline__ void init_rows(const DecodeArgs &a, int seq, int kvh, int row0, int L,
                                            float sscale, const TQ *(&qrow)[2]) {
    const int g = (threadIdx.x & 31) >> 2;
    const TQ *qb = static_cast<const TQ *>(a.q);
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
      const RowInfo ri = row_info(a, kvh, row0 + g + 8 * hr);
      lim[hr] = ri.valid ? (L - a.q_len + ri.u + 1) : 0;
      qrow[hr] = ri.valid ? qb + ((size_t)(seq * a.q_len + ri.u) * a.num_q_heads + ri.h) * D
                          : nullptr;
      m[hr] = -INFINITY;
      l[hr] = 0.f;
      rs[hr] = sscale;
    }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) o[nt][e] = 0.f;
  }

  __device__ __forceinline__ void init(const DecodeArgs &a, int seq, int kvh, int row0, int L,
                                       float sscale) {
    const int c2 = (threadIdx.x & 3) * 2;
    const T *qrow[2];
    init_rows<T>(a, seq, kvh, row0, L, sscale, qrow);
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int hr = i & 1, col = ks * 16 + c2 + (i >> 1) * 8;
        qa[ks][i] = qrow[hr] ? __ldg(reinterpret_cast<const uint32_t *>(qrow[hr] + col)) : 0u;
      }
    }
  }

  template <bool MASKED>
  __device__ __forceinline__ void tile(uint32_t kt, uint32_t vt, int tile_idx, float) {
    const int lane = threadIdx.x & 31;
    const int mi = lane >> 3, ri = lane & 7;
    // S = Q K^T: B fragments (K rows = tokens, 8 dims each) by ldmatrix.  Even and
    // odd k-steps accumulate separately (two independent mma chains), then add.
    float sc[2][4], sd[2][4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) sc[nt][e] = sd[nt][e] = 0.f;
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      uint32_t b00, b01, b10, b11;
      const int tok = ri + ((mi >> 1) << 3), ch = 2 * ks + (mi & 1);
      ldmatrix_x4(kt + sw128_offset<kTileTokens>(tok, ch), b00, b01, b10, b11);
      float (&acc)[2][4] = (ks & 1) ? sd : sc;
      Elt<T>::mma16816(acc[0], qa[ks], b00, b01);
      Elt<T>::mma16816(acc[1], qa[ks], b10, b11);
    }
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) sc[nt][e] += sd[nt][e];
    softmax_pv<MASKED>(sc, vt, tile_idx);
  }

  // P has to be rounded to the 16-bit operand type.  fp16 keeps 11 significant bits
  // (output error <= 2^-12 max|v|); bf16 keeps 8, too coarse for peaked rows, so
  // bf16 P is split into hi + lo bf16 parts and both are multiplied by V (residual
  // relative error ~2^-17).
  static constexpr bool kSplitP = Elt<T>::kMantBits < 10;

  // Online-softmax update of this tile's scores S (C fragments: rows lane/4 and
  // lane/4 + 8, tokens nt*8 + (lane%4)*2 + {0,1}), rescaling O and l when a row's
  // maximum grows.  Returns P as the A operand (rows x 16 tokens): pa, and pl for
  // the split.
  template <bool MASKED>
  __device__ __forceinline__ void softmax_p(float (&sc)[2][4], int tile_idx, uint32_t (&pa)[4],
                                            uint32_t (&pl)[4]) {
    const int lane = threadIdx.x & 31;
    // scale to base-2 units, mask, row max over the 16 tokens (4 lanes per row)
    float mx[2];
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          float v = sc[nt][2 * hr + e] * rs[hr];
          if (MASKED) {
            const int tg = tile_idx * kTileTokens + nt * 8 + (lane & 3) * 2 + e;
            if (tg >= lim[hr]) v = -INFINITY;
          }
          sc[nt][2 * hr + e] = v;
        }
      mx[hr] = fmaxf(fmaxf(sc[0][2 * hr], sc[0][2 * hr + 1]), fmaxf(sc[1][2 * hr], sc[1][2 * hr + 1]));
      mx[hr] = fmaxf(mx[hr], __shfl_xor_sync(0xffffffffu, mx[hr], 1));
      mx[hr] = fmaxf(mx[hr], __shfl_xor_sync(0xffffffffu, mx[hr], 2));
      if (mx[hr] > m[hr]) {
        const float c = fast_exp2(m[hr] - mx[hr]);
        l[hr] *= c;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          o[nt][2 * hr] *= c;
          o[nt][2 * hr + 1] *= c;
        }
        m[hr] = mx[hr];
      }
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const float v = sc[nt][2 * hr + e];
          float p;
          if (MASKED)
            p = (v == -INFINITY) ? 0.f : fast_exp2(v - m[hr]);
          else
            p = fast_exp2(v - m[hr]);
          sc[nt][2 * hr + e] = p;
          l[hr] += p;
        }
    }
    // P as the A operand, straight from the S fragments
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float p0 = sc[i >> 1][2 * (i & 1)], p1 = sc[i >> 1][2 * (i & 1) + 1];
      pa[i] = Elt<T>::from_f2(p0, p1);
      pl[i] = 0u;
      if (kSplitP) {
        const float2 hi = Elt<T>::to_f2(pa[i]);
        pl[i] = Elt<T>::from_f2(p0 - hi.x, p1 - hi.y);
      }
    }
  }

  // softmax_p, then O += P V with V^T fragments from the 16-bit tile at vt.
  template <bool MASKED>
  __device__ __forceinline__ void softmax_pv(float (&sc)[2][4], uint32_t vt, int tile_idx) {
    const int lane = threadIdx.x & 31;
    const int mi = lane >> 3, ri = lane & 7;
    uint32_t pa[4], pl[4];
    softmax_p<MASKED>(sc, tile_idx, pa, pl);
    // O += P V: B fragments (V^T) by ldmatrix.trans, two 8-dim n-tiles per load
#pragma unroll
    for (int dp = 0; dp < NT / 2; ++dp) {
      uint32_t v0, v1, v2, v3;
      const int tok = ri + ((mi & 1) << 3), ch = 2 * dp + (mi >> 1);
      ldmatrix_x4_trans(vt + sw128_offset<kTileTokens>(tok, ch), v0, v1, v2, v3);
      Elt<T>::mma16816(o[2 * dp], pa, v0, v1);
      Elt<T>::mma16816(o[2 * dp + 1], pa, v2, v3);
      if (kSplitP) {
        Elt<T>::mma16816(o[2 * dp], pl, v0, v1);
        Elt<T>::mma16816(o[2 * dp + 1], pl, v2, v3);
      }
    }
  }

  template <int STRIDE>
  __device__ __forceinline__ void publish(float *mrg_m, float *mrg_l, float *mrg_acc) {
    const int lane = threadIdx.x & 31;
    const int g = lane >> 2, c2 = (lane & 3) * 2;
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
      l[hr] += __shfl_xor_sync(0xffffffffu, l[hr], 1);
      l[hr] += __shfl_xor_sync(0xffffffffu, l[hr], 2);
      if ((lane & 3) == 0) {
        mrg_m[g + 8 * hr] = m[hr];
        mrg_l[g + 8 * hr] = l[hr];
      }
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
        *reinterpret_cast<float2 *>(mrg_acc + (g + 8 * hr) * STRIDE + nt * 8 + c2) =
            make_float2(o[nt][2 * hr], o[nt][2 * hr + 1]);
    }
  }
};

// 8x8 16-bit matrix transpose across the warp: the row-major fragment (thread t
// holds row t/4, columns 2(t%4) and 2(t%4)+1) of M in, the same fragment of M^T out.
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t a) {
  uint32_t d;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(a));
  return d;
}

// ---------------------------------------------------------------------------------
// Tensor-core path with the operands swapped, for 3..8 rows per KV head (GQA decode):
// the 16 tokens of a tile are the MMA's M, the rows its N = 8, so a padded row costs
// half of what it costs with the rows as M = 16.
//   S^T[token][row] = K[token][:] . q[row][:]   (m16n8k16: A = K by ldmatrix, B = q^T
//                                                in registers)
//   O^T[dim][row] += V^T[dim][token] P^T[token][row]   (A = V^T by ldmatrix.trans, B =
//                                                        P^T from S^T's accumulator)
// The accumulator of S^T leaves P in the row-major fragment of the 8x8 blocks
// [token][row]; one movmatrix transpose per block gives the B fragment of P^T.
// Thread (g, c) = (lane / 4, lane % 4) holds rows 2c and 2c+1 (P, l, O^T columns) and
// tokens g and g+8 of each tile.
template <typename T, int D>
struct MmaTPath {
  static constexpr int RPC = 8;
  static constexpr int KS = D / 16;  // k-steps of S (16 dims each)
  static constexpr int MT = D / 16;  // m-tiles of O^T (16 dims each)

  uint32_t qb[KS][2];  // B fragments of q^T: row g, dims ks*16 + 2c (+1) and + 8 (+9)
  float o[MT][4];      // O^T: dims mt*16 + g (+8), rows 2c, 2c+1
  float m[2], l[2];    // rows 2c + e
  float rs[2];
  int lim[2];

  // Rows 2c, 2c + 1 of this lane: causal limits, softmax state, O^T = 0.
  __device__ __forceinline__ void init_rows(const DecodeArgs &a, int kvh, int row0, int L,
                                            float sscale) {
    const int c = threadIdx.x & 3;
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const RowInfo ri = row_info(a, kvh, row0 + 2 * c + e);
      lim[e] = ri.valid ? (L - a.q_len + ri.u + 1) : 0;
      m[e] = -INFINITY;
      l[e] = 0.f;
      rs[e] = sscale;
    }
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
      for (int i = 0; i < 4; ++i) o[mt][i] = 0.f;
  }

  __device__ __forceinline__ void init(const DecodeArgs &a, int seq, int kvh, int row0, int L,
                                       float sscale) {
    const int lane = threadIdx.x & 31;
    const int g = lane >> 2, c = lane & 3;
    const T *qb_ptr = static_cast<const T *>(a.q);
    init_rows(a, kvh, row0, L, sscale);
    const RowInfo rq = row_info(a, kvh, row0 + g);
    const T *qrow = rq.valid ? qb_ptr + ((size_t)(seq * a.q_len + rq.u) * a.num_q_heads + rq.h) * D
                             : nullptr;
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      qb[ks][0] = qrow ? __ldg(reinterpret_cast<const uint32_t *>(qrow + ks * 16 + 2 * c)) : 0u;
      qb[ks][1] = qrow ? __ldg(reinterpret_cast<const uint32_t *>(qrow + ks * 16 + 2 * c + 8)) : 0u;
    }
  }

  template <bool MASKED>
  __device__ __forceinline__ void tile(uint32_t kt, uint32_t vt, int tile_idx, float) {
    const int lane = threadIdx.x & 31;
    const int mi = lane >> 3, ri = lane & 7;
    // S^T: two independent chains (even and odd k-steps), then added.  A fragment
    // of K: matrices (tokens 0-7 | 8-15) x (dims 0-7 | 8-15) of the k-step
    float sc[4] = {0.f, 0.f, 0.f, 0.f}, sd[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      uint32_t ka[4];
      const int tok = ri + ((mi & 1) << 3), ch = 2 * ks + (mi >> 1);
      ldmatrix_x4(kt + sw128_offset<kTileTokens>(tok, ch), ka[0], ka[1], ka[2], ka[3]);
      Elt<T>::mma16816((ks & 1) ? sd : sc, ka, qb[ks][0], qb[ks][1]);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) sc[i] += sd[i];
    softmax_pv<MASKED>(sc, vt, tile_idx);
  }

  // bf16 P is split into hi + lo parts as in MmaPath (8 significant bits are too
  // coarse for peaked rows); fp16 P is used directly.
  static constexpr bool kSplitP = Elt<T>::kMantBits < 10;

  // Online-softmax update from this tile's raw S^T (sc[i]: token g + 8 (i >> 1), row
  // 2c + (i & 1)), rescaling O^T and l when a row's maximum grows.  Returns P^T's B
  // fragments (tokens 0-7 and 8-15, transposed): bh, and bl for the split.
  template <bool MASKED>
  __device__ __forceinline__ void softmax_p(float (&sc)[4], int tile_idx, uint32_t (&bh)[2],
                                            uint32_t (&bl)[2]) {
    const int g = (threadIdx.x & 31) >> 2;
    // scale, mask
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float v = sc[i] * rs[i & 1];
      if (MASKED) {
        const int tg = tile_idx * kTileTokens + g + 8 * (i >> 1);
        if (tg >= lim[i & 1]) v = -INFINITY;
      }
      sc[i] = v;
    }
    // online softmax per row (the 8 threads of a row differ in g: lanes c + 4g)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      float mx = fmaxf(sc[e], sc[2 + e]);
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
      if (mx > m[e]) {
        const float f = fast_exp2(m[e] - mx);  // m = -inf -> 0
        l[e] *= f;
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          o[mt][e] *= f;
          o[mt][2 + e] *= f;
        }
        m[e] = mx;
      }
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const float v = sc[2 * h + e];
        float p;
        if (MASKED)
          p = (v == -INFINITY) ? 0.f : fast_exp2(v - m[e]);
        else
          p = fast_exp2(v - m[e]);
        sc[2 * h + e] = p;
        l[e] += p;
      }
    }
    // P^T B fragments: (tokens 0-7) and (tokens 8-15) blocks, transposed
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const float p0 = sc[2 * h], p1 = sc[2 * h + 1];
      const uint32_t hi = Elt<T>::from_f2(p0, p1);
      bh[h] = movmatrix_trans(hi);
      bl[h] = 0u;
      if (kSplitP) {
        const float2 hf = Elt<T>::to_f2(hi);
        bl[h] = movmatrix_trans(Elt<T>::from_f2(p0 - hf.x, p1 - hf.y));
      }
    }
  }

  // softmax_p, then O^T += V^T P^T with V^T fragments from the 16-bit tile at vt.
  template <bool MASKED>
  __device__ __forceinline__ void softmax_pv(float (&sc)[4], uint32_t vt, int tile_idx) {
    const int lane = threadIdx.x & 31;
    const int mi = lane >> 3, ri = lane & 7;
    uint32_t bh[2], bl[2];
    softmax_p<MASKED>(sc, tile_idx, bh, bl);
    // O^T += V^T P^T: A fragment of V^T by ldmatrix.trans, matrices (dims 0-7 | 8-15)
    // x (tokens 0-7 | 8-15) of the m-tile
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
      uint32_t va[4];
      const int tok = ri + ((mi >> 1) << 3), ch = 2 * mt + (mi & 1);
      ldmatrix_x4_trans(vt + sw128_offset<kTileTokens>(tok, ch), va[0], va[1], va[2], va[3]);
      Elt<T>::mma16816(o[mt], va, bh[0], bh[1]);
      if (kSplitP) Elt<T>::mma16816(o[mt], va, bl[0], bl[1]);
    }
  }

  template <int STRIDE>
  __device__ __forceinline__ void publish(float *mrg_m, float *mrg_l, float *mrg_acc) {
    const int lane = threadIdx.x & 31;
    const int g = lane >> 2, c = lane & 3;
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      l[e] += __shfl_xor_sync(0xffffffffu, l[e], 4);
      l[e] += __shfl_xor_sync(0xffffffffu, l[e], 8);
      l[e] += __shfl_xor_sync(0xffffffffu, l[e], 16);
      const int r = 2 * c + e;
      if (g == 0) {
        mrg_m[r] = m[e];
        mrg_l[r] = l[e];
      }
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        mrg_acc[r * STRIDE + mt * 16 + g] = o[mt][e];
        mrg_acc[r * STRIDE + mt * 16 + g + 8] = o[mt][2 + e];
      }
    }
  }
};

// Eight 16-bit values -> eight e4m3 codes of value / scale (fp32 division, nearest
// even, saturating): the quantising append of an FP8 cache.
template <typename T>
__device__ __forceinline__ uint2 quantize8(const uint4 v, float scale) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint16_t c[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = Elt<T>::to_f2(w[i]);
    c[i] = f32x2_to_e4m3x2(f.x / scale, f.y / scale);
  }
  return make_uint2((uint32_t)c[0] | ((uint32_t)c[1] << 16), (uint32_t)c[2] | ((uint32_t)c[3] << 16));
}

// Word i (compile-time after unrolling) of a 16-byte load.
__device__ __forceinline__ uint32_t word_of(const uint4 &v, int i) {
  return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}
// Codes 0, 1 (lo) or 2, 3 (hi) of a word of four e4m3 codes -> f16x2.
__device__ __forceinline__ uint32_t e4m3_lo_f16x2(uint32_t w) {
  return e4m3x2_to_f16x2(static_cast<uint16_t>(w & 0xffffu));
}
__device__ __forceinline__ uint32_t e4m3_hi_f16x2(uint32_t w) {
  return e4m3x2_to_f16x2(static_cast<uint16_t>(w >> 16));
}

// ---------------------------------------------------------------------------------
// FP8 (e4m3) cache, tensor-core path with swapped operands for 3..8 rows per KV
// head: MmaTPath's layout (tokens as the MMA's M, rows as N = 8) over fp16 MMAs,
// with both operands widened from the codes in registers (no shared-memory copy).
// - S^T = K q^T: the contraction over head dims is permuted so that lane c's k
//   slots {2c, 2c+1, 2c+8, 2c+9} of k-step ks are dims 32c + 4ks .. +3.  A lane
//   reads its 32 dims of tokens g and g + 8 with two 16-byte loads each; q^T's B
//   fragments use the same permutation, so S is unchanged.
// - O^T += V^T P^T: the m-rows of O^T are permuted so that row g of m-tile b is
//   dim 16g + 2b and row g + 8 is dim 16g + 2b + 1.  A lane then needs dims
//   16g .. 16g + 15 of tokens 2c, 2c + 1, 2c + 8, 2c + 9 (the k slots of P^T), one
//   16-byte load each; byte permutes pair the two tokens of each dim for the
//   e4m3x2 -> f16x2 conversion.
// Every load above is conflict-free under the 128-byte swizzle: the 8 lanes of a
// shared-memory phase hit 8 distinct 16-byte bank groups.  Each q row is scaled by a
// power of two into fp16's range and the score scale of its S^T column undoes it.
template <typename T>
struct Mma8TPath {
  static constexpr int D = 128;
  static constexpr int RPC = 8;
  using Inner = MmaTPath<__half, D>;
  static constexpr int KS = Inner::KS;
  Inner inner;  // inner.o[b][i]: O^T dim 16g + 2b + (i >> 1), row 2c + (i & 1)

  __device__ __forceinline__ void init(const DecodeArgs &a, int seq, int kvh, int row0, int L,
                                       float sscale) {
    const int lane = threadIdx.x & 31;
    const int g = lane >> 2, c = lane & 3;
    inner.init_rows(a, kvh, row0, L, sscale);
    // q row g, dims 32c + 4ks .. +3 of k-step ks
    const RowInfo rq = row_info(a, kvh, row0 + g);
    const T *qrow = rq.valid ? static_cast<const T *>(a.q) +
                                   ((size_t)(seq * a.q_len + rq.u) * a.num_q_heads + rq.h) * D
                             : nullptr;
    float2 qf[KS][2];
    float mx = 0.f;
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      uint2 v = make_uint2(0u, 0u);
      if (qrow) v = __ldg(reinterpret_cast<const uint2 *>(qrow + 32 * c + 4 * ks));
      qf[ks][0] = Elt<T>::to_f2(v.x);
      qf[ks][1] = Elt<T>::to_f2(v.y);
      mx = fmaxf(mx, fmaxf(fmaxf(fabsf(qf[ks][0].x), fabsf(qf[ks][0].y)),
                           fmaxf(fabsf(qf[ks][1].x), fabsf(qf[ks][1].y))));
    }
    // the 4 lanes holding row g agree on its maximum
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
    const int e_row = (mx > 0.f && isfinite(mx)) ? ilogbf(mx) : 0;
    const float down = ldexpf(1.f, -e_row);  // |q| * down < 2: well inside fp16
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      inner.qb[ks][0] = Elt<__half>::from_f2(qf[ks][0].x * down, qf[ks][0].y * down);
      inner.qb[ks][1] = Elt<__half>::from_f2(qf[ks][1].x * down, qf[ks][1].y * down);
    }
    // S^T column 2c + e is row 2c + e: its exponent comes from the lanes of that row
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int er = __shfl_sync(0xffffffffu, e_row, 4 * (2 * c + e));
      inner.rs[e] = sscale * ldexpf(1.f, er);
    }
  }

  template <bool MASKED>
  __device__ __forceinline__ void tile(uint32_t kt, uint32_t vt, int tile_idx, float) {
    const int lane = threadIdx.x & 31;
    const int g = lane >> 2, c = lane & 3;
    const uint4 k0a = lds128(kt + sw128_offset_row128(g, 2 * c));
    const uint4 k0b = lds128(kt + sw128_offset_row128(g, 2 * c + 1));
    const uint4 k8a = lds128(kt + sw128_offset_row128(g + 8, 2 * c));
    const uint4 k8b = lds128(kt + sw128_offset_row128(g + 8, 2 * c + 1));
    const uint4 v0 = lds128(vt + sw128_offset_row128(2 * c, g));
    const uint4 v1 = lds128(vt + sw128_offset_row128(2 * c + 1, g));
    const uint4 v8 = lds128(vt + sw128_offset_row128(2 * c + 8, g));
    const uint4 v9 = lds128(vt + sw128_offset_row128(2 * c + 9, g));
    // S^T: two independent chains (even and odd k-steps), then added
    float sc[4] = {0.f, 0.f, 0.f, 0.f}, sd[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      const uint32_t w0 = word_of(ks < 4 ? k0a : k0b, ks & 3);
      const uint32_t w8 = word_of(ks < 4 ? k8a : k8b, ks & 3);
      const uint32_t ka[4] = {e4m3_lo_f16x2(w0), e4m3_lo_f16x2(w8), e4m3_hi_f16x2(w0),
                              e4m3_hi_f16x2(w8)};
      Elt<__half>::mma16816((ks & 1) ? sd : sc, ka, inner.qb[ks][0], inner.qb[ks][1]);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) sc[i] += sd[i];
    uint32_t bh[2], bl[2];
    inner.template softmax_p<MASKED>(sc, tile_idx, bh, bl);  // fp16 P: no split
    // O^T += V^T P^T.  Word j of a lane's V chunk holds dims 16g + 4j .. +3: m-tile
    // 2j takes dims 4j, 4j + 1 (rows g, g + 8), m-tile 2j + 1 dims 4j + 2, 4j + 3.
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t x0 = word_of(v0, j), x1 = word_of(v1, j);
      const uint32_t x8 = word_of(v8, j), x9 = word_of(v9, j);
      const uint32_t p01 = __byte_perm(x0, x1, 0x5140), q01 = __byte_perm(x0, x1, 0x7362);
      const uint32_t p89 = __byte_perm(x8, x9, 0x5140), q89 = __byte_perm(x8, x9, 0x7362);
      const uint32_t va[4] = {e4m3_lo_f16x2(p01), e4m3_hi_f16x2(p01), e4m3_lo_f16x2(p89),
                              e4m3_hi_f16x2(p89)};
      const uint32_t vb[4] = {e4m3_lo_f16x2(q01), e4m3_hi_f16x2(q01), e4m3_lo_f16x2(q89),
                              e4m3_hi_f16x2(q89)};
      Elt<__half>::mma16816(inner.o[2 * j], va, bh[0], bh[1]);
      Elt<__half>::mma16816(inner.o[2 * j + 1], vb, bh[0], bh[1]);
    }
  }

  template <int STRIDE>
  __device__ __forceinline__ void publish(float *mrg_m, float *mrg_l, float *mrg_acc) {
    const int lane = threadIdx.x & 31;
    const int g = lane >> 2, c = lane & 3;
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      float l = inner.l[e];
      l += __shfl_xor_sync(0xffffffffu, l, 4);
      l += __shfl_xor_sync(0xffffffffu, l, 8);
      l += __shfl_xor_sync(0xffffffffu, l, 16);
      const int r = 2 * c + e;
      if (g == 0) {
        mrg_m[r] = inner.m[e];
        mrg_l[r] = l;
      }
#pragma unroll
      for (int b = 0; b < Inner::MT; ++b) {
        mrg_acc[r * STRIDE + 16 * g + 2 * b] = inner.o[b][e];
        mrg_acc[r * STRIDE + 16 * g + 2 * b + 1] = inner.o[b][2 + e];
      }
    }
  }
};

// ---------------------------------------------------------------------------------
// FP8 (e4m3) cache, CUDA-core path: head_dim 128, one 128-byte row per token,
// 4 lanes per token, each lane 2 chunks of 16 codes.  The K scale is folded into q,
// the V scale into the output.
template <typename T, int R>
struct Fma8Path {
  static constexpr int D = 128;
  static constexpr int RPC = R;
  static constexpr int K = 4;                        // lanes per token
  static constexpr int TPP = 32 / K;                 // tokens per pass
  static constexpr int PASSES = kTileTokens / TPP;
  static constexpr int CH = D / 16 / K;              // 16-code chunks per lane per token
  // Under the 128-byte swizzle the 8 lanes of a shared-memory phase (2 tokens x 4
  // parts) already land on 8 distinct bank groups: no rotation needed.

  float q[R][CH * 16];
  float acc[R][CH * 16];
  float m[R], l[R];
  int lim[R];
  int part, tip;

  __device__ __forceinline__ int chunk(int jj) const { return part * CH + jj; }

  __device__ __forceinline__ void init(const DecodeArgs &a, int seq, int kvh, int row0, int L,
                                       float sscale) {
    const int lane = threadIdx.x & 31;
    part = lane % K;
    tip = lane / K;
    const T *qb = static_cast<const T *>(a.q);
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const RowInfo ri = row_info(a, kvh, row0 + r);
      lim[r] = ri.valid ? (L - a.q_len + ri.u + 1) : 0;
      m[r] = -INFINITY;
      l[r] = 0.f;
      const T *qrow = qb + ((size_t)(seq * a.q_len + ri.u) * a.num_q_heads + ri.h) * D;
#pragma unroll
      for (int jj = 0; jj < CH; ++jj) {
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          uint4 v = make_uint4(0, 0, 0, 0);
          if (ri.valid)
            v = __ldg(reinterpret_cast<const uint4 *>(qrow + chunk(jj) * 16 + half * 8));
          const float2 f0 = Elt<T>::to_f2(v.x), f1 = Elt<T>::to_f2(v.y);
          const float2 f2 = Elt<T>::to_f2(v.z), f3 = Elt<T>::to_f2(v.w);
          const float f[8] = {f0.x, f0.y, f1.x, f1.y, f2.x, f2.y, f3.x, f3.y};
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            q[r][jj * 16 + half * 8 + e] = f[e] * sscale;
            acc[r][jj * 16 + half * 8 + e] = 0.f;
          }
        }
      }
    }
  }

  template <bool MASKED>
  __device__ __forceinline__ void tile(uint32_t kt, uint32_t vt, int tile_idx, float) {
    float s[PASSES][R];
#pragma unroll
    for (int p = 0; p < PASSES; ++p) {
      const int t = p * TPP + tip;
#pragma unroll
      for (int r = 0; r < R; ++r) s[p][r] = 0.f;
#pragma unroll
      for (int jj = 0; jj < CH; ++jj) {
        float f[16];
        e4m3x16_to_f32(lds128(kt + sw128_offset_row128(t, chunk(jj))), f);
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
          for (int e = 0; e < 16; ++e) s[p][r] = fmaf(q[r][jj * 16 + e], f[e], s[p][r]);
      }
    }
#pragma unroll
    for (int p = 0; p < PASSES; ++p)
#pragma unroll
      for (int r = 0; r < R; ++r)
#pragma unroll
        for (int o = 1; o < K; o <<= 1) s[p][r] += __shfl_xor_sync(0xffffffffu, s[p][r], o);
    if (MASKED) {
#pragma unroll
      for (int p = 0; p < PASSES; ++p) {
        const int tg = tile_idx * kTileTokens + p * TPP + tip;
#pragma unroll
        for (int r = 0; r < R; ++r)
          if (tg >= lim[r]) s[p][r] = -INFINITY;
      }
    }
#pragma unroll
    for (int r = 0; r < R; ++r) {
      float mx = s[0][r];
#pragma unroll
      for (int p = 1; p < PASSES; ++p) mx = fmaxf(mx, s[p][r]);
      if (mx > m[r]) {
        const float c = fast_exp2(m[r] - mx);
        l[r] *= c;
#pragma unroll
        for (int e = 0; e < CH * 16; ++e) acc[r][e] *= c;
        m[r] = mx;
      }
#pragma unroll
      for (int p = 0; p < PASSES; ++p) {
        float pv;
        if (MASKED)
          pv = (s[p][r] == -INFINITY) ? 0.f : fast_exp2(s[p][r] - m[r]);
        else
          pv = fast_exp2(s[p][r] - m[r]);
        s[p][r] = pv;
        l[r] += pv;
      }
    }
#pragma unroll
    for (int p = 0; p < PASSES; ++p) {
      const int t = p * TPP + tip;
#pragma unroll
      for (int jj = 0; jj < CH; ++jj) {
        float f[16];
        e4m3x16_to_f32(lds128(vt + sw128_offset_row128(t, chunk(jj))), f);
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
          for (int e = 0; e < 16; ++e) acc[r][jj * 16 + e] = fmaf(s[p][r], f[e], acc[r][jj * 16 + e]);
      }
    }
  }

  template <int STRIDE>
  __device__ __forceinline__ void publish(float *mrg_m, float *mrg_l, float *mrg_acc) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int o = K; o < 32; o <<= 1) {
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const float mo = __shfl_xor_sync(0xffffffffu, m[r], o);
        const float lo = __shfl_xor_sync(0xffffffffu, l[r], o);
        const float mn = fmaxf(m[r], mo);
        const float cs = (m[r] == -INFINITY) ? 0.f : fast_exp2(m[r] - mn);
        const float co = (mo == -INFINITY) ? 0.f : fast_exp2(mo - mn);
        l[r] = l[r] * cs + lo * co;
#pragma unroll
        for (int e = 0; e < CH * 16; ++e) {
          const float ao = __shfl_xor_sync(0xffffffffu, acc[r][e], o);
          acc[r][e] = acc[r][e] * cs + ao * co;
        }
        m[r] = mn;
      }
    }
    if (lane < K) {
#pragma unroll
      for (int r = 0; r < R; ++r) {
        if (lane == 0) {
          mrg_m[r] = m[r];
          mrg_l[r] = l[r];
        }
#pragma unroll
        for (int jj = 0; jj < CH; ++jj)
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4)
            reinterpret_cast<float4 *>(mrg_acc + r * STRIDE + chunk(jj) * 16)[q4] =
                make_float4(acc[r][jj * 16 + 4 * q4], acc[r][jj * 16 + 4 * q4 + 1],
                            acc[r][jj * 16 + 4 * q4 + 2], acc[r][jj * 16 + 4 * q4 + 3]);
      }
    }
  }
};

// FP8 (e4m3) cache, tensor-core path for 9..16 rows per KV head: MmaPath's layout
// over fp16 MMAs (every e4m3 value is exact in fp16), with both operands widened
// from the codes in registers, as in Mma8TPath.
// - S = Q K^T: inside the contraction over head dims, lane c's k slots {2c, 2c+1,
//   2c+8, 2c+9} of k-step ks are dims 32c + 4ks .. +3; each lane reads its 32 dims
//   of tokens g and g + 8 with two 16-byte loads each, and Q's A fragments use the
//   same permutation.
// - O += P V: column n of n-tile nt is dim 16n + nt.  A lane's B fragments are then
//   dims 16g .. 16g + 15 of tokens 2c, 2c + 1, 2c + 8, 2c + 9 (one 16-byte load
//   each), paired per dim by byte permutes; its accumulators hold dims 32c + nt and
//   32c + 16 + nt of rows g and g + 8.
// A bf16 q row is brought into fp16 range by an exact power-of-two factor 2^-e (e:
// exponent of the row's largest |q|), and 2^e goes into that row's score scale.  P
// is then fp16 too: no hi/lo split is needed.
template <typename T>
struct Mma8Path {
  static constexpr int D = 128;
  static constexpr int RPC = 16;
  using Inner = MmaPath<__half, D>;
  static constexpr int KS = Inner::KS;
  Inner inner;

  __device__ __forceinline__ void init(const DecodeArgs &a, int seq, int kvh, int row0, int L,
                                       float sscale) {
    const int c = threadIdx.x & 3;
    const T *qrow[2];
    inner.template init_rows<T>(a, seq, kvh, row0, L, sscale, qrow);
    float2 qf[KS][4];
    float mx[2] = {0.f, 0.f};
#pragma unroll
    for (int ks = 0; ks < KS; ++ks)
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int hr = i & 1, col = 32 * c + 4 * ks + (i >> 1) * 2;
        const uint32_t v = qrow[hr] ? __ldg(reinterpret_cast<const uint32_t *>(qrow[hr] + col)) : 0u;
        qf[ks][i] = Elt<T>::to_f2(v);
        mx[hr] = fmaxf(mx[hr], fmaxf(fabsf(qf[ks][i].x), fabsf(qf[ks][i].y)));
      }
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {  // the 4 lanes holding a row agree on its maximum
      mx[hr] = fmaxf(mx[hr], __shfl_xor_sync(0xffffffffu, mx[hr], 1));
      mx[hr] = fmaxf(mx[hr], __shfl_xor_sync(0xffffffffu, mx[hr], 2));
    }
    float down[2];
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
      const int e = (mx[hr] > 0.f && isfinite(mx[hr])) ? ilogbf(mx[hr]) : 0;
      down[hr] = ldexpf(1.f, -e);           // |q| * down < 2: well inside fp16
      inner.rs[hr] = sscale * ldexpf(1.f, e);
    }
#pragma unroll
    for (int ks = 0; ks < KS; ++ks)
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float d = down[i & 1];
        inner.qa[ks][i] = Elt<__half>::from_f2(qf[ks][i].x * d, qf[ks][i].y * d);
      }
  }

  template <bool MASKED>
  __device__ __forceinline__ void tile(uint32_t kt, uint32_t vt, int tile_idx, float) {
    const int lane = threadIdx.x & 31;
    const int g = lane >> 2, c = lane & 3;
    uint4 kw[2][2];  // [token g, g + 8][dims 32c .. +15, 32c + 16 .. +31]
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int h = 0; h < 2; ++h) kw[nt][h] = lds128(kt + sw128_offset_row128(nt * 8 + g, 2 * c + h));
    const uint4 v0 = lds128(vt + sw128_offset_row128(2 * c, g));
    const uint4 v1 = lds128(vt + sw128_offset_row128(2 * c + 1, g));
    const uint4 v8 = lds128(vt + sw128_offset_row128(2 * c + 8, g));
    const uint4 v9 = lds128(vt + sw128_offset_row128(2 * c + 9, g));
    // S = Q K^T; even and odd k-steps accumulate separately, then add
    float sc[2][4], sd[2][4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) sc[nt][e] = sd[nt][e] = 0.f;
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      float (&acc)[2][4] = (ks & 1) ? sd : sc;
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        const uint32_t w = word_of(kw[nt][ks >> 2], ks & 3);
        Elt<__half>::mma16816(acc[nt], inner.qa[ks], e4m3_lo_f16x2(w), e4m3_hi_f16x2(w));
      }
    }
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) sc[nt][e] += sd[nt][e];
    uint32_t pa[4], pl[4];
    inner.template softmax_p<MASKED>(sc, tile_idx, pa, pl);  // fp16 P: no split
    // O += P V.  Word j of a lane's V chunk holds dims 16g + 4j .. +3: the B columns
    // g of n-tiles 4j .. 4j + 3.
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t x0 = word_of(v0, j), x1 = word_of(v1, j);
      const uint32_t x8 = word_of(v8, j), x9 = word_of(v9, j);
      const uint32_t p01 = __byte_perm(x0, x1, 0x5140), q01 = __byte_perm(x0, x1, 0x7362);
      const uint32_t p89 = __byte_perm(x8, x9, 0x5140), q89 = __byte_perm(x8, x9, 0x7362);
      Elt<__half>::mma16816(inner.o[4 * j], pa, e4m3_lo_f16x2(p01), e4m3_lo_f16x2(p89));
      Elt<__half>::mma16816(inner.o[4 * j + 1], pa, e4m3_hi_f16x2(p01), e4m3_hi_f16x2(p89));
      Elt<__half>::mma16816(inner.o[4 * j + 2], pa, e4m3_lo_f16x2(q01), e4m3_lo_f16x2(q89));
      Elt<__half>::mma16816(inner.o[4 * j + 3], pa, e4m3_hi_f16x2(q01), e4m3_hi_f16x2(q89));
    }
  }

  template <int STRIDE>
  __device__ __forceinline__ void publish(float *mrg_m, float *mrg_l, float *mrg_acc) {
    const int lane = threadIdx.x & 31;
    const int g = lane >> 2, c = lane & 3;
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
      float l = inner.l[hr];
      l += __shfl_xor_sync(0xffffffffu, l, 1);
      l += __shfl_xor_sync(0xffffffffu, l, 2);
      const int r = g + 8 * hr;
      if (c == 0) {
        mrg_m[r] = inner.m[hr];
        mrg_l[r] = l;
      }
#pragma unroll
      for (int nt = 0; nt < Inner::NT; ++nt) {
        mrg_acc[r * STRIDE + 32 * c + nt] = inner.o[nt][2 * hr];
        mrg_acc[r * STRIDE + 32 * c + 16 + nt] = inner.o[nt][2 * hr + 1];
      }
    }
  }
};

// ---------------------------------------------------------------------------------
// The kernel: work unit = (sequence, KV head, split) x row group.  A unit may be
// shared by the CTAs of one thread-block cluster (launched with cluster dimension
// C > 1 along x): the C*NW warps take the unit's blocks round-robin, each CTA
// merges its warps, then the CTAs merge through distributed shared memory.  This
// splits one long sequence over several SMs without any global workspace.
// BS: the cache's block size when it is fixed at compile time (16), or 0 to read it
// from the arguments (8 or 32 tokens).
template <typename T, int D, int NW, int NSTAGE, class Path, bool PARTIAL, bool KV8, int BS>
__global__ void __launch_bounds__(NW * 32)
    paged_decode_kernel(const __grid_constant__ CUtensorMap kmap,
                        const __grid_constant__ CUtensorMap vmap, const DecodeArgs a) {
  // one head of one block: 4 KiB at D = 128 (16-bit cache), 2 KiB (FP8 cache)
  constexpr int kEltBytes = KV8 ? 1 : 2;
  constexpr int kTileBytes = kTileTokens * D * kEltBytes;
  constexpr int kStageBytes = 2 * kTileBytes;      // K tile + V tile
  constexpr int kBoxCols = 128 / kEltBytes;        // one TMA box = 16 rows x 128 bytes
  constexpr int kRowChunks = D * kEltBytes / 16;   // 16-byte chunks per cached row
  constexpr int RPC = Path::RPC;
  constexpr int kStride = D + 8;  // merge-area row stride (floats): padded against bank conflicts
  static_assert(!KV8 || D == 128, "FP8 cache: head_dim 128");
  static_assert(kStride % 4 == 0, "merge rows stay 16-byte aligned");
  static_assert((NW + 1) * RPC * (kStride + 2) * 4 + 64 <=
                    NW * NSTAGE * kStageBytes,
                "merge area");

  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bars[NW * NSTAGE];
  __shared__ int s_failed;

  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const uint32_t smem_base = (smem_u32(smem_raw) + 1023u) & ~1023u;  // 128B-swizzle tiles: 1 KiB
  uint8_t *smem_gen = smem_raw + (smem_base - smem_u32(smem_raw));

  // shared-memory state and the tensor-map descriptors: nothing another kernel writes
  if (threadIdx.x == 0) {
    s_failed = 0;
    prefetch_tensormap(&kmap);
    prefetch_tensormap(&vmap);
  }
  if (lane == 0) {
#pragma unroll
    for (int s = 0; s < NSTAGE; ++s) mbar_init(smem_u32(&bars[warp * NSTAGE + s]), 1);
    fence_mbar_init();
  }
  __syncwarp();

  // Launched as a programmatic dependent of the previous kernel on the stream (for
  // example the KV append): setup above this point overlaps that kernel's tail.
  // Wait for it to complete before the first read of global memory: any input
  // (cache, q, tables, lengths) may have been written by it.
  //
  // The one exception is the tail pass of a cascade, which merges a prior
  // partition (prior_m != nullptr) and waits only before its epilogue.
  // - The kernel before it is the cascade's shared-prefix pass.  That pass writes
  //   nothing but the prior partition, read here only after the wait, L2-only.
  // - The prefix pass reads only the shared blocks, and this kernel's append never
  //   writes those (the caller's contract).
  // - Every other input was written by kernels that completed before the prefix
  //   pass passed its own wait and allowed this launch.
  // So the prefix pass runs while this kernel walks its own blocks.
  const bool late_wait = a.prior_m != nullptr;
  if (!late_wait) griddep_wait();
  griddep_launch_dependents();  // the next kernel may start its own setup

  const int csize = static_cast<int>(cluster_nctarank());  // 1 without a cluster launch
  const int crank = static_cast<int>(cluster_ctarank());
  const int unit = blockIdx.x / csize;
  const int kvh = unit % a.num_kv_heads;
  const int rest = unit / a.num_kv_heads;
  const int split = rest % a.num_splits;
  int seq = rest / a.num_splits;
  int L;
  if (a.lpt) {
    __shared__ __align__(16) int s_lens[kLptMaxSeqs];
    __shared__ int s_pick;
    seq = lpt_sequence(a.context_lens, a.num_seqs, seq, s_lens, &s_pick);
    L = s_lens[seq];  // already loaded (and clamped at 0) for the ranking
  } else {
    L = max(0, __ldg(a.context_lens + seq));
  }
  const int row0 = blockIdx.y * RPC;

  const int bsz = BS ? BS : a.block_size;
  int nb = (L + kTileTokens - 1) / kTileTokens;  // tiles
  if ((int64_t)L > (int64_t)a.max_blocks_per_seq * bsz) {  // context longer than its table
    if (threadIdx.x == 0 && split == 0 && kvh == 0 && blockIdx.y == 0 && crank == 0)
      record_error(a.err, kErrCheck);
    nb = min(nb, a.max_tiles);
  }
  const TileRange part = partition_tiles(nb, min(nb, a.first_block), a.num_splits, split, bsz);
  const int tb = part.tb, te = part.te;
  const int first_masked = (L - a.q_len + 1) / kTileTokens;  // tiles >= this need masking
  // base-2 score scale (times the K scale of an FP8 cache) and the V scale
  const float sscale = a.scale_log2 * (KV8 ? __ldg(a.k_scale + kvh) : 1.f);
  const float vscale = KV8 ? __ldg(a.v_scale + kvh) : 1.f;

  // This warp's tiles: the unit's ntiles blocks are visited from a starting offset
  // `rot` that differs between the KV heads of a sequence, tile number
  // k = gw + TW * n (gw: warp index in the cluster) being block
  // tb + (k + rot) mod ntiles.  Staggered starts keep the CTAs of one wave in
  // different phases (e.g. some on an L2-resident shared prefix, some on private
  // blocks in HBM).  The order depends only on logical positions.
  const int gw = crank * NW + warp;
  const int TW = csize * NW;
  const int ntiles = te - tb;
  const int rot = ntiles > 0 ? (int)(((long long)kvh * ntiles) / a.num_kv_heads) : 0;
  const int n_my = (ntiles - gw > 0) ? (ntiles - gw + TW - 1) / TW : 0;
  auto tile_of = [&](int n) {
    int k = gw + TW * n + rot;
    if (k >= ntiles) k -= ntiles;
    return tb + k;
  };
  const int32_t *table = a.block_tables + (size_t)seq * a.max_blocks_per_seq;
  const uint32_t my_stages = smem_base + warp * NSTAGE * kStageBytes;
  // lane i holds the block-table entries of tile n = window + i
  int tbl = 0, tbl2 = kNoBlock;
  auto load_window = [&](int n0) {
    if (n0 + lane < n_my)
      tile_entries(table, tile_of(n0 + lane), bsz, a.max_blocks_per_seq, L, tbl, tbl2);
  };

  auto issue = [&](int n) {
    if ((n & 31) == 0 && n > 0) load_window(n);
    const int e0 = __shfl_sync(0xffffffffu, tbl, n & 31);
    const int e1 = __shfl_sync(0xffffffffu, tbl2, n & 31);
    if (lane == 0) {
      const int s = n % NSTAGE;
      const uint32_t bar = smem_u32(&bars[warp * NSTAGE + s]);
      const uint32_t kdst = my_stages + s * kStageBytes;
      // boxes outside the tensor map (bad or missing blocks) arrive zero-filled
      const int z0 = tile_box(e0, tile_of(n) & 1, kvh, a.num_kv_heads, a.num_blocks, bsz, a.err);
      mbar_arrive_expect_tx(bar, kStageBytes);
      if (bsz == 8) {  // two 8-row boxes per tile: blocks 2j (rows 0-7) and 2j + 1
        const int z1 = tile_box(e1, 0, kvh, a.num_kv_heads, a.num_blocks, bsz, a.err);
#pragma unroll
        for (int hh = 0; hh < kTileBytes / (kTileTokens * 128); ++hh) {
          const uint32_t o = hh * (kTileTokens * 128);
          tma_load_3d(kdst + o, &kmap, hh * kBoxCols, 0, z0, bar);
          tma_load_3d(kdst + o + 8 * 128, &kmap, hh * kBoxCols, 0, z1, bar);
          tma_load_3d(kdst + kTileBytes + o, &vmap, hh * kBoxCols, 0, z0, bar);
          tma_load_3d(kdst + kTileBytes + o + 8 * 128, &vmap, hh * kBoxCols, 0, z1, bar);
        }
      } else {
#pragma unroll
        for (int hh = 0; hh < kTileBytes / (kTileTokens * 128); ++hh) {
          tma_load_3d(kdst + hh * (kTileTokens * 128), &kmap, hh * kBoxCols, 0, z0, bar);
          tma_load_3d(kdst + kTileBytes + hh * (kTileTokens * 128), &vmap, hh * kBoxCols, 0, z0, bar);
        }
      }
    }
  };

  // the first block-table window and the q rows load concurrently
  if (n_my > 0) load_window(0);
  Path path;
  path.init(a, seq, kvh, row0, L, sscale);

  // Fused append: every CTA that reads a tile holding a new position writes all of
  // this unit's new rows itself (CTAs of one row group or neighbouring split that
  // also read one write identical bytes), then orders those generic-proxy stores
  // before its own TMA reads of the cache.  Tile j is read by cluster warp
  // (j - tb - rot) mod ntiles, modulo TW.  The table window and q above are already
  // in flight: neither is written here.
  bool reads_new = false;
  if (a.k_new != nullptr && ntiles > 0) {
    const int j1 = min(te, (L + kTileTokens - 1) / kTileTokens);  // past the last new tile
    for (int j = max(tb, max(0, L - a.q_len) / kTileTokens); j < j1; ++j) {
      int k = j - tb - rot;
      if (k < 0) k += ntiles;
      reads_new |= (k % TW) / NW == crank;
    }
  }
  if (reads_new) {
    const int64_t num_slots = (int64_t)a.num_blocks * bsz;
    for (int idx = threadIdx.x; idx < a.q_len * (D / 8); idx += NW * 32) {
      const int u = idx / (D / 8), c = idx % (D / 8);
      const int pos = L - a.q_len + u;
      if (pos < 0) continue;
      const int lb = pos / bsz;
      if (lb >= a.max_blocks_per_seq) {
        record_error(a.err, kErrCheck);
        continue;
      }
      const int64_t slot = (int64_t)__ldg(a.block_tables + (size_t)seq * a.max_blocks_per_seq + lb) *
                               bsz + pos % bsz;
      if (slot < 0 || slot >= num_slots) {
        record_error(a.err, kErrCheck);
        continue;
      }
      const int64_t blk = slot / bsz, off = slot % bsz;
      const size_t dst = (size_t)(((blk * a.num_kv_heads + kvh) * bsz + off) * D + c * 8);
      const size_t src = ((size_t)(seq * a.q_len + u) * a.num_kv_heads + kvh) * D + c * 8;
      const uint4 kv = __ldg(reinterpret_cast<const uint4 *>(a.k_new + src));
      const uint4 vv = __ldg(reinterpret_cast<const uint4 *>(a.v_new + src));
      if constexpr (KV8) {  // quantise: e4m3(x / scale), 8 codes per chunk
        uint8_t *kc = reinterpret_cast<uint8_t *>(a.k_cache), *vc = reinterpret_cast<uint8_t *>(a.v_cache);
        *reinterpret_cast<uint2 *>(kc + dst) = quantize8<T>(kv, __ldg(a.k_scale + kvh));
        *reinterpret_cast<uint2 *>(vc + dst) = quantize8<T>(vv, __ldg(a.v_scale + kvh));
      } else {
        *reinterpret_cast<uint4 *>(a.k_cache + dst) = kv;
        *reinterpret_cast<uint4 *>(a.v_cache + dst) = vv;
      }
    }
    fence_proxy_async_global();
    __syncthreads();
  }


  const int prologue = min(NSTAGE, n_my);
  for (int n = 0; n < prologue; ++n) issue(n);

  bool failed = false;
  int n = 0;
  for (; n < n_my; ++n) {
    const int s = n % NSTAGE;
    const uint32_t bar = smem_u32(&bars[warp * NSTAGE + s]);
    const bool ok = mbar_wait_bounded(bar, (n / NSTAGE) & 1);
    if (!__all_sync(0xffffffffu, ok)) {
      failed = true;
      break;
    }
    const int j = tile_of(n);
    const uint32_t kt = my_stages + s * kStageBytes;
    const uint32_t vt = kt + kTileBytes;
    if (j >= first_masked) {
      const int nvalid = L - j * kTileTokens;  // rows >= nvalid are past the context
      if (nvalid < kTileTokens) {
        for (int idx = lane; idx < (kTileTokens - nvalid) * kRowChunks; idx += 32) {
          const int row = nvalid + idx / kRowChunks, ch = idx % kRowChunks;
          sts128_zero(vt + (KV8 ? sw128_offset_row128(row, ch) : sw128_offset<kTileTokens>(row, ch)));
        }
        // order these generic-proxy stores before any later TMA (async proxy) write
        // into the same stage
        fence_proxy_async_smem();
        __syncwarp();
      }
      path.template tile<true>(kt, vt, j, sscale);
    } else {
      path.template tile<false>(kt, vt, j, sscale);
    }
    __syncwarp();
    if (n + NSTAGE < n_my) issue(n + NSTAGE);
  }
  if (failed) {
    // drain the loads this warp still has in flight (bounded), then report
    for (int k = n; k < min(n_my, n + NSTAGE); ++k)
      (void)mbar_wait_bounded(smem_u32(&bars[warp * NSTAGE + (k % NSTAGE)]), (k / NSTAGE) & 1);
    if (lane == 0) {
      record_error(a.err, kErrTimeout);
      s_failed = 1;
    }
  }
  __syncthreads();  // every stage consumed: the stage memory becomes the merge area
  const bool cta_failed = s_failed != 0;

  // merge area: per warp m[RPC], l[RPC], acc[RPC][kStride]; then the CTA's merged
  // state cm[RPC], cl[RPC], cacc[RPC][kStride] (read by the cluster peers)
  constexpr int kMl = (NW * RPC + 3) & ~3;  // m and l blocks padded to 16 bytes
  float *mrg_m = reinterpret_cast<float *>(smem_gen);
  float *mrg_l = mrg_m + kMl;
  float *mrg_acc = mrg_l + kMl;  // 16-byte aligned for its float4 accesses
  float *cta_acc = mrg_acc + NW * RPC * kStride;
  float *cta_m = cta_acc + RPC * kStride;
  float *cta_l = cta_m + RPC;
  if (!cta_failed) path.template publish<kStride>(mrg_m + warp * RPC, mrg_l + warp * RPC,
                                                   mrg_acc + warp * RPC * kStride);
  __syncthreads();

  if (late_wait) griddep_wait();  // the prior partition is complete and visible
  auto emit = [&](int r, int d8, float M, float den, const float (&num)[8]) {
    const RowInfo ri = row_info(a, kvh, row0 + r);
    if (!ri.valid) return;
    if constexpr (PARTIAL) {
      const size_t wrow = ((size_t)seq * a.ws_splits + a.ws_split0 + split) * (a.q_len * a.num_q_heads) +
                          (size_t)ri.u * a.num_q_heads + ri.h;
      float4 *dst = reinterpret_cast<float4 *>(a.ws_acc + wrow * D + d8 * 8);
      dst[0] = make_float4(num[0] * vscale, num[1] * vscale, num[2] * vscale, num[3] * vscale);
      dst[1] = make_float4(num[4] * vscale, num[5] * vscale, num[6] * vscale, num[7] * vscale);
      if (d8 == 0) {
        a.ws_m[wrow] = M;
        a.ws_l[wrow] = den;
      }
    } else {
      const size_t orow = (size_t)(seq * a.q_len + ri.u) * a.num_q_heads + ri.h;
      float inv = den > 0.f ? vscale / den : 0.f;
      float o[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) o[i] = num[i] * inv;
      if (a.prior_m != nullptr) {
        // merge the prior partition (m0, l0, acc0): the same rescale as the online
        // softmax, once more
        const size_t prow = (size_t)seq * a.prior_splits * (a.q_len * a.num_q_heads) +
                            (size_t)ri.u * a.num_q_heads + ri.h;
        const float m0 = __ldcg(a.prior_m + prow), l0 = __ldcg(a.prior_l + prow);
        const float Mx = fmaxf(M, m0);
        const float w1 = (M == -INFINITY) ? 0.f : fast_exp2(M - Mx);
        const float w0 = (m0 == -INFINITY) ? 0.f : fast_exp2(m0 - Mx);
        const float dd = w1 * den + w0 * l0;
        inv = dd > 0.f ? 1.f / dd : 0.f;
        const float4 *src = reinterpret_cast<const float4 *>(a.prior_acc + prow * D + d8 * 8);
        const float4 p0 = __ldcg(src), p1 = __ldcg(src + 1);
        const float pv[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
#pragma unroll
        for (int i = 0; i < 8; ++i) o[i] = (w1 * num[i] * vscale + w0 * pv[i]) * inv;
      }
      uint4 packed;
      packed.x = Elt<T>::from_f2(o[0], o[1]);
      packed.y = Elt<T>::from_f2(o[2], o[3]);
      packed.z = Elt<T>::from_f2(o[4], o[5]);
      packed.w = Elt<T>::from_f2(o[6], o[7]);
      *reinterpret_cast<uint4 *>(static_cast<T *>(a.out) + orow * D + d8 * 8) = packed;
    }
  };

  // level 1: merge this CTA's warps, item = (row, 8 dims)
  if (!cta_failed) {
    for (int item = threadIdx.x; item < RPC * (D / 8); item += NW * 32) {
      const int r = item / (D / 8), d8 = item % (D / 8);
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < NW; ++w) M = fmaxf(M, mrg_m[w * RPC + r]);
      float den = 0.f, num[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int w = 0; w < NW; ++w) {
        const float mw = mrg_m[w * RPC + r];
        const float wt = (mw == -INFINITY) ? 0.f : fast_exp2(mw - M);
        den += wt * mrg_l[w * RPC + r];
        const float4 *src =
            reinterpret_cast<const float4 *>(mrg_acc + (w * RPC + r) * kStride + d8 * 8);
        const float4 x0 = src[0], x1 = src[1];
        num[0] += wt * x0.x; num[1] += wt * x0.y; num[2] += wt * x0.z; num[3] += wt * x0.w;
        num[4] += wt * x1.x; num[5] += wt * x1.y; num[6] += wt * x1.z; num[7] += wt * x1.w;
      }
      if (csize == 1) {
        emit(r, d8, M, den, num);
      } else {
        float4 *dst = reinterpret_cast<float4 *>(cta_acc + r * kStride + d8 * 8);
        dst[0] = make_float4(num[0], num[1], num[2], num[3]);
        dst[1] = make_float4(num[4], num[5], num[6], num[7]);
        if (d8 == 0) {
          cta_m[r] = M;
          cta_l[r] = den;
        }
      }
    }
  }
  if (csize == 1) return;

  // level 2: merge the cluster's CTAs through distributed shared memory; CTA crank
  // takes every csize-th item.  Every CTA reaches both cluster barriers.
  cluster_sync_all();
  bool any_failed = false;
  for (int c = 0; c < csize; ++c)
    any_failed |= dsmem_ld_s32(dsmem_map(smem_u32(&s_failed), c)) != 0;
  if (!any_failed) {
    for (int item = crank + csize * threadIdx.x; item < RPC * (D / 8); item += csize * NW * 32) {
      const int r = item / (D / 8), d8 = item % (D / 8);
      float M = -INFINITY;
      for (int c = 0; c < csize; ++c)
        M = fmaxf(M, dsmem_ld_f32(dsmem_map(smem_u32(cta_m + r), c)));
      float den = 0.f, num[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      for (int c = 0; c < csize; ++c) {
        const float mc = dsmem_ld_f32(dsmem_map(smem_u32(cta_m + r), c));
        const float wt = (mc == -INFINITY) ? 0.f : fast_exp2(mc - M);
        den += wt * dsmem_ld_f32(dsmem_map(smem_u32(cta_l + r), c));
        const uint32_t src = dsmem_map(smem_u32(cta_acc + r * kStride + d8 * 8), c);
        const float4 x0 = dsmem_ld_f32x4(src), x1 = dsmem_ld_f32x4(src + 16);
        num[0] += wt * x0.x; num[1] += wt * x0.y; num[2] += wt * x0.z; num[3] += wt * x0.w;
        num[4] += wt * x1.x; num[5] += wt * x1.y; num[6] += wt * x1.z; num[7] += wt * x1.w;
      }
      emit(r, d8, M, den, num);
    }
  }
  cluster_sync_all();  // peers' shared memory stays alive until every read is done
}

// ---------------------------------------------------------------------------------
// Split-KV combine: one warp per (sequence, row), lanes covering head_dim (or, in
// split_combine_spread_kernel below, head_dim / 32 warps per row).
struct CombineArgs {
  void *out;
  const float *ws_acc, *ws_m, *ws_l;
  int num_seqs, rows_per_seq, num_splits;
};

template <typename T, int D>
__global__ void __launch_bounds__(128) split_combine_kernel(const CombineArgs a) {
  constexpr int PER = D / 32;  // dims per lane
  const int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (gw >= a.num_seqs * a.rows_per_seq) return;
  griddep_wait();  // the workspace comes from the partial pass just before
  griddep_launch_dependents();
  const int seq = gw / a.rows_per_seq, r = gw % a.rows_per_seq;
  const size_t base = (size_t)seq * a.num_splits * a.rows_per_seq + r;
  const size_t pstride = a.rows_per_seq;
  // statistics: lanes take partitions (all loads independent), then warp reductions
  float M = -INFINITY;
  for (int p = lane; p < a.num_splits; p += 32) {
    const size_t w = base + p * pstride;
    if (a.ws_l[w] > 0.f) M = fmaxf(M, a.ws_m[w]);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  float den = 0.f, num[PER];
#pragma unroll
  for (int k = 0; k < PER; ++k) num[k] = 0.f;
  if (M != -INFINITY) {
    for (int p0 = 0; p0 < a.num_splits; p0 += 32) {
      // lane holds the weight of partition p0 + lane
      float wt = 0.f;
      if (p0 + lane < a.num_splits) {
        const size_t w = base + (p0 + lane) * pstride;
        const float lw = a.ws_l[w];
        wt = lw > 0.f ? fast_exp2(a.ws_m[w] - M) : 0.f;
        den += wt * lw;
      }
      const int cnt = min(32, a.num_splits - p0);
#pragma unroll 8
      for (int k = 0; k < cnt; ++k) {
        const float wk = __shfl_sync(0xffffffffu, wt, k);
        const float *acc = a.ws_acc + (base + (p0 + k) * pstride) * D + lane * PER;
#pragma unroll
        for (int q = 0; q < PER; q += 2) {
          const float2 x = *reinterpret_cast<const float2 *>(acc + q);
          num[q] += wk * x.x;
          num[q + 1] += wk * x.y;
        }
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
  }
  const float inv = den > 0.f ? 1.f / den : 0.f;
  T *o = static_cast<T *>(a.out) + ((size_t)seq * a.rows_per_seq + r) * D + lane * PER;
#pragma unroll
  for (int k = 0; k < PER; k += 2)
    *reinterpret_cast<uint32_t *>(o + k) = Elt<T>::from_f2(num[k] * inv, num[k + 1] * inv);
}

// With few rows and many partitions the warps of the form above are too few to
// hide the partitions' load latency: this form gives each row D / 32 warps, one
// dimension per lane, every partition's load of that dimension in flight at once.
// The partitions are summed in the same order, so both forms give the same bits.
template <typename T, int D>
__global__ void __launch_bounds__(128) split_combine_spread_kernel(const CombineArgs a) {
  constexpr int kWarpsPerRow = D / 32;
  const int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  const int row_id = gw / kWarpsPerRow, dim = (gw % kWarpsPerRow) * 32 + lane;
  if (row_id >= a.num_seqs * a.rows_per_seq) return;
  griddep_wait();  // the workspace comes from the partial pass just before
  griddep_launch_dependents();
  const int seq = row_id / a.rows_per_seq, r = row_id % a.rows_per_seq;
  const size_t base = (size_t)seq * a.num_splits * a.rows_per_seq + r;
  const size_t pstride = a.rows_per_seq;
  float M = -INFINITY;
  for (int p = lane; p < a.num_splits; p += 32) {
    const size_t w = base + p * pstride;
    if (a.ws_l[w] > 0.f) M = fmaxf(M, a.ws_m[w]);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  float den = 0.f, num = 0.f;
  if (M != -INFINITY) {
    for (int p0 = 0; p0 < a.num_splits; p0 += 32) {
      float wt = 0.f;
      if (p0 + lane < a.num_splits) {
        const size_t w = base + (p0 + lane) * pstride;
        const float lw = a.ws_l[w];
        wt = lw > 0.f ? fast_exp2(a.ws_m[w] - M) : 0.f;
        den += wt * lw;
      }
      const int cnt = min(32, a.num_splits - p0);
#pragma unroll 16
      for (int k = 0; k < cnt; ++k) {
        const float wk = __shfl_sync(0xffffffffu, wt, k);
        num += wk * a.ws_acc[(base + (p0 + k) * pstride) * D + dim];
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
  }
  const float inv = den > 0.f ? 1.f / den : 0.f;
  static_cast<uint16_t *>(a.out)[((size_t)seq * a.rows_per_seq + r) * D + dim] =
      Elt<T>::from_f(num * inv);
}

}  // namespace pa
