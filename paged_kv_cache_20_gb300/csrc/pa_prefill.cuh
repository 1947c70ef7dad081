// pa_prefill.cuh -- paged attention for many query rows per KV head: chunked
// prefill (q_len new tokens of a sequence, causal) and the shared-prefix pass of
// cascade attention (the query rows of every sequence against prefix blocks that all
// sequences share).
//
// What is computed is the attention of pa_decode: softmax(scale q K^T) V over the
// visible positions ("LLM 推理优化全景实战" §2.4; the causal offset of
// "09-inference-optimization.md", AttentionWithKVCache.forward), with online
// softmax ("推理机制动态图解（进阶）" §5).  Sharing one physical copy of a common
// prefix ("LLM推理与服务：面试问题与推荐回答" Q2-Q3) makes its attention one dense
// product over all rows that share it.
//
// Design: one CTA = one KV head x 16*NW query rows.  A producer warp streams the
// K/V tiles of the block list into an NSTAGE ring by TMA (full barrier per stage,
// completed by the transaction count; empty barrier per stage, one arrival per
// consumer warp).  Each of the NW consumer warps owns 16 distinct rows and runs the
// tensor-core tile (S = Q K^T, online softmax, O += P V with mma.sync m16n8k16), so
// every K/V tile is read from memory once for 16*NW rows and no cross-warp merge is
// needed.  All waits are bounded.
#pragma once

#include "pa_decode.cuh"

namespace pa {

template <typename T, int D, int NW, int NSTAGE, bool PARTIAL>
__global__ void __launch_bounds__((NW + 1) * 32)
    paged_prefill_kernel(const __grid_constant__ CUtensorMap kmap,
                         const __grid_constant__ CUtensorMap vmap, const DecodeArgs a) {
  constexpr int kTileBytes = kTileTokens * D * 2;
  constexpr int kStageBytes = 2 * kTileBytes;
  constexpr int kRows = 16 * NW;

  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full_bar[NSTAGE];
  __shared__ __align__(8) uint64_t empty_bar[NSTAGE];
  __shared__ int s_failed;
  __shared__ int s_maxlim;

  griddep_wait();
  griddep_launch_dependents();

  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const bool producer = warp == NW;
  const uint32_t smem_base = (smem_u32(smem_raw) + 1023u) & ~1023u;

  // grid.x = (sequence, partition, row block) with the row block fastest; y = KV head
  const bool shared = a.shared_prefix > 0;
  const int kvh = blockIdx.y;
  const int rows_per_seq = a.q_len * a.group;
  const int rows_total = shared ? a.num_seqs * rows_per_seq : rows_per_seq;
  const int nrb = (rows_total + kRows - 1) / kRows;
  const int zz = blockIdx.x / nrb;
  const int split = zz % a.num_splits;
  const int zseq = zz / a.num_splits;                 // the sequence (chunked prefill)
  // the last row blocks see the most positions (causal): they are scheduled first
  const int row_base = (nrb - 1 - (int)(blockIdx.x % nrb)) * kRows;
  const int tseq = shared ? 0 : zseq;                 // block-table row that is walked

  // this unit's block list and its partition
  int nb;
  const int Lt = max(0, __ldg(a.context_lens + tseq));
  if (shared) {
    nb = min(a.shared_prefix, a.max_blocks_per_seq);
  } else {
    nb = (Lt + kTileTokens - 1) / kTileTokens;
    if (nb > a.max_blocks_per_seq) {
      if (threadIdx.x == 0 && kvh == 0) record_error(a.err, kErrCheck);
      nb = a.max_blocks_per_seq;
    }
  }
  // blocks before first_block are covered by another pass (the shared prefix of a
  // cascade); the rest is cut into num_splits equal partitions
  const int fb = shared ? 0 : min(nb, a.first_block);
  const int per = (nb - fb + a.num_splits - 1) / a.num_splits;
  const int tb = min(nb, fb + split * per);
  const int te = min(nb, tb + per);

  // this warp's two rows per lane: row = row_base + warp*16 + lane/4 (+8)
  const T *qrow[2] = {nullptr, nullptr};
  int lim[2] = {0, 0};
  int rseq[2] = {0, 0}, ru[2] = {0, 0}, rh[2] = {0, 0};
  if (threadIdx.x == 0) {
    s_failed = 0;
    s_maxlim = 0;
  }
  __syncthreads();
  if (!producer) {
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
      const int rho = row_base + warp * 16 + (lane >> 2) + 8 * hr;
      if (rho < rows_total) {
        const int sq = shared ? rho / rows_per_seq : zseq;
        const int rr = rho % rows_per_seq;
        const int u = rr / a.group, h = kvh * a.group + rr % a.group;
        const int L = max(0, __ldg(a.context_lens + sq));
        int visible = L - a.q_len + u + 1;            // causal limit
        if (shared) visible = min(visible, nb * kTileTokens);
        rseq[hr] = sq;
        ru[hr] = u;
        rh[hr] = h;
        lim[hr] = visible;
        qrow[hr] = static_cast<const T *>(a.q) + ((size_t)(sq * a.q_len + u) * a.num_q_heads + h) * D;
        atomicMax(&s_maxlim, visible);
      }
    }
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < NSTAGE; ++s) {
      mbar_init(smem_u32(&full_bar[s]), 1);
      mbar_init(smem_u32(&empty_bar[s]), NW);
    }
    fence_mbar_init();
    prefetch_tensormap(&kmap);
    prefetch_tensormap(&vmap);
  }
  __syncthreads();
  // the tiles any row of this CTA can see
  const int t_end = min(te, max(tb, (s_maxlim + kTileTokens - 1) / kTileTokens));
  const int ntiles = max(0, t_end - tb);
  const int32_t *table = a.block_tables + (size_t)tseq * a.max_blocks_per_seq;

  if (producer) {
    int issued = 0;
    bool ok = true;
    int tbl = 0;
    for (int n = 0; n < ntiles; ++n) {
      if ((n & 31) == 0) tbl = (n + lane < ntiles) ? __ldg(table + tb + n + lane) : 0;
      const int phys = __shfl_sync(0xffffffffu, tbl, n & 31);
      const int s = n % NSTAGE;
      // the stage is free once every consumer released its previous use (a fresh
      // barrier counts as released: parity 1 of phase -1)
      bool free_ok = mbar_wait_bounded(smem_u32(&empty_bar[s]), ((n / NSTAGE) & 1) ^ 1);
      free_ok = __all_sync(0xffffffffu, free_ok);
      if (!free_ok) {
        ok = false;
        break;
      }
      if (lane == 0) {
        int z;
        if (phys >= 0 && phys < a.num_blocks) {
          z = phys * a.num_kv_heads + kvh;
        } else {
          record_error(a.err, kErrCheck);
          z = -1;  // outside the tensor map: zero fill
        }
        const uint32_t bar = smem_u32(&full_bar[s]);
        const uint32_t kdst = smem_base + s * kStageBytes;
        mbar_arrive_expect_tx(bar, kStageBytes);
#pragma unroll
        for (int hh = 0; hh < D / 64; ++hh) {
          tma_load_3d(kdst + hh * (kTileTokens * 128), &kmap, hh * 64, 0, z, bar);
          tma_load_3d(kdst + kTileBytes + hh * (kTileTokens * 128), &vmap, hh * 64, 0, z, bar);
        }
      }
      issued = n + 1;
    }
    if (!ok) {
      if (lane == 0) {
        record_error(a.err, kErrTimeout);
        atomicExch(&s_failed, 1);
      }
      // drain the loads that may still be in flight (bounded)
      for (int k = max(0, issued - NSTAGE); k < issued; ++k)
        (void)mbar_wait_bounded(smem_u32(&full_bar[k % NSTAGE]), (k / NSTAGE) & 1);
    }
  } else {
    MmaPath<T, D> path;
    path.init_explicit(qrow, lim, a.scale_log2);
    // smallest limit among this warp's real rows: tiles that end at or below it need
    // no mask
    int warp_lo = 0x7fffffff;
#pragma unroll
    for (int hr = 0; hr < 2; ++hr)
      if (qrow[hr]) warp_lo = min(warp_lo, lim[hr]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) warp_lo = min(warp_lo, __shfl_xor_sync(0xffffffffu, warp_lo, o));
    // No row of this CTA sees a position at or past s_maxlim; the V rows there may
    // be unused slots (or hold anything), so a tile that reaches them zeroes them.
    const int Lv = s_maxlim;
    for (int n = 0; n < ntiles; ++n) {
      const int s = n % NSTAGE;
      bool ok = mbar_wait_bounded(smem_u32(&full_bar[s]), (n / NSTAGE) & 1);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) {
        if (lane == 0) {
          record_error(a.err, kErrTimeout);
          atomicExch(&s_failed, 1);
        }
        break;
      }
      const int j = tb + n;
      const uint32_t kt = smem_base + s * kStageBytes, vt = kt + kTileBytes;
      const int nvalid = Lv - j * kTileTokens;
      if (nvalid < kTileTokens) {
        // P is 0 on those rows, but 0 * NaN is not 0.  Every consumer warp writes
        // the same zeros before it reads the tile, so no warp waits on another.
        for (int idx = lane; idx < (kTileTokens - max(0, nvalid)) * (D / 8); idx += 32) {
          const int row = max(0, nvalid) + idx / (D / 8), ch = idx % (D / 8);
          sts128_zero(vt + sw128_offset<kTileTokens>(row, ch));
        }
        fence_proxy_async_smem();  // generic writes, before the stage returns to TMA
        __syncwarp();
      }
      if ((j + 1) * kTileTokens > warp_lo)
        path.template tile<true>(kt, vt, j, 0.f);
      else
        path.template tile<false>(kt, vt, j, 0.f);
      __syncwarp();
      if (lane == 0)
        asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(&empty_bar[s])) : "memory");
    }
    __syncwarp();
    // finalise this warp's rows (no cross-warp merge: rows are disjoint)
    const int c2 = (lane & 3) * 2;
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
      float l = path.l[hr];
      l += __shfl_xor_sync(0xffffffffu, l, 1);
      l += __shfl_xor_sync(0xffffffffu, l, 2);
      if (qrow[hr] == nullptr || s_failed) continue;
      const size_t orow = (size_t)(rseq[hr] * a.q_len + ru[hr]) * a.num_q_heads + rh[hr];
      if constexpr (PARTIAL) {
        const size_t wrow = ((size_t)rseq[hr] * a.ws_splits + a.ws_split0 + split) *
                                (a.q_len * a.num_q_heads) + (size_t)ru[hr] * a.num_q_heads + rh[hr];
#pragma unroll
        for (int nt = 0; nt < MmaPath<T, D>::NT; ++nt)
          *reinterpret_cast<float2 *>(a.ws_acc + wrow * D + nt * 8 + c2) =
              make_float2(path.o[nt][2 * hr], path.o[nt][2 * hr + 1]);
        if ((lane & 3) == 0) {
          a.ws_m[wrow] = path.m[hr];
          a.ws_l[wrow] = l;
        }
      } else {
        const float inv = l > 0.f ? 1.f / l : 0.f;
        T *dst = static_cast<T *>(a.out) + orow * D;
#pragma unroll
        for (int nt = 0; nt < MmaPath<T, D>::NT; ++nt)
          *reinterpret_cast<uint32_t *>(dst + nt * 8 + c2) =
              Elt<T>::from_f2(path.o[nt][2 * hr] * inv, path.o[nt][2 * hr + 1] * inv);
      }
    }
  }
  __syncthreads();  // no CTA exits while its loads may still land in shared memory
}

}  // namespace pa
