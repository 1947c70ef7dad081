// pa_prefill_tc.cuh -- paged attention for many query rows per KV head on the
// 5th-generation tensor cores: chunked prefill (q_len new tokens of a sequence,
// causal) and the shared-prefix pass of cascade attention (the query rows of every
// sequence against prefix blocks that all sequences share).
//
// What is computed is the attention of pa_decode: softmax(scale q K^T) V over each
// row's visible positions ("LLM 推理优化全景实战" §2.4; the causal offset of
// "09-inference-optimization.md", AttentionWithKVCache.forward), accumulated with
// online softmax ("推理机制动态图解（进阶）" §5: running max, running sum, output
// rescaled when the max moves, divided by the sum at the end).  Chunked prefill is
// "LLM推理与服务：面试问题与推荐回答" Q14; one physical copy of a shared prefix is
// Q2-Q3 of the same page and "Scaling Book 入门第 11 章" §11.4.
//
// One CTA = one KV head x 128 query rows (the MMA's M); the cache is walked in
// chunks of 128 positions (8 blocks):
//   warps 0, 1  TMA producers: the K (warp 0) and V (warp 1) tiles of a chunk's 8
//               blocks into rings of NK and NV stages (zero fill for blocks past the
//               walk or bad ids).  A K stage is released as soon as the S MMA that
//               reads it completes, a V stage after P V;
//   warp 2      owns tensor memory and issues O += P_j V_j (fp32 accumulator in
//               TMEM, P_j read from tensor memory) from one thread;
//   warp 3      issues S_j = Q K_j^T into S buffer j % 3 (fp32, TMEM) from one
//               thread, as soon as K_j has landed and P_{j-3} V_{j-3} has freed the
//               buffer: the scores run ahead of the softmax independently of P V;
//   warps 4-11  softmax, two warps per group of 32 rows (TMEM lanes), one per half
//               of the chunk's 128 columns: read S_j, mask, exchange the half-row
//               maxima with the partner warp, online-softmax update, write P_j
//               (16-bit) over the S_j columns it came from, rescale its half of O in
//               TMEM when the row max has grown by more than 2^8 since the last
//               rescale (until then P is taken against the older max, at most 2^8,
//               and the final O / l is the same quotient); at the end O / l (or
//               the partial statistics) for its half of the columns.
// S_{j+1} and S_{j+2} are computed while the softmax works on S_j.  S_{j+3} is issued
// only after the commit of P_j V_j (the last reader of buffer j % 3) has fired.  bf16 P is split into hi + lo bf16 parts, both multiplied by V, so
// that P keeps ~16 significant bits as the fp16 path does.  Every wait is bounded.
#pragma once

#include "pa_decode.cuh"
#include "pa_tc.cuh"

namespace pa {

constexpr int kTcRows = 128;                       // query rows per CTA (MMA M)
constexpr int kTcChunk = 128;                      // positions per chunk (S MMA N)
constexpr int kTcBlocks = kTcChunk / kTileTokens;  // cache blocks per chunk
constexpr int kTcCtl = 4;                          // K, V producers; P V and S issuers
constexpr int kTcSoft = 8;                         // softmax warps
constexpr int kTcThreads = 32 * (kTcCtl + kTcSoft);
constexpr float kTcRescale = 8.f;                  // base-2 growth that forces a rescale

template <typename T, int D>
struct TcLayout {
  static constexpr int kHalves = D / 64;           // 128-byte column groups of a row
  static constexpr bool kSplitP = Elt<T>::kMantBits < 10;
  static constexpr int kQBytes = kHalves * kTcRows * 128;    // [half][128 rows][128 B]
  static constexpr int kKVBytes = kHalves * kTcChunk * 128;  // [half][128 positions][128 B]
  static constexpr int kOffStages = kQBytes;                 // K ring, then V ring
  // O at columns [0, D); S buffer b (0..2) at [128 + 128b, 256 + 128b).  P_j (packed 16-bit
  // pairs) replaces S_j half by half: positions [64h, 64h + 64) in columns
  // 64h + [0, 32) (hi) and [32, 64) (lo, bf16 only) of the buffer
  static constexpr int kTmemCols = 512;
  static constexpr int kColS = 128;
  static constexpr int smem_bytes(int nk, int nv) { return kOffStages + (nk + nv) * kKVBytes + 1024; }
};

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// 2^x (PTX ex2.approx, flushing subnormal results to zero: a weight below 2^-126
// of the row maximum contributes nothing at fp32 accumulation anyway)
__device__ __forceinline__ float ex2_ftz(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

template <typename T, int D, int NK, int NV, bool PARTIAL>
__global__ void __launch_bounds__(kTcThreads, 1)
    paged_prefill_tc_kernel(const __grid_constant__ CUtensorMap kmap,
                            const __grid_constant__ CUtensorMap vmap,
                            const __grid_constant__ CUtensorMap qmap, const DecodeArgs a) {
  using Lay = TcLayout<T, D>;
  constexpr int H = Lay::kHalves;
  constexpr bool kBf16 = Elt<T>::kMantBits < 10;
  constexpr int kOCols = D / 2;  // O columns per softmax warp
  static_assert(NK >= 2 && NV >= 2, "ring depth");
  static_assert(D == 64 || D == 128, "head_dim");

  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t k_full[NK];
  __shared__ __align__(8) uint64_t k_empty[NK];
  __shared__ __align__(8) uint64_t v_full[NV];
  __shared__ __align__(8) uint64_t v_empty[NV];
  __shared__ __align__(8) uint64_t s_full[3];
  __shared__ __align__(8) uint64_t p_full;
  __shared__ __align__(8) uint64_t p_ack;        // the MMA thread has taken P_j
  __shared__ __align__(8) uint64_t o_done[2];   // P_j V_j complete, j even / odd
  __shared__ __align__(8) uint64_t bfree[3];    // P_j V_j complete, by S/P buffer j % 3
  __shared__ __align__(8) uint64_t q_ready;      // Q written by the softmax threads
  __shared__ __align__(8) uint64_t q_full;       // Q landed by TMA
  __shared__ __align__(8) uint64_t mma_fin;
  __shared__ __align__(8) uint64_t xbar[4];      // partner exchange, per group of 32 rows
  __shared__ float xval[2][2][kTcRows];           // [parity][column half][row]
  __shared__ uint32_t s_tmem;
  __shared__ int s_failed;
  __shared__ int s_maxlim;

  griddep_wait();
  griddep_launch_dependents();

  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t sK = base + Lay::kOffStages;  // K ring: NK x kKVBytes
  const uint32_t sV = sK + NK * Lay::kKVBytes;  // V ring: NV x kKVBytes

  // ---- the unit: grid.x = (sequence, partition, row block), row block fastest ----
  const bool shared = a.shared_prefix > 0;
  const int kvh = blockIdx.y;
  const int rows_per_seq = a.q_len * a.group;
  const int rows_total = shared ? a.num_seqs * rows_per_seq : rows_per_seq;
  const int nrb = (rows_total + kTcRows - 1) / kTcRows;
  const int zz = blockIdx.x / nrb;
  const int split = zz % a.num_splits;
  const int zseq = zz / a.num_splits;
  // the last row blocks see the most positions (causal): they are scheduled first
  const int row_base = (nrb - 1 - (int)(blockIdx.x % nrb)) * kTcRows;
  const int tseq = shared ? 0 : zseq;  // block-table row that is walked

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
  // blocks before first_block belong to another pass (a cascade's shared prefix);
  // the rest is cut into num_splits equal partitions
  const int fb = shared ? 0 : min(nb, a.first_block);
  const int per = (nb - fb + a.num_splits - 1) / a.num_splits;
  const int tb = min(nb, fb + split * per);
  const int te = min(nb, tb + per);

  if (threadIdx.x == 0) {
    s_failed = 0;
    s_maxlim = 0;
    for (int s = 0; s < NK; ++s) {
      mbar_init(smem_u32(&k_full[s]), 1);
      mbar_init(smem_u32(&k_empty[s]), 1);
    }
    for (int s = 0; s < NV; ++s) {
      mbar_init(smem_u32(&v_full[s]), 1);
      mbar_init(smem_u32(&v_empty[s]), 1);
    }
    for (int b = 0; b < 3; ++b) mbar_init(smem_u32(&s_full[b]), 1);
    mbar_init(smem_u32(&p_full), kTcSoft);
    mbar_init(smem_u32(&p_ack), 1);
    mbar_init(smem_u32(&o_done[0]), 1);
    mbar_init(smem_u32(&o_done[1]), 1);
    for (int b = 0; b < 3; ++b) mbar_init(smem_u32(&bfree[b]), 1);
    mbar_init(smem_u32(&q_ready), kTcSoft);
    mbar_init(smem_u32(&q_full), 1);
    mbar_init(smem_u32(&mma_fin), 2);  // one commit from each issuing thread
    for (int q = 0; q < 4; ++q) mbar_init(smem_u32(&xbar[q]), 2);
    fence_mbar_init();
    prefetch_tensormap(&kmap);
    prefetch_tensormap(&vmap);
    if (a.q_tma) prefetch_tensormap(&qmap);
  }
  if (warp == 2) {
    tc::alloc(smem_u32(&s_tmem), Lay::kTmemCols);
    tc::relinquish();
  }
  __syncthreads();  // s_maxlim, barriers initialised

  // ---- this thread's query row (softmax warps): row = TMEM lane ----
  const bool sm_warp = warp >= kTcCtl;
  const int hc = sm_warp ? (warp - kTcCtl) >> 2 : 0;  // column half of this warp
  const int q4 = warp & 3;                            // lane group (TMEM access rule)
  const int row = 32 * q4 + lane;
  const T *qrow = nullptr;
  int lim = 0, rseq = 0, ru = 0, rh = 0;
  if (sm_warp) {
    const int rho = row_base + row;
    if (rho < rows_total) {
      const int sq = shared ? rho / rows_per_seq : zseq;
      const int rr = rho % rows_per_seq;
      const int u = rr / a.group, h = kvh * a.group + rr % a.group;
      const int L = max(0, __ldg(a.context_lens + sq));
      int visible = L - a.q_len + u + 1;  // causal limit
      if (shared) visible = min(visible, nb * kTileTokens);
      rseq = sq;
      ru = u;
      rh = h;
      lim = visible;
      qrow = static_cast<const T *>(a.q) + ((size_t)(sq * a.q_len + u) * a.num_q_heads + h) * D;
      if (hc == 0) atomicMax(&s_maxlim, visible);
    }
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = s_tmem;
  // blocks any row of this CTA can see, and the chunks covering them
  const int t_end = min(te, max(tb, (s_maxlim + kTileTokens - 1) / kTileTokens));
  const int nch = (t_end - tb + kTcBlocks - 1) / kTcBlocks;
  const int vis_end = min(te * kTileTokens, s_maxlim);  // no row uses a position past it
  volatile int *failed = &s_failed;
  if (a.q_tma && nch > 0 && threadIdx.x == 0) {
    // the row block's 128 query rows (token, head): tokens [t0, t0 + 128/g) of heads
    // [kvh*g, kvh*g + g) (rows past the sequence's last token are never written
    // back; past the tensor they are zero-filled).  The S thread waits for them.
    const int t0 = (shared ? 0 : zseq * a.q_len) + row_base / a.group;
    const uint32_t bar = smem_u32(&q_full);
    mbar_arrive_expect_tx(bar, Lay::kQBytes);
#pragma unroll
    for (int hh = 0; hh < H; ++hh) tma_load_3d(base + hh * (kTcRows * 128), &qmap, hh * 64, kvh * a.group, t0, bar);
  }

  if (warp < 2) {
    // ------------------------------------------------------------ TMA producers
    const bool is_k = warp == 0;
    const CUtensorMap *map = is_k ? &kmap : &vmap;
    const uint32_t ring = is_k ? sK : sV;
    uint64_t *full = is_k ? k_full : v_full;
    uint64_t *empty = is_k ? k_empty : v_empty;
    const int NS = is_k ? NK : NV;
    const int32_t *table = a.block_tables + (size_t)tseq * a.max_blocks_per_seq;
    int issued = 0;
    bool ok = true;
    // block-table window: lane l holds entry tb + 32w + l of window w (4 chunks);
    // the next window is loaded a whole window ahead, so no TMA issue waits on a
    // table load
    auto table_at = [&](int w) -> int {
      const int blk = tb + 32 * w + lane;
      return blk < t_end ? __ldg(table + blk) : -1;
    };
    int win_cur = table_at(0), win_nxt = table_at(1);
    for (int ch = 0; ch < nch; ++ch) {
      const int s = ch % NS;
      if (ch > 0 && (ch & 3) == 0) {  // next window of 32 entries
        win_cur = win_nxt;
        win_nxt = table_at((ch >> 2) + 1);
      }
      // a fresh barrier counts as released (parity 1 of the phase before the first)
      bool fr = mbar_wait_bounded(smem_u32(&empty[s]), ((ch / NS) & 1) ^ 1);
      fr = __all_sync(0xffffffffu, fr);
      if (!fr || *failed) {
        ok = fr;
        break;
      }
      const int blk = tb + ch * kTcBlocks + lane;
      const int phys = __shfl_sync(0xffffffffu, win_cur, ((ch & 3) * kTcBlocks + lane) & 31);
      int z = -1;  // outside the tensor map: zero fill
      if (lane < kTcBlocks && blk < t_end) {
        if (phys >= 0 && phys < a.num_blocks)
          z = phys * a.num_kv_heads + kvh;
        else if (is_k)
          record_error(a.err, kErrCheck);
      }
      const uint32_t bar = smem_u32(&full[s]);
      if (lane == 0) mbar_arrive_expect_tx(bar, Lay::kKVBytes);
      __syncwarp();
      if (lane < kTcBlocks) {
        const uint32_t dst = ring + s * Lay::kKVBytes + lane * (kTileTokens * 128);
#pragma unroll
        for (int hh = 0; hh < H; ++hh) tma_load_3d(dst + hh * (kTcChunk * 128), map, hh * 64, 0, z, bar);
      }
      issued = ch + 1;
    }
    if (!ok && lane == 0) {
      record_error(a.err, kErrTimeout);
      atomicExch(&s_failed, 1);
    }
    if (*failed) {
      // the loads still in flight land before the CTA may exit (bounded)
      for (int k = max(0, issued - NS); k < issued; ++k)
        (void)mbar_wait_bounded(smem_u32(&full[k % NS]), (k / NS) & 1);
    }
  } else if (warp == 2 || warp == 3) {
    // ------------------------------------------------------------ MMA issue
    constexpr uint32_t kIdS = tc::idesc_f16(kTcRows, kTcChunk, kBf16, false);
    constexpr uint32_t kIdO = tc::idesc_f16(kTcRows, D, kBf16, true);
    // descriptors of the first stage; the others differ only in the start address
    // field (bits 0-13, address / 16), so an offset is a plain addition
    const uint64_t dQ = tc::sdesc_sw128(base, 16, 1024);
    const uint64_t dK = tc::sdesc_sw128(sK, 16, 1024);
    const uint64_t dV = tc::sdesc_sw128(sV, kTcChunk * 128, 1024);
    bool ok = true;
    auto wait_all = [&](uint64_t *bar, int parity) -> bool {
      bool w = mbar_wait_bounded(smem_u32(bar), parity);
      w = __all_sync(0xffffffffu, w);
      return w && !*failed;
    };
    if (warp == 3) {
      // S_j = Q K_j^T into S buffer j % 3
      if (nch > 0) ok = a.q_tma ? wait_all(&q_full, 0) : wait_all(&q_ready, 0);
      for (int j = 0; ok && j < nch; ++j) {
        ok = wait_all(&k_full[j % NK], (j / NK) & 1);
        // the buffer's last reader, P_{j-3} V_{j-3}, has completed (its barrier is at
        // most one phase behind: P_j V_j needs S_j first)
        if (ok && j >= 3) ok = wait_all(&bfree[j % 3], ((j - 3) / 3) & 1);
        if (!ok) break;
        tc::fence_after();
        if (lane == 0) {
          const uint64_t kd = dK + (uint64_t)(((j % NK) * Lay::kKVBytes) >> 4);
          const uint32_t dst = tmem + Lay::kColS + kTcChunk * (j % 3);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            // a K step of 16 columns: +32 bytes inside the 128-byte row, +one
            // column-group block every 4 steps (descriptor addresses count 16 bytes)
            tc::mma_f16(dst, dQ + (uint64_t)(((kk >> 2) * (kTcRows * 128) + (kk & 3) * 32) >> 4),
                        kd + (uint64_t)(((kk >> 2) * (kTcChunk * 128) + (kk & 3) * 32) >> 4), kIdS,
                        kk > 0 ? 1u : 0u);
          }
          tc::commit(smem_u32(&s_full[j % 3]));
          tc::commit(smem_u32(&k_empty[j % NK]));
        }
        __syncwarp();
      }
    } else {
      // O += P_j V_j, P from S buffer j % 3
      for (int j = 0; ok && j < nch; ++j) {
        ok = wait_all(&v_full[j % NV], (j / NV) & 1);
        if (ok) ok = wait_all(&p_full, j & 1);
        if (!ok) break;
        tc::fence_after();
        if (lane == 0) {
          mbar_arrive(smem_u32(&p_ack));  // the softmax may announce P_{j+1}
          const uint64_t vd = dV + (uint64_t)(((j % NV) * Lay::kKVBytes) >> 4);
          const uint32_t pa = tmem + Lay::kColS + kTcChunk * (j % 3);
#pragma unroll
          for (int kk = 0; kk < kTcChunk / 16; ++kk) {
            // V is N-major (head_dim contiguous): atoms of 64 columns kTcChunk*128
            // bytes apart (the descriptor's leading offset), groups of 8 positions
            // 1024 bytes apart; a K step of 16 positions is 2048 bytes of V and 8
            // tensor-memory columns of P (positions 64h.. in columns 64h.., hi then lo)
            const uint64_t bd = vd + (uint64_t)((kk * (16 * 128)) >> 4);
            const uint32_t pc = pa + (kk >> 2) * 64 + (kk & 3) * 8;
            tc::mma_f16_ts(tmem, pc, bd, kIdO, (j > 0 || kk > 0) ? 1u : 0u);
            if (Lay::kSplitP) tc::mma_f16_ts(tmem, pc + 32, bd, kIdO, 1u);
          }
          tc::commit(smem_u32(&o_done[j & 1]));
          tc::commit(smem_u32(&v_empty[j % NV]));
          tc::commit(smem_u32(&bfree[j % 3]));
        }
        __syncwarp();
      }
    }
    if (!ok && lane == 0) {
      record_error(a.err, kErrTimeout);
      atomicExch(&s_failed, 1);
    }
    // every MMA this thread issued has completed before tensor memory is released
    if (lane == 0) tc::commit(smem_u32(&mma_fin));
    __syncwarp();
    (void)mbar_wait_bounded(smem_u32(&mma_fin), 0);
  } else {
    // ------------------------------------------------------------ softmax rows
    const uint32_t trow = tmem + ((uint32_t)(32 * q4) << 16);
    // Q row -> shared memory in the swizzled K-major layout of the MMA's A operand
    // (each warp of the pair writes half of the row's 16-byte chunks), unless TMA
    // brings it
#pragma unroll
    for (int ci = 0; ci < (a.q_tma ? 0 : D / 16); ++ci) {
      const int c = hc * (D / 16) + ci;
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if (qrow) v = __ldg(reinterpret_cast<const uint4 *>(qrow) + c);
      const int hh = c >> 3, cc = c & 7;
      const uint32_t addr = base + hh * (kTcRows * 128) + row * 128 + ((cc ^ (row & 7)) << 4);
      asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y),
                   "r"(v.z), "r"(v.w)
                   : "memory");
    }
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&q_ready));

    const float rs = a.scale_log2;
    const uint64_t rs2 = tc::f2pack(rs, rs);
    const int lim_row = min(lim, te * kTileTokens);  // padding rows: 0
    float m_run = -INFINITY, l = 0.f;
    bool ok = true;
    int xph = 0;  // exchanges done (phase of xbar[q4])
    const int tid = (warp - kTcCtl) * 32 + lane;  // 0..255
    // max (or, at the end, sum) of this warp's value and the partner warp's
    auto exchange = [&](float v, bool is_max) -> float {
      xval[xph & 1][hc][row] = v;
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&xbar[q4]));
      bool w = mbar_wait_bounded(smem_u32(&xbar[q4]), xph & 1);
      w = __all_sync(0xffffffffu, w);
      if (!w) ok = false;
      const float o = xval[xph & 1][hc ^ 1][row];
      ++xph;
      return is_max ? fmaxf(v, o) : v + o;
    };
    for (int j = 0; j < nch; ++j) {
      const int b = j % 3;
      const uint32_t ts = trow + Lay::kColS + kTcChunk * b + 64 * hc;  // this warp's columns
      bool w = mbar_wait_bounded(smem_u32(&s_full[b]), (j / 3) & 1);
      w = __all_sync(0xffffffffu, w);
      if (!w) {
        ok = false;
        break;
      }
      tc::fence_after();
      const int c0 = (tb + j * kTcBlocks) * kTileTokens + 64 * hc;  // first position here
      float sv[64];
      tc::ld64(ts, sv);
      // scale to base-2 units (two lanes per instruction), mask, row maximum
#pragma unroll
      for (int c = 0; c < 64; c += 2) {
        const uint64_t x = tc::fmul2(tc::f2pack(sv[c], sv[c + 1]), rs2);
        tc::f2unpack(x, sv[c], sv[c + 1]);
      }
      if (c0 + 64 > lim_row) {
#pragma unroll
        for (int c = 0; c < 64; ++c) sv[c] = (c0 + c < lim_row) ? sv[c] : -INFINITY;
      }
      float pm[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) pm[i] = sv[i];
#pragma unroll
      for (int c = 8; c < 64; ++c) pm[c & 7] = fmaxf(pm[c & 7], sv[c]);
      float mx = fmaxf(fmaxf(fmaxf(pm[0], pm[1]), fmaxf(pm[2], pm[3])),
                       fmaxf(fmaxf(pm[4], pm[5]), fmaxf(pm[6], pm[7])));
      mx = exchange(mx, true);  // the whole chunk's row maximum
      if (!ok) break;
      const float m_new = fmaxf(m_run, mx);
      const bool need = m_new > m_run + kTcRescale;  // false while both are -inf
      const float f = need ? ex2_ftz(m_run - m_new) : 1.f;  // 0 when m_run = -inf
      if (need) {
        l *= f;
        m_run = m_new;
      }
      const float mb = (m_run == -INFINITY) ? 0.f : m_run;
      const uint64_t nmb2 = tc::f2pack(-mb, -mb);
      uint64_t ps2[2] = {0ull, 0ull};  // packed partial sums (+0.0f, +0.0f)
      {
        // P over these S columns: hi words in the first 32, lo words (bf16) next
        uint32_t hw[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          float x0, x1;
          tc::f2unpack(tc::fadd2(tc::f2pack(sv[2 * e], sv[2 * e + 1]), nmb2), x0, x1);
          const float p0 = ex2_ftz(x0), p1 = ex2_ftz(x1);
          if constexpr (Lay::kSplitP) {
            // hi = p truncated to bf16 (exact); lo = p - hi (exact in fp32), kept in sv
            const uint32_t u0 = __float_as_uint(p0), u1 = __float_as_uint(p1);
            hw[e] = __byte_perm(u0, u1, 0x7632);
            const uint64_t pp = tc::f2pack(p0, p1);
            const uint64_t hh = tc::f2pack(__uint_as_float(u0 & 0xffff0000u),
                                           __uint_as_float(u1 & 0xffff0000u));
            tc::f2unpack(tc::ffma2(hh, tc::f2pack(-1.f, -1.f), pp), sv[2 * e], sv[2 * e + 1]);
            ps2[e & 1] = tc::fadd2(ps2[e & 1], pp);
          } else {
            hw[e] = Elt<T>::from_f2(p0, p1);
            // the sum of the rounded weights P V is taken with: the quotient O / l
            // is then an exact convex combination of V rows (a dominant weight's
            // rounding cancels)
            const float2 hf = Elt<T>::to_f2(hw[e]);
            ps2[e & 1] = tc::fadd2(ps2[e & 1], tc::f2pack(hf.x, hf.y));
          }
        }
        tc::st32u(ts, hw);
        if constexpr (Lay::kSplitP) {
#pragma unroll
          for (int e = 0; e < 32; ++e) hw[e] = Elt<T>::from_f2(sv[2 * e], sv[2 * e + 1]);
          tc::st32u(ts + 32, hw);
        }
      }
      {
        float a0, a1, b0, b1;
        tc::f2unpack(ps2[0], a0, a1);
        tc::f2unpack(ps2[1], b0, b1);
        l += (a0 + a1) + (b0 + b1);
      }
      // O rescale: P_{j-1} V_{j-1} (and with it every earlier P V) must be complete.
      // S_j's completion implies P_{j-3} V_{j-3}'s and P_j V_j is not issued yet, so
      // the barrier of odd / even chunks that P_{j-1} V_{j-1} commits to is at most
      // one phase behind: a parity wait is exact
      if (j > 0 && __any_sync(0xffffffffu, need)) {  // (the pair decides alike)
        w = mbar_wait_bounded(smem_u32(&o_done[(j - 1) & 1]), ((j - 1) >> 1) & 1);
        w = __all_sync(0xffffffffu, w);
        if (!w) {
          ok = false;
          break;
        }
        tc::fence_after();
        {
          const uint64_t f2 = tc::f2pack(f, f);
#pragma unroll
          for (int qq = 0; qq < kOCols / 32; ++qq) {
            float o[32];
            const uint32_t oc = trow + hc * kOCols + 32 * qq;
            tc::ld32(oc, o);
#pragma unroll
            for (int i = 0; i < 32; i += 2) {
              const uint64_t x = tc::fmul2(tc::f2pack(o[i], o[i + 1]), f2);
              tc::f2unpack(x, o[i], o[i + 1]);
            }
            tc::st32(oc, o);
          }
        }
      }
      const int cs = (tb + j * kTcBlocks) * kTileTokens;  // the chunk's first position
      if (cs + kTcChunk > vis_end) {
        // V rows at or past vis_end may be unused slots holding anything; P is 0
        // there but 0 * NaN is not 0, so they become zeros before P V
        const int s = j % NV;
        w = mbar_wait_bounded(smem_u32(&v_full[s]), (j / NV) & 1);
        w = __all_sync(0xffffffffu, w);
        if (!w) {
          ok = false;
          break;
        }
        const int first = max(0, vis_end - cs);
        const uint32_t vb = sV + s * Lay::kKVBytes;
        for (int idx = tid; idx < (kTcChunk - first) * H * 8; idx += 32 * kTcSoft) {
          const int r = first + idx / (H * 8), rem = idx % (H * 8);
          const int hh = rem >> 3, cc = rem & 7;
          sts128_zero(vb + hh * (kTcChunk * 128) + r * 128 + ((cc ^ (r & 7)) << 4));
        }
        fence_proxy_async_smem();  // the zeros visible to the tensor core
      }
      tc::st_wait();  // P_j (and a rescaled O) are in tensor memory
      // the MMA thread has taken P_{j-1}: p_full may move on
      if (j > 0) {
        w = mbar_wait_bounded(smem_u32(&p_ack), (j - 1) & 1);
        w = __all_sync(0xffffffffu, w);
        if (!w) {
          ok = false;
          break;
        }
      }
      tc::fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&p_full));
    }
    if (!ok && lane == 0) {
      record_error(a.err, kErrTimeout);
      atomicExch(&s_failed, 1);
    }
    // ---- epilogue: O / l, or the unnormalised partial with its statistics ----
    bool have = ok && nch > 0;
    if (have) {
      // every MMA of this CTA has completed
      bool w = mbar_wait_bounded(smem_u32(&mma_fin), 0);
      w = __all_sync(0xffffffffu, w);
      if (!w) {
        have = false;
        ok = false;
        if (lane == 0) {
          record_error(a.err, kErrTimeout);
          atomicExch(&s_failed, 1);
        }
      } else {
        tc::fence_after();
      }
    }
    if (ok) l = exchange(l, false);  // the row sum over both column halves
    const bool write = ok && qrow != nullptr;
    const float inv = l > 0.f ? 1.f / l : 0.f;
    size_t wrow = 0;
    if (PARTIAL)
      wrow = ((size_t)rseq * a.ws_splits + a.ws_split0 + split) * (a.q_len * a.num_q_heads) +
             (size_t)ru * a.num_q_heads + rh;
    const size_t orow = (size_t)(rseq * a.q_len + ru) * a.num_q_heads + rh;
#pragma unroll
    for (int qq = 0; qq < kOCols / 32; ++qq) {
      const int col = hc * kOCols + 32 * qq;
      float o[32];
      if (have) {
        tc::ld32(trow + col, o);
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) o[i] = 0.f;
      }
      if (!write) continue;
      if constexpr (PARTIAL) {
        float4 *dst = reinterpret_cast<float4 *>(a.ws_acc + wrow * D + col);
#pragma unroll
        for (int i = 0; i < 8; ++i) dst[i] = make_float4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
      } else {
        uint4 *dst = reinterpret_cast<uint4 *>(static_cast<T *>(a.out) + orow * D + col);
#pragma unroll
        for (int i = 0; i < 4; ++i)
          dst[i] = make_uint4(Elt<T>::from_f2(o[8 * i] * inv, o[8 * i + 1] * inv),
                              Elt<T>::from_f2(o[8 * i + 2] * inv, o[8 * i + 3] * inv),
                              Elt<T>::from_f2(o[8 * i + 4] * inv, o[8 * i + 5] * inv),
                              Elt<T>::from_f2(o[8 * i + 6] * inv, o[8 * i + 7] * inv));
      }
    }
    if (PARTIAL && write && hc == 0) {
      a.ws_m[wrow] = have ? m_run : -INFINITY;
      a.ws_l[wrow] = have ? l : 0.f;
    }
  }

  // ---- teardown: every tensor-memory access is complete; release it ----
  tc::fence_before();
  __syncthreads();
  if (warp == 2) {
    tc::fence_after();
    tc::dealloc(tmem, Lay::kTmemCols);
  }
}

}  // namespace pa
