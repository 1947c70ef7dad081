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
// A unit = one KV head x one partition of the walked blocks x 128 query rows (the
// MMA's M).  The CTAs are persistent, one per SM, and each walks its own list of
// units (longest first, see tc_unit); the cache is walked in chunks of 128
// positions (8 blocks), and every ring, buffer and barrier runs on through the
// chunks of all the CTA's units, so the next unit's loads and scores start while
// the previous one is finishing:
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
//               and the final O / l is the same quotient).  A unit's results,
//               O / l (or the partial statistics) for the warp's half of the
//               columns, are written during the next unit's first chunk, through a
//               shared-memory transpose into whole 64-byte row pieces.
// S_{j+1} and S_{j+2} are computed while the softmax works on S_j.  S_{j+3} is issued
// only after the commit of P_j V_j (the last reader of buffer j % 3) has fired.  A
// unit's Q replaces the previous one once that unit's last S MMA has completed
// (by TMA from the S thread, or written by the softmax warps before the previous
// unit's epilogue); a unit's first P V overwrites O, which the softmax warps have
// read out before they announce that unit's first P.  bf16 P is split into hi + lo
// bf16 parts, both multiplied by V, so that P keeps ~16 significant bits as the
// fp16 path does.  Every wait is bounded.
//
// FP8 (e4m3) cache (KV8): the producers load each chunk's codes (128 positions x
// 128 bytes) into the first half of a ring stage, then widen them in place to fp16
// in the layout the 16-bit path loads (e4m3 is exact in fp16), and only then
// release the stage to the MMA issuers; the MMAs run on fp16 operands.  Each KV
// head's K scale goes into the score scale and its V scale into the output; a
// bf16 q row is scaled into fp16 by a power of two that its score scale undoes.
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
// Over an FP8 cache four more warps widen the codes (one per scheduler), and the
// softmax warps come after them
constexpr int kTcConv = 4;
constexpr int kTcThreads8 = 32 * (kTcCtl + kTcConv + kTcSoft);
// FP8 register split (setmaxnreg): the control and widening warpgroups give up
// registers to the two softmax warpgroups.  2 x 128 x 112 + 2 x 128 x 144 =
// 65 536 = 512 threads x 128, the registers the block is launched with (the
// smallest split at which no region of the kernel spills).
constexpr int kTcRegsLow8 = 112;
constexpr int kTcRegsSoft8 = 144;
constexpr int kTcRegsLaunch8 = 128;
static_assert(2 * 128 * kTcRegsLow8 + 2 * 128 * kTcRegsSoft8 == kTcThreads8 * kTcRegsLaunch8,
              "register split");
constexpr float kTcRescale = 8.f;                  // base-2 growth that forces a rescale
constexpr int kTcScrBytes = 32 * 64;               // epilogue scratch per softmax warp

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
  // after the rings: a 2 KiB scratch per softmax warp (the epilogue's transpose)
  static constexpr int kScrBytes = kTcSoft * kTcScrBytes;
  static constexpr int smem_bytes(int nk, int nv) {
    return kOffStages + (nk + nv) * kKVBytes + kScrBytes + 1024;
  }
};

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// max(a, b, c) in one instruction (sm_100 and later); NaN inputs are ignored as
// by fmaxf
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// 2^x (PTX ex2.approx, flushing subnormal results to zero: a weight below 2^-126
// of the row maximum contributes nothing at fp32 accumulation anyway)
__device__ __forceinline__ float ex2_ftz(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// n / d for 0 <= n < 2^31 by a multiply and a shift (Granlund and Montgomery,
// "Division by invariant integers using multiplication", 1994): with l = ceil(log2 d)
// and m = ceil(2^(31+l) / d) < 2^32, floor(n m / 2^(31+l)) = floor(n / d), because
// the rounding of m adds less than n / 2^(31+l) < 1 / d to n / d.
struct FastDiv {
  uint32_t m;
  int s, d;
  __device__ __forceinline__ void init(int dv) {
    d = dv;
    m = 0u;
    s = 0;
    if (dv > 1) {
      const int l = 32 - __clz(dv - 1);
      m = (uint32_t)(((1ull << (31 + l)) + (unsigned long long)(dv - 1)) / (unsigned long long)dv);
      s = l - 1;
    }
  }
  __device__ __forceinline__ int div(int n) const {
    return d <= 1 ? n : (int)(__umulhi((uint32_t)n, m) >> s);
  }
};

// The launch's unit geometry, computed once per thread.
struct TcGeo {
  FastDiv kvh, splits, nrb, group, rps;
  int rows_per_seq, rows_total, nrb_n;
  long long units;
  __device__ __forceinline__ void init(const DecodeArgs &a) {
    const bool shared = a.shared_prefix > 0;
    rows_per_seq = a.q_len * a.group;
    rows_total = shared ? a.num_seqs * rows_per_seq : rows_per_seq;
    nrb_n = (rows_total + kTcRows - 1) / kTcRows;
    units = (long long)nrb_n * a.num_splits * (shared ? 1 : a.num_seqs) * a.num_kv_heads;
    kvh.init(a.num_kv_heads);
    splits.init(a.num_splits);
    nrb.init(nrb_n);
    group.init(a.group);
    rps.init(rows_per_seq);
  }
};

// One unit of work: a KV head x a partition of the walked blocks x 128 query rows.
// Every warp derives it from the unit's index alone, so the roles agree on it
// without exchanging anything.
struct TcUnit {
  int valid;
  int kvh, zseq, split, row_base, tseq;
  int tb, te;      // the partition: 16-token tiles [tb, te) of the walked table row
  int lwalk;       // positions of the walked row that hold tokens
  int t_end, nch;  // blocks any row of the unit sees, and the chunks covering them
  int vis_end;     // no row of the unit uses a position at or past it
  // the caller's row of the unit (row >= 0)
  int rvalid, rseq, ru, rh, vis;
};

// Units are numbered longest first: sequences by decreasing context length
// (s_order), within a sequence the last row block (the one that sees the most
// positions) first, then partition, then KV head.  CTA c takes units
// c, 2G - 1 - c, 2G + c, 4G - 1 - c, ... of G CTAs (back and forth), so every CTA
// gets one long and one short unit of each pair of rounds.  All lanes of the warp
// call it (the shared-prefix limit is a warp maximum).
__device__ __forceinline__ TcUnit tc_unit(const DecodeArgs &a, const TcGeo &geo, int k,
                                          const int *s_order, const int *lens, int lane, int row,
                                          bool rec, int bsz) {
  TcUnit t;
  const int G = gridDim.x;
  const bool shared = a.shared_prefix > 0;
  const long long id = (long long)k * G + ((k & 1) ? G - 1 - (int)blockIdx.x : (int)blockIdx.x);
  t.valid = id < geo.units;
  t.nch = 0;
  t.rvalid = 0;
  if (!t.valid) return t;
  int r = (int)id;  // units < 2^31 (host check)
  int q = geo.kvh.div(r);
  t.kvh = r - q * a.num_kv_heads;
  r = q;
  q = geo.splits.div(r);
  t.split = r - q * a.num_splits;
  r = q;
  q = geo.nrb.div(r);
  const int rbi = r - q * geo.nrb_n;
  r = q;
  t.zseq = shared ? 0 : (a.lpt ? s_order[r] : r);
  t.row_base = (geo.nrb_n - 1 - rbi) * kTcRows;
  t.tseq = t.zseq;  // block-table row that is walked (row 0 for a shared prefix)

  int nb;  // tiles
  const int Lt = max(0, lens[t.tseq]);
  if (shared) {
    nb = min(a.shared_prefix, a.max_tiles);
  } else {
    nb = (Lt + kTileTokens - 1) / kTileTokens;
    if ((int64_t)Lt > (int64_t)a.max_blocks_per_seq * bsz) {
      if (rec && t.kvh == 0 && t.split == 0) record_error(a.err, kErrCheck);
      nb = min(nb, a.max_tiles);
    }
  }
  t.lwalk = shared ? nb * kTileTokens : Lt;
  // tiles before first_block belong to another pass (a cascade's shared prefix);
  // the rest is cut into num_splits partitions of whole blocks (or tiles)
  const TileRange part = partition_tiles(nb, shared ? 0 : min(nb, a.first_block), a.num_splits,
                                         t.split, bsz);
  t.tb = part.tb;
  t.te = part.te;

  // the largest causal limit of the unit's rows: its last row's (one sequence), or
  // the largest over the sequences whose rows it holds (shared prefix)
  const int row_last = min(t.row_base + kTcRows, geo.rows_total) - 1;
  int mx;
  if (!shared) {
    mx = max(0, Lt - a.q_len + geo.group.div(row_last) + 1);
  } else {
    const int rps = geo.rows_per_seq;
    const int s0 = geo.rps.div(t.row_base), s1 = geo.rps.div(row_last);
    mx = 0;
    for (int sq = s0 + lane; sq <= s1; sq += 32) {
      const int last = min(row_last, sq * rps + rps - 1) - sq * rps;
      const int visible = min(max(0, lens[sq]) - a.q_len + geo.group.div(last) + 1, nb * kTileTokens);
      mx = max(mx, visible);
    }
    mx = __reduce_max_sync(0xffffffffu, mx);
  }
  t.t_end = min(t.te, max(t.tb, (mx + kTileTokens - 1) / kTileTokens));
  t.nch = (t.t_end - t.tb + kTcBlocks - 1) / kTcBlocks;
  t.vis_end = min(t.te * kTileTokens, mx);

  t.rseq = t.ru = t.rh = t.vis = 0;
  const int rho = t.row_base + row;
  if (row >= 0 && rho < geo.rows_total) {
    int sq = t.zseq, rr = rho;
    if (shared) {
      sq = geo.rps.div(rho);
      rr = rho - sq * geo.rows_per_seq;
    }
    const int u = geo.group.div(rr);
    const int L = shared ? max(0, lens[sq]) : Lt;
    int visible = L - a.q_len + u + 1;  // causal limit
    if (shared) visible = min(visible, nb * kTileTokens);
    t.rvalid = 1;
    t.rseq = sq;
    t.ru = u;
    t.rh = t.kvh * a.group + (rr - u * a.group);
    t.vis = visible;
  }
  return t;
}

template <bool B, class X, class Y> struct TcPick { using type = X; };
template <class X, class Y> struct TcPick<false, X, Y> { using type = Y; };

__device__ __forceinline__ void sts128(uint32_t addr, const uint4 v) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}

// Widen the e4m3 codes of `rows` positions of a chunk in place, from position r0
// (one warp).  The codes of position r
// sit in bytes [128 r, 128 r + 128) of the stage, 16-byte chunk c (dims 16c ..
// 16c + 15) at chunk position c ^ (r % 8), as TMA writes them with the 128-byte
// swizzle.  The fp16 result takes the 16-bit tile layout: dims 64h .. 64h + 63 of
// position r in bytes [h * 16384 + 128 r, +128), 16-byte chunk c' at c' ^ (r % 8).
// Lane l widens positions r0 + l, r0 + l + 32, ...: it reads a position's eight
// chunks before it writes over them, and no other lane touches that position, so
// no synchronisation is needed inside the loop.  Every 8 lanes of a shared-memory
// phase hit 8 distinct 16-byte bank groups (r % 8 differs between them).
__device__ __forceinline__ void tc_widen_e4m3_rows(uint32_t st, int r0, int rows, int lane) {
#pragma unroll 1
  for (int k = 0; k < rows / 32; ++k) {
    const int r = r0 + 32 * k + lane;
    const uint32_t src = st + r * 128;
    // dims 64 .. 127 first: they go to the second half, which holds no codes; then
    // dims 0 .. 63, all four chunks read before the first write over the codes row
#pragma unroll
    for (int h = 1; h >= 0; --h) {
      uint4 v[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) v[i] = lds128(src + (((4 * h + i) ^ (r & 7)) << 4));
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        uint4 lo, hi;
        lo.x = e4m3_lo_f16x2(v[i].x);
        lo.y = e4m3_hi_f16x2(v[i].x);
        lo.z = e4m3_lo_f16x2(v[i].y);
        lo.w = e4m3_hi_f16x2(v[i].y);
        hi.x = e4m3_lo_f16x2(v[i].z);
        hi.y = e4m3_hi_f16x2(v[i].z);
        hi.z = e4m3_lo_f16x2(v[i].w);
        hi.w = e4m3_hi_f16x2(v[i].w);
        const uint32_t row = st + h * (kTcChunk * 128) + r * 128;
        sts128(row + (((2 * i) ^ (r & 7)) << 4), lo);
        sts128(row + (((2 * i + 1) ^ (r & 7)) << 4), hi);
      }
    }
  }
}

// BS16: the cache's blocks are 16 tokens (fixed at compile time); otherwise the
// block size (8 or 32) is read from the arguments.
template <typename T, int D, int NK, int NV, bool PARTIAL, bool KV8, bool BS16>
__global__ void __launch_bounds__(KV8 ? kTcThreads8 : kTcThreads, 1)
    paged_prefill_tc_kernel(const __grid_constant__ CUtensorMap kmap,
                            const __grid_constant__ CUtensorMap vmap,
                            const __grid_constant__ CUtensorMap qmap, const DecodeArgs a) {
  // MMA operand type: fp16 over an FP8 cache (codes widened; q converted), else T
  using TM = typename TcPick<KV8, __half, T>::type;
  using Lay = TcLayout<TM, D>;
  constexpr int H = Lay::kHalves;
  constexpr bool kBf16 = Elt<TM>::kMantBits < 10;
  static_assert(!KV8 || D == 128, "FP8 cache: head_dim 128");
  constexpr int kSoft0 = KV8 ? kTcCtl + kTcConv : kTcCtl;  // first softmax warp
  const int kBsz = BS16 ? 16 : a.block_size;
  constexpr int kOCols = D / 2;  // O columns per softmax warp
  static_assert(NK >= 2 && NV >= 2, "ring depth");
  static_assert(D == 64 || D == 128, "head_dim");

  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t k_full[NK];
  __shared__ __align__(8) uint64_t k_empty[NK];
  __shared__ __align__(8) uint64_t v_full[NV];
  __shared__ __align__(8) uint64_t v_empty[NV];
  __shared__ __align__(8) uint64_t k_land[NK];   // FP8: the codes have landed (TMA)
  __shared__ __align__(8) uint64_t v_land[NV];
  __shared__ __align__(8) uint64_t s_full[3];
  __shared__ __align__(8) uint64_t p_full;
  __shared__ __align__(8) uint64_t p_ack;        // the MMA thread has taken P_j
  __shared__ __align__(8) uint64_t o_done[2];   // P_j V_j complete, j even / odd
  __shared__ __align__(8) uint64_t bfree[3];    // P_j V_j complete, by S/P buffer j % 3
  __shared__ __align__(8) uint64_t q_ready;      // Q written by the softmax threads
  __shared__ __align__(8) uint64_t q_full;       // Q landed by TMA
  __shared__ __align__(8) uint64_t q_free;       // a unit's last S MMA has read Q
  __shared__ __align__(8) uint64_t mma_fin;
  __shared__ __align__(8) uint64_t xbar[4];      // partner exchange, per group of 32 rows
  __shared__ float xval[2][2][kTcRows];           // [parity][column half][row]
  __shared__ int s_order[kLptMaxSeqs];            // rank -> sequence, longest first
  __shared__ int s_lens[kLptMaxSeqs];
  __shared__ uint32_t s_tmem;
  __shared__ int s_failed;

  griddep_wait();
  griddep_launch_dependents();

  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t sK = base + Lay::kOffStages;  // K ring: NK x kKVBytes
  const uint32_t sV = sK + NK * Lay::kKVBytes;  // V ring: NV x kKVBytes
  const uint32_t sScr = sV + NV * Lay::kKVBytes;  // epilogue scratch
  const bool shared = a.shared_prefix > 0;

  // the context lengths (read at every unit: a global load there would stall each
  // role between units) and their longest-first order (rank by counting; ties by
  // index)
  const int *lens = a.context_lens;
  if (a.num_seqs <= kLptMaxSeqs) {
    const int n = a.num_seqs;
    for (int i = threadIdx.x; i < n; i += blockDim.x) s_lens[i] = max(0, __ldg(a.context_lens + i));
    lens = s_lens;
    __syncthreads();
  }
  if (!shared && a.lpt) {
    const int n = a.num_seqs;
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
      const int li = s_lens[i];
      int rk = 0;
      for (int j = 0; j < n; ++j) {
        const int lj = s_lens[j];
        rk += (lj > li) | ((lj == li) & (j < i));
      }
      s_order[rk] = i;
    }
  }
  if (threadIdx.x == 0) {
    s_failed = 0;
    // over an FP8 cache a stage is full once both of its widening warps are done
    for (int s = 0; s < NK; ++s) {
      mbar_init(smem_u32(&k_full[s]), KV8 ? 2 : 1);
      mbar_init(smem_u32(&k_empty[s]), 1);
      mbar_init(smem_u32(&k_land[s]), 1);
    }
    for (int s = 0; s < NV; ++s) {
      mbar_init(smem_u32(&v_full[s]), KV8 ? 2 : 1);
      mbar_init(smem_u32(&v_empty[s]), 1);
      mbar_init(smem_u32(&v_land[s]), 1);
    }
    for (int b = 0; b < 3; ++b) mbar_init(smem_u32(&s_full[b]), 1);
    mbar_init(smem_u32(&p_full), kTcSoft);
    mbar_init(smem_u32(&p_ack), 1);
    mbar_init(smem_u32(&o_done[0]), 1);
    mbar_init(smem_u32(&o_done[1]), 1);
    for (int b = 0; b < 3; ++b) mbar_init(smem_u32(&bfree[b]), 1);
    mbar_init(smem_u32(&q_ready), kTcSoft);
    mbar_init(smem_u32(&q_full), 1);
    mbar_init(smem_u32(&q_free), 1);
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
  tc::fence_before();
  __syncthreads();  // order, barriers and tensor memory ready
  tc::fence_after();
  const uint32_t tmem = s_tmem;
  volatile int *failed = &s_failed;
  TcGeo geo;
  geo.init(a);
  if constexpr (KV8) {
    // warpgroups 0 (producers, issuers) and 1 (widening) give registers to 2 and 3
    // (softmax); every warp of a warpgroup executes the same instruction
    if (warp < kSoft0)
      asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kTcRegsLow8));
    else
      asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kTcRegsSoft8));
  }

  if (warp < 2) {
    // ------------------------------------------------------------ TMA producers
    const bool is_k = warp == 0;
    const CUtensorMap *map = is_k ? &kmap : &vmap;
    const uint32_t ring = is_k ? sK : sV;
    uint64_t *full = is_k ? k_full : v_full;
    uint64_t *empty = is_k ? k_empty : v_empty;
    // the barrier the loads complete on: over an FP8 cache the codes land first and
    // the widening warps announce the stage (full)
    uint64_t *land = KV8 ? (is_k ? k_land : v_land) : full;
    const int NS = is_k ? NK : NV;
    int g = 0, issued = 0;  // chunks of this CTA so far (all units), loads issued
    bool ok = true;
    for (int k = 0; ok; ++k) {
      const TcUnit t = tc_unit(a, geo, k, s_order, lens, lane, -1, is_k && lane == 0, kBsz);
      if (!t.valid) break;
      const int32_t *table = a.block_tables + (size_t)t.tseq * a.max_blocks_per_seq;
      // block-table window (16-token blocks: a block is a tile): lane l holds entry
      // tb + 32w + l of window w (4 chunks); the next window is loaded a whole window
      // ahead, so no TMA issue waits on a table load.  Other block sizes read their
      // entries per chunk.
      auto table_at = [&](int w) -> int {
        const int blk = t.tb + 32 * w + lane;
        return (kBsz == 16 && blk < t.t_end) ? __ldg(table + blk) : -1;
      };
      int win_cur = 0, win_nxt = 0;
      if (t.nch > 0) {
        win_cur = table_at(0);
        win_nxt = table_at(1);
      }
      for (int ch = 0; ch < t.nch; ++ch) {
        const int gg = g + ch;
        const int s = gg % NS;
        if (ch > 0 && (ch & 3) == 0) {  // next window of 32 entries
          win_cur = win_nxt;
          win_nxt = table_at((ch >> 2) + 1);
        }
        // a fresh barrier counts as released (parity 1 of the phase before the first)
        bool fr = mbar_wait_bounded(smem_u32(&empty[s]), ((gg / NS) & 1) ^ 1);
        fr = __all_sync(0xffffffffu, fr);
        if (!fr || *failed) {
          ok = false;
          if (!fr && lane == 0) {
            record_error(a.err, kErrTimeout);
            atomicExch(&s_failed, 1);
          }
          break;
        }
        // lane l loads tile tb + 8 ch + l of the chunk (16-token blocks: the window's
        // entry; 32-token blocks: half l % 2 of a block), or with 8-token blocks the
        // 8-row box of block 2 (tb + 8 ch) + l.  z stays -1 (zero fill) past the walk.
        const int bsz = kBsz;
        const int tile = t.tb + ch * kTcBlocks + (bsz == 8 ? (lane >> 1) : lane);
        const int phys = __shfl_sync(0xffffffffu, win_cur, ((ch & 3) * kTcBlocks + lane) & 31);
        int z = -1;  // outside the tensor map: zero fill
        if (lane < (bsz == 8 ? 2 * kTcBlocks : kTcBlocks) && tile < t.t_end) {
          int id = phys;
          if (bsz == 32) {
            id = __ldg(table + (tile >> 1));
          } else if (bsz == 8) {
            const int blk = 2 * tile + (lane & 1);
            id = (blk < a.max_blocks_per_seq && blk * 8 < t.lwalk) ? __ldg(table + blk) : kNoBlock;
          }
          z = tile_box(id, tile & 1, t.kvh, a.num_kv_heads, a.num_blocks, bsz, a.err);
        }
        const uint32_t bar = smem_u32(&land[s]);
        if (lane == 0) mbar_arrive_expect_tx(bar, KV8 ? Lay::kKVBytes / 2 : Lay::kKVBytes);
        __syncwarp();
        const int box_rows = bsz == 8 ? 8 : kTileTokens;
        if (lane < kTcChunk / box_rows) {
          const uint32_t dst = ring + s * Lay::kKVBytes + lane * (box_rows * 128);
          if constexpr (KV8) {
            tma_load_3d(dst, map, 0, 0, z, bar);  // box_rows positions x 128 codes
          } else {
#pragma unroll
            for (int hh = 0; hh < H; ++hh) tma_load_3d(dst + hh * (kTcChunk * 128), map, hh * 64, 0, z, bar);
          }
        }
        issued = gg + 1;
      }
      g += t.nch;
    }
    // the last loads have landed before the CTA may exit (bounded; at once unless a
    // consumer gave up)
    for (int k = max(0, issued - NS); k < issued; ++k)
      (void)mbar_wait_bounded(smem_u32(&land[k % NS]), (k / NS) & 1);
  } else if (KV8 && warp >= kTcCtl && warp < kSoft0) {
    // ------------------------------------------------------------ FP8 widening
    // warps 4, 5: K positions [0, 64) and [64, 128) of every chunk; 6, 7: V
    const int cw = warp - kTcCtl;
    const bool is_k = cw < 2;
    const int r0 = (cw & 1) * (kTcChunk / 2);
    const uint32_t ring = is_k ? sK : sV;
    uint64_t *land = is_k ? k_land : v_land;
    uint64_t *full = is_k ? k_full : v_full;
    const int NS = is_k ? NK : NV;
    int g = 0;
    bool ok = true;
    for (int k = 0; ok; ++k) {
      const TcUnit t = tc_unit(a, geo, k, s_order, lens, lane, -1, false, kBsz);
      if (!t.valid) break;
      for (int ch = 0; ch < t.nch; ++ch) {
        const int gg = g + ch;
        const int s = gg % NS;
        bool w = mbar_wait_bounded(smem_u32(&land[s]), (gg / NS) & 1);
        w = __all_sync(0xffffffffu, w);
        if (!w || *failed) {
          ok = false;
          if (!w && lane == 0) {
            record_error(a.err, kErrTimeout);
            atomicExch(&s_failed, 1);
          }
          break;
        }
        tc_widen_e4m3_rows(ring + s * Lay::kKVBytes, r0, kTcChunk / 2, lane);
        fence_proxy_async_smem();  // the fp16 rows visible to the tensor core
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&full[s]));
      }
      g += t.nch;
    }
  } else if (warp == 2 || warp == 3) {
    // ------------------------------------------------------------ MMA issue
    // bit 13 of the instruction descriptor negates A (Q): S = -Q K^T for a negative scale
    const uint32_t kIdS = tc::idesc_f16(kTcRows, kTcChunk, kBf16, false) | (a.s_negate ? (1u << 13) : 0u);
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
    int g = 0;
    if (warp == 3) {
      // S_j = Q K_j^T into S buffer j % 3 (j counts the chunks of all units)
      int qn = 0;            // units with chunks so far: the phase of q_full / q_ready / q_free
      bool q_flight = false;  // a Q load issued and not yet seen landed
      for (int k = 0; ok; ++k) {
        const TcUnit t = tc_unit(a, geo, k, s_order, lens, lane, -1, false, kBsz);
        if (!t.valid) break;
        if (t.nch == 0) continue;
        if (a.q_tma) {
          // the unit's 128 query rows (token, head): tokens [t0, t0 + 128/g) of heads
          // [kvh*g, kvh*g + g) (rows past the sequence's last token are never written
          // back; past the tensor they are zero-filled), once the previous unit's S
          // MMAs have finished reading the buffer
          if (qn > 0) ok = wait_all(&q_free, (qn - 1) & 1);
          if (!ok) break;
          if (lane == 0) {
            const int t0 = (shared ? 0 : t.zseq * a.q_len) + t.row_base / a.group;
            const uint32_t bar = smem_u32(&q_full);
            mbar_arrive_expect_tx(bar, Lay::kQBytes);
#pragma unroll
            for (int hh = 0; hh < H; ++hh)
              tma_load_3d(base + hh * (kTcRows * 128), &qmap, hh * 64, t.kvh * a.group, t0, bar);
          }
          __syncwarp();
          q_flight = true;
          ok = wait_all(&q_full, qn & 1);
          if (!ok) break;
          q_flight = false;
        } else {
          ok = wait_all(&q_ready, qn & 1);
          if (!ok) break;
        }
        // over an FP8 cache the scores carry the unit's K scale; a negative one
        // negates Q K^T as a negative softmax scale does
        uint32_t idS = kIdS;
        if (KV8 && __ldg(a.k_scale + t.kvh) < 0.f) idS ^= 1u << 13;
        for (int j = 0; ok && j < t.nch; ++j) {
          const int gg = g + j;
          ok = wait_all(&k_full[gg % NK], (gg / NK) & 1);
          // the buffer's last reader, P_{j-3} V_{j-3}, has completed (its barrier is at
          // most one phase behind: P_j V_j needs S_j first)
          if (ok && gg >= 3) ok = wait_all(&bfree[gg % 3], ((gg - 3) / 3) & 1);
          if (!ok) break;
          tc::fence_after();
          if (lane == 0) {
            const uint64_t kd = dK + (uint64_t)(((gg % NK) * Lay::kKVBytes) >> 4);
            const uint32_t dst = tmem + Lay::kColS + kTcChunk * (gg % 3);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              // a K step of 16 columns: +32 bytes inside the 128-byte row, +one
              // column-group block every 4 steps (descriptor addresses count 16 bytes)
              tc::mma_f16(dst, dQ + (uint64_t)(((kk >> 2) * (kTcRows * 128) + (kk & 3) * 32) >> 4),
                          kd + (uint64_t)(((kk >> 2) * (kTcChunk * 128) + (kk & 3) * 32) >> 4), idS,
                          kk > 0 ? 1u : 0u);
            }
            tc::commit(smem_u32(&s_full[gg % 3]));
            tc::commit(smem_u32(&k_empty[gg % NK]));
            if (j == t.nch - 1) tc::commit(smem_u32(&q_free));  // Q may be replaced
          }
          __syncwarp();
        }
        g += t.nch;
        ++qn;
      }
      if (q_flight) (void)mbar_wait_bounded(smem_u32(&q_full), (qn & 1));  // lands before exit
    } else {
      // O += P_j V_j, P from S buffer j % 3; a unit's first chunk overwrites O
      for (int k = 0; ok; ++k) {
        const TcUnit t = tc_unit(a, geo, k, s_order, lens, lane, -1, false, kBsz);
        if (!t.valid) break;
        for (int j = 0; ok && j < t.nch; ++j) {
          const int gg = g + j;
          ok = wait_all(&v_full[gg % NV], (gg / NV) & 1);
          if (ok) ok = wait_all(&p_full, gg & 1);
          if (!ok) break;
          tc::fence_after();
          if (lane == 0) {
            mbar_arrive(smem_u32(&p_ack));  // the softmax may announce P_{j+1}
            const uint64_t vd = dV + (uint64_t)(((gg % NV) * Lay::kKVBytes) >> 4);
            const uint32_t pa = tmem + Lay::kColS + kTcChunk * (gg % 3);
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
            tc::commit(smem_u32(&o_done[gg & 1]));
            tc::commit(smem_u32(&v_empty[gg % NV]));
            tc::commit(smem_u32(&bfree[gg % 3]));
          }
          __syncwarp();
        }
        g += t.nch;
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
    const int hc = (warp - kSoft0) >> 2;  // column half of this warp
    const int q4 = warp & 3;              // lane group (TMEM access rule)
    const int row = 32 * q4 + lane;       // = TMEM lane
    const uint32_t trow = tmem + ((uint32_t)(32 * q4) << 16);
    const int tid = (warp - kSoft0) * 32 + lane;  // 0..255
    // base-2 score scale of this thread's row (positive; see the host), per unit
    // over an FP8 cache: |K scale| and the row's q exponent folded in
    float rs = a.scale_log2;
    uint64_t rs2 = tc::f2pack(rs, rs);
    float vs_u = 1.f;  // the unit's V scale (FP8 cache)
    auto unit_scales = [&](const TcUnit &t, int e_row) {
      if constexpr (KV8) {
        const float r = a.scale_log2 * fabsf(__ldg(a.k_scale + t.kvh)) * ldexpf(1.f, e_row);
        rs = r > 0.f ? r : 1e-30f;
        rs2 = tc::f2pack(rs, rs);
        vs_u = __ldg(a.v_scale + t.kvh);
      }
    };
    bool ok = true;
    int xph = 0;  // exchanges done (phase of xbar[q4])
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
    auto q_ptr = [&](const TcUnit &t) -> const T * {
      return t.rvalid ? static_cast<const T *>(a.q) +
                            ((size_t)(t.rseq * a.q_len + t.ru) * a.num_q_heads + t.rh) * D
                      : nullptr;
    };
    // Q row -> shared memory in the swizzled K-major layout of the MMA's A operand
    // (each warp of the pair writes half of the row's 16-byte chunks).  Over an FP8
    // cache a bf16 row goes in as fp16 scaled by 2^-e, e the exponent of its largest
    // magnitude (both warps of the row find the same e); returns e.
    auto write_q = [&](const TcUnit &t) -> int {
      const T *qrow = q_ptr(t);
      constexpr bool kConv = KV8 && Elt<T>::kMantBits < 10;
      int e_row = 0;
      float down = 1.f;
      if constexpr (kConv) {
        float mx = 0.f;
        if (qrow) {
#pragma unroll 4
          for (int c = 0; c < D / 8; ++c) {
            const uint4 v = __ldg(reinterpret_cast<const uint4 *>(qrow) + c);
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const float2 f = Elt<T>::to_f2(w[i]);
              mx = fmaxf(mx, fmaxf(fabsf(f.x), fabsf(f.y)));
            }
          }
        }
        e_row = (mx > 0.f && isfinite(mx)) ? ilogbf(mx) : 0;
        down = ldexpf(1.f, -e_row);  // |q| * down < 2: well inside fp16
      }
#pragma unroll
      for (int ci = 0; ci < D / 16; ++ci) {
        const int c = hc * (D / 16) + ci;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (qrow) v = __ldg(reinterpret_cast<const uint4 *>(qrow) + c);
        if constexpr (kConv) {
          uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float2 f = Elt<T>::to_f2(w[i]);
            w[i] = Elt<__half>::from_f2(f.x * down, f.y * down);
          }
          v = make_uint4(w[0], w[1], w[2], w[3]);
        }
        const int hh = c >> 3, cc = c & 7;
        const uint32_t addr = base + hh * (kTcRows * 128) + row * 128 + ((cc ^ (row & 7)) << 4);
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y),
                     "r"(v.z), "r"(v.w)
                     : "memory");
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&q_ready));
      return e_row;
    };

    // ---- epilogue of a finished unit: O / l (or the unnormalised partial and its
    // statistics) from tensor memory to global memory.  The warp's 32 rows pass
    // through its shared-memory scratch, so that a store instruction writes 64-byte
    // pieces of 8 rows instead of 16 bytes of 32 rows (32 lines an instruction).
    // roff: the row's output (or workspace) row, -1 for padding rows.
    const uint32_t scr = sScr + (uint32_t)(warp - kSoft0) * kTcScrBytes;
    // sc multiplies O on the way out (1 / l, with the V scale of an FP8 cache); a
    // partial's O is multiplied by ovs (the V scale) and sc is its l
    auto epilogue = [&](bool have, int gl, float sc, float m_fin, long long roff, float ovs) -> bool {
      if (have) {
        // the unit's last P V (and with it every earlier one) has completed; the next
        // P V to commit to that barrier needs a P this warp has not announced yet
        bool w = mbar_wait_bounded(smem_u32(&o_done[gl & 1]), (gl >> 1) & 1);
        w = __all_sync(0xffffffffu, w);
        if (!w) return false;
        tc::fence_after();
      }
      constexpr int kEsz = PARTIAL ? 4 : (int)sizeof(T);
      char *gbase = PARTIAL ? reinterpret_cast<char *>(a.ws_acc) : static_cast<char *>(a.out);
      long long rj[4];  // rows 8 j + lane / 4: the ones this lane stores
#pragma unroll
      for (int j = 0; j < 4; ++j) rj[j] = __shfl_sync(0xffffffffu, roff, 8 * j + (lane >> 2));
#pragma unroll
      for (int qq = 0; qq < kOCols / 32; ++qq) {
        float o[32];
        if (have) {
          tc::ld32(trow + hc * kOCols + 32 * qq, o);
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = 0.f;
        }
#pragma unroll
        for (int h2 = 0; h2 < 32 * kEsz / 64; ++h2) {  // 64-byte pieces of these columns
          uint32_t wv[16];
          if constexpr (PARTIAL) {
#pragma unroll
            for (int i = 0; i < 16; ++i) wv[i] = __float_as_uint(o[16 * h2 + i] * ovs);
          } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) wv[i] = Elt<T>::from_f2(o[2 * i] * sc, o[2 * i + 1] * sc);
          }
          // row `lane`, 16-byte chunk c at position c ^ ((lane >> 1) & 3): no bank
          // conflict when written by row or read by column
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const uint32_t addr = scr + lane * 64 + ((c ^ ((lane >> 1) & 3)) << 4);
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(wv[4 * c]),
                         "r"(wv[4 * c + 1]), "r"(wv[4 * c + 2]), "r"(wv[4 * c + 3])
                         : "memory");
          }
          __syncwarp();
          const int c = lane & 3;
          const int col_b = (hc * kOCols + 32 * qq) * kEsz + 64 * h2 + 16 * c;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int r = 8 * j + (lane >> 2);
            uint4 v;
            asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                         : "r"(scr + r * 64 + ((c ^ ((r >> 1) & 3)) << 4))
                         : "memory");
            if (rj[j] >= 0) *reinterpret_cast<uint4 *>(gbase + rj[j] * (D * kEsz) + col_b) = v;
          }
          __syncwarp();  // read before the next piece is written
        }
      }
      if (PARTIAL && hc == 0 && roff >= 0) {
        a.ws_m[roff] = have ? m_fin : -INFINITY;
        a.ws_l[roff] = have ? sc : 0.f;
      }
      return true;
    };
    // a finished unit whose epilogue waits for the next unit's first chunk
    bool pend = false;
    int pend_gl = 0;
    float pend_sc = 0.f, pend_m = 0.f, pend_vs = 1.f;
    long long pend_roff = -1;

    int g = 0;   // chunks of this CTA so far (all units)
    int qn = 0;  // Q buffers written (without TMA)
    int e_cur = 0, e_next = 0;  // the row's q exponent (FP8 cache, bf16 q), this unit and next
    TcUnit cu = tc_unit(a, geo, 0, s_order, lens, lane, row, false, kBsz);
    if (!a.q_tma && cu.valid && cu.nch > 0) {
      e_cur = write_q(cu);
      qn = 1;
    }
    for (int k = 0; ok && cu.valid; ++k) {
      unit_scales(cu, e_cur);
      const int lim_row = cu.rvalid ? min(cu.vis, cu.te * kTileTokens) : 0;  // padding rows: 0
      float m_run = -INFINITY, l = 0.f;
      for (int j = 0; j < cu.nch; ++j) {
        const int gg = g + j;
        const int b = gg % 3;
        const uint32_t ts = trow + Lay::kColS + kTcChunk * b + 64 * hc;  // this warp's columns
        bool w = mbar_wait_bounded(smem_u32(&s_full[b]), (gg / 3) & 1);
        w = __all_sync(0xffffffffu, w);
        if (!w) {
          ok = false;
          break;
        }
        tc::fence_after();
        const int c0 = (cu.tb + j * kTcBlocks) * kTileTokens + 64 * hc;  // first position here
        float sv[64];
        tc::ld64(ts, sv);
        // mask, then the row maximum of the raw scores (three-input max, eight
        // independent chains); the scale is positive, so scaling the maximum gives
        // the maximum in base-2 units
        if (c0 + 64 > lim_row) {
#pragma unroll
          for (int c = 0; c < 64; ++c) sv[c] = (c0 + c < lim_row) ? sv[c] : -INFINITY;
        }
        float pm[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) pm[i] = fmax3(sv[i], sv[8 + i], sv[16 + i]);  // 0..23
#pragma unroll
        for (int c = 24; c < 56; c += 16) {  // 24..55
#pragma unroll
          for (int i = 0; i < 8; ++i) pm[i] = fmax3(pm[i], sv[c + i], sv[c + 8 + i]);
        }
        // the eight chains and 56..63
        const float q0 = fmax3(pm[0], pm[1], sv[56]), q1 = fmax3(pm[2], pm[3], sv[57]);
        const float q2 = fmax3(pm[4], pm[5], sv[58]), q3 = fmax3(pm[6], pm[7], sv[59]);
        float mx = fmax3(fmax3(q0, q1, sv[60]), fmax3(q2, q3, sv[61]), fmaxf(sv[62], sv[63]));
        mx = exchange(mx * rs, true);  // the whole chunk's row maximum
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
            tc::f2unpack(tc::ffma2(tc::f2pack(sv[2 * e], sv[2 * e + 1]), rs2, nmb2), x0, x1);
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
              hw[e] = Elt<TM>::from_f2(p0, p1);
              // the sum of the rounded weights P V is taken with: the quotient O / l
              // is then an exact convex combination of V rows (a dominant weight's
              // rounding cancels)
              const float2 hf = Elt<TM>::to_f2(hw[e]);
              ps2[e & 1] = tc::fadd2(ps2[e & 1], tc::f2pack(hf.x, hf.y));
            }
          }
          tc::st32u(ts, hw);
          if constexpr (Lay::kSplitP) {
#pragma unroll
            for (int e = 0; e < 32; ++e) hw[e] = Elt<TM>::from_f2(sv[2 * e], sv[2 * e + 1]);
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
        // one phase behind: a parity wait is exact.  (A unit's first chunk overwrites O.)
        if (j > 0 && __any_sync(0xffffffffu, need)) {  // (the pair decides alike)
          w = mbar_wait_bounded(smem_u32(&o_done[(gg - 1) & 1]), ((gg - 1) >> 1) & 1);
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
        if (j == 0 && pend) {
          // the previous unit's epilogue: its last P V has been completing under this
          // chunk's softmax.  This unit's first P V overwrites O, and is announced
          // only below.
          if (!epilogue(true, pend_gl, pend_sc, pend_m, pend_roff, pend_vs)) {
            ok = false;
            break;
          }
          pend = false;
        }
        const int cs = (cu.tb + j * kTcBlocks) * kTileTokens;  // the chunk's first position
        if (cs + kTcChunk > cu.vis_end) {
          // V rows at or past vis_end may be unused slots holding anything; P is 0
          // there but 0 * NaN is not 0, so they become zeros before P V
          const int s = gg % NV;
          w = mbar_wait_bounded(smem_u32(&v_full[s]), (gg / NV) & 1);
          w = __all_sync(0xffffffffu, w);
          if (!w) {
            ok = false;
            break;
          }
          const int first = max(0, cu.vis_end - cs);
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
        if (gg > 0) {
          w = mbar_wait_bounded(smem_u32(&p_ack), (gg - 1) & 1);
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
      if (!ok) break;

      // the next unit's Q (without TMA) goes in while this unit's P V drains: its
      // buffer is free once this unit's last S MMA has completed
      const TcUnit nu = tc_unit(a, geo, k + 1, s_order, lens, lane, row, false, kBsz);
      e_next = 0;
      if (!a.q_tma && nu.valid && nu.nch > 0) {
        if (qn > 0) {
          bool w = mbar_wait_bounded(smem_u32(&q_free), (qn - 1) & 1);
          w = __all_sync(0xffffffffu, w);
          if (!w) {
            ok = false;
            break;
          }
        }
        e_next = write_q(nu);
        ++qn;
      }

      // ---- the unit's results: deferred to the next unit's first chunk ----
      long long roff = -1;
      if (cu.rvalid)
        roff = PARTIAL ? (long long)(((size_t)cu.rseq * a.ws_splits + a.ws_split0 + cu.split) *
                                         (a.q_len * a.num_q_heads) +
                                     (size_t)cu.ru * a.num_q_heads + cu.rh)
                       : (long long)((size_t)(cu.rseq * a.q_len + cu.ru) * a.num_q_heads + cu.rh);
      if (cu.nch > 0) {
        l = exchange(l, false);  // the row sum over both column halves
        if (!ok) break;
        pend = true;
        pend_gl = g + cu.nch - 1;
        pend_sc = PARTIAL ? l : (l > 0.f ? vs_u / l : 0.f);
        pend_m = m_run;
        pend_vs = vs_u;
        pend_roff = roff;
      } else {
        // no position in this unit's partition: zeros (empty statistics)
        if (pend) {
          if (!epilogue(true, pend_gl, pend_sc, pend_m, pend_roff, pend_vs)) {
            ok = false;
            break;
          }
          pend = false;
        }
        if (!epilogue(false, 0, 0.f, 0.f, roff, 1.f)) {
          ok = false;
          break;
        }
      }
      g += cu.nch;
      cu = nu;
      e_cur = e_next;
    }
    if (ok && pend) ok = epilogue(true, pend_gl, pend_sc, pend_m, pend_roff, pend_vs);
    if (!ok && lane == 0) {
      record_error(a.err, kErrTimeout);
      atomicExch(&s_failed, 1);
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
