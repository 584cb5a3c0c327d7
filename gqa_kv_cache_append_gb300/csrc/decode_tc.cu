// decode_tc.cu - tensor-core (tcgen05 + TMEM) split-KV decode attention for
// bf16 or fp16 caches with head dims d_k, d_v in {64, 128}.
//
// The step of the MQA review §2.4 / §3 per (sequence i, KV head j) tile of
// T = 128 cached positions, with the r = h/g query heads of the group padded
// to NP columns (16 or 32) and positions on the MMA's M axis.  With n new
// tokens per sequence (the batched form of §2.3 restricted to the new
// rows), the columns are the n * r query rows of the group, token-major,
// and token s (at position L_i - n + s) sees positions p <= L_i - n + s:
//
//   S^T [T x NP]  = K_tile [T x d_k] . Q_g^T          (tcgen05.mma, M=128)
//   P^T [T x NP]  = exp2(S^T * scale*log2e - m)        (CUDA cores, per head)
//   O^T [d_v x NP] = V_tile^T [d_v x T] . P^T          (tcgen05.mma, M=128)
//
// Head dims of 64 use one 64-column box where 128 use two: the S product
// runs over d_k / 16 steps, and with d_v = 64 the O product still has M =
// 128 (the unloaded half of the V stage feeds output rows 64-127, which
// are never read).
//
// Roles (224 or 352 threads, one persistent CTA per SM):
//   warp 0     TMA producer: Q block once per segment, then K and V tiles
//              (64-column boxes, 128-byte swizzle) into a 3-stage
//              ring, completing on mbarriers.  Each K/V byte is read from
//              HBM once and serves all r query heads.
//   warp 1     allocates tensor memory; one lane issues the S products as
//              soon as a tile's K has landed, so the softmax of tile n
//              overlaps the V product of tile n-1.
//   warp 2     one lane issues the O products as soon as a tile's P is
//              ready, independently of warp 1 (a stage is freed for the
//              next copy without waiting for the following tile's K).
//              S and O are double-buffered in TMEM.
//   warps 3-6  softmax and correction (128 threads; a second warpgroup,
//              warps 7-10, for 32 query rows): thread x owns TMEM lane
//              x, i.e. position x of the tile for S and output column x for
//              O.  Per tile: load S, mask p >= L_i, per-head max across the
//              128 positions (redux.sync.max.f32 + one shared-memory
//              exchange), exp2, write P in the MMA's MN-major swizzled
//              layout, then fold the previous tile's O into fp32 registers
//              with its rescale factor.  Segment end: sum the per-thread
//              softmax denominators and write the output; a unit split
//              across CTAs writes a partial instead, and the CTA that
//              finishes the unit last merges the partials (log-sum-exp).
//
// Rows >= L_i of the last tile of a unit are masked out of S, and their V
// rows are zeroed in shared memory before the O product reads them, so
// whatever the cache holds there never reaches the result.  The causal mask
// of the new tokens touches only the tiles holding rows >= L_i - n.
//
// With k_new / v_new given, the KV append of the step is fused in: the CTA
// that owns a tile holding one of the rows L_i - n .. L_i - 1 puts the new
// tokens' K and V into those rows of its staged tile and writes them to the
// cache, so one launch does append + attention.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <atomic>

#include "gqa_device.cuh"
#include "gqa_internal.h"

namespace gqa {
namespace {

constexpr int kT = 128;       // positions per tile (MMA M of the S product)
constexpr int kStages = 3;    // K/V ring depth (DEEP: ring slots, three or four)
constexpr int kBoxBytes = kT * 64 * 2;  // one [128 rows x 64 cols] bf16 box
// early streaming: a CTA copies kEarlyTiles tiles into its ring before the
// dependency wait and asks L2 for the next kPrefetchTiles.  Fewer copies in
// flight let the q copy after the wait land sooner, and the tiles that
// follow come from L2.  Measured against three copied tiles (and L2 asked
// for three more only on launches that merge in place): long-context MQA
// 85.6 -> 83.4-83.7 us per call, the b = 16 sweep at g = 4 27.0 -> 25.5-26.0,
// g = 8 43.5 -> 42.6-43.5, g = 1 15.4 -> 15.1-15.3; the Llama-3-70B shape
// the same (153.0), the Qwen-shaped batch 343 -> 344.  (Two copied tiles, no
// copied tile, or five asked of L2 were slower on the small calls.)
// Launches that merge in place, on segments of 32 tiles or more, ask L2 for
// kPrefetchLong instead (same box, twice: Llama-3-70B shape 151.7 -> 150.3
// us per call, Qwen-shaped batch 340.6 -> 338.8, g = 8 sweep point 42.4 ->
// 41.6; long-context MQA, merged by the combine kernel, and the 16-tile
// segments of the g = 4 point were slower with it).
constexpr int kEarlyTiles = 1;
constexpr int kPrefetchTiles = 3;
constexpr int kPrefetchLong = 5;
// steady state with d_k = d_v = 64 (half-size tiles, the ring holds half
// the bytes): when tile t's copies are issued, L2 is asked for tile
// t + kL2Ahead of the same segment, so a copy that a freed stage starts
// later finds its bytes in L2.  (With 128-wide heads HBM is already busy
// and the extra requests made every measured shape slower.)
constexpr int kL2Ahead = 3;

// Sum each of 16 values across the warp: each round trades half of the
// values still held with the partner lane x ^ o (o = 16, 8, 4, 2) and adds,
// then lanes x and x ^ 1 add their single values.  Lane x returns the warp
// total of value (x >> 1) & 15.
__device__ __forceinline__ float warp_sum16_scatter(const float (&in)[16], int lane) {
  float v[16];
#pragma unroll
  for (int k = 0; k < 16; ++k) v[k] = in[k];
#pragma unroll
  for (int o = 16, nv = 16; o >= 2; o >>= 1, nv >>= 1) {
    const bool up = (lane & o) != 0;
#pragma unroll
    for (int k = 0; k < nv / 2; ++k) {
      const float send = up ? v[k] : v[k + nv / 2];
      const float keep = up ? v[k + nv / 2] : v[k];
      v[k] = keep + __shfl_xor_sync(0xffffffffu, send, o);
    }
  }
  return v[0] + __shfl_xor_sync(0xffffffffu, v[0], 1);
}

// d_k = d_v = 64 takes tiles of 256 positions
bool wide_tiles(int d_k, int d_v) { return d_k == 64 && d_v == 64; }
// head dims above 128 take the DEEP variant: d_k in {128, 192, 256}, d_v in
// {128, 192, 256}, not both 128
bool deep_dims(int d_k, int d_v) {
  const bool k = d_k == 128 || d_k == 192 || d_k == 256;
  const bool v = d_v == 128 || d_v == 192 || d_v == 256;
  return k && v && (d_k > 128 || d_v > 128);
}

// MULTI: n > 1 new tokens per sequence (causal mask, several new rows).
// The one-token kernel keeps the lighter code (no mask table, one new row)
// because the 32-column variant runs at its register limit.
// WIDE: d_k = d_v = 64 with tiles of 256 positions: a stage holds K rows
// 0-255 (two [128 x 64] boxes, one after the other) then V rows 0-255, the
// bytes of a 128-wide tile, so each pass of the per-tile loop moves as much
// as with 128-wide heads.  S is two M = 128 products (positions 0-127 and
// 128-255), each softmax thread owns two positions, and O runs over 256
// positions.  P is written over the stage's K rows, which the S products
// no longer need, so no P buffers are kept.
// DEEP: head dims above 128 (d_k, d_v up to 256; 16 query rows): a tile's K
// rows [128 x d_k] and V rows [128 x d_v] are separate chunks of up to four
// boxes, each in its own ring slot (chunk 2n: K of tile n, chunk 2n + 1: its
// V; slot = chunk % 3), so a slot is freed by the product that read it; S
// runs over d_k / 16 steps, and O is two M = 128 products (output columns
// 0-127 and 128-255) with d_v > 128.  In three 64 KiB slots a slot holds K
// and V chunks by turns, so it has a full barrier for each (B_FULL_K /
// B_FULL_V of the slot), each waited on by one consumer, phase c / 6 for
// chunk c: a barrier shared by the two consumers would let one of them,
// waiting for the phase after the other's, take the older completed phase
// of the same parity.  When a K chunk is at most three boxes and a V chunk
// two (d_k = 192, d_v = 128) the ring is four 48 KiB slots instead: K
// chunks in slots 0 and 2, V chunks in 1 and 3, phase c / 4.
template <int NP, int NWG, bool MULTI, bool PAGED = false, bool BF16 = true, bool WIDE = false,
          int DEEP = 0>
struct TcCfg {
  static constexpr int THREADS = 96 + 128 * NWG;  // producer, 2 MMA issuers, NWG softmax warpgroups
  static constexpr int TT = WIDE ? 2 * kT : kT;   // positions per tile
  // K half 0/1, V half 0/1 (WIDE: K rows, V rows; DEEP: one slot of the ring
  // holds a K or a V chunk of up to four boxes)
  static constexpr int KV_BYTES = 4 * kBoxBytes;
  static constexpr int QB = DEEP ? 4 : 2;          // [NP x 64] boxes of q
  static constexpr int Q_BYTES = NP * 128 * QB;
  // O accumulators of 128 output columns (the four-slot ring has d_v <= 128)
  static constexpr int OH = DEEP == 3 ? 2 : 1;
  static constexpr int P_BYTES = WIDE ? 0 : kT * NP * 2;  // [T rows x NP] bf16 (WIDE: in the stage)
  static constexpr int OFF_Q = kStages * KV_BYTES;
  static constexpr int OFF_P = OFF_Q + 2 * Q_BYTES;
  // (WIDE: the O products' unused upper M half reads up to one box past the
  // last stage's V rows; the region after the ring is at least that long)
  static constexpr int OFF_RED_MIN = WIDE ? OFF_Q + kBoxBytes : 0;
  static constexpr int OFF_RED = (OFF_P + 2 * P_BYTES) > OFF_RED_MIN ? (OFF_P + 2 * P_BYTES)
                                                                     : OFF_RED_MIN;  // float [2][NP][4] warp maxima
  static constexpr int OFF_MAX = OFF_RED + 2 * 4 * NP * 4;   // float [2][NP] running max
  static constexpr int OFF_ALPHA = OFF_MAX + 2 * NP * 4;     // float [2][NP] rescale factors
  static constexpr int OFF_COL = OFF_ALPHA + 2 * NP * 4;     // int [NP] token, int [NP] out row
  static constexpr int OFF_BAR = OFF_COL + 2 * NP * 4;
  static constexpr int RS = DEEP == 4 ? 4 : kStages;  // ring slots
  static constexpr int NBAR = 3 * RS + 2 * 7 + 1;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  // The dynamic shared-memory base is 1024-byte aligned (the swizzled
  // layouts need it; the kernel checks), so no slack is requested: leaving
  // room on the SM lets small kernels (the combine) run beside a decode CTA.
  // OFF_MISC: TMEM address, abort flag, two split flags, then (ragged
  // cluster launches) the CTA's split units [2][u, first CTA, last CTA, last]
  static constexpr int SMEM = OFF_MISC + 48;
  // S0 S1 O0 O1 (WIDE: S0a S0b S1a S1b O0 O1; DEEP: S0 S1 O0a O0b O1a O1b),
  // a power of two
  static constexpr int NCOLS = WIDE ? (NP == 16 ? 128 : 256) : (DEEP ? 128 : 4 * NP);
  static constexpr int OFF_TO = WIDE ? 4 * NP : 2 * NP;  // first O column in TMEM
  // P rows are NP * 2 bytes: 32 B (NP=16) or 64 B (NP=32) swizzle atoms
  static constexpr uint32_t P_SWZ = (NP == 16) ? SWZ_32B : SWZ_64B;
  static constexpr uint32_t IDESC = idesc_bf16(128, NP, 0, 0, BF16);    // S: K-major A, B
  static constexpr uint32_t IDESC_O = idesc_bf16(128, NP, 1, 1, BF16);  // O: MN-major A, B
  // new-row chunks an MMA-issuing warp carries in registers per lane for the
  // fused append (one token: K only, d_k / 8 lanes; n tokens: up to 4 rows
  // of K in warp 1 and of V in warp 2); further rows are loaded when patched
  static constexpr int KCH = MULTI ? 2 : 1;
  static_assert(SMEM <= 232448, "shared memory budget");
  static_assert(NCOLS == 64 || NCOLS == 128 || NCOLS == 256,
                "TMEM allocation must be a power of two");
  static_assert(NCOLS >= OFF_TO + 2 * OH * NP, "TMEM columns");
  static_assert(!DEEP || (NP == 16 && NWG == 1 && !WIDE), "DEEP: 16 query rows, 128 positions");
  static_assert(NP % NWG == 0 && (NP / NWG) % 16 == 0, "16 heads or more per warpgroup");
};

// barrier slots, for a ring of RS slots: full (K and V kinds) and empty per
// slot, then the q, S, P and O double buffers and the drain barrier
template <int RS>
struct Bars {
  static constexpr int FULL_K = 0, FULL_V = RS, EMPTY = 2 * RS, Q_FULL = 3 * RS,
                       Q_EMPTY = Q_FULL + 2, S_FULL = Q_EMPTY + 2, S_FREE = S_FULL + 2,
                       P_READY = S_FREE + 2, O_FULL = P_READY + 2, O_FREE = O_FULL + 2,
                       DRAIN = O_FREE + 2;
};

template <int NP, int NWG, bool MULTI, bool PAGED, typename T16, bool WIDE, int DEEP>
// (register cap: 11 warps put 3 on a sub-partition, 3 x 32 x 168 of its
// 16384 registers; 7 warps put 2, so 200 fit)
__global__ void __maxnreg__(NWG == 2 ? 168 : 200)
    decode_tc_kernel(const __grid_constant__ CUtensorMap tm_q,
                     const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v, const int* __restrict__ lens,
                     int b, int h, int g, int cap, float scale_log2,
                     T16* __restrict__ out, float* __restrict__ part_o,
                     float* __restrict__ part_ml, int* __restrict__ counters,
                     const uint4* __restrict__ k_new, const uint4* __restrict__ v_new,
                     uint4* __restrict__ k_cache_w, uint4* __restrict__ v_cache_w,
                     unsigned int* status, long long budget, int early, int nq,
                     const int* __restrict__ table, int bsz, int max_blocks, int num_blocks,
                     int kh, int vh, int cl_size, int cl_k) {
  using C = TcCfg<NP, NWG, MULTI, PAGED, Half16<T16>::kBf16, WIDE, DEEP>;
  using Bs = Bars<C::RS>;
  constexpr int B_FULL_K = Bs::FULL_K, B_FULL_V = Bs::FULL_V, B_EMPTY = Bs::EMPTY,
                B_Q_FULL = Bs::Q_FULL, B_Q_EMPTY = Bs::Q_EMPTY, B_S_FULL = Bs::S_FULL,
                B_S_FREE = Bs::S_FREE, B_P_READY = Bs::P_READY, B_O_FULL = Bs::O_FULL,
                B_O_FREE = Bs::O_FREE, B_DRAIN = Bs::DRAIN;
  constexpr int TT = C::TT;  // positions per tile
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* sm = smem_raw;
  const uint32_t s_base = smem_u32(sm);
  if (s_base & 1023u) {  // never seen; the layout would not fit the allocation
    // (the same in every CTA, so no CTA of a cluster is left at a cluster
    // barrier: all of them return here)
    if (threadIdx.x == 0) atomicOr(status, GQA_DEV_INTERNAL);
    return;
  }
  float* red = reinterpret_cast<float*>(sm + C::OFF_RED);  // [NWG][2][HP][4]
  float* max_sm = reinterpret_cast<float*>(sm + C::OFF_MAX);
  float* alpha_sm = reinterpret_cast<float*>(sm + C::OFF_ALPHA);
  const uint32_t bar0 = s_base + C::OFF_BAR;
  auto BAR = [&](int k) -> uint32_t { return bar0 + 8u * k; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + C::OFF_MISC + 4);
  int* last_flag = reinterpret_cast<int*>(sm + C::OFF_MISC + 8);
  int* split_list = reinterpret_cast<int*>(sm + C::OFF_MISC + 16);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = h / g;
  const int nr = nq * r;  // query rows (columns) per KV head
  // head dims d_k = 64 * kh and d_v = 64 * vh: kh / vh 64-column boxes of K
  // (and q) and of V (1 or 2; DEEP: 2 to 4); a new row is cpk / cpv chunks
  // of 16 bytes
  const int cpk = kh * 8, cpv = vh * 8;
  // DEEP ring: ns slots of sb bytes, chunk c in slot c % ns, its full
  // barrier's phase c / pd (pd = lcm(ns, 2))
  constexpr int ns = C::RS;
  constexpr uint32_t sb = DEEP == 4 ? 3u * kBoxBytes : static_cast<uint32_t>(C::KV_BYTES);
  constexpr uint32_t pd = (ns % 2 == 0) ? ns : 2 * ns;
  const int dv = vh * 64;
  // column c = s * r + t is head t of new token s; padded columns never see
  // a position
  int* col_tok = reinterpret_cast<int*>(sm + C::OFF_COL);
  int* col_off = col_tok + NP;  // element offset of column c's output row

  if (threadIdx.x >= 64 && threadIdx.x < 64 + NP) {
    const int c = threadIdx.x - 64;
    const int s = c / r;
    col_tok[c] = c < nr ? s : -(1 << 24);
    col_off[c] = c < nr ? (s * h + (c - s * r)) * dv : 0;
  }
  if (threadIdx.x == 0) {
    for (int k = 0; k < C::NBAR; ++k) {
      uint32_t cnt = 1;
      if ((k >= B_S_FREE && k < B_S_FREE + 2) || (k >= B_P_READY && k < B_P_READY + 2) ||
          (k >= B_O_FREE && k < B_O_FREE + 2))
        cnt = 4 * NWG;  // one arrival per softmax warp
      if (k == B_DRAIN) cnt = 2;  // one per MMA issuer
      mbar_init(BAR(k), cnt);
    }
    *abort_flag = 0;
    split_list[0] = split_list[4] = -1;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tm_q);
    prefetch_tmap(&tm_k);
    prefetch_tmap(&tm_v);
  }
  if (warp == 1) tmem_alloc(smem_u32(tmem_slot), C::NCOLS);
  __syncthreads();  // barrier inits and the TMEM address (this CTA's own state)
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // Programmatic dependent launch: every thread waits for the previous
  // kernel of the stream before touching memory it may write.  With `early`
  // set, the caller guarantees that no kernel still running writes seq_lens
  // or the cache rows below L_i - 1 (e.g. it is another layer's step), so
  // the producer plans and streams its first tiles before the wait, and
  // waits before loading q; the other warps wait at once.
  if (!early || warp != 0) pdl_wait_then_release();
  if (warp == 2 && blockIdx.x == 0) report_bad_lengths(lens, b, nq, cap, status);

  Walker w;
  // (two whole units per CTA only with 128-wide heads or wide tiles, none
  // on a paged cache, whose per-block copies need every SM: see
  // Walker::init)
  w.init(lens, b, g, nq, cap, TT, blockIdx.x, gridDim.x,
         PAGED ? 0 : ((WIDE || DEEP || (kh == 2 && vh == 2)) ? 2 : 1));
  Segment seg;
  // Cluster merge: the launch is a cluster launch of cl_size CTAs, cl_k
  // clusters per unit (grid = units * cl_size * cl_k), and every unit has
  // the same number of tiles, so each CTA's range lies in unit
  // blockIdx.x / (cl_size * cl_k).  Each CTA leaves its partial (max, sum,
  // unnormalised output of every query row) in its own shared memory, and
  // after a cluster barrier the cluster's CTAs merge them over distributed
  // shared memory, each a slice of the unit's outputs.  (Uniform across the
  // grid; with ragged lengths a cluster launch takes the global-memory
  // merge below.)
  const bool cl_merge = cl_size > 1 && w.equal;

  if (warp == 0 && PAGED) {
    // ===================== TMA producer, paged cache =====================
    // The whole warp walks the tiles (block-table lookups are spread over
    // its lanes); lane 0 issues the copies.  A tile of 128 positions is one
    // box per 64-column half when blocks hold 128 rows or more, else one box
    // per block.  Blocks past L_i, and bad entries, are read out of range
    // (zero fill).
    const uint64_t pol_stream = policy_evict_first();
    const uint64_t pol_keep = policy_evict_last();
    const int oob_row = num_blocks * g * bsz;
    const int box_rows = bsz < kT ? bsz : kT;
    const int sub = TT / box_rows;  // boxes per tile and 64-column half
    uint32_t n = 0, k = 0;
    int last_n[ns];
#pragma unroll
    for (int s2 = 0; s2 < ns; ++s2) last_n[s2] = -1;
    int last_q[2] = {-1, -1};
    auto load_q = [&](uint32_t kk, const Segment& sg) {
      const uint32_t qs = kk & 1;
      const bool ok = __all_sync(0xffffffffu, mbar_wait(BAR(B_Q_EMPTY + qs), ((kk >> 1) & 1) ^ 1,
                                                        abort_flag, status, budget));
      if (ok && lane == 0) {
        const uint32_t qdst = s_base + C::OFF_Q + qs * C::Q_BYTES;
        mbar_arrive_expect_tx(BAR(B_Q_FULL + qs), nr * 128 * kh);
        for (int qb = 0; qb < kh; ++qb)
          tma_load_3d(qdst + qb * NP * 128, &tm_q, BAR(B_Q_FULL + qs), 64 * qb, sg.j * r,
                      sg.i * nq, pol_keep);
      }
      if (ok) last_q[qs] = static_cast<int>(kk);
    };
    bool waited = !early;
    PageCursor pc;
    while (w.next(seg)) {
      if (waited) {
        load_q(k, seg);
      } else if (lane == 0) {  // (as in the contiguous producer below)
        for (int qb = 0; qb < kh; ++qb) tma_prefetch_l2_3d(&tm_q, 64 * qb, seg.j * r, seg.i * nq);
      }
      pc.start(table + static_cast<size_t>(seg.i) * max_blocks, (seg.L + bsz - 1) / bsz,
               (seg.lt0 * TT) / bsz);
      for (int lt = seg.lt0; lt < seg.lt1; ++lt, ++n) {
        if (!waited && (lt - seg.lt0 == kStages)) {
          pdl_wait_then_release();
          waited = true;
          load_q(k, seg);
        }
        if constexpr (DEEP) {
          // as in the contiguous producer: K chunk 2n, then V chunk 2n + 1,
          // each into its slot; lane mm < sub copies the rows of box mm of
          // every 64-column box of the chunk
          const uint32_t ck = 2 * n, cv = 2 * n + 1;
          const int sk = ck % ns, sv = cv % ns;
          const int p_first = lt * TT;
          const int blk_l = pc.get_lanes(p_first / bsz);
          const int blk = (box_rows == bsz) ? blk_l : __shfl_sync(0xffffffffu, blk_l, 0);
          const int pm = p_first + lane * box_rows;
          bool bad = false;
          int row = oob_row;
          if (lane < sub && pm < seg.L) {
            if (blk >= 0 && blk < num_blocks)
              row = (blk * g + seg.j) * bsz + pm % bsz;
            else
              bad = true;
          }
          const uint32_t o = lane * box_rows * 128;
          if (DEEP == 4 && !waited && lt - seg.lt0 == 2) {
            pdl_wait_then_release();
            waited = true;
            load_q(k, seg);
          }
          if (!__all_sync(0xffffffffu, mbar_wait(BAR(B_EMPTY + sk), ((ck / ns) & 1) ^ 1,
                                                 abort_flag, status, budget)))
            continue;
          if (lane == 0) mbar_arrive_expect_tx(BAR(B_FULL_K + sk), kh * kBoxBytes);
          __syncwarp();
          if (lane < sub)
            for (int bx = 0; bx < kh; ++bx)
              tma_load_2d(s_base + sk * sb + bx * kBoxBytes + o, &tm_k, BAR(B_FULL_K + sk),
                          64 * bx, row, pol_stream);
          last_n[sk] = static_cast<int>(ck);  // (DEEP: chunk numbers)
          if (DEEP == 3 && !waited && lt - seg.lt0 == 1) {
            pdl_wait_then_release();
            waited = true;
            load_q(k, seg);
          }
          if (!__all_sync(0xffffffffu, mbar_wait(BAR(B_EMPTY + sv), ((cv / ns) & 1) ^ 1,
                                                 abort_flag, status, budget)))
            continue;
          if (lane == 0) mbar_arrive_expect_tx(BAR(B_FULL_V + sv), vh * kBoxBytes);
          __syncwarp();
          if (lane < sub)
            for (int bx = 0; bx < vh; ++bx)
              tma_load_2d(s_base + sv * sb + bx * kBoxBytes + o, &tm_v, BAR(B_FULL_V + sv),
                          64 * bx, row, pol_stream);
          last_n[sv] = static_cast<int>(cv);
          if (__any_sync(0xffffffffu, bad) && lane == 0) atomicOr(status, GQA_DEV_BAD_BLOCK);
          continue;
        }
        const int st = n % kStages;
        const bool ok = __all_sync(0xffffffffu,
                                   mbar_wait(BAR(B_EMPTY + st), ((n / kStages) & 1) ^ 1,
                                             abort_flag, status, budget));
        if (!ok) continue;
        const uint32_t dst = s_base + st * C::KV_BYTES;
        if (lane == 0) {
          mbar_arrive_expect_tx(BAR(B_FULL_K + st), kh * kBoxBytes * (TT / kT));
          mbar_arrive_expect_tx(BAR(B_FULL_V + st), vh * kBoxBytes * (TT / kT));
        }
        __syncwarp();
        // lane mm < sub copies box mm of the tile (its block's rows; blocks
        // longer than a box hold every box of the tile)
        const int p_first = lt * TT;
        const int blk_l = pc.get_lanes(p_first / bsz);
        const int blk = (box_rows == bsz) ? blk_l : __shfl_sync(0xffffffffu, blk_l, 0);
        const int pm = p_first + lane * box_rows;
        bool bad = false;
        if (lane < sub) {
          int row = oob_row;
          if (pm < seg.L) {
            if (blk >= 0 && blk < num_blocks)
              row = (blk * g + seg.j) * bsz + pm % bsz;
            else
              bad = true;
          }
          const uint32_t o = lane * box_rows * 128;
          tma_load_2d(dst + o, &tm_k, BAR(B_FULL_K + st), 0, row, pol_stream);
          if (kh == 2)
            tma_load_2d(dst + kBoxBytes + o, &tm_k, BAR(B_FULL_K + st), 64, row, pol_stream);
          tma_load_2d(dst + 2 * kBoxBytes + o, &tm_v, BAR(B_FULL_V + st), 0, row, pol_stream);
          if (vh == 2)
            tma_load_2d(dst + 3 * kBoxBytes + o, &tm_v, BAR(B_FULL_V + st), 64, row, pol_stream);
        }
        if (__any_sync(0xffffffffu, bad) && lane == 0) atomicOr(status, GQA_DEV_BAD_BLOCK);
        last_n[st] = static_cast<int>(n);
      }
      if (!waited) {
        pdl_wait_then_release();
        waited = true;
        load_q(k, seg);
      }
      ++k;
    }
    if (!waited) pdl_wait_then_release();
    if (*abort_flag && lane == 0) {
      for (int s = 0; s < ns + 2; ++s) {
        int idx;
        uint32_t b0, b1 = 0;
        bool two = false;
        if (s < ns) {
          idx = last_n[s];
          if (idx < 0) continue;
          b0 = BAR(B_FULL_K + s);
          b1 = BAR(B_FULL_V + s);
          two = !DEEP;
          if (DEEP) {  // the slot's last chunk: K (even) or V (odd), phase c / pd
            if (idx & 1) b0 = BAR(B_FULL_V + s);
            idx /= static_cast<int>(pd);
          } else {
            idx /= kStages;
          }
        } else {
          idx = last_q[s - ns];
          if (idx < 0) continue;
          b0 = BAR(B_Q_FULL + s - ns);
          idx >>= 1;
        }
        const long long t0 = clock64();
        while (!mbar_try_wait(b0, idx & 1) && clock64() - t0 < budget) {
        }
        while (two && !mbar_try_wait(b1, idx & 1) && clock64() - t0 < budget) {
        }
      }
    }
    __syncwarp();
  } else if (warp == 0) {
    // =========================== TMA producer ===========================
    if (lane == 0) {
      const uint64_t pol_stream = policy_evict_first();
      const uint64_t pol_keep = policy_evict_last();
      uint32_t n = 0, k = 0;
      int last_n[ns];
#pragma unroll
      for (int s2 = 0; s2 < ns; ++s2) last_n[s2] = -1;
      int last_q[2] = {-1, -1};
      auto load_q = [&](uint32_t kk, const Segment& sg) {
        const uint32_t qs = kk & 1;
        if (mbar_wait(BAR(B_Q_EMPTY + qs), ((kk >> 1) & 1) ^ 1, abort_flag, status, budget)) {
          const uint32_t qdst = s_base + C::OFF_Q + qs * C::Q_BYTES;
          // box [n tokens][r heads][64]: rows s * r + t of the operand
          mbar_arrive_expect_tx(BAR(B_Q_FULL + qs), nr * 128 * kh);
          for (int qb = 0; qb < kh; ++qb)
            tma_load_3d(qdst + qb * NP * 128, &tm_q, BAR(B_Q_FULL + qs), 64 * qb, sg.j * r,
                        sg.i * nq, pol_keep);
          last_q[qs] = static_cast<int>(kk);
        }
      };
      bool waited = !early;  // has this thread passed the dependency wait?
      while (w.next(seg)) {
        // q comes from the previous kernel: load it only after the wait
        // (early mode: after the first kEarlyTiles K/V tiles).  Before
        // the wait L2 is asked for it, ahead of the K/V copies: that moves
        // no data into this CTA, and a write by the kernel ahead lands in
        // L2 all the same, where the load after the wait finds it.
        if (waited) {
          load_q(k, seg);
        } else {
          for (int qb = 0; qb < kh; ++qb)
            tma_prefetch_l2_3d(&tm_q, 64 * qb, seg.j * r, seg.i * nq);
        }
        const int unit_row = (seg.i * g + seg.j) * cap;
        for (int lt = seg.lt0; lt < seg.lt1; ++lt, ++n) {
          if (!waited && (lt - seg.lt0 == (DEEP ? kStages : kEarlyTiles))) {
            // have L2 fetch the next tiles, so HBM stays busy until the kernel
            // ahead completes (DEEP waits inside its branch below)
            const int npf =
                (counters != nullptr && seg.lt1 - seg.lt0 >= 32) ? kPrefetchLong : kPrefetchTiles;
            for (int lp = lt; lp < seg.lt1 && lp < lt + (DEEP ? 0 : npf); ++lp) {
              const int rp = unit_row + lp * TT;
              for (int bx = 0; bx < kh; ++bx) tma_prefetch_l2_2d(&tm_k, 64 * bx, rp);
              if (WIDE) tma_prefetch_l2_2d(&tm_k, 0, rp + kT);
              for (int bx = 0; bx < vh; ++bx) tma_prefetch_l2_2d(&tm_v, 64 * bx, rp);
              if (WIDE) tma_prefetch_l2_2d(&tm_v, 0, rp + kT);
            }
            pdl_wait_then_release();
            waited = true;
            load_q(k, seg);
          }
          if constexpr (DEEP) {
            // K chunk 2n, then V chunk 2n + 1, each into the slot its chunk
            // number gives.  Chunk ns needs slot 0 back, i.e. tile 0's S
            // product, i.e. q: early streaming stops before it.
            const int row = unit_row + lt * TT;
            const uint32_t ck = 2 * n, cv = 2 * n + 1;
            const int sk = ck % ns, sv = cv % ns;
            // (four slots: chunk 4 is tile 2's K; three slots: chunk 3 is
            // tile 1's V)
            if (DEEP == 4 && !waited && lt - seg.lt0 == 2) {
              pdl_wait_then_release();
              waited = true;
              load_q(k, seg);
            }
            if (!mbar_wait(BAR(B_EMPTY + sk), ((ck / ns) & 1) ^ 1, abort_flag, status, budget))
              continue;
            mbar_arrive_expect_tx(BAR(B_FULL_K + sk), kh * kBoxBytes);
            for (int bx = 0; bx < kh; ++bx)
              tma_load_2d(s_base + sk * sb + bx * kBoxBytes, &tm_k, BAR(B_FULL_K + sk), 64 * bx,
                          row, pol_stream);
            last_n[sk] = static_cast<int>(ck);  // (DEEP: chunk numbers)
            if (DEEP == 3 && !waited && lt - seg.lt0 == 1) {
              pdl_wait_then_release();
              waited = true;
              load_q(k, seg);
            }
            if (!mbar_wait(BAR(B_EMPTY + sv), ((cv / ns) & 1) ^ 1, abort_flag, status, budget))
              continue;
            mbar_arrive_expect_tx(BAR(B_FULL_V + sv), vh * kBoxBytes);
            for (int bx = 0; bx < vh; ++bx)
              tma_load_2d(s_base + sv * sb + bx * kBoxBytes, &tm_v, BAR(B_FULL_V + sv), 64 * bx,
                          row, pol_stream);
            last_n[sv] = static_cast<int>(cv);
            continue;
          }
          const int st = n % kStages;
          if (!mbar_wait(BAR(B_EMPTY + st), ((n / kStages) & 1) ^ 1, abort_flag, status,
                         budget))
            continue;
          const int row = unit_row + lt * TT;
          const uint32_t dst = s_base + st * C::KV_BYTES;
          // (WIDE: the second box of each tensor is rows 128-255, not
          // columns 64-127)
          mbar_arrive_expect_tx(BAR(B_FULL_K + st), kh * kBoxBytes * (TT / kT));
          tma_load_2d(dst, &tm_k, BAR(B_FULL_K + st), 0, row, pol_stream);
          if (WIDE)
            tma_load_2d(dst + kBoxBytes, &tm_k, BAR(B_FULL_K + st), 0, row + kT, pol_stream);
          else if (kh == 2)
            tma_load_2d(dst + kBoxBytes, &tm_k, BAR(B_FULL_K + st), 64, row, pol_stream);
          mbar_arrive_expect_tx(BAR(B_FULL_V + st), vh * kBoxBytes * (TT / kT));
          tma_load_2d(dst + 2 * kBoxBytes, &tm_v, BAR(B_FULL_V + st), 0, row, pol_stream);
          if (WIDE)
            tma_load_2d(dst + 3 * kBoxBytes, &tm_v, BAR(B_FULL_V + st), 0, row + kT, pol_stream);
          else if (vh == 2)
            tma_load_2d(dst + 3 * kBoxBytes, &tm_v, BAR(B_FULL_V + st), 64, row, pol_stream);
          last_n[st] = static_cast<int>(n);
          if (!WIDE && kh + vh == 2 && waited && lt + kL2Ahead < seg.lt1) {
            const int rp = row + kL2Ahead * kT;
            tma_prefetch_l2_2d(&tm_k, 0, rp);
            if (kh == 2) tma_prefetch_l2_2d(&tm_k, 64, rp);
            tma_prefetch_l2_2d(&tm_v, 0, rp);
            if (vh == 2) tma_prefetch_l2_2d(&tm_v, 64, rp);
          }
        }
        if (!waited) {  // a first segment of kEarlyTiles tiles or fewer
          pdl_wait_then_release();
          waited = true;
          load_q(k, seg);
        }
        ++k;
      }
      if (!waited) pdl_wait_then_release();  // a CTA with no tiles
      if (*abort_flag) {  // copies in flight must land before the CTA exits
        for (int s = 0; s < ns + 2; ++s) {
          int idx;
          uint32_t b0, b1 = 0;
          bool two = false;
          if (s < ns) {
            idx = last_n[s];
            if (idx < 0) continue;
            b0 = BAR(B_FULL_K + s);
            b1 = BAR(B_FULL_V + s);
            two = !DEEP;
            if (DEEP) {  // the slot's last chunk: K (even) or V (odd), phase c / pd
              if (idx & 1) b0 = BAR(B_FULL_V + s);
              idx /= static_cast<int>(pd);
            } else {
              idx /= kStages;
            }
          } else {
            idx = last_q[s - ns];
            if (idx < 0) continue;
            b0 = BAR(B_Q_FULL + s - ns);
            idx >>= 1;
          }
          const long long t0 = clock64();
          while (!mbar_try_wait(b0, idx & 1) && clock64() - t0 < budget) {
          }
          while (two && !mbar_try_wait(b1, idx & 1) && clock64() - t0 < budget) {
          }
        }
      }
    }
    __syncwarp();
  } else if (warp == 1 || warp == 2) {
    // ============================ MMA issuers ===========================
    // Lane 0 of warp 1 issues the S products, lane 0 of warp 2 the O
    // products: each waits only for its own operands, so a tile's O product
    // (which frees its stage for the next copy) never queues behind the next
    // tile's K.  With the append fused in, warp 1 also carries the new
    // tokens' K rows that fall in the segment (16-byte chunks, loaded at the
    // segment start) to their tiles, where it patches them into the staged
    // tile and writes them to the cache; with n tokens warp 2 does the same
    // for V before the tile's O product.
    const bool s_role = warp == 1;
    const bool leader = lane == 0;
    const uint32_t tS = tmem, tO = tmem + C::OFF_TO;
    constexpr int NH = WIDE ? 2 : 1;  // S products (128-position halves) per tile
    // operand descriptors: a stage, a buffer or a k-step only moves the
    // start-address field (16-byte units, no carry out of it)
    // (DEEP: tile m's V is chunk 2m + 1, in slot (2m + 1) % 3 from its
    // first box)
    auto v_slot = [&](uint32_t m) -> int { return DEEP ? (2 * m + 1) % ns : m % kStages; };
    auto v_full = [&](uint32_t m) -> uint32_t { return BAR(B_FULL_V + v_slot(m)); };
    auto v_phase = [&](uint32_t m) -> uint32_t {
      return DEEP ? ((2 * m + 1) / pd) & 1 : (m / kStages) & 1;
    };
    auto v_base = [&](uint32_t m) -> uint32_t {
      return s_base + v_slot(m) * (DEEP ? sb : C::KV_BYTES) + (DEEP ? 0 : 2 * kBoxBytes);
    };
    auto issue_o = [&](uint32_t m) {
      const int st = v_slot(m);
      const uint32_t nb = m & 1;
      bool ok = mbar_wait(BAR(B_P_READY + nb), (m >> 1) & 1, abort_flag, status, budget);
      ok = ok && mbar_wait(v_full(m), v_phase(m), abort_flag, status, budget);
      ok = ok && mbar_wait(BAR(B_O_FREE + nb), ((m >> 1) & 1) ^ 1, abort_flag, status, budget);
      ok = __all_sync(0xffffffffu, ok);
      tc_fence_after();
      if (leader) {
        if (ok) {
          const uint64_t a0 = smem_desc(v_base(m), kBoxBytes, 1024, SWZ_128B);
          // (WIDE: P lies over the stage's K rows)
          const uint32_t pbase =
              WIDE ? s_base + st * C::KV_BYTES : s_base + C::OFF_P + nb * C::P_BYTES;
          const uint64_t b0 = smem_desc(pbase, TT * NP * 2, 8 * NP * 2, C::P_SWZ);
#pragma unroll
          for (int kk = 0; kk < TT / 16; ++kk) {
            // A = V^T: M = 128 head-dim columns (two 64-column boxes, LBO
            // apart), K = 16 positions (two 8-row groups, SBO apart; 2 KiB
            // a step).  With d_v = 64 the second box is not loaded: output
            // rows 64-127 are never read (WIDE: the V rows continue into the
            // second box, and the upper M half reads the box after the
            // current one).  B = P^T: N = NP heads contiguous per row, K =
            // 16 position rows (16 * NP * 2 bytes a step).
            mma_bf16(tO + nb * C::OH * NP, a0 + kk * (2048 >> 4), b0 + kk * ((16 * NP * 2) >> 4),
                     C::IDESC_O, kk > 0 ? 1u : 0u);
          }
          if (DEEP && vh > 2) {
            // output columns 128-255 from V boxes 2 and 3 (with d_v = 192
            // box 3 is not loaded: rows 192-255 are never read)
#pragma unroll
            for (int kk = 0; kk < TT / 16; ++kk)
              mma_bf16(tO + (nb * C::OH + 1) * NP, a0 + ((2 * kBoxBytes) >> 4) + kk * (2048 >> 4),
                       b0 + kk * ((16 * NP * 2) >> 4), C::IDESC_O, kk > 0 ? 1u : 0u);
          }
        }
        mma_commit(BAR(B_O_FULL + nb));
        mma_commit(BAR(B_EMPTY + st));
      }
      __syncwarp();
    };
    uint32_t n = 0, k = 0;
    while (w.next(seg)) {
      const uint32_t qs = k & 1;
      const size_t unit = static_cast<size_t>(seg.i) * g + seg.j;
      // new tokens s_lo .. s_lo + nrows - 1 have their rows here
      const int first_new = seg.L - nq;
      int s_lo = 0, nrows = 0;
      if (k_new != nullptr) {
        const int p_lo = max(first_new, seg.lt0 * TT), p_hi = min(seg.L, seg.lt1 * TT);
        if (p_lo < p_hi) {
          s_lo = p_lo - first_new;
          nrows = p_hi - p_lo;
        }
      }
      const int nchunk_k = nrows * cpk, nchunk_v = nrows * cpv;
      // chunk idx of the segment's new rows (cp chunks of 16 bytes a row):
      // token s_lo + idx / cp, chunk idx % cp of its row [b, n, g, d] of
      // k_new / v_new
      auto new_off = [&](int idx, int cp) {
        return ((static_cast<size_t>(seg.i) * nq + s_lo + idx / cp) * g + seg.j) * cp + idx % cp;
      };
      // paged cache (one token): the physical row of position L_i - 1, or -1
      // for a bad table entry (then nothing is written)
      long long prow = -1;
      if (PAGED && !MULTI && nrows > 0) {
        const int blk = __ldg(table + static_cast<size_t>(seg.i) * max_blocks + (seg.L - 1) / bsz);
        if (blk >= 0 && blk < num_blocks)
          prow = (static_cast<long long>(blk) * g + seg.j) * bsz + (seg.L - 1) % bsz;
        else if (lane == 0)
          atomicOr(status, GQA_DEV_BAD_BLOCK);
      }
      // (one token: the softmax warps carry and patch the V row)
      constexpr int VCH = MULTI ? C::KCH : 1;
      // put chunk ch (value v) into row `rho` of a staged tile (64-column
      // boxes, 128-byte swizzle) and into the cache at `pos` (rows of cp
      // chunks)
      auto put = [&](uint32_t tile_base, uint4* cache, int ch, int cp, int pos, int rho,
                     const uint4& v) {
        const uint32_t dst =
            tile_base + (ch >> 3) * kBoxBytes + rho * 128 + (((ch & 7) ^ (rho & 7)) << 4);
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(dst), "r"(v.x), "r"(v.y),
                     "r"(v.z), "r"(v.w)
                     : "memory");
        if (!PAGED) {
          cache[(unit * cap + pos) * cp + ch] = v;
        } else if (!MULTI) {
          if (prow >= 0) cache[prow * cp + ch] = v;
        } else {
          // n new rows: each through its own block-table entry
          const int blk = __ldg(table + static_cast<size_t>(seg.i) * max_blocks + pos / bsz);
          if (blk >= 0 && blk < num_blocks)
            cache[((static_cast<long long>(blk) * g + seg.j) * bsz + pos % bsz) * cp + ch] = v;
          else
            atomicOr(status, GQA_DEV_BAD_BLOCK);
        }
      };
      // patch the new rows that fall in tile lt (K or V part of the stage)
      auto patch = [&](uint32_t tile_base, uint4* cache, const uint4* src, const uint4* regs,
                       int nregs, int lt, int cp) {
        const int nchunk = nrows * cp;
#pragma unroll
        for (int c4 = 0; c4 < C::KCH; ++c4) {
          if (c4 >= nregs) break;
          const int idx = lane + 32 * c4;
          const int pos = first_new + s_lo + idx / cp;
          if (idx < nchunk && pos >= lt * TT && pos < (lt + 1) * TT)
            put(tile_base, cache, idx % cp, cp, pos, pos - lt * TT, regs[c4]);
        }
        for (int idx = lane + 32 * nregs; idx < nchunk; idx += 32) {
          const int pos = first_new + s_lo + idx / cp;
          if (pos >= lt * TT && pos < (lt + 1) * TT)
            put(tile_base, cache, idx % cp, cp, pos, pos - lt * TT,
                __ldg(src + new_off(idx, cp)));
        }
        fence_proxy_async_smem();
      };
      if (!s_role) {
        // O products, in tile order
        uint4 vnew[VCH];
#pragma unroll
        for (int c4 = 0; c4 < VCH; ++c4) {
          const int idx = lane + 32 * c4;
          vnew[c4] = make_uint4(0u, 0u, 0u, 0u);
          if (MULTI && idx < nchunk_v) vnew[c4] = __ldg(v_new + new_off(idx, cpv));
        }
        for (int lt = seg.lt0; lt < seg.lt1; ++lt, ++n) {
          const bool new_rows = nrows > 0 && (lt + 1) * TT > first_new;
          if (MULTI && new_rows) {
            // the tile's new V rows, before its O product (the softmax
            // warps zero the rows past L_i, which are other rows)
            const bool vok = __all_sync(
                0xffffffffu, mbar_wait(v_full(n), v_phase(n), abort_flag, status, budget));
            if (vok) patch(v_base(n), v_cache_w, v_new, vnew, VCH, lt, cpv);
            __syncwarp();
          }
          issue_o(n);
        }
        ++k;
        continue;
      }
      uint4 knew[C::KCH];
#pragma unroll
      for (int c4 = 0; c4 < C::KCH; ++c4) {
        const int idx = lane + 32 * c4;
        knew[c4] = make_uint4(0u, 0u, 0u, 0u);
        if (idx < nchunk_k) knew[c4] = __ldg(k_new + new_off(idx, cpk));
      }
      const bool qok = __all_sync(
          0xffffffffu, mbar_wait(BAR(B_Q_FULL + qs), (k >> 1) & 1, abort_flag, status, budget));
      for (int lt = seg.lt0; lt < seg.lt1; ++lt, ++n) {
        // (DEEP: tile n's K is chunk 2n)
        const int st = DEEP ? (2 * n) % ns : n % kStages;
        const uint32_t kph = DEEP ? ((2 * n) / pd) & 1 : (n / kStages) & 1;
        const uint32_t nb = n & 1;
        bool ok = qok && mbar_wait(BAR(B_FULL_K + st), kph, abort_flag, status, budget);
        ok = ok && mbar_wait(BAR(B_S_FREE + nb), ((n >> 1) & 1) ^ 1, abort_flag, status, budget);
        ok = __all_sync(0xffffffffu, ok);
        const uint32_t kbase = s_base + st * (DEEP ? sb : C::KV_BYTES);
        const bool new_rows = nrows > 0 && (lt + 1) * TT > first_new;
        if (new_rows) {
          // rows L_i - n .. L_i - 1 of this tile are the new tokens: use
          // k_new there, and store them into the cache (the append)
          if (ok) patch(kbase, k_cache_w, k_new, knew, C::KCH, lt, cpk);
          __syncwarp();
        }
        tc_fence_after();
        if (leader) {
          if (ok) {
            const uint64_t b0 = smem_desc(s_base + C::OFF_Q + qs * C::Q_BYTES, 16, 1024, SWZ_128B);
#pragma unroll
            for (int hf = 0; hf < NH; ++hf) {
              // (WIDE: half hf = positions 128 hf .. 128 hf + 127, the
              // stage's box hf, into its own accumulator)
              const uint64_t a0 = smem_desc(kbase + hf * kBoxBytes, 16, 1024, SWZ_128B);
#pragma unroll
              for (int kk = 0; kk < (DEEP ? 16 : 8); ++kk) {
                // A = K tile, K-major: 128 rows, 16 head-dim columns (32
                // bytes) per step; steps 4b .. 4b + 3 in 64-column box b
                // (b < kh).  B = the q block, the same way ([NP x 64]
                // boxes).
                if (kk >= 4 * kh) break;
                mma_bf16(tS + (nb * NH + hf) * NP,
                         a0 + (((kk >> 2) * kBoxBytes + (kk & 3) * 32) >> 4),
                         b0 + (((kk >> 2) * (NP * 128) + (kk & 3) * 32) >> 4), C::IDESC,
                         kk > 0 ? 1u : 0u);
              }
            }
          }
          mma_commit(BAR(B_S_FULL + nb));
          if (DEEP) mma_commit(BAR(B_EMPTY + st));  // the K chunk's slot
          if (lt == seg.lt1 - 1) mma_commit(BAR(B_Q_EMPTY + qs));
        }
        __syncwarp();
      }
      ++k;
    }
    if (leader) {
      // every MMA of both issuers must be finished before tensor memory is
      // released (the drain barrier takes one arrival from each)
      mma_commit(BAR(B_DRAIN));
      const long long t0 = clock64();
      while (!mbar_try_wait(BAR(B_DRAIN), 0) && clock64() - t0 < budget) {
      }
    }
    __syncwarp();
  } else {
    // ====================== softmax / correction ========================
    // NWG warpgroups of four warps; warpgroup wg owns heads
    // [wg * HP, wg * HP + HP) and runs on its own (own exchanges, named
    // barrier 1 + wg, own split counter); the warpgroups share only the
    // staged tiles and the MMAs.
    constexpr int HP = NP / NWG;
    const int wg = (warp - 3) >> 2;   // warpgroup
    const int wq = (warp - 3) & 3;    // warp within the warpgroup
    const int qd = warp & 3;          // TMEM lane quarter this warp may access
    const int row = qd * 32 + lane;   // tile position (S) / head-dim column (O)
    const int h0 = wg * HP;           // first head of this warpgroup
    const int bar_id = 1 + wg;
    const uint32_t lane_off = static_cast<uint32_t>(qd * 32) << 16;
    const uint32_t tS = tmem + lane_off + h0, tO = tmem + C::OFF_TO + lane_off + h0;
    constexpr int NH = WIDE ? 2 : 1;  // positions per thread and tile: row (+ 128)
    float* red_wg = red + wg * 2 * HP * 4;   // [2][HP][4]
    int* last_flag_wg = last_flag + wg;

    // l[e], o[e]: this thread's softmax sum (its positions) and output column
    // for head h0 + e.  The running max of a head is uniform across the CTA:
    // thread e of the warpgroup keeps head h0 + e's (m_own) and publishes it
    // with its rescale factor through max_sm / alpha_sm each tile.
    // (DEEP: o[1] holds output column row + 128, for d_v > 128)
    constexpr int OH = C::OH;
    float l[HP], o[OH][HP];
    float m_own = -INFINITY;
#pragma unroll
    for (int e = 0; e < HP; ++e) {
      l[e] = 0.f;
#pragma unroll
      for (int hf = 0; hf < OH; ++hf) o[hf][e] = 0.f;
    }

    // fold O of tile mt into the registers: o = o * alpha + O_tile
    auto correct = [&](uint32_t mt, const float* al) {
      const uint32_t nb = mt & 1;
      const bool ok = mbar_wait(BAR(B_O_FULL + nb), (mt >> 1) & 1, abort_flag, status, budget);
      float ov[OH][HP];
#pragma unroll
      for (int hf = 0; hf < OH; ++hf) {
        if (ok && (hf == 0 || vh > 2)) {
          tmem_ld16(tO + (nb * OH + hf) * NP, ov[hf]);
        } else {
#pragma unroll
          for (int e = 0; e < HP; ++e) ov[hf][e] = 0.f;
        }
      }
      if (ok) tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(BAR(B_O_FREE + nb));
#pragma unroll
      for (int hf = 0; hf < OH; ++hf)
#pragma unroll
        for (int e = 0; e < HP; ++e) o[hf][e] = fmaf(o[hf][e], al[h0 + e], ov[hf][e]);
    };

    uint32_t n = 0;
    bool had_seg = false;
    // cluster merge: [NP][d_v] outputs and [NP][2] (max, sum) at the start of
    // the ring (free once the CTA's last O product has completed)
    float* cl_o = reinterpret_cast<float*>(sm);
    float* cl_ml = cl_o + NP * dv;
    while (w.next(seg)) {
      had_seg = true;
      const int first_new = seg.L - nq;  // position of new token 0
      // one token: threads 0 .. d_v/8 - 1 of warpgroup 0 carry the new V
      // row (one 16-byte chunk each) to the unit's last tile
      const bool append_v = !MULTI && v_new != nullptr && seg.lt1 == seg.ti;
      const int vch = cpv;
      uint4 vnew = make_uint4(0u, 0u, 0u, 0u);
      long long vrow_w = -1;  // cache row written by the append
      if (append_v && wg == 0 && row < vch) {
        vnew = __ldg(v_new + (static_cast<size_t>(seg.i) * g + seg.j) * cpv + row);
        if (!PAGED) {
          vrow_w = (static_cast<long long>(seg.i) * g + seg.j) * cap + seg.L - 1;
        } else {
          const int blk =
              __ldg(table + static_cast<size_t>(seg.i) * max_blocks + (seg.L - 1) / bsz);
          if (blk >= 0 && blk < num_blocks)
            vrow_w = (static_cast<long long>(blk) * g + seg.j) * bsz + (seg.L - 1) % bsz;
        }
      }
      for (int lt = seg.lt0; lt < seg.lt1; ++lt, ++n) {
        const uint32_t nb = n & 1;
        const int st = n % kStages;
        const int valid = min(TT, seg.L - lt * TT);
        // ---- logits from TMEM (WIDE: both 128-position halves) ----
        const bool ok = mbar_wait(BAR(B_S_FULL + nb), (n >> 1) & 1, abort_flag, status, budget);
        float x[NH][HP];
        if (ok) {
#pragma unroll
          for (int hf = 0; hf < NH; ++hf) {
#pragma unroll
            for (int c = 0; c < HP; c += 16) {
              float tmp[16];
              tmem_ld16(tS + (nb * NH + hf) * NP + c, tmp);
#pragma unroll
              for (int e = 0; e < 16; ++e) x[hf][c + e] = tmp[e];
            }
          }
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int hf = 0; hf < NH; ++hf)
#pragma unroll
            for (int e = 0; e < HP; ++e) x[hf][e] = 0.f;
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(BAR(B_S_FREE + nb));
#pragma unroll
        for (int hf = 0; hf < NH; ++hf) {
          const int pos = row + hf * kT;  // position within the tile
          const bool live = pos < valid;
          if (!MULTI) {
#pragma unroll
            for (int e = 0; e < HP; ++e)
              x[hf][e] = (live && h0 + e < nr) ? x[hf][e] * scale_log2 : -INFINITY;
          } else if ((lt + 1) * TT <= first_new + 1) {
            // (uniform) every new token sees every position of the tile
#pragma unroll
            for (int e = 0; e < HP; ++e)
              x[hf][e] = (h0 + e < nr) ? x[hf][e] * scale_log2 : -INFINITY;
          } else {
            // token s sees this position iff s >= -vis (the causal mask; for
            // n = 1 it is the p < L_i mask; padded columns see nothing)
            const int vis = first_new - lt * TT - pos;
#pragma unroll
            for (int e4 = 0; e4 < HP; e4 += 4) {
              const int4 tk = *reinterpret_cast<const int4*>(col_tok + h0 + e4);
              const int tt[4] = {tk.x, tk.y, tk.z, tk.w};
#pragma unroll
              for (int k = 0; k < 4; ++k)
                x[hf][e4 + k] = (tt[k] >= -vis) ? x[hf][e4 + k] * scale_log2 : -INFINITY;
            }
          }
        }
        // ---- per-head max over the tile's positions ----
        float mine = -INFINITY;
#pragma unroll
        for (int e = 0; e < HP; ++e) {
          const float wm = warp_max(NH == 2 ? fmaxf(x[0][e], x[NH - 1][e]) : x[0][e]);
          if (lane == e) mine = wm;
        }
        // head-major [HP][4 warps]; thread e folds head h0 + e's four warp
        // maxima into the running max, forms the rescale factor and
        // publishes both
        float* rb = red_wg + nb * HP * 4;
        if (lane < HP) rb[lane * 4 + wq] = mine;
        named_bar_sync(bar_id, 128);
        if (row < HP) {
          if (h0 + row < nr) {
            const float4 v = *reinterpret_cast<const float4*>(rb + 4 * row);
            const float mn = fmaxf(m_own, fmaxf(fmaxf(v.x, v.y), fmaxf(v.z, v.w)));
            // a token that has seen no position yet (causal mask) keeps a
            // finite reference so that exp2 gives 0, not NaN
            const float mref = (mn == -INFINITY) ? 0.f : mn;
            alpha_sm[nb * NP + h0 + row] = ex2(m_own - mref);
            max_sm[nb * NP + h0 + row] = mref;
            m_own = mn;
          } else {
            alpha_sm[nb * NP + h0 + row] = 1.f;
            max_sm[nb * NP + h0 + row] = 0.f;
          }
        }
        named_bar_sync(bar_id, 128);
        // probabilities (x becomes p) and this thread's sums
#pragma unroll
        for (int e4 = 0; e4 < HP; e4 += 4) {
          const float4 mv = *reinterpret_cast<const float4*>(max_sm + nb * NP + h0 + e4);
          const float4 av = *reinterpret_cast<const float4*>(alpha_sm + nb * NP + h0 + e4);
          const float mm[4] = {mv.x, mv.y, mv.z, mv.w};
          const float aa[4] = {av.x, av.y, av.z, av.w};
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const int e = e4 + k;
#pragma unroll
            for (int hf = 0; hf < NH; ++hf)
              x[hf][e] = (h0 + e < nr) ? ex2(x[hf][e] - mm[k]) : 0.f;
            l[e] = fmaf(l[e], aa[k], NH == 2 ? x[0][e] + x[NH - 1][e] : x[0][e]);
          }
        }
        // ---- P^T rows (position row, + 128), this warpgroup's heads, into
        // the MN-major swizzled B operand (16-byte chunks of 8 heads; WIDE:
        // over the stage's K rows, which the S products have finished
        // reading) ----
        {
          const uint32_t pbase =
              WIDE ? s_base + st * C::KV_BYTES : s_base + C::OFF_P + nb * C::P_BYTES;
#pragma unroll
          for (int hf = 0; hf < NH; ++hf) {
            const uint32_t prow = pbase + (row + hf * kT) * (NP * 2);
#pragma unroll
            for (int c = 0; c < HP / 8; ++c) {
              uint32_t wv[4];
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                wv[k] = Half16<T16>::pack2(x[hf][8 * c + 2 * k], x[hf][8 * c + 2 * k + 1]);
              }
              const int cg = h0 / 8 + c;  // chunk index within the row
              const int phys = (NP == 16) ? (cg ^ ((row >> 2) & 1)) : (cg ^ ((row >> 1) & 3));
              asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(prow + phys * 16),
                           "r"(wv[0]), "r"(wv[1]), "r"(wv[2]), "r"(wv[3])
                           : "memory");
            }
          }
        }
        // ---- last tile of a unit (warpgroup 0): zero the V rows past L_i;
        // one token: put v_new into row L_i - 1 and into the cache (n
        // tokens: the O-issuing warp patches the new rows) ----
        const bool patch_v = append_v && lt == seg.ti - 1;
        if (wg == 0 && (valid < TT || patch_v)) {
          // (DEEP: the V chunk 2n + 1 has a slot of its own)
          const int vst = DEEP ? (2 * n + 1) % ns : st;
          const bool vok = mbar_wait(BAR(B_FULL_V + vst),
                                     DEEP ? ((2 * n + 1) / pd) & 1 : (n / kStages) & 1,
                                     abort_flag, status, budget);
          const uint32_t vbase =
              s_base + vst * (DEEP ? sb : C::KV_BYTES) + (DEEP ? 0 : 2 * kBoxBytes);
          if (vok && patch_v && row < vch) {
            // (WIDE: rows 0-255 run on through the second box)
            const int rho = valid - 1;
            const uint32_t dst =
                vbase + (row >> 3) * kBoxBytes + rho * 128 + (((row & 7) ^ (rho & 7)) << 4);
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(dst), "r"(vnew.x),
                         "r"(vnew.y), "r"(vnew.z), "r"(vnew.w)
                         : "memory");
            if (vrow_w >= 0) v_cache_w[vrow_w * cpv + row] = vnew;
          }
#pragma unroll
          for (int hf = 0; hf < NH; ++hf) {
            const int pos = row + hf * kT;
            if (vok && pos >= valid) {
              const uint32_t vrow = vbase + pos * 128;
#pragma unroll
              // (the boxes the O product reads: DEEP with three slots all
              // four, with four slots the two of d_v <= 128)
              for (int hb = 0; hb < (WIDE ? 1 : (DEEP == 3 ? 4 : 2)); ++hb)
#pragma unroll
                for (int c = 0; c < 8; ++c)
                  asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};" ::"r"(
                                   vrow + hb * kBoxBytes + c * 16),
                               "r"(0u)
                               : "memory");
            }
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(BAR(B_P_READY + nb));
        // ---- fold O into the registers: the previous tile's, and at the
        // segment end this one's ----
        if (lt > seg.lt0) correct(n - 1, alpha_sm + ((n - 1) & 1) * NP);
        if (lt == seg.lt1 - 1) correct(n, alpha_sm + nb * NP);
      }

      // ---- segment end: softmax denominators, output or partial ----
      {
        // the sixteen heads' sums across the warp, by a reduce-scatter of
        // shuffles (16 shuffles in five rounds rather than sixteen chains of
        // five dependent ones): lane x ends with head (x >> 1) & 15's
        static_assert(HP == 16, "sixteen heads per warpgroup");
        const float mine = warp_sum16_scatter(l, lane);
        // the warp-maxima slot of the segment's last tile is free here (its
        // readers all passed that tile's second barrier); the next tile uses
        // the other slot, and the one after waits at its first barrier
        const uint32_t nlast = n - 1;
        float* lred = red_wg + (nlast & 1) * HP * 4;
        const float* mfin = max_sm + (nlast & 1) * NP + h0;
        if ((lane & 1) == 0) lred[wq * HP + (lane >> 1)] = mine;
        named_bar_sync(bar_id, 128);
        const bool whole = (seg.lt0 == 0 && seg.lt1 == seg.ti);
        // output row of column c: (i * n + s) * h + j * r + t; thread `row`
        // holds output column `row` (none past d_v; DEEP: also row + 128)
        auto has_col = [&](int hf) { return row + 128 * hf < dv; };
        T16* obase = out + (static_cast<size_t>(seg.i) * nq * h + seg.j * r) * dv + row;
        const int u = seg.i * g + seg.j;
        const size_t slot = static_cast<size_t>(u) + blockIdx.x;
        // l[e] becomes the CTA-wide softmax denominator of head h0 + e
#pragma unroll
        for (int e4 = 0; e4 < HP; e4 += 4) {
          const float4 a = *reinterpret_cast<const float4*>(lred + e4);
          const float4 b2 = *reinterpret_cast<const float4*>(lred + HP + e4);
          const float4 c2 = *reinterpret_cast<const float4*>(lred + 2 * HP + e4);
          const float4 d2 = *reinterpret_cast<const float4*>(lred + 3 * HP + e4);
          l[e4] = a.x + b2.x + c2.x + d2.x;
          l[e4 + 1] = a.y + b2.y + c2.y + d2.y;
          l[e4 + 2] = a.z + b2.z + c2.z + d2.z;
          l[e4 + 3] = a.w + b2.w + c2.w + d2.w;
        }
        // the final maxima and output row offsets of four heads at a time
        // (shared memory, loaded ahead of the stores that use them)
        auto mf4 = [&](int e4) { return *reinterpret_cast<const float4*>(mfin + e4); };
        auto co4 = [&](int e4) { return *reinterpret_cast<const int4*>(col_off + h0 + e4); };
        auto pick = [](const float4& v, int k) { return k == 0 ? v.x : k == 1 ? v.y : k == 2 ? v.z : v.w; };
        auto pick_i = [](const int4& v, int k) { return k == 0 ? v.x : k == 1 ? v.y : k == 2 ? v.z : v.w; };
        if (cl_merge) {
          // this CTA's partial, for the merge across the cluster
#pragma unroll
          for (int e4 = 0; e4 < HP; e4 += 4) {
            const float4 mv = mf4(e4);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const int e = e4 + k;
              if (h0 + e < nr) {
#pragma unroll
                for (int hf = 0; hf < OH; ++hf)
                  if (has_col(hf)) cl_o[(h0 + e) * dv + row + 128 * hf] = o[hf][e];
                if (row == 0) {
                  cl_ml[2 * (h0 + e)] = l[e] > 0.f ? pick(mv, k) : -INFINITY;
                  cl_ml[2 * (h0 + e) + 1] = l[e];
                }
              }
            }
          }
        } else if (whole) {
#pragma unroll
          for (int e4 = 0; e4 < HP; e4 += 4) {
            const int4 cv = co4(e4);
#pragma unroll
            for (int k = 0; k < 4; ++k)
#pragma unroll
              for (int hf = 0; hf < OH; ++hf)
                if (h0 + e4 + k < nr && has_col(hf))
                  obase[pick_i(cv, k) + 128 * hf] =
                      Half16<T16>::from(o[hf][e4 + k] / l[e4 + k]);
          }
        } else {
#pragma unroll
          for (int e4 = 0; e4 < HP; e4 += 4) {
            const float4 mv = mf4(e4);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const int e = e4 + k;
              if (h0 + e < nr) {
                const size_t sl = slot * nr + h0 + e;
#pragma unroll
                for (int hf = 0; hf < OH; ++hf)
                  if (has_col(hf)) part_o[sl * dv + row + 128 * hf] = o[hf][e];
                if (row == 0) {
                  // a token that saw none of this CTA's positions: empty partial
                  part_ml[sl * 2 + 0] = l[e] > 0.f ? pick(mv, k) : -INFINITY;
                  part_ml[sl * 2 + 1] = l[e];
                }
              }
            }
          }
          // the unit is split across CTAs: for its heads, the warpgroup that
          // finishes last merges the other partials into its own (still in
          // registers)
          long long c0, c1;
          unit_ctas(seg.u0, seg.u0 + seg.ti, w.W, w.nc, c0, c1);
          const int np = unit_parts(c0, c1, w.W, w.nc);
          if (cl_size > 1) {
            // ragged cluster launch: the cluster holding the unit's last
            // piece merges it after the kernel's loop (below); list it
            if (wg == 0 && row == 0) {
              int* sl4 = split_list + (seg.lt0 == 0 ? 4 : 0);  // unit's first piece: the CTA's last segment
              sl4[0] = u;
              sl4[1] = static_cast<int>(c0);
              sl4[2] = static_cast<int>(c1);
              sl4[3] = np;
            }
          } else if (counters != nullptr && h0 < nr &&
              arrive_last(counters, u * NWG + wg, np, last_flag_wg, row == 0, bar_id, 128)) {
            // pieces merge in CTA order whichever CTA merges (the same bits
            // every run).  This CTA's piece is used from registers when it
            // is the first (one warpgroup: registers to spare), else read
            // back like the others.
            bool own_first = false;
            if constexpr (NWG == 1) {
              long long cfirst = c0;
              if (w.W < w.nc)
                while (cfirst < c1 && cta_empty(cfirst, w.W, w.nc)) ++cfirst;
              own_first = cfirst == blockIdx.x;
            }
            float m[HP];
#pragma unroll
            for (int e = 0; e < HP; ++e) {
              m[e] = (own_first && l[e] > 0.f) ? mfin[e] : -INFINITY;
              if (!own_first) {
#pragma unroll
                for (int hf = 0; hf < OH; ++hf) o[hf][e] = 0.f;
                l[e] = 0.f;
              }
            }
            for (long long c = c0; c <= c1; ++c) {
              if ((own_first && c == blockIdx.x) || (w.W < w.nc && cta_empty(c, w.W, w.nc)))
                continue;
              // eight heads at a time: their loads go out together
#pragma unroll
              for (int e0 = 0; e0 < HP; e0 += 8) {
                float mc[8], lc[8], oc[OH][8];
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                  if (h0 + e0 + k < nr) {
                    const long long sl = (u + c) * nr + h0 + e0 + k;
                    mc[k] = __ldcg(part_ml + sl * 2);
                    lc[k] = __ldcg(part_ml + sl * 2 + 1);
                    // (threads past d_v read a valid column and drop it)
                    oc[0][k] = __ldcg(part_o + sl * dv + min(row, dv - 1));
                    if (OH == 2)
                      oc[OH - 1][k] = __ldcg(part_o + sl * dv + min(row + 128, dv - 1));
                  }
                }
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                  const int e = e0 + k;
                  if (h0 + e < nr) {
                    const float mn = fmaxf(m[e], mc[k]);
                    const float mr = (mn == -INFINITY) ? 0.f : mn;  // both pieces empty
                    const float sa = ex2(m[e] - mr), sb = ex2(mc[k] - mr);
#pragma unroll
                    for (int hf = 0; hf < OH; ++hf) o[hf][e] = o[hf][e] * sa + oc[hf][k] * sb;
                    l[e] = l[e] * sa + lc[k] * sb;
                    m[e] = mn;
                  }
                }
              }
            }
#pragma unroll
            for (int e4 = 0; e4 < HP; e4 += 4) {
              const int4 cv = co4(e4);
#pragma unroll
              for (int k = 0; k < 4; ++k)
#pragma unroll
                for (int hf = 0; hf < OH; ++hf)
                  if (h0 + e4 + k < nr && has_col(hf))
                    obase[pick_i(cv, k) + 128 * hf] =
                        Half16<T16>::from(o[hf][e4 + k] / l[e4 + k]);
            }
          }
        }
        m_own = -INFINITY;
#pragma unroll
        for (int e = 0; e < HP; ++e) {
          l[e] = 0.f;
#pragma unroll
          for (int hf = 0; hf < OH; ++hf) o[hf][e] = 0.f;
        }
      }
    }
    if (cl_merge && !had_seg) {
      // a CTA with no tile of its unit: an empty partial
#pragma unroll
      for (int e = 0; e < HP; ++e) {
        if (h0 + e < nr) {
#pragma unroll
          for (int hf = 0; hf < OH; ++hf)
            if (row + 128 * hf < dv) cl_o[(h0 + e) * dv + row + 128 * hf] = 0.f;
          if (row == 0) {
            cl_ml[2 * (h0 + e)] = -INFINITY;
            cl_ml[2 * (h0 + e) + 1] = 0.f;
          }
        }
      }
    }
  }

  if (cl_merge) {
    // ====================== merge across the cluster ======================
    // Unit u's pieces are the partials of its cl_size * cl_k CTAs.  After the
    // barrier, CTA `rank` of a cluster merges items [rank * N / cl_size,
    // (rank + 1) * N / cl_size) of the unit's N = nr * d_v / 4 output chunks
    // (query row e, four columns) over the cluster's CTAs in rank order,
    // reading their shared memory.  With one cluster per unit that is the
    // output; with cl_k clusters, each cluster writes its merged slice as a
    // partial to global memory and, per slice, the CTA that arrives last
    // merges the cl_k of them in cluster order (the same bits every run).
    cluster_arrive();
    cluster_wait();
    const int rank = static_cast<int>(cluster_ctarank());
    const int per_unit = cl_size * cl_k;
    const int u = blockIdx.x / per_unit;
    const int kc = (blockIdx.x / cl_size) % cl_k;
    const int ui = u / g, uj = u % g;
    const int nq4 = dv >> 2;
    const int items = nr * nq4;
    const int it0 = (rank * items) / cl_size, it1 = ((rank + 1) * items) / cl_size;
    const uint32_t o_s = s_base, ml_s = s_base + NP * dv * 4;
    T16* obase_u = out + (static_cast<size_t>(ui) * nq * h + uj * r) * dv;
    auto store4 = [&](int e, int q, float4 v) {
      const uint2 pk = make_uint2(Half16<T16>::pack2(v.x, v.y), Half16<T16>::pack2(v.z, v.w));
      *reinterpret_cast<uint2*>(obase_u + col_off[e] + 4 * q) = pk;
    };
    for (int it = it0 + static_cast<int>(threadIdx.x); it < it1;
         it += static_cast<int>(blockDim.x)) {
      const int e = it / nq4, q = it - e * nq4;
      float mc[16];
      float M = -INFINITY;
#pragma unroll
      for (int c = 0; c < 16; ++c) {
        mc[c] = c < cl_size ? ld_dsmem(dsmem_addr(ml_s + 8 * e, c)) : -INFINITY;
        M = fmaxf(M, mc[c]);
      }
      const float mr = (M == -INFINITY) ? 0.f : M;  // every piece empty
      float4 num = make_float4(0.f, 0.f, 0.f, 0.f);
      float den = 0.f;
#pragma unroll
      for (int c = 0; c < 16; ++c) {
        if (c < cl_size) {
          const float wgt = ex2(mc[c] - mr);
          const float4 ov = ld_dsmem4(dsmem_addr(o_s + (e * dv + 4 * q) * 4, c));
          const float lc = ld_dsmem(dsmem_addr(ml_s + 8 * e + 4, c));
          num.x = fmaf(wgt, ov.x, num.x);
          num.y = fmaf(wgt, ov.y, num.y);
          num.z = fmaf(wgt, ov.z, num.z);
          num.w = fmaf(wgt, ov.w, num.w);
          den = fmaf(wgt, lc, den);
        }
      }
      if (cl_k == 1) {
        store4(e, q, make_float4(num.x / den, num.y / den, num.z / den, num.w / den));
      } else {
        const size_t sl = (static_cast<size_t>(u) * cl_k + kc) * nr + e;
        __stcg(reinterpret_cast<float4*>(part_o + sl * dv) + q, num);
        if (q == 0) {
          __stcg(part_ml + sl * 2, M);
          __stcg(part_ml + sl * 2 + 1, den);
        }
      }
    }
    // this CTA's shared memory is no longer read by the cluster once every
    // CTA passes the wait below
    cluster_arrive();
    if (cl_k > 1) {
      __threadfence();
      __syncthreads();
      if (threadIdx.x == 0) {
        const int old = atomicAdd(counters + u * cl_size + rank, 1);
        const int last = (old == cl_k - 1) ? 1 : 0;
        if (last) {
          counters[u * cl_size + rank] = 0;
          __threadfence();
        }
        *reinterpret_cast<volatile int*>(last_flag) = last;
      }
      __syncthreads();
      if (*reinterpret_cast<volatile int*>(last_flag)) {
        for (int it = it0 + static_cast<int>(threadIdx.x); it < it1;
             it += static_cast<int>(blockDim.x)) {
          const int e = it / nq4, q = it - e * nq4;
          float M = -INFINITY, den = 0.f;
          float4 num = make_float4(0.f, 0.f, 0.f, 0.f);
          for (int c0 = 0; c0 < cl_k; c0 += 4) {
            float mc[4], lc[4];
            float4 oc[4];
#pragma unroll
            for (int k4 = 0; k4 < 4; ++k4) {
              const int c = c0 + k4;
              const size_t sl = (static_cast<size_t>(u) * cl_k + c) * nr + e;
              mc[k4] = c < cl_k ? __ldcg(part_ml + sl * 2) : -INFINITY;
              lc[k4] = c < cl_k ? __ldcg(part_ml + sl * 2 + 1) : 0.f;
              oc[k4] = c < cl_k ? __ldcg(reinterpret_cast<const float4*>(part_o + sl * dv) + q)
                                : make_float4(0.f, 0.f, 0.f, 0.f);
            }
            float mb = M;
#pragma unroll
            for (int k4 = 0; k4 < 4; ++k4) mb = fmaxf(mb, mc[k4]);
            const float mbr = (mb == -INFINITY) ? 0.f : mb;
            const float sc = ex2(M - mbr);  // 0 while M = -inf
            den *= sc;
            num.x *= sc;
            num.y *= sc;
            num.z *= sc;
            num.w *= sc;
#pragma unroll
            for (int k4 = 0; k4 < 4; ++k4) {
              const float wgt = ex2(mc[k4] - mbr);
              den = fmaf(wgt, lc[k4], den);
              num.x = fmaf(wgt, oc[k4].x, num.x);
              num.y = fmaf(wgt, oc[k4].y, num.y);
              num.z = fmaf(wgt, oc[k4].z, num.z);
              num.w = fmaf(wgt, oc[k4].w, num.w);
            }
            M = mb;
          }
          store4(e, q, make_float4(num.x / den, num.y / den, num.z / den, num.w / den));
        }
      }
    }
    cluster_wait();
  } else if (cl_size > 1) {
    // ============ ragged lengths in a cluster launch: the unit's pieces are
    // global partials (slots u + c); the CTA whose piece completes a unit's
    // count marks it, and after the barrier its whole cluster merges that
    // unit, each CTA a slice of the outputs, the pieces in CTA order ========
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
      for (int s2 = 0; s2 < 2; ++s2) {
        int* e4 = split_list + 4 * s2;
        if (e4[0] < 0) continue;
        if (atomicAdd(counters + e4[0], 1) == e4[3] - 1)
          counters[e4[0]] = 0;  // this CTA completes the unit
        else
          e4[0] = -1;
      }
      __threadfence();
    }
    cluster_arrive();
    cluster_wait();
    const int rank = static_cast<int>(cluster_ctarank());
    const int nq4 = dv >> 2;
    const int items = nr * nq4;
    const int it0 = (rank * items) / cl_size, it1 = ((rank + 1) * items) / cl_size;
    const uint32_t lst = smem_u32(split_list);
    for (int c = 0; c < cl_size; ++c) {
      for (int s2 = 0; s2 < 2; ++s2) {
        const uint32_t ea = dsmem_addr(lst + 16 * s2, c);
        const int u = ld_dsmem_s32(ea);
        if (u < 0) continue;
        const int c0 = ld_dsmem_s32(ea + 4), c1 = ld_dsmem_s32(ea + 8);
        T16* obase_u = out + (static_cast<size_t>(u / g) * nq * h + (u % g) * r) * dv;
        for (int it = it0 + static_cast<int>(threadIdx.x); it < it1;
             it += static_cast<int>(blockDim.x)) {
          const int e = it / nq4, q = it - e * nq4;
          float M = -INFINITY, den = 0.f;
          float4 num = make_float4(0.f, 0.f, 0.f, 0.f);
          for (int cb = c0; cb <= c1; cb += 8) {
            float mc[8], lc[8];
            float4 oc[8];
#pragma unroll
            for (int k8 = 0; k8 < 8; ++k8) {
              const int cc = cb + k8;
              const bool use = cc <= c1 && (w.W >= w.nc || !cta_empty(cc, w.W, w.nc));
              const size_t sl = (static_cast<size_t>(u) + cc) * nr + e;
              mc[k8] = use ? __ldcg(part_ml + sl * 2) : -INFINITY;
              lc[k8] = use ? __ldcg(part_ml + sl * 2 + 1) : 0.f;
              oc[k8] = use ? __ldcg(reinterpret_cast<const float4*>(part_o + sl * dv) + q)
                           : make_float4(0.f, 0.f, 0.f, 0.f);
            }
            float mb = M;
#pragma unroll
            for (int k8 = 0; k8 < 8; ++k8) mb = fmaxf(mb, mc[k8]);
            const float mbr = (mb == -INFINITY) ? 0.f : mb;
            const float sc = ex2(M - mbr);  // 0 while M = -inf
            den *= sc;
            num.x *= sc;
            num.y *= sc;
            num.z *= sc;
            num.w *= sc;
#pragma unroll
            for (int k8 = 0; k8 < 8; ++k8) {
              const float wgt = ex2(mc[k8] - mbr);  // 0 for unused slots, empty pieces
              den = fmaf(wgt, lc[k8], den);
              num.x = fmaf(wgt, oc[k8].x, num.x);
              num.y = fmaf(wgt, oc[k8].y, num.y);
              num.z = fmaf(wgt, oc[k8].z, num.z);
              num.w = fmaf(wgt, oc[k8].w, num.w);
            }
            M = mb;
          }
          const uint2 pk =
              make_uint2(Half16<T16>::pack2(num.x / den, num.y / den),
                         Half16<T16>::pack2(num.z / den, num.w / den));
          *reinterpret_cast<uint2*>(obase_u + col_off[e] + 4 * q) = pk;
        }
      }
    }
    // no CTA leaves while another may still read its list
    cluster_arrive();
    cluster_wait();
  }

  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::NCOLS);
  }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
// 2-D map over a row-major [rows x d] 16-bit tensor (d = 64 or 128), box
// [box_rows x 64], 128-byte swizzle, zero fill outside.  (The query map is
// 3-D: [b * n tokens][h heads][d_k], box [n][r][64].)
bool make_map(CUtensorMap* map, const void* base, int d, uint64_t rows, uint32_t box_rows,
              bool bf16) {
  const uint64_t dims[2] = {static_cast<uint64_t>(d), rows};
  const uint64_t strides[1] = {static_cast<uint64_t>(d) * 2};
  const uint32_t box[2] = {64u, box_rows};
  return encode_bf16_map(map, base, 2, dims, strides, box, bf16);
}

bool make_q_map(CUtensorMap* map, const void* base, int b, int nq, int h, int r, int d,
                bool bf16) {
  const uint64_t dims[3] = {static_cast<uint64_t>(d), static_cast<uint64_t>(h),
                            static_cast<uint64_t>(b) * nq};
  const uint64_t strides[2] = {static_cast<uint64_t>(d) * 2,
                               static_cast<uint64_t>(h) * d * 2};
  const uint32_t box[3] = {64u, static_cast<uint32_t>(r), static_cast<uint32_t>(nq)};
  return encode_bf16_map(map, base, 3, dims, strides, box, bf16);
}

// The shared-memory opt-in and the permission for clusters of up to 16 CTAs
// are set once per device and kernel (outside any stream capture: the first
// call on a device must come before a capture).
template <typename K>
cudaError_t configure_kernel(K kern, int smem, std::atomic<unsigned long long>& configured) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!(configured.load() & (1ull << dev))) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
    configured.fetch_or(1ull << dev);
  }
  return cudaSuccess;
}

template <int NP, int NWG, bool MULTI, bool PAGED, typename T16, bool WIDE, int DEEP = 0>
cudaError_t launch_np(const DecodeLaunch& a) {
  constexpr bool kBf16 = Half16<T16>::kBf16;
  using C = TcCfg<NP, NWG, MULTI, PAGED, kBf16, WIDE, DEEP>;
  CUtensorMap mq, mk, mv;
  // contiguous caches: [b * g * cap rows x 128]; pools: [num_blocks * g * block_size rows]
  const uint64_t kv_rows = PAGED ? static_cast<uint64_t>(a.num_blocks) * a.g * a.block_size
                                 : static_cast<uint64_t>(a.b) * a.g * a.cap;
  const uint32_t box_rows = (PAGED && a.block_size < kT) ? a.block_size : kT;
  if (!make_q_map(&mq, a.q, a.b, a.nq, a.h, a.h / a.g, a.d, kBf16) ||
      !make_map(&mk, a.k_cache, a.d, kv_rows, box_rows, kBf16) ||
      !make_map(&mv, a.v_cache, a.dv, kv_rows, box_rows, kBf16))
    return cudaErrorInvalidValue;
  auto kern = decode_tc_kernel<NP, NWG, MULTI, PAGED, T16, WIDE, DEEP>;
  static std::atomic<unsigned long long> configured{0};  // devices done, this variant
  if (cudaError_t e = configure_kernel(kern, C::SMEM, configured)) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.nc);
  cfg.blockDim = dim3(C::THREADS);
  cfg.dynamicSmemBytes = C::SMEM;
  cfg.stream = a.stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (a.cluster > 1) {
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = static_cast<unsigned>(a.cluster);
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.numAttrs = 2;
  }
  return cudaLaunchKernelEx(
      &cfg, kern, mq, mk, mv, a.seq_lens, a.b, a.h, a.g, a.cap, a.scale_log2,
      static_cast<T16*>(a.out), a.part_o, a.part_ml, a.counters,
      static_cast<const uint4*>(a.k_new), static_cast<const uint4*>(a.v_new),
      static_cast<uint4*>(a.k_cache_w), static_cast<uint4*>(a.v_cache_w), a.status, a.budget,
      a.early ? 1 : 0, a.nq, a.block_table, a.block_size, a.max_blocks, a.num_blocks, a.d / 64,
      a.dv / 64, a.cluster > 1 ? a.cluster : 0, a.cluster > 1 ? a.cluster_k : 1);
}

template <typename T16, bool WIDE>
cudaError_t launch_type(const DecodeLaunch& a) {
  const int cols = a.nq * (a.h / a.g);
  const bool one = a.nq == 1;
  if (deep_dims(a.d, a.dv)) {  // (16 query rows at most)
    // four 48 KiB ring slots when a K chunk fits three boxes and V two
    const bool four = a.d <= 192 && a.dv <= 128;
    if (a.block_table != nullptr) {
      if (four)
        return one ? launch_np<16, 1, false, true, T16, false, 4>(a)
                   : launch_np<16, 1, true, true, T16, false, 4>(a);
      return one ? launch_np<16, 1, false, true, T16, false, 3>(a)
                 : launch_np<16, 1, true, true, T16, false, 3>(a);
    }
    if (four)
      return one ? launch_np<16, 1, false, false, T16, false, 4>(a)
                 : launch_np<16, 1, true, false, T16, false, 4>(a);
    return one ? launch_np<16, 1, false, false, T16, false, 3>(a)
               : launch_np<16, 1, true, false, T16, false, 3>(a);
  }
  if (a.block_table != nullptr) {
    if (one)
      return cols <= 16 ? launch_np<16, 1, false, true, T16, WIDE>(a)
                        : launch_np<32, 2, false, true, T16, WIDE>(a);
    return cols <= 16 ? launch_np<16, 1, true, true, T16, WIDE>(a)
                      : launch_np<32, 2, true, true, T16, WIDE>(a);
  }
  if (one)
    return cols <= 16 ? launch_np<16, 1, false, false, T16, WIDE>(a)
                      : launch_np<32, 2, false, false, T16, WIDE>(a);
  return cols <= 16 ? launch_np<16, 1, true, false, T16, WIDE>(a)
                    : launch_np<32, 2, true, false, T16, WIDE>(a);
}

}  // namespace

bool tc_supported(int dtype, int d_k, int d_v, int cols, bool) {
  if (dtype != GQA_BF16 && dtype != GQA_F16) return false;
  if (deep_dims(d_k, d_v)) return cols >= 1 && cols <= 16;
  return (d_k == 64 || d_k == 128) && (d_v == 64 || d_v == 128) && cols >= 1 && cols <= 32;
}

int tc_tile(int d_k, int d_v) { return wide_tiles(d_k, d_v) ? 2 * kT : kT; }

int tc_max_clusters(int csize) {
  // One CTA per SM whatever the variant (every one takes over 200 KiB of
  // shared memory), so the largest variant stands for all.  Cached per device.
  static std::atomic<int> cache[64][17];
  static std::atomic<bool> init[64][17];
  if (csize < 1 || csize > 16) return 0;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  if (init[dev][csize].load()) return cache[dev][csize].load();
  using C = TcCfg<32, 2, false, false, true, false>;
  auto kern = decode_tc_kernel<32, 2, false, false, __nv_bfloat16, false, 0>;
  static std::atomic<unsigned long long> configured{0};
  if (configure_kernel(kern, C::SMEM, configured) != cudaSuccess) return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(csize * 64);
  cfg.blockDim = dim3(C::THREADS);
  cfg.dynamicSmemBytes = C::SMEM;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(csize);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
    cudaGetLastError();  // (a query that failed leaves no sticky error)
    n = 0;
  }
  cache[dev][csize].store(n);
  init[dev][csize].store(true);
  return n;
}

int tc_ctas_per_sm(int) { return 1; }

cudaError_t launch_decode_tc(const DecodeLaunch& a) {
  if (wide_tiles(a.d, a.dv))
    return a.dtype == GQA_F16 ? launch_type<__half, true>(a) : launch_type<__nv_bfloat16, true>(a);
  return a.dtype == GQA_F16 ? launch_type<__half, false>(a) : launch_type<__nv_bfloat16, false>(a);
}

}  // namespace gqa
