// decode_simt.cu - CUDA-core split-KV decode attention (fp32 inputs, and the
// 16-bit types with head dim 64 or with different K and V head dims).
//
// One persistent CTA per SM streams its share of the (sequence, KV head)
// tiles (see Walker).  Warp 0 copies each K/V tile of T positions from HBM
// into a shared-memory ring (three 64 KiB stages for fp32, five of 32 KiB
// for 16-bit data) with one bulk copy per tensor (the
// rows of a tile are contiguous in the cache), completing on an mbarrier;
// only the rows below L_i are copied.  Warps 1-7 serve all r = h/g query
// heads of the KV head from each tile:
//   A  logits: 16-byte vector loads of K (each lane one or two chunks of a
//      row: as many as keep q within 64 registers), fp32 dot products
//      against q held in registers, summed across the lanes that share a
//      row by a reduce-scatter of xor shuffles (each round trades half of
//      the heads' partial sums with the partner lane: r - 1 + log2(lanes /
//      r) shuffles a row instead of r log2(lanes)) (the "bhk,bhmk->bhm"
//      contraction of the MQA review §2.4);
//   B  online softmax per head in base 2: warp max, rescale factor, exp2,
//      warp sum;
//   C  weighted sum of V rows (two positions a step) into fp32 register
//      accumulators ("bhm,bhmv->bhv"), rescaled by each tile's factor.
// A segment's end writes the normalised output; a unit split across CTAs
// writes a partial instead, and the CTA that finishes the unit last merges
// the partials (log-sum-exp).  With n new tokens per sequence the "heads"
// are the n * r query rows of the group (token-major) and token s, at
// position L_i - n + s, sees positions p <= L_i - n + s (the causal mask of
// the batched form, §2.3).  With k_new / v_new given, the KV append is
// fused in: the CTA owning a tile that holds rows L_i - n .. L_i - 1 patches
// them in its staged tile with the new tokens and writes them to the cache.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <atomic>

#include "gqa_device.cuh"
#include "gqa_internal.h"

namespace gqa {
namespace {

template <typename DT>
struct Elt;
template <>
struct Elt<float> {
  static constexpr int size = 4;
  __device__ static void unpack(const uint4& u, float* f) {
    f[0] = __uint_as_float(u.x);
    f[1] = __uint_as_float(u.y);
    f[2] = __uint_as_float(u.z);
    f[3] = __uint_as_float(u.w);
  }
  __device__ static void store(float* p, float v) { *p = v; }
};
template <>
struct Elt<__nv_bfloat16> {
  static constexpr int size = 2;
  __device__ static void unpack(const uint4& u, float* f) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      f[2 * k] = __uint_as_float(w[k] << 16);
      f[2 * k + 1] = __uint_as_float(w[k] & 0xFFFF0000u);
    }
  }
  __device__ static void store(__nv_bfloat16* p, float v) { *p = __float2bfloat16_rn(v); }
};
template <>
struct Elt<__half> {
  static constexpr int size = 2;
  __device__ static void unpack(const uint4& u, float* f) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 v = __half22float2(*reinterpret_cast<const __half2*>(&w[k]));
      f[2 * k] = v.x;
      f[2 * k + 1] = v.y;
    }
  }
  __device__ static void store(__half* p, float v) { *p = __float2half_rn(v); }
};

// DK / DV: head dims of K (and q) and of V (and out); they may differ.
// Seven compute warps: eight warps in all, two per SM sub-partition, so a
// thread may hold up to 255 registers (measured: fifteen compute warps of
// 128 registers were slower on the fp32 Llama-3-70B shape, 2.0 against 2.6
// TB/s, their share of the weighted sum taking twice as long).  fp32 with
// both head dims 128 and r <= 8 runs eight (two on each sub-partition
// besides the copy warp; 224 registers a thread, no spills): a tile's 32
// position pairs then take four steps of every warp instead of five of
// the busiest.  fp32 tiles
// hold 64 KiB of K + V in a three-stage ring (half the barriers and softmax
// passes a position of 32 KiB tiles: the fp32 Llama-3-70B shape 848 -> 722
// us per call), 16-bit ones 32 KiB in five stages.
template <typename DT, int DK, int DV, int RMAX>
struct SimtCfg {
  static constexpr int NCW = (sizeof(DT) == 4 && RMAX <= 8 && DK == 128 && DV == 128) ? 8 : 7;
  static constexpr int NCT = 32 * NCW;          // compute threads
  static constexpr int THREADS = 32 + NCT;      // warp 0 copies
  static constexpr int ELT = Elt<DT>::size;
  static constexpr int CHK = DK * ELT / 16;    // 16-byte chunks per K row
  static constexpr int CHV = DV * ELT / 16;    // ... per V row
  static constexpr int EPC = 16 / ELT;         // elements per chunk
  // logits pass: each lane holds CPL chunks of q per query row (at most 64
  // registers of q, and at least one head per lane after the reduction),
  // so LPR lanes share a K row and a warp step covers PPW rows
  static constexpr int CPL0 = 64 / (RMAX * EPC) < 1 ? 1 : 64 / (RMAX * EPC);
  static constexpr int CPL = CPL0 < CHK / RMAX ? CPL0 : (CHK / RMAX < 1 ? 1 : CHK / RMAX);
  static constexpr int LPR = CHK / CPL;
  static constexpr int PPW = 32 / LPR;         // K rows per warp step
  static constexpr int DM = DK > DV ? DK : DV;
  static constexpr int T = (ELT == 4 ? 32768 : 16384) / (DM * ELT);  // positions per tile
  static constexpr int PPL = T / 16;           // positions per lane in softmax
  static constexpr int NPG = NCT / CHV;        // position groups in the V pass
  static constexpr int STAGES = ELT == 4 ? 3 : 5;
  static constexpr int NSLOT = ELT == 4 ? 2 : 4;  // segment-end reduction slots
  static constexpr int K_BYTES = T * DK * ELT;
  static constexpr int STAGE_BYTES = T * (DK + DV) * ELT;
  static constexpr int OFF_P = STAGES * STAGE_BYTES;          // float [RMAX][T]
  static constexpr int OFF_RED = OFF_P + RMAX * T * 4;            // float [NSLOT][RMAX][DV]
  static constexpr int OFF_ML = OFF_RED + NSLOT * RMAX * DV * 4;  // float m,l,alpha [RMAX]
  static constexpr int OFF_BAR = OFF_ML + 3 * RMAX * 4;
  static constexpr int OFF_MISC = OFF_BAR + 2 * STAGES * 8;
  static constexpr int SMEM = OFF_MISC + 16 + 128;
  static_assert(CHK <= 32 && 32 % CHK == 0 && CHV <= 32 && 32 % CHV == 0,
                "rows must split evenly over lanes");
  static_assert(T % 32 == 0, "tile shape");
  static_assert(SMEM <= 232448, "shared memory budget");
  static_assert(RMAX <= LPR, "a row's lanes hold at least one head each after the reduction");
  static_assert(CHK % CPL == 0 && T % PPW == 0, "logits mapping");
  static_assert(K_BYTES % 16 == 0, "16-byte aligned V tile");
};


// Sum each of R values across the CHK lanes that share a row (lanes l with
// the same l / CHK; R <= CHK, both powers of two).  Each round trades half
// of the values still held with the partner lane l ^ O and adds, so lane l
// ends with the row total of value (l % CHK) / (CHK / R) in v[0] (the CHK /
// R lanes that hold it agree); R - 1 + log2(CHK / R) shuffles in all.
template <int CHK, int R>
struct RowReduce {
  template <int O, int NV>
  __device__ static void step(float (&v)[R], int lane) {
    if constexpr (O >= 1) {
      if constexpr (NV > 1) {
        const bool up = (lane & O) != 0;
#pragma unroll
        for (int k = 0; k < NV / 2; ++k) {
          const float send = up ? v[k] : v[k + NV / 2];
          const float keep = up ? v[k + NV / 2] : v[k];
          v[k] = keep + __shfl_xor_sync(0xffffffffu, send, O);
        }
        step<O / 2, NV / 2>(v, lane);
      } else {
        v[0] += __shfl_xor_sync(0xffffffffu, v[0], O);
        step<O / 2, 1>(v, lane);
      }
    }
  }
  __device__ static void run(float (&v)[R], int lane) { step<CHK / 2, R>(v, lane); }
  // the value lane l holds, and whether it is the first of its copies
  __device__ static int head(int lane) { return (lane % CHK) / (CHK / R); }
  __device__ static bool writer(int lane) { return (lane % (CHK / R)) == 0; }
};

template <typename DT, int DK, int DV, int RMAX>
__global__ void __launch_bounds__(SimtCfg<DT, DK, DV, RMAX>::THREADS, 1)
    decode_simt_kernel(const DT* __restrict__ q, const DT* __restrict__ kc,
                       const DT* __restrict__ vc, const int* __restrict__ lens, int b, int h,
                       int g, int cap, float scale_log2, DT* __restrict__ out,
                       float* __restrict__ part_o, float* __restrict__ part_ml,
                       int* __restrict__ counters, const uint4* __restrict__ k_new,
                       const uint4* __restrict__ v_new, uint4* __restrict__ k_cache_w,
                       uint4* __restrict__ v_cache_w, unsigned int* status, long long budget,
                       int nq, const int* __restrict__ table, int bsz, int max_blocks,
                       int num_blocks, int early) {
  using C = SimtCfg<DT, DK, DV, RMAX>;
  constexpr int kCompute = C::NCT, kWarps = C::NCW;
  extern __shared__ __align__(128) uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) &
                                           ~uintptr_t(127));
  float* sP = reinterpret_cast<float*>(sm + C::OFF_P);
  float* sRed = reinterpret_cast<float*>(sm + C::OFF_RED);
  float* sM = reinterpret_cast<float*>(sm + C::OFF_ML);
  float* sL = sM + RMAX;
  float* sA = sL + RMAX;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + C::OFF_BAR);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + C::OFF_MISC);
  int* last_flag = reinterpret_cast<int*>(sm + C::OFF_MISC + 4);
  const uint32_t full0 = smem_u32(bars);
  const uint32_t empty0 = smem_u32(bars + C::STAGES);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = h / g;
  const int nr = nq * r;  // query rows ("heads" below) per KV head: t = s * r + head

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (threadIdx.x >= 32 && threadIdx.x < 32 + RMAX) {
    const int t = threadIdx.x - 32;
    sM[t] = -INFINITY;
    sL[t] = 0.f;
    sA[t] = 0.f;
  }
  __syncthreads();  // barrier inits and the softmax state (this CTA's own)
  // Inputs and the split workspace are read only after the dependency wait.
  // With `early` set the caller guarantees that no kernel still running
  // writes seq_lens, the block table or the cache rows below L_i - n (e.g.
  // it is another layer's step), so the producer warp plans its tiles and
  // copies the first ring's worth before it waits.
  if (!early || warp != 0) pdl_wait_then_release();
  if (warp == 1 && blockIdx.x == 0) report_bad_lengths(lens, b, nq, cap, status);

  Walker w;
  w.init(lens, b, g, nq, cap, C::T, blockIdx.x, gridDim.x);
  Segment seg;

  if (warp == 0) {
    // ---------------- producer ----------------
    if (table != nullptr) {
      // paged cache: the whole warp walks the tiles (block-table lookups
      // over its lanes), lane 0 issues one copy per block piece of a tile;
      // pieces in bad blocks are not copied (the status word says so)
      uint32_t n = 0;
      int last_n[C::STAGES];
#pragma unroll
      for (int s = 0; s < C::STAGES; ++s) last_n[s] = -1;
      const int piece = bsz < C::T ? bsz : C::T;
      PageCursor pc;
      bool waited = !early;
      while (w.next(seg)) {
        pc.start(table + static_cast<size_t>(seg.i) * max_blocks, (seg.L + bsz - 1) / bsz,
                 (seg.lt0 * C::T) / bsz);
        for (int lt = seg.lt0; lt < seg.lt1; ++lt, ++n) {
          if (!waited && n == static_cast<uint32_t>(C::STAGES)) {  // the ring is full
            pdl_wait_then_release();
            waited = true;
          }
          const int st = n % C::STAGES;
          const bool ok = __all_sync(0xffffffffu,
                                     mbar_wait(empty0 + 8 * st, ((n / C::STAGES) & 1) ^ 1,
                                               abort_flag, status, budget));
          if (!ok) continue;
          const int p0 = lt * C::T;
          // lane mm < T / piece copies piece mm (one block's rows) of the tile
          const int e = pc.get_lanes(p0 / bsz);
          const int pm = p0 + lane * piece;
          const bool mine = lane * piece < C::T && pm < seg.L;
          const bool good = mine && e >= 0 && e < num_blocks;
          const uint32_t rows_m = good ? static_cast<uint32_t>(min(piece, seg.L - pm)) : 0u;
          const uint32_t total =
              __reduce_add_sync(0xffffffffu, rows_m * (DK + DV) * C::ELT);
          if (__any_sync(0xffffffffu, mine && !good) && lane == 0)
            atomicOr(status, GQA_DEV_BAD_BLOCK);
          uint8_t* stage = sm + st * C::STAGE_BYTES;
          if (lane == 0) mbar_arrive_expect_tx(full0 + 8 * st, total);
          __syncwarp();
          if (good) {
            const size_t prow = (static_cast<size_t>(e) * g + seg.j) * bsz + pm % bsz;
            bulk_load(smem_u32(stage + lane * piece * DK * C::ELT), kc + prow * DK,
                      rows_m * DK * C::ELT, full0 + 8 * st);
            bulk_load(smem_u32(stage + C::K_BYTES + lane * piece * DV * C::ELT), vc + prow * DV,
                      rows_m * DV * C::ELT, full0 + 8 * st);
          }
          last_n[st] = static_cast<int>(n);
        }
      }
      if (!waited) pdl_wait_then_release();
      if (*abort_flag && lane == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
          if (last_n[s] < 0) continue;
          const uint32_t par = (last_n[s] / C::STAGES) & 1;
          const long long t0 = clock64();
          while (!mbar_try_wait(full0 + 8 * s, par) && clock64() - t0 < budget) {
          }
        }
      }
    } else if (lane == 0) {
      uint32_t n = 0;
      int last_n[C::STAGES];
#pragma unroll
      for (int s = 0; s < C::STAGES; ++s) last_n[s] = -1;
      bool waited = !early;
      while (w.next(seg)) {
        const size_t unit_row = (static_cast<size_t>(seg.i) * g + seg.j) * cap;
        for (int lt = seg.lt0; lt < seg.lt1; ++lt, ++n) {
          if (!waited && n == static_cast<uint32_t>(C::STAGES)) {  // the ring is full
            pdl_wait_then_release();
            waited = true;
          }
          const int st = n % C::STAGES;
          const bool ok = mbar_wait(empty0 + 8 * st, ((n / C::STAGES) & 1) ^ 1, abort_flag,
                                    status, budget);
          if (!ok) continue;
          const int p0 = lt * C::T;
          const int rows = min(C::T, seg.L - p0);
          uint8_t* stage = sm + st * C::STAGE_BYTES;
          mbar_arrive_expect_tx(full0 + 8 * st, static_cast<uint32_t>(rows) * (DK + DV) * C::ELT);
          bulk_load(smem_u32(stage), kc + (unit_row + p0) * DK,
                    static_cast<uint32_t>(rows) * DK * C::ELT, full0 + 8 * st);
          bulk_load(smem_u32(stage + C::K_BYTES), vc + (unit_row + p0) * DV,
                    static_cast<uint32_t>(rows) * DV * C::ELT, full0 + 8 * st);
          last_n[st] = static_cast<int>(n);
        }
      }
      if (!waited) pdl_wait_then_release();
      if (*abort_flag) {  // let copies in flight land before the CTA exits
        for (int s = 0; s < C::STAGES; ++s) {
          if (last_n[s] < 0) continue;
          const uint32_t par = (last_n[s] / C::STAGES) & 1;
          const long long t0 = clock64();
          while (!mbar_try_wait(full0 + 8 * s, par) && clock64() - t0 < budget) {
          }
        }
      }
    }
    __syncwarp();
  } else {
    // ---------------- compute (NCT threads) ----------------
    const int ct = threadIdx.x - 32;
    const int cw = ct >> 5;
    // logits mapping: lane ch of a row's LPR lanes holds chunks ch, ch + LPR, ...
    const int sub = lane / C::LPR, ch = lane % C::LPR;
    const int pg = ct / C::CHV, chv = lane % C::CHV;  // V-pass mapping
    float qreg[RMAX][C::CPL * C::EPC];
    float acc[RMAX][C::EPC];
#pragma unroll
    for (int t = 0; t < RMAX; ++t)
#pragma unroll
      for (int e = 0; e < C::EPC; ++e) acc[t][e] = 0.f;

    uint32_t n = 0;
    while (w.next(seg)) {
      // query row t = s * r + head: q / out row (i * n + s) * h + j * r + head
      const size_t obase = static_cast<size_t>(seg.i) * nq * h + seg.j * r;
      const size_t unit = static_cast<size_t>(seg.i) * g + seg.j;
      // fused append: the new tokens whose rows fall in this segment,
      // 16-byte chunks idx < nchunk; thread ct carries chunk ct from here
      const int first_new = seg.L - nq;
      int s_lo = 0, nrows = 0;
      if (k_new != nullptr) {
        const int p_lo = max(first_new, seg.lt0 * C::T), p_hi = min(seg.L, seg.lt1 * C::T);
        if (p_lo < p_hi) {
          s_lo = p_lo - first_new;
          nrows = p_hi - p_lo;
        }
      }
      // chunk idx of the new rows of a tensor with `cpr` chunks per row
      auto new_chunk = [&](int idx, int cpr) -> size_t {
        return ((static_cast<size_t>(seg.i) * nq + s_lo + idx / cpr) * g + seg.j) * cpr +
               idx % cpr;
      };
      uint4 knew = make_uint4(0u, 0u, 0u, 0u), vnew = knew;
      if (ct < nrows * C::CHK) knew = __ldg(k_new + new_chunk(ct, C::CHK));
      if (ct < nrows * C::CHV) vnew = __ldg(v_new + new_chunk(ct, C::CHV));
#pragma unroll
      for (int t = 0; t < RMAX; ++t) {
        if (t < nr) {
          const int s_ = t / r;
          const DT* qrow = q + (obase + s_ * h + (t - s_ * r)) * DK;
#pragma unroll
          for (int c = 0; c < C::CPL; ++c) {
            const uint4 u =
                *reinterpret_cast<const uint4*>(qrow + (ch + c * C::LPR) * C::EPC);
            Elt<DT>::unpack(u, &qreg[t][c * C::EPC]);
          }
        } else {
#pragma unroll
          for (int e = 0; e < C::CPL * C::EPC; ++e) qreg[t][e] = 0.f;
        }
      }
      for (int lt = seg.lt0; lt < seg.lt1; ++lt, ++n) {
        const int st = n % C::STAGES;
        const int valid = min(C::T, seg.L - lt * C::T);
        const bool ok = mbar_wait(full0 + 8 * st, (n / C::STAGES) & 1, abort_flag, status,
                                  budget);
        const DT* sK = reinterpret_cast<const DT*>(sm + st * C::STAGE_BYTES);
        const DT* sV = reinterpret_cast<const DT*>(sm + st * C::STAGE_BYTES + C::K_BYTES);
        if (nrows > 0 && (lt + 1) * C::T > first_new) {
          // rows L_i - n .. L_i - 1 are the new tokens: use k_new / v_new
          // there and store them into the cache (the append)
          auto cache_row = [&](int pos) -> long long {
            if (table == nullptr) return static_cast<long long>(unit) * cap + pos;
            const int e = __ldg(table + static_cast<size_t>(seg.i) * max_blocks + pos / bsz);
            return (e >= 0 && e < num_blocks)
                       ? (static_cast<long long>(e) * g + seg.j) * bsz + pos % bsz
                       : -1;
          };
          if (ok) {
            for (int idx = ct; idx < nrows * C::CHK; idx += kCompute) {
              const int pos = first_new + s_lo + idx / C::CHK, c16 = idx % C::CHK;
              if (pos < lt * C::T || pos >= (lt + 1) * C::T) continue;
              const uint4 kv = idx == ct ? knew : __ldg(k_new + new_chunk(idx, C::CHK));
              reinterpret_cast<uint4*>(const_cast<DT*>(sK) + (pos - lt * C::T) * DK)[c16] = kv;
              const long long crow = cache_row(pos);
              if (crow >= 0) k_cache_w[crow * C::CHK + c16] = kv;
            }
            for (int idx = ct; idx < nrows * C::CHV; idx += kCompute) {
              const int pos = first_new + s_lo + idx / C::CHV, c16 = idx % C::CHV;
              if (pos < lt * C::T || pos >= (lt + 1) * C::T) continue;
              const uint4 vv = idx == ct ? vnew : __ldg(v_new + new_chunk(idx, C::CHV));
              reinterpret_cast<uint4*>(const_cast<DT*>(sV) + (pos - lt * C::T) * DV)[c16] = vv;
              const long long crow = cache_row(pos);
              if (crow >= 0) v_cache_w[crow * C::CHV + c16] = vv;
            }
          }
          named_bar_sync(1, kCompute);
        }
        // A: logits (query rows past nr have q = 0 and are not stored)
        using RR = RowReduce<C::LPR, RMAX>;
        const int hd = RR::head(lane);
        const bool wr = RR::writer(lane) && hd < nr;
#pragma unroll
        for (int pb = cw * C::PPW; pb < C::T; pb += kWarps * C::PPW) {
          const int p = pb + sub;
          float kf[C::CPL * C::EPC];
          if (ok && p < valid) {
#pragma unroll
            for (int c = 0; c < C::CPL; ++c) {
              const uint4 u =
                  *reinterpret_cast<const uint4*>(sK + p * DK + (ch + c * C::LPR) * C::EPC);
              Elt<DT>::unpack(u, &kf[c * C::EPC]);
            }
          } else {
#pragma unroll
            for (int e = 0; e < C::CPL * C::EPC; ++e) kf[e] = 0.f;
          }
          float part[RMAX];
#pragma unroll
          for (int t = 0; t < RMAX; ++t) {
            part[t] = 0.f;
#pragma unroll
            for (int e = 0; e < C::CPL * C::EPC; ++e) part[t] = fmaf(qreg[t][e], kf[e], part[t]);
          }
          RR::run(part, lane);
          if (wr && p < valid) sP[hd * C::T + p] = part[0] * scale_log2;
        }
        named_bar_sync(1, kCompute);
        // B: online softmax, one half-warp per query row (two rows a warp,
        // the 16 lanes of a half taking T / 16 positions each); row t (token
        // s) sees tile positions p <= lim
        {
          const int hw = lane >> 4, hl = lane & 15;
          for (int tb = 2 * cw; tb < nr; tb += 2 * kWarps) {
            const int t = tb + hw;
            const bool row_ok = t < nr;  // (both halves run the shuffles)
            const int lim = row_ok ? min(valid - 1, first_new + t / r - lt * C::T) : -1;
            float x[C::T / 16];
            float mx = -INFINITY;
#pragma unroll
            for (int k = 0; k < C::T / 16; ++k) {
              const int p = hl + 16 * k;
              x[k] = (p <= lim) ? sP[t * C::T + p] : -INFINITY;
              mx = fmaxf(mx, x[k]);
            }
#pragma unroll
            for (int o = 8; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
            const float m_old = row_ok ? sM[t] : -INFINITY;
            const float m_new = fmaxf(m_old, mx);
            // a row that has seen no position yet keeps a finite reference
            const float mref = (m_new == -INFINITY) ? 0.f : m_new;
            const float alpha = ex2(m_old - mref);
            float sum = 0.f;
#pragma unroll
            for (int k = 0; k < C::T / 16; ++k) {
              const float pv = ex2(x[k] - mref);
              sum += pv;
              if (row_ok) sP[t * C::T + hl + 16 * k] = pv;
            }
#pragma unroll
            for (int o = 8; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
            __syncwarp();
            if (hl == 0 && row_ok) {
              sM[t] = m_new;
              sL[t] = sL[t] * alpha + sum;
              sA[t] = alpha;
            }
          }
        }
        named_bar_sync(1, kCompute);
        // C: weighted sum of V (the accumulators are rescaled only when
        // some row's running max moved: the same branch in every thread)
        {
          float al[RMAX];
          bool moved = false;
#pragma unroll
          for (int t = 0; t < RMAX; ++t) {
            al[t] = t < nr ? sA[t] : 1.f;
            moved |= al[t] != 1.f;
          }
          if (moved) {
#pragma unroll
            for (int t = 0; t < RMAX; ++t)
#pragma unroll
              for (int e = 0; e < C::EPC; ++e) acc[t][e] *= al[t];
          }
        }
        // positions in pairs (one 8-byte load of a row's two weights); the
        // weight of a position past the valid rows is 0 (phase B), and its V
        // row is taken as 0 rather than read
        if (ok) {
          for (int p = 2 * pg; p < valid; p += 2 * C::NPG) {
            float v0[C::EPC], v1[C::EPC];
            Elt<DT>::unpack(*reinterpret_cast<const uint4*>(sV + p * DV + chv * C::EPC), v0);
            if (p + 1 < valid) {
              Elt<DT>::unpack(
                  *reinterpret_cast<const uint4*>(sV + (p + 1) * DV + chv * C::EPC), v1);
            } else {
#pragma unroll
              for (int e = 0; e < C::EPC; ++e) v1[e] = 0.f;
            }
#pragma unroll
            for (int t = 0; t < RMAX; ++t) {
              if (t < nr) {
                const float2 wgt = *reinterpret_cast<const float2*>(sP + t * C::T + p);
#pragma unroll
                for (int e = 0; e < C::EPC; ++e) {
                  acc[t][e] = fmaf(wgt.x, v0[e], acc[t][e]);
                  acc[t][e] = fmaf(wgt.y, v1[e], acc[t][e]);
                }
              }
            }
          }
        }
        named_bar_sync(1, kCompute);
        if (ct == 0) mbar_arrive(empty0 + 8 * st);
      }

      // ---- segment end: reduce the position groups, write out: each
      // warp's groups by shuffles, then the warps four at a time into four
      // slots ----
#pragma unroll
      for (int t = 0; t < RMAX; ++t) {
#pragma unroll
        for (int e = 0; e < C::EPC; ++e) {
          float v = acc[t][e];
#pragma unroll
          for (int o = C::CHV; o < 32; o <<= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
          acc[t][e] = v;
        }
      }
      // (warps NSLOT k .. NSLOT k + NSLOT - 1 add into the slots in pass k)
      constexpr int NS = C::NSLOT;
#pragma unroll
      for (int pass = 0; pass * NS < kWarps; ++pass) {
        if (cw / NS == pass && lane < C::CHV) {
#pragma unroll
          for (int t = 0; t < RMAX; ++t)
            if (t < nr)
#pragma unroll
              for (int e = 0; e < C::EPC; ++e) {
                float* dst = sRed + ((cw % NS) * RMAX + t) * DV + chv * C::EPC + e;
                *dst = pass == 0 ? acc[t][e] : *dst + acc[t][e];
              }
        }
        if (pass * NS + NS < kWarps) named_bar_sync(1, kCompute);
      }
      // the slots' sum for row t, column dd
      auto red_sum = [&](int t, int dd) {
        float o = sRed[t * DV + dd];
#pragma unroll
        for (int sl = 1; sl < NS; ++sl) o += sRed[(sl * RMAX + t) * DV + dd];
        return o;
      };
#pragma unroll
      for (int t = 0; t < RMAX; ++t)
#pragma unroll
        for (int e = 0; e < C::EPC; ++e) acc[t][e] = 0.f;
      named_bar_sync(1, kCompute);
      const bool whole = (seg.lt0 == 0 && seg.lt1 == seg.ti);
      const int u = seg.i * g + seg.j;
      const size_t slot = static_cast<size_t>(u) + blockIdx.x;
      auto out_row = [&](int t) -> size_t {
        const int s_ = t / r;
        return obase + s_ * h + (t - s_ * r);
      };
      for (int idx = ct; idx < nr * DV; idx += kCompute) {
        const int t = idx / DV, dd = idx % DV;
        const float o = red_sum(t, dd);
        if (whole) {
          Elt<DT>::store(out + out_row(t) * DV + dd, o / sL[t]);
        } else {
          // (a row that saw none of this CTA's positions has max -inf, sum 0)
          part_o[(slot * nr + t) * DV + dd] = o;
          if (dd == 0) {
            part_ml[(slot * nr + t) * 2 + 0] = sM[t];
            part_ml[(slot * nr + t) * 2 + 1] = sL[t];
          }
        }
      }
      if (!whole) {
        // the unit is split across CTAs: the last one to finish merges
        long long c0, c1;
        unit_ctas(seg.u0, seg.u0 + seg.ti, w.W, w.nc, c0, c1);
        const int np = unit_parts(c0, c1, w.W, w.nc);
        if (counters != nullptr &&
            arrive_last(counters, u, np, last_flag, ct == 0, 1, kCompute)) {
          // merge the partials in CTA order whichever CTA merges (the same
          // bits every run): this CTA's own (still in shared memory) is used
          // in place only when it is the first piece, else read back
          long long cfirst = c0;
          if (w.W < w.nc)
            while (cfirst < c1 && cta_empty(cfirst, w.W, w.nc)) ++cfirst;
          const bool own_first = cfirst == blockIdx.x;
          for (int idx = ct; idx < nr * DV; idx += kCompute) {
            const int t = idx / DV, dd = idx % DV;
            float o = 0.f, M = -INFINITY, den = 0.f;
            if (own_first) {
              o = red_sum(t, dd);
              M = sM[t];
              den = sL[t];
            }
            for (long long c = c0; c <= c1; ++c) {
              if ((own_first && c == blockIdx.x) || (w.W < w.nc && cta_empty(c, w.W, w.nc)))
                continue;
              const long long sl = (u + c) * nr + t;
              const float mc = __ldcg(part_ml + sl * 2), lc = __ldcg(part_ml + sl * 2 + 1);
              const float oc = __ldcg(part_o + sl * DV + dd);
              const float mn = fmaxf(M, mc);
              const float mr = (mn == -INFINITY) ? 0.f : mn;  // both pieces empty
              const float sa = ex2(M - mr), sb = ex2(mc - mr);
              o = o * sa + oc * sb;
              den = den * sa + lc * sb;
              M = mn;
            }
            Elt<DT>::store(out + out_row(t) * DV + dd, o / den);
          }
        }
      }
      named_bar_sync(1, kCompute);
      if (ct < RMAX) {
        sM[ct] = -INFINITY;
        sL[ct] = 0.f;
        sA[ct] = 0.f;
      }
      named_bar_sync(1, kCompute);
    }
  }
  __syncthreads();
}

template <typename DT, int DK, int DV, int RMAX>
cudaError_t launch_t(const DecodeLaunch& a) {
  using C = SimtCfg<DT, DK, DV, RMAX>;
  auto kern = decode_simt_kernel<DT, DK, DV, RMAX>;
  // the shared-memory opt-in is set once per device (not during a capture)
  static std::atomic<unsigned long long> configured{0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!(configured.load() & (1ull << dev))) {
    const cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    configured.fetch_or(1ull << dev);
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.nc);
  cfg.blockDim = dim3(C::THREADS);
  cfg.dynamicSmemBytes = C::SMEM;
  cfg.stream = a.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(
      &cfg, kern, static_cast<const DT*>(a.q), static_cast<const DT*>(a.k_cache),
      static_cast<const DT*>(a.v_cache), a.seq_lens, a.b, a.h, a.g, a.cap, a.scale_log2,
      static_cast<DT*>(a.out), a.part_o, a.part_ml, a.counters,
      static_cast<const uint4*>(a.k_new), static_cast<const uint4*>(a.v_new),
      static_cast<uint4*>(a.k_cache_w), static_cast<uint4*>(a.v_cache_w), a.status, a.budget,
      a.nq, a.block_table, a.block_size, a.max_blocks, a.num_blocks, a.early ? 1 : 0);
}

}  // namespace

bool simt_supported(int dtype, int d_k, int d_v, int cols) {
  const bool dims = (d_k == 64 || d_k == 128) && (d_v == 64 || d_v == 128);
  if (dtype == GQA_F32) return dims && cols >= 1 && cols <= 16;
  if (dtype == GQA_BF16 || dtype == GQA_F16) return dims && cols >= 1 && cols <= 8;
  return false;
}

int simt_tile(int dtype, int d_k, int d_v) {
  // (the kernel's SimtCfg::T: K + V of a tile take 64 KiB in fp32, 32 KiB otherwise)
  const int elt = dtype == GQA_F32 ? 4 : 2;
  return (dtype == GQA_F32 ? 32768 : 16384) / ((d_k > d_v ? d_k : d_v) * elt);
}

int simt_ctas_per_sm(int, int, int) { return 1; }

template <typename DT, int DK, int DV>
cudaError_t launch_dims(const DecodeLaunch& a, int r) {
  if constexpr (sizeof(DT) == 4) {
    if (r > 8) return launch_t<DT, DK, DV, 16>(a);
  }
  return launch_t<DT, DK, DV, 8>(a);
}

template <typename DT>
cudaError_t launch_dtype(const DecodeLaunch& a, int r) {
  if (a.d == 64) return a.dv == 64 ? launch_dims<DT, 64, 64>(a, r) : launch_dims<DT, 64, 128>(a, r);
  return a.dv == 64 ? launch_dims<DT, 128, 64>(a, r) : launch_dims<DT, 128, 128>(a, r);
}

cudaError_t launch_decode_simt(const DecodeLaunch& a) {
  const int r = a.nq * (a.h / a.g);  // query rows per KV head
  if (a.dtype == GQA_F32) return launch_dtype<float>(a, r);
  if (a.dtype == GQA_F16) return launch_dtype<__half>(a, r);
  return launch_dtype<__nv_bfloat16>(a, r);
}

}  // namespace gqa
