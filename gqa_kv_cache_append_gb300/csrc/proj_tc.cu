// proj_tc.cu - the projections around the decode step, on the tcgen05 tensor
// cores (MQA review §2.4 MultiheadSelfAttentionIncremental and §3
// MultiquerySelfAttentionIncremental):
//
//   q     = "bd,hdk->bhk"(x, P_q)     k_new = "bd,gdk->bgk"(x, P_k)
//   v_new = "bd,gdv->bgv"(x, P_v)     y     = "bhv,hdv->bd"(o, P_o)
//
// Each is a skinny GEMM (the batch b is small, the weights large), so it is
// computed transposed: out^T [M = output features x N = batch] = W [M x K] .
// X^T, with the weights on the MMA's M axis (128 features per tile) and the
// batch padded to NB columns.  Every weight byte is streamed from HBM once,
// by TMA, through a shared-memory ring; x (or o) is read per stage as the B
// operand.  Weight layouts are those of the pages: P_q / P_k / P_v
// [heads, D, 128] give a tile [128 features x 128 rows of D] that is MN-major
// (features contiguous), P_o [h, D, 128] gives [128 rows of D x 128 of v],
// K-major.
//
// Work split: the tiles' K chunks (128 deep) are laid end to end and each
// persistent CTA takes an equal contiguous share, so every SM streams the
// same number of weight bytes (a tile may be cut between CTAs).  A CTA's
// piece of a tile accumulates in tensor memory; a tile held whole is written
// directly, a cut tile writes fp32 partials and the CTA that finishes the
// tile last sums all pieces in CTA order (deterministic) and writes it.
//
// Roles (192 threads, one CTA per SM): warp 0 TMA producer, warp 1 tensor
// memory owner and MMA issuer (accumulators double-buffered across
// segments), warps 2-5 epilogue (thread x owns TMEM lane x = output feature
// x of the tile).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <atomic>

#include "gqa_device.cuh"
#include "gqa_internal.h"

namespace gqa {
namespace {

constexpr int kM = 128;                  // output features per tile
constexpr int kKc = 128;                 // reduction depth per chunk
constexpr int kBox = 128 * 64 * 2;       // one [128 rows x 64 cols] bf16 box
constexpr int kPrefetchChunks = 8;       // weight chunks sent to L2 ahead of the ring

template <int NB>
struct PCfg {
  static constexpr int A_BYTES = 2 * kBox;       // weight chunk [128 x 128]
  static constexpr int B_BYTES = 2 * NB * 128;   // activation chunk [NB x 128]
  static constexpr int STAGE = A_BYTES + B_BYTES;
  static constexpr int STAGES = NB <= 32 ? 5 : (NB <= 64 ? 4 : 3);
  static constexpr int OFF_BAR = STAGES * STAGE;
  static constexpr int NBAR = 2 * STAGES + 2 + 2 + 1;  // full, empty, acc full/free, drain
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int SMEM = OFF_MISC + 16;
  static constexpr int NCOLS = 2 * NB;                 // two accumulators
  static_assert(STAGE % 1024 == 0, "stages keep the 1024-byte swizzle alignment");
  static_assert(SMEM <= 232448, "shared memory budget");
  static_assert(NCOLS >= 32 && NCOLS <= 256 && (NCOLS & (NCOLS - 1)) == 0, "TMEM columns");
};

// tile t of a QKV launch: head a of the concatenated [P_q; P_k; P_v]
struct QkvHead {
  int which;  // 0 q, 1 k, 2 v
  int head;   // head within its tensor
};

__device__ __forceinline__ QkvHead qkv_head(int t, int h, int g) {
  if (t < h) return {0, t};
  if (t < h + g) return {1, t - h};
  return {2, t - h - g};
}

// MODE 0: q/k/v projection (weights MN-major, three tensors);
// MODE 1: output projection (weights K-major, one tensor).
template <int NB, int MODE>
__global__ void __launch_bounds__(192, 1)
    proj_tc_kernel(const __grid_constant__ CUtensorMap tm_w0,
                   const __grid_constant__ CUtensorMap tm_w1,
                   const __grid_constant__ CUtensorMap tm_w2,
                   const __grid_constant__ CUtensorMap tm_x, int b, int D, int h, int g,
                   int tiles, int chunks, __nv_bfloat16* __restrict__ out0,
                   __nv_bfloat16* __restrict__ out1, __nv_bfloat16* __restrict__ out2,
                   float* __restrict__ part, int* __restrict__ counters,
                   unsigned int* status, long long budget, int early) {
  using C = PCfg<NB>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* sm = smem_raw;
  const uint32_t s_base = smem_u32(sm);
  if (s_base & 1023u) {
    if (threadIdx.x == 0) atomicOr(status, GQA_DEV_INTERNAL);
    return;
  }
  const uint32_t bar0 = s_base + C::OFF_BAR;
  auto FULL = [&](int s) -> uint32_t { return bar0 + 8u * s; };
  auto EMPTY = [&](int s) -> uint32_t { return bar0 + 8u * (C::STAGES + s); };
  auto ACC_FULL = [&](int k) -> uint32_t { return bar0 + 8u * (2 * C::STAGES + k); };
  auto ACC_FREE = [&](int k) -> uint32_t { return bar0 + 8u * (2 * C::STAGES + 2 + k); };
  const uint32_t DRAIN = bar0 + 8u * (2 * C::STAGES + 4);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + C::OFF_MISC + 4);
  int* last_flag = reinterpret_cast<int*>(sm + C::OFF_MISC + 8);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  pdl_launch_dependents();
  if (threadIdx.x == 0) {
    for (int k = 0; k < C::NBAR; ++k) {
      const bool per_warp = k >= 2 * C::STAGES + 2 && k < 2 * C::STAGES + 4;  // acc free
      mbar_init(bar0 + 8u * k, per_warp ? 4u : 1u);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tm_w0);
    if (MODE == 0) {
      prefetch_tmap(&tm_w1);
      prefetch_tmap(&tm_w2);
    }
    prefetch_tmap(&tm_x);
  }
  if (warp == 1) tmem_alloc(smem_u32(tmem_slot), C::NCOLS);
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // The weights may be streamed before the dependency wait when the caller
  // allows it (`early`: no kernel ahead on the stream writes them); the
  // activations, the outputs and the workspace only after it.
  if (!early || warp != 0) pdl_wait();

  const long long W = static_cast<long long>(tiles) * chunks;
  const int nc = gridDim.x;
  const long long pos0 = W * blockIdx.x / nc, pos1 = W * (blockIdx.x + 1) / nc;

  if (warp == 0) {
    // ============================ producer ============================
    if (lane == 0) {
      const uint64_t pol_stream = policy_evict_first();
      const uint64_t pol_keep = policy_evict_last();
      bool waited = !early;
      int last_n[C::STAGES];
#pragma unroll
      for (int s = 0; s < C::STAGES; ++s) last_n[s] = -1;
      int n = 0;
      for (long long p = pos0; p < pos1; ++p, ++n) {
        const int t = static_cast<int>(p / chunks), c = static_cast<int>(p % chunks);
        const int st = n % C::STAGES;
        if (!mbar_wait(EMPTY(st), ((n / C::STAGES) & 1) ^ 1, abort_flag, status, budget))
          continue;
        const uint32_t dst = s_base + st * C::STAGE;
        mbar_arrive_expect_tx(FULL(st), C::STAGE);
        const CUtensorMap* wm = &tm_w0;
        int row;
        if (MODE == 0) {
          const QkvHead hd = qkv_head(t, h, g);
          wm = hd.which == 0 ? &tm_w0 : (hd.which == 1 ? &tm_w1 : &tm_w2);
          row = hd.head * D + c * kKc;  // rows of D, features in the columns
        } else {
          row = c * D + t * kM;         // head c, output rows t * 128 ..
        }
        tma_load_2d(dst, wm, FULL(st), 0, row, pol_stream);
        tma_load_2d(dst + kBox, wm, FULL(st), 64, row, pol_stream);
        if (!waited && n + 1 >= C::STAGES) {
          // before waiting, have L2 fetch the weights of the next chunks as
          // well, so HBM stays busy while the kernel ahead finishes
          for (long long pf = p + 1; pf < pos1 && pf <= p + kPrefetchChunks; ++pf) {
            const int tf = static_cast<int>(pf / chunks), cf = static_cast<int>(pf % chunks);
            const CUtensorMap* wf = &tm_w0;
            int rf;
            if (MODE == 0) {
              const QkvHead hd = qkv_head(tf, h, g);
              wf = hd.which == 0 ? &tm_w0 : (hd.which == 1 ? &tm_w1 : &tm_w2);
              rf = hd.head * D + cf * kKc;
            } else {
              rf = cf * D + tf * kM;
            }
            tma_prefetch_l2_2d(wf, 0, rf);
            tma_prefetch_l2_2d(wf, 64, rf);
          }
          // the activations of the stages issued so far, after the wait
          pdl_wait();
          waited = true;
          for (int m = 0; m <= n && !*abort_flag; ++m) {
            const int cm = static_cast<int>((pos0 + m) % chunks);
            const uint32_t dm = s_base + (m % C::STAGES) * C::STAGE + C::A_BYTES;
            tma_load_2d(dm, &tm_x, FULL(m % C::STAGES), cm * kKc, 0, pol_keep);
            tma_load_2d(dm + NB * 128, &tm_x, FULL(m % C::STAGES), cm * kKc + 64, 0, pol_keep);
          }
        } else if (waited) {
          tma_load_2d(dst + C::A_BYTES, &tm_x, FULL(st), c * kKc, 0, pol_keep);
          tma_load_2d(dst + C::A_BYTES + NB * 128, &tm_x, FULL(st), c * kKc + 64, 0, pol_keep);
        }
        last_n[st] = n;
      }
      if (!waited) {  // a range shorter than the ring
        pdl_wait();
        waited = true;
        for (int m = 0; m < n && !*abort_flag; ++m) {
          const int cm = static_cast<int>((pos0 + m) % chunks);
          const uint32_t dm = s_base + (m % C::STAGES) * C::STAGE + C::A_BYTES;
          tma_load_2d(dm, &tm_x, FULL(m % C::STAGES), cm * kKc, 0, pol_keep);
          tma_load_2d(dm + NB * 128, &tm_x, FULL(m % C::STAGES), cm * kKc + 64, 0, pol_keep);
        }
      }
      if (*abort_flag) {  // copies in flight land before the CTA exits
        for (int s = 0; s < C::STAGES; ++s) {
          if (last_n[s] < 0) continue;
          const long long t0 = clock64();
          while (!mbar_try_wait(FULL(s), (last_n[s] / C::STAGES) & 1) &&
                 clock64() - t0 < budget) {
          }
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ============================ MMA issuer ============================
    constexpr uint32_t IDESC = idesc_bf16(kM, NB, MODE == 0 ? 1 : 0, 0);
    int n = 0, sgi = 0;
    for (long long p = pos0; p < pos1; ++sgi) {
      const int t = static_cast<int>(p / chunks);
      const long long pend = ((static_cast<long long>(t) + 1) * chunks < pos1)
                                 ? (static_cast<long long>(t) + 1) * chunks
                                 : pos1;
      const int ab = sgi & 1;
      const uint32_t acc = tmem + ab * NB;
      bool ok = mbar_wait(ACC_FREE(ab), ((sgi >> 1) & 1) ^ 1, abort_flag, status, budget);
      ok = __all_sync(0xffffffffu, ok);
      tc_fence_after();
      for (long long q = p; q < pend; ++q, ++n) {
        const int st = n % C::STAGES;
        bool okk = ok && mbar_wait(FULL(st), (n / C::STAGES) & 1, abort_flag, status, budget);
        okk = __all_sync(0xffffffffu, okk);
        tc_fence_after();
        if (lane == 0) {
          if (okk) {
            const uint32_t a_base = s_base + st * C::STAGE;
            const uint32_t b_base = a_base + C::A_BYTES;
#pragma unroll
            for (int kk = 0; kk < kKc / 16; ++kk) {
              uint64_t ad;
              if (MODE == 0) {
                // A = W^T of rows of D (MN-major): M = 128 features (two
                // 64-column boxes, kBox apart), K = 16 rows (two 8-row groups)
                ad = smem_desc(a_base + kk * 2048, kBox, 1024, SWZ_128B);
              } else {
                // A = 128 rows of D x 16 of v (K-major), steps 0-3 in the
                // first 64-column box
                ad = smem_desc(a_base + (kk >> 2) * kBox + (kk & 3) * 32, 16, 1024, SWZ_128B);
              }
              const uint64_t bd =
                  smem_desc(b_base + (kk >> 2) * (NB * 128) + (kk & 3) * 32, 16, 1024, SWZ_128B);
              mma_bf16(acc, ad, bd, IDESC, (q > p || kk > 0) ? 1u : 0u);
            }
          }
          mma_commit(EMPTY(st));
        }
        __syncwarp();
      }
      if (lane == 0) mma_commit(ACC_FULL(ab));
      __syncwarp();
      p = pend;
    }
    if (lane == 0) {
      mma_commit(DRAIN);
      const long long t0 = clock64();
      while (!mbar_try_wait(DRAIN, 0) && clock64() - t0 < budget) {
      }
    }
    __syncwarp();
  } else {
    // ============================= epilogue =============================
    const int qd = warp & 3;                 // TMEM lane quarter of this warp
    const int row = qd * 32 + lane;          // output feature within the tile
    const uint32_t lane_off = static_cast<uint32_t>(qd * 32) << 16;
    int sgi = 0;
    for (long long p = pos0; p < pos1; ++sgi) {
      const int t = static_cast<int>(p / chunks);
      const long long tile0 = static_cast<long long>(t) * chunks, tile1 = tile0 + chunks;
      const long long pend = tile1 < pos1 ? tile1 : pos1;
      const bool whole = (p == tile0 && pend == tile1);
      const int ab = sgi & 1;
      const bool ok = mbar_wait(ACC_FULL(ab), (sgi >> 1) & 1, abort_flag, status, budget);
      // destination of column n of this tile's row: element offset and pitch
      __nv_bfloat16* dst;
      size_t pitch;
      if (MODE == 0) {
        const QkvHead hd = qkv_head(t, h, g);
        dst = hd.which == 0 ? out0 : (hd.which == 1 ? out1 : out2);
        const int heads = hd.which == 0 ? h : g;
        dst += static_cast<size_t>(hd.head) * kM + row;
        pitch = static_cast<size_t>(heads) * kM;
      } else {
        dst = out0 + static_cast<size_t>(t) * kM + row;
        pitch = static_cast<size_t>(D);
      }
      // partials are [slot][feature][NB]: each thread's columns contiguous
      float* mine = part + ((static_cast<size_t>(t) + blockIdx.x) * kM + row) * NB;
#pragma unroll
      for (int c16 = 0; c16 < NB / 16; ++c16) {
        float v[16];
        if (ok) {
          tmem_ld16(tmem + lane_off + ab * NB + c16 * 16, v);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int e = 0; e < 16; ++e) v[e] = 0.f;
        }
        if (whole) {
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const int col = c16 * 16 + e;
            if (col < b) dst[col * pitch] = __float2bfloat16_rn(v[e]);
          }
        } else {
#pragma unroll
          for (int e = 0; e < 16; e += 4)
            *reinterpret_cast<float4*>(mine + c16 * 16 + e) =
                make_float4(v[e], v[e + 1], v[e + 2], v[e + 3]);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(ACC_FREE(ab));
      if (!whole) {
        long long c0, c1;
        unit_ctas(tile0, tile1, W, nc, c0, c1);
        const int np = static_cast<int>(c1 - c0 + 1);
        if (arrive_last(counters, t, np, last_flag, row == 0, 1, 128)) {
          // every piece, this CTA's included, summed in CTA order; the
          // loads of PB pieces x HC columns (16 or 32 float4) go out together
          constexpr int HC = NB < 64 ? NB : 64;
          constexpr int PB = HC >= 64 ? 1 : 128 / HC;
          for (int c_lo = 0; c_lo < NB && c_lo < b; c_lo += HC) {
            float acc[HC];
#pragma unroll
            for (int e = 0; e < HC; ++e) acc[e] = 0.f;
            for (long long cb = c0; cb <= c1; cb += PB) {
              float4 w4[PB][HC / 4];
#pragma unroll
              for (int k = 0; k < PB; ++k) {
                const float4* src = reinterpret_cast<const float4*>(
                    part + ((static_cast<size_t>(t) + cb + k) * kM + row) * NB + c_lo);
#pragma unroll
                for (int e = 0; e < HC / 4; ++e)
                  w4[k][e] = (cb + k <= c1) ? __ldcg(src + e) : make_float4(0.f, 0.f, 0.f, 0.f);
              }
#pragma unroll
              for (int k = 0; k < PB; ++k) {
#pragma unroll
                for (int e = 0; e < HC / 4; ++e) {
                  acc[4 * e] += w4[k][e].x;
                  acc[4 * e + 1] += w4[k][e].y;
                  acc[4 * e + 2] += w4[k][e].z;
                  acc[4 * e + 3] += w4[k][e].w;
                }
              }
            }
#pragma unroll
            for (int e = 0; e < HC; ++e)
              if (c_lo + e < b) dst[(c_lo + e) * pitch] = __float2bfloat16_rn(acc[e]);
          }
        }
      }
      p = pend;
    }
  }

  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::NCOLS);
  }
}

template <int NB, int MODE>
cudaError_t launch_nb(const ProjLaunch& a) {
  using C = PCfg<NB>;
  CUtensorMap m0, m1, m2, mx;
  const uint32_t wbox[2] = {64u, 128u};
  const uint64_t wstr[1] = {static_cast<uint64_t>(kKc) * 2};
  if (MODE == 0) {
    const uint64_t dq[2] = {128u, static_cast<uint64_t>(a.h) * a.D};
    const uint64_t dk[2] = {128u, static_cast<uint64_t>(a.g) * a.D};
    if (!encode_bf16_map(&m0, a.w0, 2, dq, wstr, wbox) ||
        !encode_bf16_map(&m1, a.w1, 2, dk, wstr, wbox) ||
        !encode_bf16_map(&m2, a.w2, 2, dk, wstr, wbox))
      return cudaErrorInvalidValue;
  } else {
    const uint64_t dw[2] = {128u, static_cast<uint64_t>(a.h) * a.D};
    if (!encode_bf16_map(&m0, a.w0, 2, dw, wstr, wbox)) return cudaErrorInvalidValue;
    m1 = m0;
    m2 = m0;
  }
  // activations [b rows x K] (x: K = D; o: K = h * 128), box [NB rows x 64]
  const uint64_t kdim = MODE == 0 ? static_cast<uint64_t>(a.D) : static_cast<uint64_t>(a.h) * 128;
  const uint64_t dx[2] = {kdim, static_cast<uint64_t>(a.b)};
  const uint64_t sx[1] = {kdim * 2};
  const uint32_t xbox[2] = {64u, static_cast<uint32_t>(NB)};
  if (!encode_bf16_map(&mx, a.x, 2, dx, sx, xbox)) return cudaErrorInvalidValue;

  auto kern = proj_tc_kernel<NB, MODE>;
  static std::atomic<unsigned long long> configured{0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!(configured.load() & (1ull << dev))) {
    const cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    configured.fetch_or(1ull << dev);
  }
  const int tiles = MODE == 0 ? a.h + 2 * a.g : a.D / kM;
  const int chunks = MODE == 0 ? a.D / kKc : a.h;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.nc);
  cfg.blockDim = dim3(192);
  cfg.dynamicSmemBytes = C::SMEM;
  cfg.stream = a.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, m0, m1, m2, mx, a.b, a.D, a.h, a.g, tiles, chunks,
                            static_cast<__nv_bfloat16*>(a.out0),
                            static_cast<__nv_bfloat16*>(a.out1),
                            static_cast<__nv_bfloat16*>(a.out2), a.part, a.counters, a.status,
                            a.budget, a.early ? 1 : 0);
}

template <int MODE>
cudaError_t launch_mode(const ProjLaunch& a) {
  if (a.b <= 32) return launch_nb<32, MODE>(a);
  if (a.b <= 64) return launch_nb<64, MODE>(a);
  return launch_nb<128, MODE>(a);
}

}  // namespace

int proj_nb(int b) { return b <= 32 ? 32 : (b <= 64 ? 64 : 128); }

long long proj_work(int mode, int D, int h, int g) {
  return mode == 0 ? static_cast<long long>(h + 2 * g) * (D / kKc)
                   : static_cast<long long>(D / kM) * h;
}

int proj_tiles(int mode, int D, int h, int g) { return mode == 0 ? h + 2 * g : D / kM; }

cudaError_t launch_proj(const ProjLaunch& a) {
  return a.mode == 0 ? launch_mode<0>(a) : launch_mode<1>(a);
}

}  // namespace gqa
