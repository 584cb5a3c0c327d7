// gqa_api.cu - the C ABI of libgqa.so (declared in include/gqa.h): argument
// checks, kernel selection, the split workspace, the device status word, and
// the small kernels (KV append, wait self-test).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <type_traits>
#include <atomic>
#include <map>
#include <mutex>
#include <utility>

#include "../../include/gqa.h"
#include "gqa_device.cuh"
#include "gqa_internal.h"

namespace gqa {

// One status word per device (each device holds its own copy of the module).
__device__ unsigned int g_status_word;

namespace {

constexpr long long kWaitBudget = 1ll << 31;  // ~1 s of SM cycles per wait

// ---------------------------------------------------------------------------
// KV append: one thread per 16-byte chunk of the new rows.
// The concat of the new K/V rows on the position axis (MQA review §2.4, §3),
// done in place at rows L_i - n .. L_i - 1 (decode notes: kCache.push,
// vCache.push; n = 1 for one token per step).
// ---------------------------------------------------------------------------
__global__ void kv_append_kernel(const uint4* __restrict__ k_new, const uint4* __restrict__ v_new,
                                 uint4* __restrict__ k_cache, uint4* __restrict__ v_cache,
                                 const int* __restrict__ lens, int b, int nq, int g, int ck,
                                 int cv, int cap, unsigned int* status) {
  const long long per = ck + cv;
  const long long total = static_cast<long long>(b) * nq * g * per;
  const long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= total) return;
  const long long row = idx / per;  // (i, s, j) row of k_new / v_new
  const int c = static_cast<int>(idx % per);
  const int j = static_cast<int>(row % g);
  const int s = static_cast<int>((row / g) % nq);
  const int i = static_cast<int>(row / (static_cast<long long>(g) * nq));
  const int L = __ldg(lens + i);
  if (L < 1 || L < nq || L > cap) {
    if (c == 0) atomicOr(status, GQA_DEV_BAD_SEQ_LEN);
    return;
  }
  const long long dst_row = (static_cast<long long>(i) * g + j) * cap + (L - nq + s);
  if (c < ck) {
    k_cache[dst_row * ck + c] = __ldg(k_new + row * ck + c);
  } else {
    const int cc = c - ck;
    v_cache[dst_row * cv + cc] = __ldg(v_new + row * cv + cc);
  }
}

// The same for a paged cache: position L_i - 1 lives in row (L_i - 1) % B of
// block block_table[i, (L_i - 1) / B] of the pools [num_blocks, g, B, d].
__global__ void kv_append_paged_kernel(const uint4* __restrict__ k_new,
                                       const uint4* __restrict__ v_new, uint4* __restrict__ k_pool,
                                       uint4* __restrict__ v_pool, const int* __restrict__ table,
                                       const int* __restrict__ lens, int b, int nq, int g, int ck,
                                       int cv, int bsz, int max_blocks, int num_blocks,
                                       unsigned int* status) {
  const long long per = ck + cv;
  const long long total = static_cast<long long>(b) * nq * g * per;
  const long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= total) return;
  const long long row = idx / per;  // (i, s, j) row of k_new / v_new
  const int c = static_cast<int>(idx % per);
  const int j = static_cast<int>(row % g);
  const int s = static_cast<int>((row / g) % nq);
  const int i = static_cast<int>(row / (static_cast<long long>(g) * nq));
  const int L = __ldg(lens + i);
  if (L < 1 || L < nq || L > static_cast<long long>(max_blocks) * bsz) {
    if (c == 0) atomicOr(status, GQA_DEV_BAD_SEQ_LEN);
    return;
  }
  const int p = L - nq + s;  // this row's position
  const int blk = __ldg(table + static_cast<size_t>(i) * max_blocks + p / bsz);
  if (blk < 0 || blk >= num_blocks) {
    if (c == 0) atomicOr(status, GQA_DEV_BAD_BLOCK);
    return;
  }
  const long long dst_row = (static_cast<long long>(blk) * g + j) * bsz + p % bsz;
  if (c < ck) {
    k_pool[dst_row * ck + c] = __ldg(k_new + row * ck + c);
  } else {
    const int cc = c - ck;
    v_pool[dst_row * cv + cc] = __ldg(v_new + row * cv + cc);
  }
}

// ---------------------------------------------------------------------------
// Log-sum-exp combine for launches with many more CTAs than units (a few
// long sequences, e.g. one MQA head over 131k positions spread over 19
// CTAs): the decode kernel then only writes partials, and this kernel merges
// them with the whole GPU, one CTA per (unit, query row).  Its four warps
// take every fourth piece each (the loads of all pieces go out at once),
// each lane holding CPL = d / 32 consecutive output columns; the warps'
// results are merged in shared memory in warp order.  Query row t = s * r +
// head of a unit is head j * r + head of new token s.  With per-CTA maxima
// m_c (base 2), sums l_c and unnormalised outputs O_c of the same softmax
// over disjoint position ranges:
//     M = max_c m_c,  out = sum_c 2^(m_c - M) O_c / sum_c 2^(m_c - M) l_c.
// Units held whole by one CTA were written by the decode kernel.
// ---------------------------------------------------------------------------
constexpr int kCombineWarps = 4;

template <typename DT, int CPL>
__global__ void __launch_bounds__(32 * kCombineWarps)
    combine_kernel(const int* __restrict__ lens, int b, int h, int g, int cap, int tile, int nc,
                   int nq, const float* __restrict__ part_o, const float* __restrict__ part_ml,
                   DT* __restrict__ out) {
  constexpr int d = 32 * CPL;
  __shared__ float s_m[kCombineWarps], s_l[kCombineWarps];
  __shared__ float s_o[kCombineWarps][d];
  pdl_launch_dependents();
  const int r = h / g;
  const int nr = nq * r;
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int u = blockIdx.x / nr, t = blockIdx.x % nr;
  const int i = u / g, j = u % g;
  // the unit's tile range (warp-cooperative scan of the lengths, every warp)
  long long before = 0, all = 0;
  int ti = 0;
  for (int base = 0; base < b; base += 32) {
    const int idx = base + lane;
    const int tt = (idx < b) ? seq_tiles(__ldg(lens + idx), nq, cap, tile) : 0;
    all += tt;
    if (idx < i) before += tt;
    if (idx == i) ti = tt;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    all += __shfl_xor_sync(0xffffffffu, all, o);
    before += __shfl_xor_sync(0xffffffffu, before, o);
    ti += __shfl_xor_sync(0xffffffffu, ti, o);
  }
  if (ti == 0) return;  // (uniform across the CTA)
  const long long W = all * g;
  const long long u0 = before * g + static_cast<long long>(j) * ti;
  long long c0, c1;
  unit_ctas(u0, u0 + ti, W, nc, c0, c1);
  if (c0 == c1) return;
  // the lengths were read before the wait: the decode kernel releases this
  // launch only after the kernel ahead of it (which may write seq_lens) has
  // completed.  The partials come from the decode kernel itself.
  pdl_wait();
  // this warp's pieces c0 + wid + 4k, in batches of 8 (every load of a batch
  // issued before any use); batches merge online (running max M, sums)
  constexpr int kBatch = 8;
  float M = -INFINITY, den = 0.f, num[CPL];
#pragma unroll
  for (int e = 0; e < CPL; ++e) num[e] = 0.f;
  for (long long cb = c0 + wid; cb <= c1; cb += kBatch * kCombineWarps) {
    float mc[kBatch], lc[kBatch], oc[kBatch][CPL];
#pragma unroll
    for (int k = 0; k < kBatch; ++k) {
      const long long c = cb + k * kCombineWarps;
      const bool use = c <= c1 && (W >= nc || !cta_empty(c, W, nc));
      const long long sl = (u + c) * nr + t;
      mc[k] = use ? __ldg(part_ml + sl * 2) : -INFINITY;
      lc[k] = use ? __ldg(part_ml + sl * 2 + 1) : 0.f;
      if constexpr (CPL % 4 == 0) {  // CPL / 4 float4 loads a lane
#pragma unroll
        for (int q4 = 0; q4 < CPL / 4; ++q4) {
          const float4 v =
              use ? __ldg(reinterpret_cast<const float4*>(part_o + sl * d) + lane * (CPL / 4) + q4)
                  : make_float4(0.f, 0.f, 0.f, 0.f);
          oc[k][4 * q4] = v.x;
          oc[k][4 * q4 + 1] = v.y;
          oc[k][4 * q4 + 2] = v.z;
          oc[k][4 * q4 + 3] = v.w;
        }
      } else {  // CPL / 2 float2 loads
#pragma unroll
        for (int q2 = 0; q2 < CPL / 2; ++q2) {
          const float2 v =
              use ? __ldg(reinterpret_cast<const float2*>(part_o + sl * d) + lane * (CPL / 2) + q2)
                  : make_float2(0.f, 0.f);
          oc[k][2 * q2] = v.x;
          oc[k][2 * q2 + 1] = v.y;
        }
      }
    }
    float mb = M;
#pragma unroll
    for (int k = 0; k < kBatch; ++k) mb = fmaxf(mb, mc[k]);
    // pieces that saw no position of this row (causal mask) have max -inf
    const float mbr = (mb == -INFINITY) ? 0.f : mb;
    const float sc = ex2(M - mbr);  // 0 while M = -inf
    den *= sc;
#pragma unroll
    for (int e = 0; e < CPL; ++e) num[e] *= sc;
#pragma unroll
    for (int k = 0; k < kBatch; ++k) {
      const float wgt = ex2(mc[k] - mbr);  // 0 for unused slots and empty pieces
      den = fmaf(wgt, lc[k], den);
#pragma unroll
      for (int e = 0; e < CPL; ++e) num[e] = fmaf(wgt, oc[k][e], num[e]);
    }
    M = mb;
  }
  if (lane == 0) {
    s_m[wid] = M;
    s_l[wid] = den;
  }
#pragma unroll
  for (int e = 0; e < CPL; ++e) s_o[wid][lane * CPL + e] = num[e];
  __syncthreads();
  if (wid != 0) return;
  float mw[kCombineWarps], mx = -INFINITY;
#pragma unroll
  for (int w = 0; w < kCombineWarps; ++w) {
    mw[w] = s_m[w];
    mx = fmaxf(mx, mw[w]);
  }
  const float mref = (mx == -INFINITY) ? 0.f : mx;
  float dsum = 0.f, o[CPL];
#pragma unroll
  for (int e = 0; e < CPL; ++e) o[e] = 0.f;
#pragma unroll
  for (int w = 0; w < kCombineWarps; ++w) {
    const float wgt = ex2(mw[w] - mref);
    dsum = fmaf(wgt, s_l[w], dsum);
#pragma unroll
    for (int e = 0; e < CPL; ++e) o[e] = fmaf(wgt, s_o[w][lane * CPL + e], o[e]);
  }
  const int s = t / r;
  DT* dst = out + ((static_cast<size_t>(i) * nq + s) * h + j * r + (t - s * r)) * d + lane * CPL;
#pragma unroll
  for (int e = 0; e < CPL; ++e) {
    const float v = o[e] / dsum;
    if constexpr (std::is_same<DT, __nv_bfloat16>::value)
      dst[e] = __float2bfloat16_rn(v);
    else if constexpr (std::is_same<DT, __half>::value)
      dst[e] = __float2half_rn(v);
    else
      dst[e] = v;
  }
}

// One mbarrier that nothing ever arrives on; the bounded wait must give up.
__global__ void wait_selftest_kernel(unsigned int* status, long long budget) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait(smem_u32(&bar), 0, &abort_flag, status, budget);
}

// ---------------------------------------------------------------------------
// per-device state
// ---------------------------------------------------------------------------
struct DeviceInfo {
  bool checked = false;
  bool ok = false;
  int num_sms = 0;
  unsigned int* status = nullptr;
};

// Split workspace of one (device, stream): partials, rewritten by every call,
// and per-unit arrival counters, which must be zero before a launch.  The
// kernels put every counter they use back to zero; after a wait timeout (a
// launch that gave up half way) the counters are cleared again.
struct Workspace {
  void* ptr = nullptr;
  size_t bytes = 0;
  int* counters = nullptr;
  size_t units = 0;
  unsigned epoch = 0;
};

std::atomic<unsigned> g_reset_epoch{0};

std::mutex g_mu;
std::map<int, DeviceInfo> g_devices;
std::map<std::pair<int, cudaStream_t>, Workspace> g_ws;

int device_info(DeviceInfo** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return GQA_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceInfo& di = g_devices[dev];
  if (!di.checked) {
    di.checked = true;
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&di.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return GQA_ERR_CUDA;
    di.ok = (major == 10 && minor == 3);
    if (di.ok) {
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) {
        di.ok = false;
        return GQA_ERR_CUDA;
      }
      di.status = static_cast<unsigned int*>(p);
    }
  }
  if (!di.ok) return GQA_ERR_DEVICE;
  *out = &di;
  return GQA_OK;
}

int workspace(cudaStream_t stream, size_t bytes, size_t units, void** ptr, int** counters) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return GQA_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  Workspace& ws = g_ws[{dev, stream}];
  if (ws.bytes < bytes || ws.units < units) {
    // growing needs cudaMalloc, which a stream capture forbids: a captured
    // call must be preceded by an uncaptured one of at least its size
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess || cs != cudaStreamCaptureStatusNone)
      return GQA_ERR_CUDA;
    // the previous buffers may still be used by queued work on `stream`
    if ((ws.ptr || ws.counters) && cudaStreamSynchronize(stream) != cudaSuccess)
      return GQA_ERR_CUDA;
    if (ws.bytes < bytes) {
      if (ws.ptr && cudaFree(ws.ptr) != cudaSuccess) return GQA_ERR_CUDA;
      ws.ptr = nullptr;
      ws.bytes = 0;
      const size_t grow = bytes + bytes / 4;
      if (cudaMalloc(&ws.ptr, grow) != cudaSuccess) {
        ws.ptr = nullptr;
        return GQA_ERR_CUDA;
      }
      ws.bytes = grow;
    }
    if (ws.units < units) {
      if (ws.counters && cudaFree(ws.counters) != cudaSuccess) return GQA_ERR_CUDA;
      ws.counters = nullptr;
      ws.units = 0;
      const size_t grow = units + units / 4;
      if (cudaMalloc(&ws.counters, grow * sizeof(int)) != cudaSuccess ||
          cudaMemset(ws.counters, 0, grow * sizeof(int)) != cudaSuccess) {
        ws.counters = nullptr;
        return GQA_ERR_CUDA;
      }
      ws.units = grow;
      ws.epoch = g_reset_epoch.load();
    }
  }
  const unsigned epoch = g_reset_epoch.load();
  if (ws.epoch != epoch) {
    // (an async memset; allowed in a capture, where it becomes a graph node)
    if (cudaMemsetAsync(ws.counters, 0, ws.units * sizeof(int), stream) != cudaSuccess)
      return GQA_ERR_CUDA;
    ws.epoch = epoch;
  }
  *ptr = ws.ptr;
  *counters = ws.counters;
  return GQA_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// With more than twice as many CTAs as units, every unit is cut into three
// or more pieces and a merge by the last CTA to finish would serialise many
// partial reads at the end of the launch: those launches hand the merge to
// the combine kernel instead (counters = null tells the decode kernel).
// Units split over more CTAs than twice the unit count are merged by the
// combine kernel; fewer splits are merged inside the decode kernel.
bool use_combine_kernel(long long nc, int b, int g) { return nc > 2ll * b * g; }

// The combine kernel for the call's V head dim (d_v / 32 output columns a
// lane).
template <typename DT>
cudaError_t launch_combine(cudaLaunchConfig_t& cfg, const DecodeLaunch& a, int tile,
                           const float* po, const float* pml) {
  DT* o = static_cast<DT*>(a.out);
  switch (a.dv) {
    case 64:
      return cudaLaunchKernelEx(&cfg, combine_kernel<DT, 2>, a.seq_lens, a.b, a.h, a.g, a.cap,
                                tile, a.nc, a.nq, po, pml, o);
    case 128:
      return cudaLaunchKernelEx(&cfg, combine_kernel<DT, 4>, a.seq_lens, a.b, a.h, a.g, a.cap,
                                tile, a.nc, a.nq, po, pml, o);
    case 192:
      return cudaLaunchKernelEx(&cfg, combine_kernel<DT, 6>, a.seq_lens, a.b, a.h, a.g, a.cap,
                                tile, a.nc, a.nq, po, pml, o);
    case 256:
      return cudaLaunchKernelEx(&cfg, combine_kernel<DT, 8>, a.seq_lens, a.b, a.h, a.g, a.cap,
                                tile, a.nc, a.nq, po, pml, o);
    default:
      return cudaErrorInvalidValue;
  }
}

int launch_all(DecodeLaunch& a, int tile) {
  // (a cluster launch merges its split units itself)
  const bool separate = a.cluster <= 1 && use_combine_kernel(a.nc, a.b, a.g);
  if (separate) a.counters = nullptr;
  const bool tc = !a.cuda_cores && tc_supported(a.dtype, a.d, a.dv, a.nq * (a.h / a.g),
                                                a.block_table != nullptr);
  cudaError_t e = tc ? launch_decode_tc(a) : launch_decode_simt(a);
  if (e != cudaSuccess) return GQA_ERR_CUDA;
  if (separate) {
    const long long rows = static_cast<long long>(a.b) * a.h * a.nq;  // (unit, query row) pairs
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(rows));
    cfg.blockDim = dim3(32 * kCombineWarps);
    cfg.stream = a.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const float* po = static_cast<const float*>(a.part_o);
    const float* pml = static_cast<const float*>(a.part_ml);
    if (a.dtype == GQA_BF16)
      e = launch_combine<__nv_bfloat16>(cfg, a, tile, po, pml);
    else if (a.dtype == GQA_F16)
      e = launch_combine<__half>(cfg, a, tile, po, pml);
    else
      e = launch_combine<float>(cfg, a, tile, po, pml);
  }
  return e == cudaSuccess ? GQA_OK : GQA_ERR_CUDA;
}

int elt_bytes(int dtype) { return dtype == GQA_F32 ? 4 : 2; }

// Host checks of the paged-cache arguments (a decode_check follows).
int paged_check(const int32_t* block_table, int g, int block_size, int max_blocks,
                int num_blocks) {
  if (!block_table) return GQA_ERR_NULL;
  if (reinterpret_cast<uintptr_t>(block_table) & 3u) return GQA_ERR_ALIGN;
  if (block_size < 1 || max_blocks < 1 || num_blocks < 1 || g < 1) return GQA_ERR_SHAPE;
  if (static_cast<long long>(max_blocks) * block_size > 0x7FFFFF00ll ||
      static_cast<long long>(num_blocks) * g * block_size > 0x7FFFFF00ll)
    return GQA_ERR_SHAPE;
  // powers of two from 16: a block is a whole number of tiles or a tile a
  // whole number of blocks
  if (block_size < 16 || (block_size & (block_size - 1)) != 0 || block_size > 65536)
    return GQA_ERR_UNSUPPORTED;
  return GQA_OK;
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion,
                                   CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                         cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      p = nullptr;
    return reinterpret_cast<EncodeTiledFn>(p);
  }();
  return fn;
}

}  // namespace

bool encode_bf16_map(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                     const uint64_t* strides, const uint32_t* box, bool bf16) {
  EncodeTiledFn enc = encode_fn();
  if (!enc || rank < 1 || rank > 5) return false;
  cuuint64_t d[5], st[4];
  cuuint32_t bx[5], es[5];
  for (int k = 0; k < rank; ++k) {
    d[k] = dims[k];
    bx[k] = box[k];
    es[k] = 1u;
    if (k > 0) st[k - 1] = strides[k - 1];
  }
  return enc(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
             static_cast<cuuint32_t>(rank),
             const_cast<void*>(base), d, st, bx, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace gqa

using namespace gqa;

extern "C" {

int gqa_version(void) { return 100; }

const char* gqa_status_string(int s) {
  switch (s) {
    case GQA_OK: return "GQA_OK";
    case GQA_ERR_NULL: return "GQA_ERR_NULL";
    case GQA_ERR_SHAPE: return "GQA_ERR_SHAPE";
    case GQA_ERR_DTYPE: return "GQA_ERR_DTYPE";
    case GQA_ERR_ALIGN: return "GQA_ERR_ALIGN";
    case GQA_ERR_UNSUPPORTED: return "GQA_ERR_UNSUPPORTED";
    case GQA_ERR_CUDA: return "GQA_ERR_CUDA";
    case GQA_ERR_DEVICE: return "GQA_ERR_DEVICE";
    case GQA_ERR_SCRATCH_LIMIT: return "GQA_ERR_SCRATCH_LIMIT";
    default: return "GQA_ERR_UNKNOWN";
  }
}

int gqa_kv_append_multi(const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                        const int32_t* seq_lens, int b, int n, int g, int d_k, int d_v, int cap,
                        int dtype, void* stream) {
  if (!k_new || !v_new || !k_cache || !v_cache || !seq_lens) return GQA_ERR_NULL;
  if (dtype != GQA_F32 && dtype != GQA_BF16 && dtype != GQA_F16) return GQA_ERR_DTYPE;
  if (b < 1 || n < 1 || g < 1 || d_k < 1 || d_v < 1 || cap < 1 || n > cap) return GQA_ERR_SHAPE;
  const int elt = elt_bytes(dtype);
  if ((d_k * elt) % 16 != 0 || (d_v * elt) % 16 != 0) return GQA_ERR_UNSUPPORTED;
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) || !aligned16(v_cache) ||
      (reinterpret_cast<uintptr_t>(seq_lens) & 3u))
    return GQA_ERR_ALIGN;
  DeviceInfo* di = nullptr;
  if (int e = device_info(&di)) return e;
  const int ck = d_k * elt / 16, cv = d_v * elt / 16;
  const long long total = static_cast<long long>(b) * n * g * (ck + cv);
  const int threads = 256;
  const long long blocks = (total + threads - 1) / threads;
  if (blocks > 0x7FFFFFFFll) return GQA_ERR_SHAPE;
  kv_append_kernel<<<static_cast<unsigned>(blocks), threads, 0,
                     static_cast<cudaStream_t>(stream)>>>(
      static_cast<const uint4*>(k_new), static_cast<const uint4*>(v_new),
      static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache), seq_lens, b, n, g, ck, cv,
      cap, di->status);
  return cudaGetLastError() == cudaSuccess ? GQA_OK : GQA_ERR_CUDA;
}

int gqa_kv_append(const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                  const int32_t* seq_lens, int b, int g, int d_k, int d_v, int cap, int dtype,
                  void* stream) {
  return gqa_kv_append_multi(k_new, v_new, k_cache, v_cache, seq_lens, b, 1, g, d_k, d_v, cap,
                             dtype, stream);
}

int gqa_kv_append_paged(const void* k_new, const void* v_new, void* k_pool, void* v_pool,
                        const int32_t* block_table, const int32_t* seq_lens, int b, int n, int g,
                        int d_k, int d_v, int block_size, int max_blocks, int num_blocks,
                        int dtype, void* stream) {
  if (!k_new || !v_new || !k_pool || !v_pool || !seq_lens) return GQA_ERR_NULL;
  if (dtype != GQA_F32 && dtype != GQA_BF16 && dtype != GQA_F16) return GQA_ERR_DTYPE;
  if (b < 1 || n < 1 || d_k < 1 || d_v < 1) return GQA_ERR_SHAPE;
  if (int e = paged_check(block_table, g, block_size, max_blocks, num_blocks)) return e;
  if (static_cast<long long>(n) > static_cast<long long>(max_blocks) * block_size)
    return GQA_ERR_SHAPE;
  const int elt = elt_bytes(dtype);
  if ((d_k * elt) % 16 != 0 || (d_v * elt) % 16 != 0) return GQA_ERR_UNSUPPORTED;
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_pool) || !aligned16(v_pool) ||
      (reinterpret_cast<uintptr_t>(seq_lens) & 3u))
    return GQA_ERR_ALIGN;
  DeviceInfo* di = nullptr;
  if (int e = device_info(&di)) return e;
  const int ck = d_k * elt / 16, cv = d_v * elt / 16;
  const long long total = static_cast<long long>(b) * n * g * (ck + cv);
  const int threads = 256;
  const long long blocks = (total + threads - 1) / threads;
  if (blocks > 0x7FFFFFFFll) return GQA_ERR_SHAPE;
  kv_append_paged_kernel<<<static_cast<unsigned>(blocks), threads, 0,
                           static_cast<cudaStream_t>(stream)>>>(
      static_cast<const uint4*>(k_new), static_cast<const uint4*>(v_new),
      static_cast<uint4*>(k_pool), static_cast<uint4*>(v_pool), block_table, seq_lens, b, n, g,
      ck, cv, block_size, max_blocks, num_blocks, di->status);
  return cudaGetLastError() == cudaSuccess ? GQA_OK : GQA_ERR_CUDA;
}

}  // extern "C"

namespace gqa {
namespace {

// The arguments of one decode launch and its plan (kernel, CTAs, partials).
struct DecodeArgs {
  const void* q;
  const void* k_new;     // null: attention only
  const void* v_new;
  const void* k_cache;   // contiguous caches, or the pools of a paged cache
  const void* v_cache;
  const int32_t* seq_lens;
  int b, nq, h, g, d_k, d_v;
  float scale;
  void* out;
  int cap, dtype, flags;  // cap: rows per (sequence, KV head); paged: max_blocks * block_size
  const int32_t* block_table = nullptr;  // paged cache
  int block_size = 0, max_blocks = 0, num_blocks = 0;
};

struct DecodePlan {
  int tile = 0;
  long long nc = 0;
  int cluster = 0, cluster_k = 1;  // tensor-core cluster merge (0: none)
  size_t o_bytes = 0;     // partial outputs
  size_t ml_bytes = 0;    // partial max / sum
  size_t units = 0;       // arrival counters
};

// Host checks of a decode call (no CUDA call): GQA_OK or an error code.
// The tensor-core kernel wherever it takes the shape, unless the caller asks
// for the CUDA-core kernel.
bool use_tensor_cores(const DecodeArgs& x, int cols) {
  return !(x.flags & GQA_STEP_CUDA_CORES) &&
         tc_supported(x.dtype, x.d_k, x.d_v, cols, x.block_table != nullptr);
}

int decode_check(const DecodeArgs& x) {
  if (x.flags & ~(GQA_STEP_EARLY_STREAM | GQA_STEP_CUDA_CORES)) return GQA_ERR_UNSUPPORTED;
  if (!x.q || !x.k_cache || !x.v_cache || !x.seq_lens || !x.out) return GQA_ERR_NULL;
  if (x.dtype != GQA_F32 && x.dtype != GQA_BF16 && x.dtype != GQA_F16) return GQA_ERR_DTYPE;
  if (x.b < 1 || x.nq < 1 || x.h < 1 || x.g < 1 || x.d_k < 1 || x.d_v < 1 || x.cap < 1 ||
      x.h % x.g != 0 || x.nq > x.cap)
    return GQA_ERR_SHAPE;
  if (x.block_table == nullptr && static_cast<long long>(x.b) * x.g * x.cap + 256 > 0x7FFFFFFFll)
    return GQA_ERR_SHAPE;
  if (static_cast<long long>(x.b) * x.nq * x.h > 0x7FFFFFFFll) return GQA_ERR_SHAPE;
  if (!aligned16(x.q) || !aligned16(x.k_cache) || !aligned16(x.v_cache) || !aligned16(x.out) ||
      !aligned16(x.k_new) || !aligned16(x.v_new) ||
      (reinterpret_cast<uintptr_t>(x.seq_lens) & 3u))
    return GQA_ERR_ALIGN;
  const int r = x.h / x.g;
  if (x.b > 65535 || static_cast<long long>(x.nq) * r > 32) return GQA_ERR_UNSUPPORTED;
  const int cols = x.nq * r;  // query rows per KV head
  const bool tc = use_tensor_cores(x, cols);
  if (!tc && !simt_supported(x.dtype, x.d_k, x.d_v, cols)) return GQA_ERR_UNSUPPORTED;
  return GQA_OK;
}

// Fewer (sequence, KV head) units than CTAs, at most half as many: a whole
// number of CTAs per unit, so that every unit is cut into the same number
// of equal pieces and no CTA spans two units.  (With at least 70 % as many
// units as CTAs and equal lengths, the kernels themselves take one CTA per
// unit; see Walker::init.)
long long aligned_ctas(long long ctas, long long units) {
  return (units < ctas && 2 * units <= ctas) ? units * (ctas / units) : ctas;
}

// Tuning knobs read from the environment at every call (sweeps only; unset
// in normal use): GQA_CTAS = CTAs of a decode launch (capped at the tiles of
// the cache), GQA_CLUSTER = 0 (no cluster merge) or the cluster size 2..16.
int env_knob(const char* name) {
  const char* v = std::getenv(name);
  if (v == nullptr || *v == 0) return -1;
  char* end = nullptr;
  const long x = std::strtol(v, &end, 10);
  return (end != nullptr && *end == 0 && x >= 0 && x <= 1000000) ? static_cast<int>(x) : -1;
}

// Units cut into three or more pieces on the tensor-core kernel: cluster
// launches, clusters of C CTAs, k clusters per unit (grid = units * C * k),
// whose CTAs merge their pieces themselves instead of a combine kernel.
// Among the sizes for which k >= 1 clusters per unit fit at once (at most
// `pieces` CTAs per unit), the plan takes the most CTAs, then the fewest
// clusters per unit.  max_clusters(C): clusters of C that fit at once.
template <typename F>
void choose_cluster(long long units, long long pieces, int forced, F max_clusters,
                    DecodePlan& p) {
  long long best = 0;
  int bc = 0, bk = 0;
  for (int c = 2; c <= 16; ++c) {
    if (forced >= 2 && c != forced) continue;
    if (c > pieces) break;
    const long long fit = max_clusters(c) / units;
    const long long k = std::min(pieces / c, fit);
    if (k < 1) continue;
    const long long ctas = units * c * k;
    if (ctas > best || (ctas == best && k < bk)) {
      best = ctas;
      bc = c;
      bk = static_cast<int>(k);
    }
  }
  if (best > 0) {
    p.nc = best;
    p.cluster = bc;
    p.cluster_k = bk;
  }
}

// query_device: ask the device how many clusters fit at once (else assume
// every SM can take part in a cluster of any size).
DecodePlan decode_plan(const DecodeArgs& x, int num_sms, bool query_device = true) {
  const int r = x.h / x.g, d = x.d_k, cols = x.nq * r;
  const bool use_tc = use_tensor_cores(x, cols);
  DecodePlan p;
  p.tile = use_tc ? tc_tile(x.d_k, x.d_v) : simt_tile(x.dtype, x.d_k, x.d_v);
  const int per_sm = use_tc ? tc_ctas_per_sm(r) : simt_ctas_per_sm(x.dtype, d, r);
  const long long units = static_cast<long long>(x.b) * x.g;
  const long long unit_tiles = (x.cap + p.tile - 1) / p.tile;
  const long long max_tiles = units * unit_tiles;
  const long long ctas = static_cast<long long>(num_sms) * per_sm;
  p.nc = aligned_ctas(ctas, units);
  const int knob_ctas = env_knob("GQA_CTAS");
  if (knob_ctas > 0) p.nc = knob_ctas;
  if (p.nc > max_tiles) p.nc = max_tiles;
  if (p.nc < 1) p.nc = 1;
  const int knob_cluster = env_knob("GQA_CLUSTER");
  // Every unit cut into exactly two pieces (p.nc = 2 units): pairs of CTAs
  // in clusters of two merge over distributed shared memory, which takes
  // no round trip through L2 (an atomic arrival, then the other piece's
  // partial) at the end of the launch.  Measured: 64 units of 32 tiles
  // (b = 16, g = 4), 30.0 -> 26.9 us per call.
  const bool pairs = p.nc == 2 * units;
  if (use_tc && knob_cluster != 0 &&
      (use_combine_kernel(p.nc, x.b, x.g) || pairs || (knob_cluster >= 2 && p.nc > units))) {
    // A cluster launch saves the combine kernel (its run and one more grid
    // completion: about 2 us back to back) but fits fewer CTAs (whole
    // clusters per unit, as many as the GPCs hold), so it streams slower,
    // and with more than two clusters per unit the merge of their results
    // waits for the slowest cluster.  It is taken with at most two clusters
    // per unit when the streaming time it gives up, estimated from the
    // capacity at 7.4 TB/s, is below 2 us.  Measured: 128 cluster CTAs (4 x
    // 2 per unit) for 16 units of 32 tiles 15.7 us per call against 17.0
    // with the combine kernel; 144 (2 x 9 per unit) for 8 units of 1024
    // tiles 89.4 against 84.4.
    DecodePlan cl = p;
    const long long pieces = std::min(p.nc / units, unit_tiles);
    if (query_device)
      choose_cluster(units, pieces, knob_cluster, tc_max_clusters, cl);
    else
      choose_cluster(units, pieces, knob_cluster, [&](int c) { return ctas / c; }, cl);
    const double stream_s = static_cast<double>(units) * unit_tiles * p.tile *
                            (x.d_k + x.d_v) * elt_bytes(x.dtype) / 7.4e12;
    const double lost_s =
        stream_s * (1.0 - static_cast<double>(cl.nc) / static_cast<double>(p.nc));
    if (cl.cluster > 1 && (knob_cluster >= 2 || (cl.cluster_k <= 2 && lost_s < 2e-6))) p = cl;
  }
  const size_t slots = static_cast<size_t>(units) + static_cast<size_t>(p.nc);
  p.o_bytes = slots * cols * x.d_v * sizeof(float);
  p.ml_bytes = slots * cols * 2 * sizeof(float);
  // arrival counters: two per unit (the tensor-core kernel may run two
  // softmax warpgroups, each with its own), or one per unit and cluster rank
  p.units = std::max(2 * static_cast<size_t>(units),
                     static_cast<size_t>(units) * static_cast<size_t>(p.cluster));
  return p;
}

int decode_run(const DecodeArgs& x, const DecodePlan& p, unsigned int* status, void* parts,
               int* counters, cudaStream_t st) {
  DecodeLaunch a;
  a.q = x.q;
  a.k_cache = x.k_cache;
  a.v_cache = x.v_cache;
  a.seq_lens = x.seq_lens;
  a.b = x.b;
  a.h = x.h;
  a.g = x.g;
  a.d = x.d_k;
  a.dv = x.d_v;
  a.cap = x.cap;
  a.dtype = x.dtype;
  a.nq = x.nq;
  a.scale_log2 = static_cast<float>(static_cast<double>(x.scale) * 1.4426950408889634);
  a.out = x.out;
  a.part_o = static_cast<float*>(parts);
  a.part_ml = reinterpret_cast<float*>(static_cast<char*>(parts) + p.o_bytes);
  a.counters = counters;
  a.k_new = x.k_new;
  a.v_new = x.v_new;
  a.k_cache_w = const_cast<void*>(x.k_cache);
  a.v_cache_w = const_cast<void*>(x.v_cache);
  a.early = (x.flags & GQA_STEP_EARLY_STREAM) != 0;
  a.cuda_cores = (x.flags & GQA_STEP_CUDA_CORES) != 0;
  a.status = status;
  a.budget = kWaitBudget;
  a.nc = static_cast<int>(p.nc);
  a.cluster = p.cluster;
  a.cluster_k = p.cluster_k;
  a.stream = st;
  a.block_table = x.block_table;
  a.block_size = x.block_size;
  a.max_blocks = x.max_blocks;
  a.num_blocks = x.num_blocks;
  return launch_all(a, p.tile);
}



// gqa_decode_attn and gqa_decode_step (and their n-token forms): checks,
// kernel choice, workspace, launch.
int decode(const void* q, const void* k_new, const void* v_new, const void* k_cache,
           const void* v_cache, const int32_t* seq_lens, int b, int nq, int h, int g, int d_k,
           int d_v, float scale, void* out, int cap, int dtype, void* stream, int flags) {
  const DecodeArgs x{q, k_new, v_new, k_cache, v_cache, seq_lens, b, nq, h, g, d_k, d_v,
                     scale, out, cap, dtype, flags};
  if (int e = decode_check(x)) return e;
  DeviceInfo* di = nullptr;
  if (int e = device_info(&di)) return e;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const DecodePlan p = decode_plan(x, di->num_sms);
  void* ws = nullptr;
  int* counters = nullptr;
  if (int e = workspace(st, p.o_bytes + p.ml_bytes, p.units, &ws, &counters)) return e;
  return decode_run(x, p, di->status, ws, counters, st);
}

}  // namespace
}  // namespace gqa

extern "C" {

int gqa_decode_attn(const void* q, const void* k_cache, const void* v_cache,
                    const int32_t* seq_lens, int b, int h, int g, int d_k, int d_v, float scale,
                    void* out, int cap, int dtype, void* stream) {
  return gqa::decode(q, nullptr, nullptr, k_cache, v_cache, seq_lens, b, 1, h, g, d_k, d_v,
                     scale, out, cap, dtype, stream, 0);
}

int gqa_decode_step(const void* q, const void* k_new, const void* v_new, void* k_cache,
                    void* v_cache, const int32_t* seq_lens, int b, int h, int g, int d_k,
                    int d_v, float scale, void* out, int cap, int dtype, int flags,
                    void* stream) {
  if (!k_new || !v_new) return GQA_ERR_NULL;
  return gqa::decode(q, k_new, v_new, k_cache, v_cache, seq_lens, b, 1, h, g, d_k, d_v, scale,
                     out, cap, dtype, stream, flags);
}

int gqa_decode_attn_multi(const void* q, const void* k_cache, const void* v_cache,
                          const int32_t* seq_lens, int b, int n, int h, int g, int d_k, int d_v,
                          float scale, void* out, int cap, int dtype, void* stream) {
  return gqa::decode(q, nullptr, nullptr, k_cache, v_cache, seq_lens, b, n, h, g, d_k, d_v,
                     scale, out, cap, dtype, stream, 0);
}

int gqa_decode_step_multi(const void* q, const void* k_new, const void* v_new, void* k_cache,
                          void* v_cache, const int32_t* seq_lens, int b, int n, int h, int g,
                          int d_k, int d_v, float scale, void* out, int cap, int dtype,
                          int flags, void* stream) {
  if (!k_new || !v_new) return GQA_ERR_NULL;
  return gqa::decode(q, k_new, v_new, k_cache, v_cache, seq_lens, b, n, h, g, d_k, d_v, scale,
                     out, cap, dtype, stream, flags);
}

int gqa_decode_plan(int b, int n, int h, int g, int d_k, int d_v, int cap, int dtype,
                    int flags, int num_sms, int* kernels, int* ctas, int* tile,
                    int* tensor_core, long long* workspace_bytes, int* cluster) {
  using namespace gqa;
  // stand-in pointers: only the shapes are checked
  const void* p = reinterpret_cast<const void*>(uintptr_t(256));
  DecodeArgs x{p, p, p, p, p, static_cast<const int32_t*>(p), b, n, h, g, d_k, d_v, 1.f,
               const_cast<void*>(p), cap, dtype, flags};
  if (int e = decode_check(x)) return e;
  if (num_sms < 0) return GQA_ERR_SHAPE;
  const bool on_device = num_sms == 0;
  if (on_device) {
    DeviceInfo* di = nullptr;
    if (int e = device_info(&di)) return e;
    num_sms = di->num_sms;
  }
  const DecodePlan pl = decode_plan(x, num_sms, on_device);
  if (kernels) *kernels = (pl.cluster <= 1 && use_combine_kernel(pl.nc, b, g)) ? 2 : 1;
  if (cluster) *cluster = pl.cluster;
  if (ctas) *ctas = static_cast<int>(pl.nc);
  if (tile) *tile = pl.tile;
  if (tensor_core) *tensor_core = use_tensor_cores(x, n * (h / g)) ? 1 : 0;
  if (workspace_bytes)
    *workspace_bytes = static_cast<long long>(pl.o_bytes + pl.ml_bytes + pl.units * sizeof(int));
  return GQA_OK;
}

static int decode_paged(const void* q, const void* k_new, const void* v_new, const void* k_pool,
                        const void* v_pool, const int32_t* block_table, const int32_t* seq_lens,
                        int b, int n, int h, int g, int d_k, int d_v, float scale, void* out,
                        int block_size, int max_blocks, int num_blocks, int dtype, int flags,
                        void* stream) {
  using namespace gqa;
  if (int e = paged_check(block_table, g, block_size, max_blocks, num_blocks)) return e;
  DecodeArgs x{q, k_new, v_new, k_pool, v_pool, seq_lens, b, n, h, g, d_k, d_v, scale, out,
               max_blocks * block_size, dtype, flags};
  x.block_table = block_table;
  x.block_size = block_size;
  x.max_blocks = max_blocks;
  x.num_blocks = num_blocks;
  if (int e = decode_check(x)) return e;
  DeviceInfo* di = nullptr;
  if (int e = device_info(&di)) return e;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const DecodePlan p = decode_plan(x, di->num_sms);
  void* ws = nullptr;
  int* counters = nullptr;
  if (int e = workspace(st, p.o_bytes + p.ml_bytes, p.units, &ws, &counters)) return e;
  return decode_run(x, p, di->status, ws, counters, st);
}

int gqa_decode_attn_paged(const void* q, const void* k_pool, const void* v_pool,
                          const int32_t* block_table, const int32_t* seq_lens, int b, int n,
                          int h, int g, int d_k, int d_v, float scale, void* out, int block_size,
                          int max_blocks, int num_blocks, int dtype, void* stream) {
  return decode_paged(q, nullptr, nullptr, k_pool, v_pool, block_table, seq_lens, b, n, h, g,
                      d_k, d_v, scale, out, block_size, max_blocks, num_blocks, dtype, 0, stream);
}

int gqa_decode_step_paged(const void* q, const void* k_new, const void* v_new, void* k_pool,
                          void* v_pool, const int32_t* block_table, const int32_t* seq_lens,
                          int b, int n, int h, int g, int d_k, int d_v, float scale, void* out,
                          int block_size, int max_blocks, int num_blocks, int dtype, int flags,
                          void* stream) {
  if (!k_new || !v_new) return GQA_ERR_NULL;
  return decode_paged(q, k_new, v_new, k_pool, v_pool, block_table, seq_lens, b, n, h, g, d_k,
                      d_v, scale, out, block_size, max_blocks, num_blocks, dtype, flags, stream);
}

int gqa_device_status(void* stream, uint32_t* bits_out) {
  if (!bits_out) return GQA_ERR_NULL;
  DeviceInfo* di = nullptr;
  if (int e = device_info(&di)) return e;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) return GQA_ERR_CUDA;
  unsigned int v = 0;
  if (cudaMemcpy(&v, di->status, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess ||
      cudaMemset(di->status, 0, sizeof(v)) != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess)
    return GQA_ERR_CUDA;
  // a launch that gave up waiting may have left split counters raised
  if (v & GQA_DEV_WAIT_TIMEOUT) g_reset_epoch.fetch_add(1);
  *bits_out = v;
  return GQA_OK;
}

int gqa_selftest_wait_timeout(long long budget_cycles, void* stream) {
  DeviceInfo* di = nullptr;
  if (int e = device_info(&di)) return e;
  if (budget_cycles < 0) budget_cycles = 0;
  wait_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(di->status,
                                                                         budget_cycles);
  return cudaGetLastError() == cudaSuccess ? GQA_OK : GQA_ERR_CUDA;
}

}  // extern "C"


// ---------------------------------------------------------------------------
// the projections around the step and the whole layer (tcgen05 GEMMs in
// proj_tc.cu): bf16, 128-wide heads, d_model a multiple of 128, b <= 128
// ---------------------------------------------------------------------------
namespace gqa {
namespace {

constexpr int kProjMaxBatch = 128;

int proj_shape_check(int b, int D, int h, int g, int d_k, int d_v, int dtype) {
  if (dtype != GQA_F32 && dtype != GQA_BF16 && dtype != GQA_F16) return GQA_ERR_DTYPE;
  if (b < 1 || D < 1 || h < 1 || g < 1 || d_k < 1 || d_v < 1 || h % g != 0)
    return GQA_ERR_SHAPE;
  if (static_cast<long long>(h + 2 * g) * D > 0x7FFFFFFFll ||
      static_cast<long long>(b) * D > 0x7FFFFFFFll)
    return GQA_ERR_SHAPE;
  if (dtype != GQA_BF16 || d_k != 128 || d_v != 128 || D % 128 != 0 || b > kProjMaxBatch)
    return GQA_ERR_UNSUPPORTED;
  return GQA_OK;
}

size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

struct ProjPlan {
  long long nc = 0;
  size_t part_bytes = 0;
  size_t units = 0;
};

ProjPlan proj_plan(int mode, int b, int D, int h, int g, int num_sms) {
  ProjPlan p;
  const long long W = proj_work(mode, D, h, g);
  p.nc = W < num_sms ? W : num_sms;
  const int tiles = proj_tiles(mode, D, h, g);
  p.part_bytes = (static_cast<size_t>(tiles) + p.nc) * proj_nb(b) * 128 * sizeof(float);
  p.units = static_cast<size_t>(tiles);
  return p;
}

int proj_run(int mode, const void* w0, const void* w1, const void* w2, const void* x,
             void* out0, void* out1, void* out2, int b, int D, int h, int g, bool early,
             const ProjPlan& p, const DeviceInfo* di, void* parts, int* counters,
             cudaStream_t st) {
  ProjLaunch a;
  a.mode = mode;
  a.w0 = w0;
  a.w1 = w1;
  a.w2 = w2;
  a.x = x;
  a.out0 = out0;
  a.out1 = out1;
  a.out2 = out2;
  a.b = b;
  a.D = D;
  a.h = h;
  a.g = g;
  a.part = static_cast<float*>(parts);
  a.counters = counters;
  a.status = di->status;
  a.budget = kWaitBudget;
  a.early = early;
  a.nc = static_cast<int>(p.nc);
  a.stream = st;
  return launch_proj(a) == cudaSuccess ? GQA_OK : GQA_ERR_CUDA;
}

}  // namespace
}  // namespace gqa

extern "C" {

int gqa_project_qkv(const void* x, const void* w_q, const void* w_k, const void* w_v, void* q,
                    void* k_new, void* v_new, int b, int d_model, int h, int g, int d_k,
                    int d_v, int dtype, int flags, void* stream) {
  using namespace gqa;
  if (flags & ~GQA_STEP_EARLY_STREAM) return GQA_ERR_UNSUPPORTED;
  if (!x || !w_q || !w_k || !w_v || !q || !k_new || !v_new) return GQA_ERR_NULL;
  if (int e = proj_shape_check(b, d_model, h, g, d_k, d_v, dtype)) return e;
  if (!aligned16(x) || !aligned16(w_q) || !aligned16(w_k) || !aligned16(w_v) ||
      !aligned16(q) || !aligned16(k_new) || !aligned16(v_new))
    return GQA_ERR_ALIGN;
  DeviceInfo* di = nullptr;
  if (int e = device_info(&di)) return e;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const ProjPlan p = proj_plan(0, b, d_model, h, g, di->num_sms);
  void* ws = nullptr;
  int* counters = nullptr;
  if (int e = workspace(st, p.part_bytes, p.units, &ws, &counters)) return e;
  return proj_run(0, w_q, w_k, w_v, x, q, k_new, v_new, b, d_model, h, g,
                  (flags & GQA_STEP_EARLY_STREAM) != 0, p, di, ws, counters, st);
}

int gqa_project_out(const void* o, const void* w_o, void* y, int b, int d_model, int h,
                    int d_v, int dtype, int flags, void* stream) {
  using namespace gqa;
  if (flags & ~GQA_STEP_EARLY_STREAM) return GQA_ERR_UNSUPPORTED;
  if (!o || !w_o || !y) return GQA_ERR_NULL;
  if (int e = proj_shape_check(b, d_model, h, 1, 128, d_v, dtype)) return e;
  if (!aligned16(o) || !aligned16(w_o) || !aligned16(y)) return GQA_ERR_ALIGN;
  DeviceInfo* di = nullptr;
  if (int e = device_info(&di)) return e;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const ProjPlan p = proj_plan(1, b, d_model, h, 1, di->num_sms);
  void* ws = nullptr;
  int* counters = nullptr;
  if (int e = workspace(st, p.part_bytes, p.units, &ws, &counters)) return e;
  return proj_run(1, w_o, nullptr, nullptr, o, y, nullptr, nullptr, b, d_model, h, 1,
                  (flags & GQA_STEP_EARLY_STREAM) != 0, p, di, ws, counters, st);
}

int gqa_decode_layer(const void* x, const void* w_q, const void* w_k, const void* w_v,
                     const void* w_o, void* k_cache, void* v_cache, const int32_t* seq_lens,
                     int b, int d_model, int h, int g, int d_k, int d_v, float scale, void* y,
                     int cap, int dtype, int flags, void* stream) {
  using namespace gqa;
  if (flags & ~GQA_STEP_EARLY_STREAM) return GQA_ERR_UNSUPPORTED;
  if (!x || !w_q || !w_k || !w_v || !w_o || !y) return GQA_ERR_NULL;
  if (int e = proj_shape_check(b, d_model, h, g, d_k, d_v, dtype)) return e;
  if (!aligned16(x) || !aligned16(w_q) || !aligned16(w_k) || !aligned16(w_v) ||
      !aligned16(w_o) || !aligned16(y))
    return GQA_ERR_ALIGN;
  // the step's own checks, with stand-in (aligned, non-null) addresses for
  // the intermediate tensors the library keeps in its workspace
  const void* stand_in = reinterpret_cast<const void*>(uintptr_t(256));
  DecodeArgs dx{stand_in, stand_in, stand_in, k_cache, v_cache, seq_lens, b, 1, h, g,
                d_k, d_v, scale, const_cast<void*>(stand_in), cap, dtype, flags};
  if (int e = decode_check(dx)) return e;
  DeviceInfo* di = nullptr;
  if (int e = device_info(&di)) return e;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const ProjPlan p0 = proj_plan(0, b, d_model, h, g, di->num_sms);
  const ProjPlan p1 = proj_plan(1, b, d_model, h, 1, di->num_sms);
  const DecodePlan pd = decode_plan(dx, di->num_sms);
  // workspace: q | k_new | v_new | o | partials (the largest of the three)
  const size_t qb = align256(static_cast<size_t>(b) * h * 128 * 2);
  const size_t kb = align256(static_cast<size_t>(b) * g * 128 * 2);
  size_t parts = p0.part_bytes;
  if (p1.part_bytes > parts) parts = p1.part_bytes;
  if (pd.o_bytes + pd.ml_bytes > parts) parts = pd.o_bytes + pd.ml_bytes;
  size_t units = p0.units;
  if (p1.units > units) units = p1.units;
  if (pd.units > units) units = pd.units;
  void* ws = nullptr;
  int* counters = nullptr;
  if (int e = workspace(st, 2 * qb + 2 * kb + parts, units, &ws, &counters)) return e;
  char* base = static_cast<char*>(ws);
  void* q = base;
  void* kn = base + qb;
  void* vn = base + qb + kb;
  void* o = base + qb + 2 * kb;
  void* part = base + 2 * qb + 2 * kb;
  const bool early = (flags & GQA_STEP_EARLY_STREAM) != 0;
  if (int e = proj_run(0, w_q, w_k, w_v, x, q, kn, vn, b, d_model, h, g, early, p0, di, part,
                       counters, st))
    return e;
  dx.q = q;
  dx.k_new = kn;
  dx.v_new = vn;
  dx.out = o;
  // (early streaming only with the caller's consent: a kernel that started
  // before the projection, e.g. one writing this cache, may still run)
  if (int e = decode_run(dx, pd, di->status, part, counters, st)) return e;
  return proj_run(1, w_o, nullptr, nullptr, o, y, nullptr, nullptr, b, d_model, h, 1, early,
                  p1, di, part, counters, st);
}

}  // extern "C"

// ---------------------------------------------------------------------------
// gqa_decode_attn_noalloc: the same decode, with the split partials in a
// fixed device array instead of a cudaMalloc'd workspace, for callers that
// cannot allocate device memory (see include/gqa.h).
// ---------------------------------------------------------------------------
namespace gqa {
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(4) << 20;  // 4 MiB per device
constexpr size_t kNoAllocCounterBytes = size_t(256) << 10;  // first 256 KiB: unit counters
constexpr size_t kNoAllocMaxUnits = kNoAllocCounterBytes / sizeof(int);

// Every GPU that loads the library holds this array until the process exits.
// Host code must not use its name as an address: the device address comes
// from cudaGetSymbolAddress, once per device.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

struct NoAllocDevice {
  bool ready;
  int num_sms;
  unsigned int* status;
  unsigned char* scratch;
};

constexpr int kNoAllocMaxDevices = 64;
NoAllocDevice g_noalloc_devices[kNoAllocMaxDevices];  // zero-initialised, no heap
std::mutex g_noalloc_mu;

// One-time set-up per device, run with that device current: check the
// architecture and look up the device addresses of the scratch array and of
// the status word.
int noalloc_setup(NoAllocDevice** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return GQA_ERR_CUDA;
  if (dev < 0 || dev >= kNoAllocMaxDevices) return GQA_ERR_DEVICE;
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  NoAllocDevice& nd = g_noalloc_devices[dev];
  if (!nd.ready) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return GQA_ERR_CUDA;
    if (major != 10 || minor != 3) return GQA_ERR_DEVICE;
    void* scratch = nullptr;
    void* status = nullptr;
    if (cudaGetSymbolAddress(&scratch, g_noalloc_scratch) != cudaSuccess ||
        cudaGetSymbolAddress(&status, g_status_word) != cudaSuccess)
      return GQA_ERR_CUDA;
    nd.num_sms = sms;
    nd.scratch = static_cast<unsigned char*>(scratch);
    nd.status = static_cast<unsigned int*>(status);
    nd.ready = true;
  }
  *out = &nd;
  return GQA_OK;
}

}  // namespace
}  // namespace gqa

extern "C" int gqa_decode_attn_noalloc(const void* q, const void* k_cache, const void* v_cache,
                                       const int32_t* seq_lens, int b, int h, int g, int d_k,
                                       int d_v, float scale, void* out, int cap, int dtype,
                                       void* stream) {
  using namespace gqa;
  // the checks and the plan of gqa_decode_attn, so the two launch the same
  // grid with the same partial layout
  const DecodeArgs x{q, nullptr, nullptr, k_cache, v_cache, seq_lens, b, 1, h, g, d_k, d_v,
                     scale, out, cap, dtype, 0};
  if (int e = decode_check(x)) return e;
  NoAllocDevice* nd = nullptr;
  if (int e = noalloc_setup(&nd)) return e;
  const DecodePlan p = decode_plan(x, nd->num_sms);
  if (p.units > kNoAllocMaxUnits ||
      p.o_bytes + p.ml_bytes > kNoAllocScratchBytes - kNoAllocCounterBytes)
    return GQA_ERR_SCRATCH_LIMIT;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int* counters = reinterpret_cast<int*>(nd->scratch);
  // the arrival counters the launch uses must start at zero
  if (cudaMemsetAsync(counters, 0, p.units * sizeof(int), st) != cudaSuccess)
    return GQA_ERR_CUDA;
  return decode_run(x, p, nd->status, nd->scratch + kNoAllocCounterBytes, counters, st);
}
