// gqa_api.cu - the C ABI of libgqa.so (declared in include/gqa.h): argument
// checks, kernel selection, the split workspace, the device status word, and
// the small kernels (KV append, log-sum-exp combine, wait self-test).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
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
// The concat of the new K/V row on the position axis (MQA review §2.4, §3),
// done in place at row L_i - 1 (decode notes: kCache.push, vCache.push).
// ---------------------------------------------------------------------------
__global__ void kv_append_kernel(const uint4* __restrict__ k_new, const uint4* __restrict__ v_new,
                                 uint4* __restrict__ k_cache, uint4* __restrict__ v_cache,
                                 const int* __restrict__ lens, int b, int g, int ck, int cv,
                                 int cap, unsigned int* status) {
  const long long per = ck + cv;
  const long long total = static_cast<long long>(b) * g * per;
  const long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= total) return;
  const long long row = idx / per;  // (i, j) row of k_new / v_new
  const int c = static_cast<int>(idx % per);
  const int i = static_cast<int>(row / g);
  const int L = __ldg(lens + i);
  if (L < 1 || L > cap) {
    if (c == 0) atomicOr(status, GQA_DEV_BAD_SEQ_LEN);
    return;
  }
  const long long dst_row = row * cap + (L - 1);
  if (c < ck) {
    k_cache[dst_row * ck + c] = __ldg(k_new + row * ck + c);
  } else {
    const int cc = c - ck;
    v_cache[dst_row * cv + cc] = __ldg(v_new + row * cv + cc);
  }
}

// ---------------------------------------------------------------------------
// Log-sum-exp combine of the partials of one unit (sequence i, KV head j)
// split across CTAs.  With per-CTA maxima m_c (base 2), sums l_c and
// unnormalised outputs O_c of the same softmax over disjoint position ranges:
//     M = max_c m_c,  out = sum_c 2^(m_c - M) O_c / sum_c 2^(m_c - M) l_c,
// which is the softmax-weighted sum over the whole range.  Units covered by
// one CTA were written directly by the decode kernel and are skipped.  This
// kernel (one CTA per unit) also reports sequences whose length is outside
// [1, cap] on the device status word.
// ---------------------------------------------------------------------------
template <typename DT>
__global__ void combine_kernel(const int* __restrict__ lens, int b, int h, int g, int cap,
                               int d, int tile, int nc, const float* __restrict__ part_o,
                               const float* __restrict__ part_ml, DT* __restrict__ out,
                               unsigned int* status) {
  __shared__ long long s_u0, s_W;
  __shared__ int s_ti;
  const int u = blockIdx.x;
  const int i = u / g, j = u % g;
  const int r = h / g;
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    long long before = 0, all = 0;
    for (int base = 0; base < b; base += 32) {
      const int idx = base + lane;
      const int t = (idx < b) ? seq_tiles(__ldg(lens + idx), cap, tile) : 0;
      all += t;
      if (idx < i) before += t;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      all += __shfl_xor_sync(0xffffffffu, all, o);
      before += __shfl_xor_sync(0xffffffffu, before, o);
    }
    if (lane == 0) {
      const int Li = __ldg(lens + i);
      const int ti = seq_tiles(Li, cap, tile);
      // one report per bad sequence; its output rows are left untouched
      if (ti == 0 && j == 0) atomicOr(status, GQA_DEV_BAD_SEQ_LEN);
      s_ti = ti;
      s_u0 = before * g + static_cast<long long>(j) * ti;
      s_W = all * g;
    }
  }
  __syncthreads();
  const int ti = s_ti;
  if (ti == 0) return;
  const long long W = s_W, u0 = s_u0, u1 = u0 + ti;
  const long long c0 = ((u0 + 1) * nc - 1) / W;
  const long long c1 = (u1 * nc - 1) / W;
  if (c0 == c1) return;
  // a CTA between c0 and c1 with an empty range (possible when W < nc)
  // wrote no partial
  auto empty_cta = [&](long long c) { return (c * W) / nc == ((c + 1) * W) / nc; };
  for (int t = 0; t < r; ++t) {
    float M = -INFINITY;
    for (long long c = c0; c <= c1; ++c)
      if (!empty_cta(c)) M = fmaxf(M, part_ml[((u + c) * r + t) * 2]);
    float den = 0.f;
    for (long long c = c0; c <= c1; ++c) {
      if (empty_cta(c)) continue;
      const float* ml = part_ml + ((u + c) * r + t) * 2;
      den += exp2f(ml[0] - M) * ml[1];
    }
    const float inv = 1.f / den;
    for (int dd = threadIdx.x; dd < d; dd += blockDim.x) {
      float num = 0.f;
      for (long long c = c0; c <= c1; ++c) {
        if (empty_cta(c)) continue;
        const float wgt = exp2f(part_ml[((u + c) * r + t) * 2] - M);
        num = fmaf(wgt, part_o[((u + c) * r + t) * d + dd], num);
      }
      const float v = num * inv;
      DT* dst = out + (static_cast<size_t>(i) * h + j * r + t) * d + dd;
      if constexpr (sizeof(DT) == 2)
        *dst = __float2bfloat16_rn(v);
      else
        *dst = v;
    }
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

struct Workspace {
  void* ptr = nullptr;
  size_t bytes = 0;
};

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

int workspace(cudaStream_t stream, size_t bytes, void** ptr) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return GQA_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  Workspace& ws = g_ws[{dev, stream}];
  if (ws.bytes < bytes) {
    if (ws.ptr) {
      // the previous buffer may still be read by queued work on `stream`
      if (cudaStreamSynchronize(stream) != cudaSuccess || cudaFree(ws.ptr) != cudaSuccess)
        return GQA_ERR_CUDA;
      ws.ptr = nullptr;
      ws.bytes = 0;
    }
    const size_t grow = bytes + bytes / 4;
    if (cudaMalloc(&ws.ptr, grow) != cudaSuccess) {
      ws.ptr = nullptr;
      return GQA_ERR_CUDA;
    }
    ws.bytes = grow;
  }
  *ptr = ws.ptr;
  return GQA_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int elt_bytes(int dtype) { return dtype == GQA_F32 ? 4 : 2; }

}  // namespace
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

int gqa_kv_append(const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                  const int32_t* seq_lens, int b, int g, int d_k, int d_v, int cap, int dtype,
                  void* stream) {
  if (!k_new || !v_new || !k_cache || !v_cache || !seq_lens) return GQA_ERR_NULL;
  if (dtype != GQA_F32 && dtype != GQA_BF16) return GQA_ERR_DTYPE;
  if (b < 1 || g < 1 || d_k < 1 || d_v < 1 || cap < 1) return GQA_ERR_SHAPE;
  const int elt = elt_bytes(dtype);
  if ((d_k * elt) % 16 != 0 || (d_v * elt) % 16 != 0) return GQA_ERR_UNSUPPORTED;
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) || !aligned16(v_cache) ||
      (reinterpret_cast<uintptr_t>(seq_lens) & 3u))
    return GQA_ERR_ALIGN;
  DeviceInfo* di = nullptr;
  if (int e = device_info(&di)) return e;
  const int ck = d_k * elt / 16, cv = d_v * elt / 16;
  const long long total = static_cast<long long>(b) * g * (ck + cv);
  const int threads = 256;
  const long long blocks = (total + threads - 1) / threads;
  if (blocks > 0x7FFFFFFFll) return GQA_ERR_SHAPE;
  kv_append_kernel<<<static_cast<unsigned>(blocks), threads, 0,
                     static_cast<cudaStream_t>(stream)>>>(
      static_cast<const uint4*>(k_new), static_cast<const uint4*>(v_new),
      static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache), seq_lens, b, g, ck, cv, cap,
      di->status);
  return cudaGetLastError() == cudaSuccess ? GQA_OK : GQA_ERR_CUDA;
}

int gqa_decode_attn(const void* q, const void* k_cache, const void* v_cache,
                    const int32_t* seq_lens, int b, int h, int g, int d_k, int d_v, float scale,
                    void* out, int cap, int dtype, void* stream) {
  if (!q || !k_cache || !v_cache || !seq_lens || !out) return GQA_ERR_NULL;
  if (dtype != GQA_F32 && dtype != GQA_BF16) return GQA_ERR_DTYPE;
  if (b < 1 || h < 1 || g < 1 || d_k < 1 || d_v < 1 || cap < 1 || h % g != 0)
    return GQA_ERR_SHAPE;
  if (static_cast<long long>(b) * g * cap + 256 > 0x7FFFFFFFll ||
      static_cast<long long>(b) * h > 0x7FFFFFFFll)
    return GQA_ERR_SHAPE;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out) ||
      (reinterpret_cast<uintptr_t>(seq_lens) & 3u))
    return GQA_ERR_ALIGN;
  const int r = h / g;
  const int d = d_k;
  if (d_k != d_v || b > 65535) return GQA_ERR_UNSUPPORTED;
  const bool use_tc = tc_supported(dtype, d, r);
  if (!use_tc && !simt_supported(dtype, d, r)) return GQA_ERR_UNSUPPORTED;
  DeviceInfo* di = nullptr;
  if (int e = device_info(&di)) return e;
  cudaStream_t st = static_cast<cudaStream_t>(stream);

  const int tile = use_tc ? tc_tile() : simt_tile(dtype, d);
  const int per_sm = use_tc ? tc_ctas_per_sm(r) : simt_ctas_per_sm(dtype, d, r);
  const long long max_tiles = static_cast<long long>(b) * g * ((cap + tile - 1) / tile);
  long long nc = static_cast<long long>(di->num_sms) * per_sm;
  if (nc > max_tiles) nc = max_tiles;
  if (nc < 1) nc = 1;

  const size_t slots = static_cast<size_t>(b) * g + static_cast<size_t>(nc);
  const size_t o_bytes = slots * r * d * sizeof(float);
  const size_t ml_bytes = slots * r * 2 * sizeof(float);
  void* ws = nullptr;
  if (int e = workspace(st, o_bytes + ml_bytes, &ws)) return e;

  DecodeLaunch a;
  a.q = q;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.seq_lens = seq_lens;
  a.b = b;
  a.h = h;
  a.g = g;
  a.d = d;
  a.cap = cap;
  a.dtype = dtype;
  a.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  a.out = out;
  a.part_o = static_cast<float*>(ws);
  a.part_ml = reinterpret_cast<float*>(static_cast<char*>(ws) + o_bytes);
  a.status = di->status;
  a.budget = kWaitBudget;
  a.nc = static_cast<int>(nc);
  a.stream = st;

  cudaError_t e = use_tc ? launch_decode_tc(a) : launch_decode_simt(a);
  if (e != cudaSuccess) return GQA_ERR_CUDA;
  e = launch_combine(a, tile);
  return e == cudaSuccess ? GQA_OK : GQA_ERR_CUDA;
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

namespace gqa {

cudaError_t launch_combine(const DecodeLaunch& a, int tile) {
  const long long units = static_cast<long long>(a.b) * a.g;
  if (a.dtype == GQA_BF16)
    combine_kernel<__nv_bfloat16><<<static_cast<unsigned>(units), 128, 0, a.stream>>>(
        a.seq_lens, a.b, a.h, a.g, a.cap, a.d, tile, a.nc, a.part_o, a.part_ml,
        static_cast<__nv_bfloat16*>(a.out), a.status);
  else
    combine_kernel<float><<<static_cast<unsigned>(units), 128, 0, a.stream>>>(
        a.seq_lens, a.b, a.h, a.g, a.cap, a.d, tile, a.nc, a.part_o, a.part_ml,
        static_cast<float*>(a.out), a.status);
  return cudaGetLastError();
}

}  // namespace gqa

// ---------------------------------------------------------------------------
// gqa_decode_attn_noalloc: the same decode, with the split partials in a
// fixed device array instead of a cudaMalloc'd workspace, for callers that
// cannot allocate device memory (see include/gqa.h).
// ---------------------------------------------------------------------------
namespace gqa {
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(4) << 20;  // 4 MiB per device

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
  if (!q || !k_cache || !v_cache || !seq_lens || !out) return GQA_ERR_NULL;
  if (dtype != GQA_F32 && dtype != GQA_BF16) return GQA_ERR_DTYPE;
  if (b < 1 || h < 1 || g < 1 || d_k < 1 || d_v < 1 || cap < 1 || h % g != 0)
    return GQA_ERR_SHAPE;
  if (static_cast<long long>(b) * g * cap + 256 > 0x7FFFFFFFll ||
      static_cast<long long>(b) * h > 0x7FFFFFFFll)
    return GQA_ERR_SHAPE;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out) ||
      (reinterpret_cast<uintptr_t>(seq_lens) & 3u))
    return GQA_ERR_ALIGN;
  const int r = h / g;
  const int d = d_k;
  if (d_k != d_v || b > 65535) return GQA_ERR_UNSUPPORTED;
  const bool use_tc = tc_supported(dtype, d, r);
  if (!use_tc && !simt_supported(dtype, d, r)) return GQA_ERR_UNSUPPORTED;
  NoAllocDevice* nd = nullptr;
  if (int e = noalloc_setup(&nd)) return e;

  const int tile = use_tc ? tc_tile() : simt_tile(dtype, d);
  const int per_sm = use_tc ? tc_ctas_per_sm(r) : simt_ctas_per_sm(dtype, d, r);
  const long long max_tiles = static_cast<long long>(b) * g * ((cap + tile - 1) / tile);
  long long nc = static_cast<long long>(nd->num_sms) * per_sm;
  if (nc > max_tiles) nc = max_tiles;
  if (nc < 1) nc = 1;
  const size_t slots = static_cast<size_t>(b) * g + static_cast<size_t>(nc);
  const size_t o_bytes = slots * r * d * sizeof(float);
  const size_t ml_bytes = slots * r * 2 * sizeof(float);
  if (o_bytes + ml_bytes > kNoAllocScratchBytes) return GQA_ERR_SCRATCH_LIMIT;

  DecodeLaunch a;
  a.q = q;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.seq_lens = seq_lens;
  a.b = b;
  a.h = h;
  a.g = g;
  a.d = d;
  a.cap = cap;
  a.dtype = dtype;
  a.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  a.out = out;
  a.part_o = reinterpret_cast<float*>(nd->scratch);
  a.part_ml = reinterpret_cast<float*>(nd->scratch + o_bytes);
  a.status = nd->status;
  a.budget = kWaitBudget;
  a.nc = static_cast<int>(nc);
  a.stream = static_cast<cudaStream_t>(stream);

  cudaError_t e = use_tc ? launch_decode_tc(a) : launch_decode_simt(a);
  if (e != cudaSuccess) return GQA_ERR_CUDA;
  e = launch_combine(a, tile);
  return e == cudaSuccess ? GQA_OK : GQA_ERR_CUDA;
}
