// gqa_device.cuh - device-side helpers shared by the decode kernels:
// PTX wrappers (mbarrier, bulk/tensor copies, tcgen05), the bounded wait, and
// the work walker that splits the KV stream of all (sequence, KV head) units
// evenly across persistent CTAs.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "../../include/gqa.h"

namespace gqa {

// ---------------------------------------------------------------------------
// shared-memory addresses and mbarriers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait until the phase with the given parity of `bar` has completed, for at
// most `budget` SM cycles.  Returns false (and raises the CTA's abort flag and
// the device status bit) when the limit is hit, or at once when the abort
// flag is already up.  No wait in these kernels is unbounded.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity,
                                          volatile int* abort_flag,
                                          unsigned int* status, long long budget) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (true) {
    if (*abort_flag) return false;
    if (mbar_try_wait(bar, parity)) return true;
    if (clock64() - t0 > budget) {
      *abort_flag = 1;
      atomicOr(status, GQA_DEV_WAIT_TIMEOUT);
      return false;
    }
  }
}

// ---------------------------------------------------------------------------
// bulk copies global -> shared, completing on an mbarrier
// ---------------------------------------------------------------------------
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, "
      "[%3];" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void* tmap, uint32_t bar,
                                            int x, int y, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(bar), "r"(x), "r"(y), "l"(policy)
      : "memory");
}

// 3-D tiled load (e.g. the query rows of one KV head for n new tokens):
// the box lands as [z][y][x] rows of the swizzled layout.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const void* tmap, uint32_t bar,
                                            int x, int y, int z, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%3, %4, %5}], [%2], %6;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(bar), "r"(x), "r"(y), "r"(z), "l"(policy)
      : "memory");
}

// Bring a tile of a tensor map into L2 (no shared memory, no completion).
__device__ __forceinline__ void tma_prefetch_l2_2d(const void* tmap, int x, int y) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                   reinterpret_cast<uint64_t>(tmap)),
               "r"(x), "r"(y)
               : "memory");
}

__device__ __forceinline__ void tma_prefetch_l2_3d(const void* tmap, int x, int y, int z) {
  asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(
                   reinterpret_cast<uint64_t>(tmap)),
               "r"(x), "r"(y), "r"(z)
               : "memory");
}

__device__ __forceinline__ void prefetch_tmap(const void* tmap) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tmap))
               : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// make this thread's generic-proxy shared-memory writes visible to the async
// proxy (tensor cores, bulk copies)
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Programmatic dependent launch.  launch_dependents lets the next kernel of
// the stream be scheduled as SMs free up; wait blocks until the previous
// kernel of the stream has completed and its writes are visible (a no-op
// when the launch had no programmatic dependency).  Every input and the
// split workspace are read only after the wait.
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// The decode kernels let their dependents launch only once the kernel ahead
// of them has completed, so a dependent may read before its own wait what
// that kernel wrote (the combine kernel reads seq_lens so).  A decode CTA
// cannot leave room for the next decode kernel before it exits anyway.
__device__ __forceinline__ void pdl_wait_then_release() {
  pdl_wait();
  pdl_launch_dependents();
}

__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ---------------------------------------------------------------------------
// thread-block clusters: distributed shared memory and the cluster barrier
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Every thread of every CTA of the cluster arrives (release: this thread's
// earlier shared-memory writes become visible to the cluster) ...
__device__ __forceinline__ void cluster_arrive() {
  asm volatile("barrier.cluster.arrive.release;" ::: "memory");
}

// ... and waits for all of them (acquire).  A hardware barrier, not a spin:
// it completes once every thread of the cluster has arrived, and every path
// through the kernels that use it arrives.
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire;" ::: "memory");
}

// The address, in the cluster's shared window, of the variable at this
// CTA's shared address `addr` in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t dsmem_addr(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}

__device__ __forceinline__ float ld_dsmem(uint32_t addr) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
  return v;
}

__device__ __forceinline__ int ld_dsmem_s32(uint32_t addr) {
  int v;
  asm volatile("ld.shared::cluster.s32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}

__device__ __forceinline__ float4 ld_dsmem4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}

// ---------------------------------------------------------------------------
// tcgen05 (5th-generation tensor cores, accumulators in tensor memory)
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   dst_smem),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr),
               "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, bf16 inputs, fp32 accumulate
__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                         uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// arrive once on `bar` when every tcgen05 op issued so far by this thread is done
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          bar)
      : "memory");
}

__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// 32 lanes x 16 consecutive 32-bit columns: thread t of the warp gets lane
// (base lane + t), columns [col, col + 16)
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
      "%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
        "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]),
        "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
#pragma unroll
  for (int k = 0; k < 16; ++k) v[k] = __uint_as_float(r[k]);
}

// Shared-memory matrix descriptor of tcgen05.mma: start address, leading and
// stride byte offsets (16-byte units), descriptor version 1, swizzle mode.
enum : uint32_t { SWZ_NONE = 0, SWZ_128B = 2, SWZ_64B = 4, SWZ_32B = 6 };

__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo,
                                              uint32_t swz) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((addr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= 1ull << 46;
  d |= static_cast<uint64_t>(swz & 7u) << 61;
  return d;
}

// Instruction descriptor of tcgen05.mma kind::f16: A and B both bf16 (or
// both fp16 with bf16 = false), fp32 D, A/B K-major (0) or MN-major (1),
// shape M x N.
__host__ __device__ constexpr uint32_t idesc_bf16(int m, int n, int a_mn_major,
                                                  int b_mn_major, bool bf16 = true) {
  return (1u << 4)                                      // D format: f32
         | (static_cast<uint32_t>(bf16 ? 1 : 0) << 7)   // A format: bf16 (1) or f16 (0)
         | (static_cast<uint32_t>(bf16 ? 1 : 0) << 10)  // B format: the same
         | (static_cast<uint32_t>(a_mn_major) << 15) |
         (static_cast<uint32_t>(b_mn_major) << 16) |
         (static_cast<uint32_t>(n >> 3) << 17) | (static_cast<uint32_t>(m >> 4) << 24);
}

// The two 16-bit storage types of the tensor-core paths.
template <typename T>
struct Half16;
template <>
struct Half16<__nv_bfloat16> {
  static constexpr bool kBf16 = true;
  __device__ static uint32_t pack2(float a, float b) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<const uint32_t*>(&v);
  }
  __device__ static __nv_bfloat16 from(float v) { return __float2bfloat16_rn(v); }
};
template <>
struct Half16<__half> {
  static constexpr bool kBf16 = false;
  __device__ static uint32_t pack2(float a, float b) {
    const __half2 v = __floats2half2_rn(a, b);
    return *reinterpret_cast<const uint32_t*>(&v);
  }
  __device__ static __half from(float v) { return __float2half_rn(v); }
};

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float warp_max(float v) {
  float m;
  asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(m) : "f"(v));
  return m;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// ---------------------------------------------------------------------------
// Work walker.
//
// A "unit" is one (sequence i, KV head j); it holds t_i = ceil(L_i / T) tiles
// of T positions (0 when L_i is outside [n, cap], n being the number of new
// tokens per sequence of the step, usually 1).  Units are ordered
// u = i * g + j and their tiles laid end to end, W tiles in all.  CTA c of NC
// takes the tile range [c * W / NC, (c + 1) * W / NC), so every CTA streams
// the same number of tiles (to within one) whatever the length mix.  A CTA's
// range cuts into "segments", one per unit it touches.  A segment that covers
// a whole unit produces final outputs; any other writes a partial (running
// max, sum, unnormalised output) to slot u + c, which the combine kernel
// merges.  u + c is unique per (unit, CTA) pair with a non-empty overlap,
// so the partial buffer needs b * g + NC slots.
//
// Every warp runs its own walker (warp-uniform values, no shared state).
// ---------------------------------------------------------------------------
__device__ __forceinline__ int seq_tiles(int L, int lmin, int cap, int T) {
  return (L >= lmin && L >= 1 && L <= cap) ? (L + T - 1) / T : 0;
}

struct Segment {
  int i, j;       // sequence, KV head
  int lt0, lt1;   // local tile range within the unit
  int L;          // post-append length of sequence i
  int ti;         // tiles of the unit
  long long u0;   // global index of the unit's first tile
};

// CTA c's range is empty when W < nc leaves it no tile.
__device__ __forceinline__ bool cta_empty(long long c, long long W, int nc) {
  return (c * W) / nc == ((c + 1) * W) / nc;
}

// First and last CTA holding tiles of the unit that spans global tiles
// [u0, u1): the largest c with floor(c W / nc) <= u0, and the same for u1 - 1.
__device__ __forceinline__ void unit_ctas(long long u0, long long u1, long long W, int nc,
                                          long long& c0, long long& c1) {
  c0 = ((u0 + 1) * nc - 1) / W;
  c1 = (u1 * nc - 1) / W;
}

// Number of CTAs that write a partial for the unit (non-empty ranges only).
__device__ __forceinline__ int unit_parts(long long c0, long long c1, long long W, int nc) {
  if (W >= nc) return static_cast<int>(c1 - c0 + 1);
  int n = 0;
  for (long long c = c0; c <= c1; ++c) n += cta_empty(c, W, nc) ? 0 : 1;
  return n;
}

// Split units are merged by the CTA that finishes its share last.  Every CTA
// that wrote a partial of unit u calls this with all `nthreads` threads of its
// epilogue group: the partial stores are fenced, one leader thread counts the
// arrival, and the CTA whose arrival completes the count gets true (and puts
// the counter back to zero for the next launch).  No CTA ever waits for
// another.
__device__ __forceinline__ bool arrive_last(int* counters, int u, int nparts, int* s_flag,
                                            bool leader, int bar_id, int nthreads) {
  __threadfence();
  named_bar_sync(bar_id, nthreads);
  if (leader) {
    const int old = atomicAdd(counters + u, 1);
    const int last = (old == nparts - 1) ? 1 : 0;
    if (last) {
      counters[u] = 0;
      __threadfence();
    }
    *reinterpret_cast<volatile int*>(s_flag) = last;
  }
  named_bar_sync(bar_id, nthreads);
  return *reinterpret_cast<volatile int*>(s_flag) != 0;
}

// Warp-cooperative: flag every sequence whose length is outside [lmin, cap]
// (lmin = max(1, new tokens per sequence)).
__device__ __forceinline__ void report_bad_lengths(const int* lens, int b, int lmin, int cap,
                                                   unsigned int* status) {
  bool bad = false;
  for (int idx = threadIdx.x & 31; idx < b; idx += 32) {
    const int L = __ldg(lens + idx);
    bad |= (L < 1 || L < lmin || L > cap);
  }
  if (__any_sync(0xffffffffu, bad) && (threadIdx.x & 31) == 0)
    atomicOr(status, GQA_DEV_BAD_SEQ_LEN);
}

// Block-table lookups of a paged cache for one warp walking a sequence's
// blocks in increasing order: lane l holds entries base + l and base + 32 + l
// (the next chunk is loaded while the current one is used).  Entries past
// the sequence's used blocks read as -1.  Every lane must call get() with the
// same, non-decreasing block index.
struct PageCursor {
  const int* row;  // the sequence's table row
  int nvalid;      // blocks in use
  int base;
  int cur, nxt;

  __device__ int load(int k) const {
    return k < nvalid ? __ldg(row + k) : -1;
  }
  __device__ void start(const int* table_row, int blocks_in_use, int first_block) {
    const int lane = threadIdx.x & 31;
    row = table_row;
    nvalid = blocks_in_use;
    base = first_block & ~31;
    cur = load(base + lane);
    nxt = load(base + 32 + lane);
  }
  __device__ void advance_to(int m) {
    const int lane = threadIdx.x & 31;
    while (m >= base + 32) {
      base += 32;
      cur = nxt;
      nxt = load(base + 32 + lane);
    }
  }
  __device__ int get(int m) {
    advance_to(m);
    return __shfl_sync(0xffffffffu, cur, m - base);
  }
  // Lane l gets entry m + l, for l < 32 (m + l may lie in the next chunk).
  __device__ int get_lanes(int m) {
    const int lane = threadIdx.x & 31;
    advance_to(m);
    const int k = m - base + lane;  // 0 .. 62
    const int a = __shfl_sync(0xffffffffu, cur, k & 31);
    const int c = __shfl_sync(0xffffffffu, nxt, k & 31);
    return k < 32 ? a : c;
  }
};

struct Walker {
  const int* lens;
  int b, g, lmin, cap, T;
  long long W;         // total tiles of the launch
  int nc;              // CTAs of the launch
  bool equal;          // every sequence has the same, nonzero, number of tiles
  long long pos, end;  // global tile cursor and end of this CTA's range
  int i, j, lt, ti, L;

  // total tiles W (warp-cooperative; all lanes get the result); `equal`:
  // every sequence has the same, nonzero, number of tiles
  __device__ static long long total_tiles(const int* lens, int b, int g, int lmin, int cap,
                                         int T, bool* equal = nullptr) {
    const int lane = threadIdx.x & 31;
    long long acc = 0;
    int tmin = 0x7fffffff, tmax = 0;
    for (int base = 0; base < b; base += 32) {
      const int idx = base + lane;
      int t = 0;
      if (idx < b) {
        t = seq_tiles(__ldg(lens + idx), lmin, cap, T);
        tmin = min(tmin, t);
        tmax = max(tmax, t);
      }
      acc += t;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      acc += __shfl_xor_sync(0xffffffffu, acc, o);
      tmin = min(tmin, __shfl_xor_sync(0xffffffffu, tmin, o));
      tmax = max(tmax, __shfl_xor_sync(0xffffffffu, tmax, o));
    }
    if (equal) *equal = tmin == tmax && tmin > 0;
    return acc * g;
  }

  // Position the walker at CTA `c` of `nc`; sequences shorter than lmin
  // (the step's new tokens) are skipped.  whole_max: with equal lengths,
  // CTAs may take up to this many whole units each (0: never).
  // Warp-cooperative.
  __device__ void init(const int* lens_, int b_, int g_, int lmin_, int cap_, int T_, int c,
                       int nc, int whole_max = 0) {
    lens = lens_;
    b = b_;
    g = g_;
    lmin = lmin_;
    cap = cap_;
    T = T_;
    equal = false;
    W = total_tiles(lens, b, g, lmin, cap, T, &equal);
    // Equal lengths: k = 1 or 2 whole units per CTA when that still uses at
    // least 70 % of the CTAs, the rest idle (no piece to merge).  Measured on
    // the tensor-core kernel: 128 units on 152 SMs 46.9 -> 42.5 us per call
    // (64-wide heads 35.5 -> 31.1), 256 units of 128-wide heads two per CTA
    // 153.2 -> 151.2; slower with two per CTA at 64-wide heads (a CTA's own
    // loop is the limit there), with four per CTA, and, decided on the host,
    // with ragged lengths.
    const long long units = static_cast<long long>(b) * g;
    if (equal && whole_max > 0) {
      const long long k = (units + nc - 1) / nc;  // units per CTA
      if (k <= whole_max && units % k == 0 && units / k < nc &&
          10 * (units / k) >= 7 * static_cast<long long>(nc))
        nc = static_cast<int>(units / k);
    }
    this->nc = nc;
    pos = c < nc ? (W * c) / nc : W;
    end = c < nc ? (W * (c + 1)) / nc : W;
    i = b;
    j = 0;
    lt = 0;
    ti = 0;
    L = 0;
    if (pos >= end) return;
    // find sequence i with g * P_i <= pos < g * P_{i+1}
    const int lane = threadIdx.x & 31;
    long long carry = 0;  // g * (tiles before this chunk)
    for (int base = 0; base < b; base += 32) {
      const int idx = base + lane;
      int Lx = 0, t = 0;
      if (idx < b) {
        Lx = __ldg(lens + idx);
        t = seq_tiles(Lx, lmin, cap, T);
      }
      long long incl = static_cast<long long>(t) * g;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const long long y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      const long long lo = carry + incl - static_cast<long long>(t) * g;
      const long long hi = carry + incl;
      const unsigned hit = __ballot_sync(0xffffffffu, idx < b && t > 0 && lo <= pos && pos < hi);
      if (hit) {
        const int src = __ffs(hit) - 1;
        const long long lo_s = __shfl_sync(0xffffffffu, lo, src);
        const int t_s = __shfl_sync(0xffffffffu, t, src);
        i = base + src;
        ti = t_s;
        L = __shfl_sync(0xffffffffu, Lx, src);
        const long long off = pos - lo_s;
        j = static_cast<int>(off / t_s);
        lt = static_cast<int>(off % t_s);
        return;
      }
      carry = __shfl_sync(0xffffffffu, hi, 31);
    }
    pos = end;  // not reached for a consistent plan
  }

  // Next segment of this CTA's range; false when the range is exhausted.
  __device__ bool next(Segment& s) {
    if (pos >= end) return false;
    const long long left = end - pos;
    const int lt1 = (ti - lt <= left) ? ti : lt + static_cast<int>(left);
    s.i = i;
    s.j = j;
    s.lt0 = lt;
    s.lt1 = lt1;
    s.L = L;
    s.ti = ti;
    s.u0 = pos - lt;
    pos += lt1 - lt;
    lt = lt1;
    if (lt == ti && pos < end) {
      lt = 0;
      if (++j == g) {
        j = 0;
        do {
          ++i;
          L = (i < b) ? __ldg(lens + i) : 0;
          ti = (i < b) ? seq_tiles(L, lmin, cap, T) : 0;
        } while (i < b && ti == 0);
      }
    }
    return true;
  }
};

}  // namespace gqa
