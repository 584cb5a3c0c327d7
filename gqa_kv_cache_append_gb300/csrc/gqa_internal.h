// gqa_internal.h - host-side interface between the C-ABI layer and the
// kernel translation units (not installed, not part of the ABI).
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace gqa {

// Arguments of one decode-attention launch, already validated by the ABI.
struct DecodeLaunch {
  const void* q;
  const void* k_cache;
  const void* v_cache;
  const int* seq_lens;
  int b, h, g, d, cap, dtype;  // d: head dim of q and K (d_k)
  int dv = 0;            // head dim of V and out (d_v)
  int nq;                // new tokens (queries) per sequence, >= 1
  float scale_log2;      // scale * log2(e): logits are kept in base 2
  void* out;
  float* part_o;         // [slots, nq * r, dv] unnormalised partial outputs
  float* part_ml;        // [slots, nq * r, 2] running max (base 2) and sum
  int* counters;         // [b * g] arrivals per split unit; zero between launches
  const void* k_new;     // fused append: new K/V rows [b, nq, g, d], or null
  const void* v_new;
  void* k_cache_w;       // the caches, written at rows L_i - nq .. L_i - 1
  void* v_cache_w;
  bool early;            // stream the first tiles before the dependency wait
  bool cuda_cores = false;  // the CUDA-core kernel even where tensor cores apply
  unsigned int* status;  // device status word
  long long budget;      // wait limit in SM cycles
  int nc;                // persistent CTAs
  // tensor-core kernel: clusters of `cluster` CTAs (0: no cluster launch),
  // cluster_k of them per (sequence, KV head) unit, nc = units * cluster *
  // cluster_k; with equal lengths the split units are merged across each
  // cluster in distributed shared memory
  int cluster = 0, cluster_k = 1;
  cudaStream_t stream;
  // paged cache (null table: contiguous [b, g, cap, d]): the caches are pools
  // [num_blocks, g, block_size, d]; position p of sequence i is row
  // p % block_size of block block_table[i * max_blocks + p / block_size]
  const int* block_table = nullptr;
  int block_size = 0, max_blocks = 0, num_blocks = 0;
};

// Tiled TMA map over a row-major bf16 tensor: dims[0] is the contiguous
// (innermost) extent, strides[k] the byte stride of dimension k + 1, box the
// copied box; 128-byte swizzle, 256-byte L2 promotion, zero fill outside.
bool encode_bf16_map(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                     const uint64_t* strides, const uint32_t* box, bool bf16 = true);

// CUDA-core kernel (fp32 and bf16, d_k and d_v in {64, 128}); `cols` = nq * r
// query rows per KV head
bool simt_supported(int dtype, int d_k, int d_v, int cols);
int simt_tile(int dtype, int d_k, int d_v);
int simt_ctas_per_sm(int dtype, int d, int r);
cudaError_t launch_decode_simt(const DecodeLaunch& a);

// tcgen05 tensor-core kernel (bf16 and fp16, d_k and d_v in {64, 128}, up to
// 32 query rows per KV head; also d_k, d_v in {128, 192, 256}, up to 16
// rows)
bool tc_supported(int dtype, int d_k, int d_v, int cols, bool paged);
int tc_tile(int d_k, int d_v);  // positions per tile (256 for d_k = d_v = 64, else 128)
// clusters of csize CTAs of the tensor-core kernel that fit on the device
// at once (one CTA per SM); 0 if none or the query failed
int tc_max_clusters(int csize);
int tc_ctas_per_sm(int r);
cudaError_t launch_decode_tc(const DecodeLaunch& a);

// tcgen05 projection GEMMs around the step (bf16, 128-wide heads):
// mode 0: q / k_new / v_new = x . P_q / P_k / P_v; mode 1: y = o . P_o
struct ProjLaunch {
  int mode;
  const void* w0;        // P_q (mode 0) or P_o (mode 1), [heads, D, 128]
  const void* w1;        // P_k [g, D, 128] (mode 0)
  const void* w2;        // P_v [g, D, 128] (mode 0)
  const void* x;         // x [b, D] (mode 0) or o [b, h, 128] (mode 1)
  void* out0;            // q [b, h, 128] (mode 0) or y [b, D] (mode 1)
  void* out1;            // k_new [b, g, 128] (mode 0)
  void* out2;            // v_new [b, g, 128] (mode 0)
  int b, D, h, g;
  float* part;           // [tiles + nc, NB, 128] fp32 partial sums
  int* counters;         // [tiles] arrivals; zero between launches
  unsigned int* status;
  long long budget;
  bool early;            // stream the weights before the dependency wait
  int nc;
  cudaStream_t stream;
};

int proj_nb(int b);                                   // batch columns of the MMA
long long proj_work(int mode, int D, int h, int g);   // K chunks of the launch
int proj_tiles(int mode, int D, int h, int g);
cudaError_t launch_proj(const ProjLaunch& a);

}  // namespace gqa
