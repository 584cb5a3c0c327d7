// gqa_internal.h - host-side interface between the C-ABI layer and the
// kernel translation units (not installed, not part of the ABI).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace gqa {

// Arguments of one decode-attention launch, already validated by the ABI.
struct DecodeLaunch {
  const void* q;
  const void* k_cache;
  const void* v_cache;
  const int* seq_lens;
  int b, h, g, d, cap, dtype;
  int nq;                // new tokens (queries) per sequence, >= 1
  float scale_log2;      // scale * log2(e): logits are kept in base 2
  void* out;
  float* part_o;         // [slots, nq * r, d] unnormalised partial outputs
  float* part_ml;        // [slots, nq * r, 2] running max (base 2) and sum
  int* counters;         // [b * g] arrivals per split unit; zero between launches
  const void* k_new;     // fused append: new K/V rows [b, nq, g, d], or null
  const void* v_new;
  void* k_cache_w;       // the caches, written at rows L_i - nq .. L_i - 1
  void* v_cache_w;
  bool early;            // stream the first tiles before the dependency wait
  unsigned int* status;  // device status word
  long long budget;      // wait limit in SM cycles
  int nc;                // persistent CTAs
  cudaStream_t stream;
};

// CUDA-core kernel (fp32, and bf16 with d = 64); `cols` = nq * r query rows
// per KV head
bool simt_supported(int dtype, int d, int cols);
int simt_tile(int dtype, int d);
int simt_ctas_per_sm(int dtype, int d, int r);
cudaError_t launch_decode_simt(const DecodeLaunch& a);

// tcgen05 tensor-core kernel (bf16, d = 128)
bool tc_supported(int dtype, int d, int cols);
int tc_tile();
int tc_ctas_per_sm(int r);
cudaError_t launch_decode_tc(const DecodeLaunch& a);


}  // namespace gqa
