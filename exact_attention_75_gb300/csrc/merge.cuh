// Host <-> device interface of the merge of split partial results.
#pragma once

#include <cuda_runtime.h>
#include <cstdint>

namespace attn {

struct MergeLaunch {
  const void* o_part;     // [n_split, rows, d] 16-bit partial O
  const float* lse_part;  // [n_split, rows] partial LSE (-inf: no key in the split)
  void* o;                // [rows, d] 16-bit merged O
  float* lse;             // [rows] merged LSE
  long rows;              // B * H * N
  int n_split, d;
  bool bf16;
  int num_sms;
  cudaStream_t stream;
};

cudaError_t launch_merge(const MergeLaunch& a);

}  // namespace attn
