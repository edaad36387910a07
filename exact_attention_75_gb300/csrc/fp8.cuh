// Host <-> device interface of the FP8 quantization and FP8 forward kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

#include "fwd.cuh"

namespace attn {

struct QuantLaunch {
  const void* x;         // [B*H, N, d] bf16
  void* out;             // E4M3 codes, [B*H, N, d] or [B*H, d, N] (transposed)
  float* scales;         // [B*H, ceil(N/64)]
  const int8_t* signs;   // d values of +-1, or null (no rotation)
  int BH, N, d;
  bool transposed;
  cudaStream_t stream;
};

cudaError_t launch_quantize(const QuantLaunch& a);

struct Fp8FwdLaunch {
  CUtensorMap tmQ, tmK, tmVt;
  FwdLaunch base;        // params / grid / stream (its tensor maps are unused)
  const float* q_scale;
  const float* k_scale;
  const float* v_scale;
  bool causal;
};

cudaError_t launch_fwd_fp8(const Fp8FwdLaunch& a);

}  // namespace attn
