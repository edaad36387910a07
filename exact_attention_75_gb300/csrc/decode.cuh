// Host <-> device interface of the decoding kernel: a few query rows per
// key/value head (grouped query heads x new tokens), 16 per work unit,
// against a key/value cache, split over the keys like the tiled forward.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstddef>
#include <cstdint>

namespace attn {

// Query rows (query heads of a group x queries) one work unit holds at most:
// the M = 16 of the warp-level product.  A key/value head with more rows
// runs ceil(R / 16) units, each streaming the head's keys and values.
constexpr int kDecodeMaxRows = 16;
// Rows per key/value head beyond which the decoding kernel is not used (the
// units of one head re-read its keys and values, from L2 at best).
constexpr int kDecodeRowLimit = 128;
// Keys of one block a warp stages and multiplies (rows of the tensor-map box).
constexpr int kDecodeKeys = 16;

struct DecodeParams {
  const void* q;        // [B, Hkv * G, Nq, D]: the R = G * Nq rows of a unit are contiguous
  void* o;              // [n_split, B, Hkv * G, Nq, D] partial outputs (16-bit)
  float* lse;           // [n_split, B, Hkv * G, Nq] partial log-sum-exps
  uint32_t* status;     // device status word
  int Hkv, R, Nq, Nk;   // R = G * Nq rows per key/value head
  int n_rgroups;        // ceil(R / kDecodeMaxRows)
  int n_split, n_kblocks;  // split s covers 128-key blocks [s nb / n_split, (s+1) nb / n_split)
  int causal;           // query i sees keys j <= i + Nk - Nq
  float scale_log2;     // scale * log2(e)
  size_t o_split, lse_split;  // elements between two splits' partials
  unsigned long long wait_limit_ns;
};

struct DecodeLaunch {
  // K and V as [B * Hkv, Nk, D], box 64 columns x kDecodeKeys rows, 128-byte swizzle
  CUtensorMap tmK, tmV;
  DecodeParams params;
  int num_units;        // B * Hkv * n_split * n_rgroups
  cudaStream_t stream;
};

// d in {64, 96, 128, 192, 256}.
cudaError_t launch_decode(const DecodeLaunch& a, int d, bool bf16);

}  // namespace attn
