// Merge of partial attention results over disjoint key ranges (the combine
// step of a split over the keys: "8.3 FlashAttention-3" section 7.3 names ring
// attention, and the "Discussion Points" of the FlashAttention-2 review a
// decoding kernel that splits the keys).  Per row, from the partial
// (O_s, LSE_s):
//   m = max_s LSE_s,  l = sum_s exp(LSE_s - m),
//   LSE = m + log l,  O = sum_s exp(LSE_s - m) O_s / l.
// Splits whose LSE is -inf (no visible key) are skipped without reading their
// O; a row with no key at all gets O = 0 and LSE = -inf.
//
// One warp per row (d/32 values per lane, so each split's row is one
// coalesced 2*d-byte read), grid-stride over rows; arithmetic in fp32.
#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cstdint>

#include "merge.cuh"
#include "sm103_ptx.cuh"

namespace attn {

namespace {

template <int D, bool BF16>
__global__ void __launch_bounds__(256) merge_kernel(const uint16_t* __restrict__ o_part,
                                                    const float* __restrict__ lse_part,
                                                    int n_split, long rows,
                                                    uint16_t* __restrict__ o,
                                                    float* __restrict__ lse) {
  constexpr int E = D / 32;  // values per lane: 4 (d = 128) or 2 (d = 64)
  const long warp0 = ((long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const long nwarps = ((long)gridDim.x * blockDim.x) >> 5;
  const int lane = threadIdx.x & 31;
  for (long row = warp0; row < rows; row += nwarps) {
    float m = -INFINITY;
    for (int s = 0; s < n_split; ++s) m = fmaxf(m, lse_part[(size_t)s * rows + row]);
    float acc[E];
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] = 0.f;
    float l = 0.f;
    if (m != -INFINITY) {
      for (int s = 0; s < n_split; ++s) {
        const float ls = lse_part[(size_t)s * rows + row];
        if (ls == -INFINITY) continue;  // warp-uniform
        const float w = expf(ls - m);
        l += w;
        const uint16_t* src = o_part + ((size_t)s * rows + row) * D + lane * E;
        uint32_t word[E / 2];
        if constexpr (E == 4) {
          const uint2 t = *reinterpret_cast<const uint2*>(src);
          word[0] = t.x;
          word[1] = t.y;
        } else {
          word[0] = *reinterpret_cast<const uint32_t*>(src);
        }
#pragma unroll
        for (int e = 0; e < E / 2; ++e) {
          float lo, hi;
          if (BF16) {
            lo = __uint_as_float(word[e] << 16);
            hi = __uint_as_float(word[e] & 0xFFFF0000u);
          } else {
            lo = __half2float(__ushort_as_half((unsigned short)(word[e] & 0xFFFFu)));
            hi = __half2float(__ushort_as_half((unsigned short)(word[e] >> 16)));
          }
          acc[2 * e] = fmaf(w, lo, acc[2 * e]);
          acc[2 * e + 1] = fmaf(w, hi, acc[2 * e + 1]);
        }
      }
    }
    const float inv = l > 0.f ? 1.f / l : 0.f;
    uint32_t packed[E / 2];
#pragma unroll
    for (int e = 0; e < E / 2; ++e)
      packed[e] = BF16 ? pack_bf16x2(acc[2 * e] * inv, acc[2 * e + 1] * inv)
                       : pack_f16x2(acc[2 * e] * inv, acc[2 * e + 1] * inv);
    uint16_t* dst = o + (size_t)row * D + lane * E;
    if constexpr (E == 4)
      *reinterpret_cast<uint2*>(dst) = make_uint2(packed[0], packed[1]);
    else
      *reinterpret_cast<uint32_t*>(dst) = packed[0];
    if (lane == 0) lse[row] = l > 0.f ? m + logf(l) : -INFINITY;
  }
}

template <int D>
cudaError_t launch_d(const MergeLaunch& a) {
  long blocks = (a.rows + 7) / 8;  // 8 warps (rows) per block
  const long cap = (long)a.num_sms * 16;
  if (blocks > cap) blocks = cap;
  const auto* op = static_cast<const uint16_t*>(a.o_part);
  auto* out = static_cast<uint16_t*>(a.o);
  if (a.bf16)
    merge_kernel<D, true><<<(int)blocks, 256, 0, a.stream>>>(op, a.lse_part, a.n_split, a.rows,
                                                             out, a.lse);
  else
    merge_kernel<D, false><<<(int)blocks, 256, 0, a.stream>>>(op, a.lse_part, a.n_split,
                                                              a.rows, out, a.lse);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_merge(const MergeLaunch& a) {
  return a.d == 128 ? launch_d<128>(a) : launch_d<64>(a);
}

}  // namespace attn
