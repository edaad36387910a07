// Merge of partial attention results over disjoint key ranges (the combine
// step of a split over the keys: "8.3 FlashAttention-3" section 7.3 names ring
// attention, and the "Discussion Points" of the FlashAttention-2 review a
// decoding kernel that splits the keys).  Per row, from the partial
// (O_s, LSE_s):
//   m = max_s LSE_s,  l = sum_s exp(LSE_s - m),
//   LSE = m + log l,  O = sum_s exp(LSE_s - m) O_s / l.
// Splits whose LSE is -inf (no visible key) contribute nothing (their O is
// ignored, selected away rather than multiplied by zero); a row with no key
// at all gets O = 0 and LSE = -inf.
//
// d/8 lanes per row (8 values, one 16-byte read of each split's row per
// lane), so a warp merges 32/(d/8) rows at once (rounded down: at d = 96
// lanes 24-31 idle; at d = 192 and 256 one row per warp).  One pass over the splits, four at a time (their LSE
// and O reads in flight together): the running maximum m rises with each
// group and the sums gathered so far are scaled by exp(m_old - m_new), as in
// the online softmax, so no separate pass over the LSEs waits on memory
// first; grid-stride over rows; arithmetic in fp32.  Launched as a
// programmatic dependent of the previous kernel on the stream: its launch
// overlaps the tail of a producer that signals early (the decoding kernel
// does, once its key stream is done), and it waits for that grid's
// completion before its first read.
#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <atomic>
#include <cstdint>

#include "merge.cuh"
#include "sm103_ptx.cuh"
#include "smem_attr.cuh"

namespace attn {

namespace {

template <bool BF16>
__device__ __forceinline__ void unpack8(const uint4& w, float (&x)[8]) {
  const uint32_t wd[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    if (BF16) {
      x[2 * i] = __uint_as_float(wd[i] << 16);
      x[2 * i + 1] = __uint_as_float(wd[i] & 0xFFFF0000u);
    } else {
      x[2 * i] = __half2float(__ushort_as_half((unsigned short)(wd[i] & 0xFFFFu)));
      x[2 * i + 1] = __half2float(__ushort_as_half((unsigned short)(wd[i] >> 16)));
    }
  }
}

template <int D, bool BF16>
__global__ void __launch_bounds__(256) merge_kernel(const uint16_t* __restrict__ o_part,
                                                    const float* __restrict__ lse_part,
                                                    int n_split, long rows,
                                                    uint16_t* __restrict__ o,
                                                    float* __restrict__ lse) {
  // launched as a programmatic dependent of the kernel that wrote the
  // partials: wait until that grid has completed and its writes are visible
  asm volatile("griddepcontrol.wait;" ::: "memory");
  constexpr int kLanesPerRow = D / 8;
  constexpr int kRowsPerWarp = 32 / kLanesPerRow;
  constexpr int kBatch = 4;  // splits whose rows are read together
  const int lane = threadIdx.x & 31;
  const int sub = lane / kLanesPerRow;  // row of the warp
  const int col = (lane % kLanesPerRow) * 8;
  const long warp0 = ((long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const long nwarps = ((long)gridDim.x * blockDim.x) >> 5;
  for (long row0 = warp0 * kRowsPerWarp; row0 < rows; row0 += nwarps * kRowsPerWarp) {
    const long row = row0 + sub;
    const bool live = sub < kRowsPerWarp && row < rows;
    const long rrow = live ? row : rows - 1;  // in-range address for idle lanes
    float m = -INFINITY;  // the largest LSE_s so far
    float acc[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] = 0.f;
    float l = 0.f;
    for (int s0 = 0; s0 < n_split; s0 += kBatch) {
      uint4 w[kBatch];
      float ls[kBatch];
#pragma unroll
      for (int k = 0; k < kBatch; ++k) {
        const int sk = min(s0 + k, n_split - 1);
        ls[k] = s0 + k < n_split ? lse_part[(size_t)sk * rows + rrow] : -INFINITY;
        w[k] = *reinterpret_cast<const uint4*>(o_part + ((size_t)sk * rows + rrow) * D + col);
      }
      float mb = ls[0];
#pragma unroll
      for (int k = 1; k < kBatch; ++k) mb = fmaxf(mb, ls[k]);
      if (mb > m) {
        // a group with a larger LSE: rescale what was gathered (nothing yet
        // while m is -inf)
        const float sc = m == -INFINITY ? 0.f : expf(m - mb);
        l *= sc;
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] *= sc;
        m = mb;
      }
#pragma unroll
      for (int k = 0; k < kBatch; ++k) {
        const bool use = ls[k] != -INFINITY;
        const float wt = use ? expf(ls[k] - m) : 0.f;
        l += wt;
        float x[8];
        unpack8<BF16>(w[k], x);
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] = use ? fmaf(wt, x[e], acc[e]) : acc[e];
      }
    }
    const float inv = l > 0.f ? 1.f / l : 0.f;
    uint32_t packed[4];
#pragma unroll
    for (int e = 0; e < 4; ++e)
      packed[e] = BF16 ? pack_bf16x2(acc[2 * e] * inv, acc[2 * e + 1] * inv)
                       : pack_f16x2(acc[2 * e] * inv, acc[2 * e + 1] * inv);
    if (live) {
      *reinterpret_cast<uint4*>(o + (size_t)row * D + col) =
          make_uint4(packed[0], packed[1], packed[2], packed[3]);
      if (col == 0) lse[row] = l > 0.f ? m + logf(l) : -INFINITY;
    }
  }
}

// The grid is what the SMs hold at once (the grid-stride loop then gives
// every CTA the same number of rows, with no partial last wave).  CTAs per
// SM are queried once per device and instantiation.
template <int D, bool BF16>
cudaError_t launch_db(const MergeLaunch& a) {
  static std::atomic<int> resident[kMaxAttrDevices];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const bool tracked = dev >= 0 && dev < kMaxAttrDevices;
  int per_sm = tracked ? resident[dev].load(std::memory_order_acquire) : 0;
  if (per_sm == 0) {
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, merge_kernel<D, BF16>, 256, 0);
    if (e != cudaSuccess) return e;
    if (tracked) resident[dev].store(per_sm, std::memory_order_release);
  }
  long blocks = (a.rows + 7) / 8;  // 8 warps (rows) per block
  const long cap = (long)a.num_sms * (per_sm > 0 ? per_sm : 1);
  if (blocks > cap) blocks = cap;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)blocks);
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = a.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, merge_kernel<D, BF16>, static_cast<const uint16_t*>(a.o_part),
                            static_cast<const float*>(a.lse_part), a.n_split, a.rows,
                            static_cast<uint16_t*>(a.o), a.lse);
}

template <int D>
cudaError_t launch_d(const MergeLaunch& a) {
  return a.bf16 ? launch_db<D, true>(a) : launch_db<D, false>(a);
}

}  // namespace

cudaError_t launch_merge(const MergeLaunch& a) {
  switch (a.d) {
    case 64: return launch_d<64>(a);
    case 96: return launch_d<96>(a);
    case 192: return launch_d<192>(a);
    case 256: return launch_d<256>(a);
    default: return launch_d<128>(a);
  }
}

}  // namespace attn
