// FP8 E4M3 block quantization with the optional randomized Hadamard rotation
// ("8.3 FlashAttention-3", section 5.1 block quantization and section 5.2
// incoherent processing).
//
// One CTA per (batch*head, block of 64 rows); each warp owns 8 rows.  With the
// rotation, every row x (d values) becomes (x H_d) o signs / sqrt(d) through
// an in-register fast Walsh-Hadamard transform: lane l holds the d/32
// consecutive values [l*d/32, (l+1)*d/32); butterflies of stride < d/32 stay
// in registers, larger strides pair lanes with __shfl_xor_sync.  The block
// scale is s = amax / 448 (one IEEE fp32 division; 1 for an all-zero block)
// and the codes are E4M3(x / s), round to nearest even, saturating.
#include <cuda_runtime.h>
#include <cstdint>

#include "fp8.cuh"
#include "sm103_ptx.cuh"

namespace attn {

namespace {

constexpr int kRowsPerBlock = 64;
constexpr int kWarps = 8;
constexpr float kE4M3Max = 448.f;

template <int D, bool ROTATE, bool TRANSPOSED>
__global__ void __launch_bounds__(kWarps * 32) quantize_kernel(const uint16_t* __restrict__ x,
                                                               uint8_t* __restrict__ out,
                                                               float* __restrict__ scales,
                                                               const int8_t* __restrict__ signs,
                                                               int N, int nblk) {
  constexpr int E = D / 32;  // values per lane
  constexpr int kRowsPerWarp = kRowsPerBlock / kWarps;
  __shared__ float warp_max[kWarps];
  __shared__ __align__(16) uint8_t tile[TRANSPOSED ? kRowsPerBlock * (D + 4) : 16];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int bh = blockIdx.x / nblk;
  const int blk = blockIdx.x - bh * nblk;
  const int row0 = blk * kRowsPerBlock;

  float sgn[E];
  if (ROTATE) {
    const float inv_sqrt_d = 1.0f / sqrtf((float)D);
#pragma unroll
    for (int e = 0; e < E; ++e) sgn[e] = (float)signs[lane * E + e] * inv_sqrt_d;
  }

  float v[kRowsPerWarp][E];
  float amax = 0.f;
#pragma unroll
  for (int rr = 0; rr < kRowsPerWarp; ++rr) {
    const int row = row0 + warp * kRowsPerWarp + rr;
#pragma unroll
    for (int e = 0; e < E; ++e) v[rr][e] = 0.f;
    if (row < N) {  // warp-uniform
      const uint16_t* src = x + ((size_t)bh * N + row) * D + lane * E;
      uint32_t w[E / 2];
      if constexpr (E == 4) {
        const uint2 t = *reinterpret_cast<const uint2*>(src);
        w[0] = t.x;
        w[1] = t.y;
      } else {
        w[0] = *reinterpret_cast<const uint32_t*>(src);
      }
#pragma unroll
      for (int e = 0; e < E / 2; ++e) {
        v[rr][2 * e] = __uint_as_float(w[e] << 16);
        v[rr][2 * e + 1] = __uint_as_float(w[e] & 0xFFFF0000u);
      }
      if (ROTATE) {
        // in-register butterflies (strides 1 .. E/2)
#pragma unroll
        for (int s = 1; s < E; s <<= 1) {
#pragma unroll
          for (int e = 0; e < E; ++e) {
            if ((e & s) == 0) {
              const float a = v[rr][e], b = v[rr][e + s];
              v[rr][e] = a + b;
              v[rr][e + s] = a - b;
            }
          }
        }
        // cross-lane butterflies (strides E .. D/2)
#pragma unroll
        for (int m = 1; m < 32; m <<= 1) {
#pragma unroll
          for (int e = 0; e < E; ++e) {
            const float o = __shfl_xor_sync(0xffffffffu, v[rr][e], m);
            v[rr][e] = (lane & m) ? (o - v[rr][e]) : (v[rr][e] + o);
          }
        }
#pragma unroll
        for (int e = 0; e < E; ++e) v[rr][e] *= sgn[e];
      }
#pragma unroll
      for (int e = 0; e < E; ++e) amax = fmaxf(amax, fabsf(v[rr][e]));
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1)
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
  if (lane == 0) warp_max[warp] = amax;
  __syncthreads();
  float bmax = warp_max[0];
#pragma unroll
  for (int w2 = 1; w2 < kWarps; ++w2) bmax = fmaxf(bmax, warp_max[w2]);
  const float s = bmax > 0.f ? __fdiv_rn(bmax, kE4M3Max) : 1.0f;
  if (threadIdx.x == 0) scales[(size_t)bh * nblk + blk] = s;

#pragma unroll
  for (int rr = 0; rr < kRowsPerWarp; ++rr) {
    const int lrow = warp * kRowsPerWarp + rr;
    const int row = row0 + lrow;
    uint32_t packed = 0;
#pragma unroll
    for (int e = 0; e < E; e += 2) {
      const uint16_t two = pack_e4m3x2(__fdiv_rn(v[rr][e], s), __fdiv_rn(v[rr][e + 1], s));
      packed |= (uint32_t)two << (8 * e);
    }
    if constexpr (!TRANSPOSED) {
      if (row < N) {
        uint8_t* dst = out + ((size_t)bh * N + row) * D + lane * E;
        if constexpr (E == 4)
          *reinterpret_cast<uint32_t*>(dst) = packed;
        else
          *reinterpret_cast<uint16_t*>(dst) = (uint16_t)packed;
      }
    } else {
      uint8_t* t = tile + lrow * (D + 4) + lane * E;
#pragma unroll
      for (int e = 0; e < E; ++e) t[e] = (uint8_t)(packed >> (8 * e));
    }
  }
  if constexpr (TRANSPOSED) {
    // out is [bh][D][N]: column c of this row block becomes 64 contiguous
    // bytes of output row c (rows at or beyond N are not written).
    __syncthreads();
    const int nrows = min(kRowsPerBlock, N - row0);
    for (int idx = threadIdx.x; idx < D * 4; idx += blockDim.x) {
      const int c = idx >> 2, part = idx & 3;  // 16 rows per part
      uint32_t w4[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint32_t word = 0;
#pragma unroll
        for (int b = 0; b < 4; ++b) {
          const int lr = part * 16 + q * 4 + b;
          word |= (uint32_t)tile[lr * (D + 4) + c] << (8 * b);
        }
        w4[q] = word;
      }
      uint8_t* dst = out + ((size_t)bh * D + c) * N + row0 + part * 16;
      if (part * 16 + 16 <= nrows) {
        *reinterpret_cast<uint4*>(dst) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
      } else {
        for (int b = 0; b < 16 && part * 16 + b < nrows; ++b)
          dst[b] = (uint8_t)(w4[b >> 2] >> (8 * (b & 3)));
      }
    }
  }
}

template <int D, bool ROTATE, bool TRANSPOSED>
cudaError_t launch_q(const QuantLaunch& a) {
  const int nblk = (a.N + kRowsPerBlock - 1) / kRowsPerBlock;
  const long grid = (long)a.BH * nblk;
  if (grid > 0x7FFFFFFFL) return cudaErrorInvalidValue;
  quantize_kernel<D, ROTATE, TRANSPOSED><<<(int)grid, kWarps * 32, 0, a.stream>>>(
      static_cast<const uint16_t*>(a.x), static_cast<uint8_t*>(a.out), a.scales, a.signs, a.N,
      nblk);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_q_d(const QuantLaunch& a) {
  const bool rot = a.signs != nullptr;
  if (rot) return a.transposed ? launch_q<D, true, true>(a) : launch_q<D, true, false>(a);
  return a.transposed ? launch_q<D, false, true>(a) : launch_q<D, false, false>(a);
}

}  // namespace

cudaError_t launch_quantize(const QuantLaunch& a) {
  return a.d == 128 ? launch_q_d<128>(a) : launch_q_d<64>(a);
}

}  // namespace attn
