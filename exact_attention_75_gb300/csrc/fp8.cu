// FP8 E4M3 block quantization with the optional randomized Hadamard rotation
// ("8.3 FlashAttention-3", section 5.1 block quantization and section 5.2
// incoherent processing).
//
// One CTA per (batch*head, block of 64 rows), 8 warps of 8 rows each; four
// lanes share a row: lane (r = lane/4, q = lane%4) holds the d/4 values with
// index 32k + 8q + j (k < d/32, j < 8), loaded as d/32 chunks of 16 bytes.
//
// Rotation: x R = (x H_d) diag(signs) / sqrt(d).  The fast Walsh-Hadamard
// transform pairs index i with i ^ 2^b for every bit b; bits 0-2 and 5-6 are
// register strides 1, 2, 4, 8, 16 (packed fp32x2 adds except stride 1), bits
// 3-4 pair lanes through shuffles.  1/sqrt(d) is folded into the block's
// quantization multiplier and the signs are applied to the codes (E4M3 is
// sign-magnitude, so flipping bit 7 of a code negates it).
//
// Scale and codes: s = amax / 448 (one IEEE fp32 division; 1 for an all-zero
// block), code = E4M3(RN(x / s)), round to nearest even, saturating.  Without
// the rotation the codes are exact: t = RN(x * RN(1/s)) differs from x / s by
// less than 3 units in the last place, E4M3 rounding is monotone, so when the
// codes of t's neighbours 4 ulp below and above agree, that is the code of
// RN(x / s); a thread with any disagreeing pair (rare, and every zero)
// recomputes its codes with the IEEE division.
#include <cuda_runtime.h>
#include <cstdint>

#include "fp8.cuh"
#include "sm103_ptx.cuh"

namespace attn {

namespace {

constexpr int kRowsPerBlock = 64;
constexpr int kWarps = 8;
constexpr float kE4M3Max = 448.f;

__device__ __forceinline__ float2 f2(float a, float b) { return make_float2(a, b); }

// Codes of two values whose float bit patterns are moved by `delta` units in
// the last place (towards zero for negative delta on the magnitude).
__device__ __forceinline__ uint16_t codes_nudged(float2 t, int delta) {
  return pack_e4m3x2(__uint_as_float(__float_as_uint(t.x) + (uint32_t)delta),
                     __uint_as_float(__float_as_uint(t.y) + (uint32_t)delta));
}

template <int D, bool ROTATE, bool TRANSPOSED>
__global__ void __launch_bounds__(kWarps * 32) quantize_kernel(const uint16_t* __restrict__ x,
                                                               uint8_t* __restrict__ out,
                                                               float* __restrict__ scales,
                                                               const int8_t* __restrict__ signs,
                                                               int N, int nblk) {
  constexpr int K = D / 32;             // 16-byte chunks per lane
  constexpr int E = 8 * K;              // values per lane
  constexpr int W = 2 * K;              // code words (4 codes each) per lane
  constexpr int kTileWords = D / 4 + 1; // staging row stride (transposed output)
  __shared__ float warp_max[kWarps];
  __shared__ uint32_t tile[TRANSPOSED ? kRowsPerBlock * kTileWords : 1];
  // the d signs, staged once per CTA so that each lane reads its flip masks
  // as four-byte words (ordered before their use by the block-max barrier)
  __shared__ __align__(16) int8_t sgn[ROTATE ? D : 16];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if constexpr (ROTATE) {
    if (threadIdx.x < D) sgn[threadIdx.x] = signs[threadIdx.x];
  }
  const int q = lane & 3;
  const int bh = blockIdx.x / nblk;
  const int blk = blockIdx.x - bh * nblk;
  const int row0 = blk * kRowsPerBlock;
  const int lrow = warp * 8 + (lane >> 2);
  const int row = row0 + lrow;
  const bool live = row < N;

  float v[E];
  {
    uint4 raw[K];
    const uint16_t* src = x + ((size_t)bh * N + (live ? row : 0)) * D + 8 * q;
#pragma unroll
    for (int k = 0; k < K; ++k)
      raw[k] = live ? *reinterpret_cast<const uint4*>(src + 32 * k) : make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int k = 0; k < K; ++k) {
      const uint32_t w4[4] = {raw[k].x, raw[k].y, raw[k].z, raw[k].w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        v[8 * k + 2 * i] = __uint_as_float(w4[i] << 16);
        v[8 * k + 2 * i + 1] = __uint_as_float(w4[i] & 0xFFFF0000u);
      }
    }
  }

  if constexpr (ROTATE) {
    // register butterflies: stride 1 scalar, strides 2..E/2 on packed pairs
#pragma unroll
    for (int e = 0; e < E; e += 2) {
      const float a = v[e], b = v[e + 1];
      v[e] = a + b;
      v[e + 1] = a - b;
    }
#pragma unroll
    for (int st = 2; st < E; st <<= 1) {
#pragma unroll
      for (int e = 0; e < E; e += 2) {
        if ((e & st) == 0) {
          const float2 a = f2(v[e], v[e + 1]), b = f2(v[e + st], v[e + st + 1]);
          const float2 sum = __fadd2_rn(a, b), dif = __ffma2_rn(b, f2(-1.f, -1.f), a);
          v[e] = sum.x;
          v[e + 1] = sum.y;
          v[e + st] = dif.x;
          v[e + st + 1] = dif.y;
        }
      }
    }
    // lane butterflies (index bits 3 and 4): the upper partner keeps o - v
#pragma unroll
    for (int m = 1; m <= 2; m <<= 1) {
      const float sl = (q & m) ? -1.f : 1.f;
#pragma unroll
      for (int e = 0; e < E; e += 2) {
        const float o0 = __shfl_xor_sync(0xffffffffu, v[e], m);
        const float o1 = __shfl_xor_sync(0xffffffffu, v[e + 1], m);
        const float2 r = __ffma2_rn(f2(v[e], v[e + 1]), f2(sl, sl), f2(o0, o1));
        v[e] = r.x;
        v[e + 1] = r.y;
      }
    }
  }

  float amax = 0.f;
#pragma unroll
  for (int e = 0; e < E; e += 2) amax = fmax3(amax, fabsf(v[e]), fabsf(v[e + 1]));
#pragma unroll
  for (int off = 16; off > 0; off >>= 1)
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
  if (lane == 0) warp_max[warp] = amax;
  __syncthreads();
  float bmax = warp_max[0];
#pragma unroll
  for (int w2 = 1; w2 < kWarps; ++w2) bmax = fmaxf(bmax, warp_max[w2]);
  // with the rotation, v is x H_d; the normalised block maximum is
  // RN(max|x H_d| / sqrt(d)), the same as the maximum of the rounded values
  const float inv_sqrt_d = 1.0f / sqrtf((float)D);
  if (ROTATE) bmax *= inv_sqrt_d;
  const float s = bmax > 0.f ? __fdiv_rn(bmax, kE4M3Max) : 1.0f;
  if (threadIdx.x == 0) scales[(size_t)bh * nblk + blk] = s;

  uint32_t code[W];
  const float mult = ROTATE ? __fdiv_rn(inv_sqrt_d, s) : __frcp_rn(s);
  // 0x80 in each byte whose sign is negative (bit 7 of the int8 sign)
  uint32_t flip[W];
  if constexpr (ROTATE) {
#pragma unroll
    for (int w = 0; w < W; ++w)
      flip[w] = *reinterpret_cast<const uint32_t*>(sgn + 32 * (w >> 1) + 8 * q + 4 * (w & 1)) &
                0x80808080u;
  }
  const float2 mult2 = f2(mult, mult);
  bool agree = true;
#pragma unroll
  for (int w = 0; w < W; ++w) {
    uint32_t word = 0;
#pragma unroll
    for (int p = 0; p < 2; ++p) {
      const int e = 4 * w + 2 * p;
      const float2 t = __fmul2_rn(f2(v[e], v[e + 1]), mult2);
      uint16_t two;
      if constexpr (ROTATE) {
        two = pack_e4m3x2(t.x, t.y);
      } else {
        two = codes_nudged(t, -4);
        agree &= two == codes_nudged(t, 4);
      }
      word |= (uint32_t)two << (16 * p);
    }
    code[w] = ROTATE ? word ^ flip[w] : word;
  }
  if (!ROTATE && !agree) {
#pragma unroll
    for (int w = 0; w < W; ++w) {
      const int e = 4 * w;
      code[w] = (uint32_t)pack_e4m3x2(__fdiv_rn(v[e], s), __fdiv_rn(v[e + 1], s)) |
                ((uint32_t)pack_e4m3x2(__fdiv_rn(v[e + 2], s), __fdiv_rn(v[e + 3], s)) << 16);
    }
  }

  if constexpr (!TRANSPOSED) {
    if (live) {
      uint8_t* dst = out + ((size_t)bh * N + row) * D + 8 * q;
#pragma unroll
      for (int k = 0; k < K; ++k)
        *reinterpret_cast<uint2*>(dst + 32 * k) = make_uint2(code[2 * k], code[2 * k + 1]);
    }
  } else {
    // stage the codes row-major (word = 4 columns), then write out [bh][D][N]:
    // a task takes 4 rows x 4 columns, transposes the 4x4 bytes and stores one
    // word (4 consecutive rows) into each of the 4 output rows.
#pragma unroll
    for (int w = 0; w < W; ++w) tile[lrow * kTileWords + 8 * (w >> 1) + 2 * q + (w & 1)] = code[w];
    __syncthreads();
    const int nrows = min(kRowsPerBlock, N - row0);  // a multiple of 16
#pragma unroll
    for (int task = threadIdx.x; task < 16 * (D / 4); task += kWarps * 32) {
      const int g = task & 15, cw = task >> 4;
      if (4 * g >= nrows) continue;
      const uint32_t a0 = tile[(4 * g + 0) * kTileWords + cw];
      const uint32_t a1 = tile[(4 * g + 1) * kTileWords + cw];
      const uint32_t a2 = tile[(4 * g + 2) * kTileWords + cw];
      const uint32_t a3 = tile[(4 * g + 3) * kTileWords + cw];
      const uint32_t t0 = __byte_perm(a0, a1, 0x5140), t1 = __byte_perm(a0, a1, 0x7362);
      const uint32_t u0 = __byte_perm(a2, a3, 0x5140), u1 = __byte_perm(a2, a3, 0x7362);
      const uint32_t col[4] = {__byte_perm(t0, u0, 0x5410), __byte_perm(t0, u0, 0x7632),
                               __byte_perm(t1, u1, 0x5410), __byte_perm(t1, u1, 0x7632)};
      uint8_t* dst = out + ((size_t)bh * D + 4 * cw) * N + row0 + 4 * g;
#pragma unroll
      for (int b = 0; b < 4; ++b) *reinterpret_cast<uint32_t*>(dst + (size_t)b * N) = col[b];
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
