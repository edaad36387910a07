// Shared-memory tile conventions shared by the attention kernels.
//
// A 16-bit [128 rows][d] tile is loaded by TMA with the 128-byte swizzle as
// d/64 column halves, each [128 rows][64 values] = 16 KB, 1024-byte aligned.
#pragma once

#include <cstdint>

#include "sm103_ptx.cuh"

namespace attn {

// K-major operand (reduction dim contiguous): rows start at `tile_addr`
// (which may point at a row offset that is a multiple of 8 inside the tile);
// step k16 selects 16 values of the reduction dimension.
__device__ __forceinline__ uint64_t kmajor_desc16(uint32_t tile_addr, int k16) {
  const uint32_t addr = tile_addr + (uint32_t)(k16 >> 2) * 16384u + (uint32_t)(k16 & 3) * 32u;
  return sdesc_sw128(addr, 16, 1024);
}

// MN-major operand (the non-reduction dim contiguous, e.g. V as the B operand
// of P V): 8-row groups along the reduction dim are 1024 B apart (SBO), the
// 64-value column halves 16 KB apart (LBO); step k16 advances 16 rows.
__device__ __forceinline__ uint64_t mnmajor_desc16(uint32_t tile_addr, int k16) {
  return sdesc_sw128(tile_addr + (uint32_t)k16 * 2048u, 16384, 1024);
}

// Snake order over a persistent grid of G CTAs: round k gives CTA c the work
// unit k*G + c (k even) or k*G + G-1-c (k odd).  With units sorted by cost
// (longest first) this evens out the per-CTA totals.
__device__ __forceinline__ int snake_unit(int k, int cta, int G) {
  return k * G + ((k & 1) ? (G - 1 - cta) : cta);
}

}  // namespace attn
