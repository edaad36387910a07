// Shared-memory tile conventions shared by the attention kernels.
//
// A 16-bit [128 rows][d] tile is loaded by TMA with the 128-byte swizzle as
// column halves, each [128 rows][64 values] = 16 KB, 1024-byte aligned.  A
// head dim that is not a multiple of 64 (d = 96) occupies the columns of the
// next multiple: TMA fills the columns past d with zeros, so products that
// contract over d stop at d, and products with d outputs per row are issued
// with N = d (an MN-major operand of 96 columns reads one and a half 128-byte
// swizzle atoms from an atom-aligned base).
#pragma once

#include <cstdint>

#include "sm103_ptx.cuh"

namespace attn {

// Columns a 128-row tile of head dim D occupies in shared and tensor memory.
template <int D>
constexpr int kPaddedD = (D + 63) / 64 * 64;

// Cheap K-step addressing for the MMA issuer.  A single thread issues every
// tcgen05.mma of a CTA, so building descriptors from scratch per instruction
// (masking, shifting, OR-ing 64-bit fields) costs more issue cycles than the
// tensor core needs to execute an N=128 MMA.  Instead the issuer builds one
// base descriptor per tile and adds a compile-time byte offset >> 4 to the
// start-address field (bits 0-13; shared-memory addresses stay below 256 KB,
// so the field cannot carry into the neighbouring bits).
__device__ __forceinline__ uint64_t desc_plus(uint64_t desc, uint32_t byte_off) {
  return desc + (uint64_t)(byte_off >> 4);
}
// K-major 16-bit tile: byte offset of reduction step k16 (16 values).
__host__ __device__ constexpr uint32_t kmajor16_off(int k16) {
  return (uint32_t)(k16 >> 2) * 16384u + (uint32_t)(k16 & 3) * 32u;
}
// MN-major 16-bit tile: byte offset of reduction step k16 (16 rows).
__host__ __device__ constexpr uint32_t mnmajor16_off(int k16) { return (uint32_t)k16 * 2048u; }
// Base descriptors (K-step 0).
__device__ __forceinline__ uint64_t kmajor_base(uint32_t tile_addr) {
  return sdesc_sw128(tile_addr, 16, 1024);
}
__device__ __forceinline__ uint64_t mnmajor_base(uint32_t tile_addr) {
  return sdesc_sw128(tile_addr, 16384, 1024);
}

// Snake order over a persistent grid of G CTAs: round k gives CTA c the work
// unit k*G + c (k even) or k*G + G-1-c (k odd).  With units sorted by cost
// (longest first) this evens out the per-CTA totals.
__device__ __forceinline__ int snake_unit(int k, int cta, int G) {
  return k * G + ((k & 1) ? (G - 1 - cta) : cta);
}

}  // namespace attn
