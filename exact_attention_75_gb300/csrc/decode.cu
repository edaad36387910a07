// Decoding: a few query rows per key/value head (G grouped query heads x Nq
// new tokens, R = G Nq rows, taken 16 at a time) against a key/value cache,
// split over the keys like the tiled forward ("8.3 FlashAttention-3" section 7.3 on
// attention over parts of the keys; the FlashAttention-2 review, "Discussion
// Points", on a decoding kernel that splits the keys and combines the parts).
// Every key and value of the cache is read once, so the kernel is bound by
// those HBM reads; the tiled forward would spend a whole 128-row softmax per
// key block on these few rows.
//
// d in {64, 96, 128, 192, 256}.  One CTA of four warps per (batch,
// key/value head, split, group of 16 of the head's R rows).  The split's keys are cut into blocks of 16 and
// the warps take them in turn (warp w: blocks w, w + 4, ...).  Each warp streams its own blocks through a private
// ring of shared-memory slots: its lane 0 issues the TMA copies (K and V of a
// block, 64-column boxes with the 128-byte swizzle) and refills a slot as soon
// as the warp has multiplied it, so no warp ever waits for another before the
// end.  Per block, on the warp-level tensor-core product (m16n8k16, fp32
// accumulation; the 16 rows of its M hold the unit's R query rows):
//   S = Q K^T        A = Q (fragments in registers up to d = 128, above by
//                    ldmatrix from a copy in shared memory), B = K by ldmatrix;
//   online softmax   per row the block maximum raises the warp's running
//                    maximum m, P = exp2(S scale log2 e - m), the running sum
//                    and O scaled by exp2(m_old - m_new) (FlashAttention-2
//                    review, "Methods");
//   O += P V         A = P (the S accumulators repacked to 16 bits), B = V
//                    by the transposing ldmatrix.
// At the end the four warps' (m, l, O) are combined in shared memory and the
// split's partial O (16-bit) and LSE = (m + log2 l) ln 2 are written where
// attn_merge reads them; a row that sees no key of the split gets O = 0,
// LSE = -inf.
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <cstdint>

#include "decode.cuh"
#include "sm103_ptx.cuh"
#include "smem_attr.cuh"

namespace attn {

namespace {

constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kBoxBytes = kDecodeKeys * 128;  // one 64-column chunk of a block's K or V

template <int D>
struct DecodeLayout {
  static constexpr int kChunks = (D + 63) / 64;               // 64-column chunks of a row
  static constexpr int kSlotBytes = 2 * kChunks * kBoxBytes;  // K chunks, then V chunks
  // Ring depth of each warp: two CTAs per SM up to d = 192, one at d = 256.
  static constexpr int kSlots = D == 64 ? 6 : (D == 192 ? 2 : 3);
  static constexpr int kRingBytes = kWarps * kSlots * kSlotBytes;
  // Above d = 128 the Q fragments are read from shared memory (16 rows in
  // the layout of a staged block) rather than held in registers.
  static constexpr bool kQSmem = D > 128;
  static constexpr int kQBytes = kQSmem ? kChunks * kBoxBytes : 0;
  // After the loop the ring holds each warp's O (16 rows, padded), m and l.
  static constexpr int kRowStride = D + 4;
  static constexpr int kRedBytes = kWarps * 16 * (kRowStride + 2) * 4;
  static_assert(kRingBytes >= kRedBytes && kRingBytes % 1024 == 0, "ring layout");
  static constexpr int kQOff = kRingBytes;
  static constexpr int kBarOff = kQOff + kQBytes;  // one mbarrier per slot
  static constexpr int kFlagOff = kBarOff + kWarps * kSlots * 8;
  static constexpr int kBytes = kFlagOff + 16 + 1024;  // + room to align the base
  static_assert(kBytes <= (D == 256 ? 227 : 113) * 1024, "CTAs per SM");
};

// Byte offset of 16-byte piece `piece` (8 columns) of row `row` in a staged
// block: 64-column chunks of kDecodeKeys rows, each row's eight pieces
// permuted by the 128-byte swizzle (piece ^ row % 8).
__device__ __forceinline__ uint32_t sw_off(int row, int piece) {
  return (uint32_t)((piece >> 3) * kBoxBytes + row * 128 + (((piece & 7) ^ (row & 7)) << 4));
}

// Four 8x8 16-bit matrices from shared memory; lanes 8i..8i+7 give the row
// addresses of matrix i, register i receives it (row lane/4, columns
// 2 (lane%4) and 2 (lane%4) + 1; with .trans the transposed element).
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

// c += a b for one 16 x 8 x 16 tile (A row-major 16 x 16, B 16 x 8 given by
// columns, C 16 x 8 fp32).
template <bool BF16>
__device__ __forceinline__ void mma16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  if constexpr (BF16) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
        "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  } else {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, "
        "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  }
}

// Orders this thread's earlier generic-proxy shared-memory accesses (reads of
// a staged block) before its later async-proxy ones (a TMA copy into the same
// slot).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

template <bool BF16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  return BF16 ? pack_bf16x2(lo, hi) : pack_f16x2(lo, hi);
}

template <int D, bool BF16>
__global__ void __launch_bounds__(kThreads) decode_kernel(const __grid_constant__ CUtensorMap tmK,
                                                          const __grid_constant__ CUtensorMap tmV,
                                                          const DecodeParams p) {
  using L = DecodeLayout<D>;
  constexpr int KS = D / 16;             // k-steps of S = Q K^T
  constexpr int NT = kDecodeKeys / 8;    // 8-key column tiles of S
  constexpr int DN = D / 8;              // 8-column tiles of O
  constexpr int NS = L::kSlots;
  static_assert(KS % 2 == 0 && DN % 2 == 0 && NT == 2, "tile shapes");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kFlagOff);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  auto bar = [&](int s) { return sbase + L::kBarOff + 8u * (uint32_t)(warp * NS + s); };

  // Unit = (key/value head, split, group of 16 rows); the row groups of one
  // (head, split) are neighbours, so their K/V reads meet in L2.
  const int rg = blockIdx.x % p.n_rgroups;
  const int split = (blockIdx.x / p.n_rgroups) % p.n_split;
  const int bk = blockIdx.x / p.n_rgroups / p.n_split;  // batch * Hkv + key/value head
  const int row0 = rg * kDecodeMaxRows;                 // first row of the group in the head's R
  const int rows = min(kDecodeMaxRows, p.R - row0);     // rows of this unit
  const int k_lo = (int)((long long)split * p.n_kblocks / p.n_split) * 128;
  const int k_hi = min((int)((long long)(split + 1) * p.n_kblocks / p.n_split) * 128, p.Nk);
  const int nb = k_hi > k_lo ? (k_hi - k_lo + kDecodeKeys - 1) / kDecodeKeys : 0;
  const int nbw = nb > warp ? (nb - warp + kWarps - 1) / kWarps : 0;  // this warp's blocks

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    for (int i = 0; i < kWarps * NS; ++i) mbar_init(sbase + L::kBarOff + 8u * i, 1);
    mbar_fence_init();
  }
  __syncthreads();
  Watchdog wd{p.status, abort_flag, p.wait_limit_ns};

  // Block j of this warp -> slot j % NS (lane 0 only).
  const uint32_t ring = sbase + (uint32_t)(warp * NS * L::kSlotBytes);
  auto issue = [&](int j) {
    const int s = j % NS;
    const uint32_t dk = ring + (uint32_t)(s * L::kSlotBytes);
    const uint32_t dv = dk + L::kChunks * kBoxBytes;
    const int key0 = k_lo + (warp + j * kWarps) * kDecodeKeys;
    mbar_arrive_expect_tx(bar(s), L::kSlotBytes);
#pragma unroll
    for (int c = 0; c < L::kChunks; ++c) {
      tma_load_3d(dk + c * kBoxBytes, &tmK, bar(s), c * 64, key0, bk);
      tma_load_3d(dv + c * kBoxBytes, &tmV, bar(s), c * 64, key0, bk);
    }
  };
  int issued = min(nbw, NS);
  if (lane == 0)
    for (int j = 0; j < issued; ++j) issue(j);

  // Q fragments of the 16 rows (rows >= R are zero), A layout of m16n8k16:
  // a0 (row r0, cols c..c+1), a1 (row r0 + 8), a2 (row r0, cols c+8..),
  // a3 (row r0 + 8, cols c+8..), c = 16 ks + 2 (lane % 4).  Up to d = 128
  // they stay in registers; above, Q is staged once in shared memory and
  // each k-step's fragment read by ldmatrix (matrix i: rows 8 (i % 2)..,
  // columns 16 ks + 8 (i / 2)..).
  const int r0 = lane >> 2, cq = 2 * (lane & 3);
  const uint16_t* qu = static_cast<const uint16_t*>(p.q) + ((size_t)bk * p.R + row0) * D;
  constexpr int KSR = L::kQSmem ? 1 : KS;  // k-steps held in registers
  uint32_t qa[KSR][4];
  const uint32_t qs = sbase + L::kQOff;
  const int qrow = (lane & 7) + 8 * ((lane >> 3) & 1);
  if constexpr (L::kQSmem) {
    for (int i = threadIdx.x; i < 16 * (D / 8); i += kThreads) {
      const int r = i / (D / 8), pc = i % (D / 8);
      const uint4 x = r < rows ? *reinterpret_cast<const uint4*>(qu + (size_t)r * D + 8 * pc)
                              : make_uint4(0u, 0u, 0u, 0u);
      *reinterpret_cast<uint4*>(smem + L::kQOff + sw_off(r, pc)) = x;
    }
    __syncthreads();
  } else {
    auto qword = [&](int r, int c) -> uint32_t {
      return r < rows ? *reinterpret_cast<const uint32_t*>(qu + (size_t)r * D + c) : 0u;
    };
#pragma unroll
    for (int ks = 0; ks < KSR; ++ks) {
      qa[ks][0] = qword(r0, 16 * ks + cq);
      qa[ks][1] = qword(r0 + 8, 16 * ks + cq);
      qa[ks][2] = qword(r0, 16 * ks + cq + 8);
      qa[ks][3] = qword(r0 + 8, 16 * ks + cq + 8);
    }
  }
  // Last key each of the thread's two rows sees (-1: a padding row, no key).
  auto last_key = [&](int r) {
    if (r >= rows) return -1;
    const int lim = p.causal ? (row0 + r) % p.Nq + p.Nk - p.Nq : p.Nk - 1;
    return min(lim, k_hi - 1);
  };
  const int limA = last_key(r0), limB = last_key(r0 + 8);
  const bool hiB = rows > 8;  // rows 8..15 hold queries

  float o[DN][4];
#pragma unroll
  for (int dn = 0; dn < DN; ++dn) o[dn][0] = o[dn][1] = o[dn][2] = o[dn][3] = 0.f;
  float mA = -INFINITY, mB = -INFINITY, lA = 0.f, lB = 0.f;
  int j = 0;
  bool aborted = false;
#pragma unroll 1
  for (; j < nbw; ++j) {
    const int s = j % NS;
    if (!__all_sync(0xffffffffu, mbar_wait(bar(s), (j / NS) & 1, wd, 61))) {
      aborted = true;
      break;
    }
    const uint32_t tk = ring + (uint32_t)(s * L::kSlotBytes);
    const uint32_t tv = tk + L::kChunks * kBoxBytes;
    const int key0 = k_lo + (warp + j * kWarps) * kDecodeKeys;

    // S = Q K^T, two k-steps at a time: ldmatrix of one 8-key tile over
    // pieces 2ks..2ks+3, the two key tiles' products interleaved.
    float sc[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
#pragma unroll
    for (int ks = 0; ks < KS; ks += 2) {
      uint32_t qx[4], qy[4];
      if constexpr (L::kQSmem) {
        ldsm_x4(qs + sw_off(qrow, 2 * ks + (lane >> 4)), qx);
        ldsm_x4(qs + sw_off(qrow, 2 * ks + 2 + (lane >> 4)), qy);
      } else {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          qx[e] = qa[ks][e];
          qy[e] = qa[ks + 1][e];
        }
      }
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        uint32_t b[4];
        ldsm_x4(tk + sw_off(8 * nt + (lane & 7), 2 * ks + (lane >> 3)), b);
        mma16816<BF16>(sc[nt], qx, b[0], b[1]);
        mma16816<BF16>(sc[nt], qy, b[2], b[3]);
      }
    }

    // Online softmax.  sc[nt][e]: row r0 (e < 2) or r0 + 8, key key0 + 8 nt + cq + e % 2.
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int key = key0 + 8 * nt + cq + (e & 1);
        const float x = sc[nt][e] * p.scale_log2;
        sc[nt][e] = key <= (e < 2 ? limA : limB) ? x : -INFINITY;
      }
    float bA = fmaxf(fmaxf(sc[0][0], sc[0][1]), fmaxf(sc[1][0], sc[1][1]));
    bA = fmaxf(bA, __shfl_xor_sync(0xffffffffu, bA, 1));
    bA = fmaxf(bA, __shfl_xor_sync(0xffffffffu, bA, 2));
    const float nA = fmaxf(mA, bA);
    const float alphaA = nA == mA ? 1.f : ex2_approx(mA - nA);
    const float uA = nA == -INFINITY ? 0.f : nA;
    mA = nA;
    float psA = 0.f;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        sc[nt][e] = ex2_approx(sc[nt][e] - uA);
        psA += sc[nt][e];
      }
    lA = lA * alphaA + psA;
    float alphaB = 1.f;
    if (hiB) {
      float bB = fmaxf(fmaxf(sc[0][2], sc[0][3]), fmaxf(sc[1][2], sc[1][3]));
      bB = fmaxf(bB, __shfl_xor_sync(0xffffffffu, bB, 1));
      bB = fmaxf(bB, __shfl_xor_sync(0xffffffffu, bB, 2));
      const float nB = fmaxf(mB, bB);
      alphaB = nB == mB ? 1.f : ex2_approx(mB - nB);
      const float uB = nB == -INFINITY ? 0.f : nB;
      mB = nB;
      float psB = 0.f;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 2; e < 4; ++e) {
          sc[nt][e] = ex2_approx(sc[nt][e] - uB);
          psB += sc[nt][e];
        }
      lB = lB * alphaB + psB;
    }
    if (__any_sync(0xffffffffu, alphaA != 1.f || alphaB != 1.f)) {
#pragma unroll
      for (int dn = 0; dn < DN; ++dn) {
        o[dn][0] *= alphaA;
        o[dn][1] *= alphaA;
        o[dn][2] *= alphaB;
        o[dn][3] *= alphaB;
      }
    }

    // O += P V: P in the A layout (keys 0..7 from tile 0, 8..15 from tile 1),
    // V by the transposing ldmatrix (matrix i: keys 8 (i % 2).., columns of
    // 8-column tile dn + i / 2).
    uint32_t pa[4];
    pa[0] = pack2<BF16>(sc[0][0], sc[0][1]);
    pa[1] = hiB ? pack2<BF16>(sc[0][2], sc[0][3]) : 0u;
    pa[2] = pack2<BF16>(sc[1][0], sc[1][1]);
    pa[3] = hiB ? pack2<BF16>(sc[1][2], sc[1][3]) : 0u;
    const int vrow = 8 * ((lane >> 3) & 1) + (lane & 7);
#pragma unroll
    for (int dn = 0; dn < DN; dn += 2) {
      uint32_t b[4];
      ldsm_x4_trans(tv + sw_off(vrow, dn + (lane >> 4)), b);
      mma16816<BF16>(o[dn], pa, b[0], b[1]);
      mma16816<BF16>(o[dn + 1], pa, b[2], b[3]);
    }

    // The slot is read: refill it with this warp's block j + NS.
    __syncwarp();
    if (issued < nbw) {
      if (lane == 0) {
        fence_proxy_async_smem();
        issue(issued);
      }
      ++issued;
    }
  }
  if (aborted) {
    // Every copy this warp issued must land before the CTA may exit or reuse
    // the ring.
    Watchdog dw = wd;
    volatile int never = 0;
    dw.abort_flag = &never;
    dw.limit_ns = drain_limit_ns(wd.limit_ns);
    for (int jj = j; jj < issued; ++jj) mbar_wait(bar(jj % NS), (jj / NS) & 1, dw, 62);
  }

  // The key stream is done: a dependent launch (the merge) may start its
  // launch now; it waits for this grid's completion before reading.
  asm volatile("griddepcontrol.launch_dependents;");

  // Row sums over the four lanes of a row.
  lA += __shfl_xor_sync(0xffffffffu, lA, 1);
  lA += __shfl_xor_sync(0xffffffffu, lA, 2);
  lB += __shfl_xor_sync(0xffffffffu, lB, 1);
  lB += __shfl_xor_sync(0xffffffffu, lB, 2);

  // Combine the warps: each writes its (O, m, l) over the (now idle) ring.
  __syncthreads();
  float* red = reinterpret_cast<float*>(smem);
  float* rm = red + kWarps * 16 * L::kRowStride;  // [kWarps][16]
  float* rl = rm + kWarps * 16;                   // [kWarps][16]
  {
    float* ro = red + warp * 16 * L::kRowStride;
#pragma unroll
    for (int dn = 0; dn < DN; ++dn) {
      *reinterpret_cast<float2*>(ro + r0 * L::kRowStride + 8 * dn + cq) =
          make_float2(o[dn][0], o[dn][1]);
      *reinterpret_cast<float2*>(ro + (r0 + 8) * L::kRowStride + 8 * dn + cq) =
          make_float2(o[dn][2], o[dn][3]);
    }
    if ((lane & 3) == 0) {
      rm[warp * 16 + r0] = mA;
      rm[warp * 16 + r0 + 8] = mB;
      rl[warp * 16 + r0] = lA;
      rl[warp * 16 + r0 + 8] = lB;
    }
  }
  __syncthreads();
  if (*abort_flag != 0) return;

  uint16_t* ou = static_cast<uint16_t*>(p.o) + (size_t)split * p.o_split +
                 ((size_t)bk * p.R + row0) * D;
  float* lu = p.lse + (size_t)split * p.lse_split + (size_t)bk * p.R + row0;
  constexpr int P8 = D / 8;
  for (int idx = threadIdx.x; idx < rows * P8; idx += kThreads) {
    const int r = idx / P8, c = (idx % P8) * 8;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, rm[w * 16 + r]);
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    float lsum = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const float mw = rm[w * 16 + r];
      const float f = mw == -INFINITY ? 0.f : exp2f(mw - M);
      lsum += f * rl[w * 16 + r];
      const float4* src = reinterpret_cast<const float4*>(red + (w * 16 + r) * L::kRowStride + c);
      const float4 x0 = src[0], x1 = src[1];
      acc[0] += f * x0.x;
      acc[1] += f * x0.y;
      acc[2] += f * x0.z;
      acc[3] += f * x0.w;
      acc[4] += f * x1.x;
      acc[5] += f * x1.y;
      acc[6] += f * x1.z;
      acc[7] += f * x1.w;
    }
    const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
    *reinterpret_cast<uint4*>(ou + (size_t)r * D + c) =
        make_uint4(pack2<BF16>(acc[0] * inv, acc[1] * inv), pack2<BF16>(acc[2] * inv, acc[3] * inv),
                   pack2<BF16>(acc[4] * inv, acc[5] * inv), pack2<BF16>(acc[6] * inv, acc[7] * inv));
    if (c == 0) lu[r] = lsum > 0.f ? (M + log2f(lsum)) * 0.69314718055994531f : -INFINITY;
  }
}

template <int D, bool BF16>
cudaError_t launch_db(const DecodeLaunch& a) {
  using L = DecodeLayout<D>;
  static DeviceFlags configured;
  cudaError_t e = ensure_dyn_smem(decode_kernel<D, BF16>, L::kBytes, configured);
  if (e != cudaSuccess) return e;
  decode_kernel<D, BF16><<<a.num_units, kThreads, L::kBytes, a.stream>>>(a.tmK, a.tmV, a.params);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_d(const DecodeLaunch& a, bool bf16) {
  return bf16 ? launch_db<D, true>(a) : launch_db<D, false>(a);
}

}  // namespace

cudaError_t launch_decode(const DecodeLaunch& a, int d, bool bf16) {
  switch (d) {
    case 64: return launch_d<64>(a, bf16);
    case 96: return launch_d<96>(a, bf16);
    case 192: return launch_d<192>(a, bf16);
    case 256: return launch_d<256>(a, bf16);
    default: return launch_d<128>(a, bf16);
  }
}

}  // namespace attn
