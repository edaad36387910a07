// Forward pass for the wide head dims d in {192, 256} on sm_103a.
//
// The same algorithm as fwd.cu ("FlashAttention-2: Faster Attention with
// Better Parallelism and Work Partitioning" (review page), flowchart
// "프레임워크 개요" and "Methods": per query tile, loop over K/V tiles,
// online softmax with the 1/rowsum rescale deferred to the end, O and the
// log-sum-exp written once; causal blocks above the diagonal skipped, per
// "핵심 구성요소"), with a different overlap because the wide tiles do not
// fit twice:
//
//  * Tensor memory holds 512 columns.  Two query tiles per CTA would need two
//    S tiles (2 x 128) and two O accumulators (2 x d) -- more than 512 at
//    d >= 192.  This kernel keeps ONE query tile of 128 rows per work unit,
//    one O accumulator (d columns) and TWO S buffers (2 x 128 columns), so
//    the tensor core computes S(j+1) (and P V(j-1)) while the softmax
//    warpgroup exponentiates S(j): the overlap of "8.3 FlashAttention-3",
//    section 4 (intra-warpgroup overlap of softmax with the next GEMM),
//    recast for an MMA warp.  Issue order per unit:
//        S0 S1 | PV0 S2 | PV1 S3 | ... | PV(n-1)
//    where each "|" waits for P(j) from the softmax warpgroup.
//  * Shared memory holds the Q tile (48 or 64 KB) and a ring of 16 KB chunks
//    (128 rows x 64 columns, one TMA box each) through which K and V tiles
//    stream in the order they are consumed: K0 K1 V0 K2 V1 K3 ... V(n-1).  A
//    whole tile does not need a free 48-64 KB slot before its first chunk can
//    start loading.  The S products accumulate over the chunks of K (K-steps
//    of 16 along d); P V is issued per V chunk into the matching 64 columns
//    of O (N = 64), so a tile's chunks need not be contiguous in the ring.
//
// CTA organisation (224 threads, one CTA per SM, persistent):
//   warps 0-3  softmax warpgroup: thread = row of the query tile = TMEM lane
//   warp  4    TMA producer (Q, then the K/V chunk ring)
//   warp  5    tcgen05 issuer (one thread) + tensor-memory owner
//   warp  6    TMA relay: waits for the copies the next MMA group reads and
//              meets the issuer at a named barrier (the issuer itself never
//              waits on an mbarrier between its commits)
//
// Tensor memory: S buffers [0,128) [128,256) (fp32; P overwrites the first
// 64 columns as 16-bit pairs), O [256, 256+d).
//
// The O correction ("Methods": rescale when the running max rises) is lazy,
// as in fwd.cu: the reference max is raised only when a block's max exceeds
// it by more than 2^8 (log2 units).  When it is raised at block j, P V(j-1)
// may still be running (S(j) was issued before it), so the softmax first
// waits for its completion (an mbarrier committed after every P V).
#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

#include "fwd.cuh"
#include "sm103_ptx.cuh"
#include "smem_attr.cuh"
#include "tiles.cuh"

namespace attn {

namespace {

constexpr int kThreads = 224;
constexpr int kWarpProducer = 4;
constexpr int kWarpMma = 5;
constexpr int kWarpRelay = 6;
constexpr uint32_t kBarKv = 1, kBarP = 2;  // named barriers: issuer+relay, issuer+softmax
constexpr float kRescaleThreshold = 8.0f;  // log2 units: P stays <= 2^8
constexpr int kChunkBytes = 128 * 64 * 2;  // one TMA box: 128 rows x 64 16-bit values

template <int D>
struct WideLayout {
  static constexpr int kChunks = D / 64;                 // chunks per K or V tile
  static constexpr int kQBytes = 128 * D * 2;
  static constexpr int kRing = (D == 256) ? 10 : 11;     // K/V ring depth (chunks)
  static constexpr int kQOff = 0;
  static constexpr int kRingOff = kQBytes;
  static constexpr int kBarOff = kRingOff + kRing * kChunkBytes;
  enum { kQFull, kQEmpty, kSFull, kPvDone = kSFull + 2, kOFull, kDrain, kKvFull,
         kKvEmpty = kKvFull + kRing, kNumBars = kKvEmpty + kRing };
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;
  static constexpr int kBytes = kMiscOff + 16;
  static constexpr int kDynSmem = kBytes + 1024;  // + alignment slack
  static_assert(D == 192 || D == 256, "wide kernel: d in {192, 256}");
  static_assert(kDynSmem <= 232448, "shared memory budget (227 KB) exceeded");
};

struct WideUnit {
  int bh, tile;  // query head (batch * heads + head), query tile
  int zkv;       // key/value head (batch * heads_kv + head / group)
  int nb;        // key blocks visited
};

template <bool CAUSAL>
__device__ __forceinline__ WideUnit decode_wide_unit(int u, const FwdParams& p) {
  WideUnit w;
  if (CAUSAL) {
    // Longest first: the last query tiles of every head come first.
    const int r = u / p.BH;
    w.bh = u - r * p.BH;
    w.tile = p.n_qtiles - 1 - r;
  } else {
    w.bh = u / p.n_qtiles;
    w.tile = u - w.bh * p.n_qtiles;
  }
  const int b = w.bh / p.heads;
  w.zkv = b * p.heads_kv + (w.bh - b * p.heads) / p.group;
  w.nb = CAUSAL ? min(w.tile + 1, p.n_kblocks) : p.n_kblocks;
  return w;
}

// The order in which K and V tiles of a unit with nb key blocks are consumed
// (and therefore loaded into the ring): K0 K1 V0 K2 V1 K3 ... V(nb-1).
// visit(is_v, block) is called once per tile in that order.
template <typename F>
__device__ __forceinline__ void for_each_tile(int nb, F&& visit) {
  visit(false, 0);
  if (nb > 1) visit(false, 1);
  for (int j = 0; j < nb; ++j) {
    visit(true, j);
    if (j + 2 < nb) visit(false, j + 2);
  }
}

template <int D, bool CAUSAL, bool BF16>
__global__ void __launch_bounds__(kThreads, 1)
    fwd_wide_kernel(const __grid_constant__ CUtensorMap tmQ,
                    const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const FwdParams p) {
  using L = WideLayout<D>;
  constexpr int CH = L::kChunks;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + L::kBarOff;
  auto bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };
  auto chunk_addr = [&](uint32_t it) { return sbase + L::kRingOff + (it % L::kRing) * kChunkBytes; };
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + L::kMiscOff);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kMiscOff + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  Watchdog wd{p.status, abort_flag, p.wait_limit_ns};

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    mbar_init(bar(L::kQFull), 1);
    mbar_init(bar(L::kQEmpty), 1);
    mbar_init(bar(L::kSFull + 0), 1);
    mbar_init(bar(L::kSFull + 1), 1);
    mbar_init(bar(L::kPvDone), 1);
    mbar_init(bar(L::kOFull), 1);
    mbar_init(bar(L::kDrain), 1);
    for (int s = 0; s < L::kRing; ++s) {
      mbar_init(bar(L::kKvFull + s), 1);
      mbar_init(bar(L::kKvEmpty + s), 1);
    }
    mbar_fence_init();
  }
  if (warp == kWarpMma) {
    tmem_alloc(smem_u32(tmem_holder), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_holder;
  const int G = gridDim.x;
  const int cta = blockIdx.x;

  if (warp == kWarpProducer) {
    // ------------------------------------------------------ TMA producer ---
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      uint32_t it = 0, q_it = 0;
      bool ok = true;
      for (int k = 0; ok; ++k) {
        const int u = snake_unit(k, cta, G);
        if (u >= p.num_units) break;
        const WideUnit w = decode_wide_unit<CAUSAL>(u, p);
        ok = mbar_wait(bar(L::kQEmpty), (q_it & 1) ^ 1, wd, 1);
        if (!ok) break;
        mbar_arrive_expect_tx(bar(L::kQFull), L::kQBytes);
#pragma unroll
        for (int c = 0; c < CH; ++c)
          tma_load_3d(sbase + L::kQOff + c * kChunkBytes, &tmQ, bar(L::kQFull), 64 * c,
                      w.tile * 128, w.bh);
        ++q_it;
        for_each_tile(w.nb, [&](bool is_v, int j) {
#pragma unroll
          for (int c = 0; c < CH; ++c) {
            if (!ok) return;
            const uint32_t slot = it % L::kRing;
            ok = mbar_wait(bar(L::kKvEmpty + slot), ((it / L::kRing) & 1) ^ 1, wd, 2);
            if (!ok) return;
            mbar_arrive_expect_tx(bar(L::kKvFull + slot), kChunkBytes);
            tma_load_3d(chunk_addr(it), is_v ? &tmV : &tmK, bar(L::kKvFull + slot), 64 * c,
                        j * 128, w.zkv);
            ++it;
          }
        });
      }
      // Drain: every copy this thread issued must have landed before the CTA
      // may exit (only matters after an abort; otherwise all were consumed).
      Watchdog dw = wd;
      volatile int never = 0;
      dw.abort_flag = &never;
      dw.limit_ns = drain_limit_ns(wd.limit_ns);
      const uint32_t first = it > (uint32_t)L::kRing ? it - L::kRing : 0u;
      for (uint32_t i = first; i < it; ++i)
        mbar_wait(bar(L::kKvFull + i % L::kRing), (i / L::kRing) & 1, dw, 3);
      if (q_it > 0) mbar_wait(bar(L::kQFull), (q_it - 1) & 1, dw, 4);
    }
    __syncwarp();
  } else if (warp == kWarpRelay) {
    // ---------------------------------------------------------- TMA relay ---
    // Rendezvous schedule per unit: [Q + K0], [K1] (nb > 1), then per block
    // j: [V_j + K_{j+2}].  After an abort the schedule is still walked to the
    // end (waits skipped) so every rendezvous pairs up as in a clean run.
    uint32_t it = 0, q_it = 0;
    bool aborted = false;
    auto tile_ready = [&]() {
      for (int c = 0; c < CH; ++c) {
        const uint32_t slot = it % L::kRing;
        const uint32_t par = (it / L::kRing) & 1;
        ++it;
        if (!aborted)
          aborted = !__all_sync(0xffffffffu, mbar_wait(bar(L::kKvFull + slot), par, wd, 7));
      }
    };
    for (int k = 0;; ++k) {
      const int u = snake_unit(k, cta, G);
      if (u >= p.num_units) break;
      const WideUnit w = decode_wide_unit<CAUSAL>(u, p);
      const uint32_t qpar = q_it & 1;
      ++q_it;
      if (!aborted) aborted = !__all_sync(0xffffffffu, mbar_wait(bar(L::kQFull), qpar, wd, 5));
      tile_ready();  // K0
      aborted = named_bar_or(kBarKv, 64, aborted);
      if (w.nb > 1) {
        tile_ready();  // K1
        aborted = named_bar_or(kBarKv, 64, aborted);
      }
      for (int j = 0; j < w.nb; ++j) {
        tile_ready();                  // V_j
        if (j + 2 < w.nb) tile_ready();  // K_{j+2}
        aborted = named_bar_or(kBarKv, 64, aborted);
      }
    }
  } else if (warp == kWarpMma) {
    // ---------------------------------------------------- tcgen05 issuer ---
    constexpr uint32_t kIdS = idesc_f16(128, 128, BF16, false, false);
    constexpr uint32_t kIdO = idesc_f16(128, 64, BF16, false, true);  // per 64-column chunk
    uint32_t it = 0, s_it = 0;
    bool aborted = false;
    bool issued = false;
    const uint64_t qdesc = kmajor_base(sbase + L::kQOff);
    // S into buffer sb = Q K^T; K's chunks start at ring position it0.  Each
    // chunk's slot is released as soon as its own MMAs complete (a commit
    // right after them), so the producer can refill it while the rest of
    // the product runs.
    auto issue_s = [&](uint32_t sb, uint32_t it0) {
      const uint32_t dcol = tbase + 128 * sb;
#pragma unroll
      for (int c = 0; c < CH; ++c) {
        const uint64_t kd = kmajor_base(chunk_addr(it0 + c));
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_f16_ss(dcol, desc_plus(qdesc, kmajor16_off(4 * c + kk)),
                     desc_plus(kd, kmajor16_off(kk)), kIdS, (c | kk) ? 1u : 0u);
        mma_commit(bar(L::kKvEmpty + (it0 + c) % L::kRing));
      }
    };
    // O[:, 64c, 64c+64) += P V_c for each chunk c of V (at ring position
    // it0), each chunk's slot released after its MMAs.
    auto issue_pv = [&](uint32_t sb, uint32_t it0, uint32_t acc0) {
      const uint32_t pcol = tbase + 128 * sb;
#pragma unroll
      for (int c = 0; c < CH; ++c) {
        const uint64_t vd = mnmajor_base(chunk_addr(it0 + c));
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)  // 16 keys per MMA
          mma_f16_ts(tbase + 256 + 64 * c, pcol + kk * 8, desc_plus(vd, mnmajor16_off(kk)), kIdO,
                     kk > 0 ? 1u : acc0);
        mma_commit(bar(L::kKvEmpty + (it0 + c) % L::kRing));
      }
    };
    for (int k = 0;; ++k) {
      const int u = snake_unit(k, cta, G);
      if (u >= p.num_units) break;
      const WideUnit w = decode_wide_unit<CAUSAL>(u, p);
      const int nb = w.nb;
      const uint32_t s0 = s_it;  // S buffer of block j: (s0 + j) & 1
      // S(0) once Q and K0 have landed (ring positions advance in the
      // producer's load order)
      aborted = named_bar_or(kBarKv, 64, aborted);
      const uint32_t k0pos = it;
      it += CH;
      if (!aborted) {
        tc_fence_after();
        if (lane == 0) {
          issue_s(s0 & 1, k0pos);
          mma_commit(bar(L::kSFull + (s0 & 1)));
          if (nb == 1) mma_commit(bar(L::kQEmpty));
        }
        issued = true;
        __syncwarp();
      }
      if (nb > 1) {
        aborted = named_bar_or(kBarKv, 64, aborted);
        const uint32_t k1pos = it;
        it += CH;
        if (!aborted) {
          tc_fence_after();
          if (lane == 0) {
            issue_s((s0 + 1) & 1, k1pos);
            mma_commit(bar(L::kSFull + ((s0 + 1) & 1)));
            if (nb == 2) mma_commit(bar(L::kQEmpty));
          }
          __syncwarp();
        }
      }
      for (int j = 0; j < nb; ++j) {
        // V_j (and K_{j+2}, if any) have landed
        aborted = named_bar_or(kBarKv, 64, aborted);
        const uint32_t vpos = it;
        it += CH;
        const bool next = j + 2 < nb;
        uint32_t k2pos = 0;
        if (next) {
          k2pos = it;
          it += CH;
        }
        // P(j) is in tensor memory
        aborted = named_bar_or(kBarP, 160, aborted);
        if (!aborted) {
          tc_fence_after();
          if (lane == 0) {
            const uint32_t sb = (s0 + j) & 1;
            issue_pv(sb, vpos, j > 0 ? 1u : 0u);
            mma_commit(bar(L::kPvDone));
            if (j == nb - 1) mma_commit(bar(L::kOFull));
            if (next) {
              // S(j+2) reuses the buffer of block j (its P was read by the
              // P V just issued; MMAs of this thread execute in order).
              issue_s(sb, k2pos);
              mma_commit(bar(L::kSFull + sb));
              if (j + 2 == nb - 1) mma_commit(bar(L::kQEmpty));
            }
          }
          __syncwarp();
        }
      }
      s_it += nb;
    }
    // Drain: wait until every MMA issued above has completed.
    if (lane == 0 && issued) {
      mma_commit(bar(L::kDrain));
      Watchdog dw = wd;
      volatile int never = 0;
      dw.abort_flag = &never;
      dw.limit_ns = drain_limit_ns(wd.limit_ns);
      mbar_wait(bar(L::kDrain), 0, dw, 10);
    }
    __syncwarp();
  } else {
    // --------------------------------------------------- softmax warpgroup ---
    const int r = threadIdx.x & 127;  // row within the tile = TMEM lane
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    const uint32_t o_addr = tbase + lane_base + 256u;
    const float sl2 = p.scale_log2;
    uint32_t s_it = 0, o_it = 0, pv_it = 0;
    bool aborted = false;
    for (int k = 0;; ++k) {
      const int u = snake_unit(k, cta, G);
      if (u >= p.num_units) break;
      const WideUnit w = decode_wide_unit<CAUSAL>(u, p);
      const int row = w.tile * 128 + r;
      float m = -INFINITY;  // reference max of the log2-scaled scores
      float l = 0.f;        // running sum of exp2(x - m)
      for (int j = 0; j < w.nb; ++j) {
        const uint32_t sidx = s_it + j;
        const uint32_t sb = sidx & 1;
        const uint32_t s_addr = tbase + lane_base + 128u * sb;
        if (!aborted)
          aborted =
              !__all_sync(0xffffffffu, mbar_wait(bar(L::kSFull + sb), (sidx >> 1) & 1, wd, 11));
        if (!aborted) {
          tc_fence_after();
          uint32_t sr[4][32];
#pragma unroll
          for (int c = 0; c < 4; ++c) tmem_ld32(s_addr + c * 32, sr[c]);
          tmem_wait_ld();
#pragma unroll
          for (int c = 0; c < 4; ++c) reg_fence32(sr[c]);
          float s[128];
#pragma unroll
          for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int i = 0; i < 32; ++i) s[c * 32 + i] = __uint_as_float(sr[c][i]);
          // blocks reaching past the tile's first row's last visible key
          const bool diag = CAUSAL && (j == w.tile);
          const bool tail = (j == p.n_kblocks - 1) && (p.N & 127);
          if (diag || tail) {
            const int lim = CAUSAL ? min(row, p.N - 1) : (p.N - 1);
#pragma unroll
            for (int c = 0; c < 128; ++c) s[c] = (j * 128 + c > lim) ? -INFINITY : s[c];
          }
          const float m_blk = row_max128(s) * sl2;
          // Raise the reference max where the block's exceeds it by more
          // than the threshold; O and l of those rows are rescaled by alpha
          // after the exponentials (the scores are dead by then).
          bool rescale = false;
          float alpha = 1.f;
          if (j == 0) {
            m = m_blk;
          } else {
            const bool need = m_blk > m + kRescaleThreshold;
            rescale = __any_sync(0xffffffffu, need);
            if (need) {
              alpha = ex2_approx(m - m_blk);
              m = m_blk;
            }
          }
          if (!aborted) {
            const float mref = (m == -INFINITY) ? 0.f : m;
            const float2 nm2 = make_float2(-mref, -mref);
            const float2 sc2 = make_float2(sl2, sl2);
            float2 rs2[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                             make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              uint32_t pk[16];
#pragma unroll
              for (int i = 0; i < 16; ++i) {
                const float2 x = __ffma2_rn(make_float2(s[c * 32 + 2 * i], s[c * 32 + 2 * i + 1]),
                                            sc2, nm2);
                const float p0 = ex2_approx(x.x);
                const float p1 = ex2_approx(x.y);
                rs2[i & 3] = __fadd2_rn(rs2[i & 3], make_float2(p0, p1));
                pk[i] = BF16 ? pack_bf16x2(p0, p1) : pack_f16x2(p0, p1);
              }
              tmem_st16(s_addr + c * 16, pk);
            }
            const float2 rsum =
                __fadd2_rn(__fadd2_rn(rs2[0], rs2[1]), __fadd2_rn(rs2[2], rs2[3]));
            l = l * alpha + (rsum.x + rsum.y);
            if (rescale) {
              // P V(j-1) may still be accumulating into O (S(j) was issued
              // before it): wait for its completion, then O_row *= alpha.
              const uint32_t g = pv_it + j - 1;
              aborted = __any_sync(0xffffffffu, !mbar_wait(bar(L::kPvDone), g & 1, wd, 13));
              if (!aborted) {
                tc_fence_after();
#pragma unroll 1
                for (int c = 0; c < D / 64; ++c) {
                  uint32_t ra[32], rb[32];
                  tmem_ld32(o_addr + c * 64, ra);
                  tmem_ld32(o_addr + c * 64 + 32, rb);
                  tmem_wait_ld();
                  reg_fence32(ra);
                  reg_fence32(rb);
#pragma unroll
                  for (int i = 0; i < 32; ++i) {
                    ra[i] = __float_as_uint(__uint_as_float(ra[i]) * alpha);
                    rb[i] = __float_as_uint(__uint_as_float(rb[i]) * alpha);
                  }
                  tmem_st32(o_addr + c * 64, ra);
                  tmem_st32(o_addr + c * 64 + 32, rb);
                }
              }
            }
            tmem_wait_st();
            tc_fence_before();
          }
        }
        // Hand P(j) to the issuer (and learn whether anyone has aborted).
        aborted = named_bar_or(kBarP, 160, aborted);
      }
      s_it += w.nb;
      pv_it += w.nb;
      // ------------------------------------------------------- epilogue ---
      const uint32_t opar = o_it & 1;
      ++o_it;
      if (!aborted)
        aborted = !__all_sync(0xffffffffu, mbar_wait(bar(L::kOFull), opar, wd, 12));
      if (aborted) continue;
      tc_fence_after();
      const float inv_l = l > 0.f ? 1.0f / l : 0.f;
      const size_t grow = (size_t)w.bh * p.N + row;
      uint4* orow = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.o) + grow * D);
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t raw[32];
        tmem_ld32_sync(o_addr + c * 32, raw);
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float a = __uint_as_float(raw[2 * i]) * inv_l;
          const float b = __uint_as_float(raw[2 * i + 1]) * inv_l;
          pk[i] = BF16 ? pack_bf16x2(a, b) : pack_f16x2(a, b);
        }
        if (row < p.N) {
#pragma unroll
          for (int v = 0; v < 4; ++v)
            orow[c * 4 + v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
        }
      }
      if (row < p.N) p.lse[grow] = (m + log2f(l)) * 0.69314718055994530942f;
      tc_fence_before();
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
}

template <int D, bool CAUSAL, bool BF16>
cudaError_t launch_wide(const FwdLaunch& a) {
  using L = WideLayout<D>;
  auto kern = fwd_wide_kernel<D, CAUSAL, BF16>;
  static DeviceFlags configured;  // attribute set once per device and instantiation
  cudaError_t e = ensure_dyn_smem(kern, L::kDynSmem, configured);
  if (e != cudaSuccess) return e;
  const int grid = a.params.num_units < a.num_ctas ? a.params.num_units : a.num_ctas;
  kern<<<grid, kThreads, L::kDynSmem, a.stream>>>(a.tmQ, a.tmK, a.tmV, a.params);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_wide_d(const FwdLaunch& a, bool causal, bool bf16) {
  if (causal) return bf16 ? launch_wide<D, true, true>(a) : launch_wide<D, true, false>(a);
  return bf16 ? launch_wide<D, false, true>(a) : launch_wide<D, false, false>(a);
}

}  // namespace

// Forward for d in {192, 256}: dense [B*H, N, d] heads (grouped query heads
// allowed), one query tile per work unit; params.num_units must be
// B*H*ceil(N/128).
cudaError_t launch_fwd_wide(const FwdLaunch& a, int d, bool causal, bool bf16) {
  return d == 256 ? launch_wide_d<256>(a, causal, bf16) : launch_wide_d<192>(a, causal, bf16);
}

}  // namespace attn
