// Backward pass of exact attention on sm_103a (head dim 128).
//
// "FlashAttention-2: Faster Attention with Better Parallelism and Work
// Partitioning" (review page), "Methods" and "핵심 구성요소": the forward pass
// keeps only the log-sum-exp, and the backward pass recomputes P from it
// instead of storing the N x N matrix.  The backward of "Triton 07: Flash
// Attention v3" is staged; here the stages are
//   1. bwd_pre_kernel  D_i = sum_c dO_ic O_ic (warp-shuffle row reduction);
//   2. bwd_dkv_kernel  one CTA per 128-key K/V tile (persistent, longest
//                      first within a block of heads): for every 128-query
//                      tile i it recomputes
//                      S^T = K Q_i^T and P^T = exp2(S^T c - LSE_i log2 e),
//                      dP^T = V dO_i^T, dS^T = P^T o (dP^T - D_i), and
//                      accumulates dV += P^T dO_i, dK += dS^T Q_i in tensor
//                      memory;
//   3. bwd_dq_kernel   one CTA per 128-query tile: for every key tile j it
//                      recomputes S = Q K_j^T, P, dP = dO V_j^T and dS and
//                      accumulates dQ += dS K_j in tensor memory.
// Splitting dQ from dK/dV recomputes S and dP once more (7 instead of 5
// matrix products) but removes the cross-CTA reduction of dQ: with it, each
// step also had to stage 64 KB of fp32 partial dQ through shared memory for
// a TMA reduce-add, and shared-memory bandwidth (128 B/clock/SM, all of it
// taken by an N = 128 MMA with both operands in shared memory) is what
// bounds these kernels.  Every MMA here has N = 128 and keeps its
// accumulator in tensor memory; P and dS feed the dV / dK / dQ products
// from tensor memory, and in bwd_dq Q_i and dO_i are copied into tensor
// memory once per query tile so that S and dP read only K_j / V_j from
// shared memory.
//
// CTA organisation of both kernels (352 threads):
//   warps 0-3 / 4-7  compute warpgroups, one per half of the 128 columns of
//                    S (query columns in bwd_dkv, key columns in bwd_dq);
//                    thread = TMEM lane = row
//   warp 8           TMA producer
//   warp 9           tcgen05 issuer + tensor-memory owner
//   warp 10          relay: waits on the pipeline's mbarriers and
//                    meets the issuer at a named barrier, so that the issuer
//                    never touches shared memory between its commits
// Units (a K/V tile, or a query tile) are handed out at run time: the
// producer takes the next one from a counter in the workspace with an atomic
// add and publishes it through a small ring in shared memory (kUnitSlots
// entries), which the issuer, the relay and the compute warps read; an entry
// of -1 ends the CTA's work.  A CTA that finishes early takes more units, and
// with the causal order blocked by heads the units in flight at any time
// stream the tiles of a few heads only, which then stay in L2.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <cstdint>

#include "bwd.cuh"
#include "sm103_ptx.cuh"
#include "smem_attr.cuh"
#include "tiles.cuh"
#include "unit_ring.cuh"

namespace attn {

namespace {

constexpr int kThreads = 352;
constexpr int kWarpProducer = 8;
constexpr int kWarpMma = 9;
constexpr int kWarpRelay = 10;
constexpr uint32_t kBarRelay = 3;  // named barrier: relay warp + issuer warp (64 threads)
constexpr float kLog2e = 1.4426950408889634f;
constexpr uint32_t kStatusLayout = 5;  // shared memory not 1024-byte aligned
// Bytes of a 128-row tile of 16-bit values with D columns (padded to a
// multiple of 64).
template <int D>
constexpr int kTileBytes = 128 * kPaddedD<D> * 2;

// Column of the K-step kk (16 values of the contraction index) of a 16-bit
// operand that the two warpgroups wrote into the first 32 columns of their
// 64-column halves of a 128-column tensor-memory region.
__device__ __forceinline__ uint32_t half_packed_col(int kk) {
  return kk < 4 ? 8u * kk : 64u + 8u * (kk - 4);
}

__device__ __forceinline__ uint32_t pack16x2(bool bf16, float lo, float hi) {
  return bf16 ? pack_bf16x2(lo, hi) : pack_f16x2(lo, hi);
}

// Loads a 128 x D 16-bit tile (boxes of 64 columns; columns past D are
// zero-filled) with TMA.
template <int D>
__device__ __forceinline__ void load_tile(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                          int row0, int bh) {
#pragma unroll
  for (int h = 0; h < kPaddedD<D> / 64; ++h)
    tma_load_3d(dst + h * 16384, map, bar, 64 * h, row0, bh);
}

// ============================================================ dK, dV kernel ===

// Per step s the tensor core runs S^T(s) | dK(s-1) | dP^T(s) | dV(s), so the
// warpgroups' P^T(s) overlaps dK(s-1) and dP^T(s), and their dS^T(s)
// overlaps dV(s) and S^T(s+1).  Q_i is then read until the next step (by
// dK), so Q has a ring of 3 slots.  dO_i is last read by dV(s) and has a
// ring of 2 slots, each freed as soon as dV(s) completes; the -LSE / -D
// vectors of its queries are last read by the warpgroups' dS^T(s) phase and
// have a ring of their own (2 slots), so the next dO load need not wait for
// that phase and for dK(s).
template <int D>
struct DkvLayout {
  static constexpr int kTile = kTileBytes<D>;
  static constexpr int kK = 0;
  static constexpr int kV = kTile;
  static constexpr int kQSlots = 3, kDoSlots = 2;
  static constexpr int kQ0 = 2 * kTile;
  static constexpr int kDo0 = kQ0 + kQSlots * kTile;
  static constexpr int kVec = kDo0 + kDoSlots * kTile;  // per vector slot: -LSE2[128], -D[128]
  static constexpr int kBar = kVec + kDoSlots * 1024;
  enum {
    kKvFull, kKvEmpty, kQFull, kQEmpty = kQFull + kQSlots, kDoFull = kQEmpty + kQSlots,
    kDoEmpty = kDoFull + kDoSlots, kVecEmpty = kDoEmpty + kDoSlots,
    kSFull = kVecEmpty + kDoSlots, kDpFull = kSFull + 2, kPReady, kDsReady = kPReady + 2,
    kDkvFull, kDkvFree, kDrain, kUnitFull, kUnitEmpty = kUnitFull + kUnitSlots,
    kNumBars = kUnitEmpty + kUnitSlots
  };
  static constexpr int kMisc = kBar + kNumBars * 8;  // TMEM address, abort flag, unit ring
  static constexpr int kBytes = kMisc + 16 + 4 * kUnitSlots;
  static_assert(kBytes <= 232448, "shared memory budget (227 KB) exceeded");
};

// Tensor memory: dV [0,128)  dK [128,256)  S^T [256,384)  dP^T [384,512).
// P^T (16-bit) of warpgroup h overwrites S^T columns [256+64h, 256+64h+32),
// dS^T those of dP^T.  At d = 64 dV and dK take 64 columns each, which leaves
// room for a second S^T buffer: dV [0,64)  dK [64,128)  S^T [128,256) and
// [256,384) by step parity  dP^T [384,512); S^T(s+1) can then be issued
// before dV(s) has read P^T(s).
constexpr uint32_t kColDV = 0, kColDP = 384;
template <int D>
constexpr bool kDoubleS = kPaddedD<D> == 64;
template <int D>
constexpr uint32_t kColDK = kDoubleS<D> ? 64 : 128;
template <int D>
constexpr uint32_t kColST0 = kDoubleS<D> ? 128 : 256;

// Rows of sequence b: [row0, row0 + len) of every head.  Dense batches are
// one sequence of N rows per (batch, head) tensor-map index.
struct SeqRows {
  int row0, len;
};

__device__ __forceinline__ SeqRows seq_rows(const BwdParams& p, int b) {
  if (p.cu_seqlens == nullptr) return SeqRows{0, p.N};
  // clamped into [0, N] so that no access leaves the tensors
  const int s0 = min(max(__ldg(p.cu_seqlens + b), 0), p.N);
  const int s1 = min(max(__ldg(p.cu_seqlens + b + 1), s0), p.N);
  return SeqRows{s0, min(s1 - s0, p.max_seqlen)};
}

struct DkvUnit {
  int bhkv;      // key/value head (batch * heads_kv + head)
  int zkv, zq0;  // tensor-map index of the K/V head and of its group's first query head
  int row0, len; // the sequence's rows
  int j, i0;     // key tile; first query tile a query head sees
  int per_head;  // steps per query head (query tiles i0 .. end of the sequence)
  int nsteps;    // group * per_head (0: the key tile lies past the sequence's end)
};

// Tensor-map index of the query head and query tile of step s of a unit: the
// group's query heads one after another, each over its query tiles.
__device__ __forceinline__ void dkv_step(const DkvUnit& w, int s, int* zq, int* i) {
  const int g = s / w.per_head;
  *zq = w.zq0 + g;
  *i = w.i0 + (s - g * w.per_head);
}

template <bool CAUSAL>
__device__ __forceinline__ DkvUnit decode_dkv_unit(int u, const BwdParams& p) {
  DkvUnit w;
  if (CAUSAL || p.cu_seqlens != nullptr) {
    // K/V tile j sees query tiles j..n-1: ascending j is longest first,
    // within blocks of head_block heads.
    const BlockedUnit bu = blocked_unit(u, p.BHkv, p.head_block, p.n_kblocks, 1);
    w.j = bu.cls;
    w.bhkv = bu.head;
  } else {
    w.bhkv = u / p.n_kblocks;
    w.j = u - w.bhkv * p.n_kblocks;
  }
  w.i0 = CAUSAL ? w.j : 0;
  const int b = w.bhkv / p.heads_kv;
  const int hkv = w.bhkv - b * p.heads_kv;
  const SeqRows sr = seq_rows(p, b);
  w.row0 = sr.row0;
  w.len = sr.len;
  if (p.cu_seqlens != nullptr) {
    w.zkv = hkv;
    w.zq0 = hkv * p.group;
  } else {
    w.zkv = w.bhkv;
    w.zq0 = b * p.heads + hkv * p.group;
  }
  const int nt = (w.len + 127) >> 7;
  w.per_head = w.j < nt ? nt - w.i0 : 0;
  w.nsteps = p.group * w.per_head;
  return w;
}

template <int D, bool CAUSAL, bool BF16>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_dkv_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
                   const BwdParams p) {
  using L = DkvLayout<D>;
  constexpr int kTile = L::kTile;
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sbase = smem_u32(smem);
  if (sbase & 1023u) {  // the swizzled tiles need 1024-byte alignment
    if (threadIdx.x == 0 && p.status != nullptr)
      atomicCAS(p.status, 0u, kStatusLayout | ((blockIdx.x & 0xFFFFu) << 16));
    return;
  }
  const uint32_t bar0 = sbase + L::kBar;
  auto bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + L::kMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kMisc + 4);
  volatile int* unit_ring = reinterpret_cast<volatile int*>(smem + L::kMisc + 16);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  Watchdog wd{p.status, abort_flag, p.wait_limit_ns};

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    for (int s = 0; s < kUnitSlots; ++s) {
      mbar_init(bar(L::kUnitFull + s), 1);
      mbar_init(bar(L::kUnitEmpty + s), kUnitReaders);
    }
    mbar_init(bar(L::kKvFull), 1);
    mbar_init(bar(L::kKvEmpty), 1);
    for (int s = 0; s < L::kQSlots; ++s) {
      mbar_init(bar(L::kQFull + s), 1);
      mbar_init(bar(L::kQEmpty + s), 1);
    }
    for (int s = 0; s < L::kDoSlots; ++s) {
      mbar_init(bar(L::kDoFull + s), 2);  // TMA bytes + the -LSE/-D writer
      mbar_init(bar(L::kDoEmpty + s), 1);
      mbar_init(bar(L::kVecEmpty + s), 8);  // one arrival per compute warp
    }
    mbar_init(bar(L::kSFull), 1);
    mbar_init(bar(L::kSFull + 1), 1);
    mbar_init(bar(L::kDpFull), 1);
    mbar_init(bar(L::kPReady), 256);
    mbar_init(bar(L::kPReady + 1), 256);
    mbar_init(bar(L::kDsReady), 256);
    mbar_init(bar(L::kDkvFull), 1);
    mbar_init(bar(L::kDkvFree), 256);
    mbar_init(bar(L::kDrain), 1);
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
  const int num_units = p.BHkv * p.n_kblocks;

  if (warp == kWarpProducer) {
    // -------------------------------------------------------------- producer ---
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      tma_prefetch_desc(&tmDO);
    }
    uint32_t kv_it = 0, st_it = 0, un = 0;
    uint32_t q_issued = 0, do_issued = 0;  // copies issued (lane 0), for the drain
    bool ok = true;
    while (ok) {
      int u = -1;
      if (lane == 0)
        u = publish_unit(unit_ring, bar(L::kUnitFull), bar(L::kUnitEmpty), un, p.sched, num_units,
                         wd, ok, 38);
      ++un;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      u = __shfl_sync(0xffffffffu, u, 0);
      if (!ok || u < 0) break;
      const DkvUnit w = decode_dkv_unit<CAUSAL>(u, p);
      if (w.nsteps == 0) continue;
      if (lane == 0) {
        ok = mbar_wait(bar(L::kKvEmpty), (kv_it & 1) ^ 1, wd, 21);
        if (ok) {
          mbar_arrive_expect_tx(bar(L::kKvFull), 2 * kTile);
          load_tile<D>(sbase + L::kK, &tmK, bar(L::kKvFull), w.row0 + w.j * 128, w.zkv);
          load_tile<D>(sbase + L::kV, &tmV, bar(L::kKvFull), w.row0 + w.j * 128, w.zkv);
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      ++kv_it;
      for (int s = 0; s < w.nsteps && ok; ++s) {
        int zq, i;
        dkv_step(w, s, &zq, &i);
        const uint32_t qs = st_it % L::kQSlots, ds = st_it % L::kDoSlots;
        if (lane == 0) {
          ok = mbar_wait(bar(L::kQEmpty + qs), ((st_it / L::kQSlots) & 1) ^ 1, wd, 22);
          if (ok) {
            mbar_arrive_expect_tx(bar(L::kQFull + qs), kTile);
            load_tile<D>(sbase + L::kQ0 + qs * kTile, &tmQ, bar(L::kQFull + qs),
                      w.row0 + i * 128, zq);
            ++q_issued;
            ok = mbar_wait(bar(L::kDoEmpty + ds), ((st_it / L::kDoSlots) & 1) ^ 1, wd, 23);
          }
          if (ok) {
            mbar_arrive_expect_tx(bar(L::kDoFull + ds), kTile);
            load_tile<D>(sbase + L::kDo0 + ds * kTile, &tmDO, bar(L::kDoFull + ds),
                      w.row0 + i * 128, zq);
            ++do_issued;
            ok = mbar_wait(bar(L::kVecEmpty + ds), ((st_it / L::kDoSlots) & 1) ^ 1, wd, 37);
          }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        // -LSE * log2(e) and -D of the 128 queries (padding rows: -inf / 0,
        // so their P and dS vanish).
        float l2[4], dd[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int q = i * 128 + 4 * lane + e;
          const bool in = q < w.len;
          const size_t g = (size_t)zq * p.N + w.row0 + (in ? q : 0);
          l2[e] = in ? -p.lse[g] * kLog2e : -INFINITY;
          dd[e] = in ? -p.delta[g] : 0.f;
        }
        float4* vec = reinterpret_cast<float4*>(smem + L::kVec + ds * 1024);
        vec[lane] = make_float4(l2[0], l2[1], l2[2], l2[3]);
        vec[32 + lane] = make_float4(dd[0], dd[1], dd[2], dd[3]);
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(L::kDoFull + ds));
        ++st_it;
      }
    }
    if (lane == 0) {
      // Drain: the copies of the last ring rounds must have landed.
      Watchdog dw = wd;
      volatile int never = 0;
      dw.abort_flag = &never;
      dw.limit_ns = drain_limit_ns(wd.limit_ns);
      if (kv_it > 0) mbar_wait(bar(L::kKvFull), (kv_it - 1) & 1, dw, 24);
      for (uint32_t it = q_issued > (uint32_t)L::kQSlots ? q_issued - L::kQSlots : 0u;
           it < q_issued; ++it)
        mbar_wait(bar(L::kQFull + it % L::kQSlots), (it / L::kQSlots) & 1, dw, 24);
      for (uint32_t it = do_issued > (uint32_t)L::kDoSlots ? do_issued - L::kDoSlots : 0u;
           it < do_issued; ++it)
        mbar_wait(bar(L::kDoFull + it % L::kDoSlots), (it / L::kDoSlots) & 1, dw, 24);
    }
    __syncwarp();
  } else if (warp == kWarpMma) {
    // ------------------------------------------------------------ tcgen05 issuer ---
    // Per step s: S^T(s) | dK(s-1) | dP^T(s) | dV(s); after the unit's last
    // step its dK.  Each group is issued after a rendezvous with the relay
    // warp, which has seen its inputs complete; after an abort both warps
    // walk the rest of the unit (issuing nothing) and leave together at the
    // next unit's rendezvous, so every rendezvous pairs up.
    {
      constexpr uint32_t kIdS = idesc_f16(128, 128, BF16, false, false);   // S^T, dP^T
      constexpr uint32_t kIdKV = idesc_f16(128, D, BF16, false, true);  // dV, dK
      uint32_t st_it = 0;
      bool aborted = false;
      // K and V as K-major A operands of S^T / dP^T.
      const uint64_t kd_k = kmajor_base(sbase + L::kK), vd_k = kmajor_base(sbase + L::kV);
      // dK(s) += dS^T(s) Q_i(s) with Q from its ring slot; then Q's slot is
      // free.
      auto issue_dk = [&](uint32_t step, uint32_t acc0) {
        const uint32_t qs = step % L::kQSlots;
        const uint64_t qd_mn = mnmajor_base(sbase + L::kQ0 + qs * kTile);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_f16_ts(tbase + kColDK<D>, tbase + kColDP + half_packed_col(kk),
                     desc_plus(qd_mn, mnmajor16_off(kk)), kIdKV, kk > 0 ? 1u : acc0);
        mma_commit(bar(L::kQEmpty + qs));
      };
      for (uint32_t un = 0;; ++un) {
        // the relay has seen the next unit published (after an abort both
        // warps leave here, having met at every rendezvous so far)
        aborted = named_bar_or(kBarRelay, 64, aborted);
        if (aborted) break;
        const int u = read_unit(unit_ring, bar(L::kUnitEmpty), un);
        if (u < 0) break;
        const DkvUnit w = decode_dkv_unit<CAUSAL>(u, p);
        if (w.nsteps == 0) continue;
        // S^T(step) = K Q_i^T into its buffer (the P^T last held there was
        // consumed by a dV issued before, and its S^T read before that P^T
        // was handed over)
        auto issue_st = [&](uint32_t step) {
          const uint32_t b = kDoubleS<D> ? (step & 1) : 0;
          const uint64_t qd = kmajor_base(sbase + L::kQ0 + (step % L::kQSlots) * kTile);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            mma_f16_ss(tbase + kColST0<D> + 128 * b, desc_plus(kd_k, kmajor16_off(kk)),
                       desc_plus(qd, kmajor16_off(kk)), kIdS, kk > 0);
          mma_commit(bar(L::kSFull + b));
        };
        if constexpr (kDoubleS<D>) {
          // Q_i(0) and the unit's K, V have landed: S^T(0)
          aborted = named_bar_or(kBarRelay, 64, aborted);
          if (!aborted && lane == 0) {
            tc_fence_after();
            issue_st(st_it);
          }
        }
        for (int s = 0; s < w.nsteps; ++s) {
          const uint32_t ds = st_it % L::kDoSlots;
          const uint32_t sbuf = kDoubleS<D> ? (st_it & 1) : 0;
          if constexpr (!kDoubleS<D>) {
            // Q_i(s) (and at s = 0 the unit's K, V) have landed: S^T(s)
            aborted = named_bar_or(kBarRelay, 64, aborted);
            if (!aborted && lane == 0) {
              tc_fence_after();
              issue_st(st_it);
            }
          }
          // dK(s-1): its dS^T is in tensor memory
          if (s > 0) {
            aborted = named_bar_or(kBarRelay, 64, aborted);
            if (!aborted && lane == 0) {
              tc_fence_after();
              issue_dk(st_it - 1, s > 1 ? 1u : 0u);
            }
          }
          // dP^T = V dO_i^T once dO_i has landed (dS^T(s-1) in these
          // columns has just been consumed)
          const uint32_t doaddr = sbase + L::kDo0 + ds * kTile;
          aborted = named_bar_or(kBarRelay, 64, aborted);
          if (!aborted && lane == 0) {
            tc_fence_after();
            const uint64_t dod = kmajor_base(doaddr);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk)
              mma_f16_ss(tbase + kColDP, desc_plus(vd_k, kmajor16_off(kk)),
                         desc_plus(dod, kmajor16_off(kk)), kIdS, kk > 0);
            mma_commit(bar(L::kDpFull));
          }
          if constexpr (kDoubleS<D>) {
            // Q_i(s+1) has landed: S^T(s+1) into the other buffer, ahead of dV(s)
            if (s + 1 < w.nsteps) {
              aborted = named_bar_or(kBarRelay, 64, aborted);
              if (!aborted && lane == 0) {
                tc_fence_after();
                issue_st(st_it + 1);
              }
            }
          }
          // dV += P^T dO_i (A = P^T from tensor memory) once P^T is there
          // (and, at s = 0, the previous unit's dV / dK have been stored)
          aborted = named_bar_or(kBarRelay, 64, aborted);
          if (!aborted && lane == 0) {
            tc_fence_after();
            const uint64_t dod_mn = mnmajor_base(doaddr);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              mma_f16_ts(tbase + kColDV, tbase + kColST0<D> + 128 * sbuf + half_packed_col(kk),
                         desc_plus(dod_mn, mnmajor16_off(kk)), kIdKV, kk > 0 || s > 0 ? 1u : 0u);
            mma_commit(bar(L::kDoEmpty + ds));  // dV(s) was the last reader of dO_i
          }
          ++st_it;
        }
        // the unit's last dK, then hand dK / dV to the warpgroups
        aborted = named_bar_or(kBarRelay, 64, aborted);
        if (!aborted && lane == 0) {
          tc_fence_after();
          issue_dk(st_it - 1, w.nsteps > 1 ? 1u : 0u);
          mma_commit(bar(L::kDkvFull));
          mma_commit(bar(L::kKvEmpty));
        }
      }
      if (lane == 0) {
        mma_commit(bar(L::kDrain));
        Watchdog dw = wd;
        volatile int never = 0;
        dw.abort_flag = &never;
        dw.limit_ns = drain_limit_ns(wd.limit_ns);
        mbar_wait(bar(L::kDrain), 0, dw, 32);
      }
    }
    __syncwarp();
  } else if (warp == kWarpRelay) {
    // ------------------------------------------------------------------ relay ---
    // Walks the issuer's schedule: before each rendezvous, waits (all lanes)
    // for what the next MMA group reads.  After an abort the waits are
    // skipped but every rendezvous is still met.
    uint32_t kv_it = 0, st_it = 0, unit_it = 0;
    bool aborted = false;
    auto wait_all = [&](uint32_t b, uint32_t par, int site) {
      if (!aborted) aborted = !__all_sync(0xffffffffu, mbar_wait(b, par, wd, site));
    };
    for (uint32_t un = 0;; ++un) {
      wait_all(bar(L::kUnitFull + un % kUnitSlots), (un / kUnitSlots) & 1, 39);
      aborted = named_bar_or(kBarRelay, 64, aborted);
      if (aborted) break;
      const int u = read_unit(unit_ring, bar(L::kUnitEmpty), un);
      if (u < 0) break;
      const DkvUnit w = decode_dkv_unit<CAUSAL>(u, p);
      if (w.nsteps == 0) continue;
      wait_all(bar(L::kKvFull), kv_it & 1, 25);
      ++kv_it;
      if constexpr (kDoubleS<D>) {
        wait_all(bar(L::kQFull + st_it % L::kQSlots), (st_it / L::kQSlots) & 1, 26);
        aborted = named_bar_or(kBarRelay, 64, aborted);  // S^T(0)
      }
      for (int s = 0; s < w.nsteps; ++s) {
        const uint32_t qs = st_it % L::kQSlots, ds = st_it % L::kDoSlots;
        const uint32_t par = st_it & 1;
        if constexpr (!kDoubleS<D>) {
          wait_all(bar(L::kQFull + qs), (st_it / L::kQSlots) & 1, 26);
          aborted = named_bar_or(kBarRelay, 64, aborted);
        }
        if (s > 0) {
          wait_all(bar(L::kDsReady), par ^ 1, 27);
          aborted = named_bar_or(kBarRelay, 64, aborted);
        }
        wait_all(bar(L::kDoFull + ds), (st_it / L::kDoSlots) & 1, 28);
        aborted = named_bar_or(kBarRelay, 64, aborted);
        if constexpr (kDoubleS<D>) {
          if (s + 1 < w.nsteps) {
            const uint32_t n1 = st_it + 1;
            wait_all(bar(L::kQFull + n1 % L::kQSlots), (n1 / L::kQSlots) & 1, 26);
            aborted = named_bar_or(kBarRelay, 64, aborted);  // S^T(s+1)
          }
        }
        if (s == 0 && unit_it > 0) wait_all(bar(L::kDkvFree), (unit_it - 1) & 1, 29);
        // with two S^T buffers P^T(s+1) can be handed over before this wait,
        // so the hand-off barrier alternates with the buffer too
        if constexpr (kDoubleS<D>)
          wait_all(bar(L::kPReady + (st_it & 1)), (st_it >> 1) & 1, 30);
        else
          wait_all(bar(L::kPReady), par, 30);
        aborted = named_bar_or(kBarRelay, 64, aborted);
        ++st_it;
      }
      wait_all(bar(L::kDsReady), (st_it - 1) & 1, 31);
      aborted = named_bar_or(kBarRelay, 64, aborted);
      ++unit_it;
    }
  } else {
    // ------------------------------------------------------ compute warpgroups ---
    const int h = warp >> 2;                 // query half of every step
    const int r = threadIdx.x & 127;         // TMEM lane: key row
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t dp_addr = tbase + lane_base + kColDP + 64 * h;
    const float sl2 = p.scale_log2;
    uint32_t st_it = 0, unit_it = 0, un = 0;
    bool ok = true;
    while (ok) {
      const int u = take_unit(unit_ring, bar(L::kUnitFull), bar(L::kUnitEmpty), un++, wd, ok, 40);
      ok = named_bar_and(1 + h, 128, ok);
      if (!ok || u < 0) break;
      const DkvUnit w = decode_dkv_unit<CAUSAL>(u, p);
      if (w.nsteps == 0) continue;
      for (int s = 0; s < w.nsteps; ++s) {
        int zq, i;
        dkv_step(w, s, &zq, &i);
        (void)zq;
        const uint32_t ds = st_it % L::kDoSlots;
        const uint32_t par = st_it & 1;
        const uint32_t sbuf = kDoubleS<D> ? (st_it & 1) : 0;
        const uint32_t s_addr = tbase + lane_base + kColST0<D> + 128 * sbuf + 64 * h;
        ok = mbar_wait(bar(L::kSFull + sbuf), kDoubleS<D> ? ((st_it >> 1) & 1) : par, wd, 33);
        // dO_i's full barrier also waits for the -LSE / -D vectors' writer
        ok = ok && mbar_wait(bar(L::kDoFull + ds), (st_it / L::kDoSlots) & 1, wd, 34);
        // Exit decisions are uniform over the warpgroup (its warps meet at
        // named barriers).
        ok = named_bar_and(1 + h, 128, ok);
        if (!ok) break;
        tc_fence_after();
        const float4* nlse4 = reinterpret_cast<const float4*>(smem + L::kVec + ds * 1024) + 16 * h;
        const float4* nd4 = nlse4 + 32;
        const bool diag = CAUSAL && (i == w.j);
        const float2 sl2x2 = make_float2(sl2, sl2);
        // ---- P^T = exp2(S^T c - LSE log2 e), kept in fp32 for dS^T.  Both
        // 32-column chunks are loaded before one wait.
        float pr[64];
        {
          uint32_t sa[32], sb[32];
          tmem_ld32(s_addr, sa);
          tmem_ld32(s_addr + 32, sb);
          tmem_wait_ld();
          reg_fence32(sa);
          reg_fence32(sb);
#pragma unroll
          for (int v = 0; v < 16; ++v) {
            const uint32_t* src = v < 8 ? sa : sb;
            const int o = 4 * (v & 7);
            const float4 nl = nlse4[v];
            const float2 x01 = __ffma2_rn(
                make_float2(__uint_as_float(src[o]), __uint_as_float(src[o + 1])), sl2x2,
                make_float2(nl.x, nl.y));
            const float2 x23 = __ffma2_rn(
                make_float2(__uint_as_float(src[o + 2]), __uint_as_float(src[o + 3])), sl2x2,
                make_float2(nl.z, nl.w));
            pr[4 * v] = ex2_approx(x01.x);
            pr[4 * v + 1] = ex2_approx(x01.y);
            pr[4 * v + 2] = ex2_approx(x23.x);
            pr[4 * v + 3] = ex2_approx(x23.y);
          }
          if (diag) {
#pragma unroll
            for (int col = 0; col < 64; ++col)  // query column within the half
              if (64 * h + col < r) pr[col] = 0.f;  // query before key
          }
          uint32_t pp[16], pq[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            pp[e] = pack16x2(BF16, pr[2 * e], pr[2 * e + 1]);
            pq[e] = pack16x2(BF16, pr[32 + 2 * e], pr[32 + 2 * e + 1]);
          }
          tmem_st16(s_addr, pp);
          tmem_st16(s_addr + 16, pq);
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(bar(L::kPReady + sbuf));
        // ---- dS^T = P^T o (dP^T - D)
        ok = mbar_wait(bar(L::kDpFull), par, wd, 35);
        ok = named_bar_and(1 + h, 128, ok);
        if (!ok) break;
        tc_fence_after();
        {
          uint32_t da[32], db[32];
          tmem_ld32(dp_addr, da);
          tmem_ld32(dp_addr + 32, db);
          tmem_wait_ld();
          reg_fence32(da);
          reg_fence32(db);
          uint32_t pd[16], pe[16];
#pragma unroll
          for (int v = 0; v < 16; ++v) {
            const uint32_t* src = v < 8 ? da : db;
            const int o = 4 * (v & 7);
            const float4 nd = nd4[v];
            const float2 g01 = __fadd2_rn(
                make_float2(__uint_as_float(src[o]), __uint_as_float(src[o + 1])),
                make_float2(nd.x, nd.y));
            const float2 g23 = __fadd2_rn(
                make_float2(__uint_as_float(src[o + 2]), __uint_as_float(src[o + 3])),
                make_float2(nd.z, nd.w));
            const float2 s01 = __fmul2_rn(make_float2(pr[4 * v], pr[4 * v + 1]), g01);
            const float2 s23 = __fmul2_rn(make_float2(pr[4 * v + 2], pr[4 * v + 3]), g23);
            uint32_t* dst = v < 8 ? pd : pe;
            dst[2 * (v & 7)] = pack16x2(BF16, s01.x, s01.y);
            dst[2 * (v & 7) + 1] = pack16x2(BF16, s23.x, s23.y);
          }
          tmem_st16(dp_addr, pd);
          tmem_st16(dp_addr + 16, pe);
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(bar(L::kDsReady));
        // this warp has read its -LSE / -D for the step
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(L::kVecEmpty + ds));
        ++st_it;
      }
      if (!ok) break;
      // ---------------------------------------------------- dK / dV epilogue ---
      ok = mbar_wait(bar(L::kDkvFull), unit_it & 1, wd, 36);
      ok = named_bar_and(1 + h, 128, ok);
      if (!ok) break;
      ++unit_it;
      tc_fence_after();
      const int key = w.j * 128 + r;
      const uint32_t src = tbase + lane_base + (h == 0 ? kColDV : kColDK<D>);
      const float mult = (h == 0) ? 1.f : p.scale;
      uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(h == 0 ? p.dv : p.dk) +
                                            ((size_t)w.zkv * p.N + w.row0 + key) * D);
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t raw[32];
        tmem_ld32_sync(src + 32 * c, raw);
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e)
          pk[e] = pack16x2(BF16, __uint_as_float(raw[2 * e]) * mult,
                           __uint_as_float(raw[2 * e + 1]) * mult);
        if (key < w.len) {
#pragma unroll
          for (int v = 0; v < 4; ++v)
            dst[4 * c + v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
        }
      }
      tc_fence_before();
      mbar_arrive(bar(L::kDkvFree));
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
}

// ================================================================ dQ kernel ===

// K_j is read by S_j and, one step later, by dQ_j; V_j only by dP_j.  Each
// gets a ring sized to its lifetime (3 K slots, 2 V slots) so a slot's next
// load has about two steps of MMA work to land in.  Q_i and dO_i land here
// and are copied into tensor memory once per unit, so the S and dP MMAs read
// only K_j / V_j from shared memory.
template <int D>
struct DqLayout {
  static constexpr int kTile = kTileBytes<D>;
  static constexpr int kQ = 0;                    // Q_i staging (K-major)
  static constexpr int kDO = kTile;               // dO_i staging (K-major)
  static constexpr int kKSlots = 3, kVSlots = 2;
  static constexpr int kK0 = 2 * kTile;           // K ring
  static constexpr int kV0 = kK0 + kKSlots * kTile;  // V ring
  static constexpr int kBar = kV0 + kVSlots * kTile;
  enum {
    kQFull, kQEmpty, kKFull, kKEmpty = kKFull + kKSlots, kVFull = kKEmpty + kKSlots,
    kVEmpty = kVFull + kVSlots, kSFull = kVEmpty + kVSlots, kSRead = kSFull + 2, kDpFull,
    kDsReady, kDqFull, kDqFree, kDrain, kUnitFull, kUnitEmpty = kUnitFull + kUnitSlots,
    kNumBars = kUnitEmpty + kUnitSlots
  };
  static constexpr int kMisc = kBar + kNumBars * 8;  // TMEM address, abort flag, unit ring
  static constexpr int kBytes = kMisc + 16 + 4 * kUnitSlots;
  static_assert(kBytes <= 232448, "shared memory budget (227 KB) exceeded");
};

// Tensor memory: dQ [0,128)  two step buffers [128,256) [256,384)  Q_i
// [384,448)  dO_i [448,512) (16-bit, two values per column: the A operands of
// S and dP).  Step j uses buffer j%2 for S_j, then (once S_j has been read)
// for dP_j; dS_j (16-bit) of warpgroup h overwrites its columns
// [64h, 64h+32) after dP_j has been read.
constexpr uint32_t kColDQ = 0, kColS0 = 128, kColQ = 384, kColDO = 448;

struct DqUnit {
  int bh, i, nsteps;  // nsteps = 0: the query tile lies past the sequence's end
  int zq, zkv;        // tensor-map index of the query head and of its K/V head
  int row0, len;      // the sequence's rows
};

template <bool CAUSAL>
__device__ __forceinline__ DqUnit decode_dq_unit(int u, const BwdParams& p) {
  DqUnit w;
  if (CAUSAL || p.cu_seqlens != nullptr) {
    // Query tile i sees key tiles 0..i: descending i is longest first,
    // within blocks of head_block_q heads.
    const BlockedUnit bu = blocked_unit(u, p.BH, p.head_block_q, p.n_qtiles, 1);
    w.bh = bu.head;
    w.i = p.n_qtiles - 1 - bu.cls;
  } else {
    w.bh = u / p.n_qtiles;
    w.i = u - w.bh * p.n_qtiles;
  }
  const int b = w.bh / p.heads;
  const int hq = w.bh - b * p.heads;
  const SeqRows sr = seq_rows(p, b);
  w.row0 = sr.row0;
  w.len = sr.len;
  if (p.cu_seqlens != nullptr) {
    w.zq = hq;
    w.zkv = hq / p.group;
  } else {
    w.zq = w.bh;
    w.zkv = b * p.heads_kv + hq / p.group;
  }
  const int nt = (w.len + 127) >> 7;
  w.nsteps = w.i < nt ? (CAUSAL ? w.i + 1 : nt) : 0;
  return w;
}

template <int D, bool CAUSAL, bool BF16>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_dq_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
                  const BwdParams p) {
  using L = DqLayout<D>;
  constexpr int kTile = L::kTile;
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sbase = smem_u32(smem);
  if (sbase & 1023u) {
    if (threadIdx.x == 0 && p.status != nullptr)
      atomicCAS(p.status, 0u, kStatusLayout | ((blockIdx.x & 0xFFFFu) << 16));
    return;
  }
  const uint32_t bar0 = sbase + L::kBar;
  auto bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + L::kMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kMisc + 4);
  volatile int* unit_ring = reinterpret_cast<volatile int*>(smem + L::kMisc + 16);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  Watchdog wd{p.status, abort_flag, p.wait_limit_ns};

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    for (int s = 0; s < kUnitSlots; ++s) {
      mbar_init(bar(L::kUnitFull + s), 1);
      mbar_init(bar(L::kUnitEmpty + s), kUnitReaders);
    }
    mbar_init(bar(L::kQFull), 1);
    mbar_init(bar(L::kQEmpty), 1);
    for (int s = 0; s < L::kKSlots; ++s) {
      mbar_init(bar(L::kKFull + s), 1);
      mbar_init(bar(L::kKEmpty + s), 1);
    }
    for (int s = 0; s < L::kVSlots; ++s) {
      mbar_init(bar(L::kVFull + s), 1);
      mbar_init(bar(L::kVEmpty + s), 1);
    }
    for (int s = 0; s < 2; ++s) mbar_init(bar(L::kSFull + s), 1);
    mbar_init(bar(L::kSRead), 256);
    mbar_init(bar(L::kDpFull), 1);
    mbar_init(bar(L::kDsReady), 256);
    mbar_init(bar(L::kDqFull), 1);
    mbar_init(bar(L::kDqFree), 256);
    mbar_init(bar(L::kDrain), 1);
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
  const int num_units = p.BH * p.n_qtiles;

  if (warp == kWarpProducer) {
    // -------------------------------------------------------------- producer ---
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      tma_prefetch_desc(&tmDO);
      uint32_t k_it = 0, v_it = 0, unit_it = 0, un = 0;
      bool ok = true;
      while (ok) {
        const int u = publish_unit(unit_ring, bar(L::kUnitFull), bar(L::kUnitEmpty), un++,
                                   p.sched + 1, num_units, wd, ok, 38);
        if (u < 0) break;
        const DqUnit w = decode_dq_unit<CAUSAL>(u, p);
        if (w.nsteps == 0) continue;
        ok = mbar_wait(bar(L::kQEmpty), (unit_it & 1) ^ 1, wd, 41);
        if (!ok) break;
        mbar_arrive_expect_tx(bar(L::kQFull), 2 * kTile);
        load_tile<D>(sbase + L::kQ, &tmQ, bar(L::kQFull), w.row0 + w.i * 128, w.zq);
        load_tile<D>(sbase + L::kDO, &tmDO, bar(L::kQFull), w.row0 + w.i * 128, w.zq);
        ++unit_it;
        for (int j = 0; j < w.nsteps && ok; ++j) {
          const uint32_t ks = k_it % L::kKSlots;
          ok = mbar_wait(bar(L::kKEmpty + ks), ((k_it / L::kKSlots) & 1) ^ 1, wd, 42);
          if (!ok) break;
          mbar_arrive_expect_tx(bar(L::kKFull + ks), kTile);
          load_tile<D>(sbase + L::kK0 + ks * kTile, &tmK, bar(L::kKFull + ks), w.row0 + j * 128,
                    w.zkv);
          ++k_it;
          const uint32_t vs = v_it % L::kVSlots;
          ok = mbar_wait(bar(L::kVEmpty + vs), ((v_it / L::kVSlots) & 1) ^ 1, wd, 43);
          if (!ok) break;
          mbar_arrive_expect_tx(bar(L::kVFull + vs), kTile);
          load_tile<D>(sbase + L::kV0 + vs * kTile, &tmV, bar(L::kVFull + vs), w.row0 + j * 128,
                    w.zkv);
          ++v_it;
        }
      }
      // Drain: the copies of the last ring round (and of Q) must have landed.
      Watchdog dw = wd;
      volatile int never = 0;
      dw.abort_flag = &never;
      dw.limit_ns = drain_limit_ns(wd.limit_ns);
      if (unit_it > 0) mbar_wait(bar(L::kQFull), (unit_it - 1) & 1, dw, 44);
      for (uint32_t it = k_it > (uint32_t)L::kKSlots ? k_it - L::kKSlots : 0u; it < k_it; ++it)
        mbar_wait(bar(L::kKFull + it % L::kKSlots), (it / L::kKSlots) & 1, dw, 44);
      for (uint32_t it = v_it > (uint32_t)L::kVSlots ? v_it - L::kVSlots : 0u; it < v_it; ++it)
        mbar_wait(bar(L::kVFull + it % L::kVSlots), (it / L::kVSlots) & 1, dw, 44);
    }
    __syncwarp();
  } else if (warp == kWarpMma) {
    // ------------------------------------------------------------ tcgen05 issuer ---
    // Per unit: Q_i, dO_i copied into tensor memory.  Per step j (buffer
    // b = j%2): S_j into b | dQ += dS_{j-1} K_{j-1} | dP_j into b once the
    // warpgroups have read S_j.  The warpgroups compute P_j while dQ and dP_j
    // run, and dS_j while S_{j+1} runs.  Each group is issued after a
    // rendezvous with the relay warp, which has seen its inputs complete.
    // After an abort both warps walk the rest of the unit (issuing nothing)
    // and leave together at the next unit's rendezvous, so every rendezvous
    // pairs up.
    {
      constexpr uint32_t kIdS = idesc_f16(128, 128, BF16, false, false);  // S, dP
      constexpr uint32_t kIdQ = idesc_f16(128, D, BF16, false, true);  // dQ
      uint32_t k_it = 0, v_it = 0, step_it = 0;
      bool aborted = false;
      const uint64_t qd = kmajor_base(sbase + L::kQ), dod = kmajor_base(sbase + L::kDO);
      // dQ += dS K_j: A = dS from tensor memory (buffer sb), B = K_j read MN-major.
      auto issue_dq = [&](uint32_t kaddr, uint32_t sb, uint32_t acc0) {
        const uint64_t kd_mn = mnmajor_base(kaddr);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_f16_ts(tbase + kColDQ, tbase + kColS0 + 128 * sb + half_packed_col(kk),
                     desc_plus(kd_mn, mnmajor16_off(kk)), kIdQ, kk > 0 ? 1u : acc0);
      };
      for (uint32_t un = 0;; ++un) {
        // the relay has seen the next unit published (after an abort both
        // warps leave here, having met at every rendezvous so far)
        aborted = named_bar_or(kBarRelay, 64, aborted);
        if (aborted) break;
        const int u = read_unit(unit_ring, bar(L::kUnitEmpty), un);
        if (u < 0) break;
        const DqUnit w = decode_dq_unit<CAUSAL>(u, p);
        if (w.nsteps == 0) continue;
        uint32_t prev_kaddr = 0, prev_ks = 0, prev_sb = 0;
        for (int j = 0; j < w.nsteps; ++j) {
          const uint32_t ks = k_it % L::kKSlots;
          const uint32_t kaddr = sbase + L::kK0 + ks * kTile;
          const uint32_t sb = step_it & 1;
          // K_j (and at j = 0 Q_i, dO_i) have landed
          aborted = named_bar_or(kBarRelay, 64, aborted);
          if (!aborted && lane == 0) {
            tc_fence_after();
            if (j == 0) {
              // Q_i, dO_i into tensor memory, 16 columns of d per copy.  The
              // previous unit's S and dP (their last readers) have completed:
              // the dS that the last dQ awaited was computed from them.
#pragma unroll
              for (int kk = 0; kk < D / 16; ++kk) {
                tmem_cp_128x256b(tbase + kColQ + 8 * kk, desc_plus(qd, kmajor16_off(kk)));
                tmem_cp_128x256b(tbase + kColDO + 8 * kk, desc_plus(dod, kmajor16_off(kk)));
              }
              mma_commit(bar(L::kQEmpty));  // the staging tiles may be reloaded
            }
            // S_j = Q_i K_j^T into buffer sb (its previous contents, dS_{j-2},
            // were read by dQ_{j-2}, issued before).
            const uint64_t kd = kmajor_base(kaddr);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk)
              mma_f16_ts(tbase + kColS0 + 128 * sb, tbase + kColQ + 8 * kk,
                         desc_plus(kd, kmajor16_off(kk)), kIdS, kk > 0);
            mma_commit(bar(L::kSFull + sb));
          }
          if (j > 0) {
            // dS_{j-1} is ready (and, for the unit's first dQ, dQ is free)
            aborted = named_bar_or(kBarRelay, 64, aborted);
            if (!aborted && lane == 0) {
              tc_fence_after();
              issue_dq(prev_kaddr, prev_sb, j > 1 ? 1u : 0u);
              mma_commit(bar(L::kKEmpty + prev_ks));
            }
          }
          // V_j has landed and S_j has been read: dP_j = dO_i V_j^T into sb
          const uint32_t vs = v_it % L::kVSlots;
          aborted = named_bar_or(kBarRelay, 64, aborted);
          if (!aborted && lane == 0) {
            tc_fence_after();
            const uint64_t vd = kmajor_base(sbase + L::kV0 + vs * kTile);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk)
              mma_f16_ts(tbase + kColS0 + 128 * sb, tbase + kColDO + 8 * kk,
                         desc_plus(vd, kmajor16_off(kk)), kIdS, kk > 0);
            mma_commit(bar(L::kDpFull));
            mma_commit(bar(L::kVEmpty + vs));
          }
          prev_kaddr = kaddr;
          prev_ks = ks;
          prev_sb = sb;
          ++k_it;
          ++v_it;
          ++step_it;
        }
        // dQ += dS_last K_last, then hand dQ to the warpgroups
        aborted = named_bar_or(kBarRelay, 64, aborted);
        if (!aborted && lane == 0) {
          tc_fence_after();
          issue_dq(prev_kaddr, prev_sb, w.nsteps > 1 ? 1u : 0u);
          mma_commit(bar(L::kKEmpty + prev_ks));
          mma_commit(bar(L::kDqFull));
        }
      }
      if (lane == 0) {
        mma_commit(bar(L::kDrain));
        Watchdog dw = wd;
        volatile int never = 0;
        dw.abort_flag = &never;
        dw.limit_ns = drain_limit_ns(wd.limit_ns);
        mbar_wait(bar(L::kDrain), 0, dw, 51);
      }
    }
    __syncwarp();
  } else if (warp == kWarpRelay) {
    // ------------------------------------------------------------------ relay ---
    // Walks the issuer's schedule: before each rendezvous, waits (all lanes)
    // for what the next MMA group reads.  After an abort the waits are
    // skipped but every rendezvous is still met.
    uint32_t k_it = 0, v_it = 0, step_it = 0, unit_it = 0;
    bool aborted = false;
    auto wait_all = [&](uint32_t b, uint32_t par, int site) {
      if (!aborted) aborted = !__all_sync(0xffffffffu, mbar_wait(b, par, wd, site));
    };
    for (uint32_t un = 0;; ++un) {
      wait_all(bar(L::kUnitFull + un % kUnitSlots), (un / kUnitSlots) & 1, 39);
      aborted = named_bar_or(kBarRelay, 64, aborted);
      if (aborted) break;
      const int u = read_unit(unit_ring, bar(L::kUnitEmpty), un);
      if (u < 0) break;
      const DqUnit w = decode_dq_unit<CAUSAL>(u, p);
      if (w.nsteps == 0) continue;
      for (int j = 0; j < w.nsteps; ++j) {
        if (j == 0) wait_all(bar(L::kQFull), unit_it & 1, 45);
        wait_all(bar(L::kKFull + k_it % L::kKSlots), (k_it / L::kKSlots) & 1, 46);
        aborted = named_bar_or(kBarRelay, 64, aborted);
        if (j > 0) {
          wait_all(bar(L::kDsReady), (step_it - 1) & 1, 47);
          if (j == 1 && unit_it > 0) wait_all(bar(L::kDqFree), (unit_it - 1) & 1, 48);
          aborted = named_bar_or(kBarRelay, 64, aborted);
        }
        wait_all(bar(L::kVFull + v_it % L::kVSlots), (v_it / L::kVSlots) & 1, 55);
        wait_all(bar(L::kSRead), step_it & 1, 56);
        aborted = named_bar_or(kBarRelay, 64, aborted);
        ++k_it;
        ++v_it;
        ++step_it;
      }
      wait_all(bar(L::kDsReady), (step_it - 1) & 1, 49);
      if (w.nsteps == 1 && unit_it > 0) wait_all(bar(L::kDqFree), (unit_it - 1) & 1, 50);
      aborted = named_bar_or(kBarRelay, 64, aborted);
      ++unit_it;
    }
  } else {
    // ------------------------------------------------------ compute warpgroups ---
    const int h = warp >> 2;                 // key half of every step
    const int r = threadIdx.x & 127;         // TMEM lane: query row
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t dq_addr = tbase + lane_base + kColDQ;
    const float sl2 = p.scale_log2;
    uint32_t unit_it = 0, step_it = 0, un = 0;
    bool ok = true;
    while (ok) {
      const int u = take_unit(unit_ring, bar(L::kUnitFull), bar(L::kUnitEmpty), un++, wd, ok, 40);
      ok = named_bar_and(1 + h, 128, ok);
      if (!ok || u < 0) break;
      const DqUnit w = decode_dq_unit<CAUSAL>(u, p);
      if (w.nsteps == 0) continue;
      const int row = w.i * 128 + r;
      const bool in = row < w.len;
      const size_t grow = (size_t)w.zq * p.N + w.row0 + (in ? row : 0);
      // Padding rows: LSE = +inf, D = 0, so their P and dS vanish.
      const float nl2 = in ? -p.lse[grow] * kLog2e : -INFINITY;
      const float nd = in ? -p.delta[grow] : 0.f;
      const float2 sl2x2 = make_float2(sl2, sl2), nl2x2 = make_float2(nl2, nl2),
                   nd2x2 = make_float2(nd, nd);
      for (int j = 0; j < w.nsteps; ++j) {
        const uint32_t sb = step_it & 1;
        const uint32_t par = step_it & 1;
        ok = mbar_wait(bar(L::kSFull + sb), (step_it >> 1) & 1, wd, 52);
        ok = named_bar_and(1 + h, 128, ok);
        if (!ok) break;
        tc_fence_after();
        const bool diag = CAUSAL && (j == w.i);
        // S_j, then dP_j and dS_j, in this step's buffer
        const uint32_t s_addr = tbase + lane_base + kColS0 + 128 * sb + 64 * h;
        const uint32_t dp_addr = s_addr;
        // ---- P = exp2(S c - LSE log2 e), kept in fp32 for dS.  Both
        // 32-column chunks are loaded before one wait; then the buffer may
        // take dP_j.
        float pr[64];
        {
          uint32_t sa[32], sc[32];
          tmem_ld32(s_addr, sa);
          tmem_ld32(s_addr + 32, sc);
          tmem_wait_ld();
          reg_fence32(sa);
          reg_fence32(sc);
          tc_fence_before();
          mbar_arrive(bar(L::kSRead));
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const uint32_t* src = e < 16 ? sa : sc;
            const int o = 2 * (e & 15);
            const float2 x = __ffma2_rn(
                make_float2(__uint_as_float(src[o]), __uint_as_float(src[o + 1])), sl2x2, nl2x2);
            pr[2 * e] = ex2_approx(x.x);
            pr[2 * e + 1] = ex2_approx(x.y);
          }
          if (diag) {
#pragma unroll
            for (int col = 0; col < 64; ++col)  // key column within the half
              if (64 * h + col > r) pr[col] = 0.f;  // key after query
          }
          // keys past the sequence's end (zero-filled or another sequence's)
          const int kend = w.len - j * 128 - 64 * h;
          if (kend < 64) {
#pragma unroll
            for (int col = 0; col < 64; ++col)
              if (col >= kend) pr[col] = 0.f;
          }
        }
        // ---- dS = P o (dP - D)
        ok = mbar_wait(bar(L::kDpFull), par, wd, 53);
        ok = named_bar_and(1 + h, 128, ok);
        if (!ok) break;
        tc_fence_after();
        {
          uint32_t da[32], db[32];
          tmem_ld32(dp_addr, da);
          tmem_ld32(dp_addr + 32, db);
          tmem_wait_ld();
          reg_fence32(da);
          reg_fence32(db);
          uint32_t pd[16], pe[16];
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const uint32_t* src = e < 16 ? da : db;
            const int o = 2 * (e & 15);
            const float2 g = __fadd2_rn(
                make_float2(__uint_as_float(src[o]), __uint_as_float(src[o + 1])), nd2x2);
            const float2 sv = __fmul2_rn(make_float2(pr[2 * e], pr[2 * e + 1]), g);
            (e < 16 ? pd : pe)[e & 15] = pack16x2(BF16, sv.x, sv.y);
          }
          tmem_st16(dp_addr, pd);
          tmem_st16(dp_addr + 16, pe);
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(bar(L::kDsReady));
        ++step_it;
      }
      if (!ok) break;
      // ------------------------------------------------------------ dQ epilogue ---
      ok = mbar_wait(bar(L::kDqFull), unit_it & 1, wd, 54);
      ok = named_bar_and(1 + h, 128, ok);
      if (!ok) break;
      ++unit_it;
      tc_fence_after();
      uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.dq) + grow * D);
      // 32-column chunks alternate between the two warpgroups.
#pragma unroll
      for (int cc = 0; cc < (D / 32 + 1) / 2; ++cc) {
        const int c = 2 * cc + h;
        if (c >= D / 32) break;  // warp-uniform
        uint32_t raw[32];
        tmem_ld32_sync(dq_addr + 32 * c, raw);
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e)
          pk[e] = pack16x2(BF16, __uint_as_float(raw[2 * e]) * p.scale,
                           __uint_as_float(raw[2 * e + 1]) * p.scale);
        if (in) {
#pragma unroll
          for (int v = 0; v < 4; ++v)
            dst[4 * c + v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
        }
      }
      tc_fence_before();
      mbar_arrive(bar(L::kDqFree));
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
}

// ================================================================ D kernel ===

// D_i = sum_c dO_ic O_ic with one warp per row (up to 4 values per lane, then a
// butterfly of warp shuffles).
template <int D, bool BF16>
__global__ void __launch_bounds__(256) bwd_pre_kernel(const uint16_t* __restrict__ o,
                                                     const uint16_t* __restrict__ dout,
                                                     float* __restrict__ delta, long rows,
                                                     int* __restrict__ sched) {
  constexpr int W = (D + 63) / 64;  // 32-bit words (two values each) per lane, at most
  // the main kernels' work counters start at 0 (they run after this kernel
  // on the same stream)
  if (sched != nullptr && blockIdx.x == 0 && threadIdx.x < 2) sched[threadIdx.x] = 0;
  const long warp0 = ((long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const long nwarps = ((long)gridDim.x * blockDim.x) >> 5;
  const int lane = threadIdx.x & 31;
  for (long row = warp0; row < rows; row += nwarps) {
    uint32_t aw[W], bw[W];
    if constexpr (D == 128) {  // the whole row in one 8-byte load per lane
      const uint2 a = reinterpret_cast<const uint2*>(o + row * D)[lane];
      const uint2 b = reinterpret_cast<const uint2*>(dout + row * D)[lane];
      aw[0] = a.x;
      aw[1] = a.y;
      bw[0] = b.x;
      bw[1] = b.y;
    } else {
      // word lane + 32 e of the row (D / 2 words; D = 96 leaves lanes 16-31
      // without a second word)
#pragma unroll
      for (int e = 0; e < W; ++e) {
        const int wi = lane + 32 * e;
        const bool in = wi < D / 2;
        aw[e] = in ? reinterpret_cast<const uint32_t*>(o + row * D)[wi] : 0u;
        bw[e] = in ? reinterpret_cast<const uint32_t*>(dout + row * D)[wi] : 0u;
      }
    }
    float acc = 0.f;
#pragma unroll
    for (int e = 0; e < W; ++e) {
      float a0, a1, b0, b1;
      if (BF16) {
        a0 = __uint_as_float(aw[e] << 16);
        a1 = __uint_as_float(aw[e] & 0xFFFF0000u);
        b0 = __uint_as_float(bw[e] << 16);
        b1 = __uint_as_float(bw[e] & 0xFFFF0000u);
      } else {
        a0 = __half2float(__ushort_as_half((unsigned short)(aw[e] & 0xFFFF)));
        a1 = __half2float(__ushort_as_half((unsigned short)(aw[e] >> 16)));
        b0 = __half2float(__ushort_as_half((unsigned short)(bw[e] & 0xFFFF)));
        b1 = __half2float(__ushort_as_half((unsigned short)(bw[e] >> 16)));
      }
      acc = fmaf(a0, b0, acc);
      acc = fmaf(a1, b1, acc);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (lane == 0) delta[row] = acc;
  }
}

template <typename Kern>
cudaError_t launch_persistent(Kern kern, int threads, int bytes, DeviceFlags& configured,
                              const BwdLaunch& a, int units) {
  cudaError_t e = ensure_dyn_smem(kern, bytes, configured);
  if (e != cudaSuccess) return e;
  const int grid = units < a.num_sms ? units : a.num_sms;
  kern<<<grid, threads, bytes, a.stream>>>(a.tmQ, a.tmK, a.tmV, a.tmDO, a.params);
  return cudaGetLastError();
}

template <int D, bool CAUSAL, bool BF16>
cudaError_t launch_main(const BwdLaunch& a) {
  static DeviceFlags dkv_configured, dq_configured;  // per device and instantiation
  cudaError_t e = launch_persistent(bwd_dkv_kernel<D, CAUSAL, BF16>, kThreads,
                                    DkvLayout<D>::kBytes, dkv_configured, a,
                                    a.params.BHkv * a.params.n_kblocks);
  if (e != cudaSuccess) return e;
  return launch_persistent(bwd_dq_kernel<D, CAUSAL, BF16>, kThreads, DqLayout<D>::kBytes,
                           dq_configured, a, a.params.BH * a.params.n_qtiles);
}

// D_i = sum_c dO_ic O_ic for every row of O / dO: every (batch, head) holds
// N rows, a packed variable-length batch N per head.
template <int D, bool BF16>
cudaError_t launch_pre(const BwdParams& p, int num_sms, cudaStream_t stream) {
  const long rows = (long)(p.cu_seqlens != nullptr ? p.heads : p.BH) * p.N;
  long blocks = (rows + 7) / 8;
  const long cap = (long)num_sms * 16;
  if (blocks > cap) blocks = cap;
  bwd_pre_kernel<D, BF16><<<(int)blocks, 256, 0, stream>>>(
      static_cast<const uint16_t*>(p.o), static_cast<const uint16_t*>(p.dout), p.delta, rows,
      p.sched);
  return cudaGetLastError();
}

template <int D, bool BF16>
cudaError_t launch_all(const BwdLaunch& a) {
  cudaError_t e = launch_pre<D, BF16>(a.params, a.num_sms, a.stream);
  if (e != cudaSuccess) return e;
  return a.causal ? launch_main<D, true, BF16>(a) : launch_main<D, false, BF16>(a);
}

}  // namespace

cudaError_t launch_bwd_pre(const BwdParams& p, int d, bool bf16, int num_sms,
                           cudaStream_t stream) {
  if (d == 256)
    return bf16 ? launch_pre<256, true>(p, num_sms, stream) : launch_pre<256, false>(p, num_sms, stream);
  if (d == 192)
    return bf16 ? launch_pre<192, true>(p, num_sms, stream) : launch_pre<192, false>(p, num_sms, stream);
  if (d == 128)
    return bf16 ? launch_pre<128, true>(p, num_sms, stream) : launch_pre<128, false>(p, num_sms, stream);
  if (d == 96)
    return bf16 ? launch_pre<96, true>(p, num_sms, stream) : launch_pre<96, false>(p, num_sms, stream);
  return bf16 ? launch_pre<64, true>(p, num_sms, stream) : launch_pre<64, false>(p, num_sms, stream);
}

cudaError_t launch_bwd(const BwdLaunch& a) {
  if (a.d == 64) return a.bf16 ? launch_all<64, true>(a) : launch_all<64, false>(a);
  if (a.d == 96) return a.bf16 ? launch_all<96, true>(a) : launch_all<96, false>(a);
  return a.bf16 ? launch_all<128, true>(a) : launch_all<128, false>(a);
}

}  // namespace attn
