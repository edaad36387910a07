// Backward pass for the wide head dims d in {192, 256} on sm_103a.
//
// The same stages as bwd.cu ("FlashAttention-2: Faster Attention with Better
// Parallelism and Work Partitioning" (review page), "Methods" and "핵심
// 구성요소": the backward pass recomputes P from the stored log-sum-exp):
// the D pass (bwd.cu), a dK/dV kernel per key tile and a dQ kernel per query
// tile, each accumulating its outputs in tensor memory with no atomics.  The
// tiles change because 128 x d tiles of four tensors do not fit:
//
//  * Tensor memory (512 columns).  dK and dV of 128 keys at d = 256 take all
//    512 columns in fp32, so the dK/dV kernel splits the output columns into
//    two halves of 128 (two work units per key tile, each recomputing S^T and
//    dP^T; d = 192 keeps all 192 columns of both in one unit).  The products
//    that contract over the queries run 64 queries at a time, so S^T and dP^T
//    take 64 columns each.  The dQ kernel holds dQ (d columns) and two step
//    buffers of 64 key columns.
//  * Shared memory (227 KB).  A 128 x 256 tile is 64 KB.  The dK/dV kernel
//    keeps V (and at d = 192 also K) of its key tile resident and streams Q_i
//    and dO_i (64 rows each) through a ring of five slots; at d = 256 K is
//    copied into tensor memory once per unit (it is the A operand of S^T) after
//    arriving through the same ring.  The dQ kernel streams K_j and V_j (64
//    keys each) through a ring of five slots; Q is copied into tensor memory
//    (the A operand of S), and at d = 192 dO too, at d = 256 dO stays in
//    shared memory.  Every ring is filled in the order it is consumed.
//
// Roles (352 threads, one CTA per SM, persistent), as in bwd.cu:
//   warps 0-3 / 4-7  compute warpgroups: thread = TMEM lane = row (a key in
//                    the dK/dV kernel, a query in the dQ kernel); warpgroup w
//                    handles columns [32w, 32w+32) of each 64-column step
//   warp 8           TMA producer
//   warp 9           tcgen05 issuer + tensor-memory owner
//   warp 10          relay: waits on the pipeline's mbarriers and meets the
//                    issuer at a named barrier before each MMA group
#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

#include "bwd.cuh"
#include "sm103_ptx.cuh"
#include "smem_attr.cuh"
#include "unit_ring.cuh"
#include "tiles.cuh"

namespace attn {

namespace {

constexpr int kThreads = 352;
constexpr int kWarpProducer = 8;
constexpr int kWarpMma = 9;
constexpr int kWarpRelay = 10;
constexpr uint32_t kBarRelay = 3;  // named barrier: relay warp + issuer warp (64 threads)
constexpr float kLog2e = 1.4426950408889634f;
constexpr uint32_t kStatusLayout = 5;  // shared memory not 1024-byte aligned
constexpr int kRing = 5;               // ring slots of both kernels
constexpr int kBox128 = 128 * 64 * 2;  // TMA box: 128 rows x 64 16-bit values
constexpr int kBox64 = 64 * 64 * 2;    // TMA box: 64 rows x 64 16-bit values

// K-major operand of 64 rows in boxes of 64 columns: byte offset of the
// reduction step k16 (16 values along the columns).
__device__ __forceinline__ uint32_t kmajor_rows64_off(int k16) {
  return (uint32_t)(k16 >> 2) * kBox64 + (uint32_t)(k16 & 3) * 32u;
}
// MN-major operand of 64 rows (the reduction runs down the rows) whose N
// columns span boxes of 64 columns, kBox64 bytes apart.
__device__ __forceinline__ uint64_t mnmajor_rows64_base(uint32_t addr) {
  return sdesc_sw128(addr, kBox64, 1024);
}
// Tensor-memory column of the reduction step k16 of a 16-bit operand that
// warpgroup w wrote into the first 16 columns of its 32-column quarter.
__device__ __forceinline__ uint32_t wg_packed_col(int k16) {
  return 32u * (uint32_t)(k16 >> 1) + 8u * (uint32_t)(k16 & 1);
}
__device__ __forceinline__ uint32_t pack16x2(bool bf16, float lo, float hi) {
  return bf16 ? pack_bf16x2(lo, hi) : pack_f16x2(lo, hi);
}
// Copies a 128-row tile with D columns (boxes of 64, `box` bytes apart, two
// per ring slot when slot != 0) into tensor memory at column tcol, 8 columns
// per 16 values.
template <int D>
__device__ __forceinline__ void copy_rows128_to_tmem(uint32_t tcol, uint32_t box0_addr,
                                                     uint32_t box1_addr) {
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const int box = kk >> 2;  // 0 .. D/64-1; boxes 0,1 at box0_addr, 2,3 at box1_addr
    const uint32_t base = box < 2 ? box0_addr : box1_addr;
    tmem_cp_128x256b(tcol + 8 * kk,
                     desc_plus(kmajor_base(base), (uint32_t)(box & 1) * kBox128 + (kk & 3) * 32u));
  }
}

// =============================================================== dK, dV ===

template <int D>
struct WDkvLayout {
  static constexpr bool kKt = D == 256;        // K held in tensor memory
  static constexpr int kNC = kKt ? 128 : 192;  // output columns of dK / dV per unit
  static constexpr int kHalves = D / kNC;
  static constexpr int kTile = 128 * D * 2;    // K or V tile
  static constexpr int kItem = 64 * D * 2;     // ring slot: Q_i or dO_i (64 rows), a K half
  static constexpr int kV = 0;
  static constexpr int kK = kTile;             // resident K (not kKt)
  static constexpr int kRing0 = kKt ? kTile : 2 * kTile;
  static constexpr int kVec0 = kRing0 + kRing * kItem;  // per slot: -LSE log2e [64], -D [64]
  static constexpr int kBar = kVec0 + kRing * 512;
  enum {
    kKvFull, kKvEmpty, kFull, kEmpty = kFull + kRing, kSFull = kEmpty + kRing, kDpFull,
    kPReady, kDsReady, kDkvFull, kDkvFree, kDrain, kUnitFull,
    kUnitEmpty = kUnitFull + kUnitSlots, kNumBars = kUnitEmpty + kUnitSlots
  };
  static constexpr int kMisc = kBar + kNumBars * 8;  // TMEM address, abort flag, unit ring
  static constexpr int kBytes = kMisc + 16 + 4 * kUnitSlots;
  static_assert(kItem == 2 * kBox128 || !kKt, "a K half must fill one ring slot");
  static_assert(kBytes <= 232448, "shared memory budget (227 KB) exceeded");
  // tensor memory
  static constexpr uint32_t kColDV = 0, kColDK = kNC, kColS = 2 * kNC, kColDP = 2 * kNC + 64,
                            kColK = 2 * kNC + 128;
  static_assert(!kKt || kColK + D / 2 <= 512, "tensor memory budget exceeded");
  static_assert(kKt || kColDP + 64 <= 512, "tensor memory budget exceeded");
};

struct WDkvUnit {
  int zkv, zq0;  // tensor-map index of the K/V head and of its group's first query head
  int j, h;      // key tile, output column half
  int i0;        // first 64-row query sub-tile a query head sees
  int per_head;  // steps per query head
  int nsteps;    // group * per_head
};

template <int D, bool CAUSAL>
__device__ __forceinline__ WDkvUnit decode_wdkv(int u, const BwdParams& p) {
  using L = WDkvLayout<D>;
  WDkvUnit w;
  int bhkv;
  if (CAUSAL) {
    // Key tile j sees query sub-tiles 2j..: ascending j is longest first,
    // within blocks of head_block heads (both column halves of a key tile
    // are neighbours).
    const BlockedUnit bu = blocked_unit(u, p.BHkv, p.head_block, p.n_kblocks, L::kHalves);
    w.j = bu.cls;
    bhkv = bu.head;
    w.h = bu.inner;
  } else {
    const int per_kv = p.n_kblocks * L::kHalves;
    bhkv = u / per_kv;
    const int r = u - bhkv * per_kv;
    w.j = r / L::kHalves;
    w.h = r - w.j * L::kHalves;
  }
  const int b = bhkv / p.heads_kv;
  const int hkv = bhkv - b * p.heads_kv;
  w.zkv = bhkv;
  w.zq0 = b * p.heads + hkv * p.group;
  const int nq64 = (p.N + 63) >> 6;
  w.i0 = CAUSAL ? 2 * w.j : 0;
  w.per_head = nq64 - w.i0;
  w.nsteps = p.group * w.per_head;
  return w;
}

__device__ __forceinline__ void wdkv_step(const WDkvUnit& w, int s, int* zq, int* i) {
  const int g = s / w.per_head;
  *zq = w.zq0 + g;
  *i = w.i0 + (s - g * w.per_head);
}

template <int D, bool CAUSAL, bool BF16>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_dkv_wide_kernel(const __grid_constant__ CUtensorMap tmQ64,
                        const __grid_constant__ CUtensorMap tmK,
                        const __grid_constant__ CUtensorMap tmV,
                        const __grid_constant__ CUtensorMap tmDO64, const BwdParams p) {
  using L = WDkvLayout<D>;
  constexpr int NC = L::kNC;
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sbase = smem_u32(smem);
  if (sbase & 1023u) {  // the swizzled tiles need 1024-byte alignment
    if (threadIdx.x == 0 && p.status != nullptr)
      atomicCAS(p.status, 0u, kStatusLayout | ((blockIdx.x & 0xFFFFu) << 16));
    return;
  }
  const uint32_t bar0 = sbase + L::kBar;
  auto bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };
  auto slot_addr = [&](uint32_t it) { return sbase + L::kRing0 + (it % kRing) * L::kItem; };
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
    for (int s = 0; s < kRing; ++s) {
      mbar_init(bar(L::kFull + s), 1);
      mbar_init(bar(L::kEmpty + s), 1);
    }
    mbar_init(bar(L::kSFull), 1);
    mbar_init(bar(L::kDpFull), 1);
    mbar_init(bar(L::kPReady), 256);
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
  const int num_units = p.BHkv * p.n_kblocks * L::kHalves;

  if (warp == kWarpProducer) {
    // -------------------------------------------------------------- producer ---
    // Per unit: V (and K at d = 192) into their resident tiles; the two K
    // halves (d = 256) and then Q_i, dO_i of every step through the ring.
    if (lane == 0) {
      tma_prefetch_desc(&tmQ64);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      tma_prefetch_desc(&tmDO64);
    }
    uint32_t kv_it = 0, it = 0;
    bool ok = true;
    // wait for ring slot `it` to be free (lane 0), broadcast the outcome
    auto ring_slot_free = [&]() {
      if (lane == 0) ok = mbar_wait(bar(L::kEmpty + it % kRing), ((it / kRing) & 1) ^ 1, wd, 22);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      return ok;
    };
    uint32_t un = 0;
    while (ok) {
      int u = -1;
      if (lane == 0)
        u = publish_unit(unit_ring, bar(L::kUnitFull), bar(L::kUnitEmpty), un, p.sched, num_units,
                         wd, ok, 38);
      ++un;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      u = __shfl_sync(0xffffffffu, u, 0);
      if (!ok || u < 0) break;
      const WDkvUnit w = decode_wdkv<D, CAUSAL>(u, p);
      if (lane == 0) {
        ok = mbar_wait(bar(L::kKvEmpty), (kv_it & 1) ^ 1, wd, 21);
        if (ok) {
          mbar_arrive_expect_tx(bar(L::kKvFull), L::kKt ? L::kTile : 2 * L::kTile);
#pragma unroll
          for (int c = 0; c < D / 64; ++c) {
            tma_load_3d(sbase + L::kV + c * kBox128, &tmV, bar(L::kKvFull), 64 * c, w.j * 128,
                        w.zkv);
            if constexpr (!L::kKt)
              tma_load_3d(sbase + L::kK + c * kBox128, &tmK, bar(L::kKvFull), 64 * c,
                          w.j * 128, w.zkv);
          }
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      ++kv_it;
      if constexpr (L::kKt) {
        for (int half = 0; half < 2; ++half) {
          if (!ring_slot_free()) break;
          if (lane == 0) {
            const uint32_t s = it % kRing;
            mbar_arrive_expect_tx(bar(L::kFull + s), L::kItem);
            for (int b = 0; b < 2; ++b)
              tma_load_3d(slot_addr(it) + b * kBox128, &tmK, bar(L::kFull + s),
                          64 * (2 * half + b), w.j * 128, w.zkv);
          }
          ++it;
        }
        if (!ok) break;
      }
      for (int s = 0; s < w.nsteps && ok; ++s) {
        int zq, i;
        wdkv_step(w, s, &zq, &i);
        // Q_i
        if (!ring_slot_free()) break;
        if (lane == 0) {
          const uint32_t sl = it % kRing;
          mbar_arrive_expect_tx(bar(L::kFull + sl), L::kItem);
#pragma unroll
          for (int c = 0; c < D / 64; ++c)
            tma_load_3d(slot_addr(it) + c * kBox64, &tmQ64, bar(L::kFull + sl), 64 * c, i * 64,
                        zq);
        }
        ++it;
        // dO_i with the -LSE log2 e and -D vectors of its 64 queries
        // (padding queries: -inf and 0, so their P and dS vanish)
        if (!ring_slot_free()) break;
        {
          const uint32_t sl = it % kRing;
          float2 l2, dd;
          {
            const int q0 = i * 64 + 2 * lane;
            const bool in0 = q0 < p.N, in1 = q0 + 1 < p.N;
            const size_t g0 = (size_t)zq * p.N + (in0 ? q0 : 0);
            const size_t g1 = (size_t)zq * p.N + (in1 ? q0 + 1 : 0);
            l2 = make_float2(in0 ? -p.lse[g0] * kLog2e : -INFINITY,
                             in1 ? -p.lse[g1] * kLog2e : -INFINITY);
            dd = make_float2(in0 ? -p.delta[g0] : 0.f, in1 ? -p.delta[g1] : 0.f);
          }
          float2* vec = reinterpret_cast<float2*>(smem + L::kVec0 + sl * 512);
          vec[lane] = l2;
          vec[32 + lane] = dd;
          __syncwarp();
          if (lane == 0) {
            mbar_arrive_expect_tx(bar(L::kFull + sl), L::kItem);
#pragma unroll
            for (int c = 0; c < D / 64; ++c)
              tma_load_3d(slot_addr(it) + c * kBox64, &tmDO64, bar(L::kFull + sl), 64 * c,
                          i * 64, zq);
          }
          ++it;
        }
      }
    }
    if (lane == 0) {
      // Drain: the copies of the last ring round and of the last K/V tile
      // must have landed before the CTA may exit.
      Watchdog dw = wd;
      volatile int never = 0;
      dw.abort_flag = &never;
      dw.limit_ns = drain_limit_ns(wd.limit_ns);
      if (kv_it > 0) mbar_wait(bar(L::kKvFull), (kv_it - 1) & 1, dw, 24);
      for (uint32_t x = it > (uint32_t)kRing ? it - kRing : 0u; x < it; ++x)
        mbar_wait(bar(L::kFull + x % kRing), (x / kRing) & 1, dw, 24);
    }
    __syncwarp();
  } else if (warp == kWarpMma) {
    // ------------------------------------------------------------ tcgen05 issuer ---
    // Per step s: S^T(s) | dK(s-1) | dP^T(s) | dV(s); after the unit's last
    // step its dK.  At s = 0 (d = 256) K is first copied into tensor memory.
    constexpr uint32_t kIdS = idesc_f16(128, 64, BF16, false, false);   // S^T, dP^T
    constexpr uint32_t kIdKV = idesc_f16(128, NC, BF16, false, true);   // dV, dK
    uint32_t it = 0;
    bool aborted = false;
    const uint64_t vd = kmajor_base(sbase + L::kV);
    const uint64_t kd = kmajor_base(sbase + L::kK);
    // dK(half) += dS^T Q_i[:, half] for the step whose Q_i / dO_i sit at ring
    // positions qpos / dpos; then both slots are free (the -D vector of the
    // dO slot was last read by that step's dS^T phase).
    auto issue_dk = [&](uint32_t qpos, uint32_t dpos, int h, uint32_t acc0) {
      const uint64_t qmn = mnmajor_rows64_base(slot_addr(qpos) + h * (NC / 64) * kBox64);
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
        mma_f16_ts(tbase + L::kColDK, tbase + L::kColDP + wg_packed_col(kk),
                   desc_plus(qmn, mnmajor16_off(kk)), kIdKV, kk > 0 ? 1u : acc0);
      mma_commit(bar(L::kEmpty + qpos % kRing));
      mma_commit(bar(L::kEmpty + dpos % kRing));
    };
    for (uint32_t un = 0;; ++un) {
      // the relay has seen the next unit published (after an abort both
      // warps leave here, having met at every rendezvous so far)
      aborted = named_bar_or(kBarRelay, 64, aborted);
      if (aborted) break;
      const int u = read_unit(unit_ring, bar(L::kUnitEmpty), un);
      if (u < 0) break;
      const WDkvUnit w = decode_wdkv<D, CAUSAL>(u, p);
      const uint32_t kpos = it;
      if constexpr (L::kKt) it += 2;
      uint32_t prev_q = 0, prev_do = 0;
      for (int s = 0; s < w.nsteps; ++s) {
        const uint32_t qpos = it, dpos = it + 1;
        it += 2;
        // Q_i (and at s = 0 the unit's K / V) have landed.
        aborted = named_bar_or(kBarRelay, 64, aborted);
        if (!aborted && lane == 0) {
          tc_fence_after();
          if constexpr (L::kKt) {
            if (s == 0) {
              // K into tensor memory; the previous unit's S^T products, its
              // only readers, were issued before.
              copy_rows128_to_tmem<D>(tbase + L::kColK, slot_addr(kpos), slot_addr(kpos + 1));
              mma_commit(bar(L::kEmpty + kpos % kRing));
              mma_commit(bar(L::kEmpty + (kpos + 1) % kRing));
            }
          }
          const uint64_t qd = kmajor_base(slot_addr(qpos));
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            if constexpr (L::kKt)
              mma_f16_ts(tbase + L::kColS, tbase + L::kColK + 8 * kk,
                         desc_plus(qd, kmajor_rows64_off(kk)), kIdS, kk > 0);
            else
              mma_f16_ss(tbase + L::kColS, desc_plus(kd, kmajor16_off(kk)),
                         desc_plus(qd, kmajor_rows64_off(kk)), kIdS, kk > 0);
          }
          mma_commit(bar(L::kSFull));
        }
        if (s > 0) {
          // dK(s-1): its dS^T is in tensor memory
          aborted = named_bar_or(kBarRelay, 64, aborted);
          if (!aborted && lane == 0) {
            tc_fence_after();
            issue_dk(prev_q, prev_do, w.h, s > 1 ? 1u : 0u);
          }
        }
        // dP^T = V dO_i^T once dO_i has landed (dS^T(s-1) in these columns
        // has just been consumed by dK(s-1))
        aborted = named_bar_or(kBarRelay, 64, aborted);
        if (!aborted && lane == 0) {
          tc_fence_after();
          const uint64_t dod = kmajor_base(slot_addr(dpos));
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            mma_f16_ss(tbase + L::kColDP, desc_plus(vd, kmajor16_off(kk)),
                       desc_plus(dod, kmajor_rows64_off(kk)), kIdS, kk > 0);
          mma_commit(bar(L::kDpFull));
          if (s == w.nsteps - 1) mma_commit(bar(L::kKvEmpty));  // last reader of K and V
        }
        // dV(half) += P^T dO_i[:, half] once P^T is there (and, at s = 0, the
        // previous unit's dV / dK have been stored)
        aborted = named_bar_or(kBarRelay, 64, aborted);
        if (!aborted && lane == 0) {
          tc_fence_after();
          const uint64_t domn = mnmajor_rows64_base(slot_addr(dpos) + w.h * (NC / 64) * kBox64);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_f16_ts(tbase + L::kColDV, tbase + L::kColS + wg_packed_col(kk),
                       desc_plus(domn, mnmajor16_off(kk)), kIdKV, (kk > 0 || s > 0) ? 1u : 0u);
        }
        prev_q = qpos;
        prev_do = dpos;
      }
      // the unit's last dK, then hand dK / dV to the warpgroups
      aborted = named_bar_or(kBarRelay, 64, aborted);
      if (!aborted && lane == 0) {
        tc_fence_after();
        issue_dk(prev_q, prev_do, w.h, w.nsteps > 1 ? 1u : 0u);
        mma_commit(bar(L::kDkvFull));
      }
      __syncwarp();
    }
    if (lane == 0) {
      mma_commit(bar(L::kDrain));
      Watchdog dw = wd;
      volatile int never = 0;
      dw.abort_flag = &never;
      dw.limit_ns = drain_limit_ns(wd.limit_ns);
      mbar_wait(bar(L::kDrain), 0, dw, 32);
    }
    __syncwarp();
  } else if (warp == kWarpRelay) {
    // ------------------------------------------------------------------ relay ---
    uint32_t kv_it = 0, it = 0, st_it = 0, unit_it = 0;
    bool aborted = false;
    auto wait_all = [&](uint32_t b, uint32_t par, int site) {
      if (!aborted) aborted = !__all_sync(0xffffffffu, mbar_wait(b, par, wd, site));
    };
    auto wait_slot = [&](uint32_t pos, int site) {
      wait_all(bar(L::kFull + pos % kRing), (pos / kRing) & 1, site);
    };
    for (uint32_t un = 0;; ++un) {
      wait_all(bar(L::kUnitFull + un % kUnitSlots), (un / kUnitSlots) & 1, 39);
      aborted = named_bar_or(kBarRelay, 64, aborted);
      if (aborted) break;
      const int u = read_unit(unit_ring, bar(L::kUnitEmpty), un);
      if (u < 0) break;
      const WDkvUnit w = decode_wdkv<D, CAUSAL>(u, p);
      wait_all(bar(L::kKvFull), kv_it & 1, 25);
      ++kv_it;
      if constexpr (L::kKt) {
        wait_slot(it, 26);
        wait_slot(it + 1, 26);
        it += 2;
      }
      for (int s = 0; s < w.nsteps; ++s) {
        const uint32_t qpos = it, dpos = it + 1;
        it += 2;
        const uint32_t par = st_it & 1;
        wait_slot(qpos, 26);
        aborted = named_bar_or(kBarRelay, 64, aborted);
        if (s > 0) {
          wait_all(bar(L::kDsReady), par ^ 1, 27);
          aborted = named_bar_or(kBarRelay, 64, aborted);
        }
        wait_slot(dpos, 28);
        aborted = named_bar_or(kBarRelay, 64, aborted);
        if (s == 0 && unit_it > 0) wait_all(bar(L::kDkvFree), (unit_it - 1) & 1, 29);
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
    const int wg = warp >> 2;                // query columns [32 wg, 32 wg + 32) of a step
    const int r = threadIdx.x & 127;         // TMEM lane: key row
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t s_addr = tbase + lane_base + L::kColS + 32 * wg;
    const uint32_t dp_addr = tbase + lane_base + L::kColDP + 32 * wg;
    const float2 sl2x2 = make_float2(p.scale_log2, p.scale_log2);
    uint32_t it = 0, st_it = 0, unit_it = 0, un = 0;
    bool ok = true;
    while (ok) {
      const int u = take_unit(unit_ring, bar(L::kUnitFull), bar(L::kUnitEmpty), un++, wd, ok, 40);
      ok = named_bar_and(1 + wg, 128, ok);
      if (!ok || u < 0) break;
      const WDkvUnit w = decode_wdkv<D, CAUSAL>(u, p);
      if constexpr (L::kKt) it += 2;
      const int key = w.j * 128 + r;
      for (int s = 0; s < w.nsteps; ++s) {
        int zq, i;
        wdkv_step(w, s, &zq, &i);
        (void)zq;
        const uint32_t dpos = it + 1;
        it += 2;
        const uint32_t par = st_it & 1;
        ok = mbar_wait(bar(L::kSFull), par, wd, 33);
        // the -LSE / -D vectors travel with dO_i
        ok = ok && mbar_wait(bar(L::kFull + dpos % kRing), (dpos / kRing) & 1, wd, 34);
        ok = named_bar_and(1 + wg, 128, ok);
        if (!ok) break;
        tc_fence_after();
        const float4* nl4 =
            reinterpret_cast<const float4*>(smem + L::kVec0 + (dpos % kRing) * 512) + 8 * wg;
        const float4* nd4 = nl4 + 16;
        // ---- P^T = exp2(S^T c - LSE log2 e), kept in fp32 for dS^T
        float pr[32];
        {
          uint32_t sa[32];
          tmem_ld32(s_addr, sa);
          tmem_wait_ld();
          reg_fence32(sa);
#pragma unroll
          for (int v = 0; v < 8; ++v) {
            const float4 nl = nl4[v];
            const float2 x01 = __ffma2_rn(
                make_float2(__uint_as_float(sa[4 * v]), __uint_as_float(sa[4 * v + 1])), sl2x2,
                make_float2(nl.x, nl.y));
            const float2 x23 = __ffma2_rn(
                make_float2(__uint_as_float(sa[4 * v + 2]), __uint_as_float(sa[4 * v + 3])),
                sl2x2, make_float2(nl.z, nl.w));
            pr[4 * v] = ex2_approx(x01.x);
            pr[4 * v + 1] = ex2_approx(x01.y);
            pr[4 * v + 2] = ex2_approx(x23.x);
            pr[4 * v + 3] = ex2_approx(x23.y);
          }
          if (CAUSAL && i * 64 < w.j * 128 + 128) {
            const int q0 = i * 64 + 32 * wg;
#pragma unroll
            for (int c = 0; c < 32; ++c)
              if (q0 + c < key) pr[c] = 0.f;  // query before key
          }
          uint32_t pp[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) pp[e] = pack16x2(BF16, pr[2 * e], pr[2 * e + 1]);
          tmem_st16(s_addr, pp);
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(bar(L::kPReady));
        // ---- dS^T = P^T o (dP^T - D)
        ok = mbar_wait(bar(L::kDpFull), par, wd, 35);
        ok = named_bar_and(1 + wg, 128, ok);
        if (!ok) break;
        tc_fence_after();
        {
          uint32_t da[32];
          tmem_ld32(dp_addr, da);
          tmem_wait_ld();
          reg_fence32(da);
          uint32_t pd[16];
#pragma unroll
          for (int v = 0; v < 8; ++v) {
            const float4 nd = nd4[v];
            const float2 g01 = __fadd2_rn(
                make_float2(__uint_as_float(da[4 * v]), __uint_as_float(da[4 * v + 1])),
                make_float2(nd.x, nd.y));
            const float2 g23 = __fadd2_rn(
                make_float2(__uint_as_float(da[4 * v + 2]), __uint_as_float(da[4 * v + 3])),
                make_float2(nd.z, nd.w));
            const float2 s01 = __fmul2_rn(make_float2(pr[4 * v], pr[4 * v + 1]), g01);
            const float2 s23 = __fmul2_rn(make_float2(pr[4 * v + 2], pr[4 * v + 3]), g23);
            pd[2 * v] = pack16x2(BF16, s01.x, s01.y);
            pd[2 * v + 1] = pack16x2(BF16, s23.x, s23.y);
          }
          tmem_st16(dp_addr, pd);
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(bar(L::kDsReady));
        ++st_it;
      }
      if (!ok) break;
      // ---------------------------------------------------- dK / dV epilogue ---
      ok = mbar_wait(bar(L::kDkvFull), unit_it & 1, wd, 36);
      ok = named_bar_and(1 + wg, 128, ok);
      if (!ok) break;
      ++unit_it;
      tc_fence_after();
      const uint32_t src = tbase + lane_base + (wg == 0 ? L::kColDV : L::kColDK);
      const float mult = (wg == 0) ? 1.f : p.scale;
      uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(wg == 0 ? p.dv : p.dk) +
                                            ((size_t)w.zkv * p.N + key) * D + w.h * NC);
#pragma unroll 1
      for (int c = 0; c < NC / 32; ++c) {
        uint32_t raw[32];
        tmem_ld32_sync(src + 32 * c, raw);
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e)
          pk[e] = pack16x2(BF16, __uint_as_float(raw[2 * e]) * mult,
                           __uint_as_float(raw[2 * e + 1]) * mult);
        if (key < p.N) {
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

// ==================================================================== dQ ===

template <int D>
struct WDqLayout {
  static constexpr bool kQRing = D == 256;  // Q arrives through the ring (else a staging tile)
  static constexpr bool kDoT = D == 192;    // dO in tensor memory (else resident in shared)
  static constexpr int kTile = 128 * D * 2;
  static constexpr int kItem = 64 * D * 2;  // ring slot: K_j or V_j (64 keys), a Q half
  static constexpr int kQ = 0;              // Q staging (d = 192)
  static constexpr int kDO = kQRing ? 0 : kTile;  // dO staging (d = 192) or resident (d = 256)
  static constexpr int kRing0 = kQRing ? kTile : 2 * kTile;
  static constexpr int kBar = kRing0 + kRing * kItem;
  enum {
    kQFull, kQEmpty, kDoFull, kDoEmpty, kFull, kEmpty = kFull + kRing, kSFull = kEmpty + kRing,
    kSRead = kSFull + 2, kDpFull, kDsReady, kDqFull, kDqFree, kDrain, kUnitFull,
    kUnitEmpty = kUnitFull + kUnitSlots, kNumBars = kUnitEmpty + kUnitSlots
  };
  static constexpr int kMisc = kBar + kNumBars * 8;  // TMEM address, abort flag, unit ring
  static constexpr int kBytes = kMisc + 16 + 4 * kUnitSlots;
  static_assert(kItem == 2 * kBox128 || !kQRing, "a Q half must fill one ring slot");
  static_assert(kBytes <= 232448, "shared memory budget (227 KB) exceeded");
  // tensor memory: dQ, two 64-column step buffers, Q (and dO) as 16-bit pairs
  static constexpr uint32_t kColDQ = 0, kColB0 = D, kColQ = D + 128, kColDO = D + 128 + D / 2;
  static_assert(kColQ + D / 2 <= 512 && (!kDoT || kColDO + D / 2 <= 512),
                "tensor memory budget exceeded");
};

struct WDqUnit {
  int bh, i, nsteps;
  int zq, zkv;
};

template <bool CAUSAL>
__device__ __forceinline__ WDqUnit decode_wdq(int u, const BwdParams& p) {
  WDqUnit w;
  if (CAUSAL) {
    // Query tile i sees key sub-tiles 0..2i+1: descending i is longest first,
    // within blocks of head_block_q heads.
    const BlockedUnit bu = blocked_unit(u, p.BH, p.head_block_q, p.n_qtiles, 1);
    w.bh = bu.head;
    w.i = p.n_qtiles - 1 - bu.cls;
  } else {
    w.bh = u / p.n_qtiles;
    w.i = u - w.bh * p.n_qtiles;
  }
  const int b = w.bh / p.heads;
  w.zq = w.bh;
  w.zkv = b * p.heads_kv + (w.bh - b * p.heads) / p.group;
  const int nk64 = (p.N + 63) >> 6;
  w.nsteps = CAUSAL ? min(2 * w.i + 2, nk64) : nk64;
  return w;
}

template <int D, bool CAUSAL, bool BF16>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_dq_wide_kernel(const __grid_constant__ CUtensorMap tmQ,
                       const __grid_constant__ CUtensorMap tmK64,
                       const __grid_constant__ CUtensorMap tmV64,
                       const __grid_constant__ CUtensorMap tmDO, const BwdParams p) {
  using L = WDqLayout<D>;
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sbase = smem_u32(smem);
  if (sbase & 1023u) {
    if (threadIdx.x == 0 && p.status != nullptr)
      atomicCAS(p.status, 0u, kStatusLayout | ((blockIdx.x & 0xFFFFu) << 16));
    return;
  }
  const uint32_t bar0 = sbase + L::kBar;
  auto bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };
  auto slot_addr = [&](uint32_t it) { return sbase + L::kRing0 + (it % kRing) * L::kItem; };
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
    mbar_init(bar(L::kDoFull), 1);
    mbar_init(bar(L::kDoEmpty), 1);
    for (int s = 0; s < kRing; ++s) {
      mbar_init(bar(L::kFull + s), 1);
      mbar_init(bar(L::kEmpty + s), 1);
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
      tma_prefetch_desc(&tmK64);
      tma_prefetch_desc(&tmV64);
      tma_prefetch_desc(&tmDO);
      uint32_t it = 0, unit_it = 0;
      bool ok = true;
      auto ring_slot_free = [&]() {
        ok = mbar_wait(bar(L::kEmpty + it % kRing), ((it / kRing) & 1) ^ 1, wd, 42);
        return ok;
      };
      uint32_t un = 0;
      while (ok) {
        const int u = publish_unit(unit_ring, bar(L::kUnitFull), bar(L::kUnitEmpty), un++,
                                   p.sched + 1, num_units, wd, ok, 38);
        if (u < 0) break;
        const WDqUnit w = decode_wdq<CAUSAL>(u, p);
        if constexpr (L::kQRing) {
          for (int half = 0; half < 2 && ok; ++half) {
            if (!ring_slot_free()) break;
            const uint32_t s = it % kRing;
            mbar_arrive_expect_tx(bar(L::kFull + s), L::kItem);
            for (int b = 0; b < 2; ++b)
              tma_load_3d(slot_addr(it) + b * kBox128, &tmQ, bar(L::kFull + s),
                          64 * (2 * half + b), w.i * 128, w.zq);
            ++it;
          }
          if (!ok) break;
          ok = mbar_wait(bar(L::kDoEmpty), (unit_it & 1) ^ 1, wd, 41);
          if (!ok) break;
          mbar_arrive_expect_tx(bar(L::kDoFull), L::kTile);
#pragma unroll
          for (int c = 0; c < D / 64; ++c)
            tma_load_3d(sbase + L::kDO + c * kBox128, &tmDO, bar(L::kDoFull), 64 * c, w.i * 128,
                        w.zq);
        } else {
          ok = mbar_wait(bar(L::kQEmpty), (unit_it & 1) ^ 1, wd, 41);
          if (!ok) break;
          mbar_arrive_expect_tx(bar(L::kQFull), 2 * L::kTile);
#pragma unroll
          for (int c = 0; c < D / 64; ++c) {
            tma_load_3d(sbase + L::kQ + c * kBox128, &tmQ, bar(L::kQFull), 64 * c, w.i * 128,
                        w.zq);
            tma_load_3d(sbase + L::kDO + c * kBox128, &tmDO, bar(L::kQFull), 64 * c, w.i * 128,
                        w.zq);
          }
        }
        ++unit_it;
        for (int j = 0; j < w.nsteps && ok; ++j) {
#pragma unroll
          for (int which = 0; which < 2; ++which) {  // K_j, then V_j
            if (!ring_slot_free()) break;
            const uint32_t s = it % kRing;
            mbar_arrive_expect_tx(bar(L::kFull + s), L::kItem);
#pragma unroll
            for (int c = 0; c < D / 64; ++c)
              tma_load_3d(slot_addr(it) + c * kBox64, which ? &tmV64 : &tmK64, bar(L::kFull + s),
                          64 * c, j * 64, w.zkv);
            ++it;
          }
        }
      }
      // Drain: the copies of the last ring round, Q and dO must have landed.
      Watchdog dw = wd;
      volatile int never = 0;
      dw.abort_flag = &never;
      dw.limit_ns = drain_limit_ns(wd.limit_ns);
      if (unit_it > 0)
        mbar_wait(bar(L::kQRing ? L::kDoFull : L::kQFull), (unit_it - 1) & 1, dw, 44);
      for (uint32_t x = it > (uint32_t)kRing ? it - kRing : 0u; x < it; ++x)
        mbar_wait(bar(L::kFull + x % kRing), (x / kRing) & 1, dw, 44);
    }
    __syncwarp();
  } else if (warp == kWarpMma) {
    // ------------------------------------------------------------ tcgen05 issuer ---
    // Per unit: Q (and at d = 192 dO) copied into tensor memory.  Per step j
    // (buffer b = j%2): S_j into b | dQ += dS_{j-1} K_{j-1} | dP_j into b once
    // the warpgroups have read S_j.
    constexpr uint32_t kIdS = idesc_f16(128, 64, BF16, false, false);  // S, dP
    constexpr uint32_t kIdQ = idesc_f16(128, D, BF16, false, true);    // dQ
    uint32_t it = 0, step_it = 0;
    bool aborted = false;
    const uint64_t qd = kmajor_base(sbase + L::kQ), dod = kmajor_base(sbase + L::kDO);
    auto issue_dq = [&](uint32_t kpos, uint32_t sb, uint32_t acc0) {
      const uint64_t kmn = mnmajor_rows64_base(slot_addr(kpos));
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
        mma_f16_ts(tbase + L::kColDQ, tbase + L::kColB0 + 64 * sb + wg_packed_col(kk),
                   desc_plus(kmn, mnmajor16_off(kk)), kIdQ, kk > 0 ? 1u : acc0);
      mma_commit(bar(L::kEmpty + kpos % kRing));
    };
    for (uint32_t un = 0;; ++un) {
      // the relay has seen the next unit published (after an abort both
      // warps leave here, having met at every rendezvous so far)
      aborted = named_bar_or(kBarRelay, 64, aborted);
      if (aborted) break;
      const int u = read_unit(unit_ring, bar(L::kUnitEmpty), un);
      if (u < 0) break;
      const WDqUnit w = decode_wdq<CAUSAL>(u, p);
      const uint32_t qpos = it;
      if constexpr (L::kQRing) it += 2;
      uint32_t prev_k = 0, prev_sb = 0;
      for (int j = 0; j < w.nsteps; ++j) {
        const uint32_t kpos = it, vpos = it + 1;
        it += 2;
        const uint32_t sb = step_it & 1;
        const uint32_t buf = tbase + L::kColB0 + 64 * sb;
        // K_j (and at j = 0 Q, dO) have landed
        aborted = named_bar_or(kBarRelay, 64, aborted);
        if (!aborted && lane == 0) {
          tc_fence_after();
          if (j == 0) {
            // Q (and dO) into tensor memory: the previous unit's S and dP,
            // their last readers, were issued before.
            if constexpr (L::kQRing) {
              copy_rows128_to_tmem<D>(tbase + L::kColQ, slot_addr(qpos), slot_addr(qpos + 1));
              mma_commit(bar(L::kEmpty + qpos % kRing));
              mma_commit(bar(L::kEmpty + (qpos + 1) % kRing));
            } else {
#pragma unroll
              for (int kk = 0; kk < D / 16; ++kk) {
                tmem_cp_128x256b(tbase + L::kColQ + 8 * kk, desc_plus(qd, kmajor16_off(kk)));
                tmem_cp_128x256b(tbase + L::kColDO + 8 * kk, desc_plus(dod, kmajor16_off(kk)));
              }
              mma_commit(bar(L::kQEmpty));  // the staging tiles may be reloaded
            }
          }
          // S_j = Q K_j^T into buffer sb (its previous contents, dS_{j-2},
          // were read by dQ_{j-2}, issued before)
          const uint64_t kdk = kmajor_base(slot_addr(kpos));
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            mma_f16_ts(buf, tbase + L::kColQ + 8 * kk, desc_plus(kdk, kmajor_rows64_off(kk)),
                       kIdS, kk > 0);
          mma_commit(bar(L::kSFull + sb));
        }
        if (j > 0) {
          // dS_{j-1} is ready (and, for the unit's first dQ, dQ is free)
          aborted = named_bar_or(kBarRelay, 64, aborted);
          if (!aborted && lane == 0) {
            tc_fence_after();
            issue_dq(prev_k, prev_sb, j > 1 ? 1u : 0u);
          }
        }
        // V_j has landed and S_j has been read: dP_j = dO V_j^T into sb
        aborted = named_bar_or(kBarRelay, 64, aborted);
        if (!aborted && lane == 0) {
          tc_fence_after();
          const uint64_t vdk = kmajor_base(slot_addr(vpos));
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            if constexpr (L::kDoT)
              mma_f16_ts(buf, tbase + L::kColDO + 8 * kk, desc_plus(vdk, kmajor_rows64_off(kk)),
                         kIdS, kk > 0);
            else
              mma_f16_ss(buf, desc_plus(dod, kmajor16_off(kk)),
                         desc_plus(vdk, kmajor_rows64_off(kk)), kIdS, kk > 0);
          }
          mma_commit(bar(L::kDpFull));
          mma_commit(bar(L::kEmpty + vpos % kRing));
          if constexpr (!L::kDoT) {
            if (j == w.nsteps - 1) mma_commit(bar(L::kDoEmpty));  // last reader of dO
          }
        }
        prev_k = kpos;
        prev_sb = sb;
        ++step_it;
      }
      // dQ += dS_last K_last, then hand dQ to the warpgroups
      aborted = named_bar_or(kBarRelay, 64, aborted);
      if (!aborted && lane == 0) {
        tc_fence_after();
        issue_dq(prev_k, prev_sb, w.nsteps > 1 ? 1u : 0u);
        mma_commit(bar(L::kDqFull));
      }
      __syncwarp();
    }
    if (lane == 0) {
      mma_commit(bar(L::kDrain));
      Watchdog dw = wd;
      volatile int never = 0;
      dw.abort_flag = &never;
      dw.limit_ns = drain_limit_ns(wd.limit_ns);
      mbar_wait(bar(L::kDrain), 0, dw, 51);
    }
    __syncwarp();
  } else if (warp == kWarpRelay) {
    // ------------------------------------------------------------------ relay ---
    uint32_t it = 0, step_it = 0, unit_it = 0;
    bool aborted = false;
    auto wait_all = [&](uint32_t b, uint32_t par, int site) {
      if (!aborted) aborted = !__all_sync(0xffffffffu, mbar_wait(b, par, wd, site));
    };
    auto wait_slot = [&](uint32_t pos, int site) {
      wait_all(bar(L::kFull + pos % kRing), (pos / kRing) & 1, site);
    };
    for (uint32_t un = 0;; ++un) {
      wait_all(bar(L::kUnitFull + un % kUnitSlots), (un / kUnitSlots) & 1, 39);
      aborted = named_bar_or(kBarRelay, 64, aborted);
      if (aborted) break;
      const int u = read_unit(unit_ring, bar(L::kUnitEmpty), un);
      if (u < 0) break;
      const WDqUnit w = decode_wdq<CAUSAL>(u, p);
      const uint32_t qpos = it;
      if constexpr (L::kQRing) it += 2;
      for (int j = 0; j < w.nsteps; ++j) {
        const uint32_t kpos = it, vpos = it + 1;
        it += 2;
        if (j == 0) {
          if constexpr (L::kQRing) {
            wait_slot(qpos, 45);
            wait_slot(qpos + 1, 45);
            wait_all(bar(L::kDoFull), unit_it & 1, 45);
          } else {
            wait_all(bar(L::kQFull), unit_it & 1, 45);
          }
        }
        wait_slot(kpos, 46);
        aborted = named_bar_or(kBarRelay, 64, aborted);
        if (j > 0) {
          wait_all(bar(L::kDsReady), (step_it - 1) & 1, 47);
          if (j == 1 && unit_it > 0) wait_all(bar(L::kDqFree), (unit_it - 1) & 1, 48);
          aborted = named_bar_or(kBarRelay, 64, aborted);
        }
        wait_slot(vpos, 55);
        wait_all(bar(L::kSRead), step_it & 1, 56);
        aborted = named_bar_or(kBarRelay, 64, aborted);
        ++step_it;
      }
      wait_all(bar(L::kDsReady), (step_it - 1) & 1, 49);
      if (w.nsteps == 1 && unit_it > 0) wait_all(bar(L::kDqFree), (unit_it - 1) & 1, 50);
      aborted = named_bar_or(kBarRelay, 64, aborted);
      ++unit_it;
    }
  } else {
    // ------------------------------------------------------ compute warpgroups ---
    const int wg = warp >> 2;                // key columns [32 wg, 32 wg + 32) of a step
    const int r = threadIdx.x & 127;         // TMEM lane: query row
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t dq_addr = tbase + lane_base + L::kColDQ;
    const float sl2 = p.scale_log2;
    uint32_t unit_it = 0, step_it = 0, un = 0;
    bool ok = true;
    while (ok) {
      const int u = take_unit(unit_ring, bar(L::kUnitFull), bar(L::kUnitEmpty), un++, wd, ok, 40);
      ok = named_bar_and(1 + wg, 128, ok);
      if (!ok || u < 0) break;
      const WDqUnit w = decode_wdq<CAUSAL>(u, p);
      const int row = w.i * 128 + r;
      const bool in = row < p.N;
      const size_t grow = (size_t)w.zq * p.N + (in ? row : 0);
      // Padding rows: LSE = +inf, D = 0, so their P and dS vanish.
      const float nl2 = in ? -p.lse[grow] * kLog2e : -INFINITY;
      const float nd = in ? -p.delta[grow] : 0.f;
      const float2 sl2x2 = make_float2(sl2, sl2), nl2x2 = make_float2(nl2, nl2),
                   nd2x2 = make_float2(nd, nd);
      for (int j = 0; j < w.nsteps; ++j) {
        const uint32_t sb = step_it & 1;
        ok = mbar_wait(bar(L::kSFull + sb), (step_it >> 1) & 1, wd, 52);
        ok = named_bar_and(1 + wg, 128, ok);
        if (!ok) break;
        tc_fence_after();
        const uint32_t s_addr = tbase + lane_base + L::kColB0 + 64 * sb + 32 * wg;
        // ---- P = exp2(S c - LSE log2 e); then the buffer may take dP_j
        float pr[32];
        {
          uint32_t sa[32];
          tmem_ld32(s_addr, sa);
          tmem_wait_ld();
          reg_fence32(sa);
          tc_fence_before();
          mbar_arrive(bar(L::kSRead));
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const float2 x = __ffma2_rn(
                make_float2(__uint_as_float(sa[2 * e]), __uint_as_float(sa[2 * e + 1])), sl2x2,
                nl2x2);
            pr[2 * e] = ex2_approx(x.x);
            pr[2 * e + 1] = ex2_approx(x.y);
          }
          const int k0 = j * 64 + 32 * wg;  // first key of this warpgroup's columns
          if (CAUSAL && k0 + 31 > w.i * 128) {
#pragma unroll
            for (int c = 0; c < 32; ++c)
              if (k0 + c > row) pr[c] = 0.f;  // key after query
          }
          // keys past the end of the sequence (zero-filled by TMA)
          const int kend = p.N - k0;
          if (kend < 32) {
#pragma unroll
            for (int c = 0; c < 32; ++c)
              if (c >= kend) pr[c] = 0.f;
          }
        }
        // ---- dS = P o (dP - D)
        ok = mbar_wait(bar(L::kDpFull), step_it & 1, wd, 53);
        ok = named_bar_and(1 + wg, 128, ok);
        if (!ok) break;
        tc_fence_after();
        {
          uint32_t da[32];
          tmem_ld32(s_addr, da);
          tmem_wait_ld();
          reg_fence32(da);
          uint32_t pd[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const float2 g = __fadd2_rn(
                make_float2(__uint_as_float(da[2 * e]), __uint_as_float(da[2 * e + 1])), nd2x2);
            const float2 sv = __fmul2_rn(make_float2(pr[2 * e], pr[2 * e + 1]), g);
            pd[e] = pack16x2(BF16, sv.x, sv.y);
          }
          tmem_st16(s_addr, pd);
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(bar(L::kDsReady));
        ++step_it;
      }
      if (!ok) break;
      // ------------------------------------------------------------ dQ epilogue ---
      ok = mbar_wait(bar(L::kDqFull), unit_it & 1, wd, 54);
      ok = named_bar_and(1 + wg, 128, ok);
      if (!ok) break;
      ++unit_it;
      tc_fence_after();
      uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.dq) + grow * D);
      // 32-column chunks alternate between the two warpgroups.
#pragma unroll 1
      for (int c = wg; c < D / 32; c += 2) {
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

template <int D, bool CAUSAL, bool BF16>
cudaError_t launch_wide_main(const BwdWideLaunch& a) {
  static DeviceFlags dkv_configured, dq_configured;  // per device and instantiation
  const BwdParams& p = a.params;
  auto dkv = bwd_dkv_wide_kernel<D, CAUSAL, BF16>;
  cudaError_t e = ensure_dyn_smem(dkv, WDkvLayout<D>::kBytes, dkv_configured);
  if (e != cudaSuccess) return e;
  const int dkv_units = p.BHkv * p.n_kblocks * WDkvLayout<D>::kHalves;
  dkv<<<dkv_units < a.num_sms ? dkv_units : a.num_sms, kThreads, WDkvLayout<D>::kBytes,
        a.stream>>>(a.tmQ64, a.tmK, a.tmV, a.tmDO64, p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  auto dq = bwd_dq_wide_kernel<D, CAUSAL, BF16>;
  e = ensure_dyn_smem(dq, WDqLayout<D>::kBytes, dq_configured);
  if (e != cudaSuccess) return e;
  const int dq_units = p.BH * p.n_qtiles;
  dq<<<dq_units < a.num_sms ? dq_units : a.num_sms, kThreads, WDqLayout<D>::kBytes, a.stream>>>(
      a.tmQ, a.tmK64, a.tmV64, a.tmDO, p);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_wide_d(const BwdWideLaunch& a) {
  if (a.causal)
    return a.bf16 ? launch_wide_main<D, true, true>(a) : launch_wide_main<D, true, false>(a);
  return a.bf16 ? launch_wide_main<D, false, true>(a) : launch_wide_main<D, false, false>(a);
}

}  // namespace

cudaError_t launch_bwd_wide(const BwdWideLaunch& a) {
  cudaError_t e = launch_bwd_pre(a.params, a.d, a.bf16, a.num_sms, a.stream);
  if (e != cudaSuccess) return e;
  return a.d == 256 ? launch_wide_d<256>(a) : launch_wide_d<192>(a);
}

}  // namespace attn
