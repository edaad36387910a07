// Backward pass of exact attention on sm_103a (head dim 128).
//
// "FlashAttention-2: Faster Attention with Better Parallelism and Work
// Partitioning" (review page), "Methods" and "핵심 구성요소": the forward pass
// keeps only the log-sum-exp, and the backward pass recomputes P from it
// instead of storing the N x N matrix.  The backward kernel of "Triton 07:
// Flash Attention v3" is a three-stage one; here the three stages are
//   1. bwd_pre_kernel   D_i = sum_c dO_ic O_ic (warp-shuffle row reduction),
//                       and the fp32 dQ accumulator is zeroed;
//   2. bwd_main_kernel  one CTA per 128-key K/V tile (persistent, longest
//                       first): for every 128-query tile i it recomputes
//                       S^T = K Q_i^T and P^T = exp2(S^T c - LSE_i log2 e),
//                       dP^T = V dO_i^T, dS^T = P^T o (dP^T - D_i), and
//                       accumulates dV += P^T dO_i, dK += dS^T Q_i in tensor
//                       memory; dQ_i^T = K^T dS^T is drained into the fp32
//                       accumulator with TMA bulk reduce-adds;
//   3. bwd_post_kernel  dQ = scale * dQ_acc, rounded to 16 bit.
//
// Main-kernel CTA organisation (320 threads):
//   warps 0-3 / 4-7  compute warpgroups for query columns [0,64) / [64,128)
//                    of each step; thread = key row of the tile (TMEM lane)
//   warp 8           producer: TMA for K, V (once per unit) and Q_i, dO_i
//                    (2-stage ring); LSE*log2(e) and D for the 128 queries
//   warp 9           tcgen05 issuer + tensor-memory owner
// Tensor memory: dV [0,128)  dK [128,256)  S^T_0 [256,320)  dP^T_0 [320,384)
//                S^T_1 [384,448)  dP^T_1 [448,512); P^T_h and dS^T_h (16-bit)
//                overwrite the first 32 columns of S^T_h / dP^T_h, and
//                dQ^T_h (fp32, 64 columns) reuses the S^T_h columns once the
//                dV MMA has consumed P^T_h.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <cstdint>

#include "bwd.cuh"
#include "sm103_ptx.cuh"
#include "tiles.cuh"

namespace attn {

namespace {

constexpr int kThreads = 320;
constexpr int kWarpProducer = 8;
constexpr int kWarpMma = 9;
constexpr float kLog2e = 1.4426950408889634f;
constexpr uint32_t kStatusLayout = 5;  // shared memory not 1024-byte aligned

struct BwdLayout {
  static constexpr int kTile = 32768;             // 128 x 128 16-bit values
  static constexpr int kK = 0;
  static constexpr int kV = kTile;
  static constexpr int kStage0 = 2 * kTile;       // stage s: Q_i then dO_i
  static constexpr int kStageBytes = 2 * kTile;
  static constexpr int kStages = 2;
  static constexpr int kDS = kStage0 + kStages * kStageBytes;  // dS^T halves, 16 KB each
  static constexpr int kVec = kDS + 2 * 16384;    // per stage: LSE2[128], D[128]
  static constexpr int kBar = kVec + kStages * 1024;
  enum {
    kKvFull, kKvEmpty, kQFull, kQFull1, kQEmpty, kQEmpty1, kSFull, kSFull1, kPFull, kPFull1,
    kDqFull, kDqFull1, kDqFree, kDqFree1, kDkvFull, kDkvFree, kDrain, kNumBars
  };
  static constexpr int kMisc = kBar + kNumBars * 8;
  static constexpr int kBytes = kMisc + 16;
  static_assert(kBytes <= 232448, "shared memory budget (227 KB) exceeded");
};

constexpr uint32_t kColDV = 0, kColDK = 128;
__device__ __forceinline__ uint32_t col_s(int h) { return 256u + 128u * h; }
__device__ __forceinline__ uint32_t col_dp(int h) { return 320u + 128u * h; }

struct BwdUnit {
  int bh, j, i0, nsteps;
};

template <bool CAUSAL>
__device__ __forceinline__ BwdUnit decode_bwd_unit(int u, const BwdParams& p) {
  BwdUnit w;
  if (CAUSAL) {
    // K/V tile j sees query tiles j..n-1: ascending j is longest first.
    w.j = u / p.BH;
    w.bh = u - w.j * p.BH;
    w.i0 = w.j;
  } else {
    w.bh = u / p.n_kblocks;
    w.j = u - w.bh * p.n_kblocks;
    w.i0 = 0;
  }
  w.nsteps = p.n_qtiles - w.i0;
  return w;
}

template <bool CAUSAL, bool BF16>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_main_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
                    const __grid_constant__ CUtensorMap tmDQ, const BwdParams p) {
  using L = BwdLayout;
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
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  Watchdog wd{p.status, abort_flag, p.wait_limit_ns};

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    mbar_init(bar(L::kKvFull), 1);
    mbar_init(bar(L::kKvEmpty), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(L::kQFull + s), 2);    // TMA bytes + the LSE/D writer
      mbar_init(bar(L::kQEmpty + s), 1);
      mbar_init(bar(L::kSFull + s), 1);
      mbar_init(bar(L::kPFull + s), 128);
      mbar_init(bar(L::kDqFull + s), 1);
      mbar_init(bar(L::kDqFree + s), 128);
    }
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
  const int G = gridDim.x;
  const int cta = blockIdx.x;
  const int num_units = p.BH * p.n_kblocks;

  if (warp == kWarpProducer) {
    // -------------------------------------------------------------- producer ---
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      tma_prefetch_desc(&tmDO);
    }
    uint32_t kv_it = 0, st_it = 0;
    bool ok = true;
    for (int k = 0; ok; ++k) {
      const int u = snake_unit(k, cta, G);
      if (u >= num_units) break;
      const BwdUnit w = decode_bwd_unit<CAUSAL>(u, p);
      if (lane == 0) {
        ok = mbar_wait(bar(L::kKvEmpty), (kv_it & 1) ^ 1, wd, 21);
        if (ok) {
          mbar_arrive_expect_tx(bar(L::kKvFull), 2 * L::kTile);
          for (int h = 0; h < 2; ++h) {
            tma_load_3d(sbase + L::kK + h * 16384, &tmK, bar(L::kKvFull), h * 64, w.j * 128, w.bh);
            tma_load_3d(sbase + L::kV + h * 16384, &tmV, bar(L::kKvFull), h * 64, w.j * 128, w.bh);
          }
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      ++kv_it;
      for (int s = 0; s < w.nsteps && ok; ++s) {
        const int i = w.i0 + s;
        const uint32_t stage = st_it & 1;
        if (lane == 0) ok = mbar_wait(bar(L::kQEmpty + stage), ((st_it >> 1) & 1) ^ 1, wd, 22);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        const uint32_t qaddr = sbase + L::kStage0 + stage * L::kStageBytes;
        if (lane == 0) {
          mbar_arrive_expect_tx(bar(L::kQFull + stage), 2 * L::kTile);
          for (int h = 0; h < 2; ++h) {
            tma_load_3d(qaddr + h * 16384, &tmQ, bar(L::kQFull + stage), h * 64, i * 128, w.bh);
            tma_load_3d(qaddr + L::kTile + h * 16384, &tmDO, bar(L::kQFull + stage), h * 64,
                        i * 128, w.bh);
          }
        }
        // LSE * log2(e) and D of the 128 queries (padding rows: +inf / 0, so
        // their P and dS vanish).
        float l2[4], dd[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int q = i * 128 + 4 * lane + e;
          const bool in = q < p.N;
          const size_t g = (size_t)w.bh * p.N + (in ? q : 0);
          l2[e] = in ? p.lse[g] * kLog2e : INFINITY;
          dd[e] = in ? p.delta[g] : 0.f;
        }
        float4* vec = reinterpret_cast<float4*>(smem + L::kVec + stage * 1024);
        vec[lane] = make_float4(l2[0], l2[1], l2[2], l2[3]);
        vec[32 + lane] = make_float4(dd[0], dd[1], dd[2], dd[3]);
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(L::kQFull + stage));
        ++st_it;
      }
    }
    if (lane == 0) {
      Watchdog dw = wd;
      volatile int never = 0;
      dw.abort_flag = &never;
      dw.limit_ns = drain_limit_ns(wd.limit_ns);
      if (kv_it > 0) mbar_wait(bar(L::kKvFull), (kv_it - 1) & 1, dw, 23);
      const uint32_t first = st_it > 2u ? st_it - 2 : 0u;
      for (uint32_t it = first; it < st_it; ++it)
        mbar_wait(bar(L::kQFull + (it & 1)), (it >> 1) & 1, dw, 24);
    }
    __syncwarp();
  } else if (warp == kWarpMma) {
    // ------------------------------------------------------------ tcgen05 issuer ---
    if (lane == 0) {
      constexpr uint32_t kIdS = idesc_f16(128, 64, BF16, false, false);   // S^T, dP^T
      constexpr uint32_t kIdKV = idesc_f16(128, 128, BF16, false, true);  // dV, dK
      constexpr uint32_t kIdQ = idesc_f16(128, 64, BF16, true, true);     // dQ^T
      uint32_t kv_it = 0, st_it = 0, unit_it = 0;
      uint32_t dq_it[2] = {0, 0}, p_it[2] = {0, 0};
      bool ok = true;
      // Base descriptors: K and V as K-major A operands of S^T / dP^T, K as
      // the MN-major A operand of dQ^T, the dS^T halves as MN-major B.
      const uint64_t kd_k = kmajor_base(sbase + L::kK), vd_k = kmajor_base(sbase + L::kV);
      const uint64_t kd_mn = mnmajor_base(sbase + L::kK);
      const uint64_t dsd[2] = {mnmajor_base(sbase + L::kDS), mnmajor_base(sbase + L::kDS + 16384)};
      for (int k = 0; ok; ++k) {
        const int u = snake_unit(k, cta, G);
        if (u >= num_units) break;
        const BwdUnit w = decode_bwd_unit<CAUSAL>(u, p);
        ok = mbar_wait(bar(L::kKvFull), kv_it & 1, wd, 25);
        if (!ok) break;
        ++kv_it;
        tc_fence_after();
        for (int s = 0; s < w.nsteps && ok; ++s) {
          const uint32_t stage = st_it & 1;
          ok = mbar_wait(bar(L::kQFull + stage), (st_it >> 1) & 1, wd, 26);
          if (!ok) break;
          tc_fence_after();
          const uint32_t qaddr = sbase + L::kStage0 + stage * L::kStageBytes;
          const uint32_t doaddr = qaddr + L::kTile;
          for (int h = 0; h < 2 && ok; ++h) {
            if (dq_it[h] > 0) {
              ok = mbar_wait(bar(L::kDqFree + h), (dq_it[h] - 1) & 1, wd, 27);
              if (!ok) break;
              tc_fence_after();
            }
            const uint64_t qd = kmajor_base(qaddr + 8192u * h);
            const uint64_t dod = kmajor_base(doaddr + 8192u * h);
            const uint32_t cs = tbase + col_s(h), cdp = tbase + col_dp(h);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              mma_f16_ss(cs, desc_plus(kd_k, kmajor16_off(kk)), desc_plus(qd, kmajor16_off(kk)),
                         kIdS, kk > 0);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              mma_f16_ss(cdp, desc_plus(vd_k, kmajor16_off(kk)), desc_plus(dod, kmajor16_off(kk)),
                         kIdS, kk > 0);
            mma_commit(bar(L::kSFull + h));
          }
          if (!ok) break;
          if (s == 0 && unit_it > 0) {
            ok = mbar_wait(bar(L::kDkvFree), (unit_it - 1) & 1, wd, 28);
            if (!ok) break;
            tc_fence_after();
          }
          for (int h = 0; h < 2 && ok; ++h) {
            ok = mbar_wait(bar(L::kPFull + h), p_it[h] & 1, wd, 29);
            if (!ok) break;
            ++p_it[h];
            tc_fence_after();
            const uint64_t dod_mn = mnmajor_base(doaddr + 8192u * h);
            const uint64_t qd_mn = mnmajor_base(qaddr + 8192u * h);
            const uint32_t acc0 = (s > 0 || h > 0) ? 1u : 0u;
            const uint32_t cs = tbase + col_s(h), cdp = tbase + col_dp(h);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma_f16_ts(tbase + kColDV, cs + 8 * kk, desc_plus(dod_mn, mnmajor16_off(kk)), kIdKV,
                         kk > 0 ? 1u : acc0);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma_f16_ts(tbase + kColDK, cdp + 8 * kk, desc_plus(qd_mn, mnmajor16_off(kk)), kIdKV,
                         kk > 0 ? 1u : acc0);
            const uint64_t dsb = h ? dsd[1] : dsd[0];
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              mma_f16_ss(cs, desc_plus(kd_mn, mnmajor16_off(kk)), desc_plus(dsb, mnmajor16_off(kk)),
                         kIdQ, kk > 0);
            mma_commit(bar(L::kDqFull + h));
            ++dq_it[h];
          }
          if (!ok) break;
          mma_commit(bar(L::kQEmpty + stage));
          ++st_it;
        }
        if (!ok) break;
        mma_commit(bar(L::kDkvFull));
        mma_commit(bar(L::kKvEmpty));
        ++unit_it;
      }
      mma_commit(bar(L::kDrain));
      Watchdog dw = wd;
      volatile int never = 0;
      dw.abort_flag = &never;
      dw.limit_ns = drain_limit_ns(wd.limit_ns);
      mbar_wait(bar(L::kDrain), 0, dw, 30);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------ compute warpgroups ---
    const int h = warp >> 2;                 // query half of every step
    const int r = threadIdx.x & 127;         // TMEM lane: key row (or d for dQ^T)
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t s_addr = tbase + lane_base + col_s(h);
    const uint32_t dp_addr = tbase + lane_base + col_dp(h);
    uint8_t* ds_row = smem + L::kDS + 16384 * h + r * 128;
    const float sl2 = p.scale_log2;
    uint32_t s_it = 0, st_it = 0, unit_it = 0;
    bool ok = true;
    for (int k = 0; ok; ++k) {
      const int u = snake_unit(k, cta, G);
      if (u >= num_units) break;
      const BwdUnit w = decode_bwd_unit<CAUSAL>(u, p);
      for (int s = 0; s < w.nsteps; ++s) {
        const int i = w.i0 + s;
        const uint32_t stage = st_it & 1;
        ok = mbar_wait(bar(L::kSFull + h), s_it & 1, wd, 31);
        ok = ok && mbar_wait(bar(L::kQFull + stage), (st_it >> 1) & 1, wd, 32);
        // The dS^T buffer doubles as the dQ staging area of the previous
        // step: its TMA reads must be done before dS^T is written again.
        if ((threadIdx.x & 127) == 0) bulk_wait_group_read0();
        // Exit decisions are uniform over the warpgroup: its four warps meet
        // at named barriers further down.
        ok = named_bar_and(1 + h, 128, ok);
        if (!ok) break;
        ++s_it;
        tc_fence_after();
        const float4* lse4 = reinterpret_cast<const float4*>(smem + L::kVec + stage * 1024) + 16 * h;
        const float4* d4 = lse4 + 32;
        const bool diag = CAUSAL && (i == w.j);
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t sr[32], dr[32];
          tmem_ld32(s_addr + 32 * c, sr);
          tmem_ld32(dp_addr + 32 * c, dr);
          tmem_wait_ld();
          reg_fence32(sr);
          reg_fence32(dr);
          uint32_t pp[16], pd[16];
#pragma unroll
          for (int v = 0; v < 8; ++v) {
            const float4 lq = lse4[8 * c + v];
            const float4 dq = d4[8 * c + v];
            const float lv[4] = {lq.x, lq.y, lq.z, lq.w};
            const float dv[4] = {dq.x, dq.y, dq.z, dq.w};
            float pv[4], sv[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int col = 32 * c + 4 * v + e;  // query column within the half
              float pe = ex2_approx(fmaf(__uint_as_float(sr[4 * v + e]), sl2, -lv[e]));
              if (diag && (64 * h + col) < r) pe = 0.f;
              pv[e] = pe;
              sv[e] = pe * (__uint_as_float(dr[4 * v + e]) - dv[e]);
            }
            pp[2 * v] = BF16 ? pack_bf16x2(pv[0], pv[1]) : pack_f16x2(pv[0], pv[1]);
            pp[2 * v + 1] = BF16 ? pack_bf16x2(pv[2], pv[3]) : pack_f16x2(pv[2], pv[3]);
            pd[2 * v] = BF16 ? pack_bf16x2(sv[0], sv[1]) : pack_f16x2(sv[0], sv[1]);
            pd[2 * v + 1] = BF16 ? pack_bf16x2(sv[2], sv[3]) : pack_f16x2(sv[2], sv[3]);
          }
          tmem_st16(s_addr + 16 * c, pp);
          tmem_st16(dp_addr + 16 * c, pd);
          // dS^T row r, query columns [32c, 32c+32) = 16-byte chunks 4c..4c+3,
          // stored with the 128-byte swizzle (chunk index xor row % 8).
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            const int chunk = 4 * c + v;
            *reinterpret_cast<uint4*>(ds_row + ((chunk ^ (r & 7)) << 4)) =
                make_uint4(pd[4 * v], pd[4 * v + 1], pd[4 * v + 2], pd[4 * v + 3]);
          }
        }
        fence_proxy_async_smem();
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(bar(L::kPFull + h));
        // dQ^T_h: TMEM lane = head-dim index r, column = query of this half.
        ok = mbar_wait(bar(L::kDqFull + h), (s_it - 1) & 1, wd, 33);
        ok = named_bar_and(1 + h, 128, ok);
        if (!ok) break;
        tc_fence_after();
        uint32_t qa[32], qb[32];
        tmem_ld32(s_addr, qa);
        tmem_ld32(s_addr + 32, qb);
        tmem_wait_ld();
        reg_fence32(qa);
        reg_fence32(qb);
        // The columns are free again: the next S^T_h may be issued now.
        tc_fence_before();
        mbar_arrive(bar(L::kDqFree + h));
        // Reduce into the fp32 accumulator with TMA bulk reduce-add, staging
        // 32 queries x 128 values (16 KB) at a time in this half's dS^T
        // buffer, which the completed dQ^T MMA no longer reads.  Rows at or
        // beyond N fall outside the tensor map and are dropped by the TMA.
        float* qstage = reinterpret_cast<float*>(smem + L::kDS + 16384 * h);
        const bool leader = (threadIdx.x & 127) == 0;
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          if (c == 1) {
            if (leader) bulk_wait_group_read0();
            named_bar_sync(1 + h, 128);
          }
#pragma unroll
          for (int e = 0; e < 32; ++e) qstage[e * 128 + r] = __uint_as_float(c == 0 ? qa[e] : qb[e]);
          fence_proxy_async_smem();
          named_bar_sync(1 + h, 128);
          if (leader) {
            tma_reduce_add_3d(&tmDQ, smem_u32(qstage), 0, i * 128 + 64 * h + 32 * c, w.bh);
            bulk_commit_group();
          }
        }
        ++st_it;
      }
      if (!ok) break;
      // ---------------------------------------------------- dK / dV epilogue ---
      ok = mbar_wait(bar(L::kDkvFull), unit_it & 1, wd, 34);
      ok = named_bar_and(1 + h, 128, ok);
      if (!ok) break;
      ++unit_it;
      tc_fence_after();
      const int key = w.j * 128 + r;
      const uint32_t src = tbase + lane_base + (h == 0 ? kColDV : kColDK);
      const float mult = (h == 0) ? 1.f : p.scale;
      uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(h == 0 ? p.dv : p.dk) +
                                            ((size_t)w.bh * p.N + key) * 128);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t raw[32];
        tmem_ld32_sync(src + 32 * c, raw);
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const float a = __uint_as_float(raw[2 * e]) * mult;
          const float b = __uint_as_float(raw[2 * e + 1]) * mult;
          pk[e] = BF16 ? pack_bf16x2(a, b) : pack_f16x2(a, b);
        }
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

  if (warp < 8 && (threadIdx.x & 127) == 0) bulk_wait_group0();  // dQ reductions landed
  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
}

// D_i = sum_c dO_ic O_ic with one warp per row (4 values per lane, then a
// butterfly of warp shuffles), and zero the fp32 dQ accumulator row.
template <bool BF16>
__global__ void __launch_bounds__(256) bwd_pre_kernel(const uint16_t* __restrict__ o,
                                                     const uint16_t* __restrict__ dout,
                                                     float* __restrict__ delta,
                                                     float* __restrict__ dq_acc, long rows) {
  const long warp0 = ((long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const long nwarps = ((long)gridDim.x * blockDim.x) >> 5;
  const int lane = threadIdx.x & 31;
  for (long row = warp0; row < rows; row += nwarps) {
    const uint2 a = reinterpret_cast<const uint2*>(o + row * 128)[lane];
    const uint2 b = reinterpret_cast<const uint2*>(dout + row * 128)[lane];
    float acc = 0.f;
    const uint32_t aw[2] = {a.x, a.y}, bw[2] = {b.x, b.y};
#pragma unroll
    for (int e = 0; e < 2; ++e) {
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
    reinterpret_cast<float4*>(dq_acc + row * 128)[lane] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
}

// dQ = scale * dQ_acc, rounded to 16 bit; 8 values per thread and iteration.
template <bool BF16>
__global__ void __launch_bounds__(256) bwd_post_kernel(const float* __restrict__ dq_acc,
                                                      uint16_t* __restrict__ dq, float scale,
                                                      long n8) {
  const long t0 = (long)blockIdx.x * blockDim.x + threadIdx.x;
  const long nt = (long)gridDim.x * blockDim.x;
  for (long t = t0; t < n8; t += nt) {
    const float4 a = reinterpret_cast<const float4*>(dq_acc)[2 * t];
    const float4 b = reinterpret_cast<const float4*>(dq_acc)[2 * t + 1];
    uint4 r;
    if (BF16) {
      r = make_uint4(pack_bf16x2(a.x * scale, a.y * scale), pack_bf16x2(a.z * scale, a.w * scale),
                     pack_bf16x2(b.x * scale, b.y * scale), pack_bf16x2(b.z * scale, b.w * scale));
    } else {
      r = make_uint4(pack_f16x2(a.x * scale, a.y * scale), pack_f16x2(a.z * scale, a.w * scale),
                     pack_f16x2(b.x * scale, b.y * scale), pack_f16x2(b.z * scale, b.w * scale));
    }
    reinterpret_cast<uint4*>(dq)[t] = r;
  }
}

template <bool CAUSAL, bool BF16>
cudaError_t launch_main(const BwdLaunch& a) {
  auto kern = bwd_main_kernel<CAUSAL, BF16>;
  static bool configured = false;
  if (!configured) {
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, BwdLayout::kBytes);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  const int units = a.params.BH * a.params.n_kblocks;
  const int grid = units < a.num_sms ? units : a.num_sms;
  kern<<<grid, kThreads, BwdLayout::kBytes, a.stream>>>(a.tmQ, a.tmK, a.tmV, a.tmDO, a.tmDQacc,
                                                        a.params);
  return cudaGetLastError();
}

template <bool BF16>
cudaError_t launch_all(const BwdLaunch& a) {
  const BwdParams& p = a.params;
  const long rows = (long)p.BH * p.N;
  long blocks = (rows + 7) / 8;
  const long cap = (long)a.num_sms * 16;
  if (blocks > cap) blocks = cap;
  bwd_pre_kernel<BF16><<<(int)blocks, 256, 0, a.stream>>>(
      static_cast<const uint16_t*>(p.o), static_cast<const uint16_t*>(p.dout), p.delta, p.dq_acc,
      rows);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  e = a.causal ? launch_main<true, BF16>(a) : launch_main<false, BF16>(a);
  if (e != cudaSuccess) return e;
  const long n8 = rows * 128 / 8;
  long pblocks = (n8 + 255) / 256;
  if (pblocks > (long)a.num_sms * 8) pblocks = (long)a.num_sms * 8;
  bwd_post_kernel<BF16><<<(int)pblocks, 256, 0, a.stream>>>(p.dq_acc, static_cast<uint16_t*>(p.dq),
                                                           p.scale, n8);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd(const BwdLaunch& a) {
  return a.bf16 ? launch_all<true>(a) : launch_all<false>(a);
}

}  // namespace attn
