// Forward pass of exact attention on sm_103a: TMA-fed, tcgen05 tensor cores
// with S and O accumulated in tensor memory, online softmax in base 2.
//
// Algorithm: "FlashAttention-2: Faster Attention with Better Parallelism and
// Work Partitioning" (review page), flowchart "프레임워크 개요": per query
// tile, loop over K/V tiles computing S = Q K^T and the running row max /
// row sum, accumulate P V unnormalised, rescale by 1/rowsum once at the end,
// write O and the log-sum-exp ("Methods"); blocks entirely above the causal
// diagonal are never visited ("핵심 구성요소").  The exp2 formulation with the
// scale folded into the exponent is the one "Triton 07: Flash Attention v3"
// ("Method") keeps from its FA2 core.
//
// CTA organisation (one CTA per SM, persistent):
//   warps 0-3  softmax warpgroup for query tile 0 of the current work unit
//   warps 4-7  softmax warpgroup for query tile 1
//   warp  8    TMA producer: Q tiles, then a ring of K and V tiles
//   warp  9    tcgen05 issuer (one thread) + tensor-memory owner
// A work unit is (batch*head, pair of adjacent 128-row query tiles).  The two
// tiles share every K/V tile and ping-pong on the tensor core: while one
// warpgroup exponentiates S_t, the tensor core computes the other tile's
// P V and next S ("8.3 FlashAttention-3", section 4, pingpong scheduling,
// recast for an MMA warp that issues for both tiles).
//
// Tensor memory (512 columns x 128 lanes of 32 bit):
//   [  0,128) S_0 (fp32); P_0 overwrites [0,64) (16-bit pairs) or [0,32)
//             (E4M3 quads)
//   [128,256) S_1 / P_1
//   [256,256+D) O_0 (fp32)     [256+D,256+2D) O_1
//
// Precisions: fp16 and bf16 (kind::f16 MMAs; V is the MN-major B operand of
// P V), and E4M3 ("8.3 FlashAttention-3", section 5: kind::f8f6f4 MMAs with
// fp32 accumulation).  In the E4M3 path S_ij = q8_i.k8_j sq(i/64) sk(j/64),
// V arrives transposed (a K-major B operand), and P is stored as E4M3 after
// multiplying it by sv(j/64)/max(sv): the reference max keeps P <= 2^8, so
// the product fits E4M3, and O = max(sv) * sum(P~ V8) / l.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

#include "fp8.cuh"
#include "fwd.cuh"
#include "sm103_ptx.cuh"
#include "smem_attr.cuh"
#include "tiles.cuh"

namespace attn {

namespace {

constexpr int kThreads = 352;
constexpr int kWarpProducer = 8;
constexpr int kWarpMma = 9;
constexpr int kWarpRelay = 10;
// Named barriers (0 is __syncthreads): issuer <-> relay, issuer <-> softmax t.
constexpr uint32_t kBarKv = 1, kBarP = 2;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: P stays <= 2^8
// How work units map to rows (a compile-time choice, so each kernel carries
// only its own unit decoding): dense [B*H, N, D] heads; grouped heads packed
// into one query tile (FwdParams::pack_nq); packed variable-length batches
// (FwdParams::cu_seqlens).
constexpr int kModeDense = 0, kModePacked = 1, kModeVarlen = 2;
constexpr int kPrecF16 = 0, kPrecBF16 = 1, kPrecE4M3 = 2;

template <int D, bool FP8>
struct FwdLayout {
  static constexpr int kTileBytes = 128 * kPaddedD<D> * (FP8 ? 1 : 2);  // 128 rows, padded
  // K/V ring depth (tiles): a fifth 32 KB slot fits beside the two Q tiles
  // and measured 1.3 % faster at d = 96, no different at d = 128
  static constexpr int kSlots = (FP8 || D == 64) ? 8 : (D == 96 ? 5 : 4);
  static constexpr int kQOff = 0;
  static constexpr int kKvOff = 2 * kTileBytes;
  static constexpr int kBarOff = kKvOff + kSlots * kTileBytes;
  // barrier indices
  static constexpr int kQFull = 0, kQEmpty = 2, kSFull = 4, kOFull = 8, kDrain = 10;
  static constexpr int kKvFull = 11, kKvEmpty = 11 + kSlots;
  static constexpr int kNumBars = 11 + 2 * kSlots;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;
  static constexpr int kBytes = kMiscOff + 16;
  static constexpr int kDynSmem = kBytes + 1024;  // + alignment slack
  static_assert(kDynSmem <= 232448, "shared memory budget (227 KB) exceeded");
};

struct Unit {
  int bh, qp;
  int bhkv;   // key/value head (batch * heads_kv + head / group)
  int zq, zkv;  // tensor-map head index of Q / O and of K / V
  int row0;   // first row of the sequence in its head (K / V)
  int qrow;   // tensor-map row of the unit's first query row (Q / O)
  int len;    // query rows of the sequence
  int klen;   // key rows of the sequence
  int koff;   // causal: query row i sees keys j <= i + koff
  int nkb;    // its 128-row tiles (query tiles = key blocks)
  int split;  // key split of this unit (0 without a split)
  int kb0;    // first key block of the split
  int nb[2];  // K/V blocks visited by query tile 0 / 1 (0: tile absent or no key in the split)
};

// Grouped heads packed into one query tile: u = (batch, key/value head, split).
template <bool CAUSAL>
__device__ __forceinline__ Unit decode_packed_unit(int u, const FwdParams& p) {
  Unit w;
  w.split = u % p.n_split;
  u /= p.n_split;
  const int b = u / p.heads_kv;
  const int g = u - b * p.heads_kv;
  w.bh = b * p.heads + g * p.group;
  w.qp = 0;
  w.bhkv = u;
  w.zkv = u;
  w.zq = b;
  w.row0 = 0;
  w.qrow = g * p.group * p.pack_nq;
  w.len = p.group * p.pack_nq;
  w.klen = p.Nk;
  w.koff = p.Nk - p.pack_nq;
  w.nkb = (w.klen + 127) >> 7;
  w.kb0 = (w.split * w.nkb) / p.n_split;
  const int kb1 = ((w.split + 1) * w.nkb) / p.n_split;
  // causal: the last query of a head sees keys up to pack_nq - 1 + koff
  const int visible = CAUSAL ? min((p.pack_nq - 1 + w.koff) / 128 + 1, w.nkb) : w.nkb;
  w.nb[0] = max(0, min(visible, kb1) - w.kb0);
  w.nb[1] = 0;
  return w;
}

template <bool CAUSAL, int MODE>
__device__ __forceinline__ Unit decode_unit(int u, const FwdParams& p) {
  if constexpr (MODE == kModePacked) return decode_packed_unit<CAUSAL>(u, p);
  constexpr bool VARLEN = MODE == kModeVarlen;
  Unit w;
  w.split = u % p.n_split;  // splits of one query-tile pair are neighbours
  u /= p.n_split;
  if (CAUSAL || VARLEN) {
    // Longest first: the heaviest query-tile pairs of every head come first.
    const int r = u / p.BH;
    w.bh = u - r * p.BH;
    w.qp = p.n_pairs - 1 - r;
  } else {
    w.bh = u / p.n_pairs;
    w.qp = u - w.bh * p.n_pairs;
  }
  const int b = w.bh / p.heads;
  const int hq = w.bh - b * p.heads;
  if constexpr (VARLEN) {
    // rows clamped into [0, N] so that no access leaves the tensors
    const int s0 = min(max(__ldg(p.cu_seqlens + b), 0), p.N);
    const int s1 = min(max(__ldg(p.cu_seqlens + b + 1), s0), p.N);
    w.row0 = s0;
    w.qrow = s0;
    w.len = min(s1 - s0, p.max_seqlen);
    w.klen = w.len;
    w.koff = 0;
    w.zq = hq;
    w.zkv = hq / p.group;
    w.bhkv = w.zkv;
  } else {
    w.row0 = 0;
    w.qrow = 0;
    w.len = p.N;
    w.klen = p.Nk;
    w.koff = p.Nk - p.N;
    w.zq = w.bh;
    w.bhkv = b * p.heads_kv + hq / p.group;
    w.zkv = w.bhkv;
  }
  w.nkb = (w.klen + 127) >> 7;
  w.kb0 = (w.split * w.nkb) / p.n_split;
  const int kb1 = ((w.split + 1) * w.nkb) / p.n_split;
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    const int tile = 2 * w.qp + t;
    if (tile * 128 >= w.len) {
      w.nb[t] = 0;
    } else {
      // causal: the tile's last row sees keys up to tile * 128 + 127 + koff
      const int visible = CAUSAL ? min((tile * 128 + 127 + w.koff) / 128 + 1, w.nkb) : w.nkb;
      w.nb[t] = max(0, min(visible, kb1) - w.kb0);
    }
  }
  return w;
}

template <int D, bool CAUSAL, int PREC, int MODE>
__global__ void __launch_bounds__(kThreads, 1)
    fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
               const __grid_constant__ CUtensorMap tmV, const FwdParams p) {
  constexpr bool FP8 = PREC == kPrecE4M3;
  constexpr bool BF16 = PREC == kPrecBF16;
  using L = FwdLayout<D, FP8>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + L::kBarOff;
  auto bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + L::kMiscOff);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kMiscOff + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  Watchdog wd{p.status, abort_flag, p.wait_limit_ns};

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    for (int t = 0; t < 2; ++t) {
      mbar_init(bar(L::kQFull + t), 1);
      mbar_init(bar(L::kQEmpty + t), 1);
      mbar_init(bar(L::kSFull + t), 1);
      mbar_init(bar(L::kOFull + t), 1);
    }
    mbar_init(bar(L::kDrain), 1);
    for (int s = 0; s < L::kSlots; ++s) {
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
      uint32_t kv_it = 0, q_it[2] = {0, 0};
      bool ok = true;
      for (int k = 0; ok; ++k) {
        const int u = snake_unit(k, cta, G);
        if (u >= p.num_units) break;
        const Unit w = decode_unit<CAUSAL, MODE>(u, p);
        if (max(w.nb[0], w.nb[1]) == 0) continue;  // no key of the split is visible
        for (int t = 0; t < 2 && ok; ++t) {
          if (w.nb[t] == 0) continue;
          ok = mbar_wait(bar(L::kQEmpty + t), (q_it[t] & 1) ^ 1, wd, 1);
          if (!ok) break;
          mbar_arrive_expect_tx(bar(L::kQFull + t), L::kTileBytes);
          const uint32_t dst = sbase + L::kQOff + t * L::kTileBytes;
          if constexpr (FP8) {
            tma_load_3d(dst, &tmQ, bar(L::kQFull + t), 0, w.row0 + (2 * w.qp + t) * 128, w.zq);
          } else {
#pragma unroll
            for (int h = 0; h < kPaddedD<D> / 64; ++h)
              tma_load_3d(dst + h * 16384, &tmQ, bar(L::kQFull + t), h * 64,
                          (MODE == kModePacked ? w.qrow : w.row0) + (2 * w.qp + t) * 128, w.zq);
          }
          ++q_it[t];
        }
        const int nbmax = max(w.nb[0], w.nb[1]);
        for (int j = 0; j < nbmax && ok; ++j) {
#pragma unroll
          for (int which = 0; which < 2; ++which) {
            const uint32_t slot = kv_it % L::kSlots;
            ok = mbar_wait(bar(L::kKvEmpty + slot), ((kv_it / L::kSlots) & 1) ^ 1, wd, 2);
            if (!ok) break;
            mbar_arrive_expect_tx(bar(L::kKvFull + slot), L::kTileBytes);
            const uint32_t dst = sbase + L::kKvOff + slot * L::kTileBytes;
            if constexpr (FP8) {
              // K: [128 keys][128 d] bytes; V^T: [128 d][128 keys] bytes.
              if (which == 0)
                tma_load_3d(dst, &tmK, bar(L::kKvFull + slot), 0, (w.kb0 + j) * 128, w.zkv);
              else
                tma_load_3d(dst, &tmV, bar(L::kKvFull + slot), (w.kb0 + j) * 128, 0, w.zkv);
            } else {
#pragma unroll
              for (int h = 0; h < kPaddedD<D> / 64; ++h)
                tma_load_3d(dst + h * 16384, which ? &tmV : &tmK, bar(L::kKvFull + slot),
                            h * 64, w.row0 + (w.kb0 + j) * 128, w.zkv);
            }
            ++kv_it;
          }
        }
      }
      // Drain: every copy this warp issued must have landed before the CTA
      // may exit (only matters after an abort; otherwise all were consumed).
      Watchdog dw = wd;
      volatile int never = 0;
      dw.abort_flag = &never;
      dw.limit_ns = drain_limit_ns(wd.limit_ns);
      const uint32_t first = kv_it > (uint32_t)L::kSlots ? kv_it - L::kSlots : 0u;
      for (uint32_t it = first; it < kv_it; ++it)
        mbar_wait(bar(L::kKvFull + it % L::kSlots), (it / L::kSlots) & 1, dw, 3);
      for (int t = 0; t < 2; ++t)
        if (q_it[t] > 0) mbar_wait(bar(L::kQFull + t), (q_it[t] - 1) & 1, dw, 4);
    }
    __syncwarp();
  } else if (warp == kWarpRelay) {
    // ---------------------------------------------------------- TMA relay ---
    // Waits for the TMA completions the issuer needs and meets the issuer at
    // named barrier kBarKv, so that the issuer itself never touches an
    // mbarrier between its commits (a shared-memory wait there stalls the
    // tensor pipe).  Schedule, per unit: [Q tiles + K_0], then per block j:
    // [V_j + K_{j+1}].  After an abort the schedule is still walked to the end
    // (waits skipped) so every rendezvous pairs up exactly as in a clean run.
    uint32_t kv_it = 0, q_it[2] = {0, 0};
    bool aborted = false;
    auto kv_ready = [&]() {
      const uint32_t slot = kv_it % L::kSlots;
      const uint32_t par = (kv_it / L::kSlots) & 1;
      ++kv_it;
      if (aborted) return;
      const bool ok = __all_sync(0xffffffffu, mbar_wait(bar(L::kKvFull + slot), par, wd, 7));
      aborted = !ok;
    };
    for (int k = 0;; ++k) {
      const int u = snake_unit(k, cta, G);
      if (u >= p.num_units) break;
      const Unit w = decode_unit<CAUSAL, MODE>(u, p);
      const int nbmax = max(w.nb[0], w.nb[1]);
      if (nbmax == 0) continue;  // the same skip in every role
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        if (w.nb[t] == 0) continue;
        const uint32_t par = q_it[t] & 1;
        ++q_it[t];
        if (aborted) continue;
        aborted = !__all_sync(0xffffffffu, mbar_wait(bar(L::kQFull + t), par, wd, 5));
      }
      kv_ready();
      aborted = named_bar_or(kBarKv, 64, aborted);
      for (int j = 0; j < nbmax; ++j) {
        kv_ready();
        if (j + 1 < nbmax) kv_ready();
        aborted = named_bar_or(kBarKv, 64, aborted);
      }
    }
  } else if (warp == kWarpMma) {
    // ---------------------------------------------------- tcgen05 issuer ---
    // The whole warp walks the schedule (named barriers count warps); lane 0
    // issues.  Readiness arrives only through named barriers: kBarKv from the
    // relay, kBarP + t from softmax warpgroup t.  The OR carried by those
    // barriers tells the issuer to stop issuing after an abort.
    constexpr uint32_t kIdS =
        FP8 ? idesc_e4m3(128, 128, false, false) : idesc_f16(128, 128, BF16, false, false);
    constexpr uint32_t kIdO =
        FP8 ? idesc_e4m3(128, D, false, false)
            : idesc_f16(128, D, BF16, false, true);
    uint32_t kv_it = 0;
    bool aborted = false;
    bool issued = false;
    // Base descriptors of the two Q tiles (K-major); K-steps add constants.
    const uint64_t qdesc0 = kmajor_base(sbase + L::kQOff);
    const uint64_t qdesc1 = kmajor_base(sbase + L::kQOff + L::kTileBytes);
    // S_t = Q_t K^T into tensor-memory columns [128t, 128t+128).
    auto issue_s = [&](int t, uint32_t kaddr) {
      const uint64_t kd = kmajor_base(kaddr);
      const uint64_t qd = t ? qdesc1 : qdesc0;
      const uint32_t dcol = tbase + 128 * t;
      if constexpr (FP8) {
#pragma unroll
        for (int kk = 0; kk < D / 32; ++kk)
          mma_f8_ss(dcol, desc_plus(qd, 32 * kk), desc_plus(kd, 32 * kk), kIdS, kk > 0);
      } else {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          mma_f16_ss(dcol, desc_plus(qd, kmajor16_off(kk)), desc_plus(kd, kmajor16_off(kk)),
                     kIdS, kk > 0);
      }
    };
    // O_t += P_t V_j  (A = P from tensor memory)
    auto issue_pv = [&](int t, uint32_t vaddr, uint32_t acc0) {
      const uint32_t ocol = tbase + 256 + kPaddedD<D> * t;
      const uint32_t pcol = tbase + 128 * t;
      if constexpr (FP8) {
        const uint64_t vd = kmajor_base(vaddr);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)  // 32 keys per MMA
          mma_f8_ts(ocol, pcol + kk * 8, desc_plus(vd, 32 * kk), kIdO, kk > 0 ? 1u : acc0);
      } else {
        const uint64_t vd = mnmajor_base(vaddr);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)  // 16 keys per MMA
          mma_f16_ts(ocol, pcol + kk * 8, desc_plus(vd, mnmajor16_off(kk)), kIdO,
                     kk > 0 ? 1u : acc0);
      }
    };
    for (int k = 0;; ++k) {
      const int u = snake_unit(k, cta, G);
      if (u >= p.num_units) break;
      const Unit w = decode_unit<CAUSAL, MODE>(u, p);
      const int nb0 = w.nb[0], nb1 = w.nb[1];
      const int nbmax = max(nb0, nb1);
      if (nbmax == 0) continue;  // the same skip in every role
      // Q tiles and K_0 are in shared memory: S_t(0) = Q_t K_0^T.
      aborted = named_bar_or(kBarKv, 64, aborted);
      uint32_t kslot = kv_it % L::kSlots;
      ++kv_it;
      if (!aborted) {
        tc_fence_after();
        if (lane == 0) {
          const uint32_t kaddr = sbase + L::kKvOff + kslot * L::kTileBytes;
          if (nb0 > 0) {
            issue_s(0, kaddr);
            mma_commit(bar(L::kSFull + 0));
            if (nb0 == 1) mma_commit(bar(L::kQEmpty + 0));
          }
          if (nb1 > 0) {
            issue_s(1, kaddr);
            mma_commit(bar(L::kSFull + 1));
            if (nb1 == 1) mma_commit(bar(L::kQEmpty + 1));
          }
          mma_commit(bar(L::kKvEmpty + kslot));
        }
        issued = true;
        __syncwarp();
      }
      for (int j = 0; j < nbmax; ++j) {
        // V_j and (if any) K_{j+1} are in shared memory.
        aborted = named_bar_or(kBarKv, 64, aborted);
        const uint32_t vslot = kv_it % L::kSlots;
        ++kv_it;
        const bool have_next = j + 1 < nbmax;
        if (have_next) {
          kslot = kv_it % L::kSlots;
          ++kv_it;
        }
        const uint32_t vaddr = sbase + L::kKvOff + vslot * L::kTileBytes;
        const uint32_t kaddr = sbase + L::kKvOff + kslot * L::kTileBytes;
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          const int nbt = t ? nb1 : nb0;
          if (j >= nbt) continue;
          // P_t(j) is in tensor memory.
          aborted = named_bar_or(kBarP + t, 160, aborted);
          if (aborted) continue;
          tc_fence_after();
          if (lane == 0) {
            issue_pv(t, vaddr, j > 0 ? 1u : 0u);
            if (j == nbt - 1) mma_commit(bar(L::kOFull + t));
            if (j + 1 < nbt) {
              issue_s(t, kaddr);
              mma_commit(bar(L::kSFull + t));
              if (j + 1 == nbt - 1) mma_commit(bar(L::kQEmpty + t));
            }
          }
          __syncwarp();
        }
        if (!aborted) {
          if (lane == 0) {
            mma_commit(bar(L::kKvEmpty + vslot));
            if (have_next) mma_commit(bar(L::kKvEmpty + kslot));
          }
          __syncwarp();
        }
      }
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
    // --------------------------------------------------- softmax warpgroups ---
    const int t = warp >> 2;                 // query tile of the pair
    const int r = threadIdx.x & 127;         // row within the tile = TMEM lane
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t s_addr = tbase + lane_base + 128u * t;
    const uint32_t o_addr = tbase + lane_base + 256u + kPaddedD<D> * t;
    const float sl2 = p.scale_log2;
    uint32_t s_it = 0, o_it = 0;
    // After an abort the schedule is still walked to the end with every wait
    // and all tensor-memory work skipped, so the issuer's named barriers
    // always pair up.
    bool aborted = false;
    for (int k = 0;; ++k) {
      const int u = snake_unit(k, cta, G);
      if (u >= p.num_units) break;
      const Unit w = decode_unit<CAUSAL, MODE>(u, p);
      const int nb = w.nb[t];
      const int tile = 2 * w.qp + t;
      const int row = tile * 128 + r;
      // this split's partial O and LSE
      uint16_t* const obase = static_cast<uint16_t*>(p.o) + w.split * p.o_split;
      float* const lbase = p.lse + w.split * p.lse_split;
      if (nb == 0) {
        // A query tile that sees no key of this split: O = 0, LSE = -inf.
        if (row < w.len) {
          const size_t grow = MODE == kModePacked ? (size_t)w.zq * p.q_zrows + w.qrow + row
                                : (size_t)w.zq * p.N + w.row0 + row;
          uint4* orow = reinterpret_cast<uint4*>(obase + grow * D);
#pragma unroll
          for (int c = 0; c < D / 8; ++c) orow[c] = make_uint4(0u, 0u, 0u, 0u);
          lbase[grow] = -INFINITY;
        }
        continue;
      }
      float m = -INFINITY;  // running max of the log2-scaled scores (reference value)
      float l = 0.f;        // running sum of exp2(x - m)
      // E4M3 path: this row's Q block scale and the head's largest V scale
      // (warp-shuffle max over the V block scales).
      float fq = 0.f, sv_max = 1.f;
      const float* ksc = nullptr;
      const float* vsc = nullptr;
      if constexpr (FP8) {
        const size_t sb = (size_t)w.bh * p.n_sblocks;
        ksc = p.k_scale + (size_t)w.bhkv * p.n_sblocks;
        vsc = p.v_scale + (size_t)w.bhkv * p.n_sblocks;
        fq = p.q_scale[sb + min(row, p.N - 1) / 64] * sl2;
        float mv = 0.f;
        for (int b = lane; b < p.n_sblocks; b += 32) mv = fmaxf(mv, vsc[b]);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1)
          mv = fmaxf(mv, __shfl_xor_sync(0xffffffffu, mv, off));
        sv_max = mv > 0.f ? mv : 1.f;
      }
      for (int j = 0; j < nb; ++j) {
        const uint32_t spar = s_it & 1;
        ++s_it;
        // E4M3: keys [0,64) and [64,128) of the block have their own K and V
        // scales; they are read before the wait for S, off its critical path.
        float g0 = 1.f, g1 = 1.f, f0 = 1.f, f1 = 1.f;
        if constexpr (FP8) {
          const int b0 = 2 * (w.kb0 + j), b1 = min(b0 + 1, p.n_sblocks - 1);
          f0 = fq * __ldg(ksc + b0);
          f1 = fq * __ldg(ksc + b1);
          g0 = __ldg(vsc + b0) / sv_max;
          g1 = __ldg(vsc + b1) / sv_max;
        }
        if (!aborted)
          aborted = !__all_sync(0xffffffffu, mbar_wait(bar(L::kSFull + t), spar, wd, 11));
        if (!aborted) {
        tc_fence_after();
        uint32_t sr[4][32];
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld32(s_addr + c * 32, sr[c]);
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < 4; ++c) reg_fence32(sr[c]);
        float s[128];
        // E4M3: the raw scores are scaled inside the exponent argument (f0 /
        // f1 include the Q scale and scale * log2 e) and the row max is taken
        // per half on the raw scores (scaling by f > 0 keeps the order).
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int i = 0; i < 32; ++i) s[c * 32 + i] = __uint_as_float(sr[c][i]);
        const int jk = w.kb0 + j;  // key block index
        // blocks that reach past the tile's first row's last visible key
        const bool diag = CAUSAL && (jk * 128 + 127 > tile * 128 + w.koff);
        const bool tail = (jk == w.nkb - 1) && (w.klen & 127);
        if (diag || tail) {
          const int kbase = jk * 128;
          // query index within its head (packed heads: pack_nq rows each)
          const int qi = MODE == kModePacked ? r % p.pack_nq : row;
          const int lim = CAUSAL ? min(qi + w.koff, w.klen - 1) : (w.klen - 1);
#pragma unroll
          for (int c = 0; c < 128; ++c) s[c] = (kbase + c > lim) ? -INFINITY : s[c];
        }
        float m_blk;
        if constexpr (FP8) {
          float h0 = fmax3(s[0], s[1], s[2]), h1 = fmax3(s[64], s[65], s[66]);
          float h2 = fmax3(s[3], s[4], s[5]), h3 = fmax3(s[67], s[68], s[69]);
#pragma unroll
          for (int c = 6; c < 62; c += 4) {
            h0 = fmax3(h0, s[c], s[c + 1]);
            h2 = fmax3(h2, s[c + 2], s[c + 3]);
            h1 = fmax3(h1, s[64 + c], s[64 + c + 1]);
            h3 = fmax3(h3, s[64 + c + 2], s[64 + c + 3]);
          }
          h0 = fmax3(h0, h2, fmaxf(s[62], s[63]));
          h1 = fmax3(h1, h3, fmaxf(s[126], s[127]));
          m_blk = fmaxf(h0 * f0, h1 * f1);
        } else {
          m_blk = row_max128(s) * sl2;
        }
        // Raise the reference max where the block's exceeds it by more than
        // the threshold; O and l of those rows are rescaled by alpha below,
        // after the exponentials (the scores are dead by then, so O moves
        // through registers in large pieces with few waits).
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
        const float mref = (m == -INFINITY) ? 0.f : m;
        // Exponent arguments, row sums and scalings run two lanes per
        // instruction (packed fp32); four partial sums keep the adds independent.
        const float2 nm2 = make_float2(-mref, -mref);
        float2 rs2[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                         make_float2(0.f, 0.f)};
        if constexpr (FP8) {
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            const float2 g2 = c == 0 ? make_float2(g0, g0) : make_float2(g1, g1);
            uint32_t pk[16];
            const float2 fc2 = c == 0 ? make_float2(f0, f0) : make_float2(f1, f1);
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const int col = c * 64 + 4 * i;
              const float2 x01 = __ffma2_rn(make_float2(s[col], s[col + 1]), fc2, nm2);
              const float2 x23 = __ffma2_rn(make_float2(s[col + 2], s[col + 3]), fc2, nm2);
              float2 p01 = make_float2(ex2_approx(x01.x), ex2_approx(x01.y));
              float2 p23 = make_float2(ex2_approx(x23.x), ex2_approx(x23.y));
              rs2[(2 * i) & 3] = __fadd2_rn(rs2[(2 * i) & 3], p01);
              rs2[(2 * i + 1) & 3] = __fadd2_rn(rs2[(2 * i + 1) & 3], p23);
              p01 = __fmul2_rn(p01, g2);
              p23 = __fmul2_rn(p23, g2);
              pk[i] = (uint32_t)pack_e4m3x2(p01.x, p01.y) |
                      ((uint32_t)pack_e4m3x2(p23.x, p23.y) << 16);
            }
            tmem_st16(s_addr + c * 16, pk);
          }
        } else {
          const float2 sc2 = make_float2(sl2, sl2);
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const float2 x =
                  __ffma2_rn(make_float2(s[c * 32 + 2 * i], s[c * 32 + 2 * i + 1]), sc2, nm2);
              const float p0 = ex2_approx(x.x);
              const float p1 = ex2_approx(x.y);
              rs2[i & 3] = __fadd2_rn(rs2[i & 3], make_float2(p0, p1));
              pk[i] = BF16 ? pack_bf16x2(p0, p1) : pack_f16x2(p0, p1);
            }
            tmem_st16(s_addr + c * 16, pk);
          }
        }
        const float2 rsum = __fadd2_rn(__fadd2_rn(rs2[0], rs2[1]), __fadd2_rn(rs2[2], rs2[3]));
        l = l * alpha + (rsum.x + rsum.y);
        if (rescale) {
          // O_row *= alpha (1 for rows whose max did not rise).  The previous
          // P V into O has completed: its MMA was issued before the S whose
          // completion this block waited for; the next one is issued only
          // after this block's P is handed over.
#pragma unroll 1
          for (int c = 0; c < kPaddedD<D> / 64; ++c) {
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
        tmem_wait_st();
        tc_fence_before();
        }
        // Hand P_t(j) to the issuer (and learn whether anyone has aborted).
        aborted = named_bar_or(kBarP + t, 160, aborted);
      }
      // ------------------------------------------------------- epilogue ---
      const uint32_t opar = o_it & 1;
      ++o_it;
      if (!aborted)
        aborted = !__all_sync(0xffffffffu, mbar_wait(bar(L::kOFull + t), opar, wd, 12));
      if (aborted) continue;
      tc_fence_after();
      // A row that sees no key of this split (a short query block against a
      // longer cache) has l = 0: O = 0, LSE = -inf.
      const float inv_l = l > 0.f ? (FP8 ? sv_max : 1.0f) / l : 0.f;
      const size_t grow = MODE == kModePacked ? (size_t)w.zq * p.q_zrows + w.qrow + row
                                : (size_t)w.zq * p.N + w.row0 + row;
      uint4* orow = reinterpret_cast<uint4*>(obase + grow * D);
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t raw[32];
        tmem_ld32_sync(o_addr + c * 32, raw);
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float a = __uint_as_float(raw[2 * i]) * inv_l;
          const float b = __uint_as_float(raw[2 * i + 1]) * inv_l;
          pk[i] = (BF16 || FP8) ? pack_bf16x2(a, b) : pack_f16x2(a, b);
        }
        if (row < w.len) {
#pragma unroll
          for (int v = 0; v < 4; ++v)
            orow[c * 4 + v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
        }
      }
      if (row < w.len) lbase[grow] = (m + log2f(l)) * 0.69314718055994530942f;
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

template <int D, bool CAUSAL, int PREC, int MODE>
cudaError_t launch_one(const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV,
                       const FwdParams& params, int num_ctas, cudaStream_t stream) {
  using L = FwdLayout<D, PREC == kPrecE4M3>;
  auto kern = fwd_kernel<D, CAUSAL, PREC, MODE>;
  static DeviceFlags configured;  // attribute set once per device and instantiation
  cudaError_t e = ensure_dyn_smem(kern, L::kDynSmem, configured);
  if (e != cudaSuccess) return e;
  const int grid = params.num_units < num_ctas ? params.num_units : num_ctas;
  kern<<<grid, kThreads, L::kDynSmem, stream>>>(tmQ, tmK, tmV, params);
  return cudaGetLastError();
}

template <int D, int PREC>
cudaError_t launch_dc(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                      const FwdParams& p, int n, cudaStream_t s, bool causal) {
  if constexpr (PREC != kPrecE4M3) {
    if (p.pack_nq > 0)
      return causal ? launch_one<D, true, PREC, kModePacked>(q, k, v, p, n, s)
                    : launch_one<D, false, PREC, kModePacked>(q, k, v, p, n, s);
    if (p.cu_seqlens != nullptr)
      return causal ? launch_one<D, true, PREC, kModeVarlen>(q, k, v, p, n, s)
                    : launch_one<D, false, PREC, kModeVarlen>(q, k, v, p, n, s);
  }
  return causal ? launch_one<D, true, PREC, kModeDense>(q, k, v, p, n, s)
                : launch_one<D, false, PREC, kModeDense>(q, k, v, p, n, s);
}

}  // namespace

cudaError_t launch_fwd(const FwdLaunch& a, int d, bool causal, bool bf16) {
  const auto& q = a.tmQ;
  const auto& k = a.tmK;
  const auto& v = a.tmV;
  if (d == 128)
    return bf16 ? launch_dc<128, kPrecBF16>(q, k, v, a.params, a.num_ctas, a.stream, causal)
                : launch_dc<128, kPrecF16>(q, k, v, a.params, a.num_ctas, a.stream, causal);
  if (d == 96)
    return bf16 ? launch_dc<96, kPrecBF16>(q, k, v, a.params, a.num_ctas, a.stream, causal)
                : launch_dc<96, kPrecF16>(q, k, v, a.params, a.num_ctas, a.stream, causal);
  return bf16 ? launch_dc<64, kPrecBF16>(q, k, v, a.params, a.num_ctas, a.stream, causal)
              : launch_dc<64, kPrecF16>(q, k, v, a.params, a.num_ctas, a.stream, causal);
}

cudaError_t launch_fwd_fp8(const Fp8FwdLaunch& a) {
  FwdParams p = a.base.params;
  p.q_scale = a.q_scale;
  p.k_scale = a.k_scale;
  p.v_scale = a.v_scale;
  p.n_sblocks = (p.N + 63) / 64;
  return launch_dc<128, kPrecE4M3>(a.tmQ, a.tmK, a.tmVt, p, a.base.num_ctas, a.base.stream,
                                   a.causal);
}

}  // namespace attn
