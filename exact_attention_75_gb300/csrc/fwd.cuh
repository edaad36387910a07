// Host <-> device interface of the forward kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

namespace attn {

struct FwdParams {
  void* o;              // [B*H, N, D] 16-bit output
  float* lse;           // [B*H, N] fp32 output
  uint32_t* status;     // device status word
  int BH, N;            // N: query rows per head
  // Key / value rows per head (= N except when a short block of queries
  // attends to a longer key cache).  Causal masking is aligned at the
  // bottom right: query row i sits at key position i + Nk - N.
  int Nk;
  // Rows per tensor-map head index of the Q / O layout (N; heads * N when
  // grouped heads are packed).
  int q_zrows;
  // Grouped query heads packed into one tile (pack_nq = N > 0, dense only,
  // group * N <= 128): a work unit is (batch, key/value head, split) and its
  // single query tile holds the group's query heads, N rows each, contiguous
  // in the [B, heads * N, D] view of Q and O.  Each K/V block is then read and
  // multiplied once per group instead of once per query head.
  int pack_nq = 0;
  int n_qtiles;         // ceil(N / 128)
  int n_pairs;          // ceil(n_qtiles / 2): work units per head
  int n_kblocks;        // ceil(N / 128)
  int num_units;        // n_split * BH * n_pairs
  // Split over the keys: split s covers key blocks [s nb / n_split,
  // (s+1) nb / n_split) and writes its partial O / LSE at o + s * o_split,
  // lse + s * lse_split (elements).  n_split = 1: the whole key range.
  int n_split = 1;
  size_t o_split = 0, lse_split = 0;
  // Grouped query heads: BH counts query heads (B * heads); query head h of a
  // batch uses key/value head h / group of the heads_kv of that batch.
  int heads = 1, heads_kv = 1, group = 1;
  // Variable-length batch (cu_seqlens non-null): q, o are [heads, N, D] and
  // k, v [heads_kv, N, D] with N the total rows of all sequences; sequence b
  // owns rows [cu_seqlens[b], cu_seqlens[b+1]) of every head and attends only
  // within itself.  BH = n_seq * heads; n_qtiles, n_kblocks and n_pairs count
  // tiles of max_seqlen, and units past a shorter sequence's end are empty.
  const int* cu_seqlens = nullptr;
  int max_seqlen = 0;
  float scale_log2;     // scale * log2(e)
  unsigned long long wait_limit_ns;
  // E4M3 path only: per-(head, 64-row block) fp32 scales of Q, K and V.
  const float* q_scale = nullptr;
  const float* k_scale = nullptr;
  const float* v_scale = nullptr;
  int n_sblocks = 0;    // ceil(N / 64)
};

struct FwdLaunch {
  CUtensorMap tmQ, tmK, tmV;
  FwdParams params;
  int num_ctas;         // persistent grid size (number of SMs)
  cudaStream_t stream;
};

cudaError_t launch_fwd(const FwdLaunch& a, int d, bool causal, bool bf16);
// d in {192, 256}: one query tile per work unit (fwd_wide.cu); dense or
// grouped heads, no key split, no packed or variable-length modes.
cudaError_t launch_fwd_wide(const FwdLaunch& a, int d, bool causal, bool bf16);

}  // namespace attn
