// Host <-> device interface of the backward kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

namespace attn {

struct BwdParams {
  const void* q;
  const void* k;
  const void* v;
  const void* o;
  const void* dout;
  const float* lse;      // [B*H, N] natural-log LSE from the forward pass
  void* dq;
  void* dk;
  void* dv;
  float* delta;          // workspace: D_i = sum_c dO_ic O_ic  [B*H, N]
  uint32_t* status;
  int BH, N;            // BH = B * heads (query heads)
  // Grouped query heads: query head h of a batch uses key/value head
  // h / group of its heads_kv; dK, dV ([B*heads_kv, N, D]) sum over the group.
  int heads = 1, heads_kv = 1, group = 1;
  int BHkv;              // B * heads_kv
  // Variable-length batch (cu_seqlens non-null): q, o, dO, dQ are
  // [heads, N, D], k, v, dK, dV [heads_kv, N, D] and lse, delta [heads, N],
  // with N the total rows; sequence b owns rows [cu_seqlens[b],
  // cu_seqlens[b+1]) of every head.  B counts sequences, n_qtiles and
  // n_kblocks count tiles of max_seqlen; units past a sequence's end are empty.
  const int* cu_seqlens = nullptr;
  int max_seqlen = 0;
  int n_qtiles;          // ceil(N / 128)
  int n_kblocks;         // ceil(N / 128)
  float scale;
  float scale_log2;      // scale * log2(e)
  unsigned long long wait_limit_ns;
  // Work counters of the dK/dV ([0]) and dQ ([1]) kernels in the workspace,
  // zeroed by the D pass: each CTA takes its next unit with an atomic add.
  int* sched = nullptr;
  // Causal and variable-length orders hand out the units of head_block
  // key/value heads (dK/dV) or head_block_q query heads (dQ) before those of
  // the next heads, so the tiles the CTAs stream stay in L2.
  int head_block = 1, head_block_q = 1;
};

struct BwdLaunch {
  CUtensorMap tmQ, tmK, tmV, tmDO;
  BwdParams params;
  int num_sms;
  cudaStream_t stream;
  bool causal, bf16;
  int d = 128;            // head dimension: 64, 96 or 128
};

cudaError_t launch_bwd(const BwdLaunch& a);

// The D pass alone (D_i = sum_c dO_ic O_ic into params.delta), any head dim.
cudaError_t launch_bwd_pre(const BwdParams& p, int d, bool bf16, int num_sms,
                           cudaStream_t stream);

// Head dims 192 and 256 (bwd_wide.cu): the dK/dV kernel reads Q and dO in
// tiles of 64 rows, the dQ kernel K and V in tiles of 64 rows, so both sets
// of tensor maps are needed.  Dense or grouped heads only.
struct BwdWideLaunch {
  CUtensorMap tmQ, tmK, tmV, tmDO;          // boxes of 64 columns x 128 rows
  CUtensorMap tmQ64, tmK64, tmV64, tmDO64;  // boxes of 64 columns x 64 rows
  BwdParams params;
  int num_sms;
  cudaStream_t stream;
  bool causal, bf16;
  int d;                                    // 192 or 256
};

cudaError_t launch_bwd_wide(const BwdWideLaunch& a);

}  // namespace attn
