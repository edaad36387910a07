/*
 * attn.h — C ABI of libattn: exact scaled-dot-product attention on one
 * NVIDIA GB300 (sm_103a), computed in tiles with an online softmax.
 *
 * The operation is the one described by "FlashAttention-2: Faster Attention
 * with Better Parallelism and Work Partitioning" (paper review page): the
 * flowchart under "프레임워크 개요" (Q, K, V in HBM; per (batch, head,
 * query-block) thread block; load the Q tile; iterate over K/V tiles with
 * QK^T and online-softmax statistics; accumulate softmax(S) V; rescale once at
 * the end; write O and the log-sum-exp), its "Methods" section (deferred
 * 1/rowsum scaling, only the log-sum-exp is stored and reused by the
 * backward pass) and "핵심 구성요소" (blocks entirely above the causal
 * diagonal are skipped; the backward pass recomputes with the stored
 * log-sum-exp).  The FP8 entry points follow "8.3 FlashAttention-3",
 * sections 5.1 (block quantization) and 5.2 (incoherent processing with a
 * Hadamard transform).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Layout: Q, K, V, O, dO, dQ, dK, dV are [B, H, N, d] row-major and
 *    contiguous (d innermost); LSE and the delta vector D are [B, H, N].
 *    All pointers are DEVICE pointers, 16-byte aligned (TMA requirement).
 *  - Shapes: d in {64, 96, 128}; attn_fwd, attn_fwd_gqa, attn_bwd,
 *    attn_bwd_gqa, attn_bwd_noalloc and attn_merge also take d in
 *    {192, 256}, and so do attn_fwd_split and attn_fwd_kv with at most 128
 *    query rows per key/value head (otherwise the key split, key cache and
 *    variable-length entry points return ATTN_ERR_UNSUPPORTED there; the
 *    FP8 entry points: as stated there);
 *    N >= 1 (any N: partial tiles are zero-filled on load and masked);
 *    B, H >= 1; B*H*N*d must fit in 2^31 elements.
 *  - Causal masking is top-left aligned: key j is visible to query i iff
 *    j <= i.  `scale` multiplies QK^T (1/sqrt(d) in the usual case).
 *  - LSE is the natural log of sum_j exp(scale * q_i . k_j) over the visible
 *    keys, stored as fp32.
 *  - Ownership: the caller allocates and owns all memory.  No entry point
 *    allocates device memory; the backward pass takes a caller-provided
 *    workspace (see attn_bwd_workspace_bytes).
 *  - Asynchrony: every compute call is enqueued on `stream` (a cudaStream_t;
 *    NULL = the legacy default stream) and returns ATTN_OK once the launches
 *    are accepted.  Kernel-side failures (a pipeline wait that ran out of
 *    time) are reported later by attn_poll_device_status.
 *  - Errors: invalid arguments return ATTN_ERR_INVALID_ARG / _UNSUPPORTED
 *    before anything is launched; no exception crosses the ABI.
 */
#ifndef ATTN_H_
#define ATTN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  ATTN_OK = 0,
  ATTN_ERR_INVALID_ARG = 1,  /* null/misaligned pointer, bad size or flag */
  ATTN_ERR_UNSUPPORTED = 2,  /* valid but unsupported (d, dtype, device)  */
  ATTN_ERR_CUDA = 3,         /* a CUDA runtime/driver call failed          */
  ATTN_ERR_TIMEOUT = 4       /* a kernel pipeline wait ran out of time     */
} attn_status;

typedef enum { ATTN_F16 = 0, ATTN_BF16 = 1 } attn_dtype;

/*
 * Forward pass.  O = softmax(scale * Q K^T, masked) V and
 * LSE_i = log sum_j exp(scale * q_i . k_j).
 *   q, k, v : [B,H,N,d] fp16 or bf16 (per `dtype`), read only.
 *   o       : [B,H,N,d] same dtype, written (round to nearest even).
 *   lse     : [B,H,N] fp32, written.
 *   causal  : 0 or 1.
 *   d       : 64, 96, 128, 192 or 256.
 * Cite: FlashAttention-2 review, flowchart "프레임워크 개요" and "Methods";
 * causal block skipping in "핵심 구성요소".  d in {192, 256} computes the
 * same formulas with wider heads (an extension: the pages' workloads use
 * d = 64 and 128); those run one 128-row query tile per work unit.
 */
attn_status attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                     int H, int N, int d, int causal, float scale, attn_dtype dtype,
                     void* stream);

/*
 * Forward pass with grouped query heads (GQA; Hkv = 1 is multi-query
 * attention): q, o [B,Hq,N,d], k, v [B,Hkv,N,d] with Hkv dividing Hq; query
 * head h of a batch attends with key/value head h / (Hq/Hkv).  lse [B,Hq,N].
 * Other arguments and errors as in attn_fwd (ATTN_ERR_INVALID_ARG if Hkv does
 * not divide Hq).  attn_fwd is the case Hkv = Hq.
 * Cite: the FlashAttention-2 review, "Insights" (linked work: GQA, training
 * generalized multi-query transformer models).
 */
attn_status attn_fwd_gqa(const void* q, const void* k, const void* v, void* o, float* lse,
                         int B, int Hq, int Hkv, int N, int d, int causal, float scale,
                         attn_dtype dtype, void* stream);

/*
 * Forward pass over a split of the keys: the ceil(N/128) key blocks are cut
 * into n_split contiguous runs (split s = blocks [s nb / n_split,
 * (s+1) nb / n_split), a run may be empty), and split s writes the partial
 * result of its keys alone:
 *   o_part   : [n_split, B, H, N, d] same dtype as q; partial O_s (each row
 *              normalised over the split's visible keys), written.
 *   lse_part : [n_split, B, H, N] fp32; LSE_s = log sum over the split's
 *              visible keys of exp(scale q.k); -inf (and O_s = 0) for a row
 *              that sees no key of the split.  Written.
 * Other arguments as in attn_fwd; 1 <= n_split <= 256.  With n_split = 1 the
 * output equals attn_fwd's.  attn_merge combines the partial results.
 * Cite: "8.3 FlashAttention-3" section 7.3 (ring attention: attention
 * computed over parts of the keys) and the FlashAttention-2 review,
 * "Discussion Points" (a decoding kernel that splits the keys).
 */
attn_status attn_fwd_split(const void* q, const void* k, const void* v, void* o_part,
                           float* lse_part, int n_split, int B, int H, int N, int d, int causal,
                           float scale, attn_dtype dtype, void* stream);

/*
 * Forward pass of a block of Nq queries against a longer key/value cache
 * (decoding: Nq = 1, or a few draft tokens), split over the keys like
 * attn_fwd_split and with grouped query heads like attn_fwd_gqa:
 *   q        : [B,Hq,Nq,d], read only;  k, v : [B,Hkv,Nk,d], read only.
 *   o_part   : [n_split,B,Hq,Nq,d] same dtype; lse_part [n_split,B,Hq,Nq]
 *              fp32; written as in attn_fwd_split (n_split = 1: the final
 *              O and LSE; otherwise combine them with attn_merge, whose
 *              N is Nq).
 *   1 <= Nq <= Nk.  The queries are the last Nq positions of the sequence:
 *   with causal = 1 query i sees keys j <= i + Nk - Nq (so every query sees
 *   at least Nk - Nq + 1 keys); causal = 0 sees all Nk keys.  Nq = Nk gives
 *   attn_fwd_split (attn_fwd_gqa).  The split covers ceil(Nk/128) key
 *   blocks.  Other arguments and errors as in attn_fwd_split and
 *   attn_fwd_gqa.  With at most 16 query rows per key/value head
 *   ((Hq/Hkv) * Nq <= 16) the call runs a decoding kernel that reads every
 *   key and value once (any dense forward entry point of that shape does),
 *   at d in {64, 96, 128, 192, 256}.  At d in {192, 256} the same kernel
 *   takes up to 128 rows per key/value head, 16 rows per work unit (each
 *   unit streams the head's keys and values); more rows there return
 *   ATTN_ERR_UNSUPPORTED.  The results follow the same definition.
 * Cite: the FlashAttention-2 review, "Discussion Points" (decoding with a
 * KV cache by a kernel that splits the keys, then combines the parts).
 */
attn_status attn_fwd_kv(const void* q, const void* k, const void* v, void* o_part,
                        float* lse_part, int n_split, int B, int Hq, int Hkv, int Nq, int Nk,
                        int d, int causal, float scale, attn_dtype dtype, void* stream);

/*
 * Merge partial results over disjoint key sets (as written by
 * attn_fwd_split): per row, LSE = log sum_s exp(LSE_s) and
 * O = sum_s exp(LSE_s - LSE) O_s, computed in fp32 with the running maximum;
 * rows where every LSE_s is -inf get O = 0, LSE = -inf.
 *   o_part   : [n_split, B, H, N, d] fp16/bf16 (dtype), read only.
 *   lse_part : [n_split, B, H, N] fp32, read only.
 *   o        : [B, H, N, d] dtype, written;  lse : [B, H, N] fp32, written.
 * d in {64, 96, 128, 192, 256}; 1 <= n_split <= 256.
 * Cite: the FlashAttention-2 review, "Insights" (the log-sum-exp is all that
 * has to be kept besides O); the combine formula follows from the softmax
 * definition over the union of the key sets.
 */
attn_status attn_merge(const void* o_part, const float* lse_part, int n_split, void* o,
                       float* lse, int B, int H, int N, int d, attn_dtype dtype, void* stream);

/*
 * Bytes of device workspace attn_bwd needs: the delta vector
 * D_i = sum_c dO_ic O_ic (fp32 [B,H,N]), rounded up to 256 bytes, and 256
 * bytes of counters through which the kernels hand out their work.  Returns
 * 0 for invalid sizes.
 */
size_t attn_bwd_workspace_bytes(int B, int H, int N, int d);

/*
 * Backward pass for the loss whose gradient with respect to O is `dout`.
 * Recomputes P from `lse` (written by attn_fwd on the same inputs) and writes
 *   dV = P^T dO,  dS = P o (dO V^T - D),  dQ = scale dS K,  dK = scale dS^T Q.
 *   q, k, v, o, dout : [B,H,N,d] fp16/bf16, read only.
 *   lse              : [B,H,N] fp32 from attn_fwd, read only.
 *   dq, dk, dv       : [B,H,N,d] same dtype, written.
 *   workspace        : >= attn_bwd_workspace_bytes(B,H,N,d) bytes, 256-byte
 *                      aligned, caller-owned; contents on entry are ignored
 *                      and on return are unspecified.  Two calls in flight
 *                      at once (on different streams) need two workspaces.
 * d in {64, 96, 128, 192, 256} (ATTN_ERR_UNSUPPORTED otherwise).  dK, dV
 * (per key tile; at d = 256 per key tile and half of the columns) and dQ (per
 * query tile) are each accumulated in fp32 by one CTA in a fixed order, so
 * the results are the same from run to run.
 * Cite: FlashAttention-2 review, "Methods" (log-sum-exp kept for the backward
 * pass) and "핵심 구성요소" (backward recomputation with the log-sum-exp).
 */
attn_status attn_bwd(const void* q, const void* k, const void* v, const void* o,
                     const void* dout, const float* lse, void* dq, void* dk, void* dv,
                     void* workspace, size_t workspace_bytes, int B, int H, int N, int d,
                     int causal, float scale, attn_dtype dtype, void* stream);

/*
 * Backward pass with grouped query heads: q, o, dout, dq [B,Hq,N,d];
 * k, v, dk, dv [B,Hkv,N,d]; lse [B,Hq,N]; Hkv divides Hq.  dK and dV of a
 * key/value head sum the gradients of the query heads of its group (one CTA
 * per key/value tile walks all of them, so the sum has a fixed order).
 * workspace: >= attn_bwd_workspace_bytes(B, Hq, N, d).  Other arguments and
 * errors as in attn_bwd; attn_bwd is the case Hkv = Hq.
 * Cite: as attn_bwd, and the FlashAttention-2 review, "Insights" (GQA).
 */
attn_status attn_bwd_gqa(const void* q, const void* k, const void* v, const void* o,
                         const void* dout, const float* lse, void* dq, void* dk, void* dv,
                         void* workspace, size_t workspace_bytes, int B, int Hq, int Hkv, int N,
                         int d, int causal, float scale, attn_dtype dtype, void* stream);

/*
 * Variable-length batch: n_seq independent sequences of different lengths,
 * packed back to back.  Sequence b owns rows [cu_seqlens[b], cu_seqlens[b+1])
 * of every head and attends only to its own keys (causal: key index <= query
 * index, both counted from the sequence's first row).
 *   q, o       : [Hq, total, d] fp16/bf16 (head-major, rows packed).
 *   k, v       : [Hkv, total, d];  Hkv divides Hq (query head h uses h/(Hq/Hkv)).
 *   lse        : [Hq, total] fp32, written.
 *   cu_seqlens : DEVICE array of n_seq + 1 int32, cu_seqlens[0] = 0,
 *                cu_seqlens[n_seq] = total, non-decreasing (empty sequences
 *                allowed), 4-byte aligned, read only.
 *   max_seqlen : >= the longest sequence, <= total; it sizes the launch.
 * The offsets are checked on the device: a violation records
 * ATTN_ERR_INVALID_ARG in the status word (attn_poll_device_status returns
 * it; the block field of `detail` holds the first bad index).  Every
 * sequence is clamped into [0, total) and to max_seqlen rows, so a bad array
 * gives wrong results but no access outside the tensors.  d in {64, 96, 128}.
 * Cite: the FlashAttention-2 review, "Discussion Points" (the decoding /
 * KV-cache access pattern: many sequences of their own lengths); per
 * sequence the computation is attn_fwd's.
 */
attn_status attn_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse,
                            const int* cu_seqlens, int n_seq, int max_seqlen, int total, int Hq,
                            int Hkv, int d, int causal, float scale, attn_dtype dtype,
                            void* stream);

/*
 * Backward pass of attn_fwd_varlen: q, o, dout, dq [Hq, total, d]; k, v, dk,
 * dv [Hkv, total, d]; lse [Hq, total] from attn_fwd_varlen.  workspace: >=
 * attn_bwd_workspace_bytes(1, Hq, total, d) bytes, 256-byte aligned.  Rows of
 * dq, dk, dv outside every sequence (none when the offsets are valid) are
 * not written.  d in {64, 96, 128}.  Offsets, checks and errors as in
 * attn_fwd_varlen.
 * Cite: as attn_bwd and attn_fwd_varlen.
 */
attn_status attn_bwd_varlen(const void* q, const void* k, const void* v, const void* o,
                            const void* dout, const float* lse, void* dq, void* dk, void* dv,
                            void* workspace, size_t workspace_bytes, const int* cu_seqlens,
                            int n_seq, int max_seqlen, int total, int Hq, int Hkv, int d,
                            int causal, float scale, attn_dtype dtype, void* stream);

/*
 * Backward pass that allocates nothing (no counterpart on the pages: it is a
 * library convenience, not part of the method).
 *
 * For callers that cannot hand attn_bwd a workspace: plugins whose host
 * framework owns all device memory and exposes no raw allocations, serving
 * loops that must not call cudaMalloc (which can synchronise the device) on
 * the request path, or programs with a fixed memory plan.  It computes the
 * same dQ, dK, dV as attn_bwd, with the same arguments minus the workspace;
 * the scratch (the fp32 delta vector and the kernels' work counters) lives
 * in a fixed device array inside the library.
 *   Limit: B*H*N <= 4194304 query rows and d in {64, 96, 128, 192, 256}; larger
 *   problems return ATTN_ERR_INVALID_ARG, other head dims ATTN_ERR_UNSUPPORTED.
 *   Memory: the array (16 MB) is part of the library image and is held on
 *   every GPU that loads the library until the process exits.
 *   Sharing: all calls use the same array: calls that overlap on the GPU
 *   (different streams, or different host threads, without ordering between
 *   them) race on it and give wrong results.
 *   Set-up: the first call on each device looks up the array's device
 *   address (cudaGetSymbolAddress) with that device current; make that
 *   first call before any stream capture.  The address is kept for the
 *   life of the process: calls made after cudaDeviceReset on that device
 *   are not supported (the array may then sit elsewhere).
 */
attn_status attn_bwd_noalloc(const void* q, const void* k, const void* v, const void* o,
                             const void* dout, const float* lse, void* dq, void* dk, void* dv,
                             int B, int H, int N, int d, int causal, float scale,
                             attn_dtype dtype, void* stream);

/*
 * FP8 E4M3 block quantization of one bf16 tensor, optionally after the
 * randomized Hadamard rotation x <- x H_d diag(signs) / sqrt(d).
 *   x_bf16  : [B,H,N,d] bf16, read only.
 *   x_e4m3  : [B,H,N,d] bytes (E4M3) — or [B,H,d,N] when write_transposed=1.
 *   scales  : [B,H,ceil(N/block_rows)] fp32: s = amax/448 over each block of
 *             `block_rows` rows x d columns (s = 1 if the block is all zero);
 *             codes are E4M3(x/s), round to nearest even, saturating.
 *   block_rows : 64 (the only supported value);  d in {64, 128} (the
 *             rotation is a Walsh-Hadamard transform of power-of-two size).
 *   hadamard_signs : NULL (no rotation) or a DEVICE array of d int8 values,
 *             each +1 or -1.
 *   write_transposed : 0 or 1; 1 requires N % 16 == 0.
 * Cite: "8.3 FlashAttention-3", sections 5.1 and 5.2.
 */
attn_status attn_quantize_fp8(const void* x_bf16, void* x_e4m3, float* scales, int B, int H,
                              int N, int d, int block_rows, const int8_t* hadamard_signs,
                              int write_transposed, void* stream);

/*
 * FP8 forward pass: O = softmax(scale * Q K^T) V with E4M3 inputs and fp32
 * accumulation; S_ij = q8_i . k8_j * sq(i/64) * sk(j/64).
 *   q8, k8  : [B,H,N,d] E4M3 from attn_quantize_fp8 (same rotation for both).
 *   v8t     : [B,H,d,N] E4M3 (attn_quantize_fp8 with write_transposed=1).
 *   q_scale, k_scale, v_scale : [B,H,ceil(N/64)] fp32 block scales.
 *   o       : [B,H,N,d] bf16, written.   lse : [B,H,N] fp32, written.
 * Requires d = 128 and N % 16 == 0.
 * Cite: "8.3 FlashAttention-3", section 5 and section 6.2.
 */
attn_status attn_fwd_fp8(const void* q8, const void* k8, const void* v8t, const float* q_scale,
                         const float* k_scale, const float* v_scale, void* o, float* lse, int B,
                         int H, int N, int d, int causal, float scale, void* stream);

/*
 * Synchronise `stream`, then read and clear the library's device status
 * word.  Returns ATTN_ERR_TIMEOUT if a kernel pipeline wait ran out of time
 * since the last poll (the kernel then skipped the rest of its work and
 * released its resources; outputs are incomplete), ATTN_ERR_CUDA if the
 * synchronisation failed, ATTN_ERR_INVALID_ARG if a device-side argument
 * check failed (variable-length offsets), else ATTN_OK.  `detail` (may be
 * NULL) receives the raw status word: code | site << 8 | block index << 16.
 */
attn_status attn_poll_device_status(void* stream, uint32_t* detail);

/*
 * Set the time limit of every bounded pipeline wait in later launches, in
 * microseconds (default 2,000,000 = 2 s; 0 restores the default).
 */
attn_status attn_set_wait_limit_us(uint64_t limit_us);

/*
 * Self-test of the failure path: launches one block that waits on an
 * mbarrier nothing will ever arrive at, with a `limit_us` time limit.  The
 * kernel must give up, record ATTN_ERR_TIMEOUT in the status word and exit
 * normally.  Returns the result of attn_poll_device_status.
 */
attn_status attn_selftest_wait_timeout(uint64_t limit_us, void* stream, uint32_t* detail);

/* Human-readable name of a status code (static storage). */
const char* attn_status_string(attn_status s);

/* Number of SMs the persistent kernels size their grid by (device 0 current). */
int attn_num_sms(void);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_H_ */
