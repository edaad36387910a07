// Host side of the C ABI declared in include/attn.h: argument validation,
// TMA descriptor construction, launch configuration and the device status
// word.  No function here allocates device memory.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "attn.h"
#include "bwd.cuh"
#include "decode.cuh"
#include "fp8.cuh"
#include "fwd.cuh"
#include "merge.cuh"
#include "sm103_ptx.cuh"

namespace attn {

// Status word written by kernels whose pipeline waits ran out of time.
__device__ uint32_t g_status_word;

namespace {

constexpr int kMaxDevices = 64;
constexpr unsigned long long kDefaultWaitNs = 2000000000ull;
std::atomic<unsigned long long> g_wait_limit_ns{kDefaultWaitNs};

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

struct DeviceInfo {
  bool ready = false;
  int num_sms = 0;
  bool supported = false;
  uint32_t* status = nullptr;
};

std::mutex g_mu;
DeviceInfo g_dev[kMaxDevices];
EncodeTiledFn g_encode = nullptr;

attn_status device_info(DeviceInfo** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ATTN_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceInfo& di = g_dev[dev];
  if (!di.ready) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&di.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return ATTN_ERR_CUDA;
    di.supported = (major == 10 && minor == 3);
    void* addr = nullptr;
    if (cudaGetSymbolAddress(&addr, g_status_word) != cudaSuccess) return ATTN_ERR_CUDA;
    di.status = static_cast<uint32_t*>(addr);
    if (g_encode == nullptr) {
      cudaDriverEntryPointQueryResult q;
      void* fn = nullptr;
      if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                           &q) != cudaSuccess ||
          q != cudaDriverEntryPointSuccess || fn == nullptr)
        return ATTN_ERR_CUDA;
      g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    }
    di.ready = true;
  }
  if (!di.supported) return ATTN_ERR_UNSUPPORTED;
  *out = &di;
  return ATTN_OK;
}

attn_status launch_result(cudaError_t e) {
  if (e == cudaSuccess) return ATTN_OK;
  if (e == cudaErrorNotSupported) {
    cudaGetLastError();
    return ATTN_ERR_UNSUPPORTED;
  }
  return ATTN_ERR_CUDA;
}

bool aligned16(const void* p) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

// 3-D tiled map over a contiguous [outer, rows, inner] tensor with the
// 128-byte swizzle; box = [1, box_rows, box_inner].
bool encode_3d(CUtensorMap* m, const void* ptr, CUtensorMapDataType dt, int esize, int64_t inner,
               int64_t rows, int64_t outer, int box_inner, int box_rows,
               CUtensorMapSwizzle swz = CU_TENSOR_MAP_SWIZZLE_128B) {
  cuuint64_t dims[3] = {(cuuint64_t)inner, (cuuint64_t)rows, (cuuint64_t)outer};
  cuuint64_t strides[2] = {(cuuint64_t)(inner * esize), (cuuint64_t)(inner * rows * esize)};
  cuuint32_t box[3] = {(cuuint32_t)box_inner, (cuuint32_t)box_rows, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return g_encode(m, dt, 3, const_cast<void*>(ptr), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Host-side checks of a variable-length batch description (the offsets
// themselves live on the device and are checked there).
bool varlen_args_ok(const int* cu_seqlens, int n_seq, int max_seqlen, int total) {
  if ((reinterpret_cast<uintptr_t>(cu_seqlens) & 3) != 0) return false;
  if (n_seq < 1 || total < 1) return false;
  return max_seqlen >= 1 && max_seqlen <= total;
}

// Records ATTN_ERR_INVALID_ARG (site 60, the first bad index in the block
// field) in the status word unless cu_seqlens[0] = 0, cu_seqlens[n_seq] =
// total and 0 <= cu_seqlens[b+1] - cu_seqlens[b] <= max_seqlen for every b.
// The attention kernels clamp every sequence into [0, total) themselves, so
// a bad array gives wrong numbers but no access outside the tensors.
__global__ void varlen_check_kernel(const int* cu, int n_seq, int total, int max_seqlen,
                                    uint32_t* status) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b > n_seq) return;
  bool bad = false;
  if (b == 0) bad = cu[0] != 0;
  if (b == n_seq) bad = bad || cu[n_seq] != total;
  if (b < n_seq) {
    const int len = cu[b + 1] - cu[b];
    bad = bad || len < 0 || len > max_seqlen;
  }
  if (bad)
    atomicCAS(status, 0u, (uint32_t)ATTN_ERR_INVALID_ARG | (60u << 8) |
                              ((uint32_t)min(b, 0xFFFF) << 16));
}

cudaError_t launch_varlen_check(const int* cu, int n_seq, int total, int max_seqlen,
                                uint32_t* status, cudaStream_t stream) {
  const int threads = 256;
  const int blocks = (n_seq + 1 + threads - 1) / threads;
  varlen_check_kernel<<<blocks, threads, 0, stream>>>(cu, n_seq, total, max_seqlen, status);
  return cudaGetLastError();
}

// Bytes of the backward's delta vector (fp32 per query row), rounded up to
// 256; the work counters follow it in the workspace.
size_t bwd_delta_bytes(int B, int H, int N) {
  return ((size_t)B * H * N * 4 + 255) & ~(size_t)255;
}

// Heads per block of the backward's causal unit order: as many as keep the
// tiles that one block's units stream (per_head bytes each) within 32 MiB of
// L2, at least 4 (so that enough units of similar length are in flight for
// the CTAs to finish together) and at most all of them.
int bwd_head_block(double per_head, int total) {
  int hb = (int)(33554432.0 / per_head);
  if (hb < 4) hb = 4;
  if (hb > total) hb = total;
  return hb < 1 ? 1 : hb;
}

bool head_dim_ok(int d) { return d == 64 || d == 96 || d == 128 || d == 192 || d == 256; }

bool shape_ok(int B, int H, int N, int d) {
  if (B < 1 || H < 1 || N < 1) return false;
  if (!head_dim_ok(d)) return false;
  const int64_t bh = (int64_t)B * H;
  if (bh > (1 << 30) || N > (1 << 28)) return false;
  return bh * N * d < (int64_t)1 << 40;
}

}  // namespace

attn_status fill_fwd_common(FwdLaunch* a, DeviceInfo* di, int B, int H, int N, float scale,
                            void* stream, void* o, float* lse) {
  FwdParams& p = a->params;
  p.o = o;
  p.lse = lse;
  p.status = di->status;
  p.BH = B * H;
  p.N = N;
  p.Nk = N;
  p.q_zrows = N;
  p.n_qtiles = (N + 127) / 128;
  p.n_pairs = (p.n_qtiles + 1) / 2;
  p.n_kblocks = (N + 127) / 128;
  p.num_units = p.BH * p.n_pairs;
  p.heads = H;
  p.heads_kv = H;
  p.group = 1;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.wait_limit_ns = g_wait_limit_ns.load();
  a->num_ctas = di->num_sms;
  a->stream = static_cast<cudaStream_t>(stream);
  return ATTN_OK;
}

}  // namespace attn

using namespace attn;

namespace {

// The forward pass with Hkv key/value heads for H query heads (Hkv = H: plain
// multi-head attention) and the keys cut into n_split runs of whole 128-key
// blocks, each split writing its partial O / LSE at its own offset.
//
// With cu_seqlens (device, B + 1 entries) the batch is B packed sequences of
// at most max_seqlen rows: q, o are [H, N, d], k, v [Hkv, N, d], lse [H, N],
// N the total rows.
//
// Nk > 0 (dense batches only) gives K and V their own row count Nk >= N:
// the N queries are the last N positions of a sequence of Nk keys.
attn_status fwd_impl(const void* q, const void* k, const void* v, void* o, float* lse,
                     int n_split, int B, int H, int Hkv, int N, int d, int causal, float scale,
                     attn_dtype dtype, void* stream, const int* cu_seqlens = nullptr,
                     int max_seqlen = 0, int Nk = 0) {
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
    return ATTN_ERR_INVALID_ARG;
  const bool varlen = cu_seqlens != nullptr;
  if (varlen && !varlen_args_ok(cu_seqlens, B, max_seqlen, N)) return ATTN_ERR_INVALID_ARG;
  if (varlen && n_split != 1) return ATTN_ERR_INVALID_ARG;
  if (n_split < 1 || n_split > 256) return ATTN_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return ATTN_ERR_INVALID_ARG;
  if (dtype != ATTN_F16 && dtype != ATTN_BF16) return ATTN_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !std::isfinite(scale)) return ATTN_ERR_INVALID_ARG;
  if (B < 1 || H < 1 || N < 1) return ATTN_ERR_INVALID_ARG;
  if (Hkv < 1 || H % Hkv != 0) return ATTN_ERR_INVALID_ARG;
  if (!head_dim_ok(d)) return ATTN_ERR_UNSUPPORTED;
  if (!shape_ok(B, H, N, d)) return ATTN_ERR_INVALID_ARG;
  if (Nk == 0) Nk = N;
  if (Nk < N || (varlen && Nk != N) || !shape_ok(B, Hkv, Nk, d)) return ATTN_ERR_INVALID_ARG;
  // At most 16 query rows per key/value head (decoding: one or a few new
  // tokens of each query head of a group) run on the warp-level decoding
  // kernel, which streams every key and value once, at every head dim.  At
  // the wide head dims, whose tiled kernel has no key split or key cache,
  // it also takes those modes up to 128 rows per key/value head (16 rows per
  // unit, the units of a head sharing its key/value reads through L2).
  const bool wide = d > 128;
  const int64_t rows_kv = (int64_t)(H / Hkv) * N;
  const bool decode = !varlen && (rows_kv <= kDecodeMaxRows ||
                                  (wide && (n_split != 1 || Nk != N) && rows_kv <= kDecodeRowLimit));
  // Otherwise the wide head dims run one query tile per unit, dense or
  // grouped heads only: no key split, key cache or packed variable-length
  // batch.
  if (wide && !decode && (n_split != 1 || varlen || Nk != N)) return ATTN_ERR_UNSUPPORTED;
  DeviceInfo* di = nullptr;
  attn_status st = device_info(&di);
  if (st != ATTN_OK) return st;
  const CUtensorMapDataType dt =
      dtype == ATTN_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  const int64_t BH = (int64_t)B * H, BHkv = (int64_t)B * Hkv;
  if (decode) {
    const int n_rgroups = (int)((rows_kv + kDecodeMaxRows - 1) / kDecodeMaxRows);
    if (BHkv * n_split * n_rgroups > 0x7FFFFFFF) return ATTN_ERR_INVALID_ARG;
    DecodeLaunch a;
    if (!encode_3d(&a.tmK, k, dt, 2, d, Nk, BHkv, 64, kDecodeKeys) ||
        !encode_3d(&a.tmV, v, dt, 2, d, Nk, BHkv, 64, kDecodeKeys))
      return ATTN_ERR_CUDA;
    DecodeParams& p = a.params;
    p.q = q;
    p.o = o;
    p.lse = lse;
    p.status = di->status;
    p.Hkv = Hkv;
    p.R = (int)rows_kv;
    p.n_rgroups = n_rgroups;
    p.Nq = N;
    p.Nk = Nk;
    p.n_split = n_split;
    p.n_kblocks = (Nk + 127) / 128;
    p.causal = causal;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.o_split = (size_t)BH * N * d;
    p.lse_split = (size_t)BH * N;
    p.wait_limit_ns = g_wait_limit_ns.load();
    a.num_units = (int)(BHkv * n_split * n_rgroups);
    a.stream = static_cast<cudaStream_t>(stream);
    return launch_result(launch_decode(a, d, dtype == ATTN_BF16));
  }
  FwdLaunch a;
  // tensor-map head index: (batch, head) for dense tensors, head for packed ones
  const int64_t zq = varlen ? H : BH, zkv = varlen ? Hkv : BHkv;
  // Grouped heads whose queries fit one tile together (decoding: few
  // queries per head) share it: Q / O are then viewed as [B, H * N, d].
  const bool pack = !wide && !varlen && Hkv < H && (int64_t)(H / Hkv) * N <= 128;
  const int64_t q_rows = pack ? (int64_t)H * N : N, q_z = pack ? B : zq;
  if (!encode_3d(&a.tmQ, q, dt, 2, d, q_rows, q_z, 64, 128) ||
      !encode_3d(&a.tmK, k, dt, 2, d, Nk, zkv, 64, 128) ||
      !encode_3d(&a.tmV, v, dt, 2, d, Nk, zkv, 64, 128))
    return ATTN_ERR_CUDA;
  fill_fwd_common(&a, di, B, H, N, scale, stream, o, lse);
  FwdParams& p = a.params;
  p.Nk = Nk;
  if (pack) {
    p.pack_nq = N;
    p.q_zrows = H * N;
    p.n_pairs = 1;
    p.num_units = B * Hkv;  // one unit per (batch, key/value head)
  }
  p.n_kblocks = (Nk + 127) / 128;
  p.heads_kv = Hkv;
  p.group = H / Hkv;
  if (varlen) {
    p.cu_seqlens = cu_seqlens;
    p.max_seqlen = max_seqlen;
    p.n_qtiles = (max_seqlen + 127) / 128;
    p.n_kblocks = p.n_qtiles;
    p.n_pairs = (p.n_qtiles + 1) / 2;
    if ((int64_t)p.BH * p.n_pairs > 0x7FFFFFFF) return ATTN_ERR_INVALID_ARG;
    p.num_units = p.BH * p.n_pairs;
    cudaError_t e = launch_varlen_check(cu_seqlens, B, N, max_seqlen, di->status,
                                        static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return launch_result(e);
  }
  if ((int64_t)p.num_units * n_split > 0x7FFFFFFF) return ATTN_ERR_INVALID_ARG;
  p.n_split = n_split;
  p.num_units *= n_split;
  p.o_split = (size_t)BH * N * d;
  p.lse_split = (size_t)BH * N;
  if (wide) {
    p.num_units = p.BH * p.n_qtiles;  // one query tile per unit
    return launch_result(launch_fwd_wide(a, d, causal != 0, dtype == ATTN_BF16));
  }
  cudaError_t e = launch_fwd(a, d, causal != 0, dtype == ATTN_BF16);
  return launch_result(e);
}

}  // namespace

extern "C" {

const char* attn_status_string(attn_status s) {
  switch (s) {
    case ATTN_OK: return "ATTN_OK";
    case ATTN_ERR_INVALID_ARG: return "ATTN_ERR_INVALID_ARG";
    case ATTN_ERR_UNSUPPORTED: return "ATTN_ERR_UNSUPPORTED";
    case ATTN_ERR_CUDA: return "ATTN_ERR_CUDA";
    case ATTN_ERR_TIMEOUT: return "ATTN_ERR_TIMEOUT";
  }
  return "ATTN_ERR_UNKNOWN";
}

int attn_num_sms(void) {
  DeviceInfo* di = nullptr;
  if (device_info(&di) != ATTN_OK) return 0;
  return di->num_sms;
}

attn_status attn_set_wait_limit_us(uint64_t limit_us) {
  if (limit_us > 3600ull * 1000000ull) return ATTN_ERR_INVALID_ARG;
  g_wait_limit_ns.store(limit_us == 0 ? kDefaultWaitNs : limit_us * 1000ull);
  return ATTN_OK;
}


attn_status attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                     int H, int N, int d, int causal, float scale, attn_dtype dtype,
                     void* stream) {
  return fwd_impl(q, k, v, o, lse, 1, B, H, H, N, d, causal, scale, dtype, stream);
}

attn_status attn_fwd_gqa(const void* q, const void* k, const void* v, void* o, float* lse,
                         int B, int Hq, int Hkv, int N, int d, int causal, float scale,
                         attn_dtype dtype, void* stream) {
  return fwd_impl(q, k, v, o, lse, 1, B, Hq, Hkv, N, d, causal, scale, dtype, stream);
}

attn_status attn_fwd_kv(const void* q, const void* k, const void* v, void* o_part,
                        float* lse_part, int n_split, int B, int Hq, int Hkv, int Nq, int Nk,
                        int d, int causal, float scale, attn_dtype dtype, void* stream) {
  return fwd_impl(q, k, v, o_part, lse_part, n_split, B, Hq, Hkv, Nq, d, causal, scale, dtype,
                  stream, nullptr, 0, Nk);
}

attn_status attn_fwd_split(const void* q, const void* k, const void* v, void* o_part,
                           float* lse_part, int n_split, int B, int H, int N, int d, int causal,
                           float scale, attn_dtype dtype, void* stream) {
  return fwd_impl(q, k, v, o_part, lse_part, n_split, B, H, H, N, d, causal, scale, dtype,
                  stream);
}

attn_status attn_merge(const void* o_part, const float* lse_part, int n_split, void* o,
                       float* lse, int B, int H, int N, int d, attn_dtype dtype, void* stream) {
  if (!aligned16(o_part) || !aligned16(lse_part) || !aligned16(o) || !aligned16(lse))
    return ATTN_ERR_INVALID_ARG;
  if (n_split < 1 || n_split > 256) return ATTN_ERR_INVALID_ARG;
  if (dtype != ATTN_F16 && dtype != ATTN_BF16) return ATTN_ERR_INVALID_ARG;
  if (B < 1 || H < 1 || N < 1) return ATTN_ERR_INVALID_ARG;
  if (!head_dim_ok(d)) return ATTN_ERR_UNSUPPORTED;
  if (!shape_ok(B, H, N, d)) return ATTN_ERR_INVALID_ARG;
  DeviceInfo* di = nullptr;
  attn_status st = device_info(&di);
  if (st != ATTN_OK) return st;
  MergeLaunch a;
  a.o_part = o_part;
  a.lse_part = lse_part;
  a.o = o;
  a.lse = lse;
  a.rows = (long)B * H * N;
  a.n_split = n_split;
  a.d = d;
  a.bf16 = dtype == ATTN_BF16;
  a.num_sms = di->num_sms;
  a.stream = static_cast<cudaStream_t>(stream);
  return launch_result(launch_merge(a));
}

size_t attn_bwd_workspace_bytes(int B, int H, int N, int d) {
  if (!shape_ok(B, H, N, d)) return 0;
  // D = rowsum(dO o O), fp32, then 256 bytes for the main kernels' work counters
  return bwd_delta_bytes(B, H, N) + 256;
}

}  // extern "C"

namespace {

// The backward pass at d in {192, 256} (arguments already checked): the D
// pass, then the dK/dV kernel (Q and dO read 64 rows at a time) and the dQ
// kernel (K and V read 64 rows at a time).
attn_status bwd_wide_impl(DeviceInfo* di, const void* q, const void* k, const void* v,
                          const void* o, const void* dout, const float* lse, void* dq, void* dk,
                          void* dv, void* workspace, int B, int H, int Hkv, int N, int d,
                          int causal, float scale, attn_dtype dtype, void* stream) {
  BwdWideLaunch a;
  const CUtensorMapDataType dt =
      dtype == ATTN_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  const int64_t BH = (int64_t)B * H, BHkv = (int64_t)B * Hkv;
  if (!encode_3d(&a.tmQ, q, dt, 2, d, N, BH, 64, 128) ||
      !encode_3d(&a.tmK, k, dt, 2, d, N, BHkv, 64, 128) ||
      !encode_3d(&a.tmV, v, dt, 2, d, N, BHkv, 64, 128) ||
      !encode_3d(&a.tmDO, dout, dt, 2, d, N, BH, 64, 128) ||
      !encode_3d(&a.tmQ64, q, dt, 2, d, N, BH, 64, 64) ||
      !encode_3d(&a.tmK64, k, dt, 2, d, N, BHkv, 64, 64) ||
      !encode_3d(&a.tmV64, v, dt, 2, d, N, BHkv, 64, 64) ||
      !encode_3d(&a.tmDO64, dout, dt, 2, d, N, BH, 64, 64))
    return ATTN_ERR_CUDA;
  BwdParams& p = a.params;
  p.q = q;
  p.k = k;
  p.v = v;
  p.o = o;
  p.dout = dout;
  p.lse = lse;
  p.dq = dq;
  p.dk = dk;
  p.dv = dv;
  p.delta = static_cast<float*>(workspace);
  p.status = di->status;
  p.BH = (int)BH;
  p.BHkv = (int)BHkv;
  p.heads = H;
  p.heads_kv = Hkv;
  p.group = H / Hkv;
  p.N = N;
  p.n_qtiles = (N + 127) / 128;
  p.n_kblocks = (N + 127) / 128;
  p.scale = scale;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.wait_limit_ns = g_wait_limit_ns.load();
  p.sched = reinterpret_cast<int*>(static_cast<char*>(workspace) + bwd_delta_bytes(B, H, N));
  // Only the dK/dV kernel's order is blocked by heads: blocking the wide dQ
  // kernel's (K_j, V_j streamed 64 keys at a time) measured slower at d = 192
  // (2.61 against 2.68 ms for the backward) and the same at d = 256.
  const double head_bytes = (double)N * d * 4.0;  // two streamed 16-bit tensors of a head
  p.head_block = bwd_head_block(head_bytes * p.group, p.BHkv);
  p.head_block_q = p.BH;
  a.num_sms = di->num_sms;
  a.stream = static_cast<cudaStream_t>(stream);
  a.causal = causal != 0;
  a.bf16 = dtype == ATTN_BF16;
  a.d = d;
  return launch_result(launch_bwd_wide(a));
}

// The backward pass; with cu_seqlens the packed variable-length layout of
// fwd_impl (dq like q, dk / dv like k / v).
attn_status bwd_impl(const void* q, const void* k, const void* v, const void* o,
                     const void* dout, const float* lse, void* dq, void* dk, void* dv,
                     void* workspace, size_t workspace_bytes, int B, int H, int Hkv, int N,
                     int d, int causal, float scale, attn_dtype dtype, void* stream,
                     const int* cu_seqlens = nullptr, int max_seqlen = 0) {
  const bool varlen = cu_seqlens != nullptr;
  if (varlen && !varlen_args_ok(cu_seqlens, B, max_seqlen, N)) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(dout) ||
      !aligned16(lse) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv))
    return ATTN_ERR_INVALID_ARG;
  if (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & 255) != 0)
    return ATTN_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return ATTN_ERR_INVALID_ARG;
  if (dtype != ATTN_F16 && dtype != ATTN_BF16) return ATTN_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !std::isfinite(scale)) return ATTN_ERR_INVALID_ARG;
  if (B < 1 || H < 1 || N < 1) return ATTN_ERR_INVALID_ARG;
  if (Hkv < 1 || H % Hkv != 0) return ATTN_ERR_INVALID_ARG;
  if (!head_dim_ok(d)) return ATTN_ERR_UNSUPPORTED;
  // the wide head dims: dense or grouped heads only
  if (d > 128 && varlen) return ATTN_ERR_UNSUPPORTED;
  if (!shape_ok(B, H, N, d)) return ATTN_ERR_INVALID_ARG;
  if (workspace_bytes < attn_bwd_workspace_bytes(varlen ? 1 : B, H, N, d))
    return ATTN_ERR_INVALID_ARG;
  DeviceInfo* di = nullptr;
  attn_status st = device_info(&di);
  if (st != ATTN_OK) return st;
  if (d > 128)
    return bwd_wide_impl(di, q, k, v, o, dout, lse, dq, dk, dv, workspace, B, H, Hkv, N, d,
                         causal, scale, dtype, stream);
  BwdLaunch a;
  const CUtensorMapDataType dt =
      dtype == ATTN_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  const int64_t BH = (int64_t)B * H, BHkv = (int64_t)B * Hkv;
  const int64_t zq = varlen ? H : BH, zkv = varlen ? Hkv : BHkv;
  if (!encode_3d(&a.tmQ, q, dt, 2, d, N, zq, 64, 128) ||
      !encode_3d(&a.tmK, k, dt, 2, d, N, zkv, 64, 128) ||
      !encode_3d(&a.tmV, v, dt, 2, d, N, zkv, 64, 128) ||
      !encode_3d(&a.tmDO, dout, dt, 2, d, N, zq, 64, 128))
    return ATTN_ERR_CUDA;
  BwdParams& p = a.params;
  p.q = q;
  p.k = k;
  p.v = v;
  p.o = o;
  p.dout = dout;
  p.lse = lse;
  p.dq = dq;
  p.dk = dk;
  p.dv = dv;
  p.delta = static_cast<float*>(workspace);
  p.status = di->status;
  p.BH = (int)BH;
  p.BHkv = (int)BHkv;
  p.heads = H;
  p.heads_kv = Hkv;
  p.group = H / Hkv;
  p.N = N;
  p.n_qtiles = (N + 127) / 128;
  p.n_kblocks = (N + 127) / 128;
  if (varlen) {
    p.cu_seqlens = cu_seqlens;
    p.max_seqlen = max_seqlen;
    p.n_qtiles = (max_seqlen + 127) / 128;
    p.n_kblocks = p.n_qtiles;
    if ((int64_t)p.BH * p.n_qtiles > 0x7FFFFFFF) return ATTN_ERR_INVALID_ARG;
  }
  p.scale = scale;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.wait_limit_ns = g_wait_limit_ns.load();
  p.sched = reinterpret_cast<int*>(static_cast<char*>(workspace) +
                                   bwd_delta_bytes(varlen ? 1 : B, H, N));
  // A head's two streamed tensors (rows x padded d, 16-bit): dK/dV units
  // stream Q and dO of a key/value head's whole group, dQ units K and V,
  // which the group's query heads share.
  const double head_bytes = (double)(varlen ? max_seqlen : N) * ((d + 63) / 64 * 64) * 4.0;
  p.head_block = bwd_head_block(head_bytes * p.group, p.BHkv);
  p.head_block_q = bwd_head_block(head_bytes / p.group, p.BH);
  a.num_sms = di->num_sms;
  a.stream = static_cast<cudaStream_t>(stream);
  a.causal = causal != 0;
  a.bf16 = dtype == ATTN_BF16;
  a.d = d;
  if (varlen) {
    cudaError_t e = launch_varlen_check(cu_seqlens, B, N, max_seqlen, di->status, a.stream);
    if (e != cudaSuccess) return launch_result(e);
  }
  cudaError_t e = launch_bwd(a);
  return launch_result(e);
}

}  // namespace

extern "C" {

attn_status attn_bwd_gqa(const void* q, const void* k, const void* v, const void* o,
                         const void* dout, const float* lse, void* dq, void* dk, void* dv,
                         void* workspace, size_t workspace_bytes, int B, int H, int Hkv, int N,
                         int d, int causal, float scale, attn_dtype dtype, void* stream) {
  return bwd_impl(q, k, v, o, dout, lse, dq, dk, dv, workspace, workspace_bytes, B, H, Hkv, N, d,
                  causal, scale, dtype, stream);
}

attn_status attn_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse,
                            const int* cu_seqlens, int n_seq, int max_seqlen, int total, int Hq,
                            int Hkv, int d, int causal, float scale, attn_dtype dtype,
                            void* stream) {
  if (cu_seqlens == nullptr) return ATTN_ERR_INVALID_ARG;
  return fwd_impl(q, k, v, o, lse, 1, n_seq, Hq, Hkv, total, d, causal, scale, dtype, stream,
                  cu_seqlens, max_seqlen);
}

attn_status attn_bwd_varlen(const void* q, const void* k, const void* v, const void* o,
                            const void* dout, const float* lse, void* dq, void* dk, void* dv,
                            void* workspace, size_t workspace_bytes, const int* cu_seqlens,
                            int n_seq, int max_seqlen, int total, int Hq, int Hkv, int d,
                            int causal, float scale, attn_dtype dtype, void* stream) {
  if (cu_seqlens == nullptr) return ATTN_ERR_INVALID_ARG;
  return bwd_impl(q, k, v, o, dout, lse, dq, dk, dv, workspace, workspace_bytes, n_seq, Hq, Hkv,
                  total, d, causal, scale, dtype, stream, cu_seqlens, max_seqlen);
}

attn_status attn_bwd(const void* q, const void* k, const void* v, const void* o,
                     const void* dout, const float* lse, void* dq, void* dk, void* dv,
                     void* workspace, size_t workspace_bytes, int B, int H, int N, int d,
                     int causal, float scale, attn_dtype dtype, void* stream) {
  return attn_bwd_gqa(q, k, v, o, dout, lse, dq, dk, dv, workspace, workspace_bytes, B, H, H, N,
                      d, causal, scale, dtype, stream);
}

attn_status attn_quantize_fp8(const void* x_bf16, void* x_e4m3, float* scales, int B, int H,
                              int N, int d, int block_rows, const int8_t* hadamard_signs,
                              int write_transposed, void* stream) {
  if (!aligned16(x_bf16) || !aligned16(x_e4m3) || scales == nullptr ||
      (reinterpret_cast<uintptr_t>(scales) & 3) != 0)
    return ATTN_ERR_INVALID_ARG;
  if (block_rows != 64) return ATTN_ERR_UNSUPPORTED;
  if (write_transposed != 0 && write_transposed != 1) return ATTN_ERR_INVALID_ARG;
  if (B < 1 || H < 1 || N < 1) return ATTN_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED;
  if (!shape_ok(B, H, N, d)) return ATTN_ERR_INVALID_ARG;
  if (write_transposed && (N % 16) != 0) return ATTN_ERR_INVALID_ARG;
  DeviceInfo* di = nullptr;
  attn_status st = device_info(&di);
  if (st != ATTN_OK) return st;
  QuantLaunch a;
  a.x = x_bf16;
  a.out = x_e4m3;
  a.scales = scales;
  a.signs = hadamard_signs;
  a.BH = B * H;
  a.N = N;
  a.d = d;
  a.transposed = write_transposed != 0;
  a.stream = static_cast<cudaStream_t>(stream);
  cudaError_t e = launch_quantize(a);
  return launch_result(e);
}

attn_status attn_fwd_fp8(const void* q8, const void* k8, const void* v8t, const float* q_scale,
                         const float* k_scale, const float* v_scale, void* o, float* lse, int B,
                         int H, int N, int d, int causal, float scale, void* stream) {
  if (!aligned16(q8) || !aligned16(k8) || !aligned16(v8t) || !aligned16(o) || !aligned16(lse))
    return ATTN_ERR_INVALID_ARG;
  if (q_scale == nullptr || k_scale == nullptr || v_scale == nullptr) return ATTN_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return ATTN_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !std::isfinite(scale)) return ATTN_ERR_INVALID_ARG;
  if (B < 1 || H < 1 || N < 1) return ATTN_ERR_INVALID_ARG;
  if (d != 128) return ATTN_ERR_UNSUPPORTED;
  if (!shape_ok(B, H, N, d) || (N % 16) != 0) return ATTN_ERR_INVALID_ARG;
  DeviceInfo* di = nullptr;
  attn_status st = device_info(&di);
  if (st != ATTN_OK) return st;
  Fp8FwdLaunch a;
  const int64_t BH = (int64_t)B * H;
  if (!encode_3d(&a.tmQ, q8, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, d, N, BH, 128, 128) ||
      !encode_3d(&a.tmK, k8, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, d, N, BH, 128, 128) ||
      !encode_3d(&a.tmVt, v8t, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, N, d, BH, 128, 128))
    return ATTN_ERR_CUDA;
  fill_fwd_common(&a.base, di, B, H, N, scale, stream, o, lse);
  a.q_scale = q_scale;
  a.k_scale = k_scale;
  a.v_scale = v_scale;
  a.causal = causal != 0;
  cudaError_t e = launch_fwd_fp8(a);
  return launch_result(e);
}

attn_status attn_poll_device_status(void* stream, uint32_t* detail) {
  DeviceInfo* di = nullptr;
  attn_status st = device_info(&di);
  if (st != ATTN_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return ATTN_ERR_CUDA;
  uint32_t word = 0;
  if (cudaMemcpy(&word, di->status, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess)
    return ATTN_ERR_CUDA;
  if (detail != nullptr) *detail = word;
  if (word != 0) {
    const uint32_t zero = 0;
    if (cudaMemcpy(di->status, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess)
      return ATTN_ERR_CUDA;
    const uint32_t code = word & 0xFF;
    if (code == kStatusTimeout) return ATTN_ERR_TIMEOUT;
    return code == ATTN_ERR_INVALID_ARG ? ATTN_ERR_INVALID_ARG : ATTN_ERR_CUDA;
  }
  return ATTN_OK;
}

}  // extern "C"

namespace attn {
namespace {

// One thread waits on an mbarrier that nothing arrives at; the bounded wait
// must give up, record the timeout and return.
__global__ void selftest_wait_kernel(uint32_t* status, unsigned long long limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(smem_u32(&bar), 1);
    mbar_fence_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    Watchdog wd{status, &abort_flag, limit_ns};
    mbar_wait(smem_u32(&bar), 0, wd, 99);
  }
  __syncthreads();
}

}  // namespace
}  // namespace attn

extern "C" attn_status attn_selftest_wait_timeout(uint64_t limit_us, void* stream,
                                                  uint32_t* detail) {
  if (limit_us == 0 || limit_us > 10ull * 1000000ull) return ATTN_ERR_INVALID_ARG;
  DeviceInfo* di = nullptr;
  attn_status st = device_info(&di);
  if (st != ATTN_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  selftest_wait_kernel<<<1, 32, 0, s>>>(di->status, limit_us * 1000ull);
  if (cudaGetLastError() != cudaSuccess) return ATTN_ERR_CUDA;
  return attn_poll_device_status(stream, detail);
}
