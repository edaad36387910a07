// attn_bwd_noalloc: the backward pass for callers that cannot allocate
// device memory.
//
// attn_bwd needs a caller-provided workspace (the fp32 delta vector).  Some
// callers cannot provide one: code running inside a host framework whose
// allocator owns all device memory and hands plugins no raw allocations,
// real-time serving loops where a cudaMalloc (which may synchronise the
// device) is not allowed on the request path, or embedded users with a fixed
// memory plan.  For them this file keeps the workspace in a file-scope device
// array of fixed size, so the call itself allocates nothing.
//
// The array holds kMaxRows query rows of scratch: it is part of the library
// image and occupies that much memory on every GPU that loads the library,
// until the process exits.  All calls share it.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "attn.h"

namespace {

constexpr size_t kMaxRows = 4194304;  // B * H * N of one call
// The workspace attn_bwd expects: delta, fp32 per row (a multiple of 256
// bytes), then 256 bytes of work counters.
constexpr size_t kScratchBytes = kMaxRows * 4 + 256;

static __device__ __align__(256) unsigned char g_bwd_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_bwd_scratch on the current device (looked up once per
// device; in host code the array's name is only a host-side stand-in).
attn_status scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ATTN_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_bwd_scratch) != cudaSuccess || p == nullptr)
      return ATTN_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return ATTN_OK;
}

}  // namespace

extern "C" attn_status attn_bwd_noalloc(const void* q, const void* k, const void* v,
                                        const void* o, const void* dout, const float* lse,
                                        void* dq, void* dk, void* dv, int B, int H, int N, int d,
                                        int causal, float scale, attn_dtype dtype,
                                        void* stream) {
  if (B < 1 || H < 1 || N < 1) return ATTN_ERR_INVALID_ARG;
  if (d != 64 && d != 96 && d != 128 && d != 192 && d != 256) return ATTN_ERR_UNSUPPORTED;
  if ((size_t)B * (size_t)H * (size_t)N > kMaxRows) return ATTN_ERR_INVALID_ARG;
  void* scratch = nullptr;
  const attn_status st = scratch_address(&scratch);
  if (st != ATTN_OK) return st;
  // The array holds the delta vector D and the work counters.  attn_bwd's D
  // pass writes delta[row] for every row < B*H*N and zeroes the counters on
  // this stream before either main kernel reads them, so leftovers of an
  // earlier call are never read.
  return attn_bwd(q, k, v, o, dout, lse, dq, dk, dv, scratch, kScratchBytes, B, H, N, d, causal,
                  scale, dtype, stream);
}
