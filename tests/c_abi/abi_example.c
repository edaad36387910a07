/*
 * The C ABI used from plain C (no Python): a causal fp16 forward pass of one
 * head, [1,1,N,64], on the default stream.  Causal query row 0 sees only key
 * 0, so its output row equals V's row 0 and its LSE equals scale * q0 . k0;
 * the program checks both and that every output is finite; decoding the last
 * position with attn_fwd_kv (one query against the whole sequence as a
 * key/value cache) must give the last output row and LSE; then it prints OK.
 * Build: cc -std=c99 -I include abi_example.c -L <dir of libattn.so> -lattn
 *        -L <cuda>/lib64 -lcudart -lm
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "attn.h"

/* From the CUDA runtime (declared here so that no CUDA header is needed). */
extern int cudaMalloc(void** p, size_t n);
extern int cudaFree(void* p);
extern int cudaMemcpy(void* dst, const void* src, size_t n, int kind);
#define H2D 1
#define D2H 2

/* IEEE half <-> float for normal values in the range used here. */
static uint16_t to_half(float f) {
  uint32_t x;
  memcpy(&x, &f, 4);
  uint32_t sign = (x >> 16) & 0x8000u;
  int32_t e = (int32_t)((x >> 23) & 0xFF) - 127 + 15;
  uint32_t m = (x >> 13) & 0x3FFu;
  if (e <= 0) return (uint16_t)sign;
  return (uint16_t)(sign | ((uint32_t)e << 10) | m);
}
static float from_half(uint16_t h) {
  uint32_t sign = (uint32_t)(h & 0x8000u) << 16;
  uint32_t e = (h >> 10) & 0x1F, m = h & 0x3FFu;
  uint32_t x = e == 0 ? sign : (sign | ((e - 15 + 127) << 23) | (m << 13));
  float f;
  memcpy(&f, &x, 4);
  return f;
}

int main(void) {
  enum { N = 200, D = 64 };
  const size_t elems = (size_t)N * D;
  uint16_t* host[3];
  void* dev[4];
  float* lse_d;
  unsigned seed = 12345u;
  for (int t = 0; t < 3; ++t) {
    host[t] = (uint16_t*)malloc(elems * 2);
    for (size_t i = 0; i < elems; ++i) {
      seed = seed * 1664525u + 1013904223u;
      host[t][i] = to_half(((float)(seed >> 9) / 8388608.0f - 0.5f) * 2.0f);
    }
  }
  for (int t = 0; t < 4; ++t)
    if (cudaMalloc(&dev[t], elems * 2) != 0) return 2;
  if (cudaMalloc((void**)&lse_d, N * sizeof(float)) != 0) return 2;
  for (int t = 0; t < 3; ++t)
    if (cudaMemcpy(dev[t], host[t], elems * 2, H2D) != 0) return 2;
  const float scale = 0.125f;
  attn_status st = attn_fwd(dev[0], dev[1], dev[2], dev[3], lse_d, 1, 1, N, D, 1, scale,
                            ATTN_F16, NULL);
  if (st != ATTN_OK) {
    printf("attn_fwd: %s\n", attn_status_string(st));
    return 1;
  }
  uint32_t detail = 0;
  st = attn_poll_device_status(NULL, &detail);
  if (st != ATTN_OK) {
    printf("device status: %s (0x%x)\n", attn_status_string(st), detail);
    return 1;
  }
  uint16_t* o = (uint16_t*)malloc(elems * 2);
  float lse[N];
  if (cudaMemcpy(o, dev[3], elems * 2, D2H) != 0) return 2;
  if (cudaMemcpy(lse, lse_d, sizeof(lse), D2H) != 0) return 2;
  double dot = 0.0;
  for (int c = 0; c < D; ++c) dot += (double)from_half(host[0][c]) * from_half(host[1][c]);
  int bad = 0;
  for (int c = 0; c < D; ++c)
    if (o[c] != host[2][c]) ++bad;
  if (fabs(lse[0] - scale * dot) > 1e-3) ++bad;
  for (size_t i = 0; i < elems; ++i)
    if (!isfinite(from_half(o[i]))) ++bad;
  for (int i = 0; i < N; ++i)
    if (!isfinite(lse[i])) ++bad;
  /* Decoding the last position against the whole sequence as a key/value
   * cache (Nq = 1, Nk = N, causal) gives the forward's last row. */
  void* o1_d = NULL;
  float* lse1_d = NULL;
  if (cudaMalloc(&o1_d, D * 2) != 0 || cudaMalloc((void**)&lse1_d, 16) != 0) return 2;
  const uint16_t* q_last = (const uint16_t*)dev[0] + (size_t)(N - 1) * D;
  st = attn_fwd_kv(q_last, dev[1], dev[2], o1_d, lse1_d, 1, 1, 1, 1, 1, N, D, 1, scale,
                   ATTN_F16, NULL);
  if (st != ATTN_OK) ++bad;
  uint16_t o1[D];
  float lse1 = 0.f;
  if (cudaMemcpy(o1, o1_d, sizeof(o1), D2H) != 0) return 2;
  if (cudaMemcpy(&lse1, lse1_d, sizeof(lse1), D2H) != 0) return 2;
  for (int c = 0; c < D; ++c)
    if (fabs(from_half(o1[c]) - from_half(o[(size_t)(N - 1) * D + c])) > 1e-2) ++bad;
  if (fabs(lse1 - lse[N - 1]) > 1e-3) ++bad;
  cudaFree(o1_d);
  cudaFree(lse1_d);
  /* an invalid argument is rejected before any launch */
  if (attn_fwd(dev[0], dev[1], dev[2], dev[3], lse_d, 1, 1, N, 80, 1, scale, ATTN_F16, NULL) ==
      ATTN_OK)
    ++bad;
  for (int t = 0; t < 4; ++t) cudaFree(dev[t]);
  cudaFree(lse_d);
  printf(bad ? "FAIL %d\n" : "OK\n", bad);
  return bad ? 1 : 0;
}
