/*
 * A C program that uses libfa_gb300.so through include/fa.h alone (no Python,
 * no torch): exact attention forward and backward on a small causal problem
 * with grouped heads, with the CUDA runtime for memory and streams.
 *
 * Checks what holds for any input: every status is FA_OK, O and LSE are
 * finite, each O row lies within the range of the V rows (a convex
 * combination), causal row 0 equals v_0 exactly (it sees only key 0), and the
 * gradients are finite.  Prints "fa_c_client ok" and exits 0 on success.
 *
 * Build: cc fa_c_client.c -I include -I <cuda>/include -L <lib dir> -lfa_gb300
 *        -L <cuda>/lib64 -lcudart -lm
 */
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "fa.h"

static uint16_t to_bf16(float f) {  /* round to nearest even */
  uint32_t u;
  memcpy(&u, &f, 4);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}
static float from_bf16(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}
static float urand(uint32_t* s) { /* xorshift32, uniform in [-1, 1) */
  *s ^= *s << 13;
  *s ^= *s >> 17;
  *s ^= *s << 5;
  return (float)(*s >> 8) / 8388608.0f - 1.0f;
}

#define CHECK_CUDA(x)                                                         \
  do {                                                                        \
    cudaError_t e_ = (x);                                                     \
    if (e_ != cudaSuccess) {                                                  \
      fprintf(stderr, "%s: %s\n", #x, cudaGetErrorString(e_));                \
      return 1;                                                               \
    }                                                                         \
  } while (0)
#define CHECK_FA(x)                                                           \
  do {                                                                        \
    fa_status s_ = (x);                                                       \
    if (s_ != FA_OK) {                                                        \
      fprintf(stderr, "%s: %s\n", #x, fa_strerror(s_));                       \
      return 1;                                                               \
    }                                                                         \
  } while (0)

int main(void) {
  const int B = 2, Hq = 4, Hkv = 2, N = 300, d = 64, causal = 1;
  const float scale = 0.125f;
  const size_t nq = (size_t)B * Hq * N * d, nk = (size_t)B * Hkv * N * d, nl = (size_t)B * Hq * N;
  uint16_t* hq = malloc(nq * 2);
  uint16_t* hk = malloc(nk * 2);
  uint16_t* hv = malloc(nk * 2);
  uint16_t* hdo = malloc(nq * 2);
  uint16_t* ho = malloc(nq * 2);
  uint16_t* hg = malloc(nq * 2);
  float* hl = malloc(nl * 4);
  uint32_t seed = 12345u;
  for (size_t i = 0; i < nq; ++i) hq[i] = to_bf16(urand(&seed));
  for (size_t i = 0; i < nk; ++i) hk[i] = to_bf16(urand(&seed));
  for (size_t i = 0; i < nk; ++i) hv[i] = to_bf16(urand(&seed));
  for (size_t i = 0; i < nq; ++i) hdo[i] = to_bf16(urand(&seed));

  void *q, *k, *v, *o, *dO, *dq, *dk, *dv, *ws;
  float* lse;
  CHECK_CUDA(cudaMalloc(&q, nq * 2));
  CHECK_CUDA(cudaMalloc(&k, nk * 2));
  CHECK_CUDA(cudaMalloc(&v, nk * 2));
  CHECK_CUDA(cudaMalloc(&o, nq * 2));
  CHECK_CUDA(cudaMalloc(&dO, nq * 2));
  CHECK_CUDA(cudaMalloc(&dq, nq * 2));
  CHECK_CUDA(cudaMalloc(&dk, nk * 2));
  CHECK_CUDA(cudaMalloc(&dv, nk * 2));
  CHECK_CUDA(cudaMalloc((void**)&lse, nl * 4));
  const size_t ws_bytes = fa_bwd_workspace_bytes(B, Hq, Hkv, N, d);
  if (ws_bytes == 0) {
    fprintf(stderr, "fa_bwd_workspace_bytes returned 0\n");
    return 1;
  }
  CHECK_CUDA(cudaMalloc(&ws, ws_bytes));
  CHECK_CUDA(cudaMemcpy(q, hq, nq * 2, cudaMemcpyHostToDevice));
  CHECK_CUDA(cudaMemcpy(k, hk, nk * 2, cudaMemcpyHostToDevice));
  CHECK_CUDA(cudaMemcpy(v, hv, nk * 2, cudaMemcpyHostToDevice));
  CHECK_CUDA(cudaMemcpy(dO, hdo, nq * 2, cudaMemcpyHostToDevice));
  cudaStream_t st;
  CHECK_CUDA(cudaStreamCreate(&st));

  CHECK_FA(fa_fwd(q, k, v, o, lse, B, Hq, Hkv, N, d, causal, scale, st));
  CHECK_FA(fa_bwd(q, k, v, o, dO, lse, dq, dk, dv, B, Hq, Hkv, N, d, causal, scale, ws, ws_bytes, st));
  CHECK_CUDA(cudaStreamSynchronize(st));
  CHECK_FA(fa_last_device_status(st, NULL));
  CHECK_CUDA(cudaMemcpy(ho, o, nq * 2, cudaMemcpyDeviceToHost));
  CHECK_CUDA(cudaMemcpy(hl, lse, nl * 4, cudaMemcpyDeviceToHost));

  const int G = Hq / Hkv;
  for (int b = 0; b < B; ++b)
    for (int h = 0; h < Hq; ++h) {
      const int g = h / G;
      for (int c = 0; c < d; ++c) {
        float lo = INFINITY, hi = -INFINITY;
        for (int j = 0; j < N; ++j) {
          const float x = from_bf16(hv[(((size_t)b * Hkv + g) * N + j) * d + c]);
          lo = fminf(lo, x);
          hi = fmaxf(hi, x);
        }
        for (int i = 0; i < N; ++i) {
          const float x = from_bf16(ho[(((size_t)b * Hq + h) * N + i) * d + c]);
          if (!(x >= lo - 1e-2f && x <= hi + 1e-2f)) {
            fprintf(stderr, "O outside the V range at (%d,%d,%d,%d)\n", b, h, i, c);
            return 1;
          }
        }
        /* causal row 0 sees key 0 only: O_0 = v_0 */
        if (ho[(((size_t)b * Hq + h) * N) * d + c] != hv[(((size_t)b * Hkv + g) * N) * d + c]) {
          fprintf(stderr, "causal row 0 differs from v_0 at (%d,%d,%d)\n", b, h, c);
          return 1;
        }
      }
      for (int i = 0; i < N; ++i)
        if (!isfinite(hl[((size_t)b * Hq + h) * N + i])) {
          fprintf(stderr, "non-finite LSE\n");
          return 1;
        }
    }
  void* grads[3] = {dq, dk, dv};
  const size_t counts[3] = {nq, nk, nk};
  for (int t = 0; t < 3; ++t) {
    CHECK_CUDA(cudaMemcpy(hg, grads[t], counts[t] * 2, cudaMemcpyDeviceToHost));
    for (size_t i = 0; i < counts[t]; ++i)
      if (!isfinite(from_bf16(hg[i]))) {
        fprintf(stderr, "non-finite gradient %d\n", t);
        return 1;
      }
  }
  /* An invalid call is rejected with a status, not a crash. */
  if (fa_fwd(q, k, v, o, lse, B, 3, 2, N, d, causal, scale, st) != FA_ERR_BAD_SHAPE) {
    fprintf(stderr, "bad shape not rejected\n");
    return 1;
  }
  printf("fa_c_client ok (library version %d)\n", fa_version());
  return 0;
}
