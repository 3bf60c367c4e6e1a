/*
 * A plain-C caller of the fused LM-head library (no Python, no torch): it
 * allocates device buffers with the CUDA runtime, fills them with a small
 * synthetic problem, runs lmhead_fwd and lmhead_bwd through the C ABI and
 * checks properties every result must have -- logprob <= 0,
 * 0 <= entropy <= log V, zeros on skipped rows, and dW columns summing to ~0
 * (every row's logit gradient sums to zero over the vocabulary).
 * Exit status 0 on success.
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime.h>

#include "lmhead.h"

#define CHECK_CUDA(x)                                                        \
  do {                                                                       \
    cudaError_t e_ = (x);                                                    \
    if (e_ != cudaSuccess) {                                                 \
      fprintf(stderr, "CUDA error %s at line %d\n", cudaGetErrorString(e_), __LINE__); \
      return 2;                                                              \
    }                                                                        \
  } while (0)

#define CHECK_LM(x)                                                          \
  do {                                                                       \
    lmhead_status s_ = (x);                                                  \
    if (s_ != LMHEAD_OK) {                                                   \
      fprintf(stderr, "lmhead error: %s at line %d\n", lmhead_strerror(s_), __LINE__); \
      return 3;                                                              \
    }                                                                        \
  } while (0)

static uint16_t to_bf16(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  u += 0x7FFFu + ((u >> 16) & 1u); /* round to nearest even */
  return (uint16_t)(u >> 16);
}

static float uniform(uint64_t* s) { /* xorshift64*, in [-1, 1) */
  *s ^= *s >> 12;
  *s ^= *s << 25;
  *s ^= *s >> 27;
  return (float)((*s * 2685821657736338717ull) >> 40) / (float)(1 << 23) - 1.0f;
}

int main(void) {
  const int64_t N = 1000;
  const int H = 256, V = 3000;
  uint64_t seed = 12345;
  uint16_t* h = malloc(N * H * 2);
  uint16_t* w = malloc((size_t)V * H * 2);
  int64_t* y = malloc(N * 8);
  uint8_t* keep = malloc(N);
  float* g = malloc(N * 4);
  for (int64_t i = 0; i < N * H; ++i) h[i] = to_bf16(uniform(&seed));
  for (int64_t i = 0; i < (int64_t)V * H; ++i) w[i] = to_bf16(0.1f * uniform(&seed));
  for (int64_t i = 0; i < N; ++i) {
    y[i] = (int64_t)((uniform(&seed) + 1.0f) * 0.5f * V) % V;
    keep[i] = uniform(&seed) > 0.0f;
    g[i] = uniform(&seed);
  }
  void *dh, *dw, *dy, *dkeep, *dg, *dlp, *dent, *dlse, *ddh, *ddw, *ws;
  size_t wsb = lmhead_workspace_size(N, H, V, 1, 0);
  CHECK_CUDA(cudaMalloc(&dh, N * H * 2));
  CHECK_CUDA(cudaMalloc(&dw, (size_t)V * H * 2));
  CHECK_CUDA(cudaMalloc(&dy, N * 8));
  CHECK_CUDA(cudaMalloc(&dkeep, N));
  CHECK_CUDA(cudaMalloc(&dg, N * 4));
  CHECK_CUDA(cudaMalloc(&dlp, N * 4));
  CHECK_CUDA(cudaMalloc(&dent, N * 4));
  CHECK_CUDA(cudaMalloc(&dlse, N * 4));
  CHECK_CUDA(cudaMalloc(&ddh, N * H * 2));
  CHECK_CUDA(cudaMalloc(&ddw, (size_t)V * H * 4));
  CHECK_CUDA(cudaMalloc(&ws, wsb));
  CHECK_CUDA(cudaMemcpy(dh, h, N * H * 2, cudaMemcpyHostToDevice));
  CHECK_CUDA(cudaMemcpy(dw, w, (size_t)V * H * 2, cudaMemcpyHostToDevice));
  CHECK_CUDA(cudaMemcpy(dy, y, N * 8, cudaMemcpyHostToDevice));
  CHECK_CUDA(cudaMemcpy(dkeep, keep, N, cudaMemcpyHostToDevice));
  CHECK_CUDA(cudaMemcpy(dg, g, N * 4, cudaMemcpyHostToDevice));

  CHECK_LM(lmhead_fwd(dh, dw, dy, dkeep, N, H, V, 1, dlp, dent, dlse, 0, ws, wsb, NULL));
  CHECK_LM(lmhead_bwd(dh, dw, dy, dkeep, N, H, V, dlse, dent, dg, NULL, ddh, ddw, 0, 0, ws, wsb,
                      NULL));
  {
    /* a device-side error (a bad target, a pipeline wait that ran out) is
       reported here; on a timeout the record names the wait that gave up */
    const lmhead_status st = lmhead_get_status(ws, NULL);
    if (st != LMHEAD_OK) {
      const int32_t rec = lmhead_get_timeout_record(ws, NULL);
      fprintf(stderr, "device status: %s (timeout record: site %d, cta %d)\n",
              lmhead_strerror(st), rec > 0 ? rec >> 24 : 0, rec > 0 ? rec & 0xFFFFFF : 0);
      return 3;
    }
  }

  float* lp = malloc(N * 4);
  float* ent = malloc(N * 4);
  float* dW = malloc((size_t)V * H * 4);
  CHECK_CUDA(cudaMemcpy(lp, dlp, N * 4, cudaMemcpyDeviceToHost));
  CHECK_CUDA(cudaMemcpy(ent, dent, N * 4, cudaMemcpyDeviceToHost));
  CHECK_CUDA(cudaMemcpy(dW, ddw, (size_t)V * H * 4, cudaMemcpyDeviceToHost));
  int bad = 0, kept = 0;
  for (int64_t i = 0; i < N; ++i) {
    if (keep[i]) {
      ++kept;
      if (!(lp[i] <= 1e-5f) || !(ent[i] >= -1e-5f) || !(ent[i] <= logf((float)V) + 1e-4f)) ++bad;
    } else if (lp[i] != 0.0f || ent[i] != 0.0f) {
      ++bad;
    }
  }
  double worst = 0.0, scale = 0.0;
  for (int k = 0; k < H; ++k) {
    double s = 0.0, a = 0.0;
    for (int v = 0; v < V; ++v) {
      s += dW[(size_t)v * H + k];
      a += fabs(dW[(size_t)v * H + k]);
    }
    if (fabs(s) > worst) worst = fabs(s);
    if (a > scale) scale = a;
  }
  printf("kept %d of %lld rows, %d bad rows, max |column sum of dW| %.3g (scale %.3g)\n", kept,
         (long long)N, bad, worst, scale);
  return (bad == 0 && worst <= 1e-3 * scale) ? 0 : 1;
}
