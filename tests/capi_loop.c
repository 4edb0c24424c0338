/* A plain C host loop over the library's chain call, to measure what one C-ABI call costs
 * the host: argument checks, pointer classification, the launches.  Usage:
 *
 *   capi_loop B gamma V iters
 *
 * Inputs are fp32 logits of 0 (p uniform), q uniform, drafts 0, T = 1 and u = 0.5, so
 * every draft is accepted and each call reads every row.  Prints one JSON line:
 * issue_us  -- host time per call, calls issued back to back without waiting;
 * wall_us   -- host time per call including the final synchronisation;
 * device_us -- CUDA-event time per call on the stream, over the same loop.
 * Exit status 0 when every call returned SPECDEC_OK and the outputs are as expected. */
#include <stdio.h>
#include <stdlib.h>
#include <time.h>

#include <cuda_runtime.h>

#include "specdec.h"

static double now_us(void) {
  struct timespec ts;
  clock_gettime(CLOCK_MONOTONIC, &ts);
  return (double)ts.tv_sec * 1e6 + (double)ts.tv_nsec * 1e-3;
}

#define CK(x)                                                           \
  do {                                                                  \
    cudaError_t e_ = (x);                                               \
    if (e_ != cudaSuccess) {                                            \
      fprintf(stderr, "%s: %s\n", #x, cudaGetErrorString(e_));          \
      return 2;                                                         \
    }                                                                   \
  } while (0)

int main(int argc, char** argv) {
  if (argc != 5) {
    fprintf(stderr, "usage: capi_loop B gamma V iters\n");
    return 2;
  }
  const int B = atoi(argv[1]), g = atoi(argv[2]), V = atoi(argv[3]), iters = atoi(argv[4]);
  if (B <= 0 || g <= 0 || V <= 0 || iters <= 0) return 2;
  const size_t rows = (size_t)B * (size_t)(g + 1);
  float *logits, *q, *temps, *u, *p_draft;
  int32_t *drafts, *tokens, *J, *status;
  void* ws;
  const size_t wsb = specdec_chain_workspace_bytes(B, g, V, SPECDEC_F32);
  CK(cudaMalloc((void**)&logits, rows * (size_t)V * sizeof(float)));
  CK(cudaMalloc((void**)&q, (size_t)B * g * (size_t)V * sizeof(float)));
  CK(cudaMalloc((void**)&temps, (size_t)B * sizeof(float)));
  CK(cudaMalloc((void**)&u, rows * sizeof(float)));
  CK(cudaMalloc((void**)&p_draft, (size_t)B * g * sizeof(float)));
  CK(cudaMalloc((void**)&drafts, (size_t)B * g * sizeof(int32_t)));
  CK(cudaMalloc((void**)&tokens, rows * sizeof(int32_t)));
  CK(cudaMalloc((void**)&J, (size_t)B * sizeof(int32_t)));
  CK(cudaMalloc((void**)&status, (size_t)B * sizeof(int32_t)));
  CK(cudaMalloc(&ws, wsb));

  float* hq = (float*)malloc((size_t)B * g * (size_t)V * sizeof(float));
  float* hu = (float*)malloc(rows * sizeof(float));
  float* ht = (float*)malloc((size_t)B * sizeof(float));
  if (!hq || !hu || !ht) return 2;
  for (size_t i = 0; i < (size_t)B * g * (size_t)V; ++i) hq[i] = 1.0f / (float)V;
  for (size_t i = 0; i < rows; ++i) hu[i] = 0.5f;
  for (int b = 0; b < B; ++b) ht[b] = 1.0f;
  CK(cudaMemset(logits, 0, rows * (size_t)V * sizeof(float)));
  CK(cudaMemset(drafts, 0, (size_t)B * g * sizeof(int32_t)));
  CK(cudaMemcpy(q, hq, (size_t)B * g * (size_t)V * sizeof(float), cudaMemcpyHostToDevice));
  CK(cudaMemcpy(u, hu, rows * sizeof(float), cudaMemcpyHostToDevice));
  CK(cudaMemcpy(temps, ht, (size_t)B * sizeof(float), cudaMemcpyHostToDevice));

  cudaStream_t s;
  CK(cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking));
  int bad = 0;
#define CALL()                                                                                      \
  specdec_verify_chain(logits, SPECDEC_F32, q, drafts, temps, u, B, g, V, tokens, J, p_draft, status, \
                       ws, wsb, (void*)s)
  for (int i = 0; i < 50; ++i) bad |= CALL() != SPECDEC_OK;
  CK(cudaStreamSynchronize(s));

  cudaEvent_t e0, e1;
  CK(cudaEventCreate(&e0));
  CK(cudaEventCreate(&e1));
  CK(cudaEventRecord(e0, s));
  const double t0 = now_us();
  for (int i = 0; i < iters; ++i) bad |= CALL() != SPECDEC_OK;
  const double t1 = now_us();
  CK(cudaEventRecord(e1, s));
  CK(cudaStreamSynchronize(s));
  const double t2 = now_us();
  float dev_ms = 0.f;
  CK(cudaEventElapsedTime(&dev_ms, e0, e1));

  /* every draft accepted (p = q uniform, u = 0.5): J = gamma, tokens 0 then the bonus */
  int32_t* hJ = (int32_t*)malloc((size_t)B * sizeof(int32_t));
  int32_t* hs = (int32_t*)malloc((size_t)B * sizeof(int32_t));
  if (!hJ || !hs) return 2;
  CK(cudaMemcpy(hJ, J, (size_t)B * sizeof(int32_t), cudaMemcpyDeviceToHost));
  CK(cudaMemcpy(hs, status, (size_t)B * sizeof(int32_t), cudaMemcpyDeviceToHost));
  for (int b = 0; b < B; ++b) bad |= (hJ[b] != g) || (hs[b] & 0xFF) != 0;

  printf("{\"B\": %d, \"gamma\": %d, \"V\": %d, \"iters\": %d, \"issue_us\": %.3f, \"wall_us\": %.3f, "
         "\"device_us\": %.3f, \"ok\": %s}\n",
         B, g, V, iters, (t1 - t0) / iters, (t2 - t0) / iters, 1e3 * (double)dev_ms / iters, bad ? "false" : "true");
  return bad ? 1 : 0;
}
