/*
 * A plain C client of the attention library: no Python, no torch. It reads
 * bf16 Q, K, V, dO from a raw file, runs the forward and the whole backward
 * (attn_fwd, attn_bwd_preprocess, attn_bwd, attn_bwd_finalize) on a stream of
 * its own, checks every return code and the device status word, and writes
 * O, LSE, dQ, dK, dV to a raw file.
 *
 *   c_abi_client IN OUT B H H_kv N d causal
 *
 * IN holds q [B,H,N,d], k, v [B,H_kv,N,d], do [B,H,N,d] as bf16 bit
 * patterns, back to back. OUT receives o (bf16), lse (fp32), dq, dk, dv
 * (bf16) in that order. tau = 1/sqrt(d), no softcap. Exit status 0 on
 * success.
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>

#include <cuda_runtime_api.h>

#include "attnbwd.h"

#define CHECK_CUDA(x)                                                     \
  do {                                                                    \
    cudaError_t e_ = (x);                                                 \
    if (e_ != cudaSuccess) {                                              \
      fprintf(stderr, "%s: %s\n", #x, cudaGetErrorString(e_));            \
      return 2;                                                           \
    }                                                                     \
  } while (0)

#define CHECK_ATTN(x)                                                     \
  do {                                                                    \
    int r_ = (x);                                                         \
    if (r_ != ATTN_OK) {                                                  \
      fprintf(stderr, "%s: %d (%s)\n", #x, r_, attn_strerror(r_));        \
      return 3;                                                           \
    }                                                                     \
  } while (0)

int main(int argc, char** argv) {
  if (argc != 9) {
    fprintf(stderr, "usage: %s IN OUT B H H_kv N d causal\n", argv[0]);
    return 1;
  }
  const int B = atoi(argv[3]), H = atoi(argv[4]), H_kv = atoi(argv[5]), N = atoi(argv[6]),
            d = atoi(argv[7]), causal = atoi(argv[8]);
  const size_t nq = (size_t)B * H * N * d, nk = (size_t)B * H_kv * N * d, nr = (size_t)B * H * N;
  const float scale = 1.0f / sqrtf((float)d);

  uint16_t* host_in = (uint16_t*)malloc((2 * nq + 2 * nk) * sizeof(uint16_t));
  FILE* f = fopen(argv[1], "rb");
  if (!host_in || !f || fread(host_in, sizeof(uint16_t), 2 * nq + 2 * nk, f) != 2 * nq + 2 * nk) {
    fprintf(stderr, "cannot read %s\n", argv[1]);
    return 1;
  }
  fclose(f);

  void *q, *k, *v, *dO, *o, *dq, *dk, *dv;
  float *lse, *dpsum, *dq_accum;
  CHECK_CUDA(cudaMalloc(&q, nq * 2));
  CHECK_CUDA(cudaMalloc(&k, nk * 2));
  CHECK_CUDA(cudaMalloc(&v, nk * 2));
  CHECK_CUDA(cudaMalloc(&dO, nq * 2));
  CHECK_CUDA(cudaMalloc(&o, nq * 2));
  CHECK_CUDA(cudaMalloc(&dq, nq * 2));
  CHECK_CUDA(cudaMalloc(&dk, nk * 2));
  CHECK_CUDA(cudaMalloc(&dv, nk * 2));
  CHECK_CUDA(cudaMalloc((void**)&lse, nr * 4));
  CHECK_CUDA(cudaMalloc((void**)&dpsum, nr * 4));
  CHECK_CUDA(cudaMalloc((void**)&dq_accum, nq * 4));
  CHECK_CUDA(cudaMemcpy(q, host_in, nq * 2, cudaMemcpyHostToDevice));
  CHECK_CUDA(cudaMemcpy(k, host_in + nq, nk * 2, cudaMemcpyHostToDevice));
  CHECK_CUDA(cudaMemcpy(v, host_in + nq + nk, nk * 2, cudaMemcpyHostToDevice));
  CHECK_CUDA(cudaMemcpy(dO, host_in + nq + 2 * nk, nq * 2, cudaMemcpyHostToDevice));

  cudaStream_t s;
  CHECK_CUDA(cudaStreamCreate(&s));
  CHECK_ATTN(attn_fwd(q, k, v, o, lse, B, H, H_kv, N, d, scale, causal, 0.0f, s));
  CHECK_ATTN(attn_bwd_preprocess(o, dO, dpsum, dq_accum, B, H, N, d, s));
  CHECK_ATTN(attn_bwd(q, k, v, o, dO, lse, dq_accum, dk, dv, B, H, H_kv, N, d, scale, causal,
                      0.0f, dpsum, s));
  CHECK_ATTN(attn_bwd_finalize(dq_accum, dq, scale, B, H, N, d, s));
  int status = 0;
  CHECK_ATTN(attn_device_status(&status, 1, s));
  if (status != ATTN_OK) {
    fprintf(stderr, "device status %d (%s)\n", status, attn_strerror(status));
    return 4;
  }

  const size_t out_bytes = nq * 2 + nr * 4 + nq * 2 + 2 * nk * 2;
  char* host_out = (char*)malloc(out_bytes);
  if (!host_out) return 1;
  size_t at = 0;
  CHECK_CUDA(cudaMemcpy(host_out + at, o, nq * 2, cudaMemcpyDeviceToHost));
  at += nq * 2;
  CHECK_CUDA(cudaMemcpy(host_out + at, lse, nr * 4, cudaMemcpyDeviceToHost));
  at += nr * 4;
  CHECK_CUDA(cudaMemcpy(host_out + at, dq, nq * 2, cudaMemcpyDeviceToHost));
  at += nq * 2;
  CHECK_CUDA(cudaMemcpy(host_out + at, dk, nk * 2, cudaMemcpyDeviceToHost));
  at += nk * 2;
  CHECK_CUDA(cudaMemcpy(host_out + at, dv, nk * 2, cudaMemcpyDeviceToHost));
  f = fopen(argv[2], "wb");
  if (!f || fwrite(host_out, 1, out_bytes, f) != out_bytes) {
    fprintf(stderr, "cannot write %s\n", argv[2]);
    return 1;
  }
  fclose(f);
  cudaStreamDestroy(s);
  printf("ok\n");
  return 0;
}
