/* Plain C (C11, for CUDA's runtime header) use of include/vc.h with device work: the caller allocates one
 * send and one receive buffer per rank with the CUDA runtime, copies host
 * data in, runs vc_allreduce with each schedule and vc_broadcast from a
 * non-zero root through the header, and checks every element it copies back
 * against results it computes itself.  AllReduce inputs are small integers
 * stored as fp32, so every association gives the exact sum (hccl article,
 * section "hccl_allreduce接口详解": every rank ends with the elementwise sum).
 * Exit code 0 and "ok" on success; a distinct code for each failure. */
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "vc.h"

#define NR 8

static float value(int r, size_t i) { return (float)((long)((i * 7 + (size_t)r * 13) % 201) - 100); }

int main(void) {
  const size_t count = (1u << 20) + 37; /* ragged: not a multiple of N or of 4 */
  void* d_send[NR];
  void* d_recv[NR];
  float* h = (float*)malloc(count * sizeof(float));
  float* want = (float*)malloc(count * sizeof(float));
  float* got = (float*)malloc(count * sizeof(float));
  cudaStream_t s;
  size_t i;
  int r, k;
  const vc_algo_t algos[5] = {VC_ALGO_RING, VC_ALGO_RHD, VC_ALGO_DBT, VC_ALGO_FUSED, VC_ALGO_AUTO};
  if (!h || !want || !got) return 1;
  if (cudaStreamCreate(&s) != cudaSuccess) return 2;
  for (i = 0; i < count; ++i) {
    float acc = 0.0f;
    for (r = 0; r < NR; ++r) acc += value(r, i);
    want[i] = acc;
  }
  for (r = 0; r < NR; ++r) {
    if (cudaMalloc(&d_send[r], count * sizeof(float)) != cudaSuccess) return 3;
    if (cudaMalloc(&d_recv[r], count * sizeof(float)) != cudaSuccess) return 3;
    for (i = 0; i < count; ++i) h[i] = value(r, i);
    if (cudaMemcpy(d_send[r], h, count * sizeof(float), cudaMemcpyHostToDevice) != cudaSuccess) return 4;
  }
  for (k = 0; k < 5; ++k) {
    for (r = 0; r < NR; ++r)
      if (cudaMemset(d_recv[r], 0xFF, count * sizeof(float)) != cudaSuccess) return 5;
    if (vc_allreduce((const void* const*)d_send, d_recv, NR, count, VC_FLOAT32, VC_SUM, algos[k], (vc_stream_t)s) !=
        VC_SUCCESS) {
      fprintf(stderr, "vc_allreduce: %s\n", vc_last_error());
      return 6;
    }
    if (cudaStreamSynchronize(s) != cudaSuccess) return 7;
    for (r = 0; r < NR; ++r) {
      if (cudaMemcpy(got, d_recv[r], count * sizeof(float), cudaMemcpyDeviceToHost) != cudaSuccess) return 8;
      if (memcmp(got, want, count * sizeof(float)) != 0) {
        fprintf(stderr, "allreduce algo %d rank %d differs\n", (int)algos[k], r);
        return 9;
      }
    }
  }
  /* Broadcast of rank 3's input (int32 bits) to every receive buffer */
  {
    int32_t* src = (int32_t*)h;
    for (i = 0; i < count; ++i) src[i] = (int32_t)(i * 2654435761u);
    if (cudaMemcpy(d_send[3], src, count * 4, cudaMemcpyHostToDevice) != cudaSuccess) return 10;
    if (vc_broadcast(d_send[3], d_recv, NR, count, VC_INT32, 3, VC_ALGO_BINOMIAL, (vc_stream_t)s) != VC_SUCCESS)
      return 11;
    if (cudaStreamSynchronize(s) != cudaSuccess) return 12;
    for (r = 0; r < NR; ++r) {
      if (cudaMemcpy(got, d_recv[r], count * 4, cudaMemcpyDeviceToHost) != cudaSuccess) return 13;
      if (memcmp(got, src, count * 4) != 0) return 14;
    }
  }
  for (r = 0; r < NR; ++r) {
    cudaFree(d_send[r]);
    cudaFree(d_recv[r]);
  }
  cudaStreamDestroy(s);
  free(h);
  free(want);
  free(got);
  printf("ok\n");
  return 0;
}
