/* Host cost of the library's calls, measured from plain C (no Python in the loop).
 *
 * For two single-request shapes - a 6-node root-branch tree (streaming verify kernel) and a
 * 32-node chain (tensor-core verify kernel), 48 heads, d_k = d_v = 128 - it times:
 *   host_us_verify / host_us_commit : wall time per call on the host, calls issued back to back
 *                                     (the GPU runs behind; no synchronisation inside the loop);
 *   eager_us_step                   : one verify + commit step, issued and completed, averaged
 *                                     over many steps (CUDA events around the whole loop);
 *   graph_us_step                   : the same step captured once in a CUDA graph and replayed.
 * Prints one JSON object per shape and exits 0, or prints the failing call and exits 1.
 * Built and run by tests/test_c_abi.py on a GPU. */
#define _POSIX_C_SOURCE 199309L
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>
#include <time.h>

#include <cuda_runtime.h>

#include "gdn_tree.h"

#define CK(x)                                                             \
  do {                                                                    \
    cudaError_t e_ = (x);                                                 \
    if (e_ != cudaSuccess) {                                              \
      fprintf(stderr, "%s:%d %s\n", __FILE__, __LINE__, cudaGetErrorString(e_)); \
      exit(1);                                                            \
    }                                                                     \
  } while (0)
#define GK(x)                                                             \
  do {                                                                    \
    gdn_status s_ = (x);                                                  \
    if (s_ != GDN_OK) {                                                   \
      fprintf(stderr, "%s:%d %s\n", __FILE__, __LINE__, gdn_status_str(s_)); \
      exit(1);                                                            \
    }                                                                     \
  } while (0)

static double now_us(void) {
  struct timespec ts;
  clock_gettime(CLOCK_MONOTONIC, &ts);
  return ts.tv_sec * 1e6 + ts.tv_nsec * 1e-3;
}

static void *dev_zero(size_t bytes) {
  void *p = NULL;
  CK(cudaMalloc(&p, bytes < 16 ? 16 : bytes));
  CK(cudaMemset(p, 0, bytes < 16 ? 16 : bytes));
  return p;
}

static void *dev_copy(const void *host, size_t bytes) {
  void *p = dev_zero(bytes);
  CK(cudaMemcpy(p, host, bytes, cudaMemcpyHostToDevice));
  return p;
}

static void run_shape(const char *name, const int32_t *parent_h, int n, int max_nodes) {
  const int B = 1, H = 48, D = 128, T = n;
  const int32_t cu_h[2] = {0, n};
  const int32_t path_h[1] = {0};
  const int32_t path_len_h[1] = {1};
  float *ST = (float *)dev_zero((size_t)B * H * D * D * 4);
  uint16_t *q = (uint16_t *)dev_zero((size_t)T * H * D * 2);
  uint16_t *k = (uint16_t *)dev_zero((size_t)T * H * D * 2);
  uint16_t *v = (uint16_t *)dev_zero((size_t)T * H * D * 2);
  float *beta = (float *)dev_zero((size_t)T * H * 4);
  float *g = (float *)dev_zero((size_t)T * H * 4);
  int32_t *parent = (int32_t *)dev_copy(parent_h, (size_t)n * 4);
  int32_t *cu = (int32_t *)dev_copy(cu_h, sizeof cu_h);
  int32_t *path = (int32_t *)dev_copy(path_h, sizeof path_h);
  int32_t *path_len = (int32_t *)dev_copy(path_len_h, sizeof path_len_h);
  float *o = (float *)dev_zero((size_t)T * H * D * 4);
  float *U = (float *)dev_zero((size_t)T * H * D * 4);
  float *G = (float *)dev_zero((size_t)T * H * 4);
  int32_t *status = (int32_t *)dev_zero(16);
  cudaStream_t s;
  CK(cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking));
  gdn_stream_t gs = (gdn_stream_t)s;

#define VERIFY() \
  gdn_tree_verify(ST, q, k, v, beta, g, parent, cu, B, H, T, D, D, max_nodes, o, U, G, status, gs)
#define COMMIT() gdn_tree_commit(ST, U, G, k, parent, cu, path, path_len, B, H, T, D, D, 1, status, gs)

  for (int i = 0; i < 20; ++i) {  /* first calls: device properties, kernel attributes */
    GK(VERIFY());
    GK(COMMIT());
  }
  CK(cudaStreamSynchronize(s));

  /* host cost: bursts short enough that the launch queue never fills (a full queue would make
   * the host wait for the GPU); the best of several bursts */
  const int NH = 128, N = 2000;
  double host_verify = 1e30, host_commit = 1e30;
  for (int rep = 0; rep < 8; ++rep) {
    double t0 = now_us();
    for (int i = 0; i < NH; ++i) GK(VERIFY());
    const double tv = (now_us() - t0) / NH;
    CK(cudaStreamSynchronize(s));
    t0 = now_us();
    for (int i = 0; i < NH; ++i) GK(COMMIT());
    const double tc = (now_us() - t0) / NH;
    CK(cudaStreamSynchronize(s));
    if (tv < host_verify) host_verify = tv;
    if (tc < host_commit) host_commit = tc;
  }

  cudaEvent_t e0, e1;
  CK(cudaEventCreate(&e0));
  CK(cudaEventCreate(&e1));
  CK(cudaEventRecord(e0, s));
  for (int i = 0; i < N; ++i) {
    GK(VERIFY());
    GK(COMMIT());
  }
  CK(cudaEventRecord(e1, s));
  CK(cudaEventSynchronize(e1));
  float eager_ms = 0.f;
  CK(cudaEventElapsedTime(&eager_ms, e0, e1));

  cudaGraph_t graph;
  cudaGraphExec_t exec;
  CK(cudaStreamBeginCapture(s, cudaStreamCaptureModeThreadLocal));
  GK(VERIFY());
  GK(COMMIT());
  CK(cudaStreamEndCapture(s, &graph));
  CK(cudaGraphInstantiate(&exec, graph, 0));
  for (int i = 0; i < 20; ++i) CK(cudaGraphLaunch(exec, s));
  CK(cudaEventRecord(e0, s));
  for (int i = 0; i < N; ++i) CK(cudaGraphLaunch(exec, s));
  CK(cudaEventRecord(e1, s));
  CK(cudaEventSynchronize(e1));
  float graph_ms = 0.f;
  CK(cudaEventElapsedTime(&graph_ms, e0, e1));

  int32_t st_h[4];
  CK(cudaMemcpy(st_h, status, sizeof st_h, cudaMemcpyDeviceToHost));
  if (st_h[0] != 0) {
    fprintf(stderr, "%s: device status %d\n", name, st_h[0]);
    exit(1);
  }
  printf("{\"shape\": \"%s\", \"host_us_verify\": %.3f, \"host_us_commit\": %.3f, \"eager_us_step\": %.3f, "
         "\"graph_us_step\": %.3f}\n",
         name, host_verify, host_commit, eager_ms * 1e3 / N, graph_ms * 1e3 / N);
  CK(cudaGraphExecDestroy(exec));
  CK(cudaGraphDestroy(graph));
  CK(cudaEventDestroy(e0));
  CK(cudaEventDestroy(e1));
  CK(cudaStreamDestroy(s));
  void *bufs[] = {ST, q, k, v, beta, g, parent, cu, path, path_len, o, U, G, status};
  for (size_t i = 0; i < sizeof bufs / sizeof bufs[0]; ++i) CK(cudaFree(bufs[i]));
#undef VERIFY
#undef COMMIT
}

int main(void) {
  const int32_t rootbranch[6] = {-1, 0, 0, 0, 1, 2};
  int32_t chain[32];
  for (int i = 0; i < 32; ++i) chain[i] = i - 1;
  run_shape("rootbranch6_B1", rootbranch, 6, 6);
  run_shape("chain32_B1", chain, 32, 32);
  return 0;
}
