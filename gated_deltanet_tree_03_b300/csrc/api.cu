// Host side of the C ABI declared in include/gdn_tree.h: argument checks, launch
// configuration and kernel dispatch. Nothing here allocates, synchronises or keeps state.
#include <cstdint>
#include <cstdio>

#include <cuda_runtime.h>

#include "gdn_tree.h"
#include "common.cuh"
#include "commit.cuh"
#include "storeall.cuh"
#include "verify_simt.cuh"

using namespace gdn;

namespace {

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool valid_d(int d) { return d == 32 || d == 64 || d == 128; }

gdn_status check_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return GDN_ECUDA;
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return GDN_ECUDA;
  if (major != 10 || minor != 3) return GDN_EARCH;
  return GDN_OK;
}

gdn_status launch_status() {
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    fprintf(stderr, "gdn_tree: launch failed: %s\n", cudaGetErrorString(e));
    return GDN_ECUDA;
  }
  return GDN_OK;
}

// shared argument checks of the verify family (host side only; nothing is launched here)
gdn_status check_verify_args(const float *ST, const uint16_t *q, const uint16_t *k,
                             const uint16_t *v, const float *beta, const float *g,
                             const int32_t *parent, const int32_t *cu_nodes, int32_t B, int32_t H,
                             int32_t d_k, int32_t d_v, int32_t max_nodes, const float *o,
                             const float *U, const float *G, const int32_t *status) {
  if (B < 0 || H <= 0 || max_nodes < 0) return GDN_EINVAL;
  if (B > 65535 || H > 65535) return GDN_EINVAL;  // grid y / z limits
  if (!valid_d(d_k) || !valid_d(d_v)) return GDN_EINVAL;
  if (max_nodes > kMaxNodes) return GDN_ETOOBIG;
  if (B == 0) return GDN_OK;
  if (!ST || !q || !k || !v || !beta || !g || !parent || !cu_nodes || !o || !U || !G)
    return GDN_EINVAL;
  const void *ptrs[] = {ST, q, k, v, beta, g, parent, cu_nodes, o, U, G};
  for (const void *p : ptrs)
    if (!aligned16(p)) return GDN_EALIGN;
  if (status && !aligned16(status)) return GDN_EALIGN;
  return GDN_OK;
}

gdn_status check_commit_args(const float *ST, const void *a1, const void *a2, const void *a3,
                             const int32_t *parent, const int32_t *cu_nodes, const int32_t *path,
                             const int32_t *path_len, int32_t B, int32_t H, int32_t d_k,
                             int32_t d_v, int32_t max_path, const int32_t *status) {
  if (B < 0 || H <= 0 || max_path < 0) return GDN_EINVAL;
  if (!valid_d(d_k) || !valid_d(d_v)) return GDN_EINVAL;
  if (max_path > kMaxNodes) return GDN_ETOOBIG;
  if (B == 0) return GDN_OK;
  if (!ST || !a1 || !a2 || !a3 || !parent || !cu_nodes || !path_len) return GDN_EINVAL;
  if (max_path > 0 && !path) return GDN_EINVAL;
  const void *ptrs[] = {ST, a1, a2, a3, parent, cu_nodes, path_len};
  for (const void *p : ptrs)
    if (!aligned16(p)) return GDN_EALIGN;
  if (path && !aligned16(path)) return GDN_EALIGN;
  if (status && !aligned16(status)) return GDN_EALIGN;
  return GDN_OK;
}

template <int DK>
gdn_status launch_verify_simt(const VerifyArgs &a, cudaStream_t stream) {
  const int M = a.max_nodes;
  const size_t smem = verify_simt_smem_bytes(M, DK);
  if (cudaFuncSetAttribute(verify_simt_kernel<DK>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           int(smem)) != cudaSuccess)
    return GDN_ECUDA;
  dim3 grid(a.dv / 32, a.H, a.B);
  verify_simt_kernel<DK><<<grid, kThreads, smem, stream>>>(a);
  return launch_status();
}

template <int DK>
gdn_status launch_storeall(const StoreallArgs &a, cudaStream_t stream) {
  dim3 grid(a.dv / 32, a.H, a.B);
  verify_storeall_kernel<DK><<<grid, kThreads, 0, stream>>>(a);
  return launch_status();
}

}  // namespace

extern "C" {

int32_t gdn_abi_version(void) { return 1; }

const char *gdn_status_str(gdn_status s) {
  switch (s) {
    case GDN_OK: return "GDN_OK";
    case GDN_EINVAL: return "GDN_EINVAL: invalid argument";
    case GDN_ETOOBIG: return "GDN_ETOOBIG: more than 64 nodes or path entries per request";
    case GDN_EALIGN: return "GDN_EALIGN: array not 16-byte aligned";
    case GDN_ECUDA: return "GDN_ECUDA: CUDA runtime error";
    case GDN_EARCH: return "GDN_EARCH: device is not sm_103";
  }
  return "GDN_?: unknown status";
}

gdn_status gdn_tree_verify_simt(const float *ST, const uint16_t *q, const uint16_t *k,
                                const uint16_t *v, const float *beta, const float *g,
                                const int32_t *parent, const int32_t *cu_nodes, int32_t B,
                                int32_t H, int32_t d_k, int32_t d_v, int32_t max_nodes, float *o,
                                float *U, float *G, int32_t *status, gdn_stream_t stream) {
  gdn_status st = check_verify_args(ST, q, k, v, beta, g, parent, cu_nodes, B, H, d_k, d_v,
                                    max_nodes, o, U, G, status);
  if (st != GDN_OK || B == 0) return st;
  if ((st = check_device()) != GDN_OK) return st;
  VerifyArgs a{ST, q, k, v, beta, g, parent, cu_nodes, B, H, d_k, d_v, max_nodes, o, U, G, status};
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  switch (d_k) {
    case 32: return launch_verify_simt<32>(a, s);
    case 64: return launch_verify_simt<64>(a, s);
    default: return launch_verify_simt<128>(a, s);
  }
}

gdn_status gdn_tree_verify(const float *ST, const uint16_t *q, const uint16_t *k, const uint16_t *v,
                           const float *beta, const float *g, const int32_t *parent,
                           const int32_t *cu_nodes, int32_t B, int32_t H, int32_t d_k,
                           int32_t d_v, int32_t max_nodes, float *o, float *U, float *G,
                           int32_t *status, gdn_stream_t stream) {
  return gdn_tree_verify_simt(ST, q, k, v, beta, g, parent, cu_nodes, B, H, d_k, d_v, max_nodes,
                              o, U, G, status, stream);
}

gdn_status gdn_tree_commit(float *ST, const float *U, const float *G, const uint16_t *k,
                           const int32_t *parent, const int32_t *cu_nodes, const int32_t *path,
                           const int32_t *path_len, int32_t B, int32_t H, int32_t d_k,
                           int32_t d_v, int32_t max_path, int32_t *status, gdn_stream_t stream) {
  gdn_status st = check_commit_args(ST, U, G, k, parent, cu_nodes, path, path_len, B, H, d_k, d_v,
                                    max_path, status);
  if (st != GDN_OK || B == 0) return st;
  if ((st = check_device()) != GDN_OK) return st;
  CommitArgs a{ST, U, G, k, parent, cu_nodes, path, path_len, B, H, d_k, d_v, max_path, status};
  const size_t smem = commit_smem_bytes(max_path, d_k, d_v);
  if (cudaFuncSetAttribute(commit_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)) !=
      cudaSuccess)
    return GDN_ECUDA;
  const long long nchunk = d_k / commit_rows_per_cta(d_k, d_v);
  const long long blocks = (long long)B * H * nchunk;
  if (blocks > 0x7fffffffLL) return GDN_EINVAL;
  commit_kernel<<<unsigned(blocks), kThreads, smem, reinterpret_cast<cudaStream_t>(stream)>>>(a);
  return launch_status();
}

gdn_status gdn_tree_verify_storeall(const float *ST, const uint16_t *q, const uint16_t *k,
                                    const uint16_t *v, const float *beta, const float *g,
                                    const int32_t *parent, const int32_t *cu_nodes, int32_t B,
                                    int32_t H, int32_t d_k, int32_t d_v, int32_t max_nodes,
                                    float *snapshots, float *o, float *U, float *G,
                                    int32_t *status, gdn_stream_t stream) {
  gdn_status st = check_verify_args(ST, q, k, v, beta, g, parent, cu_nodes, B, H, d_k, d_v,
                                    max_nodes, o, U, G, status);
  if (st != GDN_OK || B == 0) return st;
  if (!snapshots) return GDN_EINVAL;
  if (!aligned16(snapshots)) return GDN_EALIGN;
  if ((st = check_device()) != GDN_OK) return st;
  StoreallArgs a{ST, q, k, v, beta, g, parent, cu_nodes, B, H, d_k, d_v, max_nodes, snapshots, o, U, G, status};
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  switch (d_k) {
    case 32: return launch_storeall<32>(a, s);
    case 64: return launch_storeall<64>(a, s);
    default: return launch_storeall<128>(a, s);
  }
}

gdn_status gdn_tree_commit_storeall(float *ST, const float *snapshots, const int32_t *parent,
                                    const int32_t *cu_nodes, const int32_t *path,
                                    const int32_t *path_len, int32_t B, int32_t H, int32_t d_k,
                                    int32_t d_v, int32_t max_path, int32_t *status,
                                    gdn_stream_t stream) {
  gdn_status st = check_commit_args(ST, snapshots, snapshots, snapshots, parent, cu_nodes, path,
                                    path_len, B, H, d_k, d_v, max_path, status);
  if (st != GDN_OK || B == 0) return st;
  if ((st = check_device()) != GDN_OK) return st;
  StoreallCommitArgs a{ST, snapshots, parent, cu_nodes, path, path_len, B, H, d_k, d_v, max_path, status};
  const int per_cta = kThreads * 4;
  const long long nchunk = (d_k * d_v / 4 + per_cta - 1) / per_cta;
  const long long blocks = (long long)B * H * nchunk;
  if (blocks > 0x7fffffffLL) return GDN_EINVAL;
  commit_storeall_kernel<<<unsigned(blocks), kThreads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(a);
  return launch_status();
}

}  // extern "C"
