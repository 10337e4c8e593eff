// Device helpers shared by the verify / commit kernels.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "gdn_tree.h"

namespace gdn {

constexpr int kMaxNodes = 64;  // one uint64 ancestor mask per node
constexpr int kThreads = 256;

__device__ __forceinline__ float bf16_to_f32(uint16_t b) { return __uint_as_float(uint32_t(b) << 16); }

__device__ __forceinline__ void report(int32_t *status, unsigned bit) {
  if (status != nullptr) atomicOr(reinterpret_cast<int *>(status), int(bit));
}

// Request r's node range [t0, t0 + n) must lie inside the T allocated node rows.
__device__ __forceinline__ bool offsets_ok(int t0, int n, int T) { return t0 >= 0 && n >= 0 && t0 + n <= T; }

// Per-request tree analysis kept in shared memory.
//   anc[t]  : bit j set <=> j is on t's root-to-node path (t itself included)
//   G[t]    : sum of g over that path (cumulative log-gate)
//   beta[t] : b_t
struct TreeSmem {
  unsigned long long anc[kMaxNodes];
  float G[kMaxNodes];
  float beta[kMaxNodes];
  float g[kMaxNodes];
  int par[kMaxNodes];
};

// Loads the request's parents and (for head h) gates/betas, checks parent[t] in [-1, t-1],
// and builds ancestor masks and cumulative log-gates. Every thread of the block must call it.
// Returns false (for all threads) if the tree is malformed; the caller then writes nothing.
__device__ __forceinline__ bool analyse_tree(TreeSmem &ts, const int32_t *__restrict__ parent,
                                             const float *__restrict__ g,
                                             const float *__restrict__ beta, int t0, int n, int h,
                                             int H) {
  const int tid = threadIdx.x;
  int bad = 0;
  if (tid < n) {
    const int p = parent[t0 + tid];
    bad = (p < -1 || p >= tid);
    ts.par[tid] = p;
    ts.g[tid] = g[size_t(t0 + tid) * H + h];
    ts.beta[tid] = beta[size_t(t0 + tid) * H + h];
  }
  if (__syncthreads_or(bad)) return false;
  if (tid < n) {
    // parent indices strictly decrease along the walk, so it ends within tid + 1 steps
    unsigned long long m = 1ull << tid;
    float Gs = ts.g[tid];
    for (int x = ts.par[tid]; x >= 0; x = ts.par[x]) {
      m |= 1ull << x;
      Gs += ts.g[x];
    }
    ts.anc[tid] = m;
    ts.G[tid] = Gs;
  }
  __syncthreads();
  return true;
}

// Accepted-path check for commit: 0 <= L <= min(n, max_path), root first, each next node a
// child of the previous one. Every thread of the block must call it.
__device__ __forceinline__ bool check_path(const int32_t *__restrict__ parent,
                                           const int32_t *__restrict__ path_r, int t0, int n,
                                           int L, int max_path) {
  const int tid = threadIdx.x;
  int bad = (L < 0 || L > n || L > max_path) ? 1 : 0;
  if (!bad && tid < L) {
    const int x = path_r[tid];
    const int prev = tid == 0 ? -1 : path_r[tid - 1];
    bad = (x < 0 || x >= n) || parent[t0 + x] != prev;
  }
  return !__syncthreads_or(bad);
}

}  // namespace gdn
