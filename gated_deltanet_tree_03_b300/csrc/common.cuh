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

// Serving layout (gdn_layout after the host checks). Default-constructed it is the plain
// layout: request r owns state r, q/k have H heads, no query scale, g and beta given.
struct Serving {
  const int32_t *slot = nullptr;  // [B] state slot per request (-1 = padding request), or null
  int n_slots = 0;                // states in the pool when slot is set
  int grp = 1;                    // value heads per q/k head
  float q_scale = 1.f;            // multiplies every query
  const float *a_raw = nullptr, *b_raw = nullptr, *A_log = nullptr, *dt_bias = nullptr;
};

constexpr int kSkipRequest = -1;  // state_of: padding request
constexpr int kBadSlot = -2;      // state_of: slot outside the pool

// Serving-layout accessors. Every kernel is compiled twice: SV = false for the plain layout,
// where these reduce to compile-time identities and the kernel carries none of the layout's
// indexing, and SV = true for a serving layout.

// Index of request r's state in ST (its pool slot), or kSkipRequest / kBadSlot.
template <bool SV>
__device__ __forceinline__ int state_of(const Serving &L, int r) {
  if constexpr (!SV) {
    return r;
  } else {
    if (L.slot == nullptr) return r;
    const int s = L.slot[r];
    if (s == -1) return kSkipRequest;
    return (s >= 0 && s < L.n_slots) ? s : kBadSlot;
  }
}

// Value heads per q/k head.
template <bool SV>
__device__ __forceinline__ int qk_group(const Serving &L) {
  if constexpr (SV) return L.grp;
  else return 1;
}

// Factor on every query (applied to the outputs, which are linear in q).
template <bool SV>
__device__ __forceinline__ float query_scale(const Serving &L) {
  if constexpr (SV) return L.q_scale;
  else return 1.f;
}

// Gate g and write strength b of node row th (= node * H + h): the given arrays, or formed from
// the gate pre-activations as g = -exp(A_log[h]) softplus(a_raw + dt_bias[h]), b = sigmoid(b_raw).
template <bool SV>
__device__ __forceinline__ void gate_beta(const Serving &L, const float *g, const float *beta, size_t th, int h,
                                          float &gg, float &bb) {
  if (!SV || L.a_raw == nullptr) {
    gg = g[th];
    bb = beta[th];
    return;
  }
  const float x = L.a_raw[th] + L.dt_bias[h];
  // ln(1 + e^x) equals x to fp32 precision once e^-x is below half an ulp of x
  const float sp = x > 20.f ? x : log1pf(expf(x));
  gg = -expf(L.A_log[h]) * sp;
  bb = 1.f / (1.f + expf(-L.b_raw[th]));
}

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

// Loads the request's parents and (for head h) gates/betas (given or formed under the serving
// layout L), checks parent[t] in [-1, t-1] and builds ancestor masks and cumulative log-gates.
// Every thread of the block must call it.
// Returns false (for all threads) if the tree is malformed; the caller then writes nothing.
template <bool SV>
__device__ __forceinline__ bool analyse_tree(TreeSmem &ts, const int32_t *__restrict__ parent,
                                             const float *__restrict__ g,
                                             const float *__restrict__ beta, int t0, int n, int h,
                                             int H, const Serving &L) {
  const int tid = threadIdx.x;
  int bad = 0;
  if (tid < n) {
    const int p = parent[t0 + tid];
    bad = (p < -1 || p >= tid);
    ts.par[tid] = p;
    gate_beta<SV>(L, g, beta, size_t(t0 + tid) * H + h, h, ts.g[tid], ts.beta[tid]);
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
