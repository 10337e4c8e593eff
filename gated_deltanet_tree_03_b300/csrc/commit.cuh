// Commit: rebuild only the accepted path's state, in place (TreeWY, method section: only the
// accepted path's pseudo-values are combined into the next committed state).
//
// With l the accepted path's last node, for every (request, head):
//   ST[kk][c] <- exp(G_l) ST[kk][c] + sum_{j on path} (exp(G_l - G_j) k_j[kk]) u_j[c]
// Each CTA streams one 16 KiB slab of one state (whole rows of d_v): it issues its slab loads
// first, checks the path and stages the path's coefficients while they are in flight, then
// writes each element once. Pure HBM streaming: 8 bytes of state traffic per element.
#pragma once

#include "common.cuh"

namespace gdn {

struct CommitArgs {
  float *ST;
  const float *U, *G;
  const uint16_t *k;
  const int32_t *parent, *cu_nodes, *path, *path_len;
  int B, H, T, dk, dv, max_path;
  int32_t *status;
};

constexpr int kCommitVec = 4;  // float4 per thread per slab

__host__ __device__ inline int commit_rows_per_cta(int dk, int dv) {
  int rows = (kThreads * kCommitVec * 4) / dv;  // 1024 float4 per CTA
  return rows < dk ? rows : dk;
}

__host__ __device__ inline size_t commit_smem_bytes(int max_path, int dk, int dv) {
  return sizeof(float) * size_t(max_path) * (commit_rows_per_cta(dk, dv) + dv);
}

__global__ void __launch_bounds__(kThreads) commit_kernel(CommitArgs a) {
  extern __shared__ __align__(16) float dyn[];
  const int tid = threadIdx.x;
  const int KR = commit_rows_per_cta(a.dk, a.dv);
  const int nchunk = a.dk / KR;
  const int chunk = blockIdx.x % nchunk;
  const int pair = blockIdx.x / nchunk;
  const int h = pair % a.H, r = pair / a.H;
  const int L = a.path_len[r];
  if (L == 0) return;  // keep the committed state
  const int t0 = a.cu_nodes[r];
  const int n = a.cu_nodes[r + 1] - t0;
  if (!offsets_ok(t0, n, a.T)) {
    if (tid == 0 && blockIdx.x % (nchunk * a.H) == 0) report(a.status, GDN_STATUS_BAD_OFFSETS);
    return;
  }
  const int dv4 = a.dv >> 2;
  const int nf = KR * dv4;
  float4 *slab = reinterpret_cast<float4 *>(a.ST + ((size_t(r) * a.H + h) * a.dk + size_t(chunk) * KR) * a.dv);

  // issue the slab loads before anything else so they are in flight during the set-up
  float4 x[kCommitVec];
#pragma unroll
  for (int j = 0; j < kCommitVec; ++j) {
    const int f = tid + j * kThreads;
    if (f < nf) x[j] = __ldcs(slab + f);
  }
  const int32_t *path_r = a.path + size_t(r) * a.max_path;
  if (!check_path(a.parent, path_r, t0, n, L, a.max_path)) {
    if (tid == 0 && chunk == 0 && h == 0) report(a.status, GDN_STATUS_BAD_PATH);
    return;
  }
  float *kw = dyn;                        // [L][KR]   exp(G_l - G_j) k_j[row]
  float *us = dyn + size_t(a.max_path) * KR;  // [L][dv]   u_j
  const int l = path_r[L - 1];
  const float Gl = a.G[size_t(t0 + l) * a.H + h];
  for (int i = tid; i < L * KR; i += kThreads) {
    const int s = i / KR, row = i % KR;
    const size_t th = size_t(t0 + path_r[s]) * a.H + h;
    kw[i] = expf(Gl - a.G[th]) * bf16_to_f32(a.k[th * a.dk + size_t(chunk) * KR + row]);
  }
  for (int i = tid; i < L * dv4; i += kThreads) {
    const int s = i / dv4, c4 = i % dv4;
    const size_t th = size_t(t0 + path_r[s]) * a.H + h;
    reinterpret_cast<float4 *>(us)[i] = reinterpret_cast<const float4 *>(a.U + th * a.dv)[c4];
  }
  __syncthreads();
  const float decay = expf(Gl);
#pragma unroll
  for (int j = 0; j < kCommitVec; ++j) {
    const int f = tid + j * kThreads;
    if (f < nf) {
      const int row = f / dv4, c4 = f % dv4;
      float4 y = x[j];
      y.x *= decay; y.y *= decay; y.z *= decay; y.w *= decay;
      for (int s = 0; s < L; ++s) {
        const float w = kw[s * KR + row];
        const float4 u = reinterpret_cast<const float4 *>(us)[s * dv4 + c4];
        y.x = fmaf(w, u.x, y.x);
        y.y = fmaf(w, u.y, y.y);
        y.z = fmaf(w, u.z, y.z);
        y.w = fmaf(w, u.w, y.w);
      }
      __stcs(slab + f, y);
    }
  }
}

}  // namespace gdn
