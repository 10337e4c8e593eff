// Commit: rebuild only the accepted path's state, in place (TreeWY, method section: only the
// accepted path's pseudo-values are combined into the next committed state; novelty section:
// exactly one full state is rebuilt).
//
// With l the accepted path's last node, for every (request, head):
//   ST[kk][c] <- exp(G_l) ST[kk][c] + sum_{j on path} (exp(G_l - G_j) k_j[kk]) u_j[c]
//
// One CTA per (request, head). Thread 0 reads the path length and node offsets and, for a
// non-empty path, starts one bulk copy (cp.async.bulk, mbarrier completion) of the whole
// d_k x d_v state into shared memory. While the copy is in flight the CTA checks the path and
// stages the path's coefficients (exp(G_l - G_j) k_j and u_j). Each thread then owns one fixed
// group of four state columns, keeps the path's u_j for those columns in registers as it goes,
// accumulates its float4s and writes each one to HBM once with a streaming store. State
// traffic: one read and one write per element, nothing else.
#pragma once

#include "bounds.cuh"
#include "common.cuh"
#include "ptx.cuh"

namespace gdn {

struct CommitArgs {
  float *ST;
  const float *U, *G;
  const uint16_t *k;
  const int32_t *parent, *cu_nodes, *path, *path_len;
  int B, H, T, dk, dv, max_path;
  int32_t *status;
};

constexpr uint64_t kCommitWaitNs = 1000000000ull;  // 1 s bound on the state copy

__host__ __device__ inline size_t commit_smem_bytes(int max_path, int dk, int dv) {
  return size_t(dk) * dv * 4                       // the state
         + size_t(max_path) * (dk + dv) * 4;       // exp(G_l - G_j) k_j and u_j per path entry
}

template <int DK, int DV, bool SV>
__global__ void __launch_bounds__(kThreads) commit_kernel(CommitArgs a, Serving sv) {
  constexpr int DV4 = DV / 4;
  constexpr int J = DK * DV4 / kThreads;  // float4 of the state per thread
  constexpr int ROWSTEP = kThreads / DV4;  // state rows between a thread's float4s
  static_assert(J >= 1 && (DK * DV4) % kThreads == 0, "state must tile the block");
  constexpr uint32_t kStateBytes = DK * DV * 4;
  constexpr uint32_t kPiece = kStateBytes < 16384u ? kStateBytes : 16384u;

  extern __shared__ __align__(128) uint8_t commit_dyn[];
  float4 *xs = reinterpret_cast<float4 *>(commit_dyn);
  float *kw = reinterpret_cast<float *>(commit_dyn + kStateBytes);          // [max_path][DK]
  float4 *us = reinterpret_cast<float4 *>(kw + size_t(a.max_path) * DK);  // [max_path][DV4]
  __shared__ __align__(8) uint64_t bar;
  __shared__ int s_info[3];  // L, t0, n

  const int tid = threadIdx.x;
  const int pair = blockIdx.x;
  const int h = pair % a.H, r = pair / a.H;
  const int si = state_of<SV>(sv, r);  // the request's state (pool slot)
  if (si < 0) {  // padding request, or a slot outside the pool: the state is not touched
    if (si == kBadSlot && tid == 0 && h == 0) report(a.status, GDN_STATUS_BAD_SLOT);
    return;
  }
  const size_t st_off = (SV ? size_t(si) * a.H + h : size_t(pair)) * DK * DV;
  if (!range_in_bounds((long long)st_off, DK * DV, state_count<SV>(sv, a.B) * a.H * DK * DV, a.status)) return;
  float *ST = a.ST + st_off;
  const int HK = a.H / qk_group<SV>(sv), hk = h / qk_group<SV>(sv);  // q/k heads, this value head's q/k head

  if (tid == 0) {
    const int L = a.path_len[r];
    const int t0 = a.cu_nodes[r];
    const int n = a.cu_nodes[r + 1] - t0;
    int go = L != 0;
    if (go && !offsets_ok(t0, n, a.T)) {
      if (h == 0) report(a.status, GDN_STATUS_BAD_OFFSETS);
      go = 0;
    }
    if (go && (L < 0 || L > n || L > a.max_path)) {
      if (h == 0) report(a.status, GDN_STATUS_BAD_PATH);
      go = 0;
    }
    s_info[0] = go ? L : 0;
    s_info[1] = t0;
    s_info[2] = n;
    if (go) {
      ptx::mbar_init(&bar, 1);
      ptx::fence_mbar_init();
      ptx::mbar_arrive_expect_tx(&bar, kStateBytes);
#pragma unroll
      for (uint32_t off = 0; off < kStateBytes; off += kPiece)
        ptx::bulk_load(commit_dyn + off, reinterpret_cast<const uint8_t *>(ST) + off, kPiece, &bar);
    }
  }
  __syncthreads();
  const int L = s_info[0];
  if (L == 0) return;  // empty path (keep the state) or a rejected request: no copy in flight
  const int t0 = s_info[1], n = s_info[2];

  // path check and coefficient staging overlap the state copy
  const int32_t *path_r = a.path + size_t(r) * a.max_path;
  // a checked path names nodes 0 <= x < n, so every row t0 + x below lies inside [0, T)
  const bool path_ok = check_path(a.parent, path_r, t0, n, L, a.max_path) &&
                       range_in_bounds(t0, n, a.T, a.status);
  if (path_ok) {
    const int l = path_r[L - 1];
    const float Gl = a.G[size_t(t0 + l) * a.H + h];
    for (int i = tid; i < L * DK; i += kThreads) {
      const int s = i / DK, row = i % DK;
      const size_t th = size_t(t0 + path_r[s]) * a.H + h;
      kw[i] = expf(Gl - a.G[th]) * bf16_to_f32(a.k[(size_t(t0 + path_r[s]) * HK + hk) * DK + row]);
    }
    for (int i = tid; i < L * DV4; i += kThreads) {
      const int s = i / DV4, c4 = i % DV4;
      const size_t th = size_t(t0 + path_r[s]) * a.H + h;
      us[i] = reinterpret_cast<const float4 *>(a.U + th * DV)[c4];
    }
  }
  __syncthreads();
  const bool landed = ptx::mbar_wait(&bar, 0, kCommitWaitNs);
  if (!path_ok || !__syncthreads_and(landed)) {
    if (tid == 0 && !path_ok && h == 0) report(a.status, GDN_STATUS_BAD_PATH);
    if (tid == 0 && path_ok) report(a.status, GDN_STATUS_TIMEOUT);
    if (path_ok) ptx::mbar_wait(&bar, 0, kCommitWaitNs);  // let the copy land before leaving
    return;
  }

  const int c4 = tid % DV4, row0 = tid / DV4;
  const float decay = expf(a.G[size_t(t0 + path_r[L - 1]) * a.H + h]);
  float4 y[J];
#pragma unroll
  for (int j = 0; j < J; ++j) {
    const float4 x = xs[tid + j * kThreads];
    y[j] = make_float4(decay * x.x, decay * x.y, decay * x.z, decay * x.w);
  }
  for (int s = 0; s < L; ++s) {
    const float4 u = us[s * DV4 + c4];
    const float *w = kw + s * DK + row0;
#pragma unroll
    for (int j = 0; j < J; ++j) {
      const float wv = w[j * ROWSTEP];
      y[j].x = fmaf(wv, u.x, y[j].x);
      y[j].y = fmaf(wv, u.y, y[j].y);
      y[j].z = fmaf(wv, u.z, y[j].z);
      y[j].w = fmaf(wv, u.w, y[j].w);
    }
  }
  float4 *dst = reinterpret_cast<float4 *>(ST);
#pragma unroll
  for (int j = 0; j < J; ++j) __stcs(dst + tid + j * kThreads, y[j]);
}

}  // namespace gdn
