// Commit: rebuild only the accepted path's state, in place (TreeWY, method section: only the
// accepted path's pseudo-values are combined into the next committed state; novelty section:
// exactly one full state is rebuilt).
//
// With l the accepted path's last node, for every (request, head):
//   ST[kk][c] <- exp(G_l) ST[kk][c] + sum_{j on path} (exp(G_l - G_j) k_j[kk]) u_j[c]
//
// Two CTAs per (request, head), one per half of the state's d_k rows (each half one contiguous
// block: twice the resident CTAs per SM, and half the tail when a batch fills few waves). Thread 0
// first starts the copy of its d_k/2 x d_v rows into shared memory, as bulk copies
// (cp.async.bulk) of up to 16 KB, each completing on its own mbarrier; only then does it read
// the path length and node offsets. While the copies are in
// flight the CTA checks the path and stages the path's coefficients (exp(G_l - G_j) k_j and
// u_j). Each thread owns one fixed group of four state columns and, piece by piece as the copies
// land, accumulates its float4s of that piece and writes each one to HBM once with a streaming
// store. State traffic: one read and one write per element (an empty or rejected path reads the
// state and leaves it unchanged).
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
// CTAs per (request, head), each taking a block of d_k rows: two wherever half the rows still
// give every thread of the block a float4 of the state
__host__ __device__ constexpr int commit_row_split(int dk, int dv) { return (dk / 2) * (dv / 4) >= kThreads ? 2 : 1; }

__host__ __device__ inline size_t commit_smem_bytes(int max_path, int dk, int dv) {
  const int rdk = dk / commit_row_split(dk, dv);
  return size_t(rdk) * dv * 4                      // this CTA's state rows
         + size_t(max_path) * (rdk + dv) * 4;      // exp(G_l - G_j) k_j (its rows) and u_j per path entry
}

template <int DK, int DV, bool SV>
__global__ void __launch_bounds__(kThreads) commit_kernel(CommitArgs a, Serving sv) {
  constexpr int DV4 = DV / 4;
  constexpr int RS = commit_row_split(DK, DV);
  constexpr int RDK = DK / RS;               // state rows of this CTA
  constexpr int J = RDK * DV4 / kThreads;    // float4 of the state per thread
  constexpr int ROWSTEP = kThreads / DV4;    // state rows between a thread's float4s
  static_assert(J >= 1 && (RDK * DV4) % kThreads == 0, "the rows must tile the block");
  constexpr uint32_t kStateBytes = RDK * DV * 4;
  constexpr int NP = kStateBytes > 16384u ? int(kStateBytes / 16384u) : 1;  // copy pieces
  constexpr uint32_t kPiece = kStateBytes / NP;
  constexpr int JP = J / NP;  // a thread's float4s per piece (piece p: j = p JP .. p JP + JP - 1)
  static_assert(J % NP == 0 && (RDK / NP) % ROWSTEP == 0, "pieces must hold whole float4 groups");

  extern __shared__ __align__(128) uint8_t commit_dyn[];
  float4 *xs = reinterpret_cast<float4 *>(commit_dyn);
  float *kw = reinterpret_cast<float *>(commit_dyn + kStateBytes);           // [max_path][RDK]
  float4 *us = reinterpret_cast<float4 *>(kw + size_t(a.max_path) * RDK);  // [max_path][DV4]
  __shared__ __align__(8) uint64_t bar[NP];
  __shared__ int s_info[3];  // L, t0, n

  const int tid = threadIdx.x;
  const int pair = blockIdx.x / RS, part = blockIdx.x % RS;
  const int h = pair % a.H, r = pair / a.H;
  const int si = state_of<SV>(sv, r);  // the request's state (pool slot)
  if (si < 0) {  // padding request, or a slot outside the pool: the state is not touched
    if (si == kBadSlot && tid == 0 && h == 0 && part == 0) report(a.status, GDN_STATUS_BAD_SLOT);
    return;
  }
  const size_t st_off = (SV ? size_t(si) * a.H + h : size_t(pair)) * DK * DV + size_t(part) * RDK * DV;
  if (!range_in_bounds((long long)st_off, RDK * DV, state_count<SV>(sv, a.B) * a.H * DK * DV, a.status)) return;
  float *ST = a.ST + st_off;  // this CTA's rows part RDK .. part RDK + RDK - 1
  const int HK = a.H / qk_group<SV>(sv), hk = h / qk_group<SV>(sv);  // q/k heads, this value head's q/k head

  if (tid == 0) {
    // the state copy goes out before the dependent loads of the path
#pragma unroll
    for (int p = 0; p < NP; ++p) ptx::mbar_init(&bar[p], 1);
    ptx::fence_mbar_init();
#pragma unroll
    for (int p = 0; p < NP; ++p) {
      ptx::mbar_arrive_expect_tx(&bar[p], kPiece);
      ptx::bulk_load(commit_dyn + p * kPiece, reinterpret_cast<const uint8_t *>(ST) + p * kPiece, kPiece, &bar[p]);
    }
    const int L = a.path_len[r];
    const int t0 = a.cu_nodes[r];
    const int n = a.cu_nodes[r + 1] - t0;
    int go = L != 0;
    if (go && !offsets_ok(t0, n, a.T)) {
      if (h == 0 && part == 0) report(a.status, GDN_STATUS_BAD_OFFSETS);
      go = 0;
    }
    if (go && (L < 0 || L > n || L > a.max_path)) {
      if (h == 0 && part == 0) report(a.status, GDN_STATUS_BAD_PATH);
      go = 0;
    }
    s_info[0] = go ? L : 0;
    s_info[1] = t0;
    s_info[2] = n;
  }
  __syncthreads();
  const int L = s_info[0];
  const int t0 = s_info[1], n = s_info[2];

  // path check and coefficient staging overlap the state copy
  const int32_t *path_r = a.path + size_t(r) * a.max_path;
  // a checked path names nodes 0 <= x < n, so every row t0 + x below lies inside [0, T)
  const bool path_ok = L > 0 && check_path(a.parent, path_r, t0, n, L, a.max_path) &&
                       range_in_bounds(t0, n, a.T, a.status);
  if (path_ok) {
    const int l = path_r[L - 1];
    const float Gl = a.G[size_t(t0 + l) * a.H + h];
    for (int i = tid; i < L * RDK; i += kThreads) {
      const int s = i / RDK, row = i % RDK;
      const size_t th = size_t(t0 + path_r[s]) * a.H + h;
      kw[i] = expf(Gl - a.G[th]) * bf16_to_f32(a.k[(size_t(t0 + path_r[s]) * HK + hk) * DK + part * RDK + row]);
    }
    for (int i = tid; i < L * DV4; i += kThreads) {
      const int s = i / DV4, c4 = i % DV4;
      const size_t th = size_t(t0 + path_r[s]) * a.H + h;
      us[i] = reinterpret_cast<const float4 *>(a.U + th * DV)[c4];
    }
  }
  __syncthreads();
  if (!path_ok) {  // empty path (the state stays), or a rejected one: the copies land, nothing is written
    if (tid == 0 && L > 0 && h == 0 && part == 0) report(a.status, GDN_STATUS_BAD_PATH);
    if (tid == 0)
      for (int p = 0; p < NP; ++p) ptx::mbar_wait(&bar[p], 0, kCommitWaitNs);
    return;
  }

  const int c4 = tid % DV4, row0 = tid / DV4;
  const float decay = expf(a.G[size_t(t0 + path_r[L - 1]) * a.H + h]);
  float4 *dst = reinterpret_cast<float4 *>(ST);
#pragma unroll
  for (int p = 0; p < NP; ++p) {
    if (!ptx::mbar_wait(&bar[p], 0, kCommitWaitNs)) {  // this piece never landed: nothing more is written
      if (tid == 0) report(a.status, GDN_STATUS_TIMEOUT);
      for (int q = p; q < NP; ++q) ptx::mbar_wait(&bar[q], 0, kCommitWaitNs);  // let the copies land before leaving
      return;
    }
    float4 y[JP];
#pragma unroll
    for (int jj = 0; jj < JP; ++jj) {
      const float4 x = xs[tid + (p * JP + jj) * kThreads];
      y[jj] = make_float4(decay * x.x, decay * x.y, decay * x.z, decay * x.w);
    }
    for (int s = 0; s < L; ++s) {
      const float4 u = us[s * DV4 + c4];
      const float *w = kw + s * RDK + row0 + p * JP * ROWSTEP;
#pragma unroll
      for (int jj = 0; jj < JP; ++jj) {
        const float wv = w[jj * ROWSTEP];
        y[jj].x = fmaf(wv, u.x, y[jj].x);
        y[jj].y = fmaf(wv, u.y, y[jj].y);
        y[jj].z = fmaf(wv, u.z, y[jj].z);
        y[jj].w = fmaf(wv, u.w, y[jj].w);
      }
    }
#pragma unroll
    for (int jj = 0; jj < JP; ++jj) __stcs(dst + tid + (p * JP + jj) * kThreads, y[jj]);
  }
}

}  // namespace gdn
