// Store-all comparison path (the "storeall" baseline on the TreeWY page, comparison with prior
// methods): step every node from its parent's stored state, in parent-before-child order, and
// keep the state of every node. Commit then copies the accepted node's stored state.
//
// Per node t with parent p (S_p = S_0 for a root):
//   u_t = b_t (v_t - a_t S_p k_t),   S_t = a_t S_p + u_t k_t^T,   o_t = S_t q_t
// One CTA per (request, head, 32-column slice of d_v); warp w owns rows
// [w*DK/8, (w+1)*DK/8) of the slice of S^T, lane = column. Each thread re-reads exactly the
// snapshot elements it wrote itself, so only the two dot-product reductions need barriers.
#pragma once

#include "common.cuh"

namespace gdn {

struct StoreallArgs {
  const float *ST;
  const uint16_t *q, *k, *v;
  const float *beta, *g;
  const int32_t *parent, *cu_nodes;
  int B, H, T, dk, dv, max_nodes;
  float *snap, *o, *U, *G;
  int32_t *status;
};

template <int DK>
__global__ void __launch_bounds__(kThreads) verify_storeall_kernel(StoreallArgs a) {
  constexpr int RK = DK / (kThreads / 32);  // state rows per warp
  __shared__ TreeSmem ts;
  __shared__ float kq[2][DK];
  __shared__ float red[2][kThreads / 32][32];
  const int tile = blockIdx.x, h = blockIdx.y, r = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int t0 = a.cu_nodes[r];
  const int n = a.cu_nodes[r + 1] - t0;
  if (!offsets_ok(t0, n, a.T)) {
    if (tid == 0 && tile == 0 && h == 0) report(a.status, GDN_STATUS_BAD_OFFSETS);
    return;
  }
  if (n == 0) return;
  if (n > a.max_nodes) {
    if (tid == 0 && tile == 0 && h == 0) report(a.status, GDN_STATUS_TOO_MANY_NODES);
    return;
  }
  if (!analyse_tree<false>(ts, a.parent, a.g, a.beta, t0, n, h, a.H, Serving{})) {
    if (tid == 0 && tile == 0 && h == 0) report(a.status, GDN_STATUS_BAD_TREE);
    return;
  }
  const int H = a.H, dv = a.dv, col = tile * 32 + lane, k0 = warp * RK;
  const size_t state_elems = size_t(DK) * dv;
  float s[RK];
  for (int t = 0; t < n; ++t) {
    const size_t th = size_t(t0 + t) * H + h;
    for (int i = tid; i < 2 * DK; i += kThreads)
      kq[i / DK][i % DK] = bf16_to_f32((i < DK ? a.k : a.q)[th * DK + (i % DK)]);
    const int p = ts.par[t];
    const float *src = p < 0 ? a.ST + (size_t(r) * H + h) * state_elems
                             : a.snap + (size_t(t0 + p) * H + h) * state_elems;
#pragma unroll
    for (int i = 0; i < RK; ++i) s[i] = src[size_t(k0 + i) * dv + col];
    __syncthreads();  // kq ready
    float part = 0.f;
#pragma unroll
    for (int i = 0; i < RK; ++i) part = fmaf(s[i], kq[0][k0 + i], part);
    red[0][warp][lane] = part;
    __syncthreads();
    float sk = 0.f;
#pragma unroll
    for (int w = 0; w < kThreads / 32; ++w) sk += red[0][w][lane];
    const float at = expf(ts.g[t]);
    const float u = ts.beta[t] * (bf16_to_f32(a.v[th * dv + col]) - at * sk);
    float *dst = a.snap + th * state_elems;
    part = 0.f;
#pragma unroll
    for (int i = 0; i < RK; ++i) {
      s[i] = fmaf(at, s[i], kq[0][k0 + i] * u);
      dst[size_t(k0 + i) * dv + col] = s[i];
      part = fmaf(s[i], kq[1][k0 + i], part);
    }
    red[1][warp][lane] = part;
    __syncthreads();
    if (warp == 0) {
      float out = 0.f;
#pragma unroll
      for (int w = 0; w < kThreads / 32; ++w) out += red[1][w][lane];
      a.o[th * dv + col] = out;
      a.U[th * dv + col] = u;
      if (tile == 0 && lane == 0) a.G[th] = ts.G[t];
    }
    __syncthreads();  // kq / red reuse
  }
}

struct StoreallCommitArgs {
  float *ST;
  const float *snap;
  const int32_t *parent, *cu_nodes, *path, *path_len;
  int B, H, T, dk, dv, max_path;
  int32_t *status;
};

// copy the accepted node's stored state into ST, one 16 KiB slab per CTA
__global__ void __launch_bounds__(kThreads) commit_storeall_kernel(StoreallCommitArgs a) {
  const int tid = threadIdx.x;
  const int per_cta = kThreads * 4;  // float4
  const int nf_state = a.dk * a.dv / 4;
  const int nchunk = (nf_state + per_cta - 1) / per_cta;
  const int chunk = blockIdx.x % nchunk;
  const int pair = blockIdx.x / nchunk;
  const int h = pair % a.H, r = pair / a.H;
  const int L = a.path_len[r];
  if (L == 0) return;
  const int t0 = a.cu_nodes[r];
  const int n = a.cu_nodes[r + 1] - t0;
  if (!offsets_ok(t0, n, a.T)) {
    if (tid == 0 && chunk == 0 && h == 0) report(a.status, GDN_STATUS_BAD_OFFSETS);
    return;
  }
  const int32_t *path_r = a.path + size_t(r) * a.max_path;
  if (!check_path(a.parent, path_r, t0, n, L, a.max_path)) {
    if (tid == 0 && chunk == 0 && h == 0) report(a.status, GDN_STATUS_BAD_PATH);
    return;
  }
  const int l = path_r[L - 1];
  const float4 *src = reinterpret_cast<const float4 *>(a.snap + (size_t(t0 + l) * a.H + h) * a.dk * a.dv);
  float4 *dst = reinterpret_cast<float4 *>(a.ST + (size_t(r) * a.H + h) * a.dk * a.dv);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int f = chunk * per_cta + tid + j * kThreads;
    if (f < nf_state) __stcs(dst + f, __ldcs(src + f));
  }
}

}  // namespace gdn
