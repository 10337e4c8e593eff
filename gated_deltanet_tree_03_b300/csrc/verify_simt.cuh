// CUDA-core (fp32 FMA) tree verify: the tree-structured WY form of the gated delta rule
// (TreeWY, method section), one CTA per (request, head, 32-column slice of d_v).
//
// Per (request r, head h), with nodes in parent-before-child order:
//   G_t = sum of g over t's root-to-node path, gamma_t = exp(G_t)
//   KS = K S_0^T, QS = Q S_0^T                         (projections through the state)
//   A[t,j] = b_t exp(G_t - G_j) (k_t . k_j)              j a strict ancestor of t
//   P[t,j] = exp(G_t - G_j) (q_t . k_j)                  j an ancestor of t, or t
//   (I + A) U = R,  R_t = b_t (v_t - gamma_t KS_t)       forward substitution in node order
//   o_t = gamma_t QS_t + sum_j P[t,j] u_j
// The d_v columns of U and o are independent, so each CTA owns a 32-column slice of the state
// and recomputes the small per-node scalars (A, P) itself.
#pragma once

#include "common.cuh"

namespace gdn {

struct VerifyArgs {
  const float *ST;
  const uint16_t *q, *k, *v;
  const float *beta, *g;
  const int32_t *parent, *cu_nodes;
  int B, H, T, dk, dv, max_nodes;
  float *o, *U, *G;
  int32_t *status;
};

// dynamic shared memory of the SIMT verify kernel for capacity M nodes and key width DK
__host__ __device__ inline size_t verify_simt_smem_bytes(int M, int DK) {
  return sizeof(float) * (size_t(2 * M) * DK   // K rows then Q rows (fp32)
                          + size_t(DK) * 32    // state slice
                          + size_t(M) * 32 * 4 // KS, QS, U, V slices
                          + size_t(M) * M * 2); // A, P
}

template <int DK, bool SV>
__global__ void __launch_bounds__(kThreads) verify_simt_kernel(VerifyArgs a, Serving sv) {
  __shared__ TreeSmem ts;
  extern __shared__ __align__(16) float dyn[];
  const int tile = blockIdx.x, h = blockIdx.y, r = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int t0 = a.cu_nodes[r];
  const int n = a.cu_nodes[r + 1] - t0;
  const int M = a.max_nodes;
  const int si = state_of<SV>(sv, r);
  if (si < 0) {
    if (si == kBadSlot && tid == 0 && tile == 0 && h == 0) report(a.status, GDN_STATUS_BAD_SLOT);
    return;
  }
  if (!offsets_ok(t0, n, a.T)) {
    if (tid == 0 && tile == 0 && h == 0) report(a.status, GDN_STATUS_BAD_OFFSETS);
    return;
  }
  if (n == 0) return;
  if (n > M) {
    if (tid == 0 && tile == 0 && h == 0) report(a.status, GDN_STATUS_TOO_MANY_NODES);
    return;
  }
  if (!analyse_tree<SV>(ts, a.parent, a.g, a.beta, t0, n, h, a.H, sv)) {
    if (tid == 0 && tile == 0 && h == 0) report(a.status, GDN_STATUS_BAD_TREE);
    return;
  }
  float *Xs = dyn;                       // [2M][DK]
  float *STs = Xs + size_t(2 * M) * DK;  // [DK][32]
  float *KSs = STs + DK * 32;            // [M][32]
  float *QSs = KSs + M * 32;
  float *Us = QSs + M * 32;
  float *Vs = Us + M * 32;
  float *Ac = Vs + M * 32;  // [M][M]
  float *Pc = Ac + M * M;

  const int H = a.H, dv = a.dv, c0 = tile * 32;
  const int HK = H / qk_group<SV>(sv), hk = h / qk_group<SV>(sv);  // q/k heads, this value head's q/k head
  // stage the node block and the state slice
  for (int i = tid; i < 2 * n * DK; i += kThreads) {
    const int row = i / DK, col = i % DK;
    const int t = row < n ? row : row - n;
    const uint16_t *src = row < n ? a.k : a.q;
    Xs[(row < n ? row : M + t) * DK + col] = bf16_to_f32(src[(size_t(t0 + t) * HK + hk) * DK + col]);
  }
  const float *ST = a.ST + (size_t(si) * H + h) * DK * dv + c0;
  for (int i = tid; i < DK * 32; i += kThreads) STs[i] = ST[size_t(i >> 5) * dv + (i & 31)];
  for (int i = tid; i < n * 32; i += kThreads)
    Vs[i] = bf16_to_f32(a.v[(size_t(t0 + (i >> 5)) * H + h) * dv + c0 + (i & 31)]);
  __syncthreads();

  // projections KS = K S_0^T and QS = Q S_0^T on this column slice
  for (int row = warp; row < 2 * n; row += kThreads / 32) {
    const float *x = Xs + (row < n ? row : M + row - n) * DK;
    float acc = 0.f;
#pragma unroll 8
    for (int kk = 0; kk < DK; ++kk) acc = fmaf(x[kk], STs[kk * 32 + lane], acc);
    if (row < n) KSs[row * 32 + lane] = acc;
    else QSs[(row - n) * 32 + lane] = acc;
  }
  // ancestor-masked, gate-weighted Gram entries
  for (int t = warp; t < n; t += kThreads / 32) {
    const float *kt = Xs + t * DK;
    const float *qt = Xs + (M + t) * DK;
    unsigned long long m = ts.anc[t];
    while (m) {
      const int j = __ffsll(m) - 1;
      m &= m - 1;
      const float *kj = Xs + j * DK;
      float kk = 0.f, qk = 0.f;
      for (int e = lane; e < DK; e += 32) {
        kk = fmaf(kt[e], kj[e], kk);
        qk = fmaf(qt[e], kj[e], qk);
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        kk += __shfl_xor_sync(0xffffffffu, kk, off);
        qk += __shfl_xor_sync(0xffffffffu, qk, off);
      }
      if (lane == 0) {
        const float w = expf(ts.G[t] - ts.G[j]);
        Ac[t * M + j] = (j == t) ? 0.f : ts.beta[t] * w * kk;
        Pc[t * M + j] = w * qk;
      }
    }
  }
  __syncthreads();

  // forward substitution, one column per lane (nodes are in topological order)
  if (warp == 0) {
    for (int t = 0; t < n; ++t) {
      const float gam = expf(ts.G[t]);
      float u = ts.beta[t] * (Vs[t * 32 + lane] - gam * KSs[t * 32 + lane]);
      unsigned long long m = ts.anc[t] & ~(1ull << t);
      while (m) {
        const int j = __ffsll(m) - 1;
        m &= m - 1;
        u = fmaf(-Ac[t * M + j], Us[j * 32 + lane], u);
      }
      Us[t * 32 + lane] = u;
    }
  }
  __syncthreads();

  // outputs
  for (int i = tid; i < n * 32; i += kThreads) {
    const int t = i >> 5, c = i & 31;
    float out = expf(ts.G[t]) * QSs[i];
    unsigned long long m = ts.anc[t];
    while (m) {
      const int j = __ffsll(m) - 1;
      m &= m - 1;
      out = fmaf(Pc[t * M + j], Us[j * 32 + c], out);
    }
    const size_t row = (size_t(t0 + t) * H + h) * dv + c0 + c;
    a.o[row] = query_scale<SV>(sv) * out;  // o is linear in q
    a.U[row] = Us[i];
    if (tile == 0 && c == 0) a.G[size_t(t0 + t) * H + h] = ts.G[t];
  }
}

}  // namespace gdn
