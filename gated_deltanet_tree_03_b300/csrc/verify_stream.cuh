// CUDA-core streaming tree verify for small trees (at most NMAX <= 8 nodes per request): the
// tree-structured WY form of the gated delta rule (TreeWY, method section) with every per-node
// quantity held in registers.
//
// One CTA per (request, head), DV/2 threads; thread i owns state columns 2i and 2i+1. The CTA
// issues its first state rows before anything else, then stages the node block (keys and
// queries widened to fp32) in shared memory and analyses the tree while those loads are in
// flight. The fp32 state then streams from HBM exactly once, 16 rows ahead of use, and
// every row updates the thread's 2 x 2*NMAX projection accumulators
//     KS_t = S_0 k_t,   QS_t = S_0 q_t            (fp32 FMA, fp32 accumulate)
// Per node (registers, loops fully unrolled over the NMAX slots, ancestor tests uniform across
// the CTA):
//     R_t = b_t (v_t - gamma_t KS_t),  u_t = R_t - sum_{j strict ancestor} A[t,j] u_j
//     o_t = gamma_t QS_t + sum_{j ancestor or t} P[t,j] u_j
// with A[t,j] = b_t exp(G_t - G_j) k_t.k_j and P[t,j] = exp(G_t - G_j) q_t.k_j from one-thread
// dot products over the staged node block. At N <= 8 the 4 N d_k d_v FMAs per pair stay below the time the pair's state
// takes to arrive from HBM, so the kernel is bandwidth-bound without tensor cores or any
// shared-memory round trip of the state.
//
// With FUSE the kernel first folds the previous step's accepted path into each state row as it
// streams past (the commit update ST <- exp(G_l) ST + sum_j exp(G_l - G_j) k_j u_j^T of that path),
// writes the row back once, and projects the updated row: commit and the next verify then read
// and write every state element once between them instead of reading it twice.
#pragma once

#include "bounds.cuh"
#include "common.cuh"
#include "verify_simt.cuh"

namespace gdn {

constexpr int kStreamMaxNodes = 8;  // largest tree the streaming kernel takes

__device__ __forceinline__ float2 bf16x2_to_f32(uint32_t b) {
  return make_float2(__uint_as_float(b << 16), __uint_as_float(b & 0xffff0000u));
}

// Register cap per thread, sized so that 14 (four nodes), 12 (six) or 9 (eight) 64-thread CTAs
// share an SM (measured: 80 registers for six nodes beat 88 by 14 %; 72 for four nodes beat 68
// and 64, which spill more).
__host__ __device__ constexpr int stream_max_regs(int nmax, bool fuse) {
  return fuse ? (nmax <= 4 ? 96 : nmax <= 6 ? 112 : 128) : (nmax <= 4 ? 72 : nmax <= 6 ? 80 : 112);
}

constexpr int kFuseMaxPath = 4;  // accepted-path entries the fused kernel folds in (u_j kept in registers)

// The previous step's accepted path, folded into the state by the fused kernel.
struct PrevCommit {
  float *ST;  // the same array as VerifyArgs::ST, written in place
  const float *U, *G;
  const uint16_t *k;
  const int32_t *parent, *cu_nodes, *path, *path_len;
  int T, max_path;
};

// State rows each thread keeps in flight (more rows cost resident CTAs; 16 measured best).
__host__ __device__ constexpr int stream_prefetch_rows(int) { return 16; }

template <int DK, int DV, int NMAX, bool FUSE, bool SV>
__global__ void __launch_bounds__(DV / 2) __maxnreg__(stream_max_regs(NMAX, FUSE))
    verify_stream_kernel(VerifyArgs a, PrevCommit c, Serving sv) {
  constexpr int NT = DV / 2;    // threads
  constexpr int NX = 2 * NMAX;  // node-block rows: keys 0..NMAX-1, queries NMAX..2NMAX-1
  constexpr int DV2 = DV / 2;   // float2 per state row
  constexpr int kStreamPF = stream_prefetch_rows(NMAX);
  constexpr int LW = FUSE ? kFuseMaxPath : 1;
  static_assert(NMAX <= 8 && DK % kStreamPF == 0 && NT % 32 == 0, "shape");
  __shared__ __align__(16) float Xs[NX][DK];
  __shared__ __align__(16) float Ws[LW][DK];  // fused: exp(G_l - G_j) k_j per accepted-path entry
  __shared__ float Ac[NMAX][NMAX], Pc[NMAX][NMAX];
  __shared__ float G_s[NMAX], gam_s[NMAX], beta_s[NMAX], g_s[NMAX];
  __shared__ int par_s[NMAX];
  __shared__ uint32_t anc_s[NMAX];

  const int tid = threadIdx.x, lane = tid & 31;
  const int pair = blockIdx.x, h = pair % a.H, r = pair / a.H;
  const int col2 = tid;  // this thread's float2 column index within a state row
  const int si = state_of<SV>(sv, r);  // the request's state (pool slot)
  if (si < 0) {  // padding request, or a slot outside the pool: nothing is read or written
    if (si == kBadSlot && tid == 0 && h == 0) report(a.status, GDN_STATUS_BAD_SLOT);
    return;
  }
  const size_t st_off = (SV ? size_t(si) * a.H + h : size_t(pair)) * DK * DV;
  if (!range_in_bounds((long long)st_off, DK * DV, state_count<SV>(sv, a.B) * a.H * DK * DV, a.status)) return;
  const float2 *st = reinterpret_cast<const float2 *>(a.ST + st_off) + col2;

  // 1) the first state rows go out before any dependent load
  float2 s[kStreamPF];
#pragma unroll
  for (int i = 0; i < kStreamPF; ++i) s[i] = __ldcs(st + i * DV2);

  // 2) request bounds and checks (uniform across the CTA)
  const int t0 = a.cu_nodes[r];
  const int n = a.cu_nodes[r + 1] - t0;
  bool vok = true;
  // every node row below is t0 + t with t < n; with offsets_ok that stays inside [0, T)
  if (!offsets_ok(t0, n, a.T)) {
    if (tid == 0 && h == 0) report(a.status, GDN_STATUS_BAD_OFFSETS);
    vok = false;
  } else if (n == 0) {
    vok = false;
  } else if (n > a.max_nodes || n > NMAX) {
    if (tid == 0 && h == 0) report(a.status, GDN_STATUS_TOO_MANY_NODES);
    vok = false;
  }
  const int H = a.H;
  const int HK = H / qk_group<SV>(sv), hk = h / qk_group<SV>(sv);  // q/k heads, this value head's q/k head

  // 2b) fused: the previous step's accepted path (same checks and effect as gdn_tree_commit)
  int Lc = 0;
  float decay = 1.f;
  float2 us[LW];
#pragma unroll
  for (int q = 0; q < LW; ++q) us[q] = make_float2(0.f, 0.f);
  if constexpr (FUSE) {
    const int L = c.path_len[r];
    const int tp0 = c.cu_nodes[r];
    const int np = c.cu_nodes[r + 1] - tp0;
    bool cok = L != 0;
    if (cok && !offsets_ok(tp0, np, c.T)) {
      if (tid == 0 && h == 0) report(a.status, GDN_STATUS_BAD_OFFSETS);
      cok = false;
    }
    if (cok && (L < 0 || L > np || L > c.max_path || L > kFuseMaxPath)) {
      if (tid == 0 && h == 0) report(a.status, GDN_STATUS_BAD_PATH);
      cok = false;
    }
    const int32_t *path_r = c.path + size_t(r) * c.max_path;
    if (cok && !check_path(c.parent, path_r, tp0, np, L, c.max_path)) {
      if (tid == 0 && h == 0) report(a.status, GDN_STATUS_BAD_PATH);
      cok = false;
    }
    if (cok) {
      const float Gl = c.G[size_t(tp0 + path_r[L - 1]) * H + h];
      decay = expf(Gl);
      for (int i = tid; i < L * DK; i += NT) {
        const int q = i / DK, row = i % DK;
        const size_t th = size_t(tp0 + path_r[q]) * H + h;
        Ws[q][row] = in_bounds(tp0 + path_r[q], c.T, a.status)
                         ? expf(Gl - c.G[th]) * bf16_to_f32(c.k[(size_t(tp0 + path_r[q]) * HK + hk) * DK + row])
                         : 0.f;
      }
#pragma unroll
      for (int q = 0; q < LW; ++q)
        if (q < L && in_bounds(tp0 + path_r[q], c.T, a.status))
          us[q] = reinterpret_cast<const float2 *>(c.U + (size_t(tp0 + path_r[q]) * H + h) * DV)[col2];
      Lc = L;
    }
  }
  if (!vok && Lc == 0) return;  // nothing to fold in and nothing to verify

  // 3) node block (fp32, rows >= n zero), this thread's v pairs, tree inputs: every load goes
  // out before the first result is used (one memory round trip, not one per staged row)
  constexpr int NXI = (NX * DK / 4 + NT - 1) / NT;  // node-block words (4 bf16) per thread
  uint2 xw[NXI];
#pragma unroll
  for (int it = 0; it < NXI; ++it) {
    const int i = tid + it * NT;
    const int row = i / (DK / 4), c4 = i % (DK / 4);
    const int t = row < NMAX ? row : row - NMAX;
    xw[it] = make_uint2(0u, 0u);
    if (vok && i < NX * DK / 4 && t < n && in_bounds(t0 + t, a.T, a.status))
      xw[it] = *reinterpret_cast<const uint2 *>((row < NMAX ? a.k : a.q) + (size_t(t0 + t) * HK + hk) * DK + 4 * c4);
  }
  uint32_t vb[NMAX];
#pragma unroll
  for (int t = 0; t < NMAX; ++t)
    vb[t] = vok && t < n && in_bounds(t0 + t, a.T, a.status) ? *reinterpret_cast<const uint32_t *>(a.v + (size_t(t0 + t) * H + h) * DV + 2 * col2) : 0u;
  const bool own = vok && tid < n && in_bounds(t0 + tid, a.T, a.status);  // this thread's node
  int p_own = -1;
  float g_own = 0.f, b_own = 0.f;
  if (own) {
    p_own = a.parent[t0 + tid];
    gate_beta<SV>(sv, a.g, a.beta, size_t(t0 + tid) * H + h, h, g_own, b_own);
  }
#pragma unroll
  for (int it = 0; it < NXI; ++it) {
    const int i = tid + it * NT;
    if (vok && i < NX * DK / 4) {
      const float2 lo = bf16x2_to_f32(xw[it].x), hi = bf16x2_to_f32(xw[it].y);
      *reinterpret_cast<float4 *>(&Xs[i / (DK / 4)][4 * (i % (DK / 4))]) = make_float4(lo.x, lo.y, hi.x, hi.y);
    }
  }
  int bad = 0;
  if (own) {
    bad = (p_own < -1 || p_own >= tid);
    par_s[tid] = p_own;
    g_s[tid] = g_own;
    beta_s[tid] = b_own;
  }
  if (__syncthreads_or(bad)) {
    if (tid == 0 && h == 0) report(a.status, GDN_STATUS_BAD_TREE);
    vok = false;
    if (Lc == 0) return;
  }
  if (vok && tid < n) {
    // parent indices strictly decrease along the walk, so it ends within tid + 1 steps
    uint32_t m = 1u << tid;
    float Gs = g_s[tid];
    for (int x = par_s[tid]; x >= 0; x = par_s[x]) {
      m |= 1u << x;
      Gs += g_s[x];
    }
    anc_s[tid] = m;
    G_s[tid] = Gs;
    gam_s[tid] = expf(Gs);
  }
  __syncthreads();

  // 4) stream the state once: KS (rows 0..NMAX-1) and QS (rows NMAX..) for two columns
  float2 acc[NX];
#pragma unroll
  for (int t = 0; t < NX; ++t) acc[t] = make_float2(0.f, 0.f);
  // the fused kernel keeps the block loop rolled: unrolled, the fold's coefficient loads are
  // hoisted across blocks and the register count doubles
  constexpr int KUNROLL = FUSE ? 1 : DK / kStreamPF;
#pragma unroll KUNROLL
  for (int k0 = 0; k0 < DK; k0 += kStreamPF) {
    float2 nx[kStreamPF];
    if (k0 + kStreamPF < DK) {
#pragma unroll
      for (int i = 0; i < kStreamPF; ++i) nx[i] = __ldcs(st + (k0 + kStreamPF + i) * DV2);
    }
#pragma unroll
    for (int g4 = 0; g4 < kStreamPF; g4 += 4) {
      if constexpr (FUSE) {
        if (Lc > 0) {  // fold the accepted path into these four rows and write them back once
          float2 *stw = reinterpret_cast<float2 *>(c.ST + st_off) + col2;
#pragma unroll
          for (int i = 0; i < 4; ++i) s[g4 + i] = make_float2(decay * s[g4 + i].x, decay * s[g4 + i].y);
#pragma unroll
          for (int q = 0; q < LW; ++q) {
            if (q < Lc) {
              const float4 w = *reinterpret_cast<const float4 *>(&Ws[q][k0 + g4]);
              s[g4].x = fmaf(w.x, us[q].x, s[g4].x);
              s[g4].y = fmaf(w.x, us[q].y, s[g4].y);
              s[g4 + 1].x = fmaf(w.y, us[q].x, s[g4 + 1].x);
              s[g4 + 1].y = fmaf(w.y, us[q].y, s[g4 + 1].y);
              s[g4 + 2].x = fmaf(w.z, us[q].x, s[g4 + 2].x);
              s[g4 + 2].y = fmaf(w.z, us[q].y, s[g4 + 2].y);
              s[g4 + 3].x = fmaf(w.w, us[q].x, s[g4 + 3].x);
              s[g4 + 3].y = fmaf(w.w, us[q].y, s[g4 + 3].y);
            }
          }
#pragma unroll
          for (int i = 0; i < 4; ++i) __stcs(stw + (k0 + g4 + i) * DV2, s[g4 + i]);
        }
        if (!vok) continue;
      }
#pragma unroll
      for (int t = 0; t < NX; ++t) {
        const float4 x = *reinterpret_cast<const float4 *>(&Xs[t][k0 + g4]);
        acc[t].x = fmaf(x.x, s[g4].x, acc[t].x);
        acc[t].y = fmaf(x.x, s[g4].y, acc[t].y);
        acc[t].x = fmaf(x.y, s[g4 + 1].x, acc[t].x);
        acc[t].y = fmaf(x.y, s[g4 + 1].y, acc[t].y);
        acc[t].x = fmaf(x.z, s[g4 + 2].x, acc[t].x);
        acc[t].y = fmaf(x.z, s[g4 + 2].y, acc[t].y);
        acc[t].x = fmaf(x.w, s[g4 + 3].x, acc[t].x);
        acc[t].y = fmaf(x.w, s[g4 + 3].y, acc[t].y);
      }
    }
    if (k0 + kStreamPF < DK) {
#pragma unroll
      for (int i = 0; i < kStreamPF; ++i) s[i] = nx[i];
    }
  }

  if (!vok) return;

  // 5) masked, gated Gram entries A[t][j] (from k_t.k_j) and P[t][j] (from q_t.k_j) for every j
  // on t's path: one thread per dot product, straight from shared memory, each thread starting
  // at its own column so that the float4 reads of a warp spread over the banks
  {
    constexpr int NE = 2 * NMAX * NMAX;
    for (int e = tid; e < NE; e += NT) {
      const int kind = e / (NMAX * NMAX), t = (e / NMAX) % NMAX, j = e % NMAX;
      if (t >= n || !((anc_s[t] >> j) & 1u)) continue;
      const float *xa = Xs[kind == 0 ? t : NMAX + t];
      const float *xb = Xs[j];
      const int rot = (lane * 4) & (DK - 1);
      float d0 = 0.f, d1 = 0.f, d2 = 0.f, d3 = 0.f;
#pragma unroll 8
      for (int c = 0; c < DK; c += 4) {
        const int cc = (c + rot) & (DK - 1);
        const float4 x = *reinterpret_cast<const float4 *>(xa + cc);
        const float4 y = *reinterpret_cast<const float4 *>(xb + cc);
        d0 = fmaf(x.x, y.x, d0);
        d1 = fmaf(x.y, y.y, d1);
        d2 = fmaf(x.z, y.z, d2);
        d3 = fmaf(x.w, y.w, d3);
      }
      const float dot = (d0 + d1) + (d2 + d3);
      const float w = expf(G_s[t] - G_s[j]);
      if (kind == 0) Ac[t][j] = beta_s[t] * w * dot;
      else Pc[t][j] = w * dot;
    }
  }
  __syncthreads();

  // 6) solve and outputs in registers
  float2 u[NMAX];
#pragma unroll
  for (int t = 0; t < NMAX; ++t) {
    u[t] = make_float2(0.f, 0.f);
    if (t < n) {
      const float2 vv = bf16x2_to_f32(vb[t]);
      const float gm = gam_s[t], b = beta_s[t];
      float2 uu = make_float2(b * (vv.x - gm * acc[t].x), b * (vv.y - gm * acc[t].y));
      const uint32_t m = anc_s[t];
#pragma unroll
      for (int j = 0; j < t; ++j) {
        if ((m >> j) & 1u) {
          const float c = Ac[t][j];
          uu.x = fmaf(-c, u[j].x, uu.x);
          uu.y = fmaf(-c, u[j].y, uu.y);
        }
      }
      u[t] = uu;
    }
  }
#pragma unroll
  for (int t = 0; t < NMAX; ++t) {
    if (t < n) {
      const float gm = gam_s[t];
      float2 o = make_float2(gm * acc[NMAX + t].x, gm * acc[NMAX + t].y);
      const uint32_t m = anc_s[t];
#pragma unroll
      for (int j = 0; j <= t; ++j) {
        if ((m >> j) & 1u) {
          const float c = Pc[t][j];
          o.x = fmaf(c, u[j].x, o.x);
          o.y = fmaf(c, u[j].y, o.y);
        }
      }
      const size_t row = (size_t(t0 + t) * H + h) * DV2 + col2;
      const float qsc = query_scale<SV>(sv);  // o is linear in q
      if (in_bounds((long long)row, (long long)a.T * H * DV2, a.status)) {
        __stcs(reinterpret_cast<float2 *>(a.o) + row, make_float2(qsc * o.x, qsc * o.y));
        __stcs(reinterpret_cast<float2 *>(a.U) + row, u[t]);
      }
    }
  }
  if (tid < n && in_bounds((long long)(t0 + tid) * H + h, (long long)a.T * H, a.status))
    a.G[size_t(t0 + tid) * H + h] = G_s[tid];
}

}  // namespace gdn
