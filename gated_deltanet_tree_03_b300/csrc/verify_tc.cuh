// Tensor-core tree verify for sm_103a: the tree-structured WY form of the gated delta rule
// (TreeWY, method section), one CTA per (request, head), the whole d_v width of the state.
//
//   projections  D[v][n] = sum_k S0[v][k] X[n][k],  X = [K ; Q] (the node block)
//                -> KS = D[:, 0:Np], QS = D[:, Np:2Np]            tcgen05.mma, fp32 in TMEM
//   Gram         A[t,j] = b_t exp(G_t-G_j) k_t.k_j  (j strict ancestor of t)
//                P[t,j] = exp(G_t-G_j) q_t.k_j      (j ancestor of t, or t)     CUDA cores
//   solve        (I + A) U = R,  R_t = b_t (v_t - gamma_t KS_t)   one d_v column per thread
//   outputs      o_t = gamma_t QS_t + sum_j P[t,j] u_j
//
// Data movement:
//   * the fp32 state (d_k x d_v, 64 KiB at d = 128) is read from HBM once with coalesced loads
//     straight into registers, split into bf16 hi + lo parts (S = hi + lo + O(2^-17 |S|)) and
//     written once to shared memory as the UMMA A operand (K-major, 128-byte swizzle);
//     two MMAs per K-slice (hi, lo) give fp32-accurate products against the exact bf16 q/k;
//   * q and k rows are TMA-loaded (cp.async.bulk.tensor, 128-byte swizzle) directly into the
//     UMMA B-operand layout; v rows are TMA-loaded unswizzled;
//   * the accumulator lives in tensor memory and is read back with tcgen05.ld, one state
//     column (TMEM lane) per thread, which is exactly the column-independent triangular solve.
#pragma once

#include "common.cuh"
#include "ptx.cuh"
#include "verify_simt.cuh"

namespace gdn {

constexpr uint64_t kWaitLimitNs = 1000000000ull;  // 1 s bound on every asynchronous wait

__host__ __device__ constexpr int tc_a_bytes(int DK) { return DK * 256; }  // one of hi / lo: 128 rows x DK bf16

__host__ __device__ inline size_t tc_smem_bytes(int DK, int DV, int Np) {
  return size_t(2 * tc_a_bytes(DK))        // A operand: hi and lo
         + size_t(DK) * Np * 4             // B operand: [K ; Q], 2*Np rows x DK bf16
         + size_t(Np) * DV * 2             // v rows (bf16)
         + size_t(2) * Np * Np * 4         // A and P coefficients
         + 1024;                           // alignment slack for the 1024-byte swizzle atoms
}

__host__ __device__ inline uint32_t tc_tmem_cols(int Np) {
  uint32_t c = 32;
  while (c < uint32_t(2 * Np)) c <<= 1;
  return c;
}

template <int DK, int DV>
__global__ void __launch_bounds__(kThreads, 1)
    verify_tc_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_q,
                     const __grid_constant__ CUtensorMap tm_v, VerifyArgs a, int Np) {
  static_assert(DK == 64 || DK == 128, "tensor-core verify needs d_k in {64, 128}");
  static_assert(DV == 64 || DV == 128, "tensor-core verify needs d_v in {64, 128}");
  constexpr int SLICES = kThreads / DV;         // threads sharing one state column during the split
  constexpr int CH = DK / SLICES / 8;           // 8-element K chunks per thread
  constexpr int EPL = DK / 32;                  // key elements per lane in the Gram dot products
  __shared__ TreeSmem ts;
  __shared__ float gam[kMaxNodes];
  __shared__ __align__(8) uint64_t bars[2];
  __shared__ uint32_t tmem_holder;
  extern __shared__ uint8_t dyn_raw[];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int pair = blockIdx.x;
  const int h = pair % a.H, r = pair / a.H;
  const int t0 = a.cu_nodes[r];
  const int n = a.cu_nodes[r + 1] - t0;
  if (!offsets_ok(t0, n, a.T)) {
    if (tid == 0 && h == 0) report(a.status, GDN_STATUS_BAD_OFFSETS);
    return;
  }
  if (n == 0) return;
  if (n > a.max_nodes) {
    if (tid == 0 && h == 0) report(a.status, GDN_STATUS_TOO_MANY_NODES);
    return;
  }

  // 1) issue the state loads: thread -> (column v, K slice); 8 consecutive rows per chunk
  const int v = tid % DV, slice = tid / DV;
  const float *ST = a.ST + size_t(pair) * DK * DV;
  float x[CH][8];
#pragma unroll
  for (int c = 0; c < CH; ++c)
#pragma unroll
    for (int i = 0; i < 8; ++i) x[c][i] = __ldcs(ST + size_t((slice * CH + c) * 8 + i) * DV + v);

  // 2) tree structure (parent check, ancestor masks, cumulative log-gates) while loads fly
  if (!analyse_tree(ts, a.parent, a.g, a.beta, t0, n, h, a.H)) {
    if (tid == 0 && h == 0) report(a.status, GDN_STATUS_BAD_TREE);
    return;
  }
  if (tid < n) gam[tid] = expf(ts.G[tid]);

  uint8_t *dyn = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(dyn_raw) + 1023) & ~uintptr_t(1023));
  uint8_t *A_hi = dyn;
  uint8_t *A_lo = dyn + tc_a_bytes(DK);
  uint8_t *Bt = dyn + 2 * tc_a_bytes(DK);
  const int region_b = 2 * Np * 128;  // bytes per 64-wide K region of the B operand
  uint16_t *Vs = reinterpret_cast<uint16_t *>(Bt + size_t(DK) * Np * 4);
  float *Ac = reinterpret_cast<float *>(reinterpret_cast<uint8_t *>(Vs) + size_t(Np) * DV * 2);
  float *Pc = Ac + Np * Np;
  float *Us = reinterpret_cast<float *>(dyn);  // reuses the A operand once the MMAs are done

  // 3) barriers + tensor memory
  const uint32_t ncols = tc_tmem_cols(Np);
  if (tid == 0) {
    ptx::mbar_init(&bars[0], 1);
    ptx::mbar_init(&bars[1], 1);
    ptx::fence_mbar_init();
  }
  if (warp == 0) {
    ptx::tmem_alloc(&tmem_holder, ncols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before_sync();
  __syncthreads();
  ptx::tc_fence_after_sync();
  const uint32_t tmem = tmem_holder;

  // 4) node block via TMA: K rows -> B rows [0, Np), Q rows -> [Np, 2Np); v rows unswizzled
  if (tid == 0) {
    ptx::mbar_arrive_expect_tx(&bars[0], uint32_t((2 * DK + DV) * Np * 2));
#pragma unroll
    for (int reg = 0; reg < DK / 64; ++reg) {
      ptx::tma_load_3d(Bt + reg * region_b, &tm_k, &bars[0], reg * 64, h, t0);
      ptx::tma_load_3d(Bt + reg * region_b + Np * 128, &tm_q, &bars[0], reg * 64, h, t0);
    }
    ptx::tma_load_3d(Vs, &tm_v, &bars[0], 0, h, t0);
  }

  // 5) split the state into bf16 hi / lo and store it as the K-major A operand (row = v)
#pragma unroll
  for (int c = 0; c < CH; ++c) {
    const int kc = slice * CH + c;  // global 8-element chunk index along K
    uint32_t hi[4], lo[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const __nv_bfloat162 h2 = __floats2bfloat162_rn(x[c][2 * i], x[c][2 * i + 1]);
      const float2 hf = __bfloat1622float2(h2);
      const __nv_bfloat162 l2 = __floats2bfloat162_rn(x[c][2 * i] - hf.x, x[c][2 * i + 1] - hf.y);
      hi[i] = *reinterpret_cast<const uint32_t *>(&h2);
      lo[i] = *reinterpret_cast<const uint32_t *>(&l2);
    }
    const int off = (kc >> 3) * 16384 + v * 128 + (((kc & 7) ^ (v & 7)) << 4);
    *reinterpret_cast<uint4 *>(A_hi + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
    *reinterpret_cast<uint4 *>(A_lo + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
  }
  ptx::fence_proxy_async_smem();
  __syncthreads();

  // 6) wait for the node block; one thread issues the projection MMAs
  const bool nodes_ok = ptx::mbar_wait(&bars[0], 0, kWaitLimitNs);
  if (!__syncthreads_and(nodes_ok)) {
    if (tid == 0) report(a.status, GDN_STATUS_TIMEOUT);
    ptx::mbar_wait(&bars[0], 0, kWaitLimitNs);  // let copies in flight land before leaving
    ptx::tc_fence_before_sync();
    __syncthreads();
    if (warp == 0) ptx::tmem_dealloc(tmem, ncols);
    return;
  }
  if (tid == 0) {
    ptx::tc_fence_after_sync();
    constexpr int M = 128;
    const uint32_t idesc = ptx::idesc_bf16_f32(M, 2 * Np);
    const uint32_t a_hi = ptx::smem_u32(A_hi), a_lo = ptx::smem_u32(A_lo), b0 = ptx::smem_u32(Bt);
#pragma unroll
    for (int ks = 0; ks < DK / 16; ++ks) {
      const uint32_t aoff = (ks >> 2) * 16384 + (ks & 3) * 32;
      const uint32_t boff = (ks >> 2) * region_b + (ks & 3) * 32;
      const uint64_t bdesc = ptx::desc_kmajor_sw128(b0 + boff);
      ptx::mma_bf16_ss(tmem, ptx::desc_kmajor_sw128(a_hi + aoff), bdesc, idesc, ks > 0 ? 1u : 0u);
      ptx::mma_bf16_ss(tmem, ptx::desc_kmajor_sw128(a_lo + aoff), bdesc, idesc, 1u);
    }
    ptx::mma_commit(&bars[1]);
  }

  // 7) gate-weighted, ancestor-masked Gram entries from the swizzled node tile (CUDA cores)
  {
    const int e0 = lane * EPL;  // first key element of this lane
    const int reg = e0 >> 6, chunk = (e0 & 63) >> 3, sub = (e0 & 7) * 2;
    auto row_ptr = [&](int row) {
      return Bt + reg * region_b + row * 128 + ((chunk ^ (row & 7)) << 4) + sub;
    };
    for (int t = warp; t < n; t += kThreads / 32) {
      float kt[EPL], qt[EPL];
      const uint16_t *pk = reinterpret_cast<const uint16_t *>(row_ptr(t));
      const uint16_t *pq = reinterpret_cast<const uint16_t *>(row_ptr(Np + t));
#pragma unroll
      for (int e = 0; e < EPL; ++e) {
        kt[e] = bf16_to_f32(pk[e]);
        qt[e] = bf16_to_f32(pq[e]);
      }
      unsigned long long m = ts.anc[t];
      while (m) {
        const int j = __ffsll(m) - 1;
        m &= m - 1;
        const uint16_t *pj = reinterpret_cast<const uint16_t *>(row_ptr(j));
        float kk = 0.f, qk = 0.f;
#pragma unroll
        for (int e = 0; e < EPL; ++e) {
          const float kj = bf16_to_f32(pj[e]);
          kk = fmaf(kt[e], kj, kk);
          qk = fmaf(qt[e], kj, qk);
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
          kk += __shfl_xor_sync(0xffffffffu, kk, off);
          qk += __shfl_xor_sync(0xffffffffu, qk, off);
        }
        if (lane == 0) {
          const float w = expf(ts.G[t] - ts.G[j]);
          Ac[t * Np + j] = (j == t) ? 0.f : ts.beta[t] * w * kk;
          Pc[t * Np + j] = w * qk;
        }
      }
    }
  }
  __syncthreads();

  // 8) projections ready in TMEM
  const bool mma_ok = ptx::mbar_wait(&bars[1], 0, kWaitLimitNs);
  if (!__syncthreads_and(mma_ok)) {
    if (tid == 0) report(a.status, GDN_STATUS_TIMEOUT);
    ptx::mbar_wait(&bars[1], 0, kWaitLimitNs);
    ptx::tc_fence_before_sync();
    __syncthreads();
    if (warp == 0) ptx::tmem_dealloc(tmem, ncols);
    return;
  }
  ptx::tc_fence_after_sync();

  const int H = a.H;
  // 9) R = b (v - gamma KS) into Us, then forward substitution, one state column per thread
  if (warp < 4) {
    const int col = tid;  // TMEM lane == state column v
    const uint32_t lane_base = tmem + (uint32_t(warp * 32) << 16);
    for (int c0 = 0; c0 < n; c0 += 16) {
      float ks[16];
      ptx::tmem_ld_32x32b_x16(lane_base + uint32_t(c0), ks);
      if (col < DV) {
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int t = c0 + j;
          if (t < n) Us[t * DV + col] = ts.beta[t] * (bf16_to_f32(Vs[t * DV + col]) - gam[t] * ks[j]);
        }
      }
    }
    if (col < DV) {
      for (int t = 0; t < n; ++t) {
        float u = Us[t * DV + col];
        unsigned long long m = ts.anc[t] & ~(1ull << t);
        while (m) {
          const int j = __ffsll(m) - 1;
          m &= m - 1;
          u = fmaf(-Ac[t * Np + j], Us[j * DV + col], u);
        }
        Us[t * DV + col] = u;
      }
    }
  }
  __syncthreads();

  // 10) outputs: warps w and w+4 share TMEM lanes 32*(w%4).., split nodes by parity
  {
    const int q4 = warp & 3, half = warp >> 2;
    const int col = q4 * 32 + lane;
    const uint32_t lane_base = tmem + (uint32_t(q4 * 32) << 16) + uint32_t(Np);
    for (int c0 = 0; c0 < n; c0 += 16) {
      float qs[16];
      ptx::tmem_ld_32x32b_x16(lane_base + uint32_t(c0), qs);
      if (col < DV) {
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int t = c0 + j;
          if (t < n && (t & 1) == half) {
            float out = gam[t] * qs[j];
            unsigned long long m = ts.anc[t];
            while (m) {
              const int i = __ffsll(m) - 1;
              m &= m - 1;
              out = fmaf(Pc[t * Np + i], Us[i * DV + col], out);
            }
            const size_t row = (size_t(t0 + t) * H + h) * DV + col;
            a.o[row] = out;
            a.U[row] = Us[t * DV + col];
          }
        }
      }
    }
  }
  if (tid < n) a.G[size_t(t0 + tid) * H + h] = ts.G[tid];

  ptx::tc_fence_before_sync();
  __syncthreads();
  if (warp == 0) ptx::tmem_dealloc(tmem, ncols);
}

}  // namespace gdn
