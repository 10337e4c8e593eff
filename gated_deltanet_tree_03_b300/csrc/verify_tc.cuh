// Tensor-core tree verify for sm_103a: the tree-structured WY form of the gated delta rule
// (TreeWY, method section). Persistent, warp-specialised: one CTA per SM walks the
// (request, head) pairs p = blockIdx.x, blockIdx.x + gridDim.x, ... through a pipeline.
//
// Per pair (X = [K ; Q], the node block, rows 0..Np-1 = keys, Np..2Np-1 = queries):
//   projections  D1[v][n] = sum_k S0[v][k] X[n][k]  -> KS = D1[:, 0:Np], QS = D1[:, Np:2Np]
//   Gram         D2[m][j] = sum_k X[m][k] K[j][k]   -> k_t.k_j (m = t), q_t.k_j (m = Np + t)
//   masks        A[t,j] = b_t exp(G_t - G_j) k_t.k_j   (j a strict ancestor of t)
//                P[t,j] = exp(G_t - G_j) q_t.k_j       (j an ancestor of t, or t)
//   inverse      T = (I + A)^-1 and W = P T. Both keep the ancestor pattern, so row t has one
//                entry per node of t's root-to-node path; one thread per row sweeps it in
//                registers (no chain through other rows for T, one barrier before W)
//   solve+out    D3[v][n] = sum_j R[j][v] [T ; W][n][j],  R_t = b_t (v_t - gamma_t KS_t):
//                u_t = D3[:, t], o_t = gamma_t QS_t + D3[:, Np + t]. tcgen05.mma with R and
//                [T ; W] split into bf16 hi + lo (three products), fp32 accumulate in TMEM
//
// Warp roles (640 threads):
//   warp 0       state producer: 1-D bulk copies (cp.async.bulk) of 64-row fp32 chunks of the
//                state into a ring of 32 KiB shared-memory slots
//   warp 1       node producer: TMA (cp.async.bulk.tensor) of the K and Q rows straight into the
//                128-byte-swizzled K-major UMMA operand layout (one buffer, refilled once the
//                previous pair's MMAs are done), and of the v rows (one buffer, refilled once
//                the previous pair's R is formed)
//   warp 2       MMA issuer for the projections and the Gram (one thread) and tensor-memory
//                owner: tcgen05.mma kind::f16, fp32 accumulators in TMEM, two buffers of 256
//                columns so the epilogue of one pair overlaps the MMAs of the next
//   warp 3       tree analysis: parent check, 64-bit ancestor masks, cumulative log-gates, depths
//                and each node's root-to-node path table, double-buffered
//   warps 4-11   epilogue: Gram rows from TMEM -> masked, gated path coefficients; T and W; the
//                dense [T ; W] and R operands; the solve/output MMA; o and U stores
//   warps 12-19  splitters: each fp32 chunk is split in place into bf16 hi + lo parts
//                (S = hi + lo + O(2^-17 |S|)) written as the K-major, 128-byte-swizzled UMMA A
//                operand; two MMAs per K slice (hi, lo) give fp32-accurate products against
//                the exact bf16 q / k
// Every wait on an mbarrier is bounded (1 s); a role that gives up raises a CTA-wide abort
// flag and GDN_STATUS_TIMEOUT, all roles leave their loops, the CTA waits (bounded) for its
// copies and MMAs in flight, frees its tensor memory and returns.
#pragma once

#include "common.cuh"
#include "ptx.cuh"
#include "verify_simt.cuh"

namespace gdn {

constexpr uint64_t kWaitLimitNs = 1000000000ull;  // 1 s bound on every wait
constexpr int kTcThreads = 640;
constexpr int kChunkRows = 64;            // state rows (along d_k) per ring slot
constexpr uint32_t kSlotBytes = 32768;    // fp32 chunk, then bf16 hi (16 KiB) + lo (16 KiB)
constexpr uint32_t kRegionBytes = 16384;  // 128 rows x 128 B: one 64-wide K region of an operand
constexpr int kMaxRing = 6;
constexpr uint32_t kTmemCols = 512;       // two buffers of 256 columns
constexpr uint32_t kTmemBuf = 256;
constexpr uint32_t kGramCol = 128;        // Gram accumulator offset inside a buffer

enum : int {
  kWarpState = 0,
  kWarpNodes = 1,
  kWarpMma = 2,
  kWarpTree = 3,
  kWarpEpi = 4,
  kEpiThreads = 256,
  kWarpSplit = 12,
  kSplitThreads = 256,
};

enum : int { kBarSplit = 1, kBarEpi = 2 };  // named barriers (0 is __syncthreads)

// Shared-memory carve-up (byte offsets from a 1024-byte-aligned base).
//   ring   R slots of 32 KiB: fp32 state chunks, split in place to the bf16 hi / lo A operand
//   x      the [K ; Q] B operand of the projections and the A / B operands of the Gram
//   v      v rows (bf16)
//   aop    R^T as the A operand of the solve/output MMA (hi, lo: 128 rows x 128 B each); before
//          R exists the same bytes hold the packed path coefficients A, P and T (fp32)
//   bop    [T ; W] as its B operand (hi, lo: 2 Np rows x 128 B each)
struct TcLayout {
  int Np, R;
  uint32_t ring, x, v, aop, bop, ca, cp, ct, total;
};

__host__ __device__ inline uint32_t align_up(uint32_t x, uint32_t a) { return (x + a - 1) / a * a; }

__host__ __device__ inline TcLayout tc_layout(int DK, int DV, int Np, int R) {
  TcLayout L{};
  L.Np = Np;
  L.R = R;
  const uint32_t ncoef = align_up(uint32_t(Np) * (Np + 1) / 2 * 4, 128);  // one packed coefficient array
  uint32_t off = 0;
  L.ring = off;
  off += uint32_t(R) * kSlotBytes;
  L.x = off;
  off += uint32_t(DK / 64) * kRegionBytes;
  L.v = off;
  off = align_up(off + uint32_t(Np) * DV * 2, 1024);
  L.aop = off;
  L.ca = off;
  L.cp = off + ncoef;
  L.ct = off + 2 * ncoef;
  off += 2 * kRegionBytes;
  L.bop = off;
  off += 2u * 2u * uint32_t(Np) * 128u;
  L.total = off;
  return L;
}

// Per-pair tree analysis, double-buffered between the tree warp and the epilogue.
struct TreeStage {
  unsigned long long anc[kMaxNodes];  // bit j <=> j on t's root-to-node path (t included)
  float G[kMaxNodes];                 // cumulative log-gate
  float gam[kMaxNodes];               // exp(G)
  float beta[kMaxNodes];
  float g[kMaxNodes];
  int par[kMaxNodes];
  int off[kMaxNodes + 1];             // packed per-path offsets: row t at off[t], depth(t)+1 entries
  uint8_t dep[kMaxNodes];
  uint8_t pnode[kMaxNodes * (kMaxNodes + 1) / 2];  // pnode[off[t] + k] = t's ancestor at depth k
  uint8_t tnode[kMaxNodes * (kMaxNodes + 1) / 2];  // tnode[off[t] + k] = t
  int16_t poff[kMaxNodes * (kMaxNodes + 1) / 2];   // poff[e] = off[pnode[e]]
  int nent;                                        // path entries of the pair
  int maxd;
  int bad;
};

struct TcShared {
  TreeStage tree[2];
  uint64_t slot_full[kMaxRing], slot_split[kMaxRing], slot_empty[kMaxRing];
  uint64_t node_full[2], v_full, v_empty, gram_full[2], proj_full[2], tmem_empty[2], uo_full;
  uint64_t tree_full[2], tree_empty[2], drain, drain_epi;
  uint32_t tmem_base;
  int abort_flag;
  int split_ok, epi_ok[3];
};

// Nodes and state slot of pair p; false for a pair that is skipped (padding request, slot
// outside the pool, empty, too many nodes, bad offsets).
template <bool SV>
__device__ __forceinline__ bool tc_pair_nodes(const VerifyArgs &a, const Serving &sv, int p, int &t0, int &n,
                                              int &si) {
  const int r = p / a.H;
  t0 = a.cu_nodes[r];
  n = a.cu_nodes[r + 1] - t0;
  if constexpr (SV) {
    si = state_of<SV>(sv, r);
    return si >= 0 && offsets_ok(t0, n, a.T) && n > 0 && n <= a.max_nodes;
  } else {
    si = r;
    return offsets_ok(t0, n, a.T) && n > 0 && n <= a.max_nodes;
  }
}

// Bounded wait that also gives up when another role has raised the abort flag.
__device__ __forceinline__ bool tc_wait(uint64_t *bar, uint32_t parity, TcShared &sh, int32_t *status) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = ptx::globaltimer_ns();
  for (uint32_t i = 1; i < (1u << 26); ++i) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    if ((i & 15u) == 0) {
      if (*reinterpret_cast<volatile int *>(&sh.abort_flag)) return false;
      if (ptx::globaltimer_ns() - t0 > kWaitLimitNs) break;
    }
  }
  *reinterpret_cast<volatile int *>(&sh.abort_flag) = 1;
  report(status, GDN_STATUS_TIMEOUT);
  return false;
}

__device__ __forceinline__ void named_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(ptx::smem_u32(bar)) : "memory");
}

template <int DK, int DV, bool SV>
__global__ void __launch_bounds__(kTcThreads, 1)
    verify_tc_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_q,
                     const __grid_constant__ CUtensorMap tm_v, VerifyArgs a, TcLayout lay, Serving sv) {
  static_assert(DK == 64 || DK == 128, "tensor-core verify needs d_k in {64, 128}");
  static_assert(DV == 64 || DV == 128, "tensor-core verify needs d_v in {64, 128}");
  constexpr int NCHUNK = DK / kChunkRows;              // ring slots per pair
  constexpr uint32_t kChunkBytes = kChunkRows * DV * 4;  // fp32 bytes of one chunk

  __shared__ TcShared sh;
  extern __shared__ uint8_t tc_dyn_raw[];
  uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(tc_dyn_raw) + 1023) & ~uintptr_t(1023));

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int Np = lay.Np, R = lay.R;
  const int npairs = a.B * a.H;
  uint8_t *ring = base + lay.ring;

  if (tid == 0) {
    for (int s = 0; s < R; ++s) {
      ptx::mbar_init(&sh.slot_full[s], 1);
      ptx::mbar_init(&sh.slot_split[s], 1);
      ptx::mbar_init(&sh.slot_empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(&sh.node_full[b], 1);
      ptx::mbar_init(&sh.gram_full[b], 1);
      ptx::mbar_init(&sh.proj_full[b], 1);
      ptx::mbar_init(&sh.tmem_empty[b], kEpiThreads / 32);
      ptx::mbar_init(&sh.tree_full[b], 32);
      ptx::mbar_init(&sh.tree_empty[b], kEpiThreads / 32);
    }
    ptx::mbar_init(&sh.v_full, 1);
    ptx::mbar_init(&sh.v_empty, kEpiThreads / 32);
    ptx::mbar_init(&sh.uo_full, 1);
    ptx::mbar_init(&sh.drain, 1);
    ptx::mbar_init(&sh.drain_epi, 1);
    sh.abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == kWarpMma) {
    ptx::tmem_alloc(&sh.tmem_base, kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before_sync();
  __syncthreads();
  ptx::tc_fence_after_sync();
  const uint32_t tmem = sh.tmem_base;

  // bookkeeping for the clean-up waits
  uint32_t issued = 0;   // state producer: chunks issued; node producer: stages issued
  uint32_t v_issued = 0; // node producer: v copies issued
  bool mma_any = false;  // the MMA warp (projections, Gram) or epilogue thread 0 (solve/output) issued MMAs

  if (warp == kWarpState) {
    // ------------------------------------------------------------ state producer
    if (lane == 0) {
      uint32_t u = 0;
      for (int p = blockIdx.x; p < npairs; p += gridDim.x) {
        int t0, n, si;
        if (!tc_pair_nodes<SV>(a, sv, p, t0, n, si)) continue;
        const size_t st_idx = SV ? size_t(si) * a.H + p % a.H : size_t(p);
        const uint8_t *src = reinterpret_cast<const uint8_t *>(a.ST + st_idx * DK * DV);
        bool ok = true;
        for (int c = 0; c < NCHUNK; ++c, ++u) {
          const int s = int(u % uint32_t(R));
          if (!tc_wait(&sh.slot_empty[s], ((u / R) & 1u) ^ 1u, sh, a.status)) { ok = false; break; }
          ptx::mbar_arrive_expect_tx(&sh.slot_full[s], kChunkBytes);
#pragma unroll
          for (uint32_t off = 0; off < kChunkBytes; off += 16384u)
            ptx::bulk_load(ring + s * kSlotBytes + off, src + c * kChunkBytes + off, 16384u, &sh.slot_full[s]);
          issued = u + 1;
        }
        if (!ok) break;
      }
    }
  } else if (warp == kWarpNodes) {
    // ------------------------------------------------------------ node producer
    if (lane == 0) {
      ptx::prefetch_tensormap(&tm_k);
      ptx::prefetch_tensormap(&tm_q);
      ptx::prefetch_tensormap(&tm_v);
      const uint32_t x_bytes = uint32_t(2 * DK) * Np * 2, v_bytes = uint32_t(DV) * Np * 2;
      uint8_t *X = base + lay.x;
      uint32_t i = 0;
      for (int p = blockIdx.x; p < npairs; p += gridDim.x) {
        int t0, n, si;
        if (!tc_pair_nodes<SV>(a, sv, p, t0, n, si)) continue;
        const int h = p % a.H, b = int(i & 1u), hk = h / qk_group<SV>(sv);
        // the X buffer is free once the MMAs of pair i-1 are done, the v buffer once the
        // epilogue of pair i-1 has formed its R (neither barrier can complete again before
        // this copy is issued, so the parity cannot have moved on); X goes first so the MMAs
        // never wait on v
        if (i > 0 && !tc_wait(&sh.proj_full[(i - 1) & 1u], ((i - 1) >> 1) & 1u, sh, a.status)) break;
        ptx::mbar_arrive_expect_tx(&sh.node_full[b], x_bytes);
#pragma unroll
        for (int c = 0; c < NCHUNK; ++c) {
          ptx::tma_load_3d(X + c * kRegionBytes, &tm_k, &sh.node_full[b], c * 64, hk, t0);
          ptx::tma_load_3d(X + c * kRegionBytes + Np * 128, &tm_q, &sh.node_full[b], c * 64, hk, t0);
        }
        issued = ++i;
        if (i > 1 && !tc_wait(&sh.v_empty, (i - 2) & 1u, sh, a.status)) break;
        ptx::mbar_arrive_expect_tx(&sh.v_full, v_bytes);
        ptx::tma_load_3d(base + lay.v, &tm_v, &sh.v_full, 0, h, t0);
        v_issued = i;
      }
    }
  } else if (warp == kWarpMma) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t id_proj = ptx::idesc_bf16_f32(128, 2 * Np);
      const uint32_t id_gram = ptx::idesc_bf16_f32(128, Np);
      uint32_t u = 0, i = 0;
      for (int p = blockIdx.x; p < npairs; p += gridDim.x) {
        int t0, n, si;
        if (!tc_pair_nodes<SV>(a, sv, p, t0, n, si)) continue;
        const int b = int(i & 1u);
        const uint32_t ph = (i >> 1) & 1u;
        if (!tc_wait(&sh.tmem_empty[b], ph ^ 1u, sh, a.status)) break;
        if (!tc_wait(&sh.node_full[b], ph, sh, a.status)) break;
        ptx::tc_fence_after_sync();
        const uint32_t x0 = ptx::smem_u32(base + lay.x);
        const uint32_t d1 = tmem + uint32_t(b) * kTmemBuf, d2 = d1 + kGramCol;
        // Gram: A = all 128 rows of X, B = the key rows
#pragma unroll
        for (int ks = 0; ks < DK / 16; ++ks) {
          const uint64_t dx = ptx::desc_kmajor_sw128(x0 + (ks >> 2) * kRegionBytes + (ks & 3) * 32);
          ptx::mma_bf16_ss(d2, dx, dx, id_gram, ks > 0 ? 1u : 0u);
        }
        mma_any = true;
        ptx::mma_commit(&sh.gram_full[b]);
        // projections through the state, chunk by chunk as the splitters deliver them
        bool ok = true;
        for (int c = 0; c < NCHUNK; ++c, ++u) {
          const int s = int(u % uint32_t(R));
          if (!tc_wait(&sh.slot_split[s], (u / R) & 1u, sh, a.status)) { ok = false; break; }
          ptx::tc_fence_after_sync();
          const uint32_t a_hi = ptx::smem_u32(ring + s * kSlotBytes), a_lo = a_hi + kRegionBytes;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t bx = ptx::desc_kmajor_sw128(x0 + c * kRegionBytes + kk * 32);
            ptx::mma_bf16_ss(d1, ptx::desc_kmajor_sw128(a_hi + kk * 32), bx, id_proj, (c | kk) ? 1u : 0u);
            ptx::mma_bf16_ss(d1, ptx::desc_kmajor_sw128(a_lo + kk * 32), bx, id_proj, 1u);
          }
          ptx::mma_commit(&sh.slot_empty[s]);
        }
        if (!ok) break;
        ptx::mma_commit(&sh.proj_full[b]);
        ++i;
      }
    }
  } else if (warp == kWarpTree) {
    // ------------------------------------------------------------ tree analysis
    uint32_t i = 0;
    for (int p = blockIdx.x; p < npairs; p += gridDim.x) {
      int t0, n, si;
      const int h = p % a.H;
      if (!tc_pair_nodes<SV>(a, sv, p, t0, n, si)) {
        if (lane == 0 && h == 0) {
          if (SV && si < 0) {
            if (si == kBadSlot) report(a.status, GDN_STATUS_BAD_SLOT);
          } else if (!offsets_ok(t0, n, a.T)) report(a.status, GDN_STATUS_BAD_OFFSETS);
          else if (n > a.max_nodes) report(a.status, GDN_STATUS_TOO_MANY_NODES);
        }
        continue;
      }
      const int b = int(i & 1u);
      int ok = 1;
      if (lane == 0) ok = tc_wait(&sh.tree_empty[b], ((i >> 1) & 1u) ^ 1u, sh, a.status);
      if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      ptx::mbar_try_wait(&sh.tree_empty[b], ((i >> 1) & 1u) ^ 1u);  // acquire for every lane
      TreeStage &ts = sh.tree[b];
      int bad = 0;
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int t = lane + 32 * e;
        if (t < n) {
          const int pr = a.parent[t0 + t];
          bad |= (pr < -1 || pr >= t);
          ts.par[t] = pr;
          gate_beta<SV>(sv, a.g, a.beta, size_t(t0 + t) * a.H + h, h, ts.g[t], ts.beta[t]);
        }
      }
      bad = __any_sync(0xffffffffu, bad);
      __syncwarp();
      int cnt[2] = {0, 0};
      if (!bad) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int t = lane + 32 * e;
          if (t < n) {
            // parent indices strictly decrease along the walk, so it ends within t + 1 steps
            unsigned long long m = 1ull << t;
            float Gs = ts.g[t];
            for (int x = ts.par[t]; x >= 0; x = ts.par[x]) {
              m |= 1ull << x;
              Gs += ts.g[x];
            }
            ts.anc[t] = m;
            ts.G[t] = Gs;
            ts.gam[t] = expf(Gs);
            cnt[e] = __popcll(m);
          }
        }
        // exclusive prefix sum of the ancestor counts over t = 0..n-1
        int run = 0, offs[2] = {0, 0};
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          int x = cnt[e];
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
          }
          const int t = lane + 32 * e;
          offs[e] = run + x - cnt[e];
          if (t < n) ts.off[t] = offs[e];
          run += __shfl_sync(0xffffffffu, x, 31);
        }
        // depth, root-to-node path table and depth levels
        int dmax = 0;
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int t = lane + 32 * e;
          if (t < n) {
            const int d = cnt[e] - 1;
            ts.dep[t] = uint8_t(d);
            dmax = max(dmax, d);
            int x = t;
            for (int k = d; k >= 0; --k) {
              ts.pnode[offs[e] + k] = uint8_t(x);
              ts.tnode[offs[e] + k] = uint8_t(t);
              x = ts.par[x];
            }
          }
        }
        __syncwarp();
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int t = lane + 32 * e;
          if (t < n)
            for (int k = 0; k < cnt[e]; ++k) ts.poff[offs[e] + k] = int16_t(ts.off[ts.pnode[offs[e] + k]]);
        }
        dmax = __reduce_max_sync(0xffffffffu, dmax);
        if (lane == 0) {
          ts.maxd = dmax;
          ts.nent = run;
        }
      } else if (lane == 0 && h == 0) {
        report(a.status, GDN_STATUS_BAD_TREE);
      }
      if (lane == 0) ts.bad = bad;
      __syncwarp();
      mbar_arrive(&sh.tree_full[b]);
      ++i;
    }
  } else if (warp >= kWarpEpi && warp < kWarpEpi + kEpiThreads / 32) {
    // ------------------------------------------------------------ epilogue
    const int etid = tid - kWarpEpi * 32;
    const int q4 = warp & 3;                     // TMEM lane quarter this warp may access
    const int half = (warp - kWarpEpi) >> 2;     // two warps share each quarter
    const int row = q4 * 32 + lane;              // TMEM lane: Gram row m, or state column v
    const uint32_t lane_addr = uint32_t(q4 * 32) << 16;
    float *cA = reinterpret_cast<float *>(base + lay.ca);
    float *cP = reinterpret_cast<float *>(base + lay.cp);
    float *cT = reinterpret_cast<float *>(base + lay.ct);
    uint8_t *aop = base + lay.aop;
    uint8_t *bop = base + lay.bop;
    const uint32_t bop_lo = uint32_t(2 * Np * 128);
    const uint32_t id_uo = ptx::idesc_bf16_f32(128, 2 * Np);
    uint32_t i = 0;
    for (int p = blockIdx.x; p < npairs; p += gridDim.x) {
      int t0, n, si;
      if (!tc_pair_nodes<SV>(a, sv, p, t0, n, si)) continue;
      const int h = p % a.H, b = int(i & 1u);
      const uint32_t ph = (i >> 1) & 1u;
      // tree ready (the barrier also ends every epilogue thread's use of the previous pair).
      // Each wait's verdict has its own flag, so no flag is rewritten before every thread has
      // passed a later barrier.
      if (etid == 0) sh.epi_ok[0] = tc_wait(&sh.tree_full[b], ph, sh, a.status);
      named_sync(kBarEpi, kEpiThreads);
      if (!sh.epi_ok[0]) break;
      ptx::mbar_try_wait(&sh.tree_full[b], ph);
      const TreeStage &ts = sh.tree[b];
      const bool live = !ts.bad;
      if (etid == 0) sh.epi_ok[1] = tc_wait(&sh.gram_full[b], ph, sh, a.status);
      named_sync(kBarEpi, kEpiThreads);
      if (!sh.epi_ok[1]) break;
      ptx::mbar_try_wait(&sh.gram_full[b], ph);
      ptx::tc_fence_after_sync();
      const uint32_t d1 = tmem + uint32_t(b) * kTmemBuf + lane_addr, d2 = d1 + kGramCol;

      // (1) raw Gram rows -> the [T ; W] operand bytes, fp32 [2Np][Np] with each row's 16-byte
      // chunks rotated by the row index (fewer bank conflicts); this region is free until (3)
      float *gram = reinterpret_cast<float *>(bop);
      const int nq = Np / 4;  // 16-byte chunks per Gram row
      if (live && q4 * 32 < 2 * Np) {
        for (int c0 = 16 * half; c0 < Np; c0 += 32) {
          float vals[16];
          ptx::tmem_ld_32x32b_x16(d2 + uint32_t(c0), vals);
          if (row < 2 * Np) {
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              const int cq = (c0 / 4 + c + row) % nq;
              *reinterpret_cast<float4 *>(gram + row * Np + cq * 4) =
                  make_float4(vals[4 * c], vals[4 * c + 1], vals[4 * c + 2], vals[4 * c + 3]);
            }
          }
        }
      }
      ptx::tc_fence_before_sync();  // D2 is overwritten by the solve/output MMA below
      named_sync(kBarEpi, kEpiThreads);

      // (2a) masked, gated path coefficients, one thread per path entry e = (t, depth k of j):
      //      A = b_t exp(G_t - G_j) k_t.k_j (0 for j = t),  P = exp(G_t - G_j) q_t.k_j
      const int nent = live ? ts.nent : 0;
      for (int e = etid; e < nent; e += kEpiThreads) {
        const int t = ts.tnode[e], j = ts.pnode[e];
        const float w = __expf(ts.G[t] - ts.G[j]);
        const int cj = ((j >> 2) + t) % nq, cjq = ((j >> 2) + Np + t) % nq;
        const float kk = gram[t * Np + cj * 4 + (j & 3)];
        const float qk = gram[(Np + t) * Np + cjq * 4 + (j & 3)];
        cA[e] = j == t ? 0.f : ts.beta[t] * w * kk;
        cP[e] = w * qk;
      }
      named_sync(kBarEpi, kEpiThreads);

      // (2b) row t of T by a backward sweep in registers, reading only A rows along t's path:
      //      T[t][p_d] = 1,  T[t][p_k] = -sum_{m=k+1..d} T[t][p_m] A[p_m][p_k]
      // Meanwhile the other threads clear the [T ; W] operand (the raw Gram is consumed).
      if (live && etid < n) {
        const int t = etid, d = ts.dep[t], off = ts.off[t];
        if (d < 8) {
          int po[8];
          float x[8];
#pragma unroll
          for (int m = 0; m < 8; ++m) {
            po[m] = m <= d ? ts.poff[off + m] : 0;
            x[m] = m == d ? 1.f : 0.f;
          }
#pragma unroll
          for (int k = 6; k >= 0; --k) {
            if (k < d) {
              float sum = 0.f;
#pragma unroll
              for (int m = k + 1; m < 8; ++m)
                if (m <= d) sum = fmaf(x[m], cA[po[m] + k], sum);
              x[k] = -sum;
            }
          }
#pragma unroll
          for (int m = 0; m < 8; ++m)
            if (m <= d) cT[off + m] = x[m];
        } else {  // paths deeper than eight levels: the same sweep through shared memory
          cT[off + d] = 1.f;
          for (int k = d - 1; k >= 0; --k) {
            float sum = 0.f;
            for (int m = k + 1; m <= d; ++m) sum = fmaf(cT[off + m], cA[ts.poff[off + m] + k], sum);
            cT[off + k] = -sum;
          }
        }
      }
      for (int z = etid; z < int(bop_lo) / 8; z += kEpiThreads)  // hi and lo halves: 2 * bop_lo bytes
        reinterpret_cast<uint4 *>(bop)[z] = make_uint4(0u, 0u, 0u, 0u);
      named_sync(kBarEpi, kEpiThreads);

      // (3) W = P T, one thread per path entry: W[t][p_k] = sum_{m=k..d} P[t][p_m] T[p_m][p_k].
      // T and W go into the dense [T ; W] operand (row t and Np + t, column p_k), bf16 hi + lo.
      for (int e = etid; e < nent; e += kEpiThreads) {
        const int t = ts.tnode[e], j = ts.pnode[e], off = ts.off[t], d = ts.dep[t], k = e - off;
        float sum = 0.f;
        for (int m = k; m <= d; ++m) sum = fmaf(cP[off + m], cT[ts.poff[off + m] + k], sum);
        const float tv = cT[e];
        const __nv_bfloat16 th = __float2bfloat16_rn(tv), tl = __float2bfloat16_rn(tv - __bfloat162float(th));
        const __nv_bfloat16 wh = __float2bfloat16_rn(sum), wl = __float2bfloat16_rn(sum - __bfloat162float(wh));
        const int rt = t, rw = Np + t;
        const uint32_t ot = uint32_t(rt * 128 + ((((j * 2) >> 4) ^ (rt & 7)) << 4) + ((j * 2) & 15));
        const uint32_t ow = uint32_t(rw * 128 + ((((j * 2) >> 4) ^ (rw & 7)) << 4) + ((j * 2) & 15));
        *reinterpret_cast<__nv_bfloat16 *>(bop + ot) = th;
        *reinterpret_cast<__nv_bfloat16 *>(bop + bop_lo + ot) = tl;
        *reinterpret_cast<__nv_bfloat16 *>(bop + ow) = wh;
        *reinterpret_cast<__nv_bfloat16 *>(bop + bop_lo + ow) = wl;
      }

      // (4) projections ready: R = b (v - gamma KS) -> the R^T operand (row v, column t), as
      // bf16 hi + lo; columns t >= n are zero. The packed coefficients in these bytes are dead.
      if (etid == 0)
        sh.epi_ok[2] = tc_wait(&sh.proj_full[b], ph, sh, a.status) && tc_wait(&sh.v_full, i & 1u, sh, a.status);
      named_sync(kBarEpi, kEpiThreads);
      if (!sh.epi_ok[2]) break;
      ptx::mbar_try_wait(&sh.proj_full[b], ph);
      ptx::mbar_try_wait(&sh.v_full, i & 1u);
      ptx::tc_fence_after_sync();
      const int v = row;
      const bool col = live && q4 * 32 < DV;
      if (col) {
        const uint16_t *Vs = reinterpret_cast<const uint16_t *>(base + lay.v);
        for (int c0 = 16 * half; c0 < Np; c0 += 32) {
          float ks[16];
          ptx::tmem_ld_32x32b_x16(d1 + uint32_t(c0), ks);
#pragma unroll
          for (int g8 = 0; g8 < 2; ++g8) {
            uint32_t hi[4], lo[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              float r2[2];
#pragma unroll
              for (int z = 0; z < 2; ++z) {
                const int jj = g8 * 8 + 2 * e + z, t = c0 + jj;
                r2[z] = t < n ? ts.beta[t] * (bf16_to_f32(Vs[t * DV + v]) - ts.gam[t] * ks[jj]) : 0.f;
              }
              const __nv_bfloat162 h2 = __floats2bfloat162_rn(r2[0], r2[1]);
              const float2 hf = __bfloat1622float2(h2);
              const __nv_bfloat162 l2 = __floats2bfloat162_rn(r2[0] - hf.x, r2[1] - hf.y);
              hi[e] = *reinterpret_cast<const uint32_t *>(&h2);
              lo[e] = *reinterpret_cast<const uint32_t *>(&l2);
            }
            const int kc = (c0 >> 3) + g8;  // 16-byte chunk along K (8 nodes)
            const uint32_t off = uint32_t(v * 128 + ((kc ^ (v & 7)) << 4));
            *reinterpret_cast<uint4 *>(aop + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
            *reinterpret_cast<uint4 *>(aop + kRegionBytes + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
          }
        }
      }
      ptx::fence_proxy_async_smem();  // R^T and [T ; W] feed the MMA (async proxy)
      named_sync(kBarEpi, kEpiThreads);
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh.v_empty);

      // (5) D3 = R^T [T ; W]^T: three bf16 products (hi hi, hi lo, lo hi), fp32 accumulate
      if (etid == 0) {
        ptx::tc_fence_after_sync();
        const uint32_t a0 = ptx::smem_u32(aop), b0 = ptx::smem_u32(bop);
        const uint32_t d3 = tmem + uint32_t(b) * kTmemBuf + kGramCol;
        for (int ks = 0; ks < Np / 16; ++ks) {
          const uint64_t ah = ptx::desc_kmajor_sw128(a0 + ks * 32), al = ptx::desc_kmajor_sw128(a0 + kRegionBytes + ks * 32);
          const uint64_t bh = ptx::desc_kmajor_sw128(b0 + ks * 32), bl = ptx::desc_kmajor_sw128(b0 + bop_lo + ks * 32);
          ptx::mma_bf16_ss(d3, ah, bh, id_uo, ks > 0 ? 1u : 0u);
          ptx::mma_bf16_ss(d3, ah, bl, id_uo, 1u);
          ptx::mma_bf16_ss(d3, al, bh, id_uo, 1u);
        }
        ptx::mma_commit(&sh.uo_full);
        mma_any = true;
        sh.epi_ok[0] = tc_wait(&sh.uo_full, i & 1u, sh, a.status);
      }
      named_sync(kBarEpi, kEpiThreads);
      if (!sh.epi_ok[0]) break;
      ptx::mbar_try_wait(&sh.uo_full, i & 1u);
      ptx::tc_fence_after_sync();

      // (6) u_t = D3[:, t], o_t = gamma_t QS_t + D3[:, Np + t]
      if (col) {
        const uint32_t d3 = d2;
        for (int c0 = 16 * half; c0 < n; c0 += 32) {
          float uu[16], ww[16], qs[16];
          ptx::tmem_ld_32x32b_x16(d3 + uint32_t(c0), uu);
          ptx::tmem_ld_32x32b_x16(d3 + uint32_t(Np + c0), ww);
          ptx::tmem_ld_32x32b_x16(d1 + uint32_t(Np + c0), qs);
#pragma unroll
          for (int jj = 0; jj < 16; ++jj) {
            const int t = c0 + jj;
            if (t < n) {
              const size_t o_row = (size_t(t0 + t) * a.H + h) * DV + v;
              const float ov = fmaf(ts.gam[t], qs[jj], ww[jj]);
              __stcs(a.o + o_row, SV ? query_scale<SV>(sv) * ov : ov);  // o is linear in q
              __stcs(a.U + o_row, uu[jj]);
            }
          }
        }
      }
      if (live && etid < n) a.G[size_t(t0 + etid) * a.H + h] = ts.G[etid];
      ptx::tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&sh.tmem_empty[b]);
        mbar_arrive(&sh.tree_empty[b]);
      }
      ++i;
    }
  } else if (warp >= kWarpSplit) {
    // ------------------------------------------------------------ splitters
    const int stid = tid - kWarpSplit * 32;
    constexpr int TPT = DV * 8 / kSplitThreads;  // (column, 8-row group) tasks per thread
    const int v = stid % DV, kc0 = stid / DV;
    constexpr int KCSTEP = kSplitThreads / DV;
    uint32_t u = 0;
    for (int p = blockIdx.x; p < npairs; p += gridDim.x) {
      int t0, n, si;
      if (!tc_pair_nodes<SV>(a, sv, p, t0, n, si)) continue;
      bool ok = true;
      for (int c = 0; c < NCHUNK; ++c, ++u) {
        const int s = int(u % uint32_t(R));
        const uint32_t ph = (u / R) & 1u;
        if (stid == 0) sh.split_ok = tc_wait(&sh.slot_full[s], ph, sh, a.status);
        named_sync(kBarSplit, kSplitThreads);
        if (!sh.split_ok) { ok = false; break; }
        ptx::mbar_wait(&sh.slot_full[s], ph, kWaitLimitNs);  // completes at once: acquire for this thread
        uint8_t *slot = ring + s * kSlotBytes;
        const float *xf = reinterpret_cast<const float *>(slot);
        float x[TPT][8];
#pragma unroll
        for (int m = 0; m < TPT; ++m)
#pragma unroll
          for (int e = 0; e < 8; ++e) x[m][e] = xf[((kc0 + m * KCSTEP) * 8 + e) * DV + v];
        named_sync(kBarSplit, kSplitThreads);  // every fp32 read is done before the in-place writes
#pragma unroll
        for (int m = 0; m < TPT; ++m) {
          const int kc = kc0 + m * KCSTEP;
          uint32_t hi[4], lo[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const __nv_bfloat162 h2 = __floats2bfloat162_rn(x[m][2 * e], x[m][2 * e + 1]);
            const float2 hf = __bfloat1622float2(h2);
            const __nv_bfloat162 l2 = __floats2bfloat162_rn(x[m][2 * e] - hf.x, x[m][2 * e + 1] - hf.y);
            hi[e] = *reinterpret_cast<const uint32_t *>(&h2);
            lo[e] = *reinterpret_cast<const uint32_t *>(&l2);
          }
          const uint32_t off = v * 128 + ((kc ^ (v & 7)) << 4);
          *reinterpret_cast<uint4 *>(slot + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
          *reinterpret_cast<uint4 *>(slot + kRegionBytes + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
        }
        ptx::fence_proxy_async_smem();
        named_sync(kBarSplit, kSplitThreads);
        if (stid == 0) mbar_arrive(&sh.slot_split[s]);
      }
      if (!ok) break;
    }
  }

  // ---------------------------------------------------------------- clean-up
  __syncthreads();
  if (warp == kWarpState && lane == 0) {
    // let every issued state copy land before the shared memory goes away
    for (int s = 0; s < R; ++s) {
      if (issued > uint32_t(s)) {
        const uint32_t last = issued - 1 - ((issued - 1 - uint32_t(s)) % uint32_t(R));
        ptx::mbar_wait(&sh.slot_full[s], (last / R) & 1u, kWaitLimitNs);
      }
    }
  }
  if (warp == kWarpNodes && lane == 0) {
    for (int b = 0; b < 2; ++b) {
      if (issued > uint32_t(b)) {
        const uint32_t last = issued - 1 - ((issued - 1 - uint32_t(b)) % 2u);
        ptx::mbar_wait(&sh.node_full[b], (last >> 1) & 1u, kWaitLimitNs);
      }
    }
    if (v_issued > 0) ptx::mbar_wait(&sh.v_full, (v_issued - 1) & 1u, kWaitLimitNs);
  }
  if (warp == kWarpMma && lane == 0 && mma_any) {
    ptx::mma_commit(&sh.drain);
    ptx::mbar_wait(&sh.drain, 0, kWaitLimitNs);
  }
  if (tid == kWarpEpi * 32 && mma_any) {
    ptx::mma_commit(&sh.drain_epi);
    ptx::mbar_wait(&sh.drain_epi, 0, kWaitLimitNs);
  }
  ptx::tc_fence_before_sync();
  __syncthreads();
  if (warp == kWarpMma) {
    ptx::tc_fence_after_sync();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace gdn
