// Tensor-core tree verify for sm_103a: the tree-structured WY form of the gated delta rule
// (TreeWY, method section). Persistent, warp-specialised: one CTA per SM walks the
// (request, head) pairs p = blockIdx.x, blockIdx.x + gridDim.x, ... through a pipeline.
//
// Per pair (X = [K ; Q], the node block, rows 0..Np-1 = keys, Np..2Np-1 = queries):
//   projections  D1[v][n] = sum_k S0[v][k] X[n][k]  -> KS = D1[:, 0:Np], QS = D1[:, Np:2Np]
//   Gram         D2[m][j] = sum_k X[m][k] K[j][k]   -> k_t.k_j (m = t), q_t.k_j (m = Np + t)
//   masks        A[t,j] = b_t exp(G_t - G_j) k_t.k_j   (j a strict ancestor of t)
//                P[t,j] = exp(G_t - G_j) q_t.k_j       (j an ancestor of t, or t)
//   solve        (I + A) U = R,  R_t = b_t (v_t - gamma_t KS_t)   one state column per thread
//   outputs      o_t = gamma_t QS_t + sum_j P[t,j] u_j
//
// Warp roles (512 threads):
//   warp 0       state producer: 1-D bulk copies (cp.async.bulk) of 64-row fp32 chunks of the
//                state into a ring of 32 KiB shared-memory slots
//   warp 1       node producer: TMA (cp.async.bulk.tensor) of the K and Q rows straight into the
//                128-byte-swizzled K-major UMMA operand layout, and of the v rows, double-buffered
//   warp 2       MMA issuer (one thread) and tensor-memory owner: tcgen05.mma kind::f16, fp32
//                accumulators in TMEM, two buffers of 256 columns so the epilogue of one pair
//                overlaps the MMAs of the next
//   warp 3       tree analysis: parent check, 64-bit ancestor masks, cumulative log-gates and the
//                packed offsets of the ancestor coefficients, double-buffered
//   warps 4-7    epilogue: Gram rows from TMEM -> masked, gated coefficients in shared memory;
//                then one state column per thread (TMEM lane = column): R, forward substitution,
//                outputs, coalesced stores of o and U
//   warps 8-15   splitters: each fp32 chunk is split in place into bf16 hi + lo parts
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
constexpr int kTcThreads = 512;
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
  kEpiThreads = 128,
  kWarpSplit = 8,
  kSplitThreads = 256,
};

enum : int { kBarSplit = 1, kBarEpi = 2 };  // named barriers (0 is __syncthreads)

// Shared-memory carve-up (byte offsets from a 1024-byte-aligned base).
struct TcLayout {
  int Np, R, u_in_x;
  uint32_t ring, x, v, ap, u, total;
};

__host__ __device__ inline uint32_t align_up(uint32_t x, uint32_t a) { return (x + a - 1) / a * a; }

__host__ __device__ inline TcLayout tc_layout(int DK, int DV, int Np, int R) {
  TcLayout L{};
  L.Np = Np;
  L.R = R;
  uint32_t off = 0;
  L.ring = off;
  off += uint32_t(R) * kSlotBytes;
  L.x = off;
  off += 2u * uint32_t(DK / 64) * kRegionBytes;
  L.v = off;
  off = align_up(off + 2u * uint32_t(Np) * DV * 2, 1024);
  L.ap = off;
  off = align_up(off + uint32_t(Np) * (Np + 1) / 2 * 8, 1024);
  const uint32_t u_bytes = uint32_t(Np) * DV * 4;
  L.u_in_x = u_bytes <= uint32_t(DK / 64) * kRegionBytes;
  L.u = L.u_in_x ? L.x : off;
  if (!L.u_in_x) off += u_bytes;
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
  int off[kMaxNodes + 1];             // packed ancestor-coefficient offsets
  int bad;
};

struct TcShared {
  TreeStage tree[2];
  uint64_t slot_full[kMaxRing], slot_split[kMaxRing], slot_empty[kMaxRing];
  uint64_t node_full[2], node_empty[2], gram_full[2], proj_full[2], tmem_empty[2];
  uint64_t tree_full[2], tree_empty[2], drain;
  uint32_t tmem_base;
  int abort_flag;
  int split_ok, epi_ok[3];
};

// Nodes of pair p; false for a pair that is skipped (empty, too many nodes, bad offsets).
__device__ __forceinline__ bool tc_pair_nodes(const VerifyArgs &a, int p, int &t0, int &n) {
  const int r = p / a.H;
  t0 = a.cu_nodes[r];
  n = a.cu_nodes[r + 1] - t0;
  return offsets_ok(t0, n, a.T) && n > 0 && n <= a.max_nodes;
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

template <int DK, int DV>
__global__ void __launch_bounds__(kTcThreads, 1)
    verify_tc_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_q,
                     const __grid_constant__ CUtensorMap tm_v, VerifyArgs a, TcLayout lay) {
  static_assert(DK == 64 || DK == 128, "tensor-core verify needs d_k in {64, 128}");
  static_assert(DV == 64 || DV == 128, "tensor-core verify needs d_v in {64, 128}");
  constexpr int NCHUNK = DK / kChunkRows;              // ring slots per pair
  constexpr uint32_t kChunkBytes = kChunkRows * DV * 4;  // fp32 bytes of one chunk
  constexpr uint32_t kXBytes = NCHUNK * kRegionBytes;  // one node stage of the X operand

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
      ptx::mbar_init(&sh.node_empty[b], kEpiThreads / 32);
      ptx::mbar_init(&sh.gram_full[b], 1);
      ptx::mbar_init(&sh.proj_full[b], 1);
      ptx::mbar_init(&sh.tmem_empty[b], kEpiThreads / 32);
      ptx::mbar_init(&sh.tree_full[b], 32);
      ptx::mbar_init(&sh.tree_empty[b], kEpiThreads / 32);
    }
    ptx::mbar_init(&sh.drain, 1);
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
  bool mma_any = false;

  if (warp == kWarpState) {
    // ------------------------------------------------------------ state producer
    if (lane == 0) {
      uint32_t u = 0;
      for (int p = blockIdx.x; p < npairs; p += gridDim.x) {
        int t0, n;
        if (!tc_pair_nodes(a, p, t0, n)) continue;
        const uint8_t *src = reinterpret_cast<const uint8_t *>(a.ST + size_t(p) * DK * DV);
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
      const uint32_t node_bytes = uint32_t(2 * DK + DV) * Np * 2;
      uint32_t i = 0;
      for (int p = blockIdx.x; p < npairs; p += gridDim.x) {
        int t0, n;
        if (!tc_pair_nodes(a, p, t0, n)) continue;
        const int h = p % a.H, b = int(i & 1u);
        if (!tc_wait(&sh.node_empty[b], ((i >> 1) & 1u) ^ 1u, sh, a.status)) break;
        uint8_t *X = base + lay.x + b * kXBytes;
        ptx::mbar_arrive_expect_tx(&sh.node_full[b], node_bytes);
#pragma unroll
        for (int c = 0; c < NCHUNK; ++c) {
          ptx::tma_load_3d(X + c * kRegionBytes, &tm_k, &sh.node_full[b], c * 64, h, t0);
          ptx::tma_load_3d(X + c * kRegionBytes + Np * 128, &tm_q, &sh.node_full[b], c * 64, h, t0);
        }
        ptx::tma_load_3d(base + lay.v + b * (Np * DV * 2), &tm_v, &sh.node_full[b], 0, h, t0);
        issued = ++i;
      }
    }
  } else if (warp == kWarpMma) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t id_proj = ptx::idesc_bf16_f32(128, 2 * Np);
      const uint32_t id_gram = ptx::idesc_bf16_f32(128, Np);
      uint32_t u = 0, i = 0;
      for (int p = blockIdx.x; p < npairs; p += gridDim.x) {
        int t0, n;
        if (!tc_pair_nodes(a, p, t0, n)) continue;
        const int b = int(i & 1u);
        const uint32_t ph = (i >> 1) & 1u;
        if (!tc_wait(&sh.tmem_empty[b], ph ^ 1u, sh, a.status)) break;
        if (!tc_wait(&sh.node_full[b], ph, sh, a.status)) break;
        ptx::tc_fence_after_sync();
        const uint32_t x0 = ptx::smem_u32(base + lay.x + b * kXBytes);
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
      int t0, n;
      const int h = p % a.H;
      if (!tc_pair_nodes(a, p, t0, n)) {
        if (lane == 0 && h == 0) {
          if (!offsets_ok(t0, n, a.T)) report(a.status, GDN_STATUS_BAD_OFFSETS);
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
          ts.g[t] = a.g[size_t(t0 + t) * a.H + h];
          ts.beta[t] = a.beta[size_t(t0 + t) * a.H + h];
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
        int run = 0;
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          int x = cnt[e];
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
          }
          const int t = lane + 32 * e;
          if (t < n) ts.off[t] = run + x - cnt[e];
          run += __shfl_sync(0xffffffffu, x, 31);
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
    const int q4 = warp & 3;                // TMEM lane quarter this warp may access
    const int row = q4 * 32 + lane;         // TMEM lane: Gram row m, or state column v
    const uint32_t lane_addr = uint32_t(q4 * 32) << 16;
    float2 *ap = reinterpret_cast<float2 *>(base + lay.ap);
    uint32_t i = 0;
    for (int p = blockIdx.x; p < npairs; p += gridDim.x) {
      int t0, n;
      if (!tc_pair_nodes(a, p, t0, n)) continue;
      const int h = p % a.H, b = int(i & 1u);
      const uint32_t ph = (i >> 1) & 1u;
      // tree ready (the barrier also ends every epilogue thread's use of the previous pair)
      // (each wait's verdict has its own flag, so no flag is rewritten before every thread
      // has passed a later barrier)
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
      // masked, gated ancestor coefficients: packed {A, P} per (t, ancestor-or-self j)
      if (live && q4 * 32 < 2 * Np) {
        const bool krow = row < n;
        const bool qrow = row >= Np && row - Np < n;
        const int t = krow ? row : row - Np;
        const unsigned long long anc = (krow || qrow) ? ts.anc[t] : 0ull;
        const float Gt = (krow || qrow) ? ts.G[t] : 0.f;
        const float bt = krow ? ts.beta[t] : 0.f;
        const int off = (krow || qrow) ? ts.off[t] : 0;
        for (int c0 = 0; c0 < Np; c0 += 16) {
          float vals[16];
          ptx::tmem_ld_32x32b_x16(d2 + uint32_t(c0), vals);
#pragma unroll
          for (int jj = 0; jj < 16; ++jj) {
            const int j = c0 + jj;
            if (j < 64 && ((anc >> j) & 1ull)) {
              const int idx = __popcll(anc & ((1ull << j) - 1ull));
              const float w = expf(Gt - ts.G[j]);
              if (krow && j < t) ap[off + idx].x = bt * w * vals[jj];
              if (qrow) ap[off + idx].y = w * vals[jj];
            }
          }
        }
      }
      named_sync(kBarEpi, kEpiThreads);  // coefficients ready
      if (etid == 0) sh.epi_ok[2] = tc_wait(&sh.proj_full[b], ph, sh, a.status);
      named_sync(kBarEpi, kEpiThreads);
      if (!sh.epi_ok[2]) break;
      ptx::mbar_try_wait(&sh.proj_full[b], ph);
      ptx::tc_fence_after_sync();
      if (live && q4 * 32 < DV) {
        const int v = row;
        float *Ub = reinterpret_cast<float *>(base + lay.u + (lay.u_in_x ? b * kXBytes : 0u));
        const uint16_t *Vs = reinterpret_cast<const uint16_t *>(base + lay.v + b * (Np * DV * 2));
        // R = b (v - gamma KS)
        for (int c0 = 0; c0 < n; c0 += 16) {
          float ks[16];
          ptx::tmem_ld_32x32b_x16(d1 + uint32_t(c0), ks);
#pragma unroll
          for (int jj = 0; jj < 16; ++jj) {
            const int t = c0 + jj;
            if (t < n) Ub[t * DV + v] = ts.beta[t] * (bf16_to_f32(Vs[t * DV + v]) - ts.gam[t] * ks[jj]);
          }
        }
        // forward substitution over the ancestors (parent-before-child order)
        for (int t = 0; t < n; ++t) {
          float uu = Ub[t * DV + v];
          unsigned long long m = ts.anc[t] & ~(1ull << t);
          const float2 *c = ap + ts.off[t];
          while (m) {
            const int j = __ffsll(m) - 1;
            m &= m - 1;
            uu = fmaf(-(c++)->x, Ub[j * DV + v], uu);
          }
          Ub[t * DV + v] = uu;
        }
        // outputs
        for (int c0 = 0; c0 < n; c0 += 16) {
          float qs[16];
          ptx::tmem_ld_32x32b_x16(d1 + uint32_t(Np + c0), qs);
#pragma unroll
          for (int jj = 0; jj < 16; ++jj) {
            const int t = c0 + jj;
            if (t < n) {
              float out = ts.gam[t] * qs[jj];
              unsigned long long m = ts.anc[t];
              const float2 *c = ap + ts.off[t];
              while (m) {
                const int j = __ffsll(m) - 1;
                m &= m - 1;
                out = fmaf((c++)->y, Ub[j * DV + v], out);
              }
              const size_t o_row = (size_t(t0 + t) * a.H + h) * DV + v;
              __stcs(a.o + o_row, out);
              __stcs(a.U + o_row, Ub[t * DV + v]);
            }
          }
        }
      }
      if (live && etid < n) a.G[size_t(t0 + etid) * a.H + h] = ts.G[etid];
      ptx::tc_fence_before_sync();
      ptx::fence_proxy_async_smem();  // U was written into the node stage the TMA reuses
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&sh.tmem_empty[b]);
        mbar_arrive(&sh.node_empty[b]);
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
      int t0, n;
      if (!tc_pair_nodes(a, p, t0, n)) continue;
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
  }
  if (warp == kWarpMma && lane == 0 && mma_any) {
    ptx::mma_commit(&sh.drain);
    ptx::mbar_wait(&sh.drain, 0, kWaitLimitNs);
  }
  ptx::tc_fence_before_sync();
  __syncthreads();
  if (warp == kWarpMma) {
    ptx::tc_fence_after_sync();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace gdn
