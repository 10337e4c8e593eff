// Tensor-core tree verify for sm_103a: the tree-structured WY form of the gated delta rule
// (TreeWY, method section). Persistent, warp-specialised: one CTA per SM walks the
// (request, head) pairs p = blockIdx.x, blockIdx.x + gridDim.x, ... through a pipeline.
//
// Per pair (X = [K ; Q], the node block, rows 0..Np-1 = keys, Np..2Np-1 = queries):
//   projections  D1[v][n] = sum_k S0[v][k] X[n][k]  -> KS = D1[:, 0:Np], QS = D1[:, Np:2Np]
//   Gram         D2[m][j] = sum_k X[m][k] K[j][k]   -> k_t.k_j (m = t), q_t.k_j (m = Np + t)
//   masks        A[t,j] = b_t exp(G_t - G_j) k_t.k_j   (j a strict ancestor of t)
//                P[t,j] = exp(G_t - G_j) q_t.k_j       (j an ancestor of t, or t)
//                where exp(G_t - G_j) is the product of the gates a = exp(g) along the path
//                below j, so no factor exceeds 1
//   inverse      T = (I + A)^-1 and W = P T. Both keep the ancestor pattern: on t's root-to-node
//                path p_0 .. p_d = t, row t of T solves x (I + A_path) = e_d and row t of W solves
//                w (I + A_path) = P[t, path], one backward substitution each, in one thread
//   solve+out    D3[v][n] = sum_j R[j][v] [T ; W][n][j],  R_t = b_t (v_t - gamma_t KS_t):
//                u_t = D3[:, t], o_t = gamma_t QS_t + D3[:, Np + t]. tcgen05.mma with R^T in
//                tensor memory and [T ; W] in shared memory, both split into bf16 hi + lo
//                (three products), fp32 accumulate in TMEM
//
// Warp roles (640 threads):
//   warp 0       state producer: 1-D bulk copies (cp.async.bulk) of 64-row fp32 chunks of the
//                state into a ring of 32 KiB shared-memory slots
//   warp 1       node producer: TMA (cp.async.bulk.tensor) of the K and Q rows straight into the
//                128-byte-swizzled K-major UMMA operand layout (one buffer, refilled once the
//                previous pair's MMAs are done), and of the v rows (one buffer, refilled once
//                the previous pair's R is formed)
//   warp 2       MMA issuer for the projections and the Gram (one thread) and tensor-memory
//                owner: tcgen05.mma kind::f16, fp32 accumulators in TMEM. The 512 columns form
//                2 stages (up to 32 nodes per request: 4) of projections, Gram and outputs, so
//                the epilogues of earlier pairs overlap the MMAs of later ones
//   warp 3       tree analysis: parent check, 64-bit ancestor masks, cumulative log-gates, depths
//                and packed per-path offsets, double-buffered
//   warps 4-7    coefficient group: raw Gram rows from TMEM to shared memory; then rows of T
//                and W, two threads per node, each forming the masked, gated path coefficients
//                of its own root-to-node path, into the [T ; W] operand
//   warps 8-11   R / output group: R = b (v - gamma KS) from TMEM, written back to TMEM as the
//                bf16 hi / lo A operand of the solve/output MMA over the dead KS columns; that
//                MMA; then o and U to HBM
//   warps 12-19  splitters: each fp32 chunk is split in place into bf16 hi + lo parts
//                (S = hi + lo + O(2^-17 |S|)) written as the K-major, 128-byte-swizzled UMMA A
//                operand; two MMAs per K slice (hi, lo) give fp32-accurate products against
//                the exact bf16 q / k
// The two epilogue groups meet once per pair (an mbarrier): while the output group finishes
// pair i, the coefficient group already works on pair i+1.
// Every wait on an mbarrier is bounded (1 s); a role that gives up raises a CTA-wide abort
// flag and GDN_STATUS_TIMEOUT, all roles leave their loops, the CTA waits (bounded) for its
// copies and MMAs in flight, frees its tensor memory and returns.
#pragma once

#include "bounds.cuh"
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
constexpr uint32_t kTmemCols = 512;       // split into 2 or 4 pipeline stages
constexpr int kMaxStages = 4;
constexpr int kRegPath = 9;               // root-to-node paths of up to 9 nodes are solved in registers

enum : int {
  kWarpState = 0,
  kWarpNodes = 1,
  kWarpMma = 2,
  kWarpTree = 3,
  kWarpCoef = 4,   // coefficient group: warps 4-7
  kWarpOut = 8,    // R / output group: warps 8-11
  kGroupThreads = 128,
  kWarpSplit = 12,
  kSplitThreads = 256,
};

enum : int { kBarSplit = 1, kBarCoef = 2, kBarOut = 3 };  // named barriers (0 is __syncthreads)

// Shared-memory carve-up (byte offsets from a 1024-byte-aligned base).
//   ring   R slots of 32 KiB: fp32 state chunks, split in place to the bf16 hi / lo A operand
//   x      the [K ; Q] B operand of the projections and the A / B operands of the Gram
//   v      v rows (bf16)
//   bop    [T ; W] as the B operand of the solve/output MMA (hi, lo: 2 Np rows x 128 B each)
//   gram   the raw Gram rows copied out of TMEM (fp32 [2 Np][Np + 4]: row t = k_t . k_j, row
//          Np + t = q_t . k_j; the 4-float pad spreads each row's 16-byte chunks over the banks)
struct TcLayout {
  int Np, R, ns;  // node capacity (multiple of 16), ring slots, pipeline stages (2 or 4)
  uint32_t ring, x, v, bop, gram, total;
};

__host__ __device__ inline uint32_t align_up(uint32_t x, uint32_t a) { return (x + a - 1) / a * a; }

__host__ __device__ inline TcLayout tc_layout(int DK, int DV, int Np, int R) {
  TcLayout L{};
  L.Np = Np;
  L.R = R;
  L.ns = Np <= 32 ? 4 : 2;  // a stage holds 4 Np TMEM columns (projections, Gram / outputs)
  uint32_t off = 0;
  L.ring = off;
  off += uint32_t(R) * kSlotBytes;
  L.x = off;
  off += uint32_t(DK / 64) * kRegionBytes;
  L.v = off;
  off = align_up(off + uint32_t(Np) * DV * 2, 1024);
  L.bop = off;
  off += 2u * 2u * uint32_t(Np) * 128u;
  L.gram = off;
  off += 2u * uint32_t(Np) * uint32_t(Np + 4) * 4u;
  L.total = off;
  return L;
}

// Per-pair tree analysis, double-buffered between the tree warp and the epilogue groups.
struct __align__(16) TreeStage {
  unsigned long long anc[kMaxNodes];  // bit j <=> j on t's root-to-node path (t included)
  float G[kMaxNodes];                 // cumulative log-gate
  float gam[kMaxNodes];               // exp(G)
  float beta[kMaxNodes];
  float a[kMaxNodes];                 // exp(g): the node's gate
  int par[kMaxNodes];
  uint8_t dep[kMaxNodes];
  uint8_t pj[kMaxNodes][12];          // paths of up to kRegPath nodes: p_0 .. p_d, then t repeated
  int bad;
};

struct TcShared {
  TreeStage tree[kMaxStages];
  uint64_t slot_full[kMaxRing], slot_split[kMaxRing], slot_empty[kMaxRing];
  uint64_t node_full[2], v_full, v_empty, gram_full[kMaxStages], proj_full[kMaxStages], tmem_empty[kMaxStages];
  uint64_t uo_full, coef_done, tree_full[kMaxStages], tree_empty[kMaxStages], drain, drain_out;
  uint32_t tmem_base;
  int abort_flag;
  int split_ok, coef_ok[2], out_ok[2];
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

// Bounded wait that also gives up when another role has raised the abort flag. Not inlined: the
// kernel's roles together run more code than the instruction caches hold, so every call site
// shares one copy.
__device__ __noinline__ bool tc_wait(uint64_t *bar, uint32_t parity, TcShared &sh, int32_t *status) {
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

// Byte offset of element (row r, column j) of a bf16 K-major operand in the 128-byte swizzle
// layout (rows of 128 B, 16-byte chunks XOR-ed with the row index mod 8).
__device__ __forceinline__ uint32_t sw128_bf16(int r, int j) {
  return uint32_t(r * 128 + ((((j * 2) >> 4) ^ (r & 7)) << 4) + ((j * 2) & 15));
}

// Round to bf16 (nearest even) by the hardware conversion.
__device__ __forceinline__ uint16_t f32_to_bf16_rn(float x) {
  uint16_t b;
  asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(b) : "f"(x));
  return b;
}

// Store z as bf16 hi + lo at (row r, column j) of the [T ; W] operand.
__device__ __forceinline__ void put_hilo(uint8_t *bop, uint32_t lo_off, int r, int j, float z) {
  const uint16_t h = f32_to_bf16_rn(z);
  const uint16_t l = f32_to_bf16_rn(z - __uint_as_float(uint32_t(h) << 16));
  const uint32_t o = sw128_bf16(r, j);
  *reinterpret_cast<uint16_t *>(bop + o) = h;
  *reinterpret_cast<uint16_t *>(bop + lo_off + o) = l;
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
  // pair i uses stage i mod ns (TMEM columns, tree analysis), phase parity (i / ns) mod 2
  const int lgns = lay.ns == 4 ? 2 : 1;
  const uint32_t nsm = uint32_t(lay.ns - 1);
  const uint32_t bufcols = kTmemCols >> lgns, gcol = bufcols / 2;
  uint8_t *ring = base + lay.ring;

  if (tid == 0) {
    for (int s = 0; s < R; ++s) {
      ptx::mbar_init(&sh.slot_full[s], 1);
      ptx::mbar_init(&sh.slot_split[s], 1);
      ptx::mbar_init(&sh.slot_empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) ptx::mbar_init(&sh.node_full[b], 1);
    for (int b = 0; b < kMaxStages; ++b) {
      ptx::mbar_init(&sh.gram_full[b], 1);
      ptx::mbar_init(&sh.proj_full[b], 1);
      ptx::mbar_init(&sh.tmem_empty[b], 2 * kGroupThreads / 32);  // every warp of both epilogue groups
      ptx::mbar_init(&sh.tree_full[b], 32);
      ptx::mbar_init(&sh.tree_empty[b], 2 * kGroupThreads / 32);
    }
    ptx::mbar_init(&sh.v_full, 1);
    ptx::mbar_init(&sh.v_empty, kGroupThreads / 32);
    ptx::mbar_init(&sh.uo_full, 1);
    ptx::mbar_init(&sh.coef_done, kGroupThreads / 32);
    ptx::mbar_init(&sh.drain, 1);
    ptx::mbar_init(&sh.drain_out, 1);
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
  bool mma_any = false;  // the MMA warp (projections, Gram) or output-group thread 0 (solve/output) issued MMAs

  if (warp == kWarpState) {
    // ------------------------------------------------------------ state producer
    if (lane == 0) {
      uint32_t u = 0;
      for (int p = blockIdx.x; p < npairs; p += gridDim.x) {
        int t0, n, si;
        if (!tc_pair_nodes<SV>(a, sv, p, t0, n, si)) continue;
        const size_t st_idx = SV ? size_t(si) * a.H + p % a.H : size_t(p);
        // (a skipped state leaves its slots unfilled: the pair's waits time out and report it)
        if (!range_in_bounds((long long)(st_idx * DK * DV), DK * DV, state_count<SV>(sv, a.B) * a.H * DK * DV,
                             a.status))
          break;
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
        // pull this pair's node rows into L2 first: the copies below start only once the buffers
        // are free, and would otherwise queue behind the state ring's loads
#pragma unroll
        for (int c = 0; c < NCHUNK; ++c) {
          ptx::tma_prefetch_3d(&tm_k, c * 64, hk, t0);
          ptx::tma_prefetch_3d(&tm_q, c * 64, hk, t0);
        }
        ptx::tma_prefetch_3d(&tm_v, 0, h, t0);
        // the X buffer is free once the MMAs of pair i-1 are done, the v buffer once the
        // epilogue of pair i-1 has formed its R (neither barrier can complete again before
        // this copy is issued, so the parity cannot have moved on); X goes first so the MMAs
        // never wait on v
        if (i > 0 && !tc_wait(&sh.proj_full[(i - 1) & nsm], ((i - 1) >> lgns) & 1u, sh, a.status)) break;
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
        const int b = int(i & nsm);
        const uint32_t ph = (i >> lgns) & 1u;
        if (!tc_wait(&sh.tmem_empty[b], ph ^ 1u, sh, a.status)) break;
        if (!tc_wait(&sh.node_full[i & 1u], (i >> 1) & 1u, sh, a.status)) break;
        ptx::tc_fence_after_sync();
        const uint32_t x0 = ptx::smem_u32(base + lay.x);
        const uint32_t d1 = tmem + uint32_t(b) * bufcols, d2 = d1 + gcol;
        // Gram: A = all 128 rows of X, B = the key rows (loops kept rolled: the kernel's roles
        // together run more code than the instruction caches hold)
#pragma unroll 1
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
#pragma unroll 1
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
      const int b = int(i & nsm);
      const uint32_t ph = (i >> lgns) & 1u;
      // the pair's parents, gates and betas are read from global memory before the wait for a
      // free stage, so their latency overlaps it
      // lane handles nodes lane and lane + 32
      const int tA = lane, tB = lane + 32;
      int prA = 0, prB = 0;
      float gA = 0.f, gB = 0.f, bA = 0.f, bB = 0.f;
      if (tA < n && in_bounds(t0 + tA, a.T, a.status)) {
        prA = a.parent[t0 + tA];
        gate_beta<SV>(sv, a.g, a.beta, size_t(t0 + tA) * a.H + h, h, gA, bA);
      }
      if (tB < n && in_bounds(t0 + tB, a.T, a.status)) {
        prB = a.parent[t0 + tB];
        gate_beta<SV>(sv, a.g, a.beta, size_t(t0 + tB) * a.H + h, h, gB, bB);
      }
      int ok = 1;
      if (lane == 0) ok = tc_wait(&sh.tree_empty[b], ph ^ 1u, sh, a.status);
      if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      ptx::mbar_try_wait(&sh.tree_empty[b], ph ^ 1u);  // acquire for every lane
      TreeStage &ts = sh.tree[b];
      int bad = 0;
      if (tA < n) {
        bad |= (prA < -1 || prA >= tA);
        ts.par[tA] = prA;
        ts.beta[tA] = bA;
        ts.a[tA] = gA;  // g for now; the gate exp(g) once every path sum is formed
      }
      if (tB < n) {
        bad |= (prB < -1 || prB >= tB);
        ts.par[tB] = prB;
        ts.beta[tB] = bB;
        ts.a[tB] = gB;
      }
      bad = __any_sync(0xffffffffu, bad);
      __syncwarp();
      if (!bad) {
        // ancestor masks and cumulative log-gates (parent indices strictly decrease along the
        // walk, so it ends within t + 1 steps), then depths, gates and the node lists of paths
        // short enough to be solved in registers
#pragma unroll 1
        for (int e = 0; e < 2; ++e) {
          const int t = e ? tB : tA;
          if (t < n) {
            unsigned long long m = 1ull << t;
            float Gs = e ? gB : gA;
            for (int x = ts.par[t]; x >= 0; x = ts.par[x]) {
              m |= 1ull << x;
              Gs += ts.a[x];
            }
            ts.anc[t] = m;
            ts.G[t] = Gs;
            ts.gam[t] = expf(Gs);
            ts.dep[t] = uint8_t(__popcll(m) - 1);
          }
        }
        __syncwarp();
#pragma unroll 1
        for (int e = 0; e < 2; ++e) {
          const int t = e ? tB : tA;
          if (t < n) {
            const int d = ts.dep[t];
            ts.a[t] = expf(e ? gB : gA);
            if (d < kRegPath) {
              int x = t;
              for (int k = d; k >= 0; --k) {
                ts.pj[t][k] = uint8_t(x);
                x = ts.par[x];
              }
              for (int k = d + 1; k < kRegPath; ++k) ts.pj[t][k] = uint8_t(t);
            }
          }
        }
      } else if (lane == 0 && h == 0) {
        report(a.status, GDN_STATUS_BAD_TREE);
      }
      if (lane == 0) ts.bad = bad;
      __syncwarp();
      mbar_arrive(&sh.tree_full[b]);
      ++i;
    }
  } else if (warp >= kWarpCoef && warp < kWarpCoef + kGroupThreads / 32) {
    // ------------------------------------------------------------ coefficient group
    const int ct = tid - kWarpCoef * 32;
    const int row = (warp & 3) * 32 + lane;  // TMEM lane of this thread: Gram row
    const uint32_t lane_addr = uint32_t((warp & 3) * 32) << 16;
    float *gram = reinterpret_cast<float *>(base + lay.gram);
    const int gstride = Np + 4;  // floats per staged Gram row
    uint8_t *bop = base + lay.bop;
    const uint32_t bop_lo = uint32_t(2 * Np * 128);
    uint32_t i = 0;
    for (int p = blockIdx.x; p < npairs; p += gridDim.x) {
      int t0, n, si;
      if (!tc_pair_nodes<SV>(a, sv, p, t0, n, si)) continue;
      const int b = int(i & nsm);
      const uint32_t ph = (i >> lgns) & 1u;
      // tree and Gram ready (the barrier also ends every thread's use of the previous pair's
      // coefficients)
      if (ct == 0) sh.coef_ok[0] = tc_wait(&sh.tree_full[b], ph, sh, a.status) && tc_wait(&sh.gram_full[b], ph, sh, a.status);
      named_sync(kBarCoef, kGroupThreads);
      if (!sh.coef_ok[0]) break;
      ptx::mbar_try_wait(&sh.tree_full[b], ph);  // acquire for this thread
      ptx::mbar_try_wait(&sh.gram_full[b], ph);
      ptx::tc_fence_after_sync();
      const TreeStage &ts = sh.tree[b];
      const bool live = !ts.bad;

      // (1) raw Gram rows TMEM -> shared memory (rows 0 .. 2 Np - 1; warps past them idle)
      if (live && (warp & 3) * 32 < 2 * Np) {  // warp-uniform
        const uint32_t d2 = tmem + uint32_t(b) * bufcols + gcol + lane_addr;
        float *grow = gram + row * gstride;
#pragma unroll 1
        for (int c0 = 0; c0 < Np; c0 += 16) {
          float r[16];
          ptx::tmem_ld_32x32b_x16(d2 + uint32_t(c0), r);
#pragma unroll
          for (int q = 0; q < 4; ++q)
            *reinterpret_cast<float4 *>(grow + c0 + 4 * q) = make_float4(r[4 * q], r[4 * q + 1], r[4 * q + 2], r[4 * q + 3]);
        }
      }
      // the previous pair's solve/output MMA has read the [T ; W] operand before it is rewritten
      if (ct == 0) sh.coef_ok[1] = i == 0 || tc_wait(&sh.uo_full, (i - 1) & 1u, sh, a.status);
      ptx::tc_fence_before_sync();
      named_sync(kBarCoef, kGroupThreads);
      if (!sh.coef_ok[1]) break;
      if (i > 0) ptx::mbar_try_wait(&sh.uo_full, (i - 1) & 1u);

      // (2) rows of T and W, two threads per node (role 0: row t of T, role 1: row t of W), by
      //     backward substitution along t's root-to-node path p_0 .. p_d = t:
      //       z = rhs;  for m = d .. 1:  z[k] -= z[m] A[p_m][p_k]  (k < m)
      //     with rhs = e_d (T) or P[t][p_.] (W), from the staged Gram rows and the gates:
      //       A[p_m][p_k] = b_{p_m} (a_{p_{k+1}} ... a_{p_m}) k_{p_m}.k_{p_k}
      //       P[t][p_k]   = (a_{p_{k+1}} ... a_{p_d}) q_t.k_{p_k}
      //     The row goes into the dense [T ; W] operand (row t or Np + t, column p_k) as bf16
      //     hi + lo, zeros elsewhere.
      if (live && ct < 2 * n) {
        const int t = ct >> 1, role = ct & 1;
        const unsigned long long anc = ts.anc[t];
        const int d = ts.dep[t];
        const int r = role ? Np + t : t;
        uint8_t *rowp = bop + r * 128;
        for (int c = 0; c < Np / 8; ++c) {
          const uint32_t o = uint32_t((c ^ (r & 7)) << 4);
          *reinterpret_cast<uint4 *>(rowp + o) = make_uint4(0u, 0u, 0u, 0u);
          *reinterpret_cast<uint4 *>(rowp + bop_lo + o) = make_uint4(0u, 0u, 0u, 0u);
        }
        const float *qrow = gram + (Np + t) * gstride;
        if (d < kRegPath) {
          // branch-free over the warp's longest path: entries past a lane's own depth repeat t
          // with a zero multiplier, so they change nothing
          const int dw = __reduce_max_sync(__activemask(), d);
          const uint32_t *pw = reinterpret_cast<const uint32_t *>(ts.pj[t]);
          const uint32_t w0 = pw[0], w1 = pw[1], w2 = pw[2];
          int pj[kRegPath];
          float ga[kRegPath], gb[kRegPath], z[kRegPath];
#pragma unroll
          for (int k = 0; k < kRegPath; ++k) {
            const uint32_t w = k < 4 ? w0 : (k < 8 ? w1 : w2);
            pj[k] = int((w >> (8 * (k & 3))) & 0xffu);
            ga[k] = ts.a[pj[k]];
            gb[k] = ts.beta[pj[k]];
          }
          // entries past the lane's depth hold the diagonal entry (column t) and never change
          if (role) {
            float e = 1.f;
#pragma unroll
            for (int k = kRegPath - 1; k >= 0; --k) {
              z[k] = e * qrow[pj[k]];
              e = k <= d ? e * ga[k] : e;
            }
          } else {
#pragma unroll
            for (int k = 0; k < kRegPath; ++k) z[k] = k >= d ? 1.f : 0.f;
          }
#pragma unroll
          for (int mm = kRegPath - 1; mm >= 1; --mm) {
            if (mm <= dw) {  // warp-uniform
              const float *krow = gram + pj[mm] * gstride;
              const float zm = mm <= d ? z[mm] : 0.f;
              float e = gb[mm];
#pragma unroll
              for (int k = mm - 1; k >= 0; --k) {
                e *= ga[k + 1];
                z[k] = fmaf(-zm * e, krow[pj[k]], z[k]);
              }
            }
          }
#pragma unroll
          for (int k = 0; k < kRegPath; ++k)
            if (k <= dw) put_hilo(bop, bop_lo, r, pj[k], z[k]);
        } else {  // longer paths: the same substitution with the path in local memory
          int pj[kMaxNodes];
          float ga[kMaxNodes], z[kMaxNodes];
          unsigned long long m = anc;
          for (int k = 0; k <= d; ++k) {
            pj[k] = __ffsll(static_cast<long long>(m)) - 1;
            m &= m - 1;
            ga[k] = ts.a[pj[k]];
          }
          float e = 1.f;
          for (int k = d; k >= 0; --k) {
            z[k] = role ? e * qrow[pj[k]] : (k == d ? 1.f : 0.f);
            e *= ga[k];
          }
          for (int mm = d; mm >= 1; --mm) {
            const float *krow = gram + pj[mm] * gstride;
            const float zm = z[mm];
            float em = ts.beta[pj[mm]];
            for (int k = mm - 1; k >= 0; --k) {
              em *= ga[k + 1];
              z[k] = fmaf(-zm * em, krow[pj[k]], z[k]);
            }
          }
          for (int k = 0; k <= d; ++k) put_hilo(bop, bop_lo, r, pj[k], z[k]);
        }
      }
      ptx::fence_proxy_async_smem();  // [T ; W] feeds the MMA (async proxy)
      ptx::tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&sh.coef_done);
        mbar_arrive(&sh.tmem_empty[b]);  // this group's Gram reads are done
        mbar_arrive(&sh.tree_empty[b]);
      }
      ++i;
    }
  } else if (warp >= kWarpOut && warp < kWarpOut + kGroupThreads / 32) {
    // ------------------------------------------------------------ R / output group
    const int ot = tid - kWarpOut * 32;
    const int q4 = warp & 3;
    const int v = q4 * 32 + lane;  // TMEM lane of this thread: state column v
    const uint32_t lane_addr = uint32_t(q4 * 32) << 16;
    const bool col = q4 * 32 < DV;  // warp-uniform
    const uint8_t *bop = base + lay.bop;
    const uint32_t bop_lo = uint32_t(2 * Np * 128);
    const uint32_t id_uo = ptx::idesc_bf16_f32(128, 2 * Np);
    const uint16_t *Vs = reinterpret_cast<const uint16_t *>(base + lay.v);
    uint32_t i = 0;
    for (int p = blockIdx.x; p < npairs; p += gridDim.x) {
      int t0, n, si;
      if (!tc_pair_nodes<SV>(a, sv, p, t0, n, si)) continue;
      const int h = p % a.H, b = int(i & nsm);
      const uint32_t ph = (i >> lgns) & 1u;
      if (ot == 0)
        sh.out_ok[0] = tc_wait(&sh.tree_full[b], ph, sh, a.status) && tc_wait(&sh.proj_full[b], ph, sh, a.status) &&
                       tc_wait(&sh.v_full, i & 1u, sh, a.status);
      named_sync(kBarOut, kGroupThreads);
      if (!sh.out_ok[0]) break;
      ptx::mbar_try_wait(&sh.tree_full[b], ph);  // acquire for this thread
      ptx::mbar_try_wait(&sh.proj_full[b], ph);
      ptx::mbar_try_wait(&sh.v_full, i & 1u);
      ptx::tc_fence_after_sync();
      const TreeStage &ts = sh.tree[b];
      const bool live = !ts.bad;
      const uint32_t d1 = tmem + uint32_t(b) * bufcols + lane_addr, d3 = d1 + gcol;

      // (3) R^T = (b (v - gamma KS))^T, row v: 16 nodes at a time, read from KS columns c0..c0+15
      //     and written back over them as 8 columns of bf16 hi pairs then 8 of lo pairs (the A
      //     operand of the solve/output MMA, K = nodes); columns t >= n are zero
      if (live && col) {
#pragma unroll 1
        for (int c0 = 0; c0 < Np; c0 += 16) {
          float ks[16];
          ptx::tmem_ld_32x32b_x16(d1 + uint32_t(c0), ks);
          float bt16[16], gm16[16], vv16[16];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float4 b4 = *reinterpret_cast<const float4 *>(&ts.beta[c0 + 4 * q]);
            const float4 g4 = *reinterpret_cast<const float4 *>(&ts.gam[c0 + 4 * q]);
            bt16[4 * q] = b4.x, bt16[4 * q + 1] = b4.y, bt16[4 * q + 2] = b4.z, bt16[4 * q + 3] = b4.w;
            gm16[4 * q] = g4.x, gm16[4 * q + 1] = g4.y, gm16[4 * q + 2] = g4.z, gm16[4 * q + 3] = g4.w;
          }
#pragma unroll
          for (int e = 0; e < 16; ++e) vv16[e] = c0 + e < n ? bf16_to_f32(Vs[(c0 + e) * DV + v]) : 0.f;
          float pk[16];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            float r2[2];
#pragma unroll
            for (int z = 0; z < 2; ++z) {
              const int j = 2 * e + z;
              r2[z] = c0 + j < n ? bt16[j] * (vv16[j] - gm16[j] * ks[j]) : 0.f;
            }
            const __nv_bfloat162 h2 = __floats2bfloat162_rn(r2[0], r2[1]);
            const float2 hf = __bfloat1622float2(h2);
            const __nv_bfloat162 l2 = __floats2bfloat162_rn(r2[0] - hf.x, r2[1] - hf.y);
            pk[e] = __uint_as_float(*reinterpret_cast<const uint32_t *>(&h2));
            pk[8 + e] = __uint_as_float(*reinterpret_cast<const uint32_t *>(&l2));
          }
          ptx::tmem_st_32x32b_x16(d1 + uint32_t(c0), pk);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh.v_empty);
      ptx::tc_fence_before_sync();
      named_sync(kBarOut, kGroupThreads);

      // (4) D3 = R^T [T ; W]^T: three bf16 products (hi hi, hi lo, lo hi), fp32 accumulate,
      //     once the coefficient group has written [T ; W]
      if (ot == 0) {
        bool ok = tc_wait(&sh.coef_done, i & 1u, sh, a.status);
        if (ok) {
          ptx::tc_fence_after_sync();
          const uint32_t a0 = tmem + uint32_t(b) * bufcols, b0 = ptx::smem_u32(bop);
          const uint32_t dd = a0 + gcol;
          for (int ks = 0; ks < Np / 16; ++ks) {
            const uint32_t ah = a0 + uint32_t(16 * ks), al = ah + 8u;
            const uint64_t bh = ptx::desc_kmajor_sw128(b0 + ks * 32), bl = ptx::desc_kmajor_sw128(b0 + bop_lo + ks * 32);
            ptx::mma_bf16_ts(dd, ah, bh, id_uo, ks > 0 ? 1u : 0u);
            ptx::mma_bf16_ts(dd, ah, bl, id_uo, 1u);
            ptx::mma_bf16_ts(dd, al, bh, id_uo, 1u);
          }
          ptx::mma_commit(&sh.uo_full);
          mma_any = true;
          ok = tc_wait(&sh.uo_full, i & 1u, sh, a.status);
        }
        sh.out_ok[1] = ok;
      }
      named_sync(kBarOut, kGroupThreads);
      if (!sh.out_ok[1]) break;
      ptx::mbar_try_wait(&sh.uo_full, i & 1u);
      ptx::tc_fence_after_sync();

      // (5) u_t = D3[:, t], o_t = gamma_t QS_t + D3[:, Np + t]
      if (live && col) {
        const float qsc = query_scale<SV>(sv);  // o is linear in q
        float *o_col = a.o + (size_t(t0) * a.H + h) * DV + v;
        float *u_col = a.U + (size_t(t0) * a.H + h) * DV + v;
        const size_t node_stride = size_t(a.H) * DV;
#pragma unroll 1
        for (int c0 = 0; c0 < n; c0 += 8) {
          uint32_t x[24];  // U, the tree part of o, QS
          ptx::tmem_ld3_32x32b_x8(d3 + uint32_t(c0), d3 + uint32_t(Np + c0), d1 + uint32_t(Np + c0), x);
          const float4 ga = *reinterpret_cast<const float4 *>(&ts.gam[c0]);
          const float4 gb = *reinterpret_cast<const float4 *>(&ts.gam[c0 + 4]);
          const float g8[8] = {ga.x, ga.y, ga.z, ga.w, gb.x, gb.y, gb.z, gb.w};
          float *op = o_col + size_t(c0) * node_stride;
          float *up = u_col + size_t(c0) * node_stride;
#pragma unroll
          for (int jj = 0; jj < 8; ++jj) {
            if (c0 + jj < n && in_bounds(op - a.o, (long long)a.T * a.H * DV, a.status)) {
              const float ov = fmaf(g8[jj], __uint_as_float(x[16 + jj]), __uint_as_float(x[8 + jj]));
              __stcs(op, SV ? qsc * ov : ov);
              __stcs(up, __uint_as_float(x[jj]));
            }
            op += node_stride;
            up += node_stride;
          }
        }
      }
      if (live && ot < n && in_bounds((long long)(t0 + ot) * a.H + h, (long long)a.T * a.H, a.status))
        a.G[size_t(t0 + ot) * a.H + h] = ts.G[ot];
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
  if (tid == kWarpOut * 32 && mma_any) {
    ptx::mma_commit(&sh.drain_out);
    ptx::mbar_wait(&sh.drain_out, 0, kWaitLimitNs);
  }
  ptx::tc_fence_before_sync();
  __syncthreads();
  if (warp == kWarpMma) {
    ptx::tc_fence_after_sync();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace gdn
