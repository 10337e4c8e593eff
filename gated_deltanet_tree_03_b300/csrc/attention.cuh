// Tree-bias attention for the attention layers of a hybrid model: every draft node attends to its
// request's committed key/value prefix and to the draft nodes on its own root-to-node path (GDN
// Tree-Scan abstract: tree-bias attention beside the recurrent-state replay; an attention-only
// verifier mainly needs the ancestry mask). Grouped heads: query head h reads key/value head
// h / G.
//
// One CTA per (request, key/value head, tile of 128 query rows, key split). The query rows of a
// tile are (node, query head of the group) pairs, row = node * G + head, so one TMA box brings
// G heads x 128/G nodes straight into the K-major 128-byte-swizzled operand layout. Per block of
// keys (128 prefix keys, or the request's <= 64 draft nodes as the last block):
//     S = Q K^T        tcgen05.mma into tensor memory (two S buffers, so the next block's
//                      scores are computed while this block's softmax runs)
//     softmax          one thread per query row, its scores read once from tensor memory into
//                      registers: mask (prefix length / ancestor bits), running
//                      max and sum in the log2 domain, O rescaled in tensor memory when the max
//                      grows, probabilities written back as bf16 over the S columns they came from
//     O += P V         tcgen05.mma with P read from tensor memory and V read as an MN-major
//                      operand straight from its TMA tile
// Warp roles: 0 key (and query) TMA producer, 1 MMA issuer (S_0, S_1, then P.V_j and S_{j+2} in
// turn, each after a blocking wait), 2 tree masks, 3 value TMA producer, 4..11 softmax and epilogue in two
// warpgroups: warps 4..7 take key columns 0..63 of every block, warps 8..11 columns 64..127,
// each half with its own running max and sum and its own O accumulator in tensor memory; the
// two halves are merged once, in the epilogue.
// A row's running max is only moved (and O rescaled) when a block raises it by more than 2^8;
// the probabilities are then at most 2^8, and the final O / l uses the same reference.
//
// Long prefixes with few (request, head, tile) triples are split over CTAs; each split writes
// its unnormalised O with its running max and sum, and a combine kernel merges the splits.
// Every wait is bounded; on a timeout the CTA raises GDN_STATUS_TIMEOUT, drains its copies and
// MMAs and returns.
#pragma once

#include <cuda.h>

#include "bounds.cuh"
#include "common.cuh"
#include "ptx.cuh"

namespace gdn {

constexpr int kAttnRows = 128;      // query rows per tile (the MMA's M)
constexpr int kAttnKeys = 128;      // prefix keys per block
constexpr int kAttnTreeKeys = 64;   // the draft-node block (at most 64 nodes per request)
constexpr int kAttnKStages = 3;     // key blocks in flight (a key block is free as soon as S is formed)
constexpr int kAttnVStages = 3;     // value blocks in flight (free once P.V is done)
constexpr float kAttnRescale = 8.f;  // log2 growth of a row's max that forces a rescale of O
constexpr int kAttnThreads = 384;
constexpr int kAttnSoftmaxWarp0 = 4;
constexpr uint32_t kAttnTmemCols = 512;
constexpr uint64_t kAttnWaitNs = 1000000000ull;  // 1 s bound on every wait

struct AttnArgs {
  const int32_t *parent, *cu_nodes, *cu_prefix;
  int B, Hq, Hkv, G, T, P_total, max_nodes, max_prefix;
  int tiles, splits, blocks_per_split;
  float scale_log2;  // score scale times log2(e)
  float *o;          // [T][Hq][D] (one split)
  float *ws_o;       // [B][Hkv][tiles][splits][128][D] partial outputs (several splits)
  float *ws_ml;      // [B][Hkv][tiles][splits][128][2] running max (log2 domain) and sum
  int32_t *status;
};

// Dynamic shared memory: Q, the K and V stages (128 keys x 128 B per 64-column chunk) and
// alignment slack - never less than 120 KB, so that two CTAs (whose tensor-memory allocations
// would not both fit) never share an SM.
__host__ __device__ constexpr uint32_t attn_smem_need(int D) {
  return uint32_t(1 + kAttnKStages + kAttnVStages) * (D / 64) * 16384u + 1024u;
}
__host__ __device__ constexpr uint32_t attn_smem_bytes(int D) {
  return attn_smem_need(D) > 120u * 1024u ? attn_smem_need(D) : 120u * 1024u;
}

struct AttnShared {
  uint64_t q_full, k_full[kAttnKStages], k_empty[kAttnKStages], v_full[kAttnVStages], v_empty[kAttnVStages];
  // p_full[b]: every softmax thread has written block j's P, for blocks j with j & 1 == b. Two of
  // them, so that a thread already on block j + 1 cannot complete block j's phase: it can reach
  // block j + 2 (the same barrier) only after block j's P.V was issued.
  uint64_t s_full[2], p_full[2], pv_done, o_final, drain;
  unsigned long long anc[64];
  uint32_t tmem_base;
  int abort_flag, go;
};

__device__ __forceinline__ void attn_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

__device__ __forceinline__ bool attn_wait(uint64_t *bar, uint32_t parity, AttnShared &sh, int32_t *status) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = ptx::globaltimer_ns();
  for (uint32_t i = 1; i < (1u << 26); ++i) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    if ((i & 15u) == 0) {
      if (*reinterpret_cast<volatile int *>(&sh.abort_flag)) return false;
      if (ptx::globaltimer_ns() - t0 > kAttnWaitNs) break;
    }
  }
  *reinterpret_cast<volatile int *>(&sh.abort_flag) = 1;
  report(status, GDN_STATUS_TIMEOUT);
  return false;
}

__device__ __forceinline__ void attn_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(ptx::smem_u32(bar)) : "memory");
}

template <int D>
__global__ void __launch_bounds__(kAttnThreads, 1)
    tree_attention_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_kc,
                          const __grid_constant__ CUtensorMap tm_vc, const __grid_constant__ CUtensorMap tm_kt,
                          const __grid_constant__ CUtensorMap tm_vt, AttnArgs a) {
  static_assert(D == 64 || D == 128, "head dimension 64 or 128");
  constexpr int NCH = D / 64;                       // 64-column chunks of a row
  constexpr uint32_t kChunk = 16384u;               // 128 rows x 128 B
  constexpr uint32_t kQBytes = NCH * kChunk;
  constexpr uint32_t kKVBytes = NCH * kChunk;       // one K (or V) block of 128 keys
  __shared__ AttnShared sh;
  extern __shared__ uint8_t attn_dyn_raw[];
  uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(attn_dyn_raw) + 1023) & ~uintptr_t(1023));
  uint8_t *Qs = base;
  uint8_t *Ks = Qs + kQBytes;                        // [stage] K blocks
  uint8_t *Vs = Ks + kAttnKStages * kKVBytes;        // [stage] V blocks

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int split = blockIdx.x % a.splits, tile = blockIdx.x / a.splits;
  const int g = blockIdx.y, r = blockIdx.z;
  const int G = a.G, nodes_per_tile = kAttnRows / G;

  // ---- barriers and tensor memory first, so that the first copies start while warp 2 checks
  // the request and builds the tree's ancestor masks
  if (tid == 0) {
    sh.go = 0;
    sh.abort_flag = 0;
    ptx::mbar_init(&sh.q_full, 1);
    for (int s = 0; s < kAttnKStages; ++s) {
      ptx::mbar_init(&sh.k_full[s], 1);
      ptx::mbar_init(&sh.k_empty[s], 1);
    }
    for (int s = 0; s < kAttnVStages; ++s) {
      ptx::mbar_init(&sh.v_full[s], 1);
      ptx::mbar_init(&sh.v_empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) ptx::mbar_init(&sh.s_full[b], 1);
    ptx::mbar_init(&sh.p_full[0], 256);
    ptx::mbar_init(&sh.p_full[1], 256);
    ptx::mbar_init(&sh.pv_done, 1);
    ptx::mbar_init(&sh.o_final, 1);
    ptx::mbar_init(&sh.drain, 1);
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc(&sh.tmem_base, kAttnTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before_sync();
  __syncthreads();
  ptx::tc_fence_after_sync();
  const uint32_t tmem = sh.tmem_base;

  const int t0 = a.cu_nodes[r], n = a.cu_nodes[r + 1] - t0;
  const int p0 = a.cu_prefix[r], P = a.cu_prefix[r + 1] - p0;
  const int t_begin = tile * nodes_per_tile;

  // ---- this split's blocks: prefix blocks [b_lo, b_hi), then the draft-node block (last split)
  const int n_pre = (P + kAttnKeys - 1) / kAttnKeys;
  const int b_lo = min(n_pre, split * a.blocks_per_split), b_hi = min(n_pre, b_lo + a.blocks_per_split);
  const int nbp = b_hi - b_lo;
  const bool has_tree = split == a.splits - 1;
  const int nb = nbp + (has_tree ? 1 : 0);

  // TMA producers (lane 0 of warps 0 and 3): block j of keys (warp 0) or values (warp 3) into
  // stage j % stages. The first `stages` blocks, and the query tile, go out before the request is
  // checked: with offsets that the checks will reject, their boxes are clipped or filled by the
  // copy engine (never a fault) and the CTA waits for them before it leaves.
  const bool producer = (warp == 0 || warp == 3) && lane == 0;
  const bool keys = warp == 0;
  const int stages = keys ? kAttnKStages : kAttnVStages;
  uint64_t *const full = keys ? sh.k_full : sh.v_full;
  uint64_t *const empty = keys ? sh.k_empty : sh.v_empty;
  uint8_t *const kvbuf = keys ? Ks : Vs;
  const CUtensorMap *const pre_map = keys ? &tm_kc : &tm_vc, *const node_map = keys ? &tm_kt : &tm_vt;
  auto issue_block = [&](int j) {
    const int st = j % stages;
    const bool tree = j == nbp;
    ptx::mbar_arrive_expect_tx(&full[st], tree ? uint32_t(NCH) * kAttnTreeKeys * 128u : kKVBytes);
#pragma unroll
    for (int c = 0; c < NCH; ++c) {
      if (tree) ptx::tma_load_3d(kvbuf + st * kKVBytes + c * kChunk, node_map, &full[st], c * 64, g, t0);
      else ptx::tma_load_3d(kvbuf + st * kKVBytes + c * kChunk, pre_map, &full[st], c * 64, g,
                            p0 + (b_lo + j) * kAttnKeys);
    }
  };
  int issued = 0;  // blocks this producer has issued
  if (producer && t_begin < n) {  // (a tile without rows leaves at the checks)
    ptx::prefetch_tensormap(pre_map);
    if (keys) {
      ptx::prefetch_tensormap(&tm_q);
      ptx::mbar_arrive_expect_tx(&sh.q_full, kQBytes);
#pragma unroll
      for (int c = 0; c < NCH; ++c) ptx::tma_load_3d(Qs + c * kChunk, &tm_q, &sh.q_full, c * 64, g * G, t0 + t_begin);
    }
    for (; issued < stages && issued < nb; ++issued) issue_block(issued);
  }

  if (warp == 2) {
    bool ok = true;
    if (!offsets_ok(t0, n, a.T) || !offsets_ok(p0, P, a.P_total) || P > a.max_prefix) {
      if (lane == 0 && g == 0 && tile == 0 && split == 0) report(a.status, GDN_STATUS_BAD_OFFSETS);
      ok = false;
    } else if (n > a.max_nodes || n > 64) {
      if (lane == 0 && g == 0 && tile == 0 && split == 0) report(a.status, GDN_STATUS_TOO_MANY_NODES);
      ok = false;
    }
    ok = ok && t_begin < n;  // this tile has rows
    int bad = 0;
    if (ok) {
      for (int t = lane; t < n; t += 32) {
        const int pr = a.parent[t0 + t];
        bad |= (pr < -1 || pr >= t);
      }
      bad = __any_sync(0xffffffffu, bad);
      if (bad && lane == 0 && g == 0 && tile == 0 && split == 0) report(a.status, GDN_STATUS_BAD_TREE);
    }
    if (ok && !bad) {
      for (int t = lane; t < n; t += 32) {
        unsigned long long m = 1ull << t;
        for (int x = a.parent[t0 + t]; x >= 0; x = a.parent[t0 + x]) m |= 1ull << x;  // parents decrease
        sh.anc[t] = m;
      }
      if (lane == 0) sh.go = 1;
    }
  }
  __syncthreads();
  if (!sh.go) {  // uniform: the early copies land and the tensor memory is returned
    if (producer && t_begin < n) {  // (the copies went out only for a tile with rows)
      if (keys) ptx::mbar_wait(&sh.q_full, 0, kAttnWaitNs);
      for (int j = 0; j < issued; ++j) ptx::mbar_wait(&full[j], 0, kAttnWaitNs);
    }
    __syncthreads();
    if (warp == 1) {
      __syncwarp();
      ptx::tmem_dealloc(tmem, kAttnTmemCols);
    }
    return;
  }
  const uint32_t O_col = 2 * kAttnKeys;  // S buffers at columns 0 and 128, then O of half 0, O of half 1

  if (warp == 0 || warp == 3) {
    // ---------------------------------------------------------------- TMA producers
    if (lane == 0) {
      for (; issued < nb; ++issued) {
        const int j = issued, st = j % stages;
        if (!attn_wait(&empty[st], ((j / stages) - 1) & 1, sh, a.status)) break;
        issue_block(j);
      }
      // clean-up: the copies of the last blocks issued have landed before the CTA exits
      if (keys) ptx::mbar_wait(&sh.q_full, 0, kAttnWaitNs);
      for (int j = issued - stages; j < issued; ++j)
        if (j >= 0) ptx::mbar_wait(&full[j % stages], (j / stages) & 1, kAttnWaitNs);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t q_addr = ptx::smem_u32(Qs);
      bool ok = attn_wait(&sh.q_full, 0, sh, a.status);
      // S_j = Q K_j^T into S buffer j & 1, once key block j has landed
      auto issue_s = [&](int j) {
        const int sk = j % kAttnKStages;
        if (!attn_wait(&sh.k_full[sk], (j / kAttnKStages) & 1, sh, a.status)) return false;
        ptx::tc_fence_after_sync();
        const bool tree = j == nbp;
        const uint32_t idesc = ptx::idesc_bf16_f32(kAttnRows, tree ? kAttnTreeKeys : kAttnKeys);
        const uint32_t k_addr = ptx::smem_u32(Ks + sk * kKVBytes);
#pragma unroll
        for (int c = 0; c < NCH; ++c)
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            ptx::mma_bf16_ss(tmem + uint32_t(j & 1) * kAttnKeys, ptx::desc_kmajor_sw128(q_addr + c * kChunk + kk * 32),
                             ptx::desc_kmajor_sw128(k_addr + c * kChunk + kk * 32), idesc, (c | kk) != 0);
        ptx::mma_commit(&sh.s_full[j & 1]);
        ptx::mma_commit(&sh.k_empty[sk]);
        return true;
      };
      // Fixed issue order S_0, S_1, then P.V_j followed by S_{j+2}: S_{j+2} overwrites the buffer
      // whose probabilities P.V_j reads, and one thread's MMAs run in issue order. Every wait
      // blocks (the thread sleeps in the barrier), so this warp takes no issue slots from the
      // softmax warps that share its scheduler.
      int si = 0, pi = 0;
      bool o1_started = false;  // half 1's O has had its first (overwriting) P.V
      for (; ok && si < nb && si < 2; ++si) ok = issue_s(si);
      for (; ok && pi < nb; ++pi) {
        const int sv = pi % kAttnVStages;
        if (!attn_wait(&sh.p_full[pi & 1], (pi >> 1) & 1, sh, a.status) ||
            !attn_wait(&sh.v_full[sv], (pi / kAttnVStages) & 1, sh, a.status)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after_sync();
        // one MMA per 16 keys covers all D value columns: the value tile's 64-column chunks are
        // the operand's atoms along N, kChunk bytes apart
        const uint32_t idesc = ptx::idesc_bf16_f32_bmn(kAttnRows, D);
        const uint32_t v_addr = ptx::smem_u32(Vs + sv * kKVBytes);
        const uint32_t p_tmem = tmem + uint32_t(pi & 1) * kAttnKeys;
        // half h: keys 64 h .. 64 h + 63, whose P that half wrote (packed, 16 keys = 8 columns) at
        // columns 64 h .. 64 h + 31 of the buffer, into O of half h; the draft-node block has keys
        // for half 0 only
        const int halves = pi == nbp ? 1 : 2;
        for (int h2 = 0; h2 < halves; ++h2) {
          for (int kq = 0; kq < 4; ++kq) {
            const int ks = h2 * 4 + kq;
            const uint32_t acc = h2 == 0 ? uint32_t((pi | kq) != 0) : uint32_t(o1_started || kq != 0);
            ptx::mma_bf16_ts(tmem + O_col + uint32_t(h2 * D), p_tmem + uint32_t(h2 * 64 + kq * 8),
                             ptx::desc_mnmajor_sw128(v_addr + ks * 2048, kChunk), idesc, acc);
          }
          if (h2 == 1) o1_started = true;
        }
        ptx::mma_commit(&sh.pv_done);
        ptx::mma_commit(&sh.v_empty[sv]);
        if (si < nb) {
          ok = issue_s(si);
          ++si;
        }
      }
      // O is final once every P.V has completed (the epilogue waits on this single phase: the
      // per-block barrier may trail the last block by two phases, which a parity wait cannot tell)
      if (pi == nb && nb > 0) ptx::mma_commit(&sh.o_final);
      // clean-up: every MMA this thread issued has completed
      ptx::mma_commit(&sh.drain);
      ptx::mbar_wait(&sh.drain, 0, kAttnWaitNs);
    }
  } else if (warp >= kAttnSoftmaxWarp0) {
    // ---------------------------------------------------------------- softmax and epilogue
    const int hf = (warp - kAttnSoftmaxWarp0) / 4;           // key half of this warpgroup
    const int i = ((warp - kAttnSoftmaxWarp0) & 3) * 32 + lane;  // query row = TMEM lane
    const int t_local = i / G, hq = i % G;
    const int t = t_begin + t_local;
    const bool row_ok = t < n;
    const unsigned long long anc_t = row_ok ? sh.anc[t] : 0ull;
    const uint32_t lane_addr = uint32_t(((warp - kAttnSoftmaxWarp0) & 3) * 32) << 16;
    const uint32_t o_addr = tmem + lane_addr + O_col + uint32_t(hf * D);
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; ok && j < nb; ++j) {
      const bool tree = j == nbp;
      if (!attn_wait(&sh.s_full[j & 1], (j >> 1) & 1, sh, a.status)) {
        ok = false;
        break;
      }
      ptx::tc_fence_after_sync();
      if (!tree || hf == 0) {  // the draft-node block's <= 64 keys are all in half 0
        // mask: only a partial prefix block and the draft-node block need one
        const int lim = tree ? 0 : P - (b_lo + j) * kAttnKeys - hf * 64;  // visible prefix keys of this half
        const bool full = row_ok && !tree && lim >= 64;
        auto masked = [&](float (&x)[64]) {
          if (full) return;
          if (!row_ok) {
#pragma unroll
            for (int e = 0; e < 64; ++e) x[e] = -INFINITY;
          } else if (tree) {  // key e is visible iff bit e of the row's ancestor mask is set
            const uint32_t lo = uint32_t(anc_t), hi = uint32_t(anc_t >> 32);
#pragma unroll
            for (int e = 0; e < 64; ++e)
              if (!(((e < 32 ? lo : hi) >> (e & 31)) & 1u)) x[e] = -INFINITY;
          } else {
#pragma unroll
            for (int e = 0; e < 64; ++e)
              if (e >= lim) x[e] = -INFINITY;
          }
        };
        const uint32_t s_addr = tmem + lane_addr + uint32_t(j & 1) * kAttnKeys + uint32_t(hf * 64);
        // the row's 64 scores of this half, read once and kept in registers; block max of the raw
        // scores (the scale is positive: the scaled max is the max scaled)
        float x[64];
        ptx::tmem_ld_32x32b_x64(s_addr, x);
        masked(x);
        float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
        for (int e = 0; e < 64; ++e) mx[e & 3] = fmaxf(mx[e & 3], x[e]);
        const float bmax = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) * a.scale_log2;
        const float m_new = bmax > m + kAttnRescale ? bmax : m;  // the reference max moves only by > 2^8
        const float alpha = m_new == m ? 1.f : exp2f(m - m_new);
        const float m_sub = m_new == -INFINITY ? 0.f : m_new;  // a row with no visible key yet: every p is 0
        if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {  // rescale this warp's O rows of this half
          // O is stable once the previous block's P.V has finished. S_j was issued after
          // P.V_{j-2} and its commit covers it, so the P.V barrier is at phase j - 1 (pending)
          // or past it: the parity wait is unambiguous
          if (!attn_wait(&sh.pv_done, (j - 1) & 1, sh, a.status)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after_sync();
#pragma unroll
          for (int c0 = 0; c0 < D; c0 += 16) {
            float y[16];
            ptx::tmem_ld_32x32b_x16(o_addr + uint32_t(c0), y);
#pragma unroll
            for (int e = 0; e < 16; ++e) y[e] *= alpha;
            ptx::tmem_st_32x32b_x16(o_addr + uint32_t(c0), y);
          }
        }
        // probabilities p = 2^(scale s - m), rounded to bf16 and written back over the first 32
        // columns of this half's scores (already read), two keys per 32-bit column. Their sum is
        // taken before rounding (each rounded weight is within 2^-8 of its exact value, the same
        // bound as rounding the sum).
        float ps[4] = {0.f, 0.f, 0.f, 0.f};
        const float sl = a.scale_log2;
        {
          uint32_t w[32];
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const float e0 = ptx::ex2_approx(fmaf(x[2 * e], sl, -m_sub));
            const float e1 = ptx::ex2_approx(fmaf(x[2 * e + 1], sl, -m_sub));
            ps[e & 3] += e0 + e1;
            const __nv_bfloat162 b2 = __floats2bfloat162_rn(e0, e1);
            w[e] = *reinterpret_cast<const uint32_t *>(&b2);
          }
          ptx::tmem_st_32x32b_x32(s_addr, w);
        }
        l = l * alpha + ((ps[0] + ps[1]) + (ps[2] + ps[3]));
        m = m_new;
      }
      ptx::tc_fence_before_sync();
      attn_arrive(&sh.p_full[j & 1]);
    }
    // epilogue: the last P.V has finished; merge the halves, O = (w0 O_0 + w1 O_1) / (w0 l_0 + w1 l_1)
    // with w_h = 2^(m_h - M), M the larger max
    const bool fin = ok && nb > 0 && attn_wait(&sh.o_final, 0, sh, a.status);
    // each half's running max and sum per row, exchanged through the query buffer: every MMA
    // (the only reader of Q) has completed once O is final
    float (*ml)[kAttnRows][2] = reinterpret_cast<float (*)[kAttnRows][2]>(Qs);
    if (fin) {
      ml[hf][i][0] = m;
      ml[hf][i][1] = l;
    }
    attn_bar_sync(1, 256);  // every softmax thread, whatever happened above
    if (fin) {
      ptx::tc_fence_after_sync();
      const float m0 = ml[0][i][0], l0 = ml[0][i][1], m1 = ml[1][i][0], l1 = ml[1][i][1];
      const float M = fmaxf(m0, m1);
      const float w0 = l0 > 0.f ? exp2f(m0 - M) : 0.f, w1 = l1 > 0.f ? exp2f(m1 - M) : 0.f;
      const float L = w0 * l0 + w1 * l1;
      const int h = g * G + hq;
      float *dst;
      float inv = 1.f;
      bool dst_ok;  // (the debug build checks the row against its array)
      if (a.splits == 1) {
        dst = a.o + (size_t(t0 + t) * a.Hq + h) * D;
        inv = 1.f / L;
        dst_ok = !row_ok || in_bounds((long long)(t0 + t) * a.Hq + h, (long long)a.T * a.Hq, a.status);
      } else {
        const size_t wrow = ((((size_t(r) * a.Hkv + g) * a.tiles + tile) * a.splits + split) * kAttnRows) + i;
        dst = a.ws_o + wrow * D;
        dst_ok = !row_ok || in_bounds((long long)wrow, (long long)a.B * a.Hkv * a.tiles * a.splits * kAttnRows, a.status);
        if (row_ok && dst_ok && hf == 0) {
          a.ws_ml[2 * wrow] = M;
          a.ws_ml[2 * wrow + 1] = L;
        }
      }
      const int cb = hf * (D / 2);  // each half writes half of the output columns
#pragma unroll
      for (int c0 = 0; c0 < D / 2; c0 += 16) {
        float x0[16], x1[16];
        ptx::tmem_ld_32x32b_x16(tmem + lane_addr + O_col + uint32_t(cb + c0), x0);
        ptx::tmem_ld_32x32b_x16(tmem + lane_addr + O_col + uint32_t(D + cb + c0), x1);
        if (row_ok && dst_ok) {
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const float a0 = w0 > 0.f ? w0 * x0[e] : 0.f, a1 = w1 > 0.f ? w1 * x1[e] : 0.f;
            x0[e] = (a0 + a1) * inv;
          }
#pragma unroll
          for (int e = 0; e < 16; e += 4)
            *reinterpret_cast<float4 *>(dst + cb + c0 + e) = make_float4(x0[e], x0[e + 1], x0[e + 2], x0[e + 3]);
        }
      }
    } else if (ok && nb == 0 && a.splits > 1 && row_ok && hf == 0) {  // an empty split: weight zero
      const size_t wrow = ((((size_t(r) * a.Hkv + g) * a.tiles + tile) * a.splits + split) * kAttnRows) + i;
      if (in_bounds((long long)wrow, (long long)a.B * a.Hkv * a.tiles * a.splits * kAttnRows, a.status)) {
        a.ws_ml[2 * wrow] = -INFINITY;
        a.ws_ml[2 * wrow + 1] = 0.f;
      }
    }
  }

  ptx::tc_fence_before_sync();
  __syncthreads();
  ptx::tc_fence_after_sync();
  if (warp == 1) {
    __syncwarp();
    ptx::tmem_dealloc(tmem, kAttnTmemCols);
  }
}

// Merges the key splits of every valid query row: O = sum_s 2^(m_s - M) O_s / sum_s 2^(m_s - M) l_s.
template <int D>
__global__ void __launch_bounds__(256) tree_attention_combine_kernel(AttnArgs a) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int i = blockIdx.y * 8 + warp;  // query row of the tile
  const int tile = blockIdx.x % a.tiles;
  const int g = (blockIdx.x / a.tiles) % a.Hkv, r = blockIdx.x / (a.tiles * a.Hkv);
  const int t0 = a.cu_nodes[r], n = a.cu_nodes[r + 1] - t0;
  const int p0 = a.cu_prefix[r], P = a.cu_prefix[r + 1] - p0;
  if (!offsets_ok(t0, n, a.T) || !offsets_ok(p0, P, a.P_total) || P > a.max_prefix || n > a.max_nodes || n > 64)
    return;
  const int t = tile * (kAttnRows / a.G) + i / a.G;
  if (t >= n) return;  // warp-uniform
  // the attention kernel writes no partials for a malformed tree (and reports it)
  int bad = 0;
  for (int x = lane; x < n; x += 32) {
    const int pr = a.parent[t0 + x];
    bad |= (pr < -1 || pr >= x);
  }
  if (__any_sync(0xffffffffu, bad)) return;
  const size_t row0 = (((size_t(r) * a.Hkv + g) * a.tiles + tile) * a.splits) * kAttnRows + i;
  if (!in_bounds((long long)(row0 + size_t(a.splits - 1) * kAttnRows),
                 (long long)a.B * a.Hkv * a.tiles * a.splits * kAttnRows, a.status) ||
      !in_bounds((long long)(t0 + t) * a.Hq + g * a.G + (i % a.G), (long long)a.T * a.Hq, a.status))
    return;
  float M = -INFINITY;
  for (int s = 0; s < a.splits; ++s) M = fmaxf(M, a.ws_ml[2 * (row0 + size_t(s) * kAttnRows)]);
  constexpr int PER = D / 32;
  float acc[PER] = {};
  float L = 0.f;
  for (int s = 0; s < a.splits; ++s) {
    const size_t wr = row0 + size_t(s) * kAttnRows;
    const float ms = a.ws_ml[2 * wr], ls = a.ws_ml[2 * wr + 1];
    if (ls == 0.f) continue;  // an empty split (or a row that saw no key in it)
    const float w = exp2f(ms - M);
    L += w * ls;
#pragma unroll
    for (int e = 0; e < PER; ++e) acc[e] += w * a.ws_o[wr * D + lane * PER + e];
  }
  const int h = g * a.G + (i % a.G);
  float *dst = a.o + (size_t(t0 + t) * a.Hq + h) * D + lane * PER;
#pragma unroll
  for (int e = 0; e < PER; ++e) dst[e] = acc[e] / L;
}

}  // namespace gdn
