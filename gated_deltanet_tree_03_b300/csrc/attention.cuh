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
//     softmax          one thread per query row: mask (prefix length / ancestor bits), running
//                      max and sum in the log2 domain, O rescaled in tensor memory when the max
//                      grows, probabilities written to shared memory as bf16
//     O += P V         tcgen05.mma with V read as an MN-major operand straight from its TMA tile
// Warp roles: 0 TMA producer, 1 MMA issuer, 2 tree masks, 4..7 softmax and epilogue.
//
// Long prefixes with few (request, head, tile) triples are split over CTAs; each split writes
// its unnormalised O with its running max and sum, and a combine kernel merges the splits.
// Every wait is bounded; on a timeout the CTA raises GDN_STATUS_TIMEOUT, drains its copies and
// MMAs and returns.
#pragma once

#include <cuda.h>

#include "common.cuh"
#include "ptx.cuh"

namespace gdn {

constexpr int kAttnRows = 128;      // query rows per tile (the MMA's M)
constexpr int kAttnKeys = 128;      // prefix keys per block
constexpr int kAttnTreeKeys = 64;   // the draft-node block (at most 64 nodes per request)
constexpr int kAttnStages = 2;      // key/value blocks in flight
constexpr int kAttnThreads = 256;
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

// Dynamic shared memory: Q, the K and V stages, P and alignment slack - and never less than
// 120 KB, so that two CTAs (whose tensor-memory allocations would not both fit) never share an SM.
__host__ __device__ constexpr uint32_t attn_smem_bytes(int D) {
  return (uint32_t(D / 64) * 16384u                    // Q: 128 rows x 128 B per 64-column chunk
          + uint32_t(kAttnStages) * 2u * (D / 64) * 16384u  // K and V: 128 keys x 128 B per chunk
          + 2u * 16384u                                  // P: 128 rows x 128 keys bf16
          + 1024u) > 120u * 1024u
             ? (uint32_t(D / 64) * 16384u + uint32_t(kAttnStages) * 2u * (D / 64) * 16384u + 2u * 16384u + 1024u)
             : 120u * 1024u;
}

struct AttnShared {
  uint64_t q_full, k_full[kAttnStages], v_full[kAttnStages], kv_empty[kAttnStages];
  uint64_t s_full[2], s_free[2], p_full, pv_done, drain;
  unsigned long long anc[64];
  uint32_t tmem_base;
  int abort_flag, go;
};

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
  uint8_t *Vs = Ks + kAttnStages * kKVBytes;         // [stage] V blocks
  uint8_t *Ps = Vs + kAttnStages * kKVBytes;         // P: 2 chunks of 64 keys

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int split = blockIdx.x % a.splits, tile = blockIdx.x / a.splits;
  const int g = blockIdx.y, r = blockIdx.z;
  const int G = a.G, nodes_per_tile = kAttnRows / G;

  // ---- request checks and the tree's ancestor masks (warp 2), before anything is issued
  if (tid == 0) {
    sh.go = 0;
    sh.abort_flag = 0;
  }
  __syncthreads();
  const int t0 = a.cu_nodes[r], n = a.cu_nodes[r + 1] - t0;
  const int p0 = a.cu_prefix[r], P = a.cu_prefix[r + 1] - p0;
  const int t_begin = tile * nodes_per_tile;
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
  if (!sh.go) return;  // uniform: nothing issued, nothing allocated

  // ---- this split's blocks: prefix blocks [b_lo, b_hi), then the draft-node block (last split)
  const int n_pre = (P + kAttnKeys - 1) / kAttnKeys;
  const int b_lo = min(n_pre, split * a.blocks_per_split), b_hi = min(n_pre, b_lo + a.blocks_per_split);
  const int nbp = b_hi - b_lo;
  const bool has_tree = split == a.splits - 1;
  const int nb = nbp + (has_tree ? 1 : 0);

  if (tid == 0) {
    ptx::mbar_init(&sh.q_full, 1);
    for (int s = 0; s < kAttnStages; ++s) {
      ptx::mbar_init(&sh.k_full[s], 1);
      ptx::mbar_init(&sh.v_full[s], 1);
      ptx::mbar_init(&sh.kv_empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(&sh.s_full[b], 1);
      ptx::mbar_init(&sh.s_free[b], 128);
    }
    ptx::mbar_init(&sh.p_full, 128);
    ptx::mbar_init(&sh.pv_done, 1);
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
  const uint32_t O_col = 2 * kAttnKeys;  // S buffers at columns 0 and 128, O after them

  uint32_t issued = 0;  // TMA thread: blocks whose copies were issued

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA producer
    if (lane == 0) {
      ptx::prefetch_tensormap(&tm_q);
      ptx::prefetch_tensormap(&tm_kc);
      ptx::prefetch_tensormap(&tm_vc);
      ptx::mbar_arrive_expect_tx(&sh.q_full, kQBytes);
#pragma unroll
      for (int c = 0; c < NCH; ++c)
        ptx::tma_load_3d(Qs + c * kChunk, &tm_q, &sh.q_full, c * 64, g * G, t0 + t_begin);
      for (int j = 0; j < nb; ++j) {
        const int s = j % kAttnStages;
        if (j >= kAttnStages && !attn_wait(&sh.kv_empty[s], ((j / kAttnStages) - 1) & 1, sh, a.status)) break;
        const bool tree = j == nbp;
        const uint32_t bytes = tree ? uint32_t(NCH) * kAttnTreeKeys * 128u : kKVBytes;
        ptx::mbar_arrive_expect_tx(&sh.k_full[s], bytes);
#pragma unroll
        for (int c = 0; c < NCH; ++c) {
          if (tree) ptx::tma_load_3d(Ks + s * kKVBytes + c * kChunk, &tm_kt, &sh.k_full[s], c * 64, g, t0);
          else ptx::tma_load_3d(Ks + s * kKVBytes + c * kChunk, &tm_kc, &sh.k_full[s], c * 64, g,
                                p0 + (b_lo + j) * kAttnKeys);
        }
        ptx::mbar_arrive_expect_tx(&sh.v_full[s], bytes);
#pragma unroll
        for (int c = 0; c < NCH; ++c) {
          if (tree) ptx::tma_load_3d(Vs + s * kKVBytes + c * kChunk, &tm_vt, &sh.v_full[s], c * 64, g, t0);
          else ptx::tma_load_3d(Vs + s * kKVBytes + c * kChunk, &tm_vc, &sh.v_full[s], c * 64, g,
                                p0 + (b_lo + j) * kAttnKeys);
        }
        issued = uint32_t(j + 1);
      }
      // clean-up: the copies of the last blocks issued have landed before the CTA exits
      ptx::mbar_wait(&sh.q_full, 0, kAttnWaitNs);
      for (int j = int(issued) - kAttnStages; j < int(issued); ++j) {
        if (j < 0) continue;
        ptx::mbar_wait(&sh.k_full[j % kAttnStages], (j / kAttnStages) & 1, kAttnWaitNs);
        ptx::mbar_wait(&sh.v_full[j % kAttnStages], (j / kAttnStages) & 1, kAttnWaitNs);
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t q_addr = ptx::smem_u32(Qs), p_addr = ptx::smem_u32(Ps);
      bool ok = attn_wait(&sh.q_full, 0, sh, a.status);
      auto issue_s = [&](int j) -> bool {
        const int s = j % kAttnStages;
        if (!attn_wait(&sh.k_full[s], (j / kAttnStages) & 1, sh, a.status)) return false;
        if (j >= 2 && !attn_wait(&sh.s_free[j & 1], ((j >> 1) - 1) & 1, sh, a.status)) return false;
        ptx::tc_fence_after_sync();
        const bool tree = j == nbp;
        const uint32_t idesc = ptx::idesc_bf16_f32(kAttnRows, tree ? kAttnTreeKeys : kAttnKeys);
        const uint32_t k_addr = ptx::smem_u32(Ks + s * kKVBytes);
#pragma unroll
        for (int c = 0; c < NCH; ++c)
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            ptx::mma_bf16_ss(tmem + uint32_t(j & 1) * kAttnKeys,
                             ptx::desc_kmajor_sw128(q_addr + c * kChunk + kk * 32),
                             ptx::desc_kmajor_sw128(k_addr + c * kChunk + kk * 32), idesc, (c | kk) != 0);
        ptx::mma_commit(&sh.s_full[j & 1]);
        return true;
      };
      auto issue_pv = [&](int j) -> bool {
        const int s = j % kAttnStages;
        if (!attn_wait(&sh.p_full, j & 1, sh, a.status)) return false;
        if (!attn_wait(&sh.v_full[s], (j / kAttnStages) & 1, sh, a.status)) return false;
        ptx::tc_fence_after_sync();
        const int ksteps = (j == nbp ? kAttnTreeKeys : kAttnKeys) / 16;
        const uint32_t idesc = ptx::idesc_bf16_f32_bmn(kAttnRows, 64);
        const uint32_t v_addr = ptx::smem_u32(Vs + s * kKVBytes);
        for (int ks = 0; ks < ksteps; ++ks)
#pragma unroll
          for (int c = 0; c < NCH; ++c)
            ptx::mma_bf16_ss(tmem + O_col + uint32_t(c * 64),
                             ptx::desc_kmajor_sw128(p_addr + (ks >> 2) * kChunk + (ks & 3) * 32),
                             ptx::desc_mnmajor_sw128(v_addr + c * kChunk + ks * 2048), idesc, (j | ks) != 0);
        ptx::mma_commit(&sh.pv_done);
        ptx::mma_commit(&sh.kv_empty[s]);
        return true;
      };
      if (ok && nb > 0) ok = issue_s(0);
      for (int j = 0; ok && j < nb; ++j) {
        if (j + 1 < nb && !issue_s(j + 1)) break;
        if (!issue_pv(j)) break;
      }
      // clean-up: every MMA this thread issued has completed
      ptx::mma_commit(&sh.drain);
      ptx::mbar_wait(&sh.drain, 0, kAttnWaitNs);
    }
  } else if (warp >= kAttnSoftmaxWarp0) {
    // ---------------------------------------------------------------- softmax and epilogue
    const int i = tid - kAttnSoftmaxWarp0 * 32;  // query row = TMEM lane
    const int t_local = i / G, hq = i % G;
    const int t = t_begin + t_local;
    const bool row_ok = t < n;
    const unsigned long long anc_t = row_ok ? sh.anc[t] : 0ull;
    const uint32_t lane_addr = uint32_t((warp - kAttnSoftmaxWarp0) * 32) << 16;
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; ok && j < nb; ++j) {
      const bool tree = j == nbp;
      const int ncols = tree ? kAttnTreeKeys : kAttnKeys;
      if (!attn_wait(&sh.s_full[j & 1], (j >> 1) & 1, sh, a.status)) {
        ok = false;
        break;
      }
      ptx::tc_fence_after_sync();
      float sc[kAttnKeys];
#pragma unroll
      for (int c = 0; c < kAttnKeys; ++c) sc[c] = 0.f;
#pragma unroll
      for (int c0 = 0; c0 < kAttnKeys; c0 += 16) {
        if (c0 < ncols) {
          float x[16];
          ptx::tmem_ld_32x32b_x16(tmem + lane_addr + uint32_t(j & 1) * kAttnKeys + uint32_t(c0), x);
#pragma unroll
          for (int e = 0; e < 16; ++e) sc[c0 + e] = x[e];
        }
      }
      ptx::tc_fence_before_sync();
      attn_arrive(&sh.s_free[j & 1]);
      // mask, scale (log2 domain), block max
      const int key0 = (b_lo + j) * kAttnKeys;
      float bmax = -INFINITY;
#pragma unroll
      for (int c = 0; c < kAttnKeys; ++c) {
        bool vis;
        if (tree) vis = c < kAttnTreeKeys && c < n && ((anc_t >> (c & 63)) & 1ull);
        else vis = key0 + c < P;
        vis = vis && row_ok;
        sc[c] = vis ? sc[c] * a.scale_log2 : -INFINITY;
        bmax = fmaxf(bmax, sc[c]);
      }
      const float m_new = fmaxf(m, bmax);
      const float alpha = m_new == -INFINITY ? 1.f : exp2f(m - m_new);
      const float m_sub = m_new == -INFINITY ? 0.f : m_new;  // a row with no visible key yet: every p is 0
      // the previous block's P.V has finished: P may be overwritten, O is stable
      if (j > 0 && !attn_wait(&sh.pv_done, (j - 1) & 1, sh, a.status)) {
        ok = false;
        break;
      }
      ptx::tc_fence_after_sync();
      if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {  // rescale this warp's O rows
#pragma unroll
        for (int c0 = 0; c0 < D; c0 += 16) {
          float x[16];
          ptx::tmem_ld_32x32b_x16(tmem + lane_addr + O_col + uint32_t(c0), x);
#pragma unroll
          for (int e = 0; e < 16; ++e) x[e] *= alpha;
          ptx::tmem_st_32x32b_x16(tmem + lane_addr + O_col + uint32_t(c0), x);
        }
      }
      // probabilities, rounded to bf16 as the P.V product sees them (their sum uses the same
      // rounded values), written as row i of P: K-major with the 128-byte swizzle, 16-byte unit u
      // of the row at position u ^ (i & 7)
      float psum = 0.f;
#pragma unroll
      for (int ch = 0; ch < kAttnKeys / 64; ++ch) {
        if (ch * 64 < ncols) {
          uint8_t *row = Ps + ch * kChunk + (i >> 3) * 1024 + (i & 7) * 128;
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int c = ch * 64 + u * 8 + 2 * e;
              const __nv_bfloat162 b2 = __floats2bfloat162_rn(exp2f(sc[c] - m_sub), exp2f(sc[c + 1] - m_sub));
              psum += __low2float(b2) + __high2float(b2);
              w[e] = *reinterpret_cast<const uint32_t *>(&b2);
            }
            *reinterpret_cast<uint4 *>(row + ((u ^ (i & 7)) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
          }
        }
      }
      l = l * alpha + psum;
      m = m_new;
      ptx::fence_proxy_async_smem();
      ptx::tc_fence_before_sync();
      attn_arrive(&sh.p_full);
    }
    // epilogue: the last P.V has finished
    if (ok && nb > 0 && attn_wait(&sh.pv_done, (nb - 1) & 1, sh, a.status)) {
      ptx::tc_fence_after_sync();
      const int h = g * G + hq;
      float *dst;
      float inv = 1.f;
      if (a.splits == 1) {
        dst = a.o + (size_t(t0 + t) * a.Hq + h) * D;
        inv = 1.f / l;
      } else {
        const size_t wrow = ((((size_t(r) * a.Hkv + g) * a.tiles + tile) * a.splits + split) * kAttnRows) + i;
        dst = a.ws_o + wrow * D;
        if (row_ok) {
          a.ws_ml[2 * wrow] = m;
          a.ws_ml[2 * wrow + 1] = l;
        }
      }
#pragma unroll
      for (int c0 = 0; c0 < D; c0 += 16) {
        float x[16];
        ptx::tmem_ld_32x32b_x16(tmem + lane_addr + O_col + uint32_t(c0), x);
        if (row_ok) {
#pragma unroll
          for (int e = 0; e < 16; e += 4)
            *reinterpret_cast<float4 *>(dst + c0 + e) = make_float4(x[e] * inv, x[e + 1] * inv, x[e + 2] * inv,
                                                                    x[e + 3] * inv);
        }
      }
    } else if (ok && nb == 0 && a.splits > 1 && row_ok) {  // an empty split: weight zero in the merge
      const size_t wrow = ((((size_t(r) * a.Hkv + g) * a.tiles + tile) * a.splits + split) * kAttnRows) + i;
      a.ws_ml[2 * wrow] = -INFINITY;
      a.ws_ml[2 * wrow + 1] = 0.f;
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
