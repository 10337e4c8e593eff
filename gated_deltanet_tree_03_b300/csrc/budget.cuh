// Draft budgeting on the device: which draft positions or tree nodes a verify step checks.
//
// Top-B allocation (DSpark adaptive-verification news item): each draft token carries an
// estimated probability of passing verification; a request's survival probability at position
// i is the product of those probabilities up to i; one global budget of B positions goes to the
// (request, position) pairs of largest survival, which per request is a prefix of its drafts.
//
// Threshold best-first growth (TreeSpark page): a draft tree grows along its most promising
// branch first and stops once the best remaining candidate's value - the survival product along
// its branch - falls below a threshold. Branch values never grow along a branch (every factor is
// at most 1, and fp32 rounding is monotone), so best-first order is the order of (value desc,
// candidate index asc): the kernel forms every candidate's value, gathers those that reach the
// threshold, keeps the max_nodes best of them (radix selection of the max_nodes-th key) and sorts
// those with one warp. A parent always precedes its children in that order, so the output is a
// parent-before-child tree.
//
// Neither kernel sorts everything: top-B only needs each request's count (its keys at or before
// the B-th best key, found by radix selection), and growth sorts at most 64 keys.
//
// Survival products decide which positions and nodes are taken, so they are rounded exactly as
// written: fp32 products formed from the root outward, without fused multiply-adds.
#pragma once

#include "common.cuh"

namespace gdn {

constexpr int kTopbThreads = 256;  // few warps: the selection is a chain of block-wide barriers
constexpr int kScanThreads = 1024;
constexpr int kCopyWarps = 8;      // requests per CTA of the packing copy
constexpr int kTopbMaxItems = 16384;  // requests x positions sorted by one CTA in shared memory
constexpr int kGrowThreads = 256;
constexpr int kGrowMaxCand = 8192;    // candidates per request sorted by one CTA

struct TopbArgs {
  const float *p;  // [R][K]
  int R, K, budget;
  int32_t *n_sel;      // [R]
  float *survival;     // [R][K] or null
  int32_t *cu_nodes;   // [R+1] or null
  int32_t *parent;     // [R + min(budget, R K)] or null
  int32_t *status;
};

struct GrowArgs {
  const float *p;  // [R][C]
  int R, fanout, depth, C, max_nodes;
  float threshold;
  int32_t *n_nodes;       // [R]
  int32_t *cand;          // [R][max_nodes] or null
  int32_t *parent_local;  // [R][max_nodes]
  float *value;           // [R][max_nodes] or null
  int32_t *status;
};

struct PackArgs {
  const int32_t *n_nodes, *parent_local;
  int R, max_nodes;
  int32_t *cu_nodes, *parent;
};

// An estimated probability; anything outside [0, 1] (NaN included) counts as 0, and both zeros
// are +0 (the sort keys below rely on the sign bit being clear).
__device__ __forceinline__ float checked_prob(float x, bool &bad) {
  const bool ok = x >= 0.f && x <= 1.f;
  bad |= !ok;
  return x > 0.f && ok ? x : 0.f;
}

// Sort key, smaller = earlier: a non-negative float's bit pattern grows with its value, so the
// complemented pattern orders values descending; the low word orders equal values by index.
__device__ __forceinline__ uint64_t rank_key(float v, uint32_t idx) {
  return (uint64_t(~__float_as_uint(v)) << 32) | idx;
}
constexpr uint64_t kNoKey = ~0ull;

// Ascending bitonic sort of 64 keys in shared memory by one warp.
__device__ __forceinline__ void warp_sort64(uint64_t *keys) {
  const int lane = threadIdx.x & 31;
  for (int k = 2; k <= 64; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int i = lane + 32 * h, l = i ^ j;
        if (l > i) {
          const uint64_t x = keys[i], y = keys[l];
          if ((x > y) == ((i & k) == 0)) {
            keys[i] = y;
            keys[l] = x;
          }
        }
      }
      __syncwarp();
    }
  }
}

// The n-th smallest (1 <= n <= m) of m distinct keys keys[0..m) in shared memory, by
// most-significant-digit radix selection over 8-bit digits: per digit, a histogram of the keys
// that share the digits fixed so far, then the bin holding the n-th of them; once that bin holds
// a single key, one more pass finds it. Exactly n keys are <= the result. Every thread must call
// it; `hist` holds 256 shared ints, `pick` three, `found` one 64-bit word.
__device__ uint64_t block_select_nth(const uint64_t *keys, int m, int n, int *hist, int *pick,
                                     unsigned long long *found) {
  uint64_t prefix = 0, mask = 0;
  int rem = n;  // rank of the wanted key among the keys that match `prefix` under `mask`
  const int lane = threadIdx.x & 31;
  for (int shift = 56; shift >= 0; shift -= 8) {
    for (int i = threadIdx.x; i < 256; i += blockDim.x) hist[i] = 0;
    __syncthreads();
    for (int base = 0; base < m; base += blockDim.x) {  // uniform trip count for the warp votes
      const int i = base + int(threadIdx.x);
      const uint64_t k = i < m ? keys[i] : 0ull;
      const int bin = (i < m && (k & mask) == prefix) ? int((k >> shift) & 255u) : -1;
      const unsigned peers = __match_any_sync(0xffffffffu, bin);  // the high digits cluster: one add per group
      if (bin >= 0 && lane == __ffs(peers) - 1) atomicAdd(&hist[bin], __popc(peers));
    }
    __syncthreads();
    if (threadIdx.x < 32) {  // lane l scans bins 8l .. 8l + 7
      int c[8], tot = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        c[j] = hist[8 * lane + j];
        tot += c[j];
      }
      int incl = tot;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += y;
      }
      int run = incl - tot;
      if (run < rem && rem <= incl) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if (run + c[j] >= rem) {
            pick[0] = 8 * lane + j;
            pick[1] = rem - run;
            pick[2] = c[j];
            break;
          }
          run += c[j];
        }
      }
    }
    __syncthreads();
    prefix |= uint64_t(pick[0]) << shift;
    mask |= uint64_t(255) << shift;
    rem = pick[1];
    if (pick[2] == 1 && shift > 0) {  // the only key with this prefix is the answer
      for (int i = threadIdx.x; i < m; i += blockDim.x)
        if ((keys[i] & mask) == prefix) *found = keys[i];
      __syncthreads();
      return *found;
    }
  }
  return prefix;
}

// Exclusive prefix sums of term(i), i < n, by the whole block: out[i] for i < n, out[n] = total.
// `scratch` holds 32 ints of shared memory. Every thread must call it.
template <class Term>
__device__ void block_exclusive_scan(int n, Term term, int32_t *out, int *scratch) {
  const int nt = blockDim.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int chunk = (n + nt - 1) / nt;
  const int i0 = min(n, tid * chunk), i1 = min(n, i0 + chunk);
  int local = 0;
  for (int i = i0; i < i1; ++i) local += term(i);
  int incl = local;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += y;
  }
  if (lane == 31) scratch[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int nw = nt / 32;
    int w = lane < nw ? scratch[lane] : 0;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, off);
      if (lane >= off) w += y;
    }
    if (lane < nw) scratch[lane] = w;  // inclusive totals of the warps
  }
  __syncthreads();
  int run = (warp > 0 ? scratch[warp - 1] : 0) + incl - local;
  for (int i = i0; i < i1; ++i) {
    out[i] = run;
    run += term(i);
  }
  if (tid == nt - 1) out[n] = scratch[nt / 32 - 1];
  __syncthreads();
}

// One CTA: survival products, global top-B, per-request counts, and the chains to verify.
__global__ void __launch_bounds__(kTopbThreads) topb_kernel(TopbArgs a) {
  extern __shared__ __align__(16) uint8_t budget_dyn[];
  const int n_items = a.R * a.K;
  uint64_t *keys = reinterpret_cast<uint64_t *>(budget_dyn);
  float *ps = reinterpret_cast<float *>(keys + n_items);  // the probabilities, staged
  int *cnt = reinterpret_cast<int *>(ps + n_items);
  __shared__ int scan_scratch[32];
  __shared__ int hist[256], pick[3];
  __shared__ unsigned long long found;
  const int tid = threadIdx.x;
  bool bad = false;
  for (int i = tid; i < n_items; i += blockDim.x) ps[i] = a.p[i];  // coalesced
  __syncthreads();
  for (int r = tid; r < a.R; r += blockDim.x) {
    float acc = 1.f;
    for (int i = 0; i < a.K; ++i) {
      const int idx = r * a.K + i;
      acc = __fmul_rn(acc, checked_prob(ps[idx], bad));
      keys[idx] = rank_key(acc, uint32_t(idx));
      if (a.survival) a.survival[idx] = acc;
    }
  }
  if (__syncthreads_or(bad) && tid == 0) report(a.status, GDN_STATUS_BAD_PROB);
  const int take = min(a.budget, n_items);
  // the take-th best key; a request's chosen positions are its keys at or before it (a prefix)
  const uint64_t last = take == 0 ? 0ull : take == n_items ? kNoKey : block_select_nth(keys, n_items, take, hist, pick, &found);
  for (int r = tid; r < a.R; r += blockDim.x) {
    int c = 0;
    if (take > 0)
      for (int i = 0; i < a.K; ++i) c += keys[r * a.K + i] <= last;
    cnt[r] = c;
    a.n_sel[r] = c;
  }
  __syncthreads();
  if (a.cu_nodes == nullptr) return;  // block-uniform
  // request r verifies a chain: the token the target already produced, then n_sel[r] drafts
  block_exclusive_scan(a.R, [&](int r) { return 1 + cnt[r]; }, a.cu_nodes, scan_scratch);
  if (a.parent == nullptr) return;
  for (int r = tid; r < a.R; r += blockDim.x) {  // the chains, packed in request order
    const int base = a.cu_nodes[r], len = 1 + cnt[r];
    for (int j = 0; j < len; ++j) a.parent[base + j] = j - 1;
  }
}

// One CTA per request: branch values, threshold, top max_nodes, parents in output order.
__global__ void __launch_bounds__(kGrowThreads) grow_kernel(GrowArgs a) {
  extern __shared__ __align__(16) uint8_t budget_dyn[];
  const int C = a.C;
  uint64_t *cand_keys = reinterpret_cast<uint64_t *>(budget_dyn);  // [C]: candidates at the threshold
  float *val = reinterpret_cast<float *>(cand_keys + C);           // [C]
  int *out_pos = reinterpret_cast<int *>(cand_keys);  // [C], once the keys are consumed: candidate -> output index
  __shared__ uint64_t sel[64];  // the taken candidates' keys, sorted
  __shared__ int n_cand, n_sel_s, hist[256], pick[3];
  __shared__ unsigned long long found;
  const int r = blockIdx.x, tid = threadIdx.x;
  const float *p = a.p + size_t(r) * C;
  bool bad = false;
  if (tid == 0) {
    n_cand = 0;
    n_sel_s = 0;
    val[0] = 1.f;  // the root
  }
  __syncthreads();
  // level by level: a child multiplies its parent's value
  int first = 1, width = a.fanout;
  for (int l = 1; l <= a.depth; ++l) {
    for (int c = first + tid; c < first + width; c += blockDim.x)
      val[c] = __fmul_rn(val[(c - 1) / a.fanout], checked_prob(p[c], bad));
    __syncthreads();
    first += width;
    width *= a.fanout;
  }
  // candidates that reach the threshold (the root always does), in any order: keys are unique
  for (int c = tid; c < C; c += blockDim.x)
    if (c == 0 || val[c] >= a.threshold) cand_keys[atomicAdd(&n_cand, 1)] = rank_key(val[c], uint32_t(c));
  if (__syncthreads_or(bad) && tid == 0) report(a.status, GDN_STATUS_BAD_PROB);
  const int m = n_cand, n = min(a.max_nodes, m);
  if (n < m) {  // keep the n best: those at or before the n-th smallest key
    const uint64_t last = block_select_nth(cand_keys, m, n, hist, pick, &found);
    for (int i = tid; i < m; i += blockDim.x)
      if (cand_keys[i] <= last) sel[atomicAdd(&n_sel_s, 1)] = cand_keys[i];
  } else {
    for (int i = tid; i < m; i += blockDim.x) sel[i] = cand_keys[i];
  }
  __syncthreads();
  if (tid < 32) {
    for (int i = n + tid; i < 64; i += 32) sel[i] = kNoKey;
    __syncwarp();
    warp_sort64(sel);
  }
  __syncthreads();
  for (int t = tid; t < n; t += blockDim.x) out_pos[uint32_t(sel[t])] = t;
  __syncthreads();
  const size_t row = size_t(r) * a.max_nodes;
  for (int t = tid; t < a.max_nodes; t += blockDim.x) {
    int c = -1, par = -1;
    float v = 0.f;
    if (t < n) {
      c = int(uint32_t(sel[t]));
      v = val[c];
      par = c == 0 ? -1 : out_pos[(c - 1) / a.fanout];
    }
    a.parent_local[row + t] = par;
    if (a.cand) a.cand[row + t] = c;
    if (a.value) a.value[row + t] = v;
  }
  if (tid == 0) a.n_nodes[r] = n;
}

// One CTA: node offsets of the packed batch (exclusive prefix sums of n_nodes).
__global__ void __launch_bounds__(kScanThreads) pack_scan_kernel(PackArgs a) {
  __shared__ int scan_scratch[32];
  block_exclusive_scan(a.R, [&](int r) { return a.n_nodes[r]; }, a.cu_nodes, scan_scratch);
}

// One warp per request: its taken nodes' parents, copied to the packed batch.
__global__ void __launch_bounds__(kCopyWarps * 32) pack_copy_kernel(PackArgs a) {
  const int r = blockIdx.x * kCopyWarps + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (r >= a.R) return;
  const int n = a.n_nodes[r], base = a.cu_nodes[r];
  const int32_t *src = a.parent_local + size_t(r) * a.max_nodes;
  for (int t = lane; t < n; t += 32) a.parent[base + t] = src[t];
}

}  // namespace gdn
