// Device-side greedy acceptance: the accepted root-to-node path of every request, found on the
// GPU so that verify -> accept -> commit needs no host round trip (GDN Tree-Scan abstract:
// device-side commitment of the accepted chain; TreeWY page, method section: candidate outputs
// decide acceptance, then only the accepted path is committed).
//
// Per request: the path starts at node 0 (the root: the token the target already produced, kept
// unconditionally) and, at the current node x, takes the lowest-indexed child c whose draft token
// equals the target's greedy token after x; it stops when no child matches. One warp per request,
// two nodes per lane; each step is one ballot over the request's nodes.
#pragma once

#include "common.cuh"

namespace gdn {

struct AcceptArgs {
  const int32_t *draft, *target, *parent, *cu_nodes;
  int B, T, max_nodes, max_path;
  int32_t *path, *path_len;
  int32_t *status;
};

constexpr int kAcceptWarps = 4;  // requests per CTA

__global__ void __launch_bounds__(kAcceptWarps * 32) accept_greedy_kernel(AcceptArgs a) {
  const int lane = threadIdx.x & 31;
  const int r = blockIdx.x * kAcceptWarps + (threadIdx.x >> 5);
  if (r >= a.B) return;  // warp-uniform
  int32_t *path_r = a.path + size_t(r) * a.max_path;
  const int t0 = a.cu_nodes[r];
  const int n = a.cu_nodes[r + 1] - t0;
  int L = 0;
  bool ok = true;
  if (!offsets_ok(t0, n, a.T)) {
    if (lane == 0) report(a.status, GDN_STATUS_BAD_OFFSETS);
    ok = false;
  } else if (n > a.max_nodes || n > kMaxNodes) {
    if (lane == 0) report(a.status, GDN_STATUS_TOO_MANY_NODES);
    ok = false;
  }
  if (ok && n > 0) {
    int par[2], drf[2];
    int bad = 0;
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int t = lane + 32 * e;
      par[e] = t < n ? a.parent[t0 + t] : -2;  // -2: no node in this slot
      drf[e] = t < n ? a.draft[t0 + t] : 0;
      bad |= t < n && (par[e] < -1 || par[e] >= t);
    }
    if (__any_sync(0xffffffffu, bad)) {
      if (lane == 0) report(a.status, GDN_STATUS_BAD_TREE);
    } else {
      int x = 0;  // node 0 has parent -1: it is always the first root
      if (a.max_path > 0) {
        if (lane == 0) path_r[0] = 0;
        L = 1;
        // children have larger indices than their parent, so the walk ends within n steps
        for (int step = 1; step < n; ++step) {
          const int tgt = a.target[t0 + x];
          const unsigned lo = __ballot_sync(0xffffffffu, par[0] == x && drf[0] == tgt);
          const unsigned hi = __ballot_sync(0xffffffffu, par[1] == x && drf[1] == tgt);
          if (!(lo | hi)) break;
          const int c = lo ? __ffs(lo) - 1 : 32 + __ffs(hi) - 1;
          if (L == a.max_path) {
            if (lane == 0) report(a.status, GDN_STATUS_PATH_TRUNCATED);
            break;
          }
          if (lane == 0) path_r[L] = c;
          ++L;
          x = c;
        }
      } else {
        if (lane == 0) report(a.status, GDN_STATUS_PATH_TRUNCATED);
      }
    }
  }
  for (int i = L + lane; i < a.max_path; i += 32) path_r[i] = -1;
  if (lane == 0) a.path_len[r] = L;
}

}  // namespace gdn
