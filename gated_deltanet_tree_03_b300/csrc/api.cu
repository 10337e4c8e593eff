// Host side of the C ABI declared in include/gdn_tree.h: argument checks, launch
// configuration, TMA descriptor encoding and kernel dispatch. Nothing here allocates device
// memory, synchronises the device or keeps per-call state. What is kept across calls is
// looked up once per device and never changes afterwards: the device's properties, each
// kernel's dynamic shared-memory limit, and the address of the scratch array of
// gdn_tree_attention_noalloc (its one fixed buffer).
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <mutex>
#include <unordered_map>

#include <cuda.h>
#include <cuda_runtime.h>

#include "gdn_tree.h"
#include "accept.cuh"
#include "attention.cuh"
#include "budget.cuh"
#include "common.cuh"
#include "commit.cuh"
#include "storeall.cuh"
#include "verify_simt.cuh"
#include "verify_stream.cuh"
#include "verify_tc.cuh"

using namespace gdn;

namespace {

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Largest shared memory one block may use on this architecture (227 KiB), for host-side size checks
// that must not depend on a device being present.
constexpr size_t kSmemPerBlockMax = 232448;
bool valid_d(int d) { return d == 32 || d == 64 || d == 128; }

// Properties of one device, queried on the first call that runs on it.
struct DeviceInfo {
  int major = 0, minor = 0;
  int sms = 0;    // streaming multiprocessors
  int optin = 0;  // opt-in dynamic + static shared memory per block, bytes
};

constexpr int kMaxDevices = 64;
std::mutex g_dev_mu;
DeviceInfo g_dev_info[kMaxDevices];
bool g_dev_known[kMaxDevices] = {};

// The current device's properties (one cudaGetDevice per call after the first on a device).
gdn_status device_info(const DeviceInfo **out, int *dev_out = nullptr) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return GDN_ECUDA;
  if (dev_out) *dev_out = dev;
  std::lock_guard<std::mutex> lock(g_dev_mu);
  if (!g_dev_known[dev]) {
    DeviceInfo d;
    if (cudaDeviceGetAttribute(&d.major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
      return GDN_ECUDA;
    g_dev_info[dev] = d;
    g_dev_known[dev] = true;
  }
  *out = &g_dev_info[dev];
  return GDN_OK;
}

gdn_status check_device() {
  const DeviceInfo *d = nullptr;
  const gdn_status st = device_info(&d);
  if (st != GDN_OK) return st;
  if (d->major != 10 || d->minor != 3) return GDN_EARCH;
  return GDN_OK;
}

// Per (kernel, device): its static shared memory and the dynamic shared-memory limit set so
// far. cudaFuncSetAttribute is called only when a launch needs more than the limit already set.
struct FuncInfo {
  int static_smem = -1;
  int dyn_limit = 0;
};
std::mutex g_func_mu;
std::unordered_map<uint64_t, FuncInfo> g_func_info;

uint64_t func_key(const void *fn, int dev) { return (reinterpret_cast<uint64_t>(fn) << 6) ^ uint64_t(dev); }

// Static shared memory of `fn` on the current device (looked up once).
gdn_status func_static_smem(const void *fn, int *bytes) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return GDN_ECUDA;
  std::lock_guard<std::mutex> lock(g_func_mu);
  FuncInfo &fi = g_func_info[func_key(fn, dev)];
  if (fi.static_smem < 0) {
    cudaFuncAttributes fa{};
    if (cudaFuncGetAttributes(&fa, fn) != cudaSuccess) return GDN_ECUDA;
    fi.static_smem = int(fa.sharedSizeBytes);
  }
  *bytes = fi.static_smem;
  return GDN_OK;
}

// Make sure `fn` may be launched with `bytes` of dynamic shared memory on the current device.
gdn_status ensure_dyn_smem(const void *fn, size_t bytes) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return GDN_ECUDA;
  std::lock_guard<std::mutex> lock(g_func_mu);
  FuncInfo &fi = g_func_info[func_key(fn, dev)];
  if (size_t(fi.dyn_limit) >= bytes) return GDN_OK;
  if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, int(bytes)) != cudaSuccess) {
    (void)cudaGetLastError();  // the refused attribute must not surface as a later launch error
    return GDN_ECUDA;
  }
  fi.dyn_limit = int(bytes);
  return GDN_OK;
}

gdn_status launch_status() {
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    fprintf(stderr, "gdn_tree: launch failed: %s\n", cudaGetErrorString(e));
    return GDN_ECUDA;
  }
  return GDN_OK;
}

// shared argument checks of the verify family (host side only; nothing is launched here)
gdn_status check_verify_args(const float *ST, const uint16_t *q, const uint16_t *k,
                             const uint16_t *v, const float *beta, const float *g,
                             const int32_t *parent, const int32_t *cu_nodes, int32_t B, int32_t H,
                             int32_t T, int32_t d_k, int32_t d_v, int32_t max_nodes, const float *o,
                             const float *U, const float *G, const int32_t *status,
                             const Serving &L = Serving{}) {
  if (B < 0 || H <= 0 || T < 0 || max_nodes < 0) return GDN_EINVAL;
  if (B > 65535 || H > 65535) return GDN_EINVAL;  // grid limits
  if (!valid_d(d_k) || !valid_d(d_v)) return GDN_EINVAL;
  if (max_nodes > kMaxNodes) return GDN_ETOOBIG;
  if (B == 0 || T == 0) return GDN_OK;
  const bool fused_gates = L.a_raw != nullptr;  // beta and g are then formed in the kernels
  if (!ST || !q || !k || !v || !parent || !cu_nodes || !o || !U || !G) return GDN_EINVAL;
  if (!fused_gates && (!beta || !g)) return GDN_EINVAL;
  const void *ptrs[] = {ST, q, k, v, parent, cu_nodes, o, U, G};
  for (const void *p : ptrs)
    if (!aligned16(p)) return GDN_EALIGN;
  if (!fused_gates && (!aligned16(beta) || !aligned16(g))) return GDN_EALIGN;
  if (status && !aligned16(status)) return GDN_EALIGN;
  return GDN_OK;
}

gdn_status check_commit_args(const float *ST, const void *a1, const void *a2, const void *a3,
                             const int32_t *parent, const int32_t *cu_nodes, const int32_t *path,
                             const int32_t *path_len, int32_t B, int32_t H, int32_t T, int32_t d_k,
                             int32_t d_v, int32_t max_path, const int32_t *status) {
  if (B < 0 || H <= 0 || T < 0 || max_path < 0) return GDN_EINVAL;
  if (!valid_d(d_k) || !valid_d(d_v)) return GDN_EINVAL;
  if (max_path > kMaxNodes) return GDN_ETOOBIG;
  if (B == 0) return GDN_OK;
  if (!ST || !cu_nodes || !path_len) return GDN_EINVAL;
  if (T > 0 && (!a1 || !a2 || !a3 || !parent)) return GDN_EINVAL;
  if (max_path > 0 && !path) return GDN_EINVAL;
  const void *ptrs[] = {ST, a1, a2, a3, parent, cu_nodes, path_len, path, status};
  for (const void *p : ptrs)
    if (p && !aligned16(p)) return GDN_EALIGN;
  return GDN_OK;
}

// Host checks of a serving layout (gdn_layout, declared in gdn_tree.h) and its kernel form.
// `full` = a verify call (q_scale and the gate arrays apply); commit reads the slots and H_qk.
gdn_status make_serving(const gdn_layout *l, int32_t H, bool full, Serving &L) {
  L = Serving{};
  if (!l) return GDN_OK;
  if (H <= 0) return GDN_EINVAL;
  if (l->H_qk < 0 || (l->H_qk > 0 && H % l->H_qk != 0)) return GDN_EINVAL;
  L.grp = l->H_qk > 0 ? H / l->H_qk : 1;
  if (l->state_slot) {
    if (l->n_slots <= 0) return GDN_EINVAL;
    if (!aligned16(l->state_slot)) return GDN_EALIGN;
    L.slot = l->state_slot;
    L.n_slots = l->n_slots;
  }
  if (!full) return GDN_OK;
  if (!std::isfinite(l->q_scale)) return GDN_EINVAL;
  L.q_scale = l->q_scale == 0.f ? 1.f : l->q_scale;
  const int ngate = (l->a_raw != nullptr) + (l->b_raw != nullptr) + (l->A_log != nullptr) + (l->dt_bias != nullptr);
  if (ngate != 0 && ngate != 4) return GDN_EINVAL;
  if (ngate == 4) {
    const void *gp[] = {l->a_raw, l->b_raw, l->A_log, l->dt_bias};
    for (const void *p : gp)
      if (!aligned16(p)) return GDN_EALIGN;
    L.a_raw = l->a_raw;
    L.b_raw = l->b_raw;
    L.A_log = l->A_log;
    L.dt_bias = l->dt_bias;
  }
  return GDN_OK;
}

// ------------------------------------------------------------------ TMA descriptors
using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// [T][H][D] bf16 rows viewed as a 3-D tensor (D, H, T); box = (box0, 1, rows)
bool encode_rows(CUtensorMap *map, const uint16_t *base, int D, int H, int T, int box0, int rows,
                 CUtensorMapSwizzle swz) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[3] = {cuuint64_t(D), cuuint64_t(H), cuuint64_t(T)};
  const cuuint64_t strides[2] = {cuuint64_t(D) * 2, cuuint64_t(H) * D * 2};
  const cuuint32_t box[3] = {cuuint32_t(box0), 1u, cuuint32_t(rows)};
  const cuuint32_t estr[3] = {1u, 1u, 1u};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<uint16_t *>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// [T][H][D] bf16 rows viewed as (D, H, T); box = (box0, box_h, rows), 128-byte swizzle
bool encode_rows_box(CUtensorMap *map, const uint16_t *base, int D, int H, int T, int box0, int box_h, int rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[3] = {cuuint64_t(D), cuuint64_t(H), cuuint64_t(T)};
  const cuuint64_t strides[2] = {cuuint64_t(D) * 2, cuuint64_t(H) * D * 2};
  const cuuint32_t box[3] = {cuuint32_t(box0), cuuint32_t(box_h), cuuint32_t(rows)};
  const cuuint32_t estr[3] = {1u, 1u, 1u};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<uint16_t *>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The plain layout runs the kernels compiled without any serving-layout indexing.
bool is_plain(const Serving &L) { return !L.slot && L.grp == 1 && L.q_scale == 1.f && !L.a_raw; }

template <int DK, bool SV>
gdn_status launch_verify_simt_sv(const VerifyArgs &a, const Serving &L, cudaStream_t stream) {
  const size_t smem = verify_simt_smem_bytes(a.max_nodes, DK);
  if (ensure_dyn_smem(reinterpret_cast<const void *>(verify_simt_kernel<DK, SV>), smem) != GDN_OK) return GDN_ECUDA;
  dim3 grid(a.dv / 32, a.H, a.B);
  verify_simt_kernel<DK, SV><<<grid, kThreads, smem, stream>>>(a, L);
  return launch_status();
}

template <int DK>
gdn_status launch_verify_simt(const VerifyArgs &a, const Serving &L, cudaStream_t stream) {
  return is_plain(L) ? launch_verify_simt_sv<DK, false>(a, L, stream) : launch_verify_simt_sv<DK, true>(a, L, stream);
}

int sm_count() {
  const DeviceInfo *d = nullptr;
  return device_info(&d) == GDN_OK ? d->sms : 0;
}

template <int DK, int DV, bool SV>
gdn_status launch_verify_tc_sv(const VerifyArgs &a, const Serving &L, cudaStream_t stream) {
  const int Np = ((a.max_nodes < 1 ? 1 : a.max_nodes) + 15) / 16 * 16;
  const int HK = a.H / L.grp;  // q/k heads
  CUtensorMap tk, tq, tv;
  if (!encode_rows(&tk, a.k, DK, HK, a.T, 64, Np, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_rows(&tq, a.q, DK, HK, a.T, 64, Np, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_rows(&tv, a.v, DV, a.H, a.T, DV, Np, CU_TENSOR_MAP_SWIZZLE_NONE))
    return GDN_ECUDA;
  const DeviceInfo *di = nullptr;
  int static_smem = 0;
  const void *fn = reinterpret_cast<const void *>(verify_tc_kernel<DK, DV, SV>);
  if (device_info(&di) != GDN_OK || func_static_smem(fn, &static_smem) != GDN_OK) return GDN_ECUDA;
  // deepest state ring that fits next to the node stages (1 KiB slack aligns the base)
  const long long room = (long long)di->optin - (long long)static_smem - 1024;
  int R = kMaxRing;
  while (R > 2 && (long long)tc_layout(DK, DV, Np, R).total > room) --R;
  const TcLayout lay = tc_layout(DK, DV, Np, R);
  if ((long long)lay.total > room) return GDN_ECUDA;
  // at least ~half an SM's shared memory, so a second CTA never waits on this one's tensor memory
  size_t smem = size_t(lay.total) + 1024;
  if (smem < 120u * 1024u) smem = 120u * 1024u;
  if (ensure_dyn_smem(fn, smem) != GDN_OK) return GDN_ECUDA;
  const long long pairs = (long long)a.B * a.H;
  const int sms = di->sms;
  if (sms <= 0) return GDN_ECUDA;
  const unsigned grid = unsigned(pairs < sms ? pairs : sms);
  verify_tc_kernel<DK, DV, SV><<<grid, kTcThreads, smem, stream>>>(tk, tq, tv, a, lay, L);
  return launch_status();
}

template <int DK, int DV>
gdn_status launch_verify_tc(const VerifyArgs &a, const Serving &L, cudaStream_t stream) {
  return is_plain(L) ? launch_verify_tc_sv<DK, DV, false>(a, L, stream) : launch_verify_tc_sv<DK, DV, true>(a, L, stream);
}

template <int DK, int DV, int NMAX, bool FUSE>
gdn_status launch_verify_stream(const VerifyArgs &a, const PrevCommit &c, const Serving &L, cudaStream_t stream) {
  const long long blocks = (long long)a.B * a.H;
  if (is_plain(L))
    verify_stream_kernel<DK, DV, NMAX, FUSE, false><<<unsigned(blocks), DV / 2, 0, stream>>>(a, c, L);
  else
    verify_stream_kernel<DK, DV, NMAX, FUSE, true><<<unsigned(blocks), DV / 2, 0, stream>>>(a, c, L);
  return launch_status();
}

template <int DK, int DV, bool FUSE>
gdn_status launch_verify_stream_n(const VerifyArgs &a, const PrevCommit &c, const Serving &L, cudaStream_t stream) {
  if (a.max_nodes <= 4) return launch_verify_stream<DK, DV, 4, FUSE>(a, c, L, stream);
  if (a.max_nodes <= 6) return launch_verify_stream<DK, DV, 6, FUSE>(a, c, L, stream);
  return launch_verify_stream<DK, DV, 8, FUSE>(a, c, L, stream);
}

template <bool FUSE>
gdn_status launch_verify_stream_dims(const VerifyArgs &a, const PrevCommit &c, const Serving &L, cudaStream_t s) {
  switch (a.dk * 1000 + a.dv) {
    case 32064: return launch_verify_stream_n<32, 64, FUSE>(a, c, L, s);
    case 32128: return launch_verify_stream_n<32, 128, FUSE>(a, c, L, s);
    case 64064: return launch_verify_stream_n<64, 64, FUSE>(a, c, L, s);
    case 64128: return launch_verify_stream_n<64, 128, FUSE>(a, c, L, s);
    case 128064: return launch_verify_stream_n<128, 64, FUSE>(a, c, L, s);
    default: return launch_verify_stream_n<128, 128, FUSE>(a, c, L, s);
  }
}

template <int DK, int DV, bool SV>
gdn_status launch_commit_sv(const CommitArgs &a, const Serving &L, cudaStream_t stream) {
  const size_t smem = commit_smem_bytes(a.max_path, DK, DV);
  if (ensure_dyn_smem(reinterpret_cast<const void *>(commit_kernel<DK, DV, SV>), smem) != GDN_OK) return GDN_ECUDA;
  const long long blocks = (long long)a.B * a.H * commit_row_split(DK, DV);
  commit_kernel<DK, DV, SV><<<unsigned(blocks), kThreads, smem, stream>>>(a, L);
  return launch_status();
}

template <int DK, int DV>
gdn_status launch_commit(const CommitArgs &a, const Serving &L, cudaStream_t stream) {
  return is_plain(L) ? launch_commit_sv<DK, DV, false>(a, L, stream) : launch_commit_sv<DK, DV, true>(a, L, stream);
}

template <int DK>
gdn_status launch_storeall(const StoreallArgs &a, cudaStream_t stream) {
  dim3 grid(a.dv / 32, a.H, a.B);
  verify_storeall_kernel<DK><<<grid, kThreads, 0, stream>>>(a);
  return launch_status();
}

gdn_status verify_simt_impl(const float *ST, const uint16_t *q, const uint16_t *k, const uint16_t *v,
                            const float *beta, const float *g, const int32_t *parent, const int32_t *cu_nodes,
                            int32_t B, int32_t H, int32_t T, int32_t d_k, int32_t d_v, int32_t max_nodes,
                            const Serving &L, float *o, float *U, float *G, int32_t *status, gdn_stream_t stream) {
  gdn_status st = check_verify_args(ST, q, k, v, beta, g, parent, cu_nodes, B, H, T, d_k, d_v,
                                    max_nodes, o, U, G, status, L);
  if (st != GDN_OK || B == 0 || T == 0) return st;
  if ((st = check_device()) != GDN_OK) return st;
  VerifyArgs a{ST, q, k, v, beta, g, parent, cu_nodes, B, H, T, d_k, d_v, max_nodes, o, U, G, status};
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  switch (d_k) {
    case 32: return launch_verify_simt<32>(a, L, s);
    case 64: return launch_verify_simt<64>(a, L, s);
    default: return launch_verify_simt<128>(a, L, s);
  }
}

gdn_status verify_impl(const float *ST, const uint16_t *q, const uint16_t *k, const uint16_t *v, const float *beta,
                       const float *g, const int32_t *parent, const int32_t *cu_nodes, int32_t B, int32_t H,
                       int32_t T, int32_t d_k, int32_t d_v, int32_t max_nodes, const Serving &L, float *o, float *U,
                       float *G, int32_t *status, gdn_stream_t stream) {
  gdn_status st = check_verify_args(ST, q, k, v, beta, g, parent, cu_nodes, B, H, T, d_k, d_v,
                                    max_nodes, o, U, G, status, L);
  if (st != GDN_OK || B == 0 || T == 0) return st;
  if (d_v == 32 || (d_k == 32 && max_nodes > kStreamMaxNodes))
    return verify_simt_impl(ST, q, k, v, beta, g, parent, cu_nodes, B, H, T, d_k, d_v, max_nodes, L, o, U, G,
                            status, stream);
  if ((st = check_device()) != GDN_OK) return st;
  if ((long long)B * H > 0x7fffffffLL) return GDN_EINVAL;
  VerifyArgs a{ST, q, k, v, beta, g, parent, cu_nodes, B, H, T, d_k, d_v, max_nodes, o, U, G, status};
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (max_nodes <= kStreamMaxNodes)  // small trees: CUDA-core streaming kernel
    return launch_verify_stream_dims<false>(a, PrevCommit{}, L, s);
  if (d_k == 128) return d_v == 128 ? launch_verify_tc<128, 128>(a, L, s) : launch_verify_tc<128, 64>(a, L, s);
  return d_v == 128 ? launch_verify_tc<64, 128>(a, L, s) : launch_verify_tc<64, 64>(a, L, s);
}

gdn_status commit_impl(float *ST, const float *U, const float *G, const uint16_t *k, const int32_t *parent,
                       const int32_t *cu_nodes, const int32_t *path, const int32_t *path_len, int32_t B, int32_t H,
                       int32_t T, int32_t d_k, int32_t d_v, int32_t max_path, const Serving &L, int32_t *status,
                       gdn_stream_t stream) {
  gdn_status st = check_commit_args(ST, U, G, k, parent, cu_nodes, path, path_len, B, H, T, d_k, d_v,
                                    max_path, status);
  if (st != GDN_OK || B == 0) return st;
  if ((st = check_device()) != GDN_OK) return st;
  if ((long long)B * H * 2 > 0x7fffffffLL) return GDN_EINVAL;  // (two CTAs per pair)
  CommitArgs a{ST, U, G, k, parent, cu_nodes, path, path_len, B, H, T, d_k, d_v, max_path, status};
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  switch (d_k * 1000 + d_v) {
    case 32032: return launch_commit<32, 32>(a, L, s);
    case 32064: return launch_commit<32, 64>(a, L, s);
    case 32128: return launch_commit<32, 128>(a, L, s);
    case 64032: return launch_commit<64, 32>(a, L, s);
    case 64064: return launch_commit<64, 64>(a, L, s);
    case 64128: return launch_commit<64, 128>(a, L, s);
    case 128032: return launch_commit<128, 32>(a, L, s);
    case 128064: return launch_commit<128, 64>(a, L, s);
    default: return launch_commit<128, 128>(a, L, s);
  }
}

gdn_status commit_verify_impl(float *ST, const float *U_prev, const float *G_prev, const uint16_t *k_prev,
                              const int32_t *parent_prev, const int32_t *cu_nodes_prev, const int32_t *path,
                              const int32_t *path_len, int32_t T_prev, int32_t max_path, const uint16_t *q,
                              const uint16_t *k, const uint16_t *v, const float *beta, const float *g,
                              const int32_t *parent, const int32_t *cu_nodes, int32_t B, int32_t H, int32_t T,
                              int32_t d_k, int32_t d_v, int32_t max_nodes, const Serving &L, float *o, float *U,
                              float *G, int32_t *status, gdn_stream_t stream) {
  gdn_status st = check_commit_args(ST, U_prev, G_prev, k_prev, parent_prev, cu_nodes_prev, path, path_len, B, H,
                                    T_prev, d_k, d_v, max_path, status);
  if (st != GDN_OK) return st;
  if ((st = check_verify_args(ST, q, k, v, beta, g, parent, cu_nodes, B, H, T, d_k, d_v, max_nodes, o, U, G,
                              status, L)) != GDN_OK)
    return st;
  if (B == 0) return GDN_OK;
  if (U && U == U_prev) return GDN_EINVAL;  // this step's pseudo-values may not overwrite the previous ones
  const bool fusable = T > 0 && d_v != 32 && max_nodes <= kStreamMaxNodes && max_path <= kFuseMaxPath;
  if (!fusable) {  // the same result from the two kernels in order
    if ((st = commit_impl(ST, U_prev, G_prev, k_prev, parent_prev, cu_nodes_prev, path, path_len, B, H, T_prev, d_k,
                          d_v, max_path, L, status, stream)) != GDN_OK)
      return st;
    return verify_impl(ST, q, k, v, beta, g, parent, cu_nodes, B, H, T, d_k, d_v, max_nodes, L, o, U, G, status,
                       stream);
  }
  if ((st = check_device()) != GDN_OK) return st;
  if ((long long)B * H > 0x7fffffffLL) return GDN_EINVAL;
  VerifyArgs a{ST, q, k, v, beta, g, parent, cu_nodes, B, H, T, d_k, d_v, max_nodes, o, U, G, status};
  PrevCommit c{ST, U_prev, G_prev, k_prev, parent_prev, cu_nodes_prev, path, path_len, T_prev, max_path};
  return launch_verify_stream_dims<true>(a, c, L, reinterpret_cast<cudaStream_t>(stream));
}

// ------------------------------------------------------------------ tree-bias attention
struct AttnPlan {
  int G = 0, tiles = 0, splits = 1, blocks_per_split = 1;
  size_t ws_bytes = 0;  // workspace the plan needs (0 with one split)
};

int attn_sms() {
  const int n = sm_count();
  return n > 0 ? n : 148;
}

// Query tiles per (request, head) and key splits. The attention kernel holds one CTA per SM, so
// a grid of n CTAs runs in ceil(n / SMs) waves, each as long as its slowest CTA. A CTA costs its
// key blocks plus about one block of fixed work (query load, pipeline fill); a split CTA also
// writes a partial tile (about one key block of bytes), and the combine pass reads all partials
// back (two block-equivalents per partial, spread over the SMs). The planner takes the split
// count with the least estimated time, the fewest splits on a tie, with at most 4 CTAs per SM in
// total and no more workspace than `ws_limit` bytes. With 4096-key prefixes this keeps grids of
// 128 and 256 (request, head, tile) CTAs unsplit, where splitting them measured slower.
AttnPlan attn_plan(int B, int Hq, int Hkv, int d, int max_nodes, int max_prefix, size_t ws_limit) {
  AttnPlan p;
  p.G = Hq / Hkv;
  p.tiles = (max_nodes * p.G + kAttnRows - 1) / kAttnRows;
  if (p.tiles < 1) p.tiles = 1;
  const long long base = (long long)B * Hkv * p.tiles;
  const int nblk = (max_prefix + kAttnKeys - 1) / kAttnKeys;
  const long long sms = attn_sms();
  const size_t per_split = size_t(base) * kAttnRows * size_t(d + 2) * 4;
  auto cost = [&](int s) {
    const int bps = (nblk + s - 1) / s;
    const long long ctas = base * s;
    const double waves = double((ctas + sms - 1) / sms);
    return s == 1 ? waves * (bps + 1.0) : waves * (bps + 2.0) + 2.0 * double(ctas) / double(sms);
  };
  int splits = 1;
  double best = cost(1);
  for (int s = 2; s <= nblk && base * s <= 4 * sms && per_split * size_t(s) <= ws_limit; ++s) {
    const double c = cost(s);
    if (c < best) best = c, splits = s;
  }
  const int bps = nblk > 0 ? (nblk + splits - 1) / splits : 1;
  p.splits = nblk > 0 ? (nblk + bps - 1) / bps : 1;
  p.blocks_per_split = bps;
  p.ws_bytes = p.splits > 1 ? per_split * p.splits : 0;
  return p;
}

gdn_status check_attn_shape(int32_t B, int32_t Hq, int32_t Hkv, int32_t d, int32_t max_nodes, int32_t max_prefix) {
  if (B < 0 || Hq <= 0 || Hkv <= 0 || max_nodes < 0 || max_prefix < 0) return GDN_EINVAL;
  if (Hq % Hkv != 0) return GDN_EINVAL;
  const int G = Hq / Hkv;
  if (G > kAttnRows || (G & (G - 1)) != 0) return GDN_EINVAL;  // whole nodes per 128-row tile
  if (d != 64 && d != 128) return GDN_EINVAL;
  if (max_nodes > kMaxNodes) return GDN_ETOOBIG;
  if (B > 65535 || Hkv > 65535) return GDN_EINVAL;
  return GDN_OK;
}

template <int D>
gdn_status launch_attention(const uint16_t *q, const uint16_t *k, const uint16_t *v, const uint16_t *k_cache,
                            const uint16_t *v_cache, const AttnArgs &a, cudaStream_t s) {
  CUtensorMap tq, tkc, tvc, tkt, tvt;
  const bool have_prefix = a.P_total > 0 && k_cache && v_cache;
  // without a prefix the cache maps are never read; they describe the node arrays instead
  const uint16_t *kc = have_prefix ? k_cache : k, *vc = have_prefix ? v_cache : v;
  const int pt = have_prefix ? a.P_total : a.T;
  if (!encode_rows_box(&tq, q, D, a.Hq, a.T, 64, a.G, kAttnRows / a.G) ||
      !encode_rows(&tkc, kc, D, a.Hkv, pt, 64, kAttnKeys, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_rows(&tvc, vc, D, a.Hkv, pt, 64, kAttnKeys, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_rows(&tkt, k, D, a.Hkv, a.T, 64, kAttnTreeKeys, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_rows(&tvt, v, D, a.Hkv, a.T, 64, kAttnTreeKeys, CU_TENSOR_MAP_SWIZZLE_128B))
    return GDN_ECUDA;
  const uint32_t smem = attn_smem_bytes(D);
  if (ensure_dyn_smem(reinterpret_cast<const void *>(tree_attention_kernel<D>), smem) != GDN_OK) return GDN_ECUDA;
  dim3 grid(unsigned(a.tiles * a.splits), unsigned(a.Hkv), unsigned(a.B));
  tree_attention_kernel<D><<<grid, kAttnThreads, smem, s>>>(tq, tkc, tvc, tkt, tvt, a);
  gdn_status st = launch_status();
  if (st != GDN_OK || a.splits == 1) return st;
  dim3 cgrid(unsigned(a.B * a.Hkv * a.tiles), unsigned(kAttnRows / 8));
  tree_attention_combine_kernel<D><<<cgrid, 256, 0, s>>>(a);
  return launch_status();
}

}  // namespace

// Scratch of gdn_tree_attention_noalloc: the split partial outputs and (max, sum) pairs, in a
// fixed array of the module rather than a caller buffer. Every GPU that loads the library holds
// these 32 MiB until the process exits; every call of that entry point shares them.
constexpr size_t kAttnNoAllocScratchBytes = size_t(32) << 20;
static __device__ __align__(256) unsigned char g_attn_noalloc_scratch[kAttnNoAllocScratchBytes];

namespace {

std::mutex g_noalloc_mu;
void *g_noalloc_addr[kMaxDevices] = {};

// The device address of the scratch array on the current device, looked up once per device.
// (Host code cannot use the array's name as a device pointer.)
gdn_status noalloc_scratch(void **out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return GDN_ECUDA;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (g_noalloc_addr[dev] == nullptr) {
    void *p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_attn_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr) {
      fprintf(stderr, "gdn_tree: scratch address lookup failed: %s\n", cudaGetErrorString(e));
      return GDN_ECUDA;
    }
    g_noalloc_addr[dev] = p;
  }
  *out = g_noalloc_addr[dev];
  return GDN_OK;
}

}  // namespace

extern "C" {

int32_t gdn_abi_version(void) { return 3; }

const char *gdn_status_str(gdn_status s) {
  switch (s) {
    case GDN_OK: return "GDN_OK";
    case GDN_EINVAL: return "GDN_EINVAL: invalid argument";
    case GDN_ETOOBIG: return "GDN_ETOOBIG: more than 64 nodes or path entries per request";
    case GDN_EALIGN: return "GDN_EALIGN: array not 16-byte aligned";
    case GDN_ECUDA: return "GDN_ECUDA: CUDA runtime error";
    case GDN_EARCH: return "GDN_EARCH: device is not sm_103";
  }
  return "GDN_?: unknown status";
}

gdn_status gdn_tree_verify_simt(const float *ST, const uint16_t *q, const uint16_t *k,
                                const uint16_t *v, const float *beta, const float *g,
                                const int32_t *parent, const int32_t *cu_nodes, int32_t B,
                                int32_t H, int32_t T, int32_t d_k, int32_t d_v, int32_t max_nodes,
                                float *o, float *U, float *G, int32_t *status,
                                gdn_stream_t stream) {
  return verify_simt_impl(ST, q, k, v, beta, g, parent, cu_nodes, B, H, T, d_k, d_v, max_nodes, Serving{}, o, U, G,
                          status, stream);
}

gdn_status gdn_tree_verify(const float *ST, const uint16_t *q, const uint16_t *k, const uint16_t *v,
                           const float *beta, const float *g, const int32_t *parent,
                           const int32_t *cu_nodes, int32_t B, int32_t H, int32_t T, int32_t d_k,
                           int32_t d_v, int32_t max_nodes, float *o, float *U, float *G,
                           int32_t *status, gdn_stream_t stream) {
  return verify_impl(ST, q, k, v, beta, g, parent, cu_nodes, B, H, T, d_k, d_v, max_nodes, Serving{}, o, U, G, status,
                     stream);
}

gdn_status gdn_tree_verify_ex(const float *ST, const uint16_t *q, const uint16_t *k, const uint16_t *v,
                              const float *beta, const float *g, const int32_t *parent,
                              const int32_t *cu_nodes, int32_t B, int32_t H, int32_t T, int32_t d_k,
                              int32_t d_v, int32_t max_nodes, const gdn_layout *layout, float *o,
                              float *U, float *G, int32_t *status, gdn_stream_t stream) {
  Serving L;
  const gdn_status st = make_serving(layout, H, true, L);
  if (st != GDN_OK) return st;
  return verify_impl(ST, q, k, v, beta, g, parent, cu_nodes, B, H, T, d_k, d_v, max_nodes, L, o, U, G, status, stream);
}

gdn_status gdn_tree_commit(float *ST, const float *U, const float *G, const uint16_t *k,
                           const int32_t *parent, const int32_t *cu_nodes, const int32_t *path,
                           const int32_t *path_len, int32_t B, int32_t H, int32_t T, int32_t d_k,
                           int32_t d_v, int32_t max_path, int32_t *status, gdn_stream_t stream) {
  return commit_impl(ST, U, G, k, parent, cu_nodes, path, path_len, B, H, T, d_k, d_v, max_path, Serving{}, status,
                     stream);
}

gdn_status gdn_tree_commit_ex(float *ST, const float *U, const float *G, const uint16_t *k,
                              const int32_t *parent, const int32_t *cu_nodes, const int32_t *path,
                              const int32_t *path_len, int32_t B, int32_t H, int32_t T, int32_t d_k,
                              int32_t d_v, int32_t max_path, const gdn_layout *layout, int32_t *status,
                              gdn_stream_t stream) {
  Serving L;
  const gdn_status st = make_serving(layout, H, false, L);
  if (st != GDN_OK) return st;
  return commit_impl(ST, U, G, k, parent, cu_nodes, path, path_len, B, H, T, d_k, d_v, max_path, L, status, stream);
}

gdn_status gdn_tree_accept_greedy(const int32_t *draft_tok, const int32_t *target_tok,
                                  const int32_t *parent, const int32_t *cu_nodes, int32_t B,
                                  int32_t T, int32_t max_nodes, int32_t max_path, int32_t *path,
                                  int32_t *path_len, int32_t *status, gdn_stream_t stream) {
  if (B < 0 || T < 0 || max_nodes < 0 || max_path < 0) return GDN_EINVAL;
  if (max_nodes > kMaxNodes || max_path > kMaxNodes) return GDN_ETOOBIG;
  if (B == 0) return GDN_OK;
  if (!cu_nodes || !path_len || (max_path > 0 && !path)) return GDN_EINVAL;
  if (T > 0 && (!draft_tok || !target_tok || !parent)) return GDN_EINVAL;
  const void *ptrs[] = {draft_tok, target_tok, parent, cu_nodes, path, path_len, status};
  for (const void *p : ptrs)
    if (p && !aligned16(p)) return GDN_EALIGN;
  gdn_status st;
  if ((st = check_device()) != GDN_OK) return st;
  AcceptArgs a{draft_tok, target_tok, parent, cu_nodes, B, T, max_nodes, max_path, path, path_len, status};
  const unsigned blocks = unsigned((B + kAcceptWarps - 1) / kAcceptWarps);
  accept_greedy_kernel<<<blocks, kAcceptWarps * 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(a);
  return launch_status();
}

gdn_status gdn_tree_commit_verify(float *ST, const float *U_prev, const float *G_prev,
                                  const uint16_t *k_prev, const int32_t *parent_prev,
                                  const int32_t *cu_nodes_prev, const int32_t *path,
                                  const int32_t *path_len, int32_t T_prev, int32_t max_path,
                                  const uint16_t *q, const uint16_t *k, const uint16_t *v,
                                  const float *beta, const float *g, const int32_t *parent,
                                  const int32_t *cu_nodes, int32_t B, int32_t H, int32_t T,
                                  int32_t d_k, int32_t d_v, int32_t max_nodes, float *o, float *U,
                                  float *G, int32_t *status, gdn_stream_t stream) {
  return commit_verify_impl(ST, U_prev, G_prev, k_prev, parent_prev, cu_nodes_prev, path, path_len, T_prev, max_path,
                            q, k, v, beta, g, parent, cu_nodes, B, H, T, d_k, d_v, max_nodes, Serving{}, o, U, G,
                            status, stream);
}

gdn_status gdn_tree_commit_verify_ex(float *ST, const float *U_prev, const float *G_prev,
                                     const uint16_t *k_prev, const int32_t *parent_prev,
                                     const int32_t *cu_nodes_prev, const int32_t *path,
                                     const int32_t *path_len, int32_t T_prev, int32_t max_path,
                                     const uint16_t *q, const uint16_t *k, const uint16_t *v,
                                     const float *beta, const float *g, const int32_t *parent,
                                     const int32_t *cu_nodes, int32_t B, int32_t H, int32_t T,
                                     int32_t d_k, int32_t d_v, int32_t max_nodes, const gdn_layout *layout,
                                     float *o, float *U, float *G, int32_t *status, gdn_stream_t stream) {
  Serving L;
  const gdn_status st = make_serving(layout, H, true, L);
  if (st != GDN_OK) return st;
  return commit_verify_impl(ST, U_prev, G_prev, k_prev, parent_prev, cu_nodes_prev, path, path_len, T_prev, max_path,
                            q, k, v, beta, g, parent, cu_nodes, B, H, T, d_k, d_v, max_nodes, L, o, U, G, status,
                            stream);
}

gdn_status gdn_tree_verify_storeall(const float *ST, const uint16_t *q, const uint16_t *k,
                                    const uint16_t *v, const float *beta, const float *g,
                                    const int32_t *parent, const int32_t *cu_nodes, int32_t B,
                                    int32_t H, int32_t T, int32_t d_k, int32_t d_v,
                                    int32_t max_nodes, float *snapshots, float *o, float *U,
                                    float *G, int32_t *status, gdn_stream_t stream) {
  gdn_status st = check_verify_args(ST, q, k, v, beta, g, parent, cu_nodes, B, H, T, d_k, d_v,
                                    max_nodes, o, U, G, status);
  if (st != GDN_OK || B == 0 || T == 0) return st;
  if (!snapshots) return GDN_EINVAL;
  if (!aligned16(snapshots)) return GDN_EALIGN;
  if ((st = check_device()) != GDN_OK) return st;
  StoreallArgs a{ST, q, k, v, beta, g, parent, cu_nodes, B, H, T, d_k, d_v, max_nodes, snapshots, o, U, G,
                 status};
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  switch (d_k) {
    case 32: return launch_storeall<32>(a, s);
    case 64: return launch_storeall<64>(a, s);
    default: return launch_storeall<128>(a, s);
  }
}

gdn_status gdn_tree_commit_storeall(float *ST, const float *snapshots, const int32_t *parent,
                                    const int32_t *cu_nodes, const int32_t *path,
                                    const int32_t *path_len, int32_t B, int32_t H, int32_t T,
                                    int32_t d_k, int32_t d_v, int32_t max_path, int32_t *status,
                                    gdn_stream_t stream) {
  gdn_status st = check_commit_args(ST, snapshots, snapshots, snapshots, parent, cu_nodes, path,
                                    path_len, B, H, T, d_k, d_v, max_path, status);
  if (st != GDN_OK || B == 0) return st;
  if ((st = check_device()) != GDN_OK) return st;
  StoreallCommitArgs a{ST, snapshots, parent, cu_nodes, path, path_len, B, H, T, d_k, d_v, max_path, status};
  const int per_cta = kThreads * 4;
  const long long nchunk = (d_k * d_v / 4 + per_cta - 1) / per_cta;
  const long long blocks = (long long)B * H * nchunk;
  if (blocks > 0x7fffffffLL) return GDN_EINVAL;
  commit_storeall_kernel<<<unsigned(blocks), kThreads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(a);
  return launch_status();
}

gdn_status gdn_tree_budget_topb(const float *p_accept, int32_t R, int32_t K, int32_t budget, int32_t *n_sel,
                                float *survival, int32_t *cu_nodes, int32_t *parent, int32_t *status,
                                gdn_stream_t stream) {
  if (R < 0 || K < 1 || K > kMaxNodes - 1 || budget < 0) return GDN_EINVAL;
  if ((long long)R * K > kTopbMaxItems) return GDN_ETOOBIG;
  // keys, staged probabilities and per-request counts all sit in one CTA's shared memory
  const size_t topb_smem = size_t(R) * K * 12 + size_t(R) * 4;
  if (topb_smem > kSmemPerBlockMax) return GDN_ETOOBIG;
  if (R == 0) return GDN_OK;
  if (!p_accept || !n_sel || (parent && !cu_nodes)) return GDN_EINVAL;
  const void *ptrs[] = {p_accept, n_sel, survival, cu_nodes, parent, status};
  for (const void *p : ptrs)
    if (p && !aligned16(p)) return GDN_EALIGN;
  gdn_status st;
  if ((st = check_device()) != GDN_OK) return st;
  if (ensure_dyn_smem(reinterpret_cast<const void *>(topb_kernel), topb_smem) != GDN_OK) return GDN_ECUDA;
  TopbArgs a{p_accept, R, K, budget, n_sel, survival, cu_nodes, parent, status};
  topb_kernel<<<1, kTopbThreads, topb_smem, reinterpret_cast<cudaStream_t>(stream)>>>(a);
  return launch_status();
}

gdn_status gdn_tree_grow_best_first(const float *p_edge, int32_t R, int32_t fanout, int32_t depth, float threshold,
                                    int32_t max_nodes, int32_t *n_nodes, int32_t *parent_local, int32_t *cand,
                                    float *value, int32_t *cu_nodes, int32_t *parent, int32_t *status,
                                    gdn_stream_t stream) {
  if (R < 0 || fanout < 1 || depth < 0 || max_nodes < 0 || std::isnan(threshold)) return GDN_EINVAL;
  if (max_nodes > kMaxNodes || R > 0x7fffffff / (max_nodes > 0 ? max_nodes : 1)) return GDN_ETOOBIG;
  long long C = 0, width = 1;
  for (int l = 0; l <= depth; ++l) {
    C += width;
    if (C > kGrowMaxCand) return GDN_ETOOBIG;
    width *= fanout;
  }
  if (R == 0) return GDN_OK;
  if (!p_edge || !n_nodes || !parent_local || (!cu_nodes) != (!parent)) return GDN_EINVAL;
  const void *ptrs[] = {p_edge, n_nodes, parent_local, cand, value, cu_nodes, parent, status};
  for (const void *p : ptrs)
    if (p && !aligned16(p)) return GDN_EALIGN;
  gdn_status st;
  if ((st = check_device()) != GDN_OK) return st;
  const size_t smem = size_t(C) * 8 + size_t(C) * 4;  // candidate keys (then output positions), values
  if (ensure_dyn_smem(reinterpret_cast<const void *>(grow_kernel), smem) != GDN_OK) return GDN_ECUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  GrowArgs a{p_edge, R, fanout, depth, int(C), max_nodes, threshold, n_nodes, cand, parent_local, value, status};
  grow_kernel<<<unsigned(R), kGrowThreads, smem, s>>>(a);
  if ((st = launch_status()) != GDN_OK || !cu_nodes) return st;
  PackArgs pa{n_nodes, parent_local, R, max_nodes, cu_nodes, parent};
  pack_scan_kernel<<<1, kScanThreads, 0, s>>>(pa);
  if ((st = launch_status()) != GDN_OK) return st;
  pack_copy_kernel<<<unsigned((R + kCopyWarps - 1) / kCopyWarps), kCopyWarps * 32, 0, s>>>(pa);
  return launch_status();
}

gdn_status gdn_tree_attention_noalloc(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                                      const uint16_t *k_cache, const uint16_t *v_cache, const int32_t *cu_prefix,
                                      const int32_t *parent, const int32_t *cu_nodes, int32_t B, int32_t H_q,
                                      int32_t H_kv, int32_t T, int32_t P_total, int32_t d, int32_t max_nodes,
                                      int32_t max_prefix, float scale, float *o, int32_t *status, gdn_stream_t stream) {
  gdn_status st = check_attn_shape(B, H_q, H_kv, d, max_nodes, max_prefix);
  if (st != GDN_OK) return st;
  if (B == 0 || T == 0 || max_nodes == 0) return GDN_OK;
  if (T < 0 || P_total < 0 || !std::isfinite(scale) || !(scale > 0.f)) return GDN_EINVAL;
  // The key splits gdn_tree_attention makes with a workspace of the scratch's size: the same
  // plan as with an unlimited workspace whenever that plan fits, else fewer splits (one split
  // needs no scratch at all), so every valid size runs.
  const size_t need = attn_plan(B, H_q, H_kv, d, max_nodes, max_prefix, kAttnNoAllocScratchBytes).ws_bytes;
  if (need > kAttnNoAllocScratchBytes) {  // the planner never asks for more; kept as a guard
    fprintf(stderr, "gdn_tree_attention_noalloc: these sizes need %zu bytes of scratch, more than the built-in %zu\n",
            need, kAttnNoAllocScratchBytes);
    return GDN_ETOOBIG;
  }
  void *scratch = nullptr;
  if (need > 0) {
    if ((st = check_device()) != GDN_OK) return st;
    if ((st = noalloc_scratch(&scratch)) != GDN_OK) return st;
  }
  return gdn_tree_attention(q, k, v, k_cache, v_cache, cu_prefix, parent, cu_nodes, B, H_q, H_kv, T, P_total, d,
                            max_nodes, max_prefix, scale, o, scratch, need > 0 ? kAttnNoAllocScratchBytes : 0,
                            status, stream);
}

size_t gdn_tree_attention_workspace_size(int32_t B, int32_t H_q, int32_t H_kv, int32_t d, int32_t max_nodes,
                                         int32_t max_prefix) {
  if (check_attn_shape(B, H_q, H_kv, d, max_nodes, max_prefix) != GDN_OK || B == 0) return 0;
  return attn_plan(B, H_q, H_kv, d, max_nodes, max_prefix, ~size_t(0)).ws_bytes;
}

gdn_status gdn_tree_attention(const uint16_t *q, const uint16_t *k, const uint16_t *v, const uint16_t *k_cache,
                              const uint16_t *v_cache, const int32_t *cu_prefix, const int32_t *parent,
                              const int32_t *cu_nodes, int32_t B, int32_t H_q, int32_t H_kv, int32_t T,
                              int32_t P_total, int32_t d, int32_t max_nodes, int32_t max_prefix, float scale, float *o,
                              void *workspace, size_t workspace_bytes, int32_t *status, gdn_stream_t stream) {
  gdn_status st = check_attn_shape(B, H_q, H_kv, d, max_nodes, max_prefix);
  if (st != GDN_OK) return st;
  if (T < 0 || P_total < 0 || !std::isfinite(scale) || !(scale > 0.f)) return GDN_EINVAL;
  if (B == 0 || T == 0 || max_nodes == 0) return GDN_OK;
  if (!q || !k || !v || !cu_prefix || !parent || !cu_nodes || !o) return GDN_EINVAL;
  if (P_total > 0 && (!k_cache || !v_cache)) return GDN_EINVAL;
  const void *ptrs[] = {q, k, v, k_cache, v_cache, cu_prefix, parent, cu_nodes, o, workspace, status};
  for (const void *p : ptrs)
    if (p && !aligned16(p)) return GDN_EALIGN;
  if ((st = check_device()) != GDN_OK) return st;
  const AttnPlan plan = attn_plan(B, H_q, H_kv, d, max_nodes, max_prefix, workspace ? workspace_bytes : 0);
  if ((long long)plan.tiles * plan.splits > 0x7fffffffLL) return GDN_EINVAL;
  AttnArgs a{parent, cu_nodes, cu_prefix, B, H_q, H_kv, plan.G, T, P_total, max_nodes, max_prefix,
             plan.tiles, plan.splits, plan.blocks_per_split, scale * 1.4426950408889634f, o, nullptr, nullptr,
             status};
  if (plan.splits > 1) {  // partial outputs first, then the (max, sum) pairs
    a.ws_o = static_cast<float *>(workspace);
    a.ws_ml = a.ws_o + plan.ws_bytes / 4 / size_t(d + 2) * size_t(d);
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  return d == 128 ? launch_attention<128>(q, k, v, k_cache, v_cache, a, s)
                  : launch_attention<64>(q, k, v, k_cache, v_cache, a, s);
}

}  // extern "C"
