// C ABI of the sparse MLA library: argument validation, device checks and
// the launch sequence of each call.  Declarations and the contract of every
// entry point are in include/sparse_mla.h.
#include <errno.h>
#include <stdarg.h>
#include <stdio.h>

#include <atomic>
#include <cmath>
#include <mutex>
#include <string>

#include "../../include/sparse_mla.h"
#include "smla_common.cuh"

namespace {

thread_local std::string g_last_error;
std::atomic<uint64_t> g_launches{0};

void count_launches(uint64_t n) { g_launches.fetch_add(n, std::memory_order_relaxed); }

int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return code;
}

int cuda_fail(cudaError_t e, const char* what) {
  return fail(-EIO, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool supported_h(int H) { return H == 8 || H == 16 || H == 32 || H == 64 || H == 128; }
// The tensor-core kernels take every supported H (a 128-row head tile, rows
// past H zero) up to their top-k limit; larger top-k runs the CUDA-core kernels.
bool use_tc(int H, int topk) { (void)H; return topk <= smla::kTcMaxTopk; }
// With at most 16 heads the forward runs the slots-as-rows tensor-core kernel
// (the heads are the N = 16 columns of its MMAs instead of a 128-row tile).
bool use_small_fwd(int H) { return H <= 16; }

// The backward kernel for this head count and top-k: the slots-as-rows tensor-core
// kernel for H <= 16, the 128-row head tile above, the CUDA-core kernels past the
// tensor-core top-k limit.
cudaError_t launch_bwd_any(const smla::BwdArgs& a, cudaStream_t s) {
  if (!use_tc(a.H, a.topk)) return smla::launch_bwd_simt(a, s);
  return a.H <= 16 ? smla::launch_bwd_tc_small(a, s) : smla::launch_bwd_tc(a, s);
}

// The kernels are built for sm_103a only; refuse any other device.
int check_device() {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  int major = 0, minor = 0;
  if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess)
    return cuda_fail(e, "cudaDeviceGetAttribute");
  if ((e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess)
    return cuda_fail(e, "cudaDeviceGetAttribute");
  if (major != 10 || minor != 3)
    return fail(-ENOTSUP, "device %d is sm_%d%d; this library is built for sm_103a only", dev,
                major, minor);
  return 0;
}

int check_shape(int T, int H, int topk, float scale) {
  if (T < 0) return fail(-EINVAL, "T must be >= 0 (got %d)", T);
  if (!supported_h(H)) return fail(-EINVAL, "H must be one of 8, 16, 32, 64, 128 (got %d)", H);
  if (topk <= 0 || topk % 64 != 0)
    return fail(-EINVAL, "topk must be a positive multiple of 64 (got %d)", topk);
  if (!std::isfinite(scale)) return fail(-EINVAL, "scale must be finite");
  return 0;
}

#define SMLA_REQUIRE_PTR(p)                                                   \
  do {                                                                        \
    if ((p) == nullptr) return fail(-EINVAL, "%s must not be NULL", #p);      \
    if (!aligned16(p)) return fail(-EINVAL, "%s must be 16-byte aligned", #p); \
  } while (0)

size_t delta_bytes(int T, int H) { return (((size_t)T * H * sizeof(float)) + 255) & ~(size_t)255; }
size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }
constexpr size_t kTopkSmemLimit = 220 * 1024;   // dynamic shared memory of the top-k selection

// Workspace of the deterministic dKV mode: Delta, the per-row slot lists (CSR:
// offset, fill cursor, reduction cursor, scan scratch, sorted slot ids) and the
// per-slot contributions of one chunk of tokens.
struct DetLayout {
  size_t offset, cursor, pos, sums, seg, g;   // byte offsets
  size_t per_token;                           // contribution bytes per token of a chunk
  int ng;                                     // head groups per token (contributions per slot)
};
constexpr size_t kDetChunkBytes = size_t(4) << 30;   // default chunk: 4 GiB of contributions

DetLayout det_layout(int T, int H, int topk) {
  DetLayout L;
  L.ng = use_tc(H, topk) ? 1 : smla::simt_head_groups(H);
  size_t at = delta_bytes(T, H);
  L.offset = at; at += align256(sizeof(int) * ((size_t)T + 1));
  L.cursor = at; at += align256(sizeof(int) * (size_t)T);
  L.pos = at;    at += align256(sizeof(int) * (size_t)T);
  L.sums = at;   at += align256(sizeof(int) * (size_t)smla::det_scan_tiles(T));
  L.seg = at;    at += align256(sizeof(int) * (size_t)T * topk);
  L.g = at;
  L.per_token = (size_t)L.ng * topk * smla::kDqk * sizeof(float);
  return L;
}
size_t det_default_tokens(int T, const DetLayout& L) {
  size_t tc = kDetChunkBytes / L.per_token;
  if (tc < 1) tc = 1;
  if (tc > (size_t)T) tc = (size_t)T;
  return tc;
}

}  // namespace

extern "C" {

const char* sparse_mla_last_error(void) { return g_last_error.c_str(); }

const char* sparse_mla_version(void) { return "sparse_mla_gb300 0.1.0 (sm_103a)"; }

uint64_t sparse_mla_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

int sparse_mla_device_status(uint32_t* status, int clear) {
  g_last_error.clear();
  if (status == nullptr) return fail(-EINVAL, "status must not be NULL");
  if (int r = check_device()) return r;
  cudaError_t e = cudaDeviceSynchronize();
  if (e == cudaSuccess) e = smla::read_tc_status(status, clear != 0);
  if (e != cudaSuccess) return cuda_fail(e, "sparse_mla_device_status");
  return 0;
}

int sparse_mla_wait_selftest(void* stream) {
  g_last_error.clear();
  if (int r = check_device()) return r;
  cudaError_t e = smla::launch_wait_selftest(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "sparse_mla_wait_selftest launch");
  count_launches(1);
  return 0;
}

int sparse_mla_bounds_selftest(void* stream) {
  g_last_error.clear();
#ifdef SMLA_DEBUG
  if (int r = check_device()) return r;
  cudaError_t e = smla::launch_bounds_selftest(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "sparse_mla_bounds_selftest launch");
  count_launches(1);
  return 0;
#else
  (void)stream;
  return fail(-ENOSYS, "device bounds checks are compiled only into the debug build (-DSMLA_DEBUG)");
#endif
}

int sparse_mla_topk(const float* scores, int64_t ld, int T, int ncols, const int32_t* cu_seqlens, int B, int topk,
                    int32_t* indices, void* stream) {
  g_last_error.clear();
  if (T < 0) return fail(-EINVAL, "T must be >= 0 (got %d)", T);
  if (ncols <= 0 || ld < ncols) return fail(-EINVAL, "need 0 < ncols <= ld (got ncols %d, ld %lld)", ncols, (long long)ld);
  if (topk <= 0 || topk > 8192) return fail(-EINVAL, "topk must be in [1, 8192] (got %d)", topk);
  if (B < 1) return fail(-EINVAL, "B must be >= 1 (got %d)", B);
  if (smla::topk_smem_bytes(ncols, topk) > kTopkSmemLimit)
    return fail(-EINVAL, "ncols %d with topk %d exceeds the shared-memory selection (4 (ncols + 3) + 8 max(1024, topk "
                "rounded up to a power of two) <= %zu bytes)", ncols, topk, kTopkSmemLimit);
  if (T == 0) return 0;
  if (scores == nullptr || cu_seqlens == nullptr || indices == nullptr)
    return fail(-EINVAL, "scores, cu_seqlens and indices must not be NULL");
  if (int r = check_device()) return r;
  int dev = 0, nsm = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess)
    e = smla::launch_topk(scores, ld, ncols, cu_seqlens, B, T, topk, indices, nsm, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "sparse_mla_topk launch");
  count_launches(1);
  return 0;
}

}  // extern "C"

namespace {

int check_rows(int T, int t0, int nt) {
  if (t0 < 0 || nt < 0 || (int64_t)t0 + nt > T)
    return fail(-EINVAL, "need 0 <= t0, 0 <= nt and t0 + nt <= T (got t0 %d, nt %d, T %d)", t0, nt, T);
  return 0;
}

// forward over query rows [t0, t0 + nt); shapes and the range are checked
int fwd_rows(const smla_bf16_t* q, const smla_bf16_t* kv, const int32_t* indices, int T, int H, int topk,
             float scale, int t0, int nt, smla_bf16_t* out, float* lse, void* stream) {
  if (nt == 0) return 0;
  SMLA_REQUIRE_PTR(q);
  SMLA_REQUIRE_PTR(kv);
  SMLA_REQUIRE_PTR(indices);
  SMLA_REQUIRE_PTR(out);
  SMLA_REQUIRE_PTR(lse);
  if (int r = check_device()) return r;
  smla::FwdArgs a{q, kv, indices, out, lse, T, H, topk, scale};
  a.t0 = t0;
  a.nt = nt;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = !use_tc(H, topk) ? smla::launch_fwd_simt(a, s)
                  : use_small_fwd(H) ? smla::launch_fwd_tc_small(a, s)
                                     : smla::launch_fwd_tc(a, s);
  if (e != cudaSuccess) return cuda_fail(e, "sparse_mla_fwd launch");
  count_launches(1);
  return 0;
}

}  // namespace

extern "C" {

int sparse_mla_fwd(const smla_bf16_t* q, const smla_bf16_t* kv, const int32_t* indices,
                   const int32_t* cu_seqlens, int T, int H, int topk, int B, float scale,
                   smla_bf16_t* out, float* lse, void* stream) {
  (void)cu_seqlens;
  (void)B;
  g_last_error.clear();
  if (int r = check_shape(T, H, topk, scale)) return r;
  return fwd_rows(q, kv, indices, T, H, topk, scale, 0, T, out, lse, stream);
}

int sparse_mla_fwd_rows(const smla_bf16_t* q, const smla_bf16_t* kv, const int32_t* indices,
                        const int32_t* cu_seqlens, int T, int H, int topk, int B, float scale, int t0, int nt,
                        smla_bf16_t* out, float* lse, void* stream) {
  (void)cu_seqlens;
  (void)B;
  g_last_error.clear();
  if (int r = check_shape(T, H, topk, scale)) return r;
  if (int r = check_rows(T, t0, nt)) return r;
  return fwd_rows(q, kv, indices, T, H, topk, scale, t0, nt, out, lse, stream);
}

int sparse_mla_bwd_rows(const smla_bf16_t* q, const smla_bf16_t* kv, const smla_bf16_t* out,
                        const smla_bf16_t* dout, const float* lse, const int32_t* indices,
                        const int32_t* cu_seqlens, int T, int H, int topk, int B, float scale, int t0, int nt,
                        smla_bf16_t* dq, float* dkv_f32, void* workspace, size_t workspace_bytes, void* stream) {
  (void)cu_seqlens;
  (void)B;
  g_last_error.clear();
  if (int r = check_shape(T, H, topk, scale)) return r;
  if (int r = check_rows(T, t0, nt)) return r;
  if (nt == 0) return 0;
  SMLA_REQUIRE_PTR(q);
  SMLA_REQUIRE_PTR(kv);
  SMLA_REQUIRE_PTR(out);
  SMLA_REQUIRE_PTR(dout);
  SMLA_REQUIRE_PTR(lse);
  SMLA_REQUIRE_PTR(indices);
  SMLA_REQUIRE_PTR(dq);
  SMLA_REQUIRE_PTR(dkv_f32);
  SMLA_REQUIRE_PTR(workspace);
  if (workspace_bytes < delta_bytes(T, H))
    return fail(-EINVAL, "workspace too small: %zu bytes given, %zu needed", workspace_bytes, delta_bytes(T, H));
  if (int r = check_device()) return r;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // Delta of rows t0.. at their own place, so that ranges on other streams never share it
  float* delta = static_cast<float*>(workspace);
  const int64_t r0 = (int64_t)t0 * H;
  cudaError_t e = smla::launch_delta(out + r0 * smla::kDv, dout + r0 * smla::kDv, delta + r0, (int64_t)nt * H, s);
  if (e != cudaSuccess) return cuda_fail(e, "delta launch");
  count_launches(1);
  smla::BwdArgs a{q, kv, dout, lse, delta, indices, dq, dkv_f32, T, H, topk, scale};
  a.t0 = t0;
  a.nt = nt;
  e = launch_bwd_any(a, s);
  if (e != cudaSuccess) return cuda_fail(e, "sparse_mla_bwd_rows launch");
  count_launches(1);
  return 0;
}

int sparse_mla_dkv_cast(const float* dkv_f32, smla_bf16_t* dkv, int T, void* stream) {
  g_last_error.clear();
  if (T < 0) return fail(-EINVAL, "T must be >= 0 (got %d)", T);
  if (T == 0) return 0;
  SMLA_REQUIRE_PTR(dkv_f32);
  SMLA_REQUIRE_PTR(dkv);
  if (int r = check_device()) return r;
  cudaError_t e = smla::launch_cast_bf16(dkv_f32, dkv, (int64_t)T * smla::kDqk, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "dkv cast launch");
  count_launches(1);
  return 0;
}

size_t sparse_mla_bwd_workspace_bytes(int T, int H, int topk, int dkv_mode) {
  if (T < 0 || !supported_h(H) || topk <= 0 || topk % 64 != 0) return 0;
  if (dkv_mode == SMLA_DKV_ATOMIC) return delta_bytes(T, H);
  if (dkv_mode != SMLA_DKV_DETERMINISTIC || (int64_t)T * topk > INT32_MAX) return 0;
  const DetLayout L = det_layout(T, H, topk);
  return L.g + det_default_tokens(T, L) * L.per_token;
}

int sparse_mla_bwd(const smla_bf16_t* q, const smla_bf16_t* kv, const smla_bf16_t* out,
                   const smla_bf16_t* dout, const float* lse, const int32_t* indices,
                   const int32_t* cu_seqlens, int T, int H, int topk, int B, float scale,
                   int dkv_mode, smla_bf16_t* dq, float* dkv_f32, smla_bf16_t* dkv,
                   void* workspace, size_t workspace_bytes, void* stream) {
  (void)cu_seqlens;
  (void)B;
  g_last_error.clear();
  if (int r = check_shape(T, H, topk, scale)) return r;
  if (dkv_mode != SMLA_DKV_ATOMIC && dkv_mode != SMLA_DKV_DETERMINISTIC)
    return fail(-EINVAL, "unknown dkv_mode %d", dkv_mode);
  if (dkv_mode == SMLA_DKV_DETERMINISTIC && (int64_t)T * topk > INT32_MAX)
    return fail(-EINVAL, "SMLA_DKV_DETERMINISTIC needs T * topk <= 2^31 - 1 (got %lld)", (long long)T * topk);
  if (T == 0) return 0;
  SMLA_REQUIRE_PTR(q);
  SMLA_REQUIRE_PTR(kv);
  SMLA_REQUIRE_PTR(out);
  SMLA_REQUIRE_PTR(dout);
  SMLA_REQUIRE_PTR(lse);
  SMLA_REQUIRE_PTR(indices);
  SMLA_REQUIRE_PTR(dq);
  SMLA_REQUIRE_PTR(dkv_f32);
  if (dkv != nullptr && !aligned16(dkv)) return fail(-EINVAL, "dkv must be 16-byte aligned");
  SMLA_REQUIRE_PTR(workspace);
  const DetLayout L = det_layout(T, H, topk);
  const size_t need = dkv_mode == SMLA_DKV_ATOMIC ? delta_bytes(T, H) : L.g + L.per_token;
  if (workspace_bytes < need)
    return fail(-EINVAL, "workspace too small: %zu bytes given, %zu needed", workspace_bytes, need);
  if (int r = check_device()) return r;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  float* delta = static_cast<float*>(workspace);
  cudaError_t e = smla::launch_delta(out, dout, delta, (int64_t)T * H, s);
  if (e != cudaSuccess) return cuda_fail(e, "delta launch");
  count_launches(1);
  e = cudaMemsetAsync(dkv_f32, 0, (size_t)T * smla::kDqk * sizeof(float), s);
  if (e != cudaSuccess) return cuda_fail(e, "dkv zeroing");
  smla::BwdArgs a{q, kv, dout, lse, delta, indices, dq, dkv_f32, T, H, topk, scale};
  if (dkv_mode == SMLA_DKV_ATOMIC) {
    e = launch_bwd_any(a, s);
    if (e != cudaSuccess) return cuda_fail(e, "sparse_mla_bwd launch");
    count_launches(1);
  } else {
    // index-sorted segmented reduction: slot lists per kv row, then chunks of
    // tokens whose per-slot contributions are added to their rows in slot order
    uint8_t* w = static_cast<uint8_t*>(workspace);
    int* offset = reinterpret_cast<int*>(w + L.offset);
    int* pos = reinterpret_cast<int*>(w + L.pos);
    int* seg = reinterpret_cast<int*>(w + L.seg);
    float* gbuf = reinterpret_cast<float*>(w + L.g);
    int nl = 0;
    e = smla::launch_build_row_lists(indices, T, topk, offset, reinterpret_cast<int*>(w + L.cursor), pos, seg,
                                     reinterpret_cast<int*>(w + L.sums), s, &nl);
    if (e != cudaSuccess) return cuda_fail(e, "slot list launch");
    count_launches(nl);
    size_t tc = (workspace_bytes - L.g) / L.per_token;
    if (tc > (size_t)T) tc = (size_t)T;
    a.gbuf = gbuf;
    a.gstride = (int64_t)tc * topk * smla::kDqk;
    for (int t0 = 0; t0 < T; t0 += (int)tc) {
      a.t0 = t0;
      a.nt = (int)((size_t)(T - t0) < tc ? (size_t)(T - t0) : tc);
      e = launch_bwd_any(a, s);
      if (e != cudaSuccess) return cuda_fail(e, "sparse_mla_bwd launch");
      e = smla::launch_reduce_rows(offset, seg, pos, gbuf, L.ng, a.gstride, (int64_t)t0 * topk,
                                   (int64_t)(t0 + a.nt) * topk, T, dkv_f32, s);
      if (e != cudaSuccess) return cuda_fail(e, "dkv reduction launch");
      count_launches(2);
    }
  }
  if (dkv != nullptr) {
    e = smla::launch_cast_bf16(dkv_f32, dkv, (int64_t)T * smla::kDqk, s);
    if (e != cudaSuccess) return cuda_fail(e, "dkv cast launch");
    count_launches(1);
  }
  return 0;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Backward entry point that allocates nothing.
//
// Some callers cannot call cudaMalloc at all: code that runs inside a memory
// allocator's own callbacks (allocating there would re-enter the allocator),
// and services whose device memory is fixed at start-up (they must not grow
// or fragment it while serving).  sparse_mla_bwd needs its caller to hand it a
// workspace for Delta; this variant keeps Delta in a fixed file-scope device
// array instead, so the caller passes only inputs and outputs.
namespace {

// counter of sparse_mla_check_indices (one word per device) and the host lock
// that serialises its users
__device__ unsigned long long g_check_counter;
std::mutex g_check_mu;

constexpr size_t kNoAllocMaxRows = size_t(1) << 23;   // T * H <= 8,388,608 values (32 MiB of fp32)
__device__ __align__(256) float g_noalloc_delta[kNoAllocMaxRows];

// In host code g_noalloc_delta names a host-side stand-in, not the device
// array, so its device address is looked up with the caller's device current.
// The lookup is made on every call (it is a cheap runtime query), so the
// address is always the one of the current device and context.
int noalloc_scratch(float** out) {
  void* p = nullptr;
  cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_delta);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(no-allocation scratch)");
  *out = static_cast<float*>(p);
  return 0;
}

}  // namespace

extern "C" {

int sparse_mla_bwd_noalloc(const smla_bf16_t* q, const smla_bf16_t* kv, const smla_bf16_t* out,
                           const smla_bf16_t* dout, const float* lse, const int32_t* indices,
                           const int32_t* cu_seqlens, int T, int H, int topk, int B, float scale,
                           smla_bf16_t* dq, float* dkv_f32, smla_bf16_t* dkv, void* stream) {
  (void)cu_seqlens;
  (void)B;
  g_last_error.clear();
  if (int r = check_shape(T, H, topk, scale)) return r;
  if ((size_t)T * (size_t)H > kNoAllocMaxRows)
    return fail(-EINVAL, "T*H = %lld exceeds the no-allocation scratch limit of %zu (T*H values)",
                (long long)T * H, kNoAllocMaxRows);
  if (T == 0) return 0;
  SMLA_REQUIRE_PTR(q);
  SMLA_REQUIRE_PTR(kv);
  SMLA_REQUIRE_PTR(out);
  SMLA_REQUIRE_PTR(dout);
  SMLA_REQUIRE_PTR(lse);
  SMLA_REQUIRE_PTR(indices);
  SMLA_REQUIRE_PTR(dq);
  SMLA_REQUIRE_PTR(dkv_f32);
  if (dkv != nullptr && !aligned16(dkv)) return fail(-EINVAL, "dkv must be 16-byte aligned");
  if (int r = check_device()) return r;
  float* delta = nullptr;
  if (int r = noalloc_scratch(&delta)) return r;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // Delta is fully rewritten here before the backward kernel reads it.
  cudaError_t e = smla::launch_delta(out, dout, delta, (int64_t)T * H, s);
  if (e != cudaSuccess) return cuda_fail(e, "delta launch");
  count_launches(1);
  e = cudaMemsetAsync(dkv_f32, 0, (size_t)T * smla::kDqk * sizeof(float), s);
  if (e != cudaSuccess) return cuda_fail(e, "dkv zeroing");
  smla::BwdArgs a{q, kv, dout, lse, delta, indices, dq, dkv_f32, T, H, topk, scale};
  e = launch_bwd_any(a, s);
  if (e != cudaSuccess) return cuda_fail(e, "sparse_mla_bwd_noalloc launch");
  count_launches(1);
  if (dkv != nullptr) {
    e = smla::launch_cast_bf16(dkv_f32, dkv, (int64_t)T * smla::kDqk, s);
    if (e != cudaSuccess) return cuda_fail(e, "dkv cast launch");
    count_launches(1);
  }
  return 0;
}

int sparse_mla_check_indices(const int32_t* indices, int T, int topk, const int32_t* cu_seqlens,
                             int B, int64_t* n_bad, void* stream) {
  g_last_error.clear();
  if (n_bad == nullptr) return fail(-EINVAL, "n_bad must not be NULL");
  *n_bad = 0;
  if (T < 0) return fail(-EINVAL, "T must be >= 0 (got %d)", T);
  if (topk <= 0) return fail(-EINVAL, "topk must be positive (got %d)", topk);
  if (B < 1) return fail(-EINVAL, "B must be >= 1 (got %d)", B);
  if (T == 0) return 0;
  SMLA_REQUIRE_PTR(indices);
  if (cu_seqlens == nullptr) return fail(-EINVAL, "cu_seqlens must not be NULL");
  if (int r = check_device()) return r;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // the count goes to a counter word inside the library (one per device); the
  // call holds a host lock from zeroing it to reading it back, so concurrent
  // calls from other host threads wait instead of sharing it
  std::lock_guard<std::mutex> lock(g_check_mu);
  void* cp = nullptr;
  cudaError_t e = cudaGetSymbolAddress(&cp, g_check_counter);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(index-check counter)");
  unsigned long long* counter = static_cast<unsigned long long*>(cp);
  unsigned long long host = 0;
  e = cudaMemsetAsync(counter, 0, sizeof(*counter), s);
  if (e == cudaSuccess) {
    e = smla::launch_check_indices(indices, T, topk, cu_seqlens, B, counter, s);
    if (e == cudaSuccess) count_launches(1);
  }
  if (e == cudaSuccess) e = cudaMemcpyAsync(&host, counter, sizeof(host), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "sparse_mla_check_indices");
  *n_bad = (int64_t)host;
  return 0;
}

}  // extern "C"
