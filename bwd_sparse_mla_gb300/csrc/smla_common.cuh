// Shared device helpers and launch-argument structs of the sparse MLA library.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace smla {

constexpr int kDqk = 576;    // 512 latent + 64 rope tail
constexpr int kDv = 512;     // latent = value width
constexpr int kDtail = 64;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
// ln(1e-30): the LSE of a row with no valid slot (empty max read as 0,
// sum of exponentials floored at 1e-30).
constexpr float kLseEmpty = -69.07755278982137f;
constexpr float kSumexpFloor = 1e-30f;
// Largest top-k the H = 128 tensor-core kernels take (their lists of non-empty
// blocks live in shared memory); larger top-k runs the CUDA-core kernels.
constexpr int kTcMaxTopk = 16384;

struct FwdArgs {
  const uint16_t* q;        // [T, H, 576] bf16
  const uint16_t* kv;       // [T, 576] bf16
  const int32_t* indices;   // [T, topk]
  uint16_t* out;            // [T, H, 512] bf16
  float* lse;               // [T, H]
  int T, H, topk;
  float scale;
  // query rows [t0, t0 + nt) of this launch (nt < 0: all T rows)
  int t0 = 0, nt = -1;
  uint32_t* status = nullptr;   // device status word (debug-build bounds checks)
};

struct BwdArgs {
  const uint16_t* q;
  const uint16_t* kv;
  const uint16_t* dout;     // [T, H, 512] bf16
  const float* lse;         // [T, H]
  const float* delta;       // [T, H] (workspace, filled by the Delta pass)
  const int32_t* indices;
  uint16_t* dq;             // [T, H, 576] bf16
  float* dkv32;             // [T, 576] fp32 accumulator (zeroed before)
  int T, H, topk;
  float scale;
  // token range [t0, t0 + nt) of this launch (nt < 0: all T tokens)
  int t0 = 0, nt = -1;
  // deterministic dKV: when gbuf != nullptr the kernels store each valid slot's
  // contribution at gbuf + g * gstride + ((t - t0) * topk + j) * 576 (head group g)
  // instead of adding it into dkv32
  float* gbuf = nullptr;
  int64_t gstride = 0;
  int64_t gbuf_floats = 0;      // extent of gbuf (debug-build bounds checks)
  uint32_t* status = nullptr;   // device status word (debug-build bounds checks)
};

__device__ __forceinline__ float bf16_lo(uint32_t x) { return __uint_as_float(x << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t x) { return __uint_as_float(x & 0xffff0000u); }

// Two fp32 values -> one word of two bf16 (lo in the low half), round to nearest
// even: one cvt instruction (its first source fills the high half).
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// Pairs of fp32 in one 64-bit register ({lo, hi}) and the paired fp32 arithmetic
// of sm_100+: one instruction for two lanes of work, each rounded as the scalar op.
__device__ __forceinline__ uint64_t f32x2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f32x2_split(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t fma_f32x2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t mul_f32x2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t add_f32x2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t sub_f32x2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// ----------------------------------------------------------------- debug bounds checks
// Device status word code of a failed bounds check (the word also carries the
// bounded waits' timeout code 1; see sparse_mla_device_status).
constexpr uint32_t kErrBounds = 2u;
// The device status word (lives in tc_fwd.cu).
uint32_t* tc_status_ptr();

// Debug build (-DSMLA_DEBUG): every gathered 16-byte source and every scatter
// destination (and the row reads of the deterministic reduction) is checked against
// its buffer [lo, lo + n) before the access.  A failed check records kErrBounds in
// the status word (first error wins) and the access is skipped: a gather copies zero
// bytes from the buffer's start, a scatter or read is not issued.  Nothing traps.
// In other builds the checks compile to nothing.
template <typename T>
__device__ __forceinline__ void check_src(const T*& src, uint32_t& bytes, const T* lo, int64_t n, uint32_t* status) {
#ifdef SMLA_DEBUG
  if (src < lo || src + 16 / sizeof(T) > lo + n) {
    if (status != nullptr) atomicCAS(status, 0u, kErrBounds);
    src = lo;
    bytes = 0u;
  }
#else
  (void)src; (void)bytes; (void)lo; (void)n; (void)status;
#endif
}
template <typename T>
__device__ __forceinline__ bool check_range(const T* ptr, int count, const T* lo, int64_t n, uint32_t* status) {
#ifdef SMLA_DEBUG
  if (ptr < lo || ptr + count > lo + n) {
    if (status != nullptr) atomicCAS(status, 0u, kErrBounds);
    return false;
  }
#else
  (void)ptr; (void)count; (void)lo; (void)n; (void)status;
#endif
  return true;
}

// 16-byte vector fp32 reduction into global memory (sm_90+).
__device__ __forceinline__ void red_add_v4(float* addr, float a, float b, float c, float d) {
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(addr), "f"(a), "f"(b), "f"(c),
               "f"(d)
               : "memory");
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Host-side launchers implemented in the kernel translation units.
cudaError_t launch_fwd_simt(const FwdArgs& a, cudaStream_t s);
cudaError_t launch_bwd_simt(const BwdArgs& a, cudaStream_t s);
cudaError_t launch_delta(const uint16_t* out, const uint16_t* dout, float* delta, int64_t rows,
                         cudaStream_t s);
cudaError_t launch_cast_bf16(const float* src, uint16_t* dst, int64_t n, cudaStream_t s);
cudaError_t launch_fwd_tc(const FwdArgs& a, cudaStream_t s);   // H == 128
cudaError_t launch_fwd_tc_small(const FwdArgs& a, cudaStream_t s);   // H <= 16 (tc_fwd_small.cu)
cudaError_t launch_bwd_tc(const BwdArgs& a, cudaStream_t s);   // H == 128
cudaError_t launch_bwd_tc_small(const BwdArgs& a, cudaStream_t s);   // H <= 16 (tc_bwd_small.cu)
cudaError_t read_tc_status(uint32_t* out, bool clear);
cudaError_t launch_wait_selftest(cudaStream_t s);
cudaError_t launch_bounds_selftest(cudaStream_t s);
// deterministic dKV (dkv_det.cu)
int64_t det_scan_tiles(int T);
cudaError_t launch_build_row_lists(const int32_t* indices, int T, int topk, int* offset, int* cursor, int* pos,
                                   int* seg, int* scan_sums, cudaStream_t s, int* nlaunch);
cudaError_t launch_reduce_rows(const int* offset, const int* seg, int* pos, const float* gbuf, int ng,
                               int64_t gstride, int64_t slot_lo, int64_t slot_hi, int T, float* dkv32,
                               cudaStream_t s);
int simt_head_groups(int H);   // CUDA-core backward: CTAs (head groups) per token
// top-k index selection (topk.cu)
size_t topk_smem_bytes(int ncols, int topk);
cudaError_t launch_topk(const float* scores, int64_t ld, int ncols, const int32_t* cu, int B, int T, int topk,
                        int32_t* out, int num_sms, cudaStream_t s);
cudaError_t launch_check_indices(const int32_t* indices, int T, int topk, const int32_t* cu_seqlens,
                                 int B, unsigned long long* counter, cudaStream_t s);

}  // namespace smla
