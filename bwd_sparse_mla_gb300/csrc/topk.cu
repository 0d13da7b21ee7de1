// Top-k index selection feeding sparse MLA (Megatron-Bridge PR #17, "GLM-5 DSA
// option: tilelang (2/2)", Summary and Bug fixes): for each query row t of a
// packed sequence starting at row s0, the candidates are the causal keys
// s0 .. t scored by scores[t, 0 .. t - s0]; the k = min(topk, t - s0 + 1,
// ncols) best are written as packed kv rows s0 + c in descending score order
// (equal scores by ascending column, NaN last), and the rest of the fixed-width
// row is padded with -1.
//
// One CTA per row: the row's scores are mapped to order-preserving 32-bit keys
// in shared memory; a 4-pass radix select (8 bits per pass) finds the k-th
// largest key; an ordered pass collects every key above it and the first
// columns equal to it; a bitonic sort orders the selected (key, column) pairs.
#include "smla_common.cuh"

namespace smla {
namespace {

constexpr int kTkThreads = 1024;

// larger float -> larger key; -0 and +0 equal; NaN below everything
__device__ __forceinline__ uint32_t order_key(float f) {
  uint32_t u = __float_as_uint(f);
  if ((u & 0x7fffffffu) > 0x7f800000u) return 0u;   // NaN
  if (u == 0x80000000u) u = 0u;                      // -0 -> +0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// descending bitonic sort of a[0, n2) (n2 a power of two) in shared memory
__device__ void sort_desc(unsigned long long* a, int n2) {
  for (int k = 2; k <= n2; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int i = threadIdx.x; i < n2; i += blockDim.x) {
        const int p = i ^ j;
        if (p > i) {
          const bool desc = (i & k) == 0;            // this k-block sorts descending
          const unsigned long long x = a[i], y = a[p];
          if (desc ? (x < y) : (x > y)) { a[i] = y; a[p] = x; }
        }
      }
      __syncthreads();
    }
  }
}

__global__ void __launch_bounds__(kTkThreads) topk_kernel(const float* __restrict__ scores, int64_t ld, int ncols,
                                                          const int32_t* __restrict__ cu, int B, int T, int topk,
                                                          int kpow2, int32_t* __restrict__ out) {
  extern __shared__ __align__(16) uint8_t sm[];
  unsigned long long* sel = reinterpret_cast<unsigned long long*>(sm);   // kpow2 selected (key, column)
  uint32_t* keys = reinterpret_cast<uint32_t*>(sel + kpow2);             // ncols keys
  __shared__ int hist[256];
  __shared__ int warp_cnt[32];
  __shared__ int info[4];                 // s0, chosen bin, remaining, chunk total
  __shared__ int n_sel, n_eq;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  for (int t = blockIdx.x; t < T; t += gridDim.x) {
    if (tid == 0) {                       // start of t's sequence: largest b with cu[b] <= t
      int lo = 0, hi = B;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (cu[mid] <= t) lo = mid; else hi = mid - 1;
      }
      info[0] = cu[lo];
      n_sel = 0;
      n_eq = 0;
    }
    __syncthreads();
    const int s0 = info[0];
    const int n = min(t - s0 + 1, ncols);
    const int k = min(topk, n);
    const float* row = scores + (int64_t)t * ld;
    for (int c = tid; c < n; c += kTkThreads) keys[c] = order_key(row[c]);
    for (int i = tid; i < kpow2; i += kTkThreads) sel[i] = 0ull;   // padding sorts last
    __syncthreads();

    // radix select: thr = the k-th largest key; `remaining` keys equal to thr are taken
    uint32_t prefix = 0u, mask = 0u;
    int remaining = k;
    for (int shift = 24; shift >= 0 && k > 0; shift -= 8) {
      for (int i = tid; i < 256; i += kTkThreads) hist[i] = 0;
      __syncthreads();
      for (int c = tid; c < n; c += kTkThreads) {
        const uint32_t kk = keys[c];
        if ((kk & mask) == prefix) atomicAdd(&hist[(kk >> shift) & 255u], 1);
      }
      __syncthreads();
      if (tid == 0) {
        int cum = 0, b = 255;
        for (; b > 0; --b) {
          if (cum + hist[b] >= remaining) break;
          cum += hist[b];
        }
        info[1] = b;
        info[2] = remaining - cum;
      }
      __syncthreads();
      prefix |= (uint32_t)info[1] << shift;
      mask |= 0xffu << shift;
      remaining = info[2];
      __syncthreads();
    }
    const uint32_t thr = prefix;

    // collect, in column order: every key above thr, and the first `remaining` equal to it
    const unsigned lt_mask = (1u << lane) - 1u;
    for (int base = 0; base < n && k > 0; base += kTkThreads) {
      const int c = base + tid;
      const uint32_t kk = c < n ? keys[c] : 0u;
      const bool gt = c < n && kk > thr;
      const bool eq = c < n && kk == thr;
      const unsigned ball = __ballot_sync(0xffffffffu, eq);
      if (lane == 0) warp_cnt[warp] = __popc(ball);
      __syncthreads();
      if (warp == 0) {
        const int v = warp_cnt[lane];
        int incl = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int y = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += y;
        }
        warp_cnt[lane] = incl - v;
        if (lane == 31) info[3] = incl;
      }
      __syncthreads();
      const int eq_rank = n_eq + warp_cnt[warp] + __popc(ball & lt_mask);
      if (gt || (eq && eq_rank < remaining)) {
        const int pos = atomicAdd(&n_sel, 1);
        sel[pos] = ((unsigned long long)kk << 32) | (unsigned long long)(0xffffffffu - (uint32_t)c);
      }
      __syncthreads();
      if (tid == 0) n_eq += info[3];
      __syncthreads();
    }

    // descending (key, then ascending column); write the row, -1 past k
    sort_desc(sel, kpow2);
    int32_t* o = out + (int64_t)t * topk;
    for (int i = tid; i < topk; i += kTkThreads)
      o[i] = i < k ? s0 + (int32_t)(0xffffffffu - (uint32_t)(sel[i] & 0xffffffffull)) : -1;
    __syncthreads();
  }
}

}  // namespace

size_t topk_smem_bytes(int ncols, int topk) {
  int kp = 1;
  while (kp < topk) kp <<= 1;
  return (size_t)kp * 8 + (size_t)ncols * 4;
}

cudaError_t launch_topk(const float* scores, int64_t ld, int ncols, const int32_t* cu, int B, int T, int topk,
                        int32_t* out, int num_sms, cudaStream_t s) {
  int kp = 1;
  while (kp < topk) kp <<= 1;
  const size_t sm = topk_smem_bytes(ncols, topk);
  cudaError_t e = cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
  if (e != cudaSuccess) return e;
  const int grid = T < num_sms ? T : num_sms;
  if (grid == 0) return cudaSuccess;
  topk_kernel<<<grid, kTkThreads, sm, s>>>(scores, ld, ncols, cu, B, T, topk, kp, out);
  return cudaGetLastError();
}

}  // namespace smla
