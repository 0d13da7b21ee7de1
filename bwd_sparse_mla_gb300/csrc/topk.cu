// Top-k index selection feeding sparse MLA (Megatron-Bridge PR #17, "GLM-5 DSA
// option: tilelang (2/2)", Summary and Bug fixes): for each query row t of a
// packed sequence starting at row s0, the candidates are the causal keys
// s0 .. t scored by scores[t, 0 .. t - s0]; the k = min(topk, t - s0 + 1,
// ncols) best are written as packed kv rows s0 + c in descending score order
// (equal scores by ascending column, NaN last), and the rest of the fixed-width
// row is padded with -1.
//
// One CTA per row: the row's scores are mapped to order-preserving 32-bit keys
// in shared memory; a 4-pass radix select (8 bits per pass, the first fused
// with the load, the bin chosen by a warp-parallel suffix scan) finds the k-th
// largest key thr (stopping early once the boundary bin is taken whole).
// When every key >= thr fits in the selection buffer they
// are collected in one pass in any order; otherwise (many ties at thr) an
// ordered pass collects the keys above thr and the first columns equal to it.
// A bitonic network unrolled at compile time, held in registers (shuffles
// within a warp, shared memory across warps), sorts the (key, column) pairs.
#include "smla_common.cuh"

namespace smla {
namespace {

constexpr int kTkThreads = 1024;
constexpr int kTkCuCache = 1024;          // sequences whose starts are kept in shared memory

// larger float -> larger key; -0 and +0 equal; NaN below everything
__device__ __forceinline__ uint32_t order_key(float f) {
  uint32_t u = __float_as_uint(f);
  if ((u & 0x7fffffffu) > 0x7f800000u) return 0u;   // NaN
  if (u == 0x80000000u) u = 0u;                      // -0 -> +0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// One step (K, J) of a descending bitonic network over kTkThreads * EPT
// elements held in registers, thread tid owning elements tid * EPT + m.  The
// partner of element i is i ^ J: for J < EPT it is in the same thread, for
// J < 32 * EPT in another lane of the same warp (shuffle), otherwise in
// another warp (exchanged through shared memory a, 16-byte aligned).  In a
// descending run (bit K of i clear) the lower index keeps the larger element.
template <int EPT, int K, int J>
__device__ __forceinline__ void bitonic_step(unsigned long long (&x)[EPT], unsigned long long* a, int tid) {
  constexpr int TJ = J / EPT;             // partner thread distance
  const int base = tid * EPT;
  if constexpr (J < EPT) {
#pragma unroll
    for (int m = 0; m < EPT; ++m) {
      if ((m & J) == 0) {
        const int mp = m | J;
        const bool desc = ((base + m) & K) == 0;
        const unsigned long long lo = x[m], hi = x[mp];
        const bool swap = (lo < hi) == desc;
        x[m] = swap ? hi : lo;
        x[mp] = swap ? lo : hi;
      }
    }
  } else {
    const bool keep_max = ((base & K) == 0) == ((base & J) == 0);
    if constexpr (TJ >= 32) {
      unsigned long long y[EPT];
      const int pb = (tid ^ TJ) * EPT;
      if constexpr (EPT == 1) {
        a[base] = x[0];
        __syncthreads();
        y[0] = a[pb];
      } else {
#pragma unroll
        for (int m = 0; m < EPT; m += 2)
          *reinterpret_cast<ulonglong2*>(a + base + m) = make_ulonglong2(x[m], x[m + 1]);
        __syncthreads();
#pragma unroll
        for (int m = 0; m < EPT; m += 2) {
          const ulonglong2 v = *reinterpret_cast<const ulonglong2*>(a + pb + m);
          y[m] = v.x;
          y[m + 1] = v.y;
        }
      }
      __syncthreads();
#pragma unroll
      for (int m = 0; m < EPT; ++m) x[m] = ((x[m] > y[m]) == keep_max) ? x[m] : y[m];
    } else {
#pragma unroll
      for (int m = 0; m < EPT; ++m) {
        const unsigned long long y = __shfl_xor_sync(0xffffffffu, x[m], TJ);
        x[m] = ((x[m] > y) == keep_max) ? x[m] : y;
      }
    }
  }
}

// every step of the network for runs K = 2 .. N, J = K/2 .. 1, unrolled at compile time
template <int EPT, int N, int K, int J>
__device__ __forceinline__ void bitonic_steps(unsigned long long (&x)[EPT], unsigned long long* a, int tid) {
  if constexpr (K <= N) {
    if constexpr (J == 0) {
      bitonic_steps<EPT, N, 2 * K, K>(x, a, tid);
    } else {
      bitonic_step<EPT, K, J>(x, a, tid);
      bitonic_steps<EPT, N, K, J / 2>(x, a, tid);
    }
  }
}

// descending sort of a[0, kTkThreads * EPT) in place
template <int EPT>
__device__ void sort_desc(unsigned long long* a) {
  const int tid = threadIdx.x;
  unsigned long long x[EPT];
#pragma unroll
  for (int m = 0; m < EPT; ++m) x[m] = a[tid * EPT + m];
  __syncthreads();
  bitonic_steps<EPT, kTkThreads * EPT, 2, 1>(x, a, tid);
#pragma unroll
  for (int m = 0; m < EPT; ++m) a[tid * EPT + m] = x[m];
  __syncthreads();
}

__device__ __forceinline__ unsigned long long sel_entry(uint32_t key, int c) {
  return ((unsigned long long)key << 32) | (unsigned long long)(0xffffffffu - (uint32_t)c);
}

__global__ void __launch_bounds__(kTkThreads) topk_kernel(const float* __restrict__ scores, int64_t ld, int ncols,
                                                          const int32_t* __restrict__ cu, int B, int T, int topk,
                                                          int kpow2, int32_t* __restrict__ out) {
  extern __shared__ __align__(16) uint8_t sm[];
  unsigned long long* sel = reinterpret_cast<unsigned long long*>(sm);   // kpow2 selected (key, column)
  uint32_t* keys_base = reinterpret_cast<uint32_t*>(sel + kpow2);        // ncols + 3 keys
  __shared__ int hist[2][256];           // radix histograms, alternating between passes
  __shared__ int cu_s[kTkCuCache + 1];
  __shared__ int warp_cnt[32];
  __shared__ int info[5];                 // s0, chosen bin, remaining, chunk total, keys equal to the bin
  __shared__ int n_sel, n_eq;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const unsigned lt_mask = (1u << lane) - 1u;
  const int32_t* cus = cu;
  if (B <= kTkCuCache) {
    for (int i = tid; i <= B; i += kTkThreads) cu_s[i] = cu[i];
    cus = cu_s;
  }
  __syncthreads();

  for (int t = blockIdx.x; t < T; t += gridDim.x) {
    if (tid == 0) {                       // start of t's sequence: largest b with cu[b] <= t
      int lo = 0, hi = B;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (cus[mid] <= t) lo = mid; else hi = mid - 1;
      }
      info[0] = cus[lo];
      n_sel = 0;
      n_eq = 0;
    }
    if (tid < 256) hist[0][tid] = 0;
    __syncthreads();
    const int s0 = info[0];
    const int n = min(t - s0 + 1, ncols);
    const int k = min(topk, n);
    const float* row = scores + (int64_t)t * ld;
    // keys, with the histogram of their top byte (the first radix pass).
    // Columns [0, head) and the tail are read singly, the rest as aligned
    // float4; keys is offset so that keys + head is 16-byte aligned too.
    const int head = min((int)(((16u - ((uint32_t)(uintptr_t)row & 15u)) & 15u) >> 2), n);
    const int nv = (n - head) >> 2;
    uint32_t* keys = keys_base + ((4 - head) & 3);
#pragma unroll 2
    for (int q = tid; q < nv; q += kTkThreads) {
      const float4 v = __ldg(reinterpret_cast<const float4*>(row + head) + q);
      const uint4 kk = make_uint4(order_key(v.x), order_key(v.y), order_key(v.z), order_key(v.w));
      reinterpret_cast<uint4*>(keys + head)[q] = kk;
      atomicAdd(&hist[0][kk.x >> 24], 1);
      atomicAdd(&hist[0][kk.y >> 24], 1);
      atomicAdd(&hist[0][kk.z >> 24], 1);
      atomicAdd(&hist[0][kk.w >> 24], 1);
    }
    {
      const int rest = n - head - 4 * nv;           // at most 3 at the tail
      const int c = tid < head ? tid : head + 4 * nv + (tid - head);
      if (tid < head + rest) {
        const uint32_t kk = order_key(row[c]);
        keys[c] = kk;
        atomicAdd(&hist[0][kk >> 24], 1);
      }
    }
    for (int i = tid; i < kpow2; i += kTkThreads) sel[i] = 0ull;   // padding sorts last
    if (tid < 256) hist[1][tid] = 0;
    __syncthreads();

    // radix select: thr = the k-th largest key; `remaining` keys equal to thr
    // are taken, of eq_total such keys
    uint32_t prefix = 0u, mask = 0u;
    int remaining = k, eq_total = 0;
    for (int p = 0; p < 4; ++p) {
      const int shift = 24 - 8 * p;
      if (p > 0) {
#pragma unroll 4
        for (int c = tid; c < n; c += kTkThreads) {
          const uint32_t kk = keys[c];
          if ((kk & mask) == prefix) atomicAdd(&hist[p & 1][(kk >> shift) & 255u], 1);
        }
        if (tid < 256) hist[(p + 1) & 1][tid] = 0;   // last read by the selection two passes back
        __syncthreads();
      }
      if (warp == 0) {
        // the largest bin b with count(bins >= b) >= remaining; lane L holds bins 8L .. 8L+7
        int cnt[8], sum = 0;
#pragma unroll
        for (int e = 0; e < 8; ++e) { cnt[e] = hist[p & 1][8 * lane + e]; sum += cnt[e]; }
        // exclusive suffix sum of the lane sums (the counts of the bins of higher lanes)
        int incl = sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int y = __shfl_down_sync(0xffffffffu, incl, o);
          if (lane + o < 32) incl += y;
        }
        const int above = incl - sum;
        const bool has = above + sum >= remaining;        // this lane's lowest bin qualifies
        const unsigned qual = __ballot_sync(0xffffffffu, has);
        const int top = 31 - __clz(qual);                 // highest qualifying lane holds b
        if (lane == top) {
          int cum = above, e_sel = 0, found = 0;
#pragma unroll
          for (int e = 7; e > 0; --e) {
            if (!found && cum + cnt[e] >= remaining) { e_sel = e; found = 1; }
            if (!found) cum += cnt[e];
          }
          int c_sel = cnt[0];
#pragma unroll
          for (int e = 1; e < 8; ++e) if (e == e_sel) c_sel = cnt[e];
          info[1] = 8 * lane + e_sel;
          info[2] = remaining - cum;
          info[4] = c_sel;
        }
      }
      __syncthreads();
      prefix |= (uint32_t)info[1] << shift;
      mask |= 0xffu << shift;
      remaining = info[2];
      eq_total = info[4];
      // the chosen bin is taken whole: the keys >= prefix (lower bits zero)
      // are exactly the k wanted
      if (remaining == eq_total) break;
    }
    const uint32_t thr = prefix;

    int nsort;
    if (k - remaining + eq_total <= kpow2) {
      // every key >= thr fits: collect them in any order; sorting by (key,
      // column) then puts the k wanted first
      nsort = k - remaining + eq_total;
      for (int base = 0; base < n; base += 4 * kTkThreads) {
        uint32_t kk[4];
        unsigned ball[4];
        int cnt = 0;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int c = base + u * kTkThreads + tid;
          kk[u] = c < n ? keys[c] : 0u;
          ball[u] = __ballot_sync(0xffffffffu, c < n && kk[u] >= thr);
          cnt += __popc(ball[u]);
        }
        int pos = 0;
        if (lane == 0 && cnt) pos = atomicAdd(&n_sel, cnt);
        pos = __shfl_sync(0xffffffffu, pos, 0);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          if ((ball[u] >> lane) & 1u) sel[pos + __popc(ball[u] & lt_mask)] = sel_entry(kk[u], base + u * kTkThreads + tid);
          pos += __popc(ball[u]);
        }
      }
      __syncthreads();
    } else {
      // many keys tie at thr: collect, in column order, every key above thr and
      // the first `remaining` equal to it
      nsort = k;
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
        if (gt || (eq && eq_rank < remaining)) sel[atomicAdd(&n_sel, 1)] = sel_entry(kk, c);
        __syncthreads();
        if (tid == 0) n_eq += info[3];
        __syncthreads();
      }
    }

    // descending (key, then ascending column) over 1024 entries or the next
    // power of two above nsort (zero padding sorts last); write the row, -1 past k
    if (nsort <= kTkThreads) sort_desc<1>(sel);
    else if (nsort <= 2 * kTkThreads) sort_desc<2>(sel);
    else if (nsort <= 4 * kTkThreads) sort_desc<4>(sel);
    else sort_desc<8>(sel);
    int32_t* o = out + (int64_t)t * topk;
    for (int i = tid; i < topk; i += kTkThreads)
      o[i] = i < k ? s0 + (int32_t)(0xffffffffu - (uint32_t)(sel[i] & 0xffffffffull)) : -1;
    __syncthreads();
  }
}

}  // namespace

// the selection buffer holds max(next power of two above topk, 1024) pairs;
// the keys (ncols, shifted by up to 3 for alignment) follow it
int topk_sel_entries(int topk) {
  int kp = kTkThreads;
  while (kp < topk) kp <<= 1;
  return kp;
}

size_t topk_smem_bytes(int ncols, int topk) {
  return (size_t)topk_sel_entries(topk) * 8 + (((size_t)ncols + 3) * 4 + 15) / 16 * 16;
}

cudaError_t launch_topk(const float* scores, int64_t ld, int ncols, const int32_t* cu, int B, int T, int topk,
                        int32_t* out, int num_sms, cudaStream_t s) {
  if (topk > 8 * kTkThreads) return cudaErrorInvalidValue;   // the register sort holds 8 pairs a thread
  const int kp = topk_sel_entries(topk);
  const size_t sm = topk_smem_bytes(ncols, topk);
  cudaError_t e = cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
  if (e != cudaSuccess) return e;
  const int grid = T < num_sms ? T : num_sms;
  if (grid == 0) return cudaSuccess;
  topk_kernel<<<grid, kTkThreads, sm, s>>>(scores, ld, ncols, cu, B, T, topk, kp, out);
  return cudaGetLastError();
}

}  // namespace smla
