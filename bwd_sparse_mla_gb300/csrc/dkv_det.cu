// Deterministic dKV: an index-sorted segmented reduction.
//
// The backward kernels, run over chunks of query tokens, store each valid
// slot's dKV contribution G[t, j, 0:576] (fp32) instead of adding it into the
// row it names.  Before that, the slots are sorted by the row they name: for
// every kv row r the list of flat slot ids s = t * topk + j with
// indices[t, j] = r, in ascending order (a CSR transpose of the index tensor).
// After each chunk, one warp per row adds that chunk's contributions to the
// row in slot order.  dkv[r] is therefore the fp32 left fold, in ascending slot
// order, of the row's contributions: the same bits on every run, whatever the
// scheduling, the chunk size or the number of SMs.  (The miles PR #2079
// summary names the atomic dKV accumulation of `sparse_mla_bwd_kernel` as a
// cost and risk; this is the order-fixed alternative.)
#include "smla_common.cuh"

namespace smla {
namespace {

constexpr int kScanThreads = 1024;
constexpr int kScanItems = 4;                       // elements per thread per scan block
constexpr int kScanTile = kScanThreads * kScanItems;
constexpr int kSortThreads = 512;
constexpr int kSortCap = 16384;                     // segment length sorted in shared memory (64 KiB)

__device__ __forceinline__ bool valid_row(int r, int T) { return r >= 0 && r < T; }

// count[r] += number of valid slots naming row r
__global__ void __launch_bounds__(256) count_rows_kernel(const int32_t* __restrict__ idx, int64_t nslots, int T,
                                                         int* __restrict__ count) {
  for (int64_t s = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; s < nslots; s += (int64_t)gridDim.x * blockDim.x) {
    const int r = idx[s];
    if (valid_row(r, T)) atomicAdd(count + r, 1);
  }
}

// block-wide exclusive scan of kScanTile ints; returns the tile total
__device__ int scan_tile(int* v, int* warp_sums) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int run = 0;
#pragma unroll
  for (int k = 0; k < kScanItems; ++k) {
    const int x = v[k];
    v[k] = run;
    run += x;
  }
  int incl = run;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) warp_sums[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = warp_sums[lane];
    int wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += y;
    }
    warp_sums[lane] = wi - w;        // exclusive
    if (lane == 31) warp_sums[32] = wi;
  }
  __syncthreads();
  const int base = warp_sums[warp] + incl - run;
#pragma unroll
  for (int k = 0; k < kScanItems; ++k) v[k] += base;
  const int total = warp_sums[32];
  __syncthreads();
  return total;
}

// pass 1: exclusive scan inside each tile of count -> offset, tile totals -> sums
__global__ void __launch_bounds__(kScanThreads) scan_tiles_kernel(const int* __restrict__ count, int n,
                                                                  int* __restrict__ offset, int* __restrict__ sums) {
  __shared__ int warp_sums[33];
  const int64_t base = (int64_t)blockIdx.x * kScanTile + threadIdx.x * kScanItems;
  int v[kScanItems];
#pragma unroll
  for (int k = 0; k < kScanItems; ++k) v[k] = (base + k < n) ? count[base + k] : 0;
  const int total = scan_tile(v, warp_sums);
#pragma unroll
  for (int k = 0; k < kScanItems; ++k)
    if (base + k < n) offset[base + k] = v[k];
  if (threadIdx.x == 0) sums[blockIdx.x] = total;
}

// pass 2 (one block): exclusive scan of the tile totals, in chunks of kScanTile
__global__ void __launch_bounds__(kScanThreads) scan_sums_kernel(int* __restrict__ sums, int ntiles,
                                                                 int* __restrict__ offset, int n) {
  __shared__ int warp_sums[33];
  int carry = 0;
  for (int c0 = 0; c0 < ntiles; c0 += kScanTile) {
    const int base = c0 + threadIdx.x * kScanItems;
    int v[kScanItems];
#pragma unroll
    for (int k = 0; k < kScanItems; ++k) v[k] = (base + k < ntiles) ? sums[base + k] : 0;
    const int total = scan_tile(v, warp_sums);
#pragma unroll
    for (int k = 0; k < kScanItems; ++k)
      if (base + k < ntiles) sums[base + k] = v[k] + carry;
    carry += total;
  }
  if (threadIdx.x == 0) offset[n] = carry;   // number of valid slots
}

// pass 3: add each tile's base
__global__ void __launch_bounds__(kScanThreads) scan_add_kernel(int* __restrict__ offset, int n,
                                                                const int* __restrict__ sums) {
  const int64_t base = (int64_t)blockIdx.x * kScanTile + threadIdx.x * kScanItems;
  const int add = sums[blockIdx.x];
#pragma unroll
  for (int k = 0; k < kScanItems; ++k)
    if (base + k < n) offset[base + k] += add;
}

// seg[offset[r] ...] <- slot ids naming r (in arbitrary order; sorted next)
__global__ void __launch_bounds__(256) fill_rows_kernel(const int32_t* __restrict__ idx, int64_t nslots, int T,
                                                        const int* __restrict__ offset, int* __restrict__ cursor,
                                                        int* __restrict__ seg) {
  for (int64_t s = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; s < nslots; s += (int64_t)gridDim.x * blockDim.x) {
    const int r = idx[s];
    if (valid_row(r, T)) seg[offset[r] + atomicAdd(cursor + r, 1)] = (int)s;
  }
}

// Bitonic sort of a[0, n) ascending, for any n: the network of the next power of
// two, with the missing elements read as +infinity (a pair whose upper element is
// missing is left alone).  Each stage first compares i with its mirror in the
// 2k-block, then the usual half-cleaners, so every comparison is ascending.
__device__ void bitonic_sort(int* a, int n) {
  int np2 = 1;
  while (np2 < n) np2 <<= 1;
  for (int k = 2; k <= np2; k <<= 1) {
    // mirror step
    for (int i = threadIdx.x; i < np2 / 2; i += blockDim.x) {
      const int blk = i / (k / 2), off = i % (k / 2);
      const int lo = blk * k + off, hi = blk * k + k - 1 - off;
      if (hi < n && a[lo] > a[hi]) { const int x = a[lo]; a[lo] = a[hi]; a[hi] = x; }
    }
    __syncthreads();
    for (int j = k / 4; j >= 1; j >>= 1) {
      for (int i = threadIdx.x; i < np2 / 2; i += blockDim.x) {
        const int lo = (i / j) * 2 * j + (i % j), hi = lo + j;
        if (hi < n && a[lo] > a[hi]) { const int x = a[lo]; a[lo] = a[hi]; a[hi] = x; }
      }
      __syncthreads();
    }
  }
}

// one block per row: sort the row's slot ids ascending (shared memory up to
// kSortCap ids, in place in global memory beyond)
__global__ void __launch_bounds__(kSortThreads) sort_rows_kernel(const int* __restrict__ offset, int* __restrict__ seg,
                                                                 int T) {
  extern __shared__ int buf[];   // kSortCap ints
  for (int r = blockIdx.x; r < T; r += gridDim.x) {
    const int b = offset[r], n = offset[r + 1] - b;
    if (n <= 1) continue;
    if (n <= kSortCap) {
      for (int i = threadIdx.x; i < n; i += blockDim.x) buf[i] = seg[b + i];
      __syncthreads();
      bitonic_sort(buf, n);
      for (int i = threadIdx.x; i < n; i += blockDim.x) seg[b + i] = buf[i];
      __syncthreads();
    } else {
      bitonic_sort(seg + b, n);
    }
  }
}

__global__ void __launch_bounds__(256) copy_ints_kernel(const int* __restrict__ src, int* __restrict__ dst, int n) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) dst[i] = src[i];
}

// One warp per kv row: add the contributions of the slots in [slot_lo, slot_hi)
// that name the row, in ascending slot order, to dkv32[r].  gbuf holds, per head
// group g (stride gstride floats), the contribution of slot s at
// (s - slot_lo) * 576; the head groups of a slot are added in order.
__global__ void __launch_bounds__(256) reduce_rows_kernel(const int* __restrict__ offset, const int* __restrict__ seg,
                                                          int* __restrict__ pos, const float* __restrict__ gbuf,
                                                          int ng, int64_t gstride, int64_t slot_lo, int64_t slot_hi,
                                                          int T, float* __restrict__ dkv32, uint32_t* status) {
  const int lane = threadIdx.x & 31;
  const int r = (int)(((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5);
  if (r >= T) return;
  int p = pos[r];
  const int e = offset[r + 1];
  if (p >= e || seg[p] >= slot_hi) return;
  float acc[kDqk / 32];
  if (!check_range(dkv32 + (int64_t)r * kDqk, kDqk, dkv32, (int64_t)T * kDqk, status)) return;
  float* row = dkv32 + (int64_t)r * kDqk + lane;
  const int64_t gbuf_n = (int64_t)ng * gstride;
#pragma unroll
  for (int k = 0; k < kDqk / 32; ++k) acc[k] = row[32 * k];
  if (ng == 1) {
    // four contributions in flight at a time, added in ascending slot order (the
    // row's slot list is sorted, so the ones in this chunk form a prefix)
    for (;;) {
      int64_t s[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) s[u] = p + u < e ? (int64_t)seg[p + u] : slot_hi;
      float v[4][kDqk / 32];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        if (s[u] < slot_hi) {
          const float* gs = gbuf + (s[u] - slot_lo) * kDqk + lane;
          const bool in = check_range(gs - lane, kDqk, gbuf, gbuf_n, status);
#pragma unroll
          for (int k = 0; k < kDqk / 32; ++k) v[u][k] = in ? gs[32 * k] : 0.f;
        }
      }
      int n = 0;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        if (s[u] >= slot_hi) break;
#pragma unroll
        for (int k = 0; k < kDqk / 32; ++k) acc[k] += v[u][k];
        ++n;
      }
      p += n;
      if (n < 4) break;
    }
  } else {
    for (; p < e; ++p) {
      const int64_t s = seg[p];
      if (s >= slot_hi) break;
      const float* gs = gbuf + (s - slot_lo) * kDqk + lane;
      for (int g = 0; g < ng; ++g) {
        if (!check_range(gs - lane + (int64_t)g * gstride, kDqk, gbuf, gbuf_n, status)) continue;
#pragma unroll
        for (int k = 0; k < kDqk / 32; ++k) acc[k] += gs[(int64_t)g * gstride + 32 * k];
      }
    }
  }
#pragma unroll
  for (int k = 0; k < kDqk / 32; ++k) row[32 * k] = acc[k];
  if (lane == 0) pos[r] = p;
}

unsigned grid_for(int64_t n, int threads) {
  const int64_t b = (n + threads - 1) / threads;
  return (unsigned)(b < 1 ? 1 : (b > 65536 * 16 ? 65536 * 16 : b));
}

}  // namespace

int64_t det_scan_tiles(int T) { return ((int64_t)T + kScanTile - 1) / kScanTile; }

cudaError_t launch_build_row_lists(const int32_t* indices, int T, int topk, int* offset, int* cursor, int* pos,
                                   int* seg, int* scan_sums, cudaStream_t s, int* nlaunch) {
  const int64_t nslots = (int64_t)T * topk;
  cudaError_t e = cudaMemsetAsync(cursor, 0, sizeof(int) * (size_t)T, s);
  if (e != cudaSuccess) return e;
  count_rows_kernel<<<grid_for(nslots, 256), 256, 0, s>>>(indices, nslots, T, cursor);
  const int ntiles = (int)det_scan_tiles(T);
  scan_tiles_kernel<<<ntiles, kScanThreads, 0, s>>>(cursor, T, offset, scan_sums);
  scan_sums_kernel<<<1, kScanThreads, 0, s>>>(scan_sums, ntiles, offset, T);
  scan_add_kernel<<<ntiles, kScanThreads, 0, s>>>(offset, T, scan_sums);
  if ((e = cudaMemsetAsync(cursor, 0, sizeof(int) * (size_t)T, s)) != cudaSuccess) return e;
  fill_rows_kernel<<<grid_for(nslots, 256), 256, 0, s>>>(indices, nslots, T, offset, cursor, seg);
  if ((e = cudaFuncSetAttribute(sort_rows_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)(sizeof(int) * kSortCap))) != cudaSuccess)
    return e;
  sort_rows_kernel<<<(unsigned)(T < 65536 ? T : 65536), kSortThreads, sizeof(int) * kSortCap, s>>>(offset, seg, T);
  copy_ints_kernel<<<grid_for(T, 256), 256, 0, s>>>(offset, pos, T);
  *nlaunch = 7;
  return cudaGetLastError();
}

cudaError_t launch_reduce_rows(const int* offset, const int* seg, int* pos, const float* gbuf, int ng,
                               int64_t gstride, int64_t slot_lo, int64_t slot_hi, int T, float* dkv32,
                               cudaStream_t s) {
  reduce_rows_kernel<<<(unsigned)(((int64_t)T * 32 + 255) / 256), 256, 0, s>>>(offset, seg, pos, gbuf, ng, gstride,
                                                                                slot_lo, slot_hi, T, dkv32,
                                                                                tc_status_ptr());
  return cudaGetLastError();
}

}  // namespace smla
