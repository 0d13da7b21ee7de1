// CUDA-core kernels of the sparse MLA path: a forward and a backward that
// work for every supported head count, plus the Delta pre-pass, the
// fp32 -> bf16 cast of dKV and the index validator.
//
// Structure (one CTA per query token and group of HG heads, 256 threads):
//   * the CTA's query rows (and dO rows in the backward) are staged in shared
//     memory as fp32;
//   * the top-k list is walked in blocks of 32 slots.  Each block's indices
//     are masked (valid iff 0 <= idx < T) and only valid rows are loaded;
//     padding slots get exact-zero K/V in shared memory and their score is
//     excluded from the softmax (miles PR #2079 summary, implementation
//     breakdown items 2-3: clamp + mask so padding contributes exactly 0).
//     Blocks with no valid slot are skipped;
//   * forward: online softmax in the exp2 domain with a running max, the sum
//     of exponentials floored at 1e-30 at the end (PR #2079 forward
//     fragment), natural-log LSE out;
//   * backward: P recomputed from the saved LSE, dP = dO V^T,
//     dS = P (dP - Delta), dQ accumulated in registers, the per-block dKV
//     rows formed in registers and scatter-added with 16-byte fp32 vector
//     reductions into the named rows only (padding slots issue no write).
#include "smla_common.cuh"

namespace smla {
namespace {

constexpr int kNT = 256;       // threads per CTA
constexpr int kBK = 32;        // top-k slots per block
constexpr int kQP = 580;       // padded fp32 row pitch for 576-wide rows (float4 aligned)
constexpr int kOP = 516;       // padded fp32 row pitch for 512-wide rows
constexpr int kPP = kBK + 1;   // pitch of the [heads][slots] P / dS tiles

// Load `rows` bf16 rows of width `w` (multiple of 8) into fp32 smem rows of pitch `pitch`.
__device__ __forceinline__ void stage_rows_f32(float* dst, int pitch, const uint16_t* src,
                                               int64_t src_pitch, int rows, int w) {
  const int chunks = w / 8;
  for (int i = threadIdx.x; i < rows * chunks; i += kNT) {
    const int r = i / chunks, c = i - r * chunks;
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(src + r * src_pitch + c * 8));
    float4* d = reinterpret_cast<float4*>(dst + r * pitch + c * 8);
    d[0] = make_float4(bf16_lo(v.x), bf16_hi(v.x), bf16_lo(v.y), bf16_hi(v.y));
    d[1] = make_float4(bf16_lo(v.z), bf16_hi(v.z), bf16_lo(v.w), bf16_hi(v.w));
  }
}

// Read the block's 32 indices, mask them, and gather the valid KV rows as
// fp32 (zero rows for padding).  Returns false (uniformly) when no slot of
// the block is valid.
__device__ __forceinline__ bool gather_block(const int32_t* idx_row, int blk, int T,
                                             const uint16_t* kv, int* s_row, float* skv, uint32_t* status) {
  int valid = 0;
  if (threadIdx.x < kBK) {
    const int idx = __ldg(idx_row + blk * kBK + threadIdx.x);
    valid = (idx >= 0 && idx < T);
    s_row[threadIdx.x] = valid ? idx : -1;
  }
  if (!__syncthreads_or(valid)) return false;
  for (int i = threadIdx.x; i < kBK * (kDqk / 8); i += kNT) {
    const int j = i / (kDqk / 8), c = i - j * (kDqk / 8);
    const int row = s_row[j];
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    const uint16_t* src = kv + (int64_t)(row >= 0 ? row : 0) * kDqk + c * 8;
    if (row >= 0 && check_range(src, 8, kv, (int64_t)T * kDqk, status)) v = __ldg(reinterpret_cast<const uint4*>(src));
    float4* d = reinterpret_cast<float4*>(skv + j * kQP + c * 8);
    d[0] = make_float4(bf16_lo(v.x), bf16_hi(v.x), bf16_lo(v.y), bf16_hi(v.y));
    d[1] = make_float4(bf16_lo(v.z), bf16_hi(v.z), bf16_lo(v.w), bf16_hi(v.w));
  }
  __syncthreads();
  return true;
}

__device__ __forceinline__ float dot4(float4 a, float4 b) {
  return a.x * b.x + a.y * b.y + a.z * b.z + a.w * b.w;
}

template <int HG>
__global__ void __launch_bounds__(kNT, 1) fwd_simt_kernel(FwdArgs a) {
  static_assert(HG % 8 == 0 && HG <= 32, "head group");
  constexpr int KH = HG / 8;             // heads per warp in the score phase
  constexpr int TPH = kNT / HG;          // threads per head in the output phase
  constexpr int NO = kDv / (4 * TPH);    // float4 accumulators per thread
  extern __shared__ float4 smem_f4[];
  float* sq = reinterpret_cast<float*>(smem_f4);  // [HG][kQP]
  float* skv = sq + HG * kQP;                      // [kBK][kQP]
  float* sp = skv + kBK * kQP;                     // [HG][kPP]
  float* s_alpha = sp + HG * kPP;                  // [HG]
  float* s_m = s_alpha + HG;                       // [HG]
  float* s_l = s_m + HG;                           // [HG]
  int* s_row = reinterpret_cast<int*>(s_l + HG);   // [kBK]

  const int t = a.t0 + blockIdx.x;
  const int h0 = blockIdx.y * HG;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const float c2 = a.scale * kLog2e;

  stage_rows_f32(sq, kQP, a.q + ((int64_t)t * a.H + h0) * kDqk, kDqk, HG, kDqk);

  float m[KH], l[KH];
#pragma unroll
  for (int k = 0; k < KH; ++k) { m[k] = -INFINITY; l[k] = 0.f; }
  const int oh = threadIdx.x / TPH;
  const int od0 = (threadIdx.x % TPH) * 4;
  float4 o[NO];
#pragma unroll
  for (int n = 0; n < NO; ++n) o[n] = make_float4(0.f, 0.f, 0.f, 0.f);

  const int32_t* idx_row = a.indices + (int64_t)t * a.topk;
  const int nblk = a.topk / kBK;
  for (int blk = 0; blk < nblk; ++blk) {
    if (!gather_block(idx_row, blk, a.T, a.kv, s_row, skv, a.status)) continue;
    // scores: lane = slot, heads warp + 8k
    float s[KH];
#pragma unroll
    for (int k = 0; k < KH; ++k) s[k] = 0.f;
    const float* kr = skv + lane * kQP;
#pragma unroll 4
    for (int d = 0; d < kDqk; d += 4) {
      const float4 kk = *reinterpret_cast<const float4*>(kr + d);
#pragma unroll
      for (int k = 0; k < KH; ++k)
        s[k] += dot4(*reinterpret_cast<const float4*>(sq + (warp + 8 * k) * kQP + d), kk);
    }
    const bool valid = s_row[lane] >= 0;
#pragma unroll
    for (int k = 0; k < KH; ++k) {
      const float x = valid ? s[k] * c2 : -INFINITY;
      const float m_new = fmaxf(m[k], warp_max(x));
      float p = 0.f, alpha = 1.f;
      if (m_new != -INFINITY) {          // at least one valid slot so far
        alpha = exp2f(m[k] - m_new);     // m = -inf gives 0
        p = valid ? exp2f(x - m_new) : 0.f;
      }
      l[k] = l[k] * alpha + warp_sum(p);
      m[k] = m_new;
      const int h = warp + 8 * k;
      sp[h * kPP + lane] = p;
      if (lane == 0) s_alpha[h] = alpha;
    }
    __syncthreads();
    const float al = s_alpha[oh];
#pragma unroll
    for (int n = 0; n < NO; ++n) { o[n].x *= al; o[n].y *= al; o[n].z *= al; o[n].w *= al; }
    for (int j = 0; j < kBK; ++j) {
      const float p = sp[oh * kPP + j];
      const float* vr = skv + j * kQP + od0;
#pragma unroll
      for (int n = 0; n < NO; ++n) {
        const float4 v = *reinterpret_cast<const float4*>(vr + n * 4 * TPH);
        o[n].x += p * v.x; o[n].y += p * v.y; o[n].z += p * v.z; o[n].w += p * v.w;
      }
    }
    __syncthreads();
  }
  if (lane == 0) {
#pragma unroll
    for (int k = 0; k < KH; ++k) { s_m[warp + 8 * k] = m[k]; s_l[warp + 8 * k] = l[k]; }
  }
  __syncthreads();
  // epilogue: out = O / max(l, 1e-30); empty rows (l == 0) give exactly 0
  const float inv = 1.f / fmaxf(s_l[oh], kSumexpFloor);
  uint16_t* orow = a.out + ((int64_t)t * a.H + h0 + oh) * kDv + od0;
#pragma unroll
  for (int n = 0; n < NO; ++n) {
    uint2 pk;
    pk.x = pack_bf16x2(o[n].x * inv, o[n].y * inv);
    pk.y = pack_bf16x2(o[n].z * inv, o[n].w * inv);
    *reinterpret_cast<uint2*>(orow + n * 4 * TPH) = pk;
  }
  if (threadIdx.x < HG) {
    const float lh = s_l[threadIdx.x];
    a.lse[(int64_t)t * a.H + h0 + threadIdx.x] =
        lh > 0.f ? (s_m[threadIdx.x] + log2f(lh)) * kLn2 : kLseEmpty;
  }
}

template <int HG>
__global__ void __launch_bounds__(kNT, 1) bwd_simt_kernel(BwdArgs a) {
  static_assert(HG % 8 == 0 && HG <= 32, "head group");
  constexpr int KH = HG / 8;
  constexpr int TPH = kNT / HG;                            // threads per head (dQ phase)
  constexpr int NQ = (kDqk + 4 * TPH - 1) / (4 * TPH);     // float4 dQ accumulators
  constexpr int NK = kDqk / 32;                            // float4 dKV accumulators (18)
  extern __shared__ float4 smem_f4[];
  float* sq = reinterpret_cast<float*>(smem_f4);  // [HG][kQP]
  float* sdo = sq + HG * kQP;                      // [HG][kOP]
  float* skv = sdo + HG * kOP;                     // [kBK][kQP]
  float* sp = skv + kBK * kQP;                     // [HG][kPP]
  float* sds = sp + HG * kPP;                      // [HG][kPP]
  float* s_lse2 = sds + HG * kPP;                  // [HG]
  float* s_dl = s_lse2 + HG;                       // [HG]
  int* s_row = reinterpret_cast<int*>(s_dl + HG);  // [kBK]

  const int t = a.t0 + blockIdx.x;
  const int h0 = blockIdx.y * HG;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const float c2 = a.scale * kLog2e;

  stage_rows_f32(sq, kQP, a.q + ((int64_t)t * a.H + h0) * kDqk, kDqk, HG, kDqk);
  stage_rows_f32(sdo, kOP, a.dout + ((int64_t)t * a.H + h0) * kDv, kDv, HG, kDv);
  if (threadIdx.x < HG) {
    s_lse2[threadIdx.x] = a.lse[(int64_t)t * a.H + h0 + threadIdx.x] * kLog2e;
    s_dl[threadIdx.x] = a.delta[(int64_t)t * a.H + h0 + threadIdx.x];
  }

  const int qh = threadIdx.x / TPH;
  const int qd0 = (threadIdx.x % TPH) * 4;
  float4 dq[NQ];
#pragma unroll
  for (int n = 0; n < NQ; ++n) dq[n] = make_float4(0.f, 0.f, 0.f, 0.f);
  const int kj = threadIdx.x >> 3;            // slot of this thread in the dKV phase
  const int kd0 = (threadIdx.x & 7) * 4;

  const int32_t* idx_row = a.indices + (int64_t)t * a.topk;
  const int nblk = a.topk / kBK;
  for (int blk = 0; blk < nblk; ++blk) {
    if (!gather_block(idx_row, blk, a.T, a.kv, s_row, skv, a.status)) continue;
    // S = q.k over 576 dims and dP = dO.v over 512 dims; lane = slot
    float s[KH], dp[KH];
#pragma unroll
    for (int k = 0; k < KH; ++k) { s[k] = 0.f; dp[k] = 0.f; }
    const float* kr = skv + lane * kQP;
#pragma unroll 4
    for (int d = 0; d < kDv; d += 4) {
      const float4 kk = *reinterpret_cast<const float4*>(kr + d);
#pragma unroll
      for (int k = 0; k < KH; ++k) {
        s[k] += dot4(*reinterpret_cast<const float4*>(sq + (warp + 8 * k) * kQP + d), kk);
        dp[k] += dot4(*reinterpret_cast<const float4*>(sdo + (warp + 8 * k) * kOP + d), kk);
      }
    }
#pragma unroll
    for (int d = kDv; d < kDqk; d += 4) {
      const float4 kk = *reinterpret_cast<const float4*>(kr + d);
#pragma unroll
      for (int k = 0; k < KH; ++k)
        s[k] += dot4(*reinterpret_cast<const float4*>(sq + (warp + 8 * k) * kQP + d), kk);
    }
    const bool valid = s_row[lane] >= 0;
#pragma unroll
    for (int k = 0; k < KH; ++k) {
      const int h = warp + 8 * k;
      // padding slots: P forced to 0 (not left to the zero key)
      const float p = valid ? exp2f(s[k] * c2 - s_lse2[h]) : 0.f;
      sp[h * kPP + lane] = p;
      sds[h * kPP + lane] = p * (dp[k] - s_dl[h]);
    }
    __syncthreads();
    // dQ += dS K (scale applied at the end)
    for (int j = 0; j < kBK; ++j) {
      const float ds = sds[qh * kPP + j];
      const float* kr2 = skv + j * kQP + qd0;
#pragma unroll
      for (int n = 0; n < NQ; ++n) {
        if (qd0 + n * 4 * TPH < kDqk) {
          const float4 v = *reinterpret_cast<const float4*>(kr2 + n * 4 * TPH);
          dq[n].x += ds * v.x; dq[n].y += ds * v.y; dq[n].z += ds * v.z; dq[n].w += ds * v.w;
        }
      }
    }
    // dKV rows of this block: G[j] = sum_h P[h,j] dO[h] (latent) + scale dS[h,j] q[h]
    const int row = s_row[kj];
    if (row >= 0) {
      float4 g[NK];
#pragma unroll
      for (int n = 0; n < NK; ++n) g[n] = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int h = 0; h < HG; ++h) {
        const float p = sp[h * kPP + kj];
        const float ds = sds[h * kPP + kj] * a.scale;
        const float* qr = sq + h * kQP + kd0;
        const float* dr = sdo + h * kOP + kd0;
#pragma unroll
        for (int n = 0; n < NK; ++n) {
          const float4 qq = *reinterpret_cast<const float4*>(qr + 32 * n);
          g[n].x += ds * qq.x; g[n].y += ds * qq.y; g[n].z += ds * qq.z; g[n].w += ds * qq.w;
          if (n < kDv / 32) {
            const float4 oo = *reinterpret_cast<const float4*>(dr + 32 * n);
            g[n].x += p * oo.x; g[n].y += p * oo.y; g[n].z += p * oo.z; g[n].w += p * oo.w;
          }
        }
      }
      if (a.gbuf != nullptr) {           // deterministic mode: store this head group's part of the slot
        float* dst = a.gbuf + (int64_t)blockIdx.y * a.gstride +
                     ((int64_t)(t - a.t0) * a.topk + (int64_t)blk * kBK + kj) * kDqk + kd0;
#pragma unroll
        for (int n = 0; n < NK; ++n)
          if (check_range(dst + 32 * n, 4, a.gbuf, a.gbuf_floats, a.status))
            *reinterpret_cast<float4*>(dst + 32 * n) = g[n];
      } else {
        float* dst = a.dkv32 + (int64_t)row * kDqk + kd0;
#pragma unroll
        for (int n = 0; n < NK; ++n)
          if (check_range(dst + 32 * n, 4, a.dkv32, (int64_t)a.T * kDqk, a.status))
            red_add_v4(dst + 32 * n, g[n].x, g[n].y, g[n].z, g[n].w);
      }
    }
    __syncthreads();
  }
  uint16_t* qrow = a.dq + ((int64_t)t * a.H + h0 + qh) * kDqk + qd0;
#pragma unroll
  for (int n = 0; n < NQ; ++n) {
    if (qd0 + n * 4 * TPH < kDqk) {
      uint2 pk;
      pk.x = pack_bf16x2(dq[n].x * a.scale, dq[n].y * a.scale);
      pk.y = pack_bf16x2(dq[n].z * a.scale, dq[n].w * a.scale);
      *reinterpret_cast<uint2*>(qrow + n * 4 * TPH) = pk;
    }
  }
}

// Delta[r] = sum_d dO[r, d] * out[r, d] over 512 dims; one warp per row.
__global__ void __launch_bounds__(256) delta_kernel(const uint16_t* __restrict__ out,
                                                    const uint16_t* __restrict__ dout,
                                                    float* __restrict__ delta, int64_t rows) {
  const int64_t r = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (r >= rows) return;
  const uint4* po = reinterpret_cast<const uint4*>(out + r * kDv);
  const uint4* pd = reinterpret_cast<const uint4*>(dout + r * kDv);
  float acc = 0.f;
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const uint4 x = __ldg(po + lane + 32 * i), y = __ldg(pd + lane + 32 * i);
    acc += bf16_lo(x.x) * bf16_lo(y.x) + bf16_hi(x.x) * bf16_hi(y.x);
    acc += bf16_lo(x.y) * bf16_lo(y.y) + bf16_hi(x.y) * bf16_hi(y.y);
    acc += bf16_lo(x.z) * bf16_lo(y.z) + bf16_hi(x.z) * bf16_hi(y.z);
    acc += bf16_lo(x.w) * bf16_lo(y.w) + bf16_hi(x.w) * bf16_hi(y.w);
  }
  acc = warp_sum(acc);
  if (lane == 0) delta[r] = acc;
}

// dst = bf16(src), round to nearest even; n is a multiple of 4.
__global__ void __launch_bounds__(256) cast_bf16_kernel(const float4* __restrict__ src,
                                                        uint2* __restrict__ dst, int64_t n4) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4;
       i += (int64_t)gridDim.x * blockDim.x) {
    const float4 v = src[i];
    dst[i] = make_uint2(pack_bf16x2(v.x, v.y), pack_bf16x2(v.z, v.w));
  }
}

// Counts entries that are neither -1 nor a row of the query's own sequence.
__global__ void __launch_bounds__(256) check_indices_kernel(const int32_t* __restrict__ indices,
                                                            int T, int topk,
                                                            const int32_t* __restrict__ cu, int B,
                                                            unsigned long long* counter) {
  const int lane = threadIdx.x & 31;
  unsigned long long bad = 0;
  for (int64_t t = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5); t < T;
       t += (int64_t)gridDim.x * 8) {
    int lo = 0, hi = B;  // find b with cu[b] <= t < cu[b+1]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (__ldg(cu + mid) <= t) lo = mid; else hi = mid;
    }
    const int s0 = __ldg(cu + lo), s1 = __ldg(cu + lo + 1);
    for (int k = lane; k < topk; k += 32) {
      const int v = __ldg(indices + t * topk + k);
      bad += (v != -1) && !(v >= s0 && v < s1);
    }
  }
  for (int o = 16; o > 0; o >>= 1) bad += __shfl_xor_sync(0xffffffffu, bad, o);
  if (lane == 0 && bad) atomicAdd(counter, bad);
}

template <int HG>
size_t fwd_smem() {
  return sizeof(float) * ((size_t)HG * kQP + kBK * kQP + HG * kPP + 3 * HG) + sizeof(int) * kBK;
}
template <int HG>
size_t bwd_smem() {
  return sizeof(float) * ((size_t)HG * kQP + HG * kOP + kBK * kQP + 2 * HG * kPP + 2 * HG) +
         sizeof(int) * kBK;
}

template <int HG>
cudaError_t fwd_launch(const FwdArgs& a, cudaStream_t s) {
  const size_t sm = fwd_smem<HG>();
  cudaError_t e = cudaFuncSetAttribute(fwd_simt_kernel<HG>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
  if (e != cudaSuccess) return e;
  const int nt = a.nt < 0 ? a.T : a.nt;
  if (nt == 0) return cudaSuccess;
  fwd_simt_kernel<HG><<<dim3(nt, a.H / HG), kNT, sm, s>>>(a);
  return cudaGetLastError();
}
template <int HG>
cudaError_t bwd_launch(const BwdArgs& a, cudaStream_t s) {
  const size_t sm = bwd_smem<HG>();
  cudaError_t e = cudaFuncSetAttribute(bwd_simt_kernel<HG>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
  if (e != cudaSuccess) return e;
  const int nt = a.nt < 0 ? a.T : a.nt;
  if (nt == 0) return cudaSuccess;
  bwd_simt_kernel<HG><<<dim3(nt, a.H / HG), kNT, sm, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_simt(const FwdArgs& args, cudaStream_t s) {
  FwdArgs a = args;
  a.status = tc_status_ptr();
  if (a.H == 8) return fwd_launch<8>(a, s);
  if (a.H == 16) return fwd_launch<16>(a, s);
  return fwd_launch<32>(a, s);  // H = 32, 64, 128 in groups of 32 heads
}

int simt_head_groups(int H) { return H <= 16 ? 1 : H / 32; }

cudaError_t launch_bwd_simt(const BwdArgs& args, cudaStream_t s) {
  BwdArgs a = args;
  a.status = tc_status_ptr();
  a.gbuf_floats = a.gbuf != nullptr ? (int64_t)simt_head_groups(a.H) * a.gstride : 0;
  if (a.H == 8) return bwd_launch<8>(a, s);
  if (a.H == 16) return bwd_launch<16>(a, s);
  return bwd_launch<32>(a, s);
}

cudaError_t launch_delta(const uint16_t* out, const uint16_t* dout, float* delta, int64_t rows,
                         cudaStream_t s) {
  if (rows == 0) return cudaSuccess;
  delta_kernel<<<(unsigned)((rows + 7) / 8), 256, 0, s>>>(out, dout, delta, rows);
  return cudaGetLastError();
}

cudaError_t launch_cast_bf16(const float* src, uint16_t* dst, int64_t n, cudaStream_t s) {
  const int64_t n4 = n / 4;
  if (n4 == 0) return cudaSuccess;
  const int64_t blocks = (n4 + 255) / 256;
  cast_bf16_kernel<<<(unsigned)(blocks < 152 * 16 ? blocks : 152 * 16), 256, 0, s>>>(
      reinterpret_cast<const float4*>(src), reinterpret_cast<uint2*>(dst), n4);
  return cudaGetLastError();
}

cudaError_t launch_check_indices(const int32_t* indices, int T, int topk, const int32_t* cu_seqlens,
                                 int B, unsigned long long* counter, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  const int64_t blocks = ((int64_t)T + 7) / 8;
  check_indices_kernel<<<(unsigned)(blocks < 152 * 8 ? blocks : 152 * 8), 256, 0, s>>>(
      indices, T, topk, cu_seqlens, B, counter);
  return cudaGetLastError();
}

}  // namespace smla
