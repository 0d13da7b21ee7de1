// Tensor-core (tcgen05) forward for small head counts (H <= 16).
//
// With few heads the score tile is put on its side: the top-k slots of a block
// are the M = 128 rows of the MMA and the heads the N = 16 columns (heads past
// H are zero q rows), so the MMA work scales with H instead of a 128-row head
// tile.  One CTA per SM walks a strided list of query tokens (a persistent
// kernel); every gathered KV row is read once.
//
// Per token, q (16 heads x 576, bf16) sits in shared memory as the B operand.
// Per block of 128 top-k slots:
//   producers : masked 16-byte cp.async gather of the 128 named rows into four
//               latent units (128 rows x 128 dims, 32 KiB, the V tiles) and one
//               tail unit (the 64 rope dims), 128B-swizzled; padding slots copy
//               zero bytes (exact-zero K/V rows, the clamp + mask of the miles
//               PR #2079 fix, implementation breakdown item 2);
//   MMA       : S^T = K q^T (M = 128 slots, N = 16 heads, K = 576) into one of
//               two 16-column TMEM buffers;
//   softmax   : one thread per slot: padding slots are masked to -inf; per head
//               the block max and the sums are reduced across the 128 threads;
//               the running max moves lazily (only when a block max exceeds it
//               by more than 8 in the log2 domain; O is then rescaled in TMEM);
//               P^T is rounded to bf16 into shared memory (K-major: row h, the
//               slots along K);
//   MMA       : O^T[d, h] += V^T P^T (M = 128 dims per latent unit, N = 16,
//               K = 128 slots, V read MN-major from the unit) into four
//               16-column TMEM tiles; the latent units are then free;
//   epilogue  : at the end of a token out = O^T / (sum of the bf16-rounded
//               weights), so the rounding of P cancels; LSE = ln of the fp32
//               sum floored at 1e-30 (miles PR #2079 summary, forward
//               fragment): a row with no valid slot gets ln(1e-30) and out = 0.
#include <cuda.h>

#include "smla_common.cuh"
#include "tc_common.cuh"

namespace smla {
namespace {

using namespace tc;

constexpr int kBS = 128;                // slots per block (the M of the score MMA)
constexpr int kHN = 16;                 // heads as the N dimension (rows H..15 of q are zero)
constexpr int kProducers = 128;         // warps 0..3 gather
constexpr int kMmaWarp = 4;             // warp 4, lane 0: MMA issuer; the warp owns TMEM
constexpr int kSmWarp0 = 5;             // warps 5..8: one thread per slot (softmax), rescale, epilogue
constexpr int kThreads = 288;
constexpr int kRowsPerThread = kBS * 8 / kProducers;   // 8 rows, one 16-byte piece of each chunk
constexpr float kLazyRescale = 8.f;
constexpr int kMaskRing = 4;
constexpr int kMaxBlocks = kTcMaxTopk / 64;            // blocks of 128 slots, topk a multiple of 64
constexpr int kProdBar = 1, kSmBar = 2;                // named barriers

constexpr int kLatBytes = 2 * 128 * 128;   // two 64-dim chunks of 128 rows
constexpr int kTailBytes = 128 * 128;      // the rope chunk of 128 rows
constexpr int kNLat = 5, kNTail = 2;   // one block's four latent units + the next block's first
constexpr int kQChunk = kHN * 128;         // one 64-dim chunk of the 16 q rows

constexpr int SM_LAT = 0;
constexpr int SM_TAIL = SM_LAT + kNLat * kLatBytes;
constexpr int SM_Q = SM_TAIL + kNTail * kTailBytes;        // 9 chunks
constexpr int SM_PT = SM_Q + 9 * kQChunk;                  // P^T: 2 chunks of 64 slots x 16 rows
constexpr int SM_RMAX = SM_PT + 2 * kQChunk;               // [4 warps][16] block maxima
constexpr int SM_RSUM = SM_RMAX + 4 * kHN * 4;             // [4 warps][32] sums (fp32, bf16-rounded)
constexpr int SM_MASK = SM_RSUM + 4 * 2 * kHN * 4;         // kMaskRing x 4 x u32
constexpr int SM_TOK = SM_MASK + kMaskRing * 16;           // 2 x int
constexpr int SM_BFLAG = SM_TOK + 16;
constexpr int SM_BLIST = SM_BFLAG + kMaxBlocks;
constexpr int SM_NB = SM_BLIST + 2 * kMaxBlocks;
constexpr int SM_BAR = (SM_NB + 8 + 7) & ~7;
enum Bar { LAT_FULL = 0, LAT_EMPTY = kNLat, TAIL_FULL = 2 * kNLat, TAIL_EMPTY = TAIL_FULL + kNTail,
           Q_FULL = TAIL_EMPTY + kNTail, Q_EMPTY, M_FULL, M_EMPTY = M_FULL + kMaskRing, S_FULL = M_EMPTY + kMaskRing,
           S_FREE = S_FULL + 2, P_FULL = S_FREE + 2, PV_DONE, O_FREE, TOK_FULL, TOK_EMPTY = TOK_FULL + 2,
           NBAR = TOK_EMPTY + 2 };
constexpr int SM_TMEM = SM_BAR + 8 * NBAR;
constexpr int SM_ABORT = SM_TMEM + 4;
constexpr int kSmemBytes = SM_ABORT + 4 + 1024;
static_assert(kSmemBytes <= 232448, "shared memory budget");
static_assert(SM_TAIL % 1024 == 0 && SM_Q % 1024 == 0 && SM_PT % 1024 == 0 && kQChunk % 1024 == 0, "swizzle atoms");

// TMEM: two 16-column S^T buffers, then O^T as four 16-column tiles (one per 128 dims)
constexpr uint32_t kTmemCols = 128;
constexpr uint32_t TM_S = 0;
constexpr uint32_t TM_O = 64;

struct SmallFwdParams {
  const uint16_t* q;
  const uint16_t* kv;
  const int32_t* indices;
  uint16_t* out;
  float* lse;
  uint32_t* status;
  int T, H, topk, t0, nt;
  float c2;                             // scale * log2(e)
};

__device__ __forceinline__ uint32_t bar_addr(uint32_t base, int i) { return base + SM_BAR + 8 * i; }
__device__ __forceinline__ void named_bar_sync(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}
__device__ __forceinline__ int cta_tokens(const SmallFwdParams& p) {
  return (int)blockIdx.x < p.nt ? (p.nt - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
}

// Block count of the CTA's token k from the token ring (acknowledged on the ring's
// empty barrier); -1 on abort.
template <bool kWarp>
__device__ __forceinline__ int read_token(const SmallFwdParams& p, uint32_t sb, uint8_t* smem, int k,
                                          volatile int* abort_flag) {
  const bool ok = kWarp ? __all_sync(0xffffffffu, mbar_wait(bar_addr(sb, TOK_FULL + (k & 1)), (k >> 1) & 1, abort_flag,
                                                            p.status))
                        : mbar_wait(bar_addr(sb, TOK_FULL + (k & 1)), (k >> 1) & 1, abort_flag, p.status);
  if (!ok) return -1;
  const int nb = reinterpret_cast<volatile int*>(smem + SM_TOK)[k & 1];
  mbar_arrive(bar_addr(sb, TOK_EMPTY + (k & 1)));
  return nb;
}

// Producers: per token, list the blocks of 128 slots that hold a valid slot,
// publish the count, gather the token's q rows, then each block's rows unit by
// unit; the slot-validity mask of each block goes into the mask ring.
__device__ __forceinline__ void produce(const SmallFwdParams& p, uint32_t sb, uint8_t* smem, volatile int* abort_flag) {
  const int pt = threadIdx.x;              // 0..127
  const int warp = pt >> 5, lane = pt & 31;
  const int c16 = pt & 7, r0 = pt >> 3;    // 16-byte piece c16 of rows r0 + 16 j
  constexpr int R = kRowsPerThread;
  const int nblk = (p.topk + kBS - 1) / kBS;
  const int ntok = cta_tokens(p);
  uint8_t* flag = smem + SM_BFLAG;
  int16_t* blist = reinterpret_cast<int16_t*>(smem + SM_BLIST);
  volatile int* nbs = reinterpret_cast<volatile int*>(smem + SM_NB);
  volatile int* tok = reinterpret_cast<volatile int*>(smem + SM_TOK);
  const uint16_t* kvc = p.kv + 8 * c16;
  int nl = 0, gb = 0, kq = 0;              // latent units, blocks, tokens with blocks so far
  for (int k = 0; k < ntok; ++k) {
    const int t = p.t0 + (int)blockIdx.x + k * (int)gridDim.x;
    const int32_t* irow = p.indices + (int64_t)t * p.topk;
    for (int b = pt; b < nblk; b += kProducers) {
      const int n4 = (b * kBS + kBS <= p.topk ? kBS : p.topk - b * kBS) / 4;
      const int4* ib = reinterpret_cast<const int4*>(irow + b * kBS);
      bool v = false;
      for (int c = 0; c < n4; ++c) {
        const int4 x = __ldg(ib + c);
        v |= (x.x >= 0 && x.x < p.T) | (x.y >= 0 && x.y < p.T) | (x.z >= 0 && x.z < p.T) | (x.w >= 0 && x.w < p.T);
      }
      flag[b] = v ? 1 : 0;
    }
    named_bar_sync(kProdBar, kProducers);
    if (warp == 0) {
      int base = 0;
      for (int b0 = 0; b0 < nblk; b0 += 32) {
        const bool f = (b0 + lane < nblk) && flag[b0 + lane];
        const uint32_t m = __ballot_sync(0xffffffffu, f);
        if (f) blist[base + __popc(m & ((1u << lane) - 1u))] = (int16_t)(b0 + lane);
        base += __popc(m);
      }
      const bool ok = k < 2 || __all_sync(0xffffffffu, mbar_wait(bar_addr(sb, TOK_EMPTY + (k & 1)), ((k >> 1) - 1) & 1,
                                                                 abort_flag, p.status));
      if (lane == 0) {
        *nbs = ok ? base : -1;
        if (ok) {
          tok[k & 1] = base;
          mbar_arrive(bar_addr(sb, TOK_FULL + (k & 1)));
        }
      }
    }
    named_bar_sync(kProdBar, kProducers);
    const int nb = *nbs;
    if (nb < 0) return;                    // uniform over the producer warps
    bool ok = true;
    if (nb == 0) continue;                 // nothing to gather, and no score MMA reads q
    // this token's q rows (rows H..15 zero) once the previous token's score MMAs completed
    if (kq >= 1 && !(ok = __all_sync(0xffffffffu, mbar_wait(bar_addr(sb, Q_EMPTY), (kq - 1) & 1, abort_flag, p.status))))
      return;
    ++kq;
    {
      const int h = r0;                     // 16 rows, one per group of 8 threads
      const bool real = h < p.H;
      const uint16_t* qsrc = p.q + ((int64_t)t * p.H + (real ? h : 0)) * kDqk + 8 * c16;
#pragma unroll
      for (int c = 0; c < 9; ++c)
        gather16(sb + SM_Q + c * kQChunk + h * 128 + ((c16 ^ (h & 7)) << 4), qsrc + 64 * c, real ? 16u : 0u, p.q,
                 (int64_t)p.T * p.H * kDqk, p.status);
      cp_async_arrive(bar_addr(sb, Q_FULL));
    }
    int nxt[R], nm[4] = {-1, -1, -1, -1};
    auto fetch = [&](int i) {
      const int b = blist[i];
#pragma unroll
      for (int j = 0; j < R; ++j) {
        const int slot = b * kBS + r0 + 16 * j;
        nxt[j] = slot < p.topk ? __ldg(irow + slot) : -1;
      }
      if (warp == 0) {
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          const int slot = b * kBS + 32 * w + lane;
          nm[w] = slot < p.topk ? __ldg(irow + slot) : -1;
        }
      }
    };
    if (nb > 0) fetch(0);
    for (int i = 0; ok && i < nb; ++i, ++gb) {
      int cur[R], cm[4];
#pragma unroll
      for (int j = 0; j < R; ++j) cur[j] = nxt[j];
#pragma unroll
      for (int w = 0; w < 4; ++w) cm[w] = nm[w];
      if (i + 1 < nb) fetch(i + 1);        // indices one block ahead
      const uint16_t* src[R];
      uint32_t dsto[R], nbytes[R];
#pragma unroll
      for (int j = 0; j < R; ++j) {
        const int r = r0 + 16 * j;
        const bool v = cur[j] >= 0 && cur[j] < p.T;
        src[j] = kvc + (int64_t)(v ? cur[j] : 0) * kDqk;
        dsto[j] = r * 128 + ((c16 ^ (r & 7)) << 4);
        nbytes[j] = v ? 16u : 0u;
      }
#pragma unroll 1
      for (int u = 0; u < 4; ++u, ++nl) {  // latent units: dims 128 u .. 128 u + 127
        const int slot = nl % kNLat;
        if (nl >= kNLat &&
            !(ok = __all_sync(0xffffffffu, mbar_wait(bar_addr(sb, LAT_EMPTY + slot), ((nl / kNLat) - 1) & 1, abort_flag,
                                                     p.status))))
          break;
        const uint32_t unit = sb + SM_LAT + slot * kLatBytes;
#pragma unroll
        for (int j = 0; j < R; ++j) {
          gather16(unit + dsto[j], src[j] + 128 * u, nbytes[j], p.kv, (int64_t)p.T * kDqk, p.status);
          gather16(unit + 128 * 128 + dsto[j], src[j] + 128 * u + 64, nbytes[j], p.kv, (int64_t)p.T * kDqk, p.status);
        }
        cp_async_arrive(bar_addr(sb, LAT_FULL + slot));
      }
      if (!ok) break;
      {                                    // the tail unit: dims 512..575
        const int slot = gb % kNTail;
        if (gb >= kNTail &&
            !(ok = __all_sync(0xffffffffu, mbar_wait(bar_addr(sb, TAIL_EMPTY + slot), ((gb / kNTail) - 1) & 1,
                                                     abort_flag, p.status))))
          break;
        const uint32_t unit = sb + SM_TAIL + slot * kTailBytes;
#pragma unroll
        for (int j = 0; j < R; ++j) gather16(unit + dsto[j], src[j] + 512, nbytes[j], p.kv, (int64_t)p.T * kDqk, p.status);
        cp_async_arrive(bar_addr(sb, TAIL_FULL + slot));
      }
      if (warp == 0) {                     // slot validity of the block for the softmax
        const int mr = gb % kMaskRing;
        if (gb >= kMaskRing &&
            !(ok = __all_sync(0xffffffffu, mbar_wait(bar_addr(sb, M_EMPTY + mr), ((gb / kMaskRing) - 1) & 1, abort_flag,
                                                     p.status))))
          break;
        uint32_t m[4];
#pragma unroll
        for (int w = 0; w < 4; ++w) m[w] = __ballot_sync(0xffffffffu, cm[w] >= 0 && cm[w] < p.T);
        if (lane == 0) {
          volatile uint32_t* mk = reinterpret_cast<volatile uint32_t*>(smem + SM_MASK + 16 * mr);
#pragma unroll
          for (int w = 0; w < 4; ++w) mk[w] = m[w];
          mbar_arrive(bar_addr(sb, M_FULL + mr));
        }
      }
      ok = __all_sync(0xffffffffu, ok);
    }
    if (!ok) return;
  }
}

// One step of a transposed warp reduction: lanes whose bit o is set keep the upper
// HALF of their values and send the lower half, the others the reverse; HALF == 0
// is a plain butterfly on the single remaining value.
template <int HALF, bool kMax>
__device__ __forceinline__ void wrt_step(float* v, int lane, int o) {
  if constexpr (HALF == 0) {
    const float got = __shfl_xor_sync(0xffffffffu, v[0], o);
    v[0] = kMax ? fmaxf(v[0], got) : v[0] + got;
  } else {
    const bool up = (lane & o) != 0;
#pragma unroll
    for (int i = 0; i < HALF; ++i) {
      const float send = up ? v[i] : v[i + HALF];
      const float keep = up ? v[i + HALF] : v[i];
      const float got = __shfl_xor_sync(0xffffffffu, send, o);
      v[i] = kMax ? fmaxf(keep, got) : keep + got;
    }
  }
}
// Transposed warp reduction of N values per lane (N = 16 or 32): N - 1 (+ 1) shuffles
// instead of 5 N.  Returns, in lane L, the reduction over the warp of value index
// L >> (5 - log2 N).
template <int N, bool kMax>
__device__ __forceinline__ float warp_reduce_t(float (&v)[N], int lane) {
  static_assert(N == 16 || N == 32, "value count");
  wrt_step<(N >> 1), kMax>(v, lane, 16);
  wrt_step<(N >> 2), kMax>(v, lane, 8);
  wrt_step<(N >> 3), kMax>(v, lane, 4);
  wrt_step<(N >> 4), kMax>(v, lane, 2);
  wrt_step<(N >> 5), kMax>(v, lane, 1);
  return v[0];
}

__global__ void __launch_bounds__(kThreads, 1) tc_fwd_small_kernel(SmallFwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sb = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ntok = cta_tokens(p);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + SM_ABORT);

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    for (int k = 0; k < kNLat; ++k) {
      mbar_init(bar_addr(sb, LAT_FULL + k), kProducers);   // cp.async arrivals
      mbar_init(bar_addr(sb, LAT_EMPTY + k), 1);           // the PV MMAs that read the unit completed
    }
    for (int k = 0; k < kNTail; ++k) {
      mbar_init(bar_addr(sb, TAIL_FULL + k), kProducers);
      mbar_init(bar_addr(sb, TAIL_EMPTY + k), 1);          // the score MMAs that read it completed
    }
    mbar_init(bar_addr(sb, Q_FULL), kProducers);
    mbar_init(bar_addr(sb, Q_EMPTY), 1);
    for (int k = 0; k < kMaskRing; ++k) {
      mbar_init(bar_addr(sb, M_FULL + k), 1);
      mbar_init(bar_addr(sb, M_EMPTY + k), 128);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar_addr(sb, S_FULL + b), 1);
      mbar_init(bar_addr(sb, S_FREE + b), 128);
      mbar_init(bar_addr(sb, TOK_FULL + b), 1);
      mbar_init(bar_addr(sb, TOK_EMPTY + b), 1 + 128);     // MMA thread and the slot threads
    }
    mbar_init(bar_addr(sb, P_FULL), 128);                  // P^T written (and O rescaled where the max moved)
    mbar_init(bar_addr(sb, PV_DONE), 1);
    mbar_init(bar_addr(sb, O_FREE), 128);                  // the epilogue read O^T
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(sb + SM_TMEM, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + SM_TMEM);

  if (warp < kProducers / 32) {
    produce(p, sb, smem, abort_flag);
  } else if (warp == kMmaWarp) {
    if (lane == 0) {
      const uint32_t id_s = idesc_bf16(128, kHN, false, false);   // A = K rows, B = q (both K-major)
      const uint32_t id_o = idesc_bf16(128, kHN, true, false);    // A = V^T read MN-major, B = P^T K-major
      const uint64_t dlat = sdesc_sw128(sb + SM_LAT, 16, 1024);
      const uint64_t dlatt = sdesc_sw128(sb + SM_LAT, 128 * 128, 1024);   // MN-major: 64-dim groups 16 KiB apart
      const uint64_t dtail = sdesc_sw128(sb + SM_TAIL, 16, 1024);
      const uint64_t dq = sdesc_sw128(sb + SM_Q, 16, 1024);
      const uint64_t dpt = sdesc_sw128(sb + SM_PT, 16, 1024);
      int gb = 0, nls = 0, nlp = 0, kq = 0;   // blocks; latent units scored / multiplied; tokens with blocks
      bool ok = true;
      // PV of running block g (token-local index jl), then hand its latent units back
      auto issue_pv = [&](int g, int jl, int k) -> bool {
        if (!mbar_wait(bar_addr(sb, P_FULL), g & 1, abort_flag, p.status)) return false;
        // O^T is free once the previous token's epilogue has read it (the slot threads
        // reach a token's first P only after that epilogue, so this wait never blocks)
        if (jl == 0 && k >= 1 && !mbar_wait(bar_addr(sb, O_FREE), (k - 1) & 1, abort_flag, p.status)) return false;
        tc_fence_after();
#pragma unroll 1
        for (int u = 0; u < 4; ++u, ++nlp) {
          const int slot = nlp % kNLat;
#pragma unroll
          for (int ks = 0; ks < 8; ++ks)
            mma_bf16_ss(tmem + TM_O + 16 * u, sdesc_add(dlatt, slot * kLatBytes + ks * 16 * 128),
                        sdesc_add(dpt, (ks >> 2) * kQChunk + (ks & 3) * 32), id_o, (jl > 0 || ks > 0));
          mma_commit(bar_addr(sb, LAT_EMPTY + slot));
        }
        mma_commit(bar_addr(sb, PV_DONE));
        return true;
      };
      for (int k = 0; ok && k < ntok; ++k) {
        const int nb = read_token<false>(p, sb, smem, k, abort_flag);
        if (!(ok = nb >= 0)) break;
        if (nb == 0) continue;
        if (!(ok = mbar_wait(bar_addr(sb, Q_FULL), kq & 1, abort_flag, p.status))) break;
        ++kq;
        for (int i = 0; ok && i < nb; ++i, ++gb) {
          const int b = gb & 1;
          if (gb >= 2 && !(ok = mbar_wait(bar_addr(sb, S_FREE + b), ((gb >> 1) - 1) & 1, abort_flag, p.status))) break;
          // S^T = K q^T over the four latent units and the tail
#pragma unroll 1
          for (int u = 0; u < 4; ++u, ++nls) {
            const int slot = nls % kNLat;
            if (!(ok = mbar_wait(bar_addr(sb, LAT_FULL + slot), (nls / kNLat) & 1, abort_flag, p.status))) break;
            fence_proxy_async_smem();      // cp.async wrote the unit through the generic proxy
            tc_fence_after();
#pragma unroll
            for (int c = 0; c < 2; ++c)
#pragma unroll
              for (int ks = 0; ks < 4; ++ks)
                mma_bf16_ss(tmem + TM_S + 16 * b, sdesc_add(dlat, slot * kLatBytes + c * 128 * 128 + ks * 32),
                            sdesc_add(dq, (2 * u + c) * kQChunk + ks * 32), id_s, (u | c | ks) != 0);
          }
          if (!ok) break;
          {
            const int slot = gb % kNTail;
            if (!(ok = mbar_wait(bar_addr(sb, TAIL_FULL + slot), (gb / kNTail) & 1, abort_flag, p.status))) break;
            fence_proxy_async_smem();
            tc_fence_after();
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
              mma_bf16_ss(tmem + TM_S + 16 * b, sdesc_add(dtail, slot * kTailBytes + ks * 32),
                          sdesc_add(dq, 8 * kQChunk + ks * 32), id_s, 1);
            mma_commit(bar_addr(sb, TAIL_EMPTY + slot));
          }
          mma_commit(bar_addr(sb, S_FULL + b));
          if (i + 1 == nb) mma_commit(bar_addr(sb, Q_EMPTY));   // q may take the next token's rows
          // PV of this block as soon as its P is written: the five latent units hold one
          // block and the first unit of the next, so the next block's scores can only
          // proceed once this PV has handed its units back
          if (!(ok = issue_pv(gb, i, k))) break;
        }
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ one thread per slot
    const int q4 = warp & 3;
    const int ws = (warp - kSmWarp0);      // 0..3: index of this warp among the slot warps
    const int L = 32 * q4 + lane;          // TMEM lane: slot (scores) or dim within a tile (O^T)
    const uint32_t tl = tmem + ((uint32_t)(32 * q4) << 16);
    float* rmax = reinterpret_cast<float*>(smem + SM_RMAX);
    float* rsum = reinterpret_cast<float*>(smem + SM_RSUM);
    uint8_t* pt = smem + SM_PT;
    const int pchunk = L >> 6, pbyte = (L & 63) * 2;   // slot L along K of the P^T rows
    int gb = 0;
    bool ok = true;
    for (int k = 0; ok && k < ntok; ++k) {
      const int t = p.t0 + (int)blockIdx.x + k * (int)gridDim.x;
      const int nb = read_token<true>(p, sb, smem, k, abort_flag);
      if (!(ok = nb >= 0)) break;
      float m_run[kHN], l[kHN], l_bf[kHN];
#pragma unroll
      for (int h = 0; h < kHN; ++h) { m_run[h] = -INFINITY; l[h] = 0.f; l_bf[h] = 0.f; }
      for (int i = 0; ok && i < nb; ++i, ++gb) {
        const int b = gb & 1;
        if (!(ok = __all_sync(0xffffffffu, mbar_wait(bar_addr(sb, S_FULL + b), (gb >> 1) & 1, abort_flag, p.status))))
          break;
        tc_fence_after();
        float s[kHN];
        tmem_ld16(tl + TM_S + 16 * b, s);
        tc_fence_before();
        mbar_arrive(bar_addr(sb, S_FREE + b));
        const int mr = gb % kMaskRing;
        if (!(ok = __all_sync(0xffffffffu, mbar_wait(bar_addr(sb, M_FULL + mr), (gb / kMaskRing) & 1, abort_flag,
                                                     p.status))))
          break;
        const bool valid = (reinterpret_cast<volatile uint32_t*>(smem + SM_MASK + 16 * mr)[L >> 5] >> (L & 31)) & 1u;
        mbar_arrive(bar_addr(sb, M_EMPTY + mr));
        // block maximum of each head over the 128 slots
        float mx[kHN];
#pragma unroll
        for (int h = 0; h < kHN; ++h) {
          s[h] = valid ? s[h] * p.c2 : -INFINITY;
          mx[h] = s[h];
        }
        static_assert(kHN == 16, "lane L holds head L >> 1 after the transposed reduction");
        const float mxl = warp_reduce_t<kHN, true>(mx, lane);
        if ((lane & 1) == 0) rmax[ws * kHN + (lane >> 1)] = mxl;
        named_bar_sync(kSmBar, 128);
        float alpha[kHN], msub[kHN];
        bool moved = false;
#pragma unroll
        for (int h = 0; h < kHN; ++h) {
          const float bm = fmaxf(fmaxf(rmax[h], rmax[kHN + h]), fmaxf(rmax[2 * kHN + h], rmax[3 * kHN + h]));
          // lazily updated running max: moves only when the block max exceeds it by > 8 (log2 units)
          const bool mv = bm > m_run[h] + kLazyRescale;
          const float m_new = mv ? bm : m_run[h];
          alpha[h] = mv ? ex2(m_run[h] - m_new) : 1.f;   // m_run = -inf gives 0 (no O yet)
          moved |= mv && i > 0;
          m_run[h] = m_new;
          msub[h] = m_new == -INFINITY ? 0.f : m_new;   // a listed block has a valid slot; the guard keeps exp2(-inf + inf) out
        }
        float ps[2 * kHN];
        uint16_t pb[kHN];
#pragma unroll
        for (int h = 0; h < kHN; ++h) {
          const float pv = ex2(s[h] - msub[h]);         // -inf -> 0
          const uint32_t pk = pack_bf16x2(pv, 0.f);
          pb[h] = (uint16_t)(pk & 0xffffu);
          ps[h] = pv;
          ps[kHN + h] = bf16_lo(pk);                    // the weight the PV MMA actually uses
        }
        rsum[ws * 2 * kHN + lane] = warp_reduce_t<2 * kHN, false>(ps, lane);   // lane L: value L
        named_bar_sync(kSmBar, 128);
#pragma unroll
        for (int h = 0; h < kHN; ++h) {
          const float bs = (rsum[h] + rsum[2 * kHN + h]) + (rsum[4 * kHN + h] + rsum[6 * kHN + h]);
          const float bb = (rsum[kHN + h] + rsum[3 * kHN + h]) + (rsum[5 * kHN + h] + rsum[7 * kHN + h]);
          l[h] = l[h] * alpha[h] + bs;
          l_bf[h] = l_bf[h] * alpha[h] + bb;
        }
        // P^T of the previous block has been read (and O^T written) once its PV completed
        if (gb >= 1 && !(ok = __all_sync(0xffffffffu, mbar_wait(bar_addr(sb, PV_DONE), (gb - 1) & 1, abort_flag,
                                                                   p.status))))
          break;
        tc_fence_after();
        if (moved) {                        // uniform: every thread holds the same maxima
          float o[64];
          tmem_ld64(tl + TM_O, o);
#pragma unroll
          for (int u = 0; u < 4; ++u)
#pragma unroll
            for (int h = 0; h < kHN; ++h) o[16 * u + h] *= alpha[h];
          tmem_st64(tl + TM_O, o);
          tmem_wait_st();
        }
#pragma unroll
        for (int h = 0; h < kHN; ++h)
          *reinterpret_cast<uint16_t*>(pt + pchunk * kQChunk + h * 128 + ((((pbyte >> 4) ^ (h & 7))) << 4) + (pbyte & 15)) =
              pb[h];
        fence_proxy_async_smem();          // the PV MMA reads P^T through the async proxy
        tc_fence_before();
        mbar_arrive(bar_addr(sb, P_FULL));
      }
      if (!ok) break;
      // epilogue: out[t, h, d] = O^T[d, h] / l_bf[h]; lane L holds dim L of each 128-dim tile
      if (nb > 0 && !(ok = __all_sync(0xffffffffu, mbar_wait(bar_addr(sb, PV_DONE), (gb - 1) & 1, abort_flag,
                                                               p.status))))
        break;
      tc_fence_after();
      float o[64];
      if (nb > 0) {
        tmem_ld64(tl + TM_O, o);
      } else {
#pragma unroll
        for (int c = 0; c < 64; ++c) o[c] = 0.f;
      }
      tc_fence_before();
      mbar_arrive(bar_addr(sb, O_FREE));
#pragma unroll
      for (int h = 0; h < kHN; ++h) {
        if (h < p.H) {
          const float inv = 1.f / fmaxf(l_bf[h], kSumexpFloor);
          uint16_t* orow = p.out + ((int64_t)t * p.H + h) * kDv + L;
#pragma unroll
          for (int u = 0; u < 4; ++u) orow[128 * u] = (uint16_t)(pack_bf16x2(o[16 * u + h] * inv, 0.f) & 0xffffu);
        }
      }
      if (L < p.H) {
        float lh = l[0], mh = m_run[0];
#pragma unroll
        for (int h = 1; h < kHN; ++h) {
          lh = L == h ? l[h] : lh;
          mh = L == h ? m_run[h] : mh;
        }
        p.lse[(int64_t)t * p.H + L] = lh > 0.f ? (mh + log2f(lh)) * kLn2 : kLseEmpty;
      }
    }
  }

  // ------------------------------------------------------------ teardown
  if (*abort_flag) __nanosleep(1000000);   // let copies and MMAs already issued land
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

uint32_t* tc_status_ptr();

cudaError_t launch_fwd_tc_small(const FwdArgs& a, cudaStream_t s) {
  uint32_t* status = tc_status_ptr();
  if (!status) return cudaErrorInvalidSymbol;
  if (a.H > kHN) return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(tc_fwd_small_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  const int nt = a.nt < 0 ? a.T : a.nt;
  if (nt == 0) return cudaSuccess;
  int dev = 0, nsm = 0;
  e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const int grid = nt < nsm ? nt : nsm;    // persistent: one CTA per SM
  SmallFwdParams p{a.q, a.kv, a.indices, a.out, a.lse, status, a.T, a.H, a.topk, a.t0, nt, a.scale * kLog2e};
  tc_fwd_small_kernel<<<dim3(grid), dim3(kThreads), kSmemBytes, s>>>(p);
  return cudaGetLastError();
}

}  // namespace smla
