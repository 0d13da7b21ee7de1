// Tensor-core (tcgen05) backward for small head counts (H <= 16).
//
// As in the small-head forward, the top-k slots of a block are the M = 128
// rows of the score products and the heads the N = 16 columns (heads past H
// are zero q / dO rows with lse = +inf, so their P and dS' are exactly 0).  One
// CTA per SM walks a strided list of query tokens; q and dO of the token sit
// in shared memory, every gathered KV row is read once, and no partial result
// crosses between CTAs.
//
// Per block of 128 top-k slots:
//   producers : masked 16-byte cp.async gather of the 128 named rows into four
//               latent units (128 rows x 128 dims, 32 KiB) and one tail unit
//               (the 64 rope dims); padding slots copy zero bytes; the block's
//               row list goes into a small ring for the slot and drain threads;
//   MMA       : S^T = K q^T and dP^T = V dO^T (M = 128 slots, N = 16 heads)
//               into TMEM;
//   slots     : one thread per slot: P = exp2(S*scale*log2e - lse*log2e)
//               (0 on padding slots), dS' = scale * P * (dP - Delta), each as a
//               bf16 pair hi + lo (x - hi rounded again, about 16 significant
//               bits), stored as the slot's 128-byte row [dS'_hi | dS'_lo |
//               P_hi | P_lo] and, for dQ, transposed (rows = hi and lo heads);
//   MMA       : dQ^T[d, h] += K^T dS'^T (M = 128 dims per tile, N = 32 = hi and
//               lo heads, K = 128 slots) into TMEM across the token's blocks; the
//               gathered units are then free.  dKV^T[d, j] = q^T (dS'_hi + dS'_lo)
//               + dO^T (P_hi + P_lo) (M = 128 dims, N = 64 slots, K = 16 heads,
//               hi and lo as two K steps), ten tiles per block (five 128-dim
//               ranges x two halves of the slots) through four TMEM buffers;
//   drain     : the drain warps (even tiles) and the slot warps (odd tiles, after
//               handing over P / dS'), four warps per set, one per TMEM lane
//               quarter (a dim each): load a whole tile, hand the buffer back at
//               once, transpose 4 x 4 lane groups and issue
//               16-byte fp32 reductions into the rows the valid slots name
//               (padding slots issue no write).  Deterministic mode: the rows
//               are stored per slot instead.
//   epilogue  : at the end of a token dq = dQ^T (hi + lo columns) as bf16.
#include <cuda.h>

#include "smla_common.cuh"
#include "tc_common.cuh"

namespace smla {
namespace {

using namespace tc;

constexpr int kBS = 128;                // slots per block
constexpr int kHN = 16;                 // heads as the N dimension
constexpr int kProducers = 128;         // warps 0..3 gather
constexpr int kMmaWarp = 4;             // warp 4, lane 0: MMA issuer; the warp owns TMEM
constexpr int kSlotWarp0 = 5;           // warps 5..8: one thread per slot; dq epilogue
constexpr int kDrainWarp0 = 9;          // warps 9..12: dKV drain
constexpr int kThreads = 416;
constexpr int kRowsPerThread = kBS * 8 / kProducers;   // 8 rows, one 16-byte piece of each chunk
constexpr int kRing = 4;                // block row lists in flight
constexpr int kMaxBlocks = kTcMaxTopk / 64;
constexpr int kProdBar = 1;

constexpr int kLatBytes = 2 * 128 * 128;
constexpr int kTailBytes = 128 * 128;
constexpr int kNLat = 4, kNTail = 2;    // one block's latent units; two tail units
constexpr int kQChunk = kHN * 128;      // one 64-dim chunk of 16 head rows

constexpr int SM_LAT = 0;
constexpr int SM_TAIL = SM_LAT + kNLat * kLatBytes;
constexpr int SM_Q = SM_TAIL + kNTail * kTailBytes;        // 9 chunks of q
constexpr int SM_DO = SM_Q + 9 * kQChunk;                  // 8 chunks of dO
constexpr int SM_ROWS = SM_DO + 8 * kQChunk;               // 128 slot rows [dS'_hi|dS'_lo|P_hi|P_lo], 16 KiB
constexpr int SM_DST = SM_ROWS + kBS * 128;                // dS'^T: 2 chunks (64 slots) x 32 rows (hi, lo heads)
constexpr int SM_RLIST = SM_DST + 2 * 32 * 128;            // kRing x 128 row indices
constexpr int SM_RBASE = SM_RLIST + kRing * kBS * 4;          // kRing x first slot of the block
constexpr int SM_TOK = SM_RBASE + kRing * 4;
constexpr int SM_BFLAG = SM_TOK + 16;
constexpr int SM_BLIST = SM_BFLAG + kMaxBlocks;
constexpr int SM_NB = SM_BLIST + 2 * kMaxBlocks;
constexpr int SM_BAR = (SM_NB + 8 + 7) & ~7;
enum Bar { LAT_FULL = 0, LAT_EMPTY = kNLat, TAIL_FULL = 2 * kNLat, TAIL_EMPTY = TAIL_FULL + kNTail,
           QD_FULL = TAIL_EMPTY + kNTail, QD_EMPTY, RL_FULL, RL_EMPTY = RL_FULL + kRing, SD_FULL = RL_EMPTY + kRing,
           SD_FREE, P_FULL, PDS_FREE, DQ_DONE, DQ_FREE, DKV_FULL, DKV_FREE = DKV_FULL + 4, TOK_FULL = DKV_FREE + 4,
           TOK_EMPTY = TOK_FULL + 2, NBAR = TOK_EMPTY + 2 };
constexpr int SM_TMEM = SM_BAR + 8 * NBAR;
constexpr int SM_ABORT = SM_TMEM + 4;
constexpr int kSmemBytes = SM_ABORT + 4 + 1024;
static_assert(kSmemBytes <= 232448, "shared memory budget");
static_assert(SM_TAIL % 1024 == 0 && SM_Q % 1024 == 0 && SM_DO % 1024 == 0 && SM_ROWS % 1024 == 0 &&
                  SM_DST % 1024 == 0,
              "swizzle atoms");

// TMEM: S^T and dP^T (16 columns each), dQ^T as five 32-column tiles (hi | lo
// heads; the fifth holds the rope dims in lanes 0..63), four 64-column dKV^T buffers
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t TM_S = 0, TM_DP = 16, TM_DQ = 64, TM_DKV = 256;

struct SmallBwdParams {
  const uint16_t* q;
  const uint16_t* kv;
  const uint16_t* dout;
  const float* lse;
  const float* delta;
  const int32_t* indices;
  uint16_t* dq;
  float* dkv32;
  float* gbuf;                          // deterministic mode: per-slot contributions of this launch's tokens
  uint32_t* status;
  int T, H, topk, t0, nt;
  float scale, c2;
};

__device__ __forceinline__ uint32_t bar_addr(uint32_t base, int i) { return base + SM_BAR + 8 * i; }
__device__ __forceinline__ void named_bar_sync(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}
__device__ __forceinline__ int cta_tokens(const SmallBwdParams& p) {
  return (int)blockIdx.x < p.nt ? (p.nt - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
}

template <bool kWarp>
__device__ __forceinline__ int read_token(const SmallBwdParams& p, uint32_t sb, uint8_t* smem, int k,
                                          volatile int* abort_flag) {
  const bool ok = kWarp ? __all_sync(0xffffffffu, mbar_wait(bar_addr(sb, TOK_FULL + (k & 1)), (k >> 1) & 1, abort_flag,
                                                            p.status))
                        : mbar_wait(bar_addr(sb, TOK_FULL + (k & 1)), (k >> 1) & 1, abort_flag, p.status);
  if (!ok) return -1;
  const int nb = reinterpret_cast<volatile int*>(smem + SM_TOK)[k & 1];
  mbar_arrive(bar_addr(sb, TOK_EMPTY + (k & 1)));
  return nb;
}

// 4 x 4 transpose among the four lanes 4a + b (b = lane & 3): on entry lane
// 4a + r holds x[c] = M[r][c]; on return y[r] = M[r][b].
__device__ __forceinline__ void transpose4(float x0, float x1, float x2, float x3, int b, float* y) {
  const bool o1 = b & 1;
  const float r0 = __shfl_xor_sync(0xffffffffu, o1 ? x0 : x1, 1);
  const float r1 = __shfl_xor_sync(0xffffffffu, o1 ? x2 : x3, 1);
  const float t0 = o1 ? r0 : x0, t1 = o1 ? x1 : r0, t2 = o1 ? r1 : x2, t3 = o1 ? x3 : r1;
  const bool o2 = b & 2;
  const float v0 = __shfl_xor_sync(0xffffffffu, o2 ? t0 : t2, 2);
  const float v1 = __shfl_xor_sync(0xffffffffu, o2 ? t1 : t3, 2);
  y[0] = o2 ? v0 : t0;
  y[1] = o2 ? v1 : t1;
  y[2] = o2 ? t2 : v0;
  y[3] = o2 ? t3 : v1;
}

// Drains dKV^T tile tt of block gb (dims 128 (tt / 2).., slots 64 (tt % 2)..) by
// one set of four warps (one per TMEM lane quarter: dim L of the tile): loads
// the tile's 64 slot columns, hands the TMEM buffer back, then adds each valid
// slot's value into its kv row (4 x 4 lane transposes, 16-byte reductions), or
// stores it per slot in the deterministic mode.  rows[c]: lane k holds the row
// of slot 32 c + k of the block (-1 for padding).
__device__ __forceinline__ bool drain_tile(const SmallBwdParams& p, uint32_t sb, uint32_t tl, int L, int lane,
                                           int gb, int tt, const int (&rows)[4], float* gblk,
                                           volatile int* abort_flag) {
  const int n = 10 * gb + tt;               // tiles issued so far
  const int bb = n & 3, m = tt >> 1, hh = tt & 1, b4 = lane & 3;
  if (!__all_sync(0xffffffffu, mbar_wait(bar_addr(sb, DKV_FULL + bb), (n >> 2) & 1, abort_flag, p.status)))
    return false;
  tc_fence_after();
  float g[64];                               // the tile's 64 slots of this dim
  tmem_ld64(tl + TM_DKV + 64 * bb, g);
  tc_fence_before();
  mbar_arrive(bar_addr(sb, DKV_FREE + bb));  // the MMA may overwrite this buffer
  const int d = 128 * m + L;                 // dims 512..575 in the last range: lanes 0..63
  if (d < kDqk) {                            // warp-uniform
    const int d4 = d - b4;
#pragma unroll
    for (int c = 0; c < 2; ++c) {
#pragma unroll
      for (int gq = 0; gq < 8; ++gq) {
        float y[4];
        transpose4(g[32 * c + 4 * gq], g[32 * c + 4 * gq + 1], g[32 * c + 4 * gq + 2], g[32 * c + 4 * gq + 3], b4, y);
        const int kk = 4 * gq + b4;
        const int rsrc = c == 0 ? (hh ? rows[2] : rows[0]) : (hh ? rows[3] : rows[1]);
        const int row = __shfl_sync(0xffffffffu, rsrc, kk);
        if (row < 0) continue;
        if (gblk != nullptr) {
          float* dst = gblk + (int64_t)(64 * hh + 32 * c + kk) * kDqk + d4;
          if (check_range(dst, 4, p.gbuf, (int64_t)p.nt * p.topk * kDqk, p.status))
            *reinterpret_cast<float4*>(dst) = make_float4(y[0], y[1], y[2], y[3]);
        } else {
          float* dst = p.dkv32 + (int64_t)row * kDqk + d4;
          if (check_range(dst, 4, p.dkv32, (int64_t)p.T * kDqk, p.status)) red_add_v4(dst, y[0], y[1], y[2], y[3]);
        }
      }
    }
  }
  return true;
}

// Producers: per token, list the blocks of 128 slots that hold a valid slot,
// publish the count, gather q and dO (rows H..15 zero), then each block's rows
// unit by unit, and the block's row list (-1 for padding) into the row ring.
__device__ __forceinline__ void produce(const SmallBwdParams& p, uint32_t sb, uint8_t* smem, volatile int* abort_flag) {
  const int pt = threadIdx.x;              // 0..127
  const int warp = pt >> 5, lane = pt & 31;
  const int c16 = pt & 7, r0 = pt >> 3;
  constexpr int R = kRowsPerThread;
  const int nblk = (p.topk + kBS - 1) / kBS;
  const int ntok = cta_tokens(p);
  uint8_t* flag = smem + SM_BFLAG;
  int16_t* blist = reinterpret_cast<int16_t*>(smem + SM_BLIST);
  volatile int* nbs = reinterpret_cast<volatile int*>(smem + SM_NB);
  volatile int* tok = reinterpret_cast<volatile int*>(smem + SM_TOK);
  int* rlist = reinterpret_cast<int*>(smem + SM_RLIST);
  const uint16_t* kvc = p.kv + 8 * c16;
  int nl = 0, gb = 0, kq = 0;
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
    if (nb < 0) return;
    bool ok = true;
    if (nb == 0) continue;                 // no product reads q / dO for this token
    if (kq >= 1 && !(ok = __all_sync(0xffffffffu, mbar_wait(bar_addr(sb, QD_EMPTY), (kq - 1) & 1, abort_flag,
                                                              p.status))))
      return;
    ++kq;
    {
      const int h = r0;                    // 16 rows, one per group of 8 threads
      const bool real = h < p.H;
      const uint16_t* qsrc = p.q + ((int64_t)t * p.H + (real ? h : 0)) * kDqk + 8 * c16;
      const uint16_t* dsrc = p.dout + ((int64_t)t * p.H + (real ? h : 0)) * kDv + 8 * c16;
      const uint32_t o = h * 128 + ((c16 ^ (h & 7)) << 4);
#pragma unroll
      for (int c = 0; c < 9; ++c)
        gather16(sb + SM_Q + c * kQChunk + o, qsrc + 64 * c, real ? 16u : 0u, p.q, (int64_t)p.T * p.H * kDqk, p.status);
#pragma unroll
      for (int c = 0; c < 8; ++c)
        gather16(sb + SM_DO + c * kQChunk + o, dsrc + 64 * c, real ? 16u : 0u, p.dout, (int64_t)p.T * p.H * kDv,
                 p.status);
      cp_async_arrive(bar_addr(sb, QD_FULL));
    }
    int nxt[R], nrl[4];
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
          nrl[w] = slot < p.topk ? __ldg(irow + slot) : -1;
        }
      }
    };
    if (nb > 0) fetch(0);
    for (int i = 0; ok && i < nb; ++i, ++gb) {
      int cur[R], crl[4];
#pragma unroll
      for (int j = 0; j < R; ++j) cur[j] = nxt[j];
#pragma unroll
      for (int w = 0; w < 4; ++w) crl[w] = nrl[w];
      if (i + 1 < nb) fetch(i + 1);
      if (warp == 0) {                     // the block's row list (-1: padding) for the slot and drain threads
        const int rr = gb % kRing;
        if (gb >= kRing &&
            !(ok = __all_sync(0xffffffffu, mbar_wait(bar_addr(sb, RL_EMPTY + rr), ((gb / kRing) - 1) & 1, abort_flag,
                                                     p.status))))
          break;
#pragma unroll
        for (int w = 0; w < 4; ++w)
          rlist[rr * kBS + 32 * w + lane] = (crl[w] >= 0 && crl[w] < p.T) ? crl[w] : -1;
        if (lane == 0) reinterpret_cast<int*>(smem + SM_RBASE)[rr] = blist[i] * kBS;
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_addr(sb, RL_FULL + rr));
      }
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
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
      for (int u = 0; u < 4; ++u, ++nl) {
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
      const int ts = gb % kNTail;
      if (gb >= kNTail &&
          !(ok = __all_sync(0xffffffffu, mbar_wait(bar_addr(sb, TAIL_EMPTY + ts), ((gb / kNTail) - 1) & 1, abort_flag,
                                                   p.status))))
        break;
      const uint32_t tunit = sb + SM_TAIL + ts * kTailBytes;
#pragma unroll
      for (int j = 0; j < R; ++j) gather16(tunit + dsto[j], src[j] + 512, nbytes[j], p.kv, (int64_t)p.T * kDqk, p.status);
      cp_async_arrive(bar_addr(sb, TAIL_FULL + ts));
    }
    if (!ok) return;
  }
}

__global__ void __launch_bounds__(kThreads, 1) tc_bwd_small_kernel(SmallBwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sb = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ntok = cta_tokens(p);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + SM_ABORT);

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    for (int k = 0; k < kNLat; ++k) {
      mbar_init(bar_addr(sb, LAT_FULL + k), kProducers);
      mbar_init(bar_addr(sb, LAT_EMPTY + k), 1);         // the dQ MMAs (the unit's last reader) completed
    }
    for (int k = 0; k < kNTail; ++k) {
      mbar_init(bar_addr(sb, TAIL_FULL + k), kProducers);
      mbar_init(bar_addr(sb, TAIL_EMPTY + k), 1);
    }
    mbar_init(bar_addr(sb, QD_FULL), kProducers);
    mbar_init(bar_addr(sb, QD_EMPTY), 1);                // the token's last dKV MMAs completed
    for (int k = 0; k < kRing; ++k) {
      mbar_init(bar_addr(sb, RL_FULL + k), 1);
      mbar_init(bar_addr(sb, RL_EMPTY + k), 128 + 128);  // slot threads and drain threads read it
    }
    mbar_init(bar_addr(sb, SD_FULL), 1);
    mbar_init(bar_addr(sb, SD_FREE), 128);
    mbar_init(bar_addr(sb, P_FULL), 128);
    mbar_init(bar_addr(sb, PDS_FREE), 1);
    mbar_init(bar_addr(sb, DQ_DONE), 1);
    mbar_init(bar_addr(sb, DQ_FREE), 128);
    for (int b = 0; b < 4; ++b) {
      mbar_init(bar_addr(sb, DKV_FULL + b), 1);
      mbar_init(bar_addr(sb, DKV_FREE + b), 128);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar_addr(sb, TOK_FULL + b), 1);
      mbar_init(bar_addr(sb, TOK_EMPTY + b), 1 + 128 + 128);   // MMA thread, slot threads, drain threads
    }
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
      const uint32_t id_sd = idesc_bf16(128, kHN, false, false);        // A = K / V rows, B = q / dO rows (K-major)
      const uint32_t id_dq = idesc_bf16(128, 2 * kHN, true, false);     // A = K^T (MN-major), B = dS'^T (K-major)
      const uint32_t id_dkv = idesc_bf16(128, kBS / 2, true, false);    // A = q^T / dO^T (MN-major), B = 64 slot rows
      const uint64_t dlat = sdesc_sw128(sb + SM_LAT, 16, 1024);
      const uint64_t dlatt = sdesc_sw128(sb + SM_LAT, 128 * 128, 1024);
      const uint64_t dtail = sdesc_sw128(sb + SM_TAIL, 16, 1024);
      const uint64_t dtailt = sdesc_sw128(sb + SM_TAIL, 128 * 128, 1024);
      const uint64_t dq = sdesc_sw128(sb + SM_Q, 16, 1024);
      const uint64_t ddo = sdesc_sw128(sb + SM_DO, 16, 1024);
      const uint64_t dqt = sdesc_sw128(sb + SM_Q, kQChunk, 1024);       // q^T: 64-dim groups one chunk apart
      const uint64_t ddot = sdesc_sw128(sb + SM_DO, kQChunk, 1024);
      const uint64_t drows = sdesc_sw128(sb + SM_ROWS, 16, 1024);
      const uint64_t ddst = sdesc_sw128(sb + SM_DST, 16, 1024);
      int gb = 0, nl = 0, kq = 0, nt2 = 0;   // blocks; latent units; tokens with blocks; dKV tiles issued
      bool ok = true;
      for (int k = 0; ok && k < ntok; ++k) {
        const int nb = read_token<false>(p, sb, smem, k, abort_flag);
        if (!(ok = nb >= 0)) break;
        if (nb == 0) continue;
        if (!(ok = mbar_wait(bar_addr(sb, QD_FULL), kq & 1, abort_flag, p.status))) break;
        // dQ^T is free once the previous token's epilogue read it
        if (kq >= 1 && !(ok = mbar_wait(bar_addr(sb, DQ_FREE), (kq - 1) & 1, abort_flag, p.status))) break;
        ++kq;
        for (int i = 0; ok && i < nb; ++i, ++gb) {
          // S^T and dP^T of this block once the slot threads hold the previous block's
          if (gb >= 1 && !(ok = mbar_wait(bar_addr(sb, SD_FREE), (gb - 1) & 1, abort_flag, p.status))) break;
          const int nl0 = nl;
#pragma unroll 1
          for (int u = 0; u < 4; ++u, ++nl) {
            const int slot = nl % kNLat;
            if (!(ok = mbar_wait(bar_addr(sb, LAT_FULL + slot), (nl / kNLat) & 1, abort_flag, p.status))) break;
            fence_proxy_async_smem();      // cp.async wrote the unit through the generic proxy
            tc_fence_after();
#pragma unroll
            for (int c = 0; c < 2; ++c)
#pragma unroll
              for (int ks = 0; ks < 4; ++ks) {
                const uint64_t a = sdesc_add(dlat, slot * kLatBytes + c * 128 * 128 + ks * 32);
                mma_bf16_ss(tmem + TM_S, a, sdesc_add(dq, (2 * u + c) * kQChunk + ks * 32), id_sd, (u | c | ks) != 0);
                mma_bf16_ss(tmem + TM_DP, a, sdesc_add(ddo, (2 * u + c) * kQChunk + ks * 32), id_sd, (u | c | ks) != 0);
              }
          }
          if (!ok) break;
          const int ts = gb % kNTail;
          if (!(ok = mbar_wait(bar_addr(sb, TAIL_FULL + ts), (gb / kNTail) & 1, abort_flag, p.status))) break;
          fence_proxy_async_smem();
          tc_fence_after();
#pragma unroll
          for (int ks = 0; ks < 4; ++ks)
            mma_bf16_ss(tmem + TM_S, sdesc_add(dtail, ts * kTailBytes + ks * 32), sdesc_add(dq, 8 * kQChunk + ks * 32),
                        id_sd, 1);
          mma_commit(bar_addr(sb, SD_FULL));
          // the slot threads wrote this block's P / dS' rows
          if (!(ok = mbar_wait(bar_addr(sb, P_FULL), gb & 1, abort_flag, p.status))) break;
          tc_fence_after();
          // dQ^T += K^T dS'^T: four latent tiles, then the rope dims (lanes 0..63 of the fifth tile;
          // its other lanes read the next 16 KiB of shared memory and are never used)
#pragma unroll 1
          for (int u = 0; u < 4; ++u) {
            const int slot = (nl0 + u) % kNLat;
#pragma unroll
            for (int ks = 0; ks < 8; ++ks)
              mma_bf16_ss(tmem + TM_DQ + 32 * u, sdesc_add(dlatt, slot * kLatBytes + ks * 16 * 128),
                          sdesc_add(ddst, (ks >> 2) * 32 * 128 + (ks & 3) * 32), id_dq, (i > 0 || ks > 0));
            mma_commit(bar_addr(sb, LAT_EMPTY + slot));
          }
#pragma unroll
          for (int ks = 0; ks < 8; ++ks)
            mma_bf16_ss(tmem + TM_DQ + 128, sdesc_add(dtailt, ts * kTailBytes + ks * 16 * 128),
                        sdesc_add(ddst, (ks >> 2) * 32 * 128 + (ks & 3) * 32), id_dq, (i > 0 || ks > 0));
          mma_commit(bar_addr(sb, TAIL_EMPTY + ts));
          if (i + 1 == nb) mma_commit(bar_addr(sb, DQ_DONE));
          // dKV^T tiles (dims 128 m.., slots 64 hh..): q^T (dS'_hi + dS'_lo)
          // [+ dO^T (P_hi + P_lo) inside the value range]
#pragma unroll 1
          for (int tt = 0; tt < 10; ++tt, ++nt2) {
            const int m = tt >> 1, hh = tt & 1;
            const int bb = nt2 & 3;
            if (nt2 >= 4 && !(ok = mbar_wait(bar_addr(sb, DKV_FREE + bb), ((nt2 >> 2) - 1) & 1, abort_flag, p.status)))
              break;
            tc_fence_after();
            const uint32_t d_t = tmem + TM_DKV + 64 * bb;
            const uint64_t rb = sdesc_add(drows, hh * 64 * 128);
            mma_bf16_ss(d_t, sdesc_add(dqt, 2 * m * kQChunk), rb, id_dkv, 0);
            mma_bf16_ss(d_t, sdesc_add(dqt, 2 * m * kQChunk), sdesc_add(rb, 32), id_dkv, 1);
            if (m < 4) {
              mma_bf16_ss(d_t, sdesc_add(ddot, 2 * m * kQChunk), sdesc_add(rb, 64), id_dkv, 1);
              mma_bf16_ss(d_t, sdesc_add(ddot, 2 * m * kQChunk), sdesc_add(rb, 96), id_dkv, 1);
            }
            mma_commit(bar_addr(sb, DKV_FULL + bb));
          }
          if (!ok) break;
          mma_commit(bar_addr(sb, PDS_FREE));
          if (i + 1 == nb) mma_commit(bar_addr(sb, QD_EMPTY));   // q / dO may take the next token's rows
        }
      }
    }
    __syncwarp();
  } else if (warp < kDrainWarp0) {
    // ------------------------------------------------------------ one thread per slot
    const int q4 = warp & 3;
    const int L = 32 * q4 + lane;          // TMEM lane: slot (S^T, dP^T) or dim within a tile (dQ^T)
    const uint32_t tl = tmem + ((uint32_t)(32 * q4) << 16);
    const int* rlist = reinterpret_cast<const int*>(smem + SM_RLIST);
    uint8_t* rowp = smem + SM_ROWS + L * 128;
    const int sw = L & 7;
    uint8_t* dst = smem + SM_DST + (L >> 6) * 32 * 128;
    const int pbyte = (L & 63) * 2;
    int gb = 0, kqs = 0;                   // blocks; tokens with blocks
    bool ok = true;
    for (int k = 0; ok && k < ntok; ++k) {
      const int t = p.t0 + (int)blockIdx.x + k * (int)gridDim.x;
      const int nb = read_token<true>(p, sb, smem, k, abort_flag);
      if (!(ok = nb >= 0)) break;
      float lse2[kHN], dl[kHN];
#pragma unroll
      for (int h = 0; h < kHN; ++h) {
        const bool real = h < p.H;
        lse2[h] = real ? p.lse[(int64_t)t * p.H + h] * kLog2e : INFINITY;   // heads past H: P = 0
        dl[h] = real ? p.delta[(int64_t)t * p.H + h] : 0.f;
      }
      for (int i = 0; ok && i < nb; ++i, ++gb) {
        if (!(ok = __all_sync(0xffffffffu, mbar_wait(bar_addr(sb, SD_FULL), gb & 1, abort_flag, p.status)))) break;
        tc_fence_after();
        float s[kHN], dp[kHN];
        tmem_ld16(tl + TM_S, s);
        tmem_ld16(tl + TM_DP, dp);
        tc_fence_before();
        mbar_arrive(bar_addr(sb, SD_FREE));
        const int rr = gb % kRing;
        if (!(ok = __all_sync(0xffffffffu, mbar_wait(bar_addr(sb, RL_FULL + rr), (gb / kRing) & 1, abort_flag,
                                                     p.status))))
          break;
        const bool valid = reinterpret_cast<volatile const int*>(rlist)[rr * kBS + L] >= 0;
        int rows[4];                       // for the odd dKV tiles this warp set drains
#pragma unroll
        for (int c = 0; c < 4; ++c) rows[c] = reinterpret_cast<volatile const int*>(rlist)[rr * kBS + 32 * c + lane];
        const int sbase = reinterpret_cast<volatile const int*>(smem + SM_RBASE)[rr];
        mbar_arrive(bar_addr(sb, RL_EMPTY + rr));
        uint32_t dh[kHN / 2], dlo[kHN / 2], ph[kHN / 2], plo[kHN / 2];
#pragma unroll
        for (int h2 = 0; h2 < kHN / 2; ++h2) {
          const int h = 2 * h2;
          const float p0 = valid ? ex2(s[h] * p.c2 - lse2[h]) : 0.f;       // padding: P = 0 exactly
          const float p1 = valid ? ex2(s[h + 1] * p.c2 - lse2[h + 1]) : 0.f;
          ph[h2] = pack_bf16x2(p0, p1);
          plo[h2] = pack_bf16x2(p0 - bf16_lo(ph[h2]), p1 - bf16_hi(ph[h2]));
          const float d0 = p.scale * p0 * (dp[h] - dl[h]), d1 = p.scale * p1 * (dp[h + 1] - dl[h + 1]);
          dh[h2] = pack_bf16x2(d0, d1);
          dlo[h2] = pack_bf16x2(d0 - bf16_lo(dh[h2]), d1 - bf16_hi(dh[h2]));
        }
        // the previous block's dQ / dKV products have read the rows
        if (gb >= 1 && !(ok = __all_sync(0xffffffffu, mbar_wait(bar_addr(sb, PDS_FREE), (gb - 1) & 1, abort_flag,
                                                                   p.status))))
          break;
        // slot row [dS'_hi | dS'_lo | P_hi | P_lo] (128B swizzle: chunk c at (c ^ row) & 7)
        *reinterpret_cast<uint4*>(rowp + ((0 ^ sw) << 4)) = make_uint4(dh[0], dh[1], dh[2], dh[3]);
        *reinterpret_cast<uint4*>(rowp + ((1 ^ sw) << 4)) = make_uint4(dh[4], dh[5], dh[6], dh[7]);
        *reinterpret_cast<uint4*>(rowp + ((2 ^ sw) << 4)) = make_uint4(dlo[0], dlo[1], dlo[2], dlo[3]);
        *reinterpret_cast<uint4*>(rowp + ((3 ^ sw) << 4)) = make_uint4(dlo[4], dlo[5], dlo[6], dlo[7]);
        *reinterpret_cast<uint4*>(rowp + ((4 ^ sw) << 4)) = make_uint4(ph[0], ph[1], ph[2], ph[3]);
        *reinterpret_cast<uint4*>(rowp + ((5 ^ sw) << 4)) = make_uint4(ph[4], ph[5], ph[6], ph[7]);
        *reinterpret_cast<uint4*>(rowp + ((6 ^ sw) << 4)) = make_uint4(plo[0], plo[1], plo[2], plo[3]);
        *reinterpret_cast<uint4*>(rowp + ((7 ^ sw) << 4)) = make_uint4(plo[4], plo[5], plo[6], plo[7]);
        // dS'^T for dQ: row h (hi) and 16 + h (lo), this slot along K
#pragma unroll
        for (int h2 = 0; h2 < kHN / 2; ++h2) {
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int h = 2 * h2 + e;
            const uint16_t vh = (uint16_t)(e ? dh[h2] >> 16 : dh[h2] & 0xffffu);
            const uint16_t vl = (uint16_t)(e ? dlo[h2] >> 16 : dlo[h2] & 0xffffu);
            *reinterpret_cast<uint16_t*>(dst + h * 128 + ((((pbyte >> 4) ^ (h & 7))) << 4) + (pbyte & 15)) = vh;
            *reinterpret_cast<uint16_t*>(dst + (16 + h) * 128 + ((((pbyte >> 4) ^ ((16 + h) & 7))) << 4) + (pbyte & 15)) =
                vl;
          }
        }
        fence_proxy_async_smem();          // the MMAs read them through the async proxy
        tc_fence_before();
        mbar_arrive(bar_addr(sb, P_FULL));
        // this warp set drains the block's odd dKV tiles (the drain warps the even ones)
        float* gblk = p.gbuf == nullptr ? nullptr : p.gbuf + ((int64_t)(t - p.t0) * p.topk + sbase) * kDqk;
#pragma unroll 1
        for (int tt = 1; ok && tt < 10; tt += 2) ok = drain_tile(p, sb, tl, L, lane, gb, tt, rows, gblk, abort_flag);
      }
      if (!ok) break;
      // epilogue: dq[t, h, d] = dQ^T hi + lo columns; lane L holds dim L of each 128-dim tile
      // (the fifth tile: the rope dims 512 + L, lanes 0..63)
      if (nb > 0 && !(ok = __all_sync(0xffffffffu, mbar_wait(bar_addr(sb, DQ_DONE), kqs & 1, abort_flag, p.status))))
        break;
      tc_fence_after();
#pragma unroll 1
      for (int u = 0; u < 5; ++u) {
        float v[32];
        if (nb > 0) {
          tmem_ld32(tl + TM_DQ + 32 * u, v);
        } else {                           // no valid slot: dq is exactly 0
#pragma unroll
          for (int c = 0; c < 32; ++c) v[c] = 0.f;
        }
        const int d = 128 * u + L;
        if (d < kDqk) {
#pragma unroll
          for (int h = 0; h < kHN; ++h)
            if (h < p.H)
              p.dq[((int64_t)t * p.H + h) * kDqk + d] = (uint16_t)(pack_bf16x2(v[h] + v[kHN + h], 0.f) & 0xffffu);
        }
      }
      if (nb > 0) {
        tc_fence_before();
        mbar_arrive(bar_addr(sb, DQ_FREE));   // the next token's dQ products may overwrite dQ^T
        ++kqs;
      }
    }
  } else {
    // ------------------------------------------------------------ dKV drain
    const int q4 = warp & 3;
    const int L = 32 * q4 + lane;          // TMEM lane: dim within a tile
    const uint32_t tl = tmem + ((uint32_t)(32 * q4) << 16);
    const int* rlist = reinterpret_cast<const int*>(smem + SM_RLIST);
    int gb = 0;
    bool ok = true;
    for (int k = 0; ok && k < ntok; ++k) {
      const int t = p.t0 + (int)blockIdx.x + k * (int)gridDim.x;
      const int nb = read_token<true>(p, sb, smem, k, abort_flag);
      if (!(ok = nb >= 0)) break;
      for (int i = 0; ok && i < nb; ++i, ++gb) {
        const int rr = gb % kRing;
        if (!(ok = __all_sync(0xffffffffu, mbar_wait(bar_addr(sb, RL_FULL + rr), (gb / kRing) & 1, abort_flag,
                                                     p.status))))
          break;
        int rows[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) rows[c] = reinterpret_cast<volatile const int*>(rlist)[rr * kBS + 32 * c + lane];
        const int sbase = reinterpret_cast<volatile const int*>(smem + SM_RBASE)[rr];
        mbar_arrive(bar_addr(sb, RL_EMPTY + rr));
        // deterministic mode: where the contributions of this block's slots go
        float* gblk = p.gbuf == nullptr ? nullptr : p.gbuf + ((int64_t)(t - p.t0) * p.topk + sbase) * kDqk;
#pragma unroll 1
        for (int tt = 0; ok && tt < 10; tt += 2) ok = drain_tile(p, sb, tl, L, lane, gb, tt, rows, gblk, abort_flag);
      }
    }
  }

  // ------------------------------------------------------------ teardown
  if (*abort_flag) __nanosleep(1000000);
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

uint32_t* tc_status_ptr();

cudaError_t launch_bwd_tc_small(const BwdArgs& a, cudaStream_t s) {
  uint32_t* status = tc_status_ptr();
  if (!status) return cudaErrorInvalidSymbol;
  if (a.H > kHN) return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(tc_bwd_small_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  const int nt = a.nt < 0 ? a.T : a.nt;
  if (nt == 0) return cudaSuccess;
  int dev = 0, nsm = 0;
  e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const int grid = nt < nsm ? nt : nsm;
  SmallBwdParams p{a.q, a.kv, a.dout, a.lse, a.delta, a.indices, a.dq, a.dkv32, a.gbuf, status,
                   a.T, a.H, a.topk, a.t0, nt, a.scale, a.scale * kLog2e};
  tc_bwd_small_kernel<<<dim3(grid), dim3(kThreads), kSmemBytes, s>>>(p);
  return cudaGetLastError();
}

}  // namespace smla
