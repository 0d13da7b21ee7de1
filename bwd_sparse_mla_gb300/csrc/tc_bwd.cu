// Tensor-core (tcgen05) backward for up to 128 heads (fewer heads run as a
// 128-row tile whose rows past H are zero).
//
// Work split: as in the forward, a cluster of two CTAs handles one query
// token and splits the feature dimension: CTA 0 owns key dims [0,256) and
// value dims [0,256); CTA 1 owns key dims [256,576) (the rope tail included)
// and value dims [256,512).  Each CTA keeps its slice of q and dO for the
// token in shared memory, accumulates its slice of dQ (128 heads x 256|320
// dims) in TMEM, and produces its slice of every dKV row.
//
// Per block of 32 top-k slots:
//   producer : masked 16-byte cp.async gather of the CTA's columns of the 32
//              named rows, indices read one block ahead (padding slots copy
//              zero bytes: exact-zero K/V rows);
//   MMA      : S_half = q_half K_half^T and dP_half = dO_half V_half^T
//              (M=128 heads, N=32 slots) into TMEM;
//   exchange : one thread per head loads its partial S and dP rows and writes
//              them to this SM's slot of an L2 exchange scratch;
//   softmax  : one thread per head loads its own partial rows (the TMEM buffer
//              is then free for the next block's S / dP), adds the peer CTA's
//              rows read from the peer's slot (both CTAs obtain bit-identical
//              sums), recomputes
//              P = exp2(S*scale*log2e - lse*log2e) (0 on padding slots),
//              dS' = scale * P * (dP - Delta), and stores P and dS' each as
//              a bf16 pair hi + lo (x - hi rounded again), so the dQ and dKV
//              products see them to about 16 significant bits;
//   MMA      : dQ_half += (hi + lo) K_half (M=128, N=256|320, K=32) and the
//              transposed dKV tiles dKV^T[d, j] = dO^T (hi + lo) + q^T (hi + lo)
//              (M=128 dims, N=32 slots, K=128 heads);
//   drain    : four drain warps (one per TMEM lane quarter) read each dKV
//              tile from TMEM as soon as its MMAs complete, hand the tile back
//              to the MMA issuer at once (one barrier pair per tile, so the next
//              block's products for that tile overlap the reductions of the
//              rest), and add it into the fp32 dKV rows named by the valid slots
//              (coalesced 128-byte fp32 reductions; padding slots issue no
//              write, the no-op the miles PR #2079 summary describes for the
//              clamped atomic).
#include <cuda.h>

#include "smla_common.cuh"
#include "tc_common.cuh"

namespace smla {
namespace {

using namespace tc;

constexpr int kBK = 32;
constexpr int kProducers = 64;          // w0..1 gather, w2 MMA, w3..6 softmax, w7..10 exchange, w11..14 dKV drain
constexpr int kMmaWarp = 2;
constexpr int kXchgWarp0 = 7;
constexpr int kDrainWarp0 = 11;
constexpr int kThreads = 480;
constexpr int kRowsPerProducer = kBK * 8 / kProducers;   // 4
constexpr int kChunk = 128 * 128;       // 64-dim chunk of q / dO for 128 heads
constexpr int kChunkKV = kBK * 128;     // 64-dim chunk of a 32-row KV block
constexpr int kStage = 5 * kChunkKV;

constexpr int SM_Q = 0;                                 // 5 chunks
constexpr int SM_DO = SM_Q + 5 * kChunk;                // 4 chunks
constexpr int SM_KV = SM_DO + 4 * kChunk;               // 2 stages
// P and dS' of a block, each as 128 head rows of [hi (32 slots) | lo (32 slots)]
// bf16 = 128 bytes, 128B swizzle: K-major A of dQ (one half), MN-major B (N = 64)
// of the dKV products (both halves at once)
constexpr int SM_P = SM_KV + 2 * kStage;
constexpr int SM_DS = SM_P + 128 * 128;
constexpr int SM_ROWS = SM_DS + 128 * 128;              // 2 x 32 int32
constexpr int SM_MASK = SM_ROWS + 2 * 32 * 4;           // 2 x u32
constexpr int kMaxBlocks = kTcMaxTopk / kBK;
constexpr int SM_BFLAG = SM_MASK + 8;                   // per block: holds a valid slot (u8)
constexpr int SM_BLIST = SM_BFLAG + kMaxBlocks;         // blocks with a valid slot, in order (u16)
constexpr int SM_NB = SM_BLIST + 2 * kMaxBlocks;        // their number
constexpr int SM_BAR = SM_NB + 8;
enum Bar { KV_FULL = 0, KV_EMPTY = 2, QD_FULL = 4, SDP_FULL = 5, SDP_FREE = 6, X_FULL = 7, X_EMPTY = 9,
           P_FULL = 11, PDS_FREE = 12, DKV_FULL = 13, DKV_FREE = 16, NBAR = 19 };   // DKV_*: one per tile
constexpr int SM_TMEM = SM_BAR + 8 * NBAR;
constexpr int SM_SMID = SM_TMEM + 8;
constexpr int SM_ABORT = SM_SMID + 4;
constexpr int kSmemBytes = SM_ABORT + 4 + 1024;
static_assert(SM_P % 1024 == 0 && SM_DS % 1024 == 0, "swizzle atoms");
static_assert(kSmemBytes > 232448 / 2, "one CTA per SM: the exchange scratch is indexed by SM");
static_assert(kSmemBytes <= 232448, "shared memory budget");

constexpr uint32_t kTmemCols = 512;
// TMEM columns: dQ [0, ndq), S [ndq, +32), dP [ndq+32, +32), then the dKV^T
// tiles (64 columns each: hi half | lo half); 256+64+3*64 = 320+64+2*64 = 512
constexpr uint32_t TM_DQ = 0;

struct TcBwdParams {
  const uint16_t* kv;
  float* xchg;                          // exchange scratch, kXchgSlots slots
  const int32_t* indices;
  const float* lse;
  const float* delta;
  uint16_t* dq;
  float* dkv32;
  float* gbuf;                          // deterministic mode: per-slot contributions of this launch's tokens
  uint32_t* status;
  int T, H, topk, t0;                   // this launch handles tokens t0, t0 + 1, ...; H <= 128 heads
  float scale, c2;
};

__device__ __forceinline__ uint32_t bar_addr(uint32_t base, int i) { return base + SM_BAR + 8 * i; }


// 4 x 4 transpose among the four lanes 4a + b (b = lane & 3): on entry lane
// 4a + r holds x[c] = M[r][c]; on return y[r] = M[r][b].  Two butterfly
// exchanges (lane ^ 1, then lane ^ 2), two shuffles each.
__device__ __forceinline__ void transpose4(float x0, float x1, float x2, float x3, int b, float* y) {
  // step 1: pairs (b, b ^ 1) swap the columns whose low bit differs from b's
  const bool o1 = b & 1;
  const float r0 = __shfl_xor_sync(0xffffffffu, o1 ? x0 : x1, 1);
  const float r1 = __shfl_xor_sync(0xffffffffu, o1 ? x2 : x3, 1);
  // t[c2 | j] = M[(b & 2) | j][c2 | (b & 1)]
  const float t0 = o1 ? r0 : x0, t1 = o1 ? x1 : r0, t2 = o1 ? r1 : x2, t3 = o1 ? x3 : r1;
  // step 2: pairs (b, b ^ 2) swap the row halves
  const bool o2 = b & 2;
  const float v0 = __shfl_xor_sync(0xffffffffu, o2 ? t0 : t2, 2);
  const float v1 = __shfl_xor_sync(0xffffffffu, o2 ? t1 : t3, 2);
  y[0] = o2 ? v0 : t0;
  y[1] = o2 ? v1 : t1;
  y[2] = o2 ? t2 : v0;
  y[3] = o2 ? t3 : v1;
}

// Adds block j's dKV^T tiles into the fp32 rows the valid slots name.  `rows`:
// lane k holds the row of slot k (-1 for padding).  Dims of tile m: CTA 0 ->
// [0,128), [128,256), tail [512,576); CTA 1 -> [256,384), [384,512).  Called by
// the four drain warps (one per TMEM lane quarter).  Tile m is read once its
// MMAs completed (DKV_FULL + m) and handed back (DKV_FREE + m) before its
// reductions are issued.  With kStore (deterministic mode) the slot rows are
// stored at gslot + k * 576 (k = slot within the block) instead of added into
// dkv32.
template <bool kStore>
__device__ __forceinline__ bool drain_tiles(uint32_t sb, uint32_t tl, uint32_t tm_dkv, int j, int rows, int ntile,
                                            uint32_t crank, int L, float* dkv32, float* gslot,
                                            volatile int* abort_flag, uint32_t* status, int64_t dkv_n,
                                            const float* gbuf, int64_t gbuf_n) {
#pragma unroll 1
  for (int m = 0; m < ntile; ++m) {
    if (!__all_sync(0xffffffffu, mbar_wait(bar_addr(sb, DKV_FULL + m), j & 1, abort_flag, status))) return false;
    tc_fence_after();
    const int d = (crank == 0 ? (m < 2 ? 128 * m : 512) : 256 + 128 * m) + L;
    float gh[kBK], gl[kBK];
    tmem_ld_cols<kBK>(tl + tm_dkv + 64 * m, gh);        // hi half of the slots' columns
    tmem_ld_cols<kBK>(tl + tm_dkv + 64 * m + 32, gl);   // lo half
    tc_fence_before();
    mbar_arrive(bar_addr(sb, DKV_FREE + m));            // the MMA may overwrite this tile
    if (d < kDqk) {                     // warp-uniform: only CTA 0's tail tile has lanes past 576
      // 4 x 4 transposes among lanes 4a..4a+3: afterwards lane 4a+b holds dims
      // 4a..4a+3 (of the warp's 32) of slot 4g+b, one 16-byte reduction each
      const int b = L & 3;              // L & 31 is the lane
      const int d4 = d - b;             // first of the four dims
#pragma unroll
      for (int g = 0; g < kBK / 4; ++g) {
        float y[4];
        transpose4(gh[4 * g] + gl[4 * g], gh[4 * g + 1] + gl[4 * g + 1], gh[4 * g + 2] + gl[4 * g + 2],
                   gh[4 * g + 3] + gl[4 * g + 3], b, y);
        const int k = 4 * g + b;
        const int row = __shfl_sync(0xffffffffu, rows, k);
        if (row < 0) continue;
        if (kStore) {
          float* dst = gslot + k * kDqk + d4;
          if (check_range(dst, 4, gbuf, gbuf_n, status)) *reinterpret_cast<float4*>(dst) = make_float4(y[0], y[1], y[2], y[3]);
        } else {
          float* dst = dkv32 + (int64_t)row * kDqk + d4;
          if (check_range(dst, 4, dkv32, dkv_n, status)) red_add_v4(dst, y[0], y[1], y[2], y[3]);
        }
      }
    }
  }
  return true;
}

__device__ __forceinline__ bool drain_any(uint32_t sb, uint32_t tl, uint32_t tm_dkv, int j, int rows, int ntile,
                                          uint32_t crank, int L, float* dkv32, float* gslot, volatile int* abort_flag,
                                          uint32_t* status, int64_t dkv_n, const float* gbuf, int64_t gbuf_n) {
  return gslot != nullptr
             ? drain_tiles<true>(sb, tl, tm_dkv, j, rows, ntile, crank, L, dkv32, gslot, abort_flag, status, dkv_n,
                                 gbuf, gbuf_n)
             : drain_tiles<false>(sb, tl, tm_dkv, j, rows, ntile, crank, L, dkv32, gslot, abort_flag, status, dkv_n,
                                  gbuf, gbuf_n);
}

// kAllHeads: H == 128, no padding rows (the exchange then has no per-row test)
template <bool kAllHeads>
__global__ void __launch_bounds__(kThreads, 1) __cluster_dims__(2, 1, 1)
    tc_bwd_h128_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_do,
                       TcBwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sb = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t crank = cluster_ctarank();
  const uint32_t peer = crank ^ 1u;
  const int t = p.t0 + (blockIdx.x >> 1);
  const int nch = 4 + (int)crank;          // key chunks (64 dims each) of this CTA
  const int g0 = 4 * (int)crank;           // first global key chunk; value chunks are g0 .. g0+3
  // q chunks held: the key chunks, and for CTA 0 also the rope tail (chunk 8) in slot 4,
  // because CTA 0 computes the tail's dKV tile (this balances TMEM between the two)
  const int ntile = 3 - (int)crank;        // 128-dim dKV tiles: CTA 0 [0,256) + tail, CTA 1 [256,512)
  const int ndq = 64 * nch;                // dQ columns
  const uint32_t TM_S = ndq, TM_DP = ndq + 32, TM_DKV = ndq + 64;
  const int nblk = p.topk / kBK;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + SM_ABORT);

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    mbar_init(bar_addr(sb, KV_FULL + 0), kProducers + 1);   // cp.async arrivals + mask/rows
    mbar_init(bar_addr(sb, KV_FULL + 1), kProducers + 1);
    // MMA commit + softmax threads (mask read) + drain threads (rows read)
    mbar_init(bar_addr(sb, KV_EMPTY + 0), 1 + 128 + 128);
    mbar_init(bar_addr(sb, KV_EMPTY + 1), 1 + 128 + 128);
    mbar_init(bar_addr(sb, QD_FULL), 1);
    mbar_init(bar_addr(sb, SDP_FULL), 1);
    mbar_init(bar_addr(sb, SDP_FREE), 256);      // both warp sets loaded the partial S / dP
    mbar_init(bar_addr(sb, X_FULL + 0), 128);   // the peer's exchange warps wrote their partial rows
    mbar_init(bar_addr(sb, X_FULL + 1), 128);
    mbar_init(bar_addr(sb, X_EMPTY + 0), 128);  // the peer's softmax warps read ours
    mbar_init(bar_addr(sb, X_EMPTY + 1), 128);
    mbar_init(bar_addr(sb, P_FULL), 128);
    mbar_init(bar_addr(sb, PDS_FREE), 1);
    for (int m = 0; m < 3; ++m) {
      mbar_init(bar_addr(sb, DKV_FULL + m), 1);
      mbar_init(bar_addr(sb, DKV_FREE + m), 128);   // the drain warps loaded the tile
    }
    fence_mbar_init();
    *reinterpret_cast<volatile uint32_t*>(smem + SM_SMID) = smid();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(sb + SM_TMEM, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  tc_fence_after();
  SMLA_TRACE_T0;
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + SM_TMEM);
  // fewer than 128 heads: rows H..127 of every q / dO chunk are zero (the
  // MMAs read all 128 rows); the fence orders these stores before the MMAs
  if (p.H < 128) {
    const int per_chunk = (128 - p.H) * 8;      // 16-byte pieces
    for (int i = threadIdx.x; i < 9 * per_chunk; i += kThreads) {
      const int c = i / per_chunk, r = p.H + (i % per_chunk) / 8, piece = i % 8;
      *reinterpret_cast<uint4*>(smem + SM_Q + c * kChunk + r * 128 + piece * 16) = make_uint4(0u, 0u, 0u, 0u);
    }
    fence_proxy_async_smem();
  }
  // blocks that hold only padding contribute nothing and are skipped: list the
  // others in order (both CTAs of the pair read the same indices and agree)
  const int16_t* blist = reinterpret_cast<const int16_t*>(smem + SM_BLIST);
  // deterministic mode: where the contributions of block j (of the list) go
  auto gslot = [&](int j) -> float* {
    return p.gbuf == nullptr ? nullptr : p.gbuf + ((int64_t)(t - p.t0) * p.topk + (int64_t)blist[j] * kBK) * kDqk;
  };
  const int nb = build_block_list<kBK>(p.indices + (int64_t)t * p.topk, nblk, p.T, smem + SM_BFLAG,
                                       reinterpret_cast<int16_t*>(smem + SM_BLIST), reinterpret_cast<int*>(smem + SM_NB));

  if (warp < kProducers / 32) {
    // ------------------------------------------------------------ producers
    const int pt = threadIdx.x;              // 0..63
    if (pt == 0) {
      // the token's H head rows of each 64-dim chunk; rows H..127 were zeroed above
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_do);
      mbar_arrive_expect_tx(bar_addr(sb, QD_FULL), (5 + 4) * p.H * 128);
      // q and dO are read once: evict-first, so that they do not push the fp32
      // dKV lines the reductions keep hitting out of L2
      const uint64_t pol = l2_evict_first_policy();
      for (int k = 0; k < 5; ++k)
        tma_load_2d_hint(sb + SM_Q + k * kChunk, &tm_q, 64 * (k < nch ? g0 + k : 8), t * p.H, bar_addr(sb, QD_FULL), pol);
      for (int k = 0; k < 4; ++k)
        tma_load_2d_hint(sb + SM_DO + k * kChunk, &tm_do, 64 * (g0 + k), t * p.H, bar_addr(sb, QD_FULL), pol);
    }
    // thread pt copies 16-byte piece c16 of rows r0 + 8 j of every chunk
    const int c16 = pt & 7, r0 = pt >> 3;
    constexpr int RS = kProducers / 8;
    const int32_t* irow = p.indices + (int64_t)t * p.topk;
    const uint16_t* kvc = p.kv + 64 * g0 + 8 * c16;
    int* srows = reinterpret_cast<int*>(smem + SM_ROWS);
    int nxt[kRowsPerProducer], nm = 0;
    if (nb > 0) {
      const int32_t* ib = irow + blist[0] * kBK;
#pragma unroll
      for (int j = 0; j < kRowsPerProducer; ++j) nxt[j] = __ldg(ib + r0 + RS * j);
      if (warp == 0) nm = __ldg(ib + lane);
    }
    for (int i = 0; i < nb; ++i) {
      const int st = i & 1;
      int cur[kRowsPerProducer];
#pragma unroll
      for (int j = 0; j < kRowsPerProducer; ++j) cur[j] = nxt[j];
      const int cm = nm;
      if (i + 1 < nb) {                      // indices of the next block, one block ahead
        const int32_t* ib = irow + blist[i + 1] * kBK;
#pragma unroll
        for (int j = 0; j < kRowsPerProducer; ++j) nxt[j] = __ldg(ib + r0 + RS * j);
        if (warp == 0) nm = __ldg(ib + lane);
      }
      if (i >= 2 && !__all_sync(0xffffffffu, mbar_wait(bar_addr(sb, KV_EMPTY + st), ((i >> 1) - 1) & 1, abort_flag,
                                                       p.status)))
        break;                                 // warp-uniform exit
      const uint32_t stage = sb + SM_KV + st * kStage;
#pragma unroll
      for (int j = 0; j < kRowsPerProducer; ++j) {
        const int r = r0 + RS * j;
        const bool v = cur[j] >= 0 && cur[j] < p.T;
        const uint16_t* src = kvc + (int64_t)(v ? cur[j] : 0) * kDqk;
        const uint32_t dst = stage + r * 128 + ((c16 ^ (r & 7)) << 4);
        for (int k = 0; k < nch; ++k) {
          const uint16_t* s = src + 64 * k;
          uint32_t bytes = v ? 16u : 0u;
          check_src(s, bytes, p.kv, (int64_t)p.T * kDqk, p.status);
          cp_async16(dst + k * kChunkKV, s, bytes);
        }
      }
      cp_async_arrive(bar_addr(sb, KV_FULL + st));
      if (warp == 0) {                        // slot mask and row list of the block
        const bool v = cm >= 0 && cm < p.T;
        const uint32_t m = __ballot_sync(0xffffffffu, v);
        srows[st * 32 + lane] = v ? cm : -1;
        __syncwarp();
        if (lane == 0) {
          *reinterpret_cast<volatile uint32_t*>(smem + SM_MASK + 4 * st) = m;
          mbar_arrive(bar_addr(sb, KV_FULL + st));
        }
      }
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t id_sdp = idesc_bf16(128, kBK, false, false);
      const uint32_t id_dq256 = idesc_bf16(128, 256, false, true);
      const uint32_t id_dq64 = idesc_bf16(128, 64, false, true);
      const uint32_t id_dkv = idesc_bf16(128, 2 * kBK, true, true);   // N = 64: hi | lo
      // base descriptors; per-MMA descriptors only move the start address
      const uint64_t dq0 = sdesc_sw128(sb + SM_Q, 16, 1024);        // q, K-major (scores)
      const uint64_t ddo0 = sdesc_sw128(sb + SM_DO, 16, 1024);      // dO, K-major (dP)
      const uint64_t dk0 = sdesc_sw128(sb + SM_KV, 16, 1024);       // K rows, K-major (scores, dP)
      const uint64_t dkt0 = sdesc_sw128(sb + SM_KV, kChunkKV, 1024); // K rows read MN-major (dQ)
      const uint64_t dqt0 = sdesc_sw128(sb + SM_Q, kChunk, 1024);   // q^T, MN-major (dKV)
      const uint64_t ddot0 = sdesc_sw128(sb + SM_DO, kChunk, 1024); // dO^T, MN-major (dKV)
      const uint64_t dsa0 = sdesc_sw128(sb + SM_DS, 16, 1024);      // dS' halves as the K-major A of dQ
      const uint64_t dpb0 = sdesc_sw128(sb + SM_P, 8192, 1024);     // P / dS' rows as MN-major B of dKV
      static_assert(SM_P < SM_DS, "offsets from SM_P are non-negative");
      bool ok = mbar_wait(bar_addr(sb, QD_FULL), 0, abort_flag, p.status);
      // iteration i issues S/dP of block i, then dQ/dKV of block i-1, so the
      // score MMAs of the next block run while the softmax warps work
      for (int i = 0; ok && i <= nb; ++i) {
        if (i < nb) {
          const int st = i & 1;
          if (!(ok = mbar_wait(bar_addr(sb, KV_FULL + st), (i >> 1) & 1, abort_flag, p.status))) break;
          SMLA_STAMP(i, 0);
          if (i >= 1 && !(ok = mbar_wait(bar_addr(sb, SDP_FREE), (i - 1) & 1, abort_flag, p.status))) break;
          fence_proxy_async_smem();   // cp.async wrote the stage through the generic proxy
          tc_fence_after();
          // S_half = q_half K_half^T ; dP_half = dO_half V_half^T   (K-major operands, 128B swizzle)
#pragma unroll
          for (int k = 0; k < 5; ++k) {
            if (k < nch) {
#pragma unroll
              for (int ks = 0; ks < 4; ++ks)
                mma_bf16_ss(tmem + TM_S, sdesc_add(dq0, k * kChunk + ks * 32),
                            sdesc_add(dk0, st * kStage + k * kChunkKV + ks * 32), id_sdp, (k | ks) != 0);
            }
          }
#pragma unroll
          for (int k = 0; k < 4; ++k)
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
              mma_bf16_ss(tmem + TM_DP, sdesc_add(ddo0, k * kChunk + ks * 32),
                          sdesc_add(dk0, st * kStage + k * kChunkKV + ks * 32), id_sdp, (k | ks) != 0);
          mma_commit(bar_addr(sb, SDP_FULL));
          SMLA_STAMP(i, 1);
        }
        if (i >= 1) {
          const int j = i - 1, stj = j & 1;
          if (!(ok = mbar_wait(bar_addr(sb, P_FULL), j & 1, abort_flag, p.status))) break;
          SMLA_STAMP(j, 2);
          tc_fence_after();
          // dQ_half += (hi + lo) K_half: A = dS' (K-major, 64B swizzle), B = K block read MN-major
#pragma unroll
          for (int part = 0; part < 2; ++part) {
#pragma unroll
            for (int ks = 0; ks < 2; ++ks) {
              const uint64_t ad = sdesc_add(dsa0, part * 64 + ks * 32);
              const uint32_t acc = (j > 0 || part > 0 || ks > 0);
              const uint32_t koff = stj * kStage + ks * 16 * 128;
              mma_bf16_ss(tmem + TM_DQ, ad, sdesc_add(dkt0, koff), id_dq256, acc);
              if (nch == 5) mma_bf16_ss(tmem + TM_DQ + 256, ad, sdesc_add(dkt0, koff + 4 * kChunkKV), id_dq64, acc);
            }
          }
          // the KV stage is read only by the S / dP and dQ products: hand it to the
          // producers before the dKV products, so the gather of block j + 2 starts sooner
          mma_commit(bar_addr(sb, KV_EMPTY + stj));
          // dKV^T tiles (M = 128 dims, N = 32 slots, K = 128 heads):
          //   dKV^T = q_half^T dS' + dO_half^T P   (A MN-major 128B swizzle, B MN-major 64B swizzle)
          SMLA_STAMP(j, 3);
          for (int m = 0; ok && m < ntile; ++m) {
            if (j >= 1 && !(ok = mbar_wait(bar_addr(sb, DKV_FREE + m), (j - 1) & 1, abort_flag, p.status))) break;
            if (m >= 1) SMLA_STAMP(j, m == 1 ? 11 : 8);
            tc_fence_after();
            const uint32_t d_t = tmem + TM_DKV + 64 * m;
            // q^T for this tile: q slots 2m, 2m+1 (CTA 0's tile 2 is the rope tail in slot 4;
            // its second half reads the next buffer and only lands in TMEM lanes that are not drained)
#pragma unroll
            for (int ks = 0; ks < 8; ++ks)
              mma_bf16_ss(d_t, sdesc_add(dqt0, 2 * m * kChunk + ks * 16 * 128),
                          sdesc_add(dpb0, SM_DS - SM_P + ks * 16 * 128), id_dkv, ks != 0);
            if (2 * m < 4) {   // tiles inside the value range also get the dO^T P term
#pragma unroll
              for (int ks = 0; ks < 8; ++ks)
                mma_bf16_ss(d_t, sdesc_add(ddot0, 2 * m * kChunk + ks * 16 * 128), sdesc_add(dpb0, ks * 16 * 128),
                            id_dkv, 1);
            }
            mma_commit(bar_addr(sb, DKV_FULL + m));
          }
          if (!ok) break;
          mma_commit(bar_addr(sb, PDS_FREE));
          SMLA_STAMP(j, 4);
        }
      }
    }
    __syncwarp();
  } else if (warp < kXchgWarp0) {
    // ------------------------------------------------------------ softmax / dS
    const int q4 = warp & 3;
    const int h = 32 * q4 + lane;
    const uint32_t tl = tmem + ((uint32_t)(32 * q4) << 16);
    // heads past H: lse = +inf gives P = 0 and dS' = 0 exactly
    const bool real = h < p.H;
    const float lse2 = real ? p.lse[(int64_t)t * p.H + h] * kLog2e : INFINITY;
    const float dl = real ? p.delta[(int64_t)t * p.H + h] : 0.f;
    const uint64_t c2x2 = f32x2(p.c2, p.c2), nlse2x2 = f32x2(-lse2, -lse2);
    const uint64_t scale2 = f32x2(p.scale, p.scale), dl2x2 = f32x2(dl, dl);
    uint8_t* prow = smem + SM_P + h * 128;
    uint8_t* dsrow = smem + SM_DS + h * 128;
    const int sw = h & 7;               // 128B swizzle: 16-byte chunk index ^= row & 7
    // the peer CTA's exchange slot (its partial S / dP rows) and its X_EMPTY barriers
    const uint32_t xempty_peer = mapa(bar_addr(sb, X_EMPTY), peer);
    const uint32_t peer_sm = ld_cluster_u32(mapa(sb + SM_SMID, peer));
    const float4* xpeer = reinterpret_cast<const float4*>(p.xchg + (size_t)(peer_sm % kXchgSlots) * kXchgSlotFloats) + h;
    bool ok = true;
    for (int i = 0; i < nb; ++i) {
      const int st = i & 1, xb = i & 1;
      // own partial rows; the TMEM buffer is free once both warp sets hold them
      if (!(ok = __all_sync(0xffffffffu, mbar_wait(bar_addr(sb, SDP_FULL), i & 1, abort_flag, p.status)))) break;
      if (h == 0) SMLA_STAMP(i, 5);
      tc_fence_after();
      float s[32], dp[32];
      tmem_ld32(tl + TM_S, s);
      tmem_ld32(tl + TM_DP, dp);
      tc_fence_before();
      mbar_arrive(bar_addr(sb, SDP_FREE));
      // add the peer's partial rows (published by its exchange warps)
      if (!(ok = __all_sync(0xffffffffu, mbar_wait<true>(bar_addr(sb, X_FULL + xb), (i >> 1) & 1, abort_flag, p.status))))
        break;
      // heads past H (zero q and dO rows: exactly 0 partials) are not exchanged
      const float4* rd = xpeer + xb * (kXchgBufFloats / 4);
      if (kAllHeads || real) {
#pragma unroll
        for (int v = 0; v < 8; ++v) {
          const float4 a = ld_cg_v4(rd + v * 128), c = ld_cg_v4(rd + (8 + v) * 128);
          s[4 * v] += a.x; s[4 * v + 1] += a.y; s[4 * v + 2] += a.z; s[4 * v + 3] += a.w;
          dp[4 * v] += c.x; dp[4 * v + 1] += c.y; dp[4 * v + 2] += c.z; dp[4 * v + 3] += c.w;
        }
      }
      mbar_arrive_remote(xempty_peer + 8 * xb);       // the peer may reuse that buffer
      if (h == 0) SMLA_STAMP(i, 6);
      if (!(ok = __all_sync(0xffffffffu, mbar_wait(bar_addr(sb, KV_FULL + st), (i >> 1) & 1, abort_flag, p.status)))) break;
      const uint32_t mask = *reinterpret_cast<volatile uint32_t*>(smem + SM_MASK + 4 * st);
      mbar_arrive(bar_addr(sb, KV_EMPTY + st));
      // P / dS' buffers are free once this CTA's dQ / dKV MMAs of the previous block completed
      if (i >= 1 && !(ok = __all_sync(0xffffffffu, mbar_wait(bar_addr(sb, PDS_FREE), (i - 1) & 1, abort_flag, p.status))))
        break;
      // P and dS' as bf16 pairs hi + lo, 8 slots (one 16-byte chunk of each half-row) at a
      // time; two slots per paired fp32 instruction:
      //   P = exp2(S c2 - lse2), dS' = (scale P)(dP - Delta), lo = value - hi
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t pp[4], dd[4], dl2[4], pl[4];
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
          const int j = 4 * c + jj;
          const bool v0 = (mask >> (2 * j)) & 1u, v1 = (mask >> (2 * j + 1)) & 1u;
          float a0, a1;
          f32x2_split(fma_f32x2(f32x2(s[2 * j], s[2 * j + 1]), c2x2, nlse2x2), a0, a1);
          const float p0 = v0 ? ex2(a0) : 0.f;   // padding: P = 0 exactly
          const float p1 = v1 ? ex2(a1) : 0.f;
          const uint64_t pv = f32x2(p0, p1);
          pp[jj] = pack_bf16x2(p0, p1);
          float r0, r1;
          f32x2_split(sub_f32x2(pv, f32x2(bf16_lo(pp[jj]), bf16_hi(pp[jj]))), r0, r1);
          pl[jj] = pack_bf16x2(r0, r1);
          const uint64_t dv = mul_f32x2(mul_f32x2(scale2, pv), sub_f32x2(f32x2(dp[2 * j], dp[2 * j + 1]), dl2x2));
          float d0, d1;
          f32x2_split(dv, d0, d1);
          dd[jj] = pack_bf16x2(d0, d1);
          f32x2_split(sub_f32x2(dv, f32x2(bf16_lo(dd[jj]), bf16_hi(dd[jj]))), r0, r1);   // the part bf16 dropped
          dl2[jj] = pack_bf16x2(r0, r1);
        }
        *reinterpret_cast<uint4*>(prow + ((c ^ sw) << 4)) = make_uint4(pp[0], pp[1], pp[2], pp[3]);
        *reinterpret_cast<uint4*>(prow + (((c + 4) ^ sw) << 4)) = make_uint4(pl[0], pl[1], pl[2], pl[3]);
        *reinterpret_cast<uint4*>(dsrow + ((c ^ sw) << 4)) = make_uint4(dd[0], dd[1], dd[2], dd[3]);
        *reinterpret_cast<uint4*>(dsrow + (((c + 4) ^ sw) << 4)) = make_uint4(dl2[0], dl2[1], dl2[2], dl2[3]);
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(bar_addr(sb, P_FULL));
      if (h == 0) SMLA_STAMP(i, 7);
    }
    if (ok && nb > 0)
      ok = __all_sync(0xffffffffu, mbar_wait(bar_addr(sb, PDS_FREE), (nb - 1) & 1, abort_flag, p.status));
    tc_fence_after();
    if (ok) {
      uint16_t* qrow = p.dq + ((int64_t)t * p.H + h) * kDqk + 256 * crank;
#pragma unroll 1
      for (int part = 0; part < ndq / 64; ++part) {
        float o[64];
        if (nb > 0) {
          tmem_ld64(tl + TM_DQ + 64 * part, o);
        } else {                             // no valid slot: no MMA ever wrote dQ
#pragma unroll
          for (int c = 0; c < 64; ++c) o[c] = 0.f;
        }
        uint4* dst = reinterpret_cast<uint4*>(qrow + 64 * part);
        if (real) {
#pragma unroll
          for (int c = 0; c < 8; ++c)
            dst[c] = make_uint4(pack_bf16x2(o[8 * c], o[8 * c + 1]), pack_bf16x2(o[8 * c + 2], o[8 * c + 3]),
                                pack_bf16x2(o[8 * c + 4], o[8 * c + 5]), pack_bf16x2(o[8 * c + 6], o[8 * c + 7]));
        }
      }
    }
  } else if (warp < kDrainWarp0) {
    // ------------------------------------------------------------ exchange
    // Publishes this CTA's partial S / dP rows of each block to its L2 exchange
    // slot (the peer's softmax warps read them).
    const int q4 = warp & 3;
    const int L = 32 * q4 + lane;               // TMEM lane: head (exchange) or dim within a tile (drain)
    const uint32_t tl = tmem + ((uint32_t)(32 * q4) << 16);
    const uint32_t xfull_peer = mapa(bar_addr(sb, X_FULL), peer);
    const uint32_t my_sm = *reinterpret_cast<volatile uint32_t*>(smem + SM_SMID);
    float4* xmine = reinterpret_cast<float4*>(p.xchg + (size_t)(my_sm % kXchgSlots) * kXchgSlotFloats) + L;

    bool ok = true;
    for (int i = 0; i < nb; ++i) {
      // partial S / dP rows of block i into buffer i & 1 of this SM's slot
      const int xb = i & 1;
      if (!(ok = __all_sync(0xffffffffu, mbar_wait(bar_addr(sb, SDP_FULL), i & 1, abort_flag, p.status)))) break;
      tc_fence_after();
      float s[32], dp[32];
      tmem_ld32(tl + TM_S, s);
      tmem_ld32(tl + TM_DP, dp);
      tc_fence_before();
      mbar_arrive(bar_addr(sb, SDP_FREE));
      // the peer's softmax warps read this buffer two blocks ago
      if (i >= 2 && !(ok = __all_sync(0xffffffffu, mbar_wait<true>(bar_addr(sb, X_EMPTY + xb), ((i >> 1) - 1) & 1,
                                                                   abort_flag, p.status))))
        break;
      float4* wr = xmine + xb * (kXchgBufFloats / 4);
      if (kAllHeads || L < p.H) {       // heads past H have exactly 0 partials and are not exchanged
#pragma unroll
        for (int v = 0; v < 8; ++v) {
          wr[v * 128] = make_float4(s[4 * v], s[4 * v + 1], s[4 * v + 2], s[4 * v + 3]);
          wr[(8 + v) * 128] = make_float4(dp[4 * v], dp[4 * v + 1], dp[4 * v + 2], dp[4 * v + 3]);
        }
      }
      mbar_arrive_remote(xfull_peer + 8 * xb);        // release: our rows are visible to the peer
      if (L == 0) SMLA_STAMP(i, 9);
    }
  } else {
    // ------------------------------------------------------------ dKV drain
    // Reads each block's dKV^T tiles from TMEM once the MMAs have written them and
    // adds them into the fp32 rows the block's valid slots name.  A block's row list is read from its KV stage as soon as the
    // stage lands, one block ahead, so the stage is not held back.
    const int q4 = warp & 3;
    const int L = 32 * q4 + lane;               // TMEM lane: dim within a tile
    const uint32_t tl = tmem + ((uint32_t)(32 * q4) << 16);
    const int* srows = reinterpret_cast<const int*>(smem + SM_ROWS);
    bool ok = true;
    auto read_rows = [&](int j, int& out) -> bool {
      const int st = j & 1;
      if (!__all_sync(0xffffffffu, mbar_wait(bar_addr(sb, KV_FULL + st), (j >> 1) & 1, abort_flag, p.status))) return false;
      out = srows[st * 32 + lane];
      mbar_arrive(bar_addr(sb, KV_EMPTY + st));
      return true;
    };
    int rows = -1, nxt = -1;
    if (nb > 0) ok = read_rows(0, rows);
    for (int j = 0; ok && j < nb; ++j) {
      if (j + 1 < nb && !(ok = read_rows(j + 1, nxt))) break;
      if (!(ok = drain_any(sb, tl, TM_DKV, j, rows, ntile, crank, L, p.dkv32, gslot(j), abort_flag, p.status,
                           (int64_t)p.T * kDqk, p.gbuf, (int64_t)(gridDim.x >> 1) * p.topk * kDqk)))
        break;
      if (L == 0) SMLA_STAMP(j, 10);
      rows = nxt;
    }
  }

  // ------------------------------------------------------------ teardown
  if (*abort_flag) __nanosleep(1000000);
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
  }
  return fn;
}

bool make_map(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows, uint32_t box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

uint32_t* tc_status_ptr();
float* tc_xchg_ptr();

cudaError_t launch_bwd_tc(const BwdArgs& a, cudaStream_t s) {
  CUtensorMap tm_q, tm_do;
  if (!make_map(&tm_q, a.q, kDqk, (uint64_t)a.T * a.H, a.H)) return cudaErrorInvalidValue;
  if (!make_map(&tm_do, a.dout, kDv, (uint64_t)a.T * a.H, a.H)) return cudaErrorInvalidValue;
  uint32_t* status = tc_status_ptr();
  float* xchg = tc_xchg_ptr();
  if (!status || !xchg) return cudaErrorInvalidSymbol;
  const bool all = a.H == 128;
  cudaError_t e = cudaFuncSetAttribute(all ? tc_bwd_h128_kernel<true> : tc_bwd_h128_kernel<false>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  const int nt = a.nt < 0 ? a.T : a.nt;
  if (nt == 0) return cudaSuccess;
  TcBwdParams p{a.kv,   xchg,   a.indices, a.lse, a.delta, a.dq,    a.dkv32,
                a.gbuf, status, a.T,       a.H,   a.topk,  a.t0,    a.scale, a.scale * kLog2e};
  if (all)
    tc_bwd_h128_kernel<true><<<dim3(2 * nt), dim3(kThreads), kSmemBytes, s>>>(tm_q, tm_do, p);
  else
    tc_bwd_h128_kernel<false><<<dim3(2 * nt), dim3(kThreads), kSmemBytes, s>>>(tm_q, tm_do, p);
  return cudaGetLastError();
}

#ifdef SMLA_TRACE
extern "C" int smla_trace_bwd_setup(int tok0) {
  static const long long z[tc::kTraceCtas * tc::kTracePerCta] = {};
  if (cudaMemcpyToSymbol(tc::g_trace, z, sizeof(z)) != cudaSuccess) return -1;
  return cudaMemcpyToSymbol(tc::g_trace_tok0, &tok0, sizeof(int)) == cudaSuccess ? 0 : -1;
}
extern "C" int smla_trace_bwd_read(long long* dst) {
  return cudaMemcpyFromSymbol(dst, tc::g_trace, sizeof(long long) * tc::kTraceCtas * tc::kTracePerCta) == cudaSuccess ? 0 : -1;
}
#endif

}  // namespace smla
