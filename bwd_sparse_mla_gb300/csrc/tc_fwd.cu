// Tensor-core (tcgen05) forward for up to 128 heads (fewer heads run as a
// 128-row tile whose rows past H are zero).
//
// Work split: a cluster of two CTAs works through a strided list of query
// tokens (a persistent kernel: one cluster per pair of SMs), with different
// roles, so that no fp32 partial result ever crosses between the CTAs.
//
//   score CTA (cluster rank 0) holds the current token's q (128 heads x 576
//     dims, bf16) in TMEM as the A operand and gathers the full 576-wide KV
//     rows named by each block of 64 top-k slots.  q itself arrives through
//     the same ring of units as the KV rows (nine 64-dim chunks ahead of the
//     token's first block) and is copied into TMEM by the tensor pipe.  It
//     computes the complete scores S = q K^T of two blocks at a time
//     (M = 128 heads, N = 2 x 64 slots, K = 576).  Two
//     softmax groups (one thread per head each) take alternate blocks: padding
//     slots are masked to -inf, the running max moves lazily (only when a
//     block max exceeds it by more than 8 in the log2 domain) and passes from
//     group to group in block order, P = exp2(S*scale*log2e - m) is rounded to
//     bf16.  P and the block's per-head rescale factors are copied into the
//     output CTA's shared memory with one distributed-shared-memory bulk copy
//     per block.  At the end of a token the sum of exponentials is floored at
//     1e-30 (miles PR #2079 summary, forward fragment), so a row with no valid
//     slot gets LSE = ln(1e-30).
//
//   output CTA (cluster rank 1) holds O (128 heads x 512 dims, fp32) in all of
//     its TMEM.  It gathers the 512-wide value part of the same rows, rescales
//     the O rows whose running max moved, and issues O += P V (M = 128,
//     N = 256, K = 64, twice).  At the end of a token O is divided by the sum
//     of the bf16-rounded weights (so the rounding of P cancels in `out`) and
//     written as bf16; a row with no valid slot is written as exact zeros.  The
//     sum of the rounded weights is taken here, from each block's P as it arrives.
//
// Both CTAs gather with 16-byte cp.async into rings of 128B-swizzled units
// that flow from one token into the next; a padding slot copies zero bytes
// and gets an exact-zero K/V row (the clamp + mask of the miles PR #2079 fix,
// implementation breakdown item 2).  Blocks whose 64 slots are all padding
// contribute nothing and are skipped by both CTAs.
#include <cuda.h>

#include "smla_common.cuh"
#include "tc_common.cuh"

namespace smla {
namespace {

using namespace tc;

constexpr int kBK = 64;                 // slots per block
constexpr int kProducers = 128;         // warps 0..3 gather
constexpr int kMmaWarp = 4;             // warp 4: lane 0 issues the MMAs; the warp owns TMEM
constexpr int kRowWarp0 = 5;            // warps 5..8 (and 9..12 in the score CTA): one thread per head
constexpr int kAuxWarp = 13;            // warp 13, lane 0: moves P (score CTA) / keeps the P buffers (output CTA)
constexpr int kThreads = 448;
constexpr int kRowsPerProducer = kBK * 8 / kProducers;   // 4 rows, one 16-byte piece of each chunk
constexpr int kChunkKV = kBK * 128;     // one 64-dim chunk of the 64 rows of a block (8 KiB)
constexpr float kLazyRescale = 8.f;     // log2-domain slack before O is rescaled
constexpr int kMaxBlocks = kTcMaxTopk / kBK;
constexpr int kNS = 2;                  // score CTA: P staging buffers
constexpr int kNP = 3;                  // output CTA: P buffers
constexpr int kMaskRing = 4;            // score CTA: slot-validity masks of the blocks in flight
constexpr int kProdBar = 1;             // named barrier of the producer warps

// KV rows are gathered into rings of units (128B-swizzled, 8 KiB per 64-dim
// chunk of 64 rows).  A unit is refilled as soon as the MMAs that read it
// complete, so the gathers stay in flight continuously, across token boundaries.
//   score CTA:  a token's blocks go in pairs; unit c of a pair holds 64-dim chunk
//               c of both blocks (16 KiB: the block with an even running index in
//               the first half), 9 units per pair (the 576-wide K rows), so that
//               one N = 128 score MMA reads the two blocks as one B operand; a
//               token with a valid block starts with 9 q units (unit c: 64-dim
//               chunk c of the token's 128 head rows, rows past H zero)
//   output CTA: units of 4 chunks (32 KiB), 2 per block (the 512-wide V rows;
//               one unit is the B operand of one N = 256 PV MMA)
constexpr int kSPairUnit = 2 * 64 * 128;   // bytes of one score-CTA unit
constexpr int kSUnitsPerPair = 9, kSRing = 11;
constexpr int kOUnitCh = 4, kOUnits = 2, kORing = 5;

// one P buffer: 128 heads x 64 slots bf16 (128B swizzle, the PV MMA's A
// operand), then the 128 rescale factors of the block
constexpr int kPBytes = 128 * 128;
constexpr int kPXBytes = kPBytes + 128 * 4;              // what one block hands over (16896 B)
constexpr int kPBufStride = 17 * 1024;                   // 1024-aligned buffer stride
// score CTA: K ring, P staging, the running state, the mask ring
constexpr int SM_K = 0;
constexpr int SM_STG = SM_K + kSRing * kSPairUnit;
constexpr int SM_STATE = SM_STG + kNS * kPBufStride;     // 128 heads x float4 (m, l)
constexpr int SM_MASK = SM_STATE + 128 * 16;             // kMaskRing x u64
constexpr int kScoreEnd = SM_MASK + 8 * kMaskRing;
// output CTA: V ring, P buffers, the final sums of two tokens
constexpr int SM_V = 0;
constexpr int SM_P = SM_V + kORing * kOUnitCh * kChunkKV;
constexpr int kOutEnd = SM_P + kNP * kPBufStride;
// common to both roles: the token ring (block count of the two newest tokens),
// the producers' per-token block flags and list
constexpr int SM_TOK = kScoreEnd > kOutEnd ? kScoreEnd : kOutEnd;   // 2 x int
constexpr int SM_BFLAG = SM_TOK + 16;                    // per block: holds a valid slot (u8)
constexpr int SM_BLIST = SM_BFLAG + kMaxBlocks;          // blocks with a valid slot, in order (u16)
constexpr int SM_NB = SM_BLIST + 2 * kMaxBlocks;
constexpr int SM_BAR = (SM_NB + 8 + 7) & ~7;
// barriers: the same slots carry role-specific meanings
enum ScoreBar { KV_FULL = 0, KV_EMPTY = kSRing, M_FULL = 2 * kSRing, M_EMPTY = M_FULL + kMaskRing,
                Q_EMPTY = M_EMPTY + kMaskRing, S_FULL, S_FREE = S_FULL + 2, ST_FULL = S_FREE + 2,
                STG_FULL = ST_FULL + 2, STG_FREE = STG_FULL + kNS, P_FREE = STG_FREE + kNS,
                TOK_FULL_S = P_FREE + kNP, TOK_EMPTY_S = TOK_FULL_S + 2, NBAR_S = TOK_EMPTY_S + 2 };
enum OutBar { V_FULL = 0, V_EMPTY = kORing, P_FULL = 2 * kORing, R_DONE = P_FULL + kNP, PV_DONE = R_DONE + kNP,
              RS_DONE = PV_DONE + kNP, O_FREE = RS_DONE + kNP, TOK_FULL_O, TOK_EMPTY_O = TOK_FULL_O + 2,
              NBAR_O = TOK_EMPTY_O + 2 };
constexpr int kNBar = 56;
static_assert(NBAR_S <= kNBar && NBAR_O <= kNBar, "barrier slots");
constexpr int SM_TMEM = SM_BAR + 8 * kNBar;
constexpr int SM_SMID = SM_TMEM + 4;
constexpr int SM_ABORT = SM_SMID + 4;
constexpr int kSmemBytes = SM_ABORT + 4 + 1024;          // + alignment slack
static_assert(kSmemBytes <= 232448, "shared memory budget");
static_assert(kSmemBytes > 232448 / 2, "one CTA per SM");
static_assert(SM_STG % 1024 == 0 && SM_P % 1024 == 0 && kPBufStride % 1024 == 0 && kChunkKV % 1024 == 0, "swizzle atoms");
static_assert(kPXBytes % 16 == 0 && kPXBytes <= kPBufStride, "bulk copy size");
static_assert(kSPairUnit == 2 * kChunkKV && kOUnitCh * kOUnits == 8, "units cover the rows");

// every accumulator and every tcgen05.ld starts at a column that is a multiple of its width
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t TM_S = 0;            // score CTA: two 64-column score buffers (buffer g for group g)
constexpr uint32_t TM_Q = 128;          // score CTA: q as bf16 pairs, 288 columns
constexpr uint32_t TM_O = 0;            // output CTA: O, 512 columns

struct TcFwdParams {
  const uint16_t* q;                    // [T, H, 576] bf16
  const uint16_t* kv;                   // [T, 576] bf16
  const int32_t* indices;
  uint16_t* out;
  float* lse;
  uint32_t* status;
  int T, H, topk;                       // H <= 128 heads; rows H..127 of the tile are zero
  int t0, nt;                           // this launch handles query rows [t0, t0 + nt)
  float c2;                             // scale * log2(e)
};

__device__ __forceinline__ uint32_t bar_addr(uint32_t base, int i) { return base + SM_BAR + 8 * i; }

// bulk copy of `bytes` (a multiple of 16) from this CTA's shared memory into
// another CTA's (addresses from mapa); completes tx on the destination's barrier
__device__ __forceinline__ void bulk_s2s(uint32_t dst_cluster, uint32_t src, uint32_t bytes, uint32_t bar_cluster) {
  asm volatile("cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   dst_cluster),
               "r"(src), "r"(bytes), "r"(bar_cluster)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory"); }
// 16-byte cp.async (zero fill past src_bytes) with an L2 cache policy
__device__ __forceinline__ void cp_async16_hint(uint32_t dst, const void* src, uint32_t src_bytes, uint64_t pol) {
  asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2, %3;" ::"r"(dst), "l"(src), "r"(src_bytes),
               "l"(pol)
               : "memory");
}
// Tensor-pipe copy of a 128-row x 32-byte shared-memory matrix (described like an
// MMA operand) into 128 TMEM lanes x 8 columns; executes after the tcgen05 copies
// and before the MMAs that the same thread issues later
__device__ __forceinline__ void tmem_cp_128x256b(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::1.128x256b [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}
// 16-byte global store with an L2 cache policy
__device__ __forceinline__ void st_v4_hint(uint4* p, uint4 v, uint64_t pol) {
  asm volatile("st.global.L2::cache_hint.v4.u32 [%0], {%1, %2, %3, %4}, %5;" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w), "l"(pol)
               : "memory");
}
__device__ __forceinline__ void named_bar_sync(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}
__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

#ifdef SMLA_TRACE
#define SMLA_TRACE_ARGS , long long trace_t0, int trace_cta
#define SMLA_TRACE_PASS , trace_t0, trace_cta
#else
#define SMLA_TRACE_ARGS
#define SMLA_TRACE_PASS
#endif
constexpr int kTraceGb0 = 100;          // trace rows: global blocks kTraceGb0 .. kTraceGb0 + 32

// Number of tokens of this cluster (tokens cl, cl + ncl, ... of the launch).
__device__ __forceinline__ int cluster_tokens(const TcFwdParams& p, int cl, int ncl) {
  return cl < p.nt ? (p.nt - 1 - cl) / ncl + 1 : 0;
}

// Producer warps: for each token of the cluster, list the blocks that hold a
// valid slot, publish the token's block count to the other roles, then
// gather the rows unit by unit into the ring of NRING units of UCH chunks
// (UPB units per block).  With kMask the slot-validity mask of each block is
// written into the mask ring for the softmax.
template <int UCH, int UPB, int NRING, bool kMask>
__device__ __forceinline__ void produce(const TcFwdParams& p, uint32_t sb, uint8_t* smem, int cl, int ncl,
                                        volatile int* abort_flag, int full0, int empty0, int tokfull0,
                                        int tokempty0 SMLA_TRACE_ARGS) {
  const int pt = threadIdx.x;              // 0..127
  const int warp = pt >> 5, lane = pt & 31;
  const int c16 = pt & 7, r0 = pt >> 3;    // 16-byte piece c16 of rows r0 + 16 j of every chunk
  constexpr int RS = kProducers / 8;
  constexpr int kUnitBytes = UCH * kChunkKV;
  const int nblk = p.topk / kBK;
  const int ntok = cluster_tokens(p, cl, ncl);
  uint8_t* flag = smem + SM_BFLAG;
  int16_t* blist = reinterpret_cast<int16_t*>(smem + SM_BLIST);
  volatile int* nbs = reinterpret_cast<volatile int*>(smem + SM_NB);
  volatile int* tok = reinterpret_cast<volatile int*>(smem + SM_TOK);
  const uint16_t* kvc = p.kv + 8 * c16;
  int n = 0, gb = 0;                       // units and blocks gathered so far (all tokens)
  for (int k = 0; k < ntok; ++k) {
    const int t = p.t0 + cl + k * ncl;
    const int32_t* irow = p.indices + (int64_t)t * p.topk;
    // the blocks of this token that hold a valid slot (0 <= idx < T)
    for (int b = pt; b < nblk; b += kProducers) {
      const int4* ib = reinterpret_cast<const int4*>(irow + b * kBK);
      bool v = false;
#pragma unroll 4
      for (int c = 0; c < kBK / 4; ++c) {
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
      // publish the token's block count (the slot of token k - 2 must have been read)
      const bool ok = k < 2 || __all_sync(0xffffffffu, mbar_wait(bar_addr(sb, tokempty0 + (k & 1)), ((k >> 1) - 1) & 1,
                                                                 abort_flag, p.status));
      if (lane == 0) {
        *nbs = ok ? base : -1;
        if (ok) {
          tok[k & 1] = base;
          mbar_arrive(bar_addr(sb, tokfull0 + (k & 1)));
        }
      }
    }
    named_bar_sync(kProdBar, kProducers);
    const int nb = *nbs;
    if (nb < 0) return;                    // uniform over the producer warps
    int nxt[kRowsPerProducer], nm[2] = {0, 0};
    if (nb > 0) {
      const int32_t* ib = irow + blist[0] * kBK;
#pragma unroll
      for (int j = 0; j < kRowsPerProducer; ++j) nxt[j] = __ldg(ib + r0 + RS * j);
      if (kMask && warp == 0) { nm[0] = __ldg(ib + lane); nm[1] = __ldg(ib + 32 + lane); }
    }
    bool ok = true;
    for (int i = 0; ok && i < nb; ++i, ++gb) {
      int cur[kRowsPerProducer], cm[2];
#pragma unroll
      for (int j = 0; j < kRowsPerProducer; ++j) cur[j] = nxt[j];
      cm[0] = nm[0]; cm[1] = nm[1];
      if (i + 1 < nb) {                    // indices of the next block, one block ahead
        const int32_t* ib = irow + blist[i + 1] * kBK;
#pragma unroll
        for (int j = 0; j < kRowsPerProducer; ++j) nxt[j] = __ldg(ib + r0 + RS * j);
        if (kMask && warp == 0) { nm[0] = __ldg(ib + lane); nm[1] = __ldg(ib + 32 + lane); }
      }
      const uint16_t* src[kRowsPerProducer];
      uint32_t dsto[kRowsPerProducer], nbytes[kRowsPerProducer];
#pragma unroll
      for (int j = 0; j < kRowsPerProducer; ++j) {
        const int r = r0 + RS * j;
        const bool v = cur[j] >= 0 && cur[j] < p.T;
        src[j] = kvc + (int64_t)(v ? cur[j] : 0) * kDqk;
        dsto[j] = r * 128 + ((c16 ^ (r & 7)) << 4);
        nbytes[j] = v ? 16u : 0u;
      }
      if (pt == 0) SMLA_STAMP(gb - kTraceGb0, 9);
#pragma unroll 1
      for (int u = 0; u < UPB; ++u, ++n) {
        const int slot = n % NRING;
        if (n >= NRING &&
            !(ok = __all_sync(0xffffffffu, mbar_wait(bar_addr(sb, empty0 + slot), ((n / NRING) - 1) & 1, abort_flag,
                                                     p.status))))
          break;                           // warp-uniform exit
        const uint32_t unit = sb + slot * kUnitBytes;
#pragma unroll
        for (int j = 0; j < kRowsPerProducer; ++j)
#pragma unroll
          for (int c = 0; c < UCH; ++c) {
            const uint16_t* s = src[j] + 64 * (u * UCH + c);
            uint32_t bytes = nbytes[j];
            check_src(s, bytes, p.kv, (int64_t)p.T * kDqk, p.status);
            cp_async16(unit + dsto[j] + c * kChunkKV, s, bytes);
          }
        cp_async_arrive(bar_addr(sb, full0 + slot));
      }
      if (!ok) break;
      if (pt == 0) SMLA_STAMP(gb - kTraceGb0, 10);
      if (kMask && warp == 0) {            // slot validity of the block for the softmax
        const int mr = gb % kMaskRing;
        if (gb >= kMaskRing &&
            !(ok = __all_sync(0xffffffffu, mbar_wait(bar_addr(sb, M_EMPTY + mr), ((gb / kMaskRing) - 1) & 1, abort_flag,
                                                     p.status))))
          break;
        const uint32_t ma = __ballot_sync(0xffffffffu, cm[0] >= 0 && cm[0] < p.T);
        const uint32_t mb = __ballot_sync(0xffffffffu, cm[1] >= 0 && cm[1] < p.T);
        if (lane == 0) {
          *reinterpret_cast<volatile uint64_t*>(smem + SM_MASK + 8 * mr) = (uint64_t)ma | ((uint64_t)mb << 32);
          mbar_arrive(bar_addr(sb, M_FULL + mr));
        }
      }
    }
    if (!ok) return;
  }
}

// Score CTA producers: as produce(), but a token's blocks are gathered in pairs
// (its listed blocks 2i and 2i + 1): unit c of a pair holds 64-dim chunk c of
// both blocks, the block with an even running index in the first half, the
// other in the second.  A token with an odd block count ends with a single
// block in its half of the unit.  The slot-validity mask of each block goes
// into the mask ring for the softmax.
__device__ __forceinline__ void produce_score(const TcFwdParams& p, uint32_t sb, uint8_t* smem, int cl, int ncl,
                                              volatile int* abort_flag SMLA_TRACE_ARGS) {
  const int pt = threadIdx.x;              // 0..127
  const int warp = pt >> 5, lane = pt & 31;
  const int c16 = pt & 7, r0 = pt >> 3;    // 16-byte piece c16 of rows r0 + 16 j of every chunk
  constexpr int RS = kProducers / 8;
  constexpr int R = kRowsPerProducer;
  const int nblk = p.topk / kBK;
  const int ntok = cluster_tokens(p, cl, ncl);
  uint8_t* flag = smem + SM_BFLAG;
  int16_t* blist = reinterpret_cast<int16_t*>(smem + SM_BLIST);
  volatile int* nbs = reinterpret_cast<volatile int*>(smem + SM_NB);
  volatile int* tok = reinterpret_cast<volatile int*>(smem + SM_TOK);
  const uint16_t* kvc = p.kv + 8 * c16;
  int n = 0, gb = 0;                       // units and blocks gathered so far (all tokens)
  for (int k = 0; k < ntok; ++k) {
    const int t = p.t0 + cl + k * ncl;
    const int32_t* irow = p.indices + (int64_t)t * p.topk;
    // the blocks of this token that hold a valid slot (0 <= idx < T)
    for (int b = pt; b < nblk; b += kProducers) {
      const int4* ib = reinterpret_cast<const int4*>(irow + b * kBK);
      bool v = false;
#pragma unroll 4
      for (int c = 0; c < kBK / 4; ++c) {
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
      // publish the token's block count (the slot of token k - 2 must have been read)
      const bool ok = k < 2 || __all_sync(0xffffffffu, mbar_wait(bar_addr(sb, TOK_EMPTY_S + (k & 1)),
                                                                 ((k >> 1) - 1) & 1, abort_flag, p.status));
      if (lane == 0) {
        *nbs = ok ? base : -1;
        if (ok) {
          tok[k & 1] = base;
          mbar_arrive(bar_addr(sb, TOK_FULL_S + (k & 1)));
        }
      }
    }
    named_bar_sync(kProdBar, kProducers);
    const int nb = *nbs;
    if (nb < 0) return;                    // uniform over the producer warps
    // rows of this thread and mask lanes of the (up to) two blocks of a pair, one pair ahead
    int nxt[2][R], nm[2][2];
    auto fetch = [&](int i) {
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const bool in = i + q < nb;
        const int32_t* ib = irow + (in ? blist[i + q] : 0) * kBK;
#pragma unroll
        for (int j = 0; j < R; ++j) nxt[q][j] = in ? __ldg(ib + r0 + RS * j) : -1;
        nm[q][0] = (in && warp == 0) ? __ldg(ib + lane) : -1;
        nm[q][1] = (in && warp == 0) ? __ldg(ib + 32 + lane) : -1;
      }
    };
    if (nb > 0) fetch(0);
    bool ok = true;
    if (nb > 0) {                          // the token's q rows, chunk by chunk, ahead of its blocks
      const uint64_t pol = l2_evict_first_policy();   // q is read once: keep the KV rows in L2
      const uint16_t* qsrc[2][R];
      uint32_t qdst[2][R], qbytes[2][R];
#pragma unroll
      for (int q = 0; q < 2; ++q)
#pragma unroll
        for (int j = 0; j < R; ++j) {
          const int r = r0 + RS * j, h = 64 * q + r;
          const bool v = h < p.H;
          qsrc[q][j] = p.q + ((int64_t)t * p.H + (v ? h : 0)) * kDqk + 8 * c16;
          qdst[q][j] = q * kChunkKV + r * 128 + ((c16 ^ (r & 7)) << 4);
          qbytes[q][j] = v ? 16u : 0u;
        }
#pragma unroll 1
      for (int c = 0; c < kSUnitsPerPair; ++c, ++n) {
        const int slot = n % kSRing;
        if (n >= kSRing &&
            !(ok = __all_sync(0xffffffffu, mbar_wait(bar_addr(sb, KV_EMPTY + slot), ((n / kSRing) - 1) & 1, abort_flag,
                                                     p.status))))
          break;                           // warp-uniform exit
        const uint32_t unit = sb + SM_K + slot * kSPairUnit;
#pragma unroll
        for (int q = 0; q < 2; ++q)
#pragma unroll
          for (int j = 0; j < R; ++j) {
            const uint16_t* s = qsrc[q][j] + 64 * c;
            uint32_t bytes = qbytes[q][j];
            check_src(s, bytes, p.q, (int64_t)p.T * p.H * kDqk, p.status);
            cp_async16_hint(unit + qdst[q][j], s, bytes, pol);
          }
        cp_async_arrive(bar_addr(sb, KV_FULL + slot));
      }
      if (!ok) return;
    }
    for (int i = 0; ok && i < nb; i += 2) {
      const int npair = nb - i < 2 ? 1 : 2;
      int cur[2][R], cm[2][2];
#pragma unroll
      for (int q = 0; q < 2; ++q) {
#pragma unroll
        for (int j = 0; j < R; ++j) cur[q][j] = nxt[q][j];
        cm[q][0] = nm[q][0]; cm[q][1] = nm[q][1];
      }
      if (i + 2 < nb) fetch(i + 2);
      const uint16_t* src[2][R];
      uint32_t dsto[2][R], nbytes[2][R];
#pragma unroll
      for (int q = 0; q < 2; ++q)
#pragma unroll
        for (int j = 0; j < R; ++j) {
          const int r = r0 + RS * j;
          const bool v = cur[q][j] >= 0 && cur[q][j] < p.T;
          src[q][j] = kvc + (int64_t)(v ? cur[q][j] : 0) * kDqk;
          dsto[q][j] = ((gb + q) & 1) * kChunkKV + r * 128 + ((c16 ^ (r & 7)) << 4);
          nbytes[q][j] = v ? 16u : 0u;
        }
      if (pt == 0) SMLA_STAMP(gb - kTraceGb0, 9);
      int slot = n % kSRing, lap = n / kSRing;   // kept incrementally over the pair's units
#pragma unroll 1
      for (int c = 0; c < kSUnitsPerPair; ++c, ++n) {
        if (lap > 0 &&
            !(ok = __all_sync(0xffffffffu, mbar_wait(bar_addr(sb, KV_EMPTY + slot), (lap - 1) & 1, abort_flag,
                                                     p.status))))
          break;                           // warp-uniform exit
        const uint32_t unit = sb + SM_K + slot * kSPairUnit;
        const int fslot = slot;
        if (++slot == kSRing) { slot = 0; ++lap; }
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          if (q == 1 && npair < 2) break;
#pragma unroll
          for (int j = 0; j < R; ++j) {
            const uint16_t* s = src[q][j] + 64 * c;
            uint32_t bytes = nbytes[q][j];
            check_src(s, bytes, p.kv, (int64_t)p.T * kDqk, p.status);
            cp_async16(unit + dsto[q][j], s, bytes);
          }
        }
        cp_async_arrive(bar_addr(sb, KV_FULL + fslot));
      }
      if (!ok) break;
      if (pt == 0) SMLA_STAMP(gb - kTraceGb0, 10);
      if (warp == 0) {                     // slot validity of the blocks for the softmax
        for (int q = 0; ok && q < npair; ++q) {
          const int gbq = gb + q, mr = gbq % kMaskRing;
          if (gbq >= kMaskRing &&
              !(ok = __all_sync(0xffffffffu, mbar_wait(bar_addr(sb, M_EMPTY + mr), ((gbq / kMaskRing) - 1) & 1,
                                                       abort_flag, p.status))))
            break;
          const uint32_t ma = __ballot_sync(0xffffffffu, cm[q][0] >= 0 && cm[q][0] < p.T);
          const uint32_t mb = __ballot_sync(0xffffffffu, cm[q][1] >= 0 && cm[q][1] < p.T);
          if (lane == 0) {
            *reinterpret_cast<volatile uint64_t*>(smem + SM_MASK + 8 * mr) = (uint64_t)ma | ((uint64_t)mb << 32);
            mbar_arrive(bar_addr(sb, M_FULL + mr));
          }
        }
      }
      ok = __all_sync(0xffffffffu, ok);    // warp 0's mask waits decide for its warp only
      gb += npair;
    }
    if (!ok) return;
  }
}

// Block count of the cluster's token k, from the token ring (one read per
// calling thread, acknowledged on the ring's empty barrier).  -1 on abort.
template <bool kWarp>
__device__ __forceinline__ int read_token(const TcFwdParams& p, uint32_t sb, uint8_t* smem, int k, int tokfull0,
                                          int tokempty0, volatile int* abort_flag) {
  const bool ok = kWarp ? __all_sync(0xffffffffu, mbar_wait(bar_addr(sb, tokfull0 + (k & 1)), (k >> 1) & 1, abort_flag,
                                                            p.status))
                        : mbar_wait(bar_addr(sb, tokfull0 + (k & 1)), (k >> 1) & 1, abort_flag, p.status);
  if (!ok) return -1;
  const int nb = reinterpret_cast<volatile int*>(smem + SM_TOK)[k & 1];
  mbar_arrive(bar_addr(sb, tokempty0 + (k & 1)));
  return nb;
}

// kAllHeads: H == 128 (no zero rows)
template <bool kAllHeads>
__global__ void __launch_bounds__(kThreads, 1) __cluster_dims__(2, 1, 1)
    tc_fwd_h128_kernel(TcFwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);   // 1024-aligned (128B swizzle atoms)
  const uint32_t sb = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t crank = cluster_ctarank();          // 0: score CTA, 1: output CTA
  const uint32_t peer = crank ^ 1u;
  const int cl = blockIdx.x >> 1, ncl = gridDim.x >> 1;
  const int ntok = cluster_tokens(p, cl, ncl);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + SM_ABORT);

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    if (crank == 0) {
      for (int k = 0; k < kSRing; ++k) {
        mbar_init(bar_addr(sb, KV_FULL + k), kProducers);      // cp.async arrivals
        mbar_init(bar_addr(sb, KV_EMPTY + k), 1);              // the MMAs that read the unit completed
      }
      for (int k = 0; k < kMaskRing; ++k) {
        mbar_init(bar_addr(sb, M_FULL + k), 1);
        mbar_init(bar_addr(sb, M_EMPTY + k), 128);             // the softmax group read the mask
      }
      mbar_init(bar_addr(sb, Q_EMPTY), 1);                     // the token's score MMAs completed
      for (int g = 0; g < 2; ++g) {
        mbar_init(bar_addr(sb, S_FULL + g), 1);
        mbar_init(bar_addr(sb, S_FREE + g), 128);
        mbar_init(bar_addr(sb, ST_FULL + g), 128);    // group g wrote the running state after its block
        mbar_init(bar_addr(sb, TOK_FULL_S + g), 1);
        mbar_init(bar_addr(sb, TOK_EMPTY_S + g), 1 + 1 + 256);   // MMA, P mover, both softmax groups
      }
      for (int k = 0; k < kNS; ++k) {
        mbar_init(bar_addr(sb, STG_FULL + k), 128);   // a group wrote P into staging buffer k
        mbar_init(bar_addr(sb, STG_FREE + k), 1);     // the bulk copy has read it
      }
      for (int k = 0; k < kNP; ++k) mbar_init(bar_addr(sb, P_FREE + k), 1);   // the output CTA's P buffer k is free
    } else {
      for (int k = 0; k < kORing; ++k) {
        mbar_init(bar_addr(sb, V_FULL + k), kProducers);
        mbar_init(bar_addr(sb, V_EMPTY + k), 1);
      }
      for (int k = 0; k < kNP; ++k) {
        mbar_init(bar_addr(sb, P_FULL + k), 1);       // armed with expect_tx; the bulk copy completes it
        mbar_init(bar_addr(sb, R_DONE + k), 128);     // rows rescaled where the max moved
        mbar_init(bar_addr(sb, PV_DONE + k), 1);
        mbar_init(bar_addr(sb, RS_DONE + k), 128);    // the rows summed the block's weights
      }
      for (int g = 0; g < 2; ++g) {
        mbar_init(bar_addr(sb, TOK_FULL_O + g), 1);
        mbar_init(bar_addr(sb, TOK_EMPTY_O + g), 1 + 1 + 128);   // MMA, P keeper, rows
      }
      mbar_init(bar_addr(sb, O_FREE), 128);           // the epilogue read O out of TMEM
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
  cluster_sync();   // the peer's barriers are initialised before any remote arrive
  tc_fence_after();
  SMLA_TRACE_T0;
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + SM_TMEM);

  if (crank == 0) {
    // ================================================================ score CTA
    if (warp < kProducers / 32) {
      produce_score(p, sb, smem, cl, ncl, abort_flag SMLA_TRACE_PASS);
    } else if (warp == kMmaWarp) {
      if (lane == 0) {
        // MMA issuer: S of each pair of blocks, unit by unit as the K units land: one
        // N = 128 MMA per K step writes both score buffers (buffer b holds the block
        // with running index parity b); a single last block of a token uses N = 64
        const uint32_t idesc_s1 = idesc_bf16(128, kBK, false, false);
        const uint32_t idesc_s2 = idesc_bf16(128, 2 * kBK, false, false);
        const uint64_t dk0 = sdesc_sw128(sb + SM_K, 16, 1024);
        int gb = 0, n = 0, kq = 0;           // kq: tokens with a valid block so far
        bool ok = true;
        for (int k = 0; ok && k < ntok; ++k) {
          const int nb = read_token<false>(p, sb, smem, k, TOK_FULL_S, TOK_EMPTY_S, abort_flag);
          if (!(ok = nb >= 0)) break;
          if (nb == 0) continue;             // no q units, no MMAs
          // the token's q units into TMEM, once the previous token's score MMAs (which
          // read q's columns) completed; the MMAs issued after the copies see them
#pragma unroll 1
          for (int c = 0; c < kSUnitsPerPair; ++c, ++n) {
            const int slot = n % kSRing;
            if (!(ok = mbar_wait(bar_addr(sb, KV_FULL + slot), (n / kSRing) & 1, abort_flag, p.status))) break;
            if (c == 0 && kq >= 1 && !(ok = mbar_wait(bar_addr(sb, Q_EMPTY), (kq - 1) & 1, abort_flag, p.status)))
              break;
            fence_proxy_async_smem();
            tc_fence_after();
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
              tmem_cp_128x256b(tmem + TM_Q + 32 * c + 8 * ks, sdesc_add(dk0, slot * kSPairUnit + ks * 32));
            mma_commit(bar_addr(sb, KV_EMPTY + slot));
          }
          if (!ok) break;
          ++kq;
          for (int i = 0; ok && i < nb; i += 2) {
            const int npair = nb - i < 2 ? 1 : 2;
            for (int q = 0; ok && q < npair; ++q) {   // both score buffers must be free
              const int gbq = gb + q;
              if (gbq >= 2) ok = mbar_wait(bar_addr(sb, S_FREE + (gbq & 1)), ((gbq >> 1) - 1) & 1, abort_flag, p.status);
            }
            if (!ok) break;
            SMLA_STAMP(gb - kTraceGb0, 0);
            const int b1 = gb & 1;               // a single block: its buffer and half of the unit
            int slot = n % kSRing, lap = n / kSRing;   // kept incrementally over the pair's units
#pragma unroll 1
            for (int c = 0; c < kSUnitsPerPair; ++c, ++n) {
              if (!(ok = mbar_wait(bar_addr(sb, KV_FULL + slot), lap & 1, abort_flag, p.status))) break;
              if (c == 0 || c == 3 || c == 6 || c == 8) SMLA_STAMP(gb - kTraceGb0, c == 0 ? 2 : c == 3 ? 6 : c == 6 ? 7 : 8);
              fence_proxy_async_smem();   // cp.async wrote the unit through the generic proxy
              tc_fence_after();
              // S += q K^T over chunk c (A = q from TMEM)
              if (npair == 2) {
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                  mma_bf16_ts(tmem + TM_S, tmem + TM_Q + 32 * c + 8 * ks, sdesc_add(dk0, slot * kSPairUnit + ks * 32),
                              idesc_s2, (c | ks) != 0);
              } else {
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                  mma_bf16_ts(tmem + TM_S + 64 * b1, tmem + TM_Q + 32 * c + 8 * ks,
                              sdesc_add(dk0, slot * kSPairUnit + b1 * kChunkKV + ks * 32), idesc_s1, (c | ks) != 0);
              }
              mma_commit(bar_addr(sb, KV_EMPTY + slot));
              if (++slot == kSRing) { slot = 0; ++lap; }
            }
            if (!ok) break;
            mma_commit(bar_addr(sb, S_FULL + (gb & 1)));
            if (npair == 2) mma_commit(bar_addr(sb, S_FULL + ((gb + 1) & 1)));
            SMLA_STAMP(gb - kTraceGb0, 1);
            gb += npair;
          }
          if (ok) mma_commit(bar_addr(sb, Q_EMPTY));   // q's columns may take the next token once these complete
        }
      }
      __syncwarp();
    } else if (warp == kAuxWarp) {
      if (lane == 0) {
        // P mover (a warp of its own, so that it never takes issue slots from the
        // MMA issuer): one bulk copy per block from a staging buffer into the output CTA's P buffer
        const uint32_t pbuf_peer = mapa(sb + SM_P, peer), pfull_peer = mapa(bar_addr(sb, P_FULL), peer);
        int gb = 0;
        bool ok = true;
        for (int k = 0; ok && k < ntok; ++k) {
          const int nb = read_token<false>(p, sb, smem, k, TOK_FULL_S, TOK_EMPTY_S, abort_flag);
          if (!(ok = nb >= 0)) break;
          for (int j = 0; ok && j < nb; ++j, ++gb) {
            const int sg = gb % kNS, pb = gb % kNP;
            if (!(ok = mbar_wait(bar_addr(sb, STG_FULL + sg), (gb / kNS) & 1, abort_flag, p.status))) break;
            if (gb >= kNP &&
                !(ok = mbar_wait<true>(bar_addr(sb, P_FREE + pb), ((gb / kNP) - 1) & 1, abort_flag, p.status)))
              break;
            SMLA_STAMP(gb - kTraceGb0, 11);
            bulk_s2s(pbuf_peer + pb * kPBufStride, sb + SM_STG + sg * kPBufStride, kPXBytes, pfull_peer + 8 * pb);
            bulk_commit();
            if (gb >= 1) {                       // the copy before this one has read its staging buffer
              bulk_wait_read<1>();
              mbar_arrive(bar_addr(sb, STG_FREE + (gb - 1) % kNS));
            }
          }
        }
        bulk_wait_read<0>();                     // no copy still reads this CTA's shared memory
        if (ok && gb > 0) mbar_arrive(bar_addr(sb, STG_FREE + (gb - 1) % kNS));
      }
      __syncwarp();
    } else {
      // two softmax groups, one thread per head each: group g takes the blocks whose
      // running index is g mod 2; within a token the running max and sums pass from
      // group to group through shared memory in block order
      const int g = (warp - kRowWarp0) >> 2;
      const int q4 = warp & 3;                 // TMEM lane quarter of this warp
      const int h = 32 * q4 + lane;
      const uint32_t tl = tmem + ((uint32_t)(32 * q4) << 16);
      const bool real = kAllHeads || h < p.H;
      volatile float* state = reinterpret_cast<volatile float*>(smem + SM_STATE) + 4 * h;
      if (real && ntok > 0) {                  // the first token's q row into L2
        const uint8_t* q0 = reinterpret_cast<const uint8_t*>(p.q + ((int64_t)(p.t0 + cl) * p.H + h) * kDqk);
        for (int c = g; c < 9; c += 2) prefetch_l2(q0 + 128 * c);
      }
      int gb = 0;
      bool ok = true;
      for (int k = 0; ok && k < ntok; ++k) {
        const int t = p.t0 + cl + k * ncl;
        const int nb = read_token<true>(p, sb, smem, k, TOK_FULL_S, TOK_EMPTY_S, abort_flag);
        if (!(ok = nb >= 0)) break;
        if (real && k + 1 < ntok) {            // the next token's q row into L2
          const uint8_t* qn = reinterpret_cast<const uint8_t*>(p.q + ((int64_t)(t + ncl) * p.H + h) * kDqk);
          for (int c = g; c < 9; c += 2) prefetch_l2(qn + 128 * c);
        }
        // l: sum of the fp32 exponentials (gives the LSE); the output CTA sums the
        // bf16-rounded weights itself
        float m_run = -INFINITY, l = 0.f;
        const int gb0 = gb;
        for (int j = (g - gb0) & 1; j < nb; j += 2) {
          const int gbj = gb0 + j;
          if (!(ok = __all_sync(0xffffffffu, mbar_wait(bar_addr(sb, S_FULL + g), (gbj >> 1) & 1, abort_flag, p.status))))
            break;
          tc_fence_after();
          float s[64];
          tmem_ld64(tl + TM_S + 64 * g, s);
          tc_fence_before();
          mbar_arrive(bar_addr(sb, S_FREE + g));
          if (h == 0) SMLA_STAMP(gbj - kTraceGb0, 3);
          // slot validity of this block
          const int mr = gbj % kMaskRing;
          if (!(ok = __all_sync(0xffffffffu, mbar_wait(bar_addr(sb, M_FULL + mr), (gbj / kMaskRing) & 1, abort_flag,
                                                       p.status))))
            break;
          const uint64_t mask = *reinterpret_cast<volatile uint64_t*>(smem + SM_MASK + 8 * mr);
          mbar_arrive(bar_addr(sb, M_EMPTY + mr));
          float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
          // the scale (c2 > 0) is applied to the block max here and folded into the exponent
          // below, so the raw scores are only masked
          if (mask == ~0ull) {               // no padding in the block (the common case): no selects
#pragma unroll
            for (int jj = 0; jj < 64; ++jj) mx4[jj & 3] = fmaxf(mx4[jj & 3], s[jj]);
          } else {
#pragma unroll
            for (int jj = 0; jj < 64; ++jj) {
              s[jj] = ((mask >> jj) & 1ull) ? s[jj] : -INFINITY;
              mx4[jj & 3] = fmaxf(mx4[jj & 3], s[jj]);
            }
          }
          const float mx = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3])) * p.c2;
          // the running state after the token's previous block, from the other group; at
          // a token's first block the state starts afresh, but the wait still orders this
          // group's write of the shared state after the other group's last one
          if (gbj >= 1 &&
              !(ok = __all_sync(0xffffffffu, mbar_wait(bar_addr(sb, ST_FULL + (g ^ 1)), ((gbj - 1) >> 1) & 1,
                                                       abort_flag, p.status))))
            break;
          if (j >= 1) {
            m_run = state[0]; l = state[1];
          } else {
            m_run = -INFINITY; l = 0.f;
          }
          if (h == 0) SMLA_STAMP(gbj - kTraceGb0, 4);
          float alpha = 1.f;
          uint32_t pk[32];
          if (real) {
            // lazily updated running max: move it only when the block max exceeds it by > 8 (log2 units)
            const bool move = mx > m_run + kLazyRescale;
            const float m_new = move ? mx : m_run;
            alpha = move ? ex2(m_run - m_new) : 1.f;   // m_run = -inf gives 0 (first block of a token: no O yet)
            // a listed block has a valid slot, so m_new is finite; the guard keeps
            // exp2(-inf - -inf) out regardless
            const float m_sub = (m_new == -INFINITY) ? 0.f : m_new;
            const uint64_t c2x2 = f32x2(p.c2, p.c2), nmsub2 = f32x2(-m_sub, -m_sub);
            uint64_t sum2[2] = {f32x2(0.f, 0.f), f32x2(0.f, 0.f)};
#pragma unroll
            for (int jj = 0; jj < 32; ++jj) {
              float a0, a1;
              f32x2_split(fma_f32x2(f32x2(s[2 * jj], s[2 * jj + 1]), c2x2, nmsub2), a0, a1);   // S c2 - m
              const float p0 = ex2(a0), p1 = ex2(a1);   // -inf -> 0
              sum2[jj & 1] = add_f32x2(sum2[jj & 1], f32x2(p0, p1));
              pk[jj] = pack_bf16x2(p0, p1);
            }
            float u0, u1, u2, u3;
            f32x2_split(sum2[0], u0, u1); f32x2_split(sum2[1], u2, u3);
            l = l * alpha + ((u0 + u1) + (u2 + u3));
            m_run = m_new;
          } else {
#pragma unroll
            for (int jj = 0; jj < 32; ++jj) pk[jj] = 0u;   // rows past H: P = 0, O stays 0
          }
          state[0] = m_run; state[1] = l;
          mbar_arrive(bar_addr(sb, ST_FULL + g));
          // P and alpha into a staging buffer (the P mover copies it to the output CTA)
          const int sg = gbj % kNS;
          if (gbj >= kNS && !(ok = __all_sync(0xffffffffu, mbar_wait(bar_addr(sb, STG_FREE + sg), ((gbj / kNS) - 1) & 1,
                                                                      abort_flag, p.status))))
            break;
          uint8_t* xb = smem + SM_STG + sg * kPBufStride;
#pragma unroll
          for (int c = 0; c < 8; ++c)
            *reinterpret_cast<uint4*>(xb + h * 128 + ((c ^ (h & 7)) << 4)) =
                make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
          reinterpret_cast<float*>(xb + kPBytes)[h] = alpha;
          fence_proxy_async_smem();                  // the bulk copy reads it through the async proxy
          mbar_arrive(bar_addr(sb, STG_FULL + sg));
          if (h == 0) SMLA_STAMP(gbj - kTraceGb0, 5);
        }
        if (!ok) break;
        gb = gb0 + nb;
        // the group that took the token's last block holds its final state
        const bool last = (nb == 0) ? (g == 0) : (g == ((gb - 1) & 1));
        if (last && real) p.lse[(int64_t)t * p.H + h] = l > 0.f ? (m_run + log2f(l)) * kLn2 : kLseEmpty;
      }
    }
  } else {
    // ================================================================ output CTA
    if (warp < kProducers / 32) {
      produce<kOUnitCh, kOUnits, kORing, false>(p, sb, smem, cl, ncl, abort_flag, V_FULL, V_EMPTY, TOK_FULL_O,
                                                TOK_EMPTY_O SMLA_TRACE_PASS);
    } else if (warp == kMmaWarp) {
      if (lane == 0) {
        // MMA issuer: O += P V once a block's rows are rescaled, one N = 256 tile per V unit
        const uint32_t idesc_pv = idesc_bf16(128, 256, false, true);
        const uint64_t dp0 = sdesc_sw128(sb + SM_P, 16, 1024);
        // V read MN-major from the unit: LBO = stride between 64-dim chunks, SBO = 8-row groups
        const uint64_t dv0 = sdesc_sw128(sb + SM_V, kChunkKV, 1024);
        int gb = 0, n = 0;
        bool ok = true;
        for (int k = 0; ok && k < ntok; ++k) {
          const int nb = read_token<false>(p, sb, smem, k, TOK_FULL_O, TOK_EMPTY_O, abort_flag);
          if (!(ok = nb >= 0)) break;
          // O is free once the previous token's epilogue has read it
          if (k >= 1 && nb > 0 && !(ok = mbar_wait(bar_addr(sb, O_FREE), (k - 1) & 1, abort_flag, p.status))) break;
          for (int j = 0; ok && j < nb; ++j, ++gb) {
            const int pb = gb % kNP;
            if (!(ok = mbar_wait(bar_addr(sb, R_DONE + pb), (gb / kNP) & 1, abort_flag, p.status))) break;
            SMLA_STAMP(gb - kTraceGb0, 7);
#pragma unroll 1
            for (int u = 0; u < kOUnits; ++u, ++n) {
              const int slot = n % kORing;
              if (!(ok = mbar_wait(bar_addr(sb, V_FULL + slot), (n / kORing) & 1, abort_flag, p.status))) break;
              fence_proxy_async_smem();
              tc_fence_after();
#pragma unroll
              for (int ks = 0; ks < 4; ++ks)
                mma_bf16_ss(tmem + TM_O + 256 * u, sdesc_add(dp0, pb * kPBufStride + ks * 32),
                            sdesc_add(dv0, slot * kOUnitCh * kChunkKV + ks * 16 * 128), idesc_pv, (j > 0 || ks > 0));
              mma_commit(bar_addr(sb, V_EMPTY + slot));
            }
            if (!ok) break;
            mma_commit(bar_addr(sb, PV_DONE + pb));
            SMLA_STAMP(gb - kTraceGb0, 8);
          }
        }
      }
      __syncwarp();
    } else if (warp == kAuxWarp) {
      if (lane == 0) {
        // P buffer keeper (a warp of its own, like the P mover): arms each buffer for its next block's bulk copy and tells the
        // score CTA when PV and the rows' sums have finished reading it
        const uint32_t pfree_peer = mapa(bar_addr(sb, P_FREE), peer);
        for (int b = 0; b < kNP; ++b) mbar_arrive_expect_tx(bar_addr(sb, P_FULL + b), kPXBytes);
        int gb = 0;
        bool ok = true;
        for (int k = 0; ok && k < ntok; ++k) {
          const int nb = read_token<false>(p, sb, smem, k, TOK_FULL_O, TOK_EMPTY_O, abort_flag);
          if (!(ok = nb >= 0)) break;
          for (int j = 0; ok && j < nb; ++j, ++gb) {
            const int pb = gb % kNP;
            if (!(ok = mbar_wait(bar_addr(sb, PV_DONE + pb), (gb / kNP) & 1, abort_flag, p.status))) break;
            if (!(ok = mbar_wait(bar_addr(sb, RS_DONE + pb), (gb / kNP) & 1, abort_flag, p.status))) break;
            mbar_arrive_expect_tx(bar_addr(sb, P_FULL + pb), kPXBytes);   // for block gb + kNP
            mbar_arrive_remote(pfree_peer + 8 * pb);
          }
        }
      }
      __syncwarp();
    } else if (warp < kRowWarp0 + 4) {
      // one thread per head: rescale O when the max moved, then each token's epilogue
      const int q4 = warp & 3;
      const int h = 32 * q4 + lane;
      const uint32_t tl = tmem + ((uint32_t)(32 * q4) << 16);
      const bool real = kAllHeads || h < p.H;
      int gb = 0;
      bool ok = true;
      for (int k = 0; ok && k < ntok; ++k) {
        const int t = p.t0 + cl + k * ncl;
        const int nb = read_token<true>(p, sb, smem, k, TOK_FULL_O, TOK_EMPTY_O, abort_flag);
        if (!(ok = nb >= 0)) break;
        // l_bf: sum of the bf16-rounded weights the PV MMA multiplies (normalises O, so the
        // rounding of P cancels in out), rescaled with O
        float l_bf = 0.f;
        for (int j = 0; ok && j < nb; ++j, ++gb) {
          const int pb = gb % kNP;
          if (!(ok = __all_sync(0xffffffffu, mbar_wait(bar_addr(sb, P_FULL + pb), (gb / kNP) & 1, abort_flag, p.status))))
            break;
          const float alpha = reinterpret_cast<volatile float*>(smem + SM_P + pb * kPBufStride + kPBytes)[h];
          // the running max of this head moved: O (after the previous block's PV) is scaled by alpha
          const bool resc = j >= 1 && alpha != 1.f;
          if (__any_sync(0xffffffffu, resc)) {
            if (!(ok = __all_sync(0xffffffffu, mbar_wait(bar_addr(sb, PV_DONE + (gb - 1) % kNP), ((gb - 1) / kNP) & 1,
                                                         abort_flag, p.status))))
              break;
            tc_fence_after();
            // tcgen05.ld / st are warp-collective: every lane takes part, lanes whose
            // max did not move scale by exactly 1
            const float f = resc ? alpha : 1.f;
#pragma unroll 1
            for (int part = 0; part < 8; ++part) {
              float o[64];
              tmem_ld64(tl + TM_O + 64 * part, o);
#pragma unroll
              for (int jj = 0; jj < 64; ++jj) o[jj] *= f;
              tmem_st64(tl + TM_O + 64 * part, o);
            }
            tmem_wait_st();
          }
          tc_fence_before();
          mbar_arrive(bar_addr(sb, R_DONE + pb));
          {                                      // this head's sum of the block's weights, off the PV path
            const uint4* prow = reinterpret_cast<const uint4*>(smem + SM_P + pb * kPBufStride + h * 128);
            uint64_t acc2[2] = {f32x2(0.f, 0.f), f32x2(0.f, 0.f)};
#pragma unroll
            for (int c = 0; c < 8; ++c) {
              const uint4 v = prow[c];
              acc2[0] = add_f32x2(acc2[0], f32x2(bf16_lo(v.x), bf16_hi(v.x)));
              acc2[1] = add_f32x2(acc2[1], f32x2(bf16_lo(v.y), bf16_hi(v.y)));
              acc2[0] = add_f32x2(acc2[0], f32x2(bf16_lo(v.z), bf16_hi(v.z)));
              acc2[1] = add_f32x2(acc2[1], f32x2(bf16_lo(v.w), bf16_hi(v.w)));
            }
            float a0, a1, a2, a3;
            f32x2_split(acc2[0], a0, a1);
            f32x2_split(acc2[1], a2, a3);
            l_bf = l_bf * alpha + ((a0 + a1) + (a2 + a3));
          }
          mbar_arrive(bar_addr(sb, RS_DONE + pb));
        }
        if (!ok) break;
        // epilogue of the token: O once its last PV completed
        if (nb > 0 &&
            !(ok = __all_sync(0xffffffffu, mbar_wait(bar_addr(sb, PV_DONE + (gb - 1) % kNP), ((gb - 1) / kNP) & 1,
                                                     abort_flag, p.status))))
          break;
        tc_fence_after();
        const float inv = 1.f / fmaxf(l_bf, kSumexpFloor);
        uint16_t* orow = p.out + ((int64_t)t * p.H + (real ? h : 0)) * kDv;
        const uint64_t opol = l2_evict_first_policy();   // out is written once: keep the KV rows in L2
        // every lane of the warp takes part in the warp-collective tcgen05.ld; only
        // the rows of real heads are stored
#pragma unroll 1
        for (int part = 0; part < 8; ++part) {
          float o[64];
          if (nb > 0) {
            tmem_ld64(tl + TM_O + 64 * part, o);
          } else {                             // no valid slot: no PV ever wrote O
#pragma unroll
            for (int c = 0; c < 64; ++c) o[c] = 0.f;
          }
          if (real) {
            uint4* dst = reinterpret_cast<uint4*>(orow + 64 * part);
#pragma unroll
            for (int c = 0; c < 8; ++c)
              st_v4_hint(dst + c, make_uint4(pack_bf16x2(o[8 * c] * inv, o[8 * c + 1] * inv), pack_bf16x2(o[8 * c + 2] * inv, o[8 * c + 3] * inv),
                                  pack_bf16x2(o[8 * c + 4] * inv, o[8 * c + 5] * inv), pack_bf16x2(o[8 * c + 6] * inv, o[8 * c + 7] * inv)), opol);
          }
        }
        tc_fence_before();
        mbar_arrive(bar_addr(sb, O_FREE));     // the next token's PV may overwrite O
      }
    }
  }

  // ------------------------------------------------------------ teardown
  if (*abort_flag) __nanosleep(1000000);   // let copies and MMAs already issued land
  tc_fence_before();
  __syncthreads();
  cluster_sync();   // the peer no longer touches this CTA's shared memory or barriers
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

__device__ uint32_t g_status = 0;


// Failure-detection self-test: one thread waits, through the same bounded
// wait the tensor-core kernels use, on an mbarrier that nothing arrives on.
// The wait gives up after its limit, records the timeout in the status word
// and the kernel returns normally.
__global__ void __launch_bounds__(32) wait_selftest_kernel(uint32_t* status) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait(smem_u32(&bar), 0, &abort_flag, status);
}
// Bounds-check self-test of the debug build: one gather source and one scatter
// destination that lie past the logical buffers (the first 16 elements of these
// arrays) but inside the arrays; both checks must fail, record kErrBounds and skip
// the access.  Product builds compile an empty kernel (the export refuses to run it).
#ifdef SMLA_DEBUG
__device__ __align__(16) uint16_t g_bounds_buf[64];
__device__ __align__(16) float g_bounds_fbuf[64];
#endif
__global__ void __launch_bounds__(32) bounds_selftest_kernel(uint32_t* status) {
#ifdef SMLA_DEBUG
  __shared__ __align__(16) uint16_t sdst[8];
  if (threadIdx.x == 0) {
    const uint16_t* src = g_bounds_buf + 24;
    uint32_t bytes = 16u;
    check_src(src, bytes, static_cast<const uint16_t*>(g_bounds_buf), 16, status);
    cp_async16(smem_u32(sdst), src, bytes);
    asm volatile("cp.async.wait_all;" ::: "memory");
    if (check_range(g_bounds_fbuf + 32, 4, static_cast<float*>(g_bounds_fbuf), 16, status)) g_bounds_fbuf[32] = 1.f;
  }
#else
  (void)status;
#endif
}
// exchange scratch of the tensor-core kernels (16 MiB), one slot per SM
__device__ __align__(256) float g_xchg[kXchgSlots * kXchgSlotFloats];

}  // namespace

uint32_t* tc_status_ptr() {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_status) != cudaSuccess) return nullptr;
  return static_cast<uint32_t*>(p);
}

float* tc_xchg_ptr() {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_xchg) != cudaSuccess) return nullptr;
  return static_cast<float*>(p);
}

cudaError_t read_tc_status(uint32_t* out, bool clear) {
  cudaError_t e = cudaMemcpyFromSymbol(out, g_status, sizeof(uint32_t));
  if (e == cudaSuccess && clear) {
    const uint32_t z = 0;
    e = cudaMemcpyToSymbol(g_status, &z, sizeof(z));
  }
  return e;
}

cudaError_t launch_wait_selftest(cudaStream_t s) {
  uint32_t* status = tc_status_ptr();
  if (!status) return cudaErrorInvalidSymbol;
  wait_selftest_kernel<<<1, 32, 0, s>>>(status);
  return cudaGetLastError();
}

cudaError_t launch_bounds_selftest(cudaStream_t s) {
  uint32_t* status = tc_status_ptr();
  if (!status) return cudaErrorInvalidSymbol;
  bounds_selftest_kernel<<<1, 32, 0, s>>>(status);
  return cudaGetLastError();
}

cudaError_t launch_fwd_tc(const FwdArgs& a, cudaStream_t s) {
  uint32_t* status = tc_status_ptr();
  if (!status) return cudaErrorInvalidSymbol;
  const bool all = a.H == 128;
  cudaError_t e = cudaFuncSetAttribute(all ? tc_fwd_h128_kernel<true> : tc_fwd_h128_kernel<false>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  const int nt = a.nt < 0 ? a.T : a.nt;
  if (nt == 0) return cudaSuccess;
  int dev = 0, nsm = 0;
  e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  // persistent: one cluster per pair of SMs, each walking a strided list of tokens
  const int nclusters = nt < nsm / 2 ? nt : nsm / 2;
  TcFwdParams p{a.q, a.kv, a.indices, a.out, a.lse, status, a.T, a.H, a.topk, a.t0, nt, a.scale * kLog2e};
  if (all)
    tc_fwd_h128_kernel<true><<<dim3(2 * nclusters), dim3(kThreads), kSmemBytes, s>>>(p);
  else
    tc_fwd_h128_kernel<false><<<dim3(2 * nclusters), dim3(kThreads), kSmemBytes, s>>>(p);
  return cudaGetLastError();
}

#ifdef SMLA_TRACE
extern "C" int smla_trace_setup(int tok0) {
  static const long long z[tc::kTraceCtas * tc::kTracePerCta] = {};
  if (cudaMemcpyToSymbol(tc::g_trace, z, sizeof(z)) != cudaSuccess) return -1;
  return cudaMemcpyToSymbol(tc::g_trace_tok0, &tok0, sizeof(int)) == cudaSuccess ? 0 : -1;
}
extern "C" int smla_trace_read(long long* dst) {
  return cudaMemcpyFromSymbol(dst, tc::g_trace, sizeof(long long) * tc::kTraceCtas * tc::kTracePerCta) == cudaSuccess ? 0 : -1;
}
#endif

}  // namespace smla
