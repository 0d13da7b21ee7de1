// Tensor-core (tcgen05) forward for up to 128 heads (fewer heads run as a
// 128-row tile whose rows past H are zero).
//
// Work split: a cluster of two CTAs handles one query token.  The 576-wide
// key dimension is split between them (CTA 0: dims [0,256), CTA 1: dims
// [256,576)), and so is the 512-wide value/output dimension (CTA 0: [0,256),
// CTA 1: [256,512)).  Each CTA gathers only its own columns of the named KV
// rows, so the pair reads every gathered byte exactly once, and each CTA
// holds an O accumulator of 128 heads x 256 dims (256 TMEM columns).  The
// partial scores of the two halves are exchanged through an L2 scratch and
// summed in both CTAs (a + b == b + a, so both see bit-identical scores and
// take identical softmax decisions).
//
// Per block of 64 top-k slots:
//   producer warps: read the 64 indices (one block ahead), mask them (valid
//                   iff 0 <= idx < T) and gather this CTA's columns of the
//                   named rows with 16-byte cp.async into 128B-swizzled shared
//                   memory; a padding slot copies zero bytes and gets an
//                   exact-zero K/V row (the clamp + mask of the miles PR #2079
//                   fix, implementation breakdown item 2);
//   MMA thread    : S_half = Q_half K_half^T  (M=128 heads, N=64, K=256|320)
//                   into one of two TMEM score buffers, and O += P V_half
//                   (M=128, N=256, K=64), each issued as soon as its inputs
//                   are ready;
//   two groups of four warps, one thread per head, take alternate blocks:
//                   load the 64 partial scores, write them to this SM's slot
//                   of the L2 exchange scratch, signal the peer CTA through
//                   its mbarrier, add the peer's partials, mask padding to
//                   -inf and run the online softmax in the exp2 domain with a
//                   lazily updated running max (handed from group to group
//                   through shared memory), rescale O in TMEM when the max
//                   moves, and write P (bf16) for the PV MMA.  One group's
//                   exchange overlaps the other's softmax.  At the end the sum
//                   of exponentials is floored at 1e-30 (PR #2079 forward
//                   fragment), so a row with no valid slot gets out = 0 and
//                   LSE = ln(1e-30).
#include <cuda.h>

#include "smla_common.cuh"
#include "tc_common.cuh"

namespace smla {
namespace {

using namespace tc;

constexpr int kBK = 64;                 // slots per block
constexpr int kProducers = 64;          // warps 0..1 gather, warp 2 MMA, warps 3..10 two exchange + softmax groups
constexpr int kMmaWarp = 2;
constexpr int kGroup0 = 3;
constexpr int kRowsPerProducer = kBK * 8 / kProducers;   // 8 rows, one 16-byte piece of each chunk
constexpr int kThreads = kProducers + 32 + 128 + 128;
constexpr int kChunkKV = kBK * 128;     // one 64-dim chunk of a KV block
constexpr int kStageBytes = 5 * kChunkKV;
constexpr float kLazyRescale = 8.f;     // log2-domain slack before O is rescaled
constexpr int kMaxBlocks = kTcMaxTopk / kBK;

// shared memory map (offsets from a 1024-aligned base); Q lives in TMEM
constexpr int kStages = 5;
constexpr int SM_KV = 0;                           // kStages stages
constexpr int SM_P = SM_KV + kStages * kStageBytes;
constexpr int SM_MASK = SM_P + 128 * 128;          // kStages x u64
constexpr int SM_STATE = SM_MASK + 8 * kStages;    // running max and sums, 128 heads x float4
constexpr int SM_BFLAG = SM_STATE + 128 * 16;      // per block: holds a valid slot (u8)
constexpr int SM_BLIST = SM_BFLAG + kMaxBlocks;     // blocks with a valid slot, in order (u16)
constexpr int SM_NB = SM_BLIST + 2 * kMaxBlocks;    // their number
constexpr int SM_BAR = SM_NB + 8;
// S_FULL, X_FULL, X_EMPTY, ST_FULL and O_DONE come in pairs indexed by block parity:
// each is then waited on only by one group, one phase at a time
enum Bar { KV_FULL = 0, KV_EMPTY = kStages, Q_FULL = 2 * kStages, S_FULL, S_FREE = S_FULL + 2, X_FULL,
           X_EMPTY = X_FULL + 2, ST_FULL = X_EMPTY + 2, P_FULL = ST_FULL + 2, O_DONE, NBAR = O_DONE + 2 };
constexpr int SM_TMEM = SM_BAR + 8 * NBAR;
constexpr int SM_SMID = SM_TMEM + 4;
constexpr int SM_ABORT = SM_SMID + 4;
constexpr int kSmemBytes = SM_ABORT + 4 + 1024;     // + alignment slack
static_assert(kSmemBytes <= 232448, "shared memory budget");
static_assert(kSmemBytes > 232448 / 2, "one CTA per SM: the exchange scratch is indexed by SM");

constexpr uint32_t kTmemCols = 512;
constexpr uint32_t TM_O = 0;            // O: 256 columns
constexpr uint32_t TM_S = 256;          // partial then full scores of one block: 64 columns
constexpr uint32_t TM_Q = 320;          // this CTA's q slice, bf16 pairs: 128 | 160 columns
static_assert(SM_P % 1024 == 0, "swizzle atoms");

struct TcFwdParams {
  const uint16_t* q;                    // [T, H, 576] bf16
  const uint16_t* kv;                   // [T, 576] bf16
  float* xchg;                          // exchange scratch, kXchgSlots slots
  const int32_t* indices;
  uint16_t* out;
  float* lse;
  uint32_t* status;
  int T, H, topk;                       // H <= 128 heads; rows H..127 of the tile are zero
  int t0;                               // this launch handles query rows t0, t0 + 1, ...
  float c2;                             // scale * log2(e)
};

__device__ __forceinline__ uint32_t bar_addr(uint32_t base, int i) { return base + SM_BAR + 8 * i; }

// kAllHeads: H == 128, no padding rows (the exchange then has no per-row test)
template <bool kAllHeads>
__global__ void __launch_bounds__(kThreads, 1) __cluster_dims__(2, 1, 1)
    tc_fwd_h128_kernel(TcFwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);   // 1024-aligned (128B swizzle atoms)
  const uint32_t sb = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t crank = cluster_ctarank();          // 0 or 1
  const uint32_t peer = crank ^ 1u;
  const int t = p.t0 + (blockIdx.x >> 1);
  const int nch = 4 + (int)crank;                     // 64-dim key chunks of this CTA
  const int g0 = 4 * (int)crank;                      // first global chunk
  const int nblk = p.topk / kBK;           // blocks of the token's slot list
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + SM_ABORT);

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    for (int k = 0; k < kStages; ++k) {
      mbar_init(bar_addr(sb, KV_FULL + k), kProducers + 1);   // cp.async arrivals + the slot mask
      mbar_init(bar_addr(sb, KV_EMPTY + k), 1);
    }
    mbar_init(bar_addr(sb, Q_FULL), 256);       // both groups stored their part of q into TMEM
    mbar_init(bar_addr(sb, S_FULL + 0), 1);
    mbar_init(bar_addr(sb, S_FULL + 1), 1);
    mbar_init(bar_addr(sb, S_FREE), 128);       // a group loaded the partial scores into registers
    mbar_init(bar_addr(sb, ST_FULL + 0), 128);  // the group wrote the running state after its block
    mbar_init(bar_addr(sb, ST_FULL + 1), 128);
    mbar_init(bar_addr(sb, X_FULL + 0), 128);   // the peer's 128 threads wrote their partial rows
    mbar_init(bar_addr(sb, X_FULL + 1), 128);
    mbar_init(bar_addr(sb, X_EMPTY + 0), 128);  // the peer's 128 threads read ours
    mbar_init(bar_addr(sb, X_EMPTY + 1), 128);
    mbar_init(bar_addr(sb, P_FULL), 128);
    mbar_init(bar_addr(sb, O_DONE + 0), 1);
    mbar_init(bar_addr(sb, O_DONE + 1), 1);
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
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + SM_TMEM);
  // blocks that hold only padding contribute nothing and are skipped: list the
  // others in order (both CTAs of the pair read the same indices and agree)
  const int16_t* blist = reinterpret_cast<const int16_t*>(smem + SM_BLIST);
  const int nb = build_block_list<kBK>(p.indices + (int64_t)t * p.topk, nblk, p.T, smem + SM_BFLAG,
                                  reinterpret_cast<int16_t*>(smem + SM_BLIST), reinterpret_cast<int*>(smem + SM_NB));

  if (warp < kProducers / 32) {
    // ------------------------------------------------------------ producers
    const int pt = threadIdx.x;              // 0..63
    // thread pt copies 16-byte piece c16 of rows r0 + 8 j of every chunk
    const int c16 = pt & 7, r0 = pt >> 3;
    constexpr int RS = kProducers / 8;       // row stride between a thread's rows
    const int32_t* irow = p.indices + (int64_t)t * p.topk;
    const uint16_t* kvc = p.kv + 64 * g0 + 8 * c16;
    int nxt[kRowsPerProducer], nm[2];
    if (nb > 0) {
      const int32_t* ib = irow + blist[0] * kBK;
#pragma unroll
      for (int j = 0; j < kRowsPerProducer; ++j) nxt[j] = __ldg(ib + r0 + RS * j);
      if (warp == 0) { nm[0] = __ldg(ib + lane); nm[1] = __ldg(ib + 32 + lane); }
    }
    for (int i = 0; i < nb; ++i) {
      const int st = i % kStages, use = i / kStages;
      int cur[kRowsPerProducer], cm[2];
#pragma unroll
      for (int j = 0; j < kRowsPerProducer; ++j) cur[j] = nxt[j];
      cm[0] = nm[0]; cm[1] = nm[1];
      if (i + 1 < nb) {                      // indices of the next block, one block ahead
        const int32_t* ib = irow + blist[i + 1] * kBK;
#pragma unroll
        for (int j = 0; j < kRowsPerProducer; ++j) nxt[j] = __ldg(ib + r0 + RS * j);
        if (warp == 0) { nm[0] = __ldg(ib + lane); nm[1] = __ldg(ib + 32 + lane); }
      }
      if (use >= 1 && !__all_sync(0xffffffffu, mbar_wait(bar_addr(sb, KV_EMPTY + st), (use - 1) & 1, abort_flag,
                                                        p.status)))
        break;                                 // warp-uniform exit
      const uint32_t stage = sb + SM_KV + st * kStageBytes;
#pragma unroll
      for (int j = 0; j < kRowsPerProducer; ++j) {
        const int r = r0 + RS * j;
        const bool v = cur[j] >= 0 && cur[j] < p.T;
        const uint16_t* src = kvc + (int64_t)(v ? cur[j] : 0) * kDqk;
        const uint32_t dst = stage + r * 128 + ((c16 ^ (r & 7)) << 4);
        for (int k = 0; k < nch; ++k) cp_async16(dst + k * kChunkKV, src + 64 * k, v ? 16u : 0u);
      }
      cp_async_arrive(bar_addr(sb, KV_FULL + st));
      if (warp == 0) {                        // slot validity mask of the block for the softmax warps
        const uint32_t ma = __ballot_sync(0xffffffffu, cm[0] >= 0 && cm[0] < p.T);
        const uint32_t mb = __ballot_sync(0xffffffffu, cm[1] >= 0 && cm[1] < p.T);
        if (lane == 0) {
          *reinterpret_cast<volatile uint64_t*>(smem + SM_MASK + 8 * st) = (uint64_t)ma | ((uint64_t)mb << 32);
          mbar_arrive(bar_addr(sb, KV_FULL + st));
        }
      }
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    // Event driven: the score MMAs of block i are issued as soon as its KV stage
    // has landed and its TMEM score buffer is free, the PV MMA of block j as soon
    // as P(j) is written, whichever comes first.
    if (lane == 0) {
      const uint32_t idesc_s = idesc_bf16(128, kBK, false, false);
      const uint32_t idesc_pv = idesc_bf16(128, 256, false, true);
      // base descriptors; per-MMA descriptors only move the start address
      const uint64_t dk0 = sdesc_sw128(sb + SM_KV, 16, 1024);
      const uint64_t dp0 = sdesc_sw128(sb + SM_P, 16, 1024);
      // V is the first four chunks of the stage, read MN-major:
      // LBO = stride between 64-dim chunks, SBO = stride between 8-row groups
      const uint64_t dv0 = sdesc_sw128(sb + SM_KV, kChunkKV, 1024);
      bool ok = mbar_wait(bar_addr(sb, Q_FULL), 0, abort_flag, p.status);
      tc_fence_after();
      int ns = 0, npv = 0;                    // next block for the score MMAs / for PV
      unsigned long long idle_since = 0;
      while (ok && npv < nb) {
        bool progress = false;
        if (ns < nb) {
          const int st = ns % kStages;
          if (mbar_try_wait(bar_addr(sb, KV_FULL + st), (ns / kStages) & 1) &&
              (ns < 1 || mbar_try_wait(bar_addr(sb, S_FREE), (ns - 1) & 1))) {
            fence_proxy_async_smem();   // cp.async wrote the stage through the generic proxy
            tc_fence_after();
#pragma unroll
            for (int k = 0; k < 5; ++k) {
              if (k < nch) {
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                  mma_bf16_ts(tmem + TM_S, tmem + TM_Q + 32 * k + 8 * ks,
                              sdesc_add(dk0, st * kStageBytes + k * kChunkKV + ks * 32), idesc_s, (k | ks) != 0);
              }
            }
            mma_commit(bar_addr(sb, S_FULL + (ns & 1)));
            ++ns;
            progress = true;
          }
        }
        if (npv < ns && mbar_try_wait(bar_addr(sb, P_FULL), npv & 1)) {
          const int stj = npv % kStages;
          tc_fence_after();
#pragma unroll
          for (int ks = 0; ks < 4; ++ks)
            mma_bf16_ss(tmem + TM_O, sdesc_add(dp0, ks * 32), sdesc_add(dv0, stj * kStageBytes + ks * 16 * 128),
                        idesc_pv, (npv > 0 || ks > 0));
          mma_commit(bar_addr(sb, O_DONE + (npv & 1)));
          mma_commit(bar_addr(sb, KV_EMPTY + stj));
          ++npv;
          progress = true;
        }
        if (progress) {
          idle_since = 0;
        } else if (*abort_flag) {
          break;
        } else {
          const unsigned long long now = globaltimer();
          if (idle_since == 0) {
            idle_since = now;
          } else if (now - idle_since > kWaitLimitNs) {
            *abort_flag = 1;
            atomicCAS(p.status, 0u, kErrWaitTimeout);
            break;
          }
        }
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ exchange + softmax
    // Two groups of four warps take alternate blocks (group g: blocks i = g mod 2)
    // so that one group's score exchange overlaps the other's softmax.  The
    // running max and the two sums pass from group to group through shared
    // memory, in block order.
    const int g = (warp - kGroup0) >> 2;
    const int q4 = warp & 3;                 // TMEM lane quarter of this warp
    const int h = 32 * q4 + lane;            // head == TMEM lane
    const uint32_t tl = tmem + ((uint32_t)(32 * q4) << 16);
    uint8_t* prow = smem + SM_P + h * 128;
    volatile float* state = reinterpret_cast<volatile float*>(smem + SM_STATE) + 4 * h;
    const uint32_t xfull_peer = mapa(bar_addr(sb, X_FULL), peer);
    const uint32_t xempty_peer = mapa(bar_addr(sb, X_EMPTY), peer);
    // exchange slots of this CTA's SM and of the peer's SM
    const uint32_t peer_sm = ld_cluster_u32(mapa(sb + SM_SMID, peer));
    const uint32_t my_sm = *reinterpret_cast<volatile uint32_t*>(smem + SM_SMID);
    float4* xmine = reinterpret_cast<float4*>(p.xchg + (size_t)(my_sm % kXchgSlots) * kXchgSlotFloats) + h;
    const float4* xpeer = reinterpret_cast<const float4*>(p.xchg + (size_t)(peer_sm % kXchgSlots) * kXchgSlotFloats) + h;
    // l: sum of the fp32 exponentials (gives the LSE); l_bf: sum of the bf16-rounded
    // weights fed to the PV MMA (normalises O, so the rounding of P cancels in out)
    float m_run = -INFINITY, l = 0.f, l_bf = 0.f;
    // this CTA's q slice into TMEM (the A operand of the score MMAs): head h in
    // lane h, dims packed two per column; group g stores chunks g, g+2, ...
    {
      const bool real = h < p.H;             // heads past H are zero rows of the tile
      const uint4* qrow = reinterpret_cast<const uint4*>(p.q + ((int64_t)t * p.H + (real ? h : 0)) * kDqk + 64 * g0);
      for (int k = g; k < nch; k += 2) {
        uint4 v[8];
#pragma unroll
        for (int c = 0; c < 8; ++c) v[c] = real ? __ldg(qrow + 8 * k + c) : make_uint4(0u, 0u, 0u, 0u);
        tmem_st32(tl + TM_Q + 32 * k, reinterpret_cast<const float*>(v));
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar_addr(sb, Q_FULL));
    }
    bool ok = true;
    for (int i = g; i < nb; i += 2) {
      const int b = g, st = i % kStages, k2 = i >> 1;
      // own partial scores; the TMEM buffer is free again once they are in registers
      if (!(ok = __all_sync(0xffffffffu, mbar_wait(bar_addr(sb, S_FULL + b), k2 & 1, abort_flag, p.status)))) break;
      tc_fence_after();
      float s[64];
      tmem_ld64(tl + TM_S, s);
      tc_fence_before();
      mbar_arrive(bar_addr(sb, S_FREE));
      // publish them to the peer, then add the peer's
      if (k2 >= 1 && !(ok = __all_sync(0xffffffffu, mbar_wait<true>(bar_addr(sb, X_EMPTY + b), (k2 - 1) & 1, abort_flag,
                                                                   p.status))))
        break;
      // rows past H (zero q rows: their partial scores are exactly 0 on both
      // CTAs) skip the exchange; every thread still arrives
      const bool xreal = kAllHeads || h < p.H;
      float4* wr = xmine + b * (kXchgBufFloats / 4);
      if (xreal) {
#pragma unroll
        for (int v4 = 0; v4 < 16; ++v4) wr[v4 * 128] = make_float4(s[4 * v4], s[4 * v4 + 1], s[4 * v4 + 2], s[4 * v4 + 3]);
      }
      mbar_arrive_remote(xfull_peer + 8 * b);     // release: the rows are visible to the peer
      if (!(ok = __all_sync(0xffffffffu, mbar_wait<true>(bar_addr(sb, X_FULL + b), k2 & 1, abort_flag, p.status))))
        break;
      const float4* rd = xpeer + b * (kXchgBufFloats / 4);
      if (xreal) {
#pragma unroll
        for (int v4 = 0; v4 < 16; ++v4) {
          const float4 o = ld_cg_v4(rd + v4 * 128);
          s[4 * v4] += o.x; s[4 * v4 + 1] += o.y; s[4 * v4 + 2] += o.z; s[4 * v4 + 3] += o.w;
        }
      }
      mbar_arrive_remote(xempty_peer + 8 * b);    // the peer may reuse that buffer
      // slot validity of this block (written by the producer before it armed KV_FULL)
      if (!(ok = __all_sync(0xffffffffu, mbar_wait(bar_addr(sb, KV_FULL + st), (i / kStages) & 1, abort_flag, p.status)))) break;
      const uint64_t mask = *reinterpret_cast<volatile uint64_t*>(smem + SM_MASK + 8 * st);
      float mx = -INFINITY;
#pragma unroll
      for (int j = 0; j < 64; ++j) {
        s[j] = ((mask >> j) & 1ull) ? s[j] * p.c2 : -INFINITY;
        mx = fmaxf(mx, s[j]);
      }
      // running state after block i-1, from the other group
      if (i >= 1) {
        if (!(ok = __all_sync(0xffffffffu, mbar_wait(bar_addr(sb, ST_FULL + (g ^ 1)), ((i - 1) >> 1) & 1, abort_flag,
                                                     p.status))))
          break;
        m_run = state[0]; l = state[1]; l_bf = state[2];
      }
      // lazily updated running max: move it only when the block max exceeds it by > 8 (log2 units)
      const bool move = mx > m_run + kLazyRescale;
      const float m_new = move ? mx : m_run;
      const float alpha = move ? ex2(m_run - m_new) : 1.f;   // m_run = -inf gives 0
      // while no valid slot has been seen m_new is -inf; subtract 0 instead so
      // that padding gives exp2(-inf) = 0 and never exp2(-inf - -inf) = NaN
      const float m_sub = (m_new == -INFINITY) ? 0.f : m_new;
      float sum = 0.f, sum_bf = 0.f;
      uint32_t pk[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const float p0 = ex2(s[2 * j] - m_sub), p1 = ex2(s[2 * j + 1] - m_sub);   // -inf -> 0
        sum += p0 + p1;
        pk[j] = pack_bf16x2(p0, p1);
        sum_bf += bf16_lo(pk[j]) + bf16_hi(pk[j]);    // the weights the PV MMA actually uses
      }
      l = l * alpha + sum;
      l_bf = l_bf * alpha + sum_bf;
      m_run = m_new;
      state[0] = m_run; state[1] = l; state[2] = l_bf;
      mbar_arrive(bar_addr(sb, ST_FULL + g));
      // P buffer and O are free once the previous PV has completed
      if (i >= 1 && !(ok = __all_sync(0xffffffffu, mbar_wait(bar_addr(sb, O_DONE + (b ^ 1)), ((i - 1) >> 1) & 1, abort_flag,
                                                             p.status))))
        break;
      tc_fence_after();
      if (i >= 1 && __any_sync(0xffffffffu, move)) {
#pragma unroll 1
        for (int part = 0; part < 8; ++part) {
          float o[32];
          tmem_ld32(tl + TM_O + 32 * part, o);
#pragma unroll
          for (int j = 0; j < 32; ++j) o[j] *= alpha;
          tmem_st32(tl + TM_O + 32 * part, o);
        }
        tmem_wait_st();
      }
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const uint4 v = make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
        *reinterpret_cast<uint4*>(prow + ((c ^ (h & 7)) << 4)) = v;
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(bar_addr(sb, P_FULL));
    }
    // the group that took the last block holds the final state and writes the outputs
    const bool last = (nb == 0) ? (g == 0) : (g == ((nb - 1) & 1));
    if (ok && last && nb > 0)
      ok = __all_sync(0xffffffffu, mbar_wait(bar_addr(sb, O_DONE + ((nb - 1) & 1)), ((nb - 1) >> 1) & 1, abort_flag,
                                             p.status));
    tc_fence_after();
    if (ok && last) {
      const float inv = 1.f / fmaxf(l_bf, kSumexpFloor);
      const bool real = h < p.H;
      uint16_t* orow = p.out + ((int64_t)t * p.H + h) * kDv + 256 * crank;
#pragma unroll 1
      for (int part = 0; part < 8; ++part) {
        float o[32];
        if (nb > 0) {
          tmem_ld32(tl + TM_O + 32 * part, o);
        } else {                             // no valid slot: no PV ever wrote O
#pragma unroll
          for (int c = 0; c < 32; ++c) o[c] = 0.f;
        }
        uint4* dst = reinterpret_cast<uint4*>(orow + 32 * part);
        if (real) {
#pragma unroll
          for (int c = 0; c < 4; ++c)
            dst[c] = make_uint4(pack_bf16x2(o[8 * c] * inv, o[8 * c + 1] * inv), pack_bf16x2(o[8 * c + 2] * inv, o[8 * c + 3] * inv),
                                pack_bf16x2(o[8 * c + 4] * inv, o[8 * c + 5] * inv), pack_bf16x2(o[8 * c + 6] * inv, o[8 * c + 7] * inv));
        }
      }
      if (crank == 0 && real) p.lse[(int64_t)t * p.H + h] = l > 0.f ? (m_run + log2f(l)) * kLn2 : kLseEmpty;
    }
  }

  // ------------------------------------------------------------ teardown
  if (*abort_flag) __nanosleep(1000000);   // let copies and MMAs already issued land
  tc_fence_before();
  __syncthreads();
  cluster_sync();   // the peer no longer touches this CTA's shared memory
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

cudaError_t launch_fwd_tc(const FwdArgs& a, cudaStream_t s) {
  uint32_t* status = tc_status_ptr();
  if (!status) return cudaErrorInvalidSymbol;
  const bool all = a.H == 128;
  cudaError_t e = cudaFuncSetAttribute(all ? tc_fwd_h128_kernel<true> : tc_fwd_h128_kernel<false>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  float* xchg = tc_xchg_ptr();
  if (!xchg) return cudaErrorInvalidSymbol;
  const int nt = a.nt < 0 ? a.T : a.nt;
  if (nt == 0) return cudaSuccess;
  TcFwdParams p{a.q, a.kv, xchg, a.indices, a.out, a.lse, status, a.T, a.H, a.topk, a.t0, a.scale * kLog2e};
  if (all)
    tc_fwd_h128_kernel<true><<<dim3(2 * nt), dim3(kThreads), kSmemBytes, s>>>(p);
  else
    tc_fwd_h128_kernel<false><<<dim3(2 * nt), dim3(kThreads), kSmemBytes, s>>>(p);
  return cudaGetLastError();
}

}  // namespace smla
