/*
 * sparse_mla.h -- C ABI of the GB300 (sm_103a) sparse MLA attention library.
 *
 * DSA-style sparse MLA attention: each query token t has H heads; all heads
 * attend to the same top-k rows of one latent KV tensor (a single KV group),
 * named by an int32 index tensor in which -1 marks an unused slot.  A KV row
 * has 576 elements: a 512-wide latent part, which is also the value V, and a
 * 64-wide rope tail, which is only part of the key K.
 *
 * Sources (web pages, cited by title and section):
 *   slime issue #2201 "GLM-5.2 SparseMLA TileLang backward returns NaN
 *     gradients from finite inputs" -- "Strongest repro evidence" gives the
 *     backward call sparse_mla_bwd(q, kv, tl_out, grad_output, indices,
 *     tl_lse, sm_scale) and the outputs tl_dq / tl_dkv; "Suspected area" the
 *     D = 512 latent width and the atomic dKV accumulation.
 *   miles PR #2079 summary "fix -1 index OOB and NaN gradients in the GLM-5
 *     sparse-MLA kernel" -- implementation breakdown items 1-3 and the key
 *     code fragments of the forward `main` and `sparse_mla_bwd_kernel`:
 *     clamp + mask of -1 slots to exact-zero K/V, the 1e-30 floor on the sum
 *     of exponentials, and the clamped (no-op) dKV atomic add.
 *   Megatron-Bridge PR #17 "GLM-5 DSA option: tilelang (2/2)" -- Summary and
 *     Bug fixes: packed thd layout, top-k padded to a fixed width with -1.
 *
 * Conventions shared by every call
 *   - All tensor pointers are DEVICE pointers owned by the caller, contiguous
 *     (row-major, last index fastest) and 16-byte aligned.  The library never
 *     allocates, frees or retains them.
 *   - bf16 tensors are IEEE bfloat16 bit patterns (uint16_t storage).
 *   - T is the number of packed tokens; the query and KV token axes coincide
 *     (packed thd layout), so kv has T rows and every index addresses a row of
 *     that packed axis directly.
 *   - A top-k slot is valid iff 0 <= index < T.  -1 is the padding sentinel;
 *     any other out-of-range value is a caller error (see
 *     sparse_mla_check_indices) and is treated exactly like -1.
 *   - Supported shapes: H in {8, 16, 32, 64, 128}; topk > 0 and topk % 64 == 0;
 *     the head dims are fixed at 576 (q, k) and 512 (v, out).
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Compute calls are asynchronous on it and never synchronize
 *     the host, except sparse_mla_check_indices.
 *   - Return value: 0 on success, else a negative errno value and a message
 *     readable with sparse_mla_last_error() on the same host thread:
 *        -EINVAL  (-22) bad shape, pointer, alignment, scale or workspace size
 *        -ENOTSUP (-95) the current device is not sm_103, or a mode that is
 *                       not built
 *        -EIO     (-5)  a CUDA error was reported while launching
 *     No work is launched when the call returns -EINVAL or -ENOTSUP.
 *     Exceptions never cross this boundary.
 *   - The library needs the CUDA device that owns the pointers to be current.
 */
#ifndef SPARSE_MLA_H_
#define SPARSE_MLA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t smla_bf16_t;  /* bfloat16 bit pattern */

#define SMLA_D_QK 576          /* 512 latent + 64 rope tail */
#define SMLA_D_V 512           /* latent width = value width */
#define SMLA_DKV_ATOMIC 0         /* dKV scatter by fp32 atomic adds (order varies run to run) */
#define SMLA_DKV_DETERMINISTIC 1  /* dKV by an index-sorted segmented reduction (bitwise reproducible) */

/* fp32 LSE written for a row with no valid slot: ln(1e-30) rounded to fp32
 * (the 1e-30 floor of the miles PR #2079 forward fragment, empty max read
 * as 0). */
#define SMLA_LSE_EMPTY (-69.0775527898f)

/*
 * Forward (miles PR #2079, forward fragment `main`).
 *   q        [T, H, 576] bf16   queries (absorbed latent 512 + rope 64)
 *   kv       [T, 1, 576] bf16   latent KV rows; kv[:, :, :512] is also V
 *   indices  [T, 1, topk] int32 top-k KV rows per query, -1 = padding
 *   cu_seqlens [B+1] int32 or NULL  sequence boundaries of the packed layout;
 *            accepted for interface parity, not read by this call
 *   scale    softmax scale applied to q.k (e.g. 1/sqrt(576)); must be finite
 *   out      [T, H, 512] bf16   softmax(scale q K^T) V over the valid slots;
 *            exactly 0 for a row with no valid slot
 *   lse      [T, H] fp32        natural-log log-sum-exp of the scaled scores;
 *            SMLA_LSE_EMPTY for a row with no valid slot
 */
int sparse_mla_fwd(const smla_bf16_t* q, const smla_bf16_t* kv, const int32_t* indices,
                   const int32_t* cu_seqlens, int T, int H, int topk, int B, float scale,
                   smla_bf16_t* out, float* lse, void* stream);

/*
 * Forward over the query rows [t0, t0 + nt) only (an interface addition: the
 * pages compute all rows in one call).  Same arguments and results as
 * sparse_mla_fwd; q, indices, out and lse are still the full [T, ...]
 * arrays, of which only rows t0 .. t0 + nt - 1 are read (q, indices) or
 * written (out, lse); every kv row may be gathered.  A caller that streams
 * q to the device in pieces computes each piece as soon as it has landed.
 * The rows' results are bit-identical to those of sparse_mla_fwd.
 * Needs 0 <= t0, 0 <= nt, t0 + nt <= T (else -EINVAL); nt = 0 launches nothing.
 */
int sparse_mla_fwd_rows(const smla_bf16_t* q, const smla_bf16_t* kv, const int32_t* indices,
                        const int32_t* cu_seqlens, int T, int H, int topk, int B, float scale, int t0, int nt,
                        smla_bf16_t* out, float* lse, void* stream);

/* Bytes of device workspace sparse_mla_bwd needs for these sizes (0 if the
 * sizes are invalid).  SMLA_DKV_ATOMIC: Delta = rowsum(dO * out), [T, H] fp32.
 * SMLA_DKV_DETERMINISTIC: Delta, the kv rows' sorted slot lists (about
 * 4 * (3 T + T * topk) bytes) and the per-slot dKV contributions of one chunk of
 * query tokens (the default chunk holds 4 GiB of them; any workspace of at least
 * one token's worth is accepted, and a smaller one only means more chunks).
 * Fully overwritten by each call. */
size_t sparse_mla_bwd_workspace_bytes(int T, int H, int topk, int dkv_mode);

/*
 * Backward (slime issue #2201 "Strongest repro evidence";
 * miles PR #2079, backward fragment `sparse_mla_bwd_kernel`).
 *   q, kv, indices, cu_seqlens, scale  as for sparse_mla_fwd
 *   out      [T, H, 512] bf16   forward output (used only for Delta)
 *   dout     [T, H, 512] bf16   gradient of the loss w.r.t. out
 *   lse      [T, H] fp32        forward LSE (natural log)
 *   dkv_mode SMLA_DKV_ATOMIC: each valid slot's dKV row is added into dkv_f32
 *            with fp32 atomic adds, whose order (and so the last bits) varies
 *            from run to run.
 *            SMLA_DKV_DETERMINISTIC: the slots are first sorted by the kv row
 *            they name; dkv_f32[r] is then the fp32 sum of row r's per-slot
 *            contributions taken left to right in ascending slot order
 *            (t * topk + j), the same bits on every run and for any workspace
 *            size.  Needs T * topk <= 2^31 - 1.
 *   dq       [T, H, 576] bf16   gradient w.r.t. q; exactly 0 on empty rows
 *   dkv_f32  [T, 1, 576] fp32   gradient w.r.t. kv; zeroed and then
 *            scatter-added by this call (rows no valid slot names stay 0)
 *   dkv      [T, 1, 576] bf16 or NULL  round-to-nearest-even copy of dkv_f32
 *   workspace, workspace_bytes  device scratch of at least
 *            sparse_mla_bwd_workspace_bytes(T, H, topk, dkv_mode) bytes,
 *            owned by the caller; it must not be used by another call that
 *            runs concurrently on the GPU
 */
int sparse_mla_bwd(const smla_bf16_t* q, const smla_bf16_t* kv, const smla_bf16_t* out,
                   const smla_bf16_t* dout, const float* lse, const int32_t* indices,
                   const int32_t* cu_seqlens, int T, int H, int topk, int B, float scale,
                   int dkv_mode, smla_bf16_t* dq, float* dkv_f32, smla_bf16_t* dkv,
                   void* workspace, size_t workspace_bytes, void* stream);

/*
 * Backward contribution of the query rows [t0, t0 + nt) (an interface
 * addition for callers that stream the step through the device in pieces),
 * with dKV accumulated by fp32 atomic adds (SMLA_DKV_ATOMIC).
 *   q, kv, out, dout, lse, indices, cu_seqlens, scale  as for sparse_mla_bwd
 *            (full [T, ...] arrays; only rows t0 .. t0 + nt - 1 of q, out,
 *            dout, lse and indices are read)
 *   dq       rows t0 .. t0 + nt - 1 of [T, H, 576] bf16 are written, bit-
 *            identical to those of sparse_mla_bwd
 *   dkv_f32  [T, 1, 576] fp32: the rows' dKV contributions are ADDED; the
 *            caller zeroes it once before the first range (e.g. with
 *            cudaMemsetAsync) and may then cast it with sparse_mla_dkv_cast.
 *            After all ranges of a step it equals sparse_mla_bwd's dkv_f32 up
 *            to the order of the fp32 additions.
 *   workspace, workspace_bytes  at least
 *            sparse_mla_bwd_workspace_bytes(T, H, topk, SMLA_DKV_ATOMIC) bytes;
 *            Delta of row t is kept at row t, so ranges that do not overlap
 *            may share one workspace, on one stream or on several.
 * Needs 0 <= t0, 0 <= nt, t0 + nt <= T (else -EINVAL); nt = 0 launches nothing.
 */
int sparse_mla_bwd_rows(const smla_bf16_t* q, const smla_bf16_t* kv, const smla_bf16_t* out,
                        const smla_bf16_t* dout, const float* lse, const int32_t* indices,
                        const int32_t* cu_seqlens, int T, int H, int topk, int B, float scale, int t0, int nt,
                        smla_bf16_t* dq, float* dkv_f32, void* workspace, size_t workspace_bytes, void* stream);

/* dkv [T, 1, 576] bf16 = round-to-nearest-even of dkv_f32 [T, 1, 576] fp32
 * (the cast sparse_mla_bwd applies when its dkv is not NULL). */
int sparse_mla_dkv_cast(const float* dkv_f32, smla_bf16_t* dkv, int T, void* stream);

/*
 * Backward that allocates nothing (the pages have no counterpart: this is an
 * interface addition for callers that cannot call cudaMalloc: code running
 * inside a memory allocator's own callbacks, where allocating would re-enter
 * the allocator, and services whose device memory is fixed at start-up).
 *
 * Same arguments, results and error codes as sparse_mla_bwd with
 * dkv_mode = SMLA_DKV_ATOMIC, minus the workspace: the Delta scratch lives in
 * a fixed device array inside the library, 2^23 fp32 values (32 MiB), which
 * every GPU that loads the library holds until the process exits.
 *   - T * H must be <= 8,388,608 (e.g. T = 65536 at H = 128); larger sizes
 *     return -EINVAL with a message and launch nothing.
 *   - No cudaMalloc, cudaFree or other allocating call is made.  Every call
 *     looks up the device address of the array for the current device (a
 *     runtime query that allocates nothing); the first call on a device may
 *     also load the library's kernels there, so make that first call before
 *     any stream capture.
 *   - All calls share the one array and it keeps the last call's contents
 *     (each call rewrites the part it uses before reading it).  Calls that
 *     overlap on the GPU -- on different streams, or from different host
 *     threads -- race on it and must be serialised by the caller.
 */
int sparse_mla_bwd_noalloc(const smla_bf16_t* q, const smla_bf16_t* kv, const smla_bf16_t* out,
                           const smla_bf16_t* dout, const float* lse, const int32_t* indices,
                           const int32_t* cu_seqlens, int T, int H, int topk, int B, float scale,
                           smla_bf16_t* dq, float* dkv_f32, smla_bf16_t* dkv, void* stream);

/*
 * Index validation (Megatron-Bridge PR #17, Bug fixes: top-k padded with
 * -1).  Counts the entries of indices [T, 1, topk] that are neither -1 nor a
 * row of their own query's sequence [cu_seqlens[b], cu_seqlens[b+1]).
 * cu_seqlens [B+1] int32 (device) must start at 0, be non-decreasing and end
 * at T.  Writes the count to *n_bad (HOST pointer).  The count is taken in a
 * counter word inside the library (one per device, nothing is allocated);
 * the call synchronizes `stream` before it returns and holds a host lock
 * meanwhile, so calls from several host threads run one after another.
 */
int sparse_mla_check_indices(const int32_t* indices, int T, int topk, const int32_t* cu_seqlens,
                             int B, int64_t* n_bad, void* stream);

/*
 * Top-k index selection that produces `indices` for the calls above
 * (Megatron-Bridge PR #17, "GLM-5 DSA option: tilelang (2/2)", Summary and Bug
 * fixes: the indexer's top-k is capped at the keys a query can see in its own
 * sequence and padded to the fixed width with -1).
 *   scores   [T, ld] fp32 (device): row t scores its causal candidates, the rows
 *            s0 .. t of its own sequence, in columns 0 .. t - s0 (s0 = start of
 *            t's sequence); columns past t - s0 are not read
 *   ncols    columns that may hold candidates (a longer sequence is capped at
 *            its first ncols keys); ncols <= ld
 *   cu_seqlens [B+1] int32 (device): 0 = cu[0] <= cu[1] <= ... <= cu[B] = T
 *   topk     width of each index row, 1 .. 8192
 *   indices  [T, 1, topk] int32 (device, written): the k = min(topk, t - s0 + 1,
 *            ncols) best candidates as packed kv rows s0 + c, in descending
 *            score order (equal scores by ascending c; NaN scores last),
 *            then -1
 * Needs 4 * (ncols + 3) + 8 * max(1024, topk rounded up to a power of two)
 * <= 220 KiB of shared memory (e.g. ncols 32768 with topk 8192), else -EINVAL.
 * Asynchronous on `stream`.  The pages have no kernel for this step beyond the
 * padding rule; one CTA per row selects by a radix select in shared memory and
 * sorts the selection with a bitonic network.
 */
int sparse_mla_topk(const float* scores, int64_t ld, int T, int ncols, const int32_t* cu_seqlens, int B, int topk,
                    int32_t* indices, void* stream);

/* Message of the last failed call on this host thread ("" if none). */
const char* sparse_mla_last_error(void);

/* Library version string. */
const char* sparse_mla_version(void);

/* Reads the device status word of the library's kernels on the current
 * device into *status (HOST pointer): 0 = every bounded wait inside the
 * tensor-core kernels completed (and, in the debug build, every bounds check
 * passed); 1 = some wait gave up after its time limit, the kernel returned
 * early and the outputs of that call are not valid; 2 = (debug build only) a
 * gathered row or scatter address fell outside its buffer and that access was
 * skipped, so the outputs are not valid.  The first error is kept.  With
 * clear != 0 the word is reset to 0.  Synchronizes with the device. */
int sparse_mla_device_status(uint32_t* status, int clear);

/* Failure-detection self-test (no counterpart in the source pages).  Enqueues
 * on `stream` one small kernel whose single thread waits, through the same
 * bounded wait the tensor-core kernels use, on a barrier that nothing ever
 * releases.  After the wait limit (1 s) the wait gives up, sets the status
 * word read by sparse_mla_device_status to 1 and the kernel returns normally:
 * the CUDA context stays usable.  Callers clear the status word afterwards
 * (sparse_mla_device_status(&s, 1)); until then it also reports 1 for the
 * other kernels.  Returns 0, or -EINVAL / -EIO as the other calls. */
int sparse_mla_wait_selftest(void* stream);

/* Bounds-check self-test (no counterpart in the source pages; the library's
 * debug build, compiled with -DSMLA_DEBUG, checks every 16-byte gather source
 * and every scatter destination against its buffer before the access, records
 * status 2 on a failure and skips the access, never trapping).  Enqueues on
 * `stream` one small kernel whose checks probe addresses past a logical buffer
 * (but inside its allocation): both must fail, so the status word becomes 2
 * and nothing is read or written there.  Returns 0 in the debug build,
 * -ENOSYS in the product build (whose checks compile to nothing), or -EINVAL /
 * -EIO as the other calls. */
int sparse_mla_bounds_selftest(void* stream);

/* Number of CUDA kernels this process has launched through the library so
 * far (all threads, all devices).  Diagnostics only: benchmarks read it
 * before and after a timed region to count the library's launches. */
uint64_t sparse_mla_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* SPARSE_MLA_H_ */
