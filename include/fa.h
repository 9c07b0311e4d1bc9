/*
 * fa.h -- C ABI of the GB300 (sm_103a) exact attention forward library.
 *
 * The operation (FlashAttention v4 Blackwell pipeline diagram, pseudo-code
 * panel; FlashAttention v2 work-partitioning diagram, pseudo-code panel; the
 * "flash attention v2 论文" search page, which states the result is exact
 * attention, not an approximation):
 *
 *   O[b,h,i,:] = sum_{j in A(i)} softmax_j(scale * <Q[b,h,i,:], K[b,h,j,:]>) V[b,h,j,:]
 *   LSE[b,h,i] = ln sum_{j in A(i)} exp(scale * <Q[b,h,i,:], K[b,h,j,:]>)
 *
 * with A(i) = {0..N-1}, or {0..i} when causal.  The scores S and the
 * probabilities P are computed tile by tile on chip with the online-softmax
 * recurrence and never written to memory.
 *
 * Layout (all entry points): q, k, v, o are dense, contiguous, row-major
 * [B, H, N, d] arrays of 16-bit elements; element (b,h,n,c) is at index
 * ((b*H + h)*N + n)*d + c.  lse is a dense [B, H, N] fp32 array.  Q, K and V
 * share N (self-attention shape).  Every pointer is a DEVICE pointer on the
 * current CUDA device.
 *
 * Ownership: the caller allocates and owns q, k, v, o and lse.  Non-causal
 * calls whose last round of work items is split along the keys (the
 * wave-tail split: when fewer than half the SMs would have an item in the
 * last round) need scratch memory for the pieces' partial results -- at
 * most one piece per SM, 1 KiB * d + 3 KiB each, plus 4 bytes per split
 * item; about 20 MB on 152 SMs.  It comes from a stream-ordered memory pool
 * that the library creates per device when it first sets the device up,
 * and that it fills there and then with the largest amount any call can
 * need.  A call takes its scratch from the pool and gives it back behind
 * the kernel on the same stream; the pool keeps its memory.  So after
 * set-up, calls issued one stream at a time allocate no device memory.
 * Split calls running at the same time on several streams each take their
 * own scratch, and the pool grows (once) to the most that ran at the same
 * time.  If the pool cannot supply it the call runs unsplit.  Per-device
 * state (SM count, kernel attributes, one 4-byte status word, the pool, the
 * causal item order per shape) is created on first use and lives until
 * process exit.  o and lse must not overlap q, k, v or each other.
 *
 * Execution: asynchronous on `stream` (0 = legacy default stream); no host
 * synchronisation.  Safe to call from several host threads.  fa_fwd,
 * fa_fwd_fp16 and fa_fwd_ex may be captured into a CUDA graph (stream
 * capture): the split schedule's scratch then becomes a graph allocation
 * (cudaMallocAsync / cudaFreeAsync nodes) instead of pool memory.
 *
 * Errors: 0 on success, a negative FA_ERR_* code otherwise.  On an argument
 * error nothing is launched and o/lse are not written.  Faults seen while
 * the kernel runs (a pipeline wait that gave up) are recorded in the
 * device status word and returned by fa_get_status().
 */
#ifndef FA_GB300_H
#define FA_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t, passed as an opaque pointer so this header needs no CUDA
 * headers. */
typedef void *fa_stream_t;

#define FA_OK 0
#define FA_ERR_NULL (-1)           /* a required pointer is NULL */
#define FA_ERR_SHAPE (-2)          /* B, H or N < 1, or B*H*N*d overflows */
#define FA_ERR_HEADDIM (-3)        /* d is not 64 or 128 */
#define FA_ERR_UNSUPPORTED_N (-4)  /* N above FA_MAX_N */
#define FA_ERR_ALIGN (-5)          /* a pointer is not 16-byte aligned */
#define FA_ERR_SCALE (-6)          /* scale is not finite and > 0 */
#define FA_ERR_DEVICE (-7)         /* current device is not compute capability 10.3 */
#define FA_ERR_CUDA (-8)           /* a CUDA runtime/driver call failed */
#define FA_ERR_TIMEOUT (-9)        /* a pipeline wait inside the kernel gave up */
#define FA_ERR_ALIAS (-10)         /* an output overlaps an input or the other output */
#define FA_ERR_OPTION (-11)        /* an option (rescale threshold, self-test limit) out of range */
#define FA_ERR_SCRATCH (-12)       /* fa_fwd_noalloc: the call needs more than its fixed scratch */
#define FA_ERR_WORKSPACE (-13)     /* fa_bwd: the workspace is smaller than fa_bwd_workspace_size */
#define FA_ERR_INTERNAL (-14)      /* (fa_get_status) a kernel found its shared memory unusable */

#define FA_MAX_N (1 << 20)         /* longest sequence accepted */

/* Bytes of the fixed device array that serves fa_fwd_noalloc's scratch. */
#define FA_NOALLOC_SCRATCH_BYTES (16u << 20)

/* fa_fwd_variant: let the library choose the causal item order. */
#define FA_ORDER_AUTO (-2)

/* Rescale threshold used by fa_fwd and fa_fwd_fp16, in log2 units of the
 * scaled logits (see fa_fwd_ex). */
#define FA_DEFAULT_RESCALE_THRESHOLD 8.0f
#define FA_MAX_RESCALE_THRESHOLD 12.0f

/*
 * fa_fwd -- attention forward on bf16 inputs.
 *   q, k, v : [B,H,N,d] bf16, read only
 *   o       : [B,H,N,d] bf16, written (softmax-weighted sum of V rows,
 *             fp32 accumulation, rounded to nearest even)
 *   lse     : [B,H,N] fp32, written (natural-log logsumexp of the scaled
 *             logits over the visible keys)
 *   d       : 64 or 128
 *   causal  : nonzero => query i sees keys 0..i only (top-left aligned)
 *   scale   : multiplies Q K^T before the mask and softmax; finite, > 0
 *             (usually 1/sqrt(d))
 *   stream  : cudaStream_t to launch on.  The kernel is launched as a
 *             programmatic dependent of the previous kernel in the stream:
 *             its CTAs may start while that kernel drains, but each waits
 *             for its completion before touching memory, so the call is
 *             ordered in the stream like any other launch.
 */
int fa_fwd(const void *q, const void *k, const void *v, void *o, float *lse, int64_t B,
           int64_t H, int64_t N, int64_t d, int causal, float scale, fa_stream_t stream);

/* fa_fwd_fp16 -- identical to fa_fwd with fp16 q, k, v and o.
 * Both use the rescale threshold FA_DEFAULT_RESCALE_THRESHOLD (fa_fwd_ex). */
int fa_fwd_fp16(const void *q, const void *k, const void *v, void *o, float *lse, int64_t B,
                int64_t H, int64_t N, int64_t d, int causal, float scale,
                fa_stream_t stream);

/*
 * fa_fwd_ex -- fa_fwd / fa_fwd_fp16 with the online-softmax rescale rule
 * exposed (FlashAttention v4 Blackwell pipeline diagram, pseudo-code panel:
 * "maybe skip rescale if max change small"; softmax and correction lanes:
 * rescale the old accumulator only when the max change calls for it).
 *
 *   fp16              : 0 = bf16 q/k/v/o, 1 = fp16
 *   rescale_threshold : tau >= 0 in log2 units of the scaled logits.  For
 *       each query row, the running max m used to form P = 2^(S*log2e*scale
 *       - m) is raised (and O, l rescaled by 2^(m_old - m_new)) only when a
 *       block's max exceeds m by more than tau; otherwise m is kept and the
 *       block's probabilities may reach 2^tau.  Numerator and denominator
 *       use the same m, so the result is the same softmax for any tau; tau
 *       = 0 rescales whenever the max grows ("skip when the max does not
 *       change").  Must lie in [0, FA_MAX_RESCALE_THRESHOLD] so 2^tau stays
 *       far inside the fp16 range of P; otherwise FA_ERR_OPTION.
 *
 * All other arguments, the layout and the error behaviour are fa_fwd's.
 */
int fa_fwd_ex(const void *q, const void *k, const void *v, void *o, float *lse, int64_t B,
              int64_t H, int64_t N, int64_t d, int causal, float scale, int fp16,
              float rescale_threshold, fa_stream_t stream);

/*
 * fa_fwd_noalloc -- fa_fwd_ex that never allocates device memory.
 *
 * The pages have no counterpart to this entry point.  It serves callers that
 * cannot call cudaMalloc or take memory from a pool while they run: an
 * inference server that reserves all device memory for its own caching
 * allocator at start-up (so a driver allocation would fail or steal from
 * that reservation), a real-time loop that must not hit the allocator's
 * locks and implicit synchronisation, or code that runs inside another
 * library's allocation-free contract.  For them the wave-tail split's
 * scratch (see Ownership above) is one fixed array of
 * FA_NOALLOC_SCRATCH_BYTES (16 MiB) in the library's own device memory: it
 * exists from the moment the library's device code is loaded, on every GPU
 * that loads it, until the process exits.  Host code cannot use the array's
 * name as a device address, so the first call on a device looks the
 * address up once (cudaGetSymbolAddress) with that device current; make
 * that first call before any stream capture.  Neither that set-up nor any
 * later call allocates device memory or calls an allocating routine; the
 * split-scratch pool of the other entry points is never created by this
 * one.
 *
 * Limit: a split needs 1024 * d + 3072 bytes per piece plus 4 per split
 * item, so at most 125 pieces fit at d = 128.  A call whose split needs more
 * (e.g. the 144 pieces of a non-causal [8,16,4096,128] call on 152 SMs) is
 * rejected with FA_ERR_SCRATCH before anything is launched; o and lse are
 * not written, and fa_fwd_ex serves the same call.  Calls that need no
 * scratch (causal, or a last round that is not split) are always accepted.
 * Results are bitwise those of fa_fwd_ex.
 *
 * Every call on a device shares the one array, which keeps what the last
 * call left in it; each call clears the piece counters it uses before its
 * kernel runs.  Calls that overlap on the GPU race on the array and give
 * undefined results: issue them on one stream, or order them with events.
 * Arguments, layout, ownership of q/k/v/o/lse and the other errors are
 * fa_fwd_ex's.
 */
int fa_fwd_noalloc(const void *q, const void *k, const void *v, void *o, float *lse, int64_t B,
                   int64_t H, int64_t N, int64_t d, int causal, float scale, int fp16,
                   float rescale_threshold, fa_stream_t stream);

/*
 * fa_fwd_variant -- the forward through one of the kernel variants built
 * into the library, for tuning and measurement (the product entry points
 * above always use the default variant of their head dim and dtype).
 *
 * The FlashAttention-from-scratch blog index (its auto-tuning post and the
 * block-size trade-offs of its appendix) tunes a kernel's pipeline depth
 * and tile shape per GPU; the FlashAttention v4 Blackwell pipeline diagram
 * (pseudo-code panel, v3 -> v4 comparison) moves part of the softmax's
 * exponentials from the special-function unit to the FMA pipes.  The
 * variants expose those choices:
 *   stages    : K/V ring slots in shared memory (0 = the default: 4 at
 *               d = 128, 8 at d = 64)
 *   exp_split : 0, or n: every n-th pair of the softmax's exponentials is
 *               computed by a polynomial on the FMA pipes
 *   causal_order : FA_ORDER_AUTO (the library's choice, see
 *               fa_causal_order), or an order to force on causal launches:
 *               -1 or g in [0, B*H] with fa_causal_order's meaning
 *   stats     : NULL, or a DEVICE array of 4 unsigned 64-bit counters that
 *               the kernel adds to (the caller zeroes it): [0] (row, K/V
 *               block) pairs after a tile's first block where the running
 *               max grew past the rescale threshold, [1] all such pairs,
 *               [2] warp-blocks that ran the O rescale, [3] all warp-blocks
 *               after a tile's first block.  Only the default ring depth
 *               without exp split has a counting build.
 * fa_variant_count / fa_variant_info list what is built (stages resolved
 * to the actual slot count).  A combination that is not built gives
 * FA_ERR_OPTION before anything is launched; all other arguments and
 * errors are fa_fwd_ex's.  Every variant computes the same attention.
 */
int fa_fwd_variant(const void *q, const void *k, const void *v, void *o, float *lse, int64_t B,
                   int64_t H, int64_t N, int64_t d, int causal, float scale, int fp16,
                   float rescale_threshold, int stages, int exp_split, int causal_order,
                   unsigned long long *stats, fa_stream_t stream);
int fa_variant_count(void);
int fa_variant_info(int index, int *d, int *fp16, int *stages, int *exp_split, int *stats);

/*
 * fa_causal_order -- the order in which a causal launch of [B,H,N,d] on a
 * GPU with sm_count SMs takes its work items (pairs of 128-row Q tiles),
 * as the library chooses it (host computation only, no device call):
 *   -1     heaviest pair first across all heads (also whenever K and V of
 *          all heads total at most 64 MiB);
 *   g >= 0 head by head, heaviest pair first within a head, with the last
 *          g heads taken together, heaviest pair first across them.
 * FA_ERR_SHAPE / FA_ERR_HEADDIM on bad arguments.  For tests and tuning.
 */
int fa_causal_order(int64_t B, int64_t H, int64_t N, int64_t d, int sm_count);

/*
 * fa_bwd -- gradients of the attention forward (the backward pass).
 *
 * The FlashAttention v4 Blackwell pipeline diagram names the backward pass
 * (pseudo-code panel, "backward idea"; CTA-role panel: the backward adds
 * dQ up with atomic additions, which larger MMA tiles reduce).  Given the
 * forward's inputs q, k, v, its outputs o and lse (from fa_fwd /
 * fa_fwd_fp16 / fa_fwd_ex with the same causal and scale), and dout = dL/dO
 * for some loss L, fa_bwd writes dq = dL/dQ, dk = dL/dK, dv = dL/dV:
 *
 *   P_ij = exp(scale q_i.k_j - lse_i)   (j visible to i; else 0)
 *   dv_j = sum_i P_ij dout_i            D_i  = dout_i . o_i
 *   dS_ij = P_ij (dout_i . v_j - D_i)
 *   dq_i = scale sum_j dS_ij k_j        dk_j = scale sum_i dS_ij q_i
 *
 * P and dS are recomputed tile by tile and never stored; P and dS are
 * rounded to the 16-bit input type for the tensor-core products, with fp32
 * accumulation; dq is accumulated in fp32 in the workspace.
 *
 *   q, k, v, o, dout : [B,H,N,d] 16-bit (fp16 != 0: fp16, else bf16), read only
 *   lse              : [B,H,N] fp32, read only
 *   dq, dk, dv       : [B,H,N,d] 16-bit, written (round to nearest even)
 *   workspace        : DEVICE memory of at least fa_bwd_workspace_size(B,H,N,d)
 *                      bytes, 256-byte aligned, owned by the caller;
 *                      overwritten (nothing needs to be cleared before the
 *                      call, nothing is kept after it).  Calls that run at the
 *                      same time need separate workspaces.
 *   B*H              : at most 65535
 * Layout, d, causal, scale, alignment (16 bytes; lse 4) and stream as for
 * fa_fwd.  The library allocates no memory.  Errors: as fa_fwd, plus
 * FA_ERR_WORKSPACE (too small) and FA_ERR_ALIAS when an output overlaps an
 * input, another output or the workspace.  Nothing is launched on an
 * argument error.  Three kernels run on `stream`.
 */
int fa_bwd(const void *q, const void *k, const void *v, const void *o, const float *lse,
           const void *dout, void *dq, void *dk, void *dv, void *workspace,
           size_t workspace_bytes, int64_t B, int64_t H, int64_t N, int64_t d, int causal,
           float scale, int fp16, fa_stream_t stream);

/* fa_bwd_variant -- fa_bwd with its kernel chosen: cta_pairs = 0 runs one
 * CTA per 128-key block, each adding its dQ products into the fp32
 * workspace; cta_pairs = 1 runs clusters of two CTAs over adjacent key
 * blocks that exchange halves of their dQ products through distributed
 * shared memory, so that each query block's dQ gets half as many additions
 * (the saving the pages' backward notes obtain with two CTAs sharing one
 * larger MMA tile).  Same arguments, results and errors as fa_bwd (within
 * rounding: the additions are grouped differently), plus FA_ERR_OPTION for
 * another cta_pairs value. */
int fa_bwd_variant(const void *q, const void *k, const void *v, const void *o, const float *lse,
                   const void *dout, void *dq, void *dk, void *dv, void *workspace,
                   size_t workspace_bytes, int64_t B, int64_t H, int64_t N, int64_t d,
                   int causal, float scale, int fp16, int cta_pairs, fa_stream_t stream);

/* fa_bwd_workspace_size -- bytes of workspace fa_bwd needs for [B,H,N,d]:
 * B*H*Np*(4*d + 8) with Np = N rounded up to a multiple of 128.  Host only.
 * FA_ERR_NULL / FA_ERR_SHAPE / FA_ERR_HEADDIM / FA_ERR_UNSUPPORTED_N. */
int fa_bwd_workspace_size(int64_t B, int64_t H, int64_t N, int64_t d, size_t *bytes);

/* Work split of fa_fwd_host. */
#define FA_HOST_DEFAULT_CHUNKS 8
#define FA_HOST_MAX_CHUNKS 1024

/*
 * fa_fwd_host -- the forward on HOST buffers.
 *
 * q, k, v are read from, and o, lse written to, host memory in the layout
 * above (page-locked memory -- cudaHostAlloc, cudaHostRegister -- for full
 * copy speed; pageable memory works, staged by the CUDA driver).  The B*H heads
 * are processed in `chunks` groups (0 = FA_HOST_DEFAULT_CHUNKS, at most
 * FA_HOST_MAX_CHUNKS, at most B*H): while chunk c is computed, chunk c+1 is
 * copied to the device and chunk c-1 back to the host, on three streams of
 * the library's own, through three rotating device staging buffers (kept by
 * the library per device, grown to the largest call seen).  Every chunk is
 * one fa_fwd_ex launch with the default rescale threshold.  The call returns
 * when o and lse are written; it does not wait for, or order itself after,
 * work on other streams.  Calls on one device from several host threads run
 * one at a time.
 *
 *   fp16   : 0 = bf16 q/k/v/o, 1 = fp16
 *   chunks : see above; out of range gives FA_ERR_OPTION
 *
 * Errors are fa_fwd's (alignment is not required of host pointers); a CUDA
 * failure during the pipeline gives FA_ERR_CUDA, and o/lse may then be
 * partly written.  A pipeline wait that gave up is reported by
 * fa_get_status, as for fa_fwd.
 */
int fa_fwd_host(const void *q, const void *k, const void *v, void *o, float *lse, int64_t B,
                int64_t H, int64_t N, int64_t d, int causal, float scale, int fp16, int chunks);

/*
 * fa_get_status -- synchronises `stream`, then returns and clears the
 * current device's status word: FA_OK, or FA_ERR_TIMEOUT if some launch
 * since the last call had a pipeline wait give up (its outputs are then
 * undefined).  FA_ERR_CUDA if the synchronisation itself failed.
 */
int fa_get_status(fa_stream_t stream);

/*
 * fa_selftest_wait_timeout -- exercises the kernels' failure path without a
 * fault: launches one warp that waits, with the same bounded wait the
 * attention kernel uses, on a barrier nothing ever arrives on.  After
 * timeout_us microseconds (1 .. 1e6) the wait gives up, writes 1 to the
 * device int *gave_up, sets the status word (so the next fa_get_status
 * returns FA_ERR_TIMEOUT) and the kernel returns normally.  Asynchronous on
 * `stream`.  FA_ERR_NULL / FA_ERR_OPTION on bad arguments.
 */
int fa_selftest_wait_timeout(int64_t timeout_us, int *gave_up, fa_stream_t stream);

/* fa_strerror -- static, human-readable text for a FA_* code. */
const char *fa_strerror(int code);

/* fa_last_cuda_error -- the cudaError_t behind the calling thread's most
 * recent FA_ERR_CUDA (0 if none). */
int fa_last_cuda_error(void);

/* fa_version -- library version, major*10000 + minor*100 + patch. */
int fa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FA_GB300_H */
