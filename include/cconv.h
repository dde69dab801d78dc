/*
 * cconv.h -- C ABI of the GB300 (sm_103a) depthwise causal short convolution with fused
 * SiLU: forward, backward and the single-token decode update.
 *
 * What the calls compute (sources: the kernel-fun 0.2.0.dev1 wheel, files
 * kernel_fun/cconv/__init__.py and kernel_fun/cconv/_kernels/strip.py; and the pull
 * request "Add experimental causal conv1d decode update - #797" on NVIDIA/cudnn-frontend,
 * PR summary):
 *
 *   forward   z[b,t,d] = bias[d] + sum_{k<W} w[d, W-1-k] * x[b, t-k, d]   (x = 0 for t-k < 0)
 *             y[b,t,d] = silu(z) = z * sigmoid(z)
 *   backward  g = dy * sigmoid(z) * (1 + z * (1 - sigmoid(z)))            (z recomputed)
 *             dx[b,t,d]     = sum_{k<W} w[d, W-1-k] * g[b, t+k, d]      (g = 0 for t+k >= T)
 *             dw[d, W-1-k]  = sum_{b,t} g[b,t,d] * x[b, t-k, d]
 *             dbias[d]      = sum_{b,t} g[b,t,d]
 *   decode    per row i, slot s = state_indices[i] (or i): window = (state[s,d,0..W-2], x[i,d]),
 *             y[i,d] = silu(bias[d] + sum_{j<W} w[d,j] * window[j]),
 *             state[s,d,:] <- window[1..W-1]  (state[...,0] is the oldest; bits copied exactly)
 *
 * Conventions shared by every call:
 *   - 1 <= W <= 4.  Narrower widths are the width-4 case with zero taps on the old side.
 *   - Activations (x, dy, y, dx, decode state) are bf16; the weight, bias, dw and dbias
 *     share one dtype, `wdt` (bf16 or fp32).  Arithmetic is fp32; y, dx, dw and dbias are
 *     rounded to nearest-even on store.  The sigmoid uses the hardware tanh approximation
 *     (sigmoid(z) = 0.5 * tanh(z / 2) + 0.5), whose relative error is about 2^-11.
 *   - All pointers are DEVICE pointers owned by the caller; the library allocates nothing,
 *     keeps no tensor cache and never aliases one call's buffers into another (the one
 *     fixed device array of cconv_bwd_noalloc aside).
 *   - All work is enqueued on `stream` (NULL = the legacy default stream) with no host
 *     synchronisation.  The forward, backward, decode, packed-sequence and multi-problem
 *     calls may be captured in a CUDA graph.
 *   - Argument errors are found on the host, before anything is enqueued: the call returns
 *     a negative cconv_status and launches nothing.  CCONV_OK means "enqueued".
 *   - Strides are in elements.  The channel stride is 1 for every [.., D] tensor.
 *   - Fast-path alignment: bf16 row strides must be multiples of 8 elements (16 bytes) and
 *     every base pointer 16-byte aligned; D must be a multiple of 8 for the forward and
 *     backward.  Anything else returns CCONV_ERR_ALIGN (no slow path is taken silently).
 *     The decode update also accepts unaligned rows (ldx == D with any D) on a scalar path.
 */
#ifndef CCONV_H
#define CCONV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define CCONV_API __attribute__((visibility("default")))
#else
#define CCONV_API
#endif

/* Same type as cudaStream_t / CUstream. */
typedef struct CUstream_st* cconv_stream_t;

typedef enum {
  CCONV_BF16 = 0,
  CCONV_F32 = 1
} cconv_dtype;

/* Activation applied to z (packed-sequence calls; the batched calls always apply SiLU). */
typedef enum {
  CCONV_ACT_SILU = 0,       /* y = z * sigmoid(z) */
  CCONV_ACT_NONE = 1        /* y = z */
} cconv_activation;

typedef enum {
  CCONV_OK = 0,
  CCONV_ERR_NULL = -1,      /* a required pointer is NULL */
  CCONV_ERR_SHAPE = -2,     /* a size is out of range (B, T, D, N < 1; S < N without indices; ...) */
  CCONV_ERR_WIDTH = -3,     /* W outside [1, 4] */
  CCONV_ERR_ALIGN = -4,     /* a base pointer, row stride or D breaks the 16-byte rule */
  CCONV_ERR_STRIDE = -5,    /* a stride is not positive (or ldx < D) */
  CCONV_ERR_DTYPE = -6,     /* unknown cconv_dtype */
  CCONV_ERR_WORKSPACE = -7, /* workspace NULL or smaller than cconv_bwd_workspace_bytes() */
  CCONV_ERR_INDEX = -8,     /* decode: state_indices invalid (written to status_dev only) */
  CCONV_ERR_CUDA = -9,      /* a CUDA runtime / driver call failed */
  CCONV_ERR_DEVICE = -10    /* a kernel gave up a bounded wait (see cconv_device_fault) */
} cconv_status;

/* Offence bits of an invalid state_indices vector (status_dev[1] of cconv_update). */
#define CCONV_IDX_NEGATIVE 1
#define CCONV_IDX_OUT_OF_RANGE 2
#define CCONV_IDX_DUPLICATE 4

/* Largest slot pool cconv_update validates in one pass (one bit per slot in shared memory). */
#define CCONV_UPDATE_MAX_SLOTS 393216

/*
 * cconv_fwd -- forward of the causal depthwise convolution + SiLU.
 * Source: kernel-fun 0.2.0.dev1 wheel, cconv/_kernels/strip.py (`_tap`, `_ld_ring`,
 * `_silu`, `cconv_fwd_strip`); bias added inside the activation.
 *
 *   x     [B,T,D] bf16, element (b,t,d) at x[b*sxb + t*sxt + d]; sxt, sxb positive
 *         multiples of 8 (ignored where the dimension they step over has extent 1); rows
 *         may overlap (x is only read); base 16-byte aligned.
 *   w     [D,W] contiguous, dtype wdt.
 *   bias  [D] dtype wdt, or NULL for no bias.
 *   y     [B,T,D] bf16 contiguous output, 16-byte aligned.  Must not overlap x.
 *   B, T, D >= 1, D % 8 == 0, B*T < 2^31 - 16.
 */
CCONV_API int cconv_fwd(const void* x, int64_t B, int64_t T, int64_t D, int64_t sxb,
                        int64_t sxt, const void* w, const void* bias, cconv_dtype wdt, int W,
                        void* y, cconv_stream_t stream);

/*
 * cconv_bwd_workspace_bytes -- scratch that cconv_bwd needs for its fp32 partial sums of dw
 * and dbias (one record per channel strip and CTA), for the CURRENT device (the split of
 * work follows its SM count and D).
 * Returns CCONV_OK and writes *bytes, or an error for invalid sizes / no device.
 */
CCONV_API int cconv_bwd_workspace_bytes(int64_t B, int64_t T, int64_t D, int W,
                                        size_t* bytes);

/*
 * cconv_bwd -- backward: dx, dw and (optionally) dbias, with z recomputed from x.
 * Source: kernel-fun 0.2.0.dev1 wheel, cconv/_kernels/strip.py (`_dsilu`, `_bwd4`,
 * `cconv_bwd_strip`, `cconv_bwd`): one streaming pass, then a fixed-order (deterministic,
 * atomic-free) reduction of the partial sums.  Two kernels on `stream`.
 *
 *   x, dy   [B,T,D] bf16 with strides (sxb, sxt) and (sdb, sdt); same rules as cconv_fwd.
 *   w, bias as cconv_fwd (bias may be NULL).
 *   dx      [B,T,D] bf16 contiguous output, 16-byte aligned, overlapping neither x nor dy.
 *   dw      [D,W] output in wdt.
 *   dbias   [D] output in wdt, or NULL to skip it (sum of g; written whether or not a bias
 *           was passed).
 *   workspace, workspace_bytes: device scratch of at least cconv_bwd_workspace_bytes(),
 *           16-byte aligned; contents on entry do not matter.  It must not be shared with
 *           a concurrently running cconv_bwd.
 * Results are bit-identical from run to run for the same inputs and device.
 */
CCONV_API int cconv_bwd(const void* x, int64_t sxb, int64_t sxt, const void* dy, int64_t sdb,
                        int64_t sdt, int64_t B, int64_t T, int64_t D, const void* w,
                        const void* bias, cconv_dtype wdt, int W, void* dx, void* dw,
                        void* dbias, void* workspace, size_t workspace_bytes,
                        cconv_stream_t stream);

/*
 * cconv_update -- single-token decode update of a pooled bf16 convolution state.
 * Source: "Add experimental causal conv1d decode update - #797" (NVIDIA/cudnn-frontend),
 * PR summary: the state rows named by state_indices are read, y is emitted for the new
 * token, the state shifts by one; invalid indices fail closed.
 *
 *   x       [N,D] bf16, row i at x + i*ldx, ldx >= D.
 *   state   [S,D,W-1] bf16 contiguous pool, read and written in place.
 *   state_indices [N] int32 slot per row, or NULL (row i uses slot i; needs S >= N).
 *   w, bias as cconv_fwd.
 *   y       [N,D] bf16 contiguous output.
 *   status_dev  int32[2] in device memory, written by the kernel on every call:
 *           [0] = CCONV_OK or CCONV_ERR_INDEX, [1] = OR of CCONV_IDX_* offence bits.
 *           An index is invalid when negative, >= S, or (in range and) named twice.  On an
 *           invalid vector NOTHING is written: neither the state pool nor y.
 *   S <= CCONV_UPDATE_MAX_SLOTS when state_indices is given.
 * The vector path needs ldx % 8 == 0, D % 8 == 0 and 16-byte aligned x, state and y;
 * otherwise a scalar path of the same kernel runs.  Rows must name distinct slots for the
 * update to be well defined, which the validation enforces.
 */
CCONV_API int cconv_update(const void* x, int64_t N, int64_t D, int64_t ldx, void* state,
                           int64_t S, const int32_t* state_indices, const void* w,
                           const void* bias, cconv_dtype wdt, int W, void* y,
                           int32_t* status_dev, cconv_stream_t stream);

/*
 * cconv_update_ex -- cconv_update with the decode variants the cuDNN decode-update PR names
 * ("Add experimental causal conv1d decode update - #797", NVIDIA/cudnn-frontend, PR
 * summary: state length L in {3, 4} for W = 4; index -1 as a non-mutating padding row;
 * circular-buffer cache_seqlens metadata) and fla's activation keyword.  cconv_update(...)
 * is cconv_update_ex(..., L = W-1, pad_rows = 0, cache_seqlens = NULL,
 * act = CCONV_ACT_SILU).
 *
 *   state    [S, D, L] bf16 contiguous pool, L = W-1 or L = W.  The newest W-1 entries and
 *            the token form the window; the new state is the last L of (old state, token),
 *            so L = W keeps one token more than the convolution needs.
 *   pad_rows nonzero: a state index of -1 marks a padding row, which reads and writes no
 *            state and whose y row is not written; it is left out of the validation.
 *            Other negative indices are invalid as before.  Zero: -1 is invalid.
 *   cache_seqlens  int32[N] in device memory, or NULL.  Given, the state is a circular
 *            buffer (the mode the PR's signature reserves; the reading taken here): the
 *            state of a slot is a ring of L entries per channel, cache_seqlens[i] counts the
 *            tokens row i's slot has already seen, the token is written to ring entry
 *            cache_seqlens[i] mod L (taken non-negative), and the window is the W-1 entries
 *            before it, oldest first.  Nothing is shifted and cache_seqlens is not changed
 *            (the caller advances it).  Needs L >= 1.
 *   act      CCONV_ACT_SILU or CCONV_ACT_NONE.
 * Everything else, including the status words and the fail-closed rule, is cconv_update's.
 */
CCONV_API int cconv_update_ex(const void* x, int64_t N, int64_t D, int64_t ldx, void* state,
                              int64_t S, int L, const int32_t* state_indices, int pad_rows,
                              const int32_t* cache_seqlens, const void* w, const void* bias,
                              cconv_dtype wdt, int W, cconv_activation act, void* y,
                              int32_t* status_dev, cconv_stream_t stream);

/*
 * cconv_bwd_noalloc -- cconv_bwd without a workspace argument, for callers that cannot
 * allocate device memory where they run the backward (a runtime that hands out memory only
 * from a pre-sized arena, a plugin inside a framework that owns every allocation, a thread
 * that must not call cudaMalloc because it can synchronise the device).  The pages have no
 * counterpart to this call; it exists for those callers.
 *
 * Arguments and results are those of cconv_bwd minus (workspace, workspace_bytes), and so
 * are the results: the same kernels run with the same work split, so dx, dw and dbias are
 * bit-identical to cconv_bwd's.  The partial sums live in a fixed 8 MiB device array inside
 * the library (held by every GPU that loads it until the process exits); a problem whose
 * cconv_bwd_workspace_bytes() exceeds 8 MiB returns CCONV_ERR_WORKSPACE before anything is
 * enqueued.  The call itself never calls cudaMalloc, cudaFree or any allocating routine.
 * Set-up: the first call in a context (with that device current) may load the library's
 * device code there, which reserves the 8 MiB array, and looks up the array's device
 * address; so make one warm-up call before any stream capture and before sizing a memory
 * arena from the free memory.  Every call repeats the address lookup, which is cheap once
 * the code is loaded and stays valid after a device reset.  All calls on a device share the
 * array: calls whose work overlaps on the GPU (e.g. on two streams) race on it and must be
 * serialised by the caller.  Calls queued one after another on one stream do not overlap.
 */
CCONV_API int cconv_bwd_noalloc(const void* x, int64_t sxb, int64_t sxt, const void* dy,
                                int64_t sdb, int64_t sdt, int64_t B, int64_t T, int64_t D,
                                const void* w, const void* bias, cconv_dtype wdt, int W,
                                void* dx, void* dw, void* dbias, cconv_stream_t stream);

/*
 * Packed variable-length sequences with initial and final states.
 * Sources: the keyword set of fla's causal_conv1d that the kernel-fun 0.2.0.dev1 wheel
 * forwards (kernel_fun/_common/compat.py: initial_state, output_final_state, activation,
 * cu_seqlens), and the full-sequence-to-decode state handoff named in "Add experimental
 * causal conv1d decode update - #797" (NVIDIA/cudnn-frontend), whose decode state layout
 * [.., D, W-1] the states here share, so a final state can be the decode pool itself.
 *
 * nseq sequences are packed along the rows of a [total, D] tensor: sequence i is rows
 * [cu_seqlens[i], cu_seqlens[i+1]).  Inside a sequence the computation is the batched one,
 * except that the W-1 rows before its first row are its initial state (entry j = row
 * cu[i] - (W-1) + j, oldest first) instead of zeros, and the activation may be left out:
 *
 *   z[t,d]   = bias[d] + sum_{k<W} w[d, W-1-k] * xe[t-k, d]     xe: x extended by the state
 *   y        = silu(z) (CCONV_ACT_SILU) or z (CCONV_ACT_NONE)
 *   final[i][d][j] = xe[cu[i+1] - (W-1) + j, d]   (the state a decode update continues from)
 *
 *   cu_seqlens  int32[nseq+1] in DEVICE memory: cu[0] = 0, non-decreasing, cu[nseq] = total.
 *           Empty sequences are allowed (their final state is their initial state).  The
 *           host never reads it.  An ill-formed vector gives unspecified results, every
 *           access still stays inside the buffers, and cconv_device_fault() then reports
 *           bit 4.
 *   x, dy   [total, D] bf16, row t at x + t*sxt (sxt a positive multiple of 8, ignored when
 *           total == 1), 16-byte aligned.  total may be 0 (x, dy, y, dx may then be NULL).
 *   states  bf16 arrays of S slots x [D, W-1], contiguous, 16-byte aligned (forward) or
 *           2-byte aligned (backward).  Ignored when W == 1.
 *   1 <= nseq < 2^31 - 1, total < 2^31 - 16, D % 8 == 0.
 */

/*
 * cconv_fwd_varlen -- forward over packed sequences.  One stream kernel, plus a small state
 * kernel when final_state or state_indices is given; both on `stream`.
 *
 *   initial_state  [S, D, W-1] bf16, or NULL (every sequence starts from zeros).
 *   final_state    [S, D, W-1] bf16 output, or NULL.  May be the same array as
 *                  initial_state: the final states are written after every initial state
 *                  has been read (chunked prefill into a decode pool, in place).
 *   state_indices  int32[nseq] in device memory, or NULL: sequence i's state lives in slot
 *                  state_indices[i] (else slot i, and S >= nseq).  With indices,
 *                  1 <= S <= CCONV_UPDATE_MAX_SLOTS, status_dev is required, and the
 *                  indices are validated on the device as cconv_update does (negative, >= S,
 *                  repeated): on an invalid vector no state is written, status_dev gets
 *                  [CCONV_ERR_INDEX, offence bits], and y is computed with zero initial
 *                  states for the unusable slots.  Otherwise status_dev gets [CCONV_OK, 0].
 *   status_dev     int32[2] in device memory (only written when state_indices is given).
 *   y              [total, D] bf16 contiguous output, 16-byte aligned.
 * final_state must not overlap x or y; y must not overlap x.
 */
CCONV_API int cconv_fwd_varlen(const void* x, int64_t total, int64_t D, int64_t sxt,
                               const int32_t* cu_seqlens, int64_t nseq, const void* w,
                               const void* bias, cconv_dtype wdt, int W, cconv_activation act,
                               const void* initial_state, void* final_state,
                               const int32_t* state_indices, int64_t S, int32_t* status_dev,
                               void* y, cconv_stream_t stream);

/* Workspace cconv_bwd_varlen needs on the current device (0 <= total < 2^31 - 16). */
CCONV_API int cconv_bwd_varlen_workspace_bytes(int64_t total, int64_t D, int W, size_t* bytes);

/*
 * cconv_bwd_varlen -- backward over packed sequences: dx, dw, dbias and the gradient of
 * the initial states, with z recomputed (two kernels on `stream`, deterministic; a third,
 * small one checks state_indices when they are given).
 *
 *   g = dy * silu'(z) (CCONV_ACT_SILU) or dy (CCONV_ACT_NONE)
 *   dx[t]          = sum_{k<W} w[d, W-1-k] g[t+k]   over t+k inside t's sequence
 *   dw[d, W-1-k]   = sum over all rows t of g[t] * xe[t-k]
 *   dbias[d]       = sum of g
 *   d_initial_state[i][d][j] = sum_{k<W} w[d, W-1-k] g[u+k] over u+k inside sequence i,
 *                              u = cu[i] - (W-1) + j   (zero for an empty sequence)
 *
 *   initial_state    [S, D, W-1] bf16 or NULL (zeros).  Sequence i's initial state is slot
 *                    state_indices[i] when indices are given (the decode pool a chunked
 *                    prefill read from), else slot i (then S is ignored and the array holds
 *                    nseq slots).
 *   state_indices    int32[nseq] in device memory, or NULL.  Given, 1 <= S <=
 *                    CCONV_UPDATE_MAX_SLOTS, status_dev is required, and the indices are
 *                    checked on the device as cconv_fwd_varlen checks them (negative, >= S,
 *                    repeated): status_dev gets [CCONV_OK, 0] or [CCONV_ERR_INDEX, offence
 *                    bits].  A negative or out-of-range slot reads as a zero initial state
 *                    (as in the forward); repeated slots are read as they are (the backward
 *                    writes no state).
 *   status_dev       int32[2] in device memory (only written when state_indices is given).
 *   dx               [total, D] bf16 contiguous, 16-byte aligned, overlapping neither x nor dy.
 *   dw, dbias        as cconv_bwd (dbias may be NULL).
 *   d_initial_state  [nseq, D, W-1] bf16 output (one per sequence, also with indices), or NULL.
 *   workspace        at least cconv_bwd_varlen_workspace_bytes(total, D, W), 16-byte
 *                    aligned (unused when total == 0).
 */
CCONV_API int cconv_bwd_varlen(const void* x, int64_t sxt, const void* dy, int64_t sdt,
                               int64_t total, int64_t D, const int32_t* cu_seqlens,
                               int64_t nseq, const void* w, const void* bias, cconv_dtype wdt,
                               int W, cconv_activation act, const void* initial_state,
                               const int32_t* state_indices, int64_t S, int32_t* status_dev,
                               void* dx, void* dw, void* dbias, void* d_initial_state,
                               void* workspace, size_t workspace_bytes, cconv_stream_t stream);

/*
 * Several convolutions in one launch: the q, k and v short convolutions of a KDA layer
 * (kernel-fun 0.2.0.dev1 wheel, kernel_fun/cconv/__init__.py module docstring: three calls
 * per layer forward, q and k at D = n_heads*128 and v at twice that).  Each problem k has
 * its own x, weights, bias and outputs and its own D[k]; B, T, W and the weight dtype are
 * shared.  The arrays of pointers, strides and sizes are HOST arrays of n entries
 * (1 <= n <= 4); the pointers in them are device pointers with the rules of cconv_fwd /
 * cconv_bwd.  One stream kernel covers every problem (plus one reduction kernel for the
 * backward), so the per-launch tails are paid once.  Results are those of n separate
 * calls: y and dx bit for bit, dw and dbias up to the order of the partial sums.
 */
CCONV_API int cconv_fwd_multi(int n, const void* const* x, const int64_t* D, const int64_t* sxb,
                              const int64_t* sxt, const void* const* w, const void* const* bias,
                              void* const* y, int64_t B, int64_t T, cconv_dtype wdt, int W,
                              cconv_stream_t stream);

/* Workspace cconv_bwd_multi needs on the current device. */
CCONV_API int cconv_bwd_multi_workspace_bytes(int n, const int64_t* D, int64_t B, int64_t T,
                                              int W, size_t* bytes);

/* bias and dbias may be NULL arrays (no bias / no dbias for any problem) or hold NULLs. */
CCONV_API int cconv_bwd_multi(int n, const void* const* x, const int64_t* sxb,
                              const int64_t* sxt, const void* const* dy, const int64_t* sdb,
                              const int64_t* sdt, const int64_t* D, const void* const* w,
                              const void* const* bias, void* const* dx, void* const* dw,
                              void* const* dbias, int64_t B, int64_t T, cconv_dtype wdt, int W,
                              void* workspace, size_t workspace_bytes, cconv_stream_t stream);

/*
 * Launch descriptions (a measurement and tuning aid; the pages have no counterpart).
 *
 * Between cconv_describe_begin() and cconv_describe_end() on one host thread, every call of
 * this library on that thread runs its host-side checks and planning as usual but records
 * the kernels it would launch instead of enqueueing them: nothing runs on the GPU and no
 * output is written.  cconv_describe_end() stops recording, writes up to `max` descriptions
 * into `out` (in launch order) and sets *count to the number of launches recorded.  The
 * attributes come from the CUDA runtime (cudaFuncGetAttributes and the occupancy
 * calculator, for the launch's block size and dynamic shared memory).  Returns CCONV_OK,
 * CCONV_ERR_NULL, or CCONV_ERR_CUDA if an attribute query failed.
 */
typedef struct {
  char name[160];            /* kernel name with its template arguments (may be truncated) */
  int registers;             /* registers per thread */
  int local_bytes;           /* local memory per thread (register spills and stack) */
  int static_shared_bytes;   /* per CTA */
  int dynamic_shared_bytes;  /* per CTA, as launched */
  int threads;               /* per CTA */
  int ctas_per_sm;           /* CTAs of this launch that fit on one SM at once */
  int64_t ctas;              /* CTAs in the grid */
} cconv_kernel_desc;

CCONV_API int cconv_describe_begin(void);
CCONV_API int cconv_describe_end(cconv_kernel_desc* out, int max, int* count);

/* Human-readable name of a cconv_status value (static storage). */
CCONV_API const char* cconv_status_str(int status);

/*
 * cconv_device_fault -- reads (and clears) the library's device fault word on the current
 * device after synchronising it.  *fault = 0 when nothing went wrong; otherwise an OR of:
 * 1 = a forward kernel gave up a bounded wait, 2 = a backward kernel did, 4 = an ill-formed
 * cu_seqlens was passed to a packed-sequence call.  Returns CCONV_OK or CCONV_ERR_CUDA.
 */
CCONV_API int cconv_device_fault(int32_t* fault);

#ifdef __cplusplus
}
#endif

#endif /* CCONV_H */
