/*
 * dg.h -- C ABI of libdg: the local compute of expert- and tensor-parallel
 * linear layers on one GB300 (sm_103a).
 *
 * Every entry point takes plain pointers and sizes.  Conventions that hold
 * for all of them:
 *
 *  - Tensors are caller-owned DEVICE memory, contiguous (row-major, last
 *    dimension fastest) in the shapes written beside each argument, and
 *    16-byte aligned.  bf16 means IEEE bfloat16 bit patterns (uint16),
 *    e4m3 means OCP E4M3FN bit patterns (uint8, the element format of
 *    cutlass::float_e4m3_t and torch.float8_e4m3fn).
 *  - The library never allocates device memory.  Scratch space comes from
 *    the caller through a (pointer `ws`, bytes) pair whose required size is
 *    given by the matching *_bytes() query; too small a buffer is an error.
 *  - Inputs are never written.  Outputs must not overlap inputs or scratch.
 *  - Calls are asynchronous and stream-ordered on `stream` (a cudaStream_t,
 *    NULL = legacy default stream): they return once the work is enqueued.
 *  - Every call returns a dg_status.  On failure nothing is enqueued and
 *    dg_last_error() names the offending argument (thread-local message).
 *    There is no silent fallback: an unsupported case is an error.
 *  - Error block.  The first DG_ERROR_BLOCK_BYTES bytes of every workspace
 *    hold that workspace's device-side error word.  A kernel whose bounded
 *    pipeline wait runs out of time records the failure there instead of
 *    trapping, and later kernels of calls given the same workspace return
 *    early without touching memory until dg_check_device_error() reads and
 *    clears the word.  Calls with different workspaces (for example one per
 *    stream) do not see each other's failures.  The word must be zero before
 *    a workspace's first use: zero-filled memory, or dg_workspace_init().
 *  - Tensor cores accumulate in fp32; bf16 results are rounded to nearest
 *    even once, at the end.
 */
#ifndef DG_H
#define DG_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Bytes at the start of every workspace that hold its error word. */
#define DG_ERROR_BLOCK_BYTES 256

typedef enum {
  DG_OK = 0,
  DG_ERR_INVALID_ARGUMENT = 1, /* a size, pointer, alignment or overlap rule was broken */
  DG_ERR_UNSUPPORTED = 2,      /* a valid request the library does not implement */
  DG_ERR_CUDA = 3,             /* a CUDA runtime/driver call failed */
  DG_ERR_TIMEOUT = 4,          /* a device-side wait exceeded its limit (see dg_check_device_error) */
  DG_ERR_DEVICE_CHECK = 5,     /* a device-side consistency check failed */
  DG_ERR_WORKSPACE = 6         /* the scratch buffer is missing or smaller than the query says */
} dg_status;

/* Thread-local description of the last failure on this thread ("" if none). */
const char* dg_last_error(void);

/* Library version string. */
const char* dg_version(void);

/*
 * Zeroes the error block of a freshly allocated workspace (stream-ordered;
 * ws_bytes >= DG_ERROR_BLOCK_BYTES).  Not needed for zero-filled memory.
 */
dg_status dg_workspace_init(void* ws, size_t ws_bytes, void* stream);

/*
 * Synchronises `stream`, then reads and clears the error word in the error
 * block of `ws` (a workspace given to earlier calls), or, with ws = NULL, the
 * library's own error word, which only dg_tp_swiglu_noalloc writes.  Returns
 * DG_OK, DG_ERR_TIMEOUT (a bounded pipeline wait expired),
 * DG_ERR_DEVICE_CHECK, or DG_ERR_CUDA.  When not DG_OK, *site (if non-NULL)
 * receives the raw code, whose low byte names the wait that expired.
 */
dg_status dg_check_device_error(void* ws, void* stream, uint32_t* site);

/* ------------------------------------------------------------------------
 * (a) FP8 GEMM   D = alpha * (A @ B^T) + beta * C
 *
 * Source: "Pytorch Op for blackwell distributed gemm" (pytorch-distributed-
 * gemm README), sections "Usage" and "Limitations & Important Notes":
 * A is [M,K], B is [N,K] row-major (the transpose of torch.matmul's second
 * operand), C is the [M,N] bias term; elements are e4m3.
 *
 *   A      e4m3 [M, K]         K % 16 == 0 (TMA rows must be 16-byte multiples)
 *   B      e4m3 [N, K]
 *   C      bf16 [M, N]         may be NULL only when beta == 0; N % 8 == 0
 *   D      bf16 [M, N]         output, D = bf16_rne(alpha*acc + beta*C),
 *                              acc = sum_k A[m,k]*B[n,k] exact products, fp32 sum
 *   M, N >= 0 (0 = nothing to do); K >= 0 (K == 0 gives D = beta*C).
 *   ws     the error block only (dg_gemm_fp8_workspace_bytes = 256 bytes)
 * ------------------------------------------------------------------------ */
size_t dg_gemm_fp8_workspace_bytes(int64_t M, int64_t N, int64_t K);

dg_status dg_gemm_fp8(int64_t M, int64_t N, int64_t K,
                      const void* A, const void* B, const void* C, void* D,
                      float alpha, float beta, void* ws, size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------------
 * (b) All-to-all expert-parallel FFN layer, P logical ranks on one GPU.
 *
 * Source: the A2A-FFN project statement (problems/p04), sections
 * "Interface, layout, and parameters" and "Computation and communication
 * example".  With H = D*k, L = T/P and a token position t = r*L + l
 * (rank r, slice l):
 *   Xlocal[r][n, l] = inputs[s][b, t]            n = s*B + b   (dispatch)
 *   Z  = Xlocal[r][:, l] @ w1[r][l] + b1[r][l]                 ([P*B, 2H])
 *   U, G = Z[:, :H], Z[:, H:]
 *   LN(z) = (z - mean z) / sqrt(mean((z - mean z)^2) + eps) * gamma + beta
 *   Hl = LN_x(U) * silu(LN_gate(G))       (LN params: norm_x / norm_gate of rank r)
 *   Ylocal[r][:, l] = Hl @ wout[r][l] + bout[r][l]
 *   output[s][b, t] = Ylocal[r][n, l]                           (combine)
 * The two exchanges are index maps folded into the TMA coordinates of the
 * GEMMs: no data moves for them.
 *
 * Layouts (bf16, leading dimension = rank):
 *   inputs, output, dY, d_inputs : [P, B, T, D]
 *   w1 [P, L, D, 2H]   b1 [P, L, 2H]   wout [P, L, H, D]   bout [P, L, D]
 *   nx_w, nx_b, ng_w, ng_b : [P, H]   (LayerNorm weight/bias for U and G)
 * Requirements: T % P == 0, D % 8 == 0, P*B >= 1; H = D*k <= 65536 (larger H
 * returns DG_ERR_UNSUPPORTED).
 *
 * saved  (size dg_a2a_ffn_saved_bytes) training: the forward writes Z, Hl
 *        and the per-row LayerNorm statistics there, and the backward reads
 *        them.  NULL = inference: nothing is kept, and Z, the statistics
 *        and Hl live in the workspace instead (Hl only when D is wider than
 *        one column pass of the gated GEMM, 512, or with
 *        DG_FFN_SEPARATE_GATE).
 * ws     size dg_a2a_ffn_fwd_workspace_bytes(shape, saved == NULL, flags):
 *        the error block, plus the inference scratch and the comp_only
 *        buffers when they apply.
 * flags  DG_FFN_COMP_ONLY: no exchange; each rank's own [B, T, D] rows, viewed
 *        as [B, P, L, D], feed its L slices (the project statement's
 *        comp_only mode of forward_ffn; the output keeps the input's layout).
 *        The normalise-and-gate is computed inside the second GEMM by
 *        default: producer warps normalise and gate Z while building its A
 *        operand for the first 512 output columns and store Hl as they go,
 *        and a plain GEMM on that Hl computes the remaining columns.
 *        DG_FFN_SEPARATE_GATE: compute Hl in a separate pass through HBM
 *        first, then the whole second GEMM on it.  Same results bit for bit
 *        (slower at the page's shapes).  DG_FFN_FUSED_GATE asks for the
 *        default explicitly; giving both is an invalid argument.
 * ------------------------------------------------------------------------ */
typedef struct {
  int32_t P, B, T, D, k;
  float eps; /* LayerNorm epsilon, 1e-5 on the page */
} dg_ffn_shape;

#define DG_FFN_COMP_ONLY 1u
#define DG_FFN_FUSED_GATE 2u
#define DG_FFN_SEPARATE_GATE 4u

size_t dg_a2a_ffn_saved_bytes(const dg_ffn_shape* shape);
size_t dg_a2a_ffn_fwd_workspace_bytes(const dg_ffn_shape* shape, int32_t inference, uint32_t flags);

dg_status dg_a2a_ffn_fwd(const dg_ffn_shape* shape,
                         const void* inputs, const void* w1, const void* b1,
                         const void* wout, const void* bout,
                         const void* nx_w, const void* nx_b,
                         const void* ng_w, const void* ng_b,
                         void* output, void* saved, size_t saved_bytes,
                         void* ws, size_t ws_bytes, uint32_t flags, void* stream);

/*
 * Backward of dg_a2a_ffn_fwd for the same shape, parameters and flags, given
 * the upstream gradient dY [P,B,T,D] and the `saved` buffer the forward
 * filled.  Gradient outputs are OVERWRITTEN (not accumulated), bf16, same
 * layouts as the tensors they belong to; d_nx_* / d_ng_* of rank r sum over
 * its rows and its L slices.  Any gradient pointer may be NULL: that gradient
 * is not computed, nothing is written there, and work that only it needs is
 * skipped (d_inputs: the dX GEMM; d_w1: the dw1 GEMM; d_wout: the dwout GEMM;
 * d_bout: its column sum; with d_inputs, d_w1, d_b1 and the four norm
 * gradients all NULL, also the dHl GEMM and the LayerNorm-gate backward).
 * Inputs only a skipped gradient needs may be NULL too (inputs for d_w1, w1
 * for d_inputs, saved for all but d_bout).
 * flags  the forward's flags.  DG_FFN_COMP_ONLY as in the forward.  The gate
 *        flags are checked as in the forward (both together are an invalid
 *        argument) and do not change the backward: its LayerNorm-gate row
 *        sums are always a pass of their own over Z and dHl.
 * Scratch: `ws` of dg_a2a_ffn_bwd_workspace_bytes(shape, flags) (0 for
 * invalid flags).
 */
size_t dg_a2a_ffn_bwd_workspace_bytes(const dg_ffn_shape* shape, uint32_t flags);

dg_status dg_a2a_ffn_bwd(const dg_ffn_shape* shape,
                         const void* inputs, const void* w1, const void* b1,
                         const void* wout, const void* bout,
                         const void* nx_w, const void* nx_b,
                         const void* ng_w, const void* ng_b,
                         const void* saved, size_t saved_bytes, const void* dY,
                         void* d_inputs, void* d_w1, void* d_b1,
                         void* d_wout, void* d_bout,
                         void* d_nx_w, void* d_nx_b, void* d_ng_w, void* d_ng_b,
                         void* ws, size_t ws_bytes, uint32_t flags, void* stream);

/*
 * The two exchanges as explicit permutation copies (bit-exact bf16 moves),
 * for layout checks and for callers that want the dispatched tensors:
 *   dg_a2a_dispatch: inputs [P,B,T,D] -> xlocal [P, P*B, L, D]
 *   dg_a2a_combine:  ylocal [P, P*B, L, D] -> output [P,B,T,D]
 */
dg_status dg_a2a_dispatch(int32_t P, int32_t B, int32_t T, int32_t D,
                          const void* inputs, void* xlocal, void* stream);
dg_status dg_a2a_combine(int32_t P, int32_t B, int32_t T, int32_t D,
                         const void* ylocal, void* output, void* stream);

/* ------------------------------------------------------------------------
 * A2A FFN forward with both GEMMs on e4m3 operands.
 *
 * Source: the A2A-FFN project statement (problems/p04), "Public checks and
 * instructor coverage", which lists optional FP8 paths of the layer without a
 * recipe.  Reading taken here: GEMM1 and GEMM2 run on e4m3 operands with fp32
 * accumulation and dequantise in their epilogues; everything else (bias,
 * LayerNorm statistics and normalise-and-gate, dispatch/combine) is the bf16
 * forward's.  Activations (the input rows and Hl) carry one scale per row,
 * weights one scale per output column; a scale is amax / 448 (1 for an
 * all-zero vector) and a code is the e4m3 value nearest to x * (448 / amax)
 * (binary32 quotient and product, ties to even, saturating at +-448).
 *
 * dg_a2a_ffn_fp8_pack_weights quantises w1 and wout once into `packed`
 * (dg_a2a_ffn_fp8_weights_bytes), laid out with 256-byte aligned regions:
 *   w1 codes [T, 2H, D] e4m3, w1 scales [T, 2H] f32,
 *   wout codes [T, D, H] e4m3, wout scales [T, D] f32,
 *   w1 inverse scales [T, 2H] f32, wout inverse scales [T, D] f32
 * (T = P*L problems in the order of w1's [P, L] leading dimensions).
 * dg_a2a_ffn_fwd_fp8 computes `output` (bf16 [P,B,T,D]) from bf16 inputs,
 * the packed weights, and the bf16 b1, bout and LayerNorm parameters (layouts
 * of dg_a2a_ffn_fwd).  Its workspace (dg_a2a_ffn_fp8_workspace_bytes) starts
 * with the error block, then the input codes [P,B,T,D] e4m3 followed, at the
 * next 256-byte boundary, by their scales [T, P*B] f32 (scale of input row
 * (s, b, t) at t*P*B + s*B + b); both are left there after the call.
 * Requirements: those of dg_a2a_ffn_fwd, D % 16 == 0, H % 16 == 0, H <= 8192
 * (an e4m3 Hl row is scaled inside one CTA); otherwise the query functions
 * return 0 and the calls fail with DG_ERR_INVALID_ARGUMENT / UNSUPPORTED.
 * No backward: training uses the bf16 path.
 * ------------------------------------------------------------------------ */
size_t dg_a2a_ffn_fp8_weights_bytes(const dg_ffn_shape* shape);
size_t dg_a2a_ffn_fp8_workspace_bytes(const dg_ffn_shape* shape);

dg_status dg_a2a_ffn_fp8_pack_weights(const dg_ffn_shape* shape, const void* w1, const void* wout,
                                      void* packed, size_t packed_bytes, void* stream);

dg_status dg_a2a_ffn_fwd_fp8(const dg_ffn_shape* shape, const void* inputs,
                             const void* packed, size_t packed_bytes,
                             const void* b1, const void* bout,
                             const void* nx_w, const void* nx_b, const void* ng_w, const void* ng_b,
                             void* output, void* ws, size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------------
 * (c) SwiGLU column/row-parallel pair over W tensor-parallel shards.
 *
 * Source: "Add dist GEMM attention and FFN backend" (torchtitan PR #4044),
 * sections "Structure" and "Row ordering": the column-parallel w1/w3 pair
 * shares one gathered input, h_s = silu(X w1_s^T) * (X w3_s^T), and the
 * row-parallel w2 sums the shards' partials before scattering rows back.
 *
 *   x_shards [W, bsz, S/W, d]   sequence shard of each rank
 *   w13      [W, 2*ffn/W, d]    rows [w1_s ; w3_s] of shard s
 *   w2       [d, ffn]           stock layout; shard s = columns s*ffn/W ...
 *   y_shards [W, bsz, S/W, d]   y = sum_s h_s @ w2_s^T, rows back in place
 * The layer is row-local, so gathering rows (rank, batch, seq_local) and
 * scattering them back is the identity on memory order.  The shard sum is
 * the K loop of one GEMM accumulating in TMEM.
 * Requirements: S % W == 0, ffn % W == 0, d % 8 == 0, (ffn/W) % 8 == 0.
 * Scratch (dg_tp_swiglu_workspace_bytes): the error block, then h
 * [W*bsz*S/W, ffn] bf16.
 * ------------------------------------------------------------------------ */
size_t dg_tp_swiglu_workspace_bytes(int64_t S, int64_t d, int64_t ffn, int32_t W, int32_t bsz);

dg_status dg_tp_swiglu(int64_t S, int64_t d, int64_t ffn, int32_t W, int32_t bsz,
                       const void* x_shards, const void* w13, const void* w2,
                       void* y_shards, void* ws, size_t ws_bytes, void* stream);

/*
 * dg_tp_swiglu_bwd: gradients of the SwiGLU pair above with respect to the
 * gathered input and both weights, given dY = dL/dy.
 *
 * Source: "Add dist GEMM attention and FFN backend" (torchtitan PR #4044),
 * section "Structure": the backward of the column-parallel pair is one
 * product over the concatenated [w1_s ; w3_s] rows of every shard, so its
 * input gradient (the row-parallel reduction across shards) is a single K
 * loop.  With a = X w1_s^T, b = X w3_s^T, h = silu(a) * b and
 * sig = sigmoid(a):
 *   dh_s   = dY w2_s                 da = dh * b * (sig + a*sig*(1-sig))
 *   d_w2_s = dY^T h_s                db = dh * a * sig
 *   d_w13_s = [da | db]^T X          dX = sum_s [da | db] [w1_s ; w3_s]
 * a and b are recomputed from X (nothing from the forward is kept).
 *
 *   x_shards, w13, w2   as for dg_tp_swiglu (inputs)
 *   dy_shards [W, bsz, S/W, d]   dL/dy, same layout as y_shards (input)
 *   dx_shards [W, bsz, S/W, d]   dL/dx (output, overwritten)
 *   d_w13     [W, 2*ffn/W, d]    dL/dw13 in w13's layout (output, overwritten)
 *   d_w2      [d, ffn]           dL/dw2 (output, overwritten)
 * Scratch: the error block, then [a|b] [rows, 2*ffn] and dh [rows, ffn] bf16
 * in `ws` (dg_tp_swiglu_bwd_workspace_bytes); no written buffer may overlap
 * any other.
 * Requirements and errors are those of dg_tp_swiglu.
 */
size_t dg_tp_swiglu_bwd_workspace_bytes(int64_t S, int64_t d, int64_t ffn, int32_t W, int32_t bsz);

dg_status dg_tp_swiglu_bwd(int64_t S, int64_t d, int64_t ffn, int32_t W, int32_t bsz,
                           const void* x_shards, const void* w13, const void* w2,
                           const void* dy_shards, void* dx_shards, void* d_w13, void* d_w2,
                           void* ws, size_t ws_bytes, void* stream);

/*
 * dg_tp_swiglu_noalloc: the same SwiGLU pair as dg_tp_swiglu, for callers
 * that cannot allocate device memory -- for example code that runs under a
 * framework which owns the device's memory pool and accounts for every
 * allocation, or a latency-critical path where cudaMalloc/cudaFree (which can
 * synchronise the device) are not allowed.  No source page has a counterpart
 * of this call; it exists for such callers only.
 *
 * The h activations live in a 32 MiB array built into the library instead of
 * a caller workspace, so the call takes no scratch argument and allocates
 * nothing: S*bsz*ffn*2 bytes must not exceed 32 MiB (33554432), otherwise
 * the call returns DG_ERR_UNSUPPORTED without enqueuing anything.  Every
 * device that loads the library holds that array until the process exits.
 * Having no workspace, it records device-side failures in the library's own
 * error word: read it with dg_check_device_error(NULL, stream, site).
 * The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current; make that first call
 * before any stream capture.  All calls on a device share the one array, so
 * calls whose executions overlap on the GPU (different streams, no ordering
 * between them) race on it; calls ordered on one stream are safe.  Each call
 * overwrites all of h before reading it, so nothing needs clearing between
 * calls.  Tensors, layouts and requirements are those of dg_tp_swiglu.
 */
dg_status dg_tp_swiglu_noalloc(int64_t S, int64_t d, int64_t ffn, int32_t W, int32_t bsz,
                               const void* x_shards, const void* w13, const void* w2,
                               void* y_shards, void* stream);

/* ------------------------------------------------------------------------
 * Attention projections over W tensor-parallel shards: the column-parallel
 * all-gather linear (fused QKV) and the row-parallel linear reduce-scatter
 * (output projection wo).
 *
 * Source: "Add dist GEMM attention and FFN backend" (torchtitan PR #4044),
 * sections "Structure" and "Row ordering".  Both keep the stock parameter
 * layout weight [out_features, in_features] (+ bias [out_features]).
 *   column parallel: rank s owns weight rows [s*out/W, (s+1)*out/W) and
 *     multiplies the all-gathered rows by them; its output is the column block
 *     s of y.
 *   row parallel: rank s owns input columns [s*in/W, (s+1)*in/W) and the same
 *     weight columns; the ranks' partial products are summed (reduce) and the
 *     rows split back into sequence shards (scatter).
 * On one GPU both are y = x weight^T (+ bias) over all shards at once: the
 * rank blocks are column blocks of x, y and weight, the shard sum of the row
 * parallel form is the K loop, and gathering/scattering rows is the identity
 * on memory order because every output row depends on its own input row only.
 *
 *   x [rows, in_features], y [rows, out_features]   (row-major, bf16)
 *   weight [out_features, in_features], bias [out_features] or NULL
 * dg_tp_linear_bwd writes dx = dy weight [rows, in], d_weight = dy^T x
 * [out, in] and d_bias = column sums of dy [out]; any of the three may be NULL
 * (not computed).  Outputs are overwritten.
 * Requirements: rows, in_features, out_features >= 1; in_features and
 * out_features multiples of 8; 16-byte aligned tensors; outputs disjoint from
 * each other and from the inputs.  ws: the error block only
 * (dg_tp_linear_workspace_bytes = 256 bytes).
 * ------------------------------------------------------------------------ */
size_t dg_tp_linear_workspace_bytes(int64_t rows, int64_t in_features, int64_t out_features);

dg_status dg_tp_linear_fwd(int64_t rows, int64_t in_features, int64_t out_features,
                           const void* x, const void* weight, const void* bias,
                           void* y, void* ws, size_t ws_bytes, void* stream);

dg_status dg_tp_linear_bwd(int64_t rows, int64_t in_features, int64_t out_features,
                           const void* x, const void* weight, const void* dy,
                           void* dx, void* d_weight, void* d_bias,
                           void* ws, size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------------
 * Diagnostics.
 * dg_debug_wait_timeout launches one small kernel that waits, with the
 * library's bounded wait, on a barrier nothing will ever arrive at; after
 * `limit_us` microseconds the wait gives up and records DG_ERR_TIMEOUT in the
 * error block of `ws` (ws_bytes >= DG_ERROR_BLOCK_BYTES), which
 * dg_check_device_error(ws, ...) then reports.  It exists to test the
 * failure path without faulting or hanging the GPU.
 * ------------------------------------------------------------------------ */
dg_status dg_debug_wait_timeout(void* ws, size_t ws_bytes, uint32_t limit_us, void* stream);

/* ------------------------------------------------------------------------
 * Launch tracing.
 * Between dg_trace_begin() and dg_trace_end(), every kernel the library
 * enqueues (on any stream, from any thread) is bracketed by two CUDA events
 * and recorded with its name and its algorithmic work: FLOPs (2*M*N*K per
 * GEMM problem) and the minimum HBM bytes the kernel must move.
 * dg_trace_end() synchronises the recorded events, aggregates them by kernel
 * name into `out` (up to `max_entries`, in first-launch order), stops
 * recording and returns the number of distinct kernels (or -1 on a CUDA
 * error).  Tracing adds two event records per launch and is off by default.
 * ------------------------------------------------------------------------ */
typedef struct {
  char name[40];
  int64_t launches;
  double total_ms;   /* sum of event-timed durations */
  double flops;      /* algorithmic FLOPs summed over launches */
  double bytes;      /* algorithmic HBM bytes summed over launches */
} dg_trace_entry;

dg_status dg_trace_begin(void);
int32_t dg_trace_end(dg_trace_entry* out, int32_t max_entries);

/* dg_trace_begin_only: as dg_trace_begin, but records only the launches named
 * `name` (a NUL-terminated kernel name as reported by dg_trace_end; NULL or ""
 * records every launch).  Launches not recorded get no events, so the
 * kernels around them keep their programmatic-launch overlap. */
dg_status dg_trace_begin_only(const char* name);

#ifdef __cplusplus
}
#endif

#endif /* DG_H */
