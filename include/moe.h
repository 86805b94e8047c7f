/*
 * moe.h -- C-ABI of the GB300 (sm_103a) grouped MoE prefill library.
 *
 * The path computed here is the heterogeneous MoE prefill batched by expert
 * of the page "perf(ds4): batch heterogeneous MoE prefill by expert"
 * (Luce-Org/lucebox PR #640), Summary: every token is routed to its top-k of
 * up to 256 routed experts; a route histogram, an exclusive prefix over the
 * expert counts and a scatter put the token rows in expert-major order;
 * grouped gate/up projections with SwiGLU and a grouped down projection run
 * per expert; a weighted combine returns the expert outputs to token order,
 * and masked (non-owned) routes contribute exactly zero.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Every pointer argument is a DEVICE pointer owned by the caller, unless
 *   its description says otherwise.  The library never allocates device
 *   memory and never frees caller memory.
 * - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *   stream).  Every call only enqueues work on `stream` and returns; nothing
 *   synchronises except moe_check_device_error().
 * - Matrices are dense and row-major.  Notation: T tokens, E experts
 *   (1..256), k experts per token (1..min(E,16)), d hidden size, f expert FFN
 *   size, R = number of unmasked routes (<= T*k), "route" r = t*k + s for
 *   token t and slot s.
 * - Expert weights are stored K-contiguous (the nn.Linear convention):
 *   w_gate and w_up are [E][f][d], w_down is [E][d][f].
 * - Compact (expert-major) buffers xs, h and y are sized for the worst case,
 *   T*k rows ("capacity"); rows R .. T*k-1 are zero-filled by the call that
 *   produces the buffer.  R itself stays on the device in offsets[E].
 * - Operand types: MOE_BF16 (bf16 operands, fp32 accumulation in tensor
 *   memory, h stored as bf16) or MOE_F32 (fp32 operands and fp32 FMA
 *   arithmetic, h stored as fp32).  y and out are always fp32.
 * - Row starts of x, xs, h, y and out must be 16-byte aligned: the base
 *   pointers must be 16-byte aligned and d*sizeof(operand), f*sizeof(operand)
 *   multiples of 16 bytes.  The bf16 tensor-core path needs d and f to be
 *   multiples of 128.
 * - Errors: a call returns MOE_ERR_INVALID_ARG without enqueuing anything
 *   when an argument is out of range, null where it must not be, or
 *   misaligned; MOE_ERR_UNSUPPORTED when the current device is not an
 *   sm_103 GPU or the operand type is unknown; MOE_ERR_CUDA when a launch
 *   fails (moe_last_cuda_error() gives the cudaError_t).  Conditions that are
 *   only visible on the device (inconsistent offsets, a bounded wait that ran
 *   out) set a sticky device error word instead; moe_check_device_error()
 *   reports and clears it.
 * - The calls keep no host state between calls apart from a per-device
 *   cache (SM count, kernel attributes, the address of the device error
 *   word); they are safe to call from several host threads.  Device
 *   addresses in the cache are tied to the CUDA context they were looked up
 *   in and are looked up again when another context is current (after
 *   cudaDeviceReset, for instance).
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum moe_status {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,  /* bad size, null pointer or misalignment (host check), or bad offsets (device check) */
    MOE_ERR_UNSUPPORTED = 2,  /* not an sm_103 device, or an unknown operand type */
    MOE_ERR_CUDA = 3,         /* a CUDA runtime/driver call failed; see moe_last_cuda_error() */
    MOE_ERR_TIMEOUT = 4,      /* a bounded wait inside a kernel ran out (device error word) */
    MOE_ERR_RANGE = 5         /* a value did not fit the fp16 operands of the FP8-weight path (device error word) */
} moe_status;

typedef enum moe_dtype {
    MOE_F32 = 0,
    MOE_BF16 = 1
} moe_dtype;

/* Library version as 10000*major + 100*minor + patch. */
int moe_version(void);

/* Static text for a status code (never NULL). */
const char* moe_status_string(int status);

/* The cudaError_t of the last failed CUDA call made by this library on this
 * host thread (0 if none). */
int moe_last_cuda_error(void);

/* Synchronises `stream`, then reads and clears the sticky device error word
 * of the current device.  Returns MOE_OK, MOE_ERR_TIMEOUT (a bounded wait in
 * a kernel ran out; that kernel's outputs are undefined),
 * MOE_ERR_INVALID_ARG (a kernel found inconsistent offsets and skipped its
 * work) or MOE_ERR_RANGE (the FP8-weight path met an activation beyond the
 * fp16 range; the affected outputs hold infinities). */
moe_status moe_check_device_error(void* stream);

/* Enqueues on `stream` the clearing of the current device's sticky error
 * word, without synchronising (moe_check_device_error reads and clears it
 * after a synchronisation).  For a caller that has handled a reported error
 * and wants the word clear before its next calls on `stream`. */
moe_status moe_clear_device_error(void* stream);

/* Diagnostic of the failure detection.  Every wait of the tensor-core
 * kernels on a copy or an MMA is bounded (2 s); when one runs out the kernel
 * abandons its work, drains what it has in flight, frees its tensor memory
 * and records MOE_ERR_TIMEOUT in the device error word (the runs on the page
 * "perf(ds4): extend sparse prefill scheduling to 10K" are likewise bounded
 * by a guard and a timeout, and an aborted run counts as failed).  This call
 * runs that same bounded wait on a barrier that nothing completes, giving up
 * after limit_ms (1..5000) milliseconds, so that a caller can check the
 * detection end to end: the following moe_check_device_error() returns
 * MOE_ERR_TIMEOUT and clears the word.  It faults nothing and leaves the
 * context usable. */
moe_status moe_selftest_bounded_wait(int limit_ms, void* stream);

/* Bytes of scratch workspace `ws` needed by moe_route_histogram,
 * moe_prefix_offsets, moe_scatter_rows and moe_forward for T tokens and
 * k slots.  The workspace must be zero-filled once before its first use
 * (e.g. cudaMemset); the calls leave it ready for the next call.  One
 * workspace serves one stream at a time.  T >= 0, 1 <= k <= 16. */
moe_status moe_workspace_size(int T, int k, size_t* bytes);

/* The router projection in front of A1, with A1 in its epilogue.  Page
 * "perf(ds4): extend sparse prefill scheduling to 10K", Summary (native
 * top-6 routing over the routed experts, from the router logits).
 *   x      [T][d] bf16 token rows; d a multiple of 64.
 *   wr     [E][d] bf16 router matrix (K-contiguous, like the expert weights).
 *   logits [T][E] fp32 out, or NULL: logits[t][e] = x[t] . wr[e], bf16
 *          products accumulated in fp32 on the tensor cores.
 *   ids, w [T][k] out: as moe_route_topk applied to those logits (the k
 *          largest in descending order, ties to the lower expert id; softmax
 *          over the k selected, summed in slot order). */
moe_status moe_router_topk(const void* x, const void* wr, int T, int E, int d, int k,
                           float* logits, int32_t* ids, float* w, void* stream);

/* A1 -- top-k routing.  Page "perf(ds4): batch heterogeneous MoE prefill by
 * expert", Summary (routed experts, up to 256) and page "perf(ds4): extend
 * sparse prefill scheduling to 10K", Summary (native top-6 routing).
 *   logits [T][E] fp32 (finite values).
 *   ids    [T][k] int32 out: the k largest logits in descending order, ties
 *          to the lower expert id (-0.0 equals +0.0).
 *   w      [T][k] fp32 out: softmax over the k selected logits. */
moe_status moe_route_topk(const float* logits, int T, int E, int k,
                          int32_t* ids, float* w, void* stream);

/* A2 -- route histogram.  Page "perf(ds4): batch heterogeneous MoE prefill
 * by expert", Summary (GPU-native route histogram for up to 256 experts).
 *   ids    [T][k] int32, each in [0, E).
 *   mask   [T][k] uint8 or NULL; nonzero = route masked (owned elsewhere),
 *          not counted.
 *   counts [E] int32 out: unmasked routes per expert.
 *   ws     workspace (moe_workspace_size); receives per-chunk counts and the
 *          stable rank of every route inside its chunk. */
moe_status moe_route_histogram(const int32_t* ids, const uint8_t* mask, int T, int k, int E,
                               int32_t* counts, void* ws, void* stream);

/* A1 + A2 + A3 in one launch: the outputs of moe_route_topk,
 * moe_route_histogram and moe_prefix_offsets (ids, w, counts, offsets, and
 * the workspace the scatter reads), bit for bit.  One CTA per workspace
 * chunk of tokens routes its tokens (a warp per token), ranks their routes
 * and counts them; the last CTA to finish sums the counts and writes the
 * prefix and the chunk bases.  The gate weights equal moe_route_topk's bit
 * for bit when E is a multiple of 4 (its streaming kernel sums the softmax
 * in slot order, as this one does); for other E they may differ from it in
 * the last bit.  Chunks of more than 8,192 tokens run the three step kernels
 * (the streaming top-k scales better there).
 *   logits [T][E], mask [T][k] or NULL, ids, w [T][k], counts [E],
 *   offsets [E+1], ws: as for the three calls. */
moe_status moe_route_topk_offsets(const float* logits, const uint8_t* mask, int T, int E, int k,
                                  int32_t* ids, float* w, int32_t* counts, int32_t* offsets, void* ws,
                                  void* stream);

/* Allocation-free variant of moe_route_histogram.  The pages have no
 * counterpart of this entry point: it serves callers that cannot allocate
 * device memory, such as code plugged into a host framework that owns every
 * device allocation and hands its kernels no workspace, or runtimes that
 * forbid allocation once they have started.  Such a caller passes only
 * inputs and outputs:
 *   ids, mask, T, k, E, counts  as for moe_route_histogram (same counts).
 * The scratch (per-chunk counts, in-chunk ranks and a completion counter,
 * 512 KB) is a static device array inside the library; every GPU that loads
 * the library keeps it until the process exits.
 *   Limit: T*k <= 65536 routes; a larger chunk returns MOE_ERR_INVALID_ARG
 *   without enqueuing anything.
 *   The first call on a device looks up the array's device address (with
 *   that device current) and caches it for the CUDA context that is current;
 *   when another context is current later (after cudaDeviceReset, say) the
 *   next call looks it up again.  Make the first call before any stream
 *   capture.
 *   Every call on a device shares the one array and it keeps the previous
 *   call's contents; the call clears what must start at zero itself.  Calls
 *   that can overlap on the GPU (other streams, other host threads) race and
 *   give wrong counts: serialise them.
 *   Nothing is allocated: no cudaMalloc, no cudaFree. */
moe_status moe_route_histogram_noalloc(const int32_t* ids, const uint8_t* mask, int T, int k, int E,
                                       int32_t* counts, void* stream);

/* A3 -- exclusive prefix over expert counts.  Same page, Summary
 * (GPU-native prefix).
 *   counts  [E] int32 from moe_route_histogram with the same T, k, E, ws.
 *   offsets [E+1] int32 out: offsets[0] = 0, offsets[e+1] = offsets[e] +
 *           counts[e]; offsets[E] = R.
 *   ws      the workspace moe_route_histogram filled; the per-chunk counts
 *           are read (not modified) and per-chunk row bases for the scatter
 *           are written to another part of it, so the call may be repeated. */
moe_status moe_prefix_offsets(const int32_t* counts, int T, int k, int E,
                              int32_t* offsets, void* ws, void* stream);

/* A4 -- scatter to expert-major order (every expert id, compact row and R is
 * range-checked on the device before a write; a workspace that was not
 * prepared by moe_route_histogram + moe_prefix_offsets for these ids makes
 * moe_check_device_error() report MOE_ERR_INVALID_ARG, with no write outside
 * xs, row_of_route and route_of_row).  Same page, Summary (GPU-native
 * scatter) and "Correctness and validation" (compact destinations are
 * zero-initialised).
 *   x            [T][d] operand type `dtype`.
 *   ids, mask    as for moe_route_histogram (same values).
 *   offsets      [E+1] from moe_prefix_offsets.
 *   xs           [T*k][d] out: row offsets[e] + j holds the token row of the
 *                j-th unmasked route to expert e in ascending route order;
 *                rows R .. T*k-1 are zero-filled.
 *   row_of_route [T*k] int32 out: compact row of route r, -1 when masked.
 *   route_of_row [T*k] int32 out: route of compact row i, -1 for i >= R.
 *   ws           the workspace moe_prefix_offsets prepared. */
moe_status moe_scatter_rows(const void* x, int dtype, const int32_t* ids, const uint8_t* mask,
                            const int32_t* offsets, int T, int k, int d, int E,
                            void* xs, int32_t* row_of_route, int32_t* route_of_row,
                            void* ws, void* stream);

/* A1-A4 in one launch for small chunks -- the verification-width batches of
 * the page "perf(ds4): accelerate ROCm decode and long-context selection"
 * (q=4 verification) and any chunk with T <= 128 and T*k <= 512.  Every CTA
 * recomputes the routing of the whole chunk (cheaper than three more
 * launches at these sizes) and copies its share of the token rows.
 * Outputs are those of moe_route_topk + moe_route_histogram +
 * moe_prefix_offsets + moe_scatter_rows (or moe_scatter_rows_f16 when
 * xs_f16 != 0, x bf16), bit for bit when E is a multiple of 4 (for other E
 * the gate weights sum the softmax in slot order, which may differ from
 * moe_route_topk in the last bit).  No workspace.
 *   logits [T][E], x [T][d] (dtype), mask [T][k] or NULL: as above.
 *   ids, w, counts, offsets, xs, row_of_route, route_of_row: out, as above.
 * moe_forward and moe_forward_fp8 use this call for such chunks. */
moe_status moe_route_scatter_small(const float* logits, const void* x, int dtype, int xs_f16,
                                   const uint8_t* mask, int T, int E, int k, int d,
                                   int32_t* ids, float* w, int32_t* counts, int32_t* offsets,
                                   void* xs, int32_t* row_of_route, int32_t* route_of_row, void* stream);

/* A5 -- grouped gate/up projection with SwiGLU.  Same page, Summary
 * (grouped gate/up MMID graphs instead of a serial graph per active expert);
 * the SwiGLU is the "DS4 SwiGLU split op" of the page "perf(ggml): reuse
 * ROCmFP4 weights across q=4 columns".
 *   xs      [cap][d] compact rows (moe_scatter_rows), cap = capacity rows.
 *   offsets [E+1] expert segments of xs; offsets[E] <= cap (checked on the
 *           device: a violation skips the work and sets MOE_ERR_INVALID_ARG
 *           in the device error word).
 *   w_gate, w_up [E][f][d].
 *   h       [cap][f] out: h[i] = silu(xs[i].Wg_e) * (xs[i].Wu_e) for the
 *           expert e whose segment holds row i; rows R .. cap-1 zero-filled.
 * bf16: tcgen05 tensor cores, fp32 accumulation, h rounded to bf16.
 * fp32: fp32 FMA, h fp32. */
moe_status moe_grouped_gate_up(const void* xs, const int32_t* offsets, int cap, int E, int d, int f,
                               const void* w_gate, const void* w_up, int dtype, void* h, void* stream);

/* A6 -- grouped down projection.  Same page, Summary (grouped down MMID).
 *   h       [cap][f] from moe_grouped_gate_up.
 *   w_down  [E][d][f].
 *   y       [cap][d] fp32 out: y[i] = h[i].Wd_e; rows R .. cap-1
 *           zero-filled. */
moe_status moe_grouped_down(const void* h, const int32_t* offsets, int cap, int E, int d, int f,
                            const void* w_down, int dtype, float* y, void* stream);

/* Which tensor-core kernels the bf16 and E4M3 (W8A8) grouped projections
 * run for a capacity of `cap` compact rows: *paired = 1 when clusters of two
 * CTAs issue M = 256 MMAs over two SMs (chunks of many routes), 0 when each
 * CTA works alone.  The results agree within the fp32 accumulation's
 * rounding either way.  Host only; MOE_ERR_INVALID_ARG if paired is NULL or
 * cap < 0. */
moe_status moe_ffn_paired(int cap, int* paired);

/* A5 + A6 in one call (two kernels on `stream`). */
moe_status moe_grouped_ffn(const void* xs, const int32_t* offsets, int cap, int E, int d, int f,
                           const void* w_gate, const void* w_up, const void* w_down, int dtype,
                           void* h, float* y, void* stream);

/* A7 -- weighted combine back to token order.  Page "perf(ds4): accelerate
 * ROCm decode and long-context selection", lucebox8 A/B (fused expert-major
 * route combine) and page "perf(ds4): batch heterogeneous MoE prefill by
 * expert", Summary (masked owner routes are exact zero contributions).
 *   y            [cap][d] fp32 expert outputs.
 *   row_of_route [T*k] int32, -1 = masked (skipped, never multiplied); an
 *                entry >= T*k is not a row of y: it is skipped and makes
 *                moe_check_device_error() report MOE_ERR_INVALID_ARG.
 *   w            [T][k] fp32 gate weights.
 *   out          [T][d] fp32 out: out[t] = +0.0 + sum over ascending
 *                unmasked s of w[t][s] * y[row_of_route[t*k+s]], fp32
 *                fused multiply-adds in that fixed order (deterministic). */
moe_status moe_combine(const float* y, const int32_t* row_of_route, const float* w,
                       int T, int k, int d, float* out, void* stream);

/* The whole path (A1..A7) on `stream`, with every intermediate written to
 * the caller's buffers (shapes as above; mask may be NULL). */
moe_status moe_forward(const float* logits, const void* x, const uint8_t* mask,
                       int T, int E, int k, int d, int f,
                       const void* w_gate, const void* w_up, const void* w_down, int dtype,
                       int32_t* ids, float* w, int32_t* counts, int32_t* offsets,
                       void* xs, int32_t* row_of_route, int32_t* route_of_row,
                       void* h, float* y, float* out, void* ws, void* stream);

/* A4 for the FP8-weight path: moe_scatter_rows with bf16 x, writing the
 * compact rows xs as fp16 ([T*k][d], same layout).  The conversion is exact
 * for |x| <= 65504 down to 2^-17 (smaller magnitudes round to fp16
 * subnormals); a finite |x| > 65504 is written as an infinity and makes
 * moe_check_device_error() report MOE_ERR_RANGE. */
moe_status moe_scatter_rows_f16(const void* x, const int32_t* ids, const uint8_t* mask,
                                const int32_t* offsets, int T, int k, int d, int E,
                                void* xs, int32_t* row_of_route, int32_t* route_of_row,
                                void* ws, void* stream);

/* ------------------------------------------------------------------------
 * Low-bit expert weights: FP8 E4M3 with one scale per output channel.
 * The pages run their routed experts on low-bit weights (page "perf(ds4):
 * batch heterogeneous MoE prefill by expert", "Fresh main-snapshot
 * requalification": a ROCmFP2 expert model; page "perf(ggml): reuse ROCmFP4
 * weights across q=4 columns": ROCmFP4/FPX weights).  Here a weight row
 * (one output channel, K values) is stored as K OCP FP8 E4M3 codes (sign,
 * 4 exponent bits with bias 7, 3 mantissa bits, largest finite 448) and one
 * fp32 scale; the weight the FFN uses is scale * value(code), exactly.
 * The codes are widened inside the SM to fp16 (exact: every E4M3 value is an
 * fp16 value), so the compact activations xs and h of this path are fp16
 * (tcgen05 kind::f16 takes both operands in one type), the products
 * accumulate in fp32 and y and out are fp32.
 * ------------------------------------------------------------------------ */

/* Quantizes `rows` weight rows of K values (load-time step, not part of the
 * per-chunk path).
 *   w       [rows][K] operand type `dtype` (MOE_BF16 or MOE_F32), finite.
 *   codes   [rows][K] uint8 out: E4M3 code of w / scale (fp32 division,
 *           round to nearest even, saturating at +-448).
 *   scales  [rows] fp32 out: max over the row of |w|, divided by 448 in
 *           fp32; 1 for an all-zero row.
 * K must be a multiple of 16; w and codes 16-byte aligned.  For expert
 * banks pass rows = E*f (w_gate, w_up; K = d) or E*d (w_down; K = f). */
moe_status moe_quantize_weights_fp8(const void* w, int dtype, long long rows, int K,
                                    uint8_t* codes, float* scales, void* stream);

/* A5 with FP8 weights: h[i] = silu(g) * u with g = s_gate[e][j] *
 * (xs[i] . value(w_gate_q[e][j])) and u likewise from w_up_q, s_up.
 *   xs       [cap][d] fp16 compact rows (moe_scatter_rows_f16); offsets as
 *            for moe_grouped_gate_up.
 *   w_gate_q, w_up_q [E][f][d] uint8 codes; s_gate, s_up [E][f] fp32.
 *   h        [cap][f] fp16 out (round to nearest even); rows R .. cap-1
 *            zero-filled; |h| > 65504 is written as an infinity and makes
 *            moe_check_device_error() report MOE_ERR_RANGE.
 * d and f multiples of 128. */
moe_status moe_grouped_gate_up_fp8(const void* xs, const int32_t* offsets, int cap, int E, int d, int f,
                                   const uint8_t* w_gate_q, const float* s_gate,
                                   const uint8_t* w_up_q, const float* s_up, void* h, void* stream);

/* A6 with FP8 weights: y[i][j] = s_down[e][j] * (h[i] . value(w_down_q[e][j])).
 *   h        [cap][f] fp16; w_down_q [E][d][f] uint8; s_down [E][d] fp32.
 *   y        [cap][d] fp32 out; rows R .. cap-1 zero-filled. */
moe_status moe_grouped_down_fp8(const void* h, const int32_t* offsets, int cap, int E, int d, int f,
                                const uint8_t* w_down_q, const float* s_down, float* y, void* stream);

/* A5 + A6 with FP8 weights (two kernels on `stream`). */
moe_status moe_grouped_ffn_fp8(const void* xs, const int32_t* offsets, int cap, int E, int d, int f,
                               const uint8_t* w_gate_q, const float* s_gate,
                               const uint8_t* w_up_q, const float* s_up,
                               const uint8_t* w_down_q, const float* s_down,
                               void* h, float* y, void* stream);

/* The whole path (A1..A7) with FP8 expert weights: x is bf16, xs and h are
 * fp16 (moe_scatter_rows_f16 is the scatter), every other argument as for
 * moe_forward. */
moe_status moe_forward_fp8(const float* logits, const void* x, const uint8_t* mask,
                           int T, int E, int k, int d, int f,
                           const uint8_t* w_gate_q, const float* s_gate,
                           const uint8_t* w_up_q, const float* s_up,
                           const uint8_t* w_down_q, const float* s_down,
                           int32_t* ids, float* w, int32_t* counts, int32_t* offsets,
                           void* xs, int32_t* row_of_route, int32_t* route_of_row,
                           void* h, float* y, float* out, void* ws, void* stream);

/* ------------------------------------------------------------------------
 * 4-bit block-scaled expert weights.  The pages stream ROCmFP4 (and FP2/3)
 * expert weights (page "perf(ggml): reuse ROCmFP4 weights across q=4
 * columns"; page "perf(ds4): batch heterogeneous MoE prefill by expert",
 * "Fresh main-snapshot requalification").  Here a weight row of K values is
 * stored as K E2M1 codes (the 4-bit OCP MX element type: values 0, 0.5, 1,
 * 1.5, 2, 3, 4, 6 and their negatives), one E4M3 scale per block of 16
 * consecutive values and one fp32 scale per row -- the block-scaled layout
 * of NVFP4 with its per-tensor scale taken per channel.  The weight the FFN
 * uses is row scale * block scale * E2M1 value, exactly.  The codes are
 * widened inside the SM to fp16 (exact: code value times block scale has at
 * most 6 significant bits), as on the FP8-weight path, so xs and h are fp16
 * and the MMAs are kind::f16 with A in tensor memory.
 * ------------------------------------------------------------------------ */

/* Quantizes E banks of M rows of K values (load-time step), in fp32:
 *   scale  = max|row| / 2688 (2688 = 6 * 448; 1 for an all-zero row);
 *   block  = E4M3 code (nearest even, saturating) of (block max / 6) / scale;
 *   code   = E2M1 code (nearest even, saturating at 6) of w / (value(block) *
 *            scale), 0 when value(block) is 0.
 *   w             [E][M][K] operand type `dtype` (MOE_BF16 or MOE_F32).
 *   codes         [E][M][K/2] uint8 out: two codes per byte, the lower K
 *                 index in the low nibble.
 *   block_scales  [E][K/64][M][4] uint8 out: the four block scales of row m
 *                 in 64-value tile t of expert e at [e][t][m][0..3] (one
 *                 32-bit word per row and tile, the layout the FFN loads).
 *   scales        [E][M] fp32 out.
 * K a multiple of 64; w, codes and block_scales 16-byte aligned. */
moe_status moe_quantize_weights_fp4(const void* w, int dtype, int E, int M, int K, uint8_t* codes,
                                    uint8_t* block_scales, float* scales, void* stream);

/* A5 with 4-bit weights: as moe_grouped_gate_up_fp8 with (codes, block
 * scales, row scales) of moe_quantize_weights_fp4 for each bank: xs [cap][d]
 * fp16, h [cap][f] fp16 out (|h| > 65504 reported as MOE_ERR_RANGE).  d and
 * f multiples of 128. */
moe_status moe_grouped_gate_up_fp4(const void* xs, const int32_t* offsets, int cap, int E, int d, int f,
                                   const uint8_t* w_gate_q, const uint8_t* b_gate, const float* s_gate,
                                   const uint8_t* w_up_q, const uint8_t* b_up, const float* s_up, void* h,
                                   void* stream);

/* A6 with 4-bit weights: y [cap][d] fp32 out from h [cap][f] fp16. */
moe_status moe_grouped_down_fp4(const void* h, const int32_t* offsets, int cap, int E, int d, int f,
                                const uint8_t* w_down_q, const uint8_t* b_down, const float* s_down, float* y,
                                void* stream);

/* The whole path with 4-bit weights (x bf16; xs and h fp16; every other
 * argument as for moe_forward_fp8). */
moe_status moe_forward_fp4(const float* logits, const void* x, const uint8_t* mask, int T, int E, int k, int d,
                           int f, const uint8_t* w_gate_q, const uint8_t* b_gate, const float* s_gate,
                           const uint8_t* w_up_q, const uint8_t* b_up, const float* s_up, const uint8_t* w_down_q,
                           const uint8_t* b_down, const float* s_down, int32_t* ids, float* w, int32_t* counts,
                           int32_t* offsets, void* xs, int32_t* row_of_route, int32_t* route_of_row, void* h,
                           float* y, float* out, void* ws, void* stream);

/* ------------------------------------------------------------------------
 * FP8 E4M3 weights AND activations on the FP8 tensor cores.  The pages'
 * quantized expert matmuls take quantized activations too (the MMQ path of
 * the page "perf(ggml): reuse ROCmFP4 weights across q=4 columns", whose
 * weights come in ROCmFP4/FPX formats; page "perf(ds4): batch heterogeneous
 * MoE prefill by expert", "Fresh main-snapshot requalification": a ROCmFP2
 * model).  Here both operands of every expert GEMM are OCP E4M3 codes with
 * one fp32 scale per row -- per output channel for the weights (the codes of
 * moe_quantize_weights_fp8), per token row for x and per compact row for h
 * (the same quantizer applied to the activation rows) -- and the tensor
 * cores multiply the codes directly (tcgen05.mma kind::f8f6f4, K = 32 per
 * instruction), the epilogue applying the two scales.  The method computed
 * is the FFN on the values the codes stand for: x' = s_x * value(code_x),
 * h = silu(x'.Wg') * (x'.Wu') rounded to bf16, h' = s_h * value(code_h) of
 * that bf16 h, y = h'.Wd'; products accumulate in fp32.
 * ------------------------------------------------------------------------ */

/* A4 with E4M3 rows: the codes x_q [T][d] and row scales x_scales [T] of the
 * token rows (moe_quantize_weights_fp8 applied to x, rows = T, K = d) are
 * scattered like moe_scatter_rows scatters x: xs [T*k][d] uint8 (rows R ..
 * T*k-1 zero codes) and xs_scales [T*k] (the token row's scale; 0 for rows
 * R .. T*k-1).  ids, mask, offsets, row_of_route, route_of_row, ws: as for
 * moe_scatter_rows.  d a multiple of 16. */
moe_status moe_scatter_rows_e4m3(const uint8_t* x_q, const float* x_scales, const int32_t* ids, const uint8_t* mask,
                                 const int32_t* offsets, int T, int k, int d, int E, uint8_t* xs, float* xs_scales,
                                 int32_t* row_of_route, int32_t* route_of_row, void* ws, void* stream);

/* A4 with E4M3 rows straight from the bf16 token rows x [T][d]: every token
 * row is read once and quantized -- x_q [T][d] codes and x_scales [T], the
 * codes and scales moe_quantize_weights_fp8 would give -- and its codes and
 * scale written to its compact rows as moe_scatter_rows_e4m3 writes them.
 * d a multiple of 16 and at most 8192. */
moe_status moe_scatter_rows_quant_e4m3(const void* x, const int32_t* ids, const uint8_t* mask,
                                       const int32_t* offsets, int T, int k, int d, int E, uint8_t* x_q,
                                       float* x_scales, uint8_t* xs, float* xs_scales, int32_t* row_of_route,
                                       int32_t* route_of_row, void* ws, void* stream);

/* A1-A4 with E4M3 rows in one launch for small chunks (T <= 128 and T*k <=
 * 512): the routing outputs of moe_route_topk_offsets (no workspace) and the
 * rows of moe_scatter_rows_quant_e4m3, bit for bit.  d a multiple of 16. */
moe_status moe_route_scatter_quant_small_e4m3(const float* logits, const void* x, const uint8_t* mask, int T, int E,
                                              int k, int d, int32_t* ids, float* w, int32_t* counts,
                                              int32_t* offsets, uint8_t* x_q, float* x_scales, uint8_t* xs,
                                              float* xs_scales, int32_t* row_of_route, int32_t* route_of_row,
                                              void* stream);

/* E4M3 codes and one scale per row of the compact bf16 rows a [cap][K] (h
 * of the FP8-activation path), the arithmetic of moe_quantize_weights_fp8;
 * rows at or beyond R = offsets[E] (zero rows) get zero codes and scale 1
 * without being read.  K a multiple of 16 and at most 2048. */
moe_status moe_quantize_rows_e4m3(const void* a, const int32_t* offsets, int E, int cap, int K, uint8_t* codes,
                                  float* scales, void* stream);

/* A5 on E4M3 operands: h[i][j] = silu(g) * u, g = s_gate[e][j] *
 * xs_scales[i] * (codes of xs[i] . codes of w_gate_q[e][j]) and u likewise;
 * h [cap][f] bf16 out (rows R .. cap-1 zero-filled).  d and f multiples of
 * 128; offsets checked on the device as for moe_grouped_gate_up. */
moe_status moe_grouped_gate_up_w8a8(const uint8_t* xs, const float* xs_scales, const int32_t* offsets, int cap,
                                    int E, int d, int f, const uint8_t* w_gate_q, const float* s_gate,
                                    const uint8_t* w_up_q, const float* s_up, void* h, void* stream);

/* A6 on E4M3 operands: y[i][j] = s_down[e][j] * h_scales[i] * (codes of
 * h_q[i] . codes of w_down_q[e][j]); y [cap][d] fp32 out, rows R .. cap-1
 * zero-filled.  h_q, h_scales: moe_quantize_weights_fp8 applied to the bf16
 * h (rows = cap, K = f). */
moe_status moe_grouped_down_w8a8(const uint8_t* h_q, const float* h_scales, const int32_t* offsets, int cap, int E,
                                 int d, int f, const uint8_t* w_down_q, const float* s_down, float* y, void* stream);

/* The whole path on E4M3 weights and activations: routing in one launch
 * (moe_route_topk_offsets), the token rows quantized (x_q [T][d], x_scales
 * [T]) and scattered (xs, xs_scales) by moe_scatter_rows_quant_e4m3 (small
 * chunks: the three in one launch, moe_route_scatter_quant_small_e4m3),
 * moe_grouped_gate_up_w8a8 into h [T*k][f] bf16, h quantized by
 * moe_quantize_rows_e4m3 (h_q [T*k][f], h_scales [T*k]),
 * moe_grouped_down_w8a8 into y, moe_combine into out.  x is bf16; every
 * other argument as for moe_forward. */
moe_status moe_forward_w8a8(const float* logits, const void* x, const uint8_t* mask, int T, int E, int k, int d,
                            int f, const uint8_t* w_gate_q, const float* s_gate, const uint8_t* w_up_q,
                            const float* s_up, const uint8_t* w_down_q, const float* s_down, int32_t* ids, float* w,
                            int32_t* counts, int32_t* offsets, uint8_t* x_q, float* x_scales, uint8_t* xs,
                            float* xs_scales, int32_t* row_of_route, int32_t* route_of_row, void* h, uint8_t* h_q,
                            float* h_scales, float* y, float* out, void* ws, void* stream);

/* ------------------------------------------------------------------------
 * 4-bit operands on both sides (W4A4).  The weights are the 4-bit banks of
 * moe_quantize_weights_fp4; the token rows and the rows of h are quantized
 * into the same format (E2M1 codes, an E4M3 scale per 16 values, an fp32
 * scale per row) -- the NVIDIA "NVFP4" layout, and the 4-bit counterpart of
 * the FP8-activation path above (page "perf(ggml): reuse ROCmFP4 weights
 * across q=4 columns": 4-bit weights on a quantized-activation matrix path).
 * The tensor cores multiply the codes with their block scales directly
 * (tcgen05.mma kind::mxf4nvf4 with block scaling, K = 64 per instruction);
 * the epilogue applies the two row scales.  The method computed is the FFN
 * on the values the codes stand for: x' = s_x * b_x * value(code_x), h =
 * silu(x'.Wg') * (x'.Wu') rounded to bf16, h' the same quantizer applied to
 * that bf16 h, y = h'.Wd'; products accumulate in fp32.
 *
 * Rows of activations keep their block scales tile-major like the weights:
 * [K/64][ld][4] uint8, the four scales of row r in 64-value tile t at
 * [t][r][0..3], ld >= rows a multiple of 4 (the path uses ld = 4*ceil(rows/4)).
 * ------------------------------------------------------------------------ */

/* The 4-bit quantizer of moe_quantize_weights_fp4 applied to `rows` rows of
 * activations a [rows][K] (dtype MOE_BF16 or MOE_F32): codes [rows][K/2],
 * block_scales [K/64][ld][4] (columns rows .. ld-1 untouched), scales
 * [rows].  K a multiple of 64; a, codes, block_scales 16-byte aligned. */
moe_status moe_quantize_rows_fp4(const void* a, int dtype, int rows, int ld, int K, uint8_t* codes,
                                 uint8_t* block_scales, float* scales, void* stream);

/* A4 with 4-bit rows: the token rows' codes x_codes [T][d/2], block scales
 * x_block_scales [d/64][ld_x][4] and scales x_scales [T] (moe_quantize_rows_fp4
 * of x) are scattered like moe_scatter_rows scatters x, into xs_codes
 * [T*k][d/2], xs_block_scales [d/64][ld_xs][4] and xs_scales [T*k]; rows R ..
 * T*k-1 get zero codes, zero block scales and scale 0.  ld_x >= T and ld_xs
 * >= T*k multiples of 4; d a multiple of 64; other arguments as for
 * moe_scatter_rows. */
moe_status moe_scatter_rows_fp4(const uint8_t* x_codes, const uint8_t* x_block_scales, int ld_x,
                                const float* x_scales, const int32_t* ids, const uint8_t* mask,
                                const int32_t* offsets, int T, int k, int d, int E, uint8_t* xs_codes,
                                uint8_t* xs_block_scales, int ld_xs, float* xs_scales, int32_t* row_of_route,
                                int32_t* route_of_row, void* ws, void* stream);

/* A4 with 4-bit rows straight from the bf16 token rows x [T][d]: every token
 * row is read once and quantized -- x_codes, x_block_scales, x_scales, what
 * moe_quantize_rows_fp4 would give -- and written to its compact rows as
 * moe_scatter_rows_fp4 writes them.  d a multiple of 64 and at most 8192. */
moe_status moe_scatter_rows_quant_fp4(const void* x, const int32_t* ids, const uint8_t* mask, const int32_t* offsets,
                                      int T, int k, int d, int E, uint8_t* x_codes, uint8_t* x_block_scales,
                                      int ld_x, float* x_scales, uint8_t* xs_codes, uint8_t* xs_block_scales,
                                      int ld_xs, float* xs_scales, int32_t* row_of_route, int32_t* route_of_row,
                                      void* ws, void* stream);

/* A1-A4 with 4-bit rows in one launch for small chunks (T <= 128 and T*k
 * <= 512, as moe_route_scatter_small): the routing outputs of
 * moe_route_topk_offsets (ids, w, counts, offsets, row_of_route,
 * route_of_row; no workspace) and the quantized, scattered rows of
 * moe_scatter_rows_quant_fp4, bit for bit.  d a multiple of 64. */
moe_status moe_route_scatter_quant_small_fp4(const float* logits, const void* x, const uint8_t* mask, int T, int E,
                                             int k, int d, int32_t* ids, float* w, int32_t* counts, int32_t* offsets,
                                             uint8_t* x_codes, uint8_t* x_block_scales, int ld_x, float* x_scales,
                                             uint8_t* xs_codes, uint8_t* xs_block_scales, int ld_xs,
                                             float* xs_scales, int32_t* row_of_route, int32_t* route_of_row,
                                             void* stream);

/* A5 on 4-bit operands: h[i][j] = silu(g) * u with g = s_gate[e][j] *
 * xs_scales[i] * sum over K of (b_gate * value(code)) (xs block scale *
 * value(code)) and u likewise; h [cap][f] bf16 out (rows R .. cap-1
 * zero-filled).  xs_*: compact rows in the 4-bit row format (leading
 * dimension ld of the block scales, ld >= cap a multiple of 4); weights as
 * moe_quantize_weights_fp4 writes them.  d and f multiples of 128. */
moe_status moe_grouped_gate_up_w4a4(const uint8_t* xs_codes, const uint8_t* xs_block_scales, int ld,
                                    const float* xs_scales, const int32_t* offsets, int cap, int E, int d, int f,
                                    const uint8_t* w_gate_q, const uint8_t* b_gate, const float* s_gate,
                                    const uint8_t* w_up_q, const uint8_t* b_up, const float* s_up, void* h,
                                    void* stream);

/* A6 on 4-bit operands: y [cap][d] fp32 out (rows R .. cap-1 zero-filled)
 * from the 4-bit rows of h (moe_quantize_rows_fp4 of the bf16 h, rows = cap,
 * K = f, leading dimension ld). */
moe_status moe_grouped_down_w4a4(const uint8_t* h_codes, const uint8_t* h_block_scales, int ld,
                                 const float* h_scales, const int32_t* offsets, int cap, int E, int d, int f,
                                 const uint8_t* w_down_q, const uint8_t* b_down, const float* s_down, float* y,
                                 void* stream);

/* The whole path on 4-bit weights and activations: moe_route_topk_offsets;
 * x quantized and scattered by moe_scatter_rows_quant_fp4 (small chunks: the
 * routing and this step in one launch, moe_route_scatter_quant_small_fp4;
 * above d = 8192:
 * moe_quantize_rows_fp4, then moe_scatter_rows_fp4): x_codes [T][d/2],
 * x_block_scales [d/64][4*ceil(T/4)][4], x_scales [T]; xs_codes [T*k][d/2], xs_block_scales
 * [d/64][4*ceil(T*k/4)][4], xs_scales [T*k]); moe_grouped_gate_up_w4a4 into
 * h [T*k][f] bf16; h quantized (h_codes [T*k][f/2], h_block_scales
 * [f/64][4*ceil(T*k/4)][4], h_scales [T*k]); moe_grouped_down_w4a4 into y;
 * moe_combine into out.  x is bf16; every other argument as for moe_forward. */
moe_status moe_forward_w4a4(const float* logits, const void* x, const uint8_t* mask, int T, int E, int k, int d,
                            int f, const uint8_t* w_gate_q, const uint8_t* b_gate, const float* s_gate,
                            const uint8_t* w_up_q, const uint8_t* b_up, const float* s_up, const uint8_t* w_down_q,
                            const uint8_t* b_down, const float* s_down, int32_t* ids, float* w, int32_t* counts,
                            int32_t* offsets, uint8_t* x_codes, uint8_t* x_block_scales, float* x_scales,
                            uint8_t* xs_codes, uint8_t* xs_block_scales, float* xs_scales, int32_t* row_of_route,
                            int32_t* route_of_row, void* h, uint8_t* h_codes, uint8_t* h_block_scales,
                            float* h_scales, float* y, float* out, void* ws, void* stream);

/* ------------------------------------------------------------------------
 * Fused permutation (bf16 operands only).  The pages fuse the combine into
 * one expert-major kernel (page "perf(ds4): accelerate ROCm decode and
 * long-context selection", lucebox8 gfx1151 A/B; page "perf(ds4): extend
 * sparse prefill scheduling to 10K", historical fused-combine
 * discriminator).  Here the permutation moves into the GEMMs themselves:
 * the gate/up kernel gathers token rows from x (no compact copy xs), and the
 * down kernel adds each token's slots into out as soon as the last of them
 * is stored (no separate combine).  out is bit-identical to the unfused
 * path's (same values of h and y, same fixed-order fp32 combine).
 * ------------------------------------------------------------------------ */

/* Bytes of the slot counters `tile_counts` of the fused combine for T
 * tokens of width d: T * ceil(d/128) int32. */
moe_status moe_tile_counts_size(int T, int d, size_t* bytes);

/* A4 with the fused combine's preparation.  Writes row_of_route and
 * route_of_row exactly as moe_scatter_rows does (same checks), sets
 * tile_counts to zero, and sets out[t] to +0.0 for every token whose k slots
 * are all masked (no down item reaches such a token).  With x and xs given
 * it also writes the compact rows xs as moe_scatter_rows does; with both
 * NULL it copies no rows (for moe_grouped_gate_up_gather).
 *   ids, mask, offsets, ws: as for moe_scatter_rows.
 *   x, xs        [T][d], [T*k][d] bf16, both or neither.
 *   tile_counts  [T][ceil(d/128)] int32 out, zeroed.
 *   out          [T][d] fp32; only the rows of all-masked tokens are written.
 * d a multiple of 8; out, x and xs 16-byte aligned. */
moe_status moe_scatter_index(const int32_t* ids, const uint8_t* mask, const int32_t* offsets,
                             int T, int k, int d, int E, const void* x, void* xs,
                             int32_t* row_of_route, int32_t* route_of_row,
                             int32_t* tile_counts, float* out, void* ws, void* stream);

/* moe_route_scatter_small (bf16 x) with the preparation of moe_scatter_index:
 * A1-A4 in one launch for a chunk with T <= 128 and T*k <= 512, tile_counts
 * zeroed and out[t] = +0.0 for every token whose slots are all masked; xs
 * NULL copies no rows (for moe_grouped_gate_up_gather).  d a multiple of 8;
 * x, xs and out 16-byte aligned. */
moe_status moe_route_scatter_small_fused(const float* logits, const void* x, const uint8_t* mask,
                                         int T, int E, int k, int d,
                                         int32_t* ids, float* w, int32_t* counts, int32_t* offsets,
                                         void* xs, int32_t* row_of_route, int32_t* route_of_row,
                                         int32_t* tile_counts, float* out, void* stream);

/* A5 reading the token rows directly: h[i] = silu(x[t].Wg_e) * (x[t].Wu_e)
 * with t = route_of_row[i] / k, for every compact row i < offsets[E] (the
 * expert e whose segment holds i); rows R .. T*k-1 of h are zero-filled.
 * Bit-identical to moe_scatter_rows + moe_grouped_gate_up.
 *   x             [T][d] bf16, 16-byte aligned.
 *   route_of_row  [T*k] from moe_scatter_index / moe_scatter_rows; an entry
 *                 outside [0, T*k) for a row below R makes
 *                 moe_check_device_error() report MOE_ERR_INVALID_ARG.
 *   offsets, w_gate, w_up, h: as for moe_grouped_gate_up with cap = T*k.
 * d and f multiples of 128. */
moe_status moe_grouped_gate_up_gather(const void* x, int T, int k, const int32_t* route_of_row,
                                      const int32_t* offsets, int E, int d, int f,
                                      const void* w_gate, const void* w_up, void* h, void* stream);

/* A6 + A7: the down projection with the weighted combine in the same kernel.
 * out[t] for every token with at least one unmasked slot is written exactly
 * as moe_combine writes it (+0.0, then w[t][s] * y_s by fp32 FMAs in
 * ascending unmasked slot order); rows of all-masked tokens are left to
 * moe_scatter_index.
 *   h, offsets, w_down: as for moe_grouped_down with cap = T*k (bf16).
 *   route_of_row, row_of_route  [T*k] from moe_scatter_index.
 *   w            [T][k] fp32 gate weights.
 *   y            [T*k][d] fp32 scratch (the exchange buffer between the CTAs
 *                that own a token's slots); its contents are undefined after
 *                the call.  128-byte aligned.
 *   tile_counts  [T][ceil(d/128)] int32, zero on entry (moe_scatter_index
 *                zeroes them); left nonzero.
 *   out          [T][d] fp32 out, 16-byte aligned.
 * d and f multiples of 128. */
moe_status moe_grouped_down_combine(const void* h, const int32_t* offsets, int T, int k, int E, int d, int f,
                                    const void* w_down, const int32_t* route_of_row,
                                    const int32_t* row_of_route, const float* w, float* y,
                                    int32_t* tile_counts, float* out, void* stream);

/* Modes of moe_forward_fused. */
enum {
    MOE_FUSED_AUTO = 0,     /* GATHER while T*k <= 16*E (few rows per expert); else COMPACT while y
                               (T*k*d*4 bytes) fits in twice the L2; else NONE */
    MOE_FUSED_GATHER = 1,   /* rows gathered by the gate/up kernel; xs unused (may be NULL) */
    MOE_FUSED_COMPACT = 2,  /* compact copy xs, the plain gate/up kernel, the fused down + combine */
    MOE_FUSED_NONE = 3      /* the unfused path (moe_forward): y is written as moe_grouped_down writes it */
};

/* The mode moe_forward_fused chooses for MOE_FUSED_AUTO on the current
 * device for a chunk of T tokens of width d (have_xs: a compact buffer xs
 * is passed; without one the gather mode is the only choice).  *mode gets
 * MOE_FUSED_GATHER, MOE_FUSED_COMPACT or MOE_FUSED_NONE. */
moe_status moe_forward_fused_mode(int T, int E, int k, int d, int have_xs, int* mode);

/* The whole path with the fused combine (bf16): the routing (one launch for
 * chunks with T <= 128 and T*k <= 512, else moe_route_topk,
 * moe_route_histogram, moe_prefix_offsets and moe_scatter_index), the gate/up
 * projection (moe_grouped_gate_up_gather, or moe_grouped_gate_up on the
 * compact rows), moe_grouped_down_combine.  Arguments as for moe_forward
 * without dtype; xs may be NULL (then the gather mode is used); y is scratch
 * except in mode NONE; tile_counts as above.  Every mode gives the same out,
 * bit for bit, as moe_forward. */
moe_status moe_forward_fused(const float* logits, const void* x, const uint8_t* mask,
                             int T, int E, int k, int d, int f,
                             const void* w_gate, const void* w_up, const void* w_down, int mode,
                             int32_t* ids, float* w, int32_t* counts, int32_t* offsets, void* xs,
                             int32_t* row_of_route, int32_t* route_of_row,
                             void* h, float* y, int32_t* tile_counts, float* out, void* ws, void* stream);

/* ------------------------------------------------------------------------
 * Plans: the path for fixed shapes, weights and buffers, prepared once.
 * The verification batches of the page "perf(ggml): reuse ROCmFP4 weights
 * across q=4 columns" (q=4 columns) and the decode-like chunks of the page
 * "perf(ds4): accelerate ROCm decode and long-context selection" run the
 * same small path over and over on the same buffers; a plan does the host
 * work that depends only on shapes and pointers once -- the argument
 * checks, the device lookup and the TMA tensor maps of the expert weights
 * and of the compact buffers xs and h -- so that each call only launches.
 * ------------------------------------------------------------------------ */
typedef struct moe_plan moe_plan;

/* Creates a plan for chunks of exactly T tokens (T >= 1) with the given
 * weights and buffers, on the current device and CUDA context.  Arguments as
 * for moe_forward (dtype MOE_BF16 or MOE_F32; the same shapes, alignment
 * and workspace rules).  The plan records the pointers; it owns none of the
 * memory, which must stay allocated while the plan is used.  The plan itself
 * is host memory, released by moe_plan_destroy; nothing is allocated on the
 * device.  *plan is set to NULL when creation fails. */
moe_status moe_plan_create(int T, int E, int k, int d, int f, int dtype,
                           const void* w_gate, const void* w_up, const void* w_down,
                           int32_t* ids, float* w, int32_t* counts, int32_t* offsets, void* xs,
                           int32_t* row_of_route, int32_t* route_of_row, void* h, float* y, void* ws,
                           moe_plan** plan);

/* Releases a plan (NULL is accepted). */
moe_status moe_plan_destroy(moe_plan* plan);

/* A5 and A6 on the plan's buffers (moe_grouped_gate_up / moe_grouped_down
 * with the plan's xs, offsets, weights, h and y), launched from the
 * prepared tensor maps.  MOE_ERR_INVALID_ARG when the current device or
 * context is not the plan's. */
moe_status moe_plan_grouped_gate_up(const moe_plan* plan, void* stream);
moe_status moe_plan_grouped_down(const moe_plan* plan, void* stream);

/* moe_forward on the plan's weights and buffers for one chunk: logits
 * [T][E], x [T][d] (the plan's operand type), mask [T][k] or NULL, out
 * [T][d] fp32.  Same kernels, same results bit for bit, as moe_forward. */
moe_status moe_plan_forward(const moe_plan* plan, const float* logits, const void* x, const uint8_t* mask,
                            float* out, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_GB300_H */
