/*
 * ffn.h -- C ABI of the GB300 (sm_103a) pre-norm SwiGLU feed-forward block.
 *
 *   n = RMSNorm(x) = x * rsqrt(mean(x^2) + eps) * g
 *   y = W_down * ( silu(W_gate * n) (*) (W_up * n) ),   silu(z) = z / (1 + e^-z)
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Tensor pointers are DEVICE pointers owned by the caller.  The library never
 *   allocates, frees or synchronises device memory (ffn_device_status and
 *   ffn_timing_collect are the only calls that synchronise).
 * - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy default
 *   stream).  Every buffer must stay alive and unmodified until the stream has
 *   passed the call: the library does not track buffer lifetimes ("How
 *   Megakernels Work", section "Dependencies and synchronization": buffers may
 *   not be released while submitted work can still read them).
 * - Row-major layouts.  Activations are [rows x d]; weights are [out x in] with
 *   the input (reduction) dimension contiguous.
 * - All arithmetic is fp32 on fp32/fp16/bf16 storage; every stored output is
 *   rounded once, round-to-nearest-even, to the storage type.
 * - Arguments are validated on the host before any launch.  A violation
 *   returns an error status and launches nothing.  rows == 0 (an empty batch)
 *   is valid and launches nothing (x, y and n may then be NULL).  Pointers
 *   must be 16-byte aligned.
 * - After launching, a failed launch is reported as FFN_ERR_CUDA.  A kernel
 *   that gives up a bounded wait records FFN_ERR_TIMEOUT in a device status
 *   word that ffn_device_status() reads; no C++ exception crosses this ABI.
 * - A workspace must not be shared by calls that may run concurrently.
 */
#ifndef FFN_GB300_H
#define FFN_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    FFN_OK = 0,
    FFN_ERR_NULL = 1,       /* a required pointer is NULL                          */
    FFN_ERR_SHAPE = 2,      /* a size is out of range or breaks a divisibility rule */
    FFN_ERR_DTYPE = 3,      /* unknown or unsupported storage type                 */
    FFN_ERR_ALIGN = 4,      /* a pointer is not 16-byte aligned                    */
    FFN_ERR_WORKSPACE = 5,  /* workspace NULL or smaller than the query returned   */
    FFN_ERR_ALIAS = 6,      /* an output overlaps an input it may not overlap      */
    FFN_ERR_CUDA = 7,       /* a CUDA runtime call failed                          */
    FFN_ERR_TIMEOUT = 8,    /* a kernel abandoned a bounded wait                   */
    FFN_ERR_FLAGS = 9,      /* contradictory or unknown flag bits                  */
    FFN_ERR_RANGE = 10      /* a weight does not fit the prepared (fp16) format    */
} ffn_status;

typedef enum { FFN_F32 = 0, FFN_F16 = 1, FFN_BF16 = 2 } ffn_dtype;

/* flags for ffn_block_forward / ffn_block_forward_q4 */
#define FFN_AUTO 0u
/* tensor-core path: silu(G)*U computed in the gate/up GEMM epilogue (default) */
#define FFN_GATEUP_FUSED 1u
/* tensor-core path: the gate/up GEMM stores G and U (fp32, so h is still
 * rounded once); a separate SwiGLU pass reads them back ("Unfusing a Kernel
 * Made It 1.63x Faster", Finding 1)                                          */
#define FFN_GATEUP_UNFUSED 2u
/* force the tcgen05 tensor-core GEMM path (16-bit dtypes, any rows)          */
#define FFN_PATH_GEMM 4u
/* force the weight-streaming decode path (16-bit dtypes, rows <= 64)         */
#define FFN_PATH_GEMV 8u
/* 16-bit paths: n (RMSNorm output) and h (silu(G)*U) enter the tensor-core
 * operations as one rounding to the storage type (fastest).  With bf16 this
 * leaves max|y - y_exact| up to about 2.2e-2 * rms(y), above the 2e-2 bound,
 * so it is opt-in.                                                          */
#define FFN_ACT_SINGLE 16u
/* 16-bit paths: n and h enter as two terms hi + lo (hi = round(v),
 * lo = round(v - hi)), each multiplied by the same weight tile: ~16
 * significant bits, at twice the MMA work.  Default for bf16 (and Q4);
 * opt-in for fp16, whose 11 bits already fit the budget.                    */
#define FFN_ACT_SPLIT 32u
/* 16-bit paths: w_gate, w_up and w_down hold ffn_prepare_weights output (fp16
 * values of w * 2^8) while x, g and y keep `dtype`.  n and h enter every
 * tensor op as one fp16 rounding (11 significant bits; h is stored times
 * 2^-8, which keeps it clear of fp16 overflow up to |h| ~ 1.6e7), at single-
 * term speed.  Not combinable with FFN_ACT_SPLIT or FFN_F32.               */
#define FFN_PREPARED_WEIGHTS 64u
/* The block's skip connection: y = x + W_down (silu(W_gate n) * (W_up n)),
 * x added in fp32 before y's one rounding (every path, ffn_block_forward and
 * ffn_block_forward_q4).  No counterpart on the pages, whose block output
 * stops at the down projection; the pre-norm layer adds its input back.    */
#define FFN_RESIDUAL 128u
/* Decode (weight-streaming) path, where its TMA-streamed kernels run: the
 * whole block as ONE persistent kernel -- a cooperative launch in which the
 * RMSNorm, gate/up and down stages hand over through counters and flags in
 * memory, and a CTA done with gate/up streams its down weights at once
 * ("Megakernels on Mac: What Fusion Saves and What It Costs", sections
 * "Dependencies and synchronization" and "Small gaps between dispatches").
 * Same results within the bounds; on GB300 slower than the default chain of
 * three programmatically dependent kernels (e.g. 8 x 4096 -> 14336 bf16: 69
 * against 62 us), so opt-in.  Also accepted by ffn_block_forward_q4 / _fp8 /
 * _q8 and ffn_block_forward_chained; ignored where the block runs otherwise. */
#define FFN_DECODE_ONE_KERNEL 256u

/* ------------------------------------------------------------------------
 * ffn_rmsnorm -- n[r,c] = x[r,c] * rsqrt(ms_r + eps) * g[c],
 *                ms_r = (1/d) sum_c x[r,c]^2 accumulated in fp32.
 * "When to hand-write a GPU kernel on Apple Silicon", Rung 2 (row reduction,
 * then the reciprocal root of mean + eps) and Rung 4 (wide loads, a warp
 * reduction, then a small cross-warp combine).
 *   x [rows x d], g [d], n [rows x d], all of `dtype`.  n may equal x (in
 *   place); any other overlap is FFN_ERR_ALIAS.  rows >= 0, d >= 1.
 * ---------------------------------------------------------------------- */
ffn_status ffn_rmsnorm(const void *x, const void *g, void *n, int64_t rows, int64_t d,
                       float eps, ffn_dtype dtype, void *stream);

/* ------------------------------------------------------------------------
 * ffn_swiglu -- h[i] = silu(gate[i]) * up[i], silu in fp32.
 * "When to hand-write a GPU kernel on Apple Silicon", Rung 1 (one pass,
 * activation upcast to fp32).
 *   gate, up, h: `count` elements of `dtype`.  h may equal gate or up (in
 *   place); any other overlap is FFN_ERR_ALIAS.  count >= 0.
 * ---------------------------------------------------------------------- */
ffn_status ffn_swiglu(const void *gate, const void *up, void *h, int64_t count,
                      ffn_dtype dtype, void *stream);

/* ------------------------------------------------------------------------
 * ffn_block_workspace_bytes -- device scratch bytes ffn_block_forward needs
 * for these sizes, dtype and flags (the same path choice the forward call
 * makes).  Host-only; writes *bytes.  Shape errors as in ffn_block_forward.
 * The size may depend on the current CUDA device: on the tensor-core path
 * with few row blocks, the down projection splits its reduction so that its
 * tiles fill the device's multiprocessors, and its fp32 partial sums live
 * in the workspace.  Query with the device current that the forward call
 * will use (a smaller workspace there is FFN_ERR_WORKSPACE, never a write
 * past its end).
 * ---------------------------------------------------------------------- */
ffn_status ffn_block_workspace_bytes(int64_t rows, int64_t d, int64_t ffn, ffn_dtype dtype,
                                     uint32_t flags, size_t *bytes);

/* ------------------------------------------------------------------------
 * ffn_block_forward -- y = W_down (silu(W_gate n) * (W_up n)), n = RMSNorm(x).
 * "Unfusing a Kernel Made It 1.63x Faster", Finding 1 (gate and up
 * projections, then the activation, then the down projection) with the norm
 * of "When to hand-write a GPU kernel on Apple Silicon", Rung 2.
 *   x [rows x d], g [d], w_gate and w_up [ffn x d], w_down [d x ffn],
 *   y [rows x d]; all of `dtype`.  y must not overlap any input.
 *   Paths: FFN_F32 -> fp32 SIMT FFMA kernels (any rows).  FFN_F16/FFN_BF16 ->
 *   rows <= 16: weight-streaming decode kernels (every weight read once for
 *   up to 2 tiles of 8 token rows); otherwise tcgen05/TMEM GEMMs fed by TMA
 *   (with few row blocks: narrower gate/up tiles and a split-K down
 *   projection, so that the tiles fill the SMs).  FFN_PATH_GEMV forces the
 *   first for any rows <= 64 (up to 8 token tiles).  Rules: d, ffn >= 1; 16-bit dtypes need d % 8 == 0 and
 *   ffn % 8 == 0; fp32 needs d % 4 == 0 and ffn % 4 == 0.
 *   workspace: at least ffn_block_workspace_bytes(...) bytes, 16-byte aligned.
 *   Intermediates (n, h, split-K partials) round to `dtype` where they feed
 *   a tensor-core operand and stay fp32 otherwise; split-K partials are
 *   added in a fixed order (results are bitwise reproducible).
 * ---------------------------------------------------------------------- */
ffn_status ffn_block_forward(const void *x, const void *g, const void *w_gate, const void *w_up,
                             const void *w_down, void *y, int64_t rows, int64_t d, int64_t ffn,
                             float eps, ffn_dtype dtype, uint32_t flags, void *workspace,
                             size_t workspace_bytes, void *stream);

/* ------------------------------------------------------------------------
 * ffn_block_forward_chained -- ffn_block_forward that hands the RMSNorm
 * reduction from one block to the next.  "Megakernels on Mac: What Fusion
 * Saves and What It Costs", section "Dependencies and synchronization": after
 * a down projection produces a hidden vector, the next RMSNorm needs the sum
 * of squares of all its elements, and a worker that finishes one part of the
 * row must leave its partial sum until the last part is done.
 *   x_sumsq (optional, NULL = reduce the row as usual): [rows] fp32 device,
 *     sum over c of x[r,c]^2; the RMSNorm uses it instead of reducing x
 *     (e.g. the previous call's y_sumsq, with x that call's y).
 *   y_sumsq (optional): [rows] fp32 device, receives sum over c of y[r,c]^2
 *     of the y this call stores.  Where the down projection finishes a part
 *     of a row (a 64-column group on the decode kernels, an output tile on
 *     the tensor-core path), it adds the squares of the values it stored;
 *     the last part of a row to finish adds the parts in column order
 *     (fp32, the same bits every run).  Where that projection splits its
 *     reduction, the kernel that adds the splits sums each row; on the fp32
 *     path one pass over y sums each row.  With FFN_RESIDUAL, y is the next
 *     block's x and y_sumsq its x_sumsq.
 *   Both 16-byte aligned; y_sumsq overlaps no other argument or the
 *   workspace.  Everything else as ffn_block_forward (same workspace size).
 * ---------------------------------------------------------------------- */
ffn_status ffn_block_forward_chained(const void *x, const float *x_sumsq, const void *g, const void *w_gate,
                                     const void *w_up, const void *w_down, void *y, float *y_sumsq, int64_t rows,
                                     int64_t d, int64_t ffn, float eps, ffn_dtype dtype, uint32_t flags,
                                     void *workspace, size_t workspace_bytes, void *stream);

/* ------------------------------------------------------------------------
 * ffn_block_forward_host -- ffn_block_forward with x and y in HOST memory
 * (page-locked for the copies to overlap; pageable memory works, serialised).
 * The same block as ffn_block_forward ("Unfusing a Kernel Made It 1.63x
 * Faster", Finding 1); the host copies have no counterpart on the pages.
 *   x_host, y_host: [rows x d] of `dtype` in host memory, not overlapping.
 *   g, w_gate, w_up, w_down: device pointers as in ffn_block_forward.
 *   workspace: device scratch of ffn_block_host_workspace_bytes() bytes
 *   (two sets of x and y staging buffers, used by consecutive calls in
 *   turn so that a call's input copies overlap the compute of the call
 *   before it, plus the block's own scratch).
 * The rows are split into chunks (above 1024 rows: a last chunk of 1024
 * rows, the rows before it in chunks of at most 4096); the input copy of
 * every chunk is queued at once on a copy stream owned by the library, each
 * chunk's block runs on `stream` when its rows have landed, and its output
 * copy runs on a second library stream while the next chunk computes.
 * `stream` waits for the last output copy: once `stream` has passed the call,
 * y_host holds the result.  Concurrent calls on one device are serialised on
 * the host while they are queued; the workspace must not be shared by calls
 * that may run concurrently.  Errors as ffn_block_forward; FFN_ERR_ALIAS if
 * x_host and y_host overlap.
 * ---------------------------------------------------------------------- */
ffn_status ffn_block_host_workspace_bytes(int64_t rows, int64_t d, int64_t ffn, ffn_dtype dtype,
                                          uint32_t flags, size_t *bytes);
ffn_status ffn_block_forward_host(const void *x_host, const void *g, const void *w_gate,
                                  const void *w_up, const void *w_down, void *y_host, int64_t rows,
                                  int64_t d, int64_t ffn, float eps, ffn_dtype dtype, uint32_t flags,
                                  void *workspace, size_t workspace_bytes, void *stream);

/* ------------------------------------------------------------------------
 * Q4 weights ("Unfusing a Kernel Made It 1.63x Faster", section "The finding
 * that keeps us honest about microbenchmarks": 18-byte blocks of 32 weights,
 * 16 bytes of nibbles plus a half-precision scale, repacked so each block is
 * read once and coalesced).
 *   Canonical block: weight j (0..31) is q_j in [-8, 7] stored offset-binary
 *   u_j = q_j + 8; canonical byte i (0..15) holds u_i in the low nibble and
 *   u_(i+16) in the high nibble; the weight is w_j = (u_j - 8) * s.
 *   Device layout of qs: blocks go four at a time along the input dimension
 *   (128 weights, 64 bytes per group); byte 16*t + 4*b + e of a group is
 *   canonical byte 4*t + e of block b of the group (t, b, e in 0..3).  Each
 *   weight row holds ceil(in/128) groups (in/2 bytes when in % 128 == 0); the
 *   blocks of a last, partial group past in/32 are padding: zero bytes.
 *   scales: [out][4*ceil(in/128)] IEEE fp16 bit patterns, zero past in/32.
 *   Both arrays are device pointers (16-byte aligned) owned by the caller.
 * ---------------------------------------------------------------------- */
typedef struct {
    const uint8_t *qs;
    const uint16_t *scales;
} ffn_q4_weight;

ffn_status ffn_block_q4_workspace_bytes(int64_t rows, int64_t d, int64_t ffn, size_t *bytes);

/* ------------------------------------------------------------------------
 * ffn_block_forward_q4 -- the block with Q4 weights, dequantised in registers.
 * "Megakernels on Mac: What Fusion Saves and What It Costs", section "Threadgroup staging" (stream Q4 weights
 * to registers; staging through shared memory lost).
 *   x [rows x d] bf16, g [d] bf16, y [rows x d] bf16; w_gate/w_up are Q4
 *   [ffn x d], w_down is Q4 [d x ffn].  Needs d % 32 == 0, ffn % 32 == 0
 *   (multiples of 256 stream through the TMA kernels, the rest through the
 *   register kernels).  Rows are processed in groups of up to 16; each group
 *   streams the weights once.  The codes (u - 8) are exact in fp16, so the
 *   MMAs run on fp16: activations enter as one fp16 rounding (h stored times
 *   2^-8).  On the TMA kernels the nibbles enter the MMAs as 1024 + u (low)
 *   and 1024 + 16u (high nibble, against activations stored divided by 16),
 *   each block's offset removed in fp32 (to ~2^-22 of it) after the
 *   products; h is stored times 2^-4 in the low-nibble positions of a block
 *   and 2^-8 in the high ones, so |h| must stay below 2^20 there.  flags:
 *   FFN_AUTO, FFN_RESIDUAL, FFN_DECODE_ONE_KERNEL.
 * ---------------------------------------------------------------------- */
ffn_status ffn_block_forward_q4(const void *x, const void *g, ffn_q4_weight w_gate,
                                ffn_q4_weight w_up, ffn_q4_weight w_down, void *y, int64_t rows,
                                int64_t d, int64_t ffn, float eps, uint32_t flags, void *workspace,
                                size_t workspace_bytes, void *stream);

/* ------------------------------------------------------------------------
 * e4m3 weights with one float scale per output row.  The pages store 8-bit
 * quantised data only for the KV cache ("Unfusing a Kernel Made It 1.63x
 * Faster", section "Finding 2: a quantized KV cache buys nothing while
 * you're occupancy-bound": halving the bytes pays once the kernel is bound
 * by memory); these are the projection weights at one byte each, half the
 * stream of bf16, which is the whole cost of a decode step.
 *   codes: [out x in] row-major bytes, each an 8-bit float e4m3 in the "fn"
 *   encoding (sign, 4 exponent bits with bias 7, 3 fraction bits; exponent 0
 *   is subnormal, f * 2^-9; 0x7F and 0xFF are NaN; no infinities; largest
 *   value 448).  scales: [out] float32.  The weight is
 *   w[o][i] = e4m3(codes[o][i]) * scales[o].  Both arrays are device
 *   pointers (16-byte aligned) owned by the caller.
 * ---------------------------------------------------------------------- */
typedef struct {
    const uint8_t *codes;
    const float *scales;
} ffn_fp8_weight;

ffn_status ffn_block_fp8_workspace_bytes(int64_t rows, int64_t d, int64_t ffn, size_t *bytes);

/* ------------------------------------------------------------------------
 * ffn_block_forward_fp8 -- the block with e4m3 weights ("How Megakernels
 * Work", section "Projection shape changes the achieved rate": the decode
 * projections are weight streams).
 *   x [rows x d] bf16, g [d] bf16, y [rows x d] bf16; w_gate/w_up are e4m3
 *   [ffn x d], w_down is e4m3 [d x ffn].  Needs d % 256 == 0 and
 *   ffn % 256 == 0 (FFN_ERR_SHAPE otherwise).  Rows are processed in groups
 *   of up to 16; each group streams the weights once.  Every code is exact in
 *   fp16, so the MMAs multiply the codes themselves on fp16 operands
 *   (activations as one fp16 rounding, h stored times 2^-8) and each output
 *   is multiplied by its row scale once, in fp32.  flags: FFN_AUTO or
 *   FFN_RESIDUAL.  Errors: FFN_ERR_NULL (a pointer missing),
 *   FFN_ERR_FLAGS, FFN_ERR_SHAPE, FFN_ERR_WORKSPACE (workspace smaller than
 *   ffn_block_fp8_workspace_bytes), FFN_ERR_ALIGN, FFN_ERR_ALIAS (y or the
 *   workspace overlaps an input, or each other), FFN_ERR_CUDA (a launch
 *   failed).  Nothing is launched on an error found on the host.
 * ---------------------------------------------------------------------- */
ffn_status ffn_block_forward_fp8(const void *x, const void *g, ffn_fp8_weight w_gate,
                                 ffn_fp8_weight w_up, ffn_fp8_weight w_down, void *y, int64_t rows,
                                 int64_t d, int64_t ffn, float eps, uint32_t flags, void *workspace,
                                 size_t workspace_bytes, void *stream);

/* ------------------------------------------------------------------------
 * ffn_block_forward_decode_static -- the decode block (same kernels and
 * results as ffn_block_forward on its weight-streaming path) for callers that
 * cannot hand the library a workspace: runtimes that plan all device memory
 * up front and allow no allocation while serving, plugins that receive only
 * their input and output buffers, and decode loops that must not call
 * cudaMalloc (it can synchronise the device).  The pages describe no such
 * call; it has no counterpart there.
 *   Scratch: one 12 MiB array in device memory owned by the library, present
 *   on every GPU that loads the library until the process exits.  No
 *   allocation, no free, no allocating library call is made.  Limits (checked,
 *   FFN_ERR_SHAPE beyond them): rows <= 16, d <= 8192, ffn <= 32768, plus
 *   d % 8 == 0 and ffn % 8 == 0; dtype FFN_F16 or FFN_BF16.
 *   Every call looks up the array's device address in the current device's
 *   context (a host-side query that allocates nothing), so the address stays
 *   right after cudaDeviceReset; the first call in a context also loads the
 *   library's device code there -- make that first call before any stream
 *   capture.
 *   Every call reuses the same array: calls that may run at the same time on
 *   the GPU (other streams, other host threads) race and must be serialised
 *   by the caller.  Other arguments, layouts and errors as ffn_block_forward.
 * ---------------------------------------------------------------------- */
ffn_status ffn_block_forward_decode_static(const void *x, const void *g, const void *w_gate,
                                           const void *w_up, const void *w_down, void *y,
                                           int64_t rows, int64_t d, int64_t ffn, float eps,
                                           ffn_dtype dtype, void *stream);

/* ------------------------------------------------------------------------
 * ffn_prepare_weights -- one-time re-encoding of a weight matrix for
 * FFN_PREPARED_WEIGHTS: dst[i] = fp16(src[i] * 2^8), round to nearest even.
 * No page describes this step; it exists because the tensor-core instruction
 * needs both operands in one type and fp16 keeps 11 significant bits of the
 * activations where bf16 keeps 8.  For bf16 src every value with
 * 2^-25 <= |w| < 256 is represented exactly; smaller ones round by at most
 * 2^-33 absolute; |w| >= 255.9375 becomes infinite and FFN_ERR_RANGE is
 * recorded in the device status word (see ffn_device_status).
 *   src: `count` device values of src_dtype (FFN_BF16 or FFN_F16);
 *   dst: `count` device fp16 values (may equal src, then in place).
 * ---------------------------------------------------------------------- */
ffn_status ffn_prepare_weights(const void *src, void *dst, int64_t count, ffn_dtype src_dtype,
                               void *stream);

/* ------------------------------------------------------------------------
 * Q8_0 weights: blocks of 32 signed 8-bit codes along the input dimension,
 * one IEEE fp16 scale per block ("Unfusing a Kernel Made It 1.63x Faster",
 * section "Finding 2: a quantized KV cache buys nothing while you're
 * occupancy-bound" names the format, there for the KV cache; here the
 * projection weights, at 34 bytes per 32 weights).
 *   codes: [out x in] int8, row-major (natural order); scales: [out x in/32]
 *   fp16 bit patterns; w[o][i] = codes[o][i] * scales[o][i / 32].  Both are
 *   device pointers (16-byte aligned) owned by the caller.
 * ---------------------------------------------------------------------- */
typedef struct {
    const int8_t *codes;
    const uint16_t *scales;
} ffn_q8_weight;

ffn_status ffn_block_q8_workspace_bytes(int64_t rows, int64_t d, int64_t ffn, size_t *bytes);

/* ------------------------------------------------------------------------
 * ffn_block_forward_q8 -- the block with Q8_0 weights (decode: the weights
 * are streamed; "Megakernels on Mac: What Fusion Saves and What It Costs", section "Projection shape changes
 * the achieved rate").
 *   x [rows x d] bf16, g [d] bf16, y [rows x d] bf16; w_gate/w_up are Q8_0
 *   [ffn x d], w_down is Q8_0 [d x ffn].  Needs d % 256 == 0 and
 *   ffn % 256 == 0 (FFN_ERR_SHAPE otherwise).  Rows are processed in groups
 *   of up to 16; each group streams the weights once.  The codes are exact in
 *   fp16; each 32-weight block's MMA result is multiplied by its scale in
 *   fp32; activations enter as one fp16 rounding (h stored times 2^-8).
 *   flags: FFN_AUTO or FFN_RESIDUAL.  Errors as ffn_block_forward_fp8.
 * ---------------------------------------------------------------------- */
ffn_status ffn_block_forward_q8(const void *x, const void *g, ffn_q8_weight w_gate, ffn_q8_weight w_up,
                                ffn_q8_weight w_down, void *y, int64_t rows, int64_t d, int64_t ffn, float eps,
                                uint32_t flags, void *workspace, size_t workspace_bytes, void *stream);

/* ------------------------------------------------------------------------
 * ffn_prepare_weights_fp8 / ffn_prepare_weights_q4 / ffn_prepare_weights_q8
 * -- the same prepared form
 * (fp16 values of w * 2^8, [out x in] row-major) from quantised weights, for
 * many-row batches: ffn_block_forward_fp8 and ffn_block_forward_q4 stream the
 * whole quantised weight set once per group of 16 rows, the fast path for a
 * prefill batch is to prepare once and call ffn_block_forward with
 * FFN_PREPARED_WEIGHTS (tensor-core GEMMs).  No page describes the step.
 *   fp8: w = e4m3(codes[o][i]) * scales[o]; in % 16 == 0.  The product times
 *   2^8 is rounded to fp16 once (round to nearest even), i.e. to 11
 *   significant bits of the exact w.
 *   Q4: w = (u - 8) * s in the device layout above; in % 32 == 0.  Exact
 *   before the one rounding to fp16 as well.
 *   dst: out * in device fp16 values, 16-byte aligned, overlapping neither
 *   input (FFN_ERR_ALIAS).  Values whose |w| * 2^8 exceeds fp16's range
 *   become infinite and record FFN_ERR_RANGE in the device status word.
 *   FFN_ERR_NULL, FFN_ERR_SHAPE, FFN_ERR_ALIGN are found before any launch;
 *   out == 0 or in == 0 launches nothing.
 * ---------------------------------------------------------------------- */
ffn_status ffn_prepare_weights_fp8(ffn_fp8_weight w, void *dst, int64_t out, int64_t in, void *stream);
ffn_status ffn_prepare_weights_q4(ffn_q4_weight w, void *dst, int64_t out, int64_t in, void *stream);
/* Q8_0: w = q * s; in % 32 == 0; exact before the one rounding to fp16. */
ffn_status ffn_prepare_weights_q8(ffn_q8_weight w, void *dst, int64_t out, int64_t in, void *stream);

/* Host helper (not on the hot path): pack int8 q [out x in] (values -8..7) and
 * fp16 scale bits [out x in/32] into the device layout above.  Host pointers;
 * qs_out holds out * 64 * ceil(in/128) bytes, scales_out out * 4 *
 * ceil(in/128) entries (the padding written as zeros).  in % 32 == 0. */
ffn_status ffn_q4_pack_host(const int8_t *q, const uint16_t *scales, int64_t out, int64_t in,
                            uint8_t *qs_out, uint16_t *scales_out);

/* Text for a status code (static storage). */
const char *ffn_status_string(ffn_status status);

/* Synchronises the current device, then returns and clears the device status
 * word: FFN_OK; FFN_ERR_TIMEOUT if a kernel abandoned a bounded wait since
 * the last call; else FFN_ERR_RANGE if ffn_prepare_weights met a weight out
 * of range; FFN_ERR_CUDA if the synchronisation itself failed. */
ffn_status ffn_device_status(void);

/* Failure-detection self test (no counterpart on the pages; the pages ask
 * for explicit failure behaviour -- "Megakernels on Mac: What Fusion Saves and What It Costs", section
 * "Dependencies and synchronization").  Launches on `stream` one CTA in which
 * one role waits on an mbarrier phase that nothing completes, with the same
 * bounded wait every streaming kernel of this library uses, and gives up after
 * limit_ns nanoseconds (clamped to [1 us, 1 s]); a second role, waiting with a
 * 1000x longer limit, is released by the first one's abort flag.  The kernel
 * records FFN_ERR_TIMEOUT in the device status word and returns normally, so
 * the next ffn_device_status() returns FFN_ERR_TIMEOUT and the device stays
 * usable.  Returns FFN_OK when launched, FFN_ERR_CUDA if the launch failed. */
ffn_status ffn_selftest_bounded_wait(uint64_t limit_ns, void *stream);

/* Number of kernels this library has launched since it was loaded (host count). */
uint64_t ffn_launch_count(void);

/* ------------------------------------------------------------------------
 * Measurement hooks.  With timing on, every launch is bracketed by CUDA events
 * recorded on its own stream.  ffn_timing_collect() synchronises the pending
 * events and adds their durations to per-kernel totals; ffn_timing_read()
 * returns the totals for kernel kind `kind` (0 <= kind < ffn_kernel_kinds()).
 * ---------------------------------------------------------------------- */
ffn_status ffn_timing_enable(int on);
ffn_status ffn_timing_collect(void);
ffn_status ffn_timing_reset(void);
int ffn_kernel_kinds(void);
const char *ffn_kernel_name(int kind);
ffn_status ffn_timing_read(int kind, uint64_t *launches, double *total_ms);

#ifdef __cplusplus
}
#endif

#endif /* FFN_GB300_H */
