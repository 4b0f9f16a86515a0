/*
 * mxq.h -- C ABI of libmxq, GB300 (sm_103a) block-scaled quantization.
 *
 * The library turns a bf16 matrix into OCP-MX MXFP8 (E4M3 codes, one E8M0
 * scale per 32-element block) rowwise and colwise from a single HBM read,
 * optionally fused with a dbias column sum, a tanh-GELU or a SwiGLU gate, and
 * into NVFP4 (E2M1 codes, one E4M3 scale per 16 elements, one fp32 tensor
 * scale) rowwise and transposed.
 *
 * Kernel families this covers (TransformerEngine PR #3291 "Fix pointer
 * arithmatic to generate correct LDS/STS instructions", results tables
 * "MXFP8 generic quantize kernel", "MXFP8 specialized cast-only kernel
 * (bidimensional)", "MXFP8 gated (swiglu / geglu) kernel" and "NVFP4 2D
 * quantize-transpose kernel"; the colwise-only cast is the "dim1" cast of
 * torchao PR #12 "Multiply with inverse scale in loop instead of dividing",
 * section "Performance").
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  * All pointers are DEVICE pointers unless stated otherwise; the caller
 *    owns every buffer.  The library never allocates, frees or synchronises:
 *    all work is enqueued on `stream` (NULL = the legacy default stream), and
 *    every buffer must stay valid until the stream has passed this call.
 *  * Matrices are row-major.  `x` is bf16 (raw 16-bit patterns) with a row
 *    stride of `ldx` elements; outputs are dense (row stride = width).
 *  * Host-checkable problems return a status synchronously and enqueue
 *    nothing.  A launch failure returns MXQ_ECUDA.
 *  * `dev_err` (optional, device, 4 bytes): every wait inside the kernels is
 *    bounded; if one runs out, the kernel ORs MXQ_DEVERR_TIMEOUT into
 *    *dev_err, waits (bounded) for its own copies in flight and exits
 *    without writing the remaining tiles.  The library never clears
 *    *dev_err; the caller zeroes it and reads it back after the stream.
 *    When *dev_err is nonzero after a call, every output of that call
 *    (codes, scales, dbias, the global scale) is undefined.
 *  * Alignment: `x`, every output and the workspace 16-byte aligned, `ldx`
 *    a multiple of 8.  Violations return MXQ_EALIGN.
 *  * The device must be compute capability 10.3 (GB300): else MXQ_EARCH.
 *  * NaN or infinite inputs are outside the contract.
 */
#ifndef MXQ_H
#define MXQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define MXQ_API __attribute__((visibility("default")))
#else
#define MXQ_API
#endif

/* Same object as cudaStream_t. */
typedef struct CUstream_st* mxq_stream_t;

typedef enum {
    MXQ_OK = 0,
    MXQ_EINVAL = 1,      /* NULL pointer, bad flag combination            */
    MXQ_ESHAPE = 2,      /* negative size or size not a block multiple    */
    MXQ_EALIGN = 3,      /* pointer or stride misaligned                  */
    MXQ_EARCH = 4,       /* current device is not sm_103                  */
    MXQ_EWORKSPACE = 5,  /* workspace missing or too small                */
    MXQ_ECUDA = 6        /* CUDA runtime error while launching            */
} mxq_status;

/* flags */
enum {
    MXQ_ROWWISE = 1,        /* 1x32 (MX) / 1x16 (NVFP4) blocks along K     */
    MXQ_COLWISE = 2,        /* 32x1 (MX) / 16x1 (NVFP4) blocks along M,    */
                            /* stored transposed: [K][M]                   */
    MXQ_DBIAS = 4,          /* fp32 column sums of x (mx_quantize_rowcol)  */
    MXQ_ACT_GELU_TANH = 8,  /* gelu_tanh: of x (mx_quantize_rowcol), of the */
                            /* gate (mx_quantize_gated: GeGLU), its         */
                            /* derivative (mx_quantize_dact / _dgated)     */
    MXQ_NVFP4_2D = 16,      /* 16x16 blocks (nvfp4_quantize_transpose)     */
    MXQ_ACT_SILU = 32,      /* silu: SwiGLU gate (the default of the gated */
                            /* calls), its derivative (mx_quantize_dact)   */
    MXQ_SCALE_RCEIL = 64,   /* MXFP8 calls: ceil-style E8M0 rule, below    */
    MXQ_SCALE_SWIZZLED = 128 /* MXFP8 calls: scales in 128x4 tiles, below   */
};

/* bits of *dev_err */
enum { MXQ_DEVERR_TIMEOUT = 1 };

/* operation ids for mxq_workspace_bytes */
enum { MXQ_OP_ROWCOL = 0, MXQ_OP_NVFP4 = 1, MXQ_OP_DACT = 2, MXQ_OP_ROWCOL_HOST = 3 };

/* Human-readable name of a status code (static string, never NULL). */
MXQ_API const char* mxq_status_string(int status);

/* Workspace bytes `op` needs for an M x K input with `flags` on the current
 * device (0 when none is needed).  MXQ_OP_ROWCOL needs one only with
 * MXQ_DBIAS; MXQ_OP_NVFP4 needs 4 bytes when no amax_in is given. */
MXQ_API size_t mxq_workspace_bytes(int op, int64_t M, int64_t K, uint32_t flags);

/*
 * mx_quantize_rowcol -- bf16 -> MXFP8 rowwise and/or colwise, one HBM read.
 *
 * Operation (per 32-value block B of y, y = x, or y = gelu_tanh(x) in fp32
 * with MXQ_ACT_GELU_TANH, gelu_tanh(x) = 0.5 x (1 + tanh(sqrt(2/pi)
 * (x + 0.044715 x^3)))):  a = max|y| over B;  e = floor(log2 a) - 8 clamped
 * to [-127, 127] (a = 0 -> scale code 0);  scale code = e + 127 (E8M0);
 * codes = E4M3(y * 2^-e), round-to-nearest-even, saturating to +-448.
 * With MXQ_SCALE_RCEIL (any MXFP8 call) e = ceil(log2(a / 448)) instead,
 * clamped the same way: the smallest power of two for which no element
 * exceeds 448, so nothing saturates.
 * With MXQ_SCALE_SWIZZLED (any MXFP8 call) each scale matrix [R][C] (R = M,
 * C = K/32 rowwise; R = K, C = M/32 colwise) is written in the tiled layout
 * block-scaled GEMMs read instead of row-major: padded to R' =
 * ceil(R/128)*128 rows and C' = ceil(C/4)*4 columns (padding bytes 0), cut
 * into 128x4 tiles stored one after another in row-major tile order (tile
 * (i, j) at byte (i * C'/4 + j) * 512); inside a tile, entry (r, c) is at
 * byte (r % 32) * 16 + (r / 32) * 4 + c.  The buffers must hold R' * C'
 * bytes.  (mx_quantize_dgated additionally needs N % 128 == 0.)  The
 * multiply by the exact power of two 2^-e replaces a per-element division
 * (torchao PR #12, rationale section).  Rowwise blocks are 1x32 along K,
 * colwise blocks 32x1 along M (TE PR #3291 tables, dir "row"/"col"/"both").
 * MXQ_DBIAS adds dbias[k] = sum_m x[m][k] in fp32 (TE PR #3291 fusion
 * "dbias"; not combinable with MXQ_ACT_GELU_TANH).
 *
 *   x       [M][ldx] bf16, M % 32 == 0, K % 32 == 0, ldx >= K.
 *   flags   MXQ_ROWWISE | MXQ_COLWISE (at least one), optional MXQ_DBIAS or
 *           MXQ_ACT_GELU_TANH.
 *   q_row   [M][K] E4M3 codes, s_row [M][K/32] E8M0 (needed with ROWWISE,
 *           else ignored).
 *   q_col   [K][M] E4M3 codes (row k holds column k of the blocks),
 *           s_col [K][M/32] E8M0 (needed with COLWISE, else ignored).
 *   dbias   [K] fp32 (needed with MXQ_DBIAS).
 *   workspace / workspace_bytes: device scratch of at least
 *           mxq_workspace_bytes(MXQ_OP_ROWCOL, M, K, flags) bytes, 16-byte
 *           aligned (dbias partial sums); may be NULL when that is 0.
 *   M == 0 or K == 0 is a valid empty call (dbias is zero-filled).
 */
MXQ_API mxq_status mx_quantize_rowcol(const void* x, int64_t M, int64_t K, int64_t ldx, uint32_t flags,
                              uint8_t* q_row, uint8_t* s_row, uint8_t* q_col, uint8_t* s_col,
                              float* dbias, void* workspace, size_t workspace_bytes,
                              uint32_t* dev_err, mxq_stream_t stream);

/*
 * mx_quantize_rowcol_dbias_noalloc -- mx_quantize_rowcol with MXQ_DBIAS for
 * callers that cannot allocate device memory.  The pages have no
 * counterpart to this entry point.
 *
 * Some callers cannot provide the dbias workspace: code inside a framework
 * that owns all device memory through its own pool (an extra cudaMalloc
 * would bypass the pool and synchronise the device), loops that forbid
 * allocation after start-up, and plugin hosts that pass this library only
 * the tensors it reads and writes.  This entry point takes the same
 * arguments as mx_quantize_rowcol minus the workspace, always computes
 * dbias (MXQ_DBIAS is implied; MXQ_ACT_GELU_TANH is refused with
 * MXQ_EINVAL), and keeps its scratch in a device array the library owns:
 * 8 MiB, held on every GPU that loads the library until the process exits.
 *   - Limit: shapes needing more than 8 MiB of band sums
 *     (mxq_workspace_bytes(MXQ_OP_ROWCOL, M, K, MXQ_DBIAS) > 8 MiB, e.g.
 *     more than 16384 x 16384) return MXQ_EWORKSPACE; nothing is enqueued.
 *   - Every call looks up the array's device address in the current
 *     context; the first call with a device current also loads the
 *     library's device code there, so make that first call before any
 *     stream capture begins.
 *   - All calls share the array.  Nothing in it needs clearing (every value
 *     read is written earlier in the same call), but calls that overlap on
 *     the GPU race on it: order them, e.g. on one stream.  Calls queued one
 *     after another on one stream do not overlap.
 *   - As for every entry point, the outputs are undefined when the call
 *     reports a timeout through *dev_err.
 *   - It never calls cudaMalloc, cudaFree or any allocating routine.
 */
MXQ_API mxq_status mx_quantize_rowcol_dbias_noalloc(const void* x, int64_t M, int64_t K,
                                                    int64_t ldx, uint32_t flags, uint8_t* q_row,
                                                    uint8_t* s_row, uint8_t* q_col,
                                                    uint8_t* s_col, float* dbias,
                                                    uint32_t* dev_err, mxq_stream_t stream);

/*
 * mx_quantize_rowcol_host -- mx_quantize_rowcol on a matrix in host memory.
 * The pages have no counterpart: it is the path for callers whose data is
 * on the host, and what the benchmark's end-to-end figure measures.
 *
 * The same cast (plain, no dbias or activation) of x in row panels of up to
 * 2048 rows: each panel is copied to the device, quantized, and its outputs
 * copied back (colwise codes as 2-D copies into the [K][M] host layout;
 * row-major colwise scales gathered on the device for the whole matrix and
 * copied back once, after the last panel); two sets of device buffers
 * alternate and the copies run on two library-owned streams, so copies in,
 * casts and copies out of consecutive panels overlap.
 *
 *   x, q_row, s_row, q_col, s_col  host memory with the layouts of
 *           mx_quantize_rowcol; page-locked memory lets the copies run
 *           asynchronously (pageable memory works, without overlap).
 *   flags   MXQ_ROWWISE and/or MXQ_COLWISE.
 *   workspace  device memory, 256-byte aligned, at least
 *           mxq_workspace_bytes(MXQ_OP_ROWCOL_HOST, M, K, flags) bytes.
 *   stream  the call starts after the work already on `stream`, and work
 *           enqueued on `stream` afterwards starts after the outputs are on
 *           the host (synchronise the stream before reading them).
 * Calls from several host threads are serialised inside the library (they
 * share the per-device streams).
 */
MXQ_API mxq_status mx_quantize_rowcol_host(const void* x, int64_t M, int64_t K, int64_t ldx,
                                           uint32_t flags, uint8_t* q_row, uint8_t* s_row,
                                           uint8_t* q_col, uint8_t* s_col, void* workspace,
                                           size_t workspace_bytes, mxq_stream_t stream);

/*
 * mx_quantize_gated -- SwiGLU or GeGLU gate fused with MXFP8 quantization.
 *
 * Operation: y[m][n] = act(x[m][n]) * x[m][N + n] for n < N, computed in
 * fp32 (no intermediate bf16 rounding), then quantized exactly as
 * mx_quantize_rowcol quantizes y (TE PR #3291 table "MXFP8 gated (swiglu /
 * geglu) kernel", fusions "swiglu" and "geglu").  act is silu(g) =
 * g / (1 + e^-g) (SwiGLU; the default, or MXQ_ACT_SILU) or gelu_tanh
 * (GeGLU, MXQ_ACT_GELU_TANH).
 *
 *   x       [M][ldx] bf16 holding [gate | up], each N wide; ldx >= 2N.
 *   flags   MXQ_ROWWISE and/or MXQ_COLWISE, at most one activation flag.
 *   M % 32 == 0, N % 32 == 0.
 *   q_row [M][N], s_row [M][N/32], q_col [N][M], s_col [N][M/32] as above.
 */
MXQ_API mxq_status mx_quantize_gated(const void* x, int64_t M, int64_t N, int64_t ldx, uint32_t flags,
                             uint8_t* q_row, uint8_t* s_row, uint8_t* q_col, uint8_t* s_col,
                             uint32_t* dev_err, mxq_stream_t stream);

/*
 * mx_quantize_dact -- backward activation fused with MXFP8 quantization.
 *
 * Operation (TE PR #3291 table "MXFP8 generic quantize kernel", fusions
 * "dgelu", "dsilu" and "dbias_dgelu"): y[m][k] = grad[m][k] * act'(x[m][k])
 * in fp32, with act' the derivative of gelu_tanh (MXQ_ACT_GELU_TANH) or of
 * silu (MXQ_ACT_SILU) -- exactly one of the two; y is quantized exactly as
 * mx_quantize_rowcol quantizes its input, and MXQ_DBIAS writes
 * dbias[k] = sum_m y[m][k].
 *
 *   grad    [M][ldg] bf16, the incoming gradient; x [M][ldx] bf16, the
 *           activation's input; M % 32 == 0, K % 32 == 0, ldg, ldx >= K,
 *           multiples of 8, both 16-byte aligned.
 *   outputs, dbias, workspace (mxq_workspace_bytes(MXQ_OP_DACT, M, K,
 *           flags) bytes with MXQ_DBIAS), dev_err, stream: as for
 *           mx_quantize_rowcol.
 */
MXQ_API mxq_status mx_quantize_dact(const void* grad, const void* x, int64_t M, int64_t K,
                                    int64_t ldg, int64_t ldx, uint32_t flags, uint8_t* q_row,
                                    uint8_t* s_row, uint8_t* q_col, uint8_t* s_col, float* dbias,
                                    void* workspace, size_t workspace_bytes, uint32_t* dev_err,
                                    mxq_stream_t stream);

/*
 * mx_quantize_dgated -- backward of the gated activation fused with MXFP8
 * quantization (TE PR #3291 table "MXFP8 gated (swiglu / geglu) kernel",
 * fusion "dswiglu", and its GeGLU counterpart).
 *
 * Operation: with gate = x[m][n], up = x[m][N + n] and g = grad[m][n],
 * y[m][n] = g * up * act'(gate) (the gradient of the gate) and
 * y[m][N + n] = g * act(gate) (the gradient of up), n < N, in fp32; act is
 * silu (the default, or MXQ_ACT_SILU) or gelu_tanh (MXQ_ACT_GELU_TANH).  y
 * ([M][2N]) is quantized exactly as mx_quantize_rowcol quantizes its input.
 *
 *   grad    [M][ldg] bf16, ldg >= N; x [M][ldx] bf16 holding [gate | up],
 *           ldx >= 2N; M % 32 == 0, N % 32 == 0.
 *   q_row [M][2N], s_row [M][2N/32], q_col [2N][M], s_col [2N][M/32].
 */
MXQ_API mxq_status mx_quantize_dgated(const void* grad, const void* x, int64_t M, int64_t N,
                                      int64_t ldg, int64_t ldx, uint32_t flags, uint8_t* q_row,
                                      uint8_t* s_row, uint8_t* q_col, uint8_t* s_col,
                                      uint32_t* dev_err, mxq_stream_t stream);

/*
 * bf16_amax -- largest |x| of a bf16 matrix, written as fp32 to *amax_out
 * (device).  The exact maximum, so the result does not depend on the order
 * of the reduction.  Needed for the NVFP4 tensor scale.
 *   x [M][ldx], K % 8 == 0.  M == 0 or K == 0 writes 0.
 */
MXQ_API mxq_status bf16_amax(const void* x, int64_t M, int64_t K, int64_t ldx, float* amax_out,
                     mxq_stream_t stream);

/*
 * nvfp4_quantize_transpose -- bf16 -> NVFP4, rowwise and transposed.
 *
 * Operation (TE PR #3291, "NVFP4 quantize-transpose" family: the 1D kernel
 * named in "Patched but not measurable" and the results table "NVFP4 2D
 * quantize-transpose kernel"; every step one fp32 IEEE operation in this
 * order):
 *   A = tensor amax (from amax_in, else from an internal bf16_amax pass);
 *   G = A / 2688 (2688 = 448 * 6), written to *global_scale;
 *   per block of 16 values (1x16 along K rowwise; 16x1 along M for the
 *   transposed output): b = block amax; s = E4M3((b / 6) / G) (RNE,
 *   saturating); d = value(s) * G; inv = 1 / d (0 when s == 0 or d == 0,
 *   the largest finite float if 1 / d overflows);
 *   codes = E2M1(x * inv), round-to-nearest-even, saturating to +-6,
 *   packed two per byte, element 2i in the low nibble.  A == 0 gives
 *   G = 0 and all-zero scales.
 *   With MXQ_NVFP4_2D the block is 16x16 (rows 16i.., columns 16j..): b is
 *   its amax and every element of it is quantized with its one scale in
 *   both outputs; the scale arrays keep the shapes below, each block's
 *   scale repeated in its 16 rows (s_row) or 16 columns (s_t), so q_t is
 *   exactly the transpose of q_row.
 *
 *   x       [M][ldx] bf16, M % 32 == 0, K % 32 == 0 (so that every packed
 *           code row is a multiple of 16 bytes, as the bulk-copy engine
 *           that writes them needs).
 *   flags   MXQ_ROWWISE and/or MXQ_COLWISE (= the transposed output),
 *           optional MXQ_NVFP4_2D.
 *   amax_in device fp32 tensor amax, or NULL to compute it here (then the
 *           workspace must hold 4 bytes).
 *   global_scale  device fp32, receives G (required).
 *   q_row [M][K/2], s_row [M][K/16] (E4M3); q_t [K][M/2], s_t [K][M/16].
 */
MXQ_API mxq_status nvfp4_quantize_transpose(const void* x, int64_t M, int64_t K, int64_t ldx,
                                    uint32_t flags, const float* amax_in, float* global_scale,
                                    uint8_t* q_row, uint8_t* s_row, uint8_t* q_t, uint8_t* s_t,
                                    void* workspace, size_t workspace_bytes, uint32_t* dev_err,
                                    mxq_stream_t stream);

/*
 * mxq_selftest_bounded_wait -- launches one warp that waits on a barrier
 * nothing will ever complete, through the same bounded-wait routine the
 * quantization kernels use, with a limit of `timeout_ns` nanoseconds
 * (1e3..5e9).  The kernel ORs MXQ_DEVERR_TIMEOUT into *dev_err (required)
 * and returns, leaving the context usable.  Lets a test check the timeout
 * path without faulting or hanging a GPU.
 */
MXQ_API mxq_status mxq_selftest_bounded_wait(uint64_t timeout_ns, uint32_t* dev_err, mxq_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* MXQ_H */
