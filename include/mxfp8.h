/*
 * mxfp8.h -- C ABI of the GB300 (sm_103a) MXFP8 block-scaled quantize library.
 *
 * The operation is the MXFP8 cast of "[Common] Experimental CuTeDSL MXFP8
 * backends in C++ via TVM-FFI" (TransformerEngine PR #3137): a BF16 matrix
 * becomes FP8 data plus one E8M0 power-of-two scale per 32-element block.
 * The quantization-config review on that page (`to_key()`) names the options
 * this ABI exposes: fp8_dtype, rowwise, colwise, with_dbias and with_noop;
 * the "non-32-divisible shapes" review fixes the 32-element block.  Shapes
 * that are not multiples of 32 are accepted here: M may be any size and N
 * any multiple of 8 (a 16-byte BF16 row pitch, which the TMA loads need); a
 * row's (column's) last block then holds the remaining N % 32 (M % 32)
 * elements and takes its amax over those only.
 *
 * Arithmetic, per 32-element block with amax = max |x| over the block:
 *     e = clamp(ceil(log2(amax / Fmax)) + 127, 0, 254)   (amax == 0 -> e = 127)
 *     q = round-to-nearest-even, saturate-finite (x * 2^(127 - e))
 * with Fmax = 448 (E4M3) or 57344 (E5M2).  Results are bit-exact with that
 * definition for every finite BF16 input.
 *
 * Layouts (all row-major, all buffers device memory owned by the caller):
 *     x          bf16  [M, N]
 *     out_row    uint8 [M, N]            FP8 codes, block = 1x32 along a row
 *     scale_row  uint8 [M, ceil(N/32)]   E8M0 of block (i, j/32)
 *     out_col    uint8 [M, N]            FP8 codes, block = 32x1 down a column;
 *                                        element (i, j) uses scale_col[i/32, j]
 *     scale_col  uint8 [ceil(M/32), N]   E8M0 of block (i/32, j)
 *     dbias      fp32  [N]        column sums of x (unquantized)
 *
 * Conventions shared by every call:
 *   - The library allocates no device memory for a call: every buffer is the
 *     caller's.  It keeps per-device cached kernel attributes, a launch
 *     counter, a fault word, the internal streams and events of
 *     mxfp8_quantize_host (created on its first call on a device) and the
 *     static 8 MiB scratch array of mxfp8_quantize_dbias_noalloc.
 *   - All validation happens on the host before any launch; every rejection
 *     is a status code, nothing throws or aborts across this boundary.
 *   - Work is stream-ordered on `stream` (a cudaStream_t; NULL = the legacy
 *     default stream).  No call synchronizes the host or reads device memory
 *     from the host, except mxfp8_device_fault_word().  The quantize kernels
 *     and the dbias reduces are launched with programmatic stream
 *     serialization: each may start while the kernel before it drains, but
 *     waits on the device for that kernel to finish before it touches global
 *     memory, so results are as for plain stream order.  (Captured in a CUDA
 *     graph, consecutive calls are joined by programmatic edges.)
 *   - The device is the calling thread's current device; x must live on it.
 *   - noop: optional device fp32 scalar.  When *noop == 1.0f every kernel of
 *     the call returns without writing anything (the "Perform noop tensor
 *     check on device" change on the PR #3137 page), dbias included.
 */
#ifndef MXFP8_GB300_H
#define MXFP8_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* FP8 element format (the `fp8_dtype` field of the PR #3137 config key). */
typedef enum {
    MXFP8_E4M3 = 0, /* 1 sign, 4 exponent (bias 7), 3 mantissa; max 448   */
    MXFP8_E5M2 = 1  /* 1 sign, 5 exponent (bias 15), 2 mantissa; max 57344 */
} mxfp8_fmt_t;

typedef enum {
    MXFP8_OK = 0,
    MXFP8_ERR_NULL = 1,      /* required pointer NULL, a data/scale pair half set, or no direction */
    MXFP8_ERR_SHAPE = 2,     /* M or N negative, N not a multiple of 8, or too large */
    MXFP8_ERR_ALIGN = 3,     /* x/out/workspace not 16-byte aligned, scale_col/dbias not 4-byte */
    MXFP8_ERR_FORMAT = 4,    /* fp8_fmt not MXFP8_E4M3 / MXFP8_E5M2, or an unknown option value */
    MXFP8_ERR_WORKSPACE = 5, /* dbias requested and workspace NULL */
    MXFP8_ERR_DEVICE = 6,    /* no usable CUDA device, or a buffer not on the current device */
    MXFP8_ERR_LAUNCH = 7,    /* a CUDA call of this library failed (driver/launch error) */
    MXFP8_ERR_GROUPS = 8     /* num_groups < 1 or above MXFP8_MAX_GROUPS, or offsets NULL */
} mxfp8_status_t;

/* Largest num_groups mxfp8_quantize_grouped accepts. */
#define MXFP8_MAX_GROUPS 512

/*
 * Bytes of device workspace mxfp8_quantize needs for (M, N, with_dbias).
 * 0 when with_dbias == 0.  With dbias it holds one fp32 partial column sum
 * per 128-row tile: ceil(M/128) * N * 4 bytes.  Returns 0 for invalid shapes.
 * (The workspace query precedes any launch, as on the PR #3137 page.)
 */
size_t mxfp8_quantize_workspace_bytes(int64_t M, int64_t N, int with_dbias);

/*
 * Quantize x[M,N] rowwise and/or columnwise (PR #3137: rowwise / colwise /
 * with_dbias / with_noop config fields).
 *
 *   x           device, bf16 [M,N], 16-byte aligned.
 *   M, N        M >= 0, N >= 0 a multiple of 8 (the TMA loads need a 16-byte
 *               BF16 row pitch; FP8 rows of N % 16 == 8 bytes are written with
 *               8-byte stores).  M == 0 or N == 0: nothing to quantize,
 *               x and the output pointers may then be NULL (dbias, if
 *               requested, is set to zeros unless noop).
 *   fp8_fmt     MXFP8_E4M3 or MXFP8_E5M2.
 *   out_row, scale_row   rowwise outputs; both NULL skips the rowwise direction.
 *   out_col, scale_col   columnwise outputs; both NULL skips that direction.
 *               Setting only one pointer of a pair is MXFP8_ERR_NULL, and so
 *               is skipping both directions.  out_* 16-byte aligned,
 *               scale_col 4-byte aligned.
 *   dbias       device fp32 [N] or NULL.  Written with the column sums of x,
 *               accumulated deterministically (fixed order, no atomics):
 *               per-tile fp32 partials, then a fixed-order fp32 sum over
 *               tiles; error below about 2.5e-6 * sum_i |x[i,j]|.
 *   workspace   device, >= mxfp8_quantize_workspace_bytes(M, N, dbias != NULL)
 *               bytes, 16-byte aligned; may be NULL when dbias is NULL.
 *   noop        device fp32 scalar or NULL (see above).
 *   stream      cudaStream_t.
 *
 * Returns MXFP8_OK once the work is enqueued.  The outputs must not overlap x
 * or each other.
 */
mxfp8_status_t mxfp8_quantize(const void *x, int64_t M, int64_t N, int fp8_fmt,
                              void *out_row, void *scale_row,
                              void *out_col, void *scale_col,
                              float *dbias, void *workspace, const float *noop,
                              void *stream);

/*
 * Workspace bytes for mxfp8_quantize_grouped: currently always 0 (the grouped
 * call keeps its schedule in shared memory); reserved so callers can size it.
 */
size_t mxfp8_quantize_grouped_workspace_bytes(int64_t total_rows, int64_t N, int num_groups);

/*
 * Grouped (MoE) quantize in one launch: rows [offsets[g], offsets[g+1]) of x
 * belong to expert g.  The ragged-offset convention follows the grouped
 * expert routing of "Lightning W4A16 grouped NVFP4 GEMM" (cudnn-frontend
 * PR #811, API section: per-expert offsets read on the device, one kernel,
 * zero workspace, no host copy of the offsets), here as a full prefix vector.
 *
 *   x            device bf16 [total_rows, N], 16-byte aligned.
 *   num_groups   1 .. MXFP8_MAX_GROUPS.
 *   offsets      device int64 [num_groups + 1]: offsets[0] == 0,
 *                offsets[num_groups] == total_rows, non-decreasing.  Read
 *                only on the device.  Empty groups produce no work.  No tile
 *                straddles two groups.
 *   outputs      every group is quantized as its own flat problem (the
 *                "non-32-divisible shapes" review: its columnwise blocks
 *                start at its first row and its last block holds the rows it
 *                has left, so no block mixes two groups).  out_row,
 *                scale_row and out_col are indexed by row as for
 *                mxfp8_quantize on the concatenated rows.  scale_col holds
 *                S = sum_g ceil(rows_g / 32) rows: group g's ceil(rows_g / 32)
 *                scale rows start at row sum_{h<g} ceil(rows_h / 32).  With
 *                every offset a multiple of 32, S = total_rows / 32 and the
 *                result equals the flat call on x; in general
 *                ceil(total_rows / 32) <= S <= total_rows / 32 + num_groups,
 *                and the caller allocates at least S rows.  No dbias.
 *   workspace    may be NULL (see mxfp8_quantize_grouped_workspace_bytes).
 *   err_flag     device int or NULL.  If the offsets break a rule above, the
 *                kernel writes nothing and sets *err_flag = 1.  It is never
 *                cleared by the library.
 *
 * total_rows is any size below 2^31; N a multiple of 8.
 */
mxfp8_status_t mxfp8_quantize_grouped(const void *x, int64_t total_rows, int64_t N,
                                      int num_groups, const int64_t *offsets, int fp8_fmt,
                                      void *out_row, void *scale_row,
                                      void *out_col, void *scale_col,
                                      void *workspace, const float *noop, int *err_flag,
                                      void *stream);

/*
 * Device staging bytes mxfp8_quantize_host needs for (M, N, with_dbias):
 * three chunk slots (input chunk plus its outputs) and, with dbias, the dbias
 * workspace of the whole matrix and an fp32 [N] vector.  0 for invalid or
 * empty shapes.
 */
size_t mxfp8_quantize_host_staging_bytes(int64_t M, int64_t N, int with_dbias);

/*
 * The same quantize with x and every output in HOST memory: the call moves
 * x to the device, quantizes it and moves the outputs back, pipelined over
 * row chunks (at most about 32 MiB of BF16 each, smaller at both ends) so
 * that the host-to-device copies,
 * the kernels and the device-to-host copies overlap.  Results are identical
 * to mxfp8_quantize on the same data (dbias included: the chunks write the
 * per-tile partials of one workspace and one reduce follows).
 *
 *   x_host, out_*_host, dbias_host   host buffers in the layouts of
 *               mxfp8_quantize; a direction is skipped as there.  Pinned
 *               memory (cudaHostAlloc / cudaHostRegister) lets the copies
 *               overlap; pageable memory works but serialises them.
 *   M, N        M > 0, N > 0 a multiple of 8.
 *   staging     device buffer, 256-byte aligned, at least
 *               mxfp8_quantize_host_staging_bytes(M, N, dbias_host != NULL)
 *               bytes (otherwise MXFP8_ERR_WORKSPACE); owned by the caller.
 *   stream      the kernels run on it; the copies run on two internal streams
 *               that wait for `stream` first, and `stream` waits for the last
 *               copy, so synchronising `stream` means every host output is
 *               written.  The library creates those two streams and a few
 *               events once per device, on the first call.
 * No noop flag: a skipped quantize would still copy stale staging bytes out.
 * Calls from several host threads are serialised while they enqueue.
 */
mxfp8_status_t mxfp8_quantize_host(const void *x_host, int64_t M, int64_t N, int fp8_fmt,
                                   void *out_row_host, void *scale_row_host,
                                   void *out_col_host, void *scale_col_host,
                                   float *dbias_host, void *staging, size_t staging_bytes,
                                   void *stream);

/*
 * The backward fusion, the gated cast and its backward with every input and
 * output in HOST memory, pipelined over row chunks (whole 128-row tiles,
 * about 32 MiB of input each) like mxfp8_quantize_host: the same arguments
 * as mxfp8_quantize_dact / mxfp8_quantize_gated / mxfp8_quantize_dgated,
 * host buffers in their layouts, a device staging buffer (256-byte aligned,
 * at least the matching *_host_staging_bytes) instead of the workspace, and
 * no noop.  Results are identical to the device calls on the same data (the
 * backward fusion's dbias too: every chunk writes its tile partials into one
 * workspace in the staging buffer and one reduce follows).  M > 0.  The
 * staging-bytes functions return 0 for invalid shapes.
 */
size_t mxfp8_quantize_dact_host_staging_bytes(int64_t M, int64_t N, int with_dbias);
mxfp8_status_t mxfp8_quantize_dact_host(const void *grad_host, const void *act_input_host,
                                        int64_t M, int64_t N, int fp8_fmt, int activation,
                                        void *out_row_host, void *scale_row_host,
                                        void *out_col_host, void *scale_col_host,
                                        float *dbias_host, void *staging, size_t staging_bytes,
                                        void *stream);
size_t mxfp8_quantize_gated_host_staging_bytes(int64_t M, int64_t N);
mxfp8_status_t mxfp8_quantize_gated_host(const void *x_host, int64_t M, int64_t N, int fp8_fmt,
                                         int activation, void *out_row_host, void *scale_row_host,
                                         void *out_col_host, void *scale_col_host, void *staging,
                                         size_t staging_bytes, void *stream);
size_t mxfp8_quantize_dgated_host_staging_bytes(int64_t M, int64_t N);
mxfp8_status_t mxfp8_quantize_dgated_host(const void *grad_host, const void *x_host, int64_t M,
                                          int64_t N, int fp8_fmt, int activation,
                                          void *out_row_host, void *scale_row_host,
                                          void *out_col_host, void *scale_col_host, void *staging,
                                          size_t staging_bytes, void *stream);

/*
 * Device staging bytes mxfp8_quantize_grouped_host needs: three chunk slots
 * (a chunk of x, its outputs, its columnwise scale rows and its group
 * offsets).  0 for invalid shapes or group counts.
 */
size_t mxfp8_quantize_grouped_host_staging_bytes(int64_t total_rows, int64_t N, int num_groups);

/*
 * The grouped cast (mxfp8_quantize_grouped; with an activation,
 * mxfp8_quantize_grouped_activated) with x, the offsets and every output in
 * HOST memory, pipelined over row chunks like mxfp8_quantize_host.  Results
 * are identical to the device call on the same data: a chunk boundary that
 * falls inside a group is moved down to a row a multiple of 32 rows after the
 * group's first row, so a group cut in two keeps its own 32-row blocks, and
 * the columnwise scale rows of the pieces are contiguous.
 *
 *   x_host        host bf16 [total_rows, N].
 *   host_offsets  host int64 [num_groups + 1], the layout of
 *                 mxfp8_quantize_grouped; checked here (offsets[0] == 0,
 *                 non-decreasing, offsets[num_groups] == total_rows), else
 *                 MXFP8_ERR_GROUPS before any work.  Read during the call
 *                 only.
 *   activation    MXFP8_ACT_NONE or one of the activations.
 *   out_*_host    host buffers in the device call's layouts (scale_col with
 *                 sum_g ceil(rows_g / 32) rows); a direction is skipped by
 *                 passing both of its pointers NULL.  Pinned memory lets the
 *                 copies overlap.
 *   staging       device buffer, 256-byte aligned, at least
 *                 mxfp8_quantize_grouped_host_staging_bytes(...) bytes.
 *   stream        as mxfp8_quantize_host.
 * No dbias, noop or err_flag.  total_rows > 0.
 */
mxfp8_status_t mxfp8_quantize_grouped_host(const void *x_host, int64_t total_rows, int64_t N,
                                           int num_groups, const int64_t *host_offsets,
                                           int fp8_fmt, int activation,
                                           void *out_row_host, void *scale_row_host,
                                           void *out_col_host, void *scale_col_host,
                                           void *staging, size_t staging_bytes, void *stream);

/*
 * Diagnostic (no counterpart on the pages): the row boundaries
 * 0 = b[0] < ... < b[k] = total_rows of the chunks mxfp8_quantize_grouped_host
 * uses for these offsets and N.  Writes min(k + 1, max_bounds) of them to
 * bounds (may be NULL) and returns k + 1, or -1 for invalid arguments.
 * Host only: it touches no device.
 */
int64_t mxfp8_grouped_host_chunks(const int64_t *host_offsets, int num_groups, int64_t total_rows,
                                  int64_t N, int64_t *bounds, int64_t max_bounds);

/* Layout of the E8M0 scale planes (the `swizzled` field of the PR #3137 config key). */
typedef enum {
    MXFP8_SCALES_PLAIN = 0,    /* scale_row [M, N/32], scale_col [M/32, N], row-major */
    MXFP8_SCALES_SWIZZLED = 1  /* GEMM-ready: see mxfp8_scale_bytes */
} mxfp8_scale_layout_t;

/*
 * Bytes of one scale plane for a scale matrix of `rows` x `scale_cols`.
 * MXFP8_SCALES_PLAIN: rows * scale_cols.  MXFP8_SCALES_SWIZZLED: the matrix
 * padded to multiples of 128 rows and 4 columns and stored as 128x4 tiles of
 * 512 bytes, tiles in row-tile-major order, entry (r, c) of a tile at byte
 * 16*(r % 32) + 4*(r / 32) + c; padding entries are written as 0.  This is
 * the scale-factor arrangement block-scaled tensor-core GEMMs read (the
 * reading taken for the config key's `swizzled` bit, which the pages leave
 * undefined).  For the rowwise plane rows = M, scale_cols = ceil(N/32); the
 * columnwise plane serves the transposed operand, rows = N, scale_cols =
 * ceil(M/32) (swizzled entry (j, i/32) holds the scale of column j, rows
 * i..i+31).
 * Returns 0 for an unknown layout or negative sizes.
 */
size_t mxfp8_scale_bytes(int64_t rows, int64_t scale_cols, int scale_layout);

/*
 * Activation applied to every element before the cast (the `with_act` /
 * `activation` fields of the PR #3137 config key).  It is evaluated in fp32
 * from the BF16 input; the block amax, the scales and the FP8 codes are those
 * of the fp32 activations, and amax (if requested) is max |act(x)|.
 *   RELU   x > 0 ? x : +0          SRELU  x > 0 ? x*x : +0   (squared ReLU)
 *   GELU   x * sigmoid(2 sqrt(2/pi) (x + 0.044715 x^3))      (tanh form)
 *   SILU   x * sigmoid(x)          QGELU  x * sigmoid(1.702 x)
 * sigmoid(t) is computed as 1/(1+e) or e/(1+e), e = exp(-|t|).  ReLU and SReLU
 * are exact; the others are within a few fp32 ulps of the exact function.
 * Not combinable with dbias (MXFP8_ERR_FORMAT).
 */
typedef enum {
    MXFP8_ACT_NONE = 0,
    MXFP8_ACT_RELU = 1,
    MXFP8_ACT_SRELU = 2,
    MXFP8_ACT_GELU = 3,
    MXFP8_ACT_SILU = 4,
    MXFP8_ACT_QGELU = 5
} mxfp8_activation_t;

/*
 * Options of mxfp8_quantize_ex: the fields of the quantization config key on
 * the PR #3137 page (fp8_dtype, rowwise, colwise, swizzled, with_amax,
 * with_dbias, with_noop) as one struct.  Zero-initialise it and set what is
 * needed; pointers and sizes mean what they mean for mxfp8_quantize.
 */
typedef struct mxfp8_quantize_config {
    const void *x;         /* device bf16 [M, N] */
    int64_t M, N;          /* M >= 0, N >= 0 a multiple of 8 */
    int fp8_fmt;           /* MXFP8_E4M3 / MXFP8_E5M2 */
    void *out_row;         /* uint8 [M, N] or NULL */
    void *scale_row;       /* mxfp8_scale_bytes(M, ceil(N/32), scale_layout) bytes */
    void *out_col;         /* uint8 [M, N] or NULL */
    void *scale_col;       /* mxfp8_scale_bytes(N, ceil(M/32), scale_layout) bytes (plain: [ceil(M/32), N]) */
    float *dbias;          /* fp32 [N] or NULL */
    void *workspace;       /* mxfp8_quantize_workspace_bytes(M, N, dbias != NULL) bytes */
    const float *noop;     /* device fp32 scalar or NULL */
    int scale_layout;      /* mxfp8_scale_layout_t */
    float *amax;           /* device fp32 scalar or NULL: receives max |x| over the tensor */
    int activation;        /* mxfp8_activation_t applied to x before the cast */
    int reserved[5];       /* must be 0 */
} mxfp8_quantize_config_t;

/*
 * mxfp8_quantize with every option of mxfp8_quantize_config_t.  With
 * MXFP8_SCALES_SWIZZLED the scale planes are written in the GEMM-ready
 * layout; swizzled scale pointers need no alignment.  amax, if set, is a
 * device fp32 written with the largest |x| of the tensor (4-byte aligned;
 * noop leaves it untouched like every other output).  activation applies an
 * mxfp8_activation_t before the cast.  Returns the status codes of
 * mxfp8_quantize, plus MXFP8_ERR_FORMAT for an unknown layout or activation,
 * an activation with dbias, or a non-zero reserved field, and MXFP8_ERR_NULL
 * for cfg == NULL.
 */
mxfp8_status_t mxfp8_quantize_ex(const mxfp8_quantize_config_t *cfg, void *stream);

/*
 * Device staging bytes mxfp8_quantize_ex_host needs for cfg (its M, N, dbias,
 * scale_layout and amax fields): three chunk slots sized for the layout, then
 * the dbias workspace and vector, then the amax.  0 for cfg == NULL or
 * invalid shapes.
 */
size_t mxfp8_quantize_ex_host_staging_bytes(const mxfp8_quantize_config_t *cfg);

/*
 * mxfp8_quantize_ex with x, every output, dbias and amax in HOST memory,
 * pipelined over row chunks as mxfp8_quantize_host (which is this call
 * without the layout, amax and activation options).  Results are identical to
 * mxfp8_quantize_ex on the same data: every chunk but the last is a whole
 * number of 128-row tiles, so a chunk's GEMM-ready rowwise plane is whole tile
 * rows of the matrix's plane and its columnwise plane a band of tile columns
 * (copied out with one strided copy); the amax is reduced on the device
 * across the chunks and copied out once.
 *   cfg->workspace and cfg->noop must be NULL (MXFP8_ERR_FORMAT otherwise):
 *   the workspace lives in the staging buffer, and a skipped call would still
 *   copy stale staging bytes out.
 *   staging   device buffer, 256-byte aligned, at least
 *             mxfp8_quantize_ex_host_staging_bytes(cfg) bytes.
 *   stream    as mxfp8_quantize_host.
 * M > 0, N > 0 a multiple of 8; otherwise the status codes of
 * mxfp8_quantize_host and of mxfp8_quantize_ex.
 */
mxfp8_status_t mxfp8_quantize_ex_host(const mxfp8_quantize_config_t *cfg, void *staging,
                                      size_t staging_bytes, void *stream);

/*
 * Backward fusion (the `with_dact` field of the PR #3137 config key): the
 * cast of y = dY * act'(X), with dbias (optional) = column sums of y.
 *   grad        device bf16 [M, N]: dY, 16-byte aligned.
 *   act_input   device bf16 [M, N]: X, the activation's input, 16-byte aligned.
 *   activation  MXFP8_ACT_RELU .. MXFP8_ACT_QGELU: act' is the derivative of
 *               that activation (as defined for mxfp8_activation_t),
 *               evaluated in fp32; y is the fp32 product.  dReLU and dSReLU
 *               are exact; the others are within a few fp32 ulps.
 *   outputs, dbias, workspace, noop, stream: as for mxfp8_quantize
 *               (workspace: mxfp8_quantize_workspace_bytes(M, N, 1) bytes).
 * Shapes as for mxfp8_quantize (M >= 0, N a multiple of 8).
 */
mxfp8_status_t mxfp8_quantize_dact(const void *grad, const void *act_input, int64_t M, int64_t N,
                                   int fp8_fmt, int activation,
                                   void *out_row, void *scale_row,
                                   void *out_col, void *scale_col,
                                   float *dbias, void *workspace, const float *noop,
                                   void *stream);

/*
 * Gated activation before the cast (the GLU family; the `activation` field of
 * the PR #3137 config key names the fused activation, the pages give no gated
 * form, so this library's reading is stated here): x = [a | b] is BF16
 * [M, 2N], a its first N columns (the activation's input) and b its last N
 * (the linear input), and the cast is of the fp32 value y = act(a) * b, an
 * [M, N] tensor quantized as by mxfp8_quantize:
 *   MXFP8_ACT_RELU   ReGLU            MXFP8_ACT_GELU   GeGLU (tanh form)
 *   MXFP8_ACT_SRELU  squared-ReLU GLU MXFP8_ACT_SILU   SwiGLU
 *   MXFP8_ACT_QGELU  QGeGLU
 *   x           device bf16 [M, 2N], row pitch 2N elements, 16-byte aligned.
 *   outputs     out_row / out_col uint8 [M, N], scale_row [M, ceil(N/32)],
 *               scale_col [ceil(M/32), N]; either direction may be NULL.
 *   noop, stream: as for mxfp8_quantize.  No dbias.
 * act is evaluated as for mxfp8_activation_t (ReGLU and the squared-ReLU GLU
 * are exact: y is a product of at most 24 significant bits; the others within
 * a few fp32 ulps).  M >= 0 and N a multiple of 8 (so that b starts on a
 * 16-byte boundary), N < 2^30.  Status codes as for mxfp8_quantize_dact.
 */
mxfp8_status_t mxfp8_quantize_gated(const void *x, int64_t M, int64_t N, int fp8_fmt, int activation,
                                    void *out_row, void *scale_row,
                                    void *out_col, void *scale_col,
                                    const float *noop, void *stream);

/*
 * mxfp8_quantize_grouped with an activation applied before the cast
 * (MXFP8_ACT_RELU .. MXFP8_ACT_QGELU, evaluated as for mxfp8_activation_t):
 * each group is its own flat problem of act(x) values, laid out as by
 * mxfp8_quantize_grouped.  No dbias.  Status codes as for
 * mxfp8_quantize_grouped, plus MXFP8_ERR_FORMAT for an unknown activation.
 */
mxfp8_status_t mxfp8_quantize_grouped_activated(const void *x, int64_t total_rows, int64_t N, int num_groups,
                                                const int64_t *offsets, int fp8_fmt, int activation,
                                                void *out_row, void *scale_row,
                                                void *out_col, void *scale_col,
                                                const float *noop, int *err_flag, void *stream);

/*
 * mxfp8_quantize_grouped (activation MXFP8_ACT_NONE, or an activation as for
 * mxfp8_quantize_grouped_activated) with each group's scale planes in the
 * GEMM-ready layout of MXFP8_SCALES_SWIZZLED, the layout a grouped
 * block-scaled GEMM reads per expert (this library's reading for the grouped
 * call; the pages define the swizzled bit for one tensor):
 *   scale_row  group g's own [rows_g, ceil(N/32)] plane, padded to 128-row x
 *              4-column tiles (padding zero), after the planes of the groups
 *              before it (at byte sum_{h<g} ceil(rows_h/128) * 128 *
 *              ceil(ceil(N/32)/4)*4);
 *   scale_col  group g's columnwise scales as the transposed operand's
 *              [N, ceil(rows_g/32)] plane in the same layout, after the planes
 *              of the groups before it (at byte sum_{h<g} ceil(rows_h/128) * 4 *
 *              ceil(N/128)*128).
 * Plane sizes: mxfp8_grouped_swizzled_scale_bytes.  out_row / out_col, offsets,
 * err_flag, noop and the checks as for mxfp8_quantize_grouped; no dbias.
 */
mxfp8_status_t mxfp8_quantize_grouped_swizzled(const void *x, int64_t total_rows, int64_t N, int num_groups,
                                               const int64_t *offsets, int fp8_fmt, int activation,
                                               void *out_row, void *scale_row,
                                               void *out_col, void *scale_col,
                                               const float *noop, int *err_flag, void *stream);

/*
 * Bytes of one GEMM-ready scale plane of mxfp8_quantize_grouped_swizzled
 * (colwise = 0: scale_row, 1: scale_col) for host_offsets (a host copy of the
 * call's offsets, num_groups + 1 entries).  0 for invalid arguments.
 */
size_t mxfp8_grouped_swizzled_scale_bytes(const int64_t *host_offsets, int num_groups, int64_t N, int colwise);

/*
 * mxfp8_quantize_gated over ragged per-expert row groups in one launch (an MoE
 * layer's gated activation before its second GEMM): rows
 * [offsets[g], offsets[g+1]) of x = [a | b] (bf16 [total_rows, 2N]) are group g,
 * each quantized as its own flat problem, laid out as by mxfp8_quantize_grouped:
 * out_row, scale_row, out_col indexed by row ([total_rows, N],
 * [total_rows, ceil(N/32)], [total_rows, N]); scale_col holds
 * S = sum_g ceil(rows_g / 32) rows, group g's after those of the groups before
 * it (total_rows / 32 rows when every offset is a multiple of 32).  offsets,
 * num_groups, err_flag and their checks as for mxfp8_quantize_grouped; noop and
 * stream as for mxfp8_quantize.  N a multiple of 8 below 2^30.
 */
mxfp8_status_t mxfp8_quantize_gated_grouped(const void *x, int64_t total_rows, int64_t N, int num_groups,
                                            const int64_t *offsets, int fp8_fmt, int activation,
                                            void *out_row, void *scale_row,
                                            void *out_col, void *scale_col,
                                            const float *noop, int *err_flag, void *stream);

/*
 * Backward of the gated activation (mxfp8_quantize_gated): for y = act(a) * b
 * and its gradient g, the cast of the gradient of x = [a | b]:
 *     da = g * b * act'(a),   db = g * act(a)     (fp32, act' as for
 *                                                  mxfp8_quantize_dact)
 * da and db are quantized as two [M, N] tensors laid side by side (this
 * library's reading; the pages do not define the gated forms):
 *   grad        device bf16 [M, N], 16-byte aligned.
 *   x           device bf16 [M, 2N] = [a | b], 16-byte aligned.
 *   out_row     uint8 [M, 2N]: da's codes in columns 0..N-1, db's in N..2N-1
 *               (block = 1x32 along a row within one half).
 *   scale_row   uint8 [M, 2 ceil(N/32)]: da's ceil(N/32) blocks, then db's.
 *   out_col     uint8 [M, 2N], scale_col uint8 [ceil(M/32), 2N] (columns as
 *               in out_col).
 *   Either direction may be NULL; noop and stream as for mxfp8_quantize.
 * With N a multiple of 32 the result is the cast of [da | db] as one [M, 2N]
 * tensor.  M >= 0, N a multiple of 8 below 2^30.  Status codes as for
 * mxfp8_quantize_dact.
 */
mxfp8_status_t mxfp8_quantize_dgated(const void *grad, const void *x, int64_t M, int64_t N, int fp8_fmt,
                                     int activation, void *out_row, void *scale_row,
                                     void *out_col, void *scale_col,
                                     const float *noop, void *stream);

/*
 * Workspace bytes for mxfp8_quantize_grouped_dbias: a header of
 * (num_groups + 1) int64 (each group's first row tile) padded to 256 bytes,
 * then one fp32 partial row per 128-row tile, tiles never spanning two
 * groups: at most (ceil(total_rows/128) + num_groups) * N * 4 bytes.  0 for
 * invalid sizes.
 */
size_t mxfp8_quantize_grouped_dbias_workspace_bytes(int64_t total_rows, int64_t N, int num_groups);

/*
 * mxfp8_quantize_grouped plus a per-expert dbias (the "grouped-call dbias per
 * expert" next to with_amax in the config fields of the PR #3137 page):
 *   dbias      device fp32 [num_groups, N]: row g = column sums of the rows of
 *              group g (zeros for an empty group), accumulated in a fixed
 *              order as in mxfp8_quantize.
 *   workspace  device, >= mxfp8_quantize_grouped_dbias_workspace_bytes(...)
 *              bytes, 16-byte aligned.
 * Everything else as for mxfp8_quantize_grouped; with invalid offsets nothing
 * is written, dbias included, and *err_flag is set.
 */
mxfp8_status_t mxfp8_quantize_grouped_dbias(const void *x, int64_t total_rows, int64_t N,
                                            int num_groups, const int64_t *offsets, int fp8_fmt,
                                            void *out_row, void *scale_row,
                                            void *out_col, void *scale_col,
                                            float *dbias, void *workspace, const float *noop,
                                            int *err_flag, void *stream);

/* Static, human-readable text for a status code. */
const char *mxfp8_status_string(int status);

/* Number of kernels this library has launched in this process (diagnostic). */
uint64_t mxfp8_kernel_launch_count(void);

/*
 * Read (and, if clear != 0, reset) the library's device fault word on the
 * current device.  Bit 0 is set when a kernel gave up waiting for its own
 * tile copies (a bounded wait expired) and returned early.  Synchronizes the
 * device.  Returns MXFP8_OK or MXFP8_ERR_DEVICE / MXFP8_ERR_LAUNCH.
 */
mxfp8_status_t mxfp8_device_fault_word(unsigned int *out, int clear);

/*
 * Diagnostic (no counterpart on the pages): exercises, without any fault, the
 * bounded wait every pipeline kernel uses.  One thread waits limit_ns
 * nanoseconds of wall time on an mbarrier phase that nothing completes; when
 * the wait expires it sets bit 0 of the fault word, as a pipeline CTA does,
 * writes 1 to *timed_out (device int; 0 if the phase had completed), and the
 * kernel returns, leaving the context usable.  0 < limit_ns <= 10 s.
 * Stream-ordered on `stream`.  Returns MXFP8_OK, MXFP8_ERR_NULL (timed_out
 * NULL), MXFP8_ERR_SHAPE (limit out of range), MXFP8_ERR_DEVICE or
 * MXFP8_ERR_LAUNCH.
 */
mxfp8_status_t mxfp8_selftest_bounded_wait(int64_t limit_ns, int *timed_out, void *stream);

/*
 * Diagnostic (no counterpart on the pages): the fp32 values the kernels form
 * from BF16 inputs, so that their accuracy can be checked on every input.
 *   x           device bf16 [n] (2-byte aligned), any bit patterns.
 *   activation  MXFP8_ACT_RELU .. MXFP8_ACT_QGELU.
 *   derivative  0: act(x) as the forward cast (mxfp8_quantize_ex with
 *               `activation`) evaluates it, for its scales and codes alike;
 *               1: act'(x) as mxfp8_quantize_dact evaluates it (the product
 *               with dY is one further fp32 multiply).
 *   out         device fp32 [n], 4-byte aligned.
 * Stream-ordered on `stream`.  Returns MXFP8_OK, MXFP8_ERR_FORMAT (activation
 * or derivative out of range), MXFP8_ERR_SHAPE (n < 0 or n >= 2^40),
 * MXFP8_ERR_NULL, MXFP8_ERR_ALIGN, MXFP8_ERR_DEVICE or MXFP8_ERR_LAUNCH.
 */
mxfp8_status_t mxfp8_activation_values(const void *x, int64_t n, int activation, int derivative, float *out,
                                       void *stream);

/* Size of the static scratch array used by mxfp8_quantize_dbias_noalloc. */
#define MXFP8_NOALLOC_SCRATCH_BYTES (8u << 20)

/*
 * mxfp8_quantize with dbias, for callers that cannot allocate device memory.
 * (The pages have no counterpart to this call.)
 *
 * Some callers have no way to allocate: a plugin or callback that is handed
 * only its input and output tensors, with no allocator or workspace to draw
 * from, or code that must not allocate once it is running.  This call takes
 * the same arguments as mxfp8_quantize minus the workspace, and keeps the
 * dbias workspace in a file-scope device array of MXFP8_NOALLOC_SCRATCH_BYTES
 * (8 MiB) inside the library.  Each GPU holds the array from the moment the
 * library's device code is loaded on it (the first use of any of its
 * kernels, or the first call of this function, on that device) until the
 * process exits.  It calls no cudaMalloc or cudaFree.
 *
 *   dbias      required (device fp32 [N]); NULL is MXFP8_ERR_NULL.
 *   M, N       as for mxfp8_quantize; shapes whose workspace
 *              (mxfp8_quantize_workspace_bytes(M, N, 1) = ceil(M/128)*N*4
 *              bytes) exceeds 8 MiB are rejected with MXFP8_ERR_SHAPE, e.g.
 *              16384 x 8192 fits (4 MiB), 32768 x 16384 does not.
 *   others     as for mxfp8_quantize.
 * Statuses come in mxfp8_quantize's order: MXFP8_ERR_FORMAT, then the shape
 * rules (MXFP8_ERR_SHAPE), then a NULL dbias (MXFP8_ERR_NULL), then a shape
 * beyond the scratch array (MXFP8_ERR_SHAPE), then mxfp8_quantize's own
 * remaining checks.
 *
 * The first call on a device looks up the array's device address on that
 * device (cudaGetSymbolAddress); make that first call before any stream
 * capture.  Every call shares the one array, and each call writes every
 * workspace entry it reads, so nothing carries over between calls; calls that
 * overlap on the GPU (other streams, other host threads) race on the array.
 */
mxfp8_status_t mxfp8_quantize_dbias_noalloc(const void *x, int64_t M, int64_t N, int fp8_fmt,
                                            void *out_row, void *scale_row,
                                            void *out_col, void *scale_col,
                                            float *dbias, const float *noop, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* MXFP8_GB300_H */
