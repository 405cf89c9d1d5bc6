/*
 * fp4q -- micro-scaled FP4 quantize / convert / block-scaled GEMM for GB300 (sm_103a).
 *
 * C ABI.  Every pointer named "device" is GPU global memory owned by the
 * caller; the library allocates no device memory.  Every call is
 * asynchronous on `stream` (never synchronises), except the status reads
 * (fp4q_device_status, fp4q_stream_status), which say so, and validates its
 * arguments before launching: an argument error is returned immediately and
 * nothing is launched.  A launch failure returns FP4Q_ERR_CUDA.  Device-side
 * wait timeouts are recorded in a device status word read by
 * fp4q_device_status() or fp4q_stream_status().  Inputs must be finite;
 * non-finite inputs give unspecified codes but never a fault.  Calls from
 * several host threads are safe; calls that share buffers are ordered by the
 * caller's streams.
 *
 * Conventions shared by all calls:
 *  - Tensors are row-major [rows, cols]; blocks run along the last
 *    (contiguous) axis (block_axis = 1).  block_axis = 0 (column-wise
 *    blocks, for the weight-gradient operands) is accepted where a call says
 *    so: the result is then the block_axis = 1 quantization of the transpose,
 *    written in the transposed layout ([cols, rows/2] codes, scales of a
 *    cols x rows/B matrix), without the transpose ever being stored.
 *  - Packed FP4 (E2M1): element i of a row sits in the low nibble of byte
 *    i/2 when i is even and in the high nibble when i is odd; a row of C
 *    elements takes C/2 bytes and rows are contiguous (row stride C/2).
 *  - Block scales come in one of two layouts (fp4q_scale_layout):
 *      ROWMAJOR: [rows, cols/B] bytes, row-major, no padding.
 *      MMA:      the layout the tcgen05 block-scaled MMA reads.  The scale
 *                matrix (rows x S, S = cols/B) is cut into 128 x 4 tiles,
 *                stored tile-row-major (tile (rt, ct) at byte
 *                (rt * ceil(S/4) + ct) * 512); inside a tile, scale (r, c)
 *                sits at byte (r % 32) * 16 + (r / 32) * 4 + c.  Size:
 *                fp4q_scales_bytes().  Padding entries are not written.
 *  - Pointers to packed data, scales and outputs must be 16-byte aligned
 *    (32-byte where a call says so).
 *
 * The operations follow three web pages:
 *  [MXN] "Pretraining large language models with MXFP4 on Native FP4
 *        Hardware" (news article): the MX format section (32-element
 *        blocks, E8M0 shared exponent, X = 2^E * Q_FP4(X / 2^E)) and the
 *        investigation section (Fprop / Dgrad / Wgrad GEMMs).
 *  [HOP] "Practical FP4 Training for Large-Scale MoE Models on Hopper GPUs"
 *        (technical summaries): section 2 (direct FP8 -> FP4, bitwise
 *        FP4 -> FP8 with hierarchical scale alignment, ragged MoE tensors).
 *  [NVF] "Pretraining Large Language Models with NVFP4" (technical
 *        summary): section 2.A (NVFP4 format) and 2.B (random Hadamard
 *        transform, stochastic rounding).
 */
#ifndef FP4Q_H
#define FP4Q_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; NULL is the legacy default stream. */
struct CUstream_st;
typedef struct CUstream_st* fp4q_stream_t;

typedef enum fp4q_status {
    FP4Q_OK = 0,
    FP4Q_ERR_INVALID_ARGUMENT = 1,   /* null pointer, bad enum, negative size   */
    FP4Q_ERR_UNSUPPORTED_SHAPE = 2,  /* partial block, K % 128, block_axis != 1  */
    FP4Q_ERR_MISALIGNED = 3,         /* pointer not 16-byte aligned              */
    FP4Q_ERR_UNSUPPORTED_DEVICE = 4, /* current device is not compute cap. 10.3  */
    FP4Q_ERR_CUDA = 5,               /* a CUDA call or launch failed             */
    FP4Q_ERR_TIMEOUT = 6             /* a device-side wait ran out (status word) */
} fp4q_status;

typedef enum fp4q_dtype { FP4Q_BF16 = 0, FP4Q_FP32 = 1, FP4Q_E4M3 = 2 } fp4q_dtype;
typedef enum fp4q_scale_layout { FP4Q_SCALES_ROWMAJOR = 0, FP4Q_SCALES_MMA = 1 } fp4q_scale_layout;
typedef enum fp4q_rounding { FP4Q_RNE = 0, FP4Q_SR = 1 } fp4q_rounding;
typedef enum fp4q_format { FP4Q_MXFP4 = 0, FP4Q_NVFP4 = 1, FP4Q_MXFP8 = 2 } fp4q_format;

/* Human-readable name of a status code (static string). */
const char* fp4q_status_string(fp4q_status status);

/* Detail of the last failing call on this host thread (static per thread). */
const char* fp4q_last_error(void);

/* Bytes of a block-scale matrix of `rows` x `scale_cols` in `layout`
 * (ROWMAJOR: rows * scale_cols; MMA: padded to 128 x 4 tiles); 0 for negative
 * sizes and for sizes whose byte count does not fit a size_t. */
size_t fp4q_scales_bytes(int64_t rows, int64_t scale_cols, fp4q_scale_layout layout);

/*
 * fp4q_mx_quantize -- BF16 / FP32 / FP8-E4M3 -> MXFP4.
 * [MXN] MX section: blocks of 32 elements share one E8M0 exponent
 * E = floor(log2(block amax)) - 2 (clamped to [-127, 127]; an all-zero block
 * takes E = -127), and each element is stored as the E2M1 code nearest to
 * x / 2^E (ties to even, saturating at +-6, sign kept also for zeros).
 * [HOP] abstract and section 1: with x_type == FP4Q_E4M3 the source is FP8
 * quantized straight to FP4 with no BF16 intermediate: element value =
 * decode(e4m3) * tile_scale[r, c / 128] (one FP32 multiply), then the rule
 * above.
 *   x          device, [rows, ld_x] elements of x_type, ld_x >= cols; x must
 *              be 32-byte aligned and ld_x * element size a multiple of 32 bytes
 *   tile_scale device FP32 [rows, cols/128] when x_type == FP4Q_E4M3
 *              (cols % 128 == 0), else NULL
 *   cols       multiple of 32
 *   q          device out, [rows, cols/2] packed codes
 *   scales     device out, E8M0 bytes in `layout` (rows x cols/32)
 *   block_axis 1; or 0 for a BF16 source with rows % 128 == 0 and
 *              cols % 128 == 0: q [cols, rows/2] and scales (cols x rows/32)
 *              of X^T ([HOP] 2.C: kernels with native support for transposed
 *              layouts, for the weight-gradient GEMM).
 */
fp4q_status fp4q_mx_quantize(const void* x, fp4q_dtype x_type, const float* tile_scale,
                             int64_t rows, int64_t cols, int64_t ld_x, int block_axis,
                             uint8_t* q, uint8_t* scales, fp4q_scale_layout layout,
                             fp4q_stream_t stream);

/*
 * fp4q_mx_dequantize -- MXFP4 -> BF16 / FP32: y = 2^E * value(code), exact
 * (rounded only where it overflows the output type).  [MXN] reconstruction.
 *   q       device, [rows, cols/2];  scales device, ROWMAJOR E8M0 [rows, cols/32]
 *   y       device out, [rows, cols] of y_type (FP4Q_BF16 or FP4Q_FP32), 32-byte aligned
 */
fp4q_status fp4q_mx_dequantize(const uint8_t* q, const uint8_t* scales, int64_t rows,
                               int64_t cols, int block_axis, void* y, fp4q_dtype y_type,
                               fp4q_stream_t stream);

/*
 * fp4q_fp4_to_fp8 -- scaled MXFP4 -> FP8-E4M3 with one FP32 scale per 1x128 tile.
 * [HOP] section 2.B: hierarchical scale alignment -- the tile scale is the
 * largest of the tile's four E8M0 block scales, 2^Emax; each element is the
 * E4M3 encoding of value(code) * 2^(E_i - Emax), produced by remapping the
 * sign / exponent / mantissa fields (no floating-point arithmetic).
 * [HOP, Spanish summary] section 2: subnormal results keep their value.
 * Magnitudes below the smallest E4M3 subnormal (2^-9) become signed zero;
 * values are exact whenever E_i - Emax >= -8.
 *   q           device, [rows, cols/2];  scales device, ROWMAJOR E8M0 [rows, cols/32]
 *   cols        multiple of 128
 *   y           device out, E4M3 [rows, cols], 32-byte aligned
 *   tile_scale  device out, FP32 [rows, cols/128]
 */
fp4q_status fp4q_fp4_to_fp8(const uint8_t* q, const uint8_t* scales, int64_t rows,
                            int64_t cols, int block_axis, uint8_t* y, float* tile_scale,
                            fp4q_stream_t stream);

/*
 * fp4q_fp8_pipeline_host -- the FP8 activation path on HOST buffers: E4M3
 * activations with 1x128 FP32 tile scales are quantized straight to MXFP4
 * ([HOP] abstract and section 1, as fp4q_mx_quantize with x_type FP4Q_E4M3)
 * and re-expanded to FP8 for an FP8 consumer ([HOP] 2.B, as fp4q_fp4_to_fp8);
 * the MXFP4 codes and scales and the FP8 copy are written back to host memory.
 * Results are bit-identical to the two device calls.
 * The rows go through the device in chunks of chunk_rows (0: 2048), using
 * three slots of `workspace`: host -> device copies, the two conversion
 * kernels (on `stream`) and device -> host copies of different chunks overlap
 * on two internal copy streams (one pair per host thread and device, created
 * on first use, destroyed by fp4q_fp8_pipeline_host_release).  The call
 * starts after the work already queued on `stream` and returns once
 * everything is queued; the host outputs are complete when
 * `stream` reaches the point of the call (e.g. after cudaStreamSynchronize).
 * Host buffers should be page-locked for the copies to overlap; pageable
 * memory gives the same results without the overlap.
 *   x             host E4M3 [rows, cols];  tile_scale host FP32 [rows, cols/128]
 *   cols          multiple of 128
 *   q, scales     host out: codes [rows, cols/2], ROWMAJOR E8M0 [rows, cols/32]
 *   y, y_tile_scale host out: E4M3 [rows, cols], FP32 [rows, cols/128]
 *   workspace     device, >= fp4q_fp8_pipeline_host_workspace_bytes(cols,
 *                 chunk_rows) bytes (chunk_rows capped at rows), 256-byte aligned;
 *                 owned by the call until `stream` passes it
 * Errors: negative sizes or a NULL pointer -> INVALID_ARGUMENT; cols % 128,
 * cols > 2^31 or a chunk of more than 2^40 elements -> UNSUPPORTED_SHAPE (the
 * workspace query then returns 0); misaligned workspace -> MISALIGNED; a
 * failed copy, event or launch -> CUDA.  rows == 0 or cols == 0 does nothing.
 */
size_t fp4q_fp8_pipeline_host_workspace_bytes(int64_t cols, int64_t chunk_rows);
fp4q_status fp4q_fp8_pipeline_host(const uint8_t* x, const float* tile_scale, int64_t rows,
                                   int64_t cols, uint8_t* q, uint8_t* scales, uint8_t* y,
                                   float* y_tile_scale, int64_t chunk_rows, void* workspace,
                                   size_t workspace_bytes, fp4q_stream_t stream);

/*
 * fp4q_fp8_pipeline_host_release -- destroys the two copy streams and the
 * events fp4q_fp8_pipeline_host created for the calling host thread on the
 * current device (otherwise they live until the process exits).  The pages
 * have no counterpart: this is library housekeeping.  Waits for those two
 * copy streams first, so no copy of an earlier call is cut short; a later
 * fp4q_fp8_pipeline_host call on this thread creates them again.  Nothing to
 * release returns FP4Q_OK.  Synchronous on the host.
 */
fp4q_status fp4q_fp8_pipeline_host_release(void);

/*
 * fp4q_nv_quantize -- BF16 -> NVFP4 (optional 16-point RHT, RNE or SR).
 * [NVF] 2.A: 16-element blocks of E2M1 with one E4M3 scale each under one
 * FP32 tensor scale.  With y the (optionally rotated) values and amax the
 * tensor max |y|:  s_t = amax / 2688;  s_b = E4M3_rn_satfinite(blockamax /
 * (6 s_t));  sf = float(s_b) * s_t;  q = ROUND(y * (1 / sf)); all in FP32
 * with IEEE round-to-nearest operations.  amax == 0 or s_b == 0 gives
 * signed-zero codes.
 * [NVF] 2.B: rht == 1 applies y = (1/4) H16 diag(d) x on every 16-element
 * tile (Sylvester H16; d_j = -1 iff bit j of word 0 of Philox4x32-10 with
 * key = rht_seed and counter 0; butterflies with strides 1, 2, 4, 8 in FP32).
 * rht == 2 applies the deterministic H16 (d = 1, the same rotation at every
 * call: [MXN] Wgrad section); rht_seed is then ignored.
 * rounding == FP4Q_SR rounds each element up with probability equal to its
 * distance fraction: up iff r < frac * 2^32, r the (i mod 4)-th word of
 * Philox4x32-10(key = sr_seed, counter = i / 4), i = row * cols + col.
 *   x                device BF16 [rows, ld_x], 32-byte aligned, ld_x % 16 == 0;
 *                    cols % 16 == 0
 *   amax_in          device FP32 scalar or NULL (NULL: computed, two passes)
 *   amax_out         device FP32 scalar out or NULL
 *   tensor_scale_out device FP32 scalar out (s_t)
 *   q                device out, [rows, cols/2];  scales device out, E4M3 in `layout`
 *   workspace        device, >= fp4q_nv_quantize_workspace_bytes() bytes, 16-B
 *                    aligned; used only when amax_in == NULL (may be NULL then
 *                    not); reset by the call itself.
 *   block_axis       1; or 0 (rows % 128 == 0, cols % 64 == 0): blocks, RHT
 *                    tiles and the stochastic-rounding index i follow X^T,
 *                    q [cols, rows/2], scales (cols x rows/16).
 */
size_t fp4q_nv_quantize_workspace_bytes(int64_t rows, int64_t cols);
fp4q_status fp4q_nv_quantize(const void* x, int64_t rows, int64_t cols, int64_t ld_x,
                             int block_axis, int rht, uint64_t rht_seed,
                             fp4q_rounding rounding, uint64_t sr_seed, const float* amax_in,
                             float* amax_out, float* tensor_scale_out, uint8_t* q,
                             uint8_t* scales, fp4q_scale_layout layout, void* workspace,
                             size_t workspace_bytes, fp4q_stream_t stream);

/*
 * fp4q_nv_quantize_sr_rne -- one NVFP4 quantization of a BF16 gradient with
 * both roundings over the same scales: the stochastically rounded codes into
 * q_sr and the round-to-nearest-even codes into q_rne, from one read of x and
 * one rotation.  [NVF] 2.B: stochastic rounding on the gradients, the RNE
 * codes being the deterministic counterpart of the same scaled values.
 * Results are bit-identical to fp4q_nv_quantize with FP4Q_SR and then with
 * FP4Q_RNE on the same x, seeds and amax (the scales of the two calls are the
 * same bytes).  Row-wise blocks only (block_axis 1).
 *   q_sr, q_rne   device out, [rows, cols/2] each, 16-byte aligned
 *   other arguments as fp4q_nv_quantize
 */
fp4q_status fp4q_nv_quantize_sr_rne(const void* x, int64_t rows, int64_t cols, int64_t ld_x, int rht,
                                    uint64_t rht_seed, uint64_t sr_seed, const float* amax_in,
                                    float* amax_out, float* tensor_scale_out, uint8_t* q_sr,
                                    uint8_t* q_rne, uint8_t* scales, fp4q_scale_layout layout,
                                    void* workspace, size_t workspace_bytes, fp4q_stream_t stream);

/*
 * fp4q_nv_quantize_2d -- BF16 weights -> NVFP4 with one E4M3 scale per 16 x 16
 * tile.  [NVF] 2.B (two-dimensional scaling): weight blocks of 16 x 16, so that
 * the forward pass and the backward pass, which reads the weight transposed,
 * use the same quantized values.  The rules of fp4q_nv_quantize with the block
 * amax taken over the 16 x 16 tile; no rotation.  The tile's scale is written
 * for each of its 16 rows (scales rows x cols/16 in `layout`), so the result
 * feeds fp4q_block_scaled_gemm unchanged; the quantization of W^T is the
 * transpose of that of W.
 *   x         device BF16 [rows, ld_x], 32-byte aligned, ld_x % 16 == 0;
 *             rows % 16 == 0, cols % 16 == 0
 *   other arguments as fp4q_nv_quantize (SR index i = row * cols + col)
 */
fp4q_status fp4q_nv_quantize_2d(const void* x, int64_t rows, int64_t cols, int64_t ld_x,
                                fp4q_rounding rounding, uint64_t sr_seed, const float* amax_in,
                                float* amax_out, float* tensor_scale_out, uint8_t* q,
                                uint8_t* scales, fp4q_scale_layout layout, void* workspace,
                                size_t workspace_bytes, fp4q_stream_t stream);

/*
 * fp4q_fp4_row_to_fp8_col -- FP4RowToFP8Col: row-wise MXFP4 [rows, cols] ->
 * FP8-E4M3 of the transpose [cols, rows] with one FP32 scale per 1x128 tile
 * along the output rows.  [HOP] Spanish summary section 2 (kernels
 * BF16ToFP4Row, FP4RowToFP8Row, FP4RowToFP8Col) and French summary 2.C: one
 * kernel dequantizes, transposes and re-quantizes the weight-gradient operand.
 * Output tile (c, rows r0 .. r0+127): scale 2^Emax, Emax the largest block
 * exponent among its 128 elements; element = E4M3 of value(code) *
 * 2^(E - Emax) by field remapping, as fp4q_fp4_to_fp8 (exact unless below
 * 2^-9 of its tile, then a signed zero).
 *   q           device, [rows, cols/2], 32-byte aligned
 *   scales      device, ROWMAJOR E8M0 [rows, cols/32], 4-byte aligned
 *   rows, cols  multiples of 128
 *   y           device out, E4M3 [cols, rows], 32-byte aligned
 *   tile_scale  device out, FP32 [cols, rows/128]
 */
fp4q_status fp4q_fp4_row_to_fp8_col(const uint8_t* q, const uint8_t* scales, int64_t rows,
                                    int64_t cols, uint8_t* y, float* tile_scale,
                                    fp4q_stream_t stream);

/*
 * fp4q_fp4_row_to_fp8_col_grouped -- FP4RowToFP8Col on ragged expert groups:
 * [HOP] French summary 2.C (per-expert tensors of ragged sizes, located by
 * precomputed offsets) with the element and tile rules of
 * fp4q_fp4_row_to_fp8_col.  The 1x128 tiles run along each group's rows and
 * restart at its first row; a group's last tile may be partial, and its scale
 * is 2^Emax over its real rows.  The output pads each group to whole tiles:
 * with T_g the tiles of the groups before g, group g's rows
 * offsets[g] .. offsets[g+1] - 1 land at columns 128 T_g .. 128 T_g + n_g - 1
 * of every output row, the rest of its last tile is 0, and columns from
 * 128 T_groups on are not written -- the padded per-group tile layout of
 * fp4q_mx_rebase_scales, which a grouped weight-gradient GEMM reads.
 *   q, scales   device, the rows' MXFP4 codes [rows, cols/2] (32-byte aligned)
 *               and ROWMAJOR E8M0 [rows, cols/32] (4-byte aligned)
 *   cols        multiple of 128;  rows, cols <= 2^31 - 1
 *   offsets     device int64 [groups + 1], 1 <= groups <= 256, clamped by the
 *               kernel like those of fp4q_mx_rebase_scales (each into
 *               [previous offset, rows]; rows past offsets[groups] ignored)
 *   y           device out, E4M3 [cols, ld], ld =
 *               fp4q_fp4_row_to_fp8_col_grouped_ld(rows, groups)
 *               = 128 * (ceil(rows / 128) + groups), 32-byte aligned
 *   tile_scale  device out, FP32 [cols, ld / 128]: tile t of output row c
 * fp4q_fp4_row_to_fp8_col_grouped_ld returns 0 for arguments the call rejects.
 */
int64_t fp4q_fp4_row_to_fp8_col_grouped_ld(int64_t rows, int64_t groups);
fp4q_status fp4q_fp4_row_to_fp8_col_grouped(const uint8_t* q, const uint8_t* scales, int64_t rows,
                                            int64_t cols, const int64_t* offsets, int64_t groups,
                                            uint8_t* y, float* tile_scale, fp4q_stream_t stream);

/*
 * fp4q_fp8_tile_scales_to_e8m0 -- FP32 power-of-two scales, one per 1x128 tile
 * (what fp4q_fp4_to_fp8 and fp4q_fp4_row_to_fp8_col write), -> E8M0 block
 * scales, one per 32 elements, so that their FP8 output feeds
 * fp4q_block_scaled_gemm as FP4Q_MXFP8 operands with no rounding: [HOP]
 * section 1 and Spanish section 2 (FP4 storage, FP8 compute; the FP8 copy of
 * an MXFP4 tensor carries a power-of-two tile scale, so E8M0 holds it exactly).
 * A scale that is not a power of two in [2^-127, 2^127] gives 0xFF and sets
 * bit 3 of the device status word.
 *   tile_scale  device FP32 [rows, cols/128];  cols % 128 == 0
 *   scales      device out, E8M0 (rows x cols/32) in `layout`
 */
fp4q_status fp4q_fp8_tile_scales_to_e8m0(const float* tile_scale, int64_t rows, int64_t cols,
                                         uint8_t* scales, fp4q_scale_layout layout, fp4q_stream_t stream);

/* One FP4 GEMM operand.  Host struct; the pointers in it are device pointers. */
typedef struct fp4q_operand {
    const uint8_t* q;           /* packed E2M1 [rows, K/2] (row stride K/2 bytes), or
                                   E4M3 [rows, K] for MXFP8                           */
    const uint8_t* scales;      /* block scales in FP4Q_SCALES_MMA layout              */
    fp4q_format format;         /* MXFP4: E8M0 per 32; NVFP4: E4M3 per 16;
                                   MXFP8: E8M0 per 32                                 */
    const float* tensor_scale;  /* NVFP4: device FP32 scalar s_t; MXFP4: NULL          */
} fp4q_operand;

/*
 * fp4q_block_scaled_gemm -- D = A . B^T on the tcgen05 block-scaled tensor cores.
 * [MXN] investigation section: the forward GEMM of a linear layer, Y = X W^T,
 * with both operands FP4 along the reduction axis K.  [NVF] 2.B: for NVFP4
 * operands the result is scaled by s_tA * s_tB, and a Hadamard rotation
 * applied to both operands along K cancels in the product.  FP4Q_MXFP8
 * operands (E4M3 codes with E8M0 scales per 32, kind::mxf8f6f4) are the FP8
 * consumer of fp4q_fp4_to_fp8 / fp4q_fp4_row_to_fp8_col ([HOP] section 1:
 * FP4 storage, FP8 GEMMs); their scales come from
 * fp4q_fp8_tile_scales_to_e8m0.
 *   A, B     operands of the same format; A has M rows, B has N rows, both K columns
 *   K        multiple of 128;  M, N >= 0 (M or N == 0: nothing is done;
 *            K == 0: D is set to zero)
 *   D        device out, [M, ldd] of d_type (FP4Q_BF16, RNE from FP32, or FP4Q_FP32),
 *            ldd >= N, ldd * element size a multiple of 16 bytes
 * FP32 accumulation.  Limits: M, N, K <= 2^30 and fewer than 2^31 output
 * tiles of 128 x 256, else FP4Q_ERR_UNSUPPORTED_SHAPE.
 */
fp4q_status fp4q_block_scaled_gemm(const fp4q_operand* A, const fp4q_operand* B, int64_t M,
                                   int64_t N, int64_t K, void* D, fp4q_dtype d_type,
                                   int64_t ldd, fp4q_stream_t stream);

/*
 * ---------------------------------------------------------------------------
 * MoE expert FFN in FP4 ("Practical FP4 Training for Large-Scale MoE Models
 * on Hopper GPUs", section 2.A: activations are quantized to MXFP4 before the
 * expert dispatch; section 2.C: ragged per-expert tensors with precomputed
 * offsets and no padding; section 4: the expert layers dominate the compute).
 * ---------------------------------------------------------------------------
 */

/*
 * fp4q_moe_dispatch -- group the MXFP4 rows of the tokens by expert.
 * Dispatched row p of expert e (offsets[e] <= p < offsets[e+1]) is a copy of
 * the codes and E8M0 bytes of one token that chose e; inside an expert the
 * tokens are in ascending order (stable).  Ragged, no padding.
 *   topk        device int32 [tokens, top_k]: the experts of each token,
 *               distinct per token, in [0, n_experts) (other ids are dropped)
 *   q, scales   device, the tokens' MXFP4 codes [tokens, cols/2] and ROWMAJOR
 *               E8M0 [tokens, cols/32]; cols % 32 == 0
 *   offsets     device int64 out [n_experts + 1]
 *   row_token   device int32 out [tokens * top_k]: token of each dispatched row
 *   q_out, scales_out  device out [tokens * top_k, cols/2], [tokens * top_k, cols/32]
 *   workspace   device, >= fp4q_moe_dispatch_workspace_bytes(), 16-byte aligned
 * Limits: 1 <= top_k <= 16, 1 <= n_experts <= 256, tokens * top_k <= 2^31 - 1
 * (else FP4Q_ERR_UNSUPPORTED_SHAPE; the workspace size is then 0).
 */
size_t fp4q_moe_dispatch_workspace_bytes(int64_t tokens, int top_k, int n_experts);
fp4q_status fp4q_moe_dispatch(const int32_t* topk, int64_t tokens, int top_k, int n_experts,
                              const uint8_t* q, const uint8_t* scales, int64_t cols,
                              int64_t* offsets, int32_t* row_token, uint8_t* q_out,
                              uint8_t* scales_out, void* workspace, size_t workspace_bytes,
                              fp4q_stream_t stream);

/*
 * fp4q_moe_dispatch_static -- fp4q_moe_dispatch for callers that cannot pass a
 * workspace.  The pages have no counterpart: this is a library convenience.
 * Who needs it: callers that cannot allocate device memory on this path --
 * processes that fix their device-memory budget at start-up and treat any
 * later allocation as an error, plain C code that only receives device
 * pointers from the framework owning the memory, and latency-sensitive loops
 * where a cudaMalloc (it can synchronize the device) is not acceptable.
 * Same arguments, results and limits as fp4q_moe_dispatch, minus the
 * workspace: the scratch is a static device array of
 * FP4Q_MOE_DISPATCH_STATIC_SCRATCH_BYTES that every GPU loading the library
 * holds until exit.  A call whose fp4q_moe_dispatch_workspace_bytes(tokens,
 * top_k, n_experts) exceeds it returns FP4Q_ERR_UNSUPPORTED_SHAPE (4 MiB covers
 * e.g. 65536 tokens x top-8 over 64 experts).  The first call on a device
 * looks up the array's device address (cudaGetSymbolAddress) with that device
 * current; make that first call before any stream capture.  The call
 * allocates nothing.  All calls share the array: calls that overlap on the GPU
 * (different streams, no ordering) race on it and give wrong results.
 */
#define FP4Q_MOE_DISPATCH_STATIC_SCRATCH_BYTES (4u * 1024u * 1024u)
fp4q_status fp4q_moe_dispatch_static(const int32_t* topk, int64_t tokens, int top_k, int n_experts,
                                     const uint8_t* q, const uint8_t* scales, int64_t cols,
                                     int64_t* offsets, int32_t* row_token, uint8_t* q_out,
                                     uint8_t* scales_out, fp4q_stream_t stream);

/*
 * fp4q_mx_rebase_scales -- MXFP4 block scales -> UE4M3 per-16 scales + a row
 * factor, so MXFP4 rows can meet NVFP4 operands in one block-scaled MMA.
 * Per row r: B_r = max_j E_j - 8; each 32-block's 2^E_j becomes the UE4M3
 * value 2^(E_j - B_r) for both 16-element halves; row_scale[r] = 2^B_r.
 * Exact when E_j >= B_r - 9 for every block; blocks below that get scale 0
 * and are counted in *violations (if non-NULL; the caller zeroes it).
 * Output in the MMA layout with every group padded to whole 128-row tiles
 * (group g's tiles follow those of groups < g); the entries of the padding
 * rows are unspecified (the GEMM's rows there are not stored).
 *   scales     device ROWMAJOR E8M0 [rows, cols/32], 4-byte aligned;  cols % 128 == 0
 *   offsets    device int64 [groups + 1] row offsets, 8-byte aligned (rows beyond
 *              offsets[groups] ignored).  The kernel clamps each offset into
 *              [previous offset, rows] (the first into [0, rows]), so offsets that
 *              decrease or exceed rows cannot make it read or write out of bounds
 *   ue4m3_mma  device out, fp4q_rebased_scales_bytes(rows, cols, groups) bytes, 16-byte aligned
 *   row_scale  device FP32 out [rows]
 * A misaligned pointer returns FP4Q_ERR_MISALIGNED.  fp4q_rebased_scales_bytes
 * returns 0 for negative sizes and for sizes whose byte count does not fit a
 * size_t.
 */
size_t fp4q_rebased_scales_bytes(int64_t rows, int64_t cols, int64_t groups);
fp4q_status fp4q_mx_rebase_scales(const uint8_t* scales, int64_t rows, int64_t cols,
                                  const int64_t* offsets, int64_t groups, uint8_t* ue4m3_mma,
                                  float* row_scale, uint32_t* violations, fp4q_stream_t stream);

typedef enum fp4q_epilogue {
    FP4Q_EPI_STORE_BF16 = 0,       /* D = BF16(acc * row_scale * tensor_scale[g])           */
    FP4Q_EPI_SILU_GATE_MXFP4 = 1   /* h = SiLU(U[:, :N/2]) * U[:, N/2:], U = acc * factors;
                                      h -> MXFP4 (codes into D, E8M0 into d_scales)         */
} fp4q_epilogue;

/*
 * fp4q_grouped_gemm -- per group g: rows offsets[g] .. offsets[g+1] of A times
 * B_g^T (the MoE expert GEMMs on tcgen05, kind::mxf4nvf4 with UE4M3 per 16).
 *   a_q            device [rows, K/2] packed codes (dispatched rows)
 *   a_scales       device, UE4M3 per 16 in the padded MMA layout of
 *                  fp4q_mx_rebase_scales (or NVFP4 scales laid out the same way)
 *   a_row_scale    device FP32 [rows]
 *   b_q            device [groups, N, K/2];  b_scales device, the groups' NVFP4
 *                  E4M3 scales in MMA layout, back to back;  b_tensor_scale
 *                  device FP32 [groups]
 *   offsets        device int64 [groups + 1], clamped by the kernel like those of
 *                  fp4q_mx_rebase_scales (each into [previous offset, rows]), so
 *                  malformed offsets cannot make it read or write out of bounds
 *   N, K           N % 128 == 0 (gated: N % 256 == 0), K % 128 == 0
 *   D              STORE_BF16: device BF16 [rows, N];  SILU_GATE: device codes
 *                  [rows, N/4] (h has N/2 columns)
 *   d_scales       SILU_GATE: device ROWMAJOR E8M0 [rows, N/64]; else unused
 *   h_debug        SILU_GATE: optional device FP32 [rows, N/2] copy of h before
 *                  quantization (NULL: not written)
 * FP32 accumulation; limits: 1 <= groups <= 256, rows, K and groups * N at
 * most 2^30, fewer than 2^31 output tiles of 128 x 256 (counting one partial
 * tile per group), else FP4Q_ERR_UNSUPPORTED_SHAPE; K == 0 is unsupported.
 */
fp4q_status fp4q_grouped_gemm(const uint8_t* a_q, const uint8_t* a_scales, const float* a_row_scale,
                              const uint8_t* b_q, const uint8_t* b_scales, const float* b_tensor_scale,
                              const int64_t* offsets, int64_t rows, int64_t groups, int64_t N,
                              int64_t K, fp4q_epilogue epilogue, void* D, uint8_t* d_scales,
                              float* h_debug, fp4q_stream_t stream);

/*
 * fp4q_device_status -- read (and, if reset != 0, clear) the device status
 * word of the current device: 0 when no device-side wait has timed out since
 * the last reset, else a bit mask of the kernels that gave up (FP4Q_ERR_TIMEOUT
 * is returned in that case): bit 0 fp4q_block_scaled_gemm (also set, with
 * D left unwritten, when the dense MXFP4 form finds its dynamic shared
 * memory starting more than 768 bytes below a 1024-byte boundary, which a
 * launch without static shared memory never does), bit 1
 * fp4q_grouped_gemm, bit 2 the shared-memory-staged conversions of
 * fp4q_mx_quantize (E4M3 source) and fp4q_fp4_to_fp8, bit 3 a tile scale
 * fp4q_fp8_tile_scales_to_e8m0 could not convert, bit 31
 * fp4q_check_wait_timeout.  Synchronous: waits for the device first.
 */
fp4q_status fp4q_device_status(uint32_t* status_out, int reset);

/*
 * fp4q_stream_status -- fp4q_device_status scoped to one stream: waits for
 * `stream` only (not the whole device), then reads the status word of the
 * current device into *status_out (optional; NULL: not written) and, if
 * reset != 0, clears it, both ordered on `stream`.  The word is per device, so
 * bits set by kernels on other streams show too.  Returns FP4Q_OK when the
 * word is 0, FP4Q_ERR_TIMEOUT when a bit is set, FP4Q_ERR_CUDA when the stream
 * cannot be waited for.  Synchronous on the host.
 */
fp4q_status fp4q_stream_status(uint32_t* status_out, int reset, fp4q_stream_t stream);

/*
 * fp4q_check_wait_timeout -- self-check of the device-side failure path.  The
 * pages have no counterpart: this is library infrastructure.  Launches one
 * thread that waits, with the same bounded mbarrier wait the GEMM kernels use,
 * on a barrier that nothing completes; after `limit_ns` (at most 2 s) it gives
 * up and sets bit 31 of the device status word, which fp4q_device_status()
 * then reports as FP4Q_ERR_TIMEOUT.  The GPU context stays usable.
 */
fp4q_status fp4q_check_wait_timeout(uint64_t limit_ns, fp4q_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* FP4Q_H */
