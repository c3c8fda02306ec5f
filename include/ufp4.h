/*
 * ufp4.h -- C ABI of libufp4, the GB300 (sm_103a) hot path of the UFP4 FP4
 * training recipe: fused Random Hadamard Transform + block-scaled 4-bit
 * quantization of GEMM operands, and block-scaled FP4 GEMMs on the tcgen05
 * tensor cores.
 *
 * Method sources (three web pages on arXiv:2606.20381, "Rethinking Shrinkage
 * Bias in LLM FP4 Pretraining: Geometric Origin, Systemic Impact, and UFP4
 * Recipe"):
 *   [ZC] zhichai.net post "Shrinkage Bias: The Hidden Geometric Trap in FP4
 *        Training ... and the UFP4 Fix" (Key points: "The cause", "Compounding
 *        decay", "The RHT paradox", "The fix -- UFP4");
 *   [AN] autonainews.com article "UFP4 Eliminates Shrinkage Bias in FP4 LLM
 *        Pretraining, Ant Group Research Finds" ("The UFP4 Recipe");
 *   [HP] hotpaper.ai card of the paper (abstract, technical approach).
 * The pages define the grids, the rounding modes and where RHT and SR apply;
 * they fix no block size, scale format, RNG, layout or interface.  The choices
 * made here (16-element blocks, E4M3 block scale, FP32 tensor scale, Philox
 * stochastic rounding, layouts below) are this library's contract.
 *
 * Conventions for every call:
 *   - All tensor pointers are DEVICE pointers unless marked "host".  The
 *     caller allocates and owns every buffer; the library never allocates,
 *     never frees, and keeps no state between calls.
 *   - Work is enqueued on `stream` and returns without synchronising, except
 *     where a call is documented to synchronise (it returns host values).
 *   - Argument errors are found on the host before anything is launched and
 *     return UFP4_ERR_INVALID (or UFP4_ERR_UNSUPPORTED for a valid request
 *     this library does not implement); a failed launch returns UFP4_ERR_CUDA.
 *     Faults inside an already-launched kernel surface through the CUDA
 *     runtime on a later synchronisation, as for any CUDA library.
 *   - Zero-sized tensors are a no-op returning UFP4_OK.
 */
#ifndef UFP4_H_
#define UFP4_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define UFP4_API __attribute__((visibility("default")))
#else
#define UFP4_API
#endif

typedef struct CUstream_st *ufp4_stream_t; /* a cudaStream_t; NULL = legacy default stream */

typedef enum {
    UFP4_OK = 0,
    UFP4_ERR_INVALID = 1,      /* bad pointer, size, alignment or enum */
    UFP4_ERR_UNSUPPORTED = 2,  /* valid request not implemented by this library */
    UFP4_ERR_NONFINITE = 3,    /* NaN/Inf input seen (reported by ufp4_check) */
    UFP4_ERR_CUDA = 4,         /* a CUDA runtime call or launch failed */
    UFP4_ERR_TIMEOUT = 5       /* a bounded device-side wait gave up */
} ufp4_status;

/* 4-bit grids.  A code is (sign << 3) | m with magnitude index m = 0..7.
 *   UFP4_E2M1:  magnitudes {0, .5, 1, 1.5, 2, 3, 4, 6} -- the non-uniform
 *               Blackwell FP4 format ([ZC] "The cause").
 *   UFP4_E1M2:  magnitudes {0, .5, 1, ..., 3.5} = m/2 -- the uniform grid of
 *               UFP4 ([ZC] "The fix -- UFP4"; [AN] "The UFP4 Recipe").
 *   UFP4_E2M1C: E2M1 clamped to its uniform part {0, .5, 1, 1.5, 2} (m <= 4,
 *               qmax = 2): the "clamp E2M1 to emulate a uniform grid"
 *               ablation that the pages report as failing ([ZC] Key points,
 *               "Validation results").  Its codes are E2M1 codes, so its
 *               GEMM is the native E2M1 one.
 *   UFP4_MXFP4: the OCP microscaling format MXFP4, a comparison format of
 *               the pages ([HP] technical approach): E2M1 elements, blocks of
 *               32 along k sharing one E8M0 scale 2^s with
 *               s = floor(log2(max |y|)) - 2 clamped to [-127, 127] (-127
 *               for an all-zero block), elements RTNE (saturating at 6) or SR
 *               of y * 2^-s, and no tensor scale (tensor_scale is written as
 *               1).  The scale byte s + 127 is stored at both of the block's
 *               16-block places of the scale layout below.  Supported by
 *               ufp4_quantize (block = UFP4_MX_BLOCK, k a multiple of 32,
 *               amax_in NULL), ufp4_dequantize, ufp4_stats and ufp4_gemm (two
 *               MXFP4 operands: the tensor cores' MXFP4 product, E2M1
 *               elements with one UE8M0 scale per 32 K-elements); the dual,
 *               grouped and GEMM-amax calls return UFP4_ERR_UNSUPPORTED.
 * A symmetric uniform INT4 grid {-7..7} needs no entry: with the same
 * two-level scaling its codes and block scales equal E1M2's bit for bit and
 * only the tensor scale (x 1/2) and the value of a code (x 2) differ. */
typedef enum { UFP4_E2M1 = 0, UFP4_E1M2 = 1, UFP4_E2M1C = 2, UFP4_MXFP4 = 3 } ufp4_grid;

/* Rounding onto the grid: round-to-nearest-even, or stochastic rounding
 * (the pages apply SR to dY only: [HP] key contributions; [ZC] "The fix"). */
typedef enum { UFP4_RTNE = 0, UFP4_SR = 1 } ufp4_round;

/* Element type of the tensor to quantize. */
typedef enum { UFP4_BF16 = 0, UFP4_FP32 = 1 } ufp4_dtype;

#define UFP4_BLOCK 16
#define UFP4_MX_BLOCK 32

/* Size limits of this library (32-bit block and tile indexing inside the
 * kernels).  A request beyond them returns UFP4_ERR_UNSUPPORTED before any
 * launch:
 *   quantize / stats / dequantize: rows, cols (k) < 2^31 and the quantized
 *   tensor's blocks, rows x kpad(k)/16, < 2^31 (about 3.4e10 elements);
 *   GEMM: M, N < 2^31 and every operand within the quantize limit. */
#define UFP4_MAX_DIM 2147483647LL
#define UFP4_MAX_BLOCKS 2147483647LL

/* Quantization parameters.
 *   grid, round  : see above.
 *   block        : must be 16 (UFP4_BLOCK); UFP4_MX_BLOCK (32) for UFP4_MXFP4.
 *   rht          : 1 = rotate every 16-block along K by y = (1/4) H16 diag(d) x
 *                  before quantizing ([ZC] "The RHT paradox"; UFP4 applies it
 *                  on all three GEMMs).  H16 is the Sylvester Hadamard matrix,
 *                  H[i][j] = (-1)^popcount(i & j); d_j = -1 iff bit j of word 0
 *                  of Philox4x32-10(key = rht_seed, counter = 0) is set.  Both
 *                  operands of a GEMM must use the same rht_seed.
 *   sr_seed, sr_counter : SR draws, for logical element i of the output
 *                  (i = row * k + col of the quantized orientation), 16 bits:
 *                  of Philox4x32-10(key = sr_seed, ctr = (i/8, sr_counter)),
 *                  word (i%8)/2, its low half for even i and its high half for
 *                  odd i; it rounds up iff bits * 2^-16 < p, p the position of
 *                  the value between its two neighbouring grid points.
 *   colwise      : 0 = 16-blocks run along the contiguous (last) dim and the
 *                  result is the quantization of X (rows x cols); 1 = blocks
 *                  run down the columns and the result is the quantization of
 *                  X^T (cols x rows), as the bwd_dx / bwd_dw GEMMs need.
 *   amax_in      : optional device pointer to the tensor amax A_t of the
 *                  (rotated) input; NULL = computed by the call.  Must be
 *                  NULL for UFP4_MXFP4 (no tensor scale).
 * Tensor scale: S_enc = fl32(448 qmax / A_t) (clamped to FLT_MAX), stored
 * S_dec = fl32(A_t / (448 qmax)); A_t = 0 gives S_enc = S_dec = 1.
 * Block scale:  e_b = E4M3_rne_satfinite(fl32(fl32(amax_b / qmax) * S_enc)).
 * Element:      q = fl32(y * fl32(S_enc / e_b)), a = min(|q|, qmax),
 *               code = signbit(q) << 3 | round(a); e_b = 0 gives code 0.   */
typedef struct {
    int32_t grid;
    int32_t block;
    int32_t rht;
    int32_t round;
    uint64_t rht_seed;
    uint64_t sr_seed;
    uint64_t sr_counter;
    int32_t colwise;
    int32_t reserved;          /* must be 0 */
    const float *amax_in;
} ufp4_qparams;

/* A quantized tensor of logical shape rows x k (16-blocks along k).
 *   kpad   = ufp4_kpad(k) = k rounded up to a multiple of 64.
 *   codes  : uint8 [rows][kpad/2]; byte j of a row holds element 2j in bits
 *            3..0 and element 2j+1 in bits 7..4 (the packed K-major FP4
 *            operand layout of the tensor cores).  Elements k..kpad-1 are 0.
 *   scales : E4M3 bytes in the tensor cores' block-scale layout: atoms of
 *            128 rows x 4 blocks (512 bytes); scale (r, b) of row r and
 *            16-block b lives at byte
 *              ((r / 128) * (kpad / 64) + b / 4) * 512
 *              + (r % 32) * 16 + ((r % 128) / 32) * 4 + (b % 4).
 *            Size ufp4_scales_bytes(rows, k); entries of rows >= rows or
 *            blocks >= k/16 are written as 0.
 *   tensor_scale : 1 fp32, S_dec.
 *   Values: x ~= v(m) * e_b * S_dec (then the inverse RHT when rht was on).
 *   eplane : optional, UFP4_E1M2 only (NULL otherwise): a buffer of the
 *            codes' size and layout holding the E1M2 correction plane.  An
 *            E1M2 value m/2 equals (R + E)/2 with R the code's nibble read as
 *            an E2M1 code and E = {0,.5,1,1.5,2,2,2,1}[m] (sign kept), stored
 *            here as E2M1 codes; a padding code 0 has E code 0.  Every
 *            quantize call that writes the tensor writes the plane too, and
 *            ufp4_gemm / ufp4_gemm_grouped load it (instead of expanding E
 *            on chip, which is slower) when both operands carry one.  The
 *            plane must stay in step with the codes: a caller that writes
 *            codes by other means sets eplane to NULL.  Costs 0.5 byte per
 *            element of device memory and of quantizer writes.
 *   Alignment: codes, scales and eplane 16-byte aligned, tensor_scale
 *   4-byte.  */
typedef struct {
    uint8_t *codes;
    uint8_t *scales;
    float *tensor_scale;
    int64_t rows;
    int64_t k;
    int32_t grid;
    int32_t reserved;          /* must be 0 */
    uint8_t *eplane;           /* E1M2 correction plane or NULL */
} ufp4_qtensor;

/* Host-side size helpers (no GPU needed): bytes of the buffers of a
 * quantized tensor in the layout above.  The pages fix no storage layout;
 * the sizes follow from the 16-element E4M3 block scaling of the NVFP4
 * recipe the pages start from ([ZC] Key points, "The symptom") and the
 * tensor cores' operand and scale layouts. */
UFP4_API int64_t ufp4_kpad(int64_t k);
UFP4_API int64_t ufp4_codes_bytes(int64_t rows, int64_t k);
UFP4_API int64_t ufp4_scales_bytes(int64_t rows, int64_t k);
/* Bytes of the scratch buffer that ufp4_quantize and ufp4_stats take (the
 * tensor amax of the two-level scaling needs every element before the first
 * code, [ZC] "The symptom"; its partial maxima live there). */
UFP4_API size_t ufp4_workspace_bytes(void);

/* Fused (RHT +) block quantization of one BF16 or FP32 matrix.
 *   x        : device, rows x cols elements of `dtype`, row stride ld
 *              elements; 16-byte aligned, ld * sizeof(elem) a multiple of 16.
 *   rows, cols: the matrix as stored.  Row-wise: cols % 16 == 0 and the
 *              result has shape rows x cols.  Column-wise: rows % 16 == 0,
 *              cols % 4 == 0 and the result has shape cols x rows.
 *   p        : host pointer to the parameters above.
 *   out      : host pointer; caller fills codes/scales/tensor_scale with
 *              device buffers and rows/k/grid with the result's shape.
 *   workspace: device scratch of workspace_bytes >= ufp4_workspace_bytes(),
 *              16-byte aligned; used when p->amax_in is NULL to hold per-CTA
 *              partial maxima and a status word (see ufp4_check).
 * ([ZC] "The fix -- UFP4"; [AN] "The UFP4 Recipe".)                        */
UFP4_API ufp4_status ufp4_quantize(const void *x, int32_t dtype, int64_t rows, int64_t cols, int64_t ld,
                          const ufp4_qparams *p, const ufp4_qtensor *out,
                          void *workspace, size_t workspace_bytes, ufp4_stream_t stream);

/* Both quantizations of one matrix that a training step needs -- row-wise
 * (blocks along the rows, result rows x cols) and column-wise (the
 * quantization of X^T, result cols x rows) -- from one read of x per pass
 * (the tensor amax pass and the quantization pass each read x once instead
 * of twice).  The three training GEMMs consume every operand in both
 * orientations ([ZC] zhichai.net post, Key points "The fix -- UFP4": the
 * transform and quantization are applied to the operands of fwd_y, bwd_dx
 * and bwd_dw).
 *   p_row, out_row: as for ufp4_quantize with p_row->colwise == 0;
 *   p_col, out_col: as for ufp4_quantize with p_col->colwise == 1;
 *   x, dtype, rows, cols, ld, workspace: as for ufp4_quantize, and every
 *   constraint of both orientations applies.
 * Each result is bit-identical to its own ufp4_quantize call (own tensor
 * scale, amax_in, SR seed and counter).  One pass serves both when the two
 * parameter sets share grid, rounding mode and transform (seed included)
 * and cols * sizeof(elem) is a multiple of 16; otherwise the call runs the
 * two quantizations one after the other.  The non-finite flag in the
 * workspace covers both. */
UFP4_API ufp4_status ufp4_quantize_dual(const void *x, int32_t dtype, int64_t rows, int64_t cols, int64_t ld,
                                        const ufp4_qparams *p_row, const ufp4_qparams *p_col,
                                        const ufp4_qtensor *out_row, const ufp4_qtensor *out_col,
                                        void *workspace, size_t workspace_bytes, ufp4_stream_t stream);

/* ufp4_quantize without a caller workspace, for callers that cannot
 * allocate device memory when they quantize (a frozen memory pool, a custom
 * allocator that owns all device memory, code that must not risk an
 * allocation's implicit synchronisation).  The paper has no counterpart:
 * this is a deployment convenience of this library.
 * Arguments and results are exactly those of ufp4_quantize, minus the
 * workspace.  Its scratch -- the amax pass's partial maxima and a status
 * word, 16,640 bytes -- is a fixed array inside the library that every GPU
 * using libufp4 holds until the process exits.  The array always fits: the
 * amax pass never launches more than 4096 CTAs, one partial maximum each,
 * whatever the tensor's size, so no size is refused for lack of scratch.
 * Every call looks up the array's device address on the current device
 * (cudaGetSymbolAddress; a failure returns UFP4_ERR_CUDA), so a device reset
 * between calls leaves nothing stale.  All calls on a device share
 * the array and it keeps the last call's contents: calls that overlap on the
 * GPU (other streams, unordered host threads) race and give wrong results.
 * Allocates nothing.  The non-finite status of this variant is not
 * reported (use ufp4_quantize with a workspace and ufp4_check for that). */
UFP4_API ufp4_status ufp4_quantize_noalloc(const void *x, int32_t dtype, int64_t rows, int64_t cols,
                                           int64_t ld, const ufp4_qparams *p, const ufp4_qtensor *out,
                                           ufp4_stream_t stream);

/* Reports device-side problems (synchronises `stream`).  The pages have no
 * counterpart: this is the library's failure reporting for the kernels of
 * the calls above.  Returns the first that applies:
 *   UFP4_ERR_TIMEOUT   -- a bounded wait inside a GEMM kernel gave up since
 *                         the last check (the flag is then cleared); that
 *                         GEMM's output is unspecified;
 *   UFP4_ERR_NONFINITE -- the last ufp4_quantize that used `workspace` saw a
 *                         NaN/Inf input (computed-amax path) or a non-finite
 *                         amax_in; its outputs are unspecified.
 * `workspace` may be NULL to check only the timeout flag. */
UFP4_API ufp4_status ufp4_check(const void *workspace, ufp4_stream_t stream);

/* Dequantization: the value a code stands for under the two-level scaling,
 * v(m) the grid value of its magnitude index ([ZC] Key points, "The cause"
 * for E2M1, "The fix -- UFP4" for E1M2), then, optionally, the inverse of
 * the orthonormal transform ([ZC] "The RHT paradox").
 * out[r][c] = v(m) * e_b * S_dec as fp32, computed as fl32(fl32(v e_b) S_dec);
 * with inverse_rht = 1, each 16-block is then rotated back with the signs of
 * rht_seed: x = diag(d) (1/4) H16 y.  out: device fp32, q->rows x q->k, row
 * stride ld_out >= q->k elements, 16-byte aligned, ld_out % 4 == 0. */
UFP4_API ufp4_status ufp4_dequantize(const ufp4_qtensor *q, int32_t inverse_rht, uint64_t rht_seed,
                            float *out, int64_t ld_out, ufp4_stream_t stream);

/* C = A B^T with FP32 accumulation: A is M x K, B is N x K (both quantized
 * along K, same grid), C is M x N fp32 row-major with row stride ldc.
 *   C[m][n] = S_A S_B sum_k (v_A e_A)(v_B e_B)
 * This is fwd_y (Y = X W^T: A = X rows, B = W rows), bwd_dx (dX = dY W:
 * A = dY rows, B = W columns) or bwd_dw (dW = dY^T X: A = dY columns,
 * B = X columns) ([ZC] "The fix -- UFP4"; [HP] technical approach).
 * E2M1 runs natively on tcgen05 block-scaled FP4 MMAs; E1M2 runs as the
 * exact split into two E2M1 planes per operand (R, the codes, and E, the
 * correction plane): four MMAs per K step.  The E planes are loaded from
 * a->eplane and b->eplane when both are given, else expanded from the codes
 * in shared memory (slower); both give the same result bit for bit.
 * Requirements: a->k == b->k, a->grid == b->grid; c 16-byte aligned,
 * ldc >= N and ldc % 4 == 0.  K = 0 writes zeros. */
UFP4_API ufp4_status ufp4_gemm(const ufp4_qtensor *a, const ufp4_qtensor *b, float *c, int64_t ldc,
                      ufp4_stream_t stream);

/* ufp4_gemm fused with the first step of quantizing its output.  The pages'
 * compounding chain re-quantizes every layer's output for the next layer
 * ([ZC] Key points, "Compounding decay"); the tensor amax of that
 * quantization needs all of C, so a plain GEMM leaves it to a second read of
 * C.  This call writes C exactly as ufp4_gemm does and, from the epilogue's
 * registers, the amax A_t that ufp4_quantize would compute for the row-wise
 * quantization of C with parameters rht / rht_seed: max |C| (rht = 0), or
 * max over C's 16-blocks along N of |(1/4) H16 diag(d) block| (rht = 1),
 * with the quantizer's own fp32 butterflies in its order.  Passing c_amax as
 * that quantization's amax_in gives bit for bit the codes, scales and tensor
 * scale of the unfused call, with C read once instead of twice.
 *   c_amax : device, 1 float, 4-byte aligned; overwritten (the call zeroes
 *            it on `stream`, then the kernel raises it); NaN if C holds one.
 *   rht    : 0 or 1; with rht = 1, N % 16 == 0.
 * Other arguments and requirements as ufp4_gemm. */
UFP4_API ufp4_status ufp4_gemm_amax(const ufp4_qtensor *a, const ufp4_qtensor *b, float *c, int64_t ldc,
                                    int32_t rht, uint64_t rht_seed, float *c_amax, ufp4_stream_t stream);

/* ---------------------------------------------------------------------
 * Grouped (mixture-of-experts) tensors.  The tokens routed to expert e form a
 * segment of T_e consecutive rows of x ([sum T_e] x cols); every segment has
 * its own tensor scale.  Segment layouts inside one quantized tensor:
 *   row-wise  (blocks along cols): segment e occupies rows
 *             [roff_e, roff_e + T_e) with roff_e = sum_{e'<e} round_up(T_e', 128),
 *             so every segment starts on a scale-atom boundary; the tensor
 *             has rows = ufp4_grouped_rows(...) and k = cols.
 *   column-wise (blocks down the tokens, the quantization of x_e^T): segment e
 *             occupies k range [koff_e, koff_e + T_e) with
 *             koff_e = sum_{e'<e} round_up(T_e', 64); the token dimension of
 *             each segment is zero-padded to a multiple of 16; rows = cols and
 *             k = ufp4_grouped_kpad(...).
 * The qtensor's tensor_scale points to n_seg floats (S_dec per segment).
 * Stochastic rounding indexes elements by their position in the whole
 * output tensor (row * k + col), so no two segments share a random word.
 * ([HP] technical approach: MoE 7.9B and 124B models; [ZC] Validation
 * results.) */
UFP4_API int64_t ufp4_grouped_rows(const int64_t *seg_rows_host, int32_t n_seg);
UFP4_API int64_t ufp4_grouped_kpad(const int64_t *seg_rows_host, int32_t n_seg);
#define UFP4_MAX_GROUPS 256

/* Grouped quantization of x (device, [sum seg_rows] x cols, row stride ld).
 * seg_rows_host: host array of n_seg >= 1 segment row counts (0 allowed),
 * n_seg <= UFP4_MAX_GROUPS.  p->colwise selects the layout above; p->amax_in
 * must be NULL (every segment's amax is computed).  out: rows/k as above,
 * tensor_scale -> n_seg floats.  workspace: ufp4_workspace_bytes(), 16-byte
 * aligned (holds the per-segment maxima and the status word). */
UFP4_API ufp4_status ufp4_quantize_grouped(const void *x, int32_t dtype, int64_t cols, int64_t ld,
                                           const int64_t *seg_rows_host, int32_t n_seg,
                                           const ufp4_qparams *p, const ufp4_qtensor *out,
                                           void *workspace, size_t workspace_bytes,
                                           ufp4_stream_t stream);

/* Both grouped quantizations of x that an MoE layer's training step needs --
 * row-wise (p_row->colwise == 0, the row-wise grouped layout above) and
 * column-wise (p_col->colwise == 1, the column-wise grouped layout) -- from
 * one read of x per pass: an amax pass that takes every segment's maxima of
 * both orientations, then one quantization pass writing both results.  The
 * three grouped GEMMs consume every operand in both orientations ([ZC]
 * zhichai.net post, Key points "The fix -- UFP4": the transform and
 * quantization on the fwd_y, bwd_dx and bwd_dw operands; [HP] technical
 * approach: the MoE models).
 * Arguments as for ufp4_quantize_grouped, one parameter set and one result
 * per orientation; every constraint of both orientations applies (cols % 16
 * == 0).  Each result is bit-identical to its own ufp4_quantize_grouped call
 * (own per-segment tensor scales, SR seed and counter).  The one-read path
 * serves BF16 input when the two parameter sets share grid, rounding mode
 * and transform (seed included); otherwise the call runs the two grouped
 * quantizations one after the other.  The workspace holds both
 * orientations' per-segment maxima (2 * n_seg floats) and the non-finite
 * status, which covers both results.  The pages have no dual-orientation
 * call of their own; this one reorders reads, not arithmetic. */
UFP4_API ufp4_status ufp4_quantize_grouped_dual(const void *x, int32_t dtype, int64_t cols, int64_t ld,
                                                const int64_t *seg_rows_host, int32_t n_seg,
                                                const ufp4_qparams *p_row, const ufp4_qparams *p_col,
                                                const ufp4_qtensor *out_row, const ufp4_qtensor *out_col,
                                                void *workspace, size_t workspace_bytes, ufp4_stream_t stream);

/* One GEMM per group, C_g = A_g B_g^T, in a single launch.  A group's
 * operands are views of two quantized tensors a and b (same grid):
 *   A_g = rows [a_row[g], a_row[g] + M[g]) and k range [a_k[g], a_k[g] + K[g]) of a,
 *   B_g = rows [b_row[g], b_row[g] + N[g]) and k range [b_k[g], b_k[g] + K[g]) of b,
 * with tensor scales a->tensor_scale[a_seg[g]] and b->tensor_scale[b_seg[g]].
 * Row offsets must be multiples of 128 and k offsets multiples of 64 (the
 * grouped layouts above guarantee both).  C_g: device fp32 pointer c[g] with
 * row stride ldc[g] (% 4 == 0, 16-byte aligned); K[g] = 0 writes zeros,
 * M[g] = 0 or N[g] = 0 does nothing.  All arrays are host arrays of n groups,
 * n <= UFP4_MAX_GROUPS.  The three training GEMMs of an MoE layer map onto
 * this with the grouped layouts: fwd_y (A = X rows, B = W rows), bwd_dx
 * (A = dY rows, B = W^T segments along k), bwd_dw (A = dY^T and B = X^T, both
 * sharing the segment's k range). */
typedef struct {
    int64_t M, N, K;
    int64_t a_row, a_k, b_row, b_k;
    int32_t a_seg, b_seg;
    float *c;
    int64_t ldc;
} ufp4_gemm_group;

UFP4_API ufp4_status ufp4_gemm_grouped(const ufp4_qtensor *a, const ufp4_qtensor *b,
                                       const ufp4_gemm_group *groups, int32_t n,
                                       ufp4_stream_t stream);

/* Quality of one quantization, in fp64 on the host ([ZC] "The cause",
 * "Compounding decay", "The RHT paradox").  A is the tensor that was
 * quantized (x, rotated when p->rht; transposed when p->colwise):
 *   alpha = <deq, A> / <A, A>       (shrinkage factor; < 1 pulls to zero)
 *   sqnr_db = 10 log10(<A, A> / ||A - deq||^2)
 *   mean_bias = mean over elements with a != 0 of (v(m) - a), grid units,
 *               a = min(|A| / (e_b S_dec), qmax); blocks with e_b = 0 skipped.
 * x, dtype, rows, cols, ld, p: exactly as given to ufp4_quantize for q.
 * Synchronises `stream`; host_out is a host pointer. */
typedef struct {
    double alpha;
    double sqnr_db;
    double mean_bias;
    double sum_aq;
    double sum_aa;
    double sum_err2;
    double bias_count;
} ufp4_stats_t;

UFP4_API ufp4_status ufp4_stats(const void *x, int32_t dtype, int64_t rows, int64_t cols, int64_t ld,
                       const ufp4_qparams *p, const ufp4_qtensor *q,
                       void *workspace, size_t workspace_bytes,
                       ufp4_stats_t *host_out, ufp4_stream_t stream);

/* ufp4_quantize and ufp4_stats of its result in one call: the quantization
 * kernel accumulates the statistics' partial sums as it writes the codes, so
 * x is read once for both, where the layout allows it (row-wise, contiguous
 * input: ld == cols); otherwise the call runs the two one after the other.
 * The pages track the shrinkage factor and SQNR of every quantization ([ZC]
 * "The cause", "Compounding decay", "The RHT paradox").  Arguments as
 * ufp4_quantize (out receives the quantization) plus host_out as ufp4_stats.
 * The quantized tensor is bit for bit ufp4_quantize's; the statistics equal
 * ufp4_stats's up to the order of the fp32 partial sums.  Synchronises
 * `stream`. */
UFP4_API ufp4_status ufp4_quantize_stats(const void *x, int32_t dtype, int64_t rows, int64_t cols, int64_t ld,
                                         const ufp4_qparams *p, const ufp4_qtensor *out,
                                         void *workspace, size_t workspace_bytes,
                                         ufp4_stats_t *host_out, ufp4_stream_t stream);

/* Static description of a status code (no counterpart on the pages). */
UFP4_API const char *ufp4_status_string(ufp4_status s);

#ifdef __cplusplus
}
#endif

#endif /* UFP4_H_ */
