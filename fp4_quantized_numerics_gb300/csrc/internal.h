// internal.h -- launchers behind the libufp4 C ABI (not exported).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace ufp4 {

// Workspace layout (bytes from the start of the caller's scratch buffer).
constexpr size_t kWsStatus = 0;            // uint32 status word
constexpr size_t kWsArrive = 8;            // uint32 grid-barrier counter of the single-pass quantizer
constexpr size_t kWsPartials = 256;        // float partial maxima
constexpr int kMaxPartials = 4096;
constexpr size_t kWsStats = 32768;         // double partial sums, 8 per CTA
constexpr int kMaxStatsCtas = 1024;
constexpr size_t kWorkspaceBytes = kWsStats + size_t(kMaxStatsCtas) * 8 * sizeof(double);

struct QuantLaunch {
    const void *x;
    int dtype;                 // 0 bf16, 1 fp32
    int64_t rows, cols, ld;    // input as stored
    int grid, rht, round, colwise;
    uint64_t rht_seed, sr_seed, sr_counter;
    const float *amax_in;      // device or null
    uint8_t *codes;
    uint8_t *eplane;           // E1M2 correction plane (codes' layout) or null
    uint8_t *scales;
    float *tensor_scale;
    int64_t out_rows, k;       // result shape
    uint64_t elem_base;        // SR element offset (grouped segments)
};

int num_sms();

constexpr int kMaxGroups = 256;

// Segment table of a grouped quantization (host-built, passed by value).
struct GroupQuant {
    int32_t n;
    int32_t colwise;
    int64_t in_row[kMaxGroups + 1];   // prefix sums of segment rows in x
    int64_t out_off[kMaxGroups];      // row offset (row-wise) or k offset (column-wise) in the output
    int64_t units[kMaxGroups + 1];    // prefix sums of work units (16-blocks / column-pair units)
};

// Segment table of a grouped quantization of both orientations (host-built,
// passed by value): segment e's input rows [in_row[e], in_row[e + 1]), its
// row-wise output rows from roff[e], its column-wise k range from koff[e],
// and the prefix sums of its 128 x 64 input tiles (ceil(T_e / 128) row tiles
// per segment times the column tiles).
struct GroupDual {
    int32_t n;
    int64_t in_row[kMaxGroups + 1];
    int64_t roff[kMaxGroups];
    int64_t koff[kMaxGroups];
    int64_t tiles[kMaxGroups + 1];
};

// GEMM output tile (rows of A x rows of B per CTA tile).
constexpr int kGemmBM = 128;
constexpr int kGemmBN = 256;

// One group of a grouped GEMM (host-built).
struct GroupGemm {
    int32_t M, N, nkt, ntn;           // nkt = kpad(K) / 64, ntn = ceil(N / kGemmBN)
    int32_t a_rt, a_kt, b_rt, b_kt;   // row offsets / 128, k offsets / 64
    int32_t a_seg, b_seg;
    float *c;
    int64_t ldc;
};
struct GroupGemmTab {
    int32_t n;
    int32_t tiles[kMaxGroups + 1];    // prefix sums of kGemmBM x kGemmBN tiles per group
    GroupGemm g[kMaxGroups];
};

// Tensor amax (when amax_in is null) + fused quantization.  `ws` is the
// caller's workspace (status word + partial maxima).
cudaError_t launch_quantize(const QuantLaunch &q, void *ws, cudaStream_t s);

cudaError_t launch_dequantize(const uint8_t *codes, const uint8_t *scales, const float *ts,
                              int64_t rows, int64_t k, int grid, int inverse_rht,
                              uint64_t rht_seed, float *out, int64_t ld_out, cudaStream_t s);

// Writes n_ctas x 8 double partial sums to ws + kWsStats; returns n_ctas.
cudaError_t launch_stats(const QuantLaunch &q, void *ws, int *n_ctas, cudaStream_t s);

// Quantization and the statistics of its result: one pass over x where the
// staged row-wise kernel applies (it accumulates the partial sums as it
// writes the codes), else launch_quantize then launch_stats.  Partial sums
// as launch_stats.
cudaError_t launch_quantize_stats(const QuantLaunch &q, void *ws, int *n_ctas, cudaStream_t s);

// 2-D TMA tensor map (CUtensorMap, 128 bytes) of a BF16 matrix rows x cols
// with row stride ld elements; tiles of box_cols x box_rows, no swizzle, out
// of range elements read as zero.
bool make_input_tile_map(void *tmap, const void *x, int64_t rows, int64_t cols, int64_t ld, int box_cols,
                         int box_rows);

// Row-wise (qr) and column-wise (qc) quantization of the same x in one pass
// over x (falls back to two passes when the parameters or the layout do not
// allow it).
cudaError_t launch_quantize_dual(const QuantLaunch &qr, const QuantLaunch &qc, void *ws, cudaStream_t s);

// Grouped quantization: x holds segments in row order; ws keeps one fp32
// maximum per segment and the status word.
cudaError_t launch_quantize_grouped(const QuantLaunch &q, const GroupQuant &gt, void *ws, cudaStream_t s);

// Both orientations of a grouped BF16 tensor from one read per pass (amax,
// then quantization): qr row-wise and qc column-wise, sharing grid, rounding
// and transform.  Each result equals its own launch_quantize_grouped.
cudaError_t launch_quantize_grouped_dual(const QuantLaunch &qr, const QuantLaunch &qc, const GroupDual &gd,
                                         void *ws, cudaStream_t s);

cudaError_t launch_gemm_grouped(const uint8_t *a_codes, const uint8_t *a_eplane, const uint8_t *a_scales,
                                const float *a_ts, int64_t a_rows, int64_t a_kpad, const uint8_t *b_codes,
                                const uint8_t *b_eplane, const uint8_t *b_scales, const float *b_ts,
                                int64_t b_rows, int64_t b_kpad, int grid, const GroupGemmTab &tab,
                                cudaStream_t s);

// a_eplane / b_eplane: E1M2 correction planes (same layout as the codes) or
// NULL; with both given the GEMM loads them instead of expanding on chip.
// c_amax (or NULL): set to the tensor amax of C's row-wise quantization
// (amax_rht: of the rotated C with the signs of amax_seed).
cudaError_t launch_gemm(const uint8_t *a_codes, const uint8_t *a_eplane, const uint8_t *a_scales,
                        const float *a_ts, const uint8_t *b_codes, const uint8_t *b_eplane,
                        const uint8_t *b_scales, const float *b_ts, int64_t M, int64_t N, int64_t K, int grid,
                        float *c, int64_t ldc, cudaStream_t s, float *c_amax = nullptr, int amax_rht = 0,
                        uint64_t amax_seed = 0);

// Reads and clears the sticky flag that a bounded device-side wait raises
// when it gives up (synchronises s).
cudaError_t read_timeout_flag(uint32_t *flag, cudaStream_t s);
cudaError_t read_quant_timeout_flag(uint32_t *flag, cudaStream_t s);

}  // namespace ufp4
