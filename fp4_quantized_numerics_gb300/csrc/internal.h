// internal.h -- launchers behind the libufp4 C ABI (not exported).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace ufp4 {

// Workspace layout (bytes from the start of the caller's scratch buffer).
constexpr size_t kWsStatus = 0;            // uint32 status word
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
    uint8_t *scales;
    float *tensor_scale;
    int64_t out_rows, k;       // result shape
    uint64_t elem_base;        // SR element offset (grouped segments)
};

int num_sms();

// Tensor amax (when amax_in is null) + fused quantization.  `ws` is the
// caller's workspace (status word + partial maxima).
cudaError_t launch_quantize(const QuantLaunch &q, void *ws, cudaStream_t s);

cudaError_t launch_dequantize(const uint8_t *codes, const uint8_t *scales, const float *ts,
                              int64_t rows, int64_t k, int grid, int inverse_rht,
                              uint64_t rht_seed, float *out, int64_t ld_out, cudaStream_t s);

// Writes n_ctas x 8 double partial sums to ws + kWsStats; returns n_ctas.
cudaError_t launch_stats(const QuantLaunch &q, void *ws, int *n_ctas, cudaStream_t s);

cudaError_t launch_gemm(const uint8_t *a_codes, const uint8_t *a_scales, const float *a_ts,
                        const uint8_t *b_codes, const uint8_t *b_scales, const float *b_ts,
                        int64_t M, int64_t N, int64_t K, int grid, float *c, int64_t ldc,
                        cudaStream_t s);

// Reads and clears the sticky flag that a bounded device-side wait raises
// when it gives up (synchronises s).
cudaError_t read_timeout_flag(uint32_t *flag, cudaStream_t s);
cudaError_t read_quant_timeout_flag(uint32_t *flag, cudaStream_t s);

}  // namespace ufp4
