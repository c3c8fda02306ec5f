// api.cu -- the libufp4 C ABI: host-side validation and launch.
//
// Every entry point checks its arguments on the host and returns
// UFP4_ERR_INVALID before anything is enqueued; the library never allocates
// device memory and never synchronises except in ufp4_check / ufp4_stats,
// which return host values.
#include "../../include/ufp4.h"
#include "common.cuh"
#include "internal.h"

#include <algorithm>
#include <cmath>
#include <cstring>
#include <memory>
#include <vector>

using namespace ufp4;

namespace {

inline bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

inline ufp4_status from_cuda(cudaError_t e) {
    return e == cudaSuccess ? UFP4_OK : (e == cudaErrorNotSupported ? UFP4_ERR_UNSUPPORTED : UFP4_ERR_CUDA);
}

// Within the 32-bit indexing of the kernels (UFP4_MAX_DIM, UFP4_MAX_BLOCKS).
bool within_limits(int64_t rows, int64_t k) {
    if (rows > UFP4_MAX_DIM || k > UFP4_MAX_DIM) return false;
    if (rows <= 0 || k <= 0) return true;
    return rows <= UFP4_MAX_BLOCKS / (kpad_of(k) / 16);
}

bool valid_qtensor(const ufp4_qtensor *q) {
    if (!q || q->reserved != 0) return false;
    if (q->rows < 0 || q->k < 0 || q->k % UFP4_BLOCK != 0) return false;
    if (q->grid != UFP4_E2M1 && q->grid != UFP4_E1M2 && q->grid != UFP4_E2M1C && q->grid != UFP4_MXFP4)
        return false;
    if (q->grid == UFP4_MXFP4 && q->k % UFP4_MX_BLOCK != 0) return false;
    if (q->rows == 0 || q->k == 0) return true;
    if (!q->codes || !q->scales || !q->tensor_scale) return false;
    if (q->eplane && (q->grid != UFP4_E1M2 || !aligned(q->eplane, 16))) return false;
    return aligned(q->codes, 16) && aligned(q->scales, 16) && aligned(q->tensor_scale, 4);
}

// Shared validation of ufp4_quantize / ufp4_stats arguments.  Fills `ql`.
ufp4_status check_quant_args(const void *x, int32_t dtype, int64_t rows, int64_t cols, int64_t ld,
                             const ufp4_qparams *p, const ufp4_qtensor *out, QuantLaunch *ql) {
    if (!p || !out) return UFP4_ERR_INVALID;
    if (dtype != UFP4_BF16 && dtype != UFP4_FP32) return UFP4_ERR_INVALID;
    if (p->grid != UFP4_E2M1 && p->grid != UFP4_E1M2 && p->grid != UFP4_E2M1C && p->grid != UFP4_MXFP4)
        return UFP4_ERR_INVALID;
    if (p->block != (p->grid == UFP4_MXFP4 ? UFP4_MX_BLOCK : UFP4_BLOCK)) return UFP4_ERR_UNSUPPORTED;
    if (p->round != UFP4_RTNE && p->round != UFP4_SR) return UFP4_ERR_INVALID;
    if ((p->rht != 0 && p->rht != 1) || (p->colwise != 0 && p->colwise != 1) || p->reserved != 0)
        return UFP4_ERR_INVALID;
    if (rows < 0 || cols < 0 || ld < cols) return UFP4_ERR_INVALID;
    const int64_t out_rows = p->colwise ? cols : rows;
    const int64_t k = p->colwise ? rows : cols;
    if (p->grid == UFP4_MXFP4 && (k % UFP4_MX_BLOCK != 0 || p->amax_in)) return UFP4_ERR_INVALID;
    if (!within_limits(out_rows, k) || !within_limits(rows, cols) || ld > UFP4_MAX_DIM)
        return UFP4_ERR_UNSUPPORTED;
    if (!valid_qtensor(out) || out->grid != p->grid || out->rows != out_rows || out->k != k)
        return UFP4_ERR_INVALID;
    if (k % UFP4_BLOCK != 0) return UFP4_ERR_INVALID;
    if (p->colwise && cols % 4 != 0) return UFP4_ERR_INVALID;
    const size_t esz = dtype == UFP4_BF16 ? 2 : 4;
    if (rows > 0 && cols > 0) {
        if (!x || !aligned(x, 16) || (ld * (int64_t)esz) % 16 != 0) return UFP4_ERR_INVALID;
    }
    if (p->amax_in && !aligned(p->amax_in, 4)) return UFP4_ERR_INVALID;
    QuantLaunch q{};
    q.x = x; q.dtype = dtype; q.rows = rows; q.cols = cols; q.ld = ld;
    q.grid = p->grid; q.rht = p->rht; q.round = p->round; q.colwise = p->colwise;
    q.rht_seed = p->rht_seed; q.sr_seed = p->sr_seed; q.sr_counter = p->sr_counter;
    q.amax_in = p->amax_in;
    q.codes = out->codes; q.scales = out->scales; q.tensor_scale = out->tensor_scale;
    q.eplane = out->eplane;
    q.out_rows = out_rows; q.k = k; q.elem_base = 0;
    *ql = q;
    return UFP4_OK;
}

bool valid_workspace(const void *ws, size_t bytes) {
    return ws && aligned(ws, 16) && bytes >= kWorkspaceBytes;
}

}  // namespace

extern "C" {

int64_t ufp4_kpad(int64_t k) { return k <= 0 ? 0 : kpad_of(k); }

int64_t ufp4_codes_bytes(int64_t rows, int64_t k) {
    if (rows <= 0 || k <= 0) return 0;
    return rows * (kpad_of(k) / 2);
}

int64_t ufp4_scales_bytes(int64_t rows, int64_t k) {
    if (rows <= 0 || k <= 0) return 0;
    return rpad_of(rows) * (kpad_of(k) / 16);
}

size_t ufp4_workspace_bytes(void) { return kWorkspaceBytes; }

const char *ufp4_status_string(ufp4_status s) {
    switch (s) {
        case UFP4_OK: return "ok";
        case UFP4_ERR_INVALID: return "invalid argument";
        case UFP4_ERR_UNSUPPORTED: return "unsupported by this library";
        case UFP4_ERR_NONFINITE: return "non-finite input";
        case UFP4_ERR_CUDA: return "CUDA runtime error";
        case UFP4_ERR_TIMEOUT: return "device-side wait timed out";
    }
    return "unknown status";
}

ufp4_status ufp4_quantize(const void *x, int32_t dtype, int64_t rows, int64_t cols, int64_t ld,
                          const ufp4_qparams *p, const ufp4_qtensor *out, void *workspace,
                          size_t workspace_bytes, ufp4_stream_t stream) {
    QuantLaunch q;
    ufp4_status st = check_quant_args(x, dtype, rows, cols, ld, p, out, &q);
    if (st != UFP4_OK) return st;
    if (!p->amax_in && !valid_workspace(workspace, workspace_bytes)) return UFP4_ERR_INVALID;
    if (workspace && !aligned(workspace, 16)) return UFP4_ERR_INVALID;
    if (rows == 0 || cols == 0) return UFP4_OK;
    return from_cuda(launch_quantize(q, workspace, reinterpret_cast<cudaStream_t>(stream)));
}

ufp4_status ufp4_quantize_dual(const void *x, int32_t dtype, int64_t rows, int64_t cols, int64_t ld,
                               const ufp4_qparams *p_row, const ufp4_qparams *p_col, const ufp4_qtensor *out_row,
                               const ufp4_qtensor *out_col, void *workspace, size_t workspace_bytes,
                               ufp4_stream_t stream) {
    if (!p_row || !p_col || p_row->colwise != 0 || p_col->colwise != 1) return UFP4_ERR_INVALID;
    if (p_row->grid == UFP4_MXFP4 || p_col->grid == UFP4_MXFP4) return UFP4_ERR_UNSUPPORTED;
    QuantLaunch qr, qc;
    ufp4_status st = check_quant_args(x, dtype, rows, cols, ld, p_row, out_row, &qr);
    if (st != UFP4_OK) return st;
    st = check_quant_args(x, dtype, rows, cols, ld, p_col, out_col, &qc);
    if (st != UFP4_OK) return st;
    if ((!p_row->amax_in || !p_col->amax_in) && !valid_workspace(workspace, workspace_bytes))
        return UFP4_ERR_INVALID;
    if (workspace && !aligned(workspace, 16)) return UFP4_ERR_INVALID;
    if (rows == 0 || cols == 0) return UFP4_OK;
    return from_cuda(launch_quantize_dual(qr, qc, workspace, reinterpret_cast<cudaStream_t>(stream)));
}

ufp4_status ufp4_check(const void *workspace, ufp4_stream_t stream) {
    if (workspace && !aligned(workspace, 16)) return UFP4_ERR_INVALID;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    uint32_t timeout = 0, qtimeout = 0;
    if (read_timeout_flag(&timeout, s) != cudaSuccess) return UFP4_ERR_CUDA;
    if (read_quant_timeout_flag(&qtimeout, s) != cudaSuccess) return UFP4_ERR_CUDA;
    if (timeout || qtimeout) return UFP4_ERR_TIMEOUT;
    if (!workspace) return UFP4_OK;
    uint32_t flag = 0;
    cudaError_t e = cudaMemcpyAsync(&flag, static_cast<const char *>(workspace) + kWsStatus,
                                    sizeof flag, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return UFP4_ERR_CUDA;
    return flag ? UFP4_ERR_NONFINITE : UFP4_OK;
}

ufp4_status ufp4_dequantize(const ufp4_qtensor *q, int32_t inverse_rht, uint64_t rht_seed,
                            float *out, int64_t ld_out, ufp4_stream_t stream) {
    if (!valid_qtensor(q) || (inverse_rht != 0 && inverse_rht != 1)) return UFP4_ERR_INVALID;
    if (q->rows == 0 || q->k == 0) return UFP4_OK;
    if (!within_limits(q->rows, q->k)) return UFP4_ERR_UNSUPPORTED;
    if (!out || !aligned(out, 16) || ld_out < q->k || ld_out % 4 != 0) return UFP4_ERR_INVALID;
    return from_cuda(launch_dequantize(q->codes, q->scales, q->tensor_scale, q->rows, q->k,
                                       q->grid, inverse_rht, rht_seed, out, ld_out,
                                       reinterpret_cast<cudaStream_t>(stream)));
}

ufp4_status ufp4_gemm(const ufp4_qtensor *a, const ufp4_qtensor *b, float *c, int64_t ldc,
                      ufp4_stream_t stream) {
    if (!valid_qtensor(a) || !valid_qtensor(b)) return UFP4_ERR_INVALID;
    if (a->k != b->k) return UFP4_ERR_INVALID;
    if (a->grid != b->grid) return UFP4_ERR_UNSUPPORTED;
    const int64_t M = a->rows, N = b->rows, K = a->k;
    if (M == 0 || N == 0) return UFP4_OK;
    if (!c || !aligned(c, 16) || ldc < N || ldc % 4 != 0) return UFP4_ERR_INVALID;
    if (!within_limits(M, K) || !within_limits(N, K)) return UFP4_ERR_UNSUPPORTED;
    return from_cuda(launch_gemm(a->codes, a->eplane, a->scales, a->tensor_scale, b->codes, b->eplane, b->scales,
                                 b->tensor_scale, M, N, K, a->grid, c, ldc,
                                 reinterpret_cast<cudaStream_t>(stream)));
}

ufp4_status ufp4_gemm_amax(const ufp4_qtensor *a, const ufp4_qtensor *b, float *c, int64_t ldc, int32_t rht,
                           uint64_t rht_seed, float *c_amax, ufp4_stream_t stream) {
    if (!valid_qtensor(a) || !valid_qtensor(b)) return UFP4_ERR_INVALID;
    if (a->k != b->k || (rht != 0 && rht != 1) || !c_amax || !aligned(c_amax, 4)) return UFP4_ERR_INVALID;
    if (a->grid != b->grid || a->grid == UFP4_MXFP4) return UFP4_ERR_UNSUPPORTED;
    const int64_t M = a->rows, N = b->rows, K = a->k;
    if (rht && N % UFP4_BLOCK != 0) return UFP4_ERR_INVALID;
    if (M == 0 || N == 0) {
        return from_cuda(cudaMemsetAsync(c_amax, 0, sizeof(float), reinterpret_cast<cudaStream_t>(stream)));
    }
    if (!c || !aligned(c, 16) || ldc < N || ldc % 4 != 0) return UFP4_ERR_INVALID;
    if (!within_limits(M, K) || !within_limits(N, K)) return UFP4_ERR_UNSUPPORTED;
    return from_cuda(launch_gemm(a->codes, a->eplane, a->scales, a->tensor_scale, b->codes, b->eplane, b->scales,
                                 b->tensor_scale, M, N, K, a->grid, c, ldc,
                                 reinterpret_cast<cudaStream_t>(stream), c_amax, rht, rht_seed));
}

int64_t ufp4_grouped_rows(const int64_t *seg_rows, int32_t n_seg) {
    if (!seg_rows || n_seg <= 0) return 0;
    int64_t t = 0;
    for (int i = 0; i < n_seg; ++i) t += seg_rows[i] > 0 ? rpad_of(seg_rows[i]) : 0;
    return t;
}

int64_t ufp4_grouped_kpad(const int64_t *seg_rows, int32_t n_seg) {
    if (!seg_rows || n_seg <= 0) return 0;
    int64_t t = 0;
    for (int i = 0; i < n_seg; ++i) t += seg_rows[i] > 0 ? kpad_of(seg_rows[i]) : 0;
    return t;
}

// Validation and segment table of one grouped quantization.  `*empty` is set
// when there is nothing to write (UFP4_OK without a launch).
static ufp4_status grouped_prepare(const void *x, int32_t dtype, int64_t cols, int64_t ld,
                                   const int64_t *seg_rows, int32_t n_seg, const ufp4_qparams *p,
                                   const ufp4_qtensor *out, void *workspace, size_t workspace_bytes,
                                   GroupQuant &gt, QuantLaunch &q, bool *empty) {
    *empty = false;
    if (!p || !out || !seg_rows || n_seg < 1 || n_seg > kMaxGroups) return UFP4_ERR_INVALID;
    if (p->grid == UFP4_MXFP4) return UFP4_ERR_UNSUPPORTED;
    if (p->amax_in) return UFP4_ERR_INVALID;
    int64_t total = 0;
    for (int i = 0; i < n_seg; ++i) {
        if (seg_rows[i] < 0) return UFP4_ERR_INVALID;
        total += seg_rows[i];
    }
    // shape checks through the common validator (k = Σ kpad for column-wise)
    const int64_t kcol = ufp4_grouped_kpad(seg_rows, n_seg);
    const int64_t out_rows = p->colwise ? cols : ufp4_grouped_rows(seg_rows, n_seg);
    const int64_t k = p->colwise ? kcol : cols;
    if (!valid_qtensor(out) || out->grid != p->grid || out->rows != out_rows || out->k != k)
        return UFP4_ERR_INVALID;
    if (dtype != UFP4_BF16 && dtype != UFP4_FP32) return UFP4_ERR_INVALID;
    if (p->block != UFP4_BLOCK) return UFP4_ERR_UNSUPPORTED;
    if (p->grid != UFP4_E2M1 && p->grid != UFP4_E1M2 && p->grid != UFP4_E2M1C) return UFP4_ERR_INVALID;
    if (p->round != UFP4_RTNE && p->round != UFP4_SR) return UFP4_ERR_INVALID;
    if ((p->rht != 0 && p->rht != 1) || (p->colwise != 0 && p->colwise != 1) || p->reserved != 0)
        return UFP4_ERR_INVALID;
    if (cols < 0 || ld < cols) return UFP4_ERR_INVALID;
    if (!within_limits(out_rows, k) || !within_limits(total, cols) || ld > UFP4_MAX_DIM)
        return UFP4_ERR_UNSUPPORTED;
    if (!p->colwise && cols % UFP4_BLOCK != 0) return UFP4_ERR_INVALID;
    if (p->colwise && cols % 4 != 0) return UFP4_ERR_INVALID;
    const size_t esz = dtype == UFP4_BF16 ? 2 : 4;
    if (total > 0 && cols > 0 && (!x || !aligned(x, 16) || (ld * (int64_t)esz) % 16 != 0)) return UFP4_ERR_INVALID;
    if (!valid_workspace(workspace, workspace_bytes)) return UFP4_ERR_INVALID;
    if (kWsPartials + (size_t)n_seg * 4 > kWsStats) return UFP4_ERR_INVALID;
    if (total == 0 || cols == 0 || out_rows == 0 || k == 0) {
        *empty = true;
        return UFP4_OK;
    }
    if (total > (int64_t)INT32_MAX) return UFP4_ERR_UNSUPPORTED;

    memset(&gt, 0, sizeof gt);
    gt.n = n_seg;
    gt.colwise = p->colwise;
    const int64_t kpadc = kpad_of(cols);
    for (int i = 0; i < n_seg; ++i) {
        const int64_t T = seg_rows[i];
        gt.in_row[i + 1] = gt.in_row[i] + T;
        if (!p->colwise) {
            gt.out_off[i] = i == 0 ? 0 : gt.out_off[i - 1] + (seg_rows[i - 1] > 0 ? rpad_of(seg_rows[i - 1]) : 0);
            gt.units[i + 1] = gt.units[i] + (T > 0 ? rpad_of(T) : 0) * (kpadc / 16);
        } else {
            gt.out_off[i] = i == 0 ? 0 : gt.out_off[i - 1] + (seg_rows[i - 1] > 0 ? kpad_of(seg_rows[i - 1]) : 0);
            gt.units[i + 1] = gt.units[i] + (T > 0 ? kpad_of(T) / 16 : 0) * (cols / 2);
        }
    }
    if (gt.units[n_seg] > (int64_t)INT32_MAX * 2) return UFP4_ERR_UNSUPPORTED;
    q = QuantLaunch{};
    q.x = x; q.dtype = dtype; q.rows = total; q.cols = cols; q.ld = ld;
    q.grid = p->grid; q.rht = p->rht; q.round = p->round; q.colwise = p->colwise;
    q.rht_seed = p->rht_seed; q.sr_seed = p->sr_seed; q.sr_counter = p->sr_counter;
    q.codes = out->codes; q.scales = out->scales; q.tensor_scale = out->tensor_scale;
    q.eplane = out->eplane;
    q.out_rows = out_rows; q.k = k;
    return UFP4_OK;
}

ufp4_status ufp4_quantize_grouped(const void *x, int32_t dtype, int64_t cols, int64_t ld,
                                  const int64_t *seg_rows, int32_t n_seg, const ufp4_qparams *p,
                                  const ufp4_qtensor *out, void *workspace, size_t workspace_bytes,
                                  ufp4_stream_t stream) {
    GroupQuant gt;
    QuantLaunch q;
    bool empty = false;
    ufp4_status st = grouped_prepare(x, dtype, cols, ld, seg_rows, n_seg, p, out, workspace, workspace_bytes, gt,
                                     q, &empty);
    if (st != UFP4_OK || empty) return st;
    return from_cuda(launch_quantize_grouped(q, gt, workspace, reinterpret_cast<cudaStream_t>(stream)));
}

ufp4_status ufp4_quantize_grouped_dual(const void *x, int32_t dtype, int64_t cols, int64_t ld,
                                       const int64_t *seg_rows, int32_t n_seg, const ufp4_qparams *p_row,
                                       const ufp4_qparams *p_col, const ufp4_qtensor *out_row,
                                       const ufp4_qtensor *out_col, void *workspace, size_t workspace_bytes,
                                       ufp4_stream_t stream) {
    if (!p_row || !p_col || p_row->colwise != 0 || p_col->colwise != 1) return UFP4_ERR_INVALID;
    GroupQuant gr, gc;
    QuantLaunch qr, qc;
    bool empty_r = false, empty_c = false;
    ufp4_status st = grouped_prepare(x, dtype, cols, ld, seg_rows, n_seg, p_row, out_row, workspace,
                                     workspace_bytes, gr, qr, &empty_r);
    if (st != UFP4_OK) return st;
    st = grouped_prepare(x, dtype, cols, ld, seg_rows, n_seg, p_col, out_col, workspace, workspace_bytes, gc, qc,
                         &empty_c);
    if (st != UFP4_OK) return st;
    if (empty_r || empty_c) return UFP4_OK;   // both empty together: no rows or no columns
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const bool same = qr.grid == qc.grid && qr.round == qc.round && qr.rht == qc.rht &&
                      (!qr.rht || qr.rht_seed == qc.rht_seed);
    // one read per pass serves both for BF16 input of 128 x 64 TMA tiles; the
    // amax slots of both orientations must fit the workspace's partial area
    if (!same || dtype != UFP4_BF16 || kWsPartials + 2 * (size_t)n_seg * 4 > kWsStats) {
        cudaError_t e = launch_quantize_grouped(qr, gr, workspace, s);
        return from_cuda(e != cudaSuccess ? e : launch_quantize_grouped(qc, gc, workspace, s));
    }
    GroupDual gd;
    memset(&gd, 0, sizeof gd);
    gd.n = n_seg;
    const int64_t nct = (cols + 63) / 64;
    for (int i = 0; i < n_seg; ++i) {
        gd.in_row[i + 1] = gr.in_row[i + 1];
        gd.roff[i] = gr.out_off[i];
        gd.koff[i] = gc.out_off[i];
        gd.tiles[i + 1] = gd.tiles[i] + (seg_rows[i] + 127) / 128 * nct;
    }
    if (gd.tiles[n_seg] > (int64_t)INT32_MAX) return UFP4_ERR_UNSUPPORTED;
    return from_cuda(launch_quantize_grouped_dual(qr, qc, gd, workspace, s));
}

ufp4_status ufp4_gemm_grouped(const ufp4_qtensor *a, const ufp4_qtensor *b, const ufp4_gemm_group *groups,
                              int32_t n, ufp4_stream_t stream) {
    if (!valid_qtensor(a) || !valid_qtensor(b) || !groups || n < 0 || n > kMaxGroups) return UFP4_ERR_INVALID;
    if (a->grid != b->grid || a->grid == UFP4_MXFP4) return UFP4_ERR_UNSUPPORTED;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    std::unique_ptr<GroupGemmTab> tab(new GroupGemmTab());
    memset(tab.get(), 0, sizeof(GroupGemmTab));
    int m = 0;
    int64_t tiles = 0;
    for (int i = 0; i < n; ++i) {
        const ufp4_gemm_group &g = groups[i];
        if (g.M < 0 || g.N < 0 || g.K < 0 || g.K % UFP4_BLOCK != 0) return UFP4_ERR_INVALID;
        if (!within_limits(g.M, g.K) || !within_limits(g.N, g.K)) return UFP4_ERR_UNSUPPORTED;
        if (g.M == 0 || g.N == 0) continue;
        if (!g.c || !aligned(g.c, 16) || g.ldc < g.N || g.ldc % 4 != 0) return UFP4_ERR_INVALID;
        if (g.a_row % 128 || g.b_row % 128 || g.a_k % 64 || g.b_k % 64) return UFP4_ERR_INVALID;
        if (g.a_row < 0 || g.b_row < 0 || g.a_k < 0 || g.b_k < 0) return UFP4_ERR_INVALID;
        if (g.a_row + g.M > a->rows || g.b_row + g.N > b->rows) return UFP4_ERR_INVALID;
        if (g.a_k + g.K > kpad_of(a->k) || g.b_k + g.K > kpad_of(b->k)) return UFP4_ERR_INVALID;
        if (g.a_seg < 0 || g.b_seg < 0) return UFP4_ERR_INVALID;
        if (g.K == 0) {
            cudaError_t e = cudaMemset2DAsync(g.c, g.ldc * sizeof(float), 0, g.N * sizeof(float), g.M, s);
            if (e != cudaSuccess) return UFP4_ERR_CUDA;
            continue;
        }
        GroupGemm &t = tab->g[m];
        t.M = (int32_t)g.M; t.N = (int32_t)g.N;
        t.nkt = (int32_t)(kpad_of(g.K) / 64);
        t.ntn = (int32_t)((g.N + kGemmBN - 1) / kGemmBN);
        t.a_rt = (int32_t)(g.a_row / 128); t.a_kt = (int32_t)(g.a_k / 64);
        t.b_rt = (int32_t)(g.b_row / 128); t.b_kt = (int32_t)(g.b_k / 64);
        t.a_seg = g.a_seg; t.b_seg = g.b_seg;
        t.c = g.c; t.ldc = g.ldc;
        tiles += (int64_t)((g.M + kGemmBM - 1) / kGemmBM) * t.ntn;
        if (tiles > INT32_MAX) return UFP4_ERR_UNSUPPORTED;
        ++m;
        tab->tiles[m] = (int32_t)tiles;
    }
    tab->n = m;
    if (m == 0) return UFP4_OK;
    return from_cuda(launch_gemm_grouped(a->codes, a->eplane, a->scales, a->tensor_scale, a->rows, kpad_of(a->k),
                                         b->codes, b->eplane, b->scales, b->tensor_scale, b->rows, kpad_of(b->k),
                                         a->grid, *tab, s));
}

// Host fp64 reduction of n sets of 8 partial sums into the statistics.
static ufp4_stats_t reduce_stats(const double *part, int n) {
    double s[5] = {0, 0, 0, 0, 0};
    for (int i = 0; i < n; ++i)
        for (int j = 0; j < 5; ++j) s[j] += part[(size_t)i * 8 + j];
    ufp4_stats_t r{};
    r.sum_aq = s[0]; r.sum_aa = s[1]; r.sum_err2 = s[2]; r.bias_count = s[4];
    r.alpha = s[1] > 0 ? s[0] / s[1] : 1.0;
    r.sqnr_db = s[2] > 0 ? 10.0 * std::log10(s[1] / s[2]) : INFINITY;
    r.mean_bias = s[4] > 0 ? s[3] / s[4] : 0.0;
    return r;
}

ufp4_status ufp4_quantize_stats(const void *x, int32_t dtype, int64_t rows, int64_t cols, int64_t ld,
                                const ufp4_qparams *p, const ufp4_qtensor *out, void *workspace,
                                size_t workspace_bytes, ufp4_stats_t *host_out, ufp4_stream_t stream) {
    if (!host_out) return UFP4_ERR_INVALID;
    QuantLaunch q;
    ufp4_status st = check_quant_args(x, dtype, rows, cols, ld, p, out, &q);
    if (st != UFP4_OK) return st;
    if (!valid_workspace(workspace, workspace_bytes)) return UFP4_ERR_INVALID;
    std::vector<double> part;
    int n = 0;
    if (rows > 0 && cols > 0) {
        cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
        cudaError_t e = launch_quantize_stats(q, workspace, &n, cs);
        if (e != cudaSuccess) return from_cuda(e);
        part.resize((size_t)n * 8);
        e = cudaMemcpyAsync(part.data(), static_cast<char *>(workspace) + kWsStats, part.size() * sizeof(double),
                            cudaMemcpyDeviceToHost, cs);
        if (e == cudaSuccess) e = cudaStreamSynchronize(cs);
        if (e != cudaSuccess) return UFP4_ERR_CUDA;
    }
    *host_out = reduce_stats(part.data(), n);
    return UFP4_OK;
}

ufp4_status ufp4_stats(const void *x, int32_t dtype, int64_t rows, int64_t cols, int64_t ld,
                       const ufp4_qparams *p, const ufp4_qtensor *qt, void *workspace,
                       size_t workspace_bytes, ufp4_stats_t *host_out, ufp4_stream_t stream) {
    if (!host_out) return UFP4_ERR_INVALID;
    QuantLaunch q;
    ufp4_status st = check_quant_args(x, dtype, rows, cols, ld, p, qt, &q);
    if (st != UFP4_OK) return st;
    if (!valid_workspace(workspace, workspace_bytes)) return UFP4_ERR_INVALID;
    std::vector<double> part;
    int n = 0;
    if (rows > 0 && cols > 0) {
        cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
        cudaError_t e = launch_stats(q, workspace, &n, cs);
        if (e != cudaSuccess) return from_cuda(e);
        part.resize((size_t)n * 8);
        e = cudaMemcpyAsync(part.data(), static_cast<char *>(workspace) + kWsStats,
                            part.size() * sizeof(double), cudaMemcpyDeviceToHost, cs);
        if (e == cudaSuccess) e = cudaStreamSynchronize(cs);
        if (e != cudaSuccess) return UFP4_ERR_CUDA;
    }
    *host_out = reduce_stats(part.data(), n);
    return UFP4_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// ufp4_quantize_noalloc: ufp4_quantize for callers that cannot allocate
// device memory.  Some host programs may not call cudaMalloc at the point
// where they quantize -- a custom allocator owns all device memory, a memory
// pool is frozen after start-up, or the code runs where an allocation could
// synchronise the device.  This variant needs no caller workspace: its
// scratch (the amax pass's per-CTA partial maxima and the status word) lives
// in the file-scope array below, which every GPU that loads libufp4 holds
// until the process exits.
//
// Layout of the array: the same as the first kNoAllocBytes of a regular
// workspace -- status word at 0, up to kMaxPartials float partial maxima at
// kWsPartials.  Nothing in it has to start at zero: the amax pass writes every
// slot that the quantization pass reads, and the quantization pass writes
// the status word.  The array keeps the last call's contents, and all calls
// on a device share it, so calls whose work overlaps on the GPU (different
// streams, or different host threads without ordering) race on it.
namespace {
constexpr size_t kNoAllocBytes = kWsPartials + size_t(kMaxPartials) * sizeof(float);  // 16,640 B
// The amax pass's grid is capped at kMaxPartials CTAs (resident_grid in
// quantize.cu), one partial maximum each, so the array holds every call's
// scratch whatever the tensor's size.
static_assert(kNoAllocBytes >= kWsPartials + size_t(kMaxPartials) * sizeof(float),
              "the no-allocation scratch must hold the status word and kMaxPartials partial maxima");
static __device__ __align__(256) unsigned char g_ufp4_noalloc_scratch[kNoAllocBytes];

// Device address of the scratch array on the current device.  Host code only
// holds a stand-in for the array's name, so the address is looked up on every
// call (a cheap runtime query): nothing is cached that a device reset or a
// reload of the module could leave stale.
ufp4_status noalloc_scratch(void **out) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_ufp4_noalloc_scratch) != cudaSuccess || !p) return UFP4_ERR_CUDA;
    *out = p;
    return UFP4_OK;
}
}  // namespace

extern "C" ufp4_status ufp4_quantize_noalloc(const void *x, int32_t dtype, int64_t rows, int64_t cols,
                                             int64_t ld, const ufp4_qparams *p,
                                             const ufp4_qtensor *out, ufp4_stream_t stream) {
    QuantLaunch q;
    ufp4_status st = check_quant_args(x, dtype, rows, cols, ld, p, out, &q);
    if (st != UFP4_OK) return st;
    if (rows == 0 || cols == 0) return UFP4_OK;
    void *scratch = nullptr;
    st = noalloc_scratch(&scratch);
    if (st != UFP4_OK) return st;
    return from_cuda(launch_quantize(q, scratch, reinterpret_cast<cudaStream_t>(stream)));
}
