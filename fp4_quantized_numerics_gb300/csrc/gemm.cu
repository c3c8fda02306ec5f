// gemm.cu -- block-scaled FP4 GEMM C = A B^T on the sm_100-family tcgen05
// tensor cores (hand-written PTX: TMA, mbarriers, TMEM, tcgen05.mma).
//
// The three training GEMMs of the recipe (fwd_y, bwd_dx, bwd_dw) consume the
// quantized operands ([ZC] zhichai.net post "Shrinkage Bias: The Hidden
// Geometric Trap in FP4 Training ... and the UFP4 Fix", Key points, "The fix
// -- UFP4"; [HP] hotpaper.ai card, technical approach).  Both operands are
// K-major packed 4-bit codes with one E4M3 scale per 16 K-elements and one
// FP32 tensor scale:  C[m][n] = S_A S_B sum_k (v_A e_A)(v_B e_B).
//
// E2M1: the codes ARE the tensor cores' E2M1 elements and the block scales
//   are UE4M3 scale_vec::4X factors, so each 64-wide K step is one
//   tcgen05.mma.kind::mxf4nvf4.block_scale.
// E1M2: not a tensor-core format.  Read as an E2M1 code, an E1M2 nibble m has
//   the value R(m) in {0,.5,1,1.5,2,3,4,6}; the E1M2 value m/2 equals
//   (R(m) + E(m)) / 2 with E(m) in {0,.5,1,1.5,2,2,2,1}, also E2M1.  The raw
//   tile is therefore used as it was loaded, the E plane of each operand is
//   either loaded (the quantizer wrote it beside the codes) or written by
//   expander warps, and four MMAs (R*R, R*E, E*R, E*E) with the shared block
//   scales accumulate 4 * A B^T, the factor 1/4 being applied (exactly) in
//   the epilogue.
//
// CTA tile 128 x 256 (one M=128, N=256 MMA per K step); the K stage depth
// and the rings differ per grid (Cfg below).  Warp 0 = TMA producer, warp 1
// = TMEM owner + single-thread MMA issuer, warps 2-9 = epilogue (two per TMEM
// lane quadrant, 128 columns each), warp 10 = scale copies (E2M1, E1M2 with
// loaded planes) or warps 10-15 = expanders (E1M2 without planes).  The
// accumulator (256 TMEM columns) is single-buffered: the epilogue pulls the
// whole tile out (registers and shared staging) and hands the columns back
// before it stores, so the stores overlap the next tile's MMAs.  Block scales
// are staged in TMEM after the accumulator, 12 columns per MMA K step.  Every
// wait is bounded: on timeout the kernel raises g_ufp4_timeout, drains its
// own copies, frees TMEM and returns.
#include "common.cuh"
#include "internal.h"
#include "ptx.cuh"

#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstring>
#include <mutex>
#include <type_traits>

namespace ufp4 {

__device__ uint32_t g_ufp4_timeout;

namespace {

constexpr int BM = kGemmBM, BN = kGemmBN;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kSfCol = 256;                   // accumulator in [0, 256), scales after
constexpr int kEpiWarps = 8;
constexpr long long kWaitBudget = 2000000000LL;

// Kernel variants (the template argument GRID): kE2M1 (also clamped E2M1,
// whose codes are E2M1 codes), kE1M2 (E planes expanded on chip) and kE1M2Pl
// (E1M2 whose E planes the quantizer wrote next to the codes).
constexpr int kE1M2Pl = 3;
// MXFP4 operands: E2M1 codes like kE2M1, one UE8M0 scale per 32 elements
// (stored at both of its 16-block places); the MMA takes scale_vec::2X.
constexpr int kMX = 4;

// Per-variant pipeline geometry.
//  E2M1: K stage of 128 bytes (4 MMA K steps, 128-byte swizzle) so that the
//        issuing thread's per-stage wait/commit latency stays below the
//        stage's tensor-core time; 4 stages (the epilogue stages 8-column
//        pieces through 1 KB per warp to make room).
//  E1M2: K stage of 64 bytes (2 K steps, 64-byte swizzle, 8 MMAs); a 3-deep
//        ring of raw tiles fed by TMA and a 3-slot ring of E planes written
//        by six expander warps (16 warps in all: the 128 registers a thread
//        then gets still hold the epilogue's accumulator chunks).
//  E1M2Pl: the same 8 MMAs per 64-byte stage, all four tiles (R_A, R_B,
//        E_A, E_B) loaded by TMA into a 4-deep ring (the epilogue stages
//        16-column halves through 2 KB per warp to make room); scale copies
//        from their own warps as for E2M1.
template <int GRID>
struct Cfg {
    static constexpr bool kFour = GRID == kE1M2 || GRID == kE1M2Pl;  // E1M2: 4 MMAs per K step
    static constexpr bool kE2M1Like = GRID == kE2M1 || GRID == kMX;  // one MMA per K step
    static constexpr bool kPl = GRID == kE1M2Pl;                     // E planes loaded by TMA
    // columns of a staged TMA-store box: E1M2Pl stages 16-column pieces
    // through a 2 KB buffer per epilogue warp, E2M1 8-column pieces through
    // 1 KB, which leaves room for a 4th operand stage
    static constexpr int kEpiCols = kPl ? 16 : (kE2M1Like ? 8 : 32);
    static constexpr uint32_t kEpiBufBytes = 32u * kEpiCols * 4u;
    static constexpr int kBK = kE2M1Like ? 128 : 64;                 // bytes of K per stage
    static constexpr int kKS = kBK / 32;                             // MMA K steps per stage
    static constexpr uint32_t kSwz = kBK == 128 ? 2 : 4;             // descriptor swizzle: 128B / 64B
    static constexpr uint32_t kSbo = 8 * kBK;                        // 8-row core-matrix group stride
    static constexpr uint32_t kABytes = BM * kBK, kBBytes = BN * kBK;
    static constexpr uint32_t kSfaBytes = kKS * 512;                 // one 128-row atom per K step
    static constexpr uint32_t kSfbBytes = 2 * kKS * 512;             // two 128-row halves
    static constexpr uint32_t kSfColsPerStage = 12 * kKS;            // SFA 4 + SFB 8 columns per K step
    static constexpr int kStages = GRID == kE1M2 ? 3 : 4;
    static constexpr int kESlots = GRID == kE1M2 ? 3 : 0;
    static constexpr int kExpWarps = GRID == kE1M2 ? 6 : 0;
    // E2M1 and E1M2Pl: one extra warp issues the block-scale copies
    // Block-scale copies cost their issuing thread ~45 cycles each: E2M1 and
    // MXFP4 need 12 per 512-cycle stage, more than one warp can issue, so two
    // warps take alternate stages (E2M1 4.2 -> 4.8 PFLOP/s, MXFP4 3.3 -> 4.6
    // at fwd_y of the MoE-124B layer); E1M2Pl, 6 per 1024 cycles, gains ~1 %
    // from the second.  A third warp would cap the registers below what the
    // epilogue holds.
    static constexpr int kScaleWarps = GRID == kE1M2 ? 0 : 2;
    static constexpr int kThreads = 32 * (2 + kEpiWarps + kScaleWarps + kExpWarps);
    // epilogue staging buffers (32 rows x kEpiCols fp32) per epilogue warp
    static constexpr int kEpiBufs = GRID == kE1M2 ? 2 : 1;
    // stage layout: A | B | (E1M2Pl: E_A | E_B) | SFA | SFB;  E slots: E_A | E_B
    static constexpr uint32_t kPlaneBytes = kPl ? kABytes + kBBytes : 0;
    static constexpr uint32_t kAOff = 0;
    static constexpr uint32_t kBOff = kABytes;
    static constexpr uint32_t kEAOff = kABytes + kBBytes;
    static constexpr uint32_t kEBOff = kEAOff + kABytes;
    static constexpr uint32_t kSfaOff = kABytes + kBBytes + kPlaneBytes;
    static constexpr uint32_t kSfbOff = kSfaOff + kSfaBytes;
    static constexpr uint32_t kStageBytes = kSfbOff + kSfbBytes;     // multiple of 1024
    static constexpr uint32_t kESlotBytes = kABytes + kBBytes;
    static constexpr uint32_t kEOff = kStages * kStageBytes;
    static constexpr uint32_t kEpiOff = kEOff + kESlots * kESlotBytes;
    static constexpr uint32_t kBarOff = kEpiOff + kEpiWarps * kEpiBufs * kEpiBufBytes;
    static constexpr uint32_t kSmemBytes = kBarOff + 256 + 1024;   // + barriers + alignment slack
    static_assert(kStageBytes % 1024 == 0 && kESlotBytes % 1024 == 0, "tile alignment");
    static_assert(kSmemBytes <= 232448, "shared memory per CTA");
    static_assert(kSfCol + kStages * kSfColsPerStage <= kTmemCols, "TMEM columns");
};

struct GemmParams {
    const uint8_t *sfa, *sfb;
    const float *ts_a, *ts_b;
    float *c;
    int64_t ldc;
    int M, N;
    int nkt;      // kpad / 64: scale atoms per 128-row tile
    int num_kb;   // ceil(nkt / K steps per stage): K stages per tile
    int ntm, ntn; // tiles along M and N
    int nkt_a, nkt_b;  // k atoms per 128-row tile of the whole A / B tensors
    int b_rt;     // 128-row scale tiles in the whole B tensor
    long long budget;  // clock cycles a role waits for another before it gives up
    int stall;         // test-only build: the MMA thread waits on a barrier nobody arrives on
    int splits;        // K halves per output tile (1 or 2); 2: partial sums added into a zeroed C
    int col_major;     // tile order: 1 = down the M tiles first (when M < N), 0 = along the N tiles first
    float *c_amax;     // or null: raised to the tensor amax of C's row-wise quantization
    int amax_rht;      // ... of the rotated C (16-blocks along N)
    uint64_t amax_seed;
};

// Where one output tile lives: operand rows / k atoms in the A and B tensors,
// its problem's sizes, output pointer and tensor scales.
struct TileInfo {
    int a_row, b_row, a_kt, b_kt, nkt, num_kb;
    int kb0, kb1;   // the K stages [kb0, kb1) of this work unit
    int m_loc, n_loc, M, N;
    float *c;
    int64_t ldc;
    const float *ts_a, *ts_b;
};

struct NoGroups {};
// A plain GEMM whose epilogue also raises the tensor amax of C's row-wise
// quantization (its own kernel, so the plain GEMM carries none of that code).
struct NoGroupsAmax : NoGroups {};

// Work unit u of a dense GEMM: K part u / tiles (outermost, so that one
// round of the persistent grid covers twice the tiles of a K half), then the
// tile, numbered along the dimension whose operand is smaller: a round of
// CTAs then shares the bigger operand's few tiles through L2 and re-reads only
// the smaller one (row-major tiles when M >= N, column-major when M < N).
template <int KS>
__device__ __forceinline__ TileInfo tile_info(const GemmParams &p, const NoGroups &, int u) {
    TileInfo ti;
    const int ntiles = p.ntm * p.ntn;
    const int part = u / ntiles, t = u - part * ntiles;
    const int per = (p.num_kb + p.splits - 1) / p.splits;
    ti.kb0 = part * per;
    ti.kb1 = min(p.num_kb, ti.kb0 + per);
    const int mt = p.col_major ? t % p.ntm : t / p.ntn;
    const int nt = p.col_major ? t / p.ntm : t % p.ntn;
    ti.m_loc = mt * BM;
    ti.n_loc = nt * BN;
    ti.a_row = ti.m_loc;
    ti.b_row = ti.n_loc;
    ti.a_kt = 0;
    ti.b_kt = 0;
    ti.nkt = p.nkt;
    ti.num_kb = p.num_kb;
    ti.M = p.M;
    ti.N = p.N;
    ti.c = p.c;
    ti.ldc = p.ldc;
    ti.ts_a = p.ts_a;
    ti.ts_b = p.ts_b;
    return ti;
}

template <int KS>
__device__ __forceinline__ TileInfo tile_info(const GemmParams &p, const GroupGemmTab &tab, int t) {
    int lo = 0, hi = tab.n;   // largest g with tiles[g] <= t
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (tab.tiles[mid] <= t) lo = mid; else hi = mid;
    }
    const GroupGemm &g = tab.g[lo];
    const int lt = t - tab.tiles[lo];
    TileInfo ti;
    ti.m_loc = (lt / g.ntn) * BM;
    ti.n_loc = (lt % g.ntn) * BN;
    ti.a_row = g.a_rt * 128 + ti.m_loc;
    ti.b_row = g.b_rt * 128 + ti.n_loc;
    ti.a_kt = g.a_kt;
    ti.b_kt = g.b_kt;
    ti.nkt = g.nkt;
    ti.num_kb = (g.nkt + KS - 1) / KS;
    ti.kb0 = 0;
    ti.kb1 = ti.num_kb;
    ti.M = g.M;
    ti.N = g.N;
    ti.c = g.c;
    ti.ldc = g.ldc;
    ti.ts_a = p.ts_a + g.a_seg;
    ti.ts_b = p.ts_b + g.b_seg;
    return ti;
}

__device__ __forceinline__ void raise_timeout() { atomicOr(&g_ufp4_timeout, 1u); }

// Epilogue amax: the running maximum over 16 consecutive output values of a
// row, c_j = (acc_j * kfix) * alpha exactly as stored.  Without the transform
// max |c_j|; with it max |4 y| for y = (1/4) H16 diag(d) c, computed with the
// same fp32 butterflies in the same order as the quantizer's row-wise path
// (pairs (c_j, c_{j+8}), index bits 0..2 on f32x2, then the halves), so that
// 0.25 * the maximum is bit for bit the tensor amax that ufp4_quantize of C
// would compute.  NaN propagates.
__device__ __forceinline__ float max_nan2(float a, float b) {
    float r;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
    return r;
}
__device__ __forceinline__ float out_block_amax(const uint32_t *w, float kfix, float alpha, bool rht,
                                                uint32_t smask, float m) {
    float c[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) c[j] = __uint_as_float(w[j]) * kfix * alpha;
    if (!rht) {
#pragma unroll
        for (int j = 0; j < 16; ++j) m = max_nan2(m, fabsf(c[j]));
        return m;
    }
    float a[8], b[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        a[j] = __uint_as_float(__float_as_uint(c[j]) ^ (((smask >> j) & 1u) << 31));
        b[j] = __uint_as_float(__float_as_uint(c[j + 8]) ^ (((smask >> (j + 8)) & 1u) << 31));
    }
#pragma unroll
    for (int st = 1; st < 8; st <<= 1) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            if ((j & st) == 0) {
                const float a0 = a[j], a1 = a[j + st], b0 = b[j], b1 = b[j + st];
                a[j] = __fadd_rn(a0, a1);
                a[j + st] = __fsub_rn(a0, a1);
                b[j] = __fadd_rn(b0, b1);
                b[j + st] = __fsub_rn(b0, b1);
            }
        }
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        m = max_nan2(m, fabsf(__fadd_rn(a[j], b[j])));
        m = max_nan2(m, fabsf(__fsub_rn(a[j], b[j])));
    }
    return m;
}

// Warp maximum of the lanes' running maxima into *dst (a non-negative float,
// or NaN, as int bits: the order of non-negative IEEE floats is that of their
// bit patterns).
__device__ __forceinline__ void flush_amax(float *dst, float m, bool rht, int lane) {
#pragma unroll
    for (int o = 16; o; o >>= 1) m = max_nan2(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (lane == 0) {
        const float v = rht ? m * 0.25f : m;
        atomicMax(reinterpret_cast<int *>(dst), v != v ? 0x7FFFFFFF : __float_as_int(v));
    }
}

// Bounded wait that also gives up as soon as another role has aborted.
__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity, volatile int *abort,
                                              long long budget) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (true) {
#pragma unroll 1
        for (int i = 0; i < 64; ++i)
            if (ptx::mbar_try_wait(bar, parity)) return true;
        if (*abort) return false;
        if (clock64() - t0 > budget) {
            *abort = 1;
            raise_timeout();
            return false;
        }
    }
}

// Persistent CTA: tiles t = blockIdx.x, blockIdx.x + gridDim.x, ... in
// row-major (M, N) tile order; the K ring is carried across tiles.
template <int GRID, class TAB>
__global__ void __launch_bounds__(Cfg<GRID>::kThreads, 1)
    k_gemm(const __grid_constant__ CUtensorMap tma_a, const __grid_constant__ CUtensorMap tma_b,
           const __grid_constant__ CUtensorMap tma_ea, const __grid_constant__ CUtensorMap tma_eb,
           const __grid_constant__ CUtensorMap tma_c, GemmParams p, const __grid_constant__ TAB tab) {
    constexpr bool kGrouped = std::is_same<TAB, GroupGemmTab>::value;
    constexpr bool kAmax = std::is_same<TAB, NoGroupsAmax>::value;
    using C = Cfg<GRID>;
    constexpr int S = C::kStages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::kBarOff);
    constexpr int ES = C::kESlots > 0 ? C::kESlots : 1;
    // bars: [0,S) full, [S,2S) empty, [2S,2S+ES) E slot written, [2S+ES,2S+2ES)
    // E slot free, then acc full, acc empty, MMA drained, then [.., +S) scales
    // of a stage issued to the tensor cores, then the scale copies drained
    constexpr int kNBars = 3 * S + 2 * ES + 4;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + kNBars);
    volatile int *abort = reinterpret_cast<volatile int *>(tmem_slot + 1);
    static_assert(kNBars * 8 + 8 <= 256, "barrier area");
    const uint32_t smem_base = ptx::smem_u32(smem);
    const uint32_t bar_base = ptx::smem_u32(bars);
    auto full = [&](int s) { return bar_base + 8u * s; };
    auto empty = [&](int s) { return bar_base + 8u * (S + s); };
    auto expd = [&](int e) { return bar_base + 8u * (2 * S + e); };
    auto efree = [&](int e) { return bar_base + 8u * (2 * S + ES + e); };
    const uint32_t accf = bar_base + 8u * (2 * S + 2 * ES);
    const uint32_t acce = accf + 8u;
    const uint32_t drained = accf + 16u;
    auto sfr = [&](int s) { return accf + 24u + 8u * s; };
    const uint32_t sfd = accf + 24u + 8u * S;
    constexpr uint32_t kSW = C::kScaleWarps > 0 ? C::kScaleWarps : 1;   // stage stride of a scale warp

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int ntiles;
    if constexpr (kGrouped) ntiles = tab.tiles[tab.n];
    else ntiles = p.ntm * p.ntn * p.splits;   // work units

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            ptx::mbar_init(full(s), 1);
            ptx::mbar_init(empty(s), 1);
            ptx::mbar_init(sfr(s), 1);
        }
        for (int e = 0; e < ES; ++e) {
            ptx::mbar_init(expd(e), GRID == kE1M2 ? C::kExpWarps : 1);   // one arrival per expander warp
            ptx::mbar_init(efree(e), 1);
        }
        ptx::mbar_init(accf, 1);
        ptx::mbar_init(acce, kEpiWarps);   // one arrival per epilogue warp
        ptx::mbar_init(drained, 1);
        ptx::mbar_init(sfd, C::kScaleWarps > 0 ? C::kScaleWarps : 1);   // one commit per scale warp
        *abort = 0;
        ptx::fence_mbar_init();
        ptx::prefetch_tmap(&tma_a);
        ptx::prefetch_tmap(&tma_b);
        if (C::kPl) {
            ptx::prefetch_tmap(&tma_ea);
            ptx::prefetch_tmap(&tma_eb);
        }
        ptx::prefetch_tmap(&tma_c);
    }
    if (warp == 1) {
        ptx::tmem_alloc(ptx::smem_u32(tmem_slot), kTmemCols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    // Block-scale copies of stage s into its TMEM columns: SFA 4 columns per
    // K step at [0, 4 KS), SFB 8 columns per K step (rows 0-127, then
    // 128-255) at [4 KS, 12 KS).  E2M1, MXFP4 and E1M2 with loaded planes
    // issue them from two warps of their own, alternate stages each, so that
    // their issue overlaps the MMAs' (sfr(s) says they are issued); E1M2 with
    // expanded planes issues them in line from the MMA thread.
    auto copy_scales = [&](uint32_t s, int atoms, bool signal) {
        const uint64_t hi_sf = ptx::sdesc(0, 0, 128, 0);   // 32 rows x 16 B scale atom
        const uint32_t st = smem_base + s * C::kStageBytes;
        const uint64_t dsa = hi_sf | (uint64_t)(((st + C::kSfaOff) & 0x3FFFFu) >> 4);
        const uint64_t dsb = hi_sf | (uint64_t)(((st + C::kSfbOff) & 0x3FFFFu) >> 4);
        const uint32_t sf_t = tmem + kSfCol + C::kSfColsPerStage * s;
        const uint32_t sfa0 = sf_t, sfb0 = sf_t + 4u * C::kKS;
        ptx::tc_fence_after();
        for (int j = 0; j < atoms; ++j) {
            ptx::tc_cp_32x128b_warpx4(sfa0 + 4u * j, dsa + 32u * j);
            ptx::tc_cp_32x128b_warpx4(sfb0 + 8u * j, dsb + 32u * j);
            ptx::tc_cp_32x128b_warpx4(sfb0 + 8u * j + 4u, dsb + 32u * (C::kKS + j));
        }
        if (signal) {
            // Copies and the MMAs that read their columns form a pipelined
            // pair in the tensor cores: ordered across threads by the fence
            // before this arrival and the MMA thread's fence after its wait,
            // so the MMAs need not wait for the copies to complete.
            ptx::tc_fence_before();
            ptx::mbar_arrive(sfr(s));
        }
    };
    // Every copy the scale thread issued must complete before TMEM is freed:
    // one commit tracks them all.
    auto drain_scales = [&]() {
        ptx::tc_commit(sfd);   // (with nothing issued it arrives at once)
        const long long t0 = clock64();
        while (!ptx::mbar_try_wait(sfd, 0))
            if (clock64() - t0 > kWaitBudget) { raise_timeout(); break; }
    };

    if (warp == 0) {
        // ---------------------------------------------------------- producer
        if (lane == 0) {
            uint32_t g = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x) {
                const TileInfo ti = tile_info<C::kKS>(p, tab, t);
                // the B tile's second 128 rows have scales only inside the tensor
                const bool b_hi = ti.b_row / 128 + 1 < p.b_rt;
                for (int kb = ti.kb0; kb < ti.kb1; ++kb, ++g) {
                    const uint32_t s = g % S, round = g / S;
                    if (round > 0 && !wait_or_abort(empty(s), (round - 1) & 1, abort, p.budget)) { ok = false; break; }
                    const uint32_t atoms = (uint32_t)min(C::kKS, ti.nkt - C::kKS * kb);
                    const uint32_t st = smem_base + s * C::kStageBytes;
                    ptx::mbar_arrive_expect_tx(full(s), C::kABytes + C::kBBytes + C::kPlaneBytes +
                                                            atoms * 512u * (b_hi ? 3u : 2u));
                    ptx::tma_load_2d(st + C::kAOff, &tma_a, ti.a_kt * 32 + kb * C::kBK, ti.a_row, full(s));
                    ptx::tma_load_2d(st + C::kBOff, &tma_b, ti.b_kt * 32 + kb * C::kBK, ti.b_row, full(s));
                    if (C::kPl) {
                        ptx::tma_load_2d(st + C::kEAOff, &tma_ea, ti.a_kt * 32 + kb * C::kBK, ti.a_row, full(s));
                        ptx::tma_load_2d(st + C::kEBOff, &tma_eb, ti.b_kt * 32 + kb * C::kBK, ti.b_row, full(s));
                    }
                    ptx::bulk_load(st + C::kSfaOff,
                                   p.sfa + ((size_t)(ti.a_row / 128) * p.nkt_a + ti.a_kt + C::kKS * kb) * 512,
                                   atoms * 512u, full(s));
                    const uint8_t *sfb =
                        p.sfb + ((size_t)(ti.b_row / 128) * p.nkt_b + ti.b_kt + C::kKS * kb) * 512;
                    ptx::bulk_load(st + C::kSfbOff, sfb, atoms * 512u, full(s));
                    if (b_hi)
                        ptx::bulk_load(st + C::kSfbOff + C::kKS * 512u, sfb + (size_t)p.nkt_b * 512, atoms * 512u,
                                       full(s));
                }
            }
            // every copy this thread started has landed before the CTA exits
            for (uint32_t h = g > (uint32_t)S ? g - S : 0; h < g; ++h) {
                const long long t0 = clock64();
                while (!ptx::mbar_try_wait(full(h % S), (h / S) & 1))
                    if (clock64() - t0 > kWaitBudget) { raise_timeout(); break; }
            }
        }
    } else if (warp == 1) {
        // --------------------------------------------------------- MMA issuer
        // One thread issues every MMA of the CTA; descriptors are built once
        // per stage and advanced by integer adds (address field = bytes >> 4).
        if (lane == 0) {
            // instruction descriptor, kind::mxf4nvf4: A/B E2M1 (1), K-major,
            // N >> 3 at [17,23), UE4M3 scales (bit 23 = 0), M >> 4 at [24,29).
            const uint32_t idesc = (1u << 7) | (1u << 10) | ((uint32_t)(BN >> 3) << 17) |
                                   (GRID == kMX ? (1u << 23) : 0u) |   // UE8M0 scales for MXFP4
                                   ((uint32_t)(BM >> 4) << 24);
            const uint64_t hi_op = ptx::sdesc(0, 16, C::kSbo, C::kSwz);   // swizzled K-major operand
            auto mk = [](uint64_t hi, uint32_t addr) { return hi | (uint64_t)((addr & 0x3FFFFu) >> 4); };
            uint32_t g = 0, it = 0;
            bool ok = true;
#ifdef UFP4_PROBE
            // test-only build: a wait that nothing ends ("drained" is committed
            // only below), so the timeout path runs
            if (p.stall && !wait_or_abort(drained, 0u, abort, p.budget)) ok = false;
#endif
            for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x, ++it) {
                const TileInfo ti = tile_info<C::kKS>(p, tab, t);
                // the epilogue must have read the previous tile out of the accumulator
                if (it > 0 && !wait_or_abort(acce, (it - 1) & 1, abort, p.budget)) { ok = false; break; }
                ptx::tc_fence_after();
                for (int kb = ti.kb0; kb < ti.kb1; ++kb, ++g) {
                    const uint32_t s = g % S, round = g / S;
                    const uint32_t e = g % ES, eround = g / ES;
                    // operands landed and (scale warp) scales in TMEM
                    if (!wait_or_abort(full(s), round & 1, abort, p.budget) ||
                        (C::kScaleWarps > 0 && !wait_or_abort(sfr(s), round & 1, abort, p.budget))) { ok = false; break; }
                    ptx::tc_fence_after();
                    const int atoms = min(C::kKS, ti.nkt - C::kKS * kb);
                    if constexpr (GRID == kE1M2) {
                        // scale copies queued while the expanders finish the E planes
                        copy_scales(s, atoms, false);
                        if (!wait_or_abort(expd(e), eround & 1, abort, p.budget)) { ok = false; break; }
                        ptx::tc_fence_after();
                    }
                    const uint32_t st = smem_base + s * C::kStageBytes;
                    const uint32_t es = smem_base + C::kEOff + e * C::kESlotBytes;
                    const uint32_t sf_t = tmem + kSfCol + C::kSfColsPerStage * s;
                    const uint64_t da = mk(hi_op, st + C::kAOff), db = mk(hi_op, st + C::kBOff);
                    const uint64_t dea = mk(hi_op, C::kPl ? st + C::kEAOff : es);
                    const uint64_t deb = mk(hi_op, C::kPl ? st + C::kEBOff : es + C::kABytes);
                    const uint32_t sfa0 = sf_t, sfb0 = sf_t + 4u * C::kKS;
                    // E1M2 per K step: R*R, R*E, E*R, E*E, each A plane read
                    // from shared memory once and reused by the next MMA from
                    // the tensor core's collector
                    using ptx::CollA;
                    auto mma = [&](auto u, uint64_t a, uint64_t b, int j, uint32_t acc) {
                        ptx::tc_mma_nvf4<decltype(u)::value>(tmem, a + 2u * (uint32_t)j, b + 2u * (uint32_t)j, idesc,
                                                             sfa0 + 4u * j, sfb0 + 8u * j, acc);
                    };
                    using None = std::integral_constant<CollA, CollA::kNone>;
                    using Fill = std::integral_constant<CollA, CollA::kFill>;
                    using Last = std::integral_constant<CollA, CollA::kLastUse>;
                    auto first = [&](int j) { return (kb == ti.kb0 && j == 0) ? 0u : 1u; };
#pragma unroll
                    for (int j = 0; j < C::kKS; ++j) {
                        if (j >= atoms) break;
                        if constexpr (C::kFour) {
                            mma(Fill{}, da, db, j, first(j));
                            mma(Last{}, da, deb, j, 1u);
                            mma(Fill{}, dea, db, j, 1u);
                            mma(Last{}, dea, deb, j, 1u);
                        } else if constexpr (GRID == kMX) {
                            ptx::tc_mma_mxf4(tmem, da + 2u * (uint32_t)j, db + 2u * (uint32_t)j, idesc, sfa0 + 4u * j,
                                             sfb0 + 8u * j, first(j));
                        } else {
                            mma(None{}, da, db, j, first(j));
                        }
                    }
                    ptx::tc_commit(empty(s));
                    if (GRID == kE1M2) ptx::tc_commit(efree(e));
                }
                if (ok) ptx::tc_commit(accf);   // fires once this tile's MMAs have completed
            }
            // TMEM is freed below only after every MMA issued here has finished.
            ptx::tc_commit(drained);
            const long long t0 = clock64();
            while (!ptx::mbar_try_wait(drained, 0))
                if (clock64() - t0 > kWaitBudget) { raise_timeout(); break; }
        }
    } else if (warp < 2 + kEpiWarps) {
        // ------------------------------------------------------------ epilogue
        // Each warp owns 32 accumulator rows x 128 columns (four 32 x 32
        // chunks), handed back to the MMA warp once read out of TMEM; the
        // values leave through swizzled shared staging as TMA stores (whole
        // lines; ragged edges clipped by the tensor map), or, for grouped
        // problems, as masked row-coalesced stores from the staging buffer.
        // E2M1 / E1M2Pl: all four chunks into registers, then 8- / 16-column
        // pieces through one small buffer.  E1M2: the first kEpiBufs chunks
        // staged before the hand-back, the rest held in registers.
        constexpr int NB = C::kEpiBufs;
        const int q = warp & 3;                  // TMEM lane quadrant of this warp
        const int ew = warp - 2;
        const int h = ew >> 2;                   // column half of the tile
        const uint32_t buf0 = smem_base + C::kEpiOff + (uint32_t)ew * NB * C::kEpiBufBytes;
        // E1M2 accumulates (R + E)(R + E) = 4 A B^T
        const float kfix = C::kFour ? 0.25f : 1.0f;
        const uint32_t smask = (kAmax && p.amax_rht) ? rht_sign_mask(p.amax_seed) : 0u;
        const uint32_t taddr = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(128 * h);
        uint32_t it = 0;
        for (int t = blockIdx.x; t < ntiles; t += gridDim.x, ++it) {
            bool ok = wait_or_abort(accf, it & 1, abort, p.budget);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            ptx::tc_fence_after();
            const TileInfo ti = tile_info<C::kKS>(p, tab, t);
            const float alpha = __fmul_rn(*ti.ts_a, *ti.ts_b);
            const int m0 = ti.m_loc + 32 * q, n0 = ti.n_loc + 128 * h;
            if constexpr (C::kEpiCols < 32) {
                // all four chunks into registers, accumulator handed back, then
                // kEpiCols-column pieces through one staging buffer (rows of
                // 4 kEpiCols bytes, swizzled as the output map) and TMA stores
                // of 32 x kEpiCols boxes
                uint32_t v[4][32];
#pragma unroll
                for (int ch = 0; ch < 4; ++ch) ptx::tc_ld_32x32b_x32(taddr + 32u * ch, v[ch]);
                ptx::tc_wait_ld();
                ptx::tc_fence_before();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(acce);
                if constexpr (kAmax) {
                    // rows and columns outside C hold zeros (zero-filled operands)
                    float am = 0.0f;
#pragma unroll
                    for (int blk = 0; blk < 8; ++blk)
                        am = out_block_amax(&v[blk >> 1][(blk & 1) * 16], kfix, alpha, p.amax_rht != 0, smask, am);
                    flush_amax(p.c_amax, am, p.amax_rht != 0, lane);
                }
                constexpr int EC = C::kEpiCols, RB = 4 * EC, NC = RB / 16;   // row bytes, 16-byte pieces
                const uint32_t rowb = buf0 + (uint32_t)lane * RB;
                const uint32_t sw = (uint32_t)(lane * RB / 128) & (NC - 1);  // swizzle of this row
#pragma unroll
                for (int hc = 0; hc < 128 / EC; ++hc) {
                    // the previous store has read the buffer
                    if (!kGrouped && lane == 0) ptx::bulk_wait_read<0>();
                    __syncwarp();
#pragma unroll
                    for (int c = 0; c < NC; ++c) {
                        const uint32_t *w = &v[(hc * EC) / 32][(hc * EC) % 32 + 4 * c];
                        const uint32_t addr = rowb + (uint32_t)((c ^ sw) << 4);
                        asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr),
                                     "f"(__uint_as_float(w[0]) * kfix * alpha),
                                     "f"(__uint_as_float(w[1]) * kfix * alpha),
                                     "f"(__uint_as_float(w[2]) * kfix * alpha),
                                     "f"(__uint_as_float(w[3]) * kfix * alpha)
                                     : "memory");
                    }
                    if constexpr (!kGrouped) {
                        ptx::fence_proxy_async();
                        __syncwarp();
                        if (lane == 0) {
                            const int col = n0 + EC * hc;
                            if (m0 < ti.M && col < ti.N) {
                                if (p.splits > 1) ptx::tma_reduce_add_2d(&tma_c, col, m0, buf0);
                                else ptx::tma_store_2d(&tma_c, col, m0, buf0);
                            }
                            ptx::bulk_commit();
                        }
                    } else {
                        // grouped: masked, row-coalesced stores within the group's bounds
                        __syncwarp();
                        constexpr int LPR = EC / 4, RPI = 32 / LPR;   // lanes per row, rows per pass
                        const int pc = lane % LPR;
#pragma unroll
                        for (int it = 0; it < LPR; ++it) {
                            const int rr = it * RPI + lane / LPR;
                            const uint32_t swr = (uint32_t)(rr * RB / 128) & (NC - 1);
                            float4 o;
                            asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                                         : "=f"(o.x), "=f"(o.y), "=f"(o.z), "=f"(o.w)
                                         : "r"(buf0 + (uint32_t)rr * RB + ((pc ^ swr) << 4))
                                         : "memory");
                            const int row = m0 + rr, col = n0 + EC * hc + 4 * pc;
                            if (row < ti.M && col < ti.N) {
                                float *cp = ti.c + (int64_t)row * ti.ldc + col;
                                if (col + 4 <= ti.N) {
                                    *reinterpret_cast<float4 *>(cp) = o;
                                } else {
                                    cp[0] = o.x;
                                    if (col + 1 < ti.N) cp[1] = o.y;
                                    if (col + 2 < ti.N) cp[2] = o.z;
                                }
                            }
                        }
                        __syncwarp();
                    }
                }
                continue;
            } else {
            auto stage = [&](uint32_t b, const uint32_t (&v)[32]) {
                if constexpr (kAmax) {
                    float am = out_block_amax(&v[0], kfix, alpha, p.amax_rht != 0, smask, 0.0f);
                    am = out_block_amax(&v[16], kfix, alpha, p.amax_rht != 0, smask, am);
                    flush_amax(p.c_amax, am, p.amax_rht != 0, lane);
                }
                const uint32_t rowb = b + (uint32_t)lane * 128u;
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const uint32_t addr = rowb + (uint32_t)((c ^ (lane & 7)) << 4);
                    asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr),
                                 "f"(__uint_as_float(v[4 * c]) * kfix * alpha),
                                 "f"(__uint_as_float(v[4 * c + 1]) * kfix * alpha),
                                 "f"(__uint_as_float(v[4 * c + 2]) * kfix * alpha),
                                 "f"(__uint_as_float(v[4 * c + 3]) * kfix * alpha)
                                 : "memory");
                }
            };
            auto flush = [&](uint32_t b, int ch) {
                if constexpr (!kGrouped) {
                    ptx::fence_proxy_async();
                    __syncwarp();
                    // one bulk group per chunk, empty for boxes wholly outside C, so
                    // that the wait_group.read counts below see every chunk
                    if (lane == 0) {
                        if (m0 < p.M && n0 + 32 * ch < p.N) {
                            if (p.splits > 1) ptx::tma_reduce_add_2d(&tma_c, n0 + 32 * ch, m0, b);
                            else ptx::tma_store_2d(&tma_c, n0 + 32 * ch, m0, b);
                        }
                        ptx::bulk_commit();
                    }
                } else {
                    __syncwarp();
                    const int col = n0 + 32 * ch + 4 * (lane & 7);
#pragma unroll
                    for (int i = 0; i < 32; i += 4) {
                        const int rr = i + (lane >> 3), row = m0 + rr;
                        float4 v;
                        asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                                     : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                                     : "r"(b + (uint32_t)rr * 128u + (uint32_t)(((lane & 7) ^ (rr & 7)) << 4))
                                     : "memory");
                        if (row < ti.M && col < ti.N) {
                            float *cp = ti.c + (int64_t)row * ti.ldc + col;
                            if (col + 4 <= ti.N) {
                                *reinterpret_cast<float4 *>(cp) = v;
                            } else {
                                cp[0] = v.x;
                                if (col + 1 < ti.N) cp[1] = v.y;
                                if (col + 2 < ti.N) cp[2] = v.z;
                            }
                        }
                    }
                    __syncwarp();
                }
            };
            // the previous tile's stores must be done reading the staging buffers
            if (!kGrouped && lane == 0) ptx::bulk_wait_read<0>();
            __syncwarp();
#pragma unroll
            for (int ch = 0; ch < NB; ++ch) {
                uint32_t v[32];
                ptx::tc_ld_32x32b_x32(taddr + 32u * ch, v);
                ptx::tc_wait_ld();
                stage(buf0 + 4096u * ch, v);
            }
            uint32_t rest[4 - NB][32];
#pragma unroll
            for (int ch = NB; ch < 4; ++ch) ptx::tc_ld_32x32b_x32(taddr + 32u * ch, rest[ch - NB]);
            ptx::tc_wait_ld();
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(acce);   // accumulator fully read
#pragma unroll
            for (int ch = 0; ch < NB; ++ch) flush(buf0 + 4096u * ch, ch);
#pragma unroll
            for (int ch = NB; ch < 4; ++ch) {
                const uint32_t b = buf0 + 4096u * (ch % NB);
                if (!kGrouped && lane == 0) ptx::bulk_wait_read<NB - 1>();
                __syncwarp();
                stage(b, rest[ch - NB]);
                flush(b, ch);
            }
            }
        }
        if (lane == 0) ptx::bulk_wait_all();
        __syncwarp();
    } else if (GRID == kMX && warp >= 2 + kEpiWarps && warp < 2 + kEpiWarps + C::kScaleWarps) {
        // ---------------------------------------- MXFP4 scale repack + copies
        // A staged scale word holds one row's four 16-block places of a K step,
        // (s0, s0, s1, s1) for its two 32-blocks; scale_vec::2X reads the K
        // step's two scales from bytes 0 and 1, so the whole warp rewrites
        // each word to (s0, s1, s1, s1) before lane 0 copies it to TMEM.
        // The scale warps take alternate stages.
        const uint32_t sw = (uint32_t)(warp - 2 - kEpiWarps);
        uint32_t g = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x) {
            const TileInfo ti = tile_info<C::kKS>(p, tab, t);
            for (int kb = ti.kb0; kb < ti.kb1; ++kb, ++g) {
                if (g % kSW != sw) continue;
                const uint32_t s = g % S, round = g / S;
                ok = __all_sync(0xffffffffu, wait_or_abort(full(s), round & 1, abort, p.budget));
                if (!ok) break;
                // SFA | SFB are contiguous: 16 bytes per lane and step, all of a
                // lane's loads in flight before its first store
                const uint32_t st = smem_base + s * C::kStageBytes + C::kSfaOff + 16u * (uint32_t)lane;
                constexpr int kPer = (int)((C::kSfaBytes + C::kSfbBytes) / (16 * 32));
                static_assert((C::kSfaBytes + C::kSfbBytes) % (16 * 32) == 0, "whole 16-byte steps per lane");
                uint32_t v[kPer][4];
#pragma unroll
                for (int i = 0; i < kPer; ++i)
                    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                                 : "=r"(v[i][0]), "=r"(v[i][1]), "=r"(v[i][2]), "=r"(v[i][3])
                                 : "r"(st + 512u * (uint32_t)i));
#pragma unroll
                for (int i = 0; i < kPer; ++i) {
#pragma unroll
                    for (int j = 0; j < 4; ++j) asm("prmt.b32 %0, %0, 0, 0x3320;" : "+r"(v[i][j]));
                    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(st + 512u * (uint32_t)i),
                                 "r"(v[i][0]), "r"(v[i][1]), "r"(v[i][2]), "r"(v[i][3])
                                 : "memory");
                }
                ptx::fence_proxy_async();   // the rewritten bytes, to the tensor cores' copies
                __syncwarp();
                if (lane == 0) copy_scales(s, min(C::kKS, ti.nkt - C::kKS * kb), true);
                __syncwarp();
            }
        }
        if (lane == 0) drain_scales();
    } else if (C::kScaleWarps > 0 && warp >= 2 + kEpiWarps && warp < 2 + kEpiWarps + C::kScaleWarps) {
        // ------------------------------------------------- E2M1 scale copies
        // (two warps, alternate stages)
        const uint32_t sw = (uint32_t)(warp - 2 - kEpiWarps);
        if (lane == 0) {
            uint32_t g = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x) {
                const TileInfo ti = tile_info<C::kKS>(p, tab, t);
                for (int kb = ti.kb0; kb < ti.kb1; ++kb, ++g) {
                    if (g % kSW != sw) continue;
                    const uint32_t s = g % S, round = g / S;
                    if (!wait_or_abort(full(s), round & 1, abort, p.budget)) { ok = false; break; }
                    copy_scales(s, min(C::kKS, ti.nkt - C::kKS * kb), true);
                }
            }
            drain_scales();
        }
    } else if constexpr (GRID == kE1M2) {
        // ------------------------------------------------- E1M2 expanders
        // E planes of the staged A | B tiles, 16 bytes per thread and step;
        // the swizzle is a byte permutation within rows, so the elementwise
        // plane keeps the tile's layout.
        const int et = threadIdx.x - 32 * (2 + kEpiWarps);
        constexpr int kExpThreads = 32 * C::kExpWarps;
        uint32_t g = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x) {
            const TileInfo ti = tile_info<C::kKS>(p, tab, t);
            for (int kb = ti.kb0; kb < ti.kb1; ++kb, ++g) {
                const uint32_t s = g % S, round = g / S;
                const uint32_t e = g % ES, eround = g / ES;
                ok = wait_or_abort(full(s), round & 1, abort, p.budget);
                // the MMAs that last read this E slot have completed
                if (ok && eround > 0) ok = wait_or_abort(efree(e), (eround - 1) & 1, abort, p.budget);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                const uint4 *src = reinterpret_cast<const uint4 *>(smem + s * C::kStageBytes + C::kAOff);
                uint4 *dst = reinterpret_cast<uint4 *>(smem + C::kEOff + e * C::kESlotBytes);
#pragma unroll 4
                for (int i = et; i < (int)(C::kESlotBytes / 16); i += kExpThreads) {
                    const uint4 w = src[i];
                    dst[i] = make_uint4(e1m2_eplane(w.x), e1m2_eplane(w.y), e1m2_eplane(w.z), e1m2_eplane(w.w));
                }
                // generic-proxy writes -> visible to the tensor cores (async proxy)
                ptx::fence_proxy_async();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(expd(e));
            }
        }
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, kTmemCols);
    }
}

// ------------------------------------------------------------ host side
// Wait budget of the GEMM roles (and the test-only stall switch); a test-only
// build of the library can change them, libufp4 keeps the defaults.
long long g_wait_budget = kWaitBudget;
int g_stall = 0;

PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    });
    return fn;
}

// K-major packed codes, rows x kpad/2 bytes; box = one K stage x box_rows
// rows, swizzled as the MMA operand descriptors expect.
bool make_code_map(CUtensorMap *m, const uint8_t *codes, int64_t rows, int64_t kpad, int box_rows, int bk) {
    auto enc = get_encode();
    if (!enc) return false;
    cuuint64_t dims[2] = {(cuuint64_t)(kpad / 2), (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)(kpad / 2)};
    cuuint32_t box[2] = {(cuuint32_t)bk, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t *>(codes), dims, strides, box,
                     estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     bk == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Output map: boxes of 32 rows x box_cols fp32 (32, 16, 8: rows of 128,
// 64, 32 bytes), swizzled like the epilogue's staging buffers.
bool make_out_map(CUtensorMap *m, float *c, int64_t M, int64_t N, int64_t ldc, int box_cols) {
    auto enc = get_encode();
    if (!enc) return false;
    cuuint64_t dims[2] = {(cuuint64_t)N, (cuuint64_t)M};
    cuuint64_t strides[1] = {(cuuint64_t)(ldc * 4)};
    cuuint32_t box[2] = {(cuuint32_t)box_cols, 32};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, c, dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE,
                     box_cols == 32 ? CU_TENSOR_MAP_SWIZZLE_128B
                                    : (box_cols == 16 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_32B),
                     CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

template <int GRID, class TAB>
cudaError_t run_gemm(const CUtensorMap &ma, const CUtensorMap &mb, const CUtensorMap &mea, const CUtensorMap &meb,
                     const CUtensorMap &mc, const GemmParams &p, const TAB &tab, int ntiles, cudaStream_t s) {
    using C = Cfg<GRID>;
    static bool attr_set[64] = {false};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && !attr_set[dev]) {
        cudaError_t e = cudaFuncSetAttribute(k_gemm<GRID, TAB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)C::kSmemBytes);
        if (e != cudaSuccess) return e;
        attr_set[dev] = true;
    }
    const int sms = num_sms();
    const int grid = ntiles < sms ? ntiles : sms;
    if (grid <= 0) return cudaSuccess;
    k_gemm<GRID, TAB><<<grid, C::kThreads, C::kSmemBytes, s>>>(ma, mb, mea, meb, mc, p, tab);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gemm(const uint8_t *a_codes, const uint8_t *a_eplane, const uint8_t *a_scales,
                        const float *a_ts, const uint8_t *b_codes, const uint8_t *b_eplane,
                        const uint8_t *b_scales, const float *b_ts, int64_t M, int64_t N, int64_t K, int grid,
                        float *c, int64_t ldc, cudaStream_t s, float *c_amax, int amax_rht, uint64_t amax_seed) {
    if (c_amax) {
        // the epilogue raises it from zero (and a K = 0 product is all zeros)
        cudaError_t e = cudaMemsetAsync(c_amax, 0, sizeof(float), s);
        if (e != cudaSuccess) return e;
    }
    if (K == 0) return cudaMemset2DAsync(c, ldc * sizeof(float), 0, N * sizeof(float), M, s);
    const int64_t kpad = kpad_of(K);
    const bool planes = grid == kE1M2 && a_eplane && b_eplane;
    // K bytes per stage of the kernel that runs: the tensor maps' box width
    const int bk = planes ? Cfg<kE1M2Pl>::kBK : (grid == kE1M2 ? Cfg<kE1M2>::kBK : Cfg<kE2M1>::kBK);
    static_assert(Cfg<kMX>::kBK == Cfg<kE2M1>::kBK && Cfg<kMX>::kEpiCols == Cfg<kE2M1>::kEpiCols, "MX = E2M1 geometry");
    CUtensorMap ma, mb, mea, meb, mc;
    if (!make_code_map(&ma, a_codes, M, kpad, BM, bk) || !make_code_map(&mb, b_codes, N, kpad, BN, bk) ||
        !make_out_map(&mc, c, M, N, ldc,
                      planes ? Cfg<kE1M2Pl>::kEpiCols : (grid == kE1M2 ? Cfg<kE1M2>::kEpiCols : Cfg<kE2M1>::kEpiCols)))
        return cudaErrorInvalidValue;
    if (planes) {
        if (!make_code_map(&mea, a_eplane, M, kpad, BM, bk) || !make_code_map(&meb, b_eplane, N, kpad, BN, bk))
            return cudaErrorInvalidValue;
    } else {
        mea = ma;   // unused
        meb = mb;
    }
    GemmParams p{};
    p.sfa = a_scales; p.sfb = b_scales; p.ts_a = a_ts; p.ts_b = b_ts;
    p.c = c; p.ldc = ldc; p.M = (int)M; p.N = (int)N;
    p.nkt = (int)(kpad / 64);
    const int ks = bk / 32;   // MMA K steps per stage
    p.num_kb = (p.nkt + ks - 1) / ks;
    p.ntm = (int)((M + BM - 1) / BM);
    p.ntn = (int)((N + BN - 1) / BN);
    p.nkt_a = p.nkt_b = p.nkt;
    p.b_rt = (int)((N + 127) / 128);
    p.budget = g_wait_budget;
    p.stall = g_stall;
    // Split K in two when the tiles leave the last round of the persistent
    // grid mostly idle (e.g. 512 tiles on 152 SMs: 4 rounds for 3.4 rounds of
    // work) and two half-K units per tile fill the rounds better.  The halves
    // are added into a zeroed C by TMA reduce-add; with two terms the sum
    // does not depend on their order, so the result is deterministic.
    p.splits = 1;
    {
        const int64_t tiles = (int64_t)p.ntm * p.ntn, sms = num_sms();
        const int64_t w1 = (tiles + sms - 1) / sms, w2 = (2 * tiles + sms - 1) / sms;
        // (not with the output amax: the epilogue then sees only partial sums)
        if (!c_amax && p.num_kb >= 8 && (double)w2 < 0.92 * 2.0 * (double)w1) p.splits = 2;
    }
    p.c_amax = c_amax;
    p.amax_rht = amax_rht;
    p.amax_seed = amax_seed;
    p.col_major = M < N ? 1 : 0;
    if (p.splits > 1) {
        cudaError_t e = cudaMemset2DAsync(c, ldc * sizeof(float), 0, N * sizeof(float), M, s);
        if (e != cudaSuccess) return e;
    }
    const NoGroups none;
    const int units = p.ntm * p.ntn * p.splits;
    if (c_amax) {
        const NoGroupsAmax with_amax;
        if (grid == kMXFP4) return cudaErrorInvalidValue;
        if (grid != kE1M2) return run_gemm<kE2M1>(ma, mb, mea, meb, mc, p, with_amax, units, s);
        if (planes) return run_gemm<kE1M2Pl>(ma, mb, mea, meb, mc, p, with_amax, units, s);
        return run_gemm<kE1M2>(ma, mb, mea, meb, mc, p, with_amax, units, s);
    }
    // clamped-E2M1 codes are E2M1 codes; MXFP4 codes too, with UE8M0 scales
    if (grid == kMXFP4) return run_gemm<kMX>(ma, mb, mea, meb, mc, p, none, units, s);
    if (grid != kE1M2) return run_gemm<kE2M1>(ma, mb, mea, meb, mc, p, none, units, s);
    if (planes) return run_gemm<kE1M2Pl>(ma, mb, mea, meb, mc, p, none, units, s);
    return run_gemm<kE1M2>(ma, mb, mea, meb, mc, p, none, units, s);
}

cudaError_t launch_gemm_grouped(const uint8_t *a_codes, const uint8_t *a_eplane, const uint8_t *a_scales,
                                const float *a_ts, int64_t a_rows, int64_t a_kpad, const uint8_t *b_codes,
                                const uint8_t *b_eplane, const uint8_t *b_scales, const float *b_ts,
                                int64_t b_rows, int64_t b_kpad, int grid, const GroupGemmTab &tab,
                                cudaStream_t s) {
    const bool planes = grid == kE1M2 && a_eplane && b_eplane;
    const int bk = planes ? Cfg<kE1M2Pl>::kBK : (grid == kE1M2 ? Cfg<kE1M2>::kBK : Cfg<kE2M1>::kBK);
    CUtensorMap ma, mb, mea, meb, mc;
    if (!make_code_map(&ma, a_codes, a_rows, a_kpad, BM, bk) ||
        !make_code_map(&mb, b_codes, b_rows, b_kpad, BN, bk))
        return cudaErrorInvalidValue;
    if (planes) {
        if (!make_code_map(&mea, a_eplane, a_rows, a_kpad, BM, bk) ||
            !make_code_map(&meb, b_eplane, b_rows, b_kpad, BN, bk))
            return cudaErrorInvalidValue;
    } else {
        mea = ma;   // unused
        meb = mb;
    }
    memset(&mc, 0, sizeof mc);   // grouped epilogues store directly
    GemmParams p{};
    p.sfa = a_scales; p.sfb = b_scales; p.ts_a = a_ts; p.ts_b = b_ts;
    p.nkt_a = (int)(a_kpad / 64);
    p.nkt_b = (int)(b_kpad / 64);
    p.b_rt = (int)((b_rows + 127) / 128);
    p.M = 1; p.N = 1;
    p.budget = g_wait_budget;
    p.stall = g_stall;
    p.splits = 1;
    const int ntiles = tab.tiles[tab.n];
    if (grid != kE1M2) return run_gemm<kE2M1>(ma, mb, mea, meb, mc, p, tab, ntiles, s);
    if (planes) return run_gemm<kE1M2Pl>(ma, mb, mea, meb, mc, p, tab, ntiles, s);
    return run_gemm<kE1M2>(ma, mb, mea, meb, mc, p, tab, ntiles, s);
}

bool make_input_tile_map(void *tmap, const void *x, int64_t rows, int64_t cols, int64_t ld, int box_cols,
                         int box_rows) {
    auto enc = get_encode();
    if (!enc) return false;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)(ld * 2)};
    cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(static_cast<CUtensorMap *>(tmap), CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(x),
                     dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

cudaError_t read_timeout_flag(uint32_t *flag, cudaStream_t s) {
    cudaError_t e = cudaMemcpyFromSymbolAsync(flag, g_ufp4_timeout, sizeof(uint32_t), 0,
                                              cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e == cudaSuccess && *flag) {
        const uint32_t zero = 0;
        e = cudaMemcpyToSymbolAsync(g_ufp4_timeout, &zero, sizeof zero, 0, cudaMemcpyHostToDevice, s);
        if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    }
    return e;
}

}  // namespace ufp4

#ifdef UFP4_PROBE
#include "probe_gemm.inc"
#endif
