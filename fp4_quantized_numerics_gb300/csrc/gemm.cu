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
// E1M2: not a tensor-core format.  Each magnitude m/2 splits exactly as
//   a + b/2 with a = m >> 1 in {0,1,2,3} and b = m & 1, both representable in
//   E2M1 (a -> 0,1,2,3; b/2 -> 0 or 0.5), with the sign copied to both parts
//   and the block scale shared.  Warps expand each staged tile into a "hi"
//   and a "lo" E2M1 plane in shared memory and four MMAs (hi*hi, hi*lo,
//   lo*hi, lo*lo) accumulate into the same TMEM accumulator -- exact, since
//   every product and partial sum of the dequantized values is what the
//   single E1M2 product would give.
//
// CTA: 192 threads.  Warp 0 = TMA producer, warp 1 = TMEM owner + single-
// thread MMA issuer, warps 2-5 = epilogue (and, for E1M2, the expanders).
// Tile 128 x 128, K step per stage 256 (128 bytes per row, one 128-byte
// swizzle atom), multi-stage mbarrier ring, accumulator in TMEM.
// Every wait is bounded: on timeout the kernel raises g_ufp4_timeout, drains
// its own copies, frees TMEM and returns.
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

constexpr int BM = 128, BN = 128;
constexpr int BK_BYTES = 128;                 // 256 FP4 elements per stage
constexpr uint32_t TILE_BYTES = 128 * 128;    // 16 KB per operand tile
constexpr uint32_t SF_BYTES = 4 * 512;        // 4 scale atoms per operand per stage
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kSfCol = 256;              // accumulators in [0, 256), scales after
constexpr long long kWaitBudget = 2000000000LL;

template <int GRID>
struct Cfg {
    static constexpr int kStages = GRID == kE2M1 ? 5 : 3;
    // warps: 0 producer, 1 MMA, 2-5 epilogue, (E1M2) 6-13 expanders
    static constexpr int kThreads = GRID == kE2M1 ? 192 : 448;
    static constexpr int kExpThreads = kThreads - 192;
    // epilogue staging: per epilogue warp, kEpiBufs buffers of 32 rows x 32
    // fp32 columns (4 KB, 128-byte swizzled rows) feeding TMA stores
    static constexpr int kEpiBufs = GRID == kE2M1 ? 2 : 1;
    // stage layout: A | B | (A_lo | B_lo for E1M2) | SFA | SFB
    static constexpr uint32_t kAOff = 0;
    static constexpr uint32_t kBOff = TILE_BYTES;
    static constexpr uint32_t kALoOff = 2 * TILE_BYTES;
    static constexpr uint32_t kBLoOff = 3 * TILE_BYTES;
    static constexpr uint32_t kSfaOff = (GRID == kE2M1 ? 2 : 4) * TILE_BYTES;
    static constexpr uint32_t kSfbOff = kSfaOff + SF_BYTES;
    static constexpr uint32_t kStageBytes = kSfbOff + SF_BYTES;  // multiple of 1024
    static constexpr uint32_t kEpiOff = kStages * kStageBytes;
    static constexpr uint32_t kBarOff = kEpiOff + 4 * kEpiBufs * 4096;
    static constexpr uint32_t kSmemBytes = kBarOff + 256 + 1024;  // + barriers + alignment slack
};

struct GemmParams {
    const uint8_t *sfa, *sfb;
    const float *ts_a, *ts_b;
    float *c;
    int64_t ldc;
    int M, N;
    int nkt;      // kpad / 64: scale atoms per 128-row tile
    int num_kb;   // ceil(nkt / 4): K stages per tile
    int ntm, ntn; // tiles along M and N
    int nkt_a, nkt_b;  // k atoms per 128-row tile of the whole A / B tensors
};

// Where one output tile lives: operand rows / k atoms in the A and B tensors,
// its problem's sizes, output pointer and tensor scales.
struct TileInfo {
    int a_row, b_row, a_kt, b_kt, nkt, num_kb;
    int m_loc, n_loc, M, N;
    float *c;
    int64_t ldc;
    const float *ts_a, *ts_b;
};

struct NoGroups {};

__device__ __forceinline__ TileInfo tile_info(const GemmParams &p, const NoGroups &, int t) {
    TileInfo ti;
    ti.m_loc = (t / p.ntn) * BM;
    ti.n_loc = (t % p.ntn) * BN;
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
    ti.num_kb = (g.nkt + 3) / 4;
    ti.M = g.M;
    ti.N = g.N;
    ti.c = g.c;
    ti.ldc = g.ldc;
    ti.ts_a = p.ts_a + g.a_seg;
    ti.ts_b = p.ts_b + g.b_seg;
    return ti;
}

__device__ __forceinline__ void raise_timeout() { atomicOr(&g_ufp4_timeout, 1u); }

// Bounded wait that also gives up as soon as another role has aborted.
__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity, volatile int *abort) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (true) {
#pragma unroll 1
        for (int i = 0; i < 64; ++i)
            if (ptx::mbar_try_wait(bar, parity)) return true;
        if (*abort) return false;
        if (clock64() - t0 > kWaitBudget) {
            *abort = 1;
            raise_timeout();
            return false;
        }
    }
}

// E1M2 nibbles s|m2 m1 m0 -> (hi, lo) E2M1 nibbles, 8 at a time.  With
// a = m >> 1, the E2M1 code of a in {0,1,2,3} is {0,2,4,5} = 2a - [a == 3];
// 2a sits in bits 2..1 already, so hi = (w & 0xE...) - (m1 & m2) (no borrow
// leaves a nibble); lo keeps the sign and m0 (E2M1 code 1 = 0.5).
__device__ __forceinline__ void split_e1m2(uint32_t w, uint32_t &hi, uint32_t &lo) {
    hi = (w & 0xEEEEEEEEu) - ((w >> 1) & (w >> 2) & 0x11111111u);
    lo = w & 0x99999999u;
}

// Persistent CTA: tiles t = blockIdx.x, blockIdx.x + gridDim.x, ... in
// row-major (M, N) tile order.  The K ring and the two TMEM accumulators are
// carried across tiles, so the epilogue of one tile overlaps the main loop
// of the next.
template <int GRID, class TAB>
__global__ void __launch_bounds__(Cfg<GRID>::kThreads, 1)
    k_gemm(const __grid_constant__ CUtensorMap tma_a, const __grid_constant__ CUtensorMap tma_b,
           const __grid_constant__ CUtensorMap tma_c, GemmParams p, const __grid_constant__ TAB tab) {
    constexpr bool kGrouped = std::is_same<TAB, GroupGemmTab>::value;
    using C = Cfg<GRID>;
    constexpr int S = C::kStages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::kBarOff);
    // bars: [0,S) full, [S,2S) empty, [2S,3S) expanded, 3S+{0,1} acc full,
    // 3S+{2,3} acc empty, 3S+4 MMA drained
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 3 * S + 5);
    volatile int *abort = reinterpret_cast<volatile int *>(tmem_slot + 1);
    const uint32_t smem_base = ptx::smem_u32(smem);
    const uint32_t bar_base = ptx::smem_u32(bars);
    auto full = [&](int s) { return bar_base + 8u * s; };
    auto empty = [&](int s) { return bar_base + 8u * (S + s); };
    auto expd = [&](int s) { return bar_base + 8u * (2 * S + s); };
    auto accf = [&](int b) { return bar_base + 8u * (3 * S + b); };
    auto acce = [&](int b) { return bar_base + 8u * (3 * S + 2 + b); };
    const uint32_t drained = bar_base + 8u * (3 * S + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int ntiles;
    if constexpr (kGrouped) ntiles = tab.tiles[tab.n];
    else ntiles = p.ntm * p.ntn;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            ptx::mbar_init(full(s), 1);
            ptx::mbar_init(empty(s), 1);
            ptx::mbar_init(expd(s), GRID == kE1M2 ? C::kExpThreads / 32 : 1);   // one arrival per expander warp
        }
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(accf(b), 1);
            ptx::mbar_init(acce(b), 4);   // one arrival per epilogue warp
        }
        ptx::mbar_init(drained, 1);
        *abort = 0;
        ptx::fence_mbar_init();
        ptx::prefetch_tmap(&tma_a);
        ptx::prefetch_tmap(&tma_b);
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

    if (warp == 0) {
        // ---------------------------------------------------------- producer
        if (lane == 0) {
            uint32_t g = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x) {
                const TileInfo ti = tile_info(p, tab, t);
                for (int kb = 0; kb < ti.num_kb; ++kb, ++g) {
                    const uint32_t s = g % S, round = g / S;
                    if (round > 0 && !wait_or_abort(empty(s), (round - 1) & 1, abort)) { ok = false; break; }
                    const int atoms = min(4, ti.nkt - 4 * kb);
                    const uint32_t st = smem_base + s * C::kStageBytes;
                    ptx::mbar_arrive_expect_tx(full(s), 2 * TILE_BYTES + 2u * atoms * 512u);
                    ptx::tma_load_2d(st + C::kAOff, &tma_a, ti.a_kt * 32 + kb * BK_BYTES, ti.a_row, full(s));
                    ptx::tma_load_2d(st + C::kBOff, &tma_b, ti.b_kt * 32 + kb * BK_BYTES, ti.b_row, full(s));
                    ptx::bulk_load(st + C::kSfaOff,
                                   p.sfa + ((size_t)(ti.a_row / 128) * p.nkt_a + ti.a_kt + 4 * kb) * 512,
                                   atoms * 512u, full(s));
                    ptx::bulk_load(st + C::kSfbOff,
                                   p.sfb + ((size_t)(ti.b_row / 128) * p.nkt_b + ti.b_kt + 4 * kb) * 512,
                                   atoms * 512u, full(s));
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
        // One thread issues every tcgen05 op of the CTA, so its instruction
        // stream is kept short: descriptors are built once per stage and
        // advanced by integer adds (start address field = bytes >> 4).
        if (lane == 0) {
            // instruction descriptor, kind::mxf4nvf4: A/B E2M1 (1), K-major,
            // N >> 3 at [17,23), UE4M3 scales (bit 23 = 0), M >> 4 at [24,29).
            const uint32_t idesc = (1u << 7) | (1u << 10) | ((uint32_t)(BN >> 3) << 17) |
                                   ((uint32_t)(BM >> 4) << 24);
            const uint64_t hi_op = ptx::sdesc(0, 16, 1024, 2);   // 128B-swizzled K-major operand
            const uint64_t hi_sf = ptx::sdesc(0, 0, 128, 0);     // 32 rows x 16 B scale atom
            auto mk = [](uint64_t hi, uint32_t addr) { return hi | (uint64_t)((addr & 0x3FFFFu) >> 4); };
            uint32_t g = 0, it = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x, ++it) {
                const TileInfo ti = tile_info(p, tab, t);
                const uint32_t b = it & 1, use = it >> 1;
                if (use > 0 && !wait_or_abort(acce(b), (use - 1) & 1, abort)) { ok = false; break; }
                ptx::tc_fence_after();
                const uint32_t acc = tmem + b * BN;
                for (int kb = 0; kb < ti.num_kb; ++kb, ++g) {
                    const uint32_t s = g % S, round = g / S;
                    if (!wait_or_abort(GRID == kE2M1 ? full(s) : expd(s), round & 1, abort)) { ok = false; break; }
                    ptx::tc_fence_after();
                    const int atoms = min(4, ti.nkt - 4 * kb);
                    const uint32_t st = smem_base + s * C::kStageBytes;
                    const uint32_t sf_t = tmem + kSfCol + 32u * s;
                    const uint64_t dsa = mk(hi_sf, st + C::kSfaOff), dsb = mk(hi_sf, st + C::kSfbOff);
                    const uint64_t dah = mk(hi_op, st + C::kAOff), dbh = mk(hi_op, st + C::kBOff);
                    const uint64_t dal = mk(hi_op, st + C::kALoOff), dbl = mk(hi_op, st + C::kBLoOff);
                    auto step = [&](int j) {
                        const uint32_t sfa = sf_t + 4u * j, sfb = sf_t + 16u + 4u * j;
                        const uint32_t first = (kb == 0 && j == 0) ? 0u : 1u;
                        const uint64_t o = 2u * (uint32_t)j;   // +32 bytes per 64-element K step
                        ptx::tc_mma_nvf4(acc, dah + o, dbh + o, idesc, sfa, sfb, first);
                        if (GRID == kE1M2) {
                            ptx::tc_mma_nvf4(acc, dah + o, dbl + o, idesc, sfa, sfb, 1u);
                            ptx::tc_mma_nvf4(acc, dal + o, dbh + o, idesc, sfa, sfb, 1u);
                            ptx::tc_mma_nvf4(acc, dal + o, dbl + o, idesc, sfa, sfb, 1u);
                        }
                    };
                    if (atoms == 4) {
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            ptx::tc_cp_32x128b_warpx4(sf_t + 4u * j, dsa + 32u * j);
                            ptx::tc_cp_32x128b_warpx4(sf_t + 16u + 4u * j, dsb + 32u * j);
                        }
#pragma unroll
                        for (int j = 0; j < 4; ++j) step(j);
                    } else {
                        for (int j = 0; j < atoms; ++j) {
                            ptx::tc_cp_32x128b_warpx4(sf_t + 4u * j, dsa + 32u * j);
                            ptx::tc_cp_32x128b_warpx4(sf_t + 16u + 4u * j, dsb + 32u * j);
                        }
                        for (int j = 0; j < atoms; ++j) step(j);
                    }
                    ptx::tc_commit(empty(s));
                }
                if (ok) ptx::tc_commit(accf(b));   // fires once this tile's MMAs have completed
            }
            // TMEM is freed below only after every MMA issued here has finished.
            ptx::tc_commit(drained);
            const long long t0 = clock64();
            while (!ptx::mbar_try_wait(drained, 0))
                if (clock64() - t0 > kWaitBudget) { raise_timeout(); break; }
        }
    } else if (warp < 6) {
        // ------------------------------------------------------------ epilogue
        // TMEM -> registers (x alpha) -> swizzled shared staging -> TMA store.
        // Each warp owns 32 accumulator rows; a 32 x 32 fp32 box per store, so
        // global writes are whole lines and ragged tile edges are clipped by
        // the tensor map.
        const int q = warp & 3;                 // TMEM lane quadrant of this warp
        const uint32_t ebase = smem_base + C::kEpiOff + (uint32_t)(warp - 2) * C::kEpiBufs * 4096u;
        uint32_t it = 0, nst = 0;
        for (int t = blockIdx.x; t < ntiles; t += gridDim.x, ++it) {
            const uint32_t b = it & 1, use = it >> 1;
            bool ok = wait_or_abort(accf(b), use & 1, abort);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            ptx::tc_fence_after();
            const TileInfo ti = tile_info(p, tab, t);
            const float alpha = __fmul_rn(*ti.ts_a, *ti.ts_b);
            const int m0 = ti.m_loc, n0 = ti.n_loc;
#pragma unroll 1
            for (int ch = 0; ch < BN / 32; ++ch, ++nst) {
                uint32_t r[32];
                ptx::tc_ld_32x32b_x32(tmem + ((uint32_t)(32 * q) << 16) + b * BN + 32u * ch, r);
                if constexpr (kGrouped) {
                    // masked direct stores: a group's C is not a whole tensor map
                    ptx::tc_wait_ld();
                    if (ch == BN / 32 - 1) {
                        ptx::tc_fence_before();
                        __syncwarp();
                        if (lane == 0) ptx::mbar_arrive(acce(b));
                    }
                    const int row = m0 + 32 * q + lane, col0 = n0 + 32 * ch;
                    if (row < ti.M) {
                        float *crow = ti.c + (int64_t)row * ti.ldc;
                        if (col0 + 32 <= ti.N) {
#pragma unroll
                            for (int i = 0; i < 32; i += 4)
                                *reinterpret_cast<float4 *>(crow + col0 + i) =
                                    make_float4(__uint_as_float(r[i]) * alpha, __uint_as_float(r[i + 1]) * alpha,
                                                __uint_as_float(r[i + 2]) * alpha, __uint_as_float(r[i + 3]) * alpha);
                        } else {
                            for (int i = 0; i < 32; ++i)
                                if (col0 + i < ti.N) crow[col0 + i] = __uint_as_float(r[i]) * alpha;
                        }
                    }
                    continue;
                }
                const uint32_t buf = ebase + (nst % C::kEpiBufs) * 4096u;
                // the store that last read this buffer must be done reading it
                if (lane == 0) {
                    if (C::kEpiBufs == 2) ptx::bulk_wait_read<1>();
                    else ptx::bulk_wait_read<0>();
                }
                __syncwarp();
                ptx::tc_wait_ld();
                if (ch == BN / 32 - 1) {   // accumulator fully read: hand it back to the MMA warp
                    ptx::tc_fence_before();
                    __syncwarp();
                    if (lane == 0) ptx::mbar_arrive(acce(b));
                }
                const uint32_t rowb = buf + (uint32_t)lane * 128u;
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const uint32_t addr = rowb + (uint32_t)((c ^ (lane & 7)) << 4);
                    asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr),
                                 "f"(__uint_as_float(r[4 * c]) * alpha), "f"(__uint_as_float(r[4 * c + 1]) * alpha),
                                 "f"(__uint_as_float(r[4 * c + 2]) * alpha), "f"(__uint_as_float(r[4 * c + 3]) * alpha)
                                 : "memory");
                }
                ptx::fence_proxy_async();
                __syncwarp();
                if (lane == 0 && m0 + 32 * q < p.M && n0 + 32 * ch < p.N) {   // boxes wholly outside C: skip
                    ptx::tma_store_2d(&tma_c, n0 + 32 * ch, m0 + 32 * q, buf);
                    ptx::bulk_commit();
                }
            }
        }
        if (lane == 0) ptx::bulk_wait_all();
        __syncwarp();
    } else if constexpr (GRID == kE1M2) {
        // ------------------------------------------------- E1M2 expanders
        const int et = threadIdx.x - 192;   // 0 .. kExpThreads-1
        uint32_t g = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x) {
            const int nkb = tile_info(p, tab, t).num_kb;
            for (int kb = 0; kb < nkb; ++kb, ++g) {
                const uint32_t s = g % S, round = g / S;
                ok = wait_or_abort(full(s), round & 1, abort);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                uint8_t *st = smem + s * C::kStageBytes;
#pragma unroll 4
                for (int i = et; i < (int)(TILE_BYTES / 16); i += C::kExpThreads) {
                    uint4 *pa = reinterpret_cast<uint4 *>(st + C::kAOff) + i;
                    uint4 *pb = reinterpret_cast<uint4 *>(st + C::kBOff) + i;
                    uint4 a = *pa, bv = *pb, ah, alo, bh, blo;
                    split_e1m2(a.x, ah.x, alo.x); split_e1m2(a.y, ah.y, alo.y);
                    split_e1m2(a.z, ah.z, alo.z); split_e1m2(a.w, ah.w, alo.w);
                    split_e1m2(bv.x, bh.x, blo.x); split_e1m2(bv.y, bh.y, blo.y);
                    split_e1m2(bv.z, bh.z, blo.z); split_e1m2(bv.w, bh.w, blo.w);
                    *pa = ah;
                    *pb = bh;
                    reinterpret_cast<uint4 *>(st + C::kALoOff)[i] = alo;
                    reinterpret_cast<uint4 *>(st + C::kBLoOff)[i] = blo;
                }
                // generic-proxy writes -> visible to the tensor cores (async proxy)
                ptx::fence_proxy_async();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(expd(s));
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

bool make_code_map(CUtensorMap *m, const uint8_t *codes, int64_t rows, int64_t kpad) {
    auto enc = get_encode();
    if (!enc) return false;
    cuuint64_t dims[2] = {(cuuint64_t)(kpad / 2), (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)(kpad / 2)};
    cuuint32_t box[2] = {(cuuint32_t)BK_BYTES, 128};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t *>(codes), dims, strides, box,
                     estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool make_out_map(CUtensorMap *m, float *c, int64_t M, int64_t N, int64_t ldc) {
    auto enc = get_encode();
    if (!enc) return false;
    cuuint64_t dims[2] = {(cuuint64_t)N, (cuuint64_t)M};
    cuuint64_t strides[1] = {(cuuint64_t)(ldc * 4)};
    cuuint32_t box[2] = {32, 32};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, c, dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

template <int GRID, class TAB>
cudaError_t run_gemm(const CUtensorMap &ma, const CUtensorMap &mb, const CUtensorMap &mc, const GemmParams &p,
                     const TAB &tab, int ntiles, cudaStream_t s) {
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
    k_gemm<GRID, TAB><<<grid, C::kThreads, C::kSmemBytes, s>>>(ma, mb, mc, p, tab);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gemm(const uint8_t *a_codes, const uint8_t *a_scales, const float *a_ts,
                        const uint8_t *b_codes, const uint8_t *b_scales, const float *b_ts, int64_t M,
                        int64_t N, int64_t K, int grid, float *c, int64_t ldc, cudaStream_t s) {
    if (K == 0) return cudaMemset2DAsync(c, ldc * sizeof(float), 0, N * sizeof(float), M, s);
    const int64_t kpad = kpad_of(K);
    CUtensorMap ma, mb, mc;
    if (!make_code_map(&ma, a_codes, M, kpad) || !make_code_map(&mb, b_codes, N, kpad) ||
        !make_out_map(&mc, c, M, N, ldc))
        return cudaErrorInvalidValue;
    GemmParams p{};
    p.sfa = a_scales; p.sfb = b_scales; p.ts_a = a_ts; p.ts_b = b_ts;
    p.c = c; p.ldc = ldc; p.M = (int)M; p.N = (int)N;
    p.nkt = (int)(kpad / 64);
    p.num_kb = (p.nkt + 3) / 4;
    p.ntm = (int)((M + BM - 1) / BM);
    p.ntn = (int)((N + BN - 1) / BN);
    p.nkt_a = p.nkt_b = p.nkt;
    const NoGroups none;
    if (grid == kE2M1) return run_gemm<kE2M1>(ma, mb, mc, p, none, p.ntm * p.ntn, s);
    return run_gemm<kE1M2>(ma, mb, mc, p, none, p.ntm * p.ntn, s);
}

cudaError_t launch_gemm_grouped(const uint8_t *a_codes, const uint8_t *a_scales, const float *a_ts,
                                int64_t a_rows, int64_t a_kpad, const uint8_t *b_codes, const uint8_t *b_scales,
                                const float *b_ts, int64_t b_rows, int64_t b_kpad, int grid,
                                const GroupGemmTab &tab, cudaStream_t s) {
    CUtensorMap ma, mb, mc;
    if (!make_code_map(&ma, a_codes, a_rows, a_kpad) || !make_code_map(&mb, b_codes, b_rows, b_kpad))
        return cudaErrorInvalidValue;
    memset(&mc, 0, sizeof mc);   // grouped epilogues store directly
    GemmParams p{};
    p.sfa = a_scales; p.sfb = b_scales; p.ts_a = a_ts; p.ts_b = b_ts;
    p.nkt_a = (int)(a_kpad / 64);
    p.nkt_b = (int)(b_kpad / 64);
    p.M = 1; p.N = 1;
    const int ntiles = tab.tiles[tab.n];
    if (grid == kE2M1) return run_gemm<kE2M1>(ma, mb, mc, p, tab, ntiles, s);
    return run_gemm<kE1M2>(ma, mb, mc, p, tab, ntiles, s);
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
