// Tensor-core (tcgen05) backward pass of bidirectional GMA for bf16 inputs,
// d = dv = K = 64.
//
// "Gaussian Mixture Attention" (Huang & Raza, 2026), section 4.1: the softmax
// Jacobian ds_ik = gamma_ik (g_ik - sum_l gamma_il g_il) (Eq. 17-18), the chain
// rule through the score of Eq. 16 (Eq. 19; d s / d mu of Eq. 20; d s / d x of
// section 4.3) and the memory products of Eq. 5-8 differentiated as products:
// with den_i = gamma^Q_i Z + eps, a_i = dO_i / den_i, b_i = -(dO_i . O_i) / den_i,
//   g^Q = [a | b] [Vt | Z]^T,      [R | r] = Gamma^Q^T [a | b],
//   g^K = [V | 1] [R | r]^T,       dV = Gamma^K R,
//   dx  = ds (lambda mu) - x (ds lambda),
//   P1 = ds^T x,  P2 = ds^T x^2,  P0 = ds^T 1  (per component, summed over rows)
// and dmu, drho, dalpha from P (the finalize of the CUDA-core backward).
//
// The forward's kernels give the memory [Vt | Z] (tc_params, tc_write, tc_reduce)
// as the bf16 operand [Vt | Z | 1 | 0...]^T (80 rows of 64 components); one pass
// kernel then runs twice over 128-row tiles, persistent like the read kernel:
//   QUERY mode (rows of Qx and dO): the log-density and softmax of the forward ->
//     Gamma^Q; num = Gamma^Q [Vt | Z | 1] -> a, b on the CUDA cores;
//     g^Q = [a | b] [Vt | Z]^T (the same operand read MN-major); ds;
//     dx = ds [lambda | lambda mu] (one MMA, N = 128); [R | r]^T += [a | b]^T Gamma^Q and
//     P^T += [x | x^2]^T ds accumulate in TMEM over the head's tiles and are drained to
//     fp32 partial slots (cta + head).
//   KEY mode (rows of Kx and V), with [R | r] reduced by tc_reduce into the same
//     operand layout: Gamma^K; g^K = [V | 1] [R | r]^T and dV = Gamma^K R; ds; dx; P^T.
// Operand precisions: the log-density as in the forward (fp16 [x, x^2/256] and W);
// the two memory operands [Vt | Z] and [R | r] as two bf16 terms (hi + lo, about 16
// significant bits: the roundings of these shared operands, amplified through the
// softmax Jacobian of peaked responsibilities, dominated the error in one bf16 term);
// Gamma, a | b, ds, x, x^2 and [lambda | lambda mu] in bf16; every accumulation, the
// softmax, ds and the epilogues in fp32.  Every reduction has a fixed order, so the
// result is deterministic.
//
// Warps: 0 TMA / bulk-copy producer; 1 TMEM owner and the one MMA issuer (every MMA
// of a tile, in order); 2-5 the compute group, one thread per tile row, each warp on
// its own (its barriers count four warp arrivals, and no named barrier is used, so a
// wait that runs out never leaves another warp blocked).  Every mbarrier wait is
// bounded; a timeout posts GMA_ERR_TIMEOUT.
#include <cuda.h>
#include <cuda_bf16.h>

#include <algorithm>
#include <cstdint>

#include "gma_internal.h"
#include "gma_sm100.cuh"
#include "gma_tc_common.cuh"

namespace gma {

using namespace sm100;
using namespace tc;

namespace {

constexpr int BK = 64;                        // components
constexpr int kGroups = 2, kGroupWarps = 4;   // compute groups, warps per group
constexpr int kWProd = 0, kWMma = 1, kWCompute = 2;
constexpr int kBThreads = (kWCompute + kGroups * kGroupWarps) * 32;
constexpr int kPartRows = 2 * DR + kGroups * kGroupWarps;   // P partial rows: P1^T (x), P2^T (x^2), P0 per compute warp
constexpr int kPRows = 2 * DR + 1;                // finalize layout: P1, P2, P0
constexpr uint32_t kLamBytes = 2u * DR * 128u;    // [lambda | lambda mu] as a K-major B: 128 rows x 64 components

enum : int { kQuery = 0, kKeys = 1 };

struct BwdTcArgs {
    int G, H, N, T, Ttot;
    const uint8_t *params;     // tc_params blocks, [H][param_stride]
    uint32_t param_stride;
    const uint8_t *lamb;       // [H][kLamBytes] bf16 [lambda | lambda mu] operand
    const uint8_t *mem;        // [G][mem_stride] bf16 [M | m | 1 | 0...]^T: [Vt | Z] (query) or [R | r] (keys)
    const uint8_t *mem_lo;     // [G][mem_stride] its bf16 rounding remainder (hi + lo: a two-term operand)
    uint32_t mem_stride;
    float eps;
    float *dX;                 // [G][N][d] fp32
    float *dV;                 // keys: [G][N][dv] fp32
    float *part_r;             // query: [slot][dv + 1][K] fp32, slot = cta + head
    float *part_p;             // [slot][kPartRows][K] fp32
    unsigned *status;
    int nslots;
};

struct BwdCfg {
    static constexpr uint32_t PB = align1k(param_bytes(BK));
    static constexpr uint32_t MB = align1k(mem_bytes(BK));
    static constexpr uint32_t OFF_X = 0;                               // 2 stages: x tiles (TMA)
    static constexpr uint32_t OFF_U = OFF_X + 2 * kTileBytes;          // 2 stages: dO (query) or V (keys)
    static constexpr uint32_t OFF_GD = OFF_U + 2 * kTileBytes;         // per group: Gamma, then ds (bf16 [row][k])
    static constexpr uint32_t OFF_AX = OFF_GD + kGroups * kTileBytes;  // per group: a (query), then x^2
    static constexpr uint32_t OFF_BB = OFF_AX + kGroups * kTileBytes;  // query: per group [b, 0...]; keys: [1, 0...]
    static constexpr uint32_t OFF_P = OFF_BB + kGroups * kTileBytes;   // the head's parameter block
    static constexpr uint32_t OFF_L = OFF_P + PB;                      // [lambda | lambda mu]
    static constexpr uint32_t OFF_M = OFF_L + kLamBytes;               // the head's memory operand, hi
    static constexpr uint32_t OFF_ML = OFF_M + MB;                     // and lo
    static constexpr uint32_t OFF_CA = OFF_ML + MB;                    // constant [1, 1, 0...] A block
    static constexpr uint32_t OFF_BAR = OFF_CA + kConstABytes;
    static constexpr uint32_t BYTES = OFF_BAR + 256 + 1024;
    // TMEM: group w owns columns [128 w, 128 w + 128), used in turn for [x, x^2/256] (0-63) and
    // the scores (64-127), num (0-79), g (64-127) and the dx products (0-127); then the shared
    // [R | r]^T (query) or the groups' dV (keys), and P^T
    static constexpr uint32_t COL_GRP = 128, COL_A = 0, COL_D1 = 64, COL_NUM = 0, COL_DX = 0;
    static constexpr uint32_t TMEM_COLS = 512;
};
static_assert(BwdCfg::OFF_P % 1024 == 0 && BwdCfg::OFF_L % 1024 == 0 && BwdCfg::OFF_M % 1024 == 0 &&
                  BwdCfg::OFF_ML % 1024 == 0 && BwdCfg::OFF_GD % 1024 == 0 && BwdCfg::OFF_AX % 1024 == 0 &&
                  BwdCfg::OFF_BB % 1024 == 0 && BwdCfg::OFF_CA % 1024 == 0,
              "operand blocks must be 1024-byte aligned");
static_assert(BwdCfg::BYTES <= 232448, "backward pass exceeds the shared-memory opt-in limit");
static_assert((BwdCfg::OFF_AX - BwdCfg::OFF_X) / 16 < 16384 && (BwdCfg::OFF_BB - BwdCfg::OFF_AX) / 16 < 16384,
              "descriptor leading-byte offsets");

__device__ __forceinline__ void cta_tiles(int Ttot, int &t0, int &t1) {
    t0 = (int)(((long long)blockIdx.x * Ttot) / gridDim.x);
    t1 = (int)(((long long)(blockIdx.x + 1) * Ttot) / gridDim.x);
}

// Column sums over the warp's 32 rows of one row's 32 values.  Each of five rounds
// halves the columns a lane holds: the lane keeps the upper or lower half (by one bit
// of its index) and adds the same half from the lane whose index differs in that bit.
// Lane l ends with the sum of column l (fixed order).
__device__ __forceinline__ float warp_colsum32(const float (&v)[32], int lane) {
    float a[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) a[j] = v[j];
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {          // 2 o columns held before the round, o after
        const bool hi = lane & o;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            if (j < o) {
                const float keep = hi ? a[o + j] : a[j], send = hi ? a[j] : a[o + j];
                a[j] = keep + __shfl_xor_sync(~0u, send, o);
            }
        }
    }
    return a[0];
}

template <int MODE>
__global__ void __launch_bounds__(kBThreads, 1)
tc_bwd_pass_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_u, BwdTcArgs A) {
    using C = BwdCfg;
    constexpr int K = BK;
    constexpr uint32_t COL_R = kGroups * C::COL_GRP;                       // query: [R | r]^T
    constexpr uint32_t COL_DV = kGroups * C::COL_GRP;                      // keys: dV of group w at + 64 w
    constexpr uint32_t COL_P = MODE == kQuery ? COL_R + 64 : COL_DV + kGroups * 64;   // P^T
    static_assert(COL_P + 64 <= C::TMEM_COLS, "TMEM columns");
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + C::OFF_BAR);
    uint64_t *xfull = bars, *xempty = bars + 2, *ufull = bars + 4, *uempty = bars + 6;
    uint64_t *h_full = bars + 8, *h_empty = bars + 9;           // the head's parameter, lambda and memory blocks
    // per compute group w: [w] of each
    uint64_t *a_full = bars + 10, *d1_full = bars + 12, *g_full = bars + 14, *num_full = bars + 16;
    uint64_t *ab_full = bars + 18, *gg_full = bars + 20, *ds_full = bars + 22, *dx_full = bars + 24;
    uint64_t *acc_full = bars + 26, *acc_empty = bars + 27, *fin = bars + 28;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 29);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    grid_dep_launch();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int t0, t1;
    cta_tiles(A.Ttot, t0, t1);
    const int n = t1 - t0;

    if (threadIdx.x == 0) {
        for (int s = 0; s < 2; ++s) {
            mbar_init(&xfull[s], 1);
            mbar_init(&xempty[s], kGroupWarps + 1);               // a compute group's warps and the P^T MMA
            mbar_init(&ufull[s], 1);
            mbar_init(&uempty[s], MODE == kQuery ? kGroupWarps : 1);
        }
        mbar_init(h_full, 1);
        mbar_init(h_empty, 1);
        for (int w = 0; w < kGroups; ++w) {
            mbar_init(&a_full[w], kGroupWarps);
            mbar_init(&d1_full[w], 1);
            mbar_init(&g_full[w], kGroupWarps);
            mbar_init(&num_full[w], 1);
            mbar_init(&ab_full[w], kGroupWarps);
            mbar_init(&gg_full[w], 1);
            mbar_init(&ds_full[w], kGroupWarps);
            mbar_init(&dx_full[w], 1);
        }
        mbar_init(acc_full, 1);
        mbar_init(acc_empty, kGroupWarps);
        mbar_init(fin, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    init_const_a(sm + C::OFF_CA, threadIdx.x, blockDim.x);
    // query: the [b, 0...] blocks (column 0 written per tile); keys: the [1, 0...] block of [V | 1]
    for (uint32_t e = threadIdx.x; e < kGroups * kTileBytes / 16; e += blockDim.x)
        reinterpret_cast<uint4 *>(sm + C::OFF_BB)[e] = make_uint4(0, 0, 0, 0);
    __syncthreads();
    if (MODE == kKeys && threadIdx.x < TM)
        *reinterpret_cast<uint16_t *>(sm + C::OFF_BB + sw128_off(threadIdx.x, 0)) = 0x3F80u;   // bf16 1.0
    if (warp == kWMma) { tmem_alloc(tmem_slot, C::TMEM_COLS); tmem_relinquish(); }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const Abort ab{abort_flag, A.status};

    if (warp == kWProd) {
        if (lane == 0 && n > 0) {
            TileCursor cx(t0, n, A.T, 0, 1), cu(t0, n, A.T, 0, 1);
            for (; cx.valid() && cx.hl == 0 && cx.i < 2; cx.next()) {
                mbar_arrive_expect_tx(&xfull[cx.i], kTileBytes);
                tma_load_3d(sm + C::OFF_X + cx.i * kTileBytes, &tm_x, &xfull[cx.i], 0, cx.j * TM, cx.g);
            }
            for (; cu.valid() && cu.i < 2; cu.next()) {
                mbar_arrive_expect_tx(&ufull[cu.i], kTileBytes);
                tma_load_3d(sm + C::OFF_U + cu.i * kTileBytes, &tm_u, &ufull[cu.i], 0, cu.j * TM, cu.g);
            }
            grid_dep_wait();                                 // parameter blocks and memory operands are written
            auto load_head = [&](int g) {
                mbar_arrive_expect_tx(h_full, param_bytes(K) + kLamBytes + 2 * mem_bytes(K));
                bulk_load(sm + C::OFF_P, A.params + (size_t)(g % A.H) * A.param_stride, param_bytes(K), h_full);
                bulk_load(sm + C::OFF_L, A.lamb + (size_t)(g % A.H) * kLamBytes, kLamBytes, h_full);
                bulk_load(sm + C::OFF_M, A.mem + (size_t)g * A.mem_stride, mem_bytes(K), h_full);
                bulk_load(sm + C::OFF_ML, A.mem_lo + (size_t)g * A.mem_stride, mem_bytes(K), h_full);
            };
            load_head(t0 / A.T);
            int h_loaded = 0;
            long long last = now_ns();
            while ((cx.valid() || cu.valid()) && !*abort_flag) {
                bool progress = false;
                if (cx.valid()) {
                    // the x tiles of a head follow its blocks (single-buffered: loaded once the
                    // previous head's MMAs are done)
                    bool can = true;
                    if (cx.hl > h_loaded) {
                        if (!mbar_test(h_empty, (cx.hl - 1) & 1)) {
                            can = false;
                        } else {
                            load_head(cx.g);
                            h_loaded = cx.hl;
                            progress = true;
                        }
                    }
                    const int xi = cx.i;
                    if (can && (xi < 2 || mbar_test(&xempty[xi & 1], ((xi >> 1) - 1) & 1))) {
                        (void)GMA_IN_BOUNDS(cx.g < A.G && cx.j < A.T, A.status);
                        mbar_arrive_expect_tx(&xfull[xi & 1], kTileBytes);
                        tma_load_3d(sm + C::OFF_X + (xi & 1) * kTileBytes, &tm_x, &xfull[xi & 1], 0, cx.j * TM, cx.g);
                        cx.next();
                        progress = true;
                    }
                }
                if (cu.valid()) {
                    const int ui = cu.i;
                    if (mbar_test(&uempty[ui & 1], ((ui >> 1) - 1) & 1)) {
                        mbar_arrive_expect_tx(&ufull[ui & 1], kTileBytes);
                        tma_load_3d(sm + C::OFF_U + (ui & 1) * kTileBytes, &tm_u, &ufull[ui & 1], 0, cu.j * TM, cu.g);
                        cu.next();
                        progress = true;
                    }
                }
                if (progress) {
                    last = now_ns();
                } else {
                    __nanosleep(64);
                    if (now_ns() - last > kWaitLimitNs) {
                        *abort_flag = 1;
                        atomicOr(A.status, kDevErrTimeout);
                    }
                }
            }
            wind_down_ring(xfull, 2, cx.i < n ? cx.i : n, A.status);
            wind_down_ring(ufull, 2, cu.i < n ? cu.i : n, A.status);
            wait_ignoring_abort(h_full, h_loaded & 1, A.status);
        }
    } else if (warp == kWMma) {
        // One issuer for both groups: four stages, each taking the tiles in order (so that the
        // shared accumulators sum them in a fixed order), issued as their operands become
        // ready.  The warp stays converged; lane 0 tests the barriers and broadcasts.
        if (n > 0) {
            constexpr uint32_t id_num = idesc_f16(1, 1, 0, 0, TM, 80);     // Gamma . [M | m | 1]
            constexpr uint32_t id_g = idesc_f16(1, 1, 0, 1, TM, K);        // [A | b] . [M | m]^T (B MN-major)
            constexpr uint32_t id_dv = idesc_f16(1, 1, 0, 0, TM, DVV);     // Gamma^K . R
            constexpr uint32_t id_dx = idesc_f16(1, 1, 0, 0, TM, 2 * DR);  // ds . [lambda | lambda mu]
            constexpr uint32_t id_acc = idesc_f16(1, 1, 1, 1, TM, K);      // (MN-major A)^T . (MN-major B)
            const uint32_t pw = smem_u32(sm + C::OFF_P), ca = smem_u32(sm + C::OFF_CA);
            const uint32_t maddr = smem_u32(sm + C::OFF_M), mladdr = smem_u32(sm + C::OFF_ML);
            // K-major operands step 32 bytes (16 elements) per k-step, a descriptor address step
            // of 2; MN-major ones step 16 rows of 128 bytes, a descriptor address step of 128.
            // The memory operand as hi and lo: N = value rows, K = components (K-major), or
            // K = value rows, N = components (MN-major).
            const uint64_t m_k[2] = {sdesc_sw128(maddr, 16, 1024), sdesc_sw128(mladdr, 16, 1024)};
            const uint64_t m_mn[2] = {sdesc_sw128(maddr, kTileBytes, 1024), sdesc_sw128(mladdr, kTileBytes, 1024)};
            const uint64_t l_k = sdesc_sw128(smem_u32(sm + C::OFF_L), 16, 1024);
            auto ready = [&](uint64_t *bar, uint32_t parity) {
                const int t = lane == 0 ? (int)mbar_test(bar, parity) : 0;
                return __shfl_sync(~0u, t, 0) != 0;
            };
            auto acc_free = [&](const TileCursor &c) {       // a head's accumulators start after the last drain
                return !(c.first() && c.hl >= 1) || ready(acc_empty, (c.hl - 1) & 1);
            };
            TileCursor c1(t0, n, A.T, 0, 1), c2 = c1, c3 = c1, c4 = c1;
            long long last = now_ns();
            while (c4.valid()) {
                bool progress = false;
                // S4: dx products, then the parameter sums [x | x^2]^T ds
                if (c4.valid() && c4.i < (MODE == kQuery ? c3.i : c2.i)) {
                    const int w = c4.i & 1, s = c4.i & 1;
                    if (ready(&ds_full[w], (c4.i >> 1) & 1) && (MODE == kQuery || acc_free(c4))) {
                        tc_fence_after();
                        const uint32_t gd = smem_u32(sm + C::OFF_GD + w * kTileBytes);
                        const uint64_t ds_k = sdesc_sw128(gd, 16, 1024), ds_mn = sdesc_sw128(gd, kTileBytes, 1024);
#pragma unroll
                        for (int kk = 0; kk < K / 16; ++kk)
                            mma_ss(tmem + w * C::COL_GRP + C::COL_DX, ds_k + (uint64_t)(kk * 2), l_k + (uint64_t)(kk * 2),
                                   id_dx, kk > 0);
                        mma_commit(&dx_full[w]);
                        const uint32_t xa = smem_u32(sm + C::OFF_X + s * kTileBytes);
                        const uint32_t x2a = smem_u32(sm + C::OFF_AX + w * kTileBytes);
                        const uint64_t xp = sdesc_sw128(xa, x2a - xa, 1024);      // [x | x^2] as an MN-major A
                        const bool fresh = c4.first();
#pragma unroll
                        for (int kk = 0; kk < TM / 16; ++kk)
                            mma_ss(tmem + COL_P, xp + (uint64_t)(kk * 128), ds_mn + (uint64_t)(kk * 128), id_acc,
                                   !(fresh && kk == 0));
                        mma_commit(&xempty[s]);
                        if (c4.last()) {
                            mma_commit(acc_full);
                            mma_commit(h_empty);
                        }
                        c4.next();
                        progress = true;
                    }
                }
                // S3 (queries): g^Q = [a | b] . [Vt | Z]^T, then [R | r]^T += [a | b]^T . Gamma^Q
                if (MODE == kQuery && c3.valid() && c3.i < c2.i) {
                    const int w = c3.i & 1;
                    if (ready(&ab_full[w], (c3.i >> 1) & 1) && acc_free(c3)) {
                        tc_fence_after();
                        const uint32_t aa = smem_u32(sm + C::OFF_AX + w * kTileBytes);
                        const uint32_t ba = smem_u32(sm + C::OFF_BB + w * kTileBytes);
#pragma unroll
                        for (int hl = 0; hl < 2; ++hl)
#pragma unroll
                            for (int kk = 0; kk < 5; ++kk) {
                                const uint64_t ad = kk < 4 ? sdesc_sw128(aa + kk * 32u, 16, 1024) : sdesc_sw128(ba, 16, 1024);
                                mma_ss(tmem + w * C::COL_GRP + C::COL_D1, ad, m_mn[hl] + (uint64_t)(kk * 128), id_g,
                                       hl + kk > 0);
                            }
                        const uint64_t ab_mn = sdesc_sw128(aa, ba - aa, 1024);
                        const uint64_t g_mn = sdesc_sw128(smem_u32(sm + C::OFF_GD + w * kTileBytes), kTileBytes, 1024);
                        const bool fresh = c3.first();
#pragma unroll
                        for (int kk = 0; kk < TM / 16; ++kk)
                            mma_ss(tmem + COL_R, ab_mn + (uint64_t)(kk * 128), g_mn + (uint64_t)(kk * 128), id_acc,
                                   !(fresh && kk == 0));
                        mma_commit(&gg_full[w]);
                        c3.next();
                        progress = true;
                    }
                }
                // S2: queries num = Gamma^Q . [Vt | Z | 1]; keys g^K = [V | 1] . [R | r]^T and dV = Gamma^K . R
                if (c2.valid() && c2.i < c1.i) {
                    const int w = c2.i & 1, s = c2.i & 1;
                    bool go = ready(&g_full[w], (c2.i >> 1) & 1);
                    if (MODE == kKeys) go = go && ready(&ufull[s], (c2.i >> 1) & 1);
                    if (go) {
                        tc_fence_after();
                        const uint32_t gd = smem_u32(sm + C::OFF_GD + w * kTileBytes);
                        const uint64_t g_k = sdesc_sw128(gd, 16, 1024);
                        if (MODE == kQuery) {
#pragma unroll
                            for (int hl = 0; hl < 2; ++hl)
#pragma unroll
                                for (int kk = 0; kk < K / 16; ++kk)
                                    mma_ss(tmem + w * C::COL_GRP + C::COL_NUM, g_k + (uint64_t)(kk * 2),
                                           m_k[hl] + (uint64_t)(kk * 2), id_num, hl + kk > 0);
                            mma_commit(&num_full[w]);
                        } else {
                            const uint32_t va = smem_u32(sm + C::OFF_U + s * kTileBytes);
                            const uint32_t ones = smem_u32(sm + C::OFF_BB);
#pragma unroll
                            for (int hl = 0; hl < 2; ++hl)
#pragma unroll
                                for (int kk = 0; kk < 5; ++kk) {
                                    const uint64_t ad =
                                        kk < 4 ? sdesc_sw128(va + kk * 32u, 16, 1024) : sdesc_sw128(ones, 16, 1024);
                                    mma_ss(tmem + w * C::COL_GRP + C::COL_D1, ad, m_mn[hl] + (uint64_t)(kk * 128), id_g,
                                           hl + kk > 0);
                                }
                            mma_commit(&uempty[s]);
#pragma unroll
                            for (int hl = 0; hl < 2; ++hl)
#pragma unroll
                                for (int kk = 0; kk < K / 16; ++kk)
                                    mma_ss(tmem + COL_DV + 64 * w, g_k + (uint64_t)(kk * 2), m_k[hl] + (uint64_t)(kk * 2),
                                           id_dv, hl + kk > 0);
                            mma_commit(&gg_full[w]);
                        }
                        c2.next();
                        progress = true;
                    }
                }
                // S1: the log-density of the tile's rows (as the forward)
                if (c1.valid()) {
                    const int w = c1.i & 1;
                    if (ready(&a_full[w], (c1.i >> 1) & 1) && (!c1.first() || ready(h_full, c1.hl & 1))) {
                        tc_fence_after();
                        issue_logdensity<K>(tmem + w * C::COL_GRP + C::COL_D1, tmem + w * C::COL_GRP + C::COL_A, pw, ca);
                        mma_commit(&d1_full[w]);
                        c1.next();
                        progress = true;
                    }
                }
                if (progress) {
                    last = now_ns();
                } else {
                    const int aborted = *abort_flag != 0, late = now_ns() - last > kWaitLimitNs;
                    if (__shfl_sync(~0u, aborted | (late << 1), 0)) {
                        if (lane == 0 && !aborted) {
                            *abort_flag = 1;
                            atomicOr(A.status, kDevErrTimeout);
                        }
                        break;
                    }
                    __nanosleep(32);
                }
            }
            mma_commit(fin);
            wait_ignoring_abort(fin, 0, A.status);
        }
    } else {
        // ---------------- compute group w (warps 2-5, 6-9): tiles w, w + 2, ...; thread r owns
        // tile row r (TMEM lane r) of the group's tiles
        const int w = (warp - kWCompute) / kGroupWarps;
        const uint32_t r = 32u * (warp & 3) + lane;
        const uint32_t lane_off = (uint32_t)(32 * (warp & 3)) << 16;
        const uint32_t tg = tmem + lane_off + w * C::COL_GRP;          // the group's TMEM columns, this warp's lanes
        uint8_t *gd = sm + C::OFF_GD + w * kTileBytes;                // Gamma, then ds
        uint8_t *ax = sm + C::OFF_AX + w * kTileBytes;                // a, then x^2
        uint8_t *bb = sm + C::OFF_BB + w * kTileBytes;                // [b, 0...]
        auto warp_arrive = [&](uint64_t *bar) {
            __syncwarp();
            if (lane == 0) mbar_arrive(bar);
        };
        float p0[2] = {0.f, 0.f};           // this warp's column sums of ds: columns lane, 32 + lane
        float scale = 0.f;
        int g_scale = -1;
        // P0 rows of this warp in slot (cta + head) for every head the CTA covers: the sums at
        // the group's last tile of a head, zeros for the heads it had no tiles in
        const int g_first = t0 / A.T, g_last = (t1 - 1) / A.T;
        int g_p0 = g_first - 1;
        auto p0_row = [&](int g) -> float * {
            const int slot = (int)blockIdx.x + g;
            if (!GMA_IN_BOUNDS(slot < A.nslots, A.status)) return nullptr;
            return A.part_p + ((size_t)slot * kPartRows + 2 * DR + w * kGroupWarps + (warp & 3)) * K;
        };
        auto p0_zero_through = [&](int g_end) {          // heads g_p0 + 1 .. g_end - 1
            for (int gz = g_p0 + 1; gz < g_end; ++gz)
                if (float *row = p0_row(gz)) { row[lane] = 0.f; row[32 + lane] = 0.f; }
        };
        for (TileCursor c(t0, n, A.T, w, kGroups); c.valid(); c.next()) {
            const int i = c.i, s = i & 1;
            const uint32_t ph = (uint32_t)(i >> 1) & 1u;      // this group's tile count, parity
            const int row = c.j * TM + (int)r;
            const bool valid = row < A.N;
            if (c.g != g_scale) {
                if (g_scale < 0) grid_dep_wait();
                scale = head_scale(A.params, A.param_stride, c.g % A.H, K);
                g_scale = c.g;
            }
            // ---- [x, x^2/256] (fp16) into TMEM for the log-density
            if (!mbar_wait_warp(&xfull[s], ph, ab, kDevErrTimeout)) break;
            const uint8_t *xs = sm + C::OFF_X + s * kTileBytes;
            convert_row(xs, r, tg + C::COL_A);
            tmem_st_wait();
            tc_fence_before();
            warp_arrive(&a_full[w]);
            // ---- Gamma = softmax of the scores (Eq. 3b), rows past the end 0; bf16 into GD
            if (!mbar_wait_warp(&d1_full[w], ph, ab, kDevErrTimeout)) break;
            tc_fence_after();
            {
                uint32_t e[K / 2];
                row_exp_scaled<K>(tg + C::COL_D1, scale, e);
                float q[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int t = 0; t < K / 2; ++t) {
                    q[(2 * t) & 3] += bf16_lo(e[t]);
                    q[(2 * t + 1) & 3] += bf16_hi(e[t]);
                }
                const float inv = valid ? 1.0f / ((q[0] + q[1]) + (q[2] + q[3])) : 0.f;
#pragma unroll
                for (int j = 0; j < K / 8; ++j) {
                    uint32_t wv[4];
#pragma unroll
                    for (int u = 0; u < 4; ++u)
                        wv[u] = pack_bf16(bf16_lo(e[4 * j + u]) * inv, bf16_hi(e[4 * j + u]) * inv);
                    *reinterpret_cast<uint4 *>(gd + sw128_off(r, j)) = make_uint4(wv[0], wv[1], wv[2], wv[3]);
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            warp_arrive(&g_full[w]);
            if (MODE == kQuery) {
                // ---- a = dO / den, b = -(dO . O) / den from num = [Gamma Vt | Gamma Z | Gamma 1] (Eq. 7-8)
                bool ok = mbar_wait_warp(&num_full[w], ph, ab, kDevErrTimeout);
                ok = ok && mbar_wait_warp(&ufull[s], ph, ab, kDevErrTimeout);
                if (!ok) break;
                tc_fence_after();
                uint32_t v0[32], v1[32], dz[4];
                tmem_ld32(tg + C::COL_NUM, v0);
                tmem_ld32(tg + C::COL_NUM + 32, v1);
                tmem_ld4(tg + C::COL_NUM + 64, dz);
                tmem_ld_wait();
                // den = Gamma Z + eps sum_k Gamma (the forward's normaliser, Gamma as rounded)
                const float den = valid ? __uint_as_float(dz[0]) + A.eps * __uint_as_float(dz[1]) : 1.0f;
                const float rd = 1.0f / den;
                const uint8_t *us = sm + C::OFF_U + s * kTileBytes;
                float dq[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const uint4 dv4 = *reinterpret_cast<const uint4 *>(us + sw128_off(r, j));
                    const uint32_t dw[4] = {dv4.x, dv4.y, dv4.z, dv4.w};
                    const uint32_t *src = j < 4 ? v0 + 8 * j : v1 + 8 * (j - 4);
                    uint32_t o[4];
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const float d0 = bf16_lo(dw[u]), d1 = bf16_hi(dw[u]);
                        dq[u] = fmaf(d0, __uint_as_float(src[2 * u]), dq[u]);
                        dq[u] = fmaf(d1, __uint_as_float(src[2 * u + 1]), dq[u]);
                        o[u] = pack_bf16(d0 * rd, d1 * rd);
                    }
                    *reinterpret_cast<uint4 *>(ax + sw128_off(r, j)) = make_uint4(o[0], o[1], o[2], o[3]);
                }
                // b = -(dO . num) / den^2
                const float bv = -((dq[0] + dq[1]) + (dq[2] + dq[3])) * rd * rd;
                *reinterpret_cast<uint16_t *>(bb + sw128_off(r, 0)) = (uint16_t)(pack_bf16(bv, 0.f) & 0xFFFFu);
                fence_proxy_async_smem();
                tc_fence_before();
                warp_arrive(&ab_full[w]);
                warp_arrive(&uempty[s]);
            }
            // ---- ds = gamma (g - gamma . g) (Eq. 17-18) over Gamma in GD (bf16, written back as ds);
            // x^2 (bf16) into AX for the parameter sums; the column sums of ds for P0
            if (!mbar_wait_warp(&gg_full[w], ph, ab, kDevErrTimeout)) break;
            tc_fence_after();
            {
                uint32_t gv[K];
                tmem_ld32(tg + C::COL_D1, gv);
                tmem_ld32(tg + C::COL_D1 + 32, gv + 32);
                uint32_t gm[K / 2];
#pragma unroll
                for (int j = 0; j < K / 8; ++j) {
                    const uint4 v = *reinterpret_cast<const uint4 *>(gd + sw128_off(r, j));
                    gm[4 * j] = v.x; gm[4 * j + 1] = v.y; gm[4 * j + 2] = v.z; gm[4 * j + 3] = v.w;
                }
                tmem_ld_wait();
                float q[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int t = 0; t < K / 2; ++t) {
                    q[(2 * t) & 3] = fmaf(bf16_lo(gm[t]), __uint_as_float(gv[2 * t]), q[(2 * t) & 3]);
                    q[(2 * t + 1) & 3] = fmaf(bf16_hi(gm[t]), __uint_as_float(gv[2 * t + 1]), q[(2 * t + 1) & 3]);
                }
                const float mean = (q[0] + q[1]) + (q[2] + q[3]);
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    float ds[32];
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        uint32_t wv[4];
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            const int t = 16 * hf + 4 * j + u;          // bf16 pair index
                            wv[u] = pack_bf16(bf16_lo(gm[t]) * (__uint_as_float(gv[2 * t]) - mean),
                                              bf16_hi(gm[t]) * (__uint_as_float(gv[2 * t + 1]) - mean));
                            ds[8 * j + 2 * u] = bf16_lo(wv[u]);          // P0 sums the values the MMAs use
                            ds[8 * j + 2 * u + 1] = bf16_hi(wv[u]);
                        }
                        *reinterpret_cast<uint4 *>(gd + sw128_off(r, 4 * hf + j)) = make_uint4(wv[0], wv[1], wv[2], wv[3]);
                    }
                    p0[hf] += warp_colsum32(ds, lane);
                }
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const uint4 v = *reinterpret_cast<const uint4 *>(xs + sw128_off(r, j));
                    const uint32_t xw[4] = {v.x, v.y, v.z, v.w};
                    uint32_t o[4];
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const float lo = bf16_lo(xw[u]), hi = bf16_hi(xw[u]);
                        o[u] = pack_bf16(lo * lo, hi * hi);
                    }
                    *reinterpret_cast<uint4 *>(ax + sw128_off(r, j)) = make_uint4(o[0], o[1], o[2], o[3]);
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            warp_arrive(&ds_full[w]);
            // ---- dx = ds (lambda mu) - x (ds lambda) (section 4.3); keys: dV = Gamma^K R
            if (!mbar_wait_warp(&dx_full[w], ph, ab, kDevErrTimeout)) break;
            tc_fence_after();
            {
                const bool store = valid && GMA_IN_BOUNDS(c.g < A.G, A.status);
                float *dxr = A.dX + ((size_t)c.g * A.N + (store ? row : 0)) * DR;
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    uint32_t c1[32], c2[32];
                    tmem_ld32(tg + C::COL_DX + 32 * half, c1);
                    tmem_ld32(tg + C::COL_DX + DR + 32 * half, c2);
                    tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const uint4 xv = *reinterpret_cast<const uint4 *>(xs + sw128_off(r, 4 * half + j));
                        const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
                        float o[8];
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            const int t = 8 * j + 2 * u;
                            o[2 * u] = fmaf(-bf16_lo(xw[u]), __uint_as_float(c1[t]), __uint_as_float(c2[t]));
                            o[2 * u + 1] = fmaf(-bf16_hi(xw[u]), __uint_as_float(c1[t + 1]), __uint_as_float(c2[t + 1]));
                        }
                        if (store) {
                            float4 *d4 = reinterpret_cast<float4 *>(dxr + 32 * half + 8 * j);
                            d4[0] = make_float4(o[0], o[1], o[2], o[3]);
                            d4[1] = make_float4(o[4], o[5], o[6], o[7]);
                        }
                    }
                }
                if (MODE == kKeys) {
                    uint32_t v0[32], v1[32];
                    tmem_ld32(tmem + lane_off + COL_DV + 64 * w, v0);
                    tmem_ld32(tmem + lane_off + COL_DV + 64 * w + 32, v1);
                    tmem_ld_wait();
                    if (store) {
                        float4 *d4 = reinterpret_cast<float4 *>(A.dV + ((size_t)c.g * A.N + row) * DVV);
#pragma unroll
                        for (int t = 0; t < 16; ++t) {
                            const uint32_t *src = t < 8 ? v0 + 4 * t : v1 + 4 * (t - 8);
                            d4[t] = make_float4(__uint_as_float(src[0]), __uint_as_float(src[1]),
                                                __uint_as_float(src[2]), __uint_as_float(src[3]));
                        }
                    }
                }
            }
            tc_fence_before();
            warp_arrive(&xempty[s]);        // this group has read its x rows (the P^T MMA is the other reader)
            const int slot = (int)blockIdx.x + c.g;
            const bool slot_ok = GMA_IN_BOUNDS(slot < A.nslots, A.status);
            float *pp = A.part_p + (size_t)slot * kPartRows * K;
            // ---- the group's last tile of the head: its P0 rows (one per warp) in slot (cta + head)
            if (c.i + kGroups >= n || c.j + kGroups >= A.T) {
                p0_zero_through(c.g);
                if (float *row = p0_row(c.g)) { row[lane] = p0[0]; row[32 + lane] = p0[1]; }
                p0[0] = p0[1] = 0.f;
                g_p0 = c.g;
            }
            // ---- the head's last tile: drain [R | r]^T (query) and P^T into slot (cta + head)
            if (c.last()) {
                if (!mbar_wait_warp(acc_full, c.hl & 1, ab, kDevErrTimeout)) break;
                tc_fence_after();
                uint32_t v[K];
                if (MODE == kQuery) {
                    tmem_ld32(tmem + lane_off + COL_R, v);
                    tmem_ld32(tmem + lane_off + COL_R + 32, v + 32);
                    tmem_ld_wait();
                    if (r <= (uint32_t)DVV && slot_ok) {
                        float4 *dst = reinterpret_cast<float4 *>(A.part_r + ((size_t)slot * (DVV + 1) + r) * K);
#pragma unroll
                        for (int t = 0; t < K / 4; ++t)
                            dst[t] = make_float4(__uint_as_float(v[4 * t]), __uint_as_float(v[4 * t + 1]),
                                                 __uint_as_float(v[4 * t + 2]), __uint_as_float(v[4 * t + 3]));
                    }
                }
                tmem_ld32(tmem + lane_off + COL_P, v);
                tmem_ld32(tmem + lane_off + COL_P + 32, v + 32);
                tmem_ld_wait();
                if (slot_ok) {
                    float4 *dst = reinterpret_cast<float4 *>(pp + (size_t)r * K);
#pragma unroll
                    for (int t = 0; t < K / 4; ++t)
                        dst[t] = make_float4(__uint_as_float(v[4 * t]), __uint_as_float(v[4 * t + 1]),
                                             __uint_as_float(v[4 * t + 2]), __uint_as_float(v[4 * t + 3]));
                }
                tc_fence_before();
                warp_arrive(acc_empty);
            }
        }
        p0_zero_through(g_last + 1);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kWMma) {
        __syncwarp();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

// Per head h (blockIdx.x) and 8-component chunk j (blockIdx.y): lambda = 1 / (softplus(rho)
// + var_floor) (Eq. 14) in fp32 [K][d] for the finalize, and chunk j of every row of the
// bf16 operand [lambda | lambda mu] (K-major: row m < d holds lambda_{k, m} over the
// components k, row d + m holds lambda_{k, m} mu_{k, m}).  It has no programmatic trigger, so
// a kernel launched after it starts once it has finished.
__global__ void __launch_bounds__(256) bwd_lamb_kernel(float var_floor, const float *__restrict__ mu,
                                                       const float *__restrict__ rho, float *__restrict__ lam,
                                                       uint8_t *__restrict__ out) {
    __shared__ float ls[8 * DR], ms[8 * DR];
    const int h = blockIdx.x, j = blockIdx.y;
    const size_t base = ((size_t)h * BK + 8 * j) * DR;          // components 8 j .. 8 j + 7
    for (int e = threadIdx.x; e < 8 * DR; e += blockDim.x) {
        const float w = rho[base + e];
        const float l = 1.0f / (fmaxf(w, 0.f) + log1pf(expf(-fabsf(w))) + var_floor);
        ls[e] = l;
        ms[e] = mu[base + e];
        lam[base + e] = l;
    }
    __syncthreads();
    uint8_t *blk = out + (size_t)h * kLamBytes;
    for (int nrow = threadIdx.x; nrow < 2 * DR; nrow += blockDim.x) {
        const int m = nrow % DR;
        uint32_t w[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            float v[2];
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                const int kk = 2 * u + q;                          // component 8 j + kk
                v[q] = nrow < DR ? ls[kk * DR + m] : ls[kk * DR + m] * ms[kk * DR + m];
            }
            w[u] = pack_bf16(v[0], v[1]);
        }
        *reinterpret_cast<uint4 *>(blk + sw128_off(nrow, j)) = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

// The parameter sums of head set h (blockIdx.x), rows q0 = 8 blockIdx.y .. q0 + 7 of the
// finalize layout (q < d P1, d <= q < 2d P2, q = 2d P0), for the query (blockIdx.z = 0) or
// key rows, into out[z][h][k][q].  The (batch entry b, CTA c) pairs whose partial slot c + g
// (g = b H + h) holds a part of head g are taken in a fixed order (b, then c increasing);
// thread (k, u) sums the pairs u, u + 4, ... for its eight rows (P0: the compute warps' rows
// in group and warp order), and the four sums of each (k, q) are then added in u order.
// The CTA ranges are found once per block (dynamic shared memory, two ints per batch entry).
constexpr int kPsumSplit = 4, kPsumRows = 8;
static_assert((2 * DR) % kPsumRows == 0, "P0 starts a block row");

__global__ void __launch_bounds__(BK * kPsumSplit) bwd_psum_kernel(int B, int H, int T, int Ttot, int ncta, int nslots,
                                                                   const float *__restrict__ part_q,
                                                                   const float *__restrict__ part_k,
                                                                   float *__restrict__ out, unsigned *status) {
    extern __shared__ int crange[];
    __shared__ float red[kPsumSplit][kPsumRows][BK];
    const int h = blockIdx.x, q0 = kPsumRows * blockIdx.y, k = threadIdx.x % BK, u = threadIdx.x / BK;
    for (int b = threadIdx.x; b < B; b += blockDim.x) {
        // CTA c owns tiles [c Ttot / ncta, (c + 1) Ttot / ncta): those meeting head g
        const int g = b * H + h;
        const long long lo = (long long)g * T, hi = (long long)(g + 1) * T;
        int c = (int)((lo * ncta) / Ttot);
        while (c > 0 && ((long long)c * Ttot) / ncta > lo) --c;
        while (((long long)(c + 1) * Ttot) / ncta <= lo) ++c;
        int c_hi = c;
        while (c_hi < ncta && ((long long)c_hi * Ttot) / ncta < hi) ++c_hi;
        crange[2 * b] = c;
        crange[2 * b + 1] = c_hi;
    }
    __syncthreads();
    const float *part = blockIdx.z ? part_k : part_q;
    float s[kPsumRows];
#pragma unroll
    for (int r = 0; r < kPsumRows; ++r) s[r] = 0.f;
    int pi = 0;                                      // pair index in the fixed order
    for (int b = 0; b < B; ++b) {
        const int g = b * H + h, c_lo = crange[2 * b], c_hi = crange[2 * b + 1];
        if (!GMA_IN_BOUNDS(c_lo >= 0 && c_hi + g <= nslots, status)) break;
        for (int c = c_lo; c < c_hi; ++c, ++pi) {
            if (pi % kPsumSplit != u) continue;
            const float *pp = part + (size_t)(c + g) * kPartRows * BK + k;
            float v[kPsumRows];
#pragma unroll
            for (int r = 0; r < kPsumRows; ++r) {
                const int q = q0 + r;
                v[r] = q < 2 * DR ? pp[(size_t)q * BK] : 0.f;
            }
            if (q0 == 2 * DR) {                      // the last block row holds P0 alone
                float w0 = pp[(size_t)(2 * DR) * BK];
                for (int x = 1; x < kGroups * kGroupWarps; ++x) w0 += pp[(size_t)(2 * DR + x) * BK];
                v[0] = w0;
            }
#pragma unroll
            for (int r = 0; r < kPsumRows; ++r) s[r] += v[r];
        }
    }
#pragma unroll
    for (int r = 0; r < kPsumRows; ++r) red[u][r][k] = s[r];
    __syncthreads();
    for (int e = threadIdx.x; e < kPsumRows * BK; e += blockDim.x) {
        const int r = e / BK, kk = e % BK, q = q0 + r;
        if (q >= kPRows) continue;
        float t = red[0][r][kk];
        for (int x = 1; x < kPsumSplit; ++x) t += red[x][r][kk];
        out[(((size_t)blockIdx.z * H + h) * BK + kk) * kPRows + q] = t;
    }
}

template <int MODE>
cudaError_t launch_bwd_pass(const Problem &p, const BwdTcLayout &L, const void *X, const void *U, const char *mem,
                            const char *mem_lo, float *dX, float *dV, float *part_r, float *part_p, char *ws,
                            cudaStream_t s) {
    CUtensorMap tx, tu;
    if (!make_map(&tx, X, p.G, p.N, DR) || !make_map(&tu, U, p.G, p.N, DVV)) return cudaErrorInvalidValue;
    BwdTcArgs a{};
    a.G = p.G; a.H = p.H; a.N = p.N; a.T = L.tc.Tkv; a.Ttot = L.tc.Ttot_kv;
    a.params = reinterpret_cast<const uint8_t *>(ws + L.tc.params);
    a.param_stride = L.tc.param_stride;
    a.lamb = reinterpret_cast<const uint8_t *>(ws + L.lamb);
    a.mem = reinterpret_cast<const uint8_t *>(mem);
    a.mem_lo = reinterpret_cast<const uint8_t *>(mem_lo);
    a.mem_stride = L.tc.mem_stride;
    a.eps = p.eps;
    a.dX = dX;
    a.dV = dV;
    a.part_r = part_r;
    a.part_p = part_p;
    a.status = reinterpret_cast<unsigned *>(ws);
    a.nslots = kMaxCtas + p.G;
    auto kern = tc_bwd_pass_kernel<MODE>;
    cudaError_t e = set_dyn_smem(reinterpret_cast<const void *>(kern), BwdCfg::BYTES);
    if (e != cudaSuccess) return e;
    // the same CTA partition as the write kernel, so that tc_reduce sums the query pass's
    // [R | r] slots as it sums the write kernel's
    return launch_dependent(kern, dim3(L.tc.ncta_kv), dim3(kBThreads), BwdCfg::BYTES, s, tx, tu, a);
}

}  // namespace

bool bwd_tc_supported(const Problem &p) {
    // heads of more than one tile: a one-tile head gains nothing from the persistent passes,
    // and the CUDA-core passes keep it in fp32
    return !p.causal && p.in_dtype == GMA_BF16 && p.out_dtype == GMA_BF16 && p.d == DR && p.dv == DVV && p.K == BK &&
           p.N > TM && p.Nkv == p.N;
}

BwdTcLayout bwd_tc_layout(const Problem &p) {
    BwdTcLayout L{};
    L.tc = tc_layout(p);           // parameter blocks, memory partials and operand (the forward's layout)
    const size_t slots = (size_t)kMaxCtas + p.G;
    size_t off = L.tc.total;
    L.lam = align_up(off);
    off = L.lam + sizeof(float) * (size_t)p.H * BK * DR;
    L.lamb = align_up(off);
    off = L.lamb + (size_t)p.H * kLamBytes;
    L.mem_lo = align_up(off);
    off = L.mem_lo + (size_t)p.G * L.tc.mem_stride;
    L.part_r = align_up(off);
    off = L.part_r + sizeof(float) * slots * (DVV + 1) * BK;
    L.mem_r = align_up(off);
    off = L.mem_r + (size_t)p.G * L.tc.mem_stride;
    L.mem_rlo = align_up(off);
    off = L.mem_rlo + (size_t)p.G * L.tc.mem_stride;
    L.part_pq = align_up(off);
    off = L.part_pq + sizeof(float) * slots * kPartRows * BK;
    L.part_pk = align_up(off);
    off = L.part_pk + sizeof(float) * slots * kPartRows * BK;
    L.psum = align_up(off);
    off = L.psum + sizeof(float) * 2 * (size_t)p.H * BK * kPRows;
    L.total = align_up(off);
    return L;
}

cudaError_t bwd_tc_run(const Problem &p, const BwdTcLayout &L, const void *Qx, const void *Kx, const void *V,
                       const float *mu, const float *rho, const float *alpha, const void *dO, float *dQx, float *dKx,
                       float *dV, float *dmu, float *drho, float *dalpha, char *ws, cudaStream_t s) {
    cudaError_t e;
    float *lam = reinterpret_cast<float *>(ws + L.lam);
    float *part_pq = reinterpret_cast<float *>(ws + L.part_pq), *part_pk = reinterpret_cast<float *>(ws + L.part_pk);
    float *psum = reinterpret_cast<float *>(ws + L.psum);
    unsigned *status = reinterpret_cast<unsigned *>(ws);
    const int nslots = kMaxCtas + p.G;
    // parameter prologues: the log-density blocks of the forward, fp32 lambda, [lambda | lambda mu]
    if ((e = tc_params(p, L.tc, mu, rho, alpha, ws, s)) != cudaSuccess) return e;
    bwd_lamb_kernel<<<dim3(p.H, BK / 8), 256, 0, s>>>(p.var_floor, mu, rho, lam,
                                                      reinterpret_cast<uint8_t *>(ws + L.lamb));
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    // the forward memory [Vt | Z] (Eq. 5-6)
    if ((e = tc_write(p, L.tc, Kx, V, ws, s)) != cudaSuccess) return e;
    if ((e = tc_reduce_split(p, L.tc, L.tc.part, L.tc.mem, L.mem_lo, ws, s)) != cudaSuccess) return e;
    // the query rows: dQx, [R | r], parameter sums
    if ((e = launch_bwd_pass<kQuery>(p, L, Qx, dO, ws + L.tc.mem, ws + L.mem_lo, dQx, nullptr,
                                     reinterpret_cast<float *>(ws + L.part_r), part_pq, ws, s)) != cudaSuccess)
        return e;
    // [R | r] into the memory-operand layout: the forward's reduce over the query pass's slots
    if ((e = tc_reduce_split(p, L.tc, L.part_r, L.mem_r, L.mem_rlo, ws, s)) != cudaSuccess) return e;
    // the key rows: dKx, dV, parameter sums
    if ((e = launch_bwd_pass<kKeys>(p, L, Kx, V, ws + L.mem_r, ws + L.mem_rlo, dKx, dV, nullptr, part_pk, ws, s)) !=
        cudaSuccess)
        return e;
    // per head set: the parameter sums over every batch entry, query and key rows apart
    const dim3 psum_grid(p.H, (kPRows + kPsumRows - 1) / kPsumRows, 2);
    bwd_psum_kernel<<<psum_grid, BK * kPsumSplit, sizeof(int) * 2 * (size_t)p.B, s>>>(
        p.B, p.H, L.tc.Tkv, L.tc.Ttot_kv, L.tc.ncta_kv, nslots, part_pq, part_pk, psum, status);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    Problem p1 = p;           // the finalize over one (batch-summed) entry per head set
    p1.B = 1;
    p1.G = p.H;
    return bwd_finalize(p1, 1, psum, psum + (size_t)p.H * BK * kPRows, mu, lam, rho, alpha, dmu, drho, dalpha, s);
}

}  // namespace gma
