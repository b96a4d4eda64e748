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
constexpr int kBThreads = 192;                // 6 warps
constexpr int kWProd = 0, kWMma = 1, kGroupWarps = 4;
constexpr int kPartRows = 2 * DR + kGroupWarps;   // P partial rows: P1^T (x), P2^T (x^2), P0 per compute warp
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
    static constexpr uint32_t OFF_X2 = OFF_U + 2 * kTileBytes;         // 2 buffers: x^2 (bf16)
    static constexpr uint32_t OFF_G = OFF_X2 + 2 * kTileBytes;         // Gamma (bf16 [row][k])
    static constexpr uint32_t OFF_AB = OFF_G + kTileBytes;             // query: [a], [b, 0...]; keys: [1, 0...]
    static constexpr uint32_t OFF_DS = OFF_AB + 2 * kTileBytes;        // ds (bf16 [row][k])
    static constexpr uint32_t OFF_P = OFF_DS + kTileBytes;             // the head's parameter block
    static constexpr uint32_t OFF_L = OFF_P + PB;                      // [lambda | lambda mu]
    static constexpr uint32_t OFF_M = OFF_L + kLamBytes;               // the head's memory operand, hi
    static constexpr uint32_t OFF_ML = OFF_M + MB;                     // and lo
    static constexpr uint32_t OFF_CA = OFF_ML + MB;                    // constant [1, 1, 0...] A block
    static constexpr uint32_t OFF_BAR = OFF_CA + kConstABytes;
    static constexpr uint32_t BYTES = OFF_BAR + 256 + 1024;
    // TMEM columns: [x, x^2/256] | scores, then g | num or dV | dx | [R | r]^T | P^T
    static constexpr uint32_t COL_A = 0, COL_D1 = 64, COL_NUM = 128, COL_DX = 256, COL_R = 384, COL_P = 448;
    static constexpr uint32_t TMEM_COLS = 512;
};
static_assert(BwdCfg::OFF_P % 1024 == 0 && BwdCfg::OFF_L % 1024 == 0 && BwdCfg::OFF_M % 1024 == 0 &&
                  BwdCfg::OFF_ML % 1024 == 0 && BwdCfg::OFF_AB % 1024 == 0 && BwdCfg::OFF_DS % 1024 == 0 && BwdCfg::OFF_CA % 1024 == 0,
              "operand blocks must be 1024-byte aligned");
static_assert(BwdCfg::BYTES <= 232448, "backward pass exceeds the shared-memory opt-in limit");
static_assert(BwdCfg::COL_NUM + 80 <= BwdCfg::COL_DX && BwdCfg::COL_P + BK <= BwdCfg::TMEM_COLS, "TMEM columns");

__device__ __forceinline__ void cta_tiles(int Ttot, int &t0, int &t1) {
    t0 = (int)(((long long)blockIdx.x * Ttot) / gridDim.x);
    t1 = (int)(((long long)(blockIdx.x + 1) * Ttot) / gridDim.x);
}

// Column sums over the warp's 32 rows of one row's 64 values.  Each of five rounds
// halves the columns a lane holds: the lane keeps the upper or lower half (by one bit
// of its index) and adds the same half from the lane whose index differs in that bit.
// Lane l ends with the sums of columns 2l and 2l + 1 (fixed order).
__device__ __forceinline__ float2 warp_colsum64(const float (&v)[BK], int lane) {
    float a[32];
    {
        const bool hi = lane & 16;
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            const float keep = hi ? v[32 + j] : v[j], send = hi ? v[j] : v[32 + j];
            a[j] = keep + __shfl_xor_sync(~0u, send, 16);
        }
    }
#pragma unroll
    for (int o = 8; o >= 1; o >>= 1) {          // 4 o columns held before the round, 2 o after
        const bool hi = lane & o;
        const int hh = 2 * o;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            if (j < hh) {
                const float keep = hi ? a[hh + j] : a[j], send = hi ? a[j] : a[hh + j];
                a[j] = keep + __shfl_xor_sync(~0u, send, o);
            }
        }
    }
    return make_float2(a[0], a[1]);
}

template <int MODE>
__global__ void __launch_bounds__(kBThreads, 1)
tc_bwd_pass_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_u, BwdTcArgs A) {
    using C = BwdCfg;
    constexpr int K = BK;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + C::OFF_BAR);
    uint64_t *xfull = bars, *xempty = xfull + 2, *ufull = xempty + 2, *uempty = ufull + 2;
    uint64_t *h_full = uempty + 2, *h_empty = h_full + 1;      // the head's parameter, lambda and memory blocks
    uint64_t *a_full = h_empty + 1, *d1_full = a_full + 1, *g_full = d1_full + 1, *num_full = g_full + 1;
    uint64_t *ab_full = num_full + 1, *gg_full = ab_full + 1, *ds_full = gg_full + 1, *dx_full = ds_full + 1;
    uint64_t *acc_full = dx_full + 1, *acc_empty = acc_full + 1, *fin = acc_empty + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(fin + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    grid_dep_launch();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int t0, t1;
    cta_tiles(A.Ttot, t0, t1);
    const int n = t1 - t0;

    if (threadIdx.x == 0) {
        for (int s = 0; s < 2; ++s) {
            mbar_init(&xfull[s], 1);
            mbar_init(&xempty[s], kGroupWarps + 1);               // the compute warps and the P^T MMA
            mbar_init(&ufull[s], 1);
            mbar_init(&uempty[s], MODE == kQuery ? kGroupWarps : 1);
        }
        for (uint64_t *b = h_full; b <= fin; ++b) mbar_init(b, 1);
        mbar_init(a_full, kGroupWarps);
        mbar_init(g_full, kGroupWarps);
        mbar_init(ab_full, kGroupWarps);
        mbar_init(ds_full, kGroupWarps);
        mbar_init(acc_empty, kGroupWarps);
        *abort_flag = 0;
        fence_mbar_init();
    }
    init_const_a(sm + C::OFF_CA, threadIdx.x, blockDim.x);
    // query: the [b, 0...] block (column 0 written per tile); keys: the [1, 0...] block of [V | 1]
    for (uint32_t e = threadIdx.x; e < kTileBytes / 16; e += blockDim.x)
        reinterpret_cast<uint4 *>(sm + C::OFF_AB + (MODE == kQuery ? kTileBytes : 0))[e] = make_uint4(0, 0, 0, 0);
    __syncthreads();
    if (MODE == kKeys && threadIdx.x < TM)
        *reinterpret_cast<uint16_t *>(sm + C::OFF_AB + sw128_off(threadIdx.x, 0)) = 0x3F80u;   // bf16 1.0
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
        if (n > 0) {                                         // the whole warp, converged
            constexpr uint32_t id_num = idesc_f16(1, 1, 0, 0, TM, 80);     // Gamma . [M | m | 1]
            constexpr uint32_t id_g = idesc_f16(1, 1, 0, 1, TM, K);        // [A | b] . [M | m]^T (B MN-major)
            constexpr uint32_t id_dv = idesc_f16(1, 1, 0, 0, TM, DVV);     // Gamma^K . R
            constexpr uint32_t id_dx = idesc_f16(1, 1, 0, 0, TM, 2 * DR);  // ds . [lambda | lambda mu]
            constexpr uint32_t id_acc = idesc_f16(1, 1, 1, 1, TM, K);      // (MN-major A)^T . (MN-major B)
            const uint32_t pw = smem_u32(sm + C::OFF_P), ca = smem_u32(sm + C::OFF_CA);
            const uint32_t gaddr = smem_u32(sm + C::OFF_G), dsaddr = smem_u32(sm + C::OFF_DS);
            const uint32_t abaddr = smem_u32(sm + C::OFF_AB), maddr = smem_u32(sm + C::OFF_M);
            // K-major operands step 32 bytes (16 elements) per k-step, a descriptor address step
            // of 2; MN-major ones step 16 rows of 128 bytes, a descriptor address step of 128
            const uint64_t g_k = sdesc_sw128(gaddr, 16, 1024);              // Gamma, rows x components
            const uint64_t g_mn = sdesc_sw128(gaddr, kTileBytes, 1024);     // Gamma as the MN-major B of a row sum
            const uint64_t ds_k = sdesc_sw128(dsaddr, 16, 1024);
            const uint64_t ds_mn = sdesc_sw128(dsaddr, kTileBytes, 1024);
            // the memory operand as hi and lo (two-term): N = value rows, K = components (K-major),
            // or K = value rows, N = components (MN-major)
            const uint32_t mladdr = smem_u32(sm + C::OFF_ML);
            const uint64_t m_k[2] = {sdesc_sw128(maddr, 16, 1024), sdesc_sw128(mladdr, 16, 1024)};
            const uint64_t m_mn[2] = {sdesc_sw128(maddr, kTileBytes, 1024), sdesc_sw128(mladdr, kTileBytes, 1024)};
            const uint64_t l_k = sdesc_sw128(smem_u32(sm + C::OFF_L), 16, 1024);
            bool ok = true;
            for (TileCursor c(t0, n, A.T, 0, 1); c.valid() && ok; c.next()) {
                const int i = c.i, s = i & 1;
                const uint32_t ph = (uint32_t)i & 1u;
                if (c.first() && !(ok = mbar_wait_warp(h_full, c.hl & 1, ab, kDevErrTimeout))) break;
                // log-density of the tile's rows (as the forward)
                if (!(ok = mbar_wait_warp(a_full, ph, ab, kDevErrTimeout))) break;
                tc_fence_after();
                issue_logdensity<K>(tmem + C::COL_D1, tmem + C::COL_A, pw, ca);
                mma_commit(d1_full);
                if (!(ok = mbar_wait_warp(g_full, ph, ab, kDevErrTimeout))) break;
                // a head's accumulators start once the previous head's have been drained
                if (c.first() && c.hl >= 1 && !(ok = mbar_wait_warp(acc_empty, (c.hl - 1) & 1, ab, kDevErrTimeout)))
                    break;
                tc_fence_after();
                const bool fresh = c.first();
                if (MODE == kQuery) {
                    // num = Gamma^Q . [Vt | Z | 1] (hi, then lo)
#pragma unroll
                    for (int hl = 0; hl < 2; ++hl)
#pragma unroll
                        for (int kk = 0; kk < K / 16; ++kk)
                            mma_ss(tmem + C::COL_NUM, g_k + (uint64_t)(kk * 2), m_k[hl] + (uint64_t)(kk * 2), id_num,
                                   hl + kk > 0);
                    mma_commit(num_full);
                    if (!(ok = mbar_wait_warp(ab_full, ph, ab, kDevErrTimeout))) break;
                    tc_fence_after();
                    // g^Q = [a | b] . [Vt | Z]^T: k-steps over the value rows, then the Z row (hi, lo)
#pragma unroll
                    for (int hl = 0; hl < 2; ++hl)
#pragma unroll
                        for (int kk = 0; kk < 5; ++kk) {
                            const uint64_t ad = kk < 4 ? sdesc_sw128(abaddr + kk * 32u, 16, 1024)
                                                       : sdesc_sw128(abaddr + kTileBytes, 16, 1024);
                            mma_ss(tmem + C::COL_D1, ad, m_mn[hl] + (uint64_t)(kk * 128), id_g, hl + kk > 0);
                        }
                    mma_commit(gg_full);
                    // [R | r]^T += [a | b]^T . Gamma^Q over the tile's rows
                    const uint64_t ab_mn = sdesc_sw128(abaddr, kTileBytes, 1024);
#pragma unroll
                    for (int kk = 0; kk < TM / 16; ++kk)
                        mma_ss(tmem + C::COL_R, ab_mn + (uint64_t)(kk * 128), g_mn + (uint64_t)(kk * 128), id_acc,
                               !(fresh && kk == 0));
                } else {
                    if (!(ok = mbar_wait_warp(&ufull[s], (i >> 1) & 1, ab, kDevErrTimeout))) break;
                    tc_fence_after();
                    // g^K = [V | 1] . [R | r]^T, then dV = Gamma^K . R (hi, lo)
                    const uint32_t va = smem_u32(sm + C::OFF_U + s * kTileBytes);
#pragma unroll
                    for (int hl = 0; hl < 2; ++hl)
#pragma unroll
                        for (int kk = 0; kk < 5; ++kk) {
                            const uint64_t ad =
                                kk < 4 ? sdesc_sw128(va + kk * 32u, 16, 1024) : sdesc_sw128(abaddr, 16, 1024);
                            mma_ss(tmem + C::COL_D1, ad, m_mn[hl] + (uint64_t)(kk * 128), id_g, hl + kk > 0);
                        }
                    mma_commit(&uempty[s]);
#pragma unroll
                    for (int hl = 0; hl < 2; ++hl)
#pragma unroll
                        for (int kk = 0; kk < K / 16; ++kk)
                            mma_ss(tmem + C::COL_NUM, g_k + (uint64_t)(kk * 2), m_k[hl] + (uint64_t)(kk * 2), id_dv,
                                   hl + kk > 0);
                    mma_commit(gg_full);
                }
                // dx products and the parameter sums, once ds is in place
                if (!(ok = mbar_wait_warp(ds_full, ph, ab, kDevErrTimeout))) break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < K / 16; ++kk)
                    mma_ss(tmem + C::COL_DX, ds_k + (uint64_t)(kk * 2), l_k + (uint64_t)(kk * 2), id_dx, kk > 0);
                mma_commit(dx_full);
                const uint32_t xa = smem_u32(sm + C::OFF_X + s * kTileBytes);
                const uint64_t xp = sdesc_sw128(xa, C::OFF_X2 - C::OFF_X, 1024);   // [x | x^2] as an MN-major A
#pragma unroll
                for (int kk = 0; kk < TM / 16; ++kk)
                    mma_ss(tmem + C::COL_P, xp + (uint64_t)(kk * 128), ds_mn + (uint64_t)(kk * 128), id_acc,
                           !(fresh && kk == 0));
                mma_commit(&xempty[s]);
                if (c.last()) {
                    mma_commit(acc_full);
                    mma_commit(h_empty);
                }
            }
            mma_commit(fin);
            wait_ignoring_abort(fin, 0, A.status);
        }
    } else {
        // ---------------- compute warps: thread r owns tile row r (TMEM lane r)
        const uint32_t r = 32u * (warp & 3) + lane;
        const uint32_t lane_off = (uint32_t)(32 * (warp & 3)) << 16;
        auto warp_arrive = [&](uint64_t *bar) {
            __syncwarp();
            if (lane == 0) mbar_arrive(bar);
        };
        float p0a = 0.f, p0b = 0.f;         // this warp's column sums of ds: columns 2 lane, 2 lane + 1
        float scale = 0.f;
        for (TileCursor c(t0, n, A.T, 0, 1); c.valid(); c.next()) {
            const int i = c.i, s = i & 1;
            const uint32_t ph = (uint32_t)i & 1u;
            const int row = c.j * TM + (int)r;
            const bool valid = row < A.N;
            if (c.first()) {
                if (i == 0) grid_dep_wait();
                scale = head_scale(A.params, A.param_stride, c.g % A.H, K);
            }
            // ---- [x, x^2/256] (fp16) into TMEM for the log-density; x^2 (bf16) for the parameter sums
            if (!mbar_wait_warp(&xfull[s], (i >> 1) & 1, ab, kDevErrTimeout)) break;
            const uint8_t *xs = sm + C::OFF_X + s * kTileBytes;
            convert_row(xs, r, tmem + lane_off + C::COL_A);
            {
                uint8_t *x2 = sm + C::OFF_X2 + s * kTileBytes;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const uint4 v = *reinterpret_cast<const uint4 *>(xs + sw128_off(r, j));
                    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
                    uint32_t o[4];
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const float lo = bf16_lo(w[u]), hi = bf16_hi(w[u]);
                        o[u] = pack_bf16(lo * lo, hi * hi);
                    }
                    *reinterpret_cast<uint4 *>(x2 + sw128_off(r, j)) = make_uint4(o[0], o[1], o[2], o[3]);
                }
            }
            tmem_st_wait();
            fence_proxy_async_smem();
            tc_fence_before();
            warp_arrive(a_full);
            // ---- Gamma = softmax of the scores (Eq. 3b), rows past the end 0; bf16 into G
            if (!mbar_wait_warp(d1_full, ph, ab, kDevErrTimeout)) break;
            tc_fence_after();
            float gam[K];
            {
                uint32_t e[K / 2];
                row_exp_scaled<K>(tmem + lane_off + C::COL_D1, scale, e);
                float q[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int t = 0; t < K / 2; ++t) {
                    q[(2 * t) & 3] += bf16_lo(e[t]);
                    q[(2 * t + 1) & 3] += bf16_hi(e[t]);
                }
                const float tot = (q[0] + q[1]) + (q[2] + q[3]);
                const float inv = valid ? 1.0f / tot : 0.f;
                uint8_t *gt = sm + C::OFF_G;
#pragma unroll
                for (int j = 0; j < K / 8; ++j) {
                    uint32_t wv[4];
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        wv[u] = pack_bf16(bf16_lo(e[4 * j + u]) * inv, bf16_hi(e[4 * j + u]) * inv);
                        gam[8 * j + 2 * u] = bf16_lo(wv[u]);          // the values the MMAs use
                        gam[8 * j + 2 * u + 1] = bf16_hi(wv[u]);
                    }
                    *reinterpret_cast<uint4 *>(gt + sw128_off(r, j)) = make_uint4(wv[0], wv[1], wv[2], wv[3]);
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            warp_arrive(g_full);
            if (MODE == kQuery) {
                // ---- a = dO / den, b = -(dO . O) / den from num = [Gamma Vt | Gamma Z | Gamma 1] (Eq. 7-8)
                bool w = mbar_wait_warp(num_full, ph, ab, kDevErrTimeout);
                w = w && mbar_wait_warp(&ufull[s], (i >> 1) & 1, ab, kDevErrTimeout);
                if (!w) break;
                tc_fence_after();
                uint32_t v0[32], v1[32], dz[4];
                tmem_ld32(tmem + lane_off + C::COL_NUM, v0);
                tmem_ld32(tmem + lane_off + C::COL_NUM + 32, v1);
                tmem_ld4(tmem + lane_off + C::COL_NUM + 64, dz);
                tmem_ld_wait();
                // den = Gamma Z + eps sum_k Gamma (the forward's normaliser, Gamma as rounded)
                const float den = valid ? __uint_as_float(dz[0]) + A.eps * __uint_as_float(dz[1]) : 1.0f;
                const float rd = 1.0f / den;
                const uint8_t *us = sm + C::OFF_U + s * kTileBytes;
                uint8_t *abt = sm + C::OFF_AB;
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
                    *reinterpret_cast<uint4 *>(abt + sw128_off(r, j)) = make_uint4(o[0], o[1], o[2], o[3]);
                }
                // b = -(dO . num) / den^2
                const float bv = -((dq[0] + dq[1]) + (dq[2] + dq[3])) * rd * rd;
                *reinterpret_cast<uint16_t *>(abt + kTileBytes + sw128_off(r, 0)) = (uint16_t)(pack_bf16(bv, 0.f) & 0xFFFFu);
                fence_proxy_async_smem();
                tc_fence_before();
                warp_arrive(ab_full);
                warp_arrive(&uempty[s]);
            }
            // ---- ds = gamma (g - gamma . g) (Eq. 17-18), bf16 into DS; its column sums for P0
            if (!mbar_wait_warp(gg_full, ph, ab, kDevErrTimeout)) break;
            tc_fence_after();
            {
                uint32_t gv[K];
                tmem_ld32(tmem + lane_off + C::COL_D1, gv);
                tmem_ld32(tmem + lane_off + C::COL_D1 + 32, gv + 32);
                tmem_ld_wait();
                float q[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int t = 0; t < K; ++t) q[t & 3] = fmaf(gam[t], __uint_as_float(gv[t]), q[t & 3]);
                const float mean = (q[0] + q[1]) + (q[2] + q[3]);
                float ds[K];
                uint8_t *dst = sm + C::OFF_DS;
#pragma unroll
                for (int j = 0; j < K / 8; ++j) {
                    uint32_t wv[4];
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const int t = 8 * j + 2 * u;
                        wv[u] = pack_bf16(gam[t] * (__uint_as_float(gv[t]) - mean),
                                          gam[t + 1] * (__uint_as_float(gv[t + 1]) - mean));
                        ds[t] = bf16_lo(wv[u]);                       // P0 sums the values the MMAs use
                        ds[t + 1] = bf16_hi(wv[u]);
                    }
                    *reinterpret_cast<uint4 *>(dst + sw128_off(r, j)) = make_uint4(wv[0], wv[1], wv[2], wv[3]);
                }
                fence_proxy_async_smem();
                tc_fence_before();
                warp_arrive(ds_full);
                const float2 cs = warp_colsum64(ds, lane);
                p0a += cs.x;
                p0b += cs.y;
            }
            // ---- dx = ds (lambda mu) - x (ds lambda) (section 4.3); keys: dV = Gamma^K R
            if (!mbar_wait_warp(dx_full, ph, ab, kDevErrTimeout)) break;
            tc_fence_after();
            {
                const bool store = valid && GMA_IN_BOUNDS(c.g < A.G, A.status);
                float *dxr = A.dX + ((size_t)c.g * A.N + (store ? row : 0)) * DR;
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    uint32_t c1[32], c2[32];
                    tmem_ld32(tmem + lane_off + C::COL_DX + 32 * half, c1);
                    tmem_ld32(tmem + lane_off + C::COL_DX + DR + 32 * half, c2);
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
                    tmem_ld32(tmem + lane_off + C::COL_NUM, v0);
                    tmem_ld32(tmem + lane_off + C::COL_NUM + 32, v1);
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
            warp_arrive(&xempty[s]);        // this warp has read its x rows (the P^T MMA is the other reader)
            // ---- head end: drain [R | r]^T (query) and P^T with P0 into partial slot (cta + head)
            if (c.last()) {
                if (!mbar_wait_warp(acc_full, c.hl & 1, ab, kDevErrTimeout)) break;
                tc_fence_after();
                const int slot = (int)blockIdx.x + c.g;
                const bool slot_ok = GMA_IN_BOUNDS(slot < A.nslots, A.status);
                uint32_t v[K];
                if (MODE == kQuery) {
                    tmem_ld32(tmem + lane_off + C::COL_R, v);
                    tmem_ld32(tmem + lane_off + C::COL_R + 32, v + 32);
                    tmem_ld_wait();
                    if (r <= (uint32_t)DVV && slot_ok) {
                        float4 *dst = reinterpret_cast<float4 *>(A.part_r + ((size_t)slot * (DVV + 1) + r) * K);
#pragma unroll
                        for (int t = 0; t < K / 4; ++t)
                            dst[t] = make_float4(__uint_as_float(v[4 * t]), __uint_as_float(v[4 * t + 1]),
                                                 __uint_as_float(v[4 * t + 2]), __uint_as_float(v[4 * t + 3]));
                    }
                }
                tmem_ld32(tmem + lane_off + C::COL_P, v);
                tmem_ld32(tmem + lane_off + C::COL_P + 32, v + 32);
                tmem_ld_wait();
                if (slot_ok) {
                    float *pp = A.part_p + (size_t)slot * kPartRows * K;
                    float4 *dst = reinterpret_cast<float4 *>(pp + (size_t)r * K);
#pragma unroll
                    for (int t = 0; t < K / 4; ++t)
                        dst[t] = make_float4(__uint_as_float(v[4 * t]), __uint_as_float(v[4 * t + 1]),
                                             __uint_as_float(v[4 * t + 2]), __uint_as_float(v[4 * t + 3]));
                    *reinterpret_cast<float2 *>(pp + (size_t)(2 * DR + (warp & 3)) * K + 2 * lane) = make_float2(p0a, p0b);
                }
                p0a = p0b = 0.f;
                tc_fence_before();
                warp_arrive(acc_empty);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kWMma) {
        __syncwarp();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

// The per-head bf16 operand [lambda | lambda mu] (K-major: row m < d holds lambda_{k, m}
// over the components k, row d + m holds lambda_{k, m} mu_{k, m}), from the fp32 lambda
// of the parameter prologue (Eq. 14).  One CTA per head.  It has no programmatic
// trigger, so a kernel launched after it starts once it has finished.
__global__ void __launch_bounds__(256) bwd_lamb_kernel(const float *__restrict__ mu, const float *__restrict__ lam,
                                                       uint8_t *__restrict__ out) {
    const int h = blockIdx.x;
    const float *mu_h = mu + (size_t)h * BK * DR, *lam_h = lam + (size_t)h * BK * DR;
    uint8_t *blk = out + (size_t)h * kLamBytes;
    for (int e = threadIdx.x; e < 2 * DR * (BK / 8); e += blockDim.x) {
        const int nrow = e / (BK / 8), j = e % (BK / 8), m = nrow % DR;
        uint32_t w[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            float v[2];
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                const int k = 8 * j + 2 * u + q;
                const float l = lam_h[k * DR + m];
                v[q] = nrow < DR ? l : l * mu_h[k * DR + m];
            }
            w[u] = pack_bf16(v[0], v[1]);
        }
        *reinterpret_cast<uint4 *>(blk + sw128_off(nrow, j)) = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

// Per head g, the fixed-order sum of the parameter-sum partial slots (c + g for the CTAs c
// that covered head g, in increasing c) into the finalize layout out[g][k][q]: q < d P1,
// d <= q < 2d P2, q = 2d P0 (the compute warps' rows in warp order).
__global__ void __launch_bounds__(256) bwd_psum_kernel(int T, int Ttot, int ncta, int nslots,
                                                       const float *__restrict__ part, float *__restrict__ out,
                                                       unsigned *status) {
    const int g = blockIdx.x;
    __shared__ int crange[2];
    if (threadIdx.x == 0) {
        const long long lo = (long long)g * T, hi = (long long)(g + 1) * T;
        int c = (int)((lo * ncta) / Ttot);
        while (c > 0 && ((long long)c * Ttot) / ncta > lo) --c;
        while (((long long)(c + 1) * Ttot) / ncta <= lo) ++c;
        int c_hi = c;
        while (c_hi < ncta && ((long long)c_hi * Ttot) / ncta < hi) ++c_hi;
        crange[0] = c;
        crange[1] = c_hi;
    }
    __syncthreads();
    const int c_lo = crange[0], c_hi = crange[1];
    if (!GMA_IN_BOUNDS(c_lo >= 0 && c_hi + g <= nslots, status)) return;
    for (int e = threadIdx.x; e < kPRows * BK; e += blockDim.x) {
        const int q = e / BK, k = e % BK;
        float s = 0.f;
        for (int c = c_lo; c < c_hi; ++c) {
            const float *pp = part + (size_t)(c + g) * kPartRows * BK;
            if (q < 2 * DR) {
                s += pp[(size_t)q * BK + k];
            } else {
                float w = pp[(size_t)(2 * DR) * BK + k];
                for (int u = 1; u < kGroupWarps; ++u) w += pp[(size_t)(2 * DR + u) * BK + k];
                s += w;
            }
        }
        out[((size_t)g * BK + k) * kPRows + q] = s;
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
    L.cdir = align_up(off);
    off = L.cdir + sizeof(float) * (size_t)p.H * BK;
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
    L.pq = align_up(off);
    off = L.pq + sizeof(float) * (size_t)p.G * BK * kPRows;
    L.pk = align_up(off);
    off = L.pk + sizeof(float) * (size_t)p.G * BK * kPRows;
    L.total = align_up(off);
    return L;
}

cudaError_t bwd_tc_run(const Problem &p, const BwdTcLayout &L, const void *Qx, const void *Kx, const void *V,
                       const float *mu, const float *rho, const float *alpha, const void *dO, float *dQx, float *dKx,
                       float *dV, float *dmu, float *drho, float *dalpha, char *ws, cudaStream_t s) {
    cudaError_t e;
    float *lam = reinterpret_cast<float *>(ws + L.lam);
    float *part_pq = reinterpret_cast<float *>(ws + L.part_pq), *part_pk = reinterpret_cast<float *>(ws + L.part_pk);
    float *pq = reinterpret_cast<float *>(ws + L.pq), *pk = reinterpret_cast<float *>(ws + L.pk);
    unsigned *status = reinterpret_cast<unsigned *>(ws);
    const int nslots = kMaxCtas + p.G;
    // parameter prologues: the log-density blocks of the forward, fp32 lambda, [lambda | lambda mu]
    if ((e = tc_params(p, L.tc, mu, rho, alpha, ws, s)) != cudaSuccess) return e;
    if ((e = simt_params(p, rho, alpha, lam, reinterpret_cast<float *>(ws + L.cdir), s)) != cudaSuccess) return e;
    bwd_lamb_kernel<<<p.H, 256, 0, s>>>(mu, lam, reinterpret_cast<uint8_t *>(ws + L.lamb));
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
    bwd_psum_kernel<<<p.G, 256, 0, s>>>(L.tc.Tkv, L.tc.Ttot_kv, L.tc.ncta_kv, nslots, part_pq, pq, status);
    bwd_psum_kernel<<<p.G, 256, 0, s>>>(L.tc.Tkv, L.tc.Ttot_kv, L.tc.ncta_kv, nslots, part_pk, pk, status);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    return bwd_finalize(p, 1, pq, pk, mu, lam, rho, alpha, dmu, drho, dalpha, s);
}

}  // namespace gma
