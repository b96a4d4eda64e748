// Responsibility diagnostics on the tensor cores, for bf16 routing vectors with
// d = 64 and K in {64, 128}.
//
// "Gaussian Mixture Attention" (Huang & Raza, 2026), section 5.4, Eqs. 24-29,
// over the query responsibilities of every head (Eq. 3b):
//   gbar_{t,k} = (1/H) sum_h gamma^Q_{t,h,k}          head average of one token (Eq. 24)
//   p_k        = (1/T) sum_t gbar_{t,k}                marginal usage (Eq. 25)
//   H_usage    = -sum_k p_k log p_k / log K            (Eq. 26)
//   H_token    = (1/T) sum_t -sum_k gbar log gbar / log K   (Eq. 27)
//   R_max      = (1/T) sum_t max_k gbar_{t,k}          (Eq. 28)
//   z_t        = argmax_k gbar_{t,k}, ties to the lowest index   (Eq. 29)
//
// tc_diag: persistent CTAs over 128-token tiles (batch entry b, rows j..j+127);
// for each tile the CTA loops over the H heads: TMA load of that head's Qx tile,
// the log-density MMA of section 4.1 (the same [x, x^2/256] . W^T + c form as the
// forward, N = K score columns in TMEM), the scores read once into registers (the
// columns go back to the next head's MMA at once), softmax in registers, and the
// head's responsibilities added to a K-wide fp32 sum over the heads (in registers
// at K = 64, in TMEM columns at K = 128).  After the last
// head each thread (one token) has gbar in registers: its entropy, maximum and
// argmax, and a warp transpose-reduce adds the tile's column sums to per-warp
// partials of p.  Responsibilities never leave the SM.
// tc_diag_finalize: one CTA sums the per-CTA partials in a fixed order and
// writes p [K] and {H_usage, H_token, R_max}.
// Warps: 0 TMA producer (Qx tiles and parameter blocks); 1 TMEM owner and MMA
// issuer; 2-5 the epilogue group; 6-9 the convert group (bf16 tile -> [x, x^2/256]
// operand, double-buffered, overlapping the previous step's epilogue).  Every
// mbarrier wait is bounded.
#include <cuda.h>
#include <cuda_bf16.h>

#include <algorithm>

#include "gma_internal.h"
#include "gma_sm100.cuh"
#include "gma_tc_common.cuh"

namespace gma {

using namespace sm100;
using namespace tc;

namespace {

constexpr int kDiagThreads = 320;        // warps: producer, MMA, epilogue group, convert group
constexpr int kDiagX = 4;                 // routing-tile ring stages
constexpr int kDiagMaxHeads = 1024;       // head scales kept in shared memory

template <int K>
struct DiagCfg {
    static constexpr uint32_t PB = align1k(param_bytes(K));
    static constexpr uint32_t OFF_X = 0;
    static constexpr uint32_t OFF_P = OFF_X + kDiagX * kTileBytes;         // 2 parameter buffers
    static constexpr uint32_t OFF_CA = OFF_P + 2 * PB;
    static constexpr uint32_t OFF_SC = OFF_CA + kConstABytes;              // [kDiagMaxHeads] head scales
    static constexpr uint32_t OFF_PACC = OFF_SC + 4 * kDiagMaxHeads;       // [4 warps][K] column sums
    static constexpr uint32_t OFF_BAR = OFF_PACC + 4 * 4 * K;
    static constexpr uint32_t BYTES = OFF_BAR + 256 + 1024;
    static constexpr uint32_t COL_A = 0;          // two [x, x^2/256] operands, 64 columns each
    static constexpr uint32_t COL_D = 128;        // K fp32 scores
    static constexpr uint32_t COL_ACC = 128 + K;  // K fp32: sum over the heads so far
    static constexpr uint32_t TMEM_COLS = 512;
    static_assert(COL_ACC + K <= TMEM_COLS && BYTES <= 232448, "diagnostics kernel exceeds TMEM or shared memory");
};

struct DiagArgs {
    int B, H, N, T, Ttot;     // tiles (b, j) in that order, Ttot = B T; steps = tiles x heads
    const uint8_t *params;
    uint32_t param_stride;
    float *part;              // [gridDim.x][K + 2]: column sums of gbar, sum of entropies, sum of maxima
    int *z;                   // [B][N] or nullptr
    unsigned *status;
};

// Sums 32 values v[0..31] of each lane over the 32 lanes of the warp: afterwards
// lane l holds the sum of value l (a transpose-reduce, 31 shuffles, fixed order).
__device__ __forceinline__ float warp_column_sums(float (&v)[32], int lane) {
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
        const bool up = (lane & o) != 0;
#pragma unroll
        for (int i = 0; i < o; ++i) {
            const float give = up ? v[i] : v[i + o];
            const float keep = up ? v[i + o] : v[i];
            v[i] = keep + __shfl_xor_sync(~0u, give, o);
        }
    }
    return v[0];
}

template <int K>
__global__ void __launch_bounds__(kDiagThreads, 1)
tc_diag_kernel(const __grid_constant__ CUtensorMap tm_q, DiagArgs A) {
    using C = DiagCfg<K>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + C::OFF_BAR);
    uint64_t *xfull = bars, *xempty = xfull + kDiagX, *a_full = xempty + kDiagX;   // a_full[2]
    uint64_t *d_full = a_full + 2, *d_empty = d_full + 1, *w_full = d_empty + 1;   // w_full[2]
    uint64_t *w_empty = w_full + 2, *a_empty = w_empty + 2, *fin = a_empty + 2;   // w_empty[2], a_empty[2]
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(fin + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    float *scales = reinterpret_cast<float *>(sm + C::OFF_SC);
    float *pacc = reinterpret_cast<float *>(sm + C::OFF_PACC);

    grid_dep_launch();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // contiguous range of tiles, each taken for all H heads: steps s = (tile, head)
    const int u0 = (int)(((long long)blockIdx.x * A.Ttot) / gridDim.x);
    const int u1 = (int)(((long long)(blockIdx.x + 1) * A.Ttot) / gridDim.x);
    const int nsteps = (u1 - u0) * A.H;

    if (threadIdx.x == 0) {
        for (uint64_t *b = bars; b <= fin; ++b) mbar_init(b, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    init_const_a(sm + C::OFF_CA, threadIdx.x, blockDim.x);
    for (int e = threadIdx.x; e < 4 * K; e += blockDim.x) pacc[e] = 0.f;
    if (warp == 1) { tmem_alloc(tmem_slot, C::TMEM_COLS); tmem_relinquish(); }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const Abort ab{abort_flag, A.status};
    auto step_head = [&](int s) { return s % A.H; };
    auto step_tile = [&](int s) { return u0 + s / A.H; };

    if (warp == 0) {
        if (lane == 0 && nsteps > 0) {
            grid_dep_wait();                               // the parameter blocks are written
            int xs = 0, ws = 0;                            // next step to load: routing tile, parameters
            long long last = now_ns();
            while ((xs < nsteps || ws < nsteps) && !*abort_flag) {
                bool progress = false;
                if (ws < nsteps && (ws < 2 || mbar_test(&w_empty[ws & 1], ((ws >> 1) - 1) & 1))) {
                    mbar_arrive_expect_tx(&w_full[ws & 1], param_bytes(K));
                    bulk_load(sm + C::OFF_P + (ws & 1) * C::PB,
                              A.params + (size_t)step_head(ws) * A.param_stride, param_bytes(K), &w_full[ws & 1]);
                    ++ws;
                    progress = true;
                }
                if (xs < nsteps && (xs < kDiagX || mbar_test(&xempty[xs % kDiagX], ((xs / kDiagX) - 1) & 1))) {
                    const int u = step_tile(xs), b = u / A.T, j = u % A.T;
                    mbar_arrive_expect_tx(&xfull[xs % kDiagX], kTileBytes);
                    tma_load_3d(sm + C::OFF_X + (xs % kDiagX) * kTileBytes, &tm_q, &xfull[xs % kDiagX], 0, j * TM,
                                b * A.H + step_head(xs));
                    ++xs;
                    progress = true;
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
            wind_down_ring(xfull, kDiagX, xs, A.status);
            for (int s = ws - 2 < 0 ? 0 : ws - 2; s < ws; ++s) wait_ignoring_abort(&w_full[s & 1], (s >> 1) & 1, A.status);
        }
    } else if (warp == 1) {
        // log-density MMA of step s into the score columns, once step s - 1's scores are read
        if (nsteps > 0) {                            // the whole warp, converged
            const uint32_t ca = smem_u32(sm + C::OFF_CA);
            bool ok = true;
            for (int s = 0; s < nsteps && ok; ++s) {
                ok = mbar_wait_warp(&w_full[s & 1], (s >> 1) & 1, ab, kDevErrTimeout) &&
                     mbar_wait_warp(&a_full[s & 1], (s >> 1) & 1, ab, kDevErrTimeout);
                if (ok && s >= 1) ok = mbar_wait_warp(d_empty, (s - 1) & 1, ab, kDevErrTimeout);
                if (!ok) break;
                tc_fence_after();
                issue_logdensity<K>(tmem + C::COL_D, tmem + C::COL_A + (s & 1) * 64,
                                    smem_u32(sm + C::OFF_P + (s & 1) * C::PB), ca);
                mma_commit(d_full);
                mma_commit(&xempty[s % kDiagX]);
                mma_commit(&w_empty[s & 1]);
                mma_commit(&a_empty[s & 1]);
            }
            mma_commit(fin);
            wait_ignoring_abort(fin, 0, A.status);
        }
    } else if (warp >= 6) {
        // convert group: step s's [x, x^2/256] operand into buffer s & 1 once the MMA of step
        // s - 2 has read that buffer
        RowThread rt;
        rt.wg = 1;
        rt.r = 32u * (warp & 3) + lane;
        rt.lane_off = (uint32_t)(32 * (warp & 3)) << 16;
        rt.wtid = threadIdx.x - 192;
        const bool elected = rt.wtid == 0;
        for (int s = 0; s < nsteps; ++s) {
            bool w = mbar_wait(&xfull[s % kDiagX], (s / kDiagX) & 1, ab, kDevErrTimeout);
            if (s >= 2) w = w && mbar_wait(&a_empty[s & 1], ((s >> 1) - 1) & 1, ab, kDevErrTimeout);
            if (!wg_all(rt, w)) break;
            tc_fence_after();
            convert_row(sm + C::OFF_X + (s % kDiagX) * kTileBytes, rt.r, tmem + rt.lane_off + C::COL_A + (s & 1) * 64);
            tmem_st_wait();
            tc_fence_before();
            wg_sync(rt);
            if (elected) mbar_arrive(&a_full[s & 1]);
        }
    } else {
        RowThread rt;
        rt.wg = 0;
        rt.r = 32u * (warp & 3) + lane;
        rt.lane_off = (uint32_t)(32 * (warp & 3)) << 16;
        rt.wtid = threadIdx.x - 64;
        const bool elected = rt.wtid == 0;
        // every head's coefficient scale (the parameter blocks are the previous kernel's output)
        grid_dep_wait();
        const int hs = A.H < kDiagMaxHeads ? A.H : kDiagMaxHeads;
        for (int h = rt.wtid; h < hs; h += kWgThreads) scales[h] = head_scale(A.params, A.param_stride, h, K);
        wg_sync(rt);
        const uint32_t dcol = tmem + rt.lane_off + C::COL_D, acol = tmem + rt.lane_off + C::COL_ACC;
        float ent_sum = 0.f, max_sum = 0.f;       // over this thread's tokens
        constexpr bool kRegAcc = K <= 64;          // the sum over heads in registers (else in TMEM)
        float racc[kRegAcc ? K : 1];
        bool ok = true;
        for (int s = 0; s < nsteps && ok; ++s) {
            const int h = step_head(s), u = step_tile(s), b = u / A.T, j = u % A.T;
            const float scale = h < kDiagMaxHeads ? scales[h] : head_scale(A.params, A.param_stride, h, K);
            const bool w = mbar_wait(d_full, s & 1, ab, kDevErrTimeout);
            if (!(ok = wg_all(rt, w))) break;
            tc_fence_after();
            // this head's scores in registers (one TMEM round trip); the score columns go back to
            // the MMA of the next head at once, so that it overlaps the softmax below
            uint32_t v[K];
#pragma unroll
            for (int cc = 0; cc < K / 32; ++cc) tmem_ld32(dcol + 32 * cc, v + 32 * cc);
            tmem_ld_wait();
            tc_fence_before();
            wg_sync(rt);
            if (elected) mbar_arrive(d_empty);
            // the head's responsibilities (Eq. 3b): the row maximum, fp32 exponentials and their
            // sum, then the normalised values added to the sum over the heads
            float m = -INFINITY;
#pragma unroll
            for (int t = 0; t < K; ++t) m = fmaxf(m, __uint_as_float(v[t]));
            const float M = m * scale;
            float sum = 0.f;
#pragma unroll
            for (int t = 0; t < K; ++t) {
                const float x = ex2_approx(fmaf(__uint_as_float(v[t]), scale, -M));
                sum += x;
                v[t] = __float_as_uint(x);
            }
            const float inv = 1.0f / sum;
            const bool last = h + 1 == A.H;
            const float invH = 1.0f / (float)A.H;
            const int row = j * TM + (int)rt.r;
            const bool valid = row < A.N;
            float ent = 0.f, mx = -1.f;
            int arg = 0;
            // gbar of this token on the last head (Eq. 24): entropy (Eq. 27), maximum and argmax
            // (Eq. 28-29), and one 32-column chunk's column sums over the tile's tokens (Eq. 25),
            // one partial per warp
            auto finish_chunk = [&](float (&g)[32], int cc) {
#pragma unroll
                for (int t = 0; t < 32; ++t) {
                    const float gb = g[t] * invH;
                    ent -= gb > 0.f ? gb * __logf(gb) : 0.f;
                    if (gb > mx) { mx = gb; arg = 32 * cc + t; }
                    g[t] = valid ? gb : 0.f;
                }
                pacc[(warp & 3) * K + 32 * cc + lane] += warp_column_sums(g, lane);
            };
            if constexpr (kRegAcc) {
#pragma unroll
                for (int t = 0; t < K; ++t)
                    racc[t] = h > 0 ? fmaf(__uint_as_float(v[t]), inv, racc[t]) : __uint_as_float(v[t]) * inv;
                if (last) {
#pragma unroll
                    for (int cc = 0; cc < K / 32; ++cc) {
                        float g[32];
#pragma unroll
                        for (int t = 0; t < 32; ++t) g[t] = racc[32 * cc + t];
                        finish_chunk(g, cc);
                    }
                }
            } else {
#pragma unroll
                for (int cc = 0; cc < K / 32; ++cc) {
                    float g[32];
                    if (h > 0) {
                        uint32_t acc[32];
                        tmem_ld32(acol + 32 * cc, acc);
                        tmem_ld_wait();
#pragma unroll
                        for (int t = 0; t < 32; ++t)
                            g[t] = fmaf(__uint_as_float(v[32 * cc + t]), inv, __uint_as_float(acc[t]));
                    } else {
#pragma unroll
                        for (int t = 0; t < 32; ++t) g[t] = __uint_as_float(v[32 * cc + t]) * inv;
                    }
                    if (!last)
                        tmem_st32(acol + 32 * cc, reinterpret_cast<const uint32_t *>(g));   // the sum over heads
                    else
                        finish_chunk(g, cc);
                }
                if (!last) tmem_st_wait();
            }
            if (last && valid) {
                ent_sum += ent;
                max_sum += mx;
                if (A.z) A.z[(size_t)b * A.N + row] = arg;
            }
        }
        // this CTA's partials: column sums over the four warps, entropy and maximum sums over
        // the group (fixed orders); written even when the CTA had no tile
        for (int o = 16; o >= 1; o >>= 1) {
            ent_sum += __shfl_xor_sync(~0u, ent_sum, o);
            max_sum += __shfl_xor_sync(~0u, max_sum, o);
        }
        float *red = scales;                       // the scales are no longer needed
        wg_sync(rt);
        if (lane == 0) { red[warp & 3] = ent_sum; red[4 + (warp & 3)] = max_sum; }
        wg_sync(rt);
        float *dst = A.part + (size_t)blockIdx.x * (K + 2);
        for (int k = rt.wtid; k < K; k += kWgThreads)
            dst[k] = ((pacc[k] + pacc[K + k]) + pacc[2 * K + k]) + pacc[3 * K + k];
        if (rt.wtid == 0) {
            dst[K] = ((red[0] + red[1]) + red[2]) + red[3];
            dst[K + 1] = ((red[4] + red[5]) + red[6]) + red[7];
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) {
        __syncwarp();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

// p [K] and {H_usage, H_token, R_max} from the per-CTA partials (at most kMaxCtas of them, fp32
// sums suffice).  Thread (q, k) sums column k of the CTAs c = q (mod kFinGroups) with four
// independent accumulators (the loads stay in flight); the groups' sums and the p log p terms
// are combined in a fixed order.
constexpr int kFinGroups = 6, kFinCols = 160;      // kFinCols >= K + 2 for K <= 128

__global__ void __launch_bounds__(kFinGroups * kFinCols) tc_diag_finalize_kernel(int K, int ncta, float T,
                                                                                const float *__restrict__ part,
                                                                                float *__restrict__ p_out,
                                                                                float *__restrict__ stats_out) {
    grid_dep_launch();
    grid_dep_wait();                                       // the partials are written
    __shared__ float gsum[kFinGroups][kFinCols];
    __shared__ float term[kFinCols];
    const int k = threadIdx.x % kFinCols, q = threadIdx.x / kFinCols, w = K + 2;
    float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
    if (k < w) {
        int c = q;
        for (; c + 3 * kFinGroups < ncta; c += 4 * kFinGroups) {
            a0 += part[(size_t)c * w + k];
            a1 += part[(size_t)(c + kFinGroups) * w + k];
            a2 += part[(size_t)(c + 2 * kFinGroups) * w + k];
            a3 += part[(size_t)(c + 3 * kFinGroups) * w + k];
        }
        for (; c < ncta; c += kFinGroups) a0 += part[(size_t)c * w + k];
    }
    gsum[q][k] = (a0 + a1) + (a2 + a3);
    __syncthreads();
    if (q == 0) {
        float acc = 0.f;
        for (int g = 0; g < kFinGroups; ++g) acc += gsum[g][k];
        const float pk = acc / T;
        term[k] = k < K && pk > 0.f ? -pk * logf(pk) : 0.f;
        if (k < K) p_out[k] = pk;
        if (k == K || k == K + 1) gsum[0][k] = acc;        // read back by thread 0 below
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        float hu = 0.f;
        for (int kk = 0; kk < K; ++kk) hu += term[kk];
        const float logK = logf((float)K);
        stats_out[0] = hu / logK;
        stats_out[1] = gsum[0][K] / T / logK;
        stats_out[2] = gsum[0][K + 1] / T;
    }
}

// ------------------------------------------------------------------ tc_diag2 (K = 64)
//
// The same computation at K = 64 with two epilogue groups: group w takes the CTA's tiles
// w, w + 2, ... (each tile for all H heads, its head sum in registers) and converts its own
// routing tiles, so that one group's softmax overlaps the other's log-density MMA and
// conversion.  The MMA issuer interleaves the groups' steps, (group 0, step k), (group 1,
// step k), ...; both use head k % H at step k, so one parameter block serves both.  Each
// group converts step k + 1 once it has added step k's responsibilities to its head sum
// (its one [x, x^2/256] operand is free once step k's MMA is done), so that MMA overlaps
// the last head's statistics and the other group's work.
constexpr int kDiag2Threads = 320;        // warps: producer, MMA, epilogue groups 0 and 1
constexpr int kDiag2X = 6, kDiag2W = 4;   // routing-tile and parameter-block ring stages

struct Diag2Cfg {
    static constexpr int K = 64;
    static constexpr uint32_t PB = align1k(param_bytes(K));
    static constexpr uint32_t OFF_X = 0;
    static constexpr uint32_t OFF_P = OFF_X + kDiag2X * kTileBytes;         // kDiag2W parameter buffers
    static constexpr uint32_t OFF_CA = OFF_P + kDiag2W * PB;
    static constexpr uint32_t OFF_SC = OFF_CA + kConstABytes;               // [kDiagMaxHeads] head scales
    static constexpr uint32_t OFF_PACC = OFF_SC + 4 * kDiagMaxHeads;        // [8 warps][K] column sums
    static constexpr uint32_t OFF_RED = OFF_PACC + 8 * 4 * K;               // [16]: entropy, maximum sums per warp
    static constexpr uint32_t OFF_BAR = OFF_RED + 16 * 4;
    static constexpr uint32_t BYTES = OFF_BAR + 256 + 1024;
    static constexpr uint32_t COL_GRP = 128, COL_A = 0, COL_D = 64;         // group w: operand, then K scores
    static constexpr uint32_t TMEM_COLS = 256;
    static_assert(BYTES <= 232448 && OFF_P % 1024 == 0, "diagnostics kernel layout");
};

__global__ void __launch_bounds__(kDiag2Threads, 1)
tc_diag2_kernel(const __grid_constant__ CUtensorMap tm_q, DiagArgs A) {
    using C = Diag2Cfg;
    constexpr int K = C::K;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + C::OFF_BAR);
    uint64_t *xfull = bars, *xempty = xfull + kDiag2X, *w_full = xempty + kDiag2X, *w_empty = w_full + kDiag2W;
    uint64_t *a_full = w_empty + kDiag2W, *d_full = a_full + 2, *d_empty = d_full + 2, *fin = d_empty + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(fin + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    float *scales = reinterpret_cast<float *>(sm + C::OFF_SC);
    float *pacc = reinterpret_cast<float *>(sm + C::OFF_PACC);
    float *red = reinterpret_cast<float *>(sm + C::OFF_RED);

    grid_dep_launch();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // contiguous range of tiles; group w takes tiles u0 + w + 2 m, each for all H heads
    const int u0 = (int)(((long long)blockIdx.x * A.Ttot) / gridDim.x);
    const int u1 = (int)(((long long)(blockIdx.x + 1) * A.Ttot) / gridDim.x);
    const int nt = u1 - u0;
    const int n0 = ((nt + 1) / 2) * A.H, n1 = (nt / 2) * A.H;       // steps of groups 0 and 1 (n0 >= n1)
    const int ntot = n0 + n1;
    // global order of the steps: (0, k), (1, k) while both groups have steps, then group 0's rest
    auto gidx = [&](int w, int k) { return k < n1 ? 2 * k + w : 2 * n1 + (k - n1); };
    auto gstep = [&](int idx, int &w, int &k) {
        if (idx < 2 * n1) { w = idx & 1; k = idx >> 1; } else { w = 0; k = n1 + (idx - 2 * n1); }
    };
    auto step_tile = [&](int w, int k) { return u0 + w + 2 * (k / A.H); };

    if (threadIdx.x == 0) {
        for (uint64_t *b = bars; b <= fin; ++b) mbar_init(b, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    init_const_a(sm + C::OFF_CA, threadIdx.x, blockDim.x);
    for (int e = threadIdx.x; e < 8 * K; e += blockDim.x) pacc[e] = 0.f;
    if (warp == 1) { tmem_alloc(tmem_slot, C::TMEM_COLS); tmem_relinquish(); }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const Abort ab{abort_flag, A.status};

    if (warp == 0) {
        if (lane == 0 && ntot > 0) {
            grid_dep_wait();                               // the parameter blocks are written
            int xs = 0, ws = 0;                            // next to load: global step (routing tile), k (parameters)
            long long last = now_ns();
            while ((xs < ntot || ws < n0) && !*abort_flag) {
                bool progress = false;
                if (ws < n0 && (ws < kDiag2W || mbar_test(&w_empty[ws % kDiag2W], ((ws / kDiag2W) - 1) & 1))) {
                    mbar_arrive_expect_tx(&w_full[ws % kDiag2W], param_bytes(K));
                    bulk_load(sm + C::OFF_P + (ws % kDiag2W) * C::PB, A.params + (size_t)(ws % A.H) * A.param_stride,
                              param_bytes(K), &w_full[ws % kDiag2W]);
                    ++ws;
                    progress = true;
                }
                if (xs < ntot && (xs < kDiag2X || mbar_test(&xempty[xs % kDiag2X], ((xs / kDiag2X) - 1) & 1))) {
                    int w, k;
                    gstep(xs, w, k);
                    const int u = step_tile(w, k), b = u / A.T, j = u % A.T;
                    (void)GMA_IN_BOUNDS(u < A.Ttot && b < A.B, A.status);
                    mbar_arrive_expect_tx(&xfull[xs % kDiag2X], kTileBytes);
                    tma_load_3d(sm + C::OFF_X + (xs % kDiag2X) * kTileBytes, &tm_q, &xfull[xs % kDiag2X], 0, j * TM,
                                b * A.H + k % A.H);
                    ++xs;
                    progress = true;
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
            wind_down_ring(xfull, kDiag2X, xs, A.status);
            wind_down_ring(w_full, kDiag2W, ws, A.status);
        }
    } else if (warp == 1) {
        // the log-density MMA of each step, in the global order, into the group's score columns
        if (ntot > 0) {                               // the whole warp, converged
            const uint32_t ca = smem_u32(sm + C::OFF_CA);
            bool ok = true;
            for (int idx = 0; idx < ntot && ok; ++idx) {
                int w, k;
                gstep(idx, w, k);
                if (w == 0) ok = mbar_wait_warp(&w_full[k % kDiag2W], (k / kDiag2W) & 1, ab, kDevErrTimeout);
                ok = ok && mbar_wait_warp(&a_full[w], k & 1, ab, kDevErrTimeout);
                if (ok && k >= 1) ok = mbar_wait_warp(&d_empty[w], (k - 1) & 1, ab, kDevErrTimeout);
                if (!ok) break;
                tc_fence_after();
                issue_logdensity<K>(tmem + w * C::COL_GRP + C::COL_D, tmem + w * C::COL_GRP + C::COL_A,
                                    smem_u32(sm + C::OFF_P + (k % kDiag2W) * C::PB), ca);
                mma_commit(&d_full[w]);
                if (w == 1 || k >= n1) mma_commit(&w_empty[k % kDiag2W]);   // the last step to use parameters k
            }
            mma_commit(fin);
            wait_ignoring_abort(fin, 0, A.status);
        }
    } else {
        // ---------------- epilogue group w (warps 2-5, 6-9): one thread per token of the group's tiles
        const int w = (warp - 2) >> 2;
        RowThread rt;
        rt.wg = w;
        rt.r = 32u * (warp & 3) + lane;
        rt.lane_off = (uint32_t)(32 * (warp & 3)) << 16;
        rt.wtid = threadIdx.x - 64 - w * kWgThreads;
        const bool elected = rt.wtid == 0;
        const int nw = w == 0 ? n0 : n1;
        grid_dep_wait();
        const int hs = A.H < kDiagMaxHeads ? A.H : kDiagMaxHeads;
        if (w == 0)
            for (int h = rt.wtid; h < hs; h += kWgThreads) scales[h] = head_scale(A.params, A.param_stride, h, K);
        group_sync(3, 2 * kWgThreads);                   // both groups, once, before any wait: the scales are in place
        const uint32_t acol = tmem + rt.lane_off + w * C::COL_GRP + C::COL_A;
        const uint32_t dcol = tmem + rt.lane_off + w * C::COL_GRP + C::COL_D;
        float ent_sum = 0.f, max_sum = 0.f;
        uint64_t racc[K / 2];                            // the sum over heads, as fp32 pairs
        // step k's routing tile into the operand (once step k - 1's MMA is done: its scores are read)
        auto convert = [&](int k) -> bool {
            const int idx = gidx(w, k);
            const bool ok = mbar_wait(&xfull[idx % kDiag2X], (idx / kDiag2X) & 1, ab, kDevErrTimeout);
            if (!wg_all(rt, ok)) return false;
            convert_row(sm + C::OFF_X + (idx % kDiag2X) * kTileBytes, rt.r, acol);
            tmem_st_wait();
            tc_fence_before();
            wg_sync(rt);
            if (elected) { mbar_arrive(&a_full[w]); mbar_arrive(&xempty[idx % kDiag2X]); }
            return true;
        };
        bool ok = nw == 0 || convert(0);
        for (int k = 0; k < nw && ok; ++k) {
            const int h = k % A.H, u = step_tile(w, k), b = u / A.T, j = u % A.T;
            const float scale = h < kDiagMaxHeads ? scales[h] : head_scale(A.params, A.param_stride, h, K);
            const bool wt = mbar_wait(&d_full[w], k & 1, ab, kDevErrTimeout);
            if (!(ok = wg_all(rt, wt))) break;
            tc_fence_after();
            uint32_t v[K];
            tmem_ld32(dcol, v);
            tmem_ld32(dcol + 32, v + 32);
            tmem_ld_wait();
            tc_fence_before();
            wg_sync(rt);
            if (elected) mbar_arrive(&d_empty[w]);
            // four independent chains for the maximum and the sum (fixed order), the exponent
            // arguments and the head sum as fp32 pairs
            float m4[4] = {__uint_as_float(v[0]), __uint_as_float(v[1]), __uint_as_float(v[2]), __uint_as_float(v[3])};
#pragma unroll
            for (int t = 4; t < K; t += 4)
#pragma unroll
                for (int q = 0; q < 4; ++q) m4[q] = fmaxf(m4[q], __uint_as_float(v[t + q]));
            const float M = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3])) * scale;
            const uint64_t sc2 = f2_pack(scale, scale), nm2 = f2_pack(-M, -M);
            float s4[4] = {0.f, 0.f, 0.f, 0.f};
            uint64_t e2[K / 2];
#pragma unroll
            for (int t = 0; t < K / 2; ++t) {
                float xa, xb;
                f2_unpack(f2_fma(f2_pack(__uint_as_float(v[2 * t]), __uint_as_float(v[2 * t + 1])), sc2, nm2), xa, xb);
                xa = ex2_approx(xa);
                xb = ex2_approx(xb);
                s4[(2 * t) & 3] += xa;
                s4[(2 * t + 1) & 3] += xb;
                e2[t] = f2_pack(xa, xb);
            }
            const float inv = 1.0f / ((s4[0] + s4[1]) + (s4[2] + s4[3]));
            const uint64_t inv2 = f2_pack(inv, inv);
#pragma unroll
            for (int t = 0; t < K / 2; ++t) racc[t] = h > 0 ? f2_fma(e2[t], inv2, racc[t]) : f2_mul(e2[t], inv2);
            // the next step's operand (its MMA overlaps this step's statistics and the other group)
            if (k + 1 < nw && !(ok = convert(k + 1))) break;
            if (h + 1 == A.H) {
                // gbar of this token (Eq. 24): entropy (Eq. 27), maximum and argmax (Eq. 28-29),
                // and the tile's column sums (Eq. 25), one partial per warp
                const float invH = 1.0f / (float)A.H;
                const int row = j * TM + (int)rt.r;
                const bool valid = row < A.N;
                float ent4[4] = {0.f, 0.f, 0.f, 0.f}, mx = -1.f;
                int arg = 0;
#pragma unroll
                for (int cc = 0; cc < K / 32; ++cc) {
                    float g[32];
#pragma unroll
                    for (int t = 0; t < 16; ++t) {
                        float ga, gb2;
                        f2_unpack(racc[16 * cc + t], ga, gb2);
                        g[2 * t] = ga * invH;
                        g[2 * t + 1] = gb2 * invH;
                    }
#pragma unroll
                    for (int t = 0; t < 32; ++t) {
                        const float gb = g[t];
                        ent4[t & 3] -= gb > 0.f ? gb * __logf(gb) : 0.f;
                        if (gb > mx) { mx = gb; arg = 32 * cc + t; }
                        g[t] = valid ? gb : 0.f;
                    }
                    pacc[(4 * w + (warp & 3)) * K + 32 * cc + lane] += warp_column_sums(g, lane);
                }
                const float ent = (ent4[0] + ent4[1]) + (ent4[2] + ent4[3]);
                if (valid) {
                    ent_sum += ent;
                    max_sum += mx;
                    if (A.z) A.z[(size_t)b * A.N + row] = arg;
                }
            }
        }
        for (int o = 16; o >= 1; o >>= 1) {
            ent_sum += __shfl_xor_sync(~0u, ent_sum, o);
            max_sum += __shfl_xor_sync(~0u, max_sum, o);
        }
        if (lane == 0) { red[4 * w + (warp & 3)] = ent_sum; red[8 + 4 * w + (warp & 3)] = max_sum; }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // this CTA's partials: column sums over the eight warps, entropy and maximum sums (fixed
    // orders); written even when the CTA had no tile
    if (warp >= 2 && warp < 6) {
        const int t = threadIdx.x - 64;
        float *dst = A.part + (size_t)blockIdx.x * (K + 2);
        for (int k = t; k < K; k += kWgThreads) {
            float acc = pacc[k];
            for (int x = 1; x < 8; ++x) acc += pacc[x * K + k];
            dst[k] = acc;
        }
        if (t == 0) {
            float e = red[0], m = red[8];
            for (int x = 1; x < 8; ++x) { e += red[x]; m += red[8 + x]; }
            dst[K] = e;
            dst[K + 1] = m;
        }
    }
    if (warp == 1) {
        __syncwarp();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

template <int K>
cudaError_t launch_diag(const Problem &p, const TcLayout &L, const void *Qx, int *z, char *ws, cudaStream_t s) {
    CUtensorMap tq;
    if (!make_map(&tq, Qx, p.G, p.N, DR)) return cudaErrorInvalidValue;
    DiagArgs a{};
    a.B = p.B; a.H = p.H; a.N = p.N; a.T = L.T; a.Ttot = L.Ttot;
    a.params = reinterpret_cast<const uint8_t *>(ws + L.params);
    a.param_stride = L.param_stride;
    a.part = reinterpret_cast<float *>(ws + L.part);
    a.z = z;
    a.status = reinterpret_cast<unsigned *>(ws);
    auto kern = tc_diag_kernel<K>;
    cudaError_t e = set_dyn_smem(reinterpret_cast<const void *>(kern), DiagCfg<K>::BYTES);
    if (e != cudaSuccess) return e;
    return launch_dependent(kern, dim3(L.ncta), dim3(kDiagThreads), DiagCfg<K>::BYTES, s, tq, a);
}

}  // namespace

bool tc_diag_supported(const Problem &p) {
    return p.in_dtype == GMA_BF16 && p.d == DR && (p.K == 64 || p.K == 128) && p.N > 0;
}

TcLayout tc_diag_layout(const Problem &p) {
    TcLayout L{};
    L.T = (p.N + TM - 1) / TM;
    L.Ttot = L.T * p.B;                                   // 128-token tiles (b, j)
    const int nsm = sm_count();
    L.ncta = std::max(1, std::min({nsm > 0 ? nsm : kMaxCtas, kMaxCtas, L.Ttot}));
    L.param_stride = align1k(param_bytes(p.K));
    L.params = align_up(kHeaderBytes);
    L.part = align_up(L.params + (size_t)p.H * L.param_stride);
    L.mem = L.part;
    L.total = align_up(L.part + sizeof(float) * (size_t)L.ncta * (p.K + 2));
    return L;
}

cudaError_t tc_diag(const Problem &p, const TcLayout &L, const void *Qx, int *z, char *ws, cudaStream_t s) {
    if (p.K != 64) return launch_diag<128>(p, L, Qx, z, ws, s);
    CUtensorMap tq;
    if (!make_map(&tq, Qx, p.G, p.N, DR)) return cudaErrorInvalidValue;
    DiagArgs a{};
    a.B = p.B; a.H = p.H; a.N = p.N; a.T = L.T; a.Ttot = L.Ttot;
    a.params = reinterpret_cast<const uint8_t *>(ws + L.params);
    a.param_stride = L.param_stride;
    a.part = reinterpret_cast<float *>(ws + L.part);
    a.z = z;
    a.status = reinterpret_cast<unsigned *>(ws);
    cudaError_t e = set_dyn_smem(reinterpret_cast<const void *>(tc_diag2_kernel), Diag2Cfg::BYTES);
    if (e != cudaSuccess) return e;
    return launch_dependent(tc_diag2_kernel, dim3(L.ncta), dim3(kDiag2Threads), Diag2Cfg::BYTES, s, tq, a);
}

cudaError_t tc_diag_finalize(const Problem &p, const TcLayout &L, float *p_out, float *stats_out, char *ws,
                             cudaStream_t s) {
    return launch_dependent(tc_diag_finalize_kernel, dim3(1), dim3(kFinGroups * kFinCols), 0, s, p.K, L.ncta,
                            (float)((double)p.B * (double)p.N), reinterpret_cast<const float *>(ws + L.part), p_out,
                            stats_out);
}

}  // namespace gma
