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
    return p.K == 64 ? launch_diag<64>(p, L, Qx, z, ws, s) : launch_diag<128>(p, L, Qx, z, ws, s);
}

cudaError_t tc_diag_finalize(const Problem &p, const TcLayout &L, float *p_out, float *stats_out, char *ws,
                             cudaStream_t s) {
    return launch_dependent(tc_diag_finalize_kernel, dim3(1), dim3(kFinGroups * kFinCols), 0, s, p.K, L.ncta,
                            (float)((double)p.B * (double)p.N), reinterpret_cast<const float *>(ws + L.part), p_out,
                            stats_out);
}

}  // namespace gma
