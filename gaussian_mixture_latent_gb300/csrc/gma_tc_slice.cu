// Component-sliced causal GMA forward for bf16 inputs with d = 64 and larger K
// or dv (K, dv multiples of 64, K <= 256): the configuration whose fp32 state
// [K x (dv + 1)] and K-wide scores do not fit one SM's tensor memory.
//
// "Gaussian Mixture Attention" (Huang & Raza, 2026), Eq. 6b / 8b.  Every term
// of the causal read is a sum over components k:
//   num_i = sum_k e^Q_ik (S_k + sum_{j <= i in chunk} gamma^K_jk V_j)
//   den_i = sum_k e^Q_ik (z_k + sum_{j <= i in chunk} gamma^K_jk) + eps sum_k e^Q_ik
// once gamma^K is normalised over all K components (Eq. 3b) and e^Q is taken
// relative to one per-row offset.  So the forward splits exactly into slices of
// 64 components (and 64 value columns):
//   tc_rowstats     per query row M_i = max_k score, per key row
//                   L_j = log2 sum_k 2^score (scores in log2 units)
//   tc_causal<true> one CTA per (head, component slice, value slice): the
//                   K = 64 chunked scan with gamma^K = 2^(score - L), e^Q = 2^(score - M),
//                   writing bf16 partial numerators and fp32 partial denominators
//   tc_combine      O = sum over component slices of num / sum of den
#include <cuda.h>
#include <cuda_bf16.h>

#include "gma_internal.h"
#include "gma_sm100.cuh"
#include "gma_tc_common.cuh"

namespace gma {

using namespace sm100;
using namespace tc;

namespace {

// ------------------------------------------------------------------ tc_rowstats

constexpr int kStatThreads = 192;        // warp 0 producer, 1 MMA issuer, 2-5 one compute group
constexpr int kStatX = 4;                // routing-tile ring stages

template <int K>
struct StatCfg {
    static constexpr uint32_t PB = align1k(param_bytes(K));
    static constexpr uint32_t OFF_X = 0;
    static constexpr uint32_t OFF_P = OFF_X + kStatX * kTileBytes;
    static constexpr uint32_t OFF_CA = OFF_P + PB;
    static constexpr uint32_t OFF_BAR = OFF_CA + kConstABytes;
    static constexpr uint32_t BYTES = OFF_BAR + 256 + 1024;
    static constexpr uint32_t COL_A = 0;      // two [x, x^2/256] operands, 64 columns each
    static constexpr uint32_t COL_D = 128;    // K fp32 scores
    static constexpr uint32_t TMEM_COLS = 512;
    static_assert(COL_D + K <= TMEM_COLS && BYTES <= 232448, "row statistics kernel exceeds TMEM or shared memory");
};

struct StatArgs {
    int G, H, N, T, Ttot;     // tiles: (head, routing tensor, 128-row tile) in that order, Ttot = 2 G T
    const uint8_t *params;
    uint32_t param_stride;
    float *mrow_q, *lse_k;    // [G][N]
    unsigned *status;
};

template <int K>
__global__ void __launch_bounds__(kStatThreads, 1)
tc_rowstats_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   StatArgs A) {
    using C = StatCfg<K>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + C::OFF_BAR);
    uint64_t *xfull = bars, *xempty = xfull + kStatX, *a_full = xempty + kStatX;   // a_full[2]
    uint64_t *d_full = a_full + 2, *d_empty = d_full + 1, *w_full = d_empty + 1, *w_empty = w_full + 1;
    uint64_t *fin = w_empty + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(fin + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    grid_dep_launch();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // contiguous range of the tile list; "heads" of the cursor are (head, tensor) pairs of T tiles
    const int t0 = (int)(((long long)blockIdx.x * A.Ttot) / gridDim.x);
    const int n = (int)(((long long)(blockIdx.x + 1) * A.Ttot) / gridDim.x) - t0;

    if (threadIdx.x == 0) {
        for (uint64_t *b = bars; b <= fin; ++b) mbar_init(b, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    init_const_a(sm + C::OFF_CA, threadIdx.x, blockDim.x);
    if (warp == 1) { tmem_alloc(tmem_slot, C::TMEM_COLS); tmem_relinquish(); }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const Abort ab{abort_flag, A.status};

    if (warp == 0) {
        if (lane == 0 && n > 0) {
            // the parameter block changes with the head, every second cursor "head"
            TileCursor cx(t0, n, A.T, 0, 1);
            int hp = -1;          // head whose parameters are loaded
            int nloads = 0;
            long long last = now_ns();
            while (cx.valid() && !*abort_flag) {
                bool progress = false, can = true;
                const int head = cx.g >> 1;
                if (head != hp) {
                    if (nloads >= 1 && !mbar_test(w_empty, (nloads - 1) & 1)) {
                        can = false;
                    } else {
                        if (nloads == 0) grid_dep_wait();          // the parameter blocks are written
                        mbar_arrive_expect_tx(w_full, param_bytes(K));
                        bulk_load(sm + C::OFF_P, A.params + (size_t)(head % A.H) * A.param_stride, param_bytes(K),
                                  w_full);
                        hp = head;
                        ++nloads;
                        progress = true;
                    }
                }
                const int xi = cx.i;
                if (can && (xi < kStatX || mbar_test(&xempty[xi % kStatX], ((xi / kStatX) - 1) & 1))) {
                    mbar_arrive_expect_tx(&xfull[xi % kStatX], kTileBytes);
                    tma_load_3d(sm + C::OFF_X + (xi % kStatX) * kTileBytes, (cx.g & 1) ? &tm_k : &tm_q,
                                &xfull[xi % kStatX], 0, cx.j * TM, head);
                    cx.next();
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
            wind_down_ring(xfull, kStatX, cx.i < n ? cx.i : n, A.status);
            if (nloads >= 1) wait_ignoring_abort(w_full, (nloads - 1) & 1, A.status);
        }
    } else if (warp == 1) {
        // log-density MMA of tile i into the score columns, once tile i - 1's scores are read
        if (n > 0) {                                 // the whole warp, converged
            const uint32_t ca = smem_u32(sm + C::OFF_CA), pw = smem_u32(sm + C::OFF_P);
            int hp = -1, nloads = 0;
            bool ok = true;
            for (TileCursor c(t0, n, A.T, 0, 1); c.valid() && ok; c.next()) {
                const int i = c.i, head = c.g >> 1;
                if (head != hp) {
                    if (!(ok = mbar_wait_warp(w_full, nloads & 1, ab, kDevErrTimeout))) break;
                    hp = head;
                    ++nloads;
                }
                ok = mbar_wait_warp(&a_full[i & 1], (i >> 1) & 1, ab, kDevErrTimeout);
                if (ok && i >= 1) ok = mbar_wait_warp(d_empty, (i - 1) & 1, ab, kDevErrTimeout);
                if (!ok) break;
                tc_fence_after();
                issue_logdensity<K>(tmem + C::COL_D, tmem + C::COL_A + (i & 1) * 64, pw, ca);
                mma_commit(d_full);
                mma_commit(&xempty[i % kStatX]);
                // last tile of this head in the range: its parameter block may be replaced
                const bool head_last = i == n - 1 || (c.j == A.T - 1 && (c.g & 1));
                if (head_last) mma_commit(w_empty);
            }
            mma_commit(fin);
            wait_ignoring_abort(fin, 0, A.status);
        }
    } else {
        RowThread rt;
        rt.wg = 0;
        rt.r = 32u * (warp & 3) + lane;
        rt.lane_off = (uint32_t)(32 * (warp & 3)) << 16;
        rt.wtid = threadIdx.x - 64;
        const bool elected = rt.wtid == 0;
        auto convert = [&](int i) -> bool {
            const bool w = mbar_wait(&xfull[i % kStatX], (i / kStatX) & 1, ab, kDevErrTimeout);
            if (!wg_all(rt, w)) return false;
            convert_row(sm + C::OFF_X + (i % kStatX) * kTileBytes, rt.r, tmem + rt.lane_off + C::COL_A + (i & 1) * 64);
            tmem_st_wait();
            tc_fence_before();
            wg_sync(rt);
            if (elected) mbar_arrive(&a_full[i & 1]);
            return true;
        };
        bool ok = n > 0 && convert(0);
        int hs = -1;
        float scale = 0.f;
        for (TileCursor c(t0, n, A.T, 0, 1); c.valid() && ok; c.next()) {
            const int i = c.i, head = c.g >> 1;
            // tile i + 1's operand (its buffer was read by the MMA of tile i - 1, complete)
            if (i + 1 < n && !(ok = convert(i + 1))) break;
            if (head != hs) {
                grid_dep_wait();
                scale = head_scale(A.params, A.param_stride, head % A.H, K);
                hs = head;
            }
            const bool w = mbar_wait(d_full, i & 1, ab, kDevErrTimeout);
            if (!(ok = wg_all(rt, w))) break;
            tc_fence_after();
            const uint32_t dcol = tmem + rt.lane_off + C::COL_D;
            // pass 1: row maximum of the raw scores (scale > 0 commutes with max)
            float m = -INFINITY;
#pragma unroll
            for (int cc = 0; cc < K / 32; ++cc) {
                uint32_t v[32];
                tmem_ld32(dcol + 32 * cc, v);
                tmem_ld_wait();
#pragma unroll
                for (int t = 0; t < 32; t += 2) m = max3(m, __uint_as_float(v[t]), __uint_as_float(v[t + 1]));
            }
            const float M = m * scale;
            const int row = c.j * TM + (int)rt.r;
            if (c.g & 1) {
                // keys: L = M + log2 sum_k 2^(scale d_k - M), fp32 exponentials
                const uint64_t sc2 = f2_pack(scale, scale), nm2 = f2_pack(-M, -M);
                float s = 0.f;
#pragma unroll
                for (int cc = 0; cc < K / 32; ++cc) {
                    uint32_t v[32];
                    tmem_ld32(dcol + 32 * cc, v);
                    tmem_ld_wait();
                    float part = 0.f;
#pragma unroll
                    for (int t = 0; t < 32; t += 2) {
                        float a, b;
                        f2_unpack(f2_fma(f2_pack(__uint_as_float(v[t]), __uint_as_float(v[t + 1])), sc2, nm2), a, b);
                        part += ex2_approx(a) + ex2_approx(b);
                    }
                    s += part;
                }
                if (row < A.N) A.lse_k[(size_t)head * A.N + row] = M + __log2f(s);
            } else if (row < A.N) {
                A.mrow_q[(size_t)head * A.N + row] = M;
            }
            tc_fence_before();
            wg_sync(rt);
            if (elected) mbar_arrive(d_empty);
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

// ------------------------------------------------------------------ tc_combine

// O[g][i][:] = sum_s num[s][g][i][:] / sum_s den[s][g][i], a fixed order over slices.
// A thread owns 16-byte pieces (eight value columns of one row); it issues the
// loads of all NS slices of two pieces before it uses any of them.
constexpr int kCombineThreads = 256;

template <int NS>
__device__ __forceinline__ void combine_piece(size_t rows, int dv, size_t piece, const uint16_t *__restrict__ pnum,
                                              const float *__restrict__ pden, uint16_t *__restrict__ out,
                                              const uint4 (&v)[NS], const float (&d)[NS]) {
    const int per_row = dv / 8;
    const size_t row = piece / per_row;
    const int c0 = 8 * (int)(piece % per_row);
    float den = 0.f;
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int s = 0; s < NS; ++s) {
        den += d[s];
        const uint32_t w[4] = {v[s].x, v[s].y, v[s].z, v[s].w};
#pragma unroll
        for (int u = 0; u < 4; ++u) { acc[2 * u] += bf16_lo(w[u]); acc[2 * u + 1] += bf16_hi(w[u]); }
    }
    const float rd = 1.0f / den;
    *reinterpret_cast<uint4 *>(out + row * dv + c0) =
        make_uint4(pack_bf16(acc[0] * rd, acc[1] * rd), pack_bf16(acc[2] * rd, acc[3] * rd),
                   pack_bf16(acc[4] * rd, acc[5] * rd), pack_bf16(acc[6] * rd, acc[7] * rd));
}

template <int NS>
__global__ void __launch_bounds__(kCombineThreads) tc_combine_kernel(int G, int N, int dv,
                                                                     const uint16_t *__restrict__ pnum,
                                                                     const float *__restrict__ pden,
                                                                     uint16_t *__restrict__ out) {
    grid_dep_launch();
    grid_dep_wait();                                       // the partial numerators and denominators are written
    const size_t rows = (size_t)G * N, pieces = rows * (dv / 8);
    const size_t half = (pieces + 1) / 2;                  // a thread takes pieces p and p + half
    const size_t p0 = (size_t)blockIdx.x * kCombineThreads + threadIdx.x;
    if (p0 >= half) return;
    const size_t p1 = p0 + half;
    const bool two = p1 < pieces;
    const int per_row = dv / 8;
    uint4 v0[NS], v1[NS];
    float d0[NS], d1[NS];
#pragma unroll
    for (int s = 0; s < NS; ++s) {
        const size_t r0 = p0 / per_row, r1 = p1 / per_row;
        v0[s] = __ldg(reinterpret_cast<const uint4 *>(pnum + ((size_t)s * rows + r0) * dv + 8 * (p0 % per_row)));
        d0[s] = __ldg(pden + (size_t)s * rows + r0);
        if (two) {
            v1[s] = __ldg(reinterpret_cast<const uint4 *>(pnum + ((size_t)s * rows + r1) * dv + 8 * (p1 % per_row)));
            d1[s] = __ldg(pden + (size_t)s * rows + r1);
        }
    }
    combine_piece<NS>(rows, dv, p0, pnum, pden, out, v0, d0);
    if (two) combine_piece<NS>(rows, dv, p1, pnum, pden, out, v1, d1);
}

template <int K>
cudaError_t launch_rowstats(const Problem &p, const TcLayout &L, const void *Qx, const void *Kx, char *ws,
                            cudaStream_t s) {
    CUtensorMap tq, tk;
    if (!make_map(&tq, Qx, p.G, p.N, DR) || !make_map(&tk, Kx, p.G, p.N, DR)) return cudaErrorInvalidValue;
    StatArgs a{};
    a.G = p.G; a.H = p.H; a.N = p.N; a.T = L.T; a.Ttot = 2 * L.T * p.G;
    a.params = reinterpret_cast<const uint8_t *>(ws + L.params);
    a.param_stride = L.param_stride;
    a.mrow_q = reinterpret_cast<float *>(ws + L.stats);
    a.lse_k = a.mrow_q + (size_t)p.G * p.N;
    a.status = reinterpret_cast<unsigned *>(ws);
    auto kern = tc_rowstats_kernel<K>;
    cudaError_t e = set_dyn_smem(reinterpret_cast<const void *>(kern), StatCfg<K>::BYTES);
    if (e != cudaSuccess) return e;
    const int ncta = std::max(1, std::min(sm_count() > 0 ? sm_count() : kMaxCtas, a.Ttot));
    return launch_dependent(kern, dim3(ncta), dim3(kStatThreads), StatCfg<K>::BYTES, s, tq, tk, a);
}

}  // namespace

cudaError_t tc_rowstats(const Problem &p, const TcLayout &L, const void *Qx, const void *Kx, char *ws,
                        cudaStream_t s) {
    switch (p.K) {
        case 64: return launch_rowstats<64>(p, L, Qx, Kx, ws, s);
        case 128: return launch_rowstats<128>(p, L, Qx, Kx, ws, s);
        case 192: return launch_rowstats<192>(p, L, Qx, Kx, ws, s);
        case 256: return launch_rowstats<256>(p, L, Qx, Kx, ws, s);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t tc_combine(const Problem &p, const TcLayout &L, void *out, char *ws, cudaStream_t s) {
    const size_t pieces = (size_t)p.G * p.N * (p.dv / 8), half = (pieces + 1) / 2;
    const dim3 grid((unsigned)((half + kCombineThreads - 1) / kCombineThreads));
    const auto *pn = reinterpret_cast<const uint16_t *>(ws + L.pnum);
    const auto *pd = reinterpret_cast<const float *>(ws + L.pden);
    auto *o = static_cast<uint16_t *>(out);
    switch (L.ns) {
        case 1: return launch_dependent(tc_combine_kernel<1>, grid, dim3(kCombineThreads), 0, s, p.G, p.N, p.dv, pn, pd, o);
        case 2: return launch_dependent(tc_combine_kernel<2>, grid, dim3(kCombineThreads), 0, s, p.G, p.N, p.dv, pn, pd, o);
        case 3: return launch_dependent(tc_combine_kernel<3>, grid, dim3(kCombineThreads), 0, s, p.G, p.N, p.dv, pn, pd, o);
        case 4: return launch_dependent(tc_combine_kernel<4>, grid, dim3(kCombineThreads), 0, s, p.G, p.N, p.dv, pn, pd, o);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace gma
