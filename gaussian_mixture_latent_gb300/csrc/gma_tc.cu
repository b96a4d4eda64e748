// Tensor-core (tcgen05) path of the bidirectional GMA forward for bf16
// inputs and outputs, routing dimension d = 64, value dimension dv = 64 and
// K = 64 or 128 components.
//
// "Gaussian Mixture Attention" (Huang & Raza, 2026): responsibilities
// (section 3.2 Eq. 3, in the log-density form of section 4.1 Eq. 16 / 3b),
// latent write (section 3.3 Eq. 5-6) and normalised read (Eq. 7-8), with the
// parameterisation of section 3.6 (Eq. 14-15).
//
// The log-density of all K diagonal Gaussians for a tile of 128 rows is one
// contraction:  s = [x, x^2 / 256] . W^T + c  with
//   W_k = [mu_k * lam_k, 256 * (-lam_k / 2 - beta)] * log2(e),   lam = 1 / var,
//   c_k = (log pi_k - 1/2 sum_m log var_km - 1/2 sum_m mu_km^2 lam_km) * log2(e),
// where beta_m = mean_k(-lam_km / 2) is a k-independent shift (it changes every
// score of a row by the same amount, which the softmax cancels) that centres
// the quadratic coefficients.  Scores are in log2 units, so exp2 gives the
// responsibilities.  Operands are fp16 (x exact; x^2 and W rounded to 11
// bits; W carries a per-head power-of-two scale), accumulation fp32.
//
// Kernels (tc_write / tc_read are persistent, one CTA per SM):
//   tc_params  per head: fp16 W in the MMA's shared-memory layout, c, scale
//   tc_write   per tile of Kx, V (each CTA a contiguous range of the (head,
//              128-row tile) list):  [x, x^2] -> TMEM; MMA -> scores in TMEM;
//              softmax -> Gamma^K (bf16, shared memory); MMA accumulates
//              [V | 1]^T Gamma^K (= [Vt | Z]^T) in TMEM; drained per head to a
//              fp32 partial slot (slot index = cta + head)
//   tc_reduce  per head: fixed-order sum of the partial slots -> [Vt | Z | 1]^T
//              as the bf16 B operand of the read
//   tc_read    per tile of Qx (a contiguous range per CTA, or, beside a
//              concurrent kernel, units of tiles claimed from a counter):
//              scores as above; unnormalised exp2 -> TMEM (bf16); MMA with
//              [Vt | Z | 1]; out = num / (den + eps * sum) -> TMA store
//
// Warp roles inside tc_write / tc_read ((3 + 4 NW) warps, NW = 3 compute groups
// at K = 64 and 2 at K = 128): warp 0 issues every TMA and bulk copy from one
// thread (the write's producer polls its rings without blocking; the read's
// waits on one ring slot at a time); warp 1 allocates TMEM and issues the
// log-density MMAs; warp 2 issues the write / read MMAs (two issuers, because an
// MMA issue blocks while the tensor pipe fills); warps 3 onwards are the NW
// compute warpgroups that take tiles in turn (one thread per row), each with its
// own TMEM columns, so one group's softmax overlaps the others' MMAs.  The read
// at K = 128 forms a tile's scores in two parts of 64 components through one
// 64-column region, so that three groups fit in TMEM: warp 1 issues the first
// parts, warp 3 the second ones, and the compute groups are warps 4 onwards
// ((4 + 4 * 3) warps).  Every mbarrier wait is bounded; a timeout posts
// GMA_ERR_TIMEOUT to the workspace status word and the CTA winds down.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <algorithm>
#include <cmath>
#include <cstring>
#include <mutex>

#include "gma_internal.h"
#include "gma_sm100.cuh"
#include "gma_tc_common.cuh"

namespace gma {

using namespace sm100;
using namespace tc;

namespace {

constexpr int kWarpProducer = 0, kWarpMma1 = 1, kWarpMma2 = 2, kWarpCompute = 3;
// Compute groups per CTA: three at K = 64 (TMEM holds three groups' operands and
// scores), two at K = 128 (the read fits three there by forming its scores in two
// parts, ReadCfg).  More groups hide more of each group's serial convert ->
// log-density MMA -> softmax latency.
__host__ __device__ constexpr int groups_for(int K) { return K <= 64 ? 3 : 2; }

struct TcArgs {
    int G, H, N, T, Ttot, K;
    const uint8_t *params;   // [H][param_stride]
    uint32_t param_stride;
    float *partials;         // [slots][DVV + 1][K]
    uint8_t *mem;            // [G][mem_stride]
    uint32_t mem_stride;
    float eps;
    unsigned *status;
    int nslots;              // partial slots in the workspace (index checks of the debug build)
    int *claim;              // the read's unit counter (zeroed by tc_reduce)
    int dyn;                 // the read takes units from the counter (1) or a static range (0)
};

__device__ __forceinline__ void cta_range(int Ttot, int &t0, int &t1) {
    t0 = (int)(((long long)blockIdx.x * Ttot) / gridDim.x);
    t1 = (int)(((long long)(blockIdx.x + 1) * Ttot) / gridDim.x);
}

// ------------------------------------------------------------------ tc_params

constexpr int kParamThreads = 512;

template <int K>
__global__ void __launch_bounds__(kParamThreads) tc_params_kernel(float var_floor, const float *__restrict__ mu,
                                                                  const float *__restrict__ rho,
                                                                  const float *__restrict__ alpha,
                                                                  uint8_t *__restrict__ out, uint32_t stride) {
    __shared__ __align__(16) float scratch[param_scratch_floats(K, kParamThreads)];
    grid_dep_launch();
    const int h = blockIdx.x;
    ParamLoads<K, kParamThreads> ld;
    ld.issue(threadIdx.x, mu + (size_t)h * K * DR, rho + (size_t)h * K * DR, alpha + (size_t)h * K);
    build_param_block<K, kParamThreads>(threadIdx.x, ld, var_floor, out + (size_t)h * stride, scratch,
                                        [] { __syncthreads(); });
}

// ------------------------------------------------------------------ tc_write


template <int K>
struct WriteCfg {
    static constexpr int KCH = (K + 63) / 64;
    static constexpr int NW = groups_for(K);
    static constexpr int THREADS = (kWarpCompute + 4 * NW) * 32;
    static constexpr int SX = K <= 64 ? 4 : 3;                       // X ring stages
    static constexpr int SV = K <= 64 ? 4 : 3;                       // V ring stages
    static constexpr int PN = 1;                                     // parameter buffers
    static constexpr uint32_t PB = align1k(param_bytes(K));
    static constexpr uint32_t OFF_X = 0;
    static constexpr uint32_t OFF_V = OFF_X + SX * kTileBytes;
    static constexpr uint32_t OFF_ONES = OFF_V + SV * kTileBytes;      // after every V stage (positive LBO)
    static constexpr uint32_t OFF_G = OFF_ONES + kTileBytes;           // one Gamma buffer per warpgroup
    static constexpr uint32_t OFF_P = OFF_G + NW * KCH * kTileBytes;
    static constexpr uint32_t OFF_CA = OFF_P + PN * PB;               // constant [1, 1, 0...] A block
    static constexpr uint32_t OFF_BAR = OFF_CA + kConstABytes;
    static constexpr uint32_t BYTES = OFF_BAR + 512 + 1024;            // barriers + alignment slack
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr uint32_t wg_cols = 64 + K;
    static constexpr uint32_t col_a(int w) { return w * wg_cols; }
    static constexpr uint32_t col_d1(int w) { return w * wg_cols + 64; }
    static constexpr uint32_t COL_D2 = NW * wg_cols;
    static_assert(BYTES <= 232448 && COL_D2 + K <= TMEM_COLS, "write kernel exceeds shared memory or TMEM");
    // A group waits on tile i's routing stage by parity; the stage's previous tile (i - SX)
    // must then be its own or one whose conversion it has seen (the log-density MMA of its
    // previous tile i - NW follows the conversion of tile i - NW - 1), so SX >= NW.
    static_assert(SX >= NW, "fewer routing stages than compute groups");
};

// SEG = false: the CTA's range of the (head, tile) list, one partial slot per (CTA, head).
// SEG = true: the prefix pass of the segment-parallel causal scan, the same walk over the
// concatenated prefix segments of S, one partial slot per (CTA, segment).
template <int K, bool SEG>
__global__ void __launch_bounds__(WriteCfg<K>::THREADS, 1)
tc_write_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v, TcArgs A,
                const __grid_constant__ typename SegArg<SEG>::type S) {
    using C = WriteCfg<K>;
    constexpr int SX = C::SX, SV = C::SV, PN = C::PN, NW = C::NW;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + C::OFF_BAR);
    uint64_t *xfull = bars, *xempty = xfull + SX;
    uint64_t *vfull = xempty + SX, *vempty = vfull + SV;
    uint64_t *a_full = vempty + SV, *d1_full = a_full + NW, *g_full = d1_full + NW, *g_empty = g_full + NW;
    uint64_t *w_full = g_empty + NW, *w_empty = w_full + PN;
    // d2_full[hl % NW]: the accumulation of local head hl is complete.  The group that drains
    // head hl has seen the write MMA of its previous tile (tile - NW) complete, hence every head
    // up to hl - NW, so it is never more than one phase ahead of the barrier it waits on.
    uint64_t *d2_full = w_empty + PN, *d2_empty = d2_full + NW, *fin1 = d2_empty + 1, *fin2 = fin1 + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(fin2 + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    grid_dep_launch();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int t0, t1;
    cta_range(A.Ttot, t0, t1);
    const int n = t1 - t0;
    auto cursor = [&](int start, int step) {
        if constexpr (SEG) return SegCursor(&S, blockIdx.x, n, start, step);
        else return TileCursor(t0, n, A.T, start, step);
    };

    if (threadIdx.x == 0) {
        for (int s = 0; s < SX; ++s) { mbar_init(&xfull[s], 1); mbar_init(&xempty[s], 1); }
        for (int s = 0; s < SV; ++s) { mbar_init(&vfull[s], 1); mbar_init(&vempty[s], 1); }
        for (int b = 0; b < NW; ++b) {
            mbar_init(&a_full[b], 1); mbar_init(&d1_full[b], 1); mbar_init(&g_full[b], 1); mbar_init(&g_empty[b], 1);
            mbar_init(&d2_full[b], 1);
        }
        for (int b = 0; b < PN; ++b) { mbar_init(&w_full[b], 1); mbar_init(&w_empty[b], 1); }
        mbar_init(d2_empty, 1);
        mbar_init(fin1, 1); mbar_init(fin2, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    init_const_a(sm + C::OFF_CA, threadIdx.x, blockDim.x);
    // ONES atom column: element 0 of every row is 1.0 (bf16), the rest 0.
    for (uint32_t e = threadIdx.x; e < kTileBytes / 16; e += blockDim.x)
        reinterpret_cast<uint4 *>(sm + C::OFF_ONES)[e] = make_uint4(0, 0, 0, 0);
    __syncthreads();
    if (threadIdx.x < TM) *reinterpret_cast<uint16_t *>(sm + C::OFF_ONES + sw128_off(threadIdx.x, 0)) = 0x3F80u;
    if (warp == kWarpMma1) { tmem_alloc(tmem_slot, C::TMEM_COLS); tmem_relinquish(); }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const Abort ab{abort_flag, A.status};

    if (warp == kWarpProducer) {
        if (lane == 0 && n > 0) {
            auto cx = cursor(0, 1), cv = cursor(0, 1);
            // the first head's routing and value tiles do not depend on the previous kernel
            for (; cx.valid() && cx.hl == 0 && cx.i < SX; cx.next()) {
                mbar_arrive_expect_tx(&xfull[cx.i], kTileBytes);
                tma_load_3d(sm + C::OFF_X + cx.i * kTileBytes, &tm_k, &xfull[cx.i], 0, cx.j * TM, cx.g);
            }
            for (; cv.valid() && cv.hl == 0 && cv.i < SV; cv.next()) {
                mbar_arrive_expect_tx(&vfull[cv.i], kTileBytes);
                tma_load_3d(sm + C::OFF_V + cv.i * kTileBytes, &tm_v, &vfull[cv.i], 0, cv.j * TM, cv.g);
            }
            grid_dep_wait();                               // the parameter blocks are written
            mbar_arrive_expect_tx(&w_full[0], param_bytes(K));
            bulk_load(sm + C::OFF_P, A.params + (size_t)(cursor(0, 1).g % A.H) * A.param_stride, param_bytes(K),
                      &w_full[0]);
            int p_loaded = 0;
            long long last = now_ns();
            while ((cx.valid() || cv.valid()) && !*abort_flag) {
                bool progress = false;
                if (cx.valid()) {
                    const int xi = cx.i;
                    bool can = true;
                    if (cx.hl > p_loaded) {
                        const int b = cx.hl % PN;
                        if (cx.hl >= PN && !mbar_test(&w_empty[b], ((cx.hl / PN) - 1) & 1)) can = false;
                        else {
                            mbar_arrive_expect_tx(&w_full[b], param_bytes(K));
                            bulk_load(sm + C::OFF_P + b * C::PB, A.params + (size_t)(cx.g % A.H) * A.param_stride,
                                      param_bytes(K), &w_full[b]);
                            p_loaded = cx.hl;
                            progress = true;
                        }
                    }
                    if (can && (xi < SX || mbar_test(&xempty[xi % SX], ((xi / SX) - 1) & 1))) {
                        (void)GMA_IN_BOUNDS(cx.g < A.G && cx.j < A.T, A.status);
                        mbar_arrive_expect_tx(&xfull[xi % SX], kTileBytes);
                        tma_load_3d(sm + C::OFF_X + (xi % SX) * kTileBytes, &tm_k, &xfull[xi % SX], 0, cx.j * TM, cx.g);
                        cx.next();
                        progress = true;
                    }
                }
                if (cv.valid()) {
                    const int vi = cv.i;
                    if (vi < SV || mbar_test(&vempty[vi % SV], ((vi / SV) - 1) & 1)) {
                        mbar_arrive_expect_tx(&vfull[vi % SV], kTileBytes);
                        tma_load_3d(sm + C::OFF_V + (vi % SV) * kTileBytes, &tm_v, &vfull[vi % SV], 0, cv.j * TM, cv.g);
                        cv.next();
                        progress = true;
                    }
                }
                if (progress) {
                    last = now_ns();
                } else {
                    __nanosleep(64);                       // nothing to issue: yield the issue slots
                    if (now_ns() - last > kWaitLimitNs) {
                        *abort_flag = 1;
                        atomicOr(A.status, kDevErrTimeout);
                    }
                }
            }
            wind_down_ring(xfull, SX, cx.i < n ? cx.i : n, A.status);
            wind_down_ring(vfull, SV, cv.i < n ? cv.i : n, A.status);
            for (int hl = p_loaded - PN + 1 < 0 ? 0 : p_loaded - PN + 1; hl <= p_loaded; ++hl)
                wait_ignoring_abort(&w_full[hl % PN], (hl / PN) & 1, A.status);
        }
    } else if (warp == kWarpMma1) {
        // log-density MMAs: scores(i) = [x, x^2/256](i) . W^T into D1 of group i % NW
        if (n > 0) {                                 // the whole warp, converged
            for (auto c = cursor(0, 1); c.valid(); c.next()) {
                const int i = c.i, b = c.hl % PN, w = i % NW;
                if (c.first() && !mbar_wait_warp(&w_full[b], (c.hl / PN) & 1, ab, kDevErrTimeout)) break;
                if (!mbar_wait_warp(&a_full[w], (i / NW) & 1, ab, kDevErrTimeout)) break;
                tc_fence_after();
                issue_logdensity<K>(tmem + C::col_d1(w), tmem + C::col_a(w), smem_u32(sm + C::OFF_P + b * C::PB),
                                    smem_u32(sm + C::OFF_CA));
                mma_commit(&d1_full[w]);
                if (c.last()) mma_commit(&w_empty[b]);
            }
            mma_commit(fin1);
            wait_ignoring_abort(fin1, 0, A.status);
        }
    } else if (warp == kWarpMma2) {
        // write MMAs: D2 [value row x K] += [V | 1 | 0]^T (128 x rows) . Gamma (rows x K)
        if (n > 0) {                                 // the whole warp, converged
            constexpr uint32_t idesc = idesc_f16(1, 1, 1, 1, TM, K);
            const uint32_t ones = smem_u32(sm + C::OFF_ONES);
            for (auto c = cursor(0, 1); c.valid(); c.next()) {
                const int i = c.i, s = i % SV, w = i % NW;
                if (!mbar_wait_warp(&g_full[w], (i / NW) & 1, ab, kDevErrTimeout)) break;
                if (!mbar_wait_warp(&vfull[s], (i / SV) & 1, ab, kDevErrTimeout)) break;
                if (c.first() && c.hl >= 1 && !mbar_wait_warp(d2_empty, (c.hl - 1) & 1, ab, kDevErrTimeout)) break;
                tc_fence_after();
                const uint32_t va = smem_u32(sm + C::OFF_V + s * kTileBytes);
                const uint64_t ad = sdesc_sw128(va, ones - va, 1024);
                const uint64_t bd = sdesc_sw128(smem_u32(sm + C::OFF_G + w * C::KCH * kTileBytes), kTileBytes, 1024);
                const bool first = c.first();
#pragma unroll
                for (int ks = 0; ks < 8; ++ks)
                    mma_ss(tmem + C::COL_D2, ad + (uint64_t)(ks * 128), bd + (uint64_t)(ks * 128), idesc,
                           !(first && ks == 0));
                mma_commit(&g_empty[w]);
                mma_commit(&vempty[s]);
                if (c.last()) mma_commit(&d2_full[c.hl % NW]);
            }
            mma_commit(fin2);
            wait_ignoring_abort(fin2, 0, A.status);
        }
    } else {
        // ---------------- two compute warpgroups, alternate tiles
        RowThread rt;
        rt.wg = (warp - kWarpCompute) >> 2;
        rt.r = 32u * (warp & 3) + lane;
        rt.lane_off = (uint32_t)(32 * (warp & 3)) << 16;
        rt.wtid = threadIdx.x - kWarpCompute * 32 - rt.wg * kWgThreads;
        const int w = rt.wg;
        const bool elected = rt.wtid == 0;
        auto c = cursor(w, NW);
        for (; c.valid(); c.next()) {
            const int i = c.i, hl = c.hl;
            // convert tile i into this group's A operand
            bool ok = mbar_wait(&xfull[i % SX], (i / SX) & 1, ab, kDevErrTimeout);
            if (!wg_all(rt, ok)) break;
            convert_row(sm + C::OFF_X + (i % SX) * kTileBytes, rt.r, tmem + rt.lane_off + C::col_a(w));
            tmem_st_wait();
            tc_fence_before();
            wg_sync(rt);
            if (elected) { mbar_arrive(&a_full[w]); mbar_arrive(&xempty[i % SX]); }
            // softmax of tile i (Eq. 3b); rows past the sequence end get Gamma = 0
            if (i < NW) grid_dep_wait();                   // the parameter blocks are written
            const float scale = head_scale(A.params, A.param_stride, c.g % A.H, K);
            ok = mbar_wait(&d1_full[w], (i / NW) & 1, ab, kDevErrTimeout);
            if (i >= NW) ok = ok && mbar_wait(&g_empty[w], ((i / NW) - 1) & 1, ab, kDevErrTimeout);
            if (!wg_all(rt, ok)) break;
            tc_fence_after();
            uint32_t e[K / 2];
            row_exp_scaled<K>(tmem + rt.lane_off + C::col_d1(w), scale, e);
            uint64_t acc[4] = {0, 0, 0, 0};
#pragma unroll
            for (int t = 0; t < K / 2; ++t) acc[t & 3] = f2_add(acc[t & 3], f2_pack(bf16_lo(e[t]), bf16_hi(e[t])));
            float s0, s1, s2, s3, s4, s5, s6, s7;
            f2_unpack(acc[0], s0, s1); f2_unpack(acc[1], s2, s3);
            f2_unpack(acc[2], s4, s5); f2_unpack(acc[3], s6, s7);
            const float total = ((s0 + s1) + (s2 + s3)) + ((s4 + s5) + (s6 + s7));
            const bool valid = c.j * TM + (int)rt.r < A.N;
            const float inv = valid ? 1.0f / total : 0.f;
            const uint64_t inv2 = f2_pack(inv, inv);
            const uint32_t gsm = smem_u32(sm + C::OFF_G + w * C::KCH * kTileBytes);
#pragma unroll
            for (int j = 0; j < K / 8; ++j) {
                uint32_t wv[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    float ga, gb;
                    f2_unpack(f2_mul(f2_pack(bf16_lo(e[4 * j + u]), bf16_hi(e[4 * j + u])), inv2), ga, gb);
                    wv[u] = pack_bf16(ga, gb);
                }
                st_shared_v4(gsm + (j >> 3) * kTileBytes + sw128_off(rt.r, j & 7), wv[0], wv[1], wv[2], wv[3]);
            }
            fence_proxy_async_smem();
            tc_fence_before();
            wg_sync(rt);
            if (elected) mbar_arrive(&g_full[w]);
            if (c.last()) {
                // drain [Vt | Z]^T of this head (segment) into partial slot (cta + head)
                ok = mbar_wait(&d2_full[hl % NW], (hl / NW) & 1, ab, kDevErrTimeout);
                if (!wg_all(rt, ok)) break;
                tc_fence_after();
                const int slot = (int)blockIdx.x + c.slot();
                float *dst = A.partials + ((size_t)slot * (DVV + 1) + rt.r) * K;
                const bool store = rt.r <= DVV && GMA_IN_BOUNDS(slot < A.nslots && c.g < A.G, A.status);
#pragma unroll 1
                for (int cc = 0; cc < K / 32; ++cc) {         // 32 columns at a time (few live registers)
                    uint32_t v[32];
                    tmem_ld32(tmem + rt.lane_off + C::COL_D2 + 32 * cc, v);
                    tmem_ld_wait();
                    if (store) {
#pragma unroll
                        for (int t = 0; t < 32; t += 4)
                            *reinterpret_cast<float4 *>(dst + 32 * cc + t) = make_float4(
                                __uint_as_float(v[t]), __uint_as_float(v[t + 1]), __uint_as_float(v[t + 2]),
                                __uint_as_float(v[t + 3]));
                    }
                }
                tc_fence_before();
                wg_sync(rt);
                if (elected) mbar_arrive(d2_empty);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kWarpMma1) {
        __syncwarp();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

// ------------------------------------------------------------------ tc_reduce

// Fixed-order sum over the CTAs that covered head g (blockIdx.y), then the bf16
// B operand [n][k] of the read (n = value column, dv -> Z, dv+1 -> 1, rest 0)
// in the K-major 128-byte-swizzled layout, ceil(K/64) chunks of 80 rows.  With
// mem_lo given, the rounding remainder (the fp32 sum minus its bf16 value, itself
// rounded to bf16) goes to the same layout there, so that hi + lo carries the sum
// to about 16 significant bits (the backward's two-term operands).  Each
// thread owns four consecutive k of one row (a float4 of every partial), so a
// head takes 20 K / 4 threads and the grid fits on the GPU in one wave while
// the write kernel drains.
constexpr int kReduceThreads = 256;

__global__ void __launch_bounds__(kReduceThreads) tc_reduce_kernel(int K, int T, int Ttot, int ncta,
                                                                   const float *__restrict__ partials,
                                                                   uint8_t *__restrict__ mem, uint8_t *__restrict__ mem_lo,
                                                                   uint32_t mem_stride, int nslots, int *claim,
                                                                   unsigned *status) {
    grid_dep_launch();
    // the read kernel that follows claims its tile units from this counter once this grid
    // has completed; the read before it completed before this call's first kernel started
    if (claim && blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) *claim = 0;
    const int g = blockIdx.y;
    const int q = blockIdx.x * blockDim.x + threadIdx.x;   // float4 index in the 80 x K operand
    // CTA c owns tiles [c*Ttot/ncta, (c+1)*Ttot/ncta): those meeting [g*T, (g+1)*T) are
    // c_lo..c_hi - 1 (depends only on the launch shape: found before the wait)
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
    grid_dep_wait();                                       // the partial slots are written
    const int kq = K / 4;
    if (q >= 80 * kq) return;
    const int c_lo = crange[0], c_hi = crange[1];
    if (!GMA_IN_BOUNDS(c_lo >= 0 && c_hi + g <= nslots, status)) return;
    const int nrow = q / kq, k = 4 * (q % kq);
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (nrow <= DVV) {
        // slots c + g in increasing c; loads of four slots are in flight together
        const size_t step = (size_t)(DVV + 1) * kq;
        const float4 *src = reinterpret_cast<const float4 *>(partials) + ((size_t)(c_lo + g) * (DVV + 1) + nrow) * kq +
                            (k >> 2);
        int c = c_lo;
        for (; c + 4 <= c_hi; c += 4, src += 4 * step) {
            const float4 a0 = src[0], a1 = src[step], a2 = src[2 * step], a3 = src[3 * step];
            v.x = (((v.x + a0.x) + a1.x) + a2.x) + a3.x;
            v.y = (((v.y + a0.y) + a1.y) + a2.y) + a3.y;
            v.z = (((v.z + a0.z) + a1.z) + a2.z) + a3.z;
            v.w = (((v.w + a0.w) + a1.w) + a2.w) + a3.w;
        }
        for (; c < c_hi; ++c, src += step) {
            const float4 a = *src;
            v.x += a.x; v.y += a.y; v.z += a.z; v.w += a.w;
        }
    } else if (nrow == DVV + 1) {
        v = make_float4(1.f, 1.f, 1.f, 1.f);
    }
    const uint32_t off = (uint32_t)(k >> 6) * 80u * 128u + sw128_off(nrow, (k & 63) >> 3) + (k & 7) * 2;
    const uint2 hi = make_uint2(pack_bf16(v.x, v.y), pack_bf16(v.z, v.w));
    *reinterpret_cast<uint2 *>(mem + (size_t)g * mem_stride + off) = hi;
    if (mem_lo)
        *reinterpret_cast<uint2 *>(mem_lo + (size_t)g * mem_stride + off) =
            make_uint2(pack_bf16(v.x - bf16_lo(hi.x), v.y - bf16_hi(hi.x)),
                       pack_bf16(v.z - bf16_lo(hi.y), v.w - bf16_hi(hi.y)));
}

// ------------------------------------------------------------------ tc_read
//
// The read's tiles come in runs of one head.  Alone, a CTA walks a static contiguous
// range of the (head, tile) list, one run per head it meets.  Beside a concurrent
// kernel (gma_forward_multi), the list is cut into units of up to kReadUnit tiles of
// one head, and each CTA's producer claims the next unit from a counter in the
// workspace (tc_reduce zeroes it), so a CTA that starts late, on an SM that the other
// kernel held until then, takes fewer units, and every SM that frees up joins in.
// Each run is a segment of its own: the producer loads its head's parameter block and
// memory operand into one of two buffers.  The other roles learn each tile's (head,
// tile, segment, flags) from a ring in shared memory that the producer fills before
// the tile's full barrier completes; after the last run it posts one end marker per
// compute group, and the first marker's group passes the end on to the two MMA
// issuers through its own barriers.

constexpr int kReadUnit = 4;                   // tiles per claimed unit
constexpr int kInfoRing = 16;                  // tile-info entries (>= X stages + compute groups)
enum : int { kTileFirst = 1, kTileLast = 2, kTileEnd = 4, kTileEndFirst = 8 };
struct TileInfo {
    int g, j, seg, flags;
};

// HV (K = 128): the scores are formed in two parts of 64 components through one
// 64-column region (a fourth issuer warp, kWarpMma1b, issues the second parts), so
// that three compute groups fit in TMEM instead of two.  (At K = 64 the same form
// gives four groups instead of three, but measured slower: 96 registers a thread.)
constexpr bool kReadHalves = true;
constexpr int kWarpMma1b = kWarpCompute;

template <int K, bool HV = (K == 128 && kReadHalves)>
struct ReadCfg {
    static constexpr bool HALVES = HV;
    static constexpr int NW = HV ? 3 : groups_for(K);
    static constexpr int WC = HV ? kWarpCompute + 1 : kWarpCompute;    // first compute warp
    static constexpr int THREADS = (WC + 4 * NW) * 32;
    static constexpr int SX = K <= 64 ? 6 : (HV ? 3 : 4);
    static constexpr int PN = 2;
    static constexpr uint32_t PB = align1k(param_bytes(K));
    static constexpr uint32_t MB = align1k(mem_bytes(K));
    static constexpr uint32_t OFF_X = 0;
    static constexpr uint32_t OFF_O = OFF_X + SX * kTileBytes;         // one output staging tile per group
    static constexpr uint32_t OFF_P = OFF_O + NW * kTileBytes;
    static constexpr uint32_t OFF_M = OFF_P + PN * PB;
    static constexpr uint32_t OFF_CA = OFF_M + PN * MB;                // constant [1, 1, 0...] A block
    static constexpr uint32_t OFF_INFO = OFF_CA + kConstABytes;        // tile-info ring
    static constexpr uint32_t OFF_BAR = OFF_INFO + kInfoRing * sizeof(TileInfo);
    static constexpr uint32_t BYTES = OFF_BAR + 512 + 1024;
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr int NOUT = 80;                                    // [Vt | Z | 1 | 0...]
    static constexpr uint32_t wg_cols = NOUT + (HV ? K / 2 : K);       // D2 | scores (then e)
    static constexpr uint32_t col_a(int w) { return w * wg_cols; }     // A operand, later D2 (same columns)
    static constexpr uint32_t col_d1(int w) { return w * wg_cols + NOUT; }
    static_assert(BYTES <= 232448 && NW * wg_cols <= TMEM_COLS, "read kernel exceeds shared memory or TMEM");
    // An entry is rewritten only after the tile kInfoRing places earlier has passed its
    // read MMA: the producer waits for tile i - SX's conversion, which follows the
    // epilogue (hence the read MMA) of tile i - SX - NW.
    static_assert(kInfoRing >= SX + NW, "tile-info ring shorter than the tiles in flight");
    // A group waits on tile i's routing stage by parity: the stage's previous tile (i - SX)
    // must be its own or one whose conversion it has seen, so SX >= NW.
    static_assert(SX >= NW, "fewer routing stages than compute groups");
};

template <int K, bool HV>
__global__ void __launch_bounds__(ReadCfg<K, HV>::THREADS, 1)
tc_read_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_o, TcArgs A) {
    using C = ReadCfg<K, HV>;
    constexpr int SX = C::SX, PN = C::PN, NW = C::NW;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + C::OFF_BAR);
    uint64_t *xfull = bars, *xempty = xfull + SX;
    uint64_t *a_full = xempty + SX, *d1_full = a_full + NW, *e_full = d1_full + NW, *d2_full = e_full + NW;
    uint64_t *w_full = d2_full + NW, *w_empty = w_full + PN;
    uint64_t *d1b_full = w_empty + PN, *d1_free = d1b_full + NW;       // the second score parts (HV)
    uint64_t *fin1 = d1_free + NW, *fin2 = fin1 + 1, *fin3 = fin2 + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(fin3 + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    TileInfo *info = reinterpret_cast<TileInfo *>(sm + C::OFF_INFO);

    grid_dep_launch();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < SX; ++s) { mbar_init(&xfull[s], 1); mbar_init(&xempty[s], 1); }
        for (int b = 0; b < NW; ++b) {
            mbar_init(&a_full[b], 1); mbar_init(&d1_full[b], 1); mbar_init(&e_full[b], 1); mbar_init(&d2_full[b], 1);
            mbar_init(&d1b_full[b], 1); mbar_init(&d1_free[b], 1);
        }
        for (int b = 0; b < PN; ++b) { mbar_init(&w_full[b], 1); mbar_init(&w_empty[b], 1); }
        mbar_init(fin1, 1); mbar_init(fin2, 1); mbar_init(fin3, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    init_const_a(sm + C::OFF_CA, threadIdx.x, blockDim.x);
    if (warp == kWarpMma1) { tmem_alloc(tmem_slot, C::TMEM_COLS); tmem_relinquish(); }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const Abort ab{abort_flag, A.status};

    if (warp == kWarpProducer) {
        if (lane == 0) {
            const int uph = (A.T + kReadUnit - 1) / kReadUnit;      // units per head
            const int nunits = A.G * uph;
            int t = 0, t_end = 0;
            if (!A.dyn) {
                t = (int)(((long long)blockIdx.x * A.Ttot) / gridDim.x);
                t_end = (int)(((long long)(blockIdx.x + 1) * A.Ttot) / gridDim.x);
            }
            // the next run of tiles [ja, jb) of head g: a claimed unit, or the part of the CTA's
            // static range that lies in the next head
            auto next_run = [&](int &g, int &ja, int &jb) -> bool {
                if (A.dyn) {
                    const int u = atomicAdd(A.claim, 1);
                    if (u >= nunits) return false;
                    g = u / uph;
                    ja = (u - g * uph) * kReadUnit;
                    jb = min(ja + kReadUnit, A.T);
                    return true;
                }
                if (t >= t_end) return false;
                g = t / A.T;
                ja = t - g * A.T;
                jb = min(A.T, ja + (t_end - t));
                t += jb - ja;
                return true;
            };
            int i = 0, nseg = 0, g = 0, ja = 0, jb = 0, pre = 0;   // tiles (and end markers) issued, segments
            bool have = false, ok = true;
            if (!A.dyn) {
                // a static range: its first query tiles do not depend on the previous kernel
                have = next_run(g, ja, jb);
                for (; have && pre < SX && ja + pre < jb; ++pre, ++i) {
                    const int j = ja + pre;
                    info[i] = TileInfo{g, j, 0, (pre == 0 ? kTileFirst : 0) | (j == jb - 1 ? kTileLast : 0)};
                    mbar_arrive_expect_tx(&xfull[i], kTileBytes);
                    tma_load_3d(sm + C::OFF_X + i * kTileBytes, &tm_q, &xfull[i], 0, j * TM, g);
                }
            }
            grid_dep_wait();             // parameter blocks, memory operands and the zeroed unit counter
            if (A.dyn) have = next_run(g, ja, jb);
            while (ok && have && !*abort_flag) {
                const int b = nseg % PN;
                if (nseg >= PN && !(ok = mbar_wait(&w_empty[b], ((nseg / PN) - 1) & 1, ab, kDevErrTimeout))) break;
                mbar_arrive_expect_tx(&w_full[b], param_bytes(K) + mem_bytes(K));
                bulk_load(sm + C::OFF_P + b * C::PB, A.params + (size_t)(g % A.H) * A.param_stride, param_bytes(K),
                          &w_full[b]);
                (void)GMA_IN_BOUNDS(g < A.G, A.status);
                bulk_load(sm + C::OFF_M + b * C::MB, A.mem + (size_t)g * A.mem_stride, mem_bytes(K), &w_full[b]);
                const int seg = nseg++;
                for (int j = ja + pre; j < jb; ++j, ++i) {
                    if (i >= SX && !(ok = mbar_wait(&xempty[i % SX], ((i / SX) - 1) & 1, ab, kDevErrTimeout))) break;
                    info[i % kInfoRing] = TileInfo{g, j, seg, (j == ja ? kTileFirst : 0) | (j == jb - 1 ? kTileLast : 0)};
                    mbar_arrive_expect_tx(&xfull[i % SX], kTileBytes);
                    tma_load_3d(sm + C::OFF_X + (i % SX) * kTileBytes, &tm_q, &xfull[i % SX], 0, j * TM, g);
                }
                pre = 0;
                if (ok) have = next_run(g, ja, jb);
            }
            for (int k = 0; k < NW && ok; ++k, ++i) {
                if (i >= SX && !(ok = mbar_wait(&xempty[i % SX], ((i / SX) - 1) & 1, ab, kDevErrTimeout))) break;
                info[i % kInfoRing] = TileInfo{0, 0, 0, kTileEnd | (k == 0 ? kTileEndFirst : 0)};
                mbar_arrive(&xfull[i % SX]);
            }
            wind_down_ring(xfull, SX, i, A.status);
            for (int s = nseg - PN < 0 ? 0 : nseg - PN; s < nseg; ++s)
                wait_ignoring_abort(&w_full[s % PN], (s / PN) & 1, A.status);
        }
    } else if (warp == kWarpMma1) {
        for (int i = 0;; ++i) {                      // the whole warp, converged
            const int w = i % NW;
            if (!mbar_wait_warp(&a_full[w], (i / NW) & 1, ab, kDevErrTimeout)) break;
            const TileInfo t = info[i % kInfoRing];
            if (t.flags & kTileEnd) break;
            const int b = t.seg % PN;
            if ((t.flags & kTileFirst) && !mbar_wait_warp(&w_full[b], (t.seg / PN) & 1, ab, kDevErrTimeout)) break;
            tc_fence_after();
            if constexpr (HV)
                issue_logdensity_part<K, K / 2>(tmem + C::col_d1(w), tmem + C::col_a(w),
                                                smem_u32(sm + C::OFF_P + b * C::PB), smem_u32(sm + C::OFF_CA), 0);
            else
                issue_logdensity<K>(tmem + C::col_d1(w), tmem + C::col_a(w), smem_u32(sm + C::OFF_P + b * C::PB),
                                    smem_u32(sm + C::OFF_CA));
            mma_commit(&d1_full[w]);
        }
        mma_commit(fin1);
        wait_ignoring_abort(fin1, 0, A.status);
    } else if (HV && warp == kWarpMma1b) {
        // second score parts: the group has read the first part out of the region
        for (int i = 0;; ++i) {                      // the whole warp, converged
            const int w = i % NW;
            if (!mbar_wait_warp(&d1_free[w], (i / NW) & 1, ab, kDevErrTimeout)) break;
            const TileInfo t = info[i % kInfoRing];
            if (t.flags & kTileEnd) break;
            const int b = t.seg % PN;
            tc_fence_after();
            issue_logdensity_part<K, K / 2>(tmem + C::col_d1(w), tmem + C::col_a(w),
                                            smem_u32(sm + C::OFF_P + b * C::PB), smem_u32(sm + C::OFF_CA), 1);
            mma_commit(&d1b_full[w]);
        }
        mma_commit(fin3);
        wait_ignoring_abort(fin3, 0, A.status);
    } else if (warp == kWarpMma2) {
        // read MMAs: D2 (128 rows x 80) = e (rows x K, bf16 in TMEM) . [Vt | Z | 1 | 0] (K x 80)
        constexpr uint32_t idesc = idesc_f16(1, 1, 0, 0, TM, C::NOUT);
        for (int i = 0;; ++i) {                      // the whole warp, converged
            const int w = i % NW;
            if (!mbar_wait_warp(&e_full[w], (i / NW) & 1, ab, kDevErrTimeout)) break;
            const TileInfo t = info[i % kInfoRing];
            if (t.flags & kTileEnd) break;
            const int b = t.seg % PN;
            tc_fence_after();
            const uint64_t bd = sdesc_sw128(smem_u32(sm + C::OFF_M + b * C::MB), 16, 1024);
#pragma unroll
            for (int ks = 0; ks < K / 16; ++ks)
                mma_ts(tmem + C::col_a(w), tmem + C::col_d1(w) + ks * 8,
                       bd + (uint64_t)(((ks >> 2) * 80u * 128u + (ks & 3) * 32u) >> 4), idesc, ks > 0);
            mma_commit(&d2_full[w]);
            if (t.flags & kTileLast) mma_commit(&w_empty[b]);
        }
        mma_commit(fin2);
        wait_ignoring_abort(fin2, 0, A.status);
    } else {
        RowThread rt;
        rt.wg = (warp - C::WC) >> 2;
        rt.r = 32u * (warp & 3) + lane;
        rt.lane_off = (uint32_t)(32 * (warp & 3)) << 16;
        rt.wtid = threadIdx.x - C::WC * 32 - rt.wg * kWgThreads;
        const int w = rt.wg;
        const bool elected = rt.wtid == 0;
        for (int i = w;; i += NW) {
            bool ok = mbar_wait(&xfull[i % SX], (i / SX) & 1, ab, kDevErrTimeout);
            if (!wg_all(rt, ok)) break;
            const TileInfo t = info[i % kInfoRing];
            if (t.flags & kTileEnd) {
                // the first end marker: the MMA issuers wait on this group's barriers next
                if ((t.flags & kTileEndFirst) && elected) {
                    mbar_arrive(&a_full[w]);
                    mbar_arrive(&e_full[w]);
                    if (HV) mbar_arrive(&d1_free[w]);
                }
                break;
            }
            convert_row(sm + C::OFF_X + (i % SX) * kTileBytes, rt.r, tmem + rt.lane_off + C::col_a(w));
            tmem_st_wait();
            tc_fence_before();
            wg_sync(rt);
            if (elected) { mbar_arrive(&a_full[w]); mbar_arrive(&xempty[i % SX]); }
            if (i < NW) grid_dep_wait();                   // the parameter blocks are written
            const float scale = head_scale(A.params, A.param_stride, t.g % A.H, K);
            ok = mbar_wait(&d1_full[w], (i / NW) & 1, ab, kDevErrTimeout);
            if (!wg_all(rt, ok)) break;
            tc_fence_after();
            const uint32_t d1 = tmem + rt.lane_off + C::col_d1(w);
            if constexpr (HV) {
                // the two parts of K/2 scores through the one region: e of part 0 stays in
                // registers while the second part's MMA writes the region
                uint32_t e[K / 2];
                uint32_t (&ea)[K / 4] = *reinterpret_cast<uint32_t (*)[K / 4]>(&e[0]);
                uint32_t (&eb)[K / 4] = *reinterpret_cast<uint32_t (*)[K / 4]>(&e[K / 4]);
                const float ma = row_exp_part0<K / 2>(d1, scale, ea);
                tc_fence_before();
                wg_sync(rt);
                if (elected) mbar_arrive(&d1_free[w]);
                ok = mbar_wait(&d1b_full[w], (i / NW) & 1, ab, kDevErrTimeout);
                if (!wg_all(rt, ok)) break;
                tc_fence_after();
                row_exp_part1<K / 2>(d1, scale, ma, ea, eb);
#pragma unroll
                for (int cc = 0; cc < K / 64; ++cc) tmem_st32(d1 + 32 * cc, e + 32 * cc);
            } else {
                // unnormalised responsibilities (the row scale cancels in num / den),
                // bf16 pairs written over the first K/2 score columns
                uint32_t e[K / 2];
                row_exp_scaled<K>(d1, scale, e);
#pragma unroll
                for (int cc = 0; cc < K / 64; ++cc) tmem_st32(d1 + 32 * cc, e + 32 * cc);
            }
            tmem_st_wait();
            tc_fence_before();
            wg_sync(rt);
            if (elected) mbar_arrive(&e_full[w]);
            // epilogue: out = num / (den + eps * sum_k e_k)
            ok = mbar_wait(&d2_full[w], (i / NW) & 1, ab, kDevErrTimeout);
            if (!wg_all(rt, ok)) break;
            tc_fence_after();
            uint32_t v0[32], v1[32], dz[4];
            tmem_ld32(tmem + rt.lane_off + C::col_a(w), v0);
            tmem_ld32(tmem + rt.lane_off + C::col_a(w) + 32, v1);
            tmem_ld4(tmem + rt.lane_off + C::col_a(w) + 64, dz);
            tmem_ld_wait();
            const float rd = 1.0f / (__uint_as_float(dz[0]) + A.eps * __uint_as_float(dz[1]));
            const uint64_t rd2 = f2_pack(rd, rd);
            uint8_t *ob = sm + C::OFF_O + w * kTileBytes;
            if (elected) bulk_wait_group_read<0>();          // this group's previous store left the buffer
            wg_sync(rt);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const uint32_t *src = j < 4 ? v0 + 8 * j : v1 + 8 * (j - 4);
                uint32_t o[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    float oa, obv;
                    f2_unpack(f2_mul(f2_pack(__uint_as_float(src[2 * u]), __uint_as_float(src[2 * u + 1])), rd2), oa, obv);
                    o[u] = pack_bf16(oa, obv);
                }
                *reinterpret_cast<uint4 *>(ob + sw128_off(rt.r, j)) = make_uint4(o[0], o[1], o[2], o[3]);
            }
            fence_proxy_async_smem();
            tc_fence_before();
            wg_sync(rt);
            if (elected) {
                tma_store_3d(&tm_o, ob, 0, t.j * TM, t.g);
                bulk_commit_group();
            }
        }
        if (elected) bulk_wait_group<0>();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kWarpMma1) {
        __syncwarp();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

// ------------------------------------------------------------------ host side

template <int K>
cudaError_t launch_write(const Problem &p, const TcLayout &L, const void *Kx, const void *V, char *ws,
                         cudaStream_t s) {
    CUtensorMap tk, tv;
    if (!make_map(&tk, Kx, p.G, p.Nkv, DR) || !make_map(&tv, V, p.G, p.Nkv, DVV)) return cudaErrorInvalidValue;
    TcArgs a{};
    a.G = p.G; a.H = p.H; a.N = p.Nkv; a.T = L.Tkv; a.Ttot = L.Ttot_kv; a.K = K;
    a.params = reinterpret_cast<const uint8_t *>(ws + L.params); a.param_stride = L.param_stride;
    a.partials = reinterpret_cast<float *>(ws + L.part);
    a.status = reinterpret_cast<unsigned *>(ws);
    a.nslots = kMaxCtas + p.G;
    auto kern = tc_write_kernel<K, false>;
    cudaError_t e = set_dyn_smem(reinterpret_cast<const void *>(kern), WriteCfg<K>::BYTES);
    if (e != cudaSuccess) return e;
    return launch_dependent(kern, dim3(L.ncta_kv), dim3(WriteCfg<K>::THREADS), WriteCfg<K>::BYTES, s, tk, tv, a,
                            NoSeg{});
}

template <int K>
cudaError_t launch_read(const Problem &p, const TcLayout &L, const void *Qx, void *out, char *ws,
                        cudaStream_t s) {
    CUtensorMap tq, to;
    if (!make_map(&tq, Qx, p.G, p.N, DR) || !make_map(&to, out, p.G, p.N, DVV)) return cudaErrorInvalidValue;
    TcArgs a{};
    a.G = p.G; a.H = p.H; a.N = p.N; a.T = L.T; a.Ttot = L.Ttot; a.K = K;
    a.params = reinterpret_cast<const uint8_t *>(ws + L.params); a.param_stride = L.param_stride;
    a.mem = reinterpret_cast<uint8_t *>(ws + L.mem); a.mem_stride = L.mem_stride;
    a.eps = p.eps;
    a.status = reinterpret_cast<unsigned *>(ws);
    a.claim = reinterpret_cast<int *>(ws + L.claim);
    a.dyn = p.sm_budget > 0;
    using C = ReadCfg<K>;
    auto kern = tc_read_kernel<K, C::HALVES>;
    cudaError_t e = set_dyn_smem(reinterpret_cast<const void *>(kern), C::BYTES);
    if (e != cudaSuccess) return e;
    return launch_dependent(kern, dim3(L.ncta), dim3(C::THREADS), C::BYTES, s, tq, to, a);
}

}  // namespace

bool tc_bidir_supported(const Problem &p) {
    return p.in_dtype == GMA_BF16 && p.out_dtype == GMA_BF16 && !p.causal && p.d == DR && p.dv == DVV &&
           (p.K == 64 || p.K == 128) && p.N > 0 && p.Nkv > 0;
}

TcLayout tc_layout(const Problem &p) {
    TcLayout L{};
    L.T = (p.N + TM - 1) / TM;
    L.Ttot = L.T * p.G;
    const int nsm = sm_count();
    // the read: static ranges when the call runs alone, units claimed from a counter beside
    // a concurrent kernel (a CTA that starts late takes fewer)
    const int units = p.G * ((L.T + kReadUnit - 1) / kReadUnit);
    L.ncta = std::max(1, std::min({nsm > 0 ? nsm : kMaxCtas, kMaxCtas, p.sm_budget > 0 ? units : L.Ttot}));
    L.Tkv = (p.Nkv + TM - 1) / TM;
    L.Ttot_kv = L.Tkv * p.G;
    // the write kernel's static ranges: on the SMs left free by a concurrent kernel when
    // the call runs with an SM budget (gma_forward_multi), else on every SM
    const int wsm = p.sm_budget > 0 && nsm > 0 ? std::min(nsm, p.sm_budget) : nsm;
    L.ncta_kv = std::max(1, std::min({wsm > 0 ? wsm : kMaxCtas, kMaxCtas, L.Ttot_kv}));
    L.param_stride = align1k(param_bytes(p.K));
    L.mem_stride = align1k(mem_bytes(p.K));
    size_t off = kHeaderBytes;
    L.params = align_up(off);
    off = L.params + (size_t)p.H * L.param_stride;
    L.part = align_up(off);
    off = L.part + sizeof(float) * (size_t)(kMaxCtas + p.G) * (DVV + 1) * p.K;
    L.mem = align_up(off);
    off = L.mem + (size_t)p.G * L.mem_stride;
    L.claim = align_up(off);
    off = L.claim + 16;
    L.total = align_up(off);
    return L;
}

cudaError_t tc_params(const Problem &p, const TcLayout &L, const float *mu, const float *rho,
                      const float *alpha, char *ws, cudaStream_t s) {
    auto kern = p.K <= 64 ? tc_params_kernel<64> : p.K <= 128 ? tc_params_kernel<128>
              : p.K <= 192 ? tc_params_kernel<192> : tc_params_kernel<256>;
    if (p.K != 64 && p.K != 128 && p.K != 192 && p.K != 256) return cudaErrorInvalidValue;
    kern<<<p.H, kParamThreads, 0, s>>>(p.var_floor, mu, rho, alpha, reinterpret_cast<uint8_t *>(ws + L.params),
                                          L.param_stride);
    return cudaGetLastError();
}

cudaError_t tc_write(const Problem &p, const TcLayout &L, const void *Kx, const void *V, char *ws,
                     cudaStream_t s) {
    return p.K == 64 ? launch_write<64>(p, L, Kx, V, ws, s) : launch_write<128>(p, L, Kx, V, ws, s);
}

cudaError_t tc_prefix(const Problem &p, const TcLayout &L, const SegTable &T, const void *Kx, const void *V, char *ws,
                      cudaStream_t s) {
    if (T.np == 0) return cudaSuccess;
    CUtensorMap tk, tv;
    if (!make_map(&tk, Kx, p.G, p.N, DR) || !make_map(&tv, V, p.G, p.N, DVV)) return cudaErrorInvalidValue;
    TcArgs a{};
    a.G = p.G; a.H = p.H; a.N = p.N; a.T = T.nch; a.Ttot = T.vtot; a.K = 64;
    a.params = reinterpret_cast<const uint8_t *>(ws + L.params); a.param_stride = L.param_stride;
    a.partials = reinterpret_cast<float *>(ws + L.part);
    a.status = reinterpret_cast<unsigned *>(ws);
    a.nslots = T.np + T.nseg + 1;
    auto kern = tc_write_kernel<64, true>;
    cudaError_t e = set_dyn_smem(reinterpret_cast<const void *>(kern), WriteCfg<64>::BYTES);
    if (e != cudaSuccess) return e;
    return launch_dependent(kern, dim3(T.np), dim3(WriteCfg<64>::THREADS), WriteCfg<64>::BYTES, s, tk, tv, a, T);
}

cudaError_t tc_reduce(const Problem &p, const TcLayout &L, char *ws, cudaStream_t s) {
    return tc_reduce_split(p, L, L.part, L.mem, 0, ws, s, L.claim);
}

cudaError_t tc_reduce_split(const Problem &p, const TcLayout &L, size_t part, size_t mem, size_t mem_lo, char *ws,
                            cudaStream_t s, size_t claim) {
    dim3 grid((20 * p.K + kReduceThreads - 1) / kReduceThreads, p.G);
    return launch_dependent(tc_reduce_kernel, grid, dim3(kReduceThreads), 0, s, p.K, L.Tkv, L.Ttot_kv, L.ncta_kv,
                            reinterpret_cast<const float *>(ws + part), reinterpret_cast<uint8_t *>(ws + mem),
                            mem_lo ? reinterpret_cast<uint8_t *>(ws + mem_lo) : nullptr, L.mem_stride, kMaxCtas + p.G,
                            claim ? reinterpret_cast<int *>(ws + claim) : nullptr, reinterpret_cast<unsigned *>(ws));
}

cudaError_t tc_read(const Problem &p, const TcLayout &L, const void *Qx, void *out, char *ws,
                    cudaStream_t s) {
    return p.K == 64 ? launch_read<64>(p, L, Qx, out, ws, s) : launch_read<128>(p, L, Qx, out, ws, s);
}

}  // namespace gma
