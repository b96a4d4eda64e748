// Backward pass of bidirectional GMA on the CUDA cores (fp32 arithmetic).
//
// "Gaussian Mixture Attention" (Huang & Raza, 2026), section 4.1: the upstream
// gradient g at a responsibility vector enters the scores through the softmax
// Jacobian, ds_ik = gamma_ik (g_ik - sum_j gamma_ij g_ij) (Eq. 17-18); every
// quantity that enters a score collects sum_i sum_k ds_ik ds_ik/dtheta (Eq. 19),
// with ds_ik/dmu_k = Sigma_k^-1 (x_i - mu_k) (Eq. 20), ds_ik/dx_i =
// -Sigma_k^-1 (x_i - mu_k) (section 4.3), the variance derivative of the score
// of Eq. 16, and Eq. 14-15 for rho and alpha.  The memory products of
// Eq. 5-8 are differentiated as products: with den_i = gamma^Q_i . Z + eps,
// a_i = dO_i / den_i and b_i = -(dO_i . O_i) / den_i,
//   g^Q_i = Vt a_i + Z b_i,   R = sum_i gamma^Q_i a_i^T,   r = sum_i gamma^Q_i b_i,
//   g^K_j = R v_j + r,        dV_j = R^T gamma^K_j.
//
// Three passes of one kernel over 64-row tiles (one CTA per (row chunk, head),
// 256 threads):
//   MEM  key rows:   gamma^K (stored for the key pass), [Vt | Z] partials  (Eq. 5-6)
//   QRY  query rows: gamma^Q, a, b, g^Q, ds, dQx; partials of [R | r] and of the parameter sums
//   KEY  key rows:   gamma^K as stored, g^K, dV, ds, dKx; partials of the parameter sums
// with fixed-order reductions of the partials in between and a finalize that
// turns the parameter sums P1 = sum ds x, P2 = sum ds x^2, P0 = sum ds into
// dmu, drho, dalpha.  Every product is a 4 x 4 register-blocked loop over
// shared memory; the scores use the expanded form
//   s_ik = c'_k + sum_j (lambda mu)_kj x_ij - (1/2) sum_j lambda_kj x_ij^2,
//   c'_k = log pi_k - (1/2) log|Sigma_k| - (1/2) sum_j lambda_kj mu_kj^2,
// so that the score is one product [x, x^2] . W.  Shapes: d = dv = K = 64.
#include <cuda_bf16.h>

#include <algorithm>
#include <cfloat>
#include <cstdint>

#include "gma_internal.h"

namespace gma {
namespace {

constexpr int kBT = 256;          // threads of a pass CTA
constexpr int kTN = 64;           // rows per tile
constexpr int kK = 64, kD = 64, kDV = 64;
constexpr int kW = kDV + 1;       // [value columns | normaliser] of a memory
constexpr int kPW = 2 * kD + 1;   // parameter sums per component: P1 [d], P2 [d], P0
constexpr int kRS = 68;           // row stride of the per-tile arrays (16-byte rows, spread banks)

enum BwdMode { kMem = 0, kQry = 1, kKey = 2 };

// Shared memory of one pass CTA, in floats.
constexpr int OFF_W = 0;                         // [2d][K]  score weights: lambda mu, then -lambda / 2
constexpr int OFF_CP = OFF_W + 2 * kD * kK;      // [K]      c'_k
constexpr int OFF_LAM = OFF_CP + kK;             // [K][d]   lambda
constexpr int OFF_LMU = OFF_LAM + kK * kD;       // [K][d]   lambda mu
constexpr int OFF_M = OFF_LMU + kK * kD;         // [K][dv]  Vt (QRY) or R (KEY)
constexpr int OFF_MT = OFF_M + kK * kDV;         // [dv][K]  its transpose
constexpr int OFF_ZR = OFF_MT + kDV * kK;        // [K]      Z (QRY) or r (KEY)
constexpr int OFF_X = OFF_ZR + kK;               // [TN][kRS] routing rows
constexpr int OFF_A = OFF_X + kTN * kRS;         // [TN][kRS] values (MEM, KEY) / dO then a (QRY)
constexpr int OFF_G = OFF_A + kTN * kRS;         // [TN][kRS] scores, then gamma
constexpr int OFF_S = OFF_G + kTN * kRS;         // [TN][kRS] g, then ds
constexpr int OFF_DEN = OFF_S + kTN * kRS;       // [TN]     den (QRY)
constexpr int OFF_B = OFF_DEN + kTN;             // [TN]     b (QRY)
constexpr int kBwdSmemFloats = OFF_B + kTN;
constexpr size_t kBwdSmemBytes = sizeof(float) * kBwdSmemFloats;
static_assert(kBwdSmemBytes <= 227 * 1024, "pass CTA shared memory");
static_assert((OFF_X | OFF_A | OFF_G | OFF_S | OFF_M | OFF_MT | OFF_LAM | OFF_LMU | OFF_W) % 4 == 0, "float4 rows");

struct BwdArgs {
    int N, H, C, rows_per_chunk;       // rows per head, heads per batch entry, chunks per head
    float eps;
    const void *X;                     // Qx (QRY) or Kx (MEM, KEY)  [G][N][d]
    const void *U;                     // V (MEM, KEY) or dO (QRY)   [G][N][dv]
    const float *mu, *lam, *cdir;      // [H][K][d], [H][K][d], [H][K]
    const float *mem;                  // [G][K][W]: [Vt | Z] (QRY) or [R | r] (KEY)
    float *dX;                         // dQx (QRY) or dKx (KEY)     [G][N][d]
    float *dV;                         // KEY                        [G][N][dv]
    float *part_m;                     // MEM, QRY: [G][C][K][W]
    float *part_p;                     // QRY, KEY: [G][C][K][2d + 1]
    float *gam;                        // MEM writes, KEY reads gamma^K [G][N][K]
};

__device__ __forceinline__ float bwd_warp_sum(float v) {
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(~0u, v, o);
    return v;
}
__device__ __forceinline__ float bwd_warp_max(float v) {
    for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(~0u, v, o));
    return v;
}

__device__ __forceinline__ float4 ld4(const float *p) { return *reinterpret_cast<const float4 *>(p); }

// Sixteen consecutive elements of one row (a quarter of a 64-wide row), held in registers
// between their global load and their store into shared memory, so that the next tile's
// rows are in flight while the current tile computes.
template <typename TI> struct Row16;
template <> struct Row16<float> {
    float4 v[4];
    __device__ void load(const float *src, bool live) {
#pragma unroll
        for (int i = 0; i < 4; ++i) v[i] = live ? reinterpret_cast<const float4 *>(src)[i] : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    __device__ void store(float *dst) const {
#pragma unroll
        for (int i = 0; i < 4; ++i) reinterpret_cast<float4 *>(dst)[i] = v[i];
    }
};
template <> struct Row16<__nv_bfloat16> {
    uint4 v[2];
    __device__ void load(const __nv_bfloat16 *src, bool live) {
#pragma unroll
        for (int i = 0; i < 2; ++i) v[i] = live ? reinterpret_cast<const uint4 *>(src)[i] : make_uint4(0u, 0u, 0u, 0u);
    }
    __device__ void store(float *dst) const {
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {           // bf16 -> fp32 is a 16-bit shift
                dst[8 * i + 2 * q] = __uint_as_float(w[q] << 16);
                dst[8 * i + 2 * q + 1] = __uint_as_float(w[q] & 0xffff0000u);
            }
        }
    }
};

__device__ __forceinline__ void fma4x4(float (&c)[4][4], const float (&a)[4], const float4 b) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        c[i][0] = fmaf(a[i], b.x, c[i][0]);
        c[i][1] = fmaf(a[i], b.y, c[i][1]);
        c[i][2] = fmaf(a[i], b.z, c[i][2]);
        c[i][3] = fmaf(a[i], b.w, c[i][3]);
    }
}

__device__ __forceinline__ void zero4x4(float (&c)[4][4]) {
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) c[i][j] = 0.f;
}

// c[i][j] += sum_{s < S} A[(r0 + i) * as + s] * B[s * bs + c0 + j]: A row-major with the
// summed index contiguous (scalar loads, shared by a half-warp), B with the summed index
// outermost (one float4 per step).
template <int S>
__device__ __forceinline__ void mm_rows(float (&c)[4][4], const float *A, int as, int r0, const float *B, int bs,
                                        int c0) {
#pragma unroll 8
    for (int s = 0; s < S; ++s) {
        const float a[4] = {A[(r0 + 0) * as + s], A[(r0 + 1) * as + s], A[(r0 + 2) * as + s],
                            A[(r0 + 3) * as + s]};
        fma4x4(c, a, ld4(B + s * bs + c0));
    }
}

// c[i][j] += sum_{m < TN} A[m * as + r0 + i] * B[m * bs + c0 + j]: both operands with the
// summed row index outermost (the accumulations over a tile's rows).
__device__ __forceinline__ void mm_cols(float (&c)[4][4], const float *A, int as, int r0, const float *B, int bs,
                                        int c0) {
#pragma unroll 8
    for (int m = 0; m < kTN; ++m) {
        const float4 a4 = ld4(A + m * as + r0);
        const float a[4] = {a4.x, a4.y, a4.z, a4.w};
        fma4x4(c, a, ld4(B + m * bs + c0));
    }
}

// One pass over the rows [chunk * rows_per_chunk, +rows_per_chunk) of head g = blockIdx.y.
// Thread t owns the 4 x 4 output block (rows (t / 16) * 4.., columns (t % 16) * 4..) of
// every 64 x 64 product, and the same block of the accumulated memory and parameter sums.
template <int MODE, typename TI>
__global__ void __launch_bounds__(kBT, 1) bwd_pass_kernel(BwdArgs a) {
    extern __shared__ __align__(16) float sm[];
    float *W = sm + OFF_W, *cp = sm + OFF_CP, *lam = sm + OFF_LAM, *lmu = sm + OFF_LMU;
    float *M = sm + OFF_M, *MT = sm + OFF_MT, *zr = sm + OFF_ZR;
    float *xs = sm + OFF_X, *us = sm + OFF_A, *gs = sm + OFF_G, *ss = sm + OFF_S;
    float *den = sm + OFF_DEN, *bb = sm + OFF_B;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int r0 = (tid >> 4) * 4, c0 = (tid & 15) * 4;
    const int ch = blockIdx.x, g = blockIdx.y, h = g % a.H;
    const TI *X = static_cast<const TI *>(a.X) + (size_t)g * a.N * kD;
    const TI *U = static_cast<const TI *>(a.U) + (size_t)g * a.N * kDV;

    // the head's precisions, lambda mu, the score weights and constants (Eq. 14-16)
    const float *lam_h = a.lam + (size_t)h * kK * kD, *mu_h = a.mu + (size_t)h * kK * kD;
    for (int e = tid; e < kK * kD; e += kBT) {
        const float l = lam_h[e];
        lam[e] = l;
        lmu[e] = l * mu_h[e];
    }
    __syncthreads();
    for (int e = tid; e < 2 * kD * kK; e += kBT) {
        const int q = e / kK, k = e % kK;
        W[e] = q < kD ? lmu[k * kD + q] : -0.5f * lam[k * kD + q - kD];
    }
    if (tid < kK) {
        float s = 0.f;
        for (int j = 0; j < kD; ++j) s = fmaf(lmu[tid * kD + j], mu_h[tid * kD + j], s);
        cp[tid] = a.cdir[(size_t)h * kK + tid] - 0.5f * s;
    }
    if (MODE != kMem) {
        const float *mg = a.mem + (size_t)g * kK * kW;
        for (int e = tid; e < kK * kW; e += kBT) {
            const int k = e / kW, c = e - k * kW;
            const float v = mg[e];
            if (c < kDV) {
                M[k * kDV + c] = v;
                MT[c * kK + k] = v;
            } else {
                zr[k] = v;
            }
        }
    }
    float accM[4][4], accP1[4][4], accP2[4][4];
    zero4x4(accM);
    zero4x4(accP1);
    zero4x4(accP2);
    float ex_m = 0.f, ex_p = 0.f;     // the memory's last column (threads < K); P0 (threads K..2K-1)
    __syncthreads();

    const int row_begin = ch * a.rows_per_chunk;
    const int row_end = min(a.N, row_begin + a.rows_per_chunk);
    // thread t carries row t / 4, elements (t % 4) * 16 .. +15, of the X and U tiles
    const int lm = tid >> 2, lj = (tid & 3) * 16;
    Row16<TI> rx, ru;
    if (row_begin < row_end) {
        const bool live = row_begin + lm < row_end;
        rx.load(X + (size_t)(row_begin + lm) * kD + lj, live);
        ru.load(U + (size_t)(row_begin + lm) * kDV + lj, live);
    }
    for (int t0 = row_begin; t0 < row_end; t0 += kTN) {
        const int mv = min(kTN, row_end - t0);
        rx.store(xs + lm * kRS + lj);
        ru.store(us + lm * kRS + lj);
        if (MODE == kKey) {                     // gamma^K as the memory pass left it
            const float *gsrc = a.gam + ((size_t)g * a.N + t0) * kK;
            for (int e = tid; e < kTN * (kK / 4); e += kBT) {
                const int m = e / (kK / 4), q = e - m * (kK / 4);
                reinterpret_cast<float4 *>(gs + m * kRS)[q] =
                    m < mv ? reinterpret_cast<const float4 *>(gsrc + (size_t)m * kK)[q] : make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
        __syncthreads();
        if (t0 + kTN < row_end) {               // the next tile's rows, in flight during this tile
            const bool live = t0 + kTN + lm < row_end;
            rx.load(X + (size_t)(t0 + kTN + lm) * kD + lj, live);
            ru.load(U + (size_t)(t0 + kTN + lm) * kDV + lj, live);
        }
        // Eq. 16, expanded: s = c' + x . (lambda mu) - (1/2) x^2 . lambda (the key pass reuses the
        // memory pass's responsibilities)
        if (MODE != kKey) {
            float c[4][4];
            zero4x4(c);
            mm_rows<kD>(c, xs, kRS, r0, W, kK, c0);
#pragma unroll 4
            for (int s = 0; s < kD; ++s) {
                float x2[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float v = xs[(r0 + i) * kRS + s];
                    x2[i] = v * v;
                }
                fma4x4(c, x2, ld4(W + (kD + s) * kK + c0));
            }
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) gs[(r0 + i) * kRS + c0 + j] = cp[c0 + j] + c[i][j];
        }
        __syncthreads();
        // Eq. 3b, a warp per row; rows past the end get gamma = 0 and so contribute nothing
        for (int m = warp; MODE != kKey && m < kTN; m += kBT / 32) {
            const float s0 = gs[m * kRS + lane], s1 = gs[m * kRS + lane + 32];
            const float mx = bwd_warp_max(fmaxf(s0, s1));
            float e0 = expf(s0 - mx), e1 = expf(s1 - mx);
            const float inv = 1.0f / bwd_warp_sum(e0 + e1);
            const bool live = m < mv;
            e0 = live ? e0 * inv : 0.f;
            e1 = live ? e1 * inv : 0.f;
            gs[m * kRS + lane] = e0;
            gs[m * kRS + lane + 32] = e1;
            if (MODE == kMem && live) {
                a.gam[((size_t)g * a.N + t0 + m) * kK + lane] = e0;
                a.gam[((size_t)g * a.N + t0 + m) * kK + lane + 32] = e1;
            }
            if (MODE == kQry) {
                const float z = bwd_warp_sum(e0 * zr[lane] + e1 * zr[lane + 32]);
                if (lane == 0) den[m] = live ? z + a.eps : 1.f;      // rows past the end: a = b = 0 even at eps = 0
            }
        }
        __syncthreads();
        if (MODE == kQry) {
            // Eq. 7-8: O = gamma Vt / den; a = dO / den, b = -(dO . O) / den (in place of dO)
            float c[4][4];
            zero4x4(c);
            mm_rows<kK>(c, gs, kRS, r0, M, kDV, c0);
            float dot[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float dn = den[r0 + i];
                float p = 0.f;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    float *q = us + (r0 + i) * kRS + c0 + j;
                    p = fmaf(*q, c[i][j] / dn, p);
                    *q = *q / dn;
                }
                dot[i] = p;
            }
#pragma unroll
            for (int i = 0; i < 4; ++i)
                for (int o = 8; o; o >>= 1) dot[i] += __shfl_xor_sync(~0u, dot[i], o);   // the row block's 16 threads
            if ((tid & 15) == 0)
#pragma unroll
                for (int i = 0; i < 4; ++i) bb[r0 + i] = -dot[i] / den[r0 + i];
            __syncthreads();
            // g^Q = a Vt^T + b Z
            zero4x4(c);
            mm_rows<kDV>(c, us, kRS, r0, MT, kK, c0);
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) ss[(r0 + i) * kRS + c0 + j] = fmaf(bb[r0 + i], zr[c0 + j], c[i][j]);
            __syncthreads();
        } else if (MODE == kKey) {
            // g^K = R v + r and dV = gamma^K R
            float c[4][4];
            zero4x4(c);
            mm_rows<kDV>(c, us, kRS, r0, MT, kK, c0);
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) ss[(r0 + i) * kRS + c0 + j] = c[i][j] + zr[c0 + j];
            zero4x4(c);
            mm_rows<kK>(c, gs, kRS, r0, M, kDV, c0);
#pragma unroll
            for (int i = 0; i < 4; ++i)
                if (r0 + i < mv)
                    *reinterpret_cast<float4 *>(a.dV + ((size_t)g * a.N + t0 + r0 + i) * kDV + c0) =
                        make_float4(c[i][0], c[i][1], c[i][2], c[i][3]);
            __syncthreads();
        }
        if (MODE != kMem) {
            // Eq. 18: ds = gamma (g - gamma . g), a warp per row
            for (int m = warp; m < kTN; m += kBT / 32) {
                const float g0 = gs[m * kRS + lane], g1 = gs[m * kRS + lane + 32];
                const float u0 = ss[m * kRS + lane], u1 = ss[m * kRS + lane + 32];
                const float mean = bwd_warp_sum(g0 * u0 + g1 * u1);
                ss[m * kRS + lane] = g0 * (u0 - mean);
                ss[m * kRS + lane + 32] = g1 * (u1 - mean);
            }
            __syncthreads();
            // section 4.3: dx = -sum_k ds_k lambda_k (x - mu_k) = ds . (lambda mu) - x (ds . lambda)
            float c1[4][4], c2[4][4];
            zero4x4(c1);
            zero4x4(c2);
#pragma unroll 4
            for (int s = 0; s < kK; ++s) {
                const float d4[4] = {ss[(r0 + 0) * kRS + s], ss[(r0 + 1) * kRS + s], ss[(r0 + 2) * kRS + s],
                                     ss[(r0 + 3) * kRS + s]};
                fma4x4(c1, d4, ld4(lam + s * kD + c0));
                fma4x4(c2, d4, ld4(lmu + s * kD + c0));
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                if (r0 + i >= mv) continue;
                const float *x = xs + (r0 + i) * kRS + c0;
                *reinterpret_cast<float4 *>(a.dX + ((size_t)g * a.N + t0 + r0 + i) * kD + c0) =
                    make_float4(fmaf(-x[0], c1[i][0], c2[i][0]), fmaf(-x[1], c1[i][1], c2[i][1]),
                                fmaf(-x[2], c1[i][2], c2[i][2]), fmaf(-x[3], c1[i][3], c2[i][3]));
            }
            // Eq. 19-20 and the variance derivative, as sums over the rows: P1 = sum ds x, P2 = sum ds x^2
#pragma unroll 4
            for (int m = 0; m < kTN; ++m) {
                const float4 d4 = ld4(ss + m * kRS + r0);
                const float dk[4] = {d4.x, d4.y, d4.z, d4.w};
                const float4 x4 = ld4(xs + m * kRS + c0);
                fma4x4(accP1, dk, x4);
                fma4x4(accP2, dk, make_float4(x4.x * x4.x, x4.y * x4.y, x4.z * x4.z, x4.w * x4.w));
            }
            if (tid >= kK && tid < 2 * kK)
                for (int m = 0; m < kTN; ++m) ex_p += ss[m * kRS + tid - kK];
        }
        if (MODE != kKey) {
            // Eq. 5-6 (MEM: [Vt | Z]) or the same product for the backward memory (QRY: [R | r])
            mm_cols(accM, gs, kRS, r0, us, kRS, c0);
            if (tid < kK)
                for (int m = 0; m < kTN; ++m) ex_m = fmaf(gs[m * kRS + tid], MODE == kMem ? 1.f : bb[m], ex_m);
        }
        __syncthreads();
    }

    const size_t slot = (size_t)g * a.C + ch;
    if (MODE != kKey) {
        float *pm = a.part_m + slot * kK * kW;
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) pm[(r0 + i) * kW + c0 + j] = accM[i][j];
        if (tid < kK) pm[tid * kW + kDV] = ex_m;
    }
    if (MODE != kMem) {
        float *pp = a.part_p + slot * kK * kPW;
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                pp[(r0 + i) * kPW + c0 + j] = accP1[i][j];
                pp[(r0 + i) * kPW + kD + c0 + j] = accP2[i][j];
            }
        if (tid >= kK && tid < 2 * kK) pp[(tid - kK) * kPW + 2 * kD] = ex_p;
    }
}

// out[g][e] = sum over the C chunk slots of head g, in slot order.
__global__ void bwd_sum_kernel(int C, int E, const float *__restrict__ part, float *__restrict__ out) {
    const int g = blockIdx.y, e = blockIdx.x * blockDim.x + threadIdx.x;
    if (e >= E) return;
    float s = 0.f;
    for (int c = 0; c < C; ++c) s += part[((size_t)g * C + c) * E + e];
    out[(size_t)g * E + e] = s;
}

// Parameter gradients of component k = blockIdx.x of head h = blockIdx.y from the sums over
// its query and key rows of every batch entry (fixed order: queries then keys, batch
// entries, chunks); 128 threads, thread t < d sums P1 of dimension t, thread d + t sums P2:
//   Q1 = sum ds (x - mu) = P1 - mu P0,  Q2 = sum ds (x - mu)^2 = P2 - 2 mu P1 + mu^2 P0
//   dmu = lambda Q1                                             (Eq. 20)
//   dvar = (1/2) (lambda^2 Q2 - lambda P0),  drho = dvar sigmoid(rho)   (Eq. 16, 14)
//   dalpha_k = P0_k - pi_k sum_l P0_l                           (Eq. 15; every CTA of the
//   head sums the P0 column, the K values of one row of partials at a stride)
__global__ void __launch_bounds__(2 * kD) bwd_param_kernel(int B, int H, int C, const float *__restrict__ pq,
                                                           const float *__restrict__ pk,
                                                           const float *__restrict__ mu,
                                                           const float *__restrict__ lam,
                                                           const float *__restrict__ rho,
                                                           const float *__restrict__ alpha,
                                                           float *__restrict__ dmu, float *__restrict__ drho,
                                                           float *__restrict__ dalpha) {
    __shared__ float p12[2 * kD];
    __shared__ float p0[kK];
    __shared__ float red[2];
    const int k = blockIdx.x, h = blockIdx.y, t = threadIdx.x;
    auto psum = [&](int kk, int q) {
        float s = 0.f;
        for (int side = 0; side < 2; ++side) {
            const float *p = side ? pk : pq;
            for (int b = 0; b < B; ++b)
                for (int c = 0; c < C; ++c) s += p[(((size_t)(b * H + h) * C + c) * kK + kk) * kPW + q];
        }
        return s;
    };
    p12[t] = psum(k, t);                       // P1 (t < d), P2 (t >= d)
    if (t < kK) p0[t] = psum(t, 2 * kD);
    __syncthreads();
    if (t == 0) {                              // sum_l P0_l and log-sum-exp of alpha, in order
        const float *al = alpha + (size_t)h * kK;
        float tot = 0.f, mx = -FLT_MAX, se = 0.f;
        for (int l = 0; l < kK; ++l) {
            tot += p0[l];
            mx = fmaxf(mx, al[l]);
        }
        for (int l = 0; l < kK; ++l) se += expf(al[l] - mx);
        red[0] = tot;
        red[1] = mx + logf(se);
    }
    __syncthreads();
    if (t < kD) {
        const size_t o = ((size_t)h * kK + k) * kD + t;
        const float P1 = p12[t], P2 = p12[kD + t], P0 = p0[k];
        const float m = mu[o], l = lam[o];
        const float q1 = fmaf(-m, P0, P1);
        const float q2 = fmaf(m, fmaf(m, P0, -2.f * P1), P2);
        dmu[o] = l * q1;
        const float dvar = 0.5f * l * fmaf(l, q2, -P0);
        drho[o] = dvar / (1.f + expf(-rho[o]));
    } else if (t == kD) {
        dalpha[(size_t)h * kK + k] = fmaf(-expf(alpha[(size_t)h * kK + k] - red[1]), red[0], p0[k]);
    }
}

// ---------------------------------------------------------------------------------------
// Causal backward (prefix memories of Eq. 6b / 8b).  Each CTA walks the tiles of its row
// chunk in order (queries) or in reverse (keys), carrying the memory of everything before
// (S, z) or after (R, r) the tile.  Within a tile, with the causal mask [j <= i]:
//   A  = tril(G^Q G^K^T),  num = G^Q S + A V,  den = G^Q z + A 1 + eps
//   Bm = tril(a V^T + b 1^T),  g^Q = a S^T + b z^T + Bm G^K
//   Ct = (tril(a V^T + b 1^T))^T,  g^K = Ct G^Q + V R^T + r
//   Dt = (tril(G^Q G^K^T))^T,      dV  = Dt a + G^K R
// The query pass takes gamma^K from the memory pass and stores gamma^Q; the key pass
// reads both.  ds of either side goes to global memory; bwd_rows_kernel turns it into
// dX and the parameter sums.

constexpr int kTile = kTN * kRS;                  // one [TN][kRS] tile buffer
constexpr int CC_W = 0;                           // [2d][K]
constexpr int CC_CP = CC_W + 2 * kD * kK;         // [K]
constexpr int CC_M = CC_CP + kK;                  // [K][dv]   S (queries) or R (keys)
constexpr int CC_MT = CC_M + kK * kDV;            // [dv][K]   its transpose
constexpr int CC_ZR = CC_MT + kDV * kK;           // [K]       z or r
constexpr int CC_T = CC_ZR + kK;                  // nine tile buffers
constexpr int CC_DEN = CC_T + 9 * kTile;          // [TN]
constexpr int CC_B = CC_DEN + kTN;                // [TN]
constexpr int kCSmemFloats = CC_B + kTN;
constexpr size_t kCSmemBytes = sizeof(float) * kCSmemFloats;
static_assert(kCSmemBytes <= 227 * 1024, "causal pass CTA shared memory");
static_assert((CC_M | CC_MT | CC_T | kTile) % 4 == 0, "float4 rows");

struct BwdCArgs {
    int N, H, C, rows_per_chunk;
    float eps;
    const void *Qx, *Kx, *V, *dO;                 // [G][N][d] / [G][N][dv]
    const float *mu, *lam, *cdir;
    const float *mem;                             // [G][C][K][W]: S|z before (queries) / R|r after (keys) the chunk
    float *ab;                                    // [G][N][kRS]: a (dv columns), b, zeros
    float *ds;                                    // [G][N][K]
    float *dV;                                    // keys: [G][N][dv]
    float *part_m;                                // queries: [G][C][K][W] chunk totals of [R | r]
    const float *gk;                              // gamma^K [G][N][K] from the memory pass
    float *gq;                                    // gamma^Q [G][N][K]: queries write, keys read
};

// W, c' (Eq. 16, expanded; when `scores`) and the chunk's starting memory, from global memory.
__device__ void causal_prologue(const BwdCArgs &a, float *sm, int h, const float *mem_chunk, bool scores) {
    const float *lam_h = a.lam + (size_t)h * kK * kD, *mu_h = a.mu + (size_t)h * kK * kD;
    float *W = sm + CC_W, *cp = sm + CC_CP, *M = sm + CC_M, *MT = sm + CC_MT, *zr = sm + CC_ZR;
    for (int e = threadIdx.x; scores && e < 2 * kD * kK; e += kBT) {
        const int q = e / kK, k = e % kK;
        W[e] = q < kD ? lam_h[k * kD + q] * mu_h[k * kD + q] : -0.5f * lam_h[k * kD + q - kD];
    }
    if (scores && threadIdx.x < kK) {
        const int k = threadIdx.x;
        float s = 0.f;
        for (int j = 0; j < kD; ++j) {
            const float m = mu_h[k * kD + j];
            s = fmaf(lam_h[k * kD + j] * m, m, s);
        }
        cp[k] = a.cdir[(size_t)h * kK + k] - 0.5f * s;
    }
    for (int e = threadIdx.x; e < kK * kW; e += kBT) {
        const int k = e / kW, c = e - k * kW;
        const float v = mem_chunk[e];
        if (c < kDV) {
            M[k * kDV + c] = v;
            MT[c * kK + k] = v;
        } else {
            zr[k] = v;
        }
    }
}

// Rows t0 .. t0 + mv - 1 of a [G][N][64] float32 array (head base `src`) into a tile buffer,
// and its transpose into `dstT` when given; zeros below.
__device__ __forceinline__ void load_tile_f32(float *dst, const float *src, int t0, int mv) {
    for (int e = threadIdx.x; e < kTN * 16; e += kBT) {
        const int m = e >> 4, q = e & 15;
        reinterpret_cast<float4 *>(dst + m * kRS)[q] =
            m < mv ? reinterpret_cast<const float4 *>(src + (size_t)(t0 + m) * 64)[q] : make_float4(0.f, 0.f, 0.f, 0.f);
    }
}
__device__ __forceinline__ void transpose_tile(float *dstT, const float *src) {
    for (int e = threadIdx.x; e < kTN * 64; e += kBT) {
        const int m = e % kTN, c = e / kTN;
        dstT[c * kRS + m] = src[m * kRS + c];
    }
}

// Rows t0 .. t0 + mv - 1 of a [G][N][64] input (head base `src`) into a tile buffer; zeros below.
template <typename TI>
__device__ __forceinline__ void load_tile(float *dst, const TI *src, int t0, int mv) {
    const int lm = threadIdx.x >> 2, lj = (threadIdx.x & 3) * 16;
    Row16<TI> r;
    r.load(src + (size_t)(t0 + lm) * kD + lj, lm < mv);
    r.store(dst + lm * kRS + lj);
}

// Scores of the tile rows in xs into gs: s = c' + [x, x^2] . W (Eq. 16, expanded).
__device__ __forceinline__ void tile_scores(const float *W, const float *cp, const float *xs, float *gs, int r0,
                                            int c0) {
    float c[4][4];
    zero4x4(c);
    mm_rows<kD>(c, xs, kRS, r0, W, kK, c0);
#pragma unroll 4
    for (int s = 0; s < kD; ++s) {
        float x2[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float v = xs[(r0 + i) * kRS + s];
            x2[i] = v * v;
        }
        fma4x4(c, x2, ld4(W + (kD + s) * kK + c0));
    }
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) gs[(r0 + i) * kRS + c0 + j] = cp[c0 + j] + c[i][j];
}

// Eq. 3b over the rows of gs, a warp per row; rows >= mv get 0.  gT, if given, receives the
// transpose ([k][row], stride kRS).
__device__ __forceinline__ void tile_softmax(float *gs, float *gT, int mv) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int m = warp; m < kTN; m += kBT / 32) {
        const float s0 = gs[m * kRS + lane], s1 = gs[m * kRS + lane + 32];
        const float mx = bwd_warp_max(fmaxf(s0, s1));
        float e0 = expf(s0 - mx), e1 = expf(s1 - mx);
        const float inv = 1.0f / bwd_warp_sum(e0 + e1);
        const bool live = m < mv;
        e0 = live ? e0 * inv : 0.f;
        e1 = live ? e1 * inv : 0.f;
        gs[m * kRS + lane] = e0;
        gs[m * kRS + lane + 32] = e1;
        if (gT) {
            gT[lane * kRS + m] = e0;
            gT[(lane + 32) * kRS + m] = e1;
        }
    }
}

// Eq. 18 over the rows of gg (the upstream gradient g), in place: ds = gamma (g - gamma . g);
// the live rows also go to global memory (head base `out`, rows from t0).
__device__ __forceinline__ void tile_ds(const float *gam, float *gg, float *out, int t0, int mv) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int m = warp; m < kTN; m += kBT / 32) {
        const float g0 = gam[m * kRS + lane], g1 = gam[m * kRS + lane + 32];
        const float u0 = gg[m * kRS + lane], u1 = gg[m * kRS + lane + 32];
        const float mean = bwd_warp_sum(g0 * u0 + g1 * u1);
        const float d0 = g0 * (u0 - mean), d1 = g1 * (u1 - mean);
        gg[m * kRS + lane] = d0;
        gg[m * kRS + lane + 32] = d1;
        if (m < mv) {
            out[(size_t)(t0 + m) * kK + lane] = d0;
            out[(size_t)(t0 + m) * kK + lane + 32] = d1;
        }
    }
}

// Queries, tiles in order, carrying S and z (the prefix memory of Eq. 6b before the tile).
template <typename TI>
__global__ void __launch_bounds__(kBT, 1) bwd_cq_kernel(BwdCArgs a) {
    extern __shared__ __align__(16) float sm[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int r0 = (tid >> 4) * 4, c0 = (tid & 15) * 4;
    const int ch = blockIdx.x, g = blockIdx.y, h = g % a.H;
    float *W = sm + CC_W, *cp = sm + CC_CP, *M = sm + CC_M, *MT = sm + CC_MT, *zr = sm + CC_ZR;
    float *XS = sm + CC_T, *VS = XS + kTile, *VT = VS + kTile, *US = VT + kTile, *GQ = US + kTile;
    float *GK = GQ + kTile, *GKT = GK + kTile, *AS = GKT + kTile, *GG = AS + kTile;
    float *den = sm + CC_DEN, *bb = sm + CC_B;
    const size_t slot = (size_t)g * a.C + ch;
    causal_prologue(a, sm, h, a.mem + slot * kK * kW, true);
    const TI *Qx = static_cast<const TI *>(a.Qx) + (size_t)g * a.N * kD;
    const TI *V = static_cast<const TI *>(a.V) + (size_t)g * a.N * kDV;
    const TI *dO = static_cast<const TI *>(a.dO) + (size_t)g * a.N * kDV;
    const float *gkg = a.gk + (size_t)g * a.N * kK;
    float *gqg = a.gq + (size_t)g * a.N * kK;
    float *dsq = a.ds + (size_t)g * a.N * kK, *ab = a.ab + (size_t)g * a.N * kRS;
    float accM[4][4];
    zero4x4(accM);
    float ex_m = 0.f;
    __syncthreads();
    const int row_begin = ch * a.rows_per_chunk, row_end = min(a.N, row_begin + a.rows_per_chunk);
    for (int t0 = row_begin; t0 < row_end; t0 += kTN) {
        const int mv = min(kTN, row_end - t0);
        // the tile's keys: gamma^K (from the memory pass) and V, with their transposes; the
        // tile's queries and dO
        load_tile_f32(GK, gkg, t0, mv);
        load_tile(VS, V, t0, mv);
        load_tile(XS, Qx, t0, mv);
        load_tile(US, dO, t0, mv);
        __syncthreads();
        transpose_tile(VT, VS);
        transpose_tile(GKT, GK);
        tile_scores(W, cp, XS, GQ, r0, c0);
        __syncthreads();
        tile_softmax(GQ, nullptr, mv);
        __syncthreads();
        for (int m = warp; m < kTN; m += kBT / 32) {
            const float g0 = GQ[m * kRS + lane], g1 = GQ[m * kRS + lane + 32];
            const float z = bwd_warp_sum(g0 * zr[lane] + g1 * zr[lane + 32]);
            if (lane == 0) den[m] = z;
            if (m < mv) {                      // gamma^Q for the key pass
                gqg[(size_t)(t0 + m) * kK + lane] = g0;
                gqg[(size_t)(t0 + m) * kK + lane + 32] = g1;
            }
        }
        {   // A = tril(gamma^Q gamma^K^T): rows i (queries), columns j (keys)
            float c[4][4];
            zero4x4(c);
            mm_rows<kK>(c, GQ, kRS, r0, GKT, kRS, c0);
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) AS[(r0 + i) * kRS + c0 + j] = c0 + j <= r0 + i ? c[i][j] : 0.f;
        }
        __syncthreads();
        for (int m = warp; m < kTN; m += kBT / 32) {
            const float s = bwd_warp_sum(AS[m * kRS + lane] + AS[m * kRS + lane + 32]);
            if (lane == 0) den[m] = m < mv ? den[m] + s + a.eps : 1.f;   // rows past the end: a = b = 0
        }
        __syncthreads();
        {   // num = gamma^Q S + A V; O = num / den; a = dO / den, b = -(dO . O) / den
            float c[4][4];
            zero4x4(c);
            mm_rows<kK>(c, GQ, kRS, r0, M, kDV, c0);
            mm_rows<kTN>(c, AS, kRS, r0, VS, kRS, c0);
            float dot[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float dn = den[r0 + i];
                float p = 0.f;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    float *q = US + (r0 + i) * kRS + c0 + j;
                    p = fmaf(*q, c[i][j] / dn, p);
                    *q = *q / dn;
                }
                dot[i] = p;
            }
#pragma unroll
            for (int i = 0; i < 4; ++i)
                for (int o = 8; o; o >>= 1) dot[i] += __shfl_xor_sync(~0u, dot[i], o);
            if ((tid & 15) == 0)
#pragma unroll
                for (int i = 0; i < 4; ++i) bb[r0 + i] = -dot[i] / den[r0 + i];
        }
        __syncthreads();
        {   // Bm = tril(a V^T + b 1^T)
            float c[4][4];
            zero4x4(c);
            mm_rows<kDV>(c, US, kRS, r0, VT, kRS, c0);
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    AS[(r0 + i) * kRS + c0 + j] = c0 + j <= r0 + i ? c[i][j] + bb[r0 + i] : 0.f;
        }
        __syncthreads();
        {   // g^Q = a S^T + b z^T + Bm gamma^K
            float c[4][4];
            zero4x4(c);
            mm_rows<kDV>(c, US, kRS, r0, MT, kK, c0);
            mm_rows<kTN>(c, AS, kRS, r0, GK, kRS, c0);
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) GG[(r0 + i) * kRS + c0 + j] = fmaf(bb[r0 + i], zr[c0 + j], c[i][j]);
        }
        __syncthreads();
        tile_ds(GQ, GG, dsq, t0, mv);
        // a | b of the live rows for the key pass
        for (int e = tid; e < mv * kRS; e += kBT) {
            const int m = e / kRS, c = e - m * kRS;
            ab[(size_t)(t0 + m) * kRS + c] = c < kDV ? US[m * kRS + c] : (c == kDV ? bb[m] : 0.f);
        }
        // chunk totals of [R | r] = sum_i gamma^Q_i [a_i | b_i]
        mm_cols(accM, GQ, kRS, r0, US, kRS, c0);
        if (tid < kK)
            for (int m = 0; m < kTN; ++m) ex_m = fmaf(GQ[m * kRS + tid], bb[m], ex_m);
        {   // the prefix memory now includes the tile: S += gamma^K^T V, z += gamma^K^T 1
            float u[4][4];
            zero4x4(u);
            mm_cols(u, GK, kRS, r0, VS, kRS, c0);
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    M[(r0 + i) * kDV + c0 + j] += u[i][j];
                    MT[(c0 + j) * kK + r0 + i] += u[i][j];
                }
            if (tid >= kK && tid < 2 * kK) {
                float zs = 0.f;
                for (int m = 0; m < kTN; ++m) zs += GK[m * kRS + tid - kK];
                zr[tid - kK] += zs;
            }
        }
        __syncthreads();
    }
    float *pm = a.part_m + slot * kK * kW;
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) pm[(r0 + i) * kW + c0 + j] = accM[i][j];
    if (tid < kK) pm[tid * kW + kDV] = ex_m;
}

// Keys, tiles in reverse order, carrying R and r (the rows after the tile).
template <typename TI>
__global__ void __launch_bounds__(kBT, 1) bwd_ck_kernel(BwdCArgs a) {
    extern __shared__ __align__(16) float sm[];
    const int tid = threadIdx.x;
    const int r0 = (tid >> 4) * 4, c0 = (tid & 15) * 4;
    const int ch = blockIdx.x, g = blockIdx.y, h = g % a.H;
    float *M = sm + CC_M, *MT = sm + CC_MT, *zr = sm + CC_ZR;
    float *GQ = sm + CC_T + kTile, *GQT = GQ + kTile, *US = GQT + kTile, *AT = US + kTile;   // tile 0 unused
    float *GK = AT + kTile, *VS = GK + kTile, *CM = VS + kTile, *GG = CM + kTile;
    const size_t slot = (size_t)g * a.C + ch;
    causal_prologue(a, sm, h, a.mem + slot * kK * kW, false);
    const TI *V = static_cast<const TI *>(a.V) + (size_t)g * a.N * kDV;
    const float *gqg = a.gq + (size_t)g * a.N * kK, *gkg = a.gk + (size_t)g * a.N * kK;
    const float *ab = a.ab + (size_t)g * a.N * kRS;
    float *dsk = a.ds + (size_t)g * a.N * kK, *dV = a.dV + (size_t)g * a.N * kDV;
    __syncthreads();
    const int row_begin = ch * a.rows_per_chunk, row_end = min(a.N, row_begin + a.rows_per_chunk);
    const int ntiles = row_end > row_begin ? (row_end - row_begin + kTN - 1) / kTN : 0;
    for (int tt = ntiles - 1; tt >= 0; --tt) {
        const int t0 = row_begin + tt * kTN, mv = min(kTN, row_end - t0);
        // the tile's queries: gamma^Q and a | b (with transposes); its keys: gamma^K and V
        for (int e = tid; e < kTN * (kRS / 4); e += kBT) {
            const int m = e / (kRS / 4), q = e - m * (kRS / 4);
            reinterpret_cast<float4 *>(US + m * kRS)[q] =
                m < mv ? reinterpret_cast<const float4 *>(ab + (size_t)(t0 + m) * kRS)[q] : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        load_tile_f32(GQ, gqg, t0, mv);
        load_tile_f32(GK, gkg, t0, mv);
        load_tile(VS, V, t0, mv);
        __syncthreads();
        transpose_tile(AT, US);
        transpose_tile(GQT, GQ);
        __syncthreads();
        {   // Ct[j][i] = [i >= j] (v_j . a_i + b_i): rows j (keys), columns i (queries)
            float c[4][4];
            zero4x4(c);
            mm_rows<kDV>(c, VS, kRS, r0, AT, kRS, c0);
#pragma unroll
            for (int j = 0; j < 4; ++j)
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    CM[(r0 + j) * kRS + c0 + i] = c0 + i >= r0 + j ? c[j][i] + US[(c0 + i) * kRS + kDV] : 0.f;
        }
        __syncthreads();
        {   // g^K = Ct gamma^Q + V R^T + r
            float c[4][4];
            zero4x4(c);
            mm_rows<kTN>(c, CM, kRS, r0, GQ, kRS, c0);
            mm_rows<kDV>(c, VS, kRS, r0, MT, kK, c0);
#pragma unroll
            for (int j = 0; j < 4; ++j)
#pragma unroll
                for (int k = 0; k < 4; ++k) GG[(r0 + j) * kRS + c0 + k] = c[j][k] + zr[c0 + k];
        }
        __syncthreads();
        {   // Dt[j][i] = [i >= j] gamma^K_j . gamma^Q_i
            float c[4][4];
            zero4x4(c);
            mm_rows<kK>(c, GK, kRS, r0, GQT, kRS, c0);
#pragma unroll
            for (int j = 0; j < 4; ++j)
#pragma unroll
                for (int i = 0; i < 4; ++i) CM[(r0 + j) * kRS + c0 + i] = c0 + i >= r0 + j ? c[j][i] : 0.f;
        }
        __syncthreads();
        {   // dV = Dt a + gamma^K R
            float c[4][4];
            zero4x4(c);
            mm_rows<kTN>(c, CM, kRS, r0, US, kRS, c0);
            mm_rows<kK>(c, GK, kRS, r0, M, kDV, c0);
#pragma unroll
            for (int j = 0; j < 4; ++j)
                if (r0 + j < mv)
                    *reinterpret_cast<float4 *>(dV + (size_t)(t0 + r0 + j) * kDV + c0) =
                        make_float4(c[j][0], c[j][1], c[j][2], c[j][3]);
        }
        tile_ds(GK, GG, dsk, t0, mv);
        __syncthreads();
        {   // the memory of the rows after the next tile: R += gamma^Q^T a, r += gamma^Q^T b
            float u[4][4];
            zero4x4(u);
            mm_cols(u, GQ, kRS, r0, US, kRS, c0);
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    M[(r0 + i) * kDV + c0 + j] += u[i][j];
                    MT[(c0 + j) * kK + r0 + i] += u[i][j];
                }
            if (tid < kK) {
                float rs = 0.f;
                for (int m = 0; m < kTN; ++m) rs = fmaf(GQ[m * kRS + tid], US[m * kRS + kDV], rs);
                zr[tid] += rs;
            }
        }
        __syncthreads();
    }
}

// dX = -sum_k ds_k lambda_k (x - mu_k) (section 4.3) and the parameter sums P1 = sum ds x,
// P2 = sum ds x^2, P0 = sum ds of the rows of one side, from ds in global memory.
template <typename TI>
__global__ void __launch_bounds__(kBT, 1) bwd_rows_kernel(int N, int H, int C, int rows_per_chunk,
                                                          const void *Xv, const float *__restrict__ ds,
                                                          const float *__restrict__ mu,
                                                          const float *__restrict__ lam, float *__restrict__ dX,
                                                          float *__restrict__ part_p) {
    extern __shared__ __align__(16) float sm[];
    float *LAM = sm, *LMU = LAM + kK * kD, *XS = LMU + kK * kD, *DS = XS + kTile;
    const int tid = threadIdx.x;
    const int r0 = (tid >> 4) * 4, c0 = (tid & 15) * 4;
    const int ch = blockIdx.x, g = blockIdx.y, h = g % H;
    const float *lam_h = lam + (size_t)h * kK * kD, *mu_h = mu + (size_t)h * kK * kD;
    for (int e = tid; e < kK * kD; e += kBT) {
        const float l = lam_h[e];
        LAM[e] = l;
        LMU[e] = l * mu_h[e];
    }
    const TI *X = static_cast<const TI *>(Xv) + (size_t)g * N * kD;
    const float *dsg = ds + (size_t)g * N * kK;
    float *dXg = dX + (size_t)g * N * kD;
    float accP1[4][4], accP2[4][4];
    zero4x4(accP1);
    zero4x4(accP2);
    float ex_p = 0.f;
    __syncthreads();
    const int row_begin = ch * rows_per_chunk, row_end = min(N, row_begin + rows_per_chunk);
    for (int t0 = row_begin; t0 < row_end; t0 += kTN) {
        const int mv = min(kTN, row_end - t0);
        load_tile(XS, X, t0, mv);
        for (int e = tid; e < kTN * (kK / 4); e += kBT) {
            const int m = e / (kK / 4), q = e - m * (kK / 4);
            reinterpret_cast<float4 *>(DS + m * kRS)[q] =
                m < mv ? reinterpret_cast<const float4 *>(dsg + (size_t)(t0 + m) * kK)[q] : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        __syncthreads();
        float c1[4][4], c2[4][4];
        zero4x4(c1);
        zero4x4(c2);
#pragma unroll 4
        for (int s = 0; s < kK; ++s) {
            const float d4[4] = {DS[(r0 + 0) * kRS + s], DS[(r0 + 1) * kRS + s], DS[(r0 + 2) * kRS + s],
                                 DS[(r0 + 3) * kRS + s]};
            fma4x4(c1, d4, ld4(LAM + s * kD + c0));
            fma4x4(c2, d4, ld4(LMU + s * kD + c0));
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            if (r0 + i >= mv) continue;
            const float *x = XS + (r0 + i) * kRS + c0;
            *reinterpret_cast<float4 *>(dXg + (size_t)(t0 + r0 + i) * kD + c0) =
                make_float4(fmaf(-x[0], c1[i][0], c2[i][0]), fmaf(-x[1], c1[i][1], c2[i][1]),
                            fmaf(-x[2], c1[i][2], c2[i][2]), fmaf(-x[3], c1[i][3], c2[i][3]));
        }
#pragma unroll 4
        for (int m = 0; m < kTN; ++m) {
            const float4 d4 = ld4(DS + m * kRS + r0);
            const float dk[4] = {d4.x, d4.y, d4.z, d4.w};
            const float4 x4 = ld4(XS + m * kRS + c0);
            fma4x4(accP1, dk, x4);
            fma4x4(accP2, dk, make_float4(x4.x * x4.x, x4.y * x4.y, x4.z * x4.z, x4.w * x4.w));
        }
        if (tid >= kK && tid < 2 * kK)
            for (int m = 0; m < kTN; ++m) ex_p += DS[m * kRS + tid - kK];
        __syncthreads();
    }
    float *pp = part_p + ((size_t)g * C + ch) * kK * kPW;
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            pp[(r0 + i) * kPW + c0 + j] = accP1[i][j];
            pp[(r0 + i) * kPW + kD + c0 + j] = accP2[i][j];
        }
    if (tid >= kK && tid < 2 * kK) pp[(tid - kK) * kPW + 2 * kD] = ex_p;
}

// out[g][c] = sum of part[g][c'] over the chunks before c (reverse: after c), in chunk order.
__global__ void bwd_scan_kernel(int C, int E, int reverse, const float *__restrict__ part, float *__restrict__ out) {
    const int g = blockIdx.y, e = blockIdx.x * blockDim.x + threadIdx.x;
    if (e >= E) return;
    float run = 0.f;
    for (int i = 0; i < C; ++i) {
        const int c = reverse ? C - 1 - i : i;
        const size_t o = ((size_t)g * C + c) * E + e;
        out[o] = run;
        run += part[o];
    }
}

template <int MODE>
cudaError_t launch_pass(const Problem &p, const BwdLayout &L, const BwdArgs &a, cudaStream_t s) {
    auto kern = p.in_dtype == GMA_BF16 ? bwd_pass_kernel<MODE, __nv_bfloat16> : bwd_pass_kernel<MODE, float>;
    cudaError_t e = set_dyn_smem(reinterpret_cast<const void *>(kern), (int)kBwdSmemBytes);
    if (e != cudaSuccess) return e;
    kern<<<dim3(L.C, p.G), kBT, kBwdSmemBytes, s>>>(a);
    return cudaGetLastError();
}

template <template <typename> class KERN>
cudaError_t launch_causal(const Problem &p, const BwdLayout &L, const BwdCArgs &a, cudaStream_t s) {
    auto kern = p.in_dtype == GMA_BF16 ? KERN<__nv_bfloat16>::fn : KERN<float>::fn;
    cudaError_t e = set_dyn_smem(reinterpret_cast<const void *>(kern), (int)kCSmemBytes);
    if (e != cudaSuccess) return e;
    kern<<<dim3(L.C, p.G), kBT, kCSmemBytes, s>>>(a);
    return cudaGetLastError();
}
template <typename TI> struct CqKernel { static constexpr auto fn = bwd_cq_kernel<TI>; };
template <typename TI> struct CkKernel { static constexpr auto fn = bwd_ck_kernel<TI>; };

constexpr size_t kRowsSmemBytes = sizeof(float) * (2 * kK * kD + 2 * kTile);

cudaError_t launch_rows(const Problem &p, const BwdLayout &L, const void *X, const float *ds, const float *mu,
                        const float *lam, float *dX, float *part_p, cudaStream_t s) {
    auto kern = p.in_dtype == GMA_BF16 ? bwd_rows_kernel<__nv_bfloat16> : bwd_rows_kernel<float>;
    cudaError_t e = set_dyn_smem(reinterpret_cast<const void *>(kern), (int)kRowsSmemBytes);
    if (e != cudaSuccess) return e;
    kern<<<dim3(L.C, p.G), kBT, kRowsSmemBytes, s>>>(p.N, p.H, L.C, L.rows_per_chunk, X, ds, mu, lam, dX, part_p);
    return cudaGetLastError();
}

int device_sms() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return n;
}

}  // namespace

bool bwd_supported(const Problem &p) { return p.d == kD && p.K == kK && p.dv == kDV; }

BwdLayout bwd_layout(const Problem &p) {
    BwdLayout L{};
    // chunks per head: one CTA per SM (the shared memory of a pass CTA), so pick the chunk count
    // that minimises (waves of G C CTAs) / C, the smallest such count within 2 %
    const int sms = std::max(1, device_sms() > 0 ? device_sms() : 148);
    const int tiles = std::max(1, (p.N + kTN - 1) / kTN);
    const int cmax = std::min(tiles, 64);
    double best = 1e30;
    int bestC = 1;
    for (int c = 1; c <= cmax; ++c) {
        const double cost = (double)((p.G * c + sms - 1) / sms) / c;
        if (cost < best * 0.98) {
            best = cost;
            bestC = c;
        }
    }
    L.C = bestC;
    L.rows_per_chunk = ((tiles + L.C - 1) / L.C) * kTN;
    L.lam = align_up(kHeaderBytes);
    L.cdir = align_up(L.lam + sizeof(float) * (size_t)p.H * kK * kD);
    L.mem_s = align_up(L.cdir + sizeof(float) * (size_t)p.H * kK);
    L.mem_r = align_up(L.mem_s + sizeof(float) * (size_t)p.G * kK * kW);
    L.part_m = align_up(L.mem_r + sizeof(float) * (size_t)p.G * kK * kW);
    L.part_q = align_up(L.part_m + sizeof(float) * (size_t)p.G * L.C * kK * kW);
    L.part_k = align_up(L.part_q + sizeof(float) * (size_t)p.G * L.C * kK * kPW);
    L.gk = align_up(L.part_k + sizeof(float) * (size_t)p.G * L.C * kK * kPW);
    L.total = align_up(L.gk + sizeof(float) * (size_t)p.G * p.N * kK);
    if (p.causal) {     // per-chunk starting memories, a | b and ds of every row
        L.mem_pc = L.total;
        L.mem_rc = align_up(L.mem_pc + sizeof(float) * (size_t)p.G * L.C * kK * kW);
        L.ab = align_up(L.mem_rc + sizeof(float) * (size_t)p.G * L.C * kK * kW);
        L.dsq = align_up(L.ab + sizeof(float) * (size_t)p.G * p.N * kRS);
        L.dsk = align_up(L.dsq + sizeof(float) * (size_t)p.G * p.N * kK);
        L.gq = align_up(L.dsk + sizeof(float) * (size_t)p.G * p.N * kK);
        L.total = align_up(L.gq + sizeof(float) * (size_t)p.G * p.N * kK);
    }
    return L;
}

cudaError_t bwd_finalize(const Problem &p, int C, const float *pq, const float *pk, const float *mu, const float *lam,
                         const float *rho, const float *alpha, float *dmu, float *drho, float *dalpha, cudaStream_t s) {
    bwd_param_kernel<<<dim3(kK, p.H), 2 * kD, 0, s>>>(p.B, p.H, C, pq, pk, mu, lam, rho, alpha, dmu, drho, dalpha);
    return cudaGetLastError();
}

cudaError_t bwd_run(const Problem &p, const BwdLayout &L, const void *Qx, const void *Kx, const void *V,
                    const float *mu, const float *rho, const float *alpha, const void *dO, float *dQx, float *dKx,
                    float *dV, float *dmu, float *drho, float *dalpha, char *ws, cudaStream_t s) {
    float *lam = reinterpret_cast<float *>(ws + L.lam), *cdir = reinterpret_cast<float *>(ws + L.cdir);
    float *mem_s = reinterpret_cast<float *>(ws + L.mem_s), *mem_r = reinterpret_cast<float *>(ws + L.mem_r);
    float *part_m = reinterpret_cast<float *>(ws + L.part_m);
    float *part_q = reinterpret_cast<float *>(ws + L.part_q), *part_k = reinterpret_cast<float *>(ws + L.part_k);
    cudaError_t e = simt_params(p, rho, alpha, lam, cdir, s);
    if (e != cudaSuccess) return e;
    BwdArgs a{};
    a.N = p.N;
    a.H = p.H;
    a.C = L.C;
    a.rows_per_chunk = L.rows_per_chunk;
    a.eps = p.eps;
    a.mu = mu;
    a.lam = lam;
    a.cdir = cdir;
    a.gam = reinterpret_cast<float *>(ws + L.gk);
    const dim3 sum_grid((kK * kW + 255) / 256, p.G);
    if (p.causal) {
        float *mem_pc = reinterpret_cast<float *>(ws + L.mem_pc), *mem_rc = reinterpret_cast<float *>(ws + L.mem_rc);
        float *ab = reinterpret_cast<float *>(ws + L.ab);
        float *dsq = reinterpret_cast<float *>(ws + L.dsq), *dsk = reinterpret_cast<float *>(ws + L.dsk);
        // chunk totals of [S | z] (Eq. 6b), then each chunk's starting prefix
        a.X = Kx;
        a.U = V;
        a.part_m = part_m;
        if ((e = launch_pass<kMem>(p, L, a, s)) != cudaSuccess) return e;
        bwd_scan_kernel<<<sum_grid, 256, 0, s>>>(L.C, kK * kW, 0, part_m, mem_pc);
        BwdCArgs c{};
        c.N = p.N;
        c.H = p.H;
        c.C = L.C;
        c.rows_per_chunk = L.rows_per_chunk;
        c.eps = p.eps;
        c.Qx = Qx;
        c.Kx = Kx;
        c.V = V;
        c.dO = dO;
        c.mu = mu;
        c.lam = lam;
        c.cdir = cdir;
        c.ab = ab;
        c.gk = a.gam;
        c.gq = reinterpret_cast<float *>(ws + L.gq);
        // queries in order: ds^Q, a | b, chunk totals of [R | r]
        c.mem = mem_pc;
        c.ds = dsq;
        c.part_m = part_m;
        if ((e = launch_causal<CqKernel>(p, L, c, s)) != cudaSuccess) return e;
        bwd_scan_kernel<<<sum_grid, 256, 0, s>>>(L.C, kK * kW, 1, part_m, mem_rc);
        // keys in reverse: ds^K, dV
        c.mem = mem_rc;
        c.ds = dsk;
        c.dV = dV;
        if ((e = launch_causal<CkKernel>(p, L, c, s)) != cudaSuccess) return e;
        if ((e = launch_rows(p, L, Qx, dsq, mu, lam, dQx, part_q, s)) != cudaSuccess) return e;
        if ((e = launch_rows(p, L, Kx, dsk, mu, lam, dKx, part_k, s)) != cudaSuccess) return e;
        bwd_param_kernel<<<dim3(kK, p.H), 2 * kD, 0, s>>>(p.B, p.H, L.C, part_q, part_k, mu, lam, rho, alpha, dmu,
                                                        drho, dalpha);
        return cudaGetLastError();
    }
    // the forward memory [Vt | Z] (Eq. 5-6)
    a.X = Kx;
    a.U = V;
    a.part_m = part_m;
    if ((e = launch_pass<kMem>(p, L, a, s)) != cudaSuccess) return e;
    bwd_sum_kernel<<<sum_grid, 256, 0, s>>>(L.C, kK * kW, part_m, mem_s);
    // the query rows: dQx, [R | r], parameter sums
    a.X = Qx;
    a.U = dO;
    a.mem = mem_s;
    a.dX = dQx;
    a.part_p = part_q;
    if ((e = launch_pass<kQry>(p, L, a, s)) != cudaSuccess) return e;
    bwd_sum_kernel<<<sum_grid, 256, 0, s>>>(L.C, kK * kW, part_m, mem_r);
    // the key rows: dKx, dV, parameter sums
    a.X = Kx;
    a.U = V;
    a.mem = mem_r;
    a.dX = dKx;
    a.dV = dV;
    a.part_p = part_k;
    if ((e = launch_pass<kKey>(p, L, a, s)) != cudaSuccess) return e;
    bwd_param_kernel<<<dim3(kK, p.H), 2 * kD, 0, s>>>(p.B, p.H, L.C, part_q, part_k, mu, lam, rho, alpha, dmu, drho,
                                                    dalpha);
    return cudaGetLastError();
}

}  // namespace gma
