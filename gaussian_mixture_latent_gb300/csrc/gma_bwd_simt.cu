// Backward pass of GMA for every shape the CUDA-core forward takes (d, K, dv up to 256,
// float32 or bf16 inputs), bidirectional and causal, on the CUDA cores in fp32.  The
// tensor-core backward (gma_bwd_tc.cu) and the specialised CUDA-core kernels of
// gma_bwd.cu cover d = dv = K = 64; this file covers the rest.
//
// "Gaussian Mixture Attention" (Huang & Raza, 2026), section 4.1: the softmax Jacobian
// ds_ik = gamma_ik (g_ik - sum_l gamma_il g_il) (Eq. 17-18), the chain rule through the
// score of Eq. 16 (Eq. 19; d s / d mu of Eq. 20, d s / d x of section 4.3) and Eq. 14-15
// for rho and alpha.  The memory products of Eq. 5-8 (causal: the prefix memories of
// Eq. 6b, 8b) are differentiated as products: with den_i = gamma^Q_i . Z + eps,
// a_i = dO_i / den_i and b_i = -(dO_i . O_i) / den_i,
//   g^Q_ik = sum_v a_iv Vt_kv + b_i Z_k,        [R | r]_k = sum_i gamma^Q_ik [a_i | b_i],
//   g^K_jk = sum_v V_jv R_kv + r_k,             dV_j = sum_k gamma^K_jk R_k,
//   dx_im  = sum_k ds_ik lambda_km mu_km - x_im sum_k ds_ik lambda_km,
// and the parameter sums P1 = sum_i ds x, P2 = sum_i ds x^2, P0 = sum_i ds over every row
// of both sides, from which dmu, drho and dalpha follow.  In the causal form row i reads
// the memory of rows j <= i and key row j receives from query rows i >= j: the rows are
// split into P ranges with an exclusive prefix of the memory (queries) and an exclusive
// suffix of [R | r] (keys) per range, and inside a range one CTA walks chunks of C rows
// (queries forwards, keys backwards) with the masked intra-chunk products and its
// running state in shared memory.
//
// Kernels (all fp32 arithmetic, every reduction in a fixed order, so results are
// deterministic): gb_rowmat (row-times-matrix tiles of 64 x 64 or 64 x 80), gb_outer (per-range sums of
// outer products), gb_reduce (sum / exclusive prefix / exclusive suffix over ranges),
// gb_ab, gb_ds, gb_dx (per-row steps), gb_cq / gb_ck (the causal chunk walks),
// gb_param (dmu, drho, dalpha).  The responsibilities come from the forward's CUDA-core
// kernels (simt_params, simt_gamma).
#include <cuda_bf16.h>

#include <algorithm>
#include <cfloat>
#include <cstdint>

#include "gma_internal.h"

namespace gma {
namespace {

constexpr int kGbThreads = 256;
constexpr int kWalkThreads = 512;      // the causal walks: one CTA per SM (shared memory), 16 warps
constexpr int kGbChunkDefault = 16;

template <typename T>
__device__ __forceinline__ float gld(const T *p, size_t i);
template <>
__device__ __forceinline__ float gld<float>(const float *p, size_t i) { return p[i]; }
template <>
__device__ __forceinline__ float gld<__nv_bfloat16>(const __nv_bfloat16 *p, size_t i) {
    return __bfloat162float(p[i]);
}

// out[(g N + i) ldo + c] = sum_k A(g, i, k) B(k, c), c < C, for the N rows of head-row g:
//   A(g, i, k) = A[(g N + i) lda + k] for k < a_cols, 1 at k == a_cols when a_one, else 0;
//   B(k, c)    = MT ? M[mo + c ldm + k] : M[mo + k ldm + c],  k < KA,
//   mo = (m_per_head ? g % H : g) m_stride.
// 64-row x 16 JN-column output tile per CTA, 256 threads, each four rows (ty + 16 q) by JN
// columns (tx + 16 j); k in steps of 32 through shared memory, in increasing order per
// output (the last step only over the k that exist).  JN = 5 serves widths such as dv + 1
// and 2 d + 1 in fewer tiles than 64-column ones would.
constexpr int kRmTile = 64;

template <typename TA, bool MT, int JN>
__global__ void __launch_bounds__(kGbThreads) gb_rowmat_kernel(int N, int KA, int C, int H, int lda, int a_cols,
                                                               int a_one, const TA *__restrict__ A,
                                                               const float *__restrict__ M, int m_per_head,
                                                               size_t m_stride, int ldm, float *__restrict__ out,
                                                               int ldo) {
    constexpr int CW = 16 * JN;
    __shared__ float as[kRmTile][33];
    __shared__ float bs[32][CW + 1];
    const int i0 = blockIdx.x * kRmTile, c0 = blockIdx.y * CW, g = blockIdx.z;
    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
    const float *Mg = M + (size_t)(m_per_head ? g % H : g) * m_stride;
    float acc[4][JN] = {};
    for (int k0 = 0; k0 < KA; k0 += 32) {
        for (int e = threadIdx.x; e < kRmTile * 32; e += kGbThreads) {
            const int r = e >> 5, cc = e & 31;
            const int i = i0 + r, k = k0 + cc;
            float av = 0.f;
            if (i < N) {
                if (k < a_cols) av = gld(A, ((size_t)g * N + i) * lda + k);
                else if (a_one && k == a_cols) av = 1.f;
            }
            as[r][cc] = av;
        }
        for (int e = threadIdx.x; e < CW * 32; e += kGbThreads) {
            if (MT) {          // element (k0 + cc, c0 + r): a warp reads consecutive k of one row of M
                const int r = e >> 5, cc = e & 31;
                const int kk = k0 + cc, c = c0 + r;
                bs[cc][r] = (kk < KA && c < C) ? Mg[(size_t)c * ldm + kk] : 0.f;
            } else {           // element (k0 + e / CW, c0 + e % CW)
                const int kr = e / CW, cc = e - kr * CW;
                const int kk = k0 + kr, c = c0 + cc;
                bs[kr][cc] = (kk < KA && c < C) ? Mg[(size_t)kk * ldm + c] : 0.f;
            }
        }
        __syncthreads();
        auto step = [&](int kk) {
            float a[4], b[JN];
#pragma unroll
            for (int q = 0; q < 4; ++q) a[q] = as[ty + 16 * q][kk];
#pragma unroll
            for (int j = 0; j < JN; ++j) b[j] = bs[kk][tx + 16 * j];
#pragma unroll
            for (int q = 0; q < 4; ++q)
#pragma unroll
                for (int j = 0; j < JN; ++j) acc[q][j] = fmaf(a[q], b[j], acc[q][j]);
        };
        if (KA - k0 >= 32) {
#pragma unroll 4
            for (int kk = 0; kk < 32; ++kk) step(kk);
        } else {
            for (int kk = 0; kk < KA - k0; ++kk) step(kk);
        }
        __syncthreads();
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const int i = i0 + ty + 16 * q;
        if (i >= N) continue;
#pragma unroll
        for (int j = 0; j < JN; ++j) {
            const int c = c0 + tx + 16 * j;
            if (c < C) out[((size_t)g * N + i) * ldo + c] = acc[q][j];
        }
    }
}

// The column operands of gb_outer: U(row, c) for c < width.
template <typename T>
struct UValsOne {              // [V | 1]
    const T *V;
    int dv;
    __device__ float operator()(size_t row, int c) const {
        return c < dv ? gld(V, row * dv + c) : (c == dv ? 1.f : 0.f);
    }
};
struct UPlain {                // a stored fp32 [rows][w] array ([a | b])
    const float *U;
    int w;
    __device__ float operator()(size_t row, int c) const { return c < w ? U[row * w + c] : 0.f; }
};
template <typename T>
struct USquares {              // [x | x^2 | 1]
    const T *X;
    int d;
    __device__ float operator()(size_t row, int c) const {
        if (c < d) return gld(X, row * d + c);
        if (c < 2 * d) {
            const float x = gld(X, row * d + c - d);
            return x * x;
        }
        return c == 2 * d ? 1.f : 0.f;
    }
};

// part[((g P + p) K + k) W + c] = sum over rows i of range p of A[(g N + i) K + k] U(g N + i, c),
// k < K, c < W; range p = rows [p rpp, min(N, (p + 1) rpp)).  64-component x 16 JN-column
// output tile per CTA, each thread four components (ty + 16 q) by JN columns (tx + 16 j),
// rows in increasing order through shared memory 32 at a time (the last block only over
// the rows that exist).
template <typename U, int JN>
__global__ void __launch_bounds__(kGbThreads) gb_outer_kernel(int N, int K, int W, int P, int rpp,
                                                              const float *__restrict__ A, U u,
                                                              float *__restrict__ part) {
    constexpr int CW = 16 * JN;
    __shared__ float as[32][kRmTile + 1];
    __shared__ float us[32][CW + 1];
    const int ktiles = (K + kRmTile - 1) / kRmTile;
    const int kt = blockIdx.x % ktiles, ct = blockIdx.x / ktiles;
    const int p = blockIdx.y, g = blockIdx.z;
    const int r0 = p * rpp, r1 = min(N, r0 + rpp);
    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
    const int k0 = kt * kRmTile, c0 = ct * CW;
    float acc[4][JN] = {};
    for (int j0 = r0; j0 < r1; j0 += 32) {
        for (int e = threadIdx.x; e < 32 * kRmTile; e += kGbThreads) {
            const int jr = e >> 6, cc = e & 63;
            const int j = j0 + jr, k = k0 + cc;
            as[jr][cc] = (j < r1 && k < K) ? A[((size_t)g * N + j) * K + k] : 0.f;
        }
        for (int e = threadIdx.x; e < 32 * CW; e += kGbThreads) {
            const int jr = e / CW, cc = e - jr * CW;
            const int j = j0 + jr, c = c0 + cc;
            us[jr][cc] = (j < r1 && c < W) ? u((size_t)g * N + j, c) : 0.f;
        }
        __syncthreads();
        auto step = [&](int jr) {
            float a[4], v[JN];
#pragma unroll
            for (int q = 0; q < 4; ++q) a[q] = as[jr][ty + 16 * q];
#pragma unroll
            for (int jj = 0; jj < JN; ++jj) v[jj] = us[jr][tx + 16 * jj];
#pragma unroll
            for (int q = 0; q < 4; ++q)
#pragma unroll
                for (int jj = 0; jj < JN; ++jj) acc[q][jj] = fmaf(a[q], v[jj], acc[q][jj]);
        };
        if (r1 - j0 >= 32) {
#pragma unroll 4
            for (int jr = 0; jr < 32; ++jr) step(jr);
        } else {
            for (int jr = 0; jr < r1 - j0; ++jr) step(jr);
        }
        __syncthreads();
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const int k = k0 + ty + 16 * q;
        if (k >= K) continue;
#pragma unroll
        for (int jj = 0; jj < JN; ++jj) {
            const int c = c0 + tx + 16 * jj;
            if (c < W) part[(((size_t)g * P + p) * K + k) * W + c] = acc[q][jj];
        }
    }
}

// Over the P ranges of head-row g, element e < E:  mode 0: out[g][e] = sum_p part[g][p][e];
// mode 1: out[g][p][e] = sum_{q < p} part[g][q][e];  mode 2: out[g][p][e] = sum_{q > p} part[g][q][e].
__global__ void gb_reduce_kernel(int G, int P, int E, int mode, const float *__restrict__ part,
                                 float *__restrict__ out) {
    const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (size_t)G * E) return;
    const size_t g = i / E, e = i % E;
    float acc = 0.f;
    if (mode == 2) {
        for (int p = P - 1; p >= 0; --p) {
            out[(g * P + p) * E + e] = acc;
            acc += part[(g * P + p) * E + e];
        }
        return;
    }
    for (int p = 0; p < P; ++p) {
        const float v = part[(g * P + p) * E + e];
        if (mode == 1) out[(g * P + p) * E + e] = acc;
        acc += v;
    }
    if (mode == 0) out[g * E + e] = acc;
}

__device__ __forceinline__ float gb_warp_sum(float v) {
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) v += __shfl_xor_sync(~0u, v, o);
    return v;
}

// One warp per row: t = [num | den - eps] (W = dv + 1 columns), dO -> ab = [dO / den | -(dO . O) / den].
template <typename T>
__global__ void gb_ab_kernel(size_t rows, int dv, float eps, const float *__restrict__ t, const T *__restrict__ dO,
                             float *__restrict__ ab) {
    const size_t row = (size_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= rows) return;
    const int W = dv + 1;
    const float den = t[row * W + dv] + eps;
    const float inv = 1.f / den;
    float dot = 0.f;
    for (int v = lane; v < dv; v += 32) {
        const float o = t[row * W + v] * inv, d = gld(dO, row * dv + v);
        dot = fmaf(d, o, dot);
        ab[row * W + v] = d * inv;
    }
    dot = gb_warp_sum(dot);
    if (lane == 0) ab[row * W + dv] = -dot * inv;
}

// One warp per row: g <- gamma (g - sum_k gamma_k g_k), in place (Eq. 17-18).
__global__ void gb_ds_kernel(size_t rows, int K, const float *__restrict__ gam, float *__restrict__ g) {
    const size_t row = (size_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= rows) return;
    float s = 0.f;
    for (int k = lane; k < K; k += 32) s = fmaf(gam[row * K + k], g[row * K + k], s);
    s = gb_warp_sum(s);
    for (int k = lane; k < K; k += 32) g[row * K + k] = gam[row * K + k] * (g[row * K + k] - s);
}

// dX[row][m] = t[row][m] - x[row][m] t[row][d + m], t = ds [lambda mu | lambda].
template <typename T>
__global__ void gb_dx_kernel(size_t rows, int d, const float *__restrict__ t, const T *__restrict__ X,
                             float *__restrict__ dX) {
    const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= rows * d) return;
    const size_t row = i / d;
    const int m = (int)(i % d);
    dX[i] = fmaf(-gld(X, i), t[row * 2 * d + d + m], t[row * 2 * d + m]);
}

// lmu[h][k] = [lambda_k mu_k | lambda_k] (2 d columns).
__global__ void gb_lmu_kernel(int H, int K, int d, const float *__restrict__ mu, const float *__restrict__ lam,
                              float *__restrict__ lmu) {
    const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (size_t)H * K * d) return;
    const size_t hk = i / d;
    const int m = (int)(i % d);
    const float l = lam[i];
    lmu[hk * 2 * d + m] = l * mu[i];
    lmu[hk * 2 * d + d + m] = l;
}

// Parameter gradients of head h, component k (CTA (k, h)): P1, P2 [d] and P0 summed over
// both sides, the batch and the ranges in a fixed order, then
//   dmu = lambda (P1 - mu P0),  dvar = lambda/2 (lambda (P2 - 2 mu P1 + mu^2 P0) - P0),
//   drho = dvar sigmoid(rho),   dalpha_k = P0_k - pi_k sum_l P0_l.
// Partials: [G][P][K][2 d + 1] per side, G = B H, head-row g = b H + h.
__global__ void __launch_bounds__(kGbThreads) gb_param_kernel(int B, int H, int P, int K, int d,
                                                              const float *__restrict__ pq,
                                                              const float *__restrict__ pk,
                                                              const float *__restrict__ mu,
                                                              const float *__restrict__ lam,
                                                              const float *__restrict__ rho,
                                                              const float *__restrict__ alpha,
                                                              float *__restrict__ dmu, float *__restrict__ drho,
                                                              float *__restrict__ dalpha) {
    __shared__ float red[kGbThreads / 32];
    __shared__ float tot_s;
    const int k = blockIdx.x, h = blockIdx.y, t = threadIdx.x;
    const int E = 2 * d + 1;
    auto psum = [&](int kk, int q) {
        float s = 0.f;
        for (int side = 0; side < 2; ++side) {
            const float *part = side ? pk : pq;
            for (int b = 0; b < B; ++b)
                for (int p = 0; p < P; ++p) s += part[((((size_t)(b * H + h) * P + p) * K + kk) * E) + q];
        }
        return s;
    };
    // sum over l of P0_l, in l order per thread, then across threads in a fixed order
    float tp = 0.f;
    for (int l = t; l < K; l += kGbThreads) tp += psum(l, 2 * d);
    tp = gb_warp_sum(tp);
    if ((t & 31) == 0) red[t >> 5] = tp;
    __syncthreads();
    if (t == 0) {
        float s = 0.f;
        for (int w = 0; w < kGbThreads / 32; ++w) s += red[w];
        tot_s = s;
    }
    __syncthreads();
    const float P0 = psum(k, 2 * d);
    for (int m = t; m < d; m += kGbThreads) {
        const size_t o = ((size_t)h * K + k) * d + m;
        const float P1 = psum(k, m), P2 = psum(k, d + m);
        const float mm = mu[o], l = lam[o];
        dmu[o] = l * fmaf(-mm, P0, P1);
        const float q2 = fmaf(mm, fmaf(mm, P0, -2.f * P1), P2);
        drho[o] = 0.5f * l * fmaf(l, q2, -P0) / (1.f + expf(-rho[o]));
    }
    if (t == 0) {
        const float *al = alpha + (size_t)h * K;
        float mx = -FLT_MAX, se = 0.f;
        for (int l = 0; l < K; ++l) mx = fmaxf(mx, al[l]);
        for (int l = 0; l < K; ++l) se += expf(al[l] - mx);
        const float lse = mx + logf(se);
        dalpha[(size_t)h * K + k] = fmaf(-expf(al[k] - lse), tot_s, P0);
    }
}

// ---------------------------------------------------------------------------------------
// Causal chunk walks.  Shared memory (floats), C rows per chunk, W = dv + 1:
//   state [K][W], gA [C][K], gB [C][K], gg [C][K], va [C][W], ab [C][W], dO [C][dv],
//   Am [C][C], Bm [C][C].
struct GbCausalArgs {
    int N, K, dv, P, rpp, C;
    float eps;
    const float *gq, *gk;        // responsibilities [G][N][K]
    const void *V, *dO;          // [G][N][dv], input dtype
    const float *mem;            // queries: exclusive prefix of the memory per range [G][P][K][W];
                                 // keys: exclusive suffix of [R | r] per range
    float *ab;                   // [G][N][W]: written by the query walk, read by the key walk
    float *ds;                   // [G][N][K]: ds^Q (queries) or ds^K (keys)
    float *dV;                   // keys: [G][N][dv]
};

size_t gb_causal_floats(int K, int dv, int C) {
    const size_t W = (size_t)dv + 1;
    return (size_t)K * W + 3 * (size_t)C * K + 2 * (size_t)C * W + (size_t)C * dv + 2 * (size_t)C * C;
}

// Query walk of range p of head-row g (chunks in order), with the prefix state S (the
// memory of the rows before the chunk):
//   Am_ij = [j <= i] gamma^Q_i . gamma^K_j,   [num | den - eps]_i = gamma^Q_i S + sum_j Am_ij [V_j | 1],
//   ab_i = [dO_i / den_i | -(dO_i . O_i) / den_i],
//   Bm_ij = [j <= i] ab_i . [V_j | 1],         g^Q_i = S ab_i + sum_j Bm_ij gamma^K_j,
//   ds^Q_i = gamma^Q_i (g^Q_i - gamma^Q_i . g^Q_i),   S += sum_j gamma^K_j^T [V_j | 1].
template <typename T>
__global__ void __launch_bounds__(kWalkThreads) gb_cq_kernel(GbCausalArgs a) {
    extern __shared__ float sm[];
    const int K = a.K, dv = a.dv, W = dv + 1, C = a.C, N = a.N;
    const int p = blockIdx.x, g = blockIdx.y, t = threadIdx.x, lane = t & 31, warp = t >> 5;
    const int RG = (C + 3) / 4, KG = (K + 3) / 4;       // groups of four rows, of four components
    float *S = sm, *gA = S + (size_t)K * W, *gB = gA + C * K, *gg = gB + C * K, *va = gg + C * K;
    float *ab = va + C * W, *dO = ab + C * W, *Am = dO + C * dv, *Bm = Am + C * C;
    const T *V = static_cast<const T *>(a.V), *DO = static_cast<const T *>(a.dO);
    const float *m0 = a.mem + ((size_t)g * a.P + p) * K * W;
    for (int e = t; e < K * W; e += kWalkThreads) S[e] = m0[e];
    const int r0 = p * a.rpp, r1 = min(N, r0 + a.rpp);
    for (int i0 = r0; i0 < r1; i0 += C) {
        const int n = min(C, r1 - i0);
        const size_t row0 = (size_t)g * N + i0;
        __syncthreads();                                   // the previous chunk is done with the buffers
        for (int e = t; e < C * K; e += kWalkThreads) {
            const int r = e / K;
            gA[e] = r < n ? a.gq[row0 * K + e] : 0.f;
            gB[e] = r < n ? a.gk[row0 * K + e] : 0.f;
        }
        for (int e = t; e < C * W; e += kWalkThreads) {
            const int r = e / W, c = e % W;
            va[e] = r < n ? (c < dv ? gld(V, (row0 + r) * dv + c) : 1.f) : 0.f;
        }
        for (int e = t; e < C * dv; e += kWalkThreads) dO[e] = e / dv < n ? gld(DO, row0 * dv + e) : 0.f;
        __syncthreads();
        for (int e = t; e < C * C; e += kWalkThreads) {
            const int i = e / C, j = e % C;
            float s = 0.f;
            if (j <= i)
                for (int k = 0; k < K; ++k) s = fmaf(gA[i * K + k], gB[j * K + k], s);
            Am[e] = s;
        }
        __syncthreads();
        for (int e = t; e < RG * W; e += kWalkThreads) {     // [num | den - eps] into ab, four rows a thread
            const int c = e % W, i0q = (e / W) * 4;
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
            for (int k = 0; k < K; ++k) {
                const float sv = S[k * W + c];
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    if (i0q + q < C) acc[q] = fmaf(gA[(i0q + q) * K + k], sv, acc[q]);
            }
            for (int j = 0; j < C; ++j) {
                const float v = va[j * W + c];
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    if (j <= i0q + q && i0q + q < C) acc[q] = fmaf(Am[(i0q + q) * C + j], v, acc[q]);
            }
#pragma unroll
            for (int q = 0; q < 4; ++q)
                if (i0q + q < C) ab[(i0q + q) * W + c] = acc[q];
        }
        __syncthreads();
        for (int i = warp; i < n; i += kWalkThreads / 32) {  // a and b, one warp per row
            const float inv = 1.f / (ab[i * W + dv] + a.eps);
            float dot = 0.f;
            for (int v = lane; v < dv; v += 32) dot = fmaf(dO[i * dv + v], ab[i * W + v] * inv, dot);
            dot = gb_warp_sum(dot);
            __syncwarp();
            for (int v = lane; v < dv; v += 32) ab[i * W + v] = dO[i * dv + v] * inv;
            if (lane == 0) ab[i * W + dv] = -dot * inv;
        }
        __syncthreads();
        for (int e = t; e < n * W; e += kWalkThreads) a.ab[row0 * W + e] = ab[e];
        for (int e = t; e < C * C; e += kWalkThreads) {
            const int i = e / C, j = e % C;
            float s = 0.f;
            if (j <= i && i < n)
                for (int c = 0; c < W; ++c) s = fmaf(ab[i * W + c], va[j * W + c], s);
            Bm[e] = s;
        }
        __syncthreads();
        for (int e = t; e < RG * K; e += kWalkThreads) {     // g^Q, four rows a thread
            const int k = e % K, i0q = (e / K) * 4;
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
            for (int c = 0; c < W; ++c) {
                const float sv = S[k * W + c];
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    if (i0q + q < C) acc[q] = fmaf(ab[(i0q + q) * W + c], sv, acc[q]);
            }
            for (int j = 0; j < C; ++j) {
                const float gb = gB[j * K + k];
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    if (j <= i0q + q && i0q + q < C) acc[q] = fmaf(Bm[(i0q + q) * C + j], gb, acc[q]);
            }
#pragma unroll
            for (int q = 0; q < 4; ++q)
                if (i0q + q < C) gg[(i0q + q) * K + k] = acc[q];
        }
        __syncthreads();
        for (int i = warp; i < n; i += kWalkThreads / 32) {  // ds^Q, one warp per row
            float s = 0.f;
            for (int k = lane; k < K; k += 32) s = fmaf(gA[i * K + k], gg[i * K + k], s);
            s = gb_warp_sum(s);
            for (int k = lane; k < K; k += 32) a.ds[(row0 + i) * K + k] = gA[i * K + k] * (gg[i * K + k] - s);
        }
        for (int e = t; e < KG * W; e += kWalkThreads) {     // the state after this chunk, four components a thread
            const int c = e % W, k0q = (e / W) * 4;
            float acc[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) acc[q] = k0q + q < K ? S[(k0q + q) * W + c] : 0.f;
            for (int j = 0; j < n; ++j) {
                const float v = va[j * W + c];
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    if (k0q + q < K) acc[q] = fmaf(gB[j * K + k0q + q], v, acc[q]);
            }
#pragma unroll
            for (int q = 0; q < 4; ++q)
                if (k0q + q < K) S[(k0q + q) * W + c] = acc[q];
        }
    }
}

// Key walk of range p of head-row g (chunks in reverse), with the suffix state Rs ([R | r]
// of the query rows after the chunk):
//   Am_ij = [j <= i] gamma^Q_i . gamma^K_j,   Bm_ij = [j <= i] ab_i . [V_j | 1],
//   g^K_j = Rs [V_j | 1] + sum_i Bm_ij gamma^Q_i,   dV_j = gamma^K_j Rs_V + sum_i Am_ij a_i,
//   ds^K_j = gamma^K_j (g^K_j - gamma^K_j . g^K_j),  Rs += sum_i gamma^Q_i^T ab_i.
template <typename T>
__global__ void __launch_bounds__(kWalkThreads) gb_ck_kernel(GbCausalArgs a) {
    extern __shared__ float sm[];
    const int K = a.K, dv = a.dv, W = dv + 1, C = a.C, N = a.N;
    const int p = blockIdx.x, g = blockIdx.y, t = threadIdx.x, lane = t & 31, warp = t >> 5;
    const int RG = (C + 3) / 4, KG = (K + 3) / 4;       // groups of four rows, of four components
    float *Rs = sm, *gQ = Rs + (size_t)K * W, *gK = gQ + C * K, *gg = gK + C * K, *va = gg + C * K;
    float *ab = va + C * W, *Am = ab + C * W + C * dv, *Bm = Am + C * C;
    const T *V = static_cast<const T *>(a.V);
    const float *m0 = a.mem + ((size_t)g * a.P + p) * K * W;
    for (int e = t; e < K * W; e += kWalkThreads) Rs[e] = m0[e];
    const int r0 = p * a.rpp, r1 = min(N, r0 + a.rpp);
    if (r1 <= r0) return;
    const int nch = (r1 - r0 + C - 1) / C;
    for (int ci = nch - 1; ci >= 0; --ci) {
        const int i0 = r0 + ci * C, n = min(C, r1 - i0);
        const size_t row0 = (size_t)g * N + i0;
        __syncthreads();
        for (int e = t; e < C * K; e += kWalkThreads) {
            const int r = e / K;
            gQ[e] = r < n ? a.gq[row0 * K + e] : 0.f;
            gK[e] = r < n ? a.gk[row0 * K + e] : 0.f;
        }
        for (int e = t; e < C * W; e += kWalkThreads) {
            const int r = e / W, c = e % W;
            va[e] = r < n ? (c < dv ? gld(V, (row0 + r) * dv + c) : 1.f) : 0.f;
            ab[e] = r < n ? a.ab[row0 * W + e] : 0.f;
        }
        __syncthreads();
        for (int e = t; e < C * C; e += kWalkThreads) {
            const int i = e / C, j = e % C;
            float sa = 0.f, sb = 0.f;
            if (j <= i) {
                for (int k = 0; k < K; ++k) sa = fmaf(gQ[i * K + k], gK[j * K + k], sa);
                for (int c = 0; c < W; ++c) sb = fmaf(ab[i * W + c], va[j * W + c], sb);
            }
            Am[e] = sa;
            Bm[e] = sb;
        }
        __syncthreads();
        for (int e = t; e < RG * K; e += kWalkThreads) {     // g^K, four rows a thread
            const int k = e % K, j0q = (e / K) * 4;
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
            for (int c = 0; c < W; ++c) {
                const float rv = Rs[k * W + c];
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    if (j0q + q < C) acc[q] = fmaf(va[(j0q + q) * W + c], rv, acc[q]);
            }
            for (int i = 0; i < C; ++i) {
                const float gv = gQ[i * K + k];
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    if (i >= j0q + q && j0q + q < C) acc[q] = fmaf(Bm[i * C + j0q + q], gv, acc[q]);
            }
#pragma unroll
            for (int q = 0; q < 4; ++q)
                if (j0q + q < C) gg[(j0q + q) * K + k] = acc[q];
        }
        for (int e = t; e < RG * dv; e += kWalkThreads) {    // dV, four rows a thread
            const int v = e % dv, j0q = (e / dv) * 4;
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
            for (int k = 0; k < K; ++k) {
                const float rv = Rs[k * W + v];
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    if (j0q + q < C) acc[q] = fmaf(gK[(j0q + q) * K + k], rv, acc[q]);
            }
            for (int i = 0; i < C; ++i) {
                const float av = ab[i * W + v];
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    if (i >= j0q + q && j0q + q < C) acc[q] = fmaf(Am[i * C + j0q + q], av, acc[q]);
            }
#pragma unroll
            for (int q = 0; q < 4; ++q)
                if (j0q + q < n) a.dV[(row0 + j0q + q) * dv + v] = acc[q];
        }
        __syncthreads();
        for (int j = warp; j < n; j += kWalkThreads / 32) {  // ds^K, one warp per row
            float s = 0.f;
            for (int k = lane; k < K; k += 32) s = fmaf(gK[j * K + k], gg[j * K + k], s);
            s = gb_warp_sum(s);
            for (int k = lane; k < K; k += 32) a.ds[(row0 + j) * K + k] = gK[j * K + k] * (gg[j * K + k] - s);
        }
        for (int e = t; e < KG * W; e += kWalkThreads) {     // the state before this chunk, four components a thread
            const int c = e % W, k0q = (e / W) * 4;
            float acc[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) acc[q] = k0q + q < K ? Rs[(k0q + q) * W + c] : 0.f;
            for (int i = 0; i < n; ++i) {
                const float av = ab[i * W + c];
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    if (k0q + q < K) acc[q] = fmaf(gQ[i * K + k0q + q], av, acc[q]);
            }
#pragma unroll
            for (int q = 0; q < 4; ++q)
                if (k0q + q < K) Rs[(k0q + q) * W + c] = acc[q];
        }
    }
}

// ----------------------------------------------------------------- host side

unsigned blocks_for(size_t n, int per) { return (unsigned)((n + per - 1) / per); }

// Column tile of the product kernels: 80 columns (5 a thread) where that takes fewer
// columns in all than 64-column tiles (the widths dv + 1, 2 d + 1), else 64.
int col_tile_for(int C) {
    const int t64 = (C + 63) / 64 * 64, t80 = (C + 79) / 80 * 80;
    return t80 < t64 ? 80 : 64;
}

template <typename TA, bool MT>
cudaError_t rowmat(const Problem &p, int KA, int C, int lda, int a_cols, int a_one, const TA *A, const float *M,
                   int m_per_head, size_t m_stride, int ldm, float *out, int ldo, cudaStream_t s) {
    const int cw = col_tile_for(C);
    dim3 grid((p.N + kRmTile - 1) / kRmTile, (C + cw - 1) / cw, p.G);
    if (cw == 80)
        gb_rowmat_kernel<TA, MT, 5><<<grid, kGbThreads, 0, s>>>(p.N, KA, C, p.H, lda, a_cols, a_one, A, M,
                                                                m_per_head, m_stride, ldm, out, ldo);
    else
        gb_rowmat_kernel<TA, MT, 4><<<grid, kGbThreads, 0, s>>>(p.N, KA, C, p.H, lda, a_cols, a_one, A, M,
                                                                m_per_head, m_stride, ldm, out, ldo);
    return cudaGetLastError();
}

template <typename U>
cudaError_t outer(const Problem &p, const GbLayout &L, int W, const float *A, U u, float *part, cudaStream_t s) {
    const int cw = col_tile_for(W);
    dim3 grid(((p.K + kRmTile - 1) / kRmTile) * ((W + cw - 1) / cw), L.P, p.G);
    if (cw == 80)
        gb_outer_kernel<U, 5><<<grid, kGbThreads, 0, s>>>(p.N, p.K, W, L.P, L.rpp, A, u, part);
    else
        gb_outer_kernel<U, 4><<<grid, kGbThreads, 0, s>>>(p.N, p.K, W, L.P, L.rpp, A, u, part);
    return cudaGetLastError();
}

cudaError_t reduce(const Problem &p, const GbLayout &L, int E, int mode, const float *part, float *out,
                   cudaStream_t s) {
    gb_reduce_kernel<<<blocks_for((size_t)p.G * E, 256), 256, 0, s>>>(p.G, L.P, E, mode, part, out);
    return cudaGetLastError();
}

template <typename T>
cudaError_t run_t(const Problem &p, const GbLayout &L, const void *Qx_, const void *Kx_, const void *V_,
                  const float *mu, const float *rho, const float *alpha, const void *dO_, float *dQx, float *dKx,
                  float *dV, float *dmu, float *drho, float *dalpha, char *ws, cudaStream_t s) {
    const T *Qx = static_cast<const T *>(Qx_), *Kx = static_cast<const T *>(Kx_), *V = static_cast<const T *>(V_);
    const T *dO = static_cast<const T *>(dO_);
    const int K = p.K, d = p.d, dv = p.dv, W = dv + 1, E = 2 * d + 1;
    const size_t rows = (size_t)p.G * p.N;
    float *lam = reinterpret_cast<float *>(ws + L.lam), *cdir = reinterpret_cast<float *>(ws + L.cdir);
    float *lmu = reinterpret_cast<float *>(ws + L.lmu);
    float *gq = reinterpret_cast<float *>(ws + L.gq), *gk = reinterpret_cast<float *>(ws + L.gk);
    float *dsq = reinterpret_cast<float *>(ws + L.dsq), *dsk = reinterpret_cast<float *>(ws + L.dsk);
    float *tb = reinterpret_cast<float *>(ws + L.t), *ab = reinterpret_cast<float *>(ws + L.ab);
    float *part = reinterpret_cast<float *>(ws + L.part);
    float *mem = reinterpret_cast<float *>(ws + L.mem), *memr = reinterpret_cast<float *>(ws + L.memr);
    float *pq = reinterpret_cast<float *>(ws + L.pq), *pk = reinterpret_cast<float *>(ws + L.pk);
    cudaError_t e;
#define GB_TRY(x) do { if ((e = (x)) != cudaSuccess) return e; } while (0)
    GB_TRY(simt_params(p, rho, alpha, lam, cdir, s));
    gb_lmu_kernel<<<blocks_for((size_t)p.H * K * d, 256), 256, 0, s>>>(p.H, K, d, mu, lam, lmu);
    GB_TRY(cudaGetLastError());
    GB_TRY(simt_gamma(p, Qx, mu, lam, cdir, gq, s));
    GB_TRY(simt_gamma(p, Kx, mu, lam, cdir, gk, s));
    const unsigned row_blocks = blocks_for(rows, 8);       // one warp per row, eight rows per CTA
    GB_TRY(outer(p, L, W, gk, UValsOne<T>{V, dv}, part, s));
    if (!p.causal) {
        // memory [Vt | Z]; [num | den - eps]; a, b; g^Q -> ds^Q
        GB_TRY(reduce(p, L, K * W, 0, part, mem, s));
        GB_TRY((rowmat<float, false>(p, K, W, K, K, 0, gq, mem, 0, (size_t)K * W, W, tb, W, s)));
        gb_ab_kernel<T><<<row_blocks, 256, 0, s>>>(rows, dv, p.eps, tb, dO, ab);
        GB_TRY(cudaGetLastError());
        GB_TRY((rowmat<float, true>(p, W, K, W, W, 0, ab, mem, 0, (size_t)K * W, W, dsq, K, s)));
        gb_ds_kernel<<<row_blocks, 256, 0, s>>>(rows, K, gq, dsq);
        GB_TRY(cudaGetLastError());
        // [R | r]; g^K -> ds^K; dV
        GB_TRY(outer(p, L, W, gq, UPlain{ab, W}, part, s));
        GB_TRY(reduce(p, L, K * W, 0, part, memr, s));
        GB_TRY((rowmat<T, true>(p, W, K, dv, dv, 1, V, memr, 0, (size_t)K * W, W, dsk, K, s)));
        gb_ds_kernel<<<row_blocks, 256, 0, s>>>(rows, K, gk, dsk);
        GB_TRY(cudaGetLastError());
        GB_TRY((rowmat<float, false>(p, K, dv, K, K, 0, gk, memr, 0, (size_t)K * W, W, dV, dv, s)));
    } else {
        GbCausalArgs a{};
        a.N = p.N; a.K = K; a.dv = dv; a.P = L.P; a.rpp = L.rpp; a.C = L.C; a.eps = p.eps;
        a.gq = gq; a.gk = gk; a.V = V; a.dO = dO; a.ab = ab;
        const size_t smem = sizeof(float) * gb_causal_floats(K, dv, L.C);
        // queries: the memory of the rows before each range, then the walks
        GB_TRY(reduce(p, L, K * W, 1, part, mem, s));
        a.mem = mem; a.ds = dsq;
        GB_TRY(set_dyn_smem(reinterpret_cast<const void *>(gb_cq_kernel<T>), (int)smem));
        gb_cq_kernel<T><<<dim3(L.P, p.G), kWalkThreads, smem, s>>>(a);
        GB_TRY(cudaGetLastError());
        // keys: [R | r] of the query rows after each range, then the walks
        GB_TRY(outer(p, L, W, gq, UPlain{ab, W}, part, s));
        GB_TRY(reduce(p, L, K * W, 2, part, memr, s));
        a.mem = memr; a.ds = dsk; a.dV = dV;
        GB_TRY(set_dyn_smem(reinterpret_cast<const void *>(gb_ck_kernel<T>), (int)smem));
        gb_ck_kernel<T><<<dim3(L.P, p.G), kWalkThreads, smem, s>>>(a);
        GB_TRY(cudaGetLastError());
    }
    // dQx, dKx through ds [lambda mu | lambda]; the parameter sums of both sides
    const unsigned x_blocks = blocks_for(rows * d, 256);
    GB_TRY((rowmat<float, false>(p, K, 2 * d, K, K, 0, dsq, lmu, 1, (size_t)K * 2 * d, 2 * d, tb, 2 * d, s)));
    gb_dx_kernel<T><<<x_blocks, 256, 0, s>>>(rows, d, tb, Qx, dQx);
    GB_TRY(cudaGetLastError());
    GB_TRY((rowmat<float, false>(p, K, 2 * d, K, K, 0, dsk, lmu, 1, (size_t)K * 2 * d, 2 * d, tb, 2 * d, s)));
    gb_dx_kernel<T><<<x_blocks, 256, 0, s>>>(rows, d, tb, Kx, dKx);
    GB_TRY(cudaGetLastError());
    GB_TRY(outer(p, L, E, dsq, USquares<T>{Qx, d}, pq, s));
    GB_TRY(outer(p, L, E, dsk, USquares<T>{Kx, d}, pk, s));
    gb_param_kernel<<<dim3(K, p.H), kGbThreads, 0, s>>>(p.B, p.H, L.P, K, d, pq, pk, mu, lam, rho, alpha, dmu, drho,
                                                        dalpha);
    return cudaGetLastError();
#undef GB_TRY
}

}  // namespace

bool gb_supported(const Problem &p) {
    if (p.in_dtype != p.out_dtype) return false;
    if (!p.causal) return true;
    const int C = p.chunk > 0 ? p.chunk : kGbChunkDefault;
    return sizeof(float) * gb_causal_floats(p.K, p.dv, C) <= 227 * 1024;
}

GbLayout gb_layout(const Problem &p) {
    GbLayout L{};
    const long long want = (4LL * 160 + p.G - 1) / p.G;
    const long long by_rows = (p.N + 255) / 256;
    L.P = (int)std::max(1LL, std::min(want, by_rows));
    L.C = p.chunk > 0 ? p.chunk : kGbChunkDefault;
    if (p.causal) {
        // the walks hold one CTA per SM: pick the range count that minimises
        // (waves of P G CTAs) x (chunks per range), the largest such count
        int sms = 0, dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) !=
                                                     cudaSuccess || sms <= 0)
            sms = 152;
        long long best = -1;
        for (long long P = 1; P <= std::max(1LL, std::min(4 * want, by_rows)); ++P) {
            const long long rpp = (p.N + P - 1) / P;
            const long long cost = ((P * p.G + sms - 1) / sms) * ((rpp + L.C - 1) / L.C);
            if (best < 0 || cost <= best) { best = cost; L.P = (int)P; }
        }
    }
    L.rpp = std::max(1, (p.N + L.P - 1) / L.P);
    const size_t K = p.K, d = p.d, W = (size_t)p.dv + 1, E = 2 * d + 1, G = p.G, N = p.N, P = L.P;
    const size_t rows = G * N;
    size_t off = kHeaderBytes;
    auto take = [&](size_t floats) { const size_t o = align_up(off); off = o + sizeof(float) * floats; return o; };
    L.lam = take((size_t)p.H * K * d);
    L.cdir = take((size_t)p.H * K);
    L.lmu = take((size_t)p.H * K * 2 * d);
    L.gq = take(rows * K);
    L.gk = take(rows * K);
    L.dsq = take(rows * K);
    L.dsk = take(rows * K);
    L.t = take(rows * std::max(W, 2 * d));
    L.ab = take(rows * W);
    L.part = take(G * P * K * W);
    L.mem = take(G * P * K * W);
    L.memr = take(G * P * K * W);
    L.pq = take(G * P * K * E);
    L.pk = take(G * P * K * E);
    L.total = align_up(off);
    return L;
}

cudaError_t gb_run(const Problem &p, const GbLayout &L, const void *Qx, const void *Kx, const void *V,
                   const float *mu, const float *rho, const float *alpha, const void *dO, float *dQx, float *dKx,
                   float *dV, float *dmu, float *drho, float *dalpha, char *ws, cudaStream_t s) {
    if (p.in_dtype == GMA_F32)
        return run_t<float>(p, L, Qx, Kx, V, mu, rho, alpha, dO, dQx, dKx, dV, dmu, drho, dalpha, ws, s);
    return run_t<__nv_bfloat16>(p, L, Qx, Kx, V, mu, rho, alpha, dO, dQx, dKx, dV, dmu, drho, dalpha, ws, s);
}

}  // namespace gma
