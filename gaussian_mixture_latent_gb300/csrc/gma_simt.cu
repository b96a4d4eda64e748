// CUDA-core fp32 path of the GMA forward.
//
// This is the library's float32 path (float32 inputs need float32-accurate
// log-densities, which the tensor-core path's fp16 operands do not give) and
// its path for shapes outside the tensor-core kernels' range.  Every step
// runs in fp32 with the log-density in its direct Mahalanobis form:
//
//   s_ik = c_k - 1/2 sum_m lam_km (x_im - mu_km)^2,
//   c_k  = log pi_k - 1/2 sum_m log var_km,   lam = 1 / var
//
// ("Gaussian Mixture Attention", section 4.1 Eq. 16 without the constant
// -(d/2) log 2 pi, which the softmax of Eq. 3b cancels exactly).
//
// Steps (one launch each):
//   params        Eq. 14-15: var = softplus(rho) + var_floor, log pi = log_softmax(alpha)
//   scores        Eq. 16 for tiles of rows x components of Qx and Kx, in the workspace
//   softmax_rows  Eq. 3 / 3b over each row's scores, in place
//   write_partial Eq. 5-6 over one N-range per block row: [Vt | Z] partials
//   reduce        fixed-order sum of the partials (bidirectional) or their
//                 exclusive prefix over segments (causal, Eq. 6b)
//   read          Eq. 7-8 (bidirectional)
//   causal_chunk  Eq. 6b / 8b: per segment, chunks of rows with an on-chip
//                 [K x (dv+1)] state, intra-chunk masked Gamma^Q Gamma^K^T
//
// Reductions run in a fixed order, so results are bitwise reproducible.
#include <cuda_bf16.h>

#include <algorithm>
#include <cfloat>

#include "gma_internal.h"

namespace gma {
namespace {

template <typename T>
__device__ __forceinline__ float load_elem(const T *p, size_t i);
template <>
__device__ __forceinline__ float load_elem<float>(const float *p, size_t i) { return p[i]; }
template <>
__device__ __forceinline__ float load_elem<__nv_bfloat16>(const __nv_bfloat16 *p, size_t i) {
    return __bfloat162float(p[i]);
}

__device__ __forceinline__ void store_elem(float *p, size_t i, float v) { p[i] = v; }
__device__ __forceinline__ void store_elem(__nv_bfloat16 *p, size_t i, float v) {
    p[i] = __float2bfloat16_rn(v);
}

__device__ __forceinline__ float warp_max(float v) {
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ float warp_sum(float v) {
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Block-wide reduction for blockDim.x == 256.
template <bool kMax>
__device__ float block_reduce(float v, float *scratch) {
    v = kMax ? warp_max(v) : warp_sum(v);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    __syncthreads();
    if (lane == 0) scratch[warp] = v;
    __syncthreads();
    float r = lane < (int)(blockDim.x >> 5) ? scratch[lane] : (kMax ? -FLT_MAX : 0.f);
    if (warp == 0) r = kMax ? warp_max(r) : warp_sum(r);
    if (threadIdx.x == 0) scratch[0] = r;
    __syncthreads();
    return scratch[0];
}

// Eq. 14-15 and the per-component constant of the direct-form score.
// One block (256 threads) per head.
__global__ void params_kernel(int K, int d, float var_floor, const float *__restrict__ rho, const float *__restrict__ alpha,
                              float *__restrict__ lam, float *__restrict__ cdir) {
    __shared__ float scratch[32];
    const int h = blockIdx.x;
    const float *al = alpha + (size_t)h * K;
    float m = -FLT_MAX;
    for (int k = threadIdx.x; k < K; k += blockDim.x) m = fmaxf(m, al[k]);
    m = block_reduce<true>(m, scratch);
    float s = 0.f;
    for (int k = threadIdx.x; k < K; k += blockDim.x) s += expf(al[k] - m);
    s = block_reduce<false>(s, scratch);
    const float lse = m + logf(s);
    const float *rh = rho + (size_t)h * K * d;
    float *lh = lam + (size_t)h * K * d;
    for (int k = threadIdx.x; k < K; k += blockDim.x) {
        float logdet = 0.f;
        for (int j = 0; j < d; ++j) {
            const float w = rh[(size_t)k * d + j];
            const float var = fmaxf(w, 0.f) + log1pf(expf(-fabsf(w))) + var_floor;
            logdet += logf(var);
            lh[(size_t)k * d + j] = 1.0f / var;
        }
        cdir[(size_t)h * K + k] = (al[k] - lse) - 0.5f * logdet;
    }
}

// Eq. 16 (direct form) for a tile of 32 rows x 64 components of head-row g
// (blockIdx.z), written to s[g][i][k]: each thread owns four rows and two components
// (lane and lane + 32 of the tile), and the coordinates m are staged through shared
// memory 32 at a time.  Per (row, component) the operations and their order are the
// ones of the per-row form: acc += (x_m - mu_km)^2 lam_km for m = 0 .. d - 1, then
// s = c_k - acc / 2.
constexpr int kScoreRows = 32, kScoreComps = 64;

template <typename T>
__global__ void __launch_bounds__(256) scores_kernel(int N, int H, int d, int K, const T *__restrict__ X,
                                                     const float *__restrict__ mu, const float *__restrict__ lam,
                                                     const float *__restrict__ cdir, float *__restrict__ out) {
    __shared__ float xs[kScoreRows][33];
    __shared__ float ms[kScoreComps][33];
    __shared__ float ls[kScoreComps][33];
    const int i0 = blockIdx.x * kScoreRows, k0 = blockIdx.y * kScoreComps, g = blockIdx.z, h = g % H;
    const int lane = threadIdx.x & 31, ty = threadIdx.x >> 5;
    const float *mu_h = mu + (size_t)h * K * d, *lam_h = lam + (size_t)h * K * d;
    float acc[4][2] = {{0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}};
    for (int j0 = 0; j0 < d; j0 += 32) {
        for (int e = threadIdx.x; e < kScoreRows * 32; e += 256) {
            const int r = e >> 5, jj = e & 31, i = i0 + r, j = j0 + jj;
            xs[r][jj] = (i < N && j < d) ? load_elem(X, ((size_t)g * N + i) * d + j) : 0.f;
        }
        for (int e = threadIdx.x; e < kScoreComps * 32; e += 256) {
            const int kk = e >> 5, jj = e & 31, k = k0 + kk, j = j0 + jj;
            const bool ok = k < K && j < d;
            ms[kk][jj] = ok ? mu_h[(size_t)k * d + j] : 0.f;
            ls[kk][jj] = ok ? lam_h[(size_t)k * d + j] : 0.f;
        }
        __syncthreads();
#pragma unroll 4
        for (int jj = 0; jj < 32; ++jj) {
            const float m0 = ms[lane][jj], m1 = ms[lane + 32][jj];
            const float l0 = ls[lane][jj], l1 = ls[lane + 32][jj];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float x = xs[ty * 4 + q][jj];
                const float d0 = x - m0, d1 = x - m1;
                acc[q][0] = fmaf(d0 * d0, l0, acc[q][0]);
                acc[q][1] = fmaf(d1 * d1, l1, acc[q][1]);
            }
        }
        __syncthreads();
    }
#pragma unroll
    for (int c = 0; c < 2; ++c) {
        const int k = k0 + lane + 32 * c;
        if (k >= K) continue;
        const float ck = cdir[(size_t)h * K + k];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int i = i0 + ty * 4 + q;
            if (i < N) out[((size_t)g * N + i) * K + k] = ck - 0.5f * acc[q][c];
        }
    }
}

// Eq. 3 / 3b over the scores of one row, in place: one warp per row, lane l owns
// components l, l + 32, ... (K <= 256).
__global__ void softmax_rows_kernel(size_t rows, int K, float *__restrict__ gamma) {
    const size_t row = (size_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= rows) return;
    float *gr = gamma + row * K;
    float s[8];
    float mx = -FLT_MAX;
#pragma unroll
    for (int t = 0; t < 8; ++t) {
        const int k = lane + 32 * t;
        s[t] = -FLT_MAX;
        if (k < K) {
            s[t] = gr[k];
            mx = fmaxf(mx, s[t]);
        }
    }
    mx = warp_max(mx);
    float sum = 0.f;
#pragma unroll
    for (int t = 0; t < 8; ++t) {
        const int k = lane + 32 * t;
        if (k < K) {
            s[t] = expf(s[t] - mx);
            sum += s[t];
        }
    }
    sum = warp_sum(sum);
    const float inv = 1.0f / sum;
#pragma unroll
    for (int t = 0; t < 8; ++t) {
        const int k = lane + 32 * t;
        if (k < K) gr[k] = s[t] * inv;
    }
}

// Eq. 5-6 over rows [p*rpp, min(N,(p+1)*rpp)) of head g:
//   part[g][p][k][c] = sum_j gamma^K_jk * Vaug_jc,   Vaug = [V | 1]  (W = dv + 1 columns).
// 32x32 output tile per block, 256 threads, 4 outputs per thread.
template <typename T>
__global__ void write_partial_kernel(int N, int K, int dv, int P, int rpp,
                                     const float *__restrict__ gk, const T *__restrict__ V,
                                     float *__restrict__ part) {
    __shared__ float gs[32][33];
    __shared__ float vs[32][33];
    const int W = dv + 1;
    const int ktiles = (K + 31) / 32;
    const int kt = blockIdx.x % ktiles, ct = blockIdx.x / ktiles;
    const int p = blockIdx.y, g = blockIdx.z;
    const int r0 = p * rpp, r1 = min(N, r0 + rpp);
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    for (int j0 = r0; j0 < r1; j0 += 32) {
        for (int e = threadIdx.x; e < 1024; e += 256) {
            const int jr = e >> 5, cc = e & 31;
            const int j = j0 + jr;
            const int k = kt * 32 + cc, c = ct * 32 + cc;
            gs[jr][cc] = (j < r1 && k < K) ? gk[((size_t)g * N + j) * K + k] : 0.f;
            float v = 0.f;
            if (j < r1) v = c < dv ? load_elem(V, ((size_t)g * N + j) * dv + c) : (c == dv ? 1.f : 0.f);
            vs[jr][cc] = v;
        }
        __syncthreads();
#pragma unroll 8
        for (int jr = 0; jr < 32; ++jr) {
            const float v = vs[jr][tx];
#pragma unroll
            for (int q = 0; q < 4; ++q) acc[q] = fmaf(gs[jr][ty * 4 + q], v, acc[q]);
        }
        __syncthreads();
    }
    const int c = ct * 32 + tx;
    if (c < W) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int k = kt * 32 + ty * 4 + q;
            if (k < K) part[(((size_t)g * P + p) * K + k) * W + c] = acc[q];
        }
    }
}

// Bidirectional: mem[g][e] = sum_{p=0..P-1} part[g][p][e] (fixed order).
// Causal:        mem[g][p][e] = sum_{q<p} part[g][q][e] (exclusive prefix, fixed order).
__global__ void reduce_kernel(int G, int P, int KW, int exclusive_prefix,
                              const float *__restrict__ part, float *__restrict__ mem) {
    const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (size_t)G * KW) return;
    const size_t g = i / KW, e = i % KW;
    float acc = 0.f;
    for (int p = 0; p < P; ++p) {
        const float v = part[(g * P + p) * KW + e];
        if (exclusive_prefix) mem[(g * P + p) * KW + e] = acc;
        acc += v;
    }
    if (!exclusive_prefix) mem[g * KW + e] = acc;
}

// Eq. 7-8: out[i][c] = sum_k gq_ik Vt_kc / (sum_k gq_ik Z_k + eps).
// Tile: 32 rows x 32 value columns per block; den is accumulated alongside.
template <typename Tout>
__global__ void read_kernel(int N, int K, int dv, float eps, const float *__restrict__ gq,
                            const float *__restrict__ mem, Tout *__restrict__ out) {
    __shared__ float gs[32][33];
    __shared__ float ms[32][33];
    __shared__ float zs[32];
    __shared__ float dens[32];
    const int W = dv + 1;
    const int i0 = blockIdx.x * 32, c0 = blockIdx.y * 32, g = blockIdx.z;
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
    const float *memg = mem + (size_t)g * K * W;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    float den[4] = {0.f, 0.f, 0.f, 0.f};
    for (int k0 = 0; k0 < K; k0 += 32) {
        for (int e = threadIdx.x; e < 1024; e += 256) {
            const int r = e >> 5, cc = e & 31;
            const int i = i0 + r, k = k0 + cc;
            gs[r][cc] = (i < N && k < K) ? gq[((size_t)g * N + i) * K + k] : 0.f;
            const int kk = k0 + r, c = c0 + cc;
            ms[r][cc] = (kk < K && c < dv) ? memg[(size_t)kk * W + c] : 0.f;
        }
        if (threadIdx.x < 32) zs[threadIdx.x] = (k0 + threadIdx.x < K) ? memg[(size_t)(k0 + threadIdx.x) * W + dv] : 0.f;
        __syncthreads();
#pragma unroll 8
        for (int kk = 0; kk < 32; ++kk) {
            const float m = ms[kk][tx];
#pragma unroll
            for (int q = 0; q < 4; ++q) acc[q] = fmaf(gs[ty * 4 + q][kk], m, acc[q]);
        }
        if (tx == 0) {
            for (int kk = 0; kk < 32; ++kk)
#pragma unroll
                for (int q = 0; q < 4; ++q) den[q] = fmaf(gs[ty * 4 + q][kk], zs[kk], den[q]);
        }
        __syncthreads();
    }
    if (tx == 0)
#pragma unroll
        for (int q = 0; q < 4; ++q) dens[ty * 4 + q] = den[q] + eps;
    __syncthreads();
    const int c = c0 + tx;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const int i = i0 + ty * 4 + q;
        if (i < N && c < dv) store_elem(out, ((size_t)g * N + i) * dv + c, acc[q] / dens[ty * 4 + q]);
    }
}

constexpr int kCausalChunkDefault = 16;

int causal_chunk_rows(const Problem &p) { return p.chunk > 0 ? p.chunk : kCausalChunkDefault; }

// Eq. 6b / 8b for rows [p*rpp, min(N,(p+1)*rpp)) of head g, starting from the
// exclusive prefix state prefix[g][p] = [Vt | Z] of all earlier rows.
// Per chunk of C rows (i, j inside the chunk):
//   T_ij  = [j <= i] sum_k gq_ik gk_jk
//   num_i = gq_i S + sum_j T_ij Vaug_j     (column dv is the denominator without eps)
//   out_i = num_i[:dv] / (num_i[dv] + eps)
//   S    += gk^T Vaug                      (inclusive of the chunk)
template <typename T, typename Tout>
__global__ void causal_chunk_kernel(int N, int K, int dv, int P, int rpp, int C, float eps,
                                    const float *__restrict__ gq, const float *__restrict__ gk,
                                    const T *__restrict__ V, const float *__restrict__ prefix,
                                    Tout *__restrict__ out) {
    extern __shared__ float sm[];
    const int W = dv + 1;
    const int p = blockIdx.x, g = blockIdx.y;
    const int r0 = p * rpp, r1 = min(N, r0 + rpp);
    float *S = sm;                         // [K][W]
    float *q = S + (size_t)K * W;          // [C][K]
    float *kk = q + C * K;                 // [C][K]
    float *v = kk + C * K;                 // [C][W]
    float *Tm = v + C * W;                 // [C][C]
    float *num = Tm + C * C;               // [C][W]
    const float *pre = prefix + ((size_t)g * P + p) * K * W;
    for (int e = threadIdx.x; e < K * W; e += blockDim.x) S[e] = pre[e];
    for (int c0 = r0; c0 < r1; c0 += C) {
        __syncthreads();
        for (int e = threadIdx.x; e < C * K; e += blockDim.x) {
            const int r = e / K, k = e % K;
            const int i = c0 + r;
            q[e] = i < r1 ? gq[((size_t)g * N + i) * K + k] : 0.f;
            kk[e] = i < r1 ? gk[((size_t)g * N + i) * K + k] : 0.f;
        }
        for (int e = threadIdx.x; e < C * W; e += blockDim.x) {
            const int r = e / W, c = e % W;
            const int i = c0 + r;
            v[e] = i < r1 ? (c < dv ? load_elem(V, ((size_t)g * N + i) * dv + c) : 1.f) : 0.f;
        }
        __syncthreads();
        for (int e = threadIdx.x; e < C * C; e += blockDim.x) {
            const int i = e / C, j = e % C;
            float t = 0.f;
            if (j <= i)
                for (int k = 0; k < K; ++k) t = fmaf(q[i * K + k], kk[j * K + k], t);
            Tm[e] = t;
        }
        __syncthreads();
        for (int e = threadIdx.x; e < C * W; e += blockDim.x) {
            const int i = e / W, c = e % W;
            float a = 0.f;
            for (int k = 0; k < K; ++k) a = fmaf(q[i * K + k], S[(size_t)k * W + c], a);
            for (int j = 0; j <= i; ++j) a = fmaf(Tm[i * C + j], v[j * W + c], a);
            num[e] = a;
        }
        __syncthreads();
        for (int e = threadIdx.x; e < C * dv; e += blockDim.x) {
            const int i = e / dv, c = e % dv;
            if (c0 + i < r1)
                store_elem(out, ((size_t)g * N + c0 + i) * dv + c, num[i * W + c] / (num[i * W + dv] + eps));
        }
        for (int e = threadIdx.x; e < K * W; e += blockDim.x) {
            const int k = e / W, c = e % W;
            float a = S[e];
            for (int j = 0; j < C; ++j) a = fmaf(kk[j * K + k], v[j * W + c], a);
            S[e] = a;
        }
    }
}

}  // namespace

SimtLayout simt_layout(const Problem &p) {
    SimtLayout L{};
    // Enough blocks to cover the SMs a few times over; at least 256 rows each.
    const long long want = (4LL * 160 + p.G - 1) / p.G;
    const long long by_rows = (p.N + 255) / 256;
    L.P = (int)std::max(1LL, std::min(want, by_rows));
    const size_t W = (size_t)p.dv + 1;
    size_t off = kHeaderBytes;
    L.lam = off;  off = align_up(off + sizeof(float) * p.H * p.K * p.d);
    L.cdir = off; off = align_up(off + sizeof(float) * p.H * p.K);
    L.gq = off;   off = align_up(off + sizeof(float) * p.G * (size_t)p.N * p.K);
    L.gk = off;   off = align_up(off + sizeof(float) * p.G * (size_t)p.N * p.K);
    L.part = off; off = align_up(off + sizeof(float) * p.G * (size_t)L.P * p.K * W);
    L.mem = off;  off = align_up(off + sizeof(float) * p.G * (size_t)L.P * p.K * W);
    L.total = off;
    return L;
}

cudaError_t simt_params(const Problem &p, const float *rho, const float *alpha, float *lam,
                        float *cdir, cudaStream_t s) {
    params_kernel<<<p.H, 256, 0, s>>>(p.K, p.d, p.var_floor, rho, alpha, lam, cdir);
    return cudaGetLastError();
}

cudaError_t simt_gamma(const Problem &p, const void *X, const float *mu, const float *lam,
                       const float *cdir, float *gamma, cudaStream_t s) {
    const size_t rows = (size_t)p.G * p.N;
    if (rows == 0) return cudaSuccess;
    // scores by tiles of rows x components, then the softmax of every row in place
    const dim3 grid((p.N + kScoreRows - 1) / kScoreRows, (p.K + kScoreComps - 1) / kScoreComps, p.G);
    if (p.in_dtype == GMA_F32)
        scores_kernel<float><<<grid, 256, 0, s>>>(p.N, p.H, p.d, p.K, static_cast<const float *>(X), mu, lam, cdir,
                                                  gamma);
    else
        scores_kernel<__nv_bfloat16><<<grid, 256, 0, s>>>(p.N, p.H, p.d, p.K, static_cast<const __nv_bfloat16 *>(X),
                                                          mu, lam, cdir, gamma);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    softmax_rows_kernel<<<(unsigned)((rows + 7) / 8), 256, 0, s>>>(rows, p.K, gamma);
    return cudaGetLastError();
}

cudaError_t simt_write(const Problem &p, const void *V, char *ws, const SimtLayout &L,
                       cudaStream_t s) {
    const int W = p.dv + 1;
    const int rpp = (p.N + L.P - 1) / L.P;
    dim3 grid(((p.K + 31) / 32) * ((W + 31) / 32), L.P, p.G);
    const float *gk = reinterpret_cast<const float *>(ws + L.gk);
    float *part = reinterpret_cast<float *>(ws + L.part);
    if (p.in_dtype == GMA_F32)
        write_partial_kernel<float><<<grid, 256, 0, s>>>(p.N, p.K, p.dv, L.P, rpp, gk,
                                                         static_cast<const float *>(V), part);
    else
        write_partial_kernel<__nv_bfloat16><<<grid, 256, 0, s>>>(
            p.N, p.K, p.dv, L.P, rpp, gk, static_cast<const __nv_bfloat16 *>(V), part);
    return cudaGetLastError();
}

cudaError_t simt_reduce(const Problem &p, char *ws, const SimtLayout &L, cudaStream_t s) {
    const int W = p.dv + 1;
    const size_t n = (size_t)p.G * p.K * W;
    reduce_kernel<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(
        p.G, L.P, p.K * W, p.causal, reinterpret_cast<const float *>(ws + L.part),
        reinterpret_cast<float *>(ws + L.mem));
    return cudaGetLastError();
}

namespace {
template <typename Tout>
cudaError_t read_t(const Problem &p, char *ws, const SimtLayout &L, void *out, cudaStream_t s) {
    dim3 grid((p.N + 31) / 32, (p.dv + 31) / 32, p.G);
    read_kernel<Tout><<<grid, 256, 0, s>>>(p.N, p.K, p.dv, p.eps,
                                           reinterpret_cast<const float *>(ws + L.gq),
                                           reinterpret_cast<const float *>(ws + L.mem),
                                           static_cast<Tout *>(out));
    return cudaGetLastError();
}

template <typename T, typename Tout>
cudaError_t causal_t(const Problem &p, const void *V, char *ws, const SimtLayout &L, void *out,
                     cudaStream_t s) {
    const int C = causal_chunk_rows(p);
    const int rpp = (p.N + L.P - 1) / L.P;
    const size_t smem = simt_causal_smem(p);
    auto kern = causal_chunk_kernel<T, Tout>;
    cudaError_t e = set_dyn_smem(reinterpret_cast<const void *>(kern), (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid(L.P, p.G);
    kern<<<grid, 256, smem, s>>>(p.N, p.K, p.dv, L.P, rpp, C, p.eps,
                                 reinterpret_cast<const float *>(ws + L.gq),
                                 reinterpret_cast<const float *>(ws + L.gk),
                                 static_cast<const T *>(V),
                                 reinterpret_cast<const float *>(ws + L.mem),
                                 static_cast<Tout *>(out));
    return cudaGetLastError();
}
}  // namespace

cudaError_t simt_read(const Problem &p, char *ws, const SimtLayout &L, void *out, cudaStream_t s) {
    return p.out_dtype == GMA_F32 ? read_t<float>(p, ws, L, out, s)
                                  : read_t<__nv_bfloat16>(p, ws, L, out, s);
}

cudaError_t simt_causal(const Problem &p, const void *V, char *ws, const SimtLayout &L, void *out,
                        cudaStream_t s) {
    if (p.in_dtype == GMA_F32)
        return p.out_dtype == GMA_F32 ? causal_t<float, float>(p, V, ws, L, out, s)
                                      : causal_t<float, __nv_bfloat16>(p, V, ws, L, out, s);
    return p.out_dtype == GMA_F32 ? causal_t<__nv_bfloat16, float>(p, V, ws, L, out, s)
                                  : causal_t<__nv_bfloat16, __nv_bfloat16>(p, V, ws, L, out, s);
}

size_t simt_causal_smem(const Problem &p) {
    const size_t C = (size_t)causal_chunk_rows(p);
    const size_t W = (size_t)p.dv + 1;
    return sizeof(float) * ((size_t)p.K * W + 2 * C * p.K + C * W + C * C + C * W);
}

}  // namespace gma
