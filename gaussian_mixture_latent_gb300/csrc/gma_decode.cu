// Causal decode with a carried state: new positions appended to a causal GMA
// sequence, one at a time, against the prefix memory of everything before them.
//
// "Gaussian Mixture Attention" (Huang & Raza, 2026), section 3.5, Eq. 6b and 8b
// as a recurrence.  Per head, with the state [S | z] = sum over the earlier
// positions j of gamma^K_j [V_j | 1] ([K, dv + 1], fp32), each new position t:
//   [S | z] += gamma^K(k_t) [v_t | 1]                       (the prefix includes t)
//   o_t      = gamma^Q(q_t) S / (gamma^Q(q_t) z + eps)
// with gamma from the direct-form score of Eq. 16 in fp32 (the parameter
// prologue is the fp32 path's: precisions lambda = 1 / var and the constants).
//
// decode_kernel: one CTA per head, the state in shared memory for the whole
// call; for each position: both log-densities (threads over (row, component)),
// the two softmaxes, the state update (threads over state entries), then the
// read (threads over value columns, a fixed-order sum over components).
#include <cuda_bf16.h>

#include <cfloat>

#include "gma_internal.h"

namespace gma {
namespace {

constexpr int kDecThreads = 256;
constexpr size_t kDecMaxSmem = 227 * 1024;        // opt-in shared memory of one CTA

__device__ __forceinline__ float dec_load(const float *p, size_t i) { return p[i]; }
__device__ __forceinline__ float dec_load(const __nv_bfloat16 *p, size_t i) { return __bfloat162float(p[i]); }
__device__ __forceinline__ void dec_store(float *p, size_t i, float v) { p[i] = v; }
__device__ __forceinline__ void dec_store(__nv_bfloat16 *p, size_t i, float v) { p[i] = __float2bfloat16_rn(v); }

// Block-wide max or sum of one value per thread (fixed order: lanes, then warps).
template <bool kMax>
__device__ float dec_reduce(float v, float *scratch) {
    for (int o = 16; o; o >>= 1) {
        const float w = __shfl_xor_sync(~0u, v, o);
        v = kMax ? fmaxf(v, w) : v + w;
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    __syncthreads();
    if (lane == 0) scratch[warp] = v;
    __syncthreads();
    float r = kMax ? -FLT_MAX : 0.f;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) r = kMax ? fmaxf(r, scratch[w]) : r + scratch[w];
    return r;
}

template <typename TI, typename TO>
__global__ void __launch_bounds__(kDecThreads) decode_kernel(int H, int T, int d, int K, int dv, float eps,
                                                             const TI *__restrict__ Qx, const TI *__restrict__ Kx,
                                                             const TI *__restrict__ V, const float *__restrict__ mu,
                                                             const float *__restrict__ lam,
                                                             const float *__restrict__ cdir,
                                                             float *__restrict__ state, TO *__restrict__ out) {
    extern __shared__ float sm[];
    const int W = dv + 1;
    float *st = sm;                        // [K][W] state of this head
    float *xq = st + (size_t)K * W;        // [d] query routing vector
    float *xk = xq + d;                    // [d] key routing vector
    float *vv = xk + d;                    // [dv] value
    float *gq = vv + dv;                   // [K] query scores, then responsibilities
    float *gk = gq + K;                    // [K] key scores, then responsibilities
    float *scratch = gk + K;               // [32]
    const int g = blockIdx.x, h = g % H;
    const float *mu_h = mu + (size_t)h * K * d, *lam_h = lam + (size_t)h * K * d, *c_h = cdir + (size_t)h * K;
    float *st_g = state + (size_t)g * K * W;
    for (int e = threadIdx.x; e < K * W; e += blockDim.x) st[e] = st_g[e];
    for (int t = 0; t < T; ++t) {
        const size_t row = (size_t)g * T + t;
        for (int j = threadIdx.x; j < d; j += blockDim.x) {
            xq[j] = dec_load(Qx, row * d + j);
            xk[j] = dec_load(Kx, row * d + j);
        }
        for (int c = threadIdx.x; c < dv; c += blockDim.x) vv[c] = dec_load(V, row * dv + c);
        __syncthreads();
        // Eq. 16 (direct form, the shared -d/2 log 2 pi dropped): score of the key and the query
        for (int e = threadIdx.x; e < 2 * K; e += blockDim.x) {
            const int k = e >> 1;
            const float *x = (e & 1) ? xq : xk;
            float acc = 0.f;
            for (int j = 0; j < d; ++j) {
                const float diff = x[j] - mu_h[(size_t)k * d + j];
                acc = fmaf(diff * diff, lam_h[(size_t)k * d + j], acc);
            }
            ((e & 1) ? gq : gk)[k] = c_h[k] - 0.5f * acc;
        }
        __syncthreads();
        // Eq. 3b: the two softmaxes over components
        float mq = -FLT_MAX, mk = -FLT_MAX;
        for (int k = threadIdx.x; k < K; k += blockDim.x) { mq = fmaxf(mq, gq[k]); mk = fmaxf(mk, gk[k]); }
        mq = dec_reduce<true>(mq, scratch);
        mk = dec_reduce<true>(mk, scratch);
        float sq = 0.f, sk = 0.f;
        for (int k = threadIdx.x; k < K; k += blockDim.x) {
            gq[k] = expf(gq[k] - mq);
            gk[k] = expf(gk[k] - mk);
            sq += gq[k];
            sk += gk[k];
        }
        sq = dec_reduce<false>(sq, scratch);
        sk = dec_reduce<false>(sk, scratch);
        const float iq = 1.0f / sq, ik = 1.0f / sk;
        for (int k = threadIdx.x; k < K; k += blockDim.x) { gq[k] *= iq; gk[k] *= ik; }
        __syncthreads();
        // Eq. 6b: the prefix memory now includes position t
        for (int e = threadIdx.x; e < K * W; e += blockDim.x) {
            const int k = e / W, c = e - k * W;
            st[e] = fmaf(gk[k], c < dv ? vv[c] : 1.0f, st[e]);
        }
        __syncthreads();
        // Eq. 8b: the read of position t
        float den = 0.f;
        for (int k = threadIdx.x; k < K; k += blockDim.x) den = fmaf(gq[k], st[(size_t)k * W + dv], den);
        den = dec_reduce<false>(den, scratch) + eps;
        for (int c = threadIdx.x; c < dv; c += blockDim.x) {
            float num = 0.f;
            for (int k = 0; k < K; ++k) num = fmaf(gq[k], st[(size_t)k * W + c], num);
            dec_store(out, row * dv + c, num / den);
        }
        __syncthreads();
    }
    for (int e = threadIdx.x; e < K * W; e += blockDim.x) st_g[e] = st[e];
}

size_t decode_smem(const Problem &p) {
    return sizeof(float) * ((size_t)p.K * (p.dv + 1) + 2 * p.d + p.dv + 2 * p.K + 32);
}

template <typename TI, typename TO>
cudaError_t launch_decode(const Problem &p, const void *Qx, const void *Kx, const void *V, const float *mu,
                          const float *lam, const float *cdir, float *state, void *out, cudaStream_t s) {
    auto kern = decode_kernel<TI, TO>;
    const size_t smem = decode_smem(p);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<p.G, kDecThreads, smem, s>>>(p.H, p.N, p.d, p.K, p.dv, p.eps, static_cast<const TI *>(Qx),
                                       static_cast<const TI *>(Kx), static_cast<const TI *>(V), mu, lam, cdir,
                                       state, static_cast<TO *>(out));
    return cudaGetLastError();
}

}  // namespace

bool decode_supported(const Problem &p) { return decode_smem(p) <= kDecMaxSmem; }

DecodeLayout decode_layout(const Problem &p) {
    DecodeLayout L{};
    L.lam = align_up(kHeaderBytes);
    L.cdir = align_up(L.lam + sizeof(float) * (size_t)p.H * p.K * p.d);
    L.total = align_up(L.cdir + sizeof(float) * (size_t)p.H * p.K);
    return L;
}

cudaError_t decode_step(const Problem &p, const void *Qx, const void *Kx, const void *V, const float *mu,
                        const float *lam, const float *cdir, float *state, void *out, cudaStream_t s) {
    const bool bi = p.in_dtype == GMA_BF16, bo = p.out_dtype == GMA_BF16;
    if (bi && bo) return launch_decode<__nv_bfloat16, __nv_bfloat16>(p, Qx, Kx, V, mu, lam, cdir, state, out, s);
    if (bi) return launch_decode<__nv_bfloat16, float>(p, Qx, Kx, V, mu, lam, cdir, state, out, s);
    if (bo) return launch_decode<float, __nv_bfloat16>(p, Qx, Kx, V, mu, lam, cdir, state, out, s);
    return launch_decode<float, float>(p, Qx, Kx, V, mu, lam, cdir, state, out, s);
}

}  // namespace gma
