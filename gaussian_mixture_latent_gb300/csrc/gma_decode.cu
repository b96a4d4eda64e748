// Causal decode with a carried state: new positions appended to a causal GMA
// sequence, one at a time, against the prefix memory of everything before them.
//
// "Gaussian Mixture Attention" (Huang & Raza, 2026), section 3.5, Eq. 6b and 8b
// as a recurrence.  Per head, with the state [S | z] = sum over the earlier
// positions j of gamma^K_j [V_j | 1] ([K, dv + 1], fp32), each new position t:
//   [S | z] += gamma^K(k_t) [v_t | 1]                       (the prefix includes t)
//   o_t      = gamma^Q(q_t) S / (gamma^Q(q_t) z + eps)
// with gamma from the direct-form score of Eq. 16 in fp32.
//
// decode_kernel: one CTA per head and the whole call in one launch.  The
// prologue puts every global read of the call in flight at once (cp.async into
// shared memory: the state, rho, mu when it fits, the log-prior logits, and the
// first position's row), then builds the head's precisions lambda = 1 / var in
// place of rho and the per-component constants of Eq. 16 (a warp per
// component, lanes over the d dimensions).  Each position then takes four
// barriers: both log-densities (a warp per (component, side), lanes over d),
// the two softmaxes (a warp each), the state update fused with the read
// (threads over the dv + 1 state columns, a fixed-order sum over components),
// and the normalisation; the next position's row is staged meanwhile.
#include <cuda_bf16.h>

#include <cfloat>
#include <cstdint>

#include "gma_internal.h"

namespace gma {
namespace {

constexpr int kDecThreads = 512;
constexpr int kDecWarps = kDecThreads / 32;
constexpr int kDecRows = 4;                          // components a warp works on at once

// Component ranges of the fused update and read: as many copies of the dv + 1
// state columns as fit the block.
__host__ __device__ inline int dec_ranges(int dv) {
    const int r = kDecThreads / (dv + 1);
    return r < 1 ? 1 : r;
}
constexpr size_t kDecMaxSmem = 227 * 1024;        // opt-in shared memory of one CTA

__device__ __forceinline__ float dec_load(const float *p, size_t i) { return p[i]; }
__device__ __forceinline__ float dec_load(const __nv_bfloat16 *p, size_t i) { return __bfloat162float(p[i]); }
__device__ __forceinline__ void dec_store(float *p, size_t i, float v) { p[i] = v; }
__device__ __forceinline__ void dec_store(__nv_bfloat16 *p, size_t i, float v) { p[i] = __float2bfloat16_rn(v); }

// Shared-memory carve-up of one CTA, in bytes; every offset a multiple of 16.
struct DecSmem {
    uint32_t lam, mu, st, cst, gq, gk, num, stage, stage_bytes, kx, vx, total;
};

__host__ __device__ inline uint32_t dec_round16(size_t b) { return (uint32_t)((b + 15) & ~size_t(15)); }

__host__ __device__ inline DecSmem dec_smem(int d, int K, int dv, int in_bytes, bool mu_in_smem) {
    DecSmem L{};
    uint32_t o = 0;
    L.lam = o;  o += dec_round16(4ull * K * d);
    L.mu = o;   o += mu_in_smem ? dec_round16(4ull * K * d) : 0;
    L.st = o;   o += dec_round16(4ull * K * (dv + 1));
    L.cst = o;  o += dec_round16(4ull * K);
    L.gq = o;   o += dec_round16(4ull * K);
    L.gk = o;   o += dec_round16(4ull * K);
    L.num = o;  o += dec_round16(4ull * dec_ranges(dv) * (dv + 1));
    L.kx = dec_round16((size_t)in_bytes * d);                  // within a stage: q at 0, then k, then v
    L.vx = L.kx + dec_round16((size_t)in_bytes * d);
    L.stage_bytes = L.vx + dec_round16((size_t)in_bytes * dv);
    L.stage = o; o += 2 * L.stage_bytes;                       // double-buffered row of (q, k, v)
    L.total = o;
    return L;
}

__device__ __forceinline__ uint32_t dec_smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Start an asynchronous copy of n bytes from global to shared memory, spread over
// the block: 16-byte pieces when both ends and the size allow, else 4-byte
// pieces, else (odd sizes or addresses) plain loads and stores.  Complete after
// dec_copy_wait() and a barrier.
__device__ void dec_copy(void *dst, const void *src, size_t n) {
    const uint32_t d = dec_smem_u32(dst);
    const size_t g = __cvta_generic_to_global(src);
    if (((d | g | n) & 15) == 0) {
        for (size_t i = 16 * threadIdx.x; i < n; i += 16 * blockDim.x)
            asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d + (uint32_t)i), "l"(g + i) : "memory");
    } else if (((d | g | n) & 3) == 0) {
        for (size_t i = 4 * threadIdx.x; i < n; i += 4 * blockDim.x)
            asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(d + (uint32_t)i), "l"(g + i) : "memory");
    } else {
        const unsigned short *s2 = static_cast<const unsigned short *>(src);
        unsigned short *d2 = static_cast<unsigned short *>(dst);
        for (size_t i = threadIdx.x; i < n / 2; i += blockDim.x) d2[i] = s2[i];
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
}

__device__ __forceinline__ void dec_copy_wait() { asm volatile("cp.async.wait_all;" ::: "memory"); }
// Wait for all but the N most recently started copies (each dec_copy is one group).
template <int N>
__device__ __forceinline__ void dec_copy_wait_but() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

__device__ __forceinline__ float warp_sum(float v) {
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(~0u, v, o);
    return v;
}
__device__ __forceinline__ float warp_max(float v) {
    for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(~0u, v, o));
    return v;
}

// Eq. 3b over the K scores in g, by one warp, in place.
__device__ __forceinline__ void warp_softmax(float *g, int K, int lane) {
    float m = -FLT_MAX;
    for (int k = lane; k < K; k += 32) m = fmaxf(m, g[k]);
    m = warp_max(m);
    float sum = 0.f;
    for (int k = lane; k < K; k += 32) {
        const float e = expf(g[k] - m);
        g[k] = e;
        sum += e;
    }
    const float inv = 1.0f / warp_sum(sum);
    for (int k = lane; k < K; k += 32) g[k] *= inv;
}

template <typename TI, typename TO>
__global__ void __launch_bounds__(kDecThreads) decode_kernel(int H, int T, int d, int K, int dv, float eps,
                                                             float var_floor, DecSmem L, bool mu_in_smem,
                                                             const TI *__restrict__ Qx, const TI *__restrict__ Kx,
                                                             const TI *__restrict__ V, const float *__restrict__ mu,
                                                             const float *__restrict__ rho,
                                                             const float *__restrict__ alpha,
                                                             float *__restrict__ state, TO *__restrict__ out) {
    extern __shared__ __align__(16) unsigned char dsm[];
    const int W = dv + 1;
    const int P = dec_ranges(dv);
    const int g = blockIdx.x, h = g % H, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    float *lam = reinterpret_cast<float *>(dsm + L.lam);      // [K][d] rho, then 1 / var
    float *st = reinterpret_cast<float *>(dsm + L.st);        // [K][W] state of this head
    float *cst = reinterpret_cast<float *>(dsm + L.cst);      // [K] alpha, then the constants
    float *gq = reinterpret_cast<float *>(dsm + L.gq);        // [K] query scores, then responsibilities
    float *gk = reinterpret_cast<float *>(dsm + L.gk);        // [K] key scores, then responsibilities
    float *num = reinterpret_cast<float *>(dsm + L.num);      // [P][W] partial reads (numerators, denominator)
    const float *mu_h = mu + (size_t)h * K * d;
    const float *mus = mu_in_smem ? reinterpret_cast<const float *>(dsm + L.mu) : mu_h;
    float *st_g = state + (size_t)g * K * W;
    auto stage_row = [&](int t) {
        unsigned char *sb = dsm + L.stage + (t & 1) * L.stage_bytes;
        const size_t row = (size_t)g * T + t;
        dec_copy(sb, Qx + row * d, sizeof(TI) * d);
        dec_copy(sb + L.kx, Kx + row * d, sizeof(TI) * d);
        dec_copy(sb + L.vx, V + row * dv, sizeof(TI) * dv);
    };
    // rho and alpha first: the precisions are built while the rest is in flight
    dec_copy(lam, rho + (size_t)h * K * d, 4ull * K * d);
    dec_copy(cst, alpha + (size_t)h * K, 4ull * K);
    if (mu_in_smem) dec_copy(dsm + L.mu, mu_h, 4ull * K * d);
    dec_copy(st, st_g, 4ull * K * W);
    stage_row(0);
    if (mu_in_smem) dec_copy_wait_but<5>();           // all but (mu, state, q, k, v)
    else dec_copy_wait_but<4>();
    __syncthreads();
    // Eq. 14: var = softplus(rho) + floor, kept as the precision 1 / var; the log-determinant
    // of each component.  A warp takes kDecRows components at once (lanes over dimensions,
    // a fixed-order tree per component), so their dependency chains overlap.  With Eq. 15
    // this gives the constant of Eq. 16's direct form, alpha_k - (1/2) log |Sigma_k|: the
    // normaliser of log pi = log_softmax(alpha) and the shared -(d/2) log 2 pi are the
    // same for every component and cancel in the softmax over components.
    for (int k0 = warp * kDecRows; k0 < K; k0 += kDecWarps * kDecRows) {
        float ld[kDecRows];
#pragma unroll
        for (int r = 0; r < kDecRows; ++r) ld[r] = 0.f;
        for (int j = lane; j < d; j += 32) {
#pragma unroll
            for (int r = 0; r < kDecRows; ++r) {
                if (k0 + r < K) {
                    float *q = lam + (size_t)(k0 + r) * d + j;
                    const float w = *q;
                    const float var = fmaxf(w, 0.f) + log1pf(expf(-fabsf(w))) + var_floor;
                    *q = __frcp_rn(var);
                    ld[r] += logf(var);
                }
            }
        }
#pragma unroll
        for (int r = 0; r < kDecRows; ++r) {
            const float v = warp_sum(ld[r]);
            if (lane == 0 && k0 + r < K) cst[k0 + r] -= 0.5f * v;
        }
    }
    for (int t = 0; t < T; ++t) {
        dec_copy_wait();                                   // this position's row
        __syncthreads();
        const unsigned char *sb = dsm + L.stage + (t & 1) * L.stage_bytes;
        const TI *xq = reinterpret_cast<const TI *>(sb);
        const TI *xk = reinterpret_cast<const TI *>(sb + L.kx);
        const TI *vv = reinterpret_cast<const TI *>(sb + L.vx);
        if (t + 1 < T) stage_row(t + 1);                   // the other buffer was last read before t's barrier
        // Eq. 16 (direct form): the key's and the query's scores against component k share its
        // loads; kDecRows components per warp at once, as for the precisions
        for (int k0 = warp * kDecRows; k0 < K; k0 += kDecWarps * kDecRows) {
            float aq[kDecRows], ak[kDecRows];
#pragma unroll
            for (int r = 0; r < kDecRows; ++r) aq[r] = ak[r] = 0.f;
            for (int j = lane; j < d; j += 32) {
                const float q = dec_load(xq, j), x = dec_load(xk, j);
#pragma unroll
                for (int r = 0; r < kDecRows; ++r) {
                    if (k0 + r < K) {
                        const size_t e = (size_t)(k0 + r) * d + j;
                        const float m = mus[e], l = lam[e];
                        const float dq = q - m, dk = x - m;
                        aq[r] = fmaf(dq * dq, l, aq[r]);
                        ak[r] = fmaf(dk * dk, l, ak[r]);
                    }
                }
            }
#pragma unroll
            for (int r = 0; r < kDecRows; ++r) {
                const float sq = warp_sum(aq[r]), sk = warp_sum(ak[r]);
                if (lane == 0 && k0 + r < K) {
                    gq[k0 + r] = cst[k0 + r] - 0.5f * sq;
                    gk[k0 + r] = cst[k0 + r] - 0.5f * sk;
                }
            }
        }
        __syncthreads();
        // Eq. 3b: the two softmaxes over components, a warp each
        if (warp == 0) warp_softmax(gq, K, lane);
        else if (warp == 1) warp_softmax(gk, K, lane);
        __syncthreads();
        // Eq. 6b: the prefix memory now includes position t; Eq. 8b: its read.  Thread (p, c)
        // updates column c over the p-th of P component ranges and keeps that range's
        // partial of the read; the partials are summed in range order below.
        for (int u = threadIdx.x; u < P * W; u += blockDim.x) {
            const int p = u / W, c = u - p * W;
            const int k1 = (int)((long)K * p / P), k2 = (int)((long)K * (p + 1) / P);
            const float vc = c < dv ? dec_load(vv, c) : 1.0f;
            float acc = 0.f;
            for (int k = k1; k < k2; ++k) {
                const float sv = fmaf(gk[k], vc, st[(size_t)k * W + c]);
                st[(size_t)k * W + c] = sv;
                acc = fmaf(gq[k], sv, acc);
            }
            num[u] = acc;
        }
        __syncthreads();
        float den = 0.f;
        for (int p = 0; p < P; ++p) den += num[p * W + dv];
        den += eps;
        const size_t row = (size_t)g * T + t;
        for (int c = threadIdx.x; c < dv; c += blockDim.x) {
            float nc = 0.f;
            for (int p = 0; p < P; ++p) nc += num[p * W + c];
            dec_store(out, row * dv + c, nc / den);
        }
    }
    // the state back to global memory: one bulk copy when both ends and the size allow (the
    // state's writers order their shared-memory stores before the copy's async-proxy reads)
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncthreads();
    const size_t sbytes = 4ull * K * W;
    if (((__cvta_generic_to_global(st_g) | sbytes) & 15) == 0) {
        if (threadIdx.x == 0) {
            asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(
                             __cvta_generic_to_global(st_g)),
                         "r"(dec_smem_u32(st)), "r"((uint32_t)sbytes)
                         : "memory");
            asm volatile("cp.async.bulk.commit_group;" ::: "memory");
            asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");   // smem stays valid until read
        }
    } else {
        for (int e = threadIdx.x; e < K * W; e += blockDim.x) st_g[e] = st[e];
    }
}

DecSmem decode_smem(const Problem &p, bool mu_in_smem) {
    return dec_smem(p.d, p.K, p.dv, p.in_dtype == GMA_BF16 ? 2 : 4, mu_in_smem);
}

template <typename TI, typename TO>
cudaError_t launch_decode(const Problem &p, const void *Qx, const void *Kx, const void *V, const float *mu,
                          const float *rho, const float *alpha, float *state, void *out, cudaStream_t s) {
    auto kern = decode_kernel<TI, TO>;
    const bool mu_in_smem = decode_smem(p, true).total <= kDecMaxSmem;
    const DecSmem L = decode_smem(p, mu_in_smem);
    cudaError_t e = set_dyn_smem(reinterpret_cast<const void *>(kern), (int)L.total);
    if (e != cudaSuccess) return e;
    kern<<<p.G, kDecThreads, L.total, s>>>(p.H, p.N, p.d, p.K, p.dv, p.eps, p.var_floor, L, mu_in_smem,
                                          static_cast<const TI *>(Qx), static_cast<const TI *>(Kx),
                                          static_cast<const TI *>(V), mu, rho, alpha, state,
                                          static_cast<TO *>(out));
    return cudaGetLastError();
}
}  // namespace

bool decode_supported(const Problem &p) { return decode_smem(p, false).total <= kDecMaxSmem; }

size_t decode_workspace(const Problem &) { return align_up(kHeaderBytes); }

cudaError_t decode_step(const Problem &p, const void *Qx, const void *Kx, const void *V, const float *mu,
                        const float *rho, const float *alpha, float *state, void *out, cudaStream_t s) {
    const bool bi = p.in_dtype == GMA_BF16, bo = p.out_dtype == GMA_BF16;
    if (bi && bo) return launch_decode<__nv_bfloat16, __nv_bfloat16>(p, Qx, Kx, V, mu, rho, alpha, state, out, s);
    if (bi) return launch_decode<__nv_bfloat16, float>(p, Qx, Kx, V, mu, rho, alpha, state, out, s);
    if (bo) return launch_decode<float, __nv_bfloat16>(p, Qx, Kx, V, mu, rho, alpha, state, out, s);
    return launch_decode<float, float>(p, Qx, Kx, V, mu, rho, alpha, state, out, s);
}

}  // namespace gma
