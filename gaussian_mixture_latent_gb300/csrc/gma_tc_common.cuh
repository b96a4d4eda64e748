// Shared pieces of the tensor-core kernels (bidirectional and causal):
// tile geometry, the per-head parameter block produced by tc_params, the
// conversion of a bf16 routing tile into the fp16 [x, x^2/256] MMA operand,
// the row softmax helpers, wind-down waits, and host-side TMA descriptors.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "gma_internal.h"
#include "gma_sm100.cuh"

namespace gma {
namespace tc {

using namespace sm100;

constexpr int TM = 128;            // rows per tile
constexpr int DR = 64;             // routing dimension handled by this path
constexpr int DVV = 64;            // value dimension handled by this path
constexpr int kWgThreads = 128;
constexpr float kLog2e = 1.4426950408889634f;
constexpr uint32_t kTileBytes = TM * 128;   // one 128-row x 128-byte swizzled tile

__host__ __device__ constexpr uint32_t align1k(uint32_t x) { return (x + 1023u) & ~1023u; }

// Per-head parameter block written by tc_params, all fp16 MMA B operands:
//   W chunk 0 (K x 128 B, 128-byte swizzle): linear coefficients
//   W chunk 1 (K x 128 B, 128-byte swizzle): quadratic coefficients
//   Wc        (K x 32 B, no swizzle): [c_hi, c_lo, 0...] so that the constant
//             k-step [1, 1, 0...] adds c_k exactly to ~22 bits
//   scale     f32 (+ pad): the power of two W was divided by
__host__ __device__ constexpr uint32_t param_wc_off(int K) { return 256u * K; }
__host__ __device__ constexpr uint32_t param_scale_off(int K) { return 288u * K; }
__host__ __device__ constexpr uint32_t param_bytes(int K) { return 288u * K + 16u; }
constexpr uint32_t kConstABytes = TM * 32;   // [1, 1, 0 x 14] fp16 for every tile row, no swizzle

// Byte offset of fp16 element (row, col < 16) in a no-swizzle K-major block of
// 16-column rows: 8-row x 16-byte core matrices, column halves 128 B apart,
// 8-row groups 256 B apart.
__host__ __device__ constexpr uint32_t nosw16_off(uint32_t row, uint32_t col) {
    return (row >> 3) * 256u + (col >> 3) * 128u + (row & 7u) * 16u + (col & 7u) * 2u;
}
// Per-head read operand: ceil(K/64) chunks of 80 rows x 128 B.
__host__ __device__ constexpr uint32_t mem_bytes(int K) { return (uint32_t)((K + 63) / 64) * 80u * 128u; }

// Walks the CTA's tiles in steps of `step` without dividing inside the loop:
// i = local tile index, g = head, j = tile within the head, hl = g - first head;
// slot() = the unit whose sum the tile belongs to (its head).
struct TileCursor {
    int i, g, j, hl, T, n, step;
    __device__ TileCursor(int t0, int n_, int T_, int start, int step_) : T(T_), n(n_), step(step_) {
        i = start;
        g = (t0 + start) / T_;
        j = (t0 + start) - g * T_;
        hl = g - t0 / T_;
    }
    __device__ bool valid() const { return i < n; }
    __device__ bool first() const { return j == 0 || i == 0; }
    __device__ bool last() const { return j == T - 1 || i == n - 1; }
    __device__ int slot() const { return g; }
    __device__ void next() {
        i += step;
        j += step;
        while (j >= T) { j -= T; ++g; ++hl; }
    }
};

// The same walk over the prefix segments of a segment-parallel causal scan: the CTA's
// range of the concatenated segments (segment v = chunks [a, a + len) of head g), from
// the start the plan recorded for it.  j = chunk within the head, hl = v - first
// segment, slot() = v.
struct SegCursor {
    const SegTable *S;
    int i, g, j, hl, n, step, v, jj;
    __device__ SegCursor(const SegTable *S_, int cta, int n_, int start, int step_) : S(S_), n(n_), step(step_) {
        v = S->pre_v[cta];
        jj = S->pre_jj[cta];
        i = start;
        hl = 0;
        jj += start;
        settle();
    }
    __device__ void settle() {
        while (v < S->nseg && jj >= S->seg[v].len) { jj -= S->seg[v].len; ++v; ++hl; }
        if (v < S->nseg) { g = S->seg[v].g; j = S->seg[v].a + jj; }
    }
    __device__ bool valid() const { return i < n; }
    __device__ bool first() const { return jj == 0 || i == 0; }
    __device__ bool last() const { return jj == S->seg[v].len - 1 || i == n - 1; }
    __device__ int slot() const { return v; }
    __device__ void next() {
        i += step;
        jj += step;
        settle();
    }
};

// The segment table as a kernel parameter of the kernels that walk it (an empty
// struct for the others).
struct NoSeg {};
template <bool SEG> struct SegArg { using type = NoSeg; };
template <> struct SegArg<true> { using type = SegTable; };

// ------------------------------------------------------------------ wind-down helpers

// Bounded wait that runs to completion (or its time limit) even after another
// thread raised the CTA's abort flag: used before the CTA releases shared memory
// or TMEM that in-flight copies or MMAs still touch.
__device__ __forceinline__ void wait_ignoring_abort(uint64_t *bar, uint32_t parity, unsigned *status) {
    int never = 0;
    mbar_wait(bar, parity, Abort{&never, status}, kDevErrTimeout);
}

// Every TMA load issued into an S-stage ring has landed: waits for the last
// fill of each stage (fills are issued round-robin, so that is the newest phase).
__device__ __forceinline__ void wind_down_ring(uint64_t *full, int S, int issued, unsigned *status) {
    for (int i = issued > S ? issued - S : 0; i < issued; ++i) wait_ignoring_abort(&full[i % S], (i / S) & 1, status);
}

// ------------------------------------------------------------------ compute helpers
//
// A compute warpgroup is four consecutive warps; thread r of the group owns
// tile row r (= TMEM lane r): warp w may access TMEM lanes 32*(w % 4) ... +31.

struct RowThread {
    uint32_t r;          // tile row = TMEM lane
    uint32_t lane_off;   // TMEM lane field of this warp
    int wg;              // compute warpgroup
    int wtid;            // 0..127 inside the group
};

// Named barrier 1 + wg synchronises one 128-thread compute warpgroup.
__device__ __forceinline__ bool wg_all(const RowThread &t, bool v) { return group_all(v, 1 + t.wg, kWgThreads); }
__device__ __forceinline__ void wg_sync(const RowThread &t) { group_sync(1 + t.wg, kWgThreads); }

// Convert a bf16 row (128 B, swizzled) into the fp16 [x, x^2/256] row of the
// log-density A operand in TMEM (columns 0-31: x pairs, 32-63: x^2/256 pairs).
__device__ __forceinline__ void convert_row(const uint8_t *xs, uint32_t r, uint32_t tcol_a) {
    uint32_t px[32], pq[32];
    const uint64_t k16 = f2_pack(0.0625f, 0.0625f);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const uint4 v = *reinterpret_cast<const uint4 *>(xs + sw128_off(r, j));
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const float lo = bf16_lo(w[u]), hi = bf16_hi(w[u]);
            px[4 * j + u] = pack_f16(lo, hi);
            const uint64_t y = f2_mul(f2_pack(lo, hi), k16);   // x / 16, exact
            float qa, qb;
            f2_unpack(f2_mul(y, y), qa, qb);                   // x^2 / 256
            pq[4 * j + u] = pack_f16(qa, qb);
        }
    }
    tmem_st32(tcol_a, px);
    tmem_st32(tcol_a + 32, pq);
}

// One out-of-line copy of convert_row, for kernels that convert in more than
// one warp role or at more than one site (keeps their code footprint small).
static __device__ __noinline__ void convert_row_call(const uint8_t *xs, uint32_t r, uint32_t tcol_a) {
    convert_row(xs, r, tcol_a);
}

// The constant A block of the log-density MMA: row r = [1, 1, 0 x 14] (fp16).
__device__ __forceinline__ void init_const_a(uint8_t *blk, int tid, int nthreads) {
    for (int e = tid; e < (int)(kConstABytes / 16); e += nthreads) {
        const uint32_t off = (uint32_t)e * 16u;
        const bool first_half = ((off >> 7) & 1u) == 0;          // column half 0 holds columns 0..7
        reinterpret_cast<uint4 *>(blk)[e] = make_uint4(first_half ? 0x3C003C00u : 0u, 0u, 0u, 0u);
    }
}

// Issue the log-density MMA of one 128-row tile:  D = [x, x^2/256] . W^T + [1, 1] . [c_hi, c_lo]^T.
// a_tmem holds [x, x^2/256] (64 columns of fp16 pairs); pblk / consta are shared addresses.
template <int K>
__device__ __forceinline__ void issue_logdensity(uint32_t d_tmem, uint32_t a_tmem, uint32_t pblk, uint32_t consta) {
    constexpr uint32_t idesc = idesc_f16(0, 0, 0, 0, TM, K);
    const uint64_t wd = sdesc_sw128(pblk, 16, 1024);
#pragma unroll
    for (int ks = 0; ks < 8; ++ks)
        mma_ts(d_tmem, a_tmem + ks * 8, wd + (uint64_t)(((ks >> 2) * 128u * K + (ks & 3) * 32u) >> 4), idesc, ks > 0);
    mma_ss(d_tmem, sdesc_none(consta, 128, 256), sdesc_none(pblk + param_wc_off(K), 128, 256), idesc, 1);
}

// The log-density MMA of part `part` of NP components (components NP part ..
// NP part + NP - 1) of a K-component head: N = NP columns at d_tmem.  Each score
// is the same dot product as in the full-width MMA above.
template <int K, int NP>
__device__ __forceinline__ void issue_logdensity_part(uint32_t d_tmem, uint32_t a_tmem, uint32_t pblk, uint32_t consta,
                                                      int part) {
    static_assert(NP % 32 == 0 && K % NP == 0, "parts of 32 or 64 components");
    constexpr uint32_t idesc = idesc_f16(0, 0, 0, 0, TM, NP);
    const uint64_t wd = sdesc_sw128(pblk + (uint32_t)part * NP * 128u, 16, 1024);
#pragma unroll
    for (int ks = 0; ks < 8; ++ks)
        mma_ts(d_tmem, a_tmem + ks * 8, wd + (uint64_t)(((ks >> 2) * 128u * K + (ks & 3) * 32u) >> 4), idesc, ks > 0);
    mma_ss(d_tmem, sdesc_none(consta, 128, 256),
           sdesc_none(pblk + param_wc_off(K) + nosw16_off((uint32_t)(NP * part), 0), 128, 256), idesc, 1);
}

// A row's scores in two parts of NP through one NP-column TMEM region.
// Part 0: e_a = 2^(scale * (d - m_a)) as NP/2 bf16 pairs; returns m_a, the part's maximum.
template <int NP>
__device__ __forceinline__ float row_exp_part0(uint32_t taddr, float scale, uint32_t (&e)[NP / 2]) {
    uint32_t d[NP];
#pragma unroll
    for (int cc = 0; cc < NP / 32; ++cc) tmem_ld32(taddr + 32 * cc, d + 32 * cc);
    tmem_ld_wait();
    float m[4] = {__uint_as_float(d[0]), __uint_as_float(d[1]), __uint_as_float(d[2]), __uint_as_float(d[3])};
#pragma unroll
    for (int t = 4; t < NP; t += 4) {
        m[0] = fmaxf(m[0], __uint_as_float(d[t]));
        m[1] = fmaxf(m[1], __uint_as_float(d[t + 1]));
        m[2] = fmaxf(m[2], __uint_as_float(d[t + 2]));
        m[3] = fmaxf(m[3], __uint_as_float(d[t + 3]));
    }
    const float mx = fmaxf(fmaxf(m[0], m[1]), fmaxf(m[2], m[3]));
    const uint64_t sc2 = f2_pack(scale, scale), nm2 = f2_pack(-mx * scale, -mx * scale);
#pragma unroll
    for (int t = 0; t < NP; t += 2) {
        float a, b;
        f2_unpack(f2_fma(f2_pack(__uint_as_float(d[t]), __uint_as_float(d[t + 1])), sc2, nm2), a, b);
        e[t / 2] = pack_bf16(ex2_approx(a), ex2_approx(b));
    }
    return mx;
}

// Part 1: with m = max(m_a, m_b), e_b = 2^(scale * (d - m)); where m_b > m_a the
// part-0 values are brought to the common offset by one more factor
// 2^(scale * (m_a - m)) <= 1 (a second bf16 rounding, 2^-9 relative, on those only).
// Two passes over the region, 32 scores live at a time (the part-0 values are live too).
template <int NP>
__device__ __forceinline__ void row_exp_part1(uint32_t taddr, float scale, float ma, uint32_t (&ea)[NP / 2],
                                              uint32_t (&eb)[NP / 2]) {
    float m[4] = {ma, ma, ma, ma};
#pragma unroll
    for (int h = 0; h < NP / 32; ++h) {
        uint32_t d[32];
        tmem_ld32(taddr + 32 * h, d);
        tmem_ld_wait();
#pragma unroll
        for (int t = 0; t < 32; t += 4) {
            m[0] = fmaxf(m[0], __uint_as_float(d[t]));
            m[1] = fmaxf(m[1], __uint_as_float(d[t + 1]));
            m[2] = fmaxf(m[2], __uint_as_float(d[t + 2]));
            m[3] = fmaxf(m[3], __uint_as_float(d[t + 3]));
        }
    }
    const float mx = fmaxf(fmaxf(m[0], m[1]), fmaxf(m[2], m[3]));
    const uint64_t sc2 = f2_pack(scale, scale), nm2 = f2_pack(-mx * scale, -mx * scale);
#pragma unroll
    for (int h = 0; h < NP / 32; ++h) {
        uint32_t d[32];
        tmem_ld32(taddr + 32 * h, d);
        tmem_ld_wait();
#pragma unroll
        for (int t = 0; t < 32; t += 2) {
            float a, b;
            f2_unpack(f2_fma(f2_pack(__uint_as_float(d[t]), __uint_as_float(d[t + 1])), sc2, nm2), a, b);
            eb[16 * h + t / 2] = pack_bf16(ex2_approx(a), ex2_approx(b));
        }
    }
    if (mx > ma) {
        const float f = ex2_approx(fmaf(ma, scale, -mx * scale));
        const uint64_t f2 = f2_pack(f, f);
#pragma unroll
        for (int t = 0; t < NP / 2; ++t) {
            float a, b;
            f2_unpack(f2_mul(f2_pack(bf16_lo(ea[t]), bf16_hi(ea[t])), f2), a, b);
            ea[t] = pack_bf16(a, b);
        }
    }
}

// e = 2^(scale * (d - max d)) for the K raw scores d of this thread's row in
// TMEM (one round trip), as K/2 bf16 pairs.  scale > 0, so max commutes with it.
// The exponent stays in fp32 and only the result is rounded to bf16, so every e
// carries a relative error of at most 2^-9.  (Rounding the argument to bf16
// first would cost ln2 * |arg| * 2^-9 relative: about 2% at arg = -20, which
// shows in causal rows whose query routing barely overlaps the prefix keys,
// where the output is a ratio of such tail probabilities.)
template <int K>
__device__ __forceinline__ void row_exp_scaled(uint32_t taddr, float scale, uint32_t (&e)[K / 2]) {
    uint32_t d[K];
#pragma unroll
    for (int cc = 0; cc < K / 32; ++cc) tmem_ld32(taddr + 32 * cc, d + 32 * cc);
    tmem_ld_wait();
    float m[4] = {__uint_as_float(d[0]), __uint_as_float(d[1]), __uint_as_float(d[2]), __uint_as_float(d[3])};
#pragma unroll
    for (int t = 4; t + 8 <= K; t += 8) {
        m[0] = max3(m[0], __uint_as_float(d[t]), __uint_as_float(d[t + 1]));
        m[1] = max3(m[1], __uint_as_float(d[t + 2]), __uint_as_float(d[t + 3]));
        m[2] = max3(m[2], __uint_as_float(d[t + 4]), __uint_as_float(d[t + 5]));
        m[3] = max3(m[3], __uint_as_float(d[t + 6]), __uint_as_float(d[t + 7]));
    }
    m[0] = max3(m[0], __uint_as_float(d[K - 4]), __uint_as_float(d[K - 3]));
    m[1] = max3(m[1], __uint_as_float(d[K - 2]), __uint_as_float(d[K - 1]));
    const float mx = fmaxf(max3(m[0], m[1], m[2]), m[3]);
    const uint64_t sc2 = f2_pack(scale, scale), nm2 = f2_pack(-mx * scale, -mx * scale);
#pragma unroll
    for (int t = 0; t < K; t += 2) {
        float a, b;
        f2_unpack(f2_fma(f2_pack(__uint_as_float(d[t]), __uint_as_float(d[t + 1])), sc2, nm2), a, b);
        e[t / 2] = pack_bf16(ex2_approx(a), ex2_approx(b));
    }
}

// e = 2^(scale * d - off) for the K raw scores d of this thread's row (one TMEM
// round trip), as K/2 bf16 pairs: the same rounding as row_exp_scaled, with the
// row's offset (its maximum or log-sum-exp over a wider component set) given.
template <int K>
__device__ __forceinline__ void row_exp_offset(uint32_t taddr, float scale, float off, uint32_t (&e)[K / 2]) {
    uint32_t d[K];
#pragma unroll
    for (int cc = 0; cc < K / 32; ++cc) tmem_ld32(taddr + 32 * cc, d + 32 * cc);
    tmem_ld_wait();
    const uint64_t sc2 = f2_pack(scale, scale), no2 = f2_pack(-off, -off);
#pragma unroll
    for (int t = 0; t < K; t += 2) {
        float a, b;
        f2_unpack(f2_fma(f2_pack(__uint_as_float(d[t]), __uint_as_float(d[t + 1])), sc2, no2), a, b);
        e[t / 2] = pack_bf16(ex2_approx(a), ex2_approx(b));
    }
}

// ------------------------------------------------------------------ parameter block
//
// The per-head parameter block of the log-density MMA ("Gaussian Mixture
// Attention", section 3.6 Eq. 14-15 and section 4.1 Eq. 16): variances
// var = softplus(rho) + var_floor, log priors log_softmax(alpha), and in log2
// units the linear coefficients mu * lambda, the quadratic coefficients
// -lambda / 2 centred over the components (a per-column shift common to every
// component cancels in the softmax) and rescaled for the x^2 / 256 operand, and
// the per-component constant c_k.  Everything is divided by one power-of-two
// scale so that the fp16 operands keep their range.  Written to `blk`:
//   [0, 128 K)          linear coefficients, fp16, K-major 128-byte swizzle
//   [128 K, 256 K)      quadratic coefficients, same layout
//   [256 K, 288 K)      [c_hi, c_lo, 0 x 14] per component (fp16, no swizzle)
//   [288 K, 288 K + 4)  the scale (fp32)
//
// Built by a team of NT threads (a multiple of 32) with team index `tid`:
// thread tid owns float4 e4 = tid + u NT (u < V4) of the head's [K][d] arrays,
// i.e. component e4 / 16 and columns 4 (e4 % 16) .. + 3, and keeps its
// coefficients in registers until it writes them.  The loads are issued first
// (ParamLoads), so a kernel can put them in flight before its own prologue.
// `sync` is a barrier over the team; `scratch` holds param_scratch_floats(K, NT)
// floats.  Every reduction has a fixed order for a given NT.
__host__ __device__ constexpr int param_scratch_floats(int K, int NT) { return 64 + (NT / 32) * DR + K; }

template <int K, int NT>
struct ParamLoads {
    static constexpr int n4 = K * DR / 4;
    static constexpr int V4 = (n4 + NT - 1) / NT;
    float4 mv[V4], rv[V4];
    float alk;
    __device__ __forceinline__ void issue(int tid, const float *__restrict__ mu_h, const float *__restrict__ rho_h,
                                          const float *__restrict__ al) {
        const float4 *mu4 = reinterpret_cast<const float4 *>(mu_h);
        const float4 *rho4 = reinterpret_cast<const float4 *>(rho_h);
#pragma unroll
        for (int u = 0; u < V4; ++u) {
            const int e4 = tid + u * NT;
            if (e4 < n4) { mv[u] = __ldg(mu4 + e4); rv[u] = __ldg(rho4 + e4); }
        }
        alk = tid < K ? __ldg(al + tid) : -INFINITY;
    }
};

template <int K, int NT, class Sync>
__device__ __forceinline__ void build_param_block(int tid, const ParamLoads<K, NT> &ld, float var_floor,
                                                  uint8_t *blk, float *scratch, Sync sync) {
    static_assert(NT % 32 == 0 && NT / 32 <= 32 && K <= NT && K % 2 == 0, "team size");
    constexpr int NWT = NT / 32, n4 = ParamLoads<K, NT>::n4, V4 = ParamLoads<K, NT>::V4;
    float *red = scratch;                 // [64]: two reductions of NWT warps each
    float *colpart = red + 64;            // [NWT][DR]: per-warp column sums of the quadratic coefficients
    float *cbuf = colpart + NWT * DR;     // [K]: per-component constants
    const int warp = tid >> 5, lane = tid & 31, j = tid & 15;   // j: this thread's column group
    if (tid < K) cbuf[tid] = ld.alk;                            // alpha_k, replaced by c_k below

    // log-sum-exp of the prior logits (Eq. 15)
    float m = ld.alk;
    for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(~0u, m, o));
    if (lane == 0) red[warp] = m;
    sync();
    m = red[0];
    for (int w = 1; w < NWT; ++w) m = fmaxf(m, red[w]);
    float s = tid < K ? expf(ld.alk - m) : 0.f;
    for (int o = 16; o; o >>= 1) s += __shfl_xor_sync(~0u, s, o);
    sync();                                                     // every thread has read red[]
    if (lane == 0) red[warp] = s;
    sync();
    s = 0.f;
    for (int w = 0; w < NWT; ++w) s += red[w];
    const float lse = m + logf(s);

    // Eq. 14: variances; linear and quadratic coefficients in log2 units.  The 16
    // threads sharing component k (aligned, consecutive) also reduce sum_m log var_km
    // and sum_m mu_km^2 lambda_km for the constant c_k (Eq. 16).
    float av[V4][4], bq[V4][4];
    float colacc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int u = 0; u < V4; ++u) {
        if (u * NT >= n4) break;                                // uniform across the team
        const int e4 = tid + u * NT;
        const bool valid = e4 < n4;
        const float mq[4] = {ld.mv[u].x, ld.mv[u].y, ld.mv[u].z, ld.mv[u].w};
        const float rq[4] = {ld.rv[u].x, ld.rv[u].y, ld.rv[u].z, ld.rv[u].w};
        float logdet = 0.f, musq = 0.f;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            // SFU forms (relative error near 2^-21): the coefficients are rounded to
            // fp16 (2^-12) and the constant to about 22 bits afterwards
            const float w = rq[q];
            const float var = fmaxf(w, 0.f) + __logf(1.0f + __expf(-fabsf(w))) + var_floor;
            const float lam = __frcp_rn(var);
            av[u][q] = valid ? mq[q] * lam * kLog2e : 0.f;
            bq[u][q] = valid ? -0.5f * lam * kLog2e : 0.f;
            logdet += valid ? __logf(var) : 0.f;
            musq += valid ? mq[q] * av[u][q] : 0.f;
            colacc[q] += bq[u][q];
        }
        for (int o = 1; o < 16; o <<= 1) {
            logdet += __shfl_xor_sync(~0u, logdet, o);
            musq += __shfl_xor_sync(~0u, musq, o);
        }
        if (valid && j == 0) {
            const int k = e4 >> 4;
            cbuf[k] = (cbuf[k] - lse) * kLog2e - 0.5f * kLog2e * logdet - 0.5f * musq;
        }
    }
    // column sums over this warp's components: lanes l and l ^ 16 share the columns
#pragma unroll
    for (int q = 0; q < 4; ++q) colacc[q] += __shfl_xor_sync(~0u, colacc[q], 16);
    if (lane < 16)
        *reinterpret_cast<float4 *>(colpart + warp * DR + 4 * j) = make_float4(colacc[0], colacc[1], colacc[2], colacc[3]);
    sync();
    // column means (fixed warp order), centred and rescaled quadratic coefficients, max |W|
    float cm[4] = {0.f, 0.f, 0.f, 0.f};
    for (int w = 0; w < NWT; ++w) {
        const float4 p = *reinterpret_cast<const float4 *>(colpart + w * DR + 4 * j);
        cm[0] += p.x; cm[1] += p.y; cm[2] += p.z; cm[3] += p.w;
    }
    float amax = 0.f, cmax = 0.f;
#pragma unroll
    for (int u = 0; u < V4; ++u) {
        if (u * NT >= n4) break;
        const bool valid = tid + u * NT < n4;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            bq[u][q] = valid ? (bq[u][q] - cm[q] / (float)K) * 256.0f : 0.f;
            amax = fmaxf(amax, fmaxf(fabsf(av[u][q]), fabsf(bq[u][q])));
        }
    }
    for (int k = tid; k < K; k += NT) cmax = fmaxf(cmax, fabsf(cbuf[k]));
    for (int o = 16; o; o >>= 1) {
        amax = fmaxf(amax, __shfl_xor_sync(~0u, amax, o));
        cmax = fmaxf(cmax, __shfl_xor_sync(~0u, cmax, o));
    }
    if (lane == 0) { red[warp] = amax; red[32 + warp] = cmax; }
    sync();
    amax = 0.f;
    cmax = 0.f;
    for (int w = 0; w < NWT; ++w) { amax = fmaxf(amax, red[w]); cmax = fmaxf(cmax, red[32 + w]); }
    // power-of-two scale: max |W| / scale <= 2^14 and max |c| / scale <= 2^15 (fp16 range)
    int ex = 0;
    if (amax > 0.f && isfinite(amax)) ex = (int)ceilf(log2f(amax)) - 14;
    if (cmax > 0.f && isfinite(cmax)) ex = max(ex, (int)ceilf(log2f(cmax)) - 15);
    const float inv = exp2f((float)-ex);
    if (tid == 0) *reinterpret_cast<float *>(blk + param_scale_off(K)) = exp2f((float)ex);
    // Wc: [c_hi, c_lo, 0 x 14] per component, c_hi + c_lo = c / scale to about 22 bits
    for (int e = tid; e < K * 2; e += NT) {
        const int k = e >> 1, half = e & 1;
        uint4 v = make_uint4(0, 0, 0, 0);
        if (half == 0) {
            const float cs = cbuf[k] * inv;
            const float hi = __half2float(__float2half_rn(cs));
            v.x = pack_f16(hi, cs - hi);
        }
        *reinterpret_cast<uint4 *>(blk + param_wc_off(K) + nosw16_off(k, 8 * half)) = v;
    }
    // fp16 W from registers, K-major 128-byte swizzle: row k, 8-element chunk, element
#pragma unroll
    for (int u = 0; u < V4; ++u) {
        const int e4 = tid + u * NT;
        if (u * NT >= n4) break;
        if (e4 >= n4) continue;
        const int k = e4 >> 4, m0 = 4 * j;
        const uint32_t off = sw128_off(k, m0 >> 3) + (m0 & 7) * 2;
        *reinterpret_cast<uint2 *>(blk + off) =
            make_uint2(pack_f16(av[u][0] * inv, av[u][1] * inv), pack_f16(av[u][2] * inv, av[u][3] * inv));
        *reinterpret_cast<uint2 *>(blk + 128u * K + off) =
            make_uint2(pack_f16(bq[u][0] * inv, bq[u][1] * inv), pack_f16(bq[u][2] * inv, bq[u][3] * inv));
    }
}

// Per-head scale of the coefficient matrix, read from the parameter block in global memory.
__device__ __forceinline__ float head_scale(const uint8_t *params, uint32_t stride, int h, int K) {
    return __ldg(reinterpret_cast<const float *>(params + (size_t)h * stride + param_scale_off(K)));
}

// ------------------------------------------------------------------ host helpers

using EncodeTiled = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                 const cuuint64_t *, const cuuint32_t *, const cuuint32_t *,
                                 CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                 CUtensorMapFloatOOBfill);

inline EncodeTiled encode_fn() {
    static EncodeTiled fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiled>(p);
    });
    return fn;
}

// 3D bf16 tensor map over [G][N][width], box [1][box_rows][64], 128-byte swizzle.
inline bool make_map(CUtensorMap *m, const void *base, int G, int N, int width, int box_rows = TM) {
    EncodeTiled enc = encode_fn();
    if (!enc) return false;
    const cuuint64_t dims[3] = {(cuuint64_t)width, (cuuint64_t)N, (cuuint64_t)G};
    const cuuint64_t strides[2] = {(cuuint64_t)width * 2, (cuuint64_t)width * 2 * N};
    const cuuint32_t box[3] = {64, (cuuint32_t)box_rows, 1};
    const cuuint32_t es[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Launch `kern` as a programmatic dependent of the previous kernel in the stream:
// its CTAs may start while that kernel drains, and every read of that kernel's
// results sits behind grid_dep_wait() in the device code.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_dependent(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                                    Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

inline int sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return n;
}

}  // namespace tc
}  // namespace gma
