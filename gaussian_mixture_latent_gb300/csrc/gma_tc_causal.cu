// Tensor-core (tcgen05) causal GMA forward as a chunked scan, for bf16 inputs
// and outputs, d = 64, dv = 64, K = 64.
//
// "Gaussian Mixture Attention" (Huang & Raza, 2026), section 3.5: prefix
// memories over j <= i (Eq. 6b) read by each position (Eq. 8b), equivalently
// the masked affinity of Eq. 9b-10b.  Positions are processed in chunks of
// 128 rows; for chunk c with rows i, j inside the chunk:
//
//   e^Q_i      = 2^(s_i - max s_i)      unnormalised query responsibilities
//   gamma^K_j  = softmax(s_j)           key responsibilities (Eq. 3b)
//   T_ij       = [j <= i] e^Q_i . gamma^K_j                  (intra-chunk, Eq. 9b)
//   num_i      = e^Q_i S_{c-1} + sum_j T_ij V_j
//   den_i      = e^Q_i z_{c-1} + sum_j T_ij + eps * sum_k e^Q_ik
//   O_i        = num_i / den_i
//   [S | z]_c  = [S | z]_{c-1} + gamma^K^T [V | 1]           (state after the chunk)
//
// The unnormalised e^Q scales numerator and denominator by the same factor,
// so only eps needs sum_k e^Q_ik.  The state [S | z]^T accumulates in TMEM in
// fp32 and is snapshotted as a bf16 MMA operand once per chunk; the read's
// operands carry a column of ones, so the same MMAs give the numerator, the
// denominator and sum_k e^Q_ik.  Every reduction has a fixed order, so results are bitwise
// reproducible, and row i never reads rows after i (the mask selects, it does
// not multiply).
//
// One CTA per head, and the forward is this one kernel: the three compute groups
// first build the head's parameter block (Eq. 14-16, the same code as tc_params)
// in shared memory while the first tiles load.  Warps: 0 TMA producer; 1 TMEM
// owner and issuer of the log-density MMAs (keys, then queries); 2 issuer of the
// T MMAs; 3 issuer of the state update and the read; 4-7 key group (convert,
// softmax, state snapshot); 8-11 query group (convert, exp, epilogue); 12-15
// mask group.
//
// The stages of consecutive chunks overlap: e^Q has two TMEM buffers, so the
// queries of chunk c + 1 are ready before chunk c is read (the keys and queries
// share one TMEM region for the log-density operand, converted in turn); T is formed in two
// 64-key halves through one TMEM buffer, and the first half of T(c + 1) enters
// the tensor pipe as soon as the second half of T(c) has been loaded into
// registers; each masked bf16 half has its own shared-memory slot, and the read
// consumes the halves one at a time as the mask group fills them, so the mask
// of chunk c + 1 waits only for the read of the same half of chunk c.  Outputs
// leave through a staging tile by TMA, one 32-row box per warp.  Handoffs
// between warps are mbarriers with one arrival per warp.  Every mbarrier wait
// is bounded; a timeout posts GMA_ERR_TIMEOUT.
#include <cuda.h>
#include <cuda_bf16.h>

#include "gma_internal.h"
#include "gma_sm100.cuh"
#include "gma_tc_common.cuh"

namespace gma {

using namespace sm100;
using namespace tc;

namespace {

constexpr int KC = 64;                 // components handled by this kernel
constexpr int kCThreads = 512;         // 16 warps
constexpr int kWProd = 0, kWIss1 = 1, kWIssT = 2, kWIssR = 3, kWGroups = 4;

struct CausalArgs {
    int G, H, N, nch;
    const uint8_t *params;
    uint32_t param_stride;
    float eps;
    unsigned *status;
    // component-sliced form (larger K or dv): this CTA takes components [64 s, 64 s + 64) of a
    // Kfull-component head and value columns [64 t, 64 t + 64) of a dvt-wide V
    int Kfull, dvt;
    const float *mrow_q;   // [G][N] max_k scores of each query row (log2 units, scaled)
    const float *lse_k;    // [G][N] log2 sum_k 2^score of each key row
    uint16_t *pnum;        // [ns][G][N][dvt] bf16 partial numerators
    float *pden;           // [ns][G][N] partial denominators
    // one head per CTA: the CTA builds its head's parameter block from these
    const float *mu, *rho, *alpha;   // [H][K][d], [H][K][d], [H][K]
    float var_floor;
};

struct CausalCfg {
    static constexpr uint32_t PB = align1k(param_bytes(KC));
    static constexpr uint32_t SBB = 80u * 128u;                        // state operand [S^T | z | 1 | 0...] bf16
    static constexpr uint32_t OFF_Q = 0;                               // 2 stages
    static constexpr uint32_t OFF_K = OFF_Q + 2 * kTileBytes;          // 2 stages
    static constexpr uint32_t OFF_V = OFF_K + 2 * kTileBytes;          // 2 stages
    static constexpr uint32_t OFF_ONES = OFF_V + 2 * kTileBytes;       // after the V stages (positive LBO)
    static constexpr uint32_t OFF_G = OFF_ONES + kTileBytes;           // gamma^K [row][k]
    static constexpr uint32_t OFF_TB = OFF_G + kTileBytes;             // masked T halves, bf16 [row][key], 2 slots
    static constexpr uint32_t OFF_O = OFF_TB + 2 * kTileBytes;         // output staging, a 32-row quarter per warp
    static constexpr uint32_t OFF_SB = OFF_O + kTileBytes;             // state operand, 2 buffers
    static constexpr uint32_t OFF_P = OFF_SB + 2 * SBB;
    static constexpr uint32_t OFF_CA = OFF_P + PB;                     // constant [1, 1, 0...] A block
    static constexpr uint32_t OFF_BAR = OFF_CA + kConstABytes;
    static constexpr uint32_t BYTES = OFF_BAR + 1024 + 1024;
    // TMEM columns
    static constexpr uint32_t COL_A = 0;                               // [x, x^2/256] of keys, then queries
    static constexpr uint32_t COL_D1Q = 64, COL_D1K = 128;             // log-density scores (fp32)
    static constexpr uint32_t COL_T = 192;                             // one 64-key half of T (fp32)
    static constexpr uint32_t COL_D3 = 256;                            // read result [num | den | sum e^Q], 80
    static constexpr uint32_t COL_S = 384;                             // [S | z]^T state, 64 columns
    static constexpr uint32_t COL_EQ = 448;                            // e^Q as bf16 pairs, 2 x 32 columns
    static constexpr uint32_t TMEM_COLS = 512;
};
static_assert(CausalCfg::OFF_SB % 1024 == 0 && CausalCfg::OFF_P % 1024 == 0 && CausalCfg::OFF_TB % 1024 == 0 &&
                  CausalCfg::OFF_O % 1024 == 0,
              "operand blocks must be 1024-byte aligned");
static_assert(CausalCfg::BYTES <= 232448, "causal kernel exceeds the shared-memory opt-in limit");
static_assert(param_scratch_floats(KC, 3 * kWgThreads) * 4 <= (int)kTileBytes,
              "the parameter build's scratch must fit the gamma buffer");

// The parameter build as one out-of-line call, keeping it out of the compute groups' loop code.
static __device__ __noinline__ void build_param_block_team(int tid, ParamLoads<KC, 3 * kWgThreads> ld, float var_floor,
                                                           uint8_t *blk, float *scratch) {
    build_param_block<KC, 3 * kWgThreads>(tid, ld, var_floor, blk, scratch, [] { group_sync(4, 3 * kWgThreads); });
}

// One 32-key group of a masked T row into the bf16 slot: copied whole below the
// diagonal (diag = false) or selected j <= row on it (diag = true: keys key0 + u
// with u <= lane).  Groups above the diagonal are never written: those entries
// of the slot stay zero from the kernel's start.
__device__ __forceinline__ void mask_group(const uint32_t (&v)[32], bool diag, int lane, uint8_t *slot, uint32_t r,
                                           int cc) {
    uint32_t pk[16];
#pragma unroll
    for (int t = 0; t < 16; ++t) {
        float a = __uint_as_float(v[2 * t]), b = __uint_as_float(v[2 * t + 1]);
        if (diag) {
            a = 2 * t <= lane ? a : 0.f;
            b = 2 * t + 1 <= lane ? b : 0.f;
        }
        pk[t] = pack_bf16(a, b);
    }
#pragma unroll
    for (int q4 = 0; q4 < 4; ++q4)
        *reinterpret_cast<uint4 *>(slot + sw128_off(r, cc * 4 + q4)) =
            make_uint4(pk[4 * q4], pk[4 * q4 + 1], pk[4 * q4 + 2], pk[4 * q4 + 3]);
}

// 2^(scale * d - off) in fp32 for the K raw scores d of this thread's row in TMEM
// (one round trip), with off = scale * max_k d (OFFSET = false) or given; returns
// the fp32 sum of the K values.  The exponent is evaluated in fp32 and a caller
// rounds each result once, to bf16, for the MMA.
template <int K, bool OFFSET>
__device__ __forceinline__ float row_exp2(uint32_t taddr, float scale, float off, float (&x)[K]) {
    uint32_t d[K];
#pragma unroll
    for (int cc = 0; cc < K / 32; ++cc) tmem_ld32(taddr + 32 * cc, d + 32 * cc);
    tmem_ld_wait();
    if (!OFFSET) {
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
        off = fmaxf(max3(m[0], m[1], m[2]), m[3]) * scale;
    }
    const uint64_t sc2 = f2_pack(scale, scale), no2 = f2_pack(-off, -off);
    uint64_t acc[4] = {0, 0, 0, 0};
#pragma unroll
    for (int t = 0; t < K; t += 2) {
        float a, b;
        f2_unpack(f2_fma(f2_pack(__uint_as_float(d[t]), __uint_as_float(d[t + 1])), sc2, no2), a, b);
        x[t] = ex2_approx(a);
        x[t + 1] = ex2_approx(b);
        acc[(t >> 1) & 3] = f2_add(acc[(t >> 1) & 3], f2_pack(x[t], x[t + 1]));
    }
    float s0, s1, s2, s3, s4, s5, s6, s7;
    f2_unpack(acc[0], s0, s1); f2_unpack(acc[1], s2, s3);
    f2_unpack(acc[2], s4, s5); f2_unpack(acc[3], s6, s7);
    return ((s0 + s1) + (s2 + s3)) + ((s4 + s5) + (s6 + s7));
}

// SLICE = false: one head per CTA, O written directly.  SLICE = true: one (head,
// component slice, value slice) per CTA (grid G x Kfull/64 x dvt/64); the key
// responsibilities are normalised over all Kfull components with the row's
// log-sum-exp, e^Q is taken relative to the row's maximum over all components,
// and the CTA writes its partial numerator and denominator, which the combine
// kernel sums over component slices (every term is a sum over components).
template <bool SLICE>
__global__ void __launch_bounds__(kCThreads, 1)
tc_causal_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                 const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o, CausalArgs A) {
    using C = CausalCfg;
    constexpr int K = KC;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + C::OFF_BAR);
    // TMA rings (count 1: the producer's expect_tx; the empties: one arrival per consuming warp)
    uint64_t *qfull = bars, *qempty = qfull + 2, *kfull = qempty + 2, *kempty = kfull + 2;
    uint64_t *vfull = kempty + 2, *vempty = vfull + 2;
    uint64_t *w_full = vempty + 2;                       // parameter block in place
    uint64_t *ak_full = w_full + 1, *d1k_full = ak_full + 1, *aq_full = d1k_full + 1, *d1q_full = aq_full + 1;
    uint64_t *g_full = d1q_full + 1, *g_empty = g_full + 1;           // gamma^K(c): written / read by T and update
    uint64_t *e_full = g_empty + 1, *eq_free = e_full + 2;            // e^Q buffers [2]
    uint64_t *ta_full = eq_free + 2, *ta_free = ta_full + 1;          // T half 0 computed / loaded
    uint64_t *tb2_full = ta_free + 1, *t1_read = tb2_full + 1;        // T half 1 computed / loaded
    uint64_t *slot_full = t1_read + 1, *slot_free = slot_full + 2;    // masked-T half slots [2]
    uint64_t *s_upd = slot_free + 2, *s_ready = s_upd + 1, *sb_empty = s_ready + 2;   // state
    uint64_t *d3_full = sb_empty + 2, *d3_empty = d3_full + 1;        // read result
    uint64_t *fin1 = d3_empty + 1, *fin2 = fin1 + 1, *fin3 = fin2 + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(fin3 + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = blockIdx.x, nch = A.nch;
    const int ks = SLICE ? (int)blockIdx.y : 0, vs = SLICE ? (int)blockIdx.z : 0;   // component / value slice
    grid_dep_launch();
    // direct form: the compute groups put the head's parameter loads in flight before the prologue
    constexpr int kTeam = 3 * kWgThreads, kTeamBar = 4;
    const int ttid = (int)threadIdx.x - kWGroups * 32;
    ParamLoads<K, kTeam> pld;
    if (!SLICE && ttid >= 0) {
        const int h = g % A.H;
        pld.issue(ttid, A.mu + (size_t)h * K * DR, A.rho + (size_t)h * K * DR, A.alpha + (size_t)h * K);
    }

    if (threadIdx.x == 0) {
        for (int s = 0; s < 2; ++s) {
            mbar_init(&qfull[s], 1); mbar_init(&qempty[s], 4); mbar_init(&kfull[s], 1); mbar_init(&kempty[s], 4);
            mbar_init(&vfull[s], 1); mbar_init(&vempty[s], 1);
            mbar_init(&e_full[s], 4); mbar_init(&eq_free[s], 2);
            mbar_init(&s_ready[s], 4); mbar_init(&sb_empty[s], 1);
            mbar_init(&slot_full[s], 4); mbar_init(&slot_free[s], 1);
        }
        mbar_init(w_full, 1);
        mbar_init(ak_full, 4); mbar_init(d1k_full, 1); mbar_init(aq_full, 4); mbar_init(d1q_full, 1);
        mbar_init(g_full, 4); mbar_init(g_empty, 2);
        mbar_init(ta_full, 1); mbar_init(ta_free, 4); mbar_init(tb2_full, 1); mbar_init(t1_read, 4);
        mbar_init(s_upd, 1); mbar_init(d3_full, 1); mbar_init(d3_empty, 4);
        mbar_init(fin1, 1); mbar_init(fin2, 1); mbar_init(fin3, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    // ONES atom column (element 0 of every row = 1.0 bf16) for the z row of the state update;
    // the masked-T slots (entries above the diagonal are never written); the constant
    // rows of both state operands: row 65 = 1 (gives sum_k e^Q_ik), rows 66..79 = 0, and
    // rows 0..64 of buffer 0 = 0 (the state before the first chunk).
    for (uint32_t e = threadIdx.x; e < kTileBytes / 16; e += blockDim.x)
        reinterpret_cast<uint4 *>(sm + C::OFF_ONES)[e] = make_uint4(0, 0, 0, 0);
    for (uint32_t e = threadIdx.x; e < 2 * kTileBytes / 16; e += blockDim.x)
        reinterpret_cast<uint4 *>(sm + C::OFF_TB)[e] = make_uint4(0, 0, 0, 0);
    for (uint32_t e = threadIdx.x; e < 2 * C::SBB / 16; e += blockDim.x) {
        const uint32_t row = (e * 16u % C::SBB) / 128u;
        const uint32_t v = row == DVV + 1 ? 0x3F803F80u : 0u;
        reinterpret_cast<uint4 *>(sm + C::OFF_SB)[e] = make_uint4(v, v, v, v);
    }
    init_const_a(sm + C::OFF_CA, threadIdx.x, blockDim.x);
    __syncthreads();
    if (threadIdx.x < TM) *reinterpret_cast<uint16_t *>(sm + C::OFF_ONES + sw128_off(threadIdx.x, 0)) = 0x3F80u;
    if (warp == kWIss1) { tmem_alloc(tmem_slot, C::TMEM_COLS); tmem_relinquish(); }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const Abort ab{abort_flag, A.status};
    if (threadIdx.x == 0) {                                      // the state for chunk 0 is ready
        for (int w = 0; w < 4; ++w) mbar_arrive(&s_ready[0]);
    }

    if (warp == kWProd) {
        if (lane == 0) {
            // the first tiles do not depend on the previous kernel; the parameter block does
            int qi = 0, ki = 0, vi = 0;
            for (; ki < 2 && ki < nch; ++ki) {
                mbar_arrive_expect_tx(&kfull[ki], kTileBytes);
                tma_load_3d(sm + C::OFF_K + ki * kTileBytes, &tm_k, &kfull[ki], 0, ki * TM, g);
            }
            for (; qi < 2 && qi < nch; ++qi) {
                mbar_arrive_expect_tx(&qfull[qi], kTileBytes);
                tma_load_3d(sm + C::OFF_Q + qi * kTileBytes, &tm_q, &qfull[qi], 0, qi * TM, g);
            }
            for (; vi < 2 && vi < nch; ++vi) {
                mbar_arrive_expect_tx(&vfull[vi], kTileBytes);
                tma_load_3d(sm + C::OFF_V + vi * kTileBytes, &tm_v, &vfull[vi], 64 * vs, vi * TM, g);
            }
            if (SLICE) {
                grid_dep_wait();
                const uint8_t *blk = A.params + (size_t)(g % A.H) * A.param_stride;
                // the slice's 64 rows of each part of a Kfull-component block, in the K = 64 layout
                // (row groups of 8 keep their 1 KB swizzle atoms and no-swizzle core matrices)
                constexpr uint32_t kRows = 64u * 128u, kWc = 64u * 32u;
                mbar_arrive_expect_tx(w_full, 2 * kRows + kWc + 16u);
                bulk_load(sm + C::OFF_P, blk + (size_t)ks * kRows, kRows, w_full);
                bulk_load(sm + C::OFF_P + kRows, blk + 128u * A.Kfull + (size_t)ks * kRows, kRows, w_full);
                bulk_load(sm + C::OFF_P + param_wc_off(K), blk + param_wc_off(A.Kfull) + (size_t)ks * kWc, kWc, w_full);
                bulk_load(sm + C::OFF_P + param_scale_off(K), blk + param_scale_off(A.Kfull), 16u, w_full);
            }
            long long last = now_ns();
            while ((qi < nch || ki < nch || vi < nch) && !*abort_flag) {
                bool progress = false;
                if (ki < nch && (ki < 2 || mbar_test(&kempty[ki & 1], ((ki >> 1) - 1) & 1))) {
                    mbar_arrive_expect_tx(&kfull[ki & 1], kTileBytes);
                    tma_load_3d(sm + C::OFF_K + (ki & 1) * kTileBytes, &tm_k, &kfull[ki & 1], 0, ki * TM, g);
                    ++ki;
                    progress = true;
                }
                if (qi < nch && (qi < 2 || mbar_test(&qempty[qi & 1], ((qi >> 1) - 1) & 1))) {
                    mbar_arrive_expect_tx(&qfull[qi & 1], kTileBytes);
                    tma_load_3d(sm + C::OFF_Q + (qi & 1) * kTileBytes, &tm_q, &qfull[qi & 1], 0, qi * TM, g);
                    ++qi;
                    progress = true;
                }
                if (vi < nch && (vi < 2 || mbar_test(&vempty[vi & 1], ((vi >> 1) - 1) & 1))) {
                    mbar_arrive_expect_tx(&vfull[vi & 1], kTileBytes);
                    tma_load_3d(sm + C::OFF_V + (vi & 1) * kTileBytes, &tm_v, &vfull[vi & 1], 64 * vs, vi * TM, g);
                    ++vi;
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
            wind_down_ring(kfull, 2, ki, A.status);
            wind_down_ring(qfull, 2, qi, A.status);
            wind_down_ring(vfull, 2, vi, A.status);
            if (SLICE) wait_ignoring_abort(w_full, 0, A.status);
        }
    } else if (warp == kWIss1) {
        // log-density MMAs: scores = [x, x^2/256] . W^T, keys then queries of each chunk
        const uint32_t pw = smem_u32(sm + C::OFF_P), ca = smem_u32(sm + C::OFF_CA);
        bool ok = mbar_wait_warp(w_full, 0, ab, kDevErrTimeout);
        for (int c = 0; c < nch && ok; ++c) {
            if (!(ok = mbar_wait_warp(ak_full, c & 1, ab, kDevErrTimeout))) break;
            tc_fence_after();
            issue_logdensity<K>(tmem + C::COL_D1K, tmem + C::COL_A, pw, ca);
            mma_commit(d1k_full);
            if (!(ok = mbar_wait_warp(aq_full, c & 1, ab, kDevErrTimeout))) break;
            tc_fence_after();
            issue_logdensity<K>(tmem + C::COL_D1Q, tmem + C::COL_A, pw, ca);
            mma_commit(d1q_full);
        }
        mma_commit(fin1);
        wait_ignoring_abort(fin1, 0, A.status);
    } else if (warp == kWIssT) {
        // T(c) = e^Q(c) . gamma^K(c)^T in two 64-key halves through one TMEM buffer
        constexpr uint32_t idesc_t = idesc_f16(1, 1, 0, 0, TM, 64);
        const uint64_t gk = sdesc_sw128(smem_u32(sm + C::OFF_G), 16, 1024);   // gamma^K as K-major B (N = keys)
        bool ok = true;
        for (int c = 0; c < nch && ok; ++c) {
            const uint32_t eq = tmem + C::COL_EQ + 32u * (c & 1);
            // half 0 once e^Q(c) and gamma^K(c) are in place and T(c - 1)'s second half is in registers
            ok = mbar_wait_warp(&e_full[c & 1], (c >> 1) & 1, ab, kDevErrTimeout) &&
                 mbar_wait_warp(g_full, c & 1, ab, kDevErrTimeout);
            if (ok && c >= 1) ok = mbar_wait_warp(t1_read, (c - 1) & 1, ab, kDevErrTimeout);
            if (!ok) break;
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < K / 16; ++kk)
                mma_ts(tmem + C::COL_T, eq + kk * 8, gk + (uint64_t)((kk * 32u) >> 4), idesc_t, kk > 0);
            mma_commit(ta_full);
            // half 1 once the first half has been loaded
            if (!(ok = mbar_wait_warp(ta_free, c & 1, ab, kDevErrTimeout))) break;
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < K / 16; ++kk)
                mma_ts(tmem + C::COL_T, eq + kk * 8, gk + (uint64_t)((64u * 128u + kk * 32u) >> 4), idesc_t,
                       kk > 0);
            mma_commit(tb2_full);
            mma_commit(g_empty);
            mma_commit(&eq_free[c & 1]);
        }
        mma_commit(fin2);
        wait_ignoring_abort(fin2, 0, A.status);
    } else if (warp == kWIssR) {
        constexpr uint32_t idesc_u = idesc_f16(1, 1, 1, 1, TM, K);       // [V | 1]^T . gamma^K
        constexpr uint32_t idesc_r1 = idesc_f16(1, 1, 0, 0, TM, 80);     // e^Q . [S | z | 1]
        constexpr uint32_t idesc_r2 = idesc_f16(1, 1, 0, 1, TM, 80);     // T . [V | 1]
        const uint32_t gaddr = smem_u32(sm + C::OFF_G), ones = smem_u32(sm + C::OFF_ONES);
        const uint64_t gm = sdesc_sw128(gaddr, kTileBytes, 1024);        // gamma^K as MN-major B (N = k)
        bool ok = true;
        for (int c = 0; c < nch && ok; ++c) {
            const int s = c & 1;
            // state update: [S | z]^T += [V | 1 | 0]^T . gamma^K, once the previous state is snapshotted
            ok = mbar_wait_warp(g_full, c & 1, ab, kDevErrTimeout) &&
                 mbar_wait_warp(&vfull[s], (c >> 1) & 1, ab, kDevErrTimeout) &&
                 mbar_wait_warp(&s_ready[s], (c >> 1) & 1, ab, kDevErrTimeout);
            if (!ok) break;
            tc_fence_after();
            const uint32_t va = smem_u32(sm + C::OFF_V + s * kTileBytes);
            const uint64_t vd = sdesc_sw128(va, ones - va, 1024);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
                mma_ss(tmem + C::COL_S, vd + (uint64_t)(kk * 128), gm + (uint64_t)(kk * 128), idesc_u,
                       !(c == 0 && kk == 0));
            mma_commit(s_upd);
            mma_commit(g_empty);
            // read(c) = mask(T)(c) . V + e^Q(c) . S_{c-1}, half by half as the mask group fills them
            ok = c < 1 || mbar_wait_warp(d3_empty, (c - 1) & 1, ab, kDevErrTimeout);
            if (ok) ok = mbar_wait_warp(&slot_full[0], c & 1, ab, kDevErrTimeout);
            if (!ok) break;
            tc_fence_after();
            const uint64_t tbd = sdesc_sw128(smem_u32(sm + C::OFF_TB), 16, 1024);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                mma_ss(tmem + C::COL_D3, tbd + (uint64_t)((kk * 32u) >> 4), vd + (uint64_t)(kk * 128), idesc_r2,
                       kk > 0);
            mma_commit(&slot_free[0]);
            const uint32_t eq = tmem + C::COL_EQ + 32u * (c & 1);
            const uint64_t sbd = sdesc_sw128(smem_u32(sm + C::OFF_SB + (c & 1) * C::SBB), 16, 1024);
#pragma unroll
            for (int kk = 0; kk < K / 16; ++kk)
                mma_ts(tmem + C::COL_D3, eq + kk * 8, sbd + (uint64_t)((kk * 32u) >> 4), idesc_r1, 1);
            mma_commit(&eq_free[c & 1]);
            mma_commit(&sb_empty[c & 1]);
            if (!(ok = mbar_wait_warp(&slot_full[1], c & 1, ab, kDevErrTimeout))) break;
            tc_fence_after();
#pragma unroll
            for (int kk = 4; kk < 8; ++kk)
                mma_ss(tmem + C::COL_D3, tbd + (uint64_t)((kTileBytes + (kk & 3) * 32u) >> 4),
                       vd + (uint64_t)(kk * 128), idesc_r2, 1);
            mma_commit(&slot_free[1]);
            mma_commit(d3_full);
            mma_commit(&vempty[s]);
        }
        mma_commit(fin3);
        wait_ignoring_abort(fin3, 0, A.status);
    } else {
        RowThread rt;
        rt.wg = (warp - kWGroups) >> 2;
        rt.r = 32u * (warp & 3) + lane;
        rt.lane_off = (uint32_t)(32 * (warp & 3)) << 16;
        rt.wtid = threadIdx.x - kWGroups * 32 - rt.wg * kWgThreads;
        float scale = 0.f;                                 // read once the parameter blocks are written
        // component-sliced form: this row's key log-sum-exp / query maximum in chunk c (rows past
        // the sequence end: gamma^K = 0, e^Q finite); read after the grid-dependency wait
        float stat_next = 0.f;
        auto lse_row = [&](int c) -> float {
            const int row = c * TM + (int)rt.r;
            return row < A.N ? __ldg(A.lse_k + (size_t)g * A.N + row) : INFINITY;
        };
        auto max_row = [&](int c) -> float {
            const int row = c * TM + (int)rt.r;
            return row < A.N ? __ldg(A.mrow_q + (size_t)g * A.N + row) : 0.f;
        };
        // one arrival per warp once every lane's tcgen05 / shared-memory work is done
        auto warp_arrive = [&](uint64_t *bar) {
            __syncwarp();
            if (lane == 0) mbar_arrive(bar);
        };
        if (!SLICE) {
            // The three groups build the head's parameter block straight into the operand block
            // the log-density MMAs read (scratch: the gamma buffer, which holds nothing yet).
            build_param_block_team(ttid, pld, A.var_floor, sm + C::OFF_P, reinterpret_cast<float *>(sm + C::OFF_G));
            fence_proxy_async_smem();
            group_sync(kTeamBar, kTeam);
            scale = *reinterpret_cast<const float *>(sm + C::OFF_P + param_scale_off(K));
            if (ttid == 0) mbar_arrive(w_full);
        }

        if (rt.wg == 0) {
            // ---------------- key group
            // keys of chunk c into the shared operand region once the query MMA of chunk c - 1 has read it
            auto convert_k = [&](int c) -> bool {
                if (!mbar_wait_warp(&kfull[c & 1], (c >> 1) & 1, ab, kDevErrTimeout)) return false;
                if (c >= 1 && !mbar_wait_warp(d1q_full, (c - 1) & 1, ab, kDevErrTimeout)) return false;
                tc_fence_after();
                convert_row_call(sm + C::OFF_K + (c & 1) * kTileBytes, rt.r, tmem + rt.lane_off + C::COL_A);
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) { mbar_arrive(ak_full); mbar_arrive(&kempty[c & 1]); }
                return true;
            };
            bool ok = convert_k(0);
            for (int c = 0; c < nch && ok; ++c) {
                ok = mbar_wait_warp(d1k_full, c & 1, ab, kDevErrTimeout);
                if (ok && c >= 1) ok = mbar_wait_warp(g_empty, (c - 1) & 1, ab, kDevErrTimeout);
                if (!ok) break;
                tc_fence_after();
                if (SLICE && c == 0) {
                    grid_dep_wait();
                    scale = head_scale(A.params, A.param_stride, g % A.H, A.Kfull);
                    stat_next = lse_row(0);
                }
                // gamma^K = softmax of the key scores in fp32, rounded once to bf16; rows past the
                // sequence end get 0.  Component-sliced form: normalised over all components by
                // the row's log-sum-exp (loaded a chunk ahead).
                float x[K];
                float inv;
                if (SLICE) {
                    const float off = stat_next;
                    if (c + 1 < nch) stat_next = lse_row(c + 1);
                    row_exp2<K, true>(tmem + rt.lane_off + C::COL_D1K, scale, off, x);
                    inv = 1.0f;
                } else {
                    const float total = row_exp2<K, false>(tmem + rt.lane_off + C::COL_D1K, scale, 0.f, x);
                    inv = c * TM + (int)rt.r < A.N ? 1.0f / total : 0.f;
                }
                const uint64_t inv2 = f2_pack(inv, inv);
#pragma unroll
                for (int j = 0; j < K / 8; ++j) {
                    uint32_t wv[4];
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        float ga, gb;
                        f2_unpack(f2_mul(f2_pack(x[8 * j + 2 * u], x[8 * j + 2 * u + 1]), inv2), ga, gb);
                        wv[u] = pack_bf16(ga, gb);
                    }
                    *reinterpret_cast<uint4 *>(sm + C::OFF_G + sw128_off(rt.r, j)) = make_uint4(wv[0], wv[1], wv[2], wv[3]);
                }
                fence_proxy_async_smem();
                tc_fence_before();
                warp_arrive(g_full);
                // bf16 snapshot of the state after chunk c - 1, the read operand of chunk c (its
                // update went into the tensor pipe a chunk ago; the update of chunk c waits for it)
                if (c >= 1) {
                    const int b = c & 1;
                    ok = mbar_wait_warp(s_upd, (c - 1) & 1, ab, kDevErrTimeout);
                    if (ok && c >= 2) ok = mbar_wait_warp(&sb_empty[b], ((c >> 1) - 1) & 1, ab, kDevErrTimeout);
                    if (!ok) break;
                    tc_fence_after();
                    uint32_t v[K];
                    tmem_ld32(tmem + rt.lane_off + C::COL_S, v);
                    tmem_ld32(tmem + rt.lane_off + C::COL_S + 32, v + 32);
                    tmem_ld_wait();
                    if (rt.r <= DVV) {                       // S^T rows and z
                        uint8_t *row = sm + C::OFF_SB + b * C::SBB;
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            uint4 o;
                            o.x = pack_bf16(__uint_as_float(v[8 * j + 0]), __uint_as_float(v[8 * j + 1]));
                            o.y = pack_bf16(__uint_as_float(v[8 * j + 2]), __uint_as_float(v[8 * j + 3]));
                            o.z = pack_bf16(__uint_as_float(v[8 * j + 4]), __uint_as_float(v[8 * j + 5]));
                            o.w = pack_bf16(__uint_as_float(v[8 * j + 6]), __uint_as_float(v[8 * j + 7]));
                            *reinterpret_cast<uint4 *>(row + sw128_off(rt.r, j)) = o;
                        }
                    }
                    fence_proxy_async_smem();
                    tc_fence_before();
                    warp_arrive(&s_ready[b]);
                }
                if (c + 1 >= nch) break;
                if (!(ok = convert_k(c + 1))) break;
            }
        } else if (rt.wg == 1) {
            // ---------------- query group
            // queries of chunk c into the shared operand region once the key MMA of chunk c has read it
            auto convert_q = [&](int c) -> bool {
                if (!(mbar_wait_warp(&qfull[c & 1], (c >> 1) & 1, ab, kDevErrTimeout) &&
                      mbar_wait_warp(d1k_full, c & 1, ab, kDevErrTimeout)))
                    return false;
                tc_fence_after();
                convert_row_call(sm + C::OFF_Q + (c & 1) * kTileBytes, rt.r, tmem + rt.lane_off + C::COL_A);
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) { mbar_arrive(aq_full); mbar_arrive(&qempty[c & 1]); }
                return true;
            };
            // called once read(c) is known complete (d3_full(c) waited):
            // out = num / (den + eps * sum_k e^Q_k), staged and stored by TMA (one 32-row box per warp)
            uint8_t *stage = sm + C::OFF_O + (warp & 3) * 4096u;
            auto epilogue = [&](int c) {
                uint32_t v0[32], v1[32], dz[4];
                tmem_ld32(tmem + rt.lane_off + C::COL_D3, v0);
                tmem_ld32(tmem + rt.lane_off + C::COL_D3 + 32, v1);
                tmem_ld4(tmem + rt.lane_off + C::COL_D3 + 64, dz);
                tmem_ld_wait();
                tc_fence_before();
                warp_arrive(d3_empty);
                const float den = __uint_as_float(dz[0]) + A.eps * __uint_as_float(dz[1]);
                const int row = c * TM + (int)rt.r;
                const float rd = SLICE ? 1.0f : 1.0f / den;
                if (SLICE && vs == 0 && row < A.N) A.pden[((size_t)ks * A.G + g) * A.N + row] = den;
                // this warp's previous store has left the staging quarter
                if (lane == 0) bulk_wait_group_read<0>();
                __syncwarp();
                const uint64_t rd2 = f2_pack(rd, rd);
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const uint32_t *src = j < 4 ? v0 + 8 * j : v1 + 8 * (j - 4);
                    uint32_t o[4];
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        float oa, obv;
                        f2_unpack(f2_mul(f2_pack(__uint_as_float(src[2 * u]), __uint_as_float(src[2 * u + 1])), rd2),
                                  oa, obv);
                        o[u] = pack_bf16(oa, obv);
                    }
                    *reinterpret_cast<uint4 *>(stage + sw128_off(lane, j)) = make_uint4(o[0], o[1], o[2], o[3]);
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    // rows past the sequence end are clipped by the store
                    if (SLICE) tma_store_3d(&tm_o, stage, 64 * vs, c * TM + 32 * (warp & 3), ks * A.G + g);
                    else tma_store_3d(&tm_o, stage, 0, c * TM + 32 * (warp & 3), g);
                    bulk_commit_group();
                }
            };
            bool ok = convert_q(0);
            for (int c = 0; c <= nch && ok; ++c) {
                if (c < nch) {
                    if (!(ok = mbar_wait_warp(d1q_full, c & 1, ab, kDevErrTimeout))) break;
                    tc_fence_after();
                    if (SLICE && c == 0) {
                        grid_dep_wait();
                        scale = head_scale(A.params, A.param_stride, g % A.H, A.Kfull);
                        stat_next = max_row(0);
                    }
                    float x[K];
                    if (SLICE) {
                        // relative to the row's maximum over all components (loaded a chunk ahead)
                        const float off = stat_next;
                        if (c + 1 < nch) stat_next = max_row(c + 1);
                        row_exp2<K, true>(tmem + rt.lane_off + C::COL_D1Q, scale, off, x);
                    } else {
                        row_exp2<K, false>(tmem + rt.lane_off + C::COL_D1Q, scale, 0.f, x);
                    }
                    uint32_t e[K / 2];
#pragma unroll
                    for (int t = 0; t < K / 2; ++t) e[t] = pack_bf16(x[2 * t], x[2 * t + 1]);
                    // e^Q(c) goes to buffer c & 1 once chunk c - 2 (T and read) has consumed it
                    if (c >= 2) {
                        if (!(ok = mbar_wait_warp(&eq_free[c & 1], ((c >> 1) - 1) & 1, ab, kDevErrTimeout))) break;
                        tc_fence_after();
                    }
                    tmem_st32(tmem + rt.lane_off + C::COL_EQ + 32u * (c & 1), e);
                    tmem_st_wait();
                    tc_fence_before();
                    warp_arrive(&e_full[c & 1]);
                    // the scores of chunk c have been read: the next query tile may overwrite them
                    if (c + 1 < nch && !(ok = convert_q(c + 1))) break;
                }
                // read(c - 1): its epilogue, off the chunk-to-chunk chain
                if (c >= 1) {
                    if (!(ok = mbar_wait_warp(d3_full, (c - 1) & 1, ab, kDevErrTimeout))) break;
                    tc_fence_after();
                    epilogue(c - 1);
                }
            }
            if (lane == 0) bulk_wait_group<0>();
        } else {
            // ---------------- mask group
            // Row quarter q = warp & 3 holds rows 32q..32q+31.  A group of 32 keys (global
            // index gi) is copied whole below the quarter's diagonal (gi < q), selected
            // (j <= r) on it (gi == q) and never written above it (gi > q): those entries of
            // the slot stay zero from the start.
            const int q = warp & 3;
            bool ok = true;
            for (int c = 0; c < nch && ok; ++c) {
#pragma unroll 1
                for (int hh = 0; hh < 2; ++hh) {
                    // half hh (keys 64 hh .. 64 hh + 63) of T(c), once the read of chunk c - 1 has
                    // consumed that half of the masked tile
                    ok = mbar_wait_warp(hh == 0 ? ta_full : tb2_full, c & 1, ab, kDevErrTimeout);
                    if (ok && c >= 1) ok = mbar_wait_warp(&slot_free[hh], (c - 1) & 1, ab, kDevErrTimeout);
                    if (!ok) break;
                    tc_fence_after();
                    const int g0 = 2 * hh;                   // global index of the half's first group
                    uint32_t v0[32], v1[32];
                    if (q >= g0) tmem_ld32(tmem + rt.lane_off + C::COL_T, v0);
                    if (q >= g0 + 1) tmem_ld32(tmem + rt.lane_off + C::COL_T + 32, v1);
                    tmem_ld_wait();
                    tc_fence_before();
                    warp_arrive(hh == 0 ? ta_free : t1_read);   // the T buffer may take the next half
                    uint8_t *sl = sm + C::OFF_TB + hh * kTileBytes;
                    if (q >= g0) mask_group(v0, q == g0, lane, sl, rt.r, 0);
                    if (q >= g0 + 1) mask_group(v1, q == g0 + 1, lane, sl, rt.r, 1);
                    fence_proxy_async_smem();
                    warp_arrive(&slot_full[hh]);
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kWIss1) {
        __syncwarp();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

}  // namespace

bool tc_causal_supported(const Problem &p) {
    return p.in_dtype == GMA_BF16 && p.out_dtype == GMA_BF16 && p.causal && p.d == DR && p.dv == DVV &&
           p.K == KC && p.N > 0;
}

bool tc_slice_supported(const Problem &p) {
    return p.in_dtype == GMA_BF16 && p.out_dtype == GMA_BF16 && p.causal && p.d == DR && p.N > 0 &&
           p.K % KC == 0 && p.K <= 256 && p.dv % DVV == 0 && p.dv <= 256 && !tc_causal_supported(p);
}

TcLayout tc_causal_layout(const Problem &p) {
    TcLayout L{};
    L.T = (p.N + TM - 1) / TM;
    L.Ttot = L.T * p.G;
    L.ncta = p.G;
    L.ns = L.nt = 1;
    L.param_stride = align1k(param_bytes(p.K));
    L.params = L.part = L.mem = align_up(kHeaderBytes);          // only the status header
    L.total = L.params;
    return L;
}

TcLayout tc_slice_layout(const Problem &p) {
    TcLayout L{};
    L.T = (p.N + TM - 1) / TM;
    L.Ttot = L.T * p.G;
    L.ns = p.K / KC;
    L.nt = p.dv / DVV;
    L.ncta = p.G * L.ns * L.nt;
    L.param_stride = align1k(param_bytes(p.K));
    L.params = align_up(kHeaderBytes);
    const size_t rows = (size_t)p.G * p.N;
    L.stats = align_up(L.params + (size_t)p.H * L.param_stride);              // [2][G][N] f32
    L.pnum = align_up(L.stats + 2 * rows * sizeof(float));                     // [ns][G][N][dv] bf16
    L.pden = align_up(L.pnum + (size_t)L.ns * rows * p.dv * 2);                // [ns][G][N] f32
    L.part = L.mem = L.pden;
    L.total = align_up(L.pden + (size_t)L.ns * rows * sizeof(float));
    return L;
}

static cudaError_t launch_causal(const Problem &p, const TcLayout &L, const void *Qx, const void *Kx, const void *V,
                                 const float *mu, const float *rho, const float *alpha, void *out, char *ws,
                                 cudaStream_t s, bool slices) {
    // outputs leave by TMA in 32-row boxes: O [G][N][64], or the partial numerators [ns G][N][dv]
    CUtensorMap tq, tk, tv, to;
    if (!make_map(&tq, Qx, p.G, p.N, DR) || !make_map(&tk, Kx, p.G, p.N, DR) || !make_map(&tv, V, p.G, p.N, p.dv) ||
        !(slices ? make_map(&to, ws + L.pnum, L.ns * p.G, p.N, p.dv, 32) : make_map(&to, out, p.G, p.N, DVV, 32)))
        return cudaErrorInvalidValue;
    CausalArgs a{};
    a.G = p.G; a.H = p.H; a.N = p.N; a.nch = L.T;
    a.params = reinterpret_cast<const uint8_t *>(ws + L.params);
    a.param_stride = L.param_stride;
    a.eps = p.eps;
    a.status = reinterpret_cast<unsigned *>(ws);
    a.Kfull = p.K;
    a.dvt = p.dv;
    if (slices) {
        a.mrow_q = reinterpret_cast<const float *>(ws + L.stats);
        a.lse_k = a.mrow_q + (size_t)p.G * p.N;
        a.pnum = reinterpret_cast<uint16_t *>(ws + L.pnum);
        a.pden = reinterpret_cast<float *>(ws + L.pden);
    } else {
        a.mu = mu; a.rho = rho; a.alpha = alpha;
        a.var_floor = p.var_floor;
    }
    auto kern = slices ? tc_causal_kernel<true> : tc_causal_kernel<false>;
    cudaError_t e = set_dyn_smem(reinterpret_cast<const void *>(kern), CausalCfg::BYTES);
    if (e != cudaSuccess) return e;
    if (!slices) {
        // the first kernel of its forward: an ordinary launch, so that every input is final when
        // its CTAs start
        kern<<<dim3(p.G), dim3(kCThreads), CausalCfg::BYTES, s>>>(tq, tk, tv, to, a);
        return cudaGetLastError();
    }
    return launch_dependent(kern, dim3(p.G, L.ns, L.nt), dim3(kCThreads), CausalCfg::BYTES, s, tq, tk, tv, to, a);
}

cudaError_t tc_causal(const Problem &p, const TcLayout &L, const void *Qx, const void *Kx, const void *V,
                      const float *mu, const float *rho, const float *alpha, void *out, char *ws, cudaStream_t s) {
    return launch_causal(p, L, Qx, Kx, V, mu, rho, alpha, out, ws, s, false);
}

cudaError_t tc_causal_slices(const Problem &p, const TcLayout &L, const void *Qx, const void *Kx, const void *V,
                             char *ws, cudaStream_t s) {
    return launch_causal(p, L, Qx, Kx, V, nullptr, nullptr, nullptr, nullptr, ws, s, true);
}

}  // namespace gma
