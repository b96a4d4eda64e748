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
// fp32 and is snapshotted as a bf16 MMA operand once per chunk; every
// reduction has a fixed order, so results are bitwise reproducible, and row i
// never reads rows after i (the mask selects, it does not multiply).
//
// One CTA per head, and the forward is this one kernel: the three compute groups
// first build the head's parameter block (Eq. 14-16, the same code as tc_params)
// in shared memory while the first tiles load.  Warps: 0 TMA producer; 1 TMEM owner and issuer of the
// log-density MMAs (keys, then queries); 2 issuer of the chained MMAs (T, the
// state update, the read); 3-6 key group (convert, softmax, state snapshot);
// 7-10 query group (convert, exp, epilogue and store); 11-14 mask group.
//
// T is formed in two 64-key halves through one 64-column TMEM buffer: rows
// 0..63 never see keys 64..127, so that half of the masked tile stays zero.
// e^Q, T and the read result have TMEM columns of their own, so chunk c + 1's
// query scores and T proceed while chunk c is read, and the query group runs
// chunk c - 1's epilogue once it has published e^Q(c).
// Every mbarrier wait is bounded; a timeout posts GMA_ERR_TIMEOUT.
#include <cuda.h>
#include <cuda_bf16.h>

#include <algorithm>
#include <cstring>

#include "gma_internal.h"
#include "gma_sm100.cuh"
#include "gma_tc_common.cuh"

namespace gma {

using namespace sm100;
using namespace tc;

namespace {

constexpr int KC = 64;                 // components handled by this kernel
constexpr int kCThreads = 480;         // 15 warps
constexpr int kWProd = 0, kWIss1 = 1, kWIss2 = 2, kWGroups = 3;
constexpr int NOUT = 80;               // [S | z | 1 | 0...] and [V | 1 | 0...] widths

struct CausalArgs {
    int G, H, N, nch;      // nch: 128-row chunks per head
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
    // segment-parallel form: the prefix pass's partial slots [slot][dv + 1][K] f32
    const float *partials;
    int nslots;            // partial slots in the workspace (index checks of the debug build)
};

struct CausalCfg {
    static constexpr uint32_t PB = align1k(param_bytes(KC));
    static constexpr uint32_t SBB = 80u * 128u;                        // state operand [80 rows][64 k] bf16
    static constexpr uint32_t OFF_Q = 0;                               // 2 stages
    static constexpr uint32_t OFF_K = OFF_Q + 2 * kTileBytes;          // 2 stages
    static constexpr uint32_t OFF_V = OFF_K + 2 * kTileBytes;          // 2 stages
    static constexpr uint32_t OFF_ONES = OFF_V + 2 * kTileBytes;       // after the V stages (positive LBO)
    static constexpr uint32_t OFF_G = OFF_ONES + kTileBytes;           // gamma^K [row][k]
    static constexpr uint32_t OFF_TB = OFF_G + kTileBytes;             // masked T, bf16 [row][key], 2 chunks
    static constexpr uint32_t OFF_SB = OFF_TB + 2 * kTileBytes;        // state operand, 2 buffers
    static constexpr uint32_t OFF_P = OFF_SB + 2 * SBB;
    static constexpr uint32_t OFF_O = OFF_P + PB;                      // output staging tile
    static constexpr uint32_t OFF_CA = OFF_O + kTileBytes;             // constant [1, 1, 0...] A block
    static constexpr uint32_t OFF_BAR = OFF_CA + kConstABytes;
    static constexpr uint32_t BYTES = OFF_BAR + 512 + 1024;
    // TMEM columns
    static constexpr uint32_t COL_AQ = 0, COL_D1Q = 64, COL_AK = 128, COL_D1K = 192;
    static constexpr uint32_t COL_T = 256;                             // one 64-key half of T (fp32)
    static constexpr uint32_t COL_D3 = 320;                            // read result [num | den | sum e^Q], 80
    static constexpr uint32_t COL_S = 416;                             // [S | z]^T state, 64 columns
    static constexpr uint32_t COL_EQ = 480;                            // e^Q as bf16 pairs, 32 columns
    static constexpr uint32_t TMEM_COLS = 512;
};
static_assert(CausalCfg::OFF_SB % 1024 == 0 && CausalCfg::OFF_P % 1024 == 0 && CausalCfg::OFF_O % 1024 == 0,
              "operand blocks must be 1024-byte aligned");
static_assert(CausalCfg::BYTES <= 232448, "causal kernel exceeds the shared-memory opt-in limit");
static_assert(param_scratch_floats(KC, 3 * kWgThreads) * 4 <= (int)kTileBytes,
              "the parameter build's scratch must fit the gamma buffer");

// The parameter build as one out-of-line call, keeping it out of the compute groups' loop code.
static __device__ __noinline__ void build_param_block_team(int tid, ParamLoads<KC, 3 * kWgThreads> ld, float var_floor,
                                                           uint8_t *blk, float *scratch) {
    build_param_block<KC, 3 * kWgThreads>(tid, ld, var_floor, blk, scratch, [] { group_sync(4, 3 * kWgThreads); });
}

// SLICE = false: one head per CTA, O written directly.  SLICE = true: one (head,
// component slice, value slice) per CTA (grid G x Kfull/64 x dvt/64); the key
// responsibilities are normalised over all Kfull components with the row's
// log-sum-exp, e^Q is taken relative to the row's maximum over all components,
// and the CTA writes its partial numerator and denominator, which the combine
// kernel sums over component slices (every term is a sum over components).
// SEG = true (with SLICE = false): the segment-parallel form.  CTA i scans the
// chunks [t0, t1) of the (head, chunk) list given by the plan S; a range that starts
// inside a head first sums its prefix from the prefix pass's partial slots (into the
// fp32 state and its bf16 snapshot), and at a head boundary inside the range the state
// restarts from zero and the next head's parameter block is loaded.
template <bool SLICE, bool SEG>
__global__ void __launch_bounds__(kCThreads, 1)
tc_causal_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                 const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                 CausalArgs A, const __grid_constant__ typename SegArg<SEG>::type S) {
    using C = CausalCfg;
    constexpr int K = KC;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + C::OFF_BAR);
    uint64_t *qfull = bars, *qempty = qfull + 2, *kfull = qempty + 2, *kempty = kfull + 2;
    uint64_t *vfull = kempty + 2, *vempty = vfull + 2;
    uint64_t *w_full = vempty + 2, *ak_full = w_full + 1, *d1k_full = ak_full + 1, *aq_full = d1k_full + 1;
    uint64_t *d1q_full = aq_full + 1, *g_full = d1q_full + 1, *g_empty = g_full + 1, *e_full = g_empty + 1;
    // T buffer: ta_full (first half computed), ta_free (first half read), tb2_full (second half
    // computed); tb_full: the masked bf16 tile is complete (T read).  The read of chunk c
    // commits tb0_free once it has consumed the first half of the masked tile and eq_free once
    // it has consumed e^Q(c).
    uint64_t *ta_full = e_full + 1, *ta_free = ta_full + 1, *tb2_full = ta_free + 1, *tb0_free = tb2_full + 1;
    uint64_t *tb_full = tb0_free + 1, *d3_full = tb_full + 1, *d3_empty = d3_full + 1, *eq_free = d3_empty + 1;
    uint64_t *s_upd = eq_free + 1, *s_ready = s_upd + 1, *sb_empty = s_ready + 2;
    uint64_t *fin1 = sb_empty + 2, *fin2 = fin1 + 1;
    uint64_t *w_empty = fin2 + 1;                      // segment-parallel form: parameter block consumed
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(w_empty + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // this CTA's chunks: all chunks of head blockIdx.x, or (segment-parallel form) the range
    // [t0c, t0c + nch) of the (head, chunk) list, which may start inside a head (mid) and
    // cross into the next; local chunk c is chunk cc of head gh (locate)
    const int hch = A.nch;
    int t0c = (int)blockIdx.x * hch, nch = hch;
    if constexpr (SEG) {
        const long long tt = (long long)A.G * hch;
        t0c = (int)(((long long)blockIdx.x * tt) / S.ns);
        nch = (int)(((long long)(blockIdx.x + 1) * tt) / S.ns) - t0c;
    }
    const int g = t0c / hch, cc0 = t0c - g * hch;
    const bool mid = SEG && cc0 != 0;
    auto locate = [&](int c, int &gh, int &cc) {
        cc = cc0 + c;
        gh = g;
        while (cc >= hch) { cc -= hch; ++gh; }
    };
    const int ks = SLICE ? (int)blockIdx.y : 0, vs = SLICE ? (int)blockIdx.z : 0;   // component / value slice
    grid_dep_launch();
    // direct form: the compute groups put the head's parameter loads in flight before the prologue
    constexpr int kTeam = 3 * kWgThreads, kTeamBar = 4;
    const int ttid = (int)threadIdx.x - kWGroups * 32;
    ParamLoads<K, kTeam> pld;
    if (!SLICE && !SEG && ttid >= 0) {
        const int h = g % A.H;
        pld.issue(ttid, A.mu + (size_t)h * K * DR, A.rho + (size_t)h * K * DR, A.alpha + (size_t)h * K);
    }

    if (threadIdx.x == 0) {
        for (int s = 0; s < 2; ++s) {
            mbar_init(&qfull[s], 1); mbar_init(&qempty[s], 1); mbar_init(&kfull[s], 1); mbar_init(&kempty[s], 1);
            mbar_init(&vfull[s], 1); mbar_init(&vempty[s], 1); mbar_init(&s_ready[s], 1); mbar_init(&sb_empty[s], 1);
        }
        for (uint64_t *b = w_full; b <= s_upd; ++b) mbar_init(b, 1);
        mbar_init(fin1, 1); mbar_init(fin2, 1); mbar_init(w_empty, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    // ONES atom column (element 0 of every row = 1.0 bf16) and the constant rows of both
    // state operands: row 65 = 1 (gives sum_k e^Q_ik), rows 66..79 = 0, rows 0..64 of buffer 0 = 0
    // (the state before the first chunk).
    for (uint32_t e = threadIdx.x; e < kTileBytes / 16; e += blockDim.x)
        reinterpret_cast<uint4 *>(sm + C::OFF_ONES)[e] = make_uint4(0, 0, 0, 0);
    // masked T tile: groups of 32 keys above a row quarter's diagonal are never written
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
    // the state operand for chunk 0 is ready (zero), unless the range starts inside a head
    if (threadIdx.x == 0 && !mid) mbar_arrive(&s_ready[0]);

    if (warp == kWProd) {
        if (lane == 0) {
            // the first tiles do not depend on the previous kernel; the parameter block does
            int qi = 0, ki = 0, vi = 0, gh, cc;
            for (; ki < 2 && ki < nch; ++ki) {
                locate(ki, gh, cc);
                mbar_arrive_expect_tx(&kfull[ki], kTileBytes);
                tma_load_3d(sm + C::OFF_K + ki * kTileBytes, &tm_k, &kfull[ki], 0, cc * TM, gh);
            }
            for (; qi < 2 && qi < nch; ++qi) {
                locate(qi, gh, cc);
                mbar_arrive_expect_tx(&qfull[qi], kTileBytes);
                tma_load_3d(sm + C::OFF_Q + qi * kTileBytes, &tm_q, &qfull[qi], 0, cc * TM, gh);
            }
            for (; vi < 2 && vi < nch; ++vi) {
                locate(vi, gh, cc);
                mbar_arrive_expect_tx(&vfull[vi], kTileBytes);
                tma_load_3d(sm + C::OFF_V + vi * kTileBytes, &tm_v, &vfull[vi], 64 * vs, cc * TM, gh);
            }
            // segment-parallel form: the parameter blocks (tc_params) of the range's heads, one
            // at a time through the one buffer, each once the previous head's MMAs are done with it
            int p_loaded = 0;
            int nheads = 0;
            if (SEG) {
                nheads = (cc0 + nch - 1) / hch + 1;
                grid_dep_wait();
                mbar_arrive_expect_tx(w_full, param_bytes(K));
                bulk_load(sm + C::OFF_P, A.params + (size_t)(g % A.H) * A.param_stride, param_bytes(K), w_full);
                p_loaded = 1;
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
            while ((qi < nch || ki < nch || vi < nch || p_loaded < nheads) && !*abort_flag) {
                bool progress = false;
                if (SEG && p_loaded < nheads && mbar_test(w_empty, (p_loaded - 1) & 1)) {
                    mbar_arrive_expect_tx(w_full, param_bytes(K));
                    bulk_load(sm + C::OFF_P, A.params + (size_t)((g + p_loaded) % A.H) * A.param_stride,
                              param_bytes(K), w_full);
                    ++p_loaded;
                    progress = true;
                }
                if (ki < nch && (ki < 2 || mbar_test(&kempty[ki & 1], ((ki >> 1) - 1) & 1))) {
                    locate(ki, gh, cc);
                    (void)GMA_IN_BOUNDS(gh < A.G && cc < hch, A.status);
                    mbar_arrive_expect_tx(&kfull[ki & 1], kTileBytes);
                    tma_load_3d(sm + C::OFF_K + (ki & 1) * kTileBytes, &tm_k, &kfull[ki & 1], 0, cc * TM, gh);
                    ++ki;
                    progress = true;
                }
                if (qi < nch && (qi < 2 || mbar_test(&qempty[qi & 1], ((qi >> 1) - 1) & 1))) {
                    locate(qi, gh, cc);
                    mbar_arrive_expect_tx(&qfull[qi & 1], kTileBytes);
                    tma_load_3d(sm + C::OFF_Q + (qi & 1) * kTileBytes, &tm_q, &qfull[qi & 1], 0, cc * TM, gh);
                    ++qi;
                    progress = true;
                }
                if (vi < nch && (vi < 2 || mbar_test(&vempty[vi & 1], ((vi >> 1) - 1) & 1))) {
                    locate(vi, gh, cc);
                    mbar_arrive_expect_tx(&vfull[vi & 1], kTileBytes);
                    tma_load_3d(sm + C::OFF_V + (vi & 1) * kTileBytes, &tm_v, &vfull[vi & 1], 64 * vs, cc * TM, gh);
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
            if (SEG && p_loaded > 0) wait_ignoring_abort(w_full, (p_loaded - 1) & 1, A.status);
        }
    } else if (warp == kWIss1) {
        // log-density MMAs: scores = [x, x^2/256] . W^T, keys then queries of each chunk
        if (true) {                                  // the whole warp, converged
            const uint32_t pw = smem_u32(sm + C::OFF_P), ca = smem_u32(sm + C::OFF_CA);
            bool ok = mbar_wait_warp(w_full, 0, ab, kDevErrTimeout);
            for (int c = 0; c < nch && ok; ++c) {
                int gh, cc;
                locate(c, gh, cc);
                // segment-parallel form: the next head's parameter block
                if (SEG && c > 0 && cc == 0 && !(ok = mbar_wait_warp(w_full, (gh - g) & 1, ab, kDevErrTimeout))) break;
                if (!(ok = mbar_wait_warp(ak_full, c & 1, ab, kDevErrTimeout))) break;
                tc_fence_after();
                issue_logdensity<K>(tmem + C::COL_D1K, tmem + C::COL_AK, pw, ca);
                mma_commit(d1k_full);
                if (!(ok = mbar_wait_warp(aq_full, c & 1, ab, kDevErrTimeout))) break;
                tc_fence_after();
                issue_logdensity<K>(tmem + C::COL_D1Q, tmem + C::COL_AQ, pw, ca);
                mma_commit(d1q_full);
                if (SEG && cc == hch - 1 && c + 1 < nch) mma_commit(w_empty);   // the head's last chunk
            }
            mma_commit(fin1);
            wait_ignoring_abort(fin1, 0, A.status);
        }
    } else if (warp == kWIss2) {
        if (true) {                                  // the whole warp, converged
            constexpr uint32_t idesc_t = idesc_f16(1, 1, 0, 0, TM, 64);       // e^Q (TMEM) . gamma^K^T, 64 keys
            constexpr uint32_t idesc_u = idesc_f16(1, 1, 1, 1, TM, K);       // [V | 1]^T . gamma^K
            constexpr uint32_t idesc_r1 = idesc_f16(1, 1, 0, 0, TM, NOUT);   // e^Q . [S | z | 1]
            constexpr uint32_t idesc_r2 = idesc_f16(1, 1, 0, 1, TM, NOUT);   // T . [V | 1]
            const uint32_t gaddr = smem_u32(sm + C::OFF_G), ones = smem_u32(sm + C::OFF_ONES);
            const uint64_t gk = sdesc_sw128(gaddr, 16, 1024);                // gamma^K as K-major B (N = keys)
            const uint64_t gm = sdesc_sw128(gaddr, kTileBytes, 1024);        // gamma^K as MN-major B (N = k)
            const uint64_t tbd = sdesc_sw128(smem_u32(sm + C::OFF_TB), 16, 1024);
            const uint32_t eq = tmem + C::COL_EQ;
            // T(c), keys 0..63 = e^Q(c) . gamma^K(c)[0:64]^T, once e^Q(c) and gamma^K(c) are in place
            // (the T buffer is free: its previous chunk's second half has been masked)
            auto t_first_half = [&](int c) -> bool {
                if (!(mbar_wait_warp(e_full, c & 1, ab, kDevErrTimeout) &&
                      mbar_wait_warp(g_full, c & 1, ab, kDevErrTimeout)))
                    return false;
                tc_fence_after();
#pragma unroll
                for (int ks = 0; ks < K / 16; ++ks)
                    mma_ts(tmem + C::COL_T, eq + ks * 8, gk + (uint64_t)((ks * 32u) >> 4), idesc_t, ks > 0);
                mma_commit(ta_full);
                return true;
            };
            bool ok = t_first_half(0);
            for (int c = 0; c < nch && ok; ++c) {
                const int s = c & 1;
                // T(c), keys 64..127, once the first half has been read
                if (!(ok = mbar_wait_warp(ta_free, c & 1, ab, kDevErrTimeout))) break;
                tc_fence_after();
#pragma unroll
                for (int ks = 0; ks < K / 16; ++ks)
                    mma_ts(tmem + C::COL_T, eq + ks * 8, gk + (uint64_t)((64u * 128u + ks * 32u) >> 4), idesc_t,
                           ks > 0);
                mma_commit(tb2_full);
                // state update: [S | z]^T += [V | 1 | 0]^T . gamma^K, once the previous state is snapshotted
                if (!(ok = mbar_wait_warp(&vfull[s], (c >> 1) & 1, ab, kDevErrTimeout) &&
                           mbar_wait_warp(&s_ready[c & 1], (c >> 1) & 1, ab, kDevErrTimeout)))
                    break;
                tc_fence_after();
                const uint32_t va = smem_u32(sm + C::OFF_V + s * kTileBytes);
                const uint64_t vd = sdesc_sw128(va, ones - va, 1024);
                // the state restarts at a head's first chunk (a range starting inside a head holds its prefix)
                int gh, cc;
                locate(c, gh, cc);
                const bool fresh = SEG ? cc == 0 : c == 0;
#pragma unroll
                for (int ks = 0; ks < 8; ++ks)
                    mma_ss(tmem + C::COL_S, vd + (uint64_t)(ks * 128), gm + (uint64_t)(ks * 128), idesc_u,
                           !(fresh && ks == 0));
                mma_commit(s_upd);
                mma_commit(g_empty);
                // read(c) = mask(T) . [V | 1] + e^Q(c) . [S | z | 1]_{c-1}, in the order that frees
                // what chunk c + 1 needs first: the first half of the masked tile, then e^Q; T(c + 1)'s
                // first half enters the tensor pipe before the rest of the read.
                ok = mbar_wait_warp(tb_full, c & 1, ab, kDevErrTimeout);
                if (ok && c >= 1) ok = mbar_wait_warp(d3_empty, (c - 1) & 1, ab, kDevErrTimeout);
                if (!ok) break;
                tc_fence_after();
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    mma_ss(tmem + C::COL_D3, tbd + (uint64_t)((ks * 32u) >> 4), vd + (uint64_t)(ks * 128), idesc_r2,
                           ks > 0);
                mma_commit(tb0_free);
                const uint64_t sbd = sdesc_sw128(smem_u32(sm + C::OFF_SB + (c & 1) * C::SBB), 16, 1024);
#pragma unroll
                for (int ks = 0; ks < K / 16; ++ks)
                    mma_ts(tmem + C::COL_D3, eq + ks * 8, sbd + (uint64_t)((ks * 32u) >> 4), idesc_r1, 1);
                mma_commit(eq_free);
                if (c + 1 < nch && !(ok = t_first_half(c + 1))) break;
#pragma unroll
                for (int ks = 4; ks < 8; ++ks)
                    mma_ss(tmem + C::COL_D3, tbd + (uint64_t)((kTileBytes + (ks & 3) * 32u) >> 4),
                           vd + (uint64_t)(ks * 128), idesc_r2, 1);
                mma_commit(d3_full);
                mma_commit(&sb_empty[c & 1]);
                mma_commit(&vempty[s]);
            }
            mma_commit(fin2);
            wait_ignoring_abort(fin2, 0, A.status);
        }
    } else {
        RowThread rt;
        rt.wg = (warp - kWGroups) >> 2;
        rt.r = 32u * (warp & 3) + lane;
        rt.lane_off = (uint32_t)(32 * (warp & 3)) << 16;
        rt.wtid = threadIdx.x - kWGroups * 32 - rt.wg * kWgThreads;
        const bool elected = rt.wtid == 0;
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
        if (!SLICE && !SEG) {
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
            auto convert_k = [&](int c) -> bool {
                const bool w = mbar_wait(&kfull[c & 1], (c >> 1) & 1, ab, kDevErrTimeout);
                if (!wg_all(rt, w)) return false;
                convert_row_call(sm + C::OFF_K + (c & 1) * kTileBytes, rt.r, tmem + rt.lane_off + C::COL_AK);
                tmem_st_wait();
                tc_fence_before();
                wg_sync(rt);
                if (elected) { mbar_arrive(ak_full); mbar_arrive(&kempty[c & 1]); }
                return true;
            };
            bool ok = convert_k(0);
            if constexpr (SEG) {
                if (mid && ok) {
                    // the prefix state of chunks [0, cc0) of head g: the partial slots of this head's
                    // prefix segments up to this CTA's, in order, each over the prefix-pass CTAs that
                    // covered it (fixed order); into the fp32 state in TMEM and the bf16 snapshot
                    grid_dep_wait();
                    const int s_last = S.scan_seg[blockIdx.x];
                    int s_first = s_last;
                    while (s_first > 0 && S.seg[s_first - 1].g == g) --s_first;
                    uint32_t acc[K];
#pragma unroll
                    for (int k = 0; k < K; ++k) acc[k] = 0u;
                    if (rt.r <= DVV) {
                        for (int sg = s_first; sg <= s_last; ++sg)
                            for (int p = S.seg[sg].plo; p <= S.seg[sg].phi; ++p) {
                                if (!GMA_IN_BOUNDS(p + sg < A.nslots && S.seg[sg].g == g, A.status)) continue;
                                const float4 *src = reinterpret_cast<const float4 *>(
                                    A.partials + ((size_t)(p + sg) * (DVV + 1) + rt.r) * K);
#pragma unroll
                                for (int k = 0; k < K / 4; ++k) {
                                    const float4 f = src[k];
                                    acc[4 * k] = __float_as_uint(__uint_as_float(acc[4 * k]) + f.x);
                                    acc[4 * k + 1] = __float_as_uint(__uint_as_float(acc[4 * k + 1]) + f.y);
                                    acc[4 * k + 2] = __float_as_uint(__uint_as_float(acc[4 * k + 2]) + f.z);
                                    acc[4 * k + 3] = __float_as_uint(__uint_as_float(acc[4 * k + 3]) + f.w);
                                }
                            }
                        uint8_t *row = sm + C::OFF_SB;
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            uint4 o;
                            o.x = pack_bf16(__uint_as_float(acc[8 * j + 0]), __uint_as_float(acc[8 * j + 1]));
                            o.y = pack_bf16(__uint_as_float(acc[8 * j + 2]), __uint_as_float(acc[8 * j + 3]));
                            o.z = pack_bf16(__uint_as_float(acc[8 * j + 4]), __uint_as_float(acc[8 * j + 5]));
                            o.w = pack_bf16(__uint_as_float(acc[8 * j + 6]), __uint_as_float(acc[8 * j + 7]));
                            *reinterpret_cast<uint4 *>(row + sw128_off(rt.r, j)) = o;
                        }
                    }
                    tmem_st32(tmem + rt.lane_off + C::COL_S, acc);
                    tmem_st32(tmem + rt.lane_off + C::COL_S + 32, acc + 32);
                    tmem_st_wait();
                    fence_proxy_async_smem();
                    tc_fence_before();
                    wg_sync(rt);
                    if (elected) mbar_arrive(&s_ready[0]);
                }
            }
            for (int c = 0; c < nch && ok; ++c) {
                bool w = mbar_wait(d1k_full, c & 1, ab, kDevErrTimeout);
                if (c >= 1) w = w && mbar_wait(g_empty, (c - 1) & 1, ab, kDevErrTimeout);
                if (!(ok = wg_all(rt, w))) break;
                tc_fence_after();
                if (SLICE && c == 0) {
                    grid_dep_wait();
                    scale = head_scale(A.params, A.param_stride, g % A.H, A.Kfull);
                    stat_next = lse_row(0);
                }
                int gh, cc;
                locate(c, gh, cc);
                if (SEG && (c == 0 || cc == 0)) {
                    if (c == 0) grid_dep_wait();
                    scale = head_scale(A.params, A.param_stride, gh % A.H, K);
                }
                // gamma^K = softmax of the key scores; rows past the sequence end get 0
                uint32_t e[K / 2];
                float inv;
                if (SLICE) {
                    // normalised over all components by the row's log-sum-exp (loaded a chunk ahead)
                    const float off = stat_next;
                    if (c + 1 < nch) stat_next = lse_row(c + 1);
                    row_exp_offset<K>(tmem + rt.lane_off + C::COL_D1K, scale, off, e);
                    inv = 1.0f;
                } else {
                    row_exp_scaled<K>(tmem + rt.lane_off + C::COL_D1K, scale, e);
                    uint64_t acc[4] = {0, 0, 0, 0};
#pragma unroll
                    for (int t = 0; t < K / 2; ++t)
                        acc[t & 3] = f2_add(acc[t & 3], f2_pack(bf16_lo(e[t]), bf16_hi(e[t])));
                    float s0, s1, s2, s3, s4, s5, s6, s7;
                    f2_unpack(acc[0], s0, s1); f2_unpack(acc[1], s2, s3);
                    f2_unpack(acc[2], s4, s5); f2_unpack(acc[3], s6, s7);
                    const float total = ((s0 + s1) + (s2 + s3)) + ((s4 + s5) + (s6 + s7));
                    inv = cc * TM + (int)rt.r < A.N ? 1.0f / total : 0.f;
                }
                const uint64_t inv2 = f2_pack(inv, inv);
#pragma unroll
                for (int j = 0; j < K / 8; ++j) {
                    uint32_t wv[4];
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        float ga, gb;
                        f2_unpack(f2_mul(f2_pack(bf16_lo(e[4 * j + u]), bf16_hi(e[4 * j + u])), inv2), ga, gb);
                        wv[u] = pack_bf16(ga, gb);
                    }
                    *reinterpret_cast<uint4 *>(sm + C::OFF_G + sw128_off(rt.r, j)) = make_uint4(wv[0], wv[1], wv[2], wv[3]);
                }
                fence_proxy_async_smem();
                tc_fence_before();
                wg_sync(rt);
                if (elected) mbar_arrive(g_full);
                // bf16 snapshot of the state after chunk c - 1, the read operand of chunk c (its
                // update went into the tensor pipe a chunk ago; the update of chunk c waits for it)
                if (c >= 1) {
                    const int b = c & 1;
                    w = mbar_wait(s_upd, (c - 1) & 1, ab, kDevErrTimeout);
                    if (c >= 2) w = w && mbar_wait(&sb_empty[b], ((c >> 1) - 1) & 1, ab, kDevErrTimeout);
                    if (!(ok = wg_all(rt, w))) break;
                    tc_fence_after();
                    uint32_t v[K];
                    tmem_ld32(tmem + rt.lane_off + C::COL_S, v);
                    tmem_ld32(tmem + rt.lane_off + C::COL_S + 32, v + 32);
                    tmem_ld_wait();
                    if (SEG && cc == 0) {                    // a new head: its state before chunk 0 is zero
#pragma unroll
                        for (int k = 0; k < K; ++k) v[k] = 0u;
                    }
                    if (rt.r <= DVV) {
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
                    wg_sync(rt);
                    if (elected) mbar_arrive(&s_ready[b]);
                }
                if (c + 1 >= nch) break;
                if (!(ok = convert_k(c + 1))) break;
            }
        } else if (rt.wg == 1) {
            // ---------------- query group
            auto convert_q = [&](int c) -> bool {
                const bool w = mbar_wait(&qfull[c & 1], (c >> 1) & 1, ab, kDevErrTimeout);
                if (!wg_all(rt, w)) return false;
                convert_row_call(sm + C::OFF_Q + (c & 1) * kTileBytes, rt.r, tmem + rt.lane_off + C::COL_AQ);
                tmem_st_wait();
                tc_fence_before();
                wg_sync(rt);
                if (elected) { mbar_arrive(aq_full); mbar_arrive(&qempty[c & 1]); }
                return true;
            };
            auto epilogue = [&](int c) {
                // called once read(c) is known complete (d3_full(c) waited)
                // out = num / (den + eps * sum_k e^Q_k)
                uint32_t v0[32], v1[32], dz[4];
                tmem_ld32(tmem + rt.lane_off + C::COL_D3, v0);
                tmem_ld32(tmem + rt.lane_off + C::COL_D3 + 32, v1);
                tmem_ld4(tmem + rt.lane_off + C::COL_D3 + 64, dz);
                tmem_ld_wait();
                const float den = __uint_as_float(dz[0]) + A.eps * __uint_as_float(dz[1]);
                if (SLICE) {
                    // partial numerator (bf16) and denominator of this component slice
                    tc_fence_before();
                    wg_sync(rt);
                    if (elected) mbar_arrive(d3_empty);
                    const int row = c * TM + (int)rt.r;
                    if (row < A.N && GMA_IN_BOUNDS(ks < A.Kfull / KC && g < A.G && 64 * vs < A.dvt, A.status)) {
                        const size_t pr = ((size_t)ks * A.G + g) * A.N + row;
                        uint4 *dst = reinterpret_cast<uint4 *>(A.pnum + pr * A.dvt + 64 * vs);
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            const uint32_t *src = j < 4 ? v0 + 8 * j : v1 + 8 * (j - 4);
                            dst[j] = make_uint4(pack_bf16(__uint_as_float(src[0]), __uint_as_float(src[1])),
                                                pack_bf16(__uint_as_float(src[2]), __uint_as_float(src[3])),
                                                pack_bf16(__uint_as_float(src[4]), __uint_as_float(src[5])),
                                                pack_bf16(__uint_as_float(src[6]), __uint_as_float(src[7])));
                        }
                        if (vs == 0) A.pden[pr] = den;
                    }
                    return;
                }
                const float rd = 1.0f / den;
                const uint64_t rd2 = f2_pack(rd, rd);
                if (elected) bulk_wait_group_read<0>();          // the previous store has left the staging tile
                tc_fence_before();
                wg_sync(rt);
                if (elected) mbar_arrive(d3_empty);
                uint8_t *ob = sm + C::OFF_O;
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
                    *reinterpret_cast<uint4 *>(ob + sw128_off(rt.r, j)) = make_uint4(o[0], o[1], o[2], o[3]);
                }
                fence_proxy_async_smem();
                wg_sync(rt);
                if (elected) {
                    int gh, cc;
                    locate(c, gh, cc);
                    (void)GMA_IN_BOUNDS(gh < A.G && cc < hch, A.status);
                    tma_store_3d(&tm_o, ob, 0, cc * TM, gh);
                    bulk_commit_group();
                }
            };
            bool ok = convert_q(0);
            for (int c = 0; c <= nch && ok; ++c) {
                if (c < nch) {
                    bool w = mbar_wait(d1q_full, c & 1, ab, kDevErrTimeout);
                    if (!(ok = wg_all(rt, w))) break;
                    tc_fence_after();
                    if (SLICE && c == 0) {
                        grid_dep_wait();
                        scale = head_scale(A.params, A.param_stride, g % A.H, A.Kfull);
                        stat_next = max_row(0);
                    }
                    if (SEG) {
                        int gh, cc;
                        locate(c, gh, cc);
                        if (c == 0 || cc == 0) {
                            if (c == 0) grid_dep_wait();
                            scale = head_scale(A.params, A.param_stride, gh % A.H, K);
                        }
                    }
                    uint32_t e[K / 2];
                    if (SLICE) {
                        // relative to the row's maximum over all components (loaded a chunk ahead)
                        const float off = stat_next;
                        if (c + 1 < nch) stat_next = max_row(c + 1);
                        row_exp_offset<K>(tmem + rt.lane_off + C::COL_D1Q, scale, off, e);
                    } else {
                        row_exp_scaled<K>(tmem + rt.lane_off + C::COL_D1Q, scale, e);
                    }
                    // e^Q(c) replaces e^Q(c - 1) once the read of chunk c - 1 has consumed it
                    if (c >= 1) {
                        w = mbar_wait(eq_free, (c - 1) & 1, ab, kDevErrTimeout);
                        if (!(ok = wg_all(rt, w))) break;
                        tc_fence_after();
                    }
                    tmem_st32(tmem + rt.lane_off + C::COL_EQ, e);
                    tmem_st_wait();
                    tc_fence_before();
                    wg_sync(rt);
                    if (elected) mbar_arrive(e_full);
                    // the scores of chunk c have been read: the next query tile may overwrite them
                    if (c + 1 < nch && !(ok = convert_q(c + 1))) break;
                }
                // read(c - 1): its epilogue, off the chunk-to-chunk chain
                if (c >= 1) {
                    const bool w = mbar_wait(d3_full, (c - 1) & 1, ab, kDevErrTimeout);
                    if (!(ok = wg_all(rt, w))) break;
                    tc_fence_after();
                    epilogue(c - 1);
                }
            }
            if (elected) bulk_wait_group<0>();
        } else {
            // ---------------- output group
            // Row quarter q = warp & 3 holds rows 32q..32q+31.  A group of 32 keys is copied
            // whole below the quarter's diagonal, selected (j <= r) on it, and never touched
            // above it (those entries of the masked tile stay zero from the start).
            const int q = warp & 3;
            auto mask_group = [&](const uint32_t *v, int key0, bool diag, uint8_t *half, int cc) {
                uint32_t pk[16];
                if (diag) {
                    // the group straddles the diagonal: keep keys key0 + u with u <= r - key0
                    const int rr = (int)rt.r - key0;
#pragma unroll
                    for (int t = 0; t < 16; ++t) {
                        const float a = 2 * t <= rr ? __uint_as_float(v[2 * t]) : 0.f;
                        const float b2 = 2 * t + 1 <= rr ? __uint_as_float(v[2 * t + 1]) : 0.f;
                        pk[t] = pack_bf16(a, b2);
                    }
                } else {
                    // wholly below the diagonal (warp-uniform branch): convert only
#pragma unroll
                    for (int t = 0; t < 16; ++t)
                        pk[t] = pack_bf16(__uint_as_float(v[2 * t]), __uint_as_float(v[2 * t + 1]));
                }
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4)
                    *reinterpret_cast<uint4 *>(half + sw128_off(rt.r, cc * 4 + q4)) =
                        make_uint4(pk[4 * q4], pk[4 * q4 + 1], pk[4 * q4 + 2], pk[4 * q4 + 3]);
            };
            // one half of T (64 keys starting at key0) from TMEM into the masked bf16 tile
            auto mask_half = [&](int key0, uint8_t *half) {
                const int g0 = key0 / 32;                     // global index of the half's first group
                if (q < g0) return;                           // the whole half lies above the diagonal
                uint32_t v0[32], v1[32];
                tmem_ld32(tmem + rt.lane_off + C::COL_T, v0);
                tmem_ld32(tmem + rt.lane_off + C::COL_T + 32, v1);
                tmem_ld_wait();
                mask_group(v0, key0, q == g0, half, 0);
                if (q > g0) mask_group(v1, key0 + 32, q == g0 + 1, half, 1);
            };
            bool ok = true;
            for (int c = 0; c < nch && ok; ++c) {
#pragma unroll 1
                for (int hh = 0; hh < 2; ++hh) {
                    // half hh (keys 64 hh .. 64 hh + 63) of T(c); that half of the masked tile is free
                    // once the read of chunk c - 1 has passed it (its first four k-steps / all of it)
                    bool w = mbar_wait(hh == 0 ? ta_full : tb2_full, c & 1, ab, kDevErrTimeout);
                    if (c >= 1) w = w && mbar_wait(hh == 0 ? tb0_free : d3_full, (c - 1) & 1, ab, kDevErrTimeout);
                    if (!(ok = wg_all(rt, w))) break;
                    tc_fence_after();
                    mask_half(64 * hh, sm + C::OFF_TB + hh * kTileBytes);
                    if (hh == 1) fence_proxy_async_smem();
                    tc_fence_before();
                    wg_sync(rt);
                    if (elected) {
                        mbar_arrive(hh == 0 ? ta_free : tb_full);
                    }
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
                                 cudaStream_t s, bool slices, const SegTable *seg) {
    CUtensorMap tq, tk, tv, to;
    if (!make_map(&tq, Qx, p.G, p.N, DR) || !make_map(&tk, Kx, p.G, p.N, DR) || !make_map(&tv, V, p.G, p.N, p.dv) ||
        !make_map(&to, slices ? V : out, p.G, p.N, p.dv))
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
        a.partials = reinterpret_cast<const float *>(ws + L.part);
        a.nslots = seg ? seg->np + seg->nseg + 1 : 0;
    }
    if (seg) {
        auto kern = tc_causal_kernel<false, true>;
        cudaError_t e = set_dyn_smem(reinterpret_cast<const void *>(kern), CausalCfg::BYTES);
        if (e != cudaSuccess) return e;
        return launch_dependent(kern, dim3(seg->ns), dim3(kCThreads), CausalCfg::BYTES, s, tq, tk, tv, to, a, *seg);
    }
    auto kern = slices ? tc_causal_kernel<true, false> : tc_causal_kernel<false, false>;
    cudaError_t e = set_dyn_smem(reinterpret_cast<const void *>(kern), CausalCfg::BYTES);
    if (e != cudaSuccess) return e;
    if (!slices) {
        // the first kernel of its forward: an ordinary launch, so that every input is final when
        // its CTAs start
        kern<<<dim3(p.G), dim3(kCThreads), CausalCfg::BYTES, s>>>(tq, tk, tv, to, a, NoSeg{});
        return cudaGetLastError();
    }
    return launch_dependent(kern, dim3(p.G, L.ns, L.nt), dim3(kCThreads), CausalCfg::BYTES, s, tq, tk, tv, to, a,
                            NoSeg{});
}

cudaError_t tc_causal(const Problem &p, const TcLayout &L, const void *Qx, const void *Kx, const void *V,
                      const float *mu, const float *rho, const float *alpha, void *out, char *ws, cudaStream_t s) {
    return launch_causal(p, L, Qx, Kx, V, mu, rho, alpha, out, ws, s, false, nullptr);
}

cudaError_t tc_causal_slices(const Problem &p, const TcLayout &L, const void *Qx, const void *Kx, const void *V,
                             char *ws, cudaStream_t s) {
    return launch_causal(p, L, Qx, Kx, V, nullptr, nullptr, nullptr, nullptr, ws, s, true, nullptr);
}

// ------------------------------------------------------------------ segment-parallel plan

// Used when the heads fill at most half of the SMs.  (With every SM running the scan, its
// instruction fetch, not its work, sets the chunk period: at 96 heads on 152 SMs the split
// measured a 44 % longer period per chunk and no net gain, so more heads keep one CTA each.)
// Scan ranges: ns CTAs, CTA i takes chunks [i Ttot / ns, (i + 1) Ttot / ns) of the (head,
// chunk) list, at least kMinSegChunks each, and only when that gives more CTAs than heads.
// Prefix segments: for each CTA i whose range starts at chunk a > 0 of head g, the chunks of
// g before a that belong to CTA i - 1's range.  Prefix-pass ranges: np CTAs over the
// concatenated segments, balanced the same way.
bool tc_seg_plan(const Problem &p, SegTable &T) {
    constexpr int kMinSegChunks = 4;
    std::memset(&T, 0, sizeof(T));
    const int nsm = sm_count();
    const int nch = (p.N + TM - 1) / TM;
    const long long tt = (long long)p.G * nch;
    if (nsm <= 0 || tt <= 0 || 2 * p.G > nsm) return false;
    const long long ns = std::min<long long>({(long long)std::min(nsm, kMaxScanCtas), tt / kMinSegChunks, tt});
    if (ns <= p.G) return false;
    T.ns = (int)ns;
    T.nch = nch;
    auto t0 = [&](long long i) { return (i * tt) / ns; };
    T.scan_seg[0] = -1;
    int vtot = 0;
    for (int i = 1; i < T.ns; ++i) {
        const long long a0 = t0(i), g = a0 / nch, a = a0 - g * nch;
        if (a == 0) { T.scan_seg[i] = -1; continue; }
        const long long st = std::max(t0(i - 1), g * nch) - g * nch;
        SegEntry &e = T.seg[T.nseg];
        e.g = (int32_t)g;
        e.a = (int16_t)st;
        e.len = (int16_t)(a - st);
        T.scan_seg[i] = (int16_t)T.nseg++;
        vtot += (int)(a - st);
    }
    T.vtot = vtot;
    T.np = vtot > 0 ? std::min({nsm, kMaxScanCtas, vtot}) : 0;
    // prefix-pass CTA p covers [p vtot / np, (p + 1) vtot / np) of the concatenated segments
    int sg = 0, off = 0;                                  // segment and the virtual offset of its start
    for (int q = 0; q < T.np; ++q) {
        const int v0 = (int)(((long long)q * vtot) / T.np);
        while (off + T.seg[sg].len <= v0) { off += T.seg[sg].len; ++sg; }
        T.pre_v[q] = (int16_t)sg;
        T.pre_jj[q] = (int16_t)(v0 - off);
    }
    off = 0;
    for (int k = 0; k < T.nseg; ++k) {
        const int lo = off, hi = off + T.seg[k].len - 1;   // virtual range of segment k
        int plo = (int)(((long long)lo * T.np) / vtot), phi = (int)(((long long)hi * T.np) / vtot);
        while (plo > 0 && ((long long)plo * vtot) / T.np > lo) --plo;
        while (((long long)(plo + 1) * vtot) / T.np <= lo) ++plo;
        while (phi > 0 && ((long long)phi * vtot) / T.np > hi) --phi;
        while (((long long)(phi + 1) * vtot) / T.np <= hi) ++phi;
        T.seg[k].plo = (int16_t)plo;
        T.seg[k].phi = (int16_t)phi;
        off += T.seg[k].len;
    }
    return true;
}

TcLayout tc_seg_layout(const Problem &p, const SegTable &T) {
    TcLayout L{};
    L.T = T.nch;
    L.Ttot = T.nch * p.G;
    L.ncta = T.ns;
    L.ns = L.nt = 1;
    L.param_stride = align1k(param_bytes(p.K));
    L.params = align_up(kHeaderBytes);
    L.part = align_up(L.params + (size_t)p.H * L.param_stride);        // [np + nseg][dv + 1][K] f32
    L.mem = L.part;
    L.total = align_up(L.part + sizeof(float) * (size_t)(T.np + T.nseg + 1) * (DVV + 1) * p.K);
    return L;
}

cudaError_t tc_causal_seg(const Problem &p, const TcLayout &L, const SegTable &T, const void *Qx, const void *Kx,
                          const void *V, void *out, char *ws, cudaStream_t s) {
    return launch_causal(p, L, Qx, Kx, V, nullptr, nullptr, nullptr, out, ws, s, false, &T);
}

}  // namespace gma
