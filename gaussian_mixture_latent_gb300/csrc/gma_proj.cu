// Input projections ("Gaussian Mixture Attention", Huang & Raza, 2026, section 3.1,
// Eq. 4): per head h,  Qx = X W_Q[h],  Kx = X W_K[h],  V = X W_V[h].
//
// One persistent tcgen05 GEMM over the output columns of every head's
// [W_Q | W_K | W_V] (bf16 operands, fp32 accumulation in TMEM), whose epilogue
// rounds to bf16 and writes each 128-row x 64-column block by TMA straight into
// the [B, H, N, .] layout gma_forward() reads.  A tile is 128 rows of one batch
// entry by four 64-column blocks (N = 256), the k-loop runs over the model width
// D in blocks of 64 through a 4-stage TMA ring, and two TMEM accumulators let the
// epilogue of one tile overlap the MMAs of the next.
//
// CTAs work in clusters of kCl = 4 on tile groups: four adjacent row tiles of the same
// column blocks.  Each CTA loads its own X rows and a quarter of the W blocks, which TMA
// multicasts into every CTA's stage, so a CTA pulls 24 KB per stage from L2 instead of
// 48 KB.  A stage is refilled once every CTA's MMAs have read it (each MMA commit
// arrives on the stage's barrier in every CTA of the cluster).  Groups are taken in
// row-block major order (the clusters working at a time share their X rows in L2; W
// stays in L2); row tiles past the last are copies of it whose results are not stored.
//
// Warps: 0 TMA producer, 1 TMEM owner and MMA issuer, 2-5 epilogue (thread r owns
// accumulator row r).  Every wait is bounded; a timeout posts GMA_ERR_TIMEOUT.
#include <cuda.h>
#include <cuda_bf16.h>

#include <algorithm>
#include <cstdint>

#include "gma_internal.h"
#include "gma_sm100.cuh"
#include "gma_tc_common.cuh"

namespace gma {

using namespace sm100;
using namespace tc;

namespace {

// ---- cluster helpers
__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// TMA tile load written to the same shared-memory offset of every CTA in `mask`, each
// CTA's barrier at `bar`'s offset receiving the bytes it got
__device__ __forceinline__ void tma_load_3d_mc(void *dst, const CUtensorMap *map, uint64_t *bar, int c0, int c1,
                                               int c2, uint16_t mask) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.multicast::cluster"
        " [%0], [%1, {%3, %4, %5}], [%2], %6;"
        ::"r"(smem_u32(dst)), "l"(map), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2), "h"(mask)
        : "memory");
}
// Arrive on `bar` (same offset) in every CTA of `mask` once the MMAs issued so far have
// completed.  Warp-collective, like mma_commit.
__device__ __forceinline__ void mma_commit_mc(uint64_t *bar, uint16_t mask) {
    asm volatile(
        "{\n\t.reg .pred e;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;\n\t}"
        ::"r"(smem_u32(bar)), "h"(mask)
        : "memory");
}
// Arrive on the barrier at `bar`'s offset in CTA `peer` of the cluster.
__device__ __forceinline__ void mbar_arrive_peer(uint64_t *bar, uint32_t peer) {
    asm volatile(
        "{\n\t.reg .b32 ra;\n\t"
        "mapa.shared::cluster.u32 ra, %0, %1;\n\t"
        "mbarrier.arrive.release.cluster.shared::cluster.b64 _, [ra];\n\t}"
        ::"r"(smem_u32(bar)), "r"(peer)
        : "memory");
}

constexpr int kCl = 4;                        // CTAs per cluster (row tiles sharing their W blocks)
constexpr int PM = 128;                       // rows per tile
constexpr int PBN = 64;                       // output columns per block
constexpr int PNB = 4;                        // blocks per tile (MMA N up to 256)
constexpr int PKB = 64;                       // model-width columns per stage
constexpr int PS = 4;                         // ring stages
constexpr uint32_t kABytes = PM * PKB * 2;    // X stage: 128 rows x 64, K-major, 128-byte swizzle
constexpr uint32_t kBBlk = PKB * PBN * 2;     // one W block: 64 rows (k) x 64 columns, MN-major
constexpr uint32_t kStage = kABytes + PNB * kBBlk;
constexpr int kPThreads = 192;
constexpr int kWProd = 0, kWMma = 1, kWEpi = 2;

struct ProjCfg {
    static constexpr uint32_t OFF_S = 0;                          // PS stages: [X | W blocks]
    static constexpr uint32_t OFF_E = OFF_S + PS * kStage;        // 2 epilogue buffers (bf16 128 x 64)
    static constexpr uint32_t OFF_BAR = OFF_E + 2 * kTileBytes;
    static constexpr uint32_t BYTES = OFF_BAR + 256 + 1024;
    static constexpr uint32_t ACC_COLS = PBN * PNB;               // 256 fp32 columns per accumulator
    static constexpr uint32_t TMEM_COLS = 2 * ACC_COLS;
};
static_assert(ProjCfg::BYTES <= 232448, "projection kernel exceeds the shared-memory opt-in limit");
static_assert(kStage % 1024 == 0 && ProjCfg::OFF_E % 1024 == 0, "operand blocks must be 1024-byte aligned");

struct ProjArgs {
    int B, N, H, nkb;             // nkb = D / 64
    int nqb, nvb, nbh;            // 64-column blocks per head: of W_Q (= of W_K), of W_V, in all
    int mt_per_b, n_mtiles, n_ntiles, n_pairs, nblocks;   // groups: (row tiles kCl m .. kCl m + kCl - 1; column tile)
    unsigned *status;
};

// Output column block cb -> (tensor 0 = Q, 1 = K, 2 = V; head; 64-column block within it).
struct BlockMap {
    int which, h, col;
};
__device__ __forceinline__ BlockMap map_block(const ProjArgs &A, int cb) {
    BlockMap m;
    m.h = cb / A.nbh;
    const int r = cb - m.h * A.nbh;
    m.which = r < A.nqb ? 0 : (r < 2 * A.nqb ? 1 : 2);
    m.col = r - m.which * A.nqb;
    return m;
}

__global__ void __launch_bounds__(kPThreads, 1)
proj_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_wq,
            const __grid_constant__ CUtensorMap tm_wk, const __grid_constant__ CUtensorMap tm_wv,
            const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
            const __grid_constant__ CUtensorMap tm_v, ProjArgs A) {
    using C = ProjCfg;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + C::OFF_BAR);
    uint64_t *full = bars, *empty = bars + PS, *acc_full = bars + 2 * PS, *acc_empty = acc_full + 2;
    uint64_t *fin = acc_empty + 2, *done = fin + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(done + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    grid_dep_launch();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_rank();
    const int cid = (int)(blockIdx.x / kCl), ncl = (int)(gridDim.x / kCl);
    constexpr uint16_t kAll = (uint16_t)((1u << kCl) - 1u);
    if (threadIdx.x == 0) {
        for (int s = 0; s < PS; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kCl);                 // the MMAs of every CTA of the cluster have read the stage
        }
        for (int b = 0; b < 2; ++b) { mbar_init(&acc_full[b], 1); mbar_init(&acc_empty[b], 1); }
        mbar_init(fin, 1);
        mbar_init(done, kCl - 1);                      // the other CTAs are done with this CTA's memory
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == kWMma) { tmem_alloc(tmem_slot, C::TMEM_COLS); tmem_relinquish(); }
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();                                // every CTA's barriers exist before any multicast
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const Abort ab{abort_flag, A.status};
    // group q, this CTA's row tile: m = kCl mp + rank (row tiles past the last are copies of it)
    auto tile_geom = [&](int q, int &b, int &n0, int &nt, int &nbt, bool &store) {
        const int mp = q / A.n_ntiles;
        nt = q - mp * A.n_ntiles;
        int m = kCl * mp + (int)rank;
        store = m < A.n_mtiles;
        if (!store) m = A.n_mtiles - 1;
        b = m / A.mt_per_b;
        n0 = (m - b * A.mt_per_b) * PM;
        nbt = min(PNB, A.nblocks - nt * PNB);
    };

    if (warp == kWProd) {
        if (lane == 0) {
            grid_dep_wait();
            int it = 0;
            bool ok = true;
            for (int q = cid; q < A.n_pairs && ok; q += ncl) {
                int b, n0, nt, nbt;
                bool store;
                tile_geom(q, b, n0, nt, nbt, store);
                (void)GMA_IN_BOUNDS(b < A.B && n0 < A.N, A.status);
                for (int kb = 0; kb < A.nkb; ++kb, ++it) {
                    const int s = it % PS;
                    if (it >= PS && !(ok = mbar_wait(&empty[s], ((it / PS) - 1) & 1, ab, kDevErrTimeout))) break;
                    uint8_t *st = sm + C::OFF_S + s * kStage;
                    mbar_arrive_expect_tx(&full[s], kABytes + nbt * kBBlk);
                    tma_load_3d(st, &tm_x, &full[s], kb * PKB, n0, b);
                    for (int j = (int)rank; j < nbt; j += kCl) {   // this CTA's share of the W blocks, to all
                        const BlockMap m = map_block(A, nt * PNB + j);
                        const CUtensorMap *wm = m.which == 0 ? &tm_wq : (m.which == 1 ? &tm_wk : &tm_wv);
                        tma_load_3d_mc(st + kABytes + j * kBBlk, wm, &full[s], m.col * PBN, kb * PKB, m.h, kAll);
                    }
                }
            }
            // every fill has landed, and both CTAs' MMAs have released every stage (so neither
            // CTA's multicast nor commit still targets this CTA)
            wind_down_ring(full, PS, it, A.status);
            wind_down_ring(empty, PS, it, A.status);
        }
    } else if (warp == kWMma) {
        // the whole warp, converged
        int it = 0, lt = 0;
        bool ok = true;
        for (int q = cid; q < A.n_pairs && ok; q += ncl, ++lt) {
            int b, n0, nt, nbt;
            bool store;
            tile_geom(q, b, n0, nt, nbt, store);
            const int buf = lt & 1;
            if (lt >= 2 && !(ok = mbar_wait_warp(&acc_empty[buf], ((lt >> 1) - 1) & 1, ab, kDevErrTimeout))) break;
            tc_fence_after();
            const uint32_t idesc = idesc_f16(1, 1, 0, 1, PM, PBN * nbt);     // X K-major, W MN-major
            const uint32_t acc = tmem + buf * C::ACC_COLS;
            for (int kb = 0; kb < A.nkb; ++kb, ++it) {
                const int s = it % PS;
                if (!(ok = mbar_wait_warp(&full[s], (it / PS) & 1, ab, kDevErrTimeout))) break;
                tc_fence_after();
                const uint32_t sa = smem_u32(sm + C::OFF_S + s * kStage);
                const uint64_t ad = sdesc_sw128(sa, 16, 1024);
                const uint64_t bd = sdesc_sw128(sa + kABytes, kBBlk, 1024);   // 64-column blocks kBBlk apart
#pragma unroll
                for (int kk = 0; kk < PKB / 16; ++kk)
                    mma_ss(acc, ad + (uint64_t)(kk * 2), bd + (uint64_t)(kk * 128), idesc, (kb | kk) != 0);
                mma_commit_mc(&empty[s], kAll);       // the stage is free here and, for its multicast parts, elsewhere
            }
            if (ok) mma_commit(&acc_full[buf]);
        }
        mma_commit(fin);
        wait_ignoring_abort(fin, 0, A.status);
    } else {
        // ---------------- epilogue: accumulator row r -> bf16 -> staging buffer -> TMA store
        RowThread rt;
        rt.wg = 0;
        rt.r = 32u * (warp & 3) + lane;
        rt.lane_off = (uint32_t)(32 * (warp & 3)) << 16;
        rt.wtid = threadIdx.x - kWEpi * 32;
        const bool elected = rt.wtid == 0;
        if (elected) grid_dep_wait();       // the previous kernel in the stream no longer reads the outputs
        int lt = 0, ec = 0;
        for (int q = cid; q < A.n_pairs; q += ncl, ++lt) {
            int b, n0, nt, nbt;
            bool store;
            tile_geom(q, b, n0, nt, nbt, store);
            const int buf = lt & 1;
            const bool ok = mbar_wait(&acc_full[buf], (lt >> 1) & 1, ab, kDevErrTimeout);
            if (!wg_all(rt, ok)) break;
            tc_fence_after();
            for (int j = 0; j < nbt && store; ++j, ++ec) {   // (a copy of the last row tile stores nothing)
                uint32_t v0[32], v1[32];
                const uint32_t ta = tmem + rt.lane_off + buf * C::ACC_COLS + j * PBN;
                tmem_ld32(ta, v0);
                tmem_ld32(ta + 32, v1);
                tmem_ld_wait();
                uint8_t *eb = sm + C::OFF_E + (ec & 1) * kTileBytes;
                if (elected) bulk_wait_group_read<1>();       // the store that last used this buffer has read it
                wg_sync(rt);
#pragma unroll
                for (int qq = 0; qq < 8; ++qq) {
                    const uint32_t *src = qq < 4 ? v0 + 8 * qq : v1 + 8 * (qq - 4);
                    uint32_t o[4];
#pragma unroll
                    for (int u = 0; u < 4; ++u)
                        o[u] = pack_bf16(__uint_as_float(src[2 * u]), __uint_as_float(src[2 * u + 1]));
                    *reinterpret_cast<uint4 *>(eb + sw128_off(rt.r, qq)) = make_uint4(o[0], o[1], o[2], o[3]);
                }
                fence_proxy_async_smem();
                wg_sync(rt);
                if (elected) {
                    const BlockMap m = map_block(A, nt * PNB + j);
                    const CUtensorMap *om = m.which == 0 ? &tm_q : (m.which == 1 ? &tm_k : &tm_v);
                    if (GMA_IN_BOUNDS(m.h < A.H && b < A.B, A.status)) {
                        tma_store_3d(om, eb, m.col * PBN, n0, b * A.H + m.h);
                        bulk_commit_group();
                    }
                }
            }
            tc_fence_before();
            wg_sync(rt);
            if (elected) mbar_arrive(&acc_empty[buf]);
        }
        if (elected) bulk_wait_group<0>();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // no CTA leaves while another may still write into it: each tells the others it is done
    // (its loads landed, its MMAs released every stage) and waits for the same, bounded
    if (threadIdx.x == 0) {
        for (uint32_t o = 1; o < (uint32_t)kCl; ++o) mbar_arrive_peer(done, (rank + o) % kCl);
        wait_ignoring_abort(done, 0, A.status);
    }
    __syncthreads();
    if (warp == kWMma) {
        __syncwarp();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

}  // namespace

bool proj_supported(int B, int N, int D, int H, int d, int dv) {
    return B > 0 && N > 0 && H > 0 && D > 0 && D % PKB == 0 && d > 0 && d % PBN == 0 && dv > 0 && dv % PBN == 0;
}

cudaError_t proj_run(int B, int N, int D, int H, int d, int dv, const void *X, const void *Wq, const void *Wk,
                     const void *Wv, void *Qx, void *Kx, void *V, char *ws, cudaStream_t s) {
    CUtensorMap tx, twq, twk, twv, tq, tk, tv;
    if (!make_map(&tx, X, B, N, D, PM) || !make_map(&twq, Wq, H, D, d, PKB) || !make_map(&twk, Wk, H, D, d, PKB) ||
        !make_map(&twv, Wv, H, D, dv, PKB) || !make_map(&tq, Qx, B * H, N, d, PM) ||
        !make_map(&tk, Kx, B * H, N, d, PM) || !make_map(&tv, V, B * H, N, dv, PM))
        return cudaErrorInvalidValue;
    ProjArgs a{};
    a.B = B; a.N = N; a.H = H; a.nkb = D / PKB;
    a.nqb = d / PBN; a.nvb = dv / PBN; a.nbh = 2 * a.nqb + a.nvb;
    a.mt_per_b = (N + PM - 1) / PM;
    a.n_mtiles = B * a.mt_per_b;
    a.nblocks = H * a.nbh;
    a.n_ntiles = (a.nblocks + PNB - 1) / PNB;
    a.n_pairs = ((a.n_mtiles + kCl - 1) / kCl) * a.n_ntiles;
    a.status = reinterpret_cast<unsigned *>(ws);
    cudaError_t e = set_dyn_smem(reinterpret_cast<const void *>(proj_kernel), ProjCfg::BYTES);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(kPThreads);
    cfg.dynamicSmemBytes = ProjCfg::BYTES;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = kCl;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    // persistent clusters, as many as can be resident at once (tile groups are assigned
    // statically, so a second wave would double the tail)
    const int nsm = sm_count();
    int ncl = std::max(1, std::min((nsm > 0 ? nsm : kMaxCtas) / kCl, a.n_pairs));
    cfg.gridDim = dim3(kCl * ncl);
    int active = 0;
    if (cudaOccupancyMaxActiveClusters(&active, reinterpret_cast<const void *>(proj_kernel), &cfg) == cudaSuccess &&
        active > 0)
        ncl = std::min(ncl, active);
    cfg.gridDim = dim3(kCl * ncl);
    return cudaLaunchKernelEx(&cfg, proj_kernel, tx, twq, twk, twv, tq, tk, tv, a);
}

}  // namespace gma
