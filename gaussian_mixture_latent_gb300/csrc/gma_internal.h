// Internal declarations shared by the host API and the kernel translation units.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/gma.h"

namespace gma {

// Device status word bits (first 4 bytes of the workspace header).
enum : unsigned {
    kDevErrTimeout = 1u,     // a bounded mbarrier / flag wait ran out
    kDevErrBounds = 2u,      // a debug-build index check failed (the access was skipped)
};

// Index checks of the debug build (compiled with -DGMA_DEBUG_BOUNDS): a failed check
// posts kDevErrBounds to the status word and yields false, so that the caller skips
// the access; it never traps.  In the normal build every check is `true`.
#ifdef GMA_DEBUG_BOUNDS
#define GMA_IN_BOUNDS(cond, status) ((cond) ? true : (atomicOr((status), ::gma::kDevErrBounds), false))
#else
#define GMA_IN_BOUNDS(cond, status) true
#endif

constexpr size_t kHeaderBytes = 256;
constexpr int kTcChunkRows = 128;    // causal chunk of the tensor-core kernels (one MMA tile)
constexpr int kBwdChunkRows = 64;    // row tile of the causal backward's masked products
constexpr size_t kAlign = 256;

inline size_t align_up(size_t x, size_t a = kAlign) { return (x + a - 1) / a * a; }

// Problem geometry after validation.
struct Problem {
    int B, H, N, d, K, dv, G;
    int Nkv;                     // rows of Kx and V: N, or the context length of cross-attention
    gma_dtype in_dtype, out_dtype;
    float var_floor;
    float eps;
    int causal;
    int chunk;
    int sm_budget;               // > 0: SMs the call's persistent write kernel may use (a concurrent
                                 // kernel holds the rest); 0: all of them
};

// ----- workspace carving (byte offsets from the workspace base) -----
struct SimtLayout {
    size_t lam, cdir;            // parameter prologue outputs
    size_t gq, gk;               // materialised responsibilities [G][N][K] f32
    size_t part;                 // [G][P][K][dv+1] f32 partial / segment totals
    size_t mem;                  // [G][P or 1][K][dv+1] f32 reduced memory / exclusive prefixes
    size_t total;
    int P;                       // N-splits (bidirectional) or segments (causal)
};
SimtLayout simt_layout(const Problem &p);

// Raise a kernel's dynamic shared-memory limit on the current device to `bytes`:
// the attribute is set the first time a (kernel, device) pair needs that much
// and remembered, so steady-state launches make no attribute call (gma_api.cu).
cudaError_t set_dyn_smem(const void *kern, int bytes);

// ----- tensor-core bidirectional path: gma_tc.cu -----
constexpr int kMaxCtas = 256;        // upper bound on persistent CTAs (partial slots are sized for it)
struct TcLayout {
    size_t params, part, mem, total;   // workspace byte offsets
    size_t claim;                      // the read's unit counter (bidirectional path)
    size_t stats, pnum, pden;          // component-sliced causal path: row statistics, partials
    int ns, nt;                        // component slices and value slices of 64
    uint32_t param_stride, mem_stride;
    int T, Ttot, ncta;                 // tiles per head, tiles in total, persistent CTAs (queries / read)
    int Tkv, Ttot_kv, ncta_kv;         // the same for the key/value rows (write, reduce)
};
bool tc_bidir_supported(const Problem &p);
TcLayout tc_layout(const Problem &p);
cudaError_t tc_params(const Problem &p, const TcLayout &L, const float *mu, const float *rho,
                      const float *alpha, char *ws, cudaStream_t s);
cudaError_t tc_write(const Problem &p, const TcLayout &L, const void *Kx, const void *V, char *ws,
                     cudaStream_t s);
cudaError_t tc_reduce(const Problem &p, const TcLayout &L, char *ws, cudaStream_t s);
// the same over the partial slots at workspace offset `part` into the operand at `mem`,
// and (mem_lo != 0) its bf16 rounding remainder at `mem_lo`; with claim != 0 it also
// zeroes the read kernel's unit counter at that offset
cudaError_t tc_reduce_split(const Problem &p, const TcLayout &L, size_t part, size_t mem, size_t mem_lo, char *ws,
                            cudaStream_t s, size_t claim = 0);
cudaError_t tc_read(const Problem &p, const TcLayout &L, const void *Qx, void *out, char *ws,
                    cudaStream_t s);

// ----- tensor-core causal path: gma_tc_causal.cu (one kernel; each CTA builds its head's coefficients) -----
bool tc_causal_supported(const Problem &p);
TcLayout tc_causal_layout(const Problem &p);
// component-sliced causal path (gma_tc_slice.cu + gma_tc_causal.cu): larger K or dv
bool tc_slice_supported(const Problem &p);
TcLayout tc_slice_layout(const Problem &p);
cudaError_t tc_rowstats(const Problem &p, const TcLayout &L, const void *Qx, const void *Kx, char *ws,
                        cudaStream_t s);
cudaError_t tc_causal_slices(const Problem &p, const TcLayout &L, const void *Qx, const void *Kx, const void *V,
                             char *ws, cudaStream_t s);
cudaError_t tc_combine(const Problem &p, const TcLayout &L, void *out, char *ws, cudaStream_t s);
cudaError_t tc_causal(const Problem &p, const TcLayout &L, const void *Qx, const void *Kx, const void *V,
                      const float *mu, const float *rho, const float *alpha, void *out, char *ws, cudaStream_t s);

// Segment-parallel form of the causal scan (d = dv = K = 64), for problems with fewer
// heads than SMs: ns scan CTAs take balanced contiguous ranges of the (head, 128-row
// chunk) list, so a range may start inside a head and may cross into the next.  A
// range that starts at chunk a > 0 of head g needs the prefix state of chunks [0, a)
// of g (Eq. 6b): the prefix pass (tc_write over "prefix segments") sums
// gamma^K^T [V | 1] over each segment, where the segment of scan CTA i is the part of
// CTA i-1's range that lies in the head where CTA i starts; CTA i adds the partial
// slots of the segments of its head up to its own, in a fixed order.
constexpr int kMaxScanCtas = 152;
struct SegEntry {
    int32_t g;               // head
    int16_t a, len;          // chunks [a, a + len) of head g
    int16_t plo, phi;        // prefix-pass CTAs plo..phi covered it (partial slots p + segment)
};
struct SegTable {
    int32_t nseg, ns, np, nch, vtot;              // segments, scan CTAs, prefix-pass CTAs, chunks per head, total
    SegEntry seg[kMaxScanCtas];                   // prefix segments in scan-CTA order
    int16_t pre_v[kMaxScanCtas], pre_jj[kMaxScanCtas];   // prefix-pass CTA p starts at chunk pre_jj[p] of segment pre_v[p]
    int16_t scan_seg[kMaxScanCtas];               // scan CTA i: the segment that ends at its start (-1: a head start)
};
// Fills the plan and returns true when the segment-parallel form applies (fewer heads than SMs).
bool tc_seg_plan(const Problem &p, SegTable &T);
TcLayout tc_seg_layout(const Problem &p, const SegTable &T);
cudaError_t tc_prefix(const Problem &p, const TcLayout &L, const SegTable &T, const void *Kx, const void *V, char *ws,
                      cudaStream_t s);
cudaError_t tc_causal_seg(const Problem &p, const TcLayout &L, const SegTable &T, const void *Qx, const void *Kx,
                          const void *V, void *out, char *ws, cudaStream_t s);

// ----- responsibility diagnostics (section 5.4): gma_tc_diag.cu (uses tc_params) -----
bool tc_diag_supported(const Problem &p);
TcLayout tc_diag_layout(const Problem &p);
cudaError_t tc_diag(const Problem &p, const TcLayout &L, const void *Qx, int *z, char *ws, cudaStream_t s);
cudaError_t tc_diag_finalize(const Problem &p, const TcLayout &L, float *p_out, float *stats_out, char *ws,
                             cudaStream_t s);

// ----- backward pass for every other shape (d, K, dv <= 256), CUDA cores, fp32: gma_bwd_simt.cu -----
struct GbLayout {
    size_t lam, cdir, lmu;           // lambda, the direction constants, [lambda mu | lambda] per head
    size_t gq, gk, dsq, dsk;         // [G][N][K]: responsibilities and score gradients of both sides
    size_t t, ab;                    // [G][N][max(dv + 1, 2 d)] products; [G][N][dv + 1] = [a | b]
    size_t part, mem, memr;          // [G][P][K][dv + 1]: range partials; memory; [R | r]
    size_t pq, pk;                   // [G][P][K][2 d + 1]: parameter sums per range of each side
    size_t total;
    int P, rpp, C;                   // row ranges, rows per range, causal chunk rows
};
bool gb_supported(const Problem &p);
GbLayout gb_layout(const Problem &p);
cudaError_t gb_run(const Problem &p, const GbLayout &L, const void *Qx, const void *Kx, const void *V,
                   const float *mu, const float *rho, const float *alpha, const void *dO, float *dQx, float *dKx,
                   float *dV, float *dmu, float *drho, float *dalpha, char *ws, cudaStream_t s);

// ----- backward pass, bidirectional and causal, CUDA cores: gma_bwd.cu (uses simt_params) -----
struct BwdLayout {
    size_t lam, cdir;            // parameter prologue outputs
    size_t mem_s, mem_r;         // [G][K][dv+1]: the forward memory [Vt | Z] and the backward [R | r]
    size_t part_m;               // [G][C][K][dv+1] per-chunk partials of either memory
    size_t part_q, part_k;       // [G][C][K][2d+1] per-chunk parameter sums over query / key rows
    size_t mem_pc, mem_rc;       // causal: [G][C][K][dv+1] memories before / after each chunk
    size_t gk;                   // [G][N][K] gamma^K of the memory pass, reused by the key pass
    size_t ab, dsq, dsk, gq;     // causal: [G][N][68] a | b rows, [G][N][K] ds of queries / keys, gamma^Q
    size_t total;
    int C, rows_per_chunk;       // row chunks per head
};
bool bwd_supported(const Problem &p);
BwdLayout bwd_layout(const Problem &p);
cudaError_t bwd_run(const Problem &p, const BwdLayout &L, const void *Qx, const void *Kx, const void *V,
                    const float *mu, const float *rho, const float *alpha, const void *dO, float *dQx, float *dKx,
                    float *dV, float *dmu, float *drho, float *dalpha, char *ws, cudaStream_t s);
// dmu, drho, dalpha from the parameter sums pq, pk ([G][C][K][2d+1]: P1, P2, P0 over the
// query and key rows of C row chunks) and the fp32 lambda [H][K][d]
cudaError_t bwd_finalize(const Problem &p, int C, const float *pq, const float *pk, const float *mu, const float *lam,
                         const float *rho, const float *alpha, float *dmu, float *drho, float *dalpha, cudaStream_t s);

// ----- backward pass, bidirectional bf16, tensor cores: gma_bwd_tc.cu (uses the tc_* forward kernels) -----
struct BwdTcLayout {
    TcLayout tc;                  // the forward's parameter blocks, memory partials and operand [Vt | Z]
    size_t lam;                   // fp32 lambda [H][K][d]
    size_t lamb;                  // [H] bf16 [lambda | lambda mu] operands
    size_t mem_lo;                // the bf16 remainder of [Vt | Z] (hi + lo: the two-term operand)
    size_t part_r, mem_r, mem_rlo;  // [R | r] partial slots, its bf16 operand and remainder
    size_t part_pq, part_pk;      // parameter-sum partial slots of the query and key passes
    size_t psum;                  // [2][H][K][2d+1] parameter sums per head set, query rows then key rows
    size_t total;
};
bool bwd_tc_supported(const Problem &p);
BwdTcLayout bwd_tc_layout(const Problem &p);
cudaError_t bwd_tc_run(const Problem &p, const BwdTcLayout &L, const void *Qx, const void *Kx, const void *V,
                       const float *mu, const float *rho, const float *alpha, const void *dO, float *dQx, float *dKx,
                       float *dV, float *dmu, float *drho, float *dalpha, char *ws, cudaStream_t s);

// ----- Q/K/V input projections (Eq. 4): gma_proj.cu (one tcgen05 GEMM, bf16) -----
bool proj_supported(int B, int N, int D, int H, int d, int dv);
cudaError_t proj_run(int B, int N, int D, int H, int d, int dv, const void *X, const void *Wq, const void *Wk,
                     const void *Wv, void *Qx, void *Kx, void *V, char *ws, cudaStream_t s);

// ----- self-test of the bounded-wait failure path: gma_selftest.cu -----
cudaError_t selftest_timeout(void *ws, cudaStream_t s);

// ----- causal decode with a carried state: gma_decode.cu (one launch) -----
bool decode_supported(const Problem &p);
size_t decode_workspace(const Problem &p);
cudaError_t decode_step(const Problem &p, const void *Qx, const void *Kx, const void *V, const float *mu,
                        const float *rho, const float *alpha, float *state, void *out, cudaStream_t s);

// ----- SIMT (CUDA-core, fp32) path: gma_simt.cu -----
cudaError_t simt_params(const Problem &p, const float *rho, const float *alpha, float *lam,
                        float *cdir, cudaStream_t s);
cudaError_t simt_gamma(const Problem &p, const void *X, const float *mu, const float *lam,
                       const float *cdir, float *gamma, cudaStream_t s);
cudaError_t simt_write(const Problem &p, const void *V, char *ws, const SimtLayout &L,
                       cudaStream_t s);
cudaError_t simt_reduce(const Problem &p, char *ws, const SimtLayout &L, cudaStream_t s);
cudaError_t simt_read(const Problem &p, char *ws, const SimtLayout &L, void *out, cudaStream_t s);
cudaError_t simt_causal(const Problem &p, const void *V, char *ws, const SimtLayout &L, void *out,
                        cudaStream_t s);
size_t simt_causal_smem(const Problem &p);

}  // namespace gma
