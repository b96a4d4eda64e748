/*
 * gma.h -- C ABI of the GB300 (sm_103a) Gaussian Mixture Attention forward.
 *
 * Method: "Gaussian Mixture Attention: Linear-Time Sequence Mixing via
 * Probabilistic Latent Routing" (Huang & Raza, 2026).  Per head, with
 * routing vectors Qx, Kx [N, d], values V [N, dv] and K diagonal Gaussian
 * components (means mu [K, d], variance parameters rho [K, d], prior logits
 * alpha [K]):
 *
 *   sigma^2 = softplus(rho) + var_floor                    (section 3.6, Eq. 14)
 *   pi      = softmax(alpha)                               (section 3.6, Eq. 15)
 *   Gamma^Q, Gamma^K = posterior responsibilities of the rows of Qx, Kx
 *                                                          (section 3.2, Eq. 3; Eq. 16 / 3b)
 *   bidirectional:  Vt = Gamma^K^T V,  Z = Gamma^K^T 1     (section 3.3, Eq. 5-6)
 *                   O  = Gamma^Q Vt / (Gamma^Q Z + eps)    (section 3.3, Eq. 7-8)
 *   causal:         prefix memories over j <= i           (section 3.5, Eq. 6b)
 *                   O_i = gamma^Q_i Vt^(i) / (gamma^Q_i Z^(i) + eps)   (Eq. 8b)
 *
 * Layout of every tensor argument (row-major, contiguous, no padding):
 *   Qx, Kx     [B, H, N, d]   in_dtype
 *   V          [B, H, N, dv]  in_dtype
 *   out        [B, H, N, dv]  out_dtype
 *   mu, rho    [H, K, d]      float32   (one mixture per head, shared by the batch)
 *   pi_logits  [H, K]         float32
 * All pointers are DEVICE pointers (CUDA global memory of the current device)
 * unless a function says otherwise; base addresses must be 16-byte aligned.
 * `stream` is a cudaStream_t passed as void* (NULL = the legacy default stream).
 *
 * Ownership: the caller owns every buffer, including the workspace.  The
 * library allocates no device memory, keeps no global state between calls
 * and is re-entrant; calls on different streams with different workspaces
 * may run concurrently.
 *
 * Asynchrony and errors: argument errors are returned synchronously and
 * launch nothing.  A failed kernel launch returns GMA_ERR_CUDA.  Errors found
 * on the device (a bounded wait that ran out) are posted to the status word
 * at the start of the workspace and read back with gma_get_status().  No
 * function except gma_get_status() synchronises.
 */
#ifndef GMA_H_
#define GMA_H_

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    GMA_OK = 0,
    GMA_ERR_INVALID_ARG = 1,   /* null pointer, bad size, misaligned pointer      */
    GMA_ERR_UNSUPPORTED = 2,   /* valid request outside the implemented range     */
    GMA_ERR_WORKSPACE = 3,     /* workspace missing or smaller than required      */
    GMA_ERR_CUDA = 4,          /* a CUDA runtime call or kernel launch failed     */
    GMA_ERR_TIMEOUT = 5,       /* a device-side bounded wait ran out              */
    GMA_ERR_BOUNDS = 6         /* a device-side index check failed (debug build)  */
} gma_status;

typedef enum { GMA_F32 = 0, GMA_BF16 = 1 } gma_dtype;

typedef struct {
    int B, H, N;        /* batch, heads, sequence length (N >= 0)                 */
    int d;              /* routing dimension d_r, 1..256                          */
    int K;              /* number of Gaussian components, 1..256                  */
    int dv;             /* value dimension, 1..256                                */
    gma_dtype in_dtype; /* dtype of Qx, Kx and V                                  */
    gma_dtype out_dtype;/* dtype of out                                           */
    float var_floor;    /* eps_sigma of Eq. 14 (> 0)                              */
    int chunk;          /* causal chunk length in rows (see below); 0 = default   */
} gma_desc;

/*
 * desc->chunk: the number of rows over which a causal forward forms the masked
 * intra-chunk affinity before it folds the chunk into its carried prefix state
 * (section 3.5, Eq. 6b / 9b).  It changes only the rounding of the result, never
 * its value in exact arithmetic.
 *   - bf16 tensor-core causal paths (d = 64, K and dv multiples of 64): 128 rows,
 *     the MMA tile; chunk must be 0 or 128, any other value returns
 *     GMA_ERR_UNSUPPORTED.
 *   - the float32 CUDA-core causal path (every other shape): any chunk >= 1 whose
 *     per-chunk tiles fit one CTA's shared memory (4 (K (dv + 1) + 2 chunk K
 *     + 2 chunk (dv + 1) + chunk^2) bytes <= 227 KB); larger values return
 *     GMA_ERR_UNSUPPORTED.  0 selects 16.
 *   - gma_backward with causal = 1: at d = dv = K = 64, chunk 0 or 64 takes the
 *     64-row tiles of that shape's kernels; any other chunk, and every other
 *     shape, takes the general path's chunks of chunk rows (0 selects 16) within
 *     its shared-memory bound (see gma_backward), GMA_ERR_UNSUPPORTED beyond.
 *   - bidirectional calls, decode, cross-attention and diagnostics have no
 *     chunked scan and ignore the field.
 * A negative chunk is GMA_ERR_INVALID_ARG everywhere.
 *
 * Status codes are positive (GMA_OK = 0, errors 1..5) so that a caller can test
 * `if (status)`; their names, not their values, are the interface.
 */

/*
 * Size in bytes of the device workspace that gma_forward() needs for this
 * problem and direction (causal = 0 bidirectional, 1 causal).  Pure host
 * computation.  Before its first use a workspace's first 256 bytes must be
 * zero (gma_workspace_init() does that); later calls keep them zero unless
 * a device error was posted.
 */
gma_status gma_workspace_size(const gma_desc *desc, int causal, size_t *bytes);

/* Zero the workspace header (the device status word) on `stream`. */
gma_status gma_workspace_init(void *workspace, size_t workspace_bytes, void *stream);

/*
 * The GMA forward (section 3.3, Eq. 5-8; causal: section 3.5, Eq. 6b, 8b),
 * with the parameterisation of section 3.6 (Eq. 14-15) and the
 * responsibilities of section 3.2 (Eq. 3).  Writes out [B, H, N, dv].
 * eps >= 0 is added once to each row's denominator.  Enqueued on `stream`;
 * returns without synchronising.  Inputs are not modified.  `out` must not
 * overlap any input or the workspace.
 */
gma_status gma_forward(const gma_desc *desc, const void *Qx, const void *Kx, const void *V,
                       const float *mu, const float *rho, const float *pi_logits, float eps,
                       int causal, void *out, void *workspace, size_t workspace_bytes,
                       void *stream);

/*
 * gma_forward() with per-launch timing: when `events` is not NULL it holds
 * n_events cudaEvent_t handles (as void*, created by the caller); the
 * library records events[2i] on `stream` just before its i-th kernel launch
 * and events[2i+1] just after it, for every i with 2i+1 < n_events.  NULL
 * entries are skipped.  Everything else is as for gma_forward().
 */
gma_status gma_forward_ex(const gma_desc *desc, const void *Qx, const void *Kx, const void *V,
                          const float *mu, const float *rho, const float *pi_logits, float eps,
                          int causal, void *out, void *workspace, size_t workspace_bytes,
                          void *stream, void *const *events, int n_events);

/*
 * The kernel launches gma_forward() makes for this problem, without running
 * anything: their number in *n_launches (0 when N == 0) and, when `names` is
 * not NULL, the first `capacity` kernel names (static strings).
 */
gma_status gma_forward_plan(const gma_desc *desc, int causal, int *n_launches, const char **names,
                            int capacity);

/*
 * Several independent forward calls in one request.  The paper's layers apply
 * the forward of section 3.3 (Eq. 5-8) or of section 3.5 (Eq. 6b, 8b) to each
 * head; a model that needs more than one of them at a time (a bidirectional
 * and a causal mixer over the same batch, or several layers that do not depend
 * on one another) can hand them over together, so that the library runs them
 * side by side where one of them leaves SMs idle.
 *
 * Each call has gma_forward()'s arguments (its own inputs and output) and an
 * optional list of CUDA events, recorded as by gma_forward_ex() on the stream
 * where that call's kernels run.  No output may overlap any input or output of
 * any call.
 */
typedef struct {
    gma_desc desc;
    int causal;                   /* 0 bidirectional, 1 causal                    */
    float eps;
    const void *Qx, *Kx, *V;
    const float *mu, *rho, *pi_logits;
    void *out;
    void *const *events;          /* NULL, or n_events cudaEvent_t (as void*)     */
    int n_events;
} gma_forward_call;

/*
 * Workspace of gma_forward_multi(): one region per call, in call order, each
 * 256-byte aligned and of that call's gma_workspace_size().  offsets (NULL, or
 * n_calls entries) receives each region's byte offset; the first 4 bytes of a
 * region are that call's device status word (gma_get_status(workspace +
 * offsets[i], ...)).  Zero every region's first 256 bytes before the first use
 * (zeroing the whole workspace does it); later requests of the same calls keep
 * them zero unless a device error was posted.  A request of other calls or
 * shapes moves the regions: zero its regions' headers again before it runs
 * (gma_workspace_init(workspace + offsets[i], ...) for each i).
 */
gma_status gma_forward_multi_workspace_size(const gma_forward_call *calls, int n_calls, size_t *bytes,
                                            size_t *offsets);

/*
 * Runs the calls; returns once everything is enqueued, with `stream` ordered
 * after all of it.  Every call is validated before anything is launched; the
 * first failing call's status is returned.
 *
 * Scheduling.  With aux_stream == NULL (or equal to `stream`) the calls run in
 * order on `stream`, exactly as gma_forward() calls would.  Otherwise the calls that the library
 * runs as one CTA per head (those whose gma_forward_plan() is the single launch
 * "tc_causal": the bf16 causal scan with d = K = dv = 64 when the heads B*H
 * fill more than half of the SMs or the sequences are short) run in order on
 * aux_stream, and the other calls run in order on `stream`, both starting
 * after the work already queued on `stream`.  While the scan holds one SM per
 * head, the other calls' bidirectional tensor-core write kernels are sized to
 * the SMs it leaves free (when that is at least an eighth of them), and their
 * read kernels take tiles dynamically, so that they spread over every SM once
 * the scan has finished.  Such a call's key-side memory is then summed from
 * partial sums over different row ranges than gma_forward() would use: its
 * output can differ from gma_forward()'s in the last bits (both are fixed-order
 * sums; repeated calls with the same arguments on the same GPU give identical
 * results).  Causal calls, and every call when no scan is among them, give
 * exactly gma_forward()'s results.
 */
gma_status gma_forward_multi(const gma_forward_call *calls, int n_calls, void *workspace, size_t workspace_bytes,
                             void *stream, void *aux_stream);

/*
 * Responsibilities of the rows of X [B, H, N, d] (section 3.2, Eq. 3, in the
 * softmax form of Eq. 16 / 3b), written as float32 to gamma_out [B, H, N, K].
 * A diagnostic export: the forward never writes Gamma to memory.  Needs the
 * workspace of gma_workspace_size(desc, 0, ...).
 */
gma_status gma_responsibilities(const gma_desc *desc, const void *X, const float *mu,
                                const float *rho, const float *pi_logits, float *gamma_out,
                                void *workspace, size_t workspace_bytes, void *stream);

/*
 * Test of the device-side failure path: launches one CTA whose bounded wait is on
 * a barrier that nothing arrives at.  The wait gives up after about one second,
 * as every wait in the library's kernels does, and posts GMA_ERR_TIMEOUT to the
 * workspace's status word (read with gma_get_status()); the CUDA context stays
 * usable.  workspace: at least 256 bytes, 16-byte aligned.  Returns GMA_OK when
 * the kernel was launched.
 */
gma_status gma_selftest_timeout(void *workspace, size_t workspace_bytes, void *stream);

/*
 * Backward pass ("Gaussian Mixture Attention", section 4.1, Eq. 17-20, through
 * Eq. 14-15 and the memory products of Eq. 5-8): given dO = dL/dO
 * [B, H, N, dv] for the forward output O = gma_forward(...), writes
 *   dQx, dKx [B, H, N, d], dV [B, H, N, dv]          (float32)
 *   dmu, drho [H, K, d], dpi_logits [H, K]            (float32, summed over the batch)
 * every output overwritten, not accumulated.  Qx, Kx, V in desc->in_dtype and
 * dO in desc->out_dtype, which must be the same type.  Deterministic
 * (fixed-order reductions).  causal = 1 differentiates the prefix memories of
 * Eq. 6b / 8b (each key collects the gradient of the rows at or after it).
 * Three paths, by shape:
 *   - bidirectional, bf16, d = dv = K = 64, N > 128: tensor cores (bf16
 *     operands, the two memory operands as two bf16 terms, fp32 accumulation,
 *     softmax and epilogues);
 *   - d = dv = K = 64 otherwise (fp32 inputs, one-tile heads, the causal form
 *     with chunk 0 or 64): CUDA cores in fp32 over 64-row tiles;
 *   - every other shape (d, K, dv up to 256): CUDA cores in fp32 over the
 *     responsibilities of every row; the causal form in chunks of desc->chunk
 *     rows (0 selects 16) while 4 (K (dv + 1) + 3 C K + 2 C (dv + 1) + C dv +
 *     2 C^2) bytes (C the chunk) fit a CTA's 227 KB of shared memory, and
 *     GMA_ERR_UNSUPPORTED beyond.
 * N = 0 writes zero parameter gradients.  Workspace:
 * gma_backward_workspace_size() (the first two paths hold Gamma^K of every row,
 * 256 B per row of a head, the causal one also a | b, Gamma^Q and ds, about
 * 1.3 KB per row in all; the third 4 (4 K + 2 (dv + 1) + max(dv + 1, 2 d))
 * bytes per row and the partial sums).
 * Errors as for gma_forward().
 */
gma_status gma_backward_workspace_size(const gma_desc *desc, int causal, size_t *bytes);
gma_status gma_backward(const gma_desc *desc, int causal, const void *Qx, const void *Kx, const void *V,
                        const float *mu, const float *rho, const float *pi_logits, float eps, const void *dO,
                        float *dQx, float *dKx, float *dV, float *dmu, float *drho, float *dpi_logits,
                        void *workspace, size_t workspace_bytes, void *stream);

/*
 * Causal decode with a carried state ("Gaussian Mixture Attention", section
 * 3.5, Eq. 6b and 8b as a recurrence): appends desc->N new positions to each
 * head's causal sequence.  state [B, H, K, dv + 1] float32, in and out, holds
 * [S | z] = sum over the positions so far of gamma^K_j [V_j | 1] (zeros for an
 * empty prefix).  For each new position t, in order:
 *   [S | z] += gamma^K(Kx_t) [V_t | 1]                   (the prefix includes t)
 *   out_t    = gamma^Q(Qx_t) S / (gamma^Q(Qx_t) z + eps)
 * Qx, Kx [B, H, N, d] and V [B, H, N, dv] in in_dtype, out [B, H, N, dv] in
 * out_dtype; responsibilities in fp32 from the direct form of Eq. 16.  Any
 * shape whose per-head state and precisions fit a CTA's shared memory
 * (K (dv + 1 + d) floats, about 220 KB); GMA_ERR_UNSUPPORTED otherwise.  The
 * workspace holds only the status word.  Workspace:
 * gma_decode_workspace_size().  The state is read and written on `stream`;
 * calls on one state must be ordered on one stream.
 */
gma_status gma_decode_workspace_size(const gma_desc *desc, size_t *bytes);
gma_status gma_decode(const gma_desc *desc, const void *Qx, const void *Kx, const void *V, const float *mu,
                      const float *rho, const float *pi_logits, float eps, float *state, void *out,
                      void *workspace, size_t workspace_bytes, void *stream);

/*
 * Cross-attention GMA ("Gaussian Mixture Attention", section 3.1 and section 6):
 * the queries Qx [B, H, N, d] of one sequence read the latent memory of a
 * context sequence, Ky [B, H, Nkv, d] and Vy [B, H, Nkv, dv], through the head's
 * one mixture:  Vt = Gamma^K_Y^T Vy,  Z = Gamma^K_Y^T 1,
 * out [B, H, N, dv] = Gamma^Q_X Vt / (Gamma^Q_X Z + eps)   (Eq. 5-8 with the context's memory).
 * Bidirectional only: there is no causal order between two sequences.  desc->N
 * is the query length; Nkv >= 1 when N >= 1 (an empty context has no memory:
 * GMA_ERR_INVALID_ARG).  Implemented on the tensor-core path (bf16 in and out,
 * d = dv = 64, K in {64, 128}); GMA_ERR_UNSUPPORTED otherwise.  Workspace:
 * gma_cross_workspace_size().  Errors as for gma_forward().
 */
gma_status gma_cross_workspace_size(const gma_desc *desc, int Nkv, size_t *bytes);
gma_status gma_forward_cross(const gma_desc *desc, int Nkv, const void *Qx, const void *Ky, const void *Vy,
                             const float *mu, const float *rho, const float *pi_logits, float eps, void *out,
                             void *workspace, size_t workspace_bytes, void *stream);

/*
 * Responsibility diagnostics of the query routing ("Gaussian Mixture
 * Attention", section 5.4, Eqs. 24-29).  With gamma^Q the responsibilities of
 * the rows of Qx [B, H, N, d] (Eq. 3b, per head) and T = B N tokens:
 *   gbar_t   = (1/H) sum_h gamma^Q_{t,h}              head average (Eq. 24)
 *   p_out[k] = (1/T) sum_t gbar_{t,k}                 marginal usage, p_out [K] float32 (Eq. 25)
 *   stats_out[0] = H_usage = -sum_k p_k log p_k / log K                  (Eq. 26)
 *   stats_out[1] = H_token = (1/T) sum_t -sum_k gbar log gbar / log K    (Eq. 27)
 *   stats_out[2] = R_max   = (1/T) sum_t max_k gbar_{t,k}               (Eq. 28)
 *   z_out[t]     = argmax_k gbar_{t,k}, ties to the lowest k, int32 [B, N] (Eq. 29);
 *                  z_out may be NULL
 * All outputs are device pointers.  Implemented for in_dtype = GMA_BF16,
 * d = 64, K in {64, 128} (GMA_ERR_UNSUPPORTED otherwise); desc->dv and
 * desc->out_dtype are validated as for gma_forward() but not used.  N = 0
 * launches nothing.  Needs gma_diagnostics_workspace_size() bytes.
 */
gma_status gma_diagnostics_workspace_size(const gma_desc *desc, size_t *bytes);
gma_status gma_diagnostics(const gma_desc *desc, const void *Qx, const float *mu, const float *rho,
                           const float *pi_logits, float *p_out, float *stats_out, int *z_out,
                           void *workspace, size_t workspace_bytes, void *stream);

/*
 * Input projections ("Gaussian Mixture Attention", section 3.1, Eq. 4): the routing
 * vectors and values of every head from the layer input,
 *   Qx[b, h] = X[b] W_Q[h],   Kx[b, h] = X[b] W_K[h],   V[b, h] = X[b] W_V[h],
 * bf16 operands with fp32 accumulation, results rounded to bf16.  Layouts (row-major,
 * contiguous, 16-byte aligned, every tensor bf16):
 *   X           [B, N, D]
 *   Wq, Wk      [H, D, d]        Wv  [H, D, dv]
 *   Qx, Kx      [B, H, N, d]     V   [B, H, N, dv]   (the layouts gma_forward() reads)
 * Implemented for D, d and dv multiples of 64 (GMA_ERR_UNSUPPORTED otherwise); B, N, H
 * any positive size.  N = 0 launches nothing.  The workspace holds only the status
 * word: at least 256 bytes, initialised to zero (gma_workspace_init()).  One kernel
 * launch (a persistent tcgen05 GEMM).
 */
typedef struct {
    int B, N, D, H, d, dv;
} gma_proj_desc;

gma_status gma_project(const gma_proj_desc *desc, const void *X, const void *Wq, const void *Wk, const void *Wv,
                       void *Qx, void *Kx, void *V, void *workspace, size_t workspace_bytes, void *stream);

/* Size of the fixed scratch buffer gma_forward_noalloc() uses: 32 MiB. */
#define GMA_NOALLOC_SCRATCH_BYTES ((size_t)32 << 20)

/*
 * gma_forward() for callers that cannot allocate device memory.  The paper
 * has no counterpart to this entry point; it exists for callers that must not
 * call cudaMalloc -- code whose device memory is owned by another memory
 * manager (a framework's caching allocator, a server's per-model budget) and
 * latency-sensitive loops that cannot take cudaMalloc's device-wide
 * synchronisation.
 *
 * Same arguments and results as gma_forward() minus the workspace: the
 * library uses a scratch array of GMA_NOALLOC_SCRATCH_BYTES compiled into it,
 * which every GPU that loads the library holds until the process exits.  The
 * call allocates nothing.  A request whose gma_workspace_size() is larger than
 * GMA_NOALLOC_SCRATCH_BYTES returns GMA_ERR_WORKSPACE and launches nothing.
 * The first call on a device looks up the array's device address on that
 * device (the device must be current); make that first call before any
 * stream capture.  All calls on a device share the array: calls whose GPU
 * work overlaps (other streams, or before an earlier call has finished) race
 * on it.  Each call clears the array's status word at its start; device-side
 * errors of these calls are not reported through gma_get_status().
 */
gma_status gma_forward_noalloc(const gma_desc *desc, const void *Qx, const void *Kx,
                               const void *V, const float *mu, const float *rho,
                               const float *pi_logits, float eps, int causal, void *out,
                               void *stream);

/*
 * Synchronises `stream`, reads the device status word of `workspace`, clears
 * it, and returns GMA_OK or the device error that was posted: GMA_ERR_TIMEOUT,
 * or GMA_ERR_BOUNDS from a library built with GMA_DEBUG_BOUNDS defined, whose
 * kernels check their global-memory indices (partial slots, heads, rows,
 * tiles) against the problem and skip, rather than perform, an access that
 * fails (a timeout is reported first when both were posted).
 */
gma_status gma_get_status(void *workspace, void *stream);

/* Static, human-readable name of a status code. */
const char *gma_status_string(gma_status status);

/* Library version, major*10000 + minor*100 + patch. */
int gma_version(void);

#ifdef __cplusplus
}
#endif

#endif /* GMA_H_ */
