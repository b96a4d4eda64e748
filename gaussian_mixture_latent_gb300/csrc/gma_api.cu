// Host side of the C ABI declared in include/gma.h: argument validation,
// workspace sizing and carving, and the launch plan of each request.
//
// A request becomes a Plan: an ordered list of named kernel launches on one
// stream.  gma_forward() runs the plan; gma_forward_ex() runs it with
// caller-owned CUDA events recorded around each launch (per-kernel timing);
// gma_forward_plan() reports the launches without running anything.
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <functional>
#include <mutex>
#include <vector>

#include "gma_internal.h"

namespace gma {

cudaError_t set_dyn_smem(const void *kern, int bytes) {
    struct Entry {
        const void *kern;
        int dev, bytes;
    };
    static std::mutex mu;
    static std::vector<Entry> seen;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(mu);
    for (Entry &x : seen)
        if (x.kern == kern && x.dev == dev) {
            if (x.bytes >= bytes) return cudaSuccess;
            e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
            if (e == cudaSuccess) x.bytes = bytes;
            return e;
        }
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess) seen.push_back({kern, dev, bytes});
    return e;
}

namespace {

constexpr size_t kMaxDynSmem = 227 * 1024;

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

gma_status validate_desc(const gma_desc *d) {
    if (!d) return GMA_ERR_INVALID_ARG;
    if (d->B <= 0 || d->H <= 0 || d->N < 0) return GMA_ERR_INVALID_ARG;
    if (d->d <= 0 || d->K <= 0 || d->dv <= 0) return GMA_ERR_INVALID_ARG;
    if (d->in_dtype != GMA_F32 && d->in_dtype != GMA_BF16) return GMA_ERR_INVALID_ARG;
    if (d->out_dtype != GMA_F32 && d->out_dtype != GMA_BF16) return GMA_ERR_INVALID_ARG;
    if (!(d->var_floor > 0.f) || !std::isfinite(d->var_floor)) return GMA_ERR_INVALID_ARG;
    if (d->chunk < 0) return GMA_ERR_INVALID_ARG;
    if (d->d > 256 || d->K > 256 || d->dv > 256) return GMA_ERR_UNSUPPORTED;
    // Grid dimensions and row counts are 32-bit.
    if ((long long)d->B * d->H > 65535 || (long long)d->B * d->H * d->N > (1LL << 31))
        return GMA_ERR_UNSUPPORTED;
    return GMA_OK;
}

Problem make_problem(const gma_desc *d, int causal, float eps) {
    Problem p{};
    p.B = d->B; p.H = d->H; p.N = d->N; p.d = d->d; p.K = d->K; p.dv = d->dv;
    p.G = d->B * d->H;
    p.Nkv = d->N;
    p.in_dtype = d->in_dtype; p.out_dtype = d->out_dtype;
    p.var_floor = d->var_floor; p.eps = eps; p.causal = causal ? 1 : 0; p.chunk = d->chunk;
    return p;
}

struct Launch {
    const char *name;
    std::function<cudaError_t(cudaStream_t)> run;
};

struct Plan {
    static constexpr int kMax = 16;
    Launch step[kMax];
    int n = 0;
    size_t workspace = 0;
    void add(const char *name, std::function<cudaError_t(cudaStream_t)> f) { step[n++] = {name, std::move(f)}; }
};

struct Args {
    const void *Qx, *Kx, *V;
    const float *mu, *rho, *alpha;
    void *out;
    char *ws;
};

// Builds the launch list.  With args == nullptr only names and sizes are filled.
gma_status build_forward_plan(const Problem &p, const Args *a, Plan &plan) {
    Args z{};
    if (tc_bidir_supported(p)) {
        const TcLayout T = tc_layout(p);
        plan.workspace = T.total;
        const Args A = a ? *a : z;
        char *ws = A.ws;
        plan.add("tc_params", [=](cudaStream_t s) { return tc_params(p, T, A.mu, A.rho, A.alpha, ws, s); });
        plan.add("tc_write", [=](cudaStream_t s) { return tc_write(p, T, A.Kx, A.V, ws, s); });
        plan.add("tc_reduce", [=](cudaStream_t s) { return tc_reduce(p, T, ws, s); });
        plan.add("tc_read", [=](cudaStream_t s) { return tc_read(p, T, A.Qx, A.out, ws, s); });
        return GMA_OK;
    }
    // The tensor-core causal kernels scan in 128-row chunks (one MMA tile); they
    // refuse any other requested chunk rather than silently using their own.
    if ((tc_causal_supported(p) || tc_slice_supported(p)) && p.chunk != 0 && p.chunk != kTcChunkRows)
        return GMA_ERR_UNSUPPORTED;
    if (tc_causal_supported(p)) {
        const Args A = a ? *a : z;
        char *ws = A.ws;
        SegTable seg;
        if (tc_seg_plan(p, seg)) {
            // fewer heads than SMs: the segment-parallel scan over balanced chunk ranges, after
            // the prefix pass for the ranges that start inside a head
            const TcLayout T = tc_seg_layout(p, seg);
            plan.workspace = T.total;
            plan.add("tc_params", [=](cudaStream_t s) { return tc_params(p, T, A.mu, A.rho, A.alpha, ws, s); });
            if (seg.np > 0)
                plan.add("tc_prefix", [=](cudaStream_t s) { return tc_prefix(p, T, seg, A.Kx, A.V, ws, s); });
            plan.add("tc_causal_seg", [=](cudaStream_t s) {
                return tc_causal_seg(p, T, seg, A.Qx, A.Kx, A.V, A.out, ws, s); });
            return GMA_OK;
        }
        const TcLayout T = tc_causal_layout(p);
        plan.workspace = T.total;
        plan.add("tc_causal", [=](cudaStream_t s) {
            return tc_causal(p, T, A.Qx, A.Kx, A.V, A.mu, A.rho, A.alpha, A.out, ws, s); });
        return GMA_OK;
    }
    if (tc_slice_supported(p)) {
        const TcLayout T = tc_slice_layout(p);
        plan.workspace = T.total;
        const Args A = a ? *a : z;
        char *ws = A.ws;
        plan.add("tc_params", [=](cudaStream_t s) { return tc_params(p, T, A.mu, A.rho, A.alpha, ws, s); });
        plan.add("tc_rowstats", [=](cudaStream_t s) { return tc_rowstats(p, T, A.Qx, A.Kx, ws, s); });
        plan.add("tc_causal_slices", [=](cudaStream_t s) { return tc_causal_slices(p, T, A.Qx, A.Kx, A.V, ws, s); });
        plan.add("tc_combine", [=](cudaStream_t s) { return tc_combine(p, T, A.out, ws, s); });
        return GMA_OK;
    }
    const SimtLayout L = simt_layout(p);
    if (p.causal && simt_causal_smem(p) > kMaxDynSmem) return GMA_ERR_UNSUPPORTED;
    plan.workspace = L.total;
    const Args A = a ? *a : z;
    char *ws = A.ws;
    float *lam = reinterpret_cast<float *>(ws + L.lam);
    float *cdir = reinterpret_cast<float *>(ws + L.cdir);
    plan.add("simt_params", [=](cudaStream_t s) { return simt_params(p, A.rho, A.alpha, lam, cdir, s); });
    plan.add("simt_gamma_q", [=](cudaStream_t s) {
        return simt_gamma(p, A.Qx, A.mu, lam, cdir, reinterpret_cast<float *>(ws + L.gq), s); });
    plan.add("simt_gamma_k", [=](cudaStream_t s) {
        return simt_gamma(p, A.Kx, A.mu, lam, cdir, reinterpret_cast<float *>(ws + L.gk), s); });
    plan.add("simt_write", [=](cudaStream_t s) { return simt_write(p, A.V, ws, L, s); });
    plan.add("simt_reduce", [=](cudaStream_t s) { return simt_reduce(p, ws, L, s); });
    if (p.causal)
        plan.add("simt_causal_chunk", [=](cudaStream_t s) { return simt_causal(p, A.V, ws, L, A.out, s); });
    else
        plan.add("simt_read", [=](cudaStream_t s) { return simt_read(p, ws, L, A.out, s); });
    return GMA_OK;
}

gma_status run_plan(const Plan &plan, cudaStream_t s, void *const *events, int n_events) {
    for (int i = 0; i < plan.n; ++i) {
        if (events && 2 * i + 1 < n_events && events[2 * i])
            if (cudaEventRecord(static_cast<cudaEvent_t>(events[2 * i]), s) != cudaSuccess) return GMA_ERR_CUDA;
        if (plan.step[i].run(s) != cudaSuccess) return GMA_ERR_CUDA;
        if (events && 2 * i + 1 < n_events && events[2 * i + 1])
            if (cudaEventRecord(static_cast<cudaEvent_t>(events[2 * i + 1]), s) != cudaSuccess) return GMA_ERR_CUDA;
    }
    return GMA_OK;
}

// The fork and join events of gma_forward_multi: created once per host thread and
// device, outside any stream capture that comes later, and reused (a stream wait takes
// the event's state when it is enqueued, so re-recording it afterwards is safe).  Per
// thread, so that requests from two threads never wait on each other's events.
struct LaneEvents {
    int dev;
    cudaEvent_t fork, join;
};
thread_local std::vector<LaneEvents> tl_lane_events;

cudaError_t lane_events(int dev, cudaEvent_t &fork, cudaEvent_t &join) {
    for (const LaneEvents &e : tl_lane_events)
        if (e.dev == dev) {
            fork = e.fork;
            join = e.join;
            return cudaSuccess;
        }
    LaneEvents e{dev, nullptr, nullptr};
    cudaError_t err = cudaEventCreateWithFlags(&e.fork, cudaEventDisableTiming);
    if (err != cudaSuccess) return err;
    err = cudaEventCreateWithFlags(&e.join, cudaEventDisableTiming);
    if (err != cudaSuccess) {
        cudaEventDestroy(e.fork);
        return err;
    }
    tl_lane_events.push_back(e);
    fork = e.fork;
    join = e.join;
    return cudaSuccess;
}

// The backward's path for a problem: the tensor-core passes (bidirectional bf16,
// d = dv = K = 64, more than one 128-row tile), the CUDA-core kernels specialised to
// d = dv = K = 64 (causal with their 64-row tiles), or the general CUDA-core path.
enum class BwdPath { kNone, kTensor, kSimt64, kGeneral };

BwdPath backward_path(const Problem &p) {
    if (p.out_dtype != p.in_dtype) return BwdPath::kNone;
    if (bwd_tc_supported(p)) return BwdPath::kTensor;
    if (bwd_supported(p) && (!p.causal || p.chunk == 0 || p.chunk == kBwdChunkRows)) return BwdPath::kSimt64;
    return gb_supported(p) ? BwdPath::kGeneral : BwdPath::kNone;
}

gma_status check_forward_args(const gma_desc *desc, const void *Qx, const void *Kx, const void *V,
                              const float *mu, const float *rho, const float *pi_logits, float eps,
                              int causal, void *out, void *workspace) {
    gma_status st = validate_desc(desc);
    if (st != GMA_OK) return st;
    if (!(eps >= 0.f) || !std::isfinite(eps)) return GMA_ERR_INVALID_ARG;
    if (causal != 0 && causal != 1) return GMA_ERR_INVALID_ARG;
    if (!mu || !rho || !pi_logits) return GMA_ERR_INVALID_ARG;
    if (desc->N > 0 && (!Qx || !Kx || !V || !out)) return GMA_ERR_INVALID_ARG;
    const void *ptrs[] = {Qx, Kx, V, out, mu, rho, pi_logits, workspace};
    for (const void *q : ptrs)
        if (q && !aligned16(q)) return GMA_ERR_INVALID_ARG;
    return GMA_OK;
}

}  // namespace
}  // namespace gma

using namespace gma;

extern "C" {

gma_status gma_workspace_size(const gma_desc *desc, int causal, size_t *bytes) {
    gma_status st = validate_desc(desc);
    if (st != GMA_OK) return st;
    if (!bytes) return GMA_ERR_INVALID_ARG;
    Plan plan;
    st = build_forward_plan(make_problem(desc, causal, 0.f), nullptr, plan);
    if (st != GMA_OK) return st;
    *bytes = plan.workspace;
    return GMA_OK;
}

gma_status gma_workspace_init(void *workspace, size_t workspace_bytes, void *stream) {
    if (!workspace || workspace_bytes < kHeaderBytes) return GMA_ERR_WORKSPACE;
    return cudaMemsetAsync(workspace, 0, kHeaderBytes, static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? GMA_OK : GMA_ERR_CUDA;
}

gma_status gma_forward_ex(const gma_desc *desc, const void *Qx, const void *Kx, const void *V,
                          const float *mu, const float *rho, const float *pi_logits, float eps,
                          int causal, void *out, void *workspace, size_t workspace_bytes,
                          void *stream, void *const *events, int n_events) {
    gma_status st = check_forward_args(desc, Qx, Kx, V, mu, rho, pi_logits, eps, causal, out, workspace);
    if (st != GMA_OK) return st;
    const Problem p = make_problem(desc, causal, eps);
    const Args a{Qx, Kx, V, mu, rho, pi_logits, out, static_cast<char *>(workspace)};
    Plan plan;
    st = build_forward_plan(p, &a, plan);
    if (st != GMA_OK) return st;
    if (!workspace || workspace_bytes < plan.workspace) return GMA_ERR_WORKSPACE;
    if (p.N == 0) return GMA_OK;
    return run_plan(plan, static_cast<cudaStream_t>(stream), events, n_events);
}

gma_status gma_forward(const gma_desc *desc, const void *Qx, const void *Kx, const void *V,
                       const float *mu, const float *rho, const float *pi_logits, float eps,
                       int causal, void *out, void *workspace, size_t workspace_bytes,
                       void *stream) {
    return gma_forward_ex(desc, Qx, Kx, V, mu, rho, pi_logits, eps, causal, out, workspace,
                          workspace_bytes, stream, nullptr, 0);
}

gma_status gma_forward_multi_workspace_size(const gma_forward_call *calls, int n_calls, size_t *bytes,
                                            size_t *offsets) {
    if (!bytes || n_calls < 0 || (n_calls > 0 && !calls)) return GMA_ERR_INVALID_ARG;
    size_t off = 0;
    for (int i = 0; i < n_calls; ++i) {
        if (calls[i].causal != 0 && calls[i].causal != 1) return GMA_ERR_INVALID_ARG;
        size_t b = 0;
        const gma_status st = gma_workspace_size(&calls[i].desc, calls[i].causal, &b);
        if (st != GMA_OK) return st;
        if (offsets) offsets[i] = off;
        off += align_up(std::max(b, kHeaderBytes));
    }
    *bytes = off;
    return GMA_OK;
}

gma_status gma_forward_multi(const gma_forward_call *calls, int n_calls, void *workspace, size_t workspace_bytes,
                             void *stream, void *aux_stream) {
    std::vector<size_t> off(n_calls > 0 ? n_calls : 1);
    size_t need = 0;
    gma_status st = gma_forward_multi_workspace_size(calls, n_calls, &need, off.data());
    if (st != GMA_OK) return st;
    if (n_calls == 0) return GMA_OK;
    if (!workspace || workspace_bytes < need) return GMA_ERR_WORKSPACE;
    char *base = static_cast<char *>(workspace);
    for (int i = 0; i < n_calls; ++i) {
        const gma_forward_call &c = calls[i];
        st = check_forward_args(&c.desc, c.Qx, c.Kx, c.V, c.mu, c.rho, c.pi_logits, c.eps, c.causal, c.out,
                                base + off[i]);
        if (st != GMA_OK) return st;
        if (c.n_events < 0 || (c.n_events > 0 && !c.events)) return GMA_ERR_INVALID_ARG;
    }
    // Which calls run as one CTA per head, and how many SMs those hold at once (the calls
    // of the auxiliary lane run one after another).
    std::vector<Problem> prob(n_calls);
    std::vector<char> per_head(n_calls, 0);
    int held = 0, n_head = 0, n_rest = 0;
    for (int i = 0; i < n_calls; ++i) {
        const gma_forward_call &c = calls[i];
        prob[i] = make_problem(&c.desc, c.causal, c.eps);
        Plan probe;
        st = build_forward_plan(prob[i], nullptr, probe);
        if (st != GMA_OK) return st;
        if (prob[i].N == 0) continue;
        per_head[i] = probe.n == 1 && std::strcmp(probe.step[0].name, "tc_causal") == 0;
        if (per_head[i]) { held = std::max(held, prob[i].G); ++n_head; } else { ++n_rest; }
    }
    int nsm = 0, dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) !=
                                                 cudaSuccess)
        return GMA_ERR_CUDA;
    const bool side_by_side = aux_stream && aux_stream != stream && n_head > 0 && n_rest > 0 && nsm - held >= nsm / 8;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaStream_t aux = static_cast<cudaStream_t>(aux_stream);
    std::vector<Plan> plans(n_calls);
    for (int i = 0; i < n_calls; ++i) {
        const gma_forward_call &c = calls[i];
        if (side_by_side && !per_head[i]) prob[i].sm_budget = nsm - held;
        const Args a{c.Qx, c.Kx, c.V, c.mu, c.rho, c.pi_logits, c.out, base + off[i]};
        st = build_forward_plan(prob[i], &a, plans[i]);
        if (st != GMA_OK) return st;
    }
    if (!side_by_side) {
        for (int i = 0; i < n_calls; ++i) {
            if (prob[i].N == 0) continue;
            st = run_plan(plans[i], s, calls[i].events, calls[i].n_events);
            if (st != GMA_OK) return st;
        }
        return GMA_OK;
    }
    // Fork: aux_stream starts after the work queued on `stream`.  The per-head scans are
    // enqueued first, so that their CTAs take their SMs before the other calls' grids
    // spread over the rest.  Join: `stream` waits for aux_stream.
    cudaEvent_t fork = nullptr, join = nullptr;
    if (lane_events(dev, fork, join) != cudaSuccess) return GMA_ERR_CUDA;
    st = GMA_OK;
    if (cudaEventRecord(fork, s) != cudaSuccess || cudaStreamWaitEvent(aux, fork, 0) != cudaSuccess) st = GMA_ERR_CUDA;
    for (int i = 0; i < n_calls && st == GMA_OK; ++i)
        if (per_head[i]) st = run_plan(plans[i], aux, calls[i].events, calls[i].n_events);
    for (int i = 0; i < n_calls && st == GMA_OK; ++i)
        if (!per_head[i] && prob[i].N > 0) st = run_plan(plans[i], s, calls[i].events, calls[i].n_events);
    // the join is enqueued even after a failed launch, so that `stream` never runs ahead of aux_stream
    if (cudaEventRecord(join, aux) != cudaSuccess || cudaStreamWaitEvent(s, join, 0) != cudaSuccess)
        st = GMA_ERR_CUDA;
    return st;
}

gma_status gma_cross_workspace_size(const gma_desc *desc, int Nkv, size_t *bytes) {
    gma_status st = validate_desc(desc);
    if (st != GMA_OK) return st;
    if (!bytes || Nkv < 0 || (desc->N > 0 && Nkv == 0)) return GMA_ERR_INVALID_ARG;
    if ((long long)desc->B * desc->H * Nkv > (1LL << 31)) return GMA_ERR_UNSUPPORTED;
    Problem p = make_problem(desc, 0, 0.f);
    p.Nkv = Nkv;
    if (p.N == 0) { *bytes = align_up(kHeaderBytes); return GMA_OK; }
    if (!tc_bidir_supported(p)) return GMA_ERR_UNSUPPORTED;
    *bytes = tc_layout(p).total;
    return GMA_OK;
}

gma_status gma_forward_cross(const gma_desc *desc, int Nkv, const void *Qx, const void *Ky, const void *Vy,
                             const float *mu, const float *rho, const float *pi_logits, float eps, void *out,
                             void *workspace, size_t workspace_bytes, void *stream) {
    gma_status st = validate_desc(desc);
    if (st != GMA_OK) return st;
    if (Nkv < 0 || (desc->N > 0 && Nkv == 0) || !(eps >= 0.f) || !std::isfinite(eps)) return GMA_ERR_INVALID_ARG;
    if (!mu || !rho || !pi_logits) return GMA_ERR_INVALID_ARG;
    if (desc->N > 0 && (!Qx || !Ky || !Vy || !out)) return GMA_ERR_INVALID_ARG;
    const void *ptrs[] = {Qx, Ky, Vy, out, mu, rho, pi_logits, workspace};
    for (const void *q : ptrs)
        if (q && !aligned16(q)) return GMA_ERR_INVALID_ARG;
    if ((long long)desc->B * desc->H * Nkv > (1LL << 31)) return GMA_ERR_UNSUPPORTED;
    Problem p = make_problem(desc, 0, eps);
    p.Nkv = Nkv;
    if (p.N == 0) return GMA_OK;
    if (!tc_bidir_supported(p)) return GMA_ERR_UNSUPPORTED;
    const TcLayout L = tc_layout(p);
    if (!workspace || workspace_bytes < L.total) return GMA_ERR_WORKSPACE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    char *ws = static_cast<char *>(workspace);
    if (tc_params(p, L, mu, rho, pi_logits, ws, s) != cudaSuccess) return GMA_ERR_CUDA;
    if (tc_write(p, L, Ky, Vy, ws, s) != cudaSuccess) return GMA_ERR_CUDA;
    if (tc_reduce(p, L, ws, s) != cudaSuccess) return GMA_ERR_CUDA;
    return tc_read(p, L, Qx, out, ws, s) == cudaSuccess ? GMA_OK : GMA_ERR_CUDA;
}

gma_status gma_backward_workspace_size(const gma_desc *desc, int causal, size_t *bytes) {
    gma_status st = validate_desc(desc);
    if (st != GMA_OK) return st;
    if (!bytes || causal < 0 || causal > 1) return GMA_ERR_INVALID_ARG;
    const Problem p = make_problem(desc, causal, 0.f);
    switch (backward_path(p)) {
        case BwdPath::kTensor: *bytes = bwd_tc_layout(p).total; return GMA_OK;
        case BwdPath::kSimt64: *bytes = bwd_layout(p).total; return GMA_OK;
        case BwdPath::kGeneral: *bytes = gb_layout(p).total; return GMA_OK;
        default: return GMA_ERR_UNSUPPORTED;
    }
}

gma_status gma_backward(const gma_desc *desc, int causal, const void *Qx, const void *Kx, const void *V,
                        const float *mu, const float *rho, const float *pi_logits, float eps, const void *dO,
                        float *dQx, float *dKx, float *dV, float *dmu, float *drho, float *dpi_logits,
                        void *workspace, size_t workspace_bytes, void *stream) {
    gma_status st = validate_desc(desc);
    if (st != GMA_OK) return st;
    if (causal < 0 || causal > 1 || !(eps >= 0.f) || !std::isfinite(eps)) return GMA_ERR_INVALID_ARG;
    if (!mu || !rho || !pi_logits || !dmu || !drho || !dpi_logits) return GMA_ERR_INVALID_ARG;
    if (desc->N > 0 && (!Qx || !Kx || !V || !dO || !dQx || !dKx || !dV)) return GMA_ERR_INVALID_ARG;
    const void *ptrs[] = {Qx, Kx, V, dO, dQx, dKx, dV, mu, rho, pi_logits, dmu, drho, dpi_logits, workspace};
    for (const void *q : ptrs)
        if (q && !aligned16(q)) return GMA_ERR_INVALID_ARG;
    const Problem p = make_problem(desc, causal, eps);
    const BwdPath path = backward_path(p);
    if (path == BwdPath::kNone) return GMA_ERR_UNSUPPORTED;
    const size_t need = path == BwdPath::kTensor ? bwd_tc_layout(p).total
                      : path == BwdPath::kSimt64 ? bwd_layout(p).total : gb_layout(p).total;
    if (!workspace || workspace_bytes < need) return GMA_ERR_WORKSPACE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (p.N == 0) {     // the loss does not depend on the parameters
        const size_t kd = sizeof(float) * (size_t)p.H * p.K * p.d;
        if (cudaMemsetAsync(dmu, 0, kd, s) != cudaSuccess || cudaMemsetAsync(drho, 0, kd, s) != cudaSuccess ||
            cudaMemsetAsync(dpi_logits, 0, sizeof(float) * (size_t)p.H * p.K, s) != cudaSuccess)
            return GMA_ERR_CUDA;
        return GMA_OK;
    }
    char *ws = static_cast<char *>(workspace);
    const cudaError_t e =
        path == BwdPath::kTensor
            ? bwd_tc_run(p, bwd_tc_layout(p), Qx, Kx, V, mu, rho, pi_logits, dO, dQx, dKx, dV, dmu, drho, dpi_logits,
                         ws, s)
        : path == BwdPath::kSimt64
            ? bwd_run(p, bwd_layout(p), Qx, Kx, V, mu, rho, pi_logits, dO, dQx, dKx, dV, dmu, drho, dpi_logits, ws, s)
            : gb_run(p, gb_layout(p), Qx, Kx, V, mu, rho, pi_logits, dO, dQx, dKx, dV, dmu, drho, dpi_logits, ws, s);
    return e == cudaSuccess ? GMA_OK : GMA_ERR_CUDA;
}

gma_status gma_project(const gma_proj_desc *desc, const void *X, const void *Wq, const void *Wk, const void *Wv,
                       void *Qx, void *Kx, void *V, void *workspace, size_t workspace_bytes, void *stream) {
    if (!desc) return GMA_ERR_INVALID_ARG;
    const gma_proj_desc &d = *desc;
    if (d.B < 0 || d.N < 0 || d.D <= 0 || d.H <= 0 || d.d <= 0 || d.dv <= 0) return GMA_ERR_INVALID_ARG;
    if ((long long)d.B * d.H > (1LL << 30) || (long long)d.N > (1LL << 30)) return GMA_ERR_INVALID_ARG;
    if (!proj_supported(d.B > 0 ? d.B : 1, d.N > 0 ? d.N : 1, d.D, d.H, d.d, d.dv)) return GMA_ERR_UNSUPPORTED;
    if (!Wq || !Wk || !Wv) return GMA_ERR_INVALID_ARG;
    const bool empty = d.B == 0 || d.N == 0;
    if (!empty && (!X || !Qx || !Kx || !V)) return GMA_ERR_INVALID_ARG;
    const void *ptrs[] = {X, Wq, Wk, Wv, Qx, Kx, V, workspace};
    for (const void *q : ptrs)
        if (q && !aligned16(q)) return GMA_ERR_INVALID_ARG;
    if (!workspace || workspace_bytes < kHeaderBytes) return GMA_ERR_WORKSPACE;
    if (empty) return GMA_OK;
    return proj_run(d.B, d.N, d.D, d.H, d.d, d.dv, X, Wq, Wk, Wv, Qx, Kx, V, static_cast<char *>(workspace),
                    static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? GMA_OK
               : GMA_ERR_CUDA;
}

gma_status gma_decode_workspace_size(const gma_desc *desc, size_t *bytes) {
    gma_status st = validate_desc(desc);
    if (st != GMA_OK) return st;
    if (!bytes) return GMA_ERR_INVALID_ARG;
    const Problem p = make_problem(desc, 1, 0.f);
    if (!decode_supported(p)) return GMA_ERR_UNSUPPORTED;
    *bytes = decode_workspace(p);
    return GMA_OK;
}

gma_status gma_decode(const gma_desc *desc, const void *Qx, const void *Kx, const void *V, const float *mu,
                      const float *rho, const float *pi_logits, float eps, float *state, void *out,
                      void *workspace, size_t workspace_bytes, void *stream) {
    gma_status st = validate_desc(desc);
    if (st != GMA_OK) return st;
    if (!(eps >= 0.f) || !std::isfinite(eps) || !mu || !rho || !pi_logits || !state) return GMA_ERR_INVALID_ARG;
    if (desc->N > 0 && (!Qx || !Kx || !V || !out)) return GMA_ERR_INVALID_ARG;
    const void *ptrs[] = {Qx, Kx, V, out, mu, rho, pi_logits, state, workspace};
    for (const void *q : ptrs)
        if (q && !aligned16(q)) return GMA_ERR_INVALID_ARG;
    const Problem p = make_problem(desc, 1, eps);
    if (!decode_supported(p)) return GMA_ERR_UNSUPPORTED;
    if (!workspace || workspace_bytes < decode_workspace(p)) return GMA_ERR_WORKSPACE;
    if (p.N == 0) return GMA_OK;
    return decode_step(p, Qx, Kx, V, mu, rho, pi_logits, state, out, static_cast<cudaStream_t>(stream)) ==
                   cudaSuccess
               ? GMA_OK
               : GMA_ERR_CUDA;
}

gma_status gma_forward_plan(const gma_desc *desc, int causal, int *n_launches, const char **names,
                            int capacity) {
    gma_status st = validate_desc(desc);
    if (st != GMA_OK) return st;
    if (!n_launches || causal < 0 || causal > 1) return GMA_ERR_INVALID_ARG;
    Plan plan;
    st = build_forward_plan(make_problem(desc, causal, 0.f), nullptr, plan);
    if (st != GMA_OK) return st;
    *n_launches = desc->N > 0 ? plan.n : 0;
    for (int i = 0; names && i < capacity && i < plan.n; ++i) names[i] = plan.step[i].name;
    return GMA_OK;
}

gma_status gma_responsibilities(const gma_desc *desc, const void *X, const float *mu,
                                const float *rho, const float *pi_logits, float *gamma_out,
                                void *workspace, size_t workspace_bytes, void *stream) {
    gma_status st = validate_desc(desc);
    if (st != GMA_OK) return st;
    if (!mu || !rho || !pi_logits) return GMA_ERR_INVALID_ARG;
    if (desc->N > 0 && (!X || !gamma_out)) return GMA_ERR_INVALID_ARG;
    const void *ptrs[] = {X, gamma_out, mu, rho, pi_logits, workspace};
    for (const void *q : ptrs)
        if (q && !aligned16(q)) return GMA_ERR_INVALID_ARG;
    const Problem p = make_problem(desc, 0, 0.f);
    const SimtLayout L = simt_layout(p);
    if (!workspace || workspace_bytes < L.total) return GMA_ERR_WORKSPACE;
    if (p.N == 0) return GMA_OK;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    char *ws = static_cast<char *>(workspace);
    float *lam = reinterpret_cast<float *>(ws + L.lam);
    float *cdir = reinterpret_cast<float *>(ws + L.cdir);
    if (simt_params(p, rho, pi_logits, lam, cdir, s) != cudaSuccess) return GMA_ERR_CUDA;
    return simt_gamma(p, X, mu, lam, cdir, gamma_out, s) == cudaSuccess ? GMA_OK : GMA_ERR_CUDA;
}

gma_status gma_diagnostics_workspace_size(const gma_desc *desc, size_t *bytes) {
    gma_status st = validate_desc(desc);
    if (st != GMA_OK) return st;
    if (!bytes) return GMA_ERR_INVALID_ARG;
    const Problem p = make_problem(desc, 0, 0.f);
    if (p.N > 0 && !tc_diag_supported(p)) return GMA_ERR_UNSUPPORTED;
    *bytes = p.N > 0 ? tc_diag_layout(p).total : align_up(kHeaderBytes);
    return GMA_OK;
}

gma_status gma_diagnostics(const gma_desc *desc, const void *Qx, const float *mu, const float *rho,
                           const float *pi_logits, float *p_out, float *stats_out, int *z_out,
                           void *workspace, size_t workspace_bytes, void *stream) {
    gma_status st = validate_desc(desc);
    if (st != GMA_OK) return st;
    if (!mu || !rho || !pi_logits || !p_out || !stats_out) return GMA_ERR_INVALID_ARG;
    if (desc->N > 0 && !Qx) return GMA_ERR_INVALID_ARG;
    const void *ptrs[] = {Qx, mu, rho, pi_logits, workspace};
    for (const void *q : ptrs)
        if (q && !aligned16(q)) return GMA_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(p_out) | reinterpret_cast<uintptr_t>(stats_out) |
         reinterpret_cast<uintptr_t>(z_out)) & 3u)
        return GMA_ERR_INVALID_ARG;
    const Problem p = make_problem(desc, 0, 0.f);
    if (p.N == 0) return GMA_OK;
    if (!tc_diag_supported(p)) return GMA_ERR_UNSUPPORTED;
    const TcLayout L = tc_diag_layout(p);
    if (!workspace || workspace_bytes < L.total) return GMA_ERR_WORKSPACE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    char *ws = static_cast<char *>(workspace);
    if (tc_params(p, L, mu, rho, pi_logits, ws, s) != cudaSuccess) return GMA_ERR_CUDA;
    if (tc_diag(p, L, Qx, z_out, ws, s) != cudaSuccess) return GMA_ERR_CUDA;
    return tc_diag_finalize(p, L, p_out, stats_out, ws, s) == cudaSuccess ? GMA_OK : GMA_ERR_CUDA;
}

gma_status gma_selftest_timeout(void *workspace, size_t workspace_bytes, void *stream) {
    if (!workspace || workspace_bytes < kHeaderBytes) return GMA_ERR_WORKSPACE;
    if (!aligned16(workspace)) return GMA_ERR_INVALID_ARG;
    return selftest_timeout(workspace, static_cast<cudaStream_t>(stream)) == cudaSuccess ? GMA_OK : GMA_ERR_CUDA;
}

gma_status gma_get_status(void *workspace, void *stream) {
    if (!workspace) return GMA_ERR_WORKSPACE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    unsigned word = 0;
    if (cudaMemcpyAsync(&word, workspace, sizeof(word), cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return GMA_ERR_CUDA;
    if (cudaMemsetAsync(workspace, 0, sizeof(word), s) != cudaSuccess) return GMA_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return GMA_ERR_CUDA;
    if (word & kDevErrTimeout) return GMA_ERR_TIMEOUT;
    if (word & kDevErrBounds) return GMA_ERR_BOUNDS;
    return GMA_OK;
}

const char *gma_status_string(gma_status status) {
    switch (status) {
        case GMA_OK: return "GMA_OK";
        case GMA_ERR_INVALID_ARG: return "GMA_ERR_INVALID_ARG: invalid argument";
        case GMA_ERR_UNSUPPORTED: return "GMA_ERR_UNSUPPORTED: shape or dtype outside the supported range";
        case GMA_ERR_WORKSPACE: return "GMA_ERR_WORKSPACE: workspace missing or too small";
        case GMA_ERR_CUDA: return "GMA_ERR_CUDA: CUDA runtime error or failed launch";
        case GMA_ERR_TIMEOUT: return "GMA_ERR_TIMEOUT: a device-side bounded wait ran out";
        case GMA_ERR_BOUNDS: return "GMA_ERR_BOUNDS: a device-side index check failed (debug build)";
    }
    return "unknown gma_status";
}

int gma_version(void) { return 100; }

}  // extern "C"
