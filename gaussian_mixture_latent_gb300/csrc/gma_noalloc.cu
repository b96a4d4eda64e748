// gma_forward_noalloc: the forward for callers that cannot allocate device
// memory themselves.
//
// Some callers cannot call cudaMalloc: code running under a memory manager
// that owns every device allocation in the process (a framework's caching
// allocator, an inference server that hands out memory budgets), and
// latency-sensitive loops that cannot take cudaMalloc's implicit device-wide
// synchronisation.  Such callers can still run the forward: this entry point
// uses a fixed scratch buffer compiled into the library instead of a
// caller-provided workspace.  It allocates nothing.
//
// The scratch is a file-scope device array of GMA_NOALLOC_SCRATCH_BYTES.
// Every GPU that loads the library holds it until the process exits.  In
// host code the array's name is only a host-side stand-in, so its device
// address is looked up once per device with cudaGetSymbolAddress (with that
// device current) on the first call made on that device; that first call
// should therefore come before any stream capture.
//
// All calls on a device share the one array, and it keeps the contents the
// last call left.  Each call clears the status word at its start; everything
// else the kernels read from scratch they first write in the same call.
// Calls whose work overlaps on the GPU (different streams, or a call on one
// stream while another is still running) race on the shared scratch.
#include <cmath>
#include <cstdint>
#include <mutex>

#include "gma_internal.h"

namespace {

constexpr size_t kScratchBytes = GMA_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

std::mutex g_setup_mutex;
void *g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (set-up on first use).
gma_status scratch_for_current_device(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return GMA_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return GMA_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (!g_scratch_ptr[dev]) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) return GMA_ERR_CUDA;
        g_scratch_ptr[dev] = ptr;
    }
    *out = g_scratch_ptr[dev];
    return GMA_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// The pointer and scalar checks gma_forward makes, done here first so that a
// rejected call enqueues nothing (not even the status-word clear).
gma_status check_args(const gma_desc *desc, const void *Qx, const void *Kx, const void *V,
                      const float *mu, const float *rho, const float *pi_logits, float eps,
                      int causal, const void *out) {
    if (!(eps >= 0.f) || !std::isfinite(eps)) return GMA_ERR_INVALID_ARG;
    if (causal != 0 && causal != 1) return GMA_ERR_INVALID_ARG;
    if (!mu || !rho || !pi_logits) return GMA_ERR_INVALID_ARG;
    if (desc->N > 0 && (!Qx || !Kx || !V || !out)) return GMA_ERR_INVALID_ARG;
    const void *ptrs[] = {Qx, Kx, V, out, mu, rho, pi_logits};
    for (const void *q : ptrs)
        if (q && !aligned16(q)) return GMA_ERR_INVALID_ARG;
    return GMA_OK;
}

}  // namespace

extern "C" gma_status gma_forward_noalloc(const gma_desc *desc, const void *Qx, const void *Kx,
                                          const void *V, const float *mu, const float *rho,
                                          const float *pi_logits, float eps, int causal, void *out,
                                          void *stream) {
    size_t need = 0;
    gma_status st = gma_workspace_size(desc, causal, &need);
    if (st != GMA_OK) return st;
    st = check_args(desc, Qx, Kx, V, mu, rho, pi_logits, eps, causal, out);
    if (st != GMA_OK) return st;
    if (need > kScratchBytes) return GMA_ERR_WORKSPACE;
    if (desc->N == 0) return GMA_OK;
    void *scratch = nullptr;
    st = scratch_for_current_device(&scratch);
    if (st != GMA_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(scratch, 0, gma::kHeaderBytes, s) != cudaSuccess) return GMA_ERR_CUDA;
    return gma_forward(desc, Qx, Kx, V, mu, rho, pi_logits, eps, causal, out, scratch,
                       kScratchBytes, stream);
}
