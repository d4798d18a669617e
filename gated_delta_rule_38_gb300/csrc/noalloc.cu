// Forward pass without any device allocation by the caller or the library.
//
// Some callers cannot call cudaMalloc at all: code that runs inside a memory
// pool it does not own, embedded runtimes that forbid allocation after start-up,
// or callers in the middle of a region where an allocation would synchronise the
// device or change the memory map.  gdr_fwd asks them for a workspace; this entry
// point instead runs the same forward on a fixed scratch array that lives in the
// library's own device image.
//
// The scratch is a file-scope __device__ array of kNoAllocScratchBytes bytes.
// Every GPU that loads the library keeps it for the life of the process.  In host
// code the array's name is only a host-side stand-in, so its device address is
// looked up with cudaGetSymbolAddress, once per device, on that device.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "gdr.h"
#include "launch.h"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(64) << 20;  // 64 MiB
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_mu;
void *g_ptr[kMaxDevices];

// Device address of the scratch array on the current device (looked up once per device).
gdr_status scratch_ptr(void **out) {
    int dev = 0;
    cudaError_t ce = cudaGetDevice(&dev);
    if (ce != cudaSuccess) return gdr::cuda_fail(ce);
    if (dev < 0 || dev >= kMaxDevices) return GDR_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_ptr[dev]) {
        void *p = nullptr;
        if ((ce = cudaGetSymbolAddress(&p, g_noalloc_scratch)) != cudaSuccess) return gdr::cuda_fail(ce);
        if (p == nullptr) return GDR_ERR_CUDA;
        g_ptr[dev] = p;
    }
    *out = g_ptr[dev];
    return GDR_OK;
}

}  // namespace

extern "C" gdr_status gdr_fwd_noalloc(const gdr_problem *p, const void *q, const void *k, const void *v,
                                      const void *g, const void *beta, const float *h0, void *o, float *final_state,
                                      void *stream) {
    size_t need = 0;
    gdr_status st = gdr_fwd_workspace_size(p, &need);
    if (st != GDR_OK) return st;
    if (need > kNoAllocScratchBytes) return GDR_ERR_WORKSPACE;
    void *ws = nullptr;
    if ((st = scratch_ptr(&ws)) != GDR_OK) return st;
    // No byte of the workspace has to start at zero: every value the forward reads from it is
    // written earlier in the same call, so the previous call's leftovers do no harm.
    return gdr_fwd(p, q, k, v, g, beta, h0, o, final_state, nullptr, nullptr, nullptr, ws, kNoAllocScratchBytes,
                   stream);
}
