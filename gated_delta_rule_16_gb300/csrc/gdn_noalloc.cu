// gdn_noalloc.cu -- the allocation-free variant of the event-sparse prefill.
//
// Some callers cannot call cudaMalloc: a plugin inside a host runtime that owns
// every byte of device memory and hands the plugin only its inputs and outputs,
// or a latency-critical server that forbids allocation once it has started.
// gdn_prefill_sparse_noalloc() serves them: it runs the same kernels as
// gdn_prefill_sparse(), with the workspace carved from one fixed array in the
// library's own device memory instead of a caller buffer.
#include <mutex>

#include "gdn_internal.cuh"

namespace {

// The scratch: every GPU that loads the library holds these bytes until exit.
static __device__ __align__(256) unsigned char g_noalloc_scratch[GDN_NOALLOC_SCRATCH_BYTES];

// Device address of g_noalloc_scratch per device ordinal.  In host code the
// array's name is only a host-side stand-in, so the address is looked up once
// per device with cudaGetSymbolAddress (with that device current).
constexpr int kMaxDevices = 64;
void *g_scratch_addr[kMaxDevices] = {nullptr};
std::mutex g_scratch_mutex;

gdn_status scratch_for_current_device(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return GDN_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return GDN_ERR_DEVICE;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (!g_scratch_addr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return GDN_ERR_CUDA;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return GDN_OK;
}

}  // namespace

extern "C" gdn_status gdn_prefill_sparse_noalloc(const gdn_shape *shape, const void *q, const void *k,
                                                 const void *v, const float *beta, const float *g,
                                                 const float *h0, const uint8_t *mask, gdn_solver solver,
                                                 void *o, float *s_final, float *score, void *stream) {
    const size_t need = gdn_workspace_bytes(shape, solver, 1);
    if (need == 0) {
        // invalid shape or solver: let the regular entry point name the error
        // (it returns before touching any pointer or enqueuing anything)
        return gdn_prefill_sparse(shape, q, k, v, beta, g, h0, mask, solver, o, s_final, score, nullptr, 0, stream);
    }
    if (need > (size_t)GDN_NOALLOC_SCRATCH_BYTES) return GDN_ERR_WORKSPACE;
    void *scratch = nullptr;
    const gdn_status st = scratch_for_current_device(&scratch);
    if (st != GDN_OK) return st;
    // Nothing in the scratch needs to start at zero: every value the pipeline
    // reads (CSR lists, counters, prefix, U, C-bar, W, snapshots) is written
    // earlier in the same call, so the previous call's contents are harmless.
    return gdn_prefill_sparse(shape, q, k, v, beta, g, h0, mask, solver, o, s_final, score, scratch,
                              (size_t)GDN_NOALLOC_SCRATCH_BYTES, stream);
}
