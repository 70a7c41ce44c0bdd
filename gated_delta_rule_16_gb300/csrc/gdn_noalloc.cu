// gdn_noalloc.cu -- the allocation-free variant of the event-sparse prefill.
//
// Some callers cannot call cudaMalloc: a plugin inside a host runtime that owns
// every byte of device memory and hands the plugin only its inputs and outputs,
// or a latency-critical server that forbids allocation once it has started.
// gdn_prefill_sparse_noalloc() serves them: it runs the same kernels as
// gdn_prefill_sparse(), with the workspace carved from one fixed array in the
// library's own device memory instead of a caller buffer.
#include "gdn_internal.cuh"

namespace {

// The scratch: every GPU that loads the library holds these bytes until exit.
static __device__ __align__(256) unsigned char g_noalloc_scratch[GDN_NOALLOC_SCRATCH_BYTES];

// Device address of g_noalloc_scratch on the current device.  In host code the
// array's name is only a host-side stand-in, so the address is looked up with
// cudaGetSymbolAddress (with the device current) on every call: the lookup is a
// host-side table read, allocates nothing, and stays right if the context is
// reset or another context of the device is current (the module is then loaded
// again, at a new address).  The first lookup in a context loads the module and
// with it the array.
gdn_status scratch_for_current_device(void **out) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return GDN_ERR_CUDA;
    *out = p;
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
    // reads (CSR lists, counters, prefix, U, W, snapshots) is written earlier in
    // the same call, so the previous call's contents are harmless.
    // one stream: the library-owned streams of the multi-stream schedule are not made here
    return gdn::prefill_sparse_single_stream(shape, q, k, v, beta, g, h0, mask, solver, o, s_final, score, scratch,
                                             (size_t)GDN_NOALLOC_SCRATCH_BYTES, stream);
}

extern "C" gdn_status gdn_noalloc_status(void *stream) {
    void *scratch = nullptr;
    const gdn_status st = scratch_for_current_device(&scratch);
    if (st != GDN_OK) return st;
    // the status word sits where a caller workspace keeps it: the counters at offset 0
    return gdn_workspace_status(scratch, stream);
}
