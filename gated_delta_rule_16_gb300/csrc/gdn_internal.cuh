// gdn_internal.cuh -- shared declarations of libgdn's kernels (not part of the ABI).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "../../include/gdn.h"

namespace gdn {

constexpr int kChunk = 64;     // L: tokens per chunk
constexpr int kBlk = 16;       // solver block size
constexpr int kDim = 128;      // d == dv supported by this version
constexpr int kBlkAdj = 7;     // kept 16x16 blocks of the block-adjacent solver
constexpr int kBlkFull = 10;   // lower 16x16 blocks of the exact solver

// Compact coefficient blocks, stored in this order: the four diagonal blocks,
// the three sub-diagonal ones, then (exact solver only) the far blocks.
__host__ __device__ constexpr int blk_row(int b) {
    return b < 4 ? b : (b < 7 ? b - 3 : (b == 7 ? 2 : (b == 8 ? 3 : 3)));
}
__host__ __device__ constexpr int blk_col(int b) {
    return b < 4 ? b : (b < 7 ? b - 4 : (b == 7 ? 0 : (b == 8 ? 1 : 0)));
}

// Status bits latched in counts[2].
constexpr int kStatusEventOverflow = 1;
constexpr int kStatusSnapOverflow = 2;
constexpr int kStatusTimeout = 4;     // a kernel gave up a wait after its time limit

// Chunks per run of the tensor-core scan (the serial chain inside a run).
constexpr int kRunChunks = 16;  // the compaction kernel emits two runs per 32-chunk mask word

// ---- storage-type helpers --------------------------------------------------
template <typename T> struct io;
template <> struct io<float> {
    static __device__ __forceinline__ float ld(const float *p) { return *p; }
    static __device__ __forceinline__ void st(float *p, float x) { *p = x; }
};
template <> struct io<__nv_bfloat16> {
    static __device__ __forceinline__ float ld(const __nv_bfloat16 *p) { return __bfloat162float(*p); }
    static __device__ __forceinline__ void st(__nv_bfloat16 *p, float x) { *p = __float2bfloat16_rn(x); }
};

// ---- programmatic dependent launch ------------------------------------------
// A kernel launched with programmatic stream serialization may start while the
// previous kernel of the stream is still running (its CTAs fill the SMs the
// previous kernel's last wave leaves idle).  Every such kernel calls pdl_wait()
// in every CTA before it touches anything an earlier kernel wrote (and before any
// early exit, so that a kernel's completion still implies its predecessors'), and
// pdl_trigger() to let its own successor launch early.  Both are no-ops for a
// kernel launched without the attribute.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(bool pdl, void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                          Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// ---- problem description shared by the launchers -------------------------
struct Problem {
    int B, T, Nq, Nv, d, dv, C, G, P, R;
    gdn_dtype dtype;
    gdn_solver solver;
    int nblk;                  // 7 (block-adjacent) or 10 (exact)
    int online;                // workspace also holds the online-selection buffers
    int need_cbar;             // workspace holds the compact C-bar blocks (fp32 storage, online, W deferred)
    int need_runs;             // workspace holds the run maps of the run-map scan (bf16, scan_runs)
    int tail;                  // rows of the Tail-W score window (16 by default)
    int pdl;                   // launch the stage's first kernel as a programmatic dependent of the previous one
    int pdl_ok;                // programmatic dependent launch allowed in this prefill (later kernels of a stage)
    // Row range: when nrows > 0 the intra, scan and output launchers cover only the pairs of CSR
    // rows [row0, row0 + nrows) (physical pair row_pair[j]; the compaction must have completed);
    // nrows == 0: every pair, gridded by (pair, sequence).
    const int32_t *row_pair;
    int row0, nrows;
    int scan_full;             // masked full scan: W built for every chunk, the scan visits every chunk
    int states_expanded;       // one entry state per output group (slot i G + r), read by group
    const void *q, *k, *v;
    const float *beta, *g, *h0;
    const uint8_t *mask;       // NULL: every chunk is an event
    void *o;
    float *s_final, *score;
    cudaStream_t stream;
};

// Workspace layout (all offsets 256-byte aligned).
struct Workspace {
    int32_t *counts;           // [4]: E, n_snap, status, reserved
    int32_t *row_pair, *row_ptr, *ev_chunk, *grp_pred, *snap_slot;
    int32_t *run_first;        // [R, NR+1] first event of each run, per CSR row
    double *P;                 // [B, Nv, C+1] log2 decay prefix (Eq. 19)
    void *grp_info;            // [B, P, G] int4 {snapshot slot, kind, decay head 0, decay head 1}
    void *U;                   // U, then U' in place for events: bf16 head-major [B, Nv, T, dv], fp32 [B, T, Nv, dv]
    float *cbar;               // [B, Nv, C, nblk, 16, 16] compact C-bar blocks (bf16 on the tensor-core path)
    void *W;                   // [ev_cap, 2, 64, d] dtype, W of events (bf16 storage: -W, for the scan's U' product)
    void *snap;                // post-event state snapshots: fp32 [snap_cap, 2, d, dv]; bf16 storage: S^T [snap_cap, 2, dv, d]
    // tensor-core scan (bf16 storage only; NR = ceil(C / kRunChunks))
    void *amap;                // [R, 2, NR, 128, 128] bf16: A_r^T of each run
    float *bmap;               // [R, 2, NR, 128, 128] B_r^T of each run
    float *entry;              // [R, 2, NR, 128, 128] S^T entering each run
    // online selection only
    void *sel_ws;              // online selector scratch (selector_workspace_bytes)
    float *sel_score;          // [B, Nv, C] Tail-16 scores when the caller passes none
    uint8_t *sel_mask;         // [B, P, C] selected mask when the caller passes none
    int64_t ev_cap, snap_cap;
};

size_t workspace_layout(const Problem &pb, void *base, Workspace *ws);

// gdn_prefill_sparse with every kernel on the caller's stream (no library-owned streams).
gdn_status prefill_sparse_single_stream(const gdn_shape *shape, const void *q, const void *k, const void *v,
                                        const float *beta, const float *g, const float *h0, const uint8_t *mask,
                                        gdn_solver solver, void *o, float *s_final, float *score, void *workspace,
                                        size_t workspace_bytes, void *stream);

// ---- launchers (each returns cudaGetLastError()) --------------------------
// run_first (may be NULL): [R, NR+1] per CSR row, index of the first event of each run of
// kRunChunks chunks (entry NR: the row's end); needs kRunChunks = 16 (two runs per mask word).
// wait_first: the mask comes from the kernel before (else the kernel waits for it only before
// exiting); or_status: OR the status bits into counts[2] instead of overwriting it.
// part: 0 everything; 1 the row order only (row_pair); 2 everything but row_pair (after part 1).
// Masks too large for the word-parallel kernel do everything in part 1 and nothing in part 2.
cudaError_t launch_select(const Problem &pb, const gdn_events &ev, int64_t snap_cap, int32_t *run_first,
                          bool wait_first, bool or_status, int part = 0);
cudaError_t launch_prefix(const Problem &pb, const Workspace &ws);
cudaError_t launch_intra(const Problem &pb, const Workspace &ws);
cudaError_t launch_wbuild(const Problem &pb, const Workspace &ws);
cudaError_t launch_scan(const Problem &pb, const Workspace &ws);
cudaError_t launch_output(const Problem &pb, const Workspace &ws);
// part 0: run maps, 1: chain over runs, 2: per-run fix-up (writes U' and snapshots)
cudaError_t launch_scan_tc(const Problem &pb, const Workspace &ws, int part);
cudaError_t launch_output_tc(const Problem &pb, const Workspace &ws);
// The whole event scan in one launch: one warp per 16 state columns walks its CSR row
// once (writes U', the snapshots and S_final; bf16 storage only).
cudaError_t launch_scan_warp(const Problem &pb, const Workspace &ws);
// write_cbar: store the compact C-bar blocks (W is built later, after online selection)
cudaError_t launch_intra_tc(const Problem &pb, const Workspace &ws, bool write_cbar);
// online selection: mask [B,16,C] (and tiers [B,16], may be NULL) from scores [B,Nv,C]
// Single-token decode step from a state (see include/gdn.h, gdn_decode_step).
cudaError_t launch_decode(const gdn_shape &s, const void *q, const void *k, const void *v, const float *beta,
                          const float *a, float *state, void *o, cudaStream_t stream);
// Deferred W on tensor cores for the selected events, from the compact bf16 C-bar
// blocks that launch_intra_tc(..., write_cbar = true) stored (bf16 storage only).
cudaError_t launch_wbuild_tc(const Problem &pb, const Workspace &ws);
// Online selection (Eqs. 10-14) for 16 head pairs: score [B,32,C] -> mask [B,16,C],
// tier_out [B,16] (may be NULL); ws holds selector_workspace_bytes(B, C).
size_t selector_workspace_bytes(int B, int C);
// gamma [B,Nv,C] (may be NULL: read from pb.g at each chunk's last token)
cudaError_t launch_selector(const Problem &pb, const float *score, const float *eta, uint8_t *mask,
                            int32_t *tier_out, void *ws, const float *gamma = nullptr);

}  // namespace gdn
