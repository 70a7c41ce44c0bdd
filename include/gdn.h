/*
 * gdn.h -- C ABI of libgdn: the chunkwise (64-token) Gated Delta Network
 * prefill core on NVIDIA GB300 (sm_103a), dense and event-sparse forms.
 *
 * Source of the operator: "SparseGDN: Chunk Sparse in Linear Attention"
 * (arXiv 2610.41420v1), as paraphrased by its Chinese reading notes:
 *   Sec. 2.1, Eqs. 1-4   dense chunkwise recurrence and chunk output
 *   Sec. 2.3, Eqs. 5-9   local Delta system, block-adjacent solver, Tail-16 score
 *   Sec. 2.5, Eqs. 15-16 deferred W, CSR event layout, device-resident event count
 *   Sec. 2.6, Eqs. 17-21 event-sparse propagation and prefix-gap recovery
 *   Sec. 2.7, Eqs. 22-25 two-chunk group output from compact state snapshots
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * Shapes.  B sequences of T tokens; Nq query/key heads of width d; Nv = 2*Nq
 * value heads of width dv.  Value heads 2p and 2p+1 form head pair p and read
 * query/key head p.  C = ceil(T/64) chunks (a partial last chunk holds the
 * remaining T - 64 (C-1) tokens), G = ceil(C/2) output groups, P = Nq pairs.
 * This version requires d == dv == 128 and C <= 16384 (T == 0 and B == 0 are
 * accepted).
 *
 * Layouts (row-major, contiguous, innermost last):
 *   q, k      [B, T, Nq, d]      dtype (bf16 or fp32)
 *   v, o      [B, T, Nv, dv]     dtype
 *   beta      [B, T, Nv]         fp32, per-token update strength
 *   g         [B, T, Nv]         fp32, log2 retention accumulated inside each
 *                                64-token chunk, inclusive of the token's own
 *                                gate (the pages' g_{c,h,i})
 *   mask      [B, P, C]          uint8 0/1 event mask, shared by a head pair
 *   h0, s_final [B, Nv, d, dv]   fp32 recurrent state (key dim x value dim)
 *   score     [B, Nv, C]         fp32 Tail-16 write score s_{c,h} (Eq. 9)
 *   O is the GDN-core output before RMSNorm, output gate and projection,
 *   scaled by 1/sqrt(d).
 *
 * Memory and streams.  Every pointer is a caller-owned DEVICE pointer on the
 * current CUDA device, 16-byte aligned (the workspace: 256-byte aligned).  The
 * library never allocates device memory, never frees and never synchronises,
 * except in the status queries.  Work is enqueued on `stream` (a cudaStream_t;
 * NULL = legacy default stream) and is complete only when that stream is.  The
 * bf16 prefills fork part of their kernels onto library-owned streams (made
 * once per device, at higher priority) with an event recorded on `stream`,
 * and join them back with events before returning, so `stream` alone orders
 * the work; a stream capture of `stream` takes the forked kernels in.  Make
 * the first prefill on a device outside a capture (it creates those streams).
 * Calls on distinct workspaces are independent (concurrent calls share the
 * library's streams, so their forked kernels run one call after the other);
 * two calls that share a workspace must be stream-ordered.  The event count E
 * never leaves the device.
 *
 * Errors.  Argument problems are detected on the host before anything is
 * enqueued and returned synchronously (GDN_ERR_NULL / SHAPE / DTYPE / ALIGN /
 * WORKSPACE / UNSUPPORTED / DEVICE).  A failed launch returns GDN_ERR_CUDA.
 * Conditions only the GPU can see (event or snapshot capacity exceeded, a
 * wait inside a kernel that ran past its time limit) are latched in a device
 * status word; the kernels never write past a capacity and never wait
 * without a limit, and gdn_workspace_status() / gdn_events_status() report
 * the latch.
 */
#ifndef GDN_H
#define GDN_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define GDN_API __attribute__((visibility("default")))
#else
#define GDN_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    GDN_OK = 0,
    GDN_ERR_NULL = 1,        /* a required pointer is NULL */
    GDN_ERR_SHAPE = 2,       /* unsupported or inconsistent sizes */
    GDN_ERR_DTYPE = 3,       /* unknown dtype or solver enum */
    GDN_ERR_ALIGN = 4,       /* a pointer is not 16-byte (workspace: 256-byte) aligned */
    GDN_ERR_WORKSPACE = 5,   /* workspace smaller than gdn_workspace_bytes() */
    GDN_ERR_UNSUPPORTED = 6, /* valid request this library does not implement */
    GDN_ERR_CUDA = 7,        /* a CUDA runtime call or launch failed */
    GDN_ERR_DEVICE = 8,      /* current device is not a compute-capability 10.3 GPU */
    GDN_ERR_CAPACITY = 9,    /* (device-latched) more events or snapshots than capacity */
    GDN_ERR_TIMEOUT = 10     /* (device-latched) a kernel wait exceeded its 2 s limit and was abandoned */
} gdn_status;

typedef enum { GDN_BF16 = 0, GDN_F32 = 1 } gdn_dtype;

/* Intra-chunk solver for M = I + A_Delta (Sec. 2.3).
 * EXACT ("Full64"): C = M^-1.  BLOCK_ADJ: only the four diagonal and three
 * sub-diagonal 16x16 blocks of M^-1 are kept (Eq. 7). */
typedef enum { GDN_SOLVER_EXACT = 0, GDN_SOLVER_BLOCK_ADJ = 1 } gdn_solver;

typedef struct {
    int32_t B, T, Nq, Nv, d, dv;
    gdn_dtype dtype; /* storage type of q, k, v, o (and of internal U / W) */
} gdn_shape;

/* CSR event lists (Sec. 2.5).  One row per (sequence b, head pair p), physical
 * row id i = b*P + p.  Rows are ordered by event count descending, ties by
 * physical id ascending ("long chains first"; a caller mask carries no tiers).
 * Events inside a row ascend in chunk index.  All arrays are caller-owned
 * device memory written by gdn_select_events(). */
typedef struct {
    int32_t *row_pair;  /* [B*P]       physical id of row j */
    int32_t *row_ptr;   /* [B*P+1]     offset of row j's first event; row_ptr[B*P] = E */
    int32_t *ev_chunk;  /* [capacity]  chunk index of event e */
    int32_t *grp_pred;  /* [B*P*G]     indexed by physical id: global index of the last
                                       event of that pair with chunk < 2r, or -1 */
    int32_t *snap_slot; /* [capacity]  dense number (in event order) of the events some
                                       group reads as predecessor, else -1 */
    int32_t *counts;    /* [4]         E, number of snapshots, status bits, reserved */
    int32_t capacity;   /* entries available in ev_chunk and snap_slot */
} gdn_events;

/* What gdn_prefill_ex computes: every chunk an event, a caller mask, or events
 * chosen on the GPU from the Tail-W scores (Sec. 2.4). */
typedef enum { GDN_MODE_DENSE = 0, GDN_MODE_SPARSE = 1, GDN_MODE_ONLINE = 2 } gdn_mode;

/* Execution variants (the pages' ablation axes; Secs. 3.4-3.5).  Zero-initialise:
 * every field's zero value is the default.
 *   tail_window  rows of the Tail-W write-score window, the last W rows of a
 *                chunk's U: 0 (= 16), 8, 16, 32 or 64 (Fig. 10).  Changes only
 *                the scores, and through them an online selection.
 *   w_deferred   0: with a mask known up front, W = C-bar K is built inside the
 *                intra step for the event chunks;  1: the intra step stores the
 *                compact C-bar blocks and a separate tensor-core kernel builds W
 *                for the events after compaction (the order online selection
 *                needs).  The results are identical bit for bit (bf16 storage;
 *                fp32 storage always builds W separately).
 *   scan_runs    bf16 storage only.  0: the event scan walks each CSR row once,
 *                the state held on chip for the whole row (every event applied
 *                once);  1: the row is cut into runs of 16 chunks whose affine
 *                maps are built in parallel, chained, then replayed (three
 *                launches; every event applied three times, on tcgen05 tensor
 *                cores).  Both compute the same recurrence (Eqs. 1-2, 17-21);
 *                their fp32 rounding orders differ, so the results agree to
 *                rounding, not bit for bit.  scan_runs = 1 needs the larger
 *                workspace that gdn_workspace_bytes_ex() reports for it.
 *   scan_full    1: the masked full scan, the pages' reference for the CSR
 *                scan (Table 6): the intra step builds W for every chunk and
 *                the scan visits every chunk, computing both products on each
 *                but keeping them on the mask's events only, with the same
 *                decay arithmetic (the gap factors of Eq. 21).  Identical
 *                results bit for bit; more work.  bf16, given mask or dense
 *                (not online selection, not w_deferred, not scan_runs).
 *   states_expanded  1: the pages' reference for compact states and mapped
 *                output (Table 6): the scan writes the entry state of every
 *                two-chunk output group to a slot of its own (dense group
 *                states, B*P*G slots), and the output reads its group's slot
 *                directly instead of the predecessor's compact snapshot
 *                through the group map.  Identical results bit for bit.  bf16,
 *                one-pass scan.
 *   online_split online selection in two calls, for head pairs sharded over
 *                ranks (tensor parallelism: the selection couples a sequence's
 *                16 pairs, Eq. 14).  Both calls use mode GDN_MODE_ONLINE, the
 *                rank's own pairs (any number) and the same workspace.
 *                1: the intra step only; writes `score` (required) and keeps
 *                U and the C-bar blocks in the workspace.  The caller gathers
 *                every rank's scores and chunk gate tails gamma (g at each
 *                chunk's last token) and selects with
 *                gdn_select_events_gamma().  2: the rest of the pipeline
 *                (compaction, deferred W, scan, output) on the workspace of
 *                call 1, with the rank's rows of that selection in `mask`.
 *                The two calls compute what one online prefill computes, bit
 *                for bit.
 *   reserved     must be zero. */
typedef struct {
    int32_t tail_window;
    int32_t w_deferred;
    int32_t scan_runs;
    int32_t scan_full;
    int32_t states_expanded;
    int32_t online_split;
    int32_t reserved[2];
} gdn_options;

/* Bytes of workspace the prefill entry points need for `shape`: sparse = 0
 * gdn_prefill_dense, 1 gdn_prefill_sparse, 2 gdn_prefill_sparse_online (all
 * with default execution variants).  0 for invalid shapes. */
GDN_API size_t gdn_workspace_bytes(const gdn_shape *shape, gdn_solver solver, int sparse);

/* Bytes of workspace gdn_prefill_ex needs for `mode` and the options `opt`
 * (NULL = defaults; equal to gdn_workspace_bytes for the same mode).  Some
 * variants keep extra buffers: w_deferred the compact C-bar blocks, scan_runs
 * the per-run affine maps.  0 for invalid shapes or options. */
GDN_API size_t gdn_workspace_bytes_ex(const gdn_shape *shape, gdn_solver solver, gdn_mode mode,
                                      const gdn_options *opt);

/* Bytes of one device buffer that holds the arrays of a gdn_events for `shape`
 * with room for `capacity` events: row_pair, row_ptr, ev_chunk, grp_pred,
 * snap_slot and counts, in that order, each at a 256-byte aligned offset.
 * 0 for an invalid shape or a negative capacity.  A capacity of B*P*C always
 * suffices (every chunk of every pair an event); the pages' selector bounds E
 * by 16 k_H per sequence (Sec. 2.5). */
GDN_API size_t gdn_events_bytes(const gdn_shape *shape, int32_t capacity);

/* Points the arrays of *events into `buffer` (device memory of at least
 * gdn_events_bytes(shape, capacity) bytes, 256-byte aligned) in the layout
 * gdn_events_bytes() describes, and sets events->capacity.  Host-only: nothing
 * is enqueued and the buffer is not touched.  Returns GDN_ERR_NULL, _SHAPE or
 * _ALIGN on bad arguments. */
GDN_API gdn_status gdn_events_carve(const gdn_shape *shape, int32_t capacity, void *buffer, gdn_events *events);

/* Event compaction (Sec. 2.5, Eq. 16): turn the [B,P,C] 0/1 mask into CSR
 * event lists, the per-group predecessor event and the snapshot numbering.
 * E = sum of the mask stays on the device (counts[0]).  If E > capacity the
 * status bit 1 is set in counts[2], nothing past capacity is written and
 * gdn_events_status() returns GDN_ERR_CAPACITY.  No workspace needed. */
GDN_API gdn_status gdn_select_events(const gdn_shape *shape, const uint8_t *mask,
                             gdn_events *events, void *stream);

/* Online event selection (Sec. 2.4, Eqs. 10-14) for 16 head pairs (Nv == 32):
 * from the Tail-16 scores score [B,Nv,C] (fp32, Eq. 9), the gates g [B,T,Nv]
 * (gamma = g at each chunk's last token) and an optional output-visibility
 * energy eta [B,Nv] (NULL: G_h = 1), choose per sequence the tier of every pair
 * (Eq. 14) and its chunks (anchors 0 and C-1 plus the best k_tier - 2 chunks by
 * the in-pair rank q, Eqs. 10 and 13); writes mask_out [B,16,C] (0/1) and, if
 * non-NULL, tier_out [B,16] (0 low, 1 mid, 2 high).  Ties: q descending then
 * lower chunk; pair gains descending then lower pair; B(x,k) ties take the
 * smaller k.  Workspace: gdn_select_scored_workspace_bytes(shape), 256-byte
 * aligned.  Other head counts return GDN_ERR_UNSUPPORTED. */
GDN_API gdn_status gdn_select_events_scored(const gdn_shape *shape, const float *score, const float *g,
                                    const float *eta, uint8_t *mask_out, int32_t *tier_out,
                                    void *workspace, size_t workspace_bytes, void *stream);
GDN_API size_t gdn_select_scored_workspace_bytes(const gdn_shape *shape);

/* gdn_select_events_scored with the chunk gate tails given directly: gamma
 * [B,Nv,C] fp32 (gamma[b,h,c] = g at chunk c's last token) instead of g
 * [B,T,Nv].  For a selection over head pairs gathered from several ranks
 * (online_split), where each rank holds only its own heads' gates.  Same
 * results as gdn_select_events_scored on the same values.  shape gives B, C
 * (through T) and Nv == 32; workspace as gdn_select_scored_workspace_bytes. */
GDN_API gdn_status gdn_select_events_gamma(const gdn_shape *shape, const float *score, const float *gamma,
                                           const float *eta, uint8_t *mask_out, int32_t *tier_out,
                                           void *workspace, size_t workspace_bytes, void *stream);

/* Synchronises `stream` and reports the status bits of an events struct. */
GDN_API gdn_status gdn_events_status(const gdn_events *events, void *stream);

/* Dense prefill (Secs. 2.1 and 2.3; Eqs. 1-8): every chunk is a recurrent
 * event.  Writes o and s_final (the state after the last chunk, for decoding).
 * h0 may be NULL (zero initial state); score may be NULL. */
GDN_API gdn_status gdn_prefill_dense(const gdn_shape *shape,
                             const void *q, const void *k, const void *v,
                             const float *beta, const float *g, const float *h0,
                             gdn_solver solver, void *o, float *s_final, float *score,
                             void *workspace, size_t workspace_bytes, void *stream);

/* Event-sparse prefill (Secs. 2.3-2.7; Eqs. 5-25).  Runs the whole pipeline on
 * the GPU: intra-chunk solve and Tail-16 score for every chunk, mask -> CSR
 * compaction, deferred W for selected events only, the event scan (read and
 * write only on selected events, decay always), and the two-chunk group
 * output from compact state snapshots.  Selected chunks write U' in place of
 * U; unselected chunks keep U.  mask: [B,P,C] uint8 0/1.  h0 and score may be
 * NULL. */
GDN_API gdn_status gdn_prefill_sparse(const gdn_shape *shape,
                              const void *q, const void *k, const void *v,
                              const float *beta, const float *g, const float *h0,
                              const uint8_t *mask, gdn_solver solver,
                              void *o, float *s_final, float *score,
                              void *workspace, size_t workspace_bytes, void *stream);

/* Event-sparse prefill with online selection, the pages' full pipeline
 * (Secs. 2.3-2.7): intra step (U, Tail-16 scores, compact C-bar), online
 * selection (as gdn_select_events_scored), compaction, deferred W for the
 * selected events only, event scan, group output.  16 head pairs only.
 * score (may be NULL) receives the Tail-16 scores, mask_out (may be NULL) the
 * selected mask [B,16,C], tier_out (may be NULL) the tiers [B,16]; eta may be
 * NULL.  Workspace: gdn_workspace_bytes(shape, solver, 2). */
GDN_API gdn_status gdn_prefill_sparse_online(const gdn_shape *shape,
                                     const void *q, const void *k, const void *v,
                                     const float *beta, const float *g, const float *h0,
                                     const float *eta, gdn_solver solver,
                                     void *o, float *s_final, float *score, uint8_t *mask_out,
                                     int32_t *tier_out, void *workspace, size_t workspace_bytes,
                                     void *stream);

/* The general prefill: `mode` selects dense (mask ignored), sparse (mask
 * required) or online selection (eta, mask_out and tier_out as in
 * gdn_prefill_sparse_online, 16 head pairs); `opt` (NULL = defaults) selects
 * execution variants.  Arguments otherwise as gdn_prefill_sparse; workspace
 * gdn_workspace_bytes_ex(shape, solver, mode, opt).  Unknown option values return
 * GDN_ERR_UNSUPPORTED before anything is enqueued. */
GDN_API gdn_status gdn_prefill_ex(const gdn_shape *shape, gdn_mode mode,
                          const void *q, const void *k, const void *v,
                          const float *beta, const float *g, const float *h0,
                          const uint8_t *mask, const float *eta, gdn_solver solver,
                          const gdn_options *opt, void *o, float *s_final, float *score,
                          uint8_t *mask_out, int32_t *tier_out, void *workspace,
                          size_t workspace_bytes, void *stream);

/* One autoregressive decode step from a state, e.g. the S_final of a prefill
 * (the pages return S_C for the decoding that follows; Sec. 2.6).  It is
 * Eqs. 1-4 for a chunk of a single token whose log2 retention is a:
 *   U' = beta v - beta 2^a S^T k,   S <- 2^a S + k U'^T,
 *   o  = [2^a S^T q + <q,k> U'] / sqrt(d)   (= S_new^T q / sqrt(d)).
 * shape: B sequences, T == 1, Nq, Nv = 2 Nq, d = dv = 128, dtype of q, k, v, o.
 * q, k [B,Nq,d]; v [B,Nv,dv]; beta [B,Nv] fp32; a [B,Nv] fp32: this token's
 * log2 retention (the increment of g; g of a prefill is its within-chunk
 * running sum); state [B,Nv,d,dv] fp32, updated in place; o [B,Nv,dv] out.
 * Value head h reads query/key head h/2.  All device pointers, 16-byte aligned.
 * Enqueues one kernel on `stream`; no workspace. */
GDN_API gdn_status gdn_decode_step(const gdn_shape *shape, const void *q, const void *k, const void *v,
                                   const float *beta, const float *a, float *state, void *o, void *stream);

/* Prefill with HOST inputs and outputs: the same computation as
 * gdn_prefill_sparse (mask != NULL) or gdn_prefill_dense (mask == NULL), with
 * q, k, v, beta, g, h0 (may be NULL), mask and the outputs o, s_final in host
 * memory, laid out as in those calls.  On `stream` the call enqueues one
 * cudaMemcpyAsync per input into device staging carved from the workspace, the
 * prefill, and one cudaMemcpyAsync per output back to the host; it returns
 * without waiting (synchronise the stream before reading o and s_final).  Host
 * buffers should be page-locked (cudaHostAlloc / cudaHostRegister): otherwise
 * the copies do not overlap with other work.  Calls on different streams with
 * different workspaces run concurrently, so a caller can overlap one call's
 * copies with another call's kernels.  Workspace (device, 256-byte aligned):
 * gdn_prefill_host_workspace_bytes(shape, solver, mask != NULL). */
GDN_API gdn_status gdn_prefill_host(const gdn_shape *shape,
                            const void *q, const void *k, const void *v,
                            const float *beta, const float *g, const float *h0,
                            const uint8_t *mask, gdn_solver solver,
                            void *o, float *s_final, void *workspace, size_t workspace_bytes,
                            void *stream);
GDN_API size_t gdn_prefill_host_workspace_bytes(const gdn_shape *shape, gdn_solver solver, int sparse);

/* Allocation-free event-sparse prefill.  The paper has no counterpart: this
 * is a deployment aid for callers that cannot allocate device memory -- for
 * example a plugin inside a host runtime that owns all device memory and
 * passes the plugin only its inputs and outputs, or a latency-critical server
 * that forbids cudaMalloc after start-up.  Same arguments, pipeline and
 * results as gdn_prefill_sparse(), but no workspace argument: the scratch is a
 * fixed array of GDN_NOALLOC_SCRATCH_BYTES (64 MiB) in the library's device
 * memory, which every GPU that loads the library holds until the process
 * exits.  The call allocates nothing and calls no allocating routine.
 *   - Size limit: shapes with gdn_workspace_bytes(shape, solver, 1) above
 *     64 MiB are rejected with GDN_ERR_WORKSPACE before anything is enqueued
 *     (with this version's workspace layout: B=1, Nq=16, bf16 up to
 *     T = 2688; one head pair in fp32 up to T = 20352).
 *   - Set-up: the array belongs to the library's device code, which CUDA loads
 *     lazily: the first call in each context (this entry point or
 *     gdn_noalloc_status) loads it, claiming the 64 MiB then, and looks up its
 *     address with that device current.  Make that first call at start-up,
 *     before a host runtime reserves the rest of the device memory and before
 *     any stream capture.  Every call looks the address up again (no cache), so
 *     a reset context or another context of the same device is handled.
 *   - Sharing: every call uses the same array and it keeps the last call's
 *     contents.  Nothing in it must start at zero (each value read is written
 *     earlier in the same call), but calls that overlap on the GPU (other
 *     streams, other host threads) race on it: serialise them.
 *   - Failure detection: the device status word lives in that array; read it
 *     with gdn_noalloc_status(), which reports the last call on the current
 *     device. */
#define GDN_NOALLOC_SCRATCH_BYTES (64ull << 20)
GDN_API gdn_status gdn_prefill_sparse_noalloc(const gdn_shape *shape,
                                      const void *q, const void *k, const void *v,
                                      const float *beta, const float *g, const float *h0,
                                      const uint8_t *mask, gdn_solver solver,
                                      void *o, float *s_final, float *score, void *stream);

/* Synchronises `stream` and reports the device-latched status (GDN_OK,
 * GDN_ERR_CAPACITY or GDN_ERR_TIMEOUT) of the last gdn_prefill_sparse_noalloc()
 * call on the current device, read from the library's scratch array.  Also
 * loads that array when called first (see the set-up note above).  Allocates
 * nothing.  No counterpart in the paper: part of the allocation-free entry
 * point. */
GDN_API gdn_status gdn_noalloc_status(void *stream);

/* Self-test of failure detection: every wait inside the kernels is bounded in
 * time.  Launches one thread that waits on a barrier nothing arrives at, with
 * a limit of limit_ms (1..2000) milliseconds; the wait must give up, latch the
 * timeout bit (status[2] & 4, the same bit a prefill latches as
 * GDN_ERR_TIMEOUT) and return, leaving the context usable.  status: caller
 * device buffer of 4 int32 (status[3] receives the milliseconds waited).
 * Synchronises `stream`.  Returns GDN_OK when the wait timed out as designed,
 * GDN_ERR_DEVICE when it did not. */
GDN_API gdn_status gdn_selftest_wait_timeout(int32_t *status, int32_t limit_ms, void *stream);

/* Synchronises `stream` and reports the device-latched status of the last
 * prefill that used `workspace` (GDN_OK, GDN_ERR_CAPACITY or GDN_ERR_TIMEOUT). */
GDN_API gdn_status gdn_workspace_status(const void *workspace, void *stream);

GDN_API const char *gdn_status_string(gdn_status status);

/* Stage timing for benchmarks.  enable = 1: each following prefill records a
 * CUDA event before its first and after each pipeline stage on its own stream
 * (stages: 0 compaction, 1 log-decay prefix, 2 intra, 3 deferred W, 4 scan
 * run maps, 5 scan chain over runs, 6 scan (the one-pass scan, the run-map
 * fix-up, or the fp32 scan), 7 group output, 8 online selector; a stage a path
 * does not run reads 0), for up to 256 prefills; while recording, a prefill
 * runs every kernel on the caller's stream, one after another.  enable = 2:
 * nothing is recorded and the prefills keep their normal schedule; only the
 * kernels they launch are counted.  0: off.  Enabling (again) drops earlier
 * records.  Not thread-safe: one host thread drives the profiler.  The events
 * are created on the first enable = 1 (no device memory). */
GDN_API gdn_status gdn_profile_enable(int enable);

/* Synchronises on the recorded events, writes the summed milliseconds of each
 * stage over all recorded prefills to stage_ms[0..n_stages) (n_stages <= 9;
 * zeros under enable = 2), the number of prefills run since enabling to
 * *n_prefills, the number of kernels they launched to *n_launches (may be
 * NULL), and clears the records. */
GDN_API gdn_status gdn_profile_read(float *stage_ms, int32_t n_stages, int32_t *n_prefills,
                                    int64_t *n_launches);

/* Library ABI version (major*10000 + minor*100 + patch). */
GDN_API int32_t gdn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* GDN_H */
