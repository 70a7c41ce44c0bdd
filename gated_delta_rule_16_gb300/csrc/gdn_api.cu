// gdn_api.cu -- the extern "C" entry points of libgdn (declared in include/gdn.h):
// argument validation, workspace carving and the launch sequence of the
// prefill pipeline.  No allocation, no synchronisation (except the status
// queries), no host copy of the event count.
#include <cstring>
#include <mutex>

#include "gdn_internal.cuh"

namespace gdn {
namespace {

constexpr size_t kAlign = 256;

inline size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

inline bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

// ---- stage profiler (benchmark aid; see gdn_profile_enable) ----------------
// Stages: 0 select (compaction), 1 prefix, 2 intra, 3 deferred W, 4 scan run maps,
// 5 scan chain, 6 scan (fix-up / whole scan), 7 output, 8 online selector.
constexpr int kStages = 9;
constexpr int kProfSlots = 256;
struct Profiler {
    int mode = 0;                              // 0 off, 1 stage events (one stream), 2 count kernels only
    bool created = false;
    int used = 0;                              // prefills with stage events recorded
    int64_t calls = 0;                         // prefills run while enabled
    int64_t launches = 0;                      // kernels those prefills launched
    cudaEvent_t ev[kProfSlots][2 * kStages];  // start and end of every stage
};
Profiler g_prof;

// Returns the event row of this prefill, or nullptr when not recording stage events.
cudaEvent_t *prof_slot() {
    if (g_prof.mode != 1 || g_prof.used >= kProfSlots) return nullptr;
    return g_prof.ev[g_prof.used++];
}

int device_ok() {
    // cache per device: 0 unknown, 1 ok, 2 not a compute-capability 10.3 part
    static int state[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    if (state[dev] == 0) {
        int major = 0, minor = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
            return 0;
        state[dev] = (major == 10 && minor == 3) ? 1 : 2;
    }
    return state[dev] == 1;
}

gdn_status check_shape(const gdn_shape *s) {
    if (!s) return GDN_ERR_NULL;
    if (s->dtype != GDN_BF16 && s->dtype != GDN_F32) return GDN_ERR_DTYPE;
    if (s->B < 0 || s->T < 0 || s->Nq <= 0 || s->Nv != 2 * s->Nq) return GDN_ERR_SHAPE;
    if (s->d != kDim || s->dv != kDim) return GDN_ERR_UNSUPPORTED;
    // C = ceil(T / 64) chunks; a partial last chunk holds the remaining T - 64 (C - 1) tokens
    const int64_t C = ((int64_t)s->T + kChunk - 1) / kChunk;
    if (C > 16384) return GDN_ERR_UNSUPPORTED;  // compaction stages a row's mask bits in shared memory
    // index arithmetic uses int32 for chunk/row/event counts
    // event tiles are addressed by int32 TMA row coordinates: events x 128 rows < 2^31
    if ((int64_t)s->B * s->Nq * C >= (int64_t)1 << 24) return GDN_ERR_SHAPE;
    if ((int64_t)s->B * s->T >= (int64_t)1 << 31) return GDN_ERR_SHAPE;
    if ((int64_t)s->B * s->Nq > 8192) return GDN_ERR_UNSUPPORTED;  // compaction keeps rows in shared memory
    return GDN_OK;
}

void fill_problem(const gdn_shape *s, gdn_solver solver, Problem *pb) {
    std::memset(pb, 0, sizeof(*pb));
    pb->B = s->B; pb->T = s->T; pb->Nq = s->Nq; pb->Nv = s->Nv; pb->d = s->d; pb->dv = s->dv;
    pb->C = (s->T + kChunk - 1) / kChunk;
    pb->G = (pb->C + 1) / 2;
    pb->P = s->Nq;
    pb->R = s->B * s->Nq;
    pb->dtype = s->dtype;
    pb->solver = solver;
    pb->nblk = solver == GDN_SOLVER_EXACT ? kBlkFull : kBlkAdj;
    pb->tail = kBlk;
}

size_t elem_size(gdn_dtype t) { return t == GDN_BF16 ? 2 : 4; }

// Which optional workspace buffers a prefill of this mode and these options uses.
void set_buffers(Problem *pb, bool online, const gdn_options *opt) {
    pb->online = online;
    pb->need_cbar = pb->dtype == GDN_F32 || online || (opt && opt->w_deferred);
    pb->need_runs = pb->dtype == GDN_BF16 && opt && opt->scan_runs;
}

}  // namespace

size_t workspace_layout(const Problem &pb, void *base, Workspace *ws) {
    const int64_t R = pb.R, C = pb.C, G = pb.G;
    const size_t es = elem_size(pb.dtype);
    const int64_t ev_cap = R * C;            // every chunk of every pair may be an event
    const int64_t snap_cap = R * G;          // at most one predecessor per group
    size_t off = 0;
    auto take = [&](size_t bytes) { size_t o = off; off = align_up(off + bytes); return o; };
    const size_t o_counts = take(4 * sizeof(int32_t));
    const size_t o_row_pair = take(R * sizeof(int32_t));
    const size_t o_row_ptr = take((R + 1) * sizeof(int32_t));
    const size_t o_ev_chunk = take(ev_cap * sizeof(int32_t));
    const size_t o_grp_pred = take(R * G * sizeof(int32_t));
    const size_t o_snap_slot = take(ev_cap * sizeof(int32_t));
    const size_t o_run_first = take(R * ((C + kRunChunks - 1) / kRunChunks + 1) * sizeof(int32_t));
    const size_t o_P = take((size_t)pb.B * pb.Nv * (C + 1) * sizeof(double));
    const size_t o_grp_info = take((size_t)R * G * 16);
    const size_t o_U = take((size_t)pb.B * pb.T * pb.Nv * pb.dv * es);
    const size_t o_cbar = take(pb.need_cbar ? (size_t)pb.B * pb.Nv * C * pb.nblk * 256 * sizeof(float) : 0);
    const size_t o_W = take((size_t)ev_cap * 2 * kChunk * pb.d * es);
    const size_t o_snap = take((size_t)snap_cap * 2 * pb.d * pb.dv * es);
    const size_t o_sel_ws = take(pb.online ? selector_workspace_bytes(pb.B, (int)C) : 0);
    const size_t o_sel_score = take(pb.online ? (size_t)pb.B * pb.Nv * C * sizeof(float) : 0);
    const size_t o_sel_mask = take(pb.online ? (size_t)R * C : 0);
    const int64_t nr = pb.dtype == GDN_BF16 && pb.need_runs ? (C + kRunChunks - 1) / kRunChunks : 0;
    const size_t run_elems = (size_t)R * 2 * nr * kDim * kDim;
    const size_t o_amap = take(run_elems * 2);
    const size_t o_bmap = take(run_elems * sizeof(float));
    const size_t o_entry = take(run_elems * sizeof(float));
    if (ws) {
        char *b = (char *)base;
        ws->counts = (int32_t *)(b + o_counts);
        ws->row_pair = (int32_t *)(b + o_row_pair);
        ws->row_ptr = (int32_t *)(b + o_row_ptr);
        ws->ev_chunk = (int32_t *)(b + o_ev_chunk);
        ws->grp_pred = (int32_t *)(b + o_grp_pred);
        ws->snap_slot = (int32_t *)(b + o_snap_slot);
        ws->run_first = (int32_t *)(b + o_run_first);
        ws->P = (double *)(b + o_P);
        ws->grp_info = b + o_grp_info;
        ws->U = b + o_U;
        ws->cbar = (float *)(b + o_cbar);
        ws->W = b + o_W;
        ws->snap = b + o_snap;
        ws->sel_ws = b + o_sel_ws;
        ws->sel_score = (float *)(b + o_sel_score);
        ws->sel_mask = (uint8_t *)(b + o_sel_mask);
        ws->amap = b + o_amap;
        ws->bmap = (float *)(b + o_bmap);
        ws->entry = (float *)(b + o_entry);
        ws->ev_cap = ev_cap;
        ws->snap_cap = snap_cap;
    }
    return off;
}

namespace {

enum PrefillMode { kDense = 0, kSparse = 1, kOnline = 2 };

// ---- row classes on concurrent streams ----------------------------------------
// CSR rows are sorted by event count, longest first, so the scan's critical path is
// the first rows.  The bf16 prefill splits the rows into classes by CSR index (no
// event count leaves the device): class c = rows [bound_c, bound_c+1) with bounds
// from class_bounds (classes of 3/16, 4/16, 4/16 and 5/16 of the rows).  Each class
// runs its intra step (given mask), scan and output on its own stream, the longest
// class first and at the highest priority, so its scan starts once its own intra step
// is done while the other classes' intra steps, scans and outputs fill the GPU around it.  Streams and events are made once per
// device; a mutex keeps one prefill's fork / join sequence together on the host.
constexpr int kClasses = 4;
struct ClassStreams {
    bool tried = false, ok = false;
    cudaStream_t s[kClasses - 1];  // classes 0 .. 2 (the last class runs on the caller's stream)
    cudaEvent_t fork, prefix_done, join[kClasses - 1];
};
ClassStreams g_class_streams[64];
std::mutex g_class_mutex;

ClassStreams *class_streams() {  // under g_class_mutex; nullptr if they cannot be made
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    ClassStreams &cs = g_class_streams[dev];
    if (!cs.tried) {
        cs.tried = true;
        int least = 0, greatest = 0;
        cudaDeviceGetStreamPriorityRange(&least, &greatest);
        bool ok = cudaEventCreateWithFlags(&cs.fork, cudaEventDisableTiming) == cudaSuccess &&
                  cudaEventCreateWithFlags(&cs.prefix_done, cudaEventDisableTiming) == cudaSuccess;
        for (int c = 0; ok && c < kClasses - 1; ++c) {
            const int prio = greatest + c < least ? greatest + c : least;  // class 0 first
            ok = cudaStreamCreateWithPriority(&cs.s[c], cudaStreamNonBlocking, prio) == cudaSuccess &&
                 cudaEventCreateWithFlags(&cs.join[c], cudaEventDisableTiming) == cudaSuccess;
        }
        cs.ok = ok;
    }
    return cs.ok ? &cs : nullptr;
}

// Class bounds for R rows (sorted longest first): returns the number of non-empty classes.  Each
// class's intra step fills the GPU, so the classes' intra steps run one after another; classes of
// nearly equal size (3/16, 4/16, 4/16 and 5/16 of the rows) start the longest rows' scan after a
// short intra step and stagger the other classes' scans and outputs behind it.
int class_bounds(int R, int *bound) {
    const int cand[kClasses + 1] = {0, (3 * R + 15) / 16, (7 * R + 15) / 16, (11 * R + 15) / 16, R};
    int n = 0;
    bound[0] = 0;
    for (int c = 1; c <= kClasses; ++c)
        if (cand[c] > bound[n]) bound[++n] = cand[c];
    return n;
}

gdn_status check_options(const gdn_options *opt) {
    if (!opt) return GDN_OK;
    const int tw = opt->tail_window;
    if (tw != 0 && tw != 8 && tw != 16 && tw != 32 && tw != 64) return GDN_ERR_UNSUPPORTED;
    if (opt->w_deferred != 0 && opt->w_deferred != 1) return GDN_ERR_UNSUPPORTED;
    if (opt->scan_runs != 0 && opt->scan_runs != 1) return GDN_ERR_UNSUPPORTED;
    if (opt->scan_full != 0 && opt->scan_full != 1) return GDN_ERR_UNSUPPORTED;
    if (opt->states_expanded != 0 && opt->states_expanded != 1) return GDN_ERR_UNSUPPORTED;
    if (opt->online_split < 0 || opt->online_split > 2) return GDN_ERR_UNSUPPORTED;
    // the masked full scan and the expanded states are variants of the one-pass scan
    if ((opt->scan_full || opt->states_expanded) && opt->scan_runs) return GDN_ERR_UNSUPPORTED;
    // the masked full scan reads W of every chunk, built in the intra step from a mask known up front
    if (opt->scan_full && opt->w_deferred) return GDN_ERR_UNSUPPORTED;
    for (int i = 0; i < 2; ++i)
        if (opt->reserved[i] != 0) return GDN_ERR_UNSUPPORTED;
    return GDN_OK;
}

gdn_status run_prefill(const gdn_shape *shape, const void *q, const void *k, const void *v, const float *beta,
                       const float *g, const float *h0, const uint8_t *mask, const float *eta, PrefillMode mode,
                       gdn_solver solver, void *o, float *s_final, float *score, uint8_t *mask_out,
                       int32_t *tier_out, void *workspace, size_t workspace_bytes, void *stream,
                       const gdn_options *opt = nullptr, bool single_stream = false) {
    gdn_status st = check_shape(shape);
    if (st != GDN_OK) return st;
    if ((st = check_options(opt)) != GDN_OK) return st;
    if (solver != GDN_SOLVER_EXACT && solver != GDN_SOLVER_BLOCK_ADJ) return GDN_ERR_DTYPE;
    const int split = opt ? opt->online_split : 0;  // online selection in two calls (sharded head pairs)
    if (split && mode != kOnline) return GDN_ERR_UNSUPPORTED;
    // the tier table is for 16 pairs (a split call selects nothing itself)
    if (mode == kOnline && !split && shape->Nv != 32) return GDN_ERR_UNSUPPORTED;
    if (split == 1 && shape->B > 0 && shape->T > 0 && !score) return GDN_ERR_NULL;
    if (split == 2 && shape->B > 0 && shape->T > 0 && !mask) return GDN_ERR_NULL;
    if (opt && (opt->scan_full || opt->states_expanded) && shape->dtype != GDN_BF16) return GDN_ERR_UNSUPPORTED;
    if (opt && opt->scan_full && mode == kOnline) return GDN_ERR_UNSUPPORTED;
    const bool has_tokens = shape->B > 0 && shape->T > 0;
    if (shape->B > 0 && !s_final) return GDN_ERR_NULL;
    if (has_tokens && (!q || !k || !v || !beta || !g || !o || (mode == kSparse && !mask))) return GDN_ERR_NULL;
    if (shape->B > 0 && !workspace) return GDN_ERR_NULL;
    const void *ptrs[] = {q, k, v, beta, g, h0, o, s_final, score, eta, tier_out};
    for (const void *p : ptrs)
        if (p && !aligned16(p)) return GDN_ERR_ALIGN;
    if (workspace && ((uintptr_t)workspace % kAlign) != 0) return GDN_ERR_ALIGN;
    Problem pb;
    fill_problem(shape, solver, &pb);
    set_buffers(&pb, mode == kOnline, opt);
    if (opt && opt->tail_window) pb.tail = opt->tail_window;
    pb.scan_full = opt && opt->scan_full;
    pb.states_expanded = opt && opt->states_expanded;
    const bool w_deferred = opt && opt->w_deferred;
    if (shape->B == 0) return GDN_OK;
    const size_t need = workspace_layout(pb, nullptr, nullptr);
    if (workspace_bytes < need) return GDN_ERR_WORKSPACE;
    if (!device_ok()) return GDN_ERR_DEVICE;
    pb.q = q; pb.k = k; pb.v = v; pb.beta = beta; pb.g = g; pb.h0 = h0;
    pb.o = o; pb.s_final = s_final;
    pb.stream = (cudaStream_t)stream;
    Workspace ws;
    workspace_layout(pb, workspace, &ws);
    pb.score = score;
    if (mode == kOnline && split == 2) {
        pb.mask = mask;  // the rank's rows of a selection over all ranks' pairs
    } else if (mode == kOnline) {
        if (!pb.score) pb.score = ws.sel_score;
        if (!mask_out) mask_out = ws.sel_mask;
        pb.mask = mask_out;
    } else {
        pb.mask = mode == kSparse ? mask : nullptr;
    }

    gdn_events ev;
    ev.row_pair = ws.row_pair; ev.row_ptr = ws.row_ptr; ev.ev_chunk = ws.ev_chunk;
    ev.grp_pred = ws.grp_pred; ev.snap_slot = ws.snap_slot; ev.counts = ws.counts;
    ev.capacity = (int32_t)ws.ev_cap;
    cudaEvent_t *prof = prof_slot();
    auto mark = [&](int i) { if (prof) cudaEventRecord(prof[i], pb.stream); };
    const bool tc = pb.dtype == GDN_BF16;   // tensor-core path for bf16 storage
    cudaError_t e = cudaSuccess;
    // Tensor-core path: every kernel after the prefill's first is a programmatic dependent of
    // the one before (it may start while that one drains).  Not while profiling: the stage
    // events between launches serialise them anyway.
    pb.pdl_ok = tc && !prof;
    bool launched = false;
    // kernels: how many kernels the stage's launcher issues (0 for an empty stage)
    const bool counting = g_prof.mode != 0;
    if (counting) ++g_prof.calls;
    auto stage = [&](int id, int kernels, auto &&launch) {
        mark(2 * id);
        pb.pdl = pb.pdl_ok && launched;
        if (e == cudaSuccess) e = launch();
        mark(2 * id + 1);
        if (kernels > 0) launched = true;
        if (counting) g_prof.launches += kernels;
    };
    auto none = [] { return cudaSuccess; };
    // the status word collects every kernel's bits (timeouts, capacity overflows) for this prefill
    // (a second online_split call adds its bits to the first one's)
    if (split != 2 && cudaMemsetAsync(ws.counts + 2, 0, sizeof(int32_t), pb.stream) != cudaSuccess)
        return GDN_ERR_CUDA;
    if (split == 1) {  // the intra step and its scores only
        stage(2, 1, [&] { return tc ? launch_intra_tc(pb, ws, true) : launch_intra(pb, ws); });
        return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
    }
    const bool runs = pb.need_runs != 0;
    // row classes on concurrent streams (bf16 one-pass scan; not while profiling, whose stage
    // events need one stream, nor for a caller that asked for a single stream)
    std::unique_lock<std::mutex> class_lock(g_class_mutex, std::defer_lock);
    ClassStreams *cs = nullptr;
    if (tc && !runs && !prof && !single_stream && pb.R > 1) {
        class_lock.lock();
        cs = class_streams();
        if (!cs) class_lock.unlock();
    }
    if (cs) {
        // the compaction and the prefix first (the classes need the CSR rows), then per class
        // [intra (given mask) ->] scan -> output
        const bool intra_split = mode != kOnline && !w_deferred;
        if (mode == kOnline) {
            if (!split) {
                stage(2, 1, [&] { return launch_intra_tc(pb, ws, true); });
                stage(8, 2, [&] { return launch_selector(pb, pb.score, eta, mask_out, tier_out, ws.sel_ws); });
            }
            stage(0, 1, [&] { return launch_select(pb, ev, ws.snap_cap, nullptr, !split, true); });
            stage(1, 1, [&] { return launch_prefix(pb, ws); });
            stage(3, 1, [&] { return launch_wbuild_tc(pb, ws); });
        } else {
            // with the intra steps per class, only the row order comes before the fork
            stage(0, 1, [&] { return launch_select(pb, ev, ws.snap_cap, nullptr, false, true, intra_split ? 1 : 0); });
            if (!intra_split) {
                stage(1, 1, [&] { return launch_prefix(pb, ws); });
                stage(2, 1, [&] { return launch_intra_tc(pb, ws, true); });
                stage(3, 1, [&] { return launch_wbuild_tc(pb, ws); });
            }
        }
        int bound[kClasses + 1];
        const int ncls = class_bounds(pb.R, bound);
        // the classes' intra steps need only the row order: they fork after the compaction's first
        // part, and its second part and the prefix (P and the group table, for the scans and
        // outputs) run beside them
        if (e == cudaSuccess) e = cudaEventRecord(cs->fork, pb.stream);
        if (intra_split) {  // the rest of the compaction and the prefix, beside the first intra steps
            stage(0, 1, [&] { return launch_select(pb, ev, ws.snap_cap, nullptr, false, true, 2); });
            stage(1, 1, [&] { return launch_prefix(pb, ws); });
            if (e == cudaSuccess) e = cudaEventRecord(cs->prefix_done, pb.stream);
        }
        for (int c = 0; c < ncls && e == cudaSuccess; ++c) {
            Problem q = pb;
            q.row_pair = ws.row_pair;
            q.row0 = bound[c];
            q.nrows = bound[c + 1] - bound[c];
            const bool last = c == ncls - 1;
            q.stream = last ? pb.stream : cs->s[c];
            if (!last) e = cudaStreamWaitEvent(q.stream, cs->fork, 0);
            // No programmatic dependent launch inside a class: a dependent's CTAs would sit on SMs
            // waiting for their predecessor (the output for the whole scan), which the other
            // classes' kernels need.  (The first kernel of a class also reads the CSR rows.)
            q.pdl = 0;
            if (e == cudaSuccess && intra_split) e = launch_intra_tc(q, ws, false);
            if (e == cudaSuccess && intra_split && !last) e = cudaStreamWaitEvent(q.stream, cs->prefix_done, 0);
            if (e == cudaSuccess) e = launch_scan_warp(q, ws);
            if (e == cudaSuccess) e = launch_output_tc(q, ws);
            if (counting) g_prof.launches += intra_split ? 3 : 2;
            if (e == cudaSuccess && !last) e = cudaEventRecord(cs->join[c], q.stream);
        }
        for (int c = 0; c + 1 < ncls && e == cudaSuccess; ++c) e = cudaStreamWaitEvent(pb.stream, cs->join[c], 0);
        return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
    }
    if (mode == kOnline) {
        // intra first (its Tail-16 scores drive the selection), then the rest of the pipeline
        // (a second online_split call starts after both, with the caller's mask)
        if (!split) {
            stage(2, 1, [&] { return tc ? launch_intra_tc(pb, ws, true) : launch_intra(pb, ws); });
            stage(8, 2, [&] { return launch_selector(pb, pb.score, eta, mask_out, tier_out, ws.sel_ws); });
        }
        stage(0, 1, [&] { return launch_select(pb, ev, ws.snap_cap, pb.need_runs ? ws.run_first : nullptr, !split, true); });
        stage(1, 1, [&] { return launch_prefix(pb, ws); });
        stage(3, 1, [&] { return tc ? launch_wbuild_tc(pb, ws) : launch_wbuild(pb, ws); });
    } else {
        // intra needs only the caller's mask (W goes to slot row * C + chunk), so it does not wait
        // for the compaction and the prefix: their few CTAs run beside intra's first waves, and
        // intra waits for them only before it exits
        stage(0, 1, [&] { return launch_select(pb, ev, ws.snap_cap, pb.need_runs ? ws.run_first : nullptr, false, true); });
        stage(1, 1, [&] { return launch_prefix(pb, ws); });
        stage(2, 1, [&] { return tc ? launch_intra_tc(pb, ws, w_deferred) : launch_intra(pb, ws); });
        // bf16: W is built inside intra for the event chunks, or after it from C-bar (w_deferred)
        stage(3, !tc || w_deferred ? 1 : 0,
              [&] { return !tc ? launch_wbuild(pb, ws) : (w_deferred ? launch_wbuild_tc(pb, ws) : none()); });
        stage(8, 0, none);
    }
    // bf16 storage: one pass over each CSR row, or run maps + chain + fix-up (scan_runs)
    stage(4, runs ? 1 : 0, [&] { return runs ? launch_scan_tc(pb, ws, 0) : none(); });
    stage(5, runs ? 1 : 0, [&] { return runs ? launch_scan_tc(pb, ws, 1) : none(); });
    stage(6, 1, [&] {
        return !tc ? launch_scan(pb, ws) : (runs ? launch_scan_tc(pb, ws, 2) : launch_scan_warp(pb, ws));
    });
    stage(7, 1, [&] { return tc ? launch_output_tc(pb, ws) : launch_output(pb, ws); });
    return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

gdn_status read_status(const int32_t *counts, void *stream) {
    if (!counts) return GDN_ERR_NULL;
    if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return GDN_ERR_CUDA;
    int32_t host[4] = {0, 0, 0, 0};
    if (cudaMemcpy(host, counts, sizeof(host), cudaMemcpyDeviceToHost) != cudaSuccess) return GDN_ERR_CUDA;
    if (host[2] & kStatusTimeout) return GDN_ERR_TIMEOUT;
    return host[2] ? GDN_ERR_CAPACITY : GDN_OK;
}

// Device staging of gdn_prefill_host: q, k, v, beta, g, h0, mask, o, s_final (each 256-byte aligned).
struct HostStaging {
    size_t q, k, v, beta, g, h0, mask, o, s, total;
};

HostStaging host_staging(const gdn_shape *sh) {
    const size_t es = elem_size(sh->dtype), BT = (size_t)sh->B * sh->T;
    const size_t qk = BT * sh->Nq * sh->d * es, vo = BT * sh->Nv * sh->dv * es, bg = BT * sh->Nv * sizeof(float);
    const size_t st = (size_t)sh->B * sh->Nv * sh->d * sh->dv * sizeof(float);
    const size_t mk = (size_t)sh->B * sh->Nq * ((sh->T + kChunk - 1) / kChunk);
    HostStaging h;
    size_t off = 0;
    auto take = [&](size_t bytes) { size_t o = off; off = align_up(off + bytes); return o; };
    h.q = take(qk); h.k = take(qk); h.v = take(vo); h.beta = take(bg); h.g = take(bg);
    h.h0 = take(st); h.mask = take(mk); h.o = take(vo); h.s = take(st);
    h.total = off;
    return h;
}

}  // namespace

// gdn_prefill_sparse on the caller's stream alone (no library-owned streams or events, which the
// allocation-free entry point must not create); same kernels, same results.
gdn_status prefill_sparse_single_stream(const gdn_shape *shape, const void *q, const void *k, const void *v,
                                        const float *beta, const float *g, const float *h0, const uint8_t *mask,
                                        gdn_solver solver, void *o, float *s_final, float *score, void *workspace,
                                        size_t workspace_bytes, void *stream) {
    return run_prefill(shape, q, k, v, beta, g, h0, mask, nullptr, kSparse, solver, o, s_final, score, nullptr,
                       nullptr, workspace, workspace_bytes, stream, nullptr, true);
}

}  // namespace gdn

using namespace gdn;

extern "C" {

size_t gdn_workspace_bytes(const gdn_shape *shape, gdn_solver solver, int sparse) {
    // dense and sparse share one layout (the dense path is the all-events case);
    // sparse == 2 (online selection) adds the selector's buffers
    return gdn_workspace_bytes_ex(shape, solver, sparse == 2 ? GDN_MODE_ONLINE : (gdn_mode)(sparse != 0), nullptr);
}

size_t gdn_workspace_bytes_ex(const gdn_shape *shape, gdn_solver solver, gdn_mode mode, const gdn_options *opt) {
    if (check_shape(shape) != GDN_OK || check_options(opt) != GDN_OK) return 0;
    if (solver != GDN_SOLVER_EXACT && solver != GDN_SOLVER_BLOCK_ADJ) return 0;
    if (mode != GDN_MODE_DENSE && mode != GDN_MODE_SPARSE && mode != GDN_MODE_ONLINE) return 0;
    Problem pb;
    fill_problem(shape, solver, &pb);
    set_buffers(&pb, mode == GDN_MODE_ONLINE, opt);
    return workspace_layout(pb, nullptr, nullptr);
}

namespace {
struct EventsLayout {
    size_t row_pair, row_ptr, ev_chunk, grp_pred, snap_slot, counts, total;
};
EventsLayout events_layout(const gdn_shape *s, int32_t capacity) {
    const int64_t R = (int64_t)s->B * s->Nq, C = ((int64_t)s->T + kChunk - 1) / kChunk, G = (C + 1) / 2;
    EventsLayout l;
    size_t off = 0;
    auto take = [&](size_t bytes) { size_t o = off; off = align_up(off + bytes); return o; };
    l.row_pair = take(R * 4); l.row_ptr = take((R + 1) * 4); l.ev_chunk = take((size_t)capacity * 4);
    l.grp_pred = take(R * G * 4); l.snap_slot = take((size_t)capacity * 4); l.counts = take(4 * 4);
    l.total = off;
    return l;
}
}  // namespace

size_t gdn_events_bytes(const gdn_shape *shape, int32_t capacity) {
    if (check_shape(shape) != GDN_OK || capacity < 0) return 0;
    return events_layout(shape, capacity).total;
}

gdn_status gdn_events_carve(const gdn_shape *shape, int32_t capacity, void *buffer, gdn_events *events) {
    gdn_status st = check_shape(shape);
    if (st != GDN_OK) return st;
    if (!buffer || !events) return GDN_ERR_NULL;
    if (capacity < 0) return GDN_ERR_SHAPE;
    if (((uintptr_t)buffer % kAlign) != 0) return GDN_ERR_ALIGN;
    const EventsLayout l = events_layout(shape, capacity);
    char *b = (char *)buffer;
    events->row_pair = (int32_t *)(b + l.row_pair);
    events->row_ptr = (int32_t *)(b + l.row_ptr);
    events->ev_chunk = (int32_t *)(b + l.ev_chunk);
    events->grp_pred = (int32_t *)(b + l.grp_pred);
    events->snap_slot = (int32_t *)(b + l.snap_slot);
    events->counts = (int32_t *)(b + l.counts);
    events->capacity = capacity;
    return GDN_OK;
}

gdn_status gdn_select_events(const gdn_shape *shape, const uint8_t *mask, gdn_events *events, void *stream) {
    gdn_status st = check_shape(shape);
    if (st != GDN_OK) return st;
    if (!events) return GDN_ERR_NULL;
    Problem pb;
    fill_problem(shape, GDN_SOLVER_BLOCK_ADJ, &pb);
    if (pb.R == 0) return GDN_OK;
    if (!events->row_pair || !events->row_ptr || !events->grp_pred || !events->counts) return GDN_ERR_NULL;
    if (pb.C > 0 && (!mask || !events->ev_chunk || !events->snap_slot)) return GDN_ERR_NULL;
    if (events->capacity < 0) return GDN_ERR_SHAPE;
    const void *ptrs[] = {mask, events->row_pair, events->row_ptr, events->ev_chunk, events->grp_pred,
                          events->snap_slot, events->counts};
    for (const void *p : ptrs)
        if (p && !aligned16(p)) return GDN_ERR_ALIGN;
    if (!device_ok()) return GDN_ERR_DEVICE;
    pb.mask = mask;
    pb.stream = (cudaStream_t)stream;
    // the snapshot numbering needs no capacity of its own: it never exceeds E
    const cudaError_t e = launch_select(pb, *events, (int64_t)events->capacity, nullptr, true, false);
    return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

gdn_status gdn_events_status(const gdn_events *events, void *stream) {
    if (!events) return GDN_ERR_NULL;
    return read_status(events->counts, stream);
}

gdn_status gdn_prefill_dense(const gdn_shape *shape, const void *q, const void *k, const void *v,
                             const float *beta, const float *g, const float *h0, gdn_solver solver, void *o,
                             float *s_final, float *score, void *workspace, size_t workspace_bytes, void *stream) {
    return run_prefill(shape, q, k, v, beta, g, h0, nullptr, nullptr, kDense, solver, o, s_final, score, nullptr,
                       nullptr, workspace, workspace_bytes, stream);
}

gdn_status gdn_prefill_sparse(const gdn_shape *shape, const void *q, const void *k, const void *v,
                              const float *beta, const float *g, const float *h0, const uint8_t *mask,
                              gdn_solver solver, void *o, float *s_final, float *score, void *workspace,
                              size_t workspace_bytes, void *stream) {
    return run_prefill(shape, q, k, v, beta, g, h0, mask, nullptr, kSparse, solver, o, s_final, score, nullptr,
                       nullptr, workspace, workspace_bytes, stream);
}

size_t gdn_prefill_host_workspace_bytes(const gdn_shape *shape, gdn_solver solver, int sparse) {
    const size_t w = gdn_workspace_bytes(shape, solver, sparse ? 1 : 0);
    return w ? w + host_staging(shape).total : 0;
}

gdn_status gdn_prefill_host(const gdn_shape *shape, const void *q, const void *k, const void *v, const float *beta,
                            const float *g, const float *h0, const uint8_t *mask, gdn_solver solver, void *o,
                            float *s_final, void *workspace, size_t workspace_bytes, void *stream) {
    gdn_status st = check_shape(shape);
    if (st != GDN_OK) return st;
    if (solver != GDN_SOLVER_EXACT && solver != GDN_SOLVER_BLOCK_ADJ) return GDN_ERR_DTYPE;
    if (shape->B == 0) return GDN_OK;
    const bool sparse = mask != nullptr;
    const size_t wbytes = gdn_workspace_bytes(shape, solver, sparse ? 1 : 0);
    const HostStaging hs = host_staging(shape);
    if (!workspace) return GDN_ERR_NULL;
    if (((uintptr_t)workspace % kAlign) != 0) return GDN_ERR_ALIGN;
    if (workspace_bytes < wbytes + hs.total) return GDN_ERR_WORKSPACE;
    const bool has_tokens = shape->T > 0;
    if (!s_final || (has_tokens && (!q || !k || !v || !beta || !g || !o))) return GDN_ERR_NULL;
    if (!device_ok()) return GDN_ERR_DEVICE;
    char *stg = (char *)workspace + wbytes;
    const cudaStream_t cs = (cudaStream_t)stream;
    const size_t es = elem_size(shape->dtype), BT = (size_t)shape->B * shape->T;
    const size_t qk = BT * shape->Nq * shape->d * es, vo = BT * shape->Nv * shape->dv * es;
    const size_t bg = BT * shape->Nv * sizeof(float);
    const size_t stb = (size_t)shape->B * shape->Nv * shape->d * shape->dv * sizeof(float);
    const size_t mk = (size_t)shape->B * shape->Nq * ((shape->T + kChunk - 1) / kChunk);
    cudaError_t e = cudaSuccess;
    auto h2d = [&](size_t off, const void *src, size_t n) {
        if (e == cudaSuccess && n) e = cudaMemcpyAsync(stg + off, src, n, cudaMemcpyHostToDevice, cs);
    };
    if (has_tokens) {
        h2d(hs.q, q, qk); h2d(hs.k, k, qk); h2d(hs.v, v, vo); h2d(hs.beta, beta, bg); h2d(hs.g, g, bg);
        if (sparse) h2d(hs.mask, mask, mk);
    }
    if (h0) h2d(hs.h0, h0, stb);
    if (e != cudaSuccess) return GDN_ERR_CUDA;
    st = run_prefill(shape, stg + hs.q, stg + hs.k, stg + hs.v, (const float *)(stg + hs.beta),
                     (const float *)(stg + hs.g), h0 ? (const float *)(stg + hs.h0) : nullptr,
                     sparse ? (const uint8_t *)(stg + hs.mask) : nullptr, nullptr, sparse ? kSparse : kDense,
                     solver, stg + hs.o, (float *)(stg + hs.s), nullptr, nullptr, nullptr, workspace, wbytes, stream);
    if (st != GDN_OK) return st;
    if (has_tokens) e = cudaMemcpyAsync(o, stg + hs.o, vo, cudaMemcpyDeviceToHost, cs);
    if (e == cudaSuccess) e = cudaMemcpyAsync(s_final, stg + hs.s, stb, cudaMemcpyDeviceToHost, cs);
    return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

gdn_status gdn_decode_step(const gdn_shape *shape, const void *q, const void *k, const void *v, const float *beta,
                           const float *a, float *state, void *o, void *stream) {
    if (!shape) return GDN_ERR_NULL;
    if (shape->dtype != GDN_BF16 && shape->dtype != GDN_F32) return GDN_ERR_DTYPE;
    if (shape->B < 0 || shape->T != 1 || shape->Nq <= 0 || shape->Nv != 2 * shape->Nq) return GDN_ERR_SHAPE;
    if (shape->d != kDim || shape->dv != kDim) return GDN_ERR_UNSUPPORTED;
    if ((int64_t)shape->B * shape->Nv >= (int64_t)1 << 31) return GDN_ERR_SHAPE;
    if (shape->B == 0) return GDN_OK;
    if (!q || !k || !v || !beta || !a || !state || !o) return GDN_ERR_NULL;
    const void *ptrs[] = {q, k, v, beta, a, state, o};
    for (const void *p : ptrs)
        if (!aligned16(p)) return GDN_ERR_ALIGN;
    if (!device_ok()) return GDN_ERR_DEVICE;
    return launch_decode(*shape, q, k, v, beta, a, state, o, (cudaStream_t)stream) == cudaSuccess ? GDN_OK
                                                                                                  : GDN_ERR_CUDA;
}

gdn_status gdn_prefill_ex(const gdn_shape *shape, gdn_mode mode, const void *q, const void *k, const void *v,
                          const float *beta, const float *g, const float *h0, const uint8_t *mask, const float *eta,
                          gdn_solver solver, const gdn_options *opt, void *o, float *s_final, float *score,
                          uint8_t *mask_out, int32_t *tier_out, void *workspace, size_t workspace_bytes,
                          void *stream) {
    if (mode != GDN_MODE_DENSE && mode != GDN_MODE_SPARSE && mode != GDN_MODE_ONLINE) return GDN_ERR_UNSUPPORTED;
    if (mode == GDN_MODE_SPARSE && shape && shape->B > 0 && shape->T > 0 && !mask) return GDN_ERR_NULL;
    const PrefillMode m = mode == GDN_MODE_DENSE ? kDense : (mode == GDN_MODE_SPARSE ? kSparse : kOnline);
    const bool takes_mask = m == kSparse || (m == kOnline && opt && opt->online_split == 2);
    return run_prefill(shape, q, k, v, beta, g, h0, takes_mask ? mask : nullptr, eta, m, solver, o, s_final, score,
                       mask_out, tier_out, workspace, workspace_bytes, stream, opt);
}

gdn_status gdn_prefill_sparse_online(const gdn_shape *shape, const void *q, const void *k, const void *v,
                                     const float *beta, const float *g, const float *h0, const float *eta,
                                     gdn_solver solver, void *o, float *s_final, float *score, uint8_t *mask_out,
                                     int32_t *tier_out, void *workspace, size_t workspace_bytes, void *stream) {
    return run_prefill(shape, q, k, v, beta, g, h0, nullptr, eta, kOnline, solver, o, s_final, score, mask_out,
                       tier_out, workspace, workspace_bytes, stream);
}

namespace {
// The online selection on its own: gates either per token (g) or per chunk (gamma).
gdn_status select_scored(const gdn_shape *shape, const float *score, const float *g, const float *gamma,
                         const float *eta, uint8_t *mask_out, int32_t *tier_out, void *workspace,
                         size_t workspace_bytes, void *stream) {
    gdn_status st = check_shape(shape);
    if (st != GDN_OK) return st;
    if (shape->Nv != 32) return GDN_ERR_UNSUPPORTED;
    Problem pb;
    fill_problem(shape, GDN_SOLVER_BLOCK_ADJ, &pb);
    if (pb.B == 0 || pb.C == 0) return GDN_OK;
    if (!score || !(g || gamma) || !mask_out || !workspace) return GDN_ERR_NULL;
    const void *ptrs[] = {score, g, gamma, eta, tier_out};
    for (const void *p : ptrs)
        if (p && !aligned16(p)) return GDN_ERR_ALIGN;
    if (((uintptr_t)workspace % kAlign) != 0) return GDN_ERR_ALIGN;
    if (workspace_bytes < gdn_select_scored_workspace_bytes(shape)) return GDN_ERR_WORKSPACE;
    if (!device_ok()) return GDN_ERR_DEVICE;
    pb.g = g;
    pb.stream = (cudaStream_t)stream;
    const cudaError_t e = launch_selector(pb, score, eta, mask_out, tier_out, workspace, gamma);
    return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}
}  // namespace

gdn_status gdn_select_events_scored(const gdn_shape *shape, const float *score, const float *g, const float *eta,
                                    uint8_t *mask_out, int32_t *tier_out, void *workspace, size_t workspace_bytes,
                                    void *stream) {
    if (!g && shape && shape->B > 0 && shape->T > 0) return GDN_ERR_NULL;
    return select_scored(shape, score, g, nullptr, eta, mask_out, tier_out, workspace, workspace_bytes, stream);
}

gdn_status gdn_select_events_gamma(const gdn_shape *shape, const float *score, const float *gamma, const float *eta,
                                   uint8_t *mask_out, int32_t *tier_out, void *workspace, size_t workspace_bytes,
                                   void *stream) {
    if (!gamma && shape && shape->B > 0 && shape->T > 0) return GDN_ERR_NULL;
    return select_scored(shape, score, nullptr, gamma, eta, mask_out, tier_out, workspace, workspace_bytes, stream);
}

size_t gdn_select_scored_workspace_bytes(const gdn_shape *shape) {
    if (check_shape(shape) != GDN_OK || shape->Nv != 32) return 0;
    return align_up(selector_workspace_bytes(shape->B, (int)((shape->T + kChunk - 1) / kChunk)) + 1);
}

gdn_status gdn_workspace_status(const void *workspace, void *stream) {
    if (!workspace) return GDN_ERR_NULL;
    // counts live at offset 0 of the workspace
    return read_status((const int32_t *)workspace, stream);
}

const char *gdn_status_string(gdn_status status) {
    switch (status) {
        case GDN_OK: return "ok";
        case GDN_ERR_NULL: return "a required pointer is NULL";
        case GDN_ERR_SHAPE: return "unsupported or inconsistent sizes";
        case GDN_ERR_DTYPE: return "unknown dtype or solver";
        case GDN_ERR_ALIGN: return "pointer not 16-byte aligned (workspace: 256-byte)";
        case GDN_ERR_WORKSPACE: return "workspace smaller than gdn_workspace_bytes()";
        case GDN_ERR_UNSUPPORTED: return "request not implemented by this library (needs d == dv == 128, ceil(T/64) <= 16384)";
        case GDN_ERR_CUDA: return "CUDA runtime call or kernel launch failed";
        case GDN_ERR_DEVICE: return "current device is not a compute-capability 10.3 (GB300) GPU";
        case GDN_ERR_CAPACITY: return "device-side event or snapshot capacity exceeded";
        case GDN_ERR_TIMEOUT: return "a kernel gave up waiting after its time limit (device-latched)";
    }
    return "unknown status";
}

int32_t gdn_version(void) { return 100; }

gdn_status gdn_profile_enable(int enable) {
    if (enable < 0 || enable > 2) return GDN_ERR_UNSUPPORTED;
    if (enable == 1 && !g_prof.created) {
        if (!device_ok()) return GDN_ERR_DEVICE;
        for (int i = 0; i < kProfSlots; ++i)
            for (int j = 0; j < 2 * kStages; ++j)
                if (cudaEventCreate(&g_prof.ev[i][j]) != cudaSuccess) return GDN_ERR_CUDA;
        g_prof.created = true;
    }
    g_prof.mode = enable;
    g_prof.used = 0;
    g_prof.calls = 0;
    g_prof.launches = 0;
    return GDN_OK;
}

gdn_status gdn_profile_read(float *stage_ms, int32_t n_stages, int32_t *n_prefills, int64_t *n_launches) {
    if (!stage_ms || !n_prefills) return GDN_ERR_NULL;
    if (n_launches) *n_launches = g_prof.launches;
    if (n_stages < 0 || n_stages > kStages) return GDN_ERR_SHAPE;
    for (int j = 0; j < n_stages; ++j) stage_ms[j] = 0.f;
    const int recorded = g_prof.created ? g_prof.used : 0;
    *n_prefills = g_prof.mode == 2 ? (int32_t)g_prof.calls : recorded;
    for (int i = 0; i < recorded; ++i) {
        for (int j = 0; j < n_stages; ++j) {
            float ms = 0.f;
            if (cudaEventSynchronize(g_prof.ev[i][2 * j + 1]) != cudaSuccess) return GDN_ERR_CUDA;
            if (cudaEventElapsedTime(&ms, g_prof.ev[i][2 * j], g_prof.ev[i][2 * j + 1]) != cudaSuccess)
                return GDN_ERR_CUDA;
            stage_ms[j] += ms;
        }
    }
    g_prof.used = 0;
    g_prof.calls = 0;
    g_prof.launches = 0;
    return GDN_OK;
}

}  // extern "C"
