// k_scan_warp.cu -- the event-sparse state scan (SparseGDN Secs. 2.1, 2.6;
// Eqs. 1-2, 17-21) as ONE pass over each CSR row, for bf16 storage.
//
// The recurrence is serial in the events of a row, but the columns of the state
// S [d x dv] evolve independently: column j only ever meets column j of U.  So a
// row's state is cut into slices of 16 columns, one CTA per slice, and the CTA's
// four warps (one per SM sub-partition) share each event's two products by
// splitting their N dimension.  Warp w keeps the fp32 state S^T[16 dv x 32 d]
// for d in [32 w, 32 w + 32) in registers (the accumulator fragments of m16n8k16
// warp MMAs) for the whole row.  Per event (chunk c; fgap = 2^(P_c - P_prev) the
// decay over the skipped chunks, Eq. 21):
//   U'^T[:, t in 16w..]  = U^T + fgap bf16(S^T) (-W)^T        (all d; A from the
//                          shared bf16 copy of S^T, B = the stored -W tile [t][d])
//   U' -> the U buffer in place; U''^T = U'^T 2^(gamma - g_t) -> shared (bf16)
//   S^T[:, d in 32w..]  <- 2^gamma fgap S^T + U''^T K         (all t; B = the K tile
//                          [t][d] transposed on load)
//   the new bf16 S^T quarter -> the shared copy, which is also the event's
//   snapshot when some output group reads it (Eqs. 20-21).
// Two CTA barriers per event hand U'' and S between the warps.  S_final =
// 2^(P_C - P_(e_last + 1)) S.  Every event is applied once, by one CTA, and the
// state never leaves the SM.
//
// Tiles.  W [64 t][128 d] and K [64 t][128 d] arrive by TMA with the 128-byte
// swizzle (two 64-column boxes each), the U slice [64 t][16 dv] unswizzled; a
// ring of stages is refilled stages - 1 events ahead and a stage is reused once
// all four warps have arrived on its "empty" barrier.  The shared bf16 S^T copy
// and U'' use the same swizzle, so their ldmatrix / stmatrix accesses are
// conflict-free.
#include "gdn_internal.cuh"
#include "tc.cuh"
#include "tmap.cuh"

namespace gdn {
namespace {

using namespace tc;

constexpr int kWarps = 4;
constexpr int kThreads = 32 * kWarps;
constexpr int kSlice = 16;                       // state columns (dv) per CTA: the M of one warp MMA
constexpr uint32_t kTile = 16384;                // W or K tile: two swizzled boxes [64 t][64 d]
constexpr uint32_t kUBox = kChunk * kSlice * 2;  // U slice [64 t][16 dv] bf16, 32-byte rows
constexpr uint32_t kStage = 2 * kTile + kUBox;
constexpr uint32_t kSBox = kSlice * 128;         // [16 rows][64 columns] bf16, 128-byte swizzle (2 KB)
constexpr uint32_t kUpBox = 16 * kSlice * 2;     // one warp's U' rows [16 t][16 dv] (512 B)

template <int STAGES>
struct Layout {
    static constexpr uint32_t sb = STAGES * kStage;  // bf16 S^T: two boxes [16 dv][64 d]
    static constexpr uint32_t upp = sb + 2 * kSBox;  // bf16 U''^T [16 dv][64 t]
    static constexpr uint32_t ust = upp + kSBox;     // U' staging: [warp][16 t][16 dv]
    static constexpr uint32_t smem = 1024 + ust + kWarps * kUpBox;
    static_assert(kStage % 1024 == 0 && sb % 1024 == 0 && upp % 1024 == 0, "swizzled tiles 1024-byte aligned");
    static_assert(smem <= 227 * 1024, "shared memory per CTA");
};

struct WarpScanParams {
    const int32_t *row_pair, *row_ptr, *ev_chunk, *snap_slot;
    const double *P;
    const float *g, *h0;
    __nv_bfloat16 *U;       // [B,Nv,T,128] (head-major): U, replaced by U' for events
    __nv_bfloat16 *snap;    // [snap_cap,2,128 dv,128 d] post-event states S^T
    float *s_final;
    int32_t *status;
    int P_, T_, Nv, C;
    int row0;               // first CSR row of this launch (blockIdx.z = row - row0)
    int64_t ev_cap, snap_cap;
    // execution variants (bit-identical results): the masked full scan walks every chunk
    // (mask [B,P,C], the products computed on every chunk and kept on the events only);
    // expanded entry states: the state after an event goes to the slot of every output group
    // it enters (physical row i, group r: slot i G + r) instead of its compact snapshot slot
    const uint8_t *mask;
    int expanded, G;
};

__device__ __forceinline__ uint8_t *align1024(uint8_t *p) {
    return reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void ldsm4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr)
                 : "memory");
}
__device__ __forceinline__ void ldsm4t(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr)
                 : "memory");
}
__device__ __forceinline__ void stsm4(uint32_t addr, uint32_t r0, uint32_t r1, uint32_t r2, uint32_t r3) {
    asm volatile("stmatrix.sync.aligned.m8n8.x4.shared.b16 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(r0), "r"(r1),
                 "r"(r2), "r"(r3)
                 : "memory");
}
__device__ __forceinline__ void stsm4t(uint32_t addr, uint32_t r0, uint32_t r1, uint32_t r2, uint32_t r3) {
    asm volatile("stmatrix.sync.aligned.m8n8.x4.trans.shared.b16 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(r0),
                 "r"(r1), "r"(r2), "r"(r3)
                 : "memory");
}
__device__ __forceinline__ float bf16lo(uint32_t x) { return __uint_as_float(x << 16); }
__device__ __forceinline__ float bf16hi(uint32_t x) { return __uint_as_float(x & 0xFFFF0000u); }
// CTA-wide named barrier over the four warps (id 0 is __syncthreads').
__device__ __forceinline__ void cta_bar(int id) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "n"(kThreads) : "memory");
}
// The same, returning whether any thread passed a non-zero flag.
__device__ __forceinline__ bool cta_bar_any(int id, int flag) {
    uint32_t r;
    asm volatile(
        "{\n"
        ".reg .pred p, q;\n"
        "setp.ne.u32 q, %1, 0;\n"
        "bar.red.or.pred p, %2, %3, q;\n"
        "selp.u32 %0, 1, 0, p;\n"
        "}\n"
        : "=r"(r)
        : "r"((uint32_t)flag), "r"(id), "n"(kThreads)
        : "memory");
    return r != 0;
}

// Address of the 16-byte chunk holding column k (k % 8 == 0) of row r in a tile of
// 128-byte swizzled boxes [rows][64 columns] placed box_bytes apart.
__device__ __forceinline__ uint32_t sw_addr(uint32_t base, uint32_t r, uint32_t k, uint32_t box_bytes) {
    return base + (k >> 6) * box_bytes + sw128_offset(r, k & 63);
}

// grid: (dv slices 8, 2 heads, CSR rows R); block: 4 consumer warps + 1 producer warp.
// FULL: the masked full scan (every chunk a step; see WarpScanParams).
template <int STAGES, bool FULL>
__global__ void __launch_bounds__(kThreads + 32, 1)
scan_warp_kernel(const __grid_constant__ CUtensorMap tW, const __grid_constant__ CUtensorMap tK,
                 const __grid_constant__ CUtensorMap tU, WarpScanParams a) {
    using L = Layout<STAGES>;
    extern __shared__ uint8_t smraw[];
    uint8_t *sm = align1024(smraw);
    __shared__ uint64_t full[STAGES], empty[STAGES];
    __shared__ int abort_s;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int gq = lane >> 2, cq = lane & 3;           // fragment row group, column pair
    const uint32_t lrow = lane & 7, lmat = lane >> 3;  // ldmatrix / stmatrix: row in matrix, matrix id
    const int hh = blockIdx.y, j = a.row0 + (int)blockIdx.z;
    const int dv0 = blockIdx.x * kSlice;               // the CTA's first state column
    const int t0w = 16 * warp, d0w = 32 * warp;        // this warp's tokens (MMA1) and d columns (MMA2)
    pdl_trigger();
    if (tid == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kWarps);
        }
        fence_mbar_init();
        abort_s = 0;
    }
    pdl_wait();  // CSR lists, P, U and W come from the kernels before
    const int i = a.row_pair[j], b = i / a.P_, p = i % a.P_, h = 2 * p + hh;
    const int e_lo = (int)min((int64_t)a.row_ptr[j], a.ev_cap);
    const int e_hi = (int)min((int64_t)a.row_ptr[j + 1], a.ev_cap);
    const int n_ev = max(0, e_hi - e_lo);
    const double *Pu = a.P + ((int64_t)b * a.Nv + h) * (a.C + 1);
    const int64_t gbase = (int64_t)b * a.T_;
    const uint32_t sb = smem_addr(sm + L::sb), upp = smem_addr(sm + L::upp);
    const int n_steps = FULL ? a.C : n_ev;  // the masked full scan visits every chunk
    const uint8_t *mrow = FULL ? a.mask + (int64_t)i * a.C : nullptr;

    if (warp == kWarps) {  // ---- producer: the tiles of step k (event k / chunk k) into stage k % STAGES ----
        __syncthreads();
        int kk = 0;
        for (; kk < n_steps; ++kk) {
            const int s = kk % STAGES;
            if (kk >= STAGES && !mbar_wait(&empty[s], ((kk / STAGES) - 1) & 1)) {
                if (lane == 0) {
                    abort_s = 1;
                    atomicOr(a.status, kStatusTimeout);
                }
                break;
            }
            if (*(volatile int *)&abort_s) break;
            if (lane == 0) {
                const int c = FULL ? kk : a.ev_chunk[e_lo + kk];
                uint8_t *st = sm + s * kStage;
                const int wrow = (int)((((int64_t)i * a.C + c) * 2 + hh) * kChunk);  // W of (row i, chunk c): slot i C + c
                mbar_arrive_expect_tx(&full[s], kStage);
                tma_load_3d(st, &tW, 0, wrow, 0, &full[s]);
                tma_load_3d(st + 8192, &tW, 64, wrow, 0, &full[s]);
                tma_load_4d(st + kTile, &tK, 0, p, c * kChunk, b, &full[s]);  // past the sequence's end: zeros
                tma_load_4d(st + kTile + 8192, &tK, 64, p, c * kChunk, b, &full[s]);
                tma_load_4d(st + 2 * kTile, &tU, dv0, c * kChunk, h, b, &full[s]);
            }
            __syncwarp();
        }
        // every requested tile has landed before the CTA may exit (the latest phase of each stage)
        if (lane == 0)
            for (int q = max(0, kk - STAGES); q < kk; ++q) mbar_wait(&full[q % STAGES], (q / STAGES) & 1);
        return;
    }

    uint8_t *ust_w = sm + L::ust + warp * kUpBox;
    // this warp's state quarter: n-tile nd holds d = d0w + 8 nd .. + 7; fragment (row gq / gq + 8, cols 2 cq, +1)
    float S[4][4];
    if (a.h0) {
        const float *h0p = a.h0 + ((int64_t)b * a.Nv + h) * (kDim * kDim);  // h0[d][dv]
#pragma unroll
        for (int nd = 0; nd < 4; ++nd) {
            const int d = d0w + 8 * nd + 2 * cq;
            S[nd][0] = h0p[d * kDim + dv0 + gq];
            S[nd][1] = h0p[(d + 1) * kDim + dv0 + gq];
            S[nd][2] = h0p[d * kDim + dv0 + gq + 8];
            S[nd][3] = h0p[(d + 1) * kDim + dv0 + gq + 8];
        }
    } else {
#pragma unroll
        for (int nd = 0; nd < 4; ++nd) S[nd][0] = S[nd][1] = S[nd][2] = S[nd][3] = 0.f;
    }
    // the bf16 copy of S^T (rows dv, columns d): this warp's 32 columns, two x4 stmatrix
    auto publish_state = [&]() {
        const uint32_t sbb = sb;
#pragma unroll
        for (int np = 0; np < 4; np += 2) {
            // matrices: (rows 0-7, n-tile np), (rows 8-15, np), (rows 0-7, np+1), (rows 8-15, np+1)
            const uint32_t r = 8 * (lmat & 1) + lrow, col = d0w + 8 * (np + (lmat >> 1));
            stsm4(sw_addr(sbb, r, col, kSBox), pack_bf16x2(S[np][0], S[np][1]), pack_bf16x2(S[np][2], S[np][3]),
                  pack_bf16x2(S[np + 1][0], S[np + 1][1]), pack_bf16x2(S[np + 1][2], S[np + 1][3]));
        }
    };
    publish_state();

    // Event metadata in batches of 32, lane l holding event kb + l: chunk, snapshot slot, the
    // log2 gap decay before the chunk (P_c - P_(previous event's chunk + 1), Eq. 21) and P at the
    // chunk's end.  The next batch is in flight while this one is used.
    int cb = 0, slb = -1, cn = 0, sln = -1;
    double pe_b = 0.0, pe_n = 0.0;  // P at the end of the chunk
    float lg_b = 0.f, lg_n = 0.f;   // log2 gap decay
    double pe_prev = Pu[0];         // the end of the event before the batch (start: P_0)
    auto load_batch = [&](int kb, int &cc, int &sl, double &pe, float &lg, double &prev) {
        const int kk = kb + lane;
        const bool in = kk < n_ev;
        cc = in ? a.ev_chunk[e_lo + kk] : 0;
        sl = in ? a.snap_slot[e_lo + kk] : -1;
        const double ps = in ? Pu[cc] : 0.0;
        pe = in ? Pu[cc + 1] : 0.0;
        double before = __shfl_up_sync(0xffffffffu, pe, 1);
        if (lane == 0) before = prev;
        lg = (float)(ps - before);
        prev = __shfl_sync(0xffffffffu, pe, 31);
    };
    load_batch(0, cb, slb, pe_b, lg_b, pe_prev);
    if (n_ev > 32) load_batch(32, cn, sln, pe_n, lg_n, pe_prev);
    double P_end = Pu[0];  // P at the end of the last applied event's chunk (start: chunk 0)

    // per-event scalars of event k, computed one event ahead: chunk, slot, decays
    // the gates of a chunk (lane l: tokens l and l + 32): gA/gB for the scalars being computed,
    // gnA/gnB in flight for the event after that
    float gA = 0.f, gB = 0.f, gnA = 0.f, gnB = 0.f;
    auto load_g = [&](int c, float &x, float &y) {
        const int n = min(kChunk, a.T_ - c * kChunk);
        const int64_t tk = gbase + (int64_t)c * kChunk;
        x = a.g[(tk + min(lane, n - 1)) * a.Nv + h];
        y = a.g[(tk + min(lane + 32, n - 1)) * a.Nv + h];
    };
    // chunk of event kq (kq < n_ev, in batch cb or the next one, cn)
    auto chunk_of = [&](int kq, int kcur) {
        const int v0 = __shfl_sync(0xffffffffu, cb, kq & 31), v1 = __shfl_sync(0xffffffffu, cn, kq & 31);
        return (kq >> 5) == (kcur >> 5) ? v0 : v1;
    };
    int c_k = 0, slot_k = -1;
    float fgap = 1.f, fsta = 1.f, dec[2][2];
    double pe_k = 0.0;
    auto scalars = [&](int kq) {  // kq < n_ev; its batch is cb (same 32-block as kq) or cn
        const int src = kq & 31;
        c_k = __shfl_sync(0xffffffffu, cb, src);
        slot_k = __shfl_sync(0xffffffffu, slb, src);
        pe_k = __shfl_sync(0xffffffffu, pe_b, src);
        const float lgap = __shfl_sync(0xffffffffu, lg_b, src);
        const int n = min(kChunk, a.T_ - c_k * kChunk);
        const float gl_a = __shfl_sync(0xffffffffu, gA, (n - 1) & 31);
        const float gl_b = __shfl_sync(0xffffffffu, gB, (n - 1) & 31);
        const float gam = n - 1 < 32 ? gl_a : gl_b;
        fgap = ex2(lgap);
        fsta = ex2(gam + lgap);  // 2^gamma fgap: the state's decay through the chunk
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            const int t = t0w + 8 * nt + 2 * cq;
            const float x0 = __shfl_sync(0xffffffffu, warp < 2 ? gA : gB, t & 31);
            const float x1 = __shfl_sync(0xffffffffu, warp < 2 ? gA : gB, (t + 1) & 31);
            dec[nt][0] = ex2(gam - x0);
            dec[nt][1] = ex2(gam - x1);
        }
    };
    if (n_ev > 0) {
        load_g(__shfl_sync(0xffffffffu, cb, 0), gA, gB);
        scalars(0);
        if (n_ev > 1) load_g(chunk_of(1, 0), gnA, gnB);
    }
    __syncthreads();  // barriers initialised, the bf16 state published

    int k = 0;       // events applied
    int zb = 0;      // masked full scan: lane l holds the mask bit of chunk 32 (st / 32) + l
    int st = 0;      // steps (events, or chunks for the masked full scan)
    for (; st < n_steps; ++st) {
        const int s = st % STAGES;
        bool is_ev = true;
        if (FULL) {
            if ((st & 31) == 0) zb = st + lane < a.C ? mrow[st + lane] != 0 : 0;
            is_ev = __shfl_sync(0xffffffffu, zb, st & 31) != 0;
        }
        const int c = FULL ? st : c_k, slot = slot_k;
        // a failed wait leaves garbage in this step's products (all accesses stay in shared
        // memory); the CTA then stops together at the next barrier
        const int bad = !mbar_wait(&full[s], (st / STAGES) & 1) || *(volatile int *)&abort_s;
        const uint32_t wbase = smem_addr(sm + s * kStage), kbase = wbase + kTile, ubase = wbase + 2 * kTile;

        // MMA1 on this warp's 16 tokens: Pm = bf16(S^T) (-W)^T over all d (two accumulator sets
        // over alternate k steps, so the dependent chains are half as long)
        const uint32_t sbk = sb;  // the state entering this event (bf16)
        float Pm[2][2][4] = {};
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
            uint32_t af[4];
            // A (16 dv x 16 d): matrices (rows 0-7, d lo), (rows 8-15, d lo), (rows 0-7, d hi), (rows 8-15, d hi)
            ldsm4(sw_addr(sbk, 8 * (lmat & 1) + lrow, 16 * ks + 8 * (lmat >> 1), kSBox), af[0], af[1], af[2], af[3]);
            // B (16 d x 16 t): matrices (t 0-7, d lo), (t 0-7, d hi), (t 8-15, d lo), (t 8-15, d hi)
            uint32_t b0, b1, b2, b3;
            ldsm4(sw_addr(wbase, t0w + 8 * (lmat >> 1) + lrow, 16 * ks + 8 * (lmat & 1), 8192), b0, b1, b2, b3);
            mma16816(Pm[ks & 1][0], af, b0, b1);
            mma16816(Pm[ks & 1][1], af, b2, b3);
        }
        // U'^T = U^T + fgap Pm on the warp's tokens (U^T fragments from the U box, transposed on load)
        float Up[2][4];
        {
            uint32_t r0, r1, r2, r3;
            // matrices: (t 0-7, dv 0-7), (t 0-7, dv 8-15), (t 8-15, dv 0-7), (t 8-15, dv 8-15)
            const uint32_t t = t0w + 8 * (lmat >> 1) + lrow;
            ldsm4t(ubase + t * 32 + (lmat & 1) * 16, r0, r1, r2, r3);
            const uint32_t ur[2][2] = {{r0, r1}, {r2, r3}};
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                Up[nt][0] = fmaf(fgap, Pm[0][nt][0] + Pm[1][nt][0], bf16lo(ur[nt][0]));
                Up[nt][1] = fmaf(fgap, Pm[0][nt][1] + Pm[1][nt][1], bf16hi(ur[nt][0]));
                Up[nt][2] = fmaf(fgap, Pm[0][nt][2] + Pm[1][nt][2], bf16lo(ur[nt][1]));
                Up[nt][3] = fmaf(fgap, Pm[0][nt][3] + Pm[1][nt][3], bf16hi(ur[nt][1]));
            }
        }
        // U''^T = U'^T 2^(gamma - g_t) on the warp's tokens -> the shared bf16 tile [16 dv][64 t]
        {
            const uint32_t r = 8 * (lmat & 1) + lrow, col = t0w + 8 * (lmat >> 1);
            stsm4(sw_addr(upp, r, col, kSBox), pack_bf16x2(Up[0][0] * dec[0][0], Up[0][1] * dec[0][1]),
                  pack_bf16x2(Up[0][2] * dec[0][0], Up[0][3] * dec[0][1]),
                  pack_bf16x2(Up[1][0] * dec[1][0], Up[1][1] * dec[1][1]),
                  pack_bf16x2(Up[1][2] * dec[1][0], Up[1][3] * dec[1][1]));
        }
        // U'' complete, every warp done reading the bf16 state; stop together on a failed wait
        if (cta_bar_any(1, bad)) {
            if (tid == 0) {
                abort_s = 1;
                atomicOr(a.status, kStatusTimeout);
            }
            break;
        }
        // MMA2 on this warp's 32 d columns: S^T <- fsta S^T + U''^T K over all tokens (the masked
        // full scan computes it on every chunk and keeps it on the events)
        float Sx[4][4];
#pragma unroll
        for (int nd = 0; nd < 4; ++nd)
#pragma unroll
            for (int q = 0; q < 4; ++q) Sx[nd][q] = S[nd][q] * fsta;
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
            uint32_t af[4];
            ldsm4(sw_addr(upp, 8 * (lmat & 1) + lrow, 16 * ks + 8 * (lmat >> 1), kSBox), af[0], af[1], af[2], af[3]);
#pragma unroll
            for (int np = 0; np < 4; np += 2) {
                // B (16 t x 16 d): matrices (t lo, n-tile np), (t hi, np), (t lo, np+1), (t hi, np+1)
                const uint32_t t = 16 * ks + 8 * (lmat & 1) + lrow, d = d0w + 8 * (np + (lmat >> 1));
                uint32_t b0, b1, b2, b3;
                ldsm4t(sw_addr(kbase, t, d, 8192), b0, b1, b2, b3);
                mma16816(Sx[np], af, b0, b1);
                mma16816(Sx[np + 1], af, b2, b3);
            }
        }
        if (!is_ev) {  // masked full scan, a chunk that is no event: the state only decays (Eq. 18,
            // applied at the next event through its gap factor); nothing is written
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
            cta_bar(2);  // every warp has read U'' before the next step rewrites it
            continue;
        }
#pragma unroll
        for (int nd = 0; nd < 4; ++nd)
#pragma unroll
            for (int q = 0; q < 4; ++q) S[nd][q] = Sx[nd][q];
        // U' out: this warp's 16 rows, bf16, through its staging: lane l writes half of row l / 2
        // (each 32-byte row segment of U is one whole sector)
        {
            const uint32_t t = 8 * (lmat >> 1) + lrow;
            stsm4t(smem_addr(ust_w) + t * 32 + (lmat & 1) * 16, pack_bf16x2(Up[0][0], Up[0][1]),
                   pack_bf16x2(Up[0][2], Up[0][3]), pack_bf16x2(Up[1][0], Up[1][1]), pack_bf16x2(Up[1][2], Up[1][3]));
            __syncwarp();
            const int tr = lane >> 1, tok = c * kChunk + t0w + tr;
            const uint4 v = *reinterpret_cast<const uint4 *>(ust_w + tr * 32 + (lane & 1) * 16);
            if (tok < a.T_)  // rows past the sequence's end are not written
                *reinterpret_cast<uint4 *>(a.U + (((int64_t)b * a.Nv + h) * a.T_ + tok) * kDim + dv0 + (lane & 1) * 8) = v;
            __syncwarp();
        }
        P_end = pe_k;
        // chunk of the next event (expanded entry states: the groups this event enters end there)
        const int c_next = k + 1 < n_ev ? chunk_of(k + 1, k) : 2 * a.G;
        // the next event's scalars while the products complete (its gates were loaded an event
        // ago); the gates of the event after it go in flight.  Past the row's end the values
        // are computed for a clamped event and never used.
        if (((k + 1) & 31) == 0) {  // next batch
            cb = cn; slb = sln; pe_b = pe_n; lg_b = lg_n;
            if (k + 33 < n_ev) load_batch(k + 33, cn, sln, pe_n, lg_n, pe_prev);
        }
        gA = gnA; gB = gnB;
        scalars(min(k + 1, n_ev - 1));
        load_g(chunk_of(min(k + 2, n_ev - 1), k + 1), gnA, gnB);
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);  // this warp is done with the stage
        publish_state();
        cta_bar(2);  // the new bf16 state is complete
        // snapshot S_(c+1): bf16 S^T rows dv0 .. dv0 + 15 (4 KB) into its compact slot, or
        // (expanded entry states) into the slot of every group r with c < 2r <= c_next
        auto put = [&](int64_t sl) {
            __nv_bfloat16 *dst = a.snap + (sl * 2 + hh) * (kDim * kDim) + dv0 * kDim;
#pragma unroll
            for (int q = 0; q < 2; ++q) {  // 16-byte chunk (row r, columns 8 j ..): a warp writes two whole rows
                const int idx = tid + q * kThreads, r = idx >> 4, jj = idx & 15;
                const uint4 v = *reinterpret_cast<const uint4 *>(sm + L::sb + (jj >> 3) * kSBox +
                                                                 sw128_offset(r, (jj & 7) * 8));
                *reinterpret_cast<uint4 *>(dst + r * kDim + jj * 8) = v;
            }
        };
        if (a.expanded) {
            const int r_hi = min(c_next / 2, a.G - 1);
            for (int r = c / 2 + 1; r <= r_hi; ++r) put((int64_t)i * a.G + r);
        } else if (slot >= 0 && slot < a.snap_cap) {
            put(slot);
        }
        ++k;
    }

    if (!*(volatile int *)&abort_s) {  // S_final = 2^(P_C - P_end) S, written as s_final[d][dv]
        const float f = ex2((float)(Pu[a.C] - P_end));
        float *sf = a.s_final + ((int64_t)b * a.Nv + h) * (kDim * kDim);
#pragma unroll
        for (int nd = 0; nd < 4; ++nd) {
            const int d = d0w + 8 * nd + 2 * cq;
            sf[d * kDim + dv0 + gq] = S[nd][0] * f;
            sf[(d + 1) * kDim + dv0 + gq] = S[nd][1] * f;
            sf[d * kDim + dv0 + gq + 8] = S[nd][2] * f;
            sf[(d + 1) * kDim + dv0 + gq + 8] = S[nd][3] * f;
        }
    }
}

template <int STAGES, bool FULL>
cudaError_t launch_stages(const Problem &pb, const CUtensorMap &tW, const CUtensorMap &tK, const CUtensorMap &tU,
                          const WarpScanParams &a) {
    constexpr uint32_t smem = Layout<STAGES>::smem;
    cudaFuncSetAttribute(scan_warp_kernel<STAGES, FULL>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    const int nrows = pb.nrows > 0 ? pb.nrows : pb.R;
    return launch_kernel(pb.pdl, scan_warp_kernel<STAGES, FULL>, dim3(kDim / kSlice, 2, nrows), kThreads + 32, smem,
                         pb.stream, tW, tK, tU, a);
}

template <int STAGES>
cudaError_t launch_mode(const Problem &pb, const CUtensorMap &tW, const CUtensorMap &tK, const CUtensorMap &tU,
                        const WarpScanParams &a) {
    return a.mask ? launch_stages<STAGES, true>(pb, tW, tK, tU, a) : launch_stages<STAGES, false>(pb, tW, tK, tU, a);
}

}  // namespace

cudaError_t launch_scan_warp(const Problem &pb, const Workspace &ws) {
    if (pb.R == 0) return cudaSuccess;
    CUtensorMap tW, tK, tU;
    const uint64_t wrows = (uint64_t)ws.ev_cap * 2 * kChunk;
    const int T = pb.T > 0 ? pb.T : 1;  // a map needs non-empty dimensions (no tile is read when T = 0)
    if (!make_tmap_bf16_3d(&tW, ws.W, kDim, wrows > 0 ? wrows : 1, 1, kDim * 2, (wrows > 0 ? wrows : 1) * kDim * 2,
                           64, 64, 1, true) ||
        !make_tmap_tokens(&tK, pb.k ? pb.k : ws.U, pb.Nq, T, pb.B, 64, 64, true) ||
        !make_tmap_headmajor(&tU, ws.U, pb.Nv, T, pb.B, kSlice, kChunk, false))
        return cudaErrorInvalidValue;
    WarpScanParams a;
    a.row_pair = ws.row_pair; a.row_ptr = ws.row_ptr; a.ev_chunk = ws.ev_chunk; a.snap_slot = ws.snap_slot;
    a.P = ws.P; a.g = pb.g; a.h0 = pb.h0; a.s_final = pb.s_final; a.status = ws.counts + 2;
    a.U = (__nv_bfloat16 *)ws.U; a.snap = (__nv_bfloat16 *)ws.snap;
    a.P_ = pb.P; a.T_ = pb.T; a.Nv = pb.Nv; a.C = pb.C;
    a.ev_cap = ws.ev_cap; a.snap_cap = ws.snap_cap;
    a.row0 = pb.nrows > 0 ? pb.row0 : 0;
    // the masked full scan needs the mask (the dense path's full scan is its CSR scan)
    a.mask = pb.scan_full && pb.mask ? pb.mask : nullptr;
    a.expanded = pb.states_expanded;
    a.G = pb.G;
    const int nrows = pb.nrows > 0 ? pb.nrows : pb.R;
    // The whole scan alone in up to two waves: a deep ring and the SM to itself (151 KB; a
    // latency-bound loop runs slower beside another kernel's CTAs).  A row class beside the
    // other classes' kernels: 111 KB, so an intra or output CTA fits beside it.  Many CTAs: a
    // shallow ring and two scan CTAs per SM (throughput).
    int sms = 148, dev = 0;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int64_t ctas = (int64_t)nrows * 2 * (kDim / kSlice);
    if (pb.nrows == 0 && ctas <= 2 * (int64_t)sms) return launch_mode<4>(pb, tW, tK, tU, a);
    if (ctas <= 2 * (int64_t)sms) return launch_mode<3>(pb, tW, tK, tU, a);
    return launch_mode<2>(pb, tW, tK, tU, a);
}

}  // namespace gdn
