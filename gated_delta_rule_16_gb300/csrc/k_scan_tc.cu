// k_scan_tc.cu -- the event-sparse state scan (SparseGDN Secs. 2.1, 2.6;
// Eqs. 1-2, 17-21) on tcgen05 tensor cores, for bf16 storage.
//
// Splitting the serial chain.  A CSR row (one head pair) can hold hundreds of
// events, and each event needs the state left by the previous one.  Every
// event, and every skipped chunk, maps the state affinely:
//     S -> 2^gamma S + K^T D (U - W S) = A_e S + B_e,    D = diag(2^(gamma - g)),
// so a run of 16 chunks maps its entry state S_r to A_r S_r + B_r.  Three
// launches replace the row-long chain:
//   1. scan_run_kernel, "map" mode, all runs in parallel: the run's events
//      applied to the identity with U = 0 give A_r (homogeneous part), applied
//      to 0 with the true U give B_r (inhomogeneous part);
//   2. scan_chain_kernel, per (row, head) and block of 32 state rows:
//      S_{r+1} = A_r S_r + B_r, one 128x128x128 MMA per run; writes every
//      run's entry state and S_final;
//   3. scan_run_kernel, "fix-up" mode, all runs in parallel: the run's events
//      from the true entry state, writing U' = U - W S in place of U and the
//      post-event snapshots that output groups read.
// The longest serial chain is then 16 events (plus one MMA per run), not a row.
//
// Layout.  Columns of S evolve independently, so the CTA works on S^T: TMEM
// lane / state row = a column of S (d_v index), 128 rows; 512 threads, thread
// (row, segment) handles 32 of the row's 128 entries.  The state lives in TMEM
// (fp32, 128 columns), which keeps the registers per thread low enough for two
// CTAs per SM: one CTA's barriers and MMA round trips overlap the other's work.
// Scaled state.  TMEM holds S^T / sigma, sigma a CTA-uniform factor that absorbs
// every decay of the run (sigma <- 2^(P_c - P_cur) 2^gamma sigma per event), so the
// state is never rewritten for a decay; the write of an event is divided by the new
// sigma instead.  When 1/sigma would pass 2^64 the event's decay is applied to TMEM
// and sigma restarts at 1.  Per event:
//   A1 = sigma 2^(P_c - P_cur) S_tmem^T, bf16 (the state entering chunk c)
//   MMA  U'^T[128 x 64]  = U^T . I                         (A: U [t][dv] MN-major; B: identity)
//   MMA1 U'^T          += A1[128 x 128] . (-W)^T           (B: -W [t][d] K-major, as stored)
//   U''^T = U'^T * 2^(gamma - g_t) / sigma_new, bf16        (registers)
//   MMA2 S_tmem^T      += U''^T[128 x 64] . K              (A: U''^T K-major; B: K [t][d] MN-major)
// The W, K and U tiles are single-buffered; W and U are refilled for the next event
// once MMA1 is done, K once MMA2 is done, so every load has most of an event to
// land (the fix-up's U tile once its U' store has read it).  The fix-up writes U'
// into the U tile and stores it over U by TMA.  Snapshots are stored in bf16 as
// S^T [dv][d] (each thread's 32 state entries are 64 contiguous bytes, written as
// two whole 32-byte sectors), the K-major operand of the output kernel's Q S product.
#include "gdn_internal.cuh"
#include "tc.cuh"
#include "tmap.cuh"

namespace gdn {
namespace {

using namespace tc;

constexpr int kThreads = 512;  // 16 warps: 4 per TMEM lane quarter, 32 state columns each
constexpr int kRun = kRunChunks;
constexpr uint32_t kSlab = 16384;        // [128 rows][128 B]
constexpr uint32_t OFF_A1 = 0;           // S^T bf16, K-major, 2 slabs
constexpr uint32_t OFF_A2 = 2 * kSlab;   // U''^T bf16, K-major, 1 slab
constexpr uint32_t OFF_W = 3 * kSlab;    // W [64 t][128 d]: 2 K-slabs of [64][128 B], 8192 apart
constexpr uint32_t OFF_K = 4 * kSlab;    // K MN-major: 2 stacks of [64 t][64 d], 8192 apart
constexpr uint32_t OFF_U = 5 * kSlab;    // U MN-major: 2 stacks of [64 t][64 dv], 8192 apart
constexpr uint32_t OFF_I = 6 * kSlab;    // identity [64 t'][64 t] bf16, K-major (8 KB)
constexpr uint32_t kRunSmem = 1024 + 6 * kSlab + 8192;
// The run kernel keeps 1/sigma below 2^64 (sigma: the state's scale in TMEM).
constexpr float kMinLog2Scale = -64.f;
constexpr uint32_t TM_U = 0;             // TMEM columns [0, 64): U'^T accumulator
constexpr uint32_t TM_S = 128;           // TMEM columns [128, 256): the state S^T
constexpr uint32_t kBlockQuads = 32 * 4 * 32 * 4;  // one row block's 32 rows of a column-quad fp32 tile (16 KB)
constexpr int kChainBufs = 3;  // A_r / B_r buffers: runs are prefetched two steps ahead
constexpr uint32_t kChainSmem = 1024 + 2 * kSlab + kChainBufs * (2 * kSlab + kBlockQuads) + kBlockQuads;
constexpr int kMaxRuns = 1024;  // C <= 16384 chunks
// The chain of one (row, head) is split over kChainSplit CTAs, each owning kChainRows rows
// of S^T (the rows evolve independently); its MMAs keep M = 128 with the other rows zero.
constexpr int kChainSplit = 4;
constexpr int kChainRows = kDim / kChainSplit;
static_assert(kChainRows == 32, "the active rows are TMEM lanes 0..31: one warp per column segment");

enum { kModeHomog = 0, kModeInhom = 1, kModeFixup = 2 };

struct ScanParams {
    const int32_t *row_pair, *row_ptr, *ev_chunk, *snap_slot;
    const int32_t *run_first;   // [R, NR+1] first event of each run, per CSR row
    const double *P;
    const float *g, *h0;
    __nv_bfloat16 *U;       // [B,T,Nv,128]: U, replaced by U' for events (fix-up mode)
    __nv_bfloat16 *amap;    // [R,2,NR,128,128] A_r^T (row m' = column m' of A_r)
    float *bmap;            // [R,2,NR] tiles of B_r^T, column-quad layout (quad_index)
    float *entry;           // [R,2,NR] tiles of S_r^T entering each run, column-quad layout
    __nv_bfloat16 *snap;    // [snap_cap,2,128 dv,128 d] post-event states S^T (bf16)
    float *s_final;         // [B,Nv,128 d,128 dv]
    int32_t *status;
    int P_, T_, Nv, C, NR;
    int64_t ev_cap, snap_cap;
};

__device__ __forceinline__ uint8_t *align1024(uint8_t *p) {
    return reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

__device__ __forceinline__ void fail(const ScanParams &a, int *abort_flag) {
    *abort_flag = 1;
    atomicOr(a.status, kStatusTimeout);
}

// grid: (runs NR, map mode: 2 heads x {homog, inhom} | fix-up: 2 heads, CSR rows R)
__global__ void __launch_bounds__(kThreads, 2)
scan_run_kernel(const __grid_constant__ CUtensorMap tW, const __grid_constant__ CUtensorMap tK,
                const __grid_constant__ CUtensorMap tU, const __grid_constant__ CUtensorMap tA, ScanParams a,
                int fixup) {
    extern __shared__ uint8_t smraw[];
    uint8_t *sm = align1024(smraw);
    __shared__ uint64_t bar_w, bar_k, bar_u, bar_mma1, bar_mma2, bar_drain;
    __shared__ uint32_t tmem_base;
    __shared__ int abort_s, n_ev_s, e_first_s;
    __shared__ int ev_c[kRun], ev_slot[kRun];
    __shared__ double Pl[kRun + 1];
    __shared__ float dec[kRun][kChunk];  // 2^(gamma - g_t) of each event chunk
    __shared__ float gamk[kRun], dPk[kRun];  // gamma of each event chunk; log2 gap decay before it
    // scaled state: TMEM holds S / sigma with sigma a CTA-uniform factor (see the header)
    __shared__ float f_snap[kRun], f_op[kRun], f_ren[kRun], f_u[kRun], f_end;
    __shared__ int ren[kRun];

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quarter = warp & 3, seg = warp >> 2;  // TMEM lane quarter, 32-column segment
    const int row = quarter * 32 + lane;
    const int cs = 32 * seg, slab = seg >> 1, cin = 32 * (seg & 1);  // columns, slab, offset in slab
    const int rho = blockIdx.x, j = blockIdx.z;
    const int hh = fixup ? (int)blockIdx.y : (int)(blockIdx.y >> 1);
    const int mode = fixup ? kModeFixup : (int)(blockIdx.y & 1);
    const int c_lo = rho * kRun, c_hi = min(a.C, c_lo + kRun);
    pdl_wait();  // everything below reads what the kernels before wrote
    pdl_trigger();
    const int i = a.row_pair[j], b = i / a.P_, p = i % a.P_, h = 2 * p + hh;

    if (tid == 0) {
        const int64_t f = min((int64_t)a.run_first[(int64_t)j * (a.NR + 1) + rho], a.ev_cap);
        const int64_t l = min((int64_t)a.run_first[(int64_t)j * (a.NR + 1) + rho + 1], a.ev_cap);
        n_ev_s = (int)max((int64_t)0, l - f);
        e_first_s = (int)f;
        abort_s = 0;
    }
    __syncthreads();
    const int n_ev = n_ev_s;
    if (n_ev == 0) return;  // a run without events: the chain kernel applies its decay
    const int e_first = e_first_s;
    const int64_t ubase = (((int64_t)i * 2 + hh) * a.NR + rho) * (kDim * kDim);
    if (tid < n_ev) {
        ev_c[tid] = a.ev_chunk[e_first + tid];
        ev_slot[tid] = a.snap_slot[e_first + tid];
    }
    const double *Pu = a.P + ((int64_t)b * a.Nv + h) * (a.C + 1);
    if (tid <= c_hi - c_lo) Pl[tid] = Pu[c_lo + tid];
    float S0[32];  // the entering state (fix-up: the chain's entry table), loaded with the lists above
    if (mode == kModeFixup) {
        const float4 *src = reinterpret_cast<const float4 *>(a.entry + ubase) + 8 * seg * 128 + row;
#pragma unroll
        for (int v4 = 0; v4 < 8; ++v4) {
            const float4 x = src[v4 * 128];
            S0[4 * v4] = x.x; S0[4 * v4 + 1] = x.y; S0[4 * v4 + 2] = x.z; S0[4 * v4 + 3] = x.w;
        }
    } else {
#pragma unroll
        for (int jj = 0; jj < 32; ++jj) S0[jj] = mode == kModeHomog && cs + jj == row ? 1.f : 0.f;
    }
    if (tid == 0) {
        mbar_init(&bar_w, 1);
        mbar_init(&bar_k, 1);
        mbar_init(&bar_u, 1);
        mbar_init(&bar_mma1, 1);
        mbar_init(&bar_mma2, 1);
        mbar_init(&bar_drain, 1);
        fence_mbar_init();
    }
    if (warp == 0) tmem_alloc<256>(&tmem_base);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    for (int idx = tid; idx < n_ev * kChunk; idx += kThreads) {
        const int k = idx >> 6, t = idx & 63;
        const int64_t tk = (int64_t)b * a.T_ + (int64_t)ev_c[k] * kChunk;
        const int n = min(kChunk, a.T_ - ev_c[k] * kChunk);  // valid tokens (a partial last chunk has fewer)
        const float gam = a.g[(tk + n - 1) * a.Nv + h];       // gamma: g at the chunk's last token
        dec[k][t] = ex2(gam - a.g[(tk + min(t, n - 1)) * a.Nv + h]);
        if (t == 0) {
            gamk[k] = gam;
            dPk[k] = (float)(Pl[ev_c[k] - c_lo] - Pl[(k ? ev_c[k - 1] + 1 : c_lo) - c_lo]);
        }
    }
    {   // identity [64 t'][64 t], the K-major B operand that copies U^T into the U' accumulator
        const int irow = tid >> 3, ich = tid & 7;
        float v[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) v[q] = 8 * ich + q == irow ? 1.f : 0.f;
        st_sw128_8(sm + OFF_I, irow, 8 * ich, v);
    }
    const uint32_t tbase = tmem_base;
    const uint32_t t_s = tmem_addr(tbase, quarter * 32, TM_S + cs);
    uint8_t *A1 = sm + OFF_A1;
    uint8_t *A2 = sm + OFF_A2;
    const bool with_u = mode != kModeHomog;
    // loads of event k (thread 0), each once its buffer is free
    auto load_w = [&](int k) {  // W of (row i, chunk c) at slot i C + c
        const int wrow = (int)((((int64_t)i * a.C + ev_c[k]) * 2 + hh) * kChunk);
        mbar_arrive_expect_tx(&bar_w, 16384u);
        tma_load_3d(sm + OFF_W, &tW, 0, wrow, 0, &bar_w);
        tma_load_3d(sm + OFF_W + 8192, &tW, 64, wrow, 0, &bar_w);
    };
    auto load_u = [&](int k) {
        const int tok = ev_c[k] * kChunk;
        mbar_arrive_expect_tx(&bar_u, 16384u);
        tma_load_4d(sm + OFF_U, &tU, 0, tok, h, b, &bar_u);  // rows past the sequence's end read zeros
        tma_load_4d(sm + OFF_U + 8192, &tU, 64, tok, h, b, &bar_u);
    };
    auto load_k = [&](int k) {
        const int tok = ev_c[k] * kChunk;
        mbar_arrive_expect_tx(&bar_k, 16384u);
        tma_load_4d(sm + OFF_K, &tK, 0, p, tok, b, &bar_k);  // rows past the sequence's end read zeros
        tma_load_4d(sm + OFF_K + 8192, &tK, 64, p, tok, b, &bar_k);
    };
    // thread 0: events whose tiles were requested, and completed waits it observed (for the drain)
    int loads_w = 0, loads_u = 0, loads_k = 0, seen_w = 0, seen_k = 0, seen_u = 0;
    if (tid == 0) {
        load_w(0);
        load_k(0);
        loads_w = loads_k = 1;
        if (with_u) {
            load_u(0);
            loads_u = 1;
        }
    }
    tmem_st32(t_s, S0);  // the entering state: identity (A_r), zero (B_r) or the true entry (fix-up)
    tmem_st_wait();
    __syncthreads();  // dec[], gamk[], dPk[] complete
    if (warp == 0) {  // the scale sigma = 2^ls through the run: ls is a prefix sum of (dP_k + gamma_k)
        const float x = lane < n_ev ? dPk[lane] + gamk[lane] : 0.f;
        float incl = x;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
        }
        const bool low = __any_sync(0xffffffffu, lane < n_ev && incl < kMinLog2Scale);
        if (!low) {  // 1/sigma stays in range over the whole run
            const float excl = incl - x;
            if (lane < n_ev) {
                f_snap[lane] = ex2(excl);
                f_op[lane] = ex2(excl + dPk[lane]);
                ren[lane] = 0;
                f_ren[lane] = 1.f;
                f_u[lane] = ex2(-incl);
            }
            if (lane == n_ev - 1) {
                const int cl = ev_c[n_ev - 1] + 1;
                f_end = ex2(incl + (mode == kModeFixup ? 0.f : (float)(Pl[c_hi - c_lo] - Pl[cl - c_lo])));
            }
        } else if (lane == 0) {  // a renormalisation is due somewhere: the serial rule
            float ls = 0.f;
            for (int k = 0; k < n_ev; ++k) {
                f_snap[k] = ex2(ls);            // the state left by event k-1
                const float lop = ls + dPk[k];  // the state entering chunk c_k
                f_op[k] = ex2(lop);
                const float lnew = lop + gamk[k];
                ren[k] = lnew < kMinLog2Scale;  // keep 1/sigma in range: apply this decay to TMEM instead
                f_ren[k] = ex2(lnew);
                ls = ren[k] ? 0.f : lnew;
                f_u[k] = ex2(-ls);
            }
            const int cl = ev_c[n_ev - 1] + 1;
            f_end = ex2(ls + (mode == kModeFixup ? 0.f : (float)(Pl[c_hi - c_lo] - Pl[cl - c_lo])));
        }
    }
    __syncthreads();
    for (int idx = tid; idx < n_ev * kChunk; idx += kThreads) dec[idx >> 6][idx & 63] *= f_u[idx >> 6];
    __syncthreads();  // dec[k][t] = 2^(gamma - g_t) / sigma after event k
    auto snapshot = [&](int slot, const float (&S)[32], float f) {  // row `row` of f S^T, columns cs .. cs+31
        if (slot >= 0 && slot < a.snap_cap) {
            __nv_bfloat16 *sn = a.snap + ((int64_t)slot * 2 + hh) * (kDim * kDim) + row * kDim + cs;
#pragma unroll
            for (int q = 0; q < 2; ++q) {  // 32 bytes per lane and store: whole sectors (half-sector
                uint32_t w[8];             // 16-byte stores made this the fix-up's slowest part)
#pragma unroll
                for (int u = 0; u < 8; ++u) w[u] = pack_bf16x2(f * S[16 * q + 2 * u], f * S[16 * q + 2 * u + 1]);
                st_global_v8(sn + 16 * q, w);
            }
        }
    };

    const uint32_t id1 = idesc_bf16(128, 64, false, false);
    const uint32_t idu = idesc_bf16(128, 64, true, false);
    const uint32_t id2 = idesc_bf16(128, 128, false, true);
    for (int k = 0; k < n_ev; ++k) {
        const int c = ev_c[k];
        if (tid == 0 && k > 0) {  // K buffer free: MMA2 of the previous event completed
            load_k(k);
            loads_k = k + 1;
        }
        {   // the state entering chunk c, sigma 2^(P_c - P_cur) S_tmem, as the bf16 operand of MMA1
            float S[32];
            tmem_ld32(t_s, S);
            tmem_ld_wait();
            if (mode == kModeFixup && k > 0) snapshot(ev_slot[k - 1], S, f_snap[k]);
            const float fo = f_op[k];
#pragma unroll
            for (int k0 = 0; k0 < 32; k0 += 8) {
                float w[8];
#pragma unroll
                for (int q = 0; q < 8; ++q) w[q] = S[k0 + q] * fo;
                st_sw128_8(A1 + slab * kSlab, row, cin + k0, w);
            }
            if (ren[k]) {  // CTA-uniform
                const float fr = f_ren[k];
#pragma unroll
                for (int jj = 0; jj < 32; ++jj) S[jj] *= fr;
                tmem_st32(t_s, S);
                tmem_st_wait();
            }
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        if (abort_s) break;
        if (tid == 0) {  // U'^T = U^T I - S_c^T W^T (the workspace holds -W)
            const bool landed_w = mbar_wait(&bar_w, k & 1);
            const bool landed_u = landed_w && (!with_u || mbar_wait(&bar_u, k & 1));
            if (!landed_u) {
                fail(a, &abort_s);
            } else {
                seen_w = k + 1;
                if (with_u) seen_u = k + 1;
                tc_fence_after();
                if (with_u)
                    for (int ks = 0; ks < 4; ++ks)
                        mma_bf16(tbase + TM_U, mnmajor_desc(smem_addr(sm + OFF_U), ks, 8192),
                                 kmajor_desc(smem_addr(sm + OFF_I), ks, 8192), idu, ks > 0);
                for (int ks = 0; ks < 8; ++ks)
                    mma_bf16(tbase + TM_U, kmajor_desc(smem_addr(A1), ks, kSlab),
                             kmajor_desc(smem_addr(sm + OFF_W), ks, 8192), id1, with_u || ks > 0);
                mma_commit(&bar_mma1);
            }
        }
        if (!mbar_wait(&bar_mma1, k & 1)) fail(a, &abort_s);
        if (tid == 0 && k + 1 < n_ev && !abort_s) {  // the products just done have read W and U
            load_w(k + 1);
            loads_w = k + 2;
            if (mode == kModeInhom) {  // (the fix-up writes U' into the U tile first)
                load_u(k + 1);
                loads_u = k + 2;
            }
        }
        tc_fence_after();
        {
            float acc[16];
            tmem_ld16(tmem_addr(tbase, quarter * 32, TM_U + 16 * seg), acc);
            tmem_ld_wait();
            if (mode == kModeFixup) {  // U' over U in the tile (read by now), stored below
                uint8_t *ut = sm + OFF_U + (row >> 6) * 8192;
#pragma unroll
                for (int t = 0; t < 16; ++t)
                    *reinterpret_cast<__nv_bfloat16 *>(ut + sw128_offset(16 * seg + t, row & 63)) =
                        __float2bfloat16_rn(acc[t]);
            }
            float up[16];
#pragma unroll
            for (int t = 0; t < 16; ++t) up[t] = acc[t] * dec[k][16 * seg + t];
#pragma unroll
            for (int t0 = 0; t0 < 16; t0 += 8) st_sw128_8(A2, row, 16 * seg + t0, &up[t0]);
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        if (abort_s) break;
        if (tid == 0) {
            tc_fence_after();
            if (!mbar_wait(&bar_k, k & 1)) {
                fail(a, &abort_s);
            } else {
                seen_k = k + 1;
                for (int ks = 0; ks < 4; ++ks)
                    mma_bf16(tbase + TM_S, kmajor_desc(smem_addr(A2), ks, kSlab),
                             mnmajor_desc(smem_addr(sm + OFF_K), ks, 8192), id2, 1);
                mma_commit(&bar_mma2);
                if (mode == kModeFixup) {  // U' of this event back over U (clipped at the sequence's end)
                    tma_store_4d(&tU, 0, c * kChunk, h, b, sm + OFF_U);
                    tma_store_4d(&tU, 64, c * kChunk, h, b, sm + OFF_U + 8192);
                    bulk_commit();
                    if (k + 1 < n_ev) {
                        bulk_wait_read();  // the store has left the U tile
                        load_u(k + 1);
                        loads_u = k + 2;
                    }
                }
            }
        }
        if (!mbar_wait(&bar_mma2, k & 1)) fail(a, &abort_s);
        tc_fence_after();
    }
    __syncthreads();
    if (!abort_s) {
        float S[32];
        tmem_ld32(t_s, S);
        tmem_ld_wait();
        if (mode == kModeFixup) {
            snapshot(ev_slot[n_ev - 1], S, f_end);
        } else {
            const float fin = f_end;  // sigma and the decay of the run's chunks after its last event
#pragma unroll
            for (int jj = 0; jj < 32; ++jj) S[jj] *= fin;
            if (mode == kModeHomog) {
                // A_r^T rows staged as the chain's MN-major operand image, then one TMA store
#pragma unroll
                for (int k0 = 0; k0 < 32; k0 += 8) st_sw128_8(A1 + slab * kSlab, row, cin + k0, &S[k0]);
                fence_async_smem();
                __syncthreads();
                if (tid == 0) {
                    const int yrow = (int)((((int64_t)i * 2 + hh) * a.NR + rho) * kDim);
                    tma_store_3d(&tA, 0, yrow, 0, A1);
                    tma_store_3d(&tA, 64, yrow, 0, A1 + kSlab);
                    bulk_commit();
                }
            } else {
                float4 *dst = reinterpret_cast<float4 *>(a.bmap + ubase) + 8 * seg * 128 + row;
#pragma unroll
                for (int v4 = 0; v4 < 8; ++v4)
                    dst[v4 * 128] = make_float4(S[4 * v4], S[4 * v4 + 1], S[4 * v4 + 2], S[4 * v4 + 3]);
            }
        }
    }
    if (tid == 0) bulk_wait_read();  // the stores only need their shared-memory sources before exit
    if (abort_s && tid == 0) {
        // drain: tiles still in flight into shared memory (phases this thread has not seen
        // complete), then every MMA issued so far (a commit arrives after all of them)
        for (int kk = seen_w; kk < loads_w; ++kk) mbar_wait(&bar_w, kk & 1);
        for (int kk = seen_k; kk < loads_k; ++kk) mbar_wait(&bar_k, kk & 1);
        for (int kk = seen_u; kk < loads_u; ++kk) mbar_wait(&bar_u, kk & 1);
        mma_commit(&bar_drain);
        mbar_wait(&bar_drain, 0);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc<256>(tbase);
}

// grid: (2 heads x kChainSplit row blocks, CSR rows R).  S_{r+1}^T = S_r^T A_r^T + B_r^T over the runs.
__global__ void __launch_bounds__(kThreads, 1)
scan_chain_kernel(const __grid_constant__ CUtensorMap tA, const __grid_constant__ CUtensorMap tB,
                  const __grid_constant__ CUtensorMap tE, ScanParams a) {
    extern __shared__ uint8_t smraw[];
    uint8_t *sm = align1024(smraw);
    __shared__ uint64_t bar_tma[kChainBufs], bar_mma;
    __shared__ uint32_t tmem_base;
    __shared__ int abort_s;
    __shared__ int nxt[kMaxRuns + 1];  // nxt[r]: first run >= r holding events of this row (NR if none)
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quarter = warp & 3, seg = warp >> 2;
    const int row = quarter * 32 + lane;
    const int cs = 32 * seg, slab = seg >> 1, cin = 32 * (seg & 1);
    const int hh = blockIdx.x / kChainSplit, part = blockIdx.x % kChainSplit, j = blockIdx.y;
    const bool active = row < kChainRows;         // warp-uniform: TMEM lanes 0 .. 31
    const int dv = part * kChainRows + row;       // this thread's row of S^T
    pdl_wait();  // the run maps of the kernel before
    pdl_trigger();
    const int i = a.row_pair[j], b = i / a.P_, p = i % a.P_, h = 2 * p + hh;
    const double *Pu = a.P + ((int64_t)b * a.Nv + h) * (a.C + 1);
    const int64_t sbase = ((int64_t)b * a.Nv + h) * (kDim * kDim);
    const int64_t rbase = ((int64_t)i * 2 + hh) * a.NR;

    if (tid == 0) {
        for (int q = 0; q < kChainBufs; ++q) mbar_init(&bar_tma[q], 1);
        mbar_init(&bar_mma, 1);
        fence_mbar_init();
        abort_s = 0;
    }
    if (warp == 0) tmem_alloc<128>(&tmem_base);
    {   // which runs hold events: from the per-run first-event table
        const int32_t *rf = a.run_first + (int64_t)j * (a.NR + 1);
        for (int r = tid; r < a.NR; r += kThreads) nxt[r] = rf[r + 1] > rf[r] ? r : a.NR;
        if (tid == 0) nxt[a.NR] = a.NR;
    }
    __syncthreads();
    if (warp == 0) {  // suffix minimum: nxt[r] = first run >= r with events
        int carry = a.NR;
        for (int base = ((a.NR + 31) / 32 - 1) * 32; base >= 0; base -= 32) {
            const int r = base + lane;
            int v = r < a.NR ? nxt[r] : a.NR;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_down_sync(0xffffffffu, v, o);
                if (lane + o < 32) v = min(v, y);
            }
            v = min(v, carry);
            if (r < a.NR) nxt[r] = v;
            carry = __shfl_sync(0xffffffffu, v, 0);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = tmem_base;
    uint8_t *Atile = sm;                  // S^T bf16, K-major (rows of other blocks stay zero)
    uint8_t *Mbuf = sm + 2 * kSlab;                              // A_r^T, kChainBufs buffers
    uint8_t *Bbuf = Mbuf + kChainBufs * 2 * kSlab;               // this block's rows of B_r^T (fp32, column quads)
    uint8_t *Estage = Bbuf + kChainBufs * kBlockQuads;           // this block's rows of the entry state
    const int qrow = row * 16;            // byte offset of this thread's row inside a column quad

    float S[32];
#pragma unroll
    for (int jj = 0; jj < 32; ++jj) S[jj] = a.h0 && active ? a.h0[sbase + (int64_t)(cs + jj) * kDim + dv] : 0.f;
    {   // rows of the operand other than this CTA's stay zero
        uint4 *z = reinterpret_cast<uint4 *>(Atile);
        for (int q = tid; q < 2 * (int)kSlab / 16; q += kThreads) z[q] = make_uint4(0u, 0u, 0u, 0u);
    }

    auto next_run = [&](int r) -> int { return r < a.NR ? nxt[r] : a.NR; };
    // thread 0: A_r^T and this block's B_r^T rows of run rn into buffer nb
    auto load_run = [&](int rn, int nb) {
        mbar_arrive_expect_tx(&bar_tma[nb], 2 * kSlab + kBlockQuads);
        tma_load_3d(Mbuf + nb * 2 * kSlab, &tA, 0, (int)((rbase + rn) * kDim), 0, &bar_tma[nb]);
        tma_load_3d(Mbuf + nb * 2 * kSlab + kSlab, &tA, 64, (int)((rbase + rn) * kDim), 0, &bar_tma[nb]);
        tma_load_2d(Bbuf + nb * kBlockQuads, &tB, part * 4 * kChainRows, (int)((rbase + rn) * 32), &bar_tma[nb]);
    };
    int n_loads = 0, n_mma = 0, last = -1;  // thread 0: tiles requested, the last run requested
    if (tid == 0) {
        for (int q = 0; q < kChainBufs - 1; ++q) {
            const int rn = next_run(last + 1);
            if (rn >= a.NR) break;
            load_run(rn, q);
            last = rn;
            ++n_loads;
        }
    }
    const uint32_t idesc = idesc_bf16(128, 128, false, true);
    int used = 0;  // map tiles consumed
    for (int r = 0; r < a.NR; ++r) {
        const int c_lo = r * kRun, c_hi = min(a.C, c_lo + kRun);
        const bool has = nxt[r] == r;
        if (!has) {  // no events: the state only decays (the entry state goes out directly)
            if (active) {
                float4 *ent = reinterpret_cast<float4 *>(a.entry + (rbase + r) * (kDim * kDim)) + 8 * seg * 128 + dv;
#pragma unroll
                for (int v4 = 0; v4 < 8; ++v4)
                    ent[v4 * 128] = make_float4(S[4 * v4], S[4 * v4 + 1], S[4 * v4 + 2], S[4 * v4 + 3]);
            }
            const float f = ex2((float)(Pu[c_hi] - Pu[c_lo]));
#pragma unroll
            for (int jj = 0; jj < 32; ++jj) S[jj] *= f;
            continue;
        }
        if (active) {  // the entering state: fp32 for the entry table, bf16 as the MMA operand
#pragma unroll
            for (int v4 = 0; v4 < 8; ++v4)
                *reinterpret_cast<float4 *>(Estage + (cs / 4 + v4) * 512 + qrow) =
                    make_float4(S[4 * v4], S[4 * v4 + 1], S[4 * v4 + 2], S[4 * v4 + 3]);
#pragma unroll
            for (int k0 = 0; k0 < 32; k0 += 8) st_sw128_8(Atile + slab * kSlab, row, cin + k0, &S[k0]);
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        const int bufi = used % kChainBufs;
        const uint32_t par = (uint32_t)(used / kChainBufs) & 1u;
        if (tid == 0) {
            tma_store_2d(&tE, part * 4 * kChainRows, (int)((rbase + r) * 32), Estage);
            bulk_commit();
            if (!mbar_wait(&bar_tma[bufi], par)) {
                fail(a, &abort_s);
            } else {
                tc_fence_after();
                uint8_t *mt = Mbuf + bufi * 2 * kSlab;
                for (int ks = 0; ks < 8; ++ks)
                    mma_bf16(tbase, kmajor_desc(smem_addr(Atile), ks, kSlab), mnmajor_desc(smem_addr(mt), ks, kSlab),
                             idesc, ks > 0);
                mma_commit(&bar_mma);
                const int rn = next_run(last + 1);
                if (rn < a.NR) {  // the buffer the previous step read (its MMA and B rows are done)
                    load_run(rn, (used + kChainBufs - 1) % kChainBufs);
                    last = rn;
                    ++n_loads;
                }
            }
        }
        __syncthreads();
        if (abort_s) break;
        if (!mbar_wait(&bar_mma, n_mma & 1)) fail(a, &abort_s);
        ++n_mma;
        tc_fence_after();
        if (active) {
            if (tid != 0 && !mbar_wait(&bar_tma[bufi], par)) fail(a, &abort_s);  // B rows visible
            float d0[32];
            tmem_ld32(tmem_addr(tbase, quarter * 32, cs), d0);
            tmem_ld_wait();
            const uint8_t *bsrc = Bbuf + bufi * kBlockQuads + qrow;
#pragma unroll
            for (int v4 = 0; v4 < 8; ++v4) {
                const float4 x = *reinterpret_cast<const float4 *>(bsrc + (cs / 4 + v4) * 512);
                S[4 * v4] = d0[4 * v4] + x.x;
                S[4 * v4 + 1] = d0[4 * v4 + 1] + x.y;
                S[4 * v4 + 2] = d0[4 * v4 + 2] + x.z;
                S[4 * v4 + 3] = d0[4 * v4 + 3] + x.w;
            }
        }
        ++used;
        if (tid == 0) bulk_wait_read();  // the entry store has read the staging tile
        tc_fence_before();
        __syncthreads();
        if (abort_s) break;
    }
    if (!abort_s) {
        if (active) {
#pragma unroll
            for (int jj = 0; jj < 32; ++jj) a.s_final[sbase + (int64_t)(cs + jj) * kDim + dv] = S[jj];
        }
    } else if (tid == 0) {
        for (int u = used + 1; u < n_loads; ++u) mbar_wait(&bar_tma[u % kChainBufs], (u / kChainBufs) & 1);
        mma_commit(&bar_mma);
        mbar_wait(&bar_mma, n_mma & 1);
    }
    if (tid == 0) bulk_wait_read();
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc<128>(tbase);
}

}  // namespace

cudaError_t launch_scan_tc(const Problem &pb, const Workspace &ws, int part) {
    if (pb.R == 0) return cudaSuccess;
    const int NR = (pb.C + kRun - 1) / kRun;
    ScanParams a;
    a.row_pair = ws.row_pair; a.row_ptr = ws.row_ptr; a.ev_chunk = ws.ev_chunk; a.snap_slot = ws.snap_slot;
    a.run_first = ws.run_first;
    a.P = ws.P; a.g = pb.g; a.h0 = pb.h0;
    a.U = (__nv_bfloat16 *)ws.U; a.amap = (__nv_bfloat16 *)ws.amap; a.bmap = ws.bmap; a.entry = ws.entry;
    a.snap = (__nv_bfloat16 *)ws.snap; a.s_final = pb.s_final; a.status = ws.counts + 2;
    a.P_ = pb.P; a.T_ = pb.T; a.Nv = pb.Nv; a.C = pb.C; a.NR = NR;
    a.ev_cap = ws.ev_cap; a.snap_cap = ws.snap_cap;
    CUtensorMap tA;
    const uint64_t amap_rows = (uint64_t)pb.R * 2 * (NR > 0 ? NR : 1) * kDim;
    if (!make_tmap_bf16_3d(&tA, ws.amap, kDim, amap_rows, 1, kDim * 2, amap_rows * kDim * 2, 64, 128, 1, true))
        return cudaErrorInvalidValue;
    if (part == 1) {  // chain
        cudaFuncSetAttribute(scan_chain_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kChainSmem);
        // B_r^T and entry tiles as [quads][512 floats]: a box of 128 floats x 32 quads is one row block
        CUtensorMap tB, tE;
        const uint64_t quads = (uint64_t)pb.R * 2 * (NR > 0 ? NR : 1) * 32;
        if (!make_tmap_f32_2d(&tB, ws.bmap, 512, quads, 2048, 4 * kChainRows, 32) ||
            !make_tmap_f32_2d(&tE, ws.entry, 512, quads, 2048, 4 * kChainRows, 32))
            return cudaErrorInvalidValue;
        return launch_kernel(pb.pdl, scan_chain_kernel, dim3(2 * kChainSplit, pb.R), kThreads, kChainSmem, pb.stream,
                             tA, tB, tE, a);
    }
    if (NR == 0 || pb.C == 0) return cudaSuccess;
    CUtensorMap tW, tK, tU;
    if (!make_tmap_bf16_3d(&tW, ws.W, kDim, (uint64_t)ws.ev_cap * 2 * kChunk, 1, kDim * 2,
                           (uint64_t)ws.ev_cap * 2 * kChunk * kDim * 2, 64, 64, 1, true) ||
        !make_tmap_tokens(&tK, pb.k, pb.Nq, pb.T, pb.B, 64, 64, true) ||
        !make_tmap_headmajor(&tU, ws.U, pb.Nv, pb.T, pb.B, 64, 64, true))
        return cudaErrorInvalidValue;
    cudaFuncSetAttribute(scan_run_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kRunSmem);
    const int fixup = part == 2;
    return launch_kernel(pb.pdl, scan_run_kernel, dim3(NR, fixup ? 2 : 4, pb.R), kThreads, kRunSmem, pb.stream, tW,
                         tK, tU, tA, a, fixup);
}

}  // namespace gdn
